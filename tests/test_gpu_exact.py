"""The mat-vec kernels' own decoders pinned bit for bit, and adversarial
weights through the mat-vec.

* Exact arithmetic.  With power-of-two block scales, small-integer inputs
  and weights of a few significant bits, every product and every partial sum
  of every kernel is exact in binary32, so y must equal the oracle's f64 sum
  exactly -- for every format, on both engines where both apply, on the TMA
  and the plain staging paths, at m = 1, 3, 8 (and 16 / 32 on the
  tensor-core engine).  A slip in any decoder (a code bit, a nibble, a
  sub-block scale or min, the Q6_K window offset) changes y.  The blocks are
  full-range random bytes (every code value and every scale bit) and blocks
  with a single code different from the format's zero (one code lit at a
  time, at a position that moves from block to block and row to row).
* Adversarial weights (random bytes with normal, subnormal, negative and
  large binary16 scales; Q4_K blocks whose mins cancel the scaled codes
  exactly; affine groups whose bias cancels the scaled code) and an infinite
  input, against the oracle at |y - y_ref| <= 1e-4 * sum|w*x| + 1e-7
  (non-finite where the reference is).

Block layouts follow the page's RowExactWeight formats (mlx-native 0.18.0
src/ops/row_exact_matvec.rs, block constants) in the byte order the oracle
uses (tests/golden/dequant_fields.txt pins it).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import quantized_few_row_gb300 as rem
from quantized_few_row_gb300 import inputs
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

FMTS = ["f16", "bf16", "f32", "q8_0", "q5_0", "q4_K", "q6_K"]
TC = ("q8_0", "q5_0", "q6_K")
# tensor-core tile widths: 32 input rows where a scale block is 32 values, 16 for Q6_K
TC_MAX = {"q8_0": 32, "q5_0": 32, "q6_K": 16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rem.build()
    rem.load()
    torch.cuda.init()


def _pow2_h(g, shape, lo, hi):
    """binary16 bit patterns of 2^e, e uniform in [lo, hi]."""
    e = g.integers(lo, hi + 1, size=shape)
    return ((e + 15) << 10).astype(np.uint16)


def _put16(blocks, off, h):
    blocks[..., off:off + 2] = h.astype(np.uint16)[..., None].view(np.uint8).reshape(*h.shape, 2)


def exact_weights(fmt, rows, k, seed, lit=False):
    """Weight bytes whose values have few significant bits (see the module
    doc) and the small-integer input range that keeps every sum exact."""
    g = np.random.Generator(np.random.PCG64(seed))
    if fmt in ("f16", "bf16", "f32"):
        unit = {"f16": 2.0 ** -6, "bf16": 2.0 ** -4, "f32": 2.0 ** -10}[fmt]
        top = {"f16": 64, "bf16": 64, "f32": 1024}[fmt]
        v = g.integers(-top, top + 1, size=(rows, k)).astype(np.float64) * unit
        if lit:
            keep = np.zeros((rows, k), bool)
            keep[np.arange(rows), (np.arange(rows) * 7) % k] = True
            v = np.where(keep, np.where(v == 0, unit, v), 0.0)
        v = v.astype(np.float32)
        if fmt == "f16":
            return v.astype(np.float16).view(np.uint8).reshape(rows, -1), 8
        if fmt == "bf16":
            return (v.view(np.uint32) >> 16).astype(np.uint16).view(np.uint8).reshape(rows, -1), 8
        return v.view(np.uint8).reshape(rows, -1), 8
    bb, bv = oracle.block_bytes(fmt), oracle.block_values(fmt)
    nb = k // bv
    blocks = g.integers(0, 256, size=(rows, nb, bb), dtype=np.uint8)
    pos = (np.arange(rows)[:, None] * 5 + np.arange(nb)[None, :] * 3) % bv   # the lit element of each block
    if fmt == "q8_0":
        _put16(blocks, 0, _pow2_h(g, (rows, nb), -3, 1))
        if lit:
            q = blocks[:, :, 2:].copy()
            blocks[:, :, 2:] = 0
            r, b = np.meshgrid(np.arange(rows), np.arange(nb), indexing="ij")
            lit_q = q[r, b, pos]
            blocks[r, b, 2 + pos] = np.where(lit_q == 0, 1, lit_q)
        return blocks.reshape(rows, -1), 8
    if fmt == "q5_0":
        _put16(blocks, 0, _pow2_h(g, (rows, nb), -3, 1))
        if lit:   # every code 16 (weight 0: nibble 0, high bit 1) but one
            blocks[:, :, 2:6] = 0xFF
            blocks[:, :, 6:] = 0
            for r in range(rows):
                for b in range(nb):
                    e, q = int(pos[r, b]), int(g.integers(0, 32))
                    q = 17 if q == 16 else q
                    qh = int.from_bytes(blocks[r, b, 2:6].tobytes(), "little")
                    qh = (qh & ~(1 << e)) | ((q >> 4) << e)
                    blocks[r, b, 2:6] = np.frombuffer(qh.to_bytes(4, "little"), np.uint8)
                    if e < 16:
                        blocks[r, b, 6 + e] = (blocks[r, b, 6 + e] & 0xF0) | (q & 0xF)
                    else:
                        blocks[r, b, 6 + e - 16] = (blocks[r, b, 6 + e - 16] & 0x0F) | ((q & 0xF) << 4)
        return blocks.reshape(rows, -1), 8
    if fmt == "q4_K":
        _put16(blocks, 0, _pow2_h(g, (rows, nb), -3, 0))
        _put16(blocks, 2, _pow2_h(g, (rows, nb), -3, 0))
        if lit:   # every min 0 (scale bytes 4..7 and the high nibbles of 8..11 clear), every code 0 but one
            blocks[:, :, 8:12] = 0
            blocks[:, :, 12:16] &= np.uint8(0x0F)
            blocks[:, :, 16:] = 0
            for r in range(rows):
                for b in range(nb):
                    e = int(pos[r, b])
                    c, hi, l = e // 64, (e % 64) >= 32, e % 32
                    q = int(g.integers(1, 16))
                    idx = 16 + 32 * c + l
                    blocks[r, b, idx] = (q << 4) if hi else q
        return blocks.reshape(rows, -1), 2
    if fmt == "q6_K":
        _put16(blocks, 208, _pow2_h(g, (rows, nb), -2, 0))
        if lit:   # every code 32 (low nibble 0, high bits 2) but one
            blocks[:, :, 0:128] = 0
            blocks[:, :, 128:192] = 0xAA
            for r in range(rows):
                for b in range(nb):
                    e = int(pos[r, b])
                    h, t, l = e // 128, (e % 128) // 32, e % 32
                    q = int(g.integers(0, 64))
                    q = 33 if q == 32 else q
                    li = 64 * h + l + 32 * (t & 1)
                    if t < 2:
                        blocks[r, b, li] = (blocks[r, b, li] & 0xF0) | (q & 0xF)
                    else:
                        blocks[r, b, li] = (blocks[r, b, li] & 0x0F) | ((q & 0xF) << 4)
                    hi = 128 + 32 * h + l
                    keep = (~(3 << (2 * t))) & 0xFF
                    blocks[r, b, hi] = (int(blocks[r, b, hi]) & keep) | ((q >> 4) << (2 * t))
        return blocks.reshape(rows, -1), 1
    raise ValueError(fmt)


def _engines(fmt):
    return [rem.ENGINE_SIMT, rem.ENGINE_TC] if fmt in TC else [rem.ENGINE_SIMT]


def _offsets(fmt):
    """Weight byte offsets: 16-byte aligned (TMA staging) and, where the
    format's alignment allows, an offset that forces the plain staging path."""
    return [0] + {"q4_K": [], "f16": [8], "bf16": [8], "f32": [4]}.get(fmt, [2])


CASES = [(f, e, lit) for f in FMTS for e in _engines(f) for lit in (False, True)]


@pytest.mark.parametrize("fmt,engine,lit", CASES,
                         ids=[f"{f}-{'tc' if e else 'simt'}-{'lit' if l else 'full'}" for f, e, l in CASES])
def test_exact_arithmetic_is_bitwise(fmt, engine, lit):
    n = 150                                          # two tiles of 128 rows with a ragged tail
    k = {"f16": 520, "bf16": 520, "f32": 520}.get(fmt, 512)
    w, xmax = exact_weights(fmt, n, k, 700 + FMTS.index(fmt) + (50 if lit else 0), lit)
    ms = [1, 3, 8] + ([12, 16, 23] + ([29] if TC_MAX[fmt] == 32 else []) if engine == rem.ENGINE_TC else [])
    mmax = max(ms)
    x = inputs.small_ints((mmax, k), 701, -xmax, xmax)
    y_ref, _ = oracle.matvec(w, fmt, n, k, 1, x, mmax, k, 0)
    for off in _offsets(fmt):
        for m in ms:
            for split in (0, 3):
                sc = rem.Schedule(engine=engine, split=split)
                y = H.run_sched(w, fmt, n, k, 1, x[:m], m, k, 0, n, 0, m * n, sc, w_offset=off, tail=64)
                got = y[:m * n].reshape(m, n).astype(np.float64)
                bad = np.argwhere(got != y_ref[0, :m])
                assert bad.size == 0, (off, m, split, bad[:5].tolist(),
                                       [(got[tuple(b)], y_ref[0, :m][tuple(b)]) for b in bad[:3]])
                assert np.all(y[m * n:] == H.CANARY), (off, m, split)


# ---------------------------------------------------------------- adversarial weights

ADV = [(f, e) for f in FMTS for e in _engines(f)]


@pytest.mark.parametrize("fmt,engine", ADV, ids=[f"{f}-{'tc' if e else 'simt'}" for f, e in ADV])
def test_adversarial_blocks_match_oracle(fmt, engine):
    n = 140
    k = {"f16": 520, "bf16": 520, "f32": 520}.get(fmt, 1024)
    w = H.adversarial_blocks(fmt, n, k, 720)
    if fmt in ("bf16", "f32"):   # keep |w| below 2^40 so sums stay far from binary32 overflow
        if fmt == "bf16":
            h = w.view(np.uint16)
            ex = (h >> 7) & 0xFF
            h[ex > 127 + 40] = (h[ex > 127 + 40] & 0x807F) | np.uint16((127 + 40) << 7)
        else:
            u = w.view(np.uint32)
            ex = (u >> 23) & 0xFF
            u[ex > 127 + 40] = (u[ex > 127 + 40] & 0x807FFFFF) | np.uint32((127 + 40) << 23)
    x = inputs.activations(8, k, 721)
    y_ref, a_ref = oracle.matvec(w, fmt, n, k, 1, x, 8, k, 0)
    for off in _offsets(fmt):
        for m in (1, 5, 8):
            y = H.run_sched(w, fmt, n, k, 1, x[:m], m, k, 0, n, 0, m * n, rem.Schedule(engine=engine), w_offset=off)
            H.assert_close_to_oracle(y.reshape(1, m, n), y_ref[:, :m], a_ref[:, :m], f"{fmt} off={off} m={m}")


def _q4k_cancelling(rows, nsb, seed):
    """Q4_K super-blocks whose every sub-block has sc = 4, mn = 60 and d = dmin,
    so a code of 15 dequantizes to exactly zero; a few codes per row differ.
    The scale bytes encode (sc, mn) = (4, 60) for all 8 sub-blocks."""
    g = np.random.Generator(np.random.PCG64(seed))
    blocks = np.zeros((rows, nsb, 144), np.uint8)
    d = g.integers(0x0400, 0x7800, size=(rows, nsb)).astype(np.uint16)   # normal, not powers of two
    _put16(blocks, 0, d)
    _put16(blocks, 2, d)
    blocks[:, :, 4:8] = 4
    blocks[:, :, 8:12] = 252
    blocks[:, :, 12:16] = 196
    blocks[:, :, 16:] = 0xFF
    for r in range(rows):
        for _ in range(3):
            b, i = int(g.integers(0, nsb)), int(g.integers(16, 144))
            blocks[r, b, i] = int(g.integers(0, 256))
    return blocks.reshape(rows, -1)


def test_q4k_cancelling_mins_match_oracle():
    n, k = 96, 1024
    w = _q4k_cancelling(n, k // 256, 730)
    deq = oracle.dequantize(w, "q4_K", n, k)
    assert np.mean(deq == 0.0) > 0.98      # nearly every weight is an exact cancellation
    x = inputs.activations(8, k, 731) * np.float32(1000.0)
    y_ref, a_ref = oracle.matvec(w, "q4_K", n, k, 1, x, 8, k, 0)
    for m in (1, 8):
        for layout in (0, 1, 2):
            if layout == 2 and m < 2:
                continue
            y = H.run_sched(w, "q4_K", n, k, 1, x[:m], m, k, 0, n, 0, m * n,
                            rem.Schedule(layout=layout, engine=rem.ENGINE_SIMT))
            H.assert_close_to_oracle(y.reshape(1, m, n), y_ref[:, :m], a_ref[:, :m], f"q4_K cancel m={m} l={layout}")


def test_affine_cancelling_bias_matches_oracle():
    bits, gs, n, k = 4, 64, 96, 1024
    wt = rem.affine_wtype(bits, gs)
    g = np.random.Generator(np.random.PCG64(740))
    ng = k // gs
    # scale with 7 significant bits, bias = -7 * scale exactly: a code of 7 is an exact zero
    mant = g.integers(64, 128, size=(n, ng)).astype(np.float64)
    scale = (mant * 2.0 ** g.integers(-14, -8, size=(n, ng))).astype(np.float16)
    bias = (-7.0 * scale.astype(np.float64)).astype(np.float16)
    assert np.all(bias.astype(np.float64) == -7.0 * scale.astype(np.float64))
    codes = np.full((n, k * bits // 32), 0x77777777, np.uint32)
    for r in range(n):
        for _ in range(3):
            i = int(g.integers(0, codes.shape[1]))
            codes[r, i] = np.uint32(g.integers(0, 2 ** 32, dtype=np.uint64))
    sc, bi = scale.view(np.uint16), bias.view(np.uint16)
    x = inputs.activations(8, k, 741) * np.float32(1000.0)
    y_ref, a_ref = oracle.affine_matvec(codes, sc, bi, bits, gs, n, k, 1, x, 8, k, 0)
    dev = H.dev()
    cd = torch.from_numpy(codes.view(np.int32).reshape(-1)).to(dev)
    sd = torch.from_numpy(sc.view(np.int16).reshape(-1)).to(dev)
    bd = torch.from_numpy(bi.view(np.int16).reshape(-1)).to(dev)
    xd = H.to_dev_f32(x)
    for m in (1, 8):
        yd = H.canary(m * n)
        rem.check(rem.rem_matvec_affine(cd, sd, bd, wt, n, k, 1, xd, m, k, 0, yd, n, 0, 0))
        torch.cuda.synchronize()
        H.assert_close_to_oracle(yd.cpu().numpy().reshape(1, m, n), y_ref[:, :m], a_ref[:, :m], f"affine m={m}")


@pytest.mark.parametrize("fmt,engine", ADV, ids=[f"{f}-{'tc' if e else 'simt'}" for f, e in ADV])
def test_infinite_input_stays_in_its_row(fmt, engine):
    n, k, m = 70, {"f16": 520, "bf16": 520, "f32": 520}.get(fmt, 512), 3
    w, x = H.contiguous(fmt, n, k, m, 750, 751)
    x[1, 33] = np.inf
    x[2, 100] = -np.inf
    y_ref, a_ref = oracle.matvec(w, fmt, n, k, 1, x, m, k, 0)
    y = H.run_sched(w, fmt, n, k, 1, x, m, k, 0, n, 0, m * n, rem.Schedule(engine=engine)).reshape(1, m, n)
    H.assert_close_to_oracle(y, y_ref, a_ref, f"{fmt} inf")
    assert np.all(np.isfinite(y[0, 0]))
    # a weight row that is not zero at the infinite input gives an infinity of the reference's sign
    wf = oracle.dequantize(w, fmt, n, k)
    sel = wf[:, 33] != 0
    assert np.all(np.isinf(y[0, 1][sel]) == np.isinf(y_ref[0, 1][sel]))
    assert np.all(np.sign(y[0, 1][sel & np.isinf(y_ref[0, 1])]) == np.sign(y_ref[0, 1][sel & np.isinf(y_ref[0, 1])]))


# ---------------------------------------------------------------- the tensor-core engine

@pytest.mark.parametrize("fmt", TC)
def test_tc_rows_bitwise_equal_for_every_m(fmt):
    """On the tensor-core engine row j is the same bits for every m, including
    launches of 9..16 and 17..32 input rows (the wider tiles) and calls of
    more rows than one launch takes, and equal to the oracle within
    tolerance."""
    n, k = 200, 1024
    mmax = 40
    w, x = H.contiguous(fmt, n, k, mmax, 760, 761)
    y_ref, a_ref = oracle.matvec(w, fmt, n, k, 1, x, mmax, k, 0)
    tc = rem.Schedule(engine=rem.ENGINE_TC)
    alone = [H.run_sched(w, fmt, n, k, 1, x[j:j + 1], 1, k, 0, n, 0, n, tc) for j in range(mmax)]
    for m in (1, 2, 3, 5, 8, 9, 12, 16, 17, 24, 31, 32, 40):
        y = H.run_sched(w, fmt, n, k, 1, x[:m], m, k, 0, n, 0, m * n, tc).reshape(m, n)
        H.assert_close_to_oracle(y[None], y_ref[:, :m], a_ref[:, :m], f"{fmt} m={m}")
        for j in range(m):
            assert np.array_equal(y[j].view(np.uint32), alone[j].view(np.uint32)), (m, j)


@pytest.mark.parametrize("fmt", TC)
def test_tc_many_rows_one_pass_per_group(fmt):
    """rem_matvec_many on the tensor-core engine: groups of up to 16 input
    rows, each row bitwise the row of an m = 1 call."""
    n, k, m = 130, 512, 40
    w, x = H.contiguous(fmt, n, k, m, 762, 763)
    # the thread's default schedule takes every call of this test to the
    # tensor cores (Q6_K goes there by default; Q8_0 and Q5_0 on request)
    rem.check(rem.rem_set_thread_schedule(rem.Schedule(engine=rem.ENGINE_TC)))
    try:
        wh, wp = H.to_dev_bytes(w)
        xd = H.to_dev_f32(x)
        yd = H.canary(m * n + 16)
        rem.check(rem.rem_matvec_many(wp, fmt, n, k, 1, xd, m, k, 0, yd, n, 0, 0))
        torch.cuda.synchronize()
        assert "engine=tc" in rem.rem_last_plan()
        y = yd.cpu().numpy()
        assert np.all(y[m * n:] == H.CANARY)
        y = y[:m * n].reshape(m, n)
        y_ref, a_ref = oracle.matvec(w, fmt, n, k, 1, x, m, k, 0)
        H.assert_close_to_oracle(y[None], y_ref, a_ref, f"{fmt} many")
        for j in (0, 17, 39):
            one = H.run_matvec(w, fmt, n, k, 1, x[j:j + 1], 1, k, 0, n, 0, n, use_ex=False)
            assert np.array_equal(y[j].view(np.uint32), one.view(np.uint32)), j
    finally:
        rem.check(rem.rem_set_thread_schedule(None))
