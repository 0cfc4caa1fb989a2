"""GPU parity of the affine group-quantized formats (3-, 4-, 5-, 6- or 8-bit
codes, binary16 scale and bias per group of 32/64/128) through
rem_matvec_affine and rem_dequantize_affine, against the oracle's affine
dequantizer and f64 dot.  Test weights come from the oracle's affine
quantizer, from random codes and finite scales, or (for the bitwise test)
from codes, power-of-two scales, short biases and small-integer inputs whose
every sum is exact in binary32; nothing the CUDA path computes feeds the
oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import quantized_few_row_gb300 as rem
from quantized_few_row_gb300 import inputs
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

TYPES = [(b, g) for b in (3, 4, 5, 6, 8) for g in (32, 64, 128)]
IDS = [f"a{b}_g{g}" for b, g in TYPES]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rem.build()
    rem.load()


def _dev(a, offset=0):
    return H.to_dev_bytes(np.ascontiguousarray(a).view(np.uint8), offset)


def _random_affine(rows, k, bits, gs, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    codes = g.integers(0, 2 ** 32, size=(rows, k * bits // 32), dtype=np.uint64).astype(np.uint32)
    ng = k // gs
    sc = g.integers(0, 0x7C00, size=(rows, ng)).astype(np.uint16)          # finite
    sc |= (g.integers(0, 2, size=(rows, ng)) << 15).astype(np.uint16)      # either sign
    sc[:, ::5] &= 0x03FF                                                   # some subnormal
    bi = g.integers(0, 0x7C00, size=(rows, ng)).astype(np.uint16)
    bi |= (g.integers(0, 2, size=(rows, ng)) << 15).astype(np.uint16)
    return codes, sc, bi


def _run(codes, sc, bi, wt, n, k, batch, x, m, xrs, xbs, yrs, ybs, ylen, offset=0):
    ch, cp = _dev(codes, offset)
    sh, sp = _dev(sc)
    bh, bp = _dev(bi)
    xd = H.to_dev_f32(x)
    yd = H.canary(ylen)
    rem.check(rem.rem_matvec_affine(cp, sp, bp, wt, n, k, batch, xd, m, xrs, xbs, yd, yrs, ybs, 0))
    torch.cuda.synchronize()
    return yd.cpu().numpy()


@pytest.mark.parametrize("bits,gs", TYPES, ids=IDS)
def test_affine_dequantize_bit_exact(bits, gs):
    rows, k = 19, 1024
    wt = rem.affine_wtype(bits, gs)
    for codes, sc, bi in (oracle.affine_quantize(inputs.weights(rows, k, 500), bits, gs),
                          _random_affine(rows, k, bits, gs, 501)):
        ref = oracle.affine_dequantize(codes, sc, bi, bits, gs, rows, k)
        (ch, cp), (sh, sp), (bh, bp) = _dev(codes), _dev(sc), _dev(bi)
        out = H.canary(rows * k)
        rem.check(rem.rem_dequantize_affine(cp, sp, bp, wt, rows, k, out))
        torch.cuda.synchronize()
        got = out.cpu().numpy().reshape(rows, k)
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


@pytest.mark.parametrize("bits,gs", TYPES, ids=IDS)
@pytest.mark.parametrize("m", [1, 2, 5, 8])
def test_affine_matvec_matches_oracle(bits, gs, m):
    wt = rem.affine_wtype(bits, gs)
    for si, (n, k) in enumerate([(103, 1024), (40, 256), (150, 4096)]):
        codes, sc, bi = oracle.affine_quantize(inputs.weights(n, k, 510 + si), bits, gs)
        x = inputs.activations(m, k, 610 + si)
        y = _run(codes, sc, bi, wt, n, k, 1, x, m, k, 0, n, 0, m * n)
        y_ref, a_ref = oracle.affine_matvec(codes, sc, bi, bits, gs, n, k, 1, x, m, k, 0)
        H.assert_close_to_oracle(y.reshape(1, m, n), y_ref, a_ref, f"a{bits} g{gs} n={n} k={k} m={m}")


def _pack_stream(q, bits):
    """Codes [rows, k] (ints < 2^bits) packed as each row's little-endian bit
    stream, code i at stream bits [bits*i, bits*i + bits); uint32 words."""
    rows, k = q.shape
    bitpos = np.arange(k * bits)
    stream = (q[:, bitpos // bits] >> (bitpos % bits)) & 1                 # [rows, k*bits]
    by = np.packbits(stream.astype(np.uint8).reshape(rows, -1, 8), axis=2, bitorder="little").reshape(rows, -1)
    return np.ascontiguousarray(by).view("<u4").astype(np.uint32)


def _exact_affine(rows, k, bits, gs, seed, lit):
    """Codes, power-of-two binary16 scales (s * (2^bits - 1) <= 128) and
    biases that are multiples of 1/16 in [-64, 64], so every weight is a
    multiple of 1/16 below 192 in magnitude; with inputs in [-4, 4] and
    k = 512 every partial sum is an integer multiple of 1/16 below 2^23 and
    exact in binary32, in any order.  lit: one nonzero code per group."""
    g = np.random.Generator(np.random.PCG64(seed))
    ng = k // gs
    q = g.integers(0, 2 ** bits, size=(rows, k))
    if lit:
        keep = np.zeros((rows, k), bool)
        keep[np.arange(rows)[:, None], np.arange(ng)[None, :] * gs + (np.arange(rows)[:, None] * 7) % gs] = True
        q = np.where(keep, np.maximum(q, 1), 0)
    e = g.integers(-4, 8 - bits, size=(rows, ng))
    sc = ((e + 15) << 10).astype(np.uint16)
    bias = g.integers(-1024, 1025, size=(rows, ng)).astype(np.float64) / 16.0
    bi = bias.astype(np.float16).view(np.uint16)
    return _pack_stream(q, bits), sc, bi


@pytest.mark.parametrize("bits,gs", TYPES, ids=IDS)
@pytest.mark.parametrize("lit", [False, True], ids=["full", "lit"])
def test_affine_exact_arithmetic_is_bitwise(bits, gs, lit):
    """Every sum exact: y equals the oracle bit for bit, which pins the
    kernel's own code extraction and scale/bias step, on the TMA and the
    plain staging path."""
    wt = rem.affine_wtype(bits, gs)
    n, k = 130, 512
    codes, sc, bi = _exact_affine(n, k, bits, gs, 550 + bits, lit)
    x = np.random.Generator(np.random.PCG64(551)).integers(-4, 5, size=(8, k)).astype(np.float32)
    y_ref, _ = oracle.affine_matvec(codes, sc, bi, bits, gs, n, k, 1, x, 8, k, 0)
    want = y_ref.astype(np.float32)
    assert np.array_equal(want.astype(np.float64), y_ref)            # the exact sums are binary32 values
    for off in (0, 4):
        for m in (1, 5, 8):
            y = _run(codes, sc, bi, wt, n, k, 1, x[:m], m, k, 0, n, 0, m * n, offset=off).reshape(1, m, n)
            assert np.array_equal(y.view(np.uint32), want[:, :m].view(np.uint32)), (off, m)


@pytest.mark.parametrize("bits,gs", [(4, 64), (8, 32), (3, 32), (5, 128), (6, 64)],
                         ids=["a4_g64", "a8_g32", "a3_g32", "a5_g128", "a6_g64"])
def test_affine_rows_exact_across_m_packing_and_paths(bits, gs):
    """Row j of every m equals the row computed alone; the plain staging path
    (codes not 16-byte aligned) equals the TMA path bit for bit."""
    wt = rem.affine_wtype(bits, gs)
    n, k = 200, 2048
    codes, sc, bi = oracle.affine_quantize(inputs.weights(n, k, 520), bits, gs)
    x = inputs.activations(8, k, 620)
    alone = [_run(codes, sc, bi, wt, n, k, 1, x[j:j + 1], 1, k, 0, n, 0, n) for j in range(8)]
    for m in (2, 4, 7, 8):
        y = _run(codes, sc, bi, wt, n, k, 1, x[:m], m, k, 0, n, 0, m * n).reshape(m, n)
        for j in range(m):
            assert np.array_equal(y[j].view(np.uint32), alone[j].view(np.uint32)), (m, j)
    plain = _run(codes, sc, bi, wt, n, k, 1, x, 8, k, 0, n, 0, 8 * n, offset=4).reshape(8, n)
    tma = _run(codes, sc, bi, wt, n, k, 1, x, 8, k, 0, n, 0, 8 * n).reshape(8, n)
    assert np.array_equal(plain.view(np.uint32), tma.view(np.uint32))


@pytest.mark.parametrize("bits,gs", [(4, 32), (5, 32)], ids=["a4_g32", "a5_g32"])
def test_affine_grouped_token_major(bits, gs):
    wt = rem.affine_wtype(bits, gs)
    G, n, k, m = 3, 96, 512, 5
    codes, sc, bi = oracle.affine_quantize(inputs.weights(G * n, k, 530), bits, gs)
    x = inputs.activations(m, G * k, 630)
    y = _run(codes, sc, bi, wt, n, k, G, x, m, G * k, k, G * n, n, m * G * n)
    y_ref, a_ref = oracle.affine_matvec(codes, sc, bi, bits, gs, n, k, G, x, m, G * k, k)
    H.assert_close_to_oracle(H.gather_y(y, G, m, n, G * n, n), y_ref, a_ref, "affine grouped")


@pytest.mark.parametrize("bits,gs,k", [(4, 64, 320), (4, 32, 288), (4, 128, 640), (8, 32, 96), (8, 32, 224),
                                       (8, 64, 192), (3, 32, 288), (5, 64, 320), (6, 128, 384), (6, 32, 96),
                                       (3, 128, 640)])
@pytest.mark.parametrize("m", [1, 3, 8])
def test_affine_partial_last_chunk(bits, gs, k, m):
    """k a multiple of the group size but not of the staged chunk (256 4-bit,
    128 8-bit or 256 3-, 5- or 6-bit values): the groups past k read no scale
    or bias and add
    nothing.  The scale and bias arrays are followed by NaN halves on the
    device, so a read past the last row's groups would show as NaN."""
    wt = rem.affine_wtype(bits, gs)
    n = 37
    codes, sc, bi = oracle.affine_quantize(inputs.weights(n, k, 540), bits, gs)
    x = inputs.activations(m, k, 640)
    guard = np.full(64, 0x7E00, dtype=np.uint16)
    ch, cp = _dev(codes)
    sh, sp = _dev(np.concatenate([sc.reshape(-1), guard]))
    bh, bp = _dev(np.concatenate([bi.reshape(-1), guard]))
    xd = H.to_dev_f32(x)
    yd = H.canary(m * n)
    rem.check(rem.rem_matvec_affine(cp, sp, bp, wt, n, k, 1, xd, m, k, 0, yd, n, 0, 0))
    torch.cuda.synchronize()
    y = yd.cpu().numpy().reshape(1, m, n)
    y_ref, a_ref = oracle.affine_matvec(codes, sc, bi, bits, gs, n, k, 1, x, m, k, 0)
    assert np.all(np.isfinite(y))
    H.assert_close_to_oracle(y, y_ref, a_ref, f"a{bits} g{gs} k={k} m={m}")
