"""Pins of the CPU oracle against facts that do not come from the oracle.

* block sizes / row_bytes: the constants printed in mlx-native 0.18.0
  src/ops/row_exact_matvec.rs (*_BLOCK_* constants, RowExactWeight::row_bytes);
* decode layout: hand-derived single-block cases in golden/dequant_fields.txt;
* fp16 conversions: numpy / torch library conversions;
* quantize -> dequantize round trip: the half-step bound of round-to-nearest;
* the f64 dot: torch / numpy library products, exact integer arithmetic,
  one-hot weights and exact rational brute force on tiny shapes.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from quantized_few_row_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dequant_fields.txt")

# Printed on the page: Q8_0 32 values / 34 B, QK_K 256 values, Q4_K 144 B,
# Q6_K 210 B, Q5_0 32 values / 22 B; F16 rows are 2*k bytes.
PRINTED = {"f16": (1, 2), "q8_0": (32, 34), "q4_K": (256, 144), "q6_K": (256, 210), "q5_0": (32, 22)}


@pytest.mark.parametrize("fmt", list(PRINTED))
def test_block_constants(orc, fmt):
    values, nbytes = PRINTED[fmt]
    assert orc.block_values(fmt) == values
    assert orc.block_bytes(fmt) == nbytes
    for k in (256, 512, 4096, 14336):
        assert orc.row_bytes(fmt, k) == (k // values) * nbytes


def test_row_bytes_of_the_workloads(orc):
    # row sizes the workloads imply (k = 4096): 4352, 2304, 3360, 2816 B
    assert orc.row_bytes("q8_0", 4096) == 4352
    assert orc.row_bytes("q4_K", 4096) == 2304
    assert orc.row_bytes("q6_K", 4096) == 3360
    assert orc.row_bytes("q5_0", 4096) == 2816
    assert orc.row_bytes("f16", 512) == 1024


# ---------------------------------------------------------------- fp16

def test_h2f_all_patterns_match_library(orc):
    import torch
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.h2f(h)
    ref_np = h.view(np.float16).astype(np.float32)
    ref_t = torch.from_numpy(h.view(np.float16).copy()).float().numpy()
    nan = np.isnan(ref_np)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref_np[~nan].view(np.uint32))
    assert np.array_equal(ours[~nan].view(np.uint32), ref_t[~nan].view(np.uint32))


def _f32_probe_values():
    g = np.random.Generator(np.random.PCG64(7))
    parts = [
        g.standard_normal(20000).astype(np.float32) * np.float32(0.02),
        g.standard_normal(20000).astype(np.float32) * np.float32(1e-5),   # fp16 subnormal range
        (g.standard_normal(20000) * 1000).astype(np.float32),
        (g.random(5000) * 70000).astype(np.float32),                     # around overflow
    ]
    # exact halfway points between neighbouring fp16 values
    h = g.integers(0, 0x7BFF, 5000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    parts.append(((lo + hi) / 2).astype(np.float32))
    v = np.concatenate(parts)
    return np.concatenate([v, -v, np.array([0.0, -0.0, np.inf, -np.inf], np.float32)])


def test_f2h_nearest_even_matches_library(orc):
    v = _f32_probe_values()
    ours = orc.f2h(v, "rn")
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_f2h_toward_plus_inf_is_smallest_fp16_not_below(orc):
    v = _f32_probe_values()
    ours = orc.f2h(v, "ru").view(np.float16)
    with np.errstate(over="ignore"):
        rn = v.astype(np.float16)
        below = rn.astype(np.float64) < v.astype(np.float64)
        expect = rn.copy()
        expect[below] = np.nextafter(rn[below], np.float16(np.inf))
    # a negative value past the range rounds toward +inf to the largest finite magnitude
    neg_over = (v < -65504) & np.isfinite(v)
    expect[neg_over] = np.float16(-65504)
    assert np.array_equal(ours.view(np.uint16), expect.view(np.uint16))
    assert np.all(ours.astype(np.float64)[np.isfinite(v)] >= v[np.isfinite(v)].astype(np.float64))


# ---------------------------------------------------------------- decode layout

FIELDS = {  # name: (byte offset, element size, signed)
    "q8_0": {"d": (0, 2, False), "qs": (2, 1, True)},
    "q5_0": {"d": (0, 2, False), "qh": (2, 4, False), "qs": (6, 1, False)},
    "q4_K": {"d": (0, 2, False), "dmin": (2, 2, False), "scales": (4, 1, False), "qs": (16, 1, False)},
    "q6_K": {"ql": (0, 1, False), "qh": (128, 1, False), "sc": (192, 1, True), "d": (208, 2, False)},
    "f16": {"h": (0, 2, False)},
}
BLOCK = {"q8_0": (32, 34), "q5_0": (32, 22), "q4_K": (256, 144), "q6_K": (256, 210), "f16": (4, 8)}


def _num(tok):
    tok = tok.strip()
    if tok in ("inf", "-inf", "nan"):
        return float(tok)
    return Fraction(tok)


def _cases():
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fmt, assigns, default, exc = [p.strip() for p in line.split("|")]
            yield fmt, assigns, default, exc


def _idx_range(s):
    if ".." in s:
        a, b = s.split("..")
        return range(int(a), int(b) + 1)
    return range(int(s), int(s) + 1)


def _build_block(fmt, assigns):
    nvals, nbytes = BLOCK[fmt]
    blk = bytearray(nbytes)
    for tok in assigns.split():
        lhs, rhs = tok.split("=")
        val = int(rhs, 0)
        if "[" in lhs:
            name, idx = lhs[:-1].split("[")
            idxs = _idx_range(idx)
        else:
            name, idxs = lhs, range(0, 1)
        off, size, signed = FIELDS[fmt][name]
        for i in idxs:
            blk[off + size * i: off + size * (i + 1)] = val.to_bytes(size, "little", signed=signed)
    return np.frombuffer(bytes(blk), dtype=np.uint8), nvals


@pytest.mark.parametrize("case", list(_cases()), ids=lambda c: f"{c[0]}:{c[1]}")
def test_decode_golden(orc, case):
    fmt, assigns, default, exc = case
    blk, nvals = _build_block(fmt, assigns)
    got = orc.dequantize(blk, fmt, 1, nvals)[0]
    expect = [_num(default)] * nvals
    for tok in exc.split():
        lhs, rhs = tok.split("=")
        for i in _idx_range(lhs):
            expect[i] = _num(rhs)
    for i, (g, e) in enumerate(zip(got, expect)):
        if isinstance(e, float) and np.isnan(e):
            assert np.isnan(g), (i, g)
        elif isinstance(e, float):
            assert g == e, (i, g, e)
        else:
            assert Fraction(float(g)) == e, (i, float(g), e)


def test_q8_0_unit_scale_returns_codes(orc):
    codes = inputs.uniform_bytes(32 * 64, 11).view(np.int8).reshape(64, 32)
    blocks = np.zeros((64, 34), np.uint8)
    blocks[:, 0:2] = np.frombuffer(np.uint16(0x3C00).tobytes(), np.uint8)
    blocks[:, 2:] = codes.view(np.uint8)
    got = orc.dequantize(blocks.reshape(-1), "q8_0", 1, 64 * 32)[0]
    assert np.array_equal(got, codes.reshape(-1).astype(np.float32))


# ---------------------------------------------------------------- round trip

def _step_bound(orc, fmt, v, blocks):
    """Per-element half-step bound (1 + 2^-10) * step / 2 from the stored scales."""
    rows, k = v.shape
    bb = blocks.reshape(rows, -1)
    if fmt == "q8_0":
        d = orc.h2f(bb.reshape(rows, k // 32, 34)[:, :, 0:2].copy().view(np.uint16)[..., 0])
        step = np.repeat(np.abs(d), 32, axis=1)
        return step / 2
    if fmt == "q5_0":
        d = orc.h2f(bb.reshape(rows, k // 32, 22)[:, :, 0:2].copy().view(np.uint16)[..., 0])
        step = np.repeat(np.abs(d), 32, axis=1)
        # d = vmax / -16 sends the largest magnitude to code 0; values on the
        # other side past 15.5 steps clamp at code 31 (+15 steps).  Their
        # error is at most |vmax| - 15|d| <= |d| * 16 / (1 - 2^-11) - 15|d|
        # (fp16 rounding of d), i.e. just over one step.
        dd = np.repeat(d, 32, axis=1).astype(np.float64)
        clamped = v.astype(np.float64) / np.where(dd == 0, 1, dd) > 15.5
        return np.where(clamped, step * (1 + 2.0 ** -6), step / 2)
    # K-quants: step = d*sc of the element's sub-block, recovered from two
    # decoded codes differing by one, using the oracle's decoder on probes.
    raise AssertionError


@pytest.mark.parametrize("fmt", ["q8_0", "q5_0"])
def test_round_trip_half_step_32(orc, fmt):
    v = inputs.weights(64, 1024, 21)
    v[3] *= 100.0      # a row of large values
    v[5, :32] = 0.0    # an all-zero block
    v[7, :32] = 0.01   # a constant block
    blocks = orc.quantize(v, fmt)
    back = orc.dequantize(blocks, fmt, 64, 1024)
    bound = _step_bound(orc, fmt, v, blocks) * (1 + 2.0 ** -10)
    assert np.all(np.abs(back.astype(np.float64) - v) <= bound + 1e-30)


def _k_scales(orc, fmt, blocks, rows, k):
    """Sub-block step d*sc per element, from the stored header fields."""
    nb = k // 256
    b = blocks.reshape(rows, nb, -1)
    if fmt == "q4_K":
        d = orc.h2f(b[:, :, 0:2].copy().view(np.uint16)[..., 0])
        s12 = b[:, :, 4:16].astype(np.int64)
        sc = np.empty((rows, nb, 8), np.int64)
        for s in range(8):
            if s < 4:
                sc[:, :, s] = s12[:, :, s] & 63
            else:
                sc[:, :, s] = (s12[:, :, s + 4] & 15) | ((s12[:, :, s - 4] >> 6) << 4)
        step = d[:, :, None].astype(np.float64) * sc
        return np.repeat(step, 32, axis=2).reshape(rows, k)
    d = orc.h2f(b[:, :, 208:210].copy().view(np.uint16)[..., 0])
    sc = b[:, :, 192:208].view(np.int8).astype(np.int64)
    step = np.abs(d[:, :, None].astype(np.float64) * sc)
    return np.repeat(step, 16, axis=2).reshape(rows, k)


@pytest.mark.parametrize("fmt", ["q4_K", "q6_K"])
def test_round_trip_half_step_k(orc, fmt):
    v = inputs.weights(48, 1024, 22)
    v[2] = np.abs(v[2])          # all positive
    v[4] = -np.abs(v[4])         # all negative
    v[6, :256] = 0.0             # zero super-block
    v[8, :128] *= 50.0           # mixed magnitudes inside one super-block
    blocks = orc.quantize(v, fmt)
    back = orc.dequantize(blocks, fmt, 48, 1024)
    step = _k_scales(orc, fmt, blocks, 48, 1024)
    err = np.abs(back.astype(np.float64) - v)
    assert np.all(err <= step / 2 * (1 + 2.0 ** -10) + 1e-30)


def test_f16_quantize_is_round_to_nearest(orc):
    v = inputs.weights(8, 256, 23)
    blocks = orc.quantize(v, "f16")
    assert np.array_equal(blocks.view(np.uint16), v.astype(np.float16).view(np.uint16))


# ---------------------------------------------------------------- the f64 dot

def test_f16_workload_matches_torch_f64_matmul(orc):
    import torch
    n, k = 256, 512
    w = inputs.weights(n, k, 1000).astype(np.float16)
    x = inputs.activations(1, k, 2000)
    y, a = orc.matvec(w.view(np.uint8), "f16", n, k, 1, x, 1, k, 0)
    ref = (torch.from_numpy(x).double() @ torch.from_numpy(w.astype(np.float64)).T).numpy()
    assert np.all(np.abs(y[0] - ref) <= 1e-13 * a[0])


def test_exact_integer_case(orc):
    # Q8_0 with power-of-two scales and small-integer x: every product and
    # partial sum is an exact f64 integer multiple of the scale.
    n, k, m = 8, 256, 3
    codes = inputs.uniform_bytes(n * k, 31).view(np.int8).reshape(n, k // 32, 32)
    scales = np.array([0x3800, 0x3C00, 0x4000, 0x3400], np.uint16)  # 0.5, 1, 2, 0.25
    blocks = np.zeros((n, k // 32, 34), np.uint8)
    for r in range(n):
        for blk in range(k // 32):
            blocks[r, blk, 0:2] = np.frombuffer(scales[(r + blk) % 4].tobytes(), np.uint8)
    blocks[:, :, 2:] = codes.view(np.uint8)
    x = inputs.small_ints((m, k), 32, -8, 8)
    y, _ = orc.matvec(blocks.reshape(-1), "q8_0", n, k, 1, x, m, k, 0)
    sv = {0x3800: Fraction(1, 2), 0x3C00: Fraction(1), 0x4000: Fraction(2), 0x3400: Fraction(1, 4)}
    for r in range(n):
        for j in range(m):
            tot = Fraction(0)
            for blk in range(k // 32):
                d = sv[int(scales[(r + blk) % 4])]
                tot += d * sum(int(codes[r, blk, e]) * int(x[j, 32 * blk + e]) for e in range(32))
            assert Fraction(y[0, j, r]) == tot


def test_one_hot_weight_selects_input(orc):
    n, k, m = 4, 128, 2
    blocks = np.zeros((n, k // 32, 34), np.uint8)
    blocks[:, :, 0:2] = np.frombuffer(np.uint16(0x3C00).tobytes(), np.uint8)
    hot = [5, 40, 77, 127]
    for r, k0 in enumerate(hot):
        blocks[r, k0 // 32, 2 + k0 % 32] = 1
    x = inputs.activations(m, k, 33)
    y, _ = orc.matvec(blocks.reshape(-1), "q8_0", n, k, 1, x, m, k, 0)
    for r, k0 in enumerate(hot):
        assert np.array_equal(y[0, :, r], x[:, k0].astype(np.float64))


@pytest.mark.parametrize("fmt,k", [("f16", 64), ("q8_0", 128), ("q5_0", 96), ("q4_K", 512), ("q6_K", 256)])
def test_brute_force_rational(orc, fmt, k):
    n, m = 3, 5
    v = inputs.weights(n, k, 40)
    blocks = orc.quantize(v, fmt)
    wf = orc.dequantize(blocks, fmt, n, k)
    x = inputs.activations(m, k, 41)
    y, a = orc.matvec(blocks, fmt, n, k, 1, x, m, k, 0)
    for i in range(n):
        for j in range(m):
            exact = sum(Fraction(float(wf[i, kk])) * Fraction(float(x[j, kk])) for kk in range(k))
            err = abs(Fraction(y[0, j, i]) - exact)
            assert err <= Fraction(k * 2.0 ** -52) * Fraction(a[0, j, i])


def test_grouped_token_major_layout_matches_einsum(orc):
    # grouped projection: x [m, G*k], W [G*n, k], y[j, g*n+i] = W[g*n+i] . x[j, g*k:(g+1)*k]
    G, n, k, m = 3, 5, 64, 4
    v = inputs.weights(G * n, k, 50)
    blocks = orc.quantize(v, "q8_0")
    wf = orc.dequantize(blocks, "q8_0", G * n, k).astype(np.float64)
    x = inputs.activations(m, G * k, 51)
    y, _ = orc.matvec(blocks, "q8_0", n, k, G, x, m, G * k, k)   # x_row_stride=G*k, x_batch_stride=k
    ref = np.einsum("gik,jgk->gji", wf.reshape(G, n, k), x.astype(np.float64).reshape(m, G, k))
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_sampled_rows_equal_full_rows(orc):
    n, k, m = 40, 256, 3
    blocks = orc.quantize(inputs.weights(2 * n, k, 60), "q4_K")
    x = inputs.activations(m, 2 * k, 61)
    yf, af = orc.matvec(blocks, "q4_K", n, k, 2, x, m, 2 * k, k)
    rows = np.array([0, 7, 39, 40, 79], np.uint64)
    ys, as_ = orc.matvec_rows(blocks, "q4_K", n, k, x, m, 2 * k, k, rows)
    for c, r in enumerate(rows):
        b, i = divmod(int(r), n)
        assert np.array_equal(ys[c], yf[b, :, i])
        assert np.array_equal(as_[c], af[b, :, i])


# ---------------------------------------------------------------- dense BF16 / F32 weights

def test_dense_row_bytes(orc):
    # one IEEE binary32 (4 B) or bfloat16 (2 B) per element
    for k in (4, 256, 4096):
        assert orc.row_bytes("f32", k) == 4 * k
        assert orc.row_bytes("bf16", k) == 2 * k
    assert orc.block_values("bf16") == 1 and orc.block_bytes("bf16") == 2
    assert orc.block_values("f32") == 1 and orc.block_bytes("f32") == 4


def test_bf2f_all_patterns_match_library(orc):
    import torch
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.bf2f(b)
    ref = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f2bf_nearest_even_matches_library(orc):
    import torch
    g = np.random.Generator(np.random.PCG64(11))
    b = g.integers(0, 0x7F7F, 20000).astype(np.uint16)
    lo = orc.bf2f(b).astype(np.float64)
    hi = orc.bf2f((b + 1).astype(np.uint16)).astype(np.float64)
    halfway = ((lo + hi) / 2).astype(np.float32)     # exact in binary32: ties to even decide
    v = np.concatenate([_f32_probe_values(), halfway, -halfway,
                        np.array([3.4e38, -3.4e38, 1e-40, -1e-40], np.float32)])
    ours = orc.f2bf(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    nan_bits = orc.f2bf(np.array([np.nan], np.float32))
    assert np.isnan(orc.bf2f(nan_bits))[0]


def test_dense_quantize_dequantize(orc):
    v = inputs.weights(3, 64, 50)
    assert np.array_equal(orc.dequantize(orc.quantize(v, "f32"), "f32", 3, 64).view(np.uint32), v.view(np.uint32))
    bf = orc.dequantize(orc.quantize(v, "bf16"), "bf16", 3, 64)
    assert np.array_equal(orc.f2bf(bf), orc.f2bf(v))            # bf16 values, re-rounding is exact
    assert np.all(np.abs(bf - v) <= np.abs(v) * 2.0 ** -8)      # half an ulp of an 8-bit significand


@pytest.mark.parametrize("fmt,k", [("f32", 64), ("bf16", 96)])
def test_dense_brute_force_rational(orc, fmt, k):
    n, m = 3, 4
    blocks = orc.quantize(inputs.weights(n, k, 42), fmt)
    wf = orc.dequantize(blocks, fmt, n, k)
    x = inputs.activations(m, k, 43)
    y, a = orc.matvec(blocks, fmt, n, k, 1, x, m, k, 0)
    for i in range(n):
        for j in range(m):
            exact = sum(Fraction(float(wf[i, kk])) * Fraction(float(x[j, kk])) for kk in range(k))
            assert abs(Fraction(y[0, j, i]) - exact) <= Fraction(k * 2.0 ** -52) * Fraction(a[0, j, i])


# ---------------------------------------------------------------- affine (group scale and bias)

def _affine_case(bits, gs, k, codes_at, scale_bits, bias_bits):
    """codes_at: {element index: code}; scale/bias binary16 bit patterns per group."""
    per = 32 // bits
    codes = np.zeros((1, k * bits // 32), dtype=np.uint32)
    for i, q in codes_at.items():
        codes[0, i // per] |= np.uint32(q << (bits * (i % per)))
    sc = np.array([scale_bits], dtype=np.uint16).reshape(1, -1)
    bi = np.array([bias_bits], dtype=np.uint16).reshape(1, -1)
    return codes, sc, bi


@pytest.mark.parametrize("bits,gs,k,codes_at,scales,biases,expect", [
    # one code lights one element, at index i: word i // (32/bits), bits bits*(i % (32/bits)) (lowest first)
    (4, 32, 32, {0: 5}, [0x3C00], [0x0000], {0: 5.0}),
    (4, 32, 32, {1: 5}, [0x3C00], [0x0000], {1: 5.0}),
    (4, 32, 32, {7: 15}, [0x3C00], [0x0000], {7: 15.0}),
    (4, 32, 32, {8: 9}, [0x3C00], [0x0000], {8: 9.0}),
    (4, 32, 32, {31: 1}, [0x3800], [0x0000], {31: 0.5}),
    (8, 32, 32, {2: 200}, [0x3C00], [0x0000], {2: 200.0}),
    (8, 32, 32, {5: 255}, [0x3400], [0x0000], {5: 63.75}),
    # the bias adds to every element of its group, the scale multiplies the code
    (4, 32, 32, {}, [0x3C00], [0xC000], {}),                  # all -2
    (4, 32, 32, {3: 15}, [0x3800], [0xC000], {3: 5.5}),       # 0.5*15 - 2
    # group g covers elements g*gs .. g*gs+gs-1
    (4, 32, 64, {40: 3}, [0x3C00, 0x4000], [0x0000, 0x3C00], {40: 7.0}),   # group 1: 2*3 + 1
    (8, 64, 128, {63: 1, 64: 1}, [0x3C00, 0x4400], [0x0000, 0x0000], {63: 1.0, 64: 4.0}),
])
def test_affine_decode_hand_derived(orc, bits, gs, k, codes_at, scales, biases, expect):
    codes, sc, bi = _affine_case(bits, gs, k, codes_at, scales, biases)
    got = orc.affine_dequantize(codes, sc, bi, bits, gs, 1, k)[0]
    for i in range(k):
        g = i // gs
        base = float(orc.h2f(np.array([biases[g]], np.uint16))[0])
        assert got[i] == np.float32(expect.get(i, base)), (i, got[i])


def _affine_bytes_case(bits, k, byte_map):
    """Codes of one row from explicit byte values {byte index: value}; the
    row's uint32 words are those bytes read little-endian."""
    b = np.zeros(k * bits // 8, dtype=np.uint8)
    for j, v in byte_map.items():
        b[j] = v
    return b.view("<u4").astype(np.uint32).reshape(1, -1)


@pytest.mark.parametrize("bits,gs,k,byte_map,scales,biases,expect", [
    # 3 bits, 8 codes per 3-byte packing unit; code i at stream bits 3i .. 3i+2
    (3, 32, 32, {0: 0x05}, [0x3C00], [0x0000], {0: 5.0}),                 # bits 0-2 = 101
    (3, 32, 32, {0: 0xC0, 1: 0x01}, [0x3C00], [0x0000], {2: 7.0}),        # bits 6, 7 | 8
    (3, 32, 32, {2: 0x80}, [0x3C00], [0x0000], {7: 4.0}),                 # bit 23 = top bit of code 7
    (3, 32, 32, {3: 0x03}, [0x3C00], [0x0000], {8: 3.0}),                 # second unit starts at byte 3
    (3, 32, 32, {3: 0x80, 4: 0x01}, [0x3C00], [0x0000], {10: 6.0}),       # bits 30 (0), 31 (1), 32 (1)
    (3, 32, 32, {11: 0xE0}, [0x3C00], [0x0000], {31: 7.0}),               # bits 93-95
    # 5 bits, 8 codes per 5-byte unit
    (5, 32, 32, {0: 0xE0, 1: 0x03}, [0x3C00], [0x0000], {1: 31.0}),       # bits 5-9
    (5, 32, 32, {4: 0x88}, [0x3C00], [0x0000], {7: 17.0}),                # bits 35 and 39 of 35-39
    (5, 32, 32, {5: 0x01}, [0x3800], [0xC000], {8: -1.5}),                # 0.5*1 - 2, the rest -2
    (5, 32, 32, {19: 0xF8}, [0x3C00], [0x0000], {31: 31.0}),              # bits 155-159
    # 6 bits, 4 codes per 3-byte unit
    (6, 32, 32, {0: 0xC0, 1: 0x0F}, [0x3C00], [0x0000], {1: 63.0}),       # bits 6-11
    (6, 32, 32, {2: 0x84}, [0x3C00], [0x0000], {3: 33.0}),                # bits 18 and 23 of 18-23
    (6, 32, 32, {3: 0x02}, [0x3C00], [0x0000], {4: 2.0}),                 # second unit starts at byte 3
    (6, 32, 32, {4: 0x0C}, [0x3C00], [0x0000], {5: 48.0}),                # bits 34, 35 of 30-35
    (6, 32, 32, {23: 0xFC}, [0x3C00], [0x0000], {31: 63.0}),              # bits 186-191
    (6, 32, 64, {30: 0x21}, [0x3C00, 0x4000], [0x0000, 0x3C00], {40: 67.0}),   # group 1: 2*33 + 1
])
def test_affine_decode_hand_derived_bytes(orc, bits, gs, k, byte_map, scales, biases, expect):
    codes = _affine_bytes_case(bits, k, byte_map)
    sc = np.array([scales], dtype=np.uint16).reshape(1, -1)
    bi = np.array([biases], dtype=np.uint16).reshape(1, -1)
    got = orc.affine_dequantize(codes, sc, bi, bits, gs, 1, k)[0]
    for i in range(k):
        base = float(orc.h2f(np.array([biases[i // gs]], np.uint16))[0])
        assert got[i] == np.float32(expect.get(i, base)), (i, got[i])


@pytest.mark.parametrize("bits,gs", [(b, g) for b in (3, 4, 5, 6, 8) for g in (32, 64, 128)])
def test_affine_round_trip_bound(orc, bits, gs):
    k, rows = 512, 6
    v = inputs.weights(rows, k, 60)
    v[1] *= 100.0
    v[2] = np.float32(0.25)                       # constant rows: scale 0
    c, s, b = orc.affine_quantize(v, bits, gs)
    d = orc.affine_dequantize(c, s, b, bits, gs, rows, k)
    qmax = 2 ** bits - 1
    g = v.reshape(rows, k // gs, gs)
    lo, hi = g.min(axis=2).astype(np.float64), g.max(axis=2).astype(np.float64)
    sf, bf = orc.h2f(s).astype(np.float64), orc.h2f(b).astype(np.float64)
    bound = 0.5 * sf + np.abs(lo - bf) + qmax * np.abs((hi - lo) / qmax - sf) + 1e-6 * (np.abs(lo) + np.abs(hi))
    err = np.abs(d.astype(np.float64) - v.astype(np.float64)).reshape(rows, k // gs, gs).max(axis=2)
    assert np.all(err <= bound)


@pytest.mark.parametrize("bits,gs", [(4, 64), (8, 32), (3, 32), (5, 128), (6, 64)])
def test_affine_brute_force_rational(orc, bits, gs):
    n, k, m = 3, 128, 4
    c, s, b = orc.affine_quantize(inputs.weights(n, k, 61), bits, gs)
    wf = orc.affine_dequantize(c, s, b, bits, gs, n, k)
    x = inputs.activations(m, k, 62)
    y, a = orc.affine_matvec(c, s, b, bits, gs, n, k, 1, x, m, k, 0)
    for i in range(n):
        for j in range(m):
            exact = sum(Fraction(float(wf[i, kk])) * Fraction(float(x[j, kk])) for kk in range(k))
            assert abs(Fraction(y[0, j, i]) - exact) <= Fraction(k * 2.0 ** -52) * Fraction(a[0, j, i])
