"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

* decode: rem_dequantize equals the oracle's dequantizer bit for bit;
* quantize: rem_quantize equals the oracle's quantizer byte for byte;
* mat-vec: |y - y_ref| <= 1e-4 * sum|w*x| + 1e-7 element by element, on shapes
  that span several row groups, several chunks and ragged tails;
* row exactness (module doc "Row exactness" of mlx-native 0.18.0
  src/ops/row_exact_matvec.rs): row j of an m-row call is bitwise equal to
  the same row computed alone, for every m <= 8, every rows-per-CTA packing,
  both staging paths and repeated runs;
* batched / grouped products (RowExactMatvecShape) equal separate calls.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import quantized_few_row_gb300 as rem
from quantized_few_row_gb300 import inputs
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

FMTS = ["f16", "q8_0", "q5_0", "q4_K", "q6_K", "bf16", "f32"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rem.build()
    rem.load()
    torch.cuda.init()


# ---------------------------------------------------------------- decode / quantize

@pytest.mark.parametrize("fmt", FMTS)
def test_dequantize_bit_exact(fmt):
    k = {"f16": 520, "q8_0": 1024, "q5_0": 1024, "q4_K": 1024, "q6_K": 1024, "bf16": 520, "f32": 520}[fmt]
    rows = 37
    for w in (oracle.quantize(inputs.weights(rows, k, 101), fmt), H.adversarial_blocks(fmt, rows, k, 102)):
        ref = oracle.dequantize(w, fmt, rows, k)
        wh, wp = H.to_dev_bytes(w)
        out = H.canary(rows * k)
        rem.check(rem.rem_dequantize(wp, fmt, rows, k, out))
        torch.cuda.synchronize()
        got = out.cpu().numpy().reshape(rows, k)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("fmt", FMTS)
def test_quantize_bit_exact(fmt):
    k = 1024
    v = inputs.weights(24, k, 111)
    v[1] = 0.0                     # zero rows
    v[2] = np.float32(0.013)       # constant row
    v[3] *= 1000.0                 # large values
    v[4] *= 1e-4                   # subnormal fp16 scales
    v[5] = np.abs(v[5])            # one sign only
    v[6] = -np.abs(v[6])
    ref = oracle.quantize(v, fmt)
    src = H.to_dev_f32(v)
    wd = torch.zeros(ref.size, dtype=torch.uint8, device=H.dev())
    rem.check(rem.rem_quantize(src, fmt, 24, k, wd))
    torch.cuda.synchronize()
    assert np.array_equal(wd.cpu().numpy().reshape(ref.shape), ref)


# ---------------------------------------------------------------- mat-vec parity

SHAPES = {  # (n, k): several row groups, several chunks, ragged row tail
    "f16": [(103, 520), (64, 136), (7, 4096)],
    "q8_0": [(103, 1024), (40, 352), (300, 4096)],
    "q5_0": [(103, 1024), (40, 160), (77, 2048)],
    "q4_K": [(103, 1024), (33, 256), (150, 4096)],
    "q6_K": [(103, 1024), (33, 256), (150, 4096)],
    "bf16": [(103, 520), (64, 72), (7, 4096)],
    "f32": [(103, 520), (64, 36), (7, 4096)],
}


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 8])
def test_matvec_matches_oracle(fmt, m):
    for si, (n, k) in enumerate(SHAPES[fmt]):
        w, x = H.contiguous(fmt, n, k, m, 200 + si, 300 + si)
        y_ref, a_ref = oracle.matvec(w, fmt, n, k, 1, x, m, k, 0)
        y = H.run_matvec(w, fmt, n, k, 1, x, m, k, 0, n, 0, m * n, use_ex=False)
        H.assert_close_to_oracle(y.reshape(1, m, n), y_ref, a_ref, f"{fmt} n={n} k={k} m={m}")


@pytest.mark.parametrize("fmt", FMTS)
def test_strided_output_untouched_between_rows(fmt):
    n, k, m = 70, 512, 3
    w, x = H.contiguous(fmt, n, k, m, 210, 310)
    xs = np.zeros((m, k + 8), np.float32)
    xs[:, :k] = x
    y = H.run_matvec(w, fmt, n, k, 1, xs, m, k + 8, 0, n + 5, 0, m * (n + 5))
    y_ref, a_ref = oracle.matvec(w, fmt, n, k, 1, xs, m, k + 8, 0)
    H.assert_close_to_oracle(H.gather_y(y, 1, m, n, n + 5, 0), y_ref, a_ref, fmt)
    gaps = y.reshape(m, n + 5)[:, n:]
    assert np.all(gaps == H.CANARY)


# ---------------------------------------------------------------- row exactness

@pytest.mark.parametrize("fmt", FMTS)
def test_rows_bitwise_equal_for_every_m(fmt):
    n, k = 200, {"f16": 1088}.get(fmt, 1024)
    w, x = H.contiguous(fmt, n, k, 8, 220, 320)
    alone = [H.run_matvec(w, fmt, n, k, 1, x[j:j + 1], 1, k, 0, n, 0, n, use_ex=False) for j in range(8)]
    for m in range(1, 9):
        y = H.run_matvec(w, fmt, n, k, 1, x[:m], m, k, 0, n, 0, m * n, use_ex=False).reshape(m, n)
        for j in range(m):
            assert np.array_equal(y[j].view(np.uint32), alone[j].view(np.uint32)), (m, j)


@pytest.mark.parametrize("fmt", FMTS)
def test_rows_inert_to_packing_path_and_runs(fmt):
    n, k = 300, 2048
    w, x = H.contiguous(fmt, n, k, 8, 230, 330)
    split = 2
    base = H.run_matvec(w, fmt, n, k, 1, x, 8, k, 0, n, 0, 8 * n, split=split)
    variants = [dict(rows_per_cta=rpc) for rpc in (32, 64, 128)]
    if fmt in ("f16", "bf16"):
        variants.append(dict(w_offset=8))           # 8-byte alignment required: plain staging path
    elif fmt == "f32":
        variants.append(dict(w_offset=4))           # 4-byte aligned base: plain staging path
    elif fmt != "q4_K":                             # Q4_K requires 16-byte alignment
        variants.append(dict(w_offset=2))           # 2-byte aligned base: plain staging path
    for v in variants:
        y = H.run_matvec(w, fmt, n, k, 1, x, 8, k, 0, n, 0, 8 * n, split=split, **v)
        assert np.array_equal(y.view(np.uint32), base.view(np.uint32)), v
    for m in (1, 4):
        for rpc in (32, 64):
            ym = H.run_matvec(w, fmt, n, k, 1, x[:m], m, k, 0, n, 0, m * n, split=split, rows_per_cta=rpc)
            assert np.array_equal(ym.view(np.uint32), base[:m * n].view(np.uint32)), (m, rpc)
    wh, wp = H.to_dev_bytes(w)
    xd = H.to_dev_f32(x)
    outs = []
    for _ in range(10):
        yd = H.canary(8 * n)
        rem.check(rem.rem_matvec_ex(wp, fmt, n, k, 1, xd, 8, k, 0, yd, n, 0, split, 0))
        outs.append(yd)
    torch.cuda.synchronize()
    for yd in outs:
        assert np.array_equal(yd.cpu().numpy().view(np.uint32), base.view(np.uint32))


@pytest.mark.parametrize("fmt", FMTS)
def test_split_changes_only_rounding(fmt):
    n, k, m = 64, 2048, 2
    w, x = H.contiguous(fmt, n, k, m, 240, 340)
    y_ref, a_ref = oracle.matvec(w, fmt, n, k, 1, x, m, k, 0)
    for split in (1, 2, 3, 5, 8):
        y = H.run_matvec(w, fmt, n, k, 1, x, m, k, 0, n, 0, m * n, split=split)
        H.assert_close_to_oracle(y.reshape(1, m, n), y_ref, a_ref, f"{fmt} split={split}")


# ---------------------------------------------------------------- batched / grouped

@pytest.mark.parametrize("fmt", FMTS)
def test_grouped_token_major_equals_separate_calls(fmt):
    G, n, k, m = 3, 70, 512, 4
    wf = inputs.weights(G * n, k, 250)
    w = oracle.quantize(wf, fmt)
    x = inputs.activations(m, G * k, 350)
    split = rem.rem_split_factor(fmt, G * n, k)
    # grouped_token_major: x [m, G*k], W [G*n, k], y [m, G*n]
    y = H.run_matvec(w, fmt, n, k, G, x, m, G * k, k, G * n, n, m * G * n, split=split)
    y3 = H.gather_y(y, G, m, n, G * n, n)
    y_ref, a_ref = oracle.matvec(w, fmt, n, k, G, x, m, G * k, k)
    H.assert_close_to_oracle(y3, y_ref, a_ref, f"{fmt} grouped")
    # the same through rem_matvec's inferred token-major strides
    yi = H.run_matvec(w, fmt, n, k, G, x, m, 0, k, 0, n, m * G * n, use_ex=False)
    if split == rem.rem_split_factor(fmt, G * n, k):
        assert np.array_equal(yi.view(np.uint32), y.view(np.uint32))
    rb = oracle.row_bytes(fmt, k)
    for g in range(G):
        wg = w.reshape(-1)[g * n * rb:(g + 1) * n * rb]
        xg = np.ascontiguousarray(x[:, g * k:(g + 1) * k])
        yg = H.run_matvec(wg, fmt, n, k, 1, xg, m, k, 0, n, 0, m * n, split=split).reshape(m, n)
        assert np.array_equal(yg.view(np.uint32), y3[g].view(np.uint32)), g


@pytest.mark.parametrize("fmt", ["q8_0", "q4_K"])
def test_batch_major_layout(fmt):
    B, n, k, m = 2, 96, 512, 3
    w = oracle.quantize(inputs.weights(B * n, k, 260), fmt)
    x = inputs.activations(B * m, k, 360)        # x [B, m, k]
    y = H.run_matvec(w, fmt, n, k, B, x, m, k, m * k, n, m * n, B * m * n, use_ex=False)
    y_ref, a_ref = oracle.matvec(w, fmt, n, k, B, x, m, k, m * k)
    H.assert_close_to_oracle(y.reshape(B, m, n), y_ref, a_ref, f"{fmt} batch-major")


# ---------------------------------------------------------------- special cases

def test_exact_integer_case_is_bitwise():
    n, k, m = 96, 512, 5
    codes = inputs.uniform_bytes(n * k, 270).view(np.int8).reshape(n, k // 32, 32)
    scales = np.array([0x3800, 0x3C00, 0x4000, 0x3400], np.uint16)
    blocks = np.zeros((n, k // 32, 34), np.uint8)
    for r in range(n):
        for b in range(k // 32):
            blocks[r, b, 0:2] = np.frombuffer(scales[(r + b) % 4].tobytes(), np.uint8)
    blocks[:, :, 2:] = codes.view(np.uint8)
    x = inputs.small_ints((m, k), 271, -8, 8)
    y_ref, _ = oracle.matvec(blocks, "q8_0", n, k, 1, x, m, k, 0)
    y = H.run_matvec(blocks, "q8_0", n, k, 1, x, m, k, 0, n, 0, m * n, use_ex=False)
    assert np.array_equal(y.reshape(m, n).astype(np.float64), y_ref[0])


@pytest.mark.parametrize("fmt", FMTS)
def test_nan_in_input_row_stays_in_that_row(fmt):
    n, k, m = 64, 1024, 3
    w, x = H.contiguous(fmt, n, k, m, 280, 380)
    x[1, 77] = np.nan
    y = H.run_matvec(w, fmt, n, k, 1, x, m, k, 0, n, 0, m * n).reshape(m, n)
    assert np.all(np.isnan(y[1]))
    assert np.all(np.isfinite(y[0])) and np.all(np.isfinite(y[2]))


@pytest.mark.parametrize("fmt", FMTS)
def test_single_row_single_chunk(fmt):
    n, k, m = 1, {"f16": 4, "bf16": 4, "f32": 4}.get(fmt, oracle.block_values(fmt)), 1
    w, x = H.contiguous(fmt, n, k, m, 290, 390)
    y_ref, a_ref = oracle.matvec(w, fmt, n, k, 1, x, m, k, 0)
    y = H.run_matvec(w, fmt, n, k, 1, x, m, k, 0, n, 0, 1, use_ex=False)
    H.assert_close_to_oracle(y.reshape(1, 1, 1), y_ref, a_ref, fmt)


# ---------------------------------------------------------------- errors leave y alone

def test_rejected_calls_write_nothing():
    n, k, m = 64, 256, 2
    w, x = H.contiguous("q8_0", n, k, m, 295, 395)
    wh, wp = H.to_dev_bytes(w)
    xd = H.to_dev_f32(x)
    yd = H.canary(m * n)
    bad = [dict(m=9), dict(k=100), dict(yrs=n - 1), dict(wp=wp + 1)]   # wp is 256-byte aligned
    for b in bad:
        a = dict(wp=wp, m=m, k=k, yrs=n)
        a.update(b)
        rc = rem.rem_matvec_ex(a["wp"], "q8_0", n, a["k"], 1, xd, a["m"], k, 0, yd, a["yrs"], 0, 0, 0)
        assert rc == rem.REM_EINVAL, b
    # a weight pointer 64 bytes before the end of its allocation: the caching
    # allocator gives a fresh 32 MiB request a segment of its own
    torch.cuda.empty_cache()
    big = torch.zeros(32 << 20, dtype=torch.uint8, device=H.dev())
    near_end = big.data_ptr() + (32 << 20) - 64
    assert rem.rem_matvec_ex(near_end, "q8_0", n, k, 1, xd, m, k, 0, yd, n, 0, 0, 0) == rem.REM_EINVAL
    assert "holds" in rem.rem_last_error()
    # host memory that CUDA cannot see
    host = np.zeros(m * n, np.float32)
    assert rem.rem_matvec_ex(wp, "q8_0", n, k, 1, xd, m, k, 0, host.ctypes.data, n, 0, 0, 0) == rem.REM_EINVAL
    # a schedule above the kernels' thread limit is refused, not launched
    assert rem.rem_matvec_ex(wp, "q8_0", n, k, 1, xd, m, k, 0, yd, n, 0, 16, 0) == rem.REM_ELAUNCH
    torch.cuda.synchronize()
    assert np.all(yd.cpu().numpy() == H.CANARY)


# ---------------------------------------------------------------- dependent launches

def _alternating_sequence(fmt, n, k, m, stream, W, x, srcs, xs, outs):
    """rem_quantize -> input copy -> rem_matvec -> output copy, three times
    per source, on one stream with no synchronisation in between."""
    for it in range(len(outs)):
        i = it % 2
        rem.check(rem.rem_quantize(srcs[i], fmt, n, k, W, stream))
        x.copy_(xs[i])
        rem.check(rem.rem_matvec(W, fmt, n, k, 1, x, m, 0, outs[it], 0, stream))
        outs[it].mul_(1.0)   # a kernel that reads y right after the call


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("graph", [False, True])
def test_back_to_back_calls_see_previous_writes(fmt, graph):
    """Each call may start while the previous kernel of its stream is still
    running (it only prefetches weights into L2 before waiting for it): weights
    just rewritten by rem_quantize, inputs just rewritten by a copy, and an
    output read by the next kernel give exactly the synchronised result."""
    n, k, m = 640, 2048, 4
    dev = H.dev()
    wf = [inputs.weights(n, k, 260), inputs.weights(n, k, 261)]
    xf = [inputs.activations(m, k, 360), inputs.activations(m, k, 361)]
    q = [oracle.quantize(w, fmt) for w in wf]
    ref = [H.run_matvec(q[i], fmt, n, k, 1, xf[i], m, k, 0, n, 0, m * n, use_ex=False) for i in range(2)]
    for i in range(2):
        y_ref, a_ref = oracle.matvec(q[i], fmt, n, k, 1, xf[i], m, k, 0)
        H.assert_close_to_oracle(ref[i].reshape(1, m, n), y_ref, a_ref, fmt)
    srcs = [torch.from_numpy(w).to(dev) for w in wf]
    xs = [H.to_dev_f32(x) for x in xf]
    W = torch.zeros(n * oracle.row_bytes(fmt, k), dtype=torch.uint8, device=dev)
    x = torch.zeros_like(xs[0])
    outs = [H.canary(m * n) for _ in range(6)]
    torch.cuda.synchronize()
    s = torch.cuda.Stream(device=dev)
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
                _alternating_sequence(fmt, n, k, m, s, W, x, srcs, xs, outs)
        for _ in range(2):
            for o in outs:
                o.fill_(float(H.CANARY))
            with torch.cuda.stream(s):
                g.replay()
            s.synchronize()
            for it, o in enumerate(outs):
                assert np.array_equal(o.cpu().numpy().view(np.uint32), ref[it % 2].view(np.uint32)), it
    else:
        with torch.cuda.stream(s):
            _alternating_sequence(fmt, n, k, m, s, W, x, srcs, xs, outs)
        s.synchronize()
        for it, o in enumerate(outs):
            assert np.array_equal(o.cpu().numpy().view(np.uint32), ref[it % 2].view(np.uint32)), it


# ---------------------------------------------------------------- more than 8 input rows

@pytest.mark.parametrize("fmt", FMTS)
def test_many_rows_match_oracle_and_single_rows(fmt):
    """rem_matvec_many (groups of 8 input rows) against the oracle, and every
    row bitwise equal to the same row computed alone and to the same row of an
    8-row call."""
    n, k = 200, {"f16": 1088}.get(fmt, 1024)
    mmax = 24
    w, x = H.contiguous(fmt, n, k, mmax, 270, 370)
    alone = [H.run_matvec(w, fmt, n, k, 1, x[j:j + 1], 1, k, 0, n, 0, n, use_ex=False) for j in range(mmax)]
    eight = H.run_matvec(w, fmt, n, k, 1, x[8:16], 8, k, 0, n, 0, 8 * n, use_ex=False).reshape(8, n)
    wh, wp = H.to_dev_bytes(w)
    xd = H.to_dev_f32(x)
    for m in (9, 12, 16, 17, 24):
        yd = H.canary(m * n)
        rem.check(rem.rem_matvec_many(wp, fmt, n, k, 1, xd, m, k, 0, yd, n, 0, 0))
        torch.cuda.synchronize()
        y = yd.cpu().numpy().reshape(m, n)
        y_ref, a_ref = oracle.matvec(w, fmt, n, k, 1, x[:m], m, k, 0)
        H.assert_close_to_oracle(y.reshape(1, m, n), y_ref, a_ref, f"{fmt} m={m}")
        for j in range(m):
            assert np.array_equal(y[j].view(np.uint32), alone[j].view(np.uint32)), (m, j)
        if m >= 16:
            assert np.array_equal(y[8:16].view(np.uint32), eight.view(np.uint32)), m


@pytest.mark.parametrize("fmt", ["q5_0", "q4_K"])
def test_many_rows_token_major_grouped(fmt):
    """Grouped token-major layout (x [m, G*k], y [m, G*n]) with m = 11 tokens:
    equal to the oracle and bitwise equal to the 8 + 3 split done by hand."""
    G, n, k, m = 3, 96, 512, 11
    w = oracle.quantize(inputs.weights(G * n, k, 280), fmt)
    x = inputs.activations(m, G * k, 380)
    wh, wp = H.to_dev_bytes(w)
    xd = H.to_dev_f32(x)
    yd = H.canary(m * G * n)
    rem.check(rem.rem_matvec_many(wp, fmt, n, k, G, xd, m, G * k, k, yd, G * n, n, 0))
    torch.cuda.synchronize()
    y = yd.cpu().numpy()
    y_ref, a_ref = oracle.matvec(w, fmt, n, k, G, x, m, G * k, k)
    H.assert_close_to_oracle(H.gather_y(y, G, m, n, G * n, n), y_ref, a_ref, f"{fmt} grouped m={m}")
    split = rem.rem_split_factor(fmt, G * n, k)
    head = H.run_matvec(w, fmt, n, k, G, x[:8], 8, G * k, k, G * n, n, 8 * G * n, split=split)
    tail = H.run_matvec(w, fmt, n, k, G, x[8:], 3, G * k, k, G * n, n, 3 * G * n, split=split)
    assert np.array_equal(y[:8 * G * n].view(np.uint32), head.view(np.uint32))
    assert np.array_equal(y[8 * G * n:].view(np.uint32), tail.view(np.uint32))


# ---------------------------------------------------------------- fused epilogue alpha * W.x + beta * c

def _fma_f32(a, b, c):
    """Correctly rounded binary32 fma(a, b, c) from exact rational arithmetic."""
    from fractions import Fraction
    r = Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c))
    f = np.float32(float(r))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    return min(cands, key=lambda v: (abs(Fraction(float(v)) - r), int(np.float32(v).view(np.uint32)) & 1))


@pytest.mark.parametrize("fmt", FMTS)
def test_axpby_matches_oracle_and_exact_epilogue(fmt):
    n, k, m = 150, {"f16": 1088}.get(fmt, 1024), 5
    w, x = H.contiguous(fmt, n, k, m, 290, 390)
    c = inputs.activations(m, n, 490)
    alpha, beta = np.float32(-1.75), np.float32(0.3)
    wh, wp = H.to_dev_bytes(w)
    xd = H.to_dev_f32(x)
    cd = H.to_dev_f32(c)
    plain = H.canary(m * n)
    rem.check(rem.rem_matvec_ex(wp, fmt, n, k, 1, xd, m, k, 0, plain, n, 0, 0, 0))
    yd = H.canary(m * n)
    rem.check(rem.rem_matvec_axpby(wp, fmt, n, k, 1, xd, m, k, 0, yd, n, 0, float(alpha), float(beta), cd, n, 0))
    torch.cuda.synchronize()
    y = yd.cpu().numpy().reshape(m, n)
    p = plain.cpu().numpy().reshape(m, n)
    # against the oracle: alpha * y_ref + beta * c in f64, the product's tolerance scaled
    # by |alpha| plus two binary32 roundings of the epilogue
    y_ref, a_ref = oracle.matvec(w, fmt, n, k, 1, x, m, k, 0)
    ref = float(alpha) * y_ref[0] + float(beta) * c.astype(np.float64)
    tol = abs(float(alpha)) * (1e-4 * a_ref[0] + 1e-7) + 2.0 ** -22 * (np.abs(float(alpha) * y_ref[0]) +
                                                                       np.abs(float(beta) * c))
    assert np.all(np.abs(y - ref) <= tol), np.max(np.abs(y - ref) - tol)
    # the epilogue is exactly fma(alpha, acc, fl(beta * c)) on the plain result
    g = np.random.Generator(np.random.PCG64(7))
    for j, i in zip(g.integers(0, m, 200), g.integers(0, n, 200)):
        expect = _fma_f32(alpha, p[j, i], np.float32(beta) * np.float32(c[j, i]))
        assert y[j, i].view(np.uint32) == np.float32(expect).view(np.uint32), (j, i)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_K", "f16"])
def test_axpby_special_cases(fmt):
    """alpha = 1, beta = 0 is the plain call bitwise; beta = 0 reads no c;
    c == y accumulates in place; c_row_stride = 0 broadcasts one bias vector."""
    n, k, m = 130, {"f16": 1088}.get(fmt, 1024), 3
    w, x = H.contiguous(fmt, n, k, m, 291, 391)
    wh, wp = H.to_dev_bytes(w)
    xd = H.to_dev_f32(x)
    plain = H.canary(m * n)
    rem.check(rem.rem_matvec_ex(wp, fmt, n, k, 1, xd, m, k, 0, plain, n, 0, 0, 0))
    nan_c = torch.full((m * n,), float("nan"), device=H.dev())
    y1 = H.canary(m * n)
    rem.check(rem.rem_matvec_axpby(wp, fmt, n, k, 1, xd, m, k, 0, y1, n, 0, 1.0, 0.0, nan_c, n, 0))
    y2 = H.canary(m * n)
    rem.check(rem.rem_matvec_axpby(wp, fmt, n, k, 1, xd, m, k, 0, y2, n, 0, 0.5, 0.0, None, 0, 0))
    bias = inputs.activations(1, n, 492)[0]
    bd = H.to_dev_f32(bias)
    y3 = H.canary(m * n)
    rem.check(rem.rem_matvec_axpby(wp, fmt, n, k, 1, xd, m, k, 0, y3, n, 0, 1.0, 1.0, bd, 0, 0))
    acc = H.to_dev_f32(inputs.activations(m, n, 493))
    acc0 = acc.cpu().numpy().reshape(m, n)
    rem.check(rem.rem_matvec_axpby(wp, fmt, n, k, 1, xd, m, k, 0, acc, n, 0, 2.0, -1.0, acc, n, 0))
    torch.cuda.synchronize()
    p = plain.cpu().numpy().reshape(m, n)
    assert np.array_equal(y1.cpu().numpy().view(np.uint32), plain.cpu().numpy().view(np.uint32))
    assert np.array_equal(y2.cpu().numpy().reshape(m, n), p * np.float32(0.5))
    assert np.array_equal(y3.cpu().numpy().reshape(m, n), p + bias[None, :])   # fma(1, acc, b) = acc + b
    g = np.random.Generator(np.random.PCG64(8))
    got = acc.cpu().numpy().reshape(m, n)
    for j, i in zip(g.integers(0, m, 100), g.integers(0, n, 100)):
        expect = _fma_f32(np.float32(2.0), p[j, i], -acc0[j, i])
        assert got[j, i].view(np.uint32) == np.float32(expect).view(np.uint32), (j, i)
