"""GPU parity at the benchmark's full sizes, called the way bench.py calls the
library (rem_matvec, inferred strides, the automatic schedule): every output
of every m against the oracle (one f64 run over all rows at the largest m;
the oracle's row j does not depend on m), a canary past the end of y that no
call may touch, and bitwise row exactness between m = 1 and the larger m on
every row.

Workloads (all seeded and synthetic, W ~ N(0, 0.02) quantized by the
oracle's quantizer, x ~ N(0, 1)): F16 256x512 m=1; Q8_0 4096x4096 m=1..8;
Q4_K 14336x4096 m=1..8; Q6_K 128256x4096 m=1,4,8; grouped token-major Q5_0,
16 groups of 1024x4096, m=8; the >= 64 MB variants (F16 8192, Q8_0 16384,
Q4_K 28672 rows, Q5_0 32 groups) and dense BF16 8192 / F32 4096 rows; Q4_K
14336x4096 at m = 16 and 32 through rem_matvec_many; Q8_0 4096x4096 with a
bias vector through rem_matvec_axpby.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import quantized_few_row_gb300 as rem
from quantized_few_row_gb300 import inputs
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

CONFIGS = [  # format, n, k, batch, m values, token-major grouped, seed index
    ("f16", 256, 512, 1, [1], False, 0),
    ("q8_0", 4096, 4096, 1, list(range(1, 9)), False, 1),
    ("q4_K", 14336, 4096, 1, list(range(1, 9)), False, 2),
    ("q6_K", 128256, 4096, 1, [1, 4, 8], False, 3),
    ("q5_0", 1024, 4096, 16, [8], True, 4),
    # >= 64 MB variants and dense weights
    ("f16", 8192, 4096, 1, [1, 8], False, 5),
    ("q8_0", 16384, 4096, 1, [1, 8], False, 6),
    ("q4_K", 28672, 4096, 1, [1, 8], False, 7),
    ("q5_0", 1024, 4096, 32, [8], True, 8),
    ("bf16", 8192, 4096, 1, [1, 8], False, 11),
    ("f32", 4096, 4096, 1, [1, 8], False, 12),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rem.build()
    rem.load()


def _weights(fmt, rows, k, seed, slab=8192):
    """Quantized rows drawn slab by slab from one seeded stream (bounded host memory)."""
    g = np.random.Generator(np.random.PCG64(seed))
    rb = oracle.row_bytes(fmt, k)
    w = np.empty((rows, rb), dtype=np.uint8)
    for r0 in range(0, rows, slab):
        r1 = min(rows, r0 + slab)
        v = (g.standard_normal(size=(r1 - r0, k), dtype=np.float32) * np.float32(inputs.W_STD)).astype(np.float32)
        w[r0:r1] = oracle.quantize(v, fmt)
    return w


TAIL = 256   # canary floats past the last output


def _all_rows(batch, n):
    return np.arange(batch * n, dtype=np.uint64)


def _check_all(y, y_ref, a_ref, batch, n, m, yrs, ybs, what):
    """Every output (b, j, i), j < m, of a flat y against the oracle's
    [rows, mmax] arrays."""
    r = _all_rows(batch, n).astype(np.int64)
    bi, ii = r // n, r % n
    got = np.stack([y[bi * ybs + j * yrs + ii] for j in range(m)], axis=1)
    ok = oracle.within_tolerance(got, y_ref[:, :m], a_ref[:, :m])
    assert ok.all(), (what, m, int((~ok).sum()), np.argwhere(~ok)[:5].tolist())
    return got


@pytest.mark.parametrize("cfg", CONFIGS, ids=[f"{c[0]}_{c[1]}x{c[2]}_b{c[3]}" for c in CONFIGS])
def test_full_size_parity_every_output(cfg):
    fmt, n, k, batch, ms, grouped, ci = cfg
    w = _weights(fmt, batch * n, k, 1000 + ci)
    mmax = max(ms)
    dev = H.dev()
    wd = torch.from_numpy(w.reshape(-1)).to(dev)
    if grouped:   # x [m, batch*k], y [m, batch*n]; rem_matvec infers the token-major row strides
        x = inputs.activations(mmax, batch * k, 2000 + ci)
        xrs, xbs, yrs, ybs = batch * k, k, batch * n, n
    else:         # x [batch, m, k], y [batch, m, n]
        x = inputs.normal((batch, mmax, k), 2000 + ci, inputs.X_STD)
        xrs, xbs, yrs, ybs = k, mmax * k, n, mmax * n
    xd = torch.from_numpy(np.ascontiguousarray(x).reshape(-1)).to(dev)
    y_ref, a_ref = oracle.matvec_rows(w, fmt, n, k, x, mmax, xrs, xbs, _all_rows(batch, n))   # [rows, mmax]
    first = None
    for m in ms:
        yd = H.canary(batch * mmax * n + TAIL)
        rem.check(rem.rem_matvec(wd, fmt, n, k, batch, xd, m, xbs, yd, ybs))
        torch.cuda.synchronize()
        y = yd.cpu().numpy()
        assert np.all(y[batch * mmax * n:] == H.CANARY), (fmt, m, "wrote past the end of y")
        got = _check_all(y, y_ref, a_ref, batch, n, m, yrs, ybs, fmt)
        # row exactness on every row: input row 0 of every m equals the first m's
        if first is None:
            first = got[:, 0].copy()
        assert np.array_equal(got[:, 0].view(np.uint32), first.view(np.uint32)), m


def test_full_size_many_rows_and_bias():
    """Q4_K 14336x4096 at m = 16, 32 (rem_matvec_many) and Q8_0 4096x4096 m = 8
    plus a bias vector (rem_matvec_axpby, alpha = beta = 1), every output."""
    dev = H.dev()
    fmt, n, k = "q4_K", 14336, 4096
    w = _weights(fmt, n, k, 1009)
    wd = torch.from_numpy(w.reshape(-1)).to(dev)
    x = inputs.activations(32, k, 2009)
    xd = H.to_dev_f32(x)
    y_ref, a_ref = oracle.matvec_rows(w, fmt, n, k, x, 32, k, 0, _all_rows(1, n))
    for m in (16, 32):
        yd = H.canary(m * n + TAIL)
        rem.check(rem.rem_matvec_many(wd, fmt, n, k, 1, xd, m, k, 0, yd, n, 0, 0))
        torch.cuda.synchronize()
        y = yd.cpu().numpy()
        assert np.all(y[m * n:] == H.CANARY)
        _check_all(y, y_ref, a_ref, 1, n, m, n, 0, "q4_K many")
    fmt, n, k, m = "q8_0", 4096, 4096, 8
    w = _weights(fmt, n, k, 1010)
    wd = torch.from_numpy(w.reshape(-1)).to(dev)
    x = inputs.activations(m, k, 2010)
    bias = inputs.activations(1, n, 3010)[0]
    xd, bd = H.to_dev_f32(x), H.to_dev_f32(bias)
    yd = H.canary(m * n + TAIL)
    rem.check(rem.rem_matvec_axpby(wd, fmt, n, k, 1, xd, m, k, 0, yd, n, 0, 1.0, 1.0, bd, 0, n))
    torch.cuda.synchronize()
    yall = yd.cpu().numpy()
    assert np.all(yall[m * n:] == H.CANARY)
    y_ref, a_ref = oracle.matvec_rows(w, fmt, n, k, x, m, k, 0, _all_rows(1, n))
    got = yall[:m * n].reshape(m, n).T
    ref = y_ref + bias.astype(np.float64)[:, None]
    tol = 1e-4 * a_ref + 1e-7 + 2.0 ** -22 * (np.abs(y_ref) + np.abs(bias)[:, None])
    assert np.all(np.abs(got - ref) <= tol)


def test_full_size_affine_sampled():
    """Affine 4-bit codes in groups of 64, 14336x4096, m = 1..8 through
    rem_matvec_affine (the bench's affine workload shape), every output."""
    bits, gs, n, k = 4, 64, 14336, 4096
    wt = rem.affine_wtype(bits, gs)
    g = np.random.Generator(np.random.PCG64(1013))
    codes = np.empty((n, k * bits // 32), np.uint32)
    sc = np.empty((n, k // gs), np.uint16)
    bi = np.empty((n, k // gs), np.uint16)
    for r0 in range(0, n, 4096):
        r1 = min(n, r0 + 4096)
        v = (g.standard_normal(size=(r1 - r0, k), dtype=np.float32) * np.float32(inputs.W_STD)).astype(np.float32)
        codes[r0:r1], sc[r0:r1], bi[r0:r1] = oracle.affine_quantize(v, bits, gs)
    dev = H.dev()
    cd = torch.from_numpy(codes.view(np.int32).reshape(-1)).to(dev)
    sd = torch.from_numpy(sc.view(np.int16).reshape(-1)).to(dev)
    bd = torch.from_numpy(bi.view(np.int16).reshape(-1)).to(dev)
    x = inputs.activations(8, k, 2013)
    xd = H.to_dev_f32(x)
    y_ref, a_ref = oracle.affine_matvec_rows(codes, sc, bi, bits, gs, n, k, x, 8, k, 0, _all_rows(1, n))
    first = None
    for m in range(1, 9):
        yd = H.canary(m * n + TAIL)
        rem.check(rem.rem_matvec_affine(cd, sd, bd, wt, n, k, 1, xd, m, k, 0, yd, n, 0, 0))
        torch.cuda.synchronize()
        y = yd.cpu().numpy()
        assert np.all(y[m * n:] == H.CANARY)
        got = _check_all(y, y_ref, a_ref, 1, n, m, n, 0, "affine")
        if first is None:
            first = got[:, 0].copy()
        assert np.array_equal(got[:, 0].view(np.uint32), first.view(np.uint32)), m
