"""Lane layouts of the lanes-over-rows (SIMT) engine: one weight row per
lane, two rows per lane, and two lane groups that each hold two rows and half
of the input rows (include/rem.h, rem_schedule.layout; the tests pin one with
rem_set_thread_schedule, and pin the SIMT engine for the formats whose
default engine is the tensor cores).  The arithmetic of every
output is fixed by row exactness (module doc "Row exactness" of mlx-native
0.18.0 src/ops/row_exact_matvec.rs), so every layout must give the same bits,
and those bits must match the oracle.  The cases cover ragged row counts, odd
m (the second lane group repeats one input row), split 1 and split > 1,
batch-major and token-major inputs, the alpha/beta epilogue, affine weights
and the plain (non-TMA) staging path."""
import contextlib

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import quantized_few_row_gb300 as rem
from quantized_few_row_gb300 import inputs
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rem.build()
    rem.load()
    torch.cuda.init()


@contextlib.contextmanager
def pinned(layout):
    rem.check(rem.rem_set_thread_schedule(rem.Schedule(layout=layout, engine=rem.ENGINE_SIMT)))
    try:
        yield
    finally:
        rem.check(rem.rem_set_thread_schedule(None))


@contextlib.contextmanager
def simt():
    rem.check(rem.rem_set_thread_schedule(rem.Schedule(engine=rem.ENGINE_SIMT)))
    try:
        yield
    finally:
        rem.check(rem.rem_set_thread_schedule(None))


def layouts(m, fmt="q8_0"):
    """Layouts with a kernel for (m, fmt): 2 needs m >= 2, 3 needs m in (6, 8) and F16 / BF16; Q6_K has layout 0
    only."""
    if fmt == "q6_K":
        return [0]
    return [0, 1] + ([2] if m >= 2 else []) + ([3] if m in (6, 8) and fmt in ("f16", "bf16") else [])


# (format, n, k, batch, m, split, token-major, weight byte offset)
CASES = [
    ("q8_0", 100, 1024, 1, 5, 0, False, 0),    # ragged n, odd m, automatic split
    ("q4_K", 150, 1024, 1, 1, 0, False, 0),    # m = 1: one or two rows per lane
    ("q8_0", 100, 1024, 1, 8, 1, False, 0),    # split 1: direct stores
    ("q8_0", 90, 512, 1, 6, 0, False, 2),      # plain staging (rows not 16-byte aligned)
    ("q4_K", 70, 1024, 2, 7, 0, False, 0),     # batch-major, odd m
    ("q4_K", 64, 512, 1, 2, 2, False, 0),
    ("q5_0", 96, 1024, 3, 3, 2, True, 0),      # token-major grouped
    ("q5_0", 40, 2048, 1, 8, 8, False, 0),     # split 8 (a full cluster)
    ("f16", 130, 520, 1, 6, 0, False, 0),      # ragged k
    ("f16", 200, 1040, 2, 8, 0, True, 8),      # four rows per lane, token-major, plain staging
    ("f16", 70, 1040, 1, 7, 0, False, 0),
    ("bf16", 64, 264, 2, 4, 3, True, 0),
    ("bf16", 100, 1024, 1, 8, 4, False, 0),
    ("f32", 50, 260, 1, 8, 0, False, 0),
    ("q6_K", 64, 512, 1, 8, 0, False, 0),
    ("q6_K", 70, 2048, 2, 5, 0, True, 0),      # super-blocks at every 2-byte offset of the staged window
    ("q6_K", 33, 768, 1, 3, 3, False, 2),      # plain staging
]


@pytest.mark.parametrize("fmt,n,k,batch,m,split,tm,off", CASES,
                         ids=[f"{c[0]}_n{c[1]}_k{c[2]}_b{c[3]}_m{c[4]}_s{c[5]}{'_tm' if c[6] else ''}"
                              f"{'_plain' if c[7] else ''}" for c in CASES])
def test_layouts_bitwise_equal_and_match_oracle(fmt, n, k, batch, m, split, tm, off):
    w = oracle.quantize(inputs.weights(batch * n, k, 610 + m), fmt)
    if tm:   # x [m, batch*k], y [m, batch*n]
        x = inputs.activations(m, batch * k, 710 + m)
        xrs, xbs, yrs, ybs = batch * k, k, batch * n, n
    else:    # x [batch, m, k], y [batch, m, n]
        x = inputs.activations(batch * m, k, 710 + m)
        xrs, xbs, yrs, ybs = k, m * k, n, m * n
    y_ref, a_ref = oracle.matvec(w, fmt, n, k, batch, x, m, xrs, xbs)
    got = {}
    for lay in layouts(m, fmt):
        with pinned(lay):
            y = H.run_matvec(w, fmt, n, k, batch, x, m, xrs, xbs, yrs, ybs, batch * m * n, split=split,
                             w_offset=off)
        got[lay] = H.gather_y(y, batch, m, n, yrs, ybs)
        H.assert_close_to_oracle(got[lay], y_ref, a_ref, f"layout {lay}")
    with simt():
        auto = H.gather_y(H.run_matvec(w, fmt, n, k, batch, x, m, xrs, xbs, yrs, ybs, batch * m * n, split=split,
                                       w_offset=off), batch, m, n, yrs, ybs)
    for lay, y in got.items():
        assert np.array_equal(y.view(np.uint32), got[0].view(np.uint32)), f"layout {lay} differs from layout 0"
    assert np.array_equal(auto.view(np.uint32), got[0].view(np.uint32))
    # row exactness across layouts: row j alone (m = 1, layout 0) equals row j of every layout
    for j in (0, m - 1):
        xj = x.reshape(-1)
        if tm:
            x1 = xj[j * xrs:j * xrs + batch * k].reshape(1, batch * k)
            with simt():
                y1 = H.run_matvec(w, fmt, n, k, batch, x1, 1, batch * k, k, batch * n, n, batch * n, split=split)
            y1 = H.gather_y(y1, batch, 1, n, batch * n, n)
        else:
            x1 = x.reshape(batch, m, k)[:, j, :].copy()
            with simt():
                y1 = H.run_matvec(w, fmt, n, k, batch, x1, 1, k, k, n, n, batch * n, split=split)
            y1 = H.gather_y(y1, batch, 1, n, n, n)
        assert np.array_equal(y1[:, 0].view(np.uint32), got[0][:, j].view(np.uint32)), f"row {j}"


@pytest.mark.parametrize("fmt", ["q8_0", "q4_K", "f16"])
def test_layouts_epilogue(fmt):
    """alpha * W.x + beta * c: the addend is read at each lane's own input row."""
    n, k, m = 150, {"f16": 1088}.get(fmt, 1024), 5
    w, x = H.contiguous(fmt, n, k, m, 620, 720)
    c = inputs.activations(m, n, 820)
    wh, wp = H.to_dev_bytes(w)
    xd, cd = H.to_dev_f32(x), H.to_dev_f32(c)
    outs = {}
    for lay in layouts(m, fmt):
        yd = H.canary(m * n)
        with pinned(lay):
            rem.check(rem.rem_matvec_axpby(wp, fmt, n, k, 1, xd, m, k, 0, yd, n, 0, -1.75, 0.3, cd, n, 0))
        torch.cuda.synchronize()
        outs[lay] = yd.cpu().numpy()
    y_ref, a_ref = oracle.matvec(w, fmt, n, k, 1, x, m, k, 0)
    ref = -1.75 * y_ref[0] + 0.3 * c.astype(np.float64)
    tol = 1.75 * (1e-4 * a_ref[0] + 1e-7) + 2.0 ** -22 * (np.abs(1.75 * y_ref[0]) + np.abs(0.3 * c))
    for lay, y in outs.items():
        assert np.all(np.abs(y.reshape(m, n) - ref) <= tol), f"layout {lay}"
        assert np.array_equal(y.view(np.uint32), outs[0].view(np.uint32)), f"layout {lay}"


@pytest.mark.parametrize("bits,gs", [(4, 64), (8, 32)])
def test_layouts_affine(bits, gs):
    n, k, batch, m = 75, 1024, 2, 7
    wt = rem.affine_wtype(bits, gs)
    wf = inputs.weights(batch * n, k, 630)
    codes, sc, bi = oracle.affine_quantize(wf, bits, gs)
    x = inputs.activations(batch * m, k, 730)
    y_ref, a_ref = oracle.affine_matvec(codes, sc, bi, bits, gs, n, k, batch, x, m, k, m * k)
    ch, cp = H.to_dev_bytes(np.ascontiguousarray(codes).view(np.uint8))
    sh, sp = H.to_dev_bytes(np.ascontiguousarray(sc).view(np.uint8))
    bh, bp = H.to_dev_bytes(np.ascontiguousarray(bi).view(np.uint8))
    xd = H.to_dev_f32(x)
    outs = {}
    for lay in layouts(m):
        yd = H.canary(batch * m * n)
        with pinned(lay):
            rem.check(rem.rem_matvec_affine(cp, sp, bp, wt, n, k, batch, xd, m, k, m * k, yd, n, m * n, 0))
        torch.cuda.synchronize()
        outs[lay] = H.gather_y(yd.cpu().numpy(), batch, m, n, n, m * n)
        H.assert_close_to_oracle(outs[lay], y_ref, a_ref, f"layout {lay}")
        assert np.array_equal(outs[lay].view(np.uint32), outs[0].view(np.uint32)), f"layout {lay}"


def test_pinned_layout_without_kernel_is_a_launch_error():
    n, k = 64, 512
    w, x = H.contiguous("q8_0", n, k, 2, 640, 740)
    wh, wp = H.to_dev_bytes(w)
    xd = H.to_dev_f32(x)
    yd = H.canary(2 * n)
    with pinned(2):   # two lane groups exist from m = 2 only
        rc = rem.rem_matvec_ex(wp, "q8_0", n, k, 1, xd, 1, k, 0, yd, n, 0, 0, 0)
        err = rem.rem_last_error()
    assert rc == rem.REM_ELAUNCH
    assert "lane layout 2" in err
    torch.cuda.synchronize()
    assert np.all(yd.cpu().numpy() == H.CANARY)
    with pinned(1):   # two rows per lane exist at every m
        rem.check(rem.rem_matvec_ex(wp, "q8_0", n, k, 1, xd, 1, k, 0, yd, n, 0, 0, 0))
