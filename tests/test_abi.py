"""The C ABI without a GPU: the library loads, exports what include/rem.h
declares, and its host-side rules (row_bytes, split factor, argument
validation) behave as specified.  Every call here returns before any CUDA
call is made (invalid arguments are rejected first)."""
import os
import re

import pytest

import quantized_few_row_gb300 as rem

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rem.h")


@pytest.fixture(scope="module")
def lib():
    rem.build()
    return rem.load()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(rem_[a-z_]+)\s*\(", src))


def test_header_declares_the_binding_names():
    assert _declared() == set(rem.C_FUNCTIONS)


def test_exports_every_declared_symbol(lib):
    for name in _declared():
        assert getattr(lib, name) is not None
    assert rem.rem_version() == 2


@pytest.mark.parametrize("wt,k,expect", [
    ("f16", 512, 1024), ("q8_0", 4096, 4352), ("q4_K", 4096, 2304), ("q6_K", 4096, 3360),
    ("q5_0", 4096, 2816), ("q8_0", 32, 34), ("q5_0", 32, 22), ("q4_K", 256, 144), ("q6_K", 256, 210),
    ("f32", 4096, 16384), ("bf16", 4096, 8192), ("f32", 4, 16), ("bf16", 4, 8),
])
def test_row_bytes(lib, wt, k, expect):
    assert rem.rem_row_bytes(wt, k) == expect


def test_row_bytes_unknown_type(lib):
    assert rem.rem_row_bytes(99, 4096) == 0


@pytest.mark.parametrize("wt,rows,k,expect", [
    ("q8_0", 4096, 4096, 8),     # 128 row groups -> 2048/128 = 16, capped at 8
    ("q4_K", 14336, 4096, 4),    # 448 row groups -> 4
    ("q6_K", 128256, 4096, 1),   # 4008 row groups -> 1
    ("q5_0", 16384, 4096, 4),    # 512 row groups -> 4
    ("f16", 256, 512, 8),        # 8 groups -> 256, capped at 8 (8 chunks of 72 values)
    ("f16", 256, 144, 2),        # 2 chunks of 72 values
    ("q4_K", 32, 256, 1),        # one chunk per row
])
def test_split_factor_from_shape(lib, wt, rows, k, expect):
    assert rem.rem_split_factor(wt, rows, k) == expect
    assert rem.rem_split_factor(wt, rows, k) == expect   # no state, no m


def test_split_factor_degenerate(lib):
    assert rem.rem_split_factor("q8_0", 0, 4096) == 0
    assert rem.rem_split_factor("q8_0", 64, 0) == 0
    assert rem.rem_split_factor(99, 64, 256) == 0


W, X, Y = 0x100000, 0x200000, 0x300000     # aligned fake addresses, never dereferenced


def _ex(**kw):
    a = dict(W=W, wtype="q8_0", n=64, k=256, batch=1, x=X, m=2, x_row_stride=256, x_batch_stride=0,
             y=Y, y_row_stride=64, y_batch_stride=0, split=0, rows_per_cta=0)
    a.update(kw)
    return rem.rem_matvec_ex(a["W"], a["wtype"], a["n"], a["k"], a["batch"], a["x"], a["m"],
                             a["x_row_stride"], a["x_batch_stride"], a["y"], a["y_row_stride"],
                             a["y_batch_stride"], a["split"], a["rows_per_cta"], stream=0)


CASES = [
    ("m0", dict(m=0), "m (0) must be in 1..=8"),
    ("m9", dict(m=9), "m (9) must be in 1..=8"),
    ("n0", dict(n=0), "must be > 0"),
    ("k0", dict(k=0), "must be > 0"),
    ("batch0", dict(batch=0), "must be > 0"),
    ("split", dict(split=17), "split (17)"),
    ("rows_per_cta", dict(rows_per_cta=48), "rows_per_cta (48)"),
    ("rows_per_cta256", dict(rows_per_cta=256), "rows_per_cta (256)"),
    ("wtype", dict(wtype=99), "unknown weight type"),
    ("nullW", dict(W=0), "non-null"),
    ("nullx", dict(x=0), "non-null"),
    ("nully", dict(y=0), "non-null"),
    ("k_q8", dict(k=100, x_row_stride=100), "multiple of 32"),
    ("k_f16", dict(wtype="f16", k=6, x_row_stride=8), "multiple of 4"),
    ("k_f32", dict(wtype="f32", k=6, x_row_stride=8), "multiple of 4"),
    ("k_bf16", dict(wtype="bf16", k=10, x_row_stride=12), "multiple of 4"),
    ("w_f32", dict(wtype="f32", W=W + 2), "4-byte"),
    ("k_q4k", dict(wtype="q4_K", k=288, x_row_stride=288), "multiple of 256"),
    ("k_q6k", dict(wtype="q6_K", k=128, x_row_stride=128), "multiple of 256"),
    ("k_q5", dict(wtype="q5_0", k=48, x_row_stride=48), "multiple of 32"),
    ("xrs", dict(x_row_stride=258), "input strides"),
    ("xbs", dict(batch=2, x_batch_stride=514, x_row_stride=256, y_batch_stride=128), "input strides"),
    ("xalign", dict(x=X + 4), "16-byte aligned"),
    ("walign_q4k", dict(wtype="q4_K", W=W + 8), "16-byte"),
    ("walign_f16", dict(wtype="f16", W=W + 4), "8-byte"),
    ("walign_q8", dict(W=W + 1), "2-byte"),
    ("walign_q6k", dict(wtype="q6_K", W=W + 1), "2-byte"),
    ("walign_q5", dict(wtype="q5_0", W=W + 1), "2-byte"),
    ("yalign", dict(y=Y + 2), "output pointer 4-byte"),
    ("rows_overlap", dict(m=2, y_row_stride=63), "overlap"),
    ("batch_overlap_m1", dict(m=1, batch=2, x_batch_stride=256, y_batch_stride=63), "overlap"),
    ("batch_major_overlap", dict(m=2, batch=2, x_batch_stride=512, y_row_stride=64, y_batch_stride=100),
     "overlap"),
    ("token_major_overlap", dict(m=2, batch=2, x_row_stride=512, x_batch_stride=256, y_row_stride=127,
                                 y_batch_stride=64), "overlap"),
    ("row_extent_u32", dict(m=8, y_row_stride=1 << 30), "exceeds u32"),
]


@pytest.mark.parametrize("name,kw,msg", CASES, ids=[c[0] for c in CASES])
def test_validation_rejects(lib, name, kw, msg):
    assert _ex(**kw) == rem.REM_EINVAL
    err = rem.rem_last_error()
    assert err.startswith("rem_matvec:"), err
    assert msg in err, err


def test_inferred_token_major_strides_validate(lib):
    # rem_matvec with batch > 1 and x_batch_stride < m*k infers x_row_stride =
    # batch*k and y_row_stride = batch*n; overlapping inferred outputs are
    # still rejected: y_batch_stride < n
    rc = rem.rem_matvec(W, "q8_0", 64, 256, 4, X, 2, 256, Y, 32, stream=0)
    assert rc == rem.REM_EINVAL and "overlap" in rem.rem_last_error()


def test_dequantize_and_quantize_validate(lib):
    assert rem.rem_dequantize(W, "q4_K", 4, 300, Y, stream=0) == rem.REM_EINVAL
    assert "rem_dequantize" in rem.rem_last_error()
    assert rem.rem_dequantize(W + 8, "q4_K", 4, 256, Y, stream=0) == rem.REM_EINVAL
    assert rem.rem_quantize(X, "q8_0", 0, 256, W, stream=0) == rem.REM_EINVAL
    assert rem.rem_quantize(0, "q8_0", 4, 256, W, stream=0) == rem.REM_EINVAL
    assert "rem_quantize" in rem.rem_last_error()


def _many(**kw):
    a = dict(W=W, wtype="q8_0", n=64, k=256, batch=1, x=X, m=12, x_row_stride=256, x_batch_stride=0,
             y=Y, y_row_stride=64, y_batch_stride=0, split=0)
    a.update(kw)
    return rem.rem_matvec_many(a["W"], a["wtype"], a["n"], a["k"], a["batch"], a["x"], a["m"],
                               a["x_row_stride"], a["x_batch_stride"], a["y"], a["y_row_stride"],
                               a["y_batch_stride"], a["split"], stream=0)


@pytest.mark.parametrize("kw,msg", [
    (dict(m=0), "m (0) must be >= 1"),
    (dict(y_row_stride=63), "overlap"),             # rows 0..11 of 64 outputs overlap
    (dict(k=100, x_row_stride=100), "multiple of 32"),
    (dict(split=17), "split (17)"),
    (dict(m=20, y_row_stride=1 << 28), "exceeds u32"),  # (m-1)*y_row_stride + n past 2^32
], ids=["m0", "overlap", "k", "split", "extent"])
def test_many_rows_validation_rejects(lib, kw, msg):
    """rem_matvec_many checks the rules over all m rows (not only per group of
    8) before it launches anything; fake pointers are never dereferenced."""
    assert _many(**kw) == rem.REM_EINVAL
    assert msg in rem.rem_last_error(), rem.rem_last_error()


def _axpby(**kw):
    a = dict(W=W, wtype="q8_0", n=64, k=256, batch=1, x=X, m=2, x_row_stride=256, x_batch_stride=0,
             y=Y, y_row_stride=64, y_batch_stride=0, alpha=2.0, beta=0.5, c=0x400000, c_row_stride=64,
             c_batch_stride=0)
    a.update(kw)
    return rem.rem_matvec_axpby(a["W"], a["wtype"], a["n"], a["k"], a["batch"], a["x"], a["m"],
                                a["x_row_stride"], a["x_batch_stride"], a["y"], a["y_row_stride"],
                                a["y_batch_stride"], a["alpha"], a["beta"], a["c"], a["c_row_stride"],
                                a["c_batch_stride"], stream=0)


@pytest.mark.parametrize("kw,msg", [
    (dict(c=0), "c must be non-null"),
    (dict(c=0x400002), "c must be non-null and 4-byte aligned"),
    (dict(c=Y + 4), "c overlaps y"),                       # shifted by one element
    (dict(c=Y, c_row_stride=0), "c overlaps y"),           # same base, other strides
], ids=["null", "misaligned", "shifted", "strides"])
def test_axpby_addend_rules(lib, kw, msg):
    """The addend is checked before anything else happens: non-null and
    aligned when beta != 0, and either disjoint from y or y itself with the
    same strides."""
    assert _axpby(**kw) == rem.REM_EINVAL
    assert msg in rem.rem_last_error(), rem.rem_last_error()


def test_affine_types_need_the_affine_entry(lib):
    """An affine weight type through rem_matvec_ex (no scales) is refused, as
    is a non-affine type, a null scale array or a k off the group size
    through rem_matvec_affine; rem_dequantize and rem_quantize refuse affine
    types."""
    assert _ex(wtype=rem.A4_G64, k=256, x_row_stride=256) == rem.REM_EINVAL
    assert "rem_matvec_affine" in rem.rem_last_error()
    aff = lambda **kw: rem.rem_matvec_affine(kw.get("codes", W), kw.get("scales", 0x500000), kw.get("biases", 0x600000),
                                             kw.get("wtype", rem.A4_G64), 64, kw.get("k", 256), 1, X, 2, 256, 0, Y, 64,
                                             0, 0, stream=0)
    assert aff(wtype=rem.Q8_0) == rem.REM_EINVAL and "not an affine" in rem.rem_last_error()
    assert aff(scales=0) == rem.REM_EINVAL and "scales and biases" in rem.rem_last_error()
    assert aff(k=96) == rem.REM_EINVAL and "multiple of 64" in rem.rem_last_error()
    assert rem.rem_dequantize(W, rem.A8_G32, 4, 256, Y, stream=0) == rem.REM_EINVAL
    assert rem.rem_quantize(X, rem.A8_G32, 4, 256, W, stream=0) == rem.REM_EINVAL
    assert rem.rem_row_bytes(rem.A4_G32, 4096) == 2048 and rem.rem_row_bytes(rem.A8_G128, 4096) == 4096
    # 3, 5 and 6 bits: k*bits/8 bytes (packing units of 3, 5 and 3 bytes)
    assert rem.rem_row_bytes(rem.A3_G32, 4096) == 1536 and rem.rem_row_bytes(rem.A5_G64, 4096) == 2560
    assert rem.rem_row_bytes(rem.A6_G128, 4096) == 3072 and rem.rem_row_bytes(rem.A3_G128, 128) == 48


@pytest.mark.parametrize("wt,rows,k,expect", [
    ("q6_K", 128256, 4096, rem.ENGINE_TC), ("q6_K", 256, 512, rem.ENGINE_TC), ("q8_0", 4096, 4096, rem.ENGINE_SIMT),
    ("q5_0", 16384, 4096, rem.ENGINE_SIMT),
    ("q4_K", 14336, 4096, rem.ENGINE_SIMT), ("f16", 256, 512, rem.ENGINE_SIMT), ("bf16", 64, 256, rem.ENGINE_SIMT),
    ("f32", 64, 256, rem.ENGINE_SIMT), (rem.A4_G64, 64, 256, rem.ENGINE_SIMT),
])
def test_engine_from_shape(lib, wt, rows, k, expect):
    assert rem.rem_engine_of(wt, rows, k) == expect
    assert rem.rem_engine_of(wt, rows, k) == expect     # no state


def test_engine_degenerate(lib):
    assert rem.rem_engine_of(99, 64, 256) == -1
    assert rem.rem_engine_of("q8_0", 0, 256) == -1
    assert rem.rem_engine_of("q8_0", 64, 0) == -1


def _sched(sched, **kw):
    a = dict(W=W, wtype="q8_0", n=64, k=256, batch=1, x=X, m=2, x_row_stride=256, x_batch_stride=0,
             y=Y, y_row_stride=64, y_batch_stride=0)
    a.update(kw)
    return rem.rem_matvec_sched(a["W"], a["wtype"], a["n"], a["k"], a["batch"], a["x"], a["m"],
                                a["x_row_stride"], a["x_batch_stride"], a["y"], a["y_row_stride"],
                                a["y_batch_stride"], sched, stream=0)


@pytest.mark.parametrize("sched,kw,msg", [
    (rem.Schedule(layout=4), {}, "layout (4)"),
    (rem.Schedule(layout=-2), {}, "layout (-2)"),
    (rem.Schedule(engine=2), {}, "engine (2)"),
    (rem.Schedule(engine=rem.ENGINE_TC), dict(wtype="q4_K"), "tensor-core engine takes"),
    (rem.Schedule(engine=rem.ENGINE_TC), dict(wtype="f16"), "tensor-core engine takes"),
    (rem.Schedule(split=17), {}, "split (17)"),
    (rem.Schedule(), dict(m=0), "m (0) must be >= 1"),
    (rem.Schedule(), dict(m=20, y_row_stride=63), "overlap"),
], ids=["layout4", "layout-2", "engine2", "tc_q4k", "tc_f16", "split", "m0", "overlap"])
def test_schedule_rules(lib, sched, kw, msg):
    """rem_matvec_sched refuses schedule fields out of range and the
    tensor-core engine on a format it does not take, before any CUDA call."""
    assert _sched(sched, **kw) == rem.REM_EINVAL
    assert msg in rem.rem_last_error(), rem.rem_last_error()


def test_few_row_entry_points_keep_eight_rows(lib):
    """rem_matvec_ex and rem_matvec_axpby take at most 8 input rows on either
    engine (the page's per-dispatch limit); more rows go through
    rem_matvec_many or rem_matvec_sched."""
    for wt in ("q8_0", "q6_K", "q4_K"):
        k = 256
        assert _ex(wtype=wt, m=9, k=k, x_row_stride=k) == rem.REM_EINVAL
        assert "1..=8" in rem.rem_last_error(), rem.rem_last_error()
