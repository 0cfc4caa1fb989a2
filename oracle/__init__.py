"""CPU oracle for the row-exact few-row quantized mat-vec.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
(``quantized_few_row_gb300``) never does, and shares no code with it.

The arithmetic lives in ``rem_oracle.c`` (plain C, compiled with
``-ffp-contract=off`` so every f32 step is one IEEE-rounded operation).  This
module only marshals numpy arrays through ctypes.  What it follows:

* block sizes and ``row_bytes``: mlx-native 0.18.0
  ``src/ops/row_exact_matvec.rs``, the ``*_BLOCK_*`` constants and
  ``RowExactWeight::row_bytes``;
* the mat-vec: the module doc of the same file, ``y[j, :] = W . x[j, :]``
  for ``1 <= m <= 8`` rows, batched per ``RowExactMatvecShape`` (batch ``b``
  reads weight rows ``b*n..``, input at ``b*x_batch_stride``), summed in f64;
* the block layouts and quantizers: the public GGML layouts of the type names
  the page uses (readings listed in the design notes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rem_oracle.c")
_LIB = os.path.join(_HERE, "librem_oracle.so")

F16, Q8_0, Q4_K, Q6_K, Q5_0, F32, BF16 = 0, 1, 2, 3, 4, 5, 6
WTYPES = {"f16": F16, "q8_0": Q8_0, "q4_K": Q4_K, "q6_K": Q6_K, "q5_0": Q5_0, "f32": F32, "bf16": BF16}

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available); return the path."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-fno-associative-math", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    f32p = ctypes.POINTER(ctypes.c_float)
    f64p = ctypes.POINTER(ctypes.c_double)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    u64p = ctypes.POINTER(ctypes.c_uint64)
    lib.rem_oracle_block_values.argtypes = [ctypes.c_int]
    lib.rem_oracle_block_values.restype = ctypes.c_int
    lib.rem_oracle_block_bytes.argtypes = [ctypes.c_int]
    lib.rem_oracle_block_bytes.restype = ctypes.c_int
    lib.rem_oracle_row_bytes.argtypes = [ctypes.c_int, ctypes.c_uint32]
    lib.rem_oracle_row_bytes.restype = ctypes.c_uint64
    lib.rem_oracle_h2f_array.argtypes = [u16p, f32p, ctypes.c_uint64]
    lib.rem_oracle_h2f_array.restype = None
    lib.rem_oracle_f2h_array.argtypes = [f32p, u16p, ctypes.c_uint64, ctypes.c_int]
    lib.rem_oracle_f2h_array.restype = None
    u32p = ctypes.POINTER(ctypes.c_uint32)
    lib.rem_oracle_affine_dequantize.argtypes = [u32p, u16p, u16p, ctypes.c_int, ctypes.c_int, ctypes.c_uint32,
                                                 ctypes.c_uint32, f32p]
    lib.rem_oracle_affine_dequantize.restype = ctypes.c_int
    lib.rem_oracle_affine_quantize.argtypes = [f32p, ctypes.c_int, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint32,
                                               u32p, u16p, u16p]
    lib.rem_oracle_affine_quantize.restype = ctypes.c_int
    lib.rem_oracle_affine_matvec_rows.argtypes = [u32p, u16p, u16p, ctypes.c_int, ctypes.c_int, ctypes.c_uint32,
                                                  ctypes.c_uint32, f32p, ctypes.c_uint32, ctypes.c_uint64,
                                                  ctypes.c_uint64, ctypes.POINTER(ctypes.c_uint64),
                                                  ctypes.c_uint64, ctypes.POINTER(ctypes.c_double),
                                                  ctypes.POINTER(ctypes.c_double)]
    lib.rem_oracle_affine_matvec_rows.restype = ctypes.c_int
    lib.rem_oracle_bf2f_array.argtypes = [u16p, f32p, ctypes.c_uint64]
    lib.rem_oracle_bf2f_array.restype = None
    lib.rem_oracle_f2bf_array.argtypes = [f32p, u16p, ctypes.c_uint64]
    lib.rem_oracle_f2bf_array.restype = None
    lib.rem_oracle_dequantize.argtypes = [u8p, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint32, f32p]
    lib.rem_oracle_dequantize.restype = ctypes.c_int
    lib.rem_oracle_quantize.argtypes = [f32p, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint32, u8p]
    lib.rem_oracle_quantize.restype = ctypes.c_int
    lib.rem_oracle_matvec_rows.argtypes = [u8p, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint32,
                                           f32p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_uint64,
                                           u64p, ctypes.c_uint64, f64p, f64p]
    lib.rem_oracle_matvec_rows.restype = ctypes.c_int
    lib.rem_oracle_threads.argtypes = []
    lib.rem_oracle_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def wtype_of(w) -> int:
    return WTYPES[w] if isinstance(w, str) else int(w)


def block_values(wtype) -> int:
    return _load().rem_oracle_block_values(wtype_of(wtype))


def block_bytes(wtype) -> int:
    return _load().rem_oracle_block_bytes(wtype_of(wtype))


def row_bytes(wtype, k: int) -> int:
    return int(_load().rem_oracle_row_bytes(wtype_of(wtype), k))


def threads() -> int:
    return int(_load().rem_oracle_threads())


def h2f(h: np.ndarray) -> np.ndarray:
    """Exact binary16 -> binary32 widening of uint16 bit patterns."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _load().rem_oracle_h2f_array(_ptr(h, ctypes.c_uint16), _ptr(out, ctypes.c_float), h.size)
    return out


def f2h(f: np.ndarray, mode: str = "rn") -> np.ndarray:
    """binary32 -> binary16 bit patterns; mode 'rn' (nearest even) or 'ru' (toward +inf)."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    _load().rem_oracle_f2h_array(_ptr(f, ctypes.c_float), _ptr(out, ctypes.c_uint16), f.size,
                                 {"rn": 0, "ru": 1}[mode])
    return out


def bf2f(b: np.ndarray) -> np.ndarray:
    """Exact bfloat16 -> binary32 widening of uint16 bit patterns."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float32)
    _load().rem_oracle_bf2f_array(_ptr(b, ctypes.c_uint16), _ptr(out, ctypes.c_float), b.size)
    return out


def f2bf(f: np.ndarray) -> np.ndarray:
    """binary32 -> bfloat16 bit patterns, round to nearest even."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    _load().rem_oracle_f2bf_array(_ptr(f, ctypes.c_float), _ptr(out, ctypes.c_uint16), f.size)
    return out


def affine_quantize(values: np.ndarray, bits: int, group_size: int):
    """Affine test data: (codes uint32 [rows, k*bits/32], scales uint16 [rows, k/gs],
    biases uint16 [rows, k/gs]) from float rows [rows, k]."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    rows, k = v.shape
    codes = np.empty((rows, k * bits // 32), dtype=np.uint32)
    sc = np.empty((rows, k // group_size), dtype=np.uint16)
    bi = np.empty((rows, k // group_size), dtype=np.uint16)
    rc = _load().rem_oracle_affine_quantize(_ptr(v, ctypes.c_float), bits, group_size, rows, k,
                                            _ptr(codes, ctypes.c_uint32), _ptr(sc, ctypes.c_uint16),
                                            _ptr(bi, ctypes.c_uint16))
    if rc != 0:
        raise ValueError(f"affine_quantize: bad bits {bits} / group size {group_size} / k {k}")
    return codes, sc, bi


def affine_dequantize(codes, scales, biases, bits: int, group_size: int, rows: int, k: int) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint32)
    s = np.ascontiguousarray(scales, dtype=np.uint16)
    b = np.ascontiguousarray(biases, dtype=np.uint16)
    out = np.empty((rows, k), dtype=np.float32)
    rc = _load().rem_oracle_affine_dequantize(_ptr(c, ctypes.c_uint32), _ptr(s, ctypes.c_uint16),
                                              _ptr(b, ctypes.c_uint16), bits, group_size, rows, k,
                                              _ptr(out, ctypes.c_float))
    if rc != 0:
        raise ValueError("affine_dequantize: bad arguments")
    return out


def affine_matvec_rows(codes, scales, biases, bits: int, group_size: int, n: int, k: int, x: np.ndarray, m: int,
                       x_row_stride: int, x_batch_stride: int, rows):
    """f64 y and sum|w*x| for selected global rows of an affine weight; [len(rows), m]."""
    c = np.ascontiguousarray(codes, dtype=np.uint32).reshape(-1)
    s = np.ascontiguousarray(scales, dtype=np.uint16).reshape(-1)
    b = np.ascontiguousarray(biases, dtype=np.uint16).reshape(-1)
    xf = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    r = np.ascontiguousarray(rows, dtype=np.uint64).reshape(-1)
    y = np.empty((r.size, m), dtype=np.float64)
    a = np.empty((r.size, m), dtype=np.float64)
    rc = _load().rem_oracle_affine_matvec_rows(_ptr(c, ctypes.c_uint32), _ptr(s, ctypes.c_uint16),
                                               _ptr(b, ctypes.c_uint16), bits, group_size, n, k,
                                               _ptr(xf, ctypes.c_float), m, x_row_stride, x_batch_stride,
                                               _ptr(r, ctypes.c_uint64), r.size, _ptr(y, ctypes.c_double),
                                               _ptr(a, ctypes.c_double))
    if rc != 0:
        raise RuntimeError(f"oracle affine matvec failed ({rc})")
    return y, a


def affine_matvec(codes, scales, biases, bits: int, group_size: int, n: int, k: int, batch: int, x: np.ndarray,
                  m: int, x_row_stride: int, x_batch_stride: int):
    """f64 y[b, j, i] and A[b, j, i] for every output of an affine product."""
    rows = np.arange(batch * n, dtype=np.uint64)
    y, a = affine_matvec_rows(codes, scales, biases, bits, group_size, n, k, x, m, x_row_stride, x_batch_stride,
                              rows)
    return (y.reshape(batch, n, m).transpose(0, 2, 1).copy(), a.reshape(batch, n, m).transpose(0, 2, 1).copy())


def quantize(values: np.ndarray, wtype) -> np.ndarray:
    """Quantize float rows [rows, k] into block bytes [rows, row_bytes]."""
    wt = wtype_of(wtype)
    v = np.ascontiguousarray(values, dtype=np.float32)
    assert v.ndim == 2
    rows, k = v.shape
    out = np.empty((rows, row_bytes(wt, k)), dtype=np.uint8)
    rc = _load().rem_oracle_quantize(_ptr(v, ctypes.c_float), wt, rows, k, _ptr(out, ctypes.c_uint8))
    if rc != 0:
        raise ValueError(f"oracle quantize rejected wtype={wtype} k={k}")
    return out


def dequantize(w: np.ndarray, wtype, rows: int, k: int) -> np.ndarray:
    """Exact f32 weights [rows, k] of block bytes (row-major, row_bytes apart)."""
    wt = wtype_of(wtype)
    wb = np.ascontiguousarray(w, dtype=np.uint8).reshape(-1)
    assert wb.size >= rows * row_bytes(wt, k)
    out = np.empty((rows, k), dtype=np.float32)
    rc = _load().rem_oracle_dequantize(_ptr(wb, ctypes.c_uint8), wt, rows, k, _ptr(out, ctypes.c_float))
    if rc != 0:
        raise ValueError("oracle dequantize rejected its arguments")
    return out


def matvec_rows(w: np.ndarray, wtype, n: int, k: int, x: np.ndarray, m: int,
                x_row_stride: int, x_batch_stride: int, rows) -> tuple[np.ndarray, np.ndarray]:
    """f64 y and sum|w*x| for selected global weight rows (b*n + i).

    ``x`` is the flat f32 input; input row j of batch b starts at
    ``b*x_batch_stride + j*x_row_stride``.  Returns arrays [len(rows), m].
    """
    wt = wtype_of(wtype)
    wb = np.ascontiguousarray(w, dtype=np.uint8).reshape(-1)
    xf = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    r = np.ascontiguousarray(rows, dtype=np.uint64).reshape(-1)
    y = np.empty((r.size, m), dtype=np.float64)
    a = np.empty((r.size, m), dtype=np.float64)
    rc = _load().rem_oracle_matvec_rows(_ptr(wb, ctypes.c_uint8), wt, n, k, _ptr(xf, ctypes.c_float), m,
                                        x_row_stride, x_batch_stride, _ptr(r, ctypes.c_uint64), r.size,
                                        _ptr(y, ctypes.c_double), _ptr(a, ctypes.c_double))
    if rc != 0:
        raise RuntimeError(f"oracle matvec failed ({rc})")
    return y, a


def matvec(w: np.ndarray, wtype, n: int, k: int, batch: int, x: np.ndarray, m: int,
           x_row_stride: int, x_batch_stride: int) -> tuple[np.ndarray, np.ndarray]:
    """f64 y[b, j, i] and A[b, j, i] for every output of a (batched) product."""
    rows = np.arange(batch * n, dtype=np.uint64)
    y, a = matvec_rows(w, wtype, n, k, x, m, x_row_stride, x_batch_stride, rows)
    y = y.reshape(batch, n, m).transpose(0, 2, 1).copy()
    a = a.reshape(batch, n, m).transpose(0, 2, 1).copy()
    return y, a


def within_tolerance(y_gpu: np.ndarray, y_ref: np.ndarray, a_ref: np.ndarray,
                     rel: float = 1e-4, abs_: float = 1e-7) -> np.ndarray:
    """Elementwise acceptance: |y - y_ref| <= rel*A + abs where y_ref is finite;
    a non-finite reference demands a non-finite result."""
    y = np.asarray(y_gpu, dtype=np.float64)
    finite = np.isfinite(y_ref)
    ok = np.empty(y.shape, dtype=bool)
    ok[finite] = np.abs(y[finite] - y_ref[finite]) <= rel * a_ref[finite] + abs_
    ok[~finite] = ~np.isfinite(y[~finite])
    return ok


__all__ = ["build", "F16", "Q8_0", "Q4_K", "Q6_K", "Q5_0", "F32", "BF16", "WTYPES", "block_values", "block_bytes",
           "row_bytes", "threads", "h2f", "f2h", "bf2f", "f2bf", "affine_quantize", "affine_dequantize", "affine_matvec",
           "affine_matvec_rows", "quantize", "dequantize", "matvec", "matvec_rows",
           "within_tolerance", "wtype_of"]
