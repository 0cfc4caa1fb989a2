"""Row-exact few-row quantized mat-vec for GB300 (sm_103a).

Python binding of ``librem.so`` (C ABI in ``include/rem.h``).  The functions
keep the C names and only marshal arguments: tensors become device pointers
(``data_ptr()``), streams become ``cudaStream_t`` handles.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback, and a
missing library raises instead of computing anything.

The operation (mlx-native 0.18.0 src/ops/row_exact_matvec.rs):
``y[b, j, :] = W[b] . x[b, j, :]`` for ``1 <= m <= 8`` F32 input rows against
F16 / Q8_0 / Q4_K / Q6_K / Q5_0 weights, with F32 output, bitwise identical
per output row for any m.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "F16", "Q8_0", "Q4_K", "Q6_K", "Q5_0", "F32", "BF16", "A4_G32", "A4_G64", "A4_G128", "A8_G32", "A8_G64",
    "A8_G128", "A3_G32", "A3_G64", "A3_G128", "A5_G32", "A5_G64", "A5_G128", "A6_G32", "A6_G64", "A6_G128",
    "WTYPES", "affine_wtype", "rem_matvec_affine", "rem_dequantize_affine", "REM_OK", "REM_EINVAL", "REM_ELAUNCH", "REM_ECUDA",
    "RemError", "build", "library_path", "load", "rem_matvec", "rem_matvec_ex", "rem_matvec_many",
    "rem_matvec_axpby", "rem_row_bytes",
    "rem_split_factor", "rem_dequantize", "rem_quantize", "rem_last_error", "rem_version", "check",
    "C_FUNCTIONS", "Schedule", "rem_matvec_sched", "rem_engine_of", "rem_device_status", "rem_last_plan",
    "ENGINE_AUTO", "ENGINE_SIMT", "ENGINE_TC", "TEST_SKIP_FIRST_STAGE", "rem_set_thread_schedule",
]

F16, Q8_0, Q4_K, Q6_K, Q5_0, F32, BF16 = 0, 1, 2, 3, 4, 5, 6
A4_G32, A4_G64, A4_G128, A8_G32, A8_G64, A8_G128 = 7, 8, 9, 10, 11, 12
A3_G32, A3_G64, A3_G128, A5_G32, A5_G64, A5_G128, A6_G32, A6_G64, A6_G128 = 13, 14, 15, 16, 17, 18, 19, 20, 21
WTYPES = {"f16": F16, "q8_0": Q8_0, "q4_K": Q4_K, "q6_K": Q6_K, "q5_0": Q5_0, "f32": F32, "bf16": BF16,
          "a4_g32": A4_G32, "a4_g64": A4_G64, "a4_g128": A4_G128, "a8_g32": A8_G32, "a8_g64": A8_G64,
          "a8_g128": A8_G128, "a3_g32": A3_G32, "a3_g64": A3_G64, "a3_g128": A3_G128, "a5_g32": A5_G32,
          "a5_g64": A5_G64, "a5_g128": A5_G128, "a6_g32": A6_G32, "a6_g64": A6_G64, "a6_g128": A6_G128}


def affine_wtype(bits: int, group_size: int) -> int:
    """The weight type of affine codes of `bits` bits in groups of `group_size`."""
    return WTYPES[f"a{bits}_g{group_size}"]
REM_OK, REM_EINVAL, REM_ELAUNCH, REM_ECUDA = 0, -1, -2, -3
ENGINE_AUTO, ENGINE_SIMT, ENGINE_TC = -1, 0, 1
TEST_SKIP_FIRST_STAGE = 1
C_FUNCTIONS = ("rem_matvec", "rem_matvec_ex", "rem_matvec_many", "rem_matvec_axpby", "rem_matvec_affine",
               "rem_dequantize_affine", "rem_row_bytes", "rem_split_factor",
               "rem_dequantize", "rem_quantize", "rem_last_error", "rem_version", "rem_matvec_sched",
               "rem_engine_of", "rem_device_status", "rem_last_plan", "rem_set_thread_schedule")


class Schedule(ctypes.Structure):
    """rem_schedule: split, rows_per_cta, layout, engine, wait_ns, test_flags (zero / -1 = default)."""
    _fields_ = [("split", ctypes.c_uint32), ("rows_per_cta", ctypes.c_uint32), ("layout", ctypes.c_int32),
                ("engine", ctypes.c_int32), ("wait_ns", ctypes.c_uint64), ("test_flags", ctypes.c_uint32)]

    def __init__(self, split=0, rows_per_cta=0, layout=-1, engine=-1, wait_ns=0, test_flags=0):
        super().__init__(split, rows_per_cta, layout, engine, wait_ns, test_flags)

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "librem.so")
_lib = None


class RemError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def build(force: bool = False) -> str:
    """Compile librem.so in-tree with nvcc (sm_103a)."""
    from ._build import build as _b
    return _b(force=force)


def load():
    """Load librem.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with quantized_few_row_gb300.build() "
                           "(nvcc, sm_103a); there is no non-CUDA implementation")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, u32, u64, i32 = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int
    lib.rem_matvec.argtypes = [vp, i32, u32, u32, u32, vp, u32, u32, vp, u32, vp]
    lib.rem_matvec.restype = i32
    lib.rem_matvec_ex.argtypes = [vp, i32, u32, u32, u32, vp, u32, u32, u32, vp, u32, u32, u32, u32, vp]
    lib.rem_matvec_ex.restype = i32
    lib.rem_matvec_many.argtypes = [vp, i32, u32, u32, u32, vp, u32, u32, u32, vp, u32, u32, u32, vp]
    lib.rem_matvec_many.restype = i32
    f32 = ctypes.c_float
    lib.rem_matvec_axpby.argtypes = [vp, i32, u32, u32, u32, vp, u32, u32, u32, vp, u32, u32, f32, f32, vp, u32,
                                     u32, vp]
    lib.rem_matvec_axpby.restype = i32
    lib.rem_matvec_affine.argtypes = [vp, vp, vp, i32, u32, u32, u32, vp, u32, u32, u32, vp, u32, u32, u32, vp]
    lib.rem_matvec_affine.restype = i32
    lib.rem_dequantize_affine.argtypes = [vp, vp, vp, i32, u32, u32, vp, vp]
    lib.rem_dequantize_affine.restype = i32
    lib.rem_row_bytes.argtypes = [i32, u32]
    lib.rem_row_bytes.restype = u64
    lib.rem_split_factor.argtypes = [i32, u32, u32]
    lib.rem_split_factor.restype = u32
    lib.rem_dequantize.argtypes = [vp, i32, u32, u32, vp, vp]
    lib.rem_dequantize.restype = i32
    lib.rem_quantize.argtypes = [vp, i32, u32, u32, vp, vp]
    lib.rem_quantize.restype = i32
    lib.rem_last_error.argtypes = []
    lib.rem_last_error.restype = ctypes.c_char_p
    lib.rem_version.argtypes = []
    lib.rem_version.restype = i32
    lib.rem_matvec_sched.argtypes = [vp, i32, u32, u32, u32, vp, u32, u32, u32, vp, u32, u32,
                                     ctypes.POINTER(Schedule), vp]
    lib.rem_matvec_sched.restype = i32
    lib.rem_engine_of.argtypes = [i32, u32, u32]
    lib.rem_engine_of.restype = i32
    lib.rem_device_status.argtypes = [i32]
    lib.rem_device_status.restype = i32
    lib.rem_set_thread_schedule.argtypes = [ctypes.POINTER(Schedule)]
    lib.rem_set_thread_schedule.restype = i32
    lib.rem_last_plan.argtypes = []
    lib.rem_last_plan.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _wt(wtype) -> int:
    return WTYPES[wtype] if isinstance(wtype, str) else int(wtype)


def _ptr(obj) -> int:
    """Device address of a tensor, or an integer address as is."""
    if obj is None:
        return 0
    if isinstance(obj, int):
        return obj
    if hasattr(obj, "data_ptr"):
        return int(obj.data_ptr())
    raise TypeError(f"cannot take the address of {type(obj)!r}")


def _stream(stream) -> int:
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return int(torch.cuda.current_stream().cuda_stream)
        except ImportError:
            pass
        return 0
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def rem_matvec(W, wtype, n: int, k: int, batch: int, x, m: int, x_batch_stride: int, y,
               y_batch_stride: int, stream=None) -> int:
    return load().rem_matvec(_ptr(W), _wt(wtype), n, k, batch, _ptr(x), m, x_batch_stride, _ptr(y),
                             y_batch_stride, _stream(stream))


def rem_matvec_ex(W, wtype, n: int, k: int, batch: int, x, m: int, x_row_stride: int, x_batch_stride: int,
                  y, y_row_stride: int, y_batch_stride: int, split: int = 0, rows_per_cta: int = 0,
                  stream=None) -> int:
    return load().rem_matvec_ex(_ptr(W), _wt(wtype), n, k, batch, _ptr(x), m, x_row_stride, x_batch_stride,
                                _ptr(y), y_row_stride, y_batch_stride, split, rows_per_cta, _stream(stream))


def rem_matvec_many(W, wtype, n: int, k: int, batch: int, x, m: int, x_row_stride: int, x_batch_stride: int,
                    y, y_row_stride: int, y_batch_stride: int, split: int = 0, stream=None) -> int:
    return load().rem_matvec_many(_ptr(W), _wt(wtype), n, k, batch, _ptr(x), m, x_row_stride, x_batch_stride,
                                  _ptr(y), y_row_stride, y_batch_stride, split, _stream(stream))


def rem_matvec_axpby(W, wtype, n: int, k: int, batch: int, x, m: int, x_row_stride: int, x_batch_stride: int,
                     y, y_row_stride: int, y_batch_stride: int, alpha: float, beta: float, c=None,
                     c_row_stride: int = 0, c_batch_stride: int = 0, stream=None) -> int:
    return load().rem_matvec_axpby(_ptr(W), _wt(wtype), n, k, batch, _ptr(x), m, x_row_stride, x_batch_stride,
                                   _ptr(y), y_row_stride, y_batch_stride, alpha, beta, _ptr(c), c_row_stride,
                                   c_batch_stride, _stream(stream))


def rem_matvec_affine(codes, scales, biases, wtype, n: int, k: int, batch: int, x, m: int, x_row_stride: int,
                      x_batch_stride: int, y, y_row_stride: int, y_batch_stride: int, split: int = 0,
                      stream=None) -> int:
    return load().rem_matvec_affine(_ptr(codes), _ptr(scales), _ptr(biases), _wt(wtype), n, k, batch, _ptr(x), m,
                                    x_row_stride, x_batch_stride, _ptr(y), y_row_stride, y_batch_stride, split,
                                    _stream(stream))


def rem_dequantize_affine(codes, scales, biases, wtype, rows: int, k: int, out, stream=None) -> int:
    return load().rem_dequantize_affine(_ptr(codes), _ptr(scales), _ptr(biases), _wt(wtype), rows, k, _ptr(out),
                                        _stream(stream))


def rem_matvec_sched(W, wtype, n: int, k: int, batch: int, x, m: int, x_row_stride: int, x_batch_stride: int,
                     y, y_row_stride: int, y_batch_stride: int, sched: Schedule | None = None, stream=None) -> int:
    return load().rem_matvec_sched(_ptr(W), _wt(wtype), n, k, batch, _ptr(x), m, x_row_stride, x_batch_stride,
                                   _ptr(y), y_row_stride, y_batch_stride,
                                   ctypes.byref(sched) if sched is not None else None, _stream(stream))


def rem_engine_of(wtype, rows: int, k: int) -> int:
    return int(load().rem_engine_of(_wt(wtype), rows, k))


def rem_device_status(clear: bool = False) -> int:
    return int(load().rem_device_status(1 if clear else 0))


def rem_set_thread_schedule(sched: Schedule | None) -> int:
    return int(load().rem_set_thread_schedule(ctypes.byref(sched) if sched is not None else None))


def rem_last_plan() -> str:
    return load().rem_last_plan().decode()


def rem_row_bytes(wtype, k: int) -> int:
    return int(load().rem_row_bytes(_wt(wtype), k))


def rem_split_factor(wtype, rows: int, k: int) -> int:
    return int(load().rem_split_factor(_wt(wtype), rows, k))


def rem_dequantize(W, wtype, rows: int, k: int, out, stream=None) -> int:
    return load().rem_dequantize(_ptr(W), _wt(wtype), rows, k, _ptr(out), _stream(stream))


def rem_quantize(src, wtype, rows: int, k: int, W, stream=None) -> int:
    return load().rem_quantize(_ptr(src), _wt(wtype), rows, k, _ptr(W), _stream(stream))


def rem_last_error() -> str:
    return load().rem_last_error().decode()


def rem_version() -> int:
    return int(load().rem_version())


def check(status: int) -> None:
    """Raise RemError with the library's message unless status is REM_OK."""
    if status != REM_OK:
        raise RemError(status, rem_last_error())
