"""Helpers for the GPU parity tests: move oracle-made inputs to the device,
call the library through its C ABI, and bring results back.

Inputs are always produced on the host by the seeded generators and the
oracle's quantizer; nothing the CUDA path computes is ever fed to the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import quantized_few_row_gb300 as rem

CANARY = np.float32(-1234.5)


def dev():
    return torch.device("cuda:0")


def to_dev_bytes(w: np.ndarray, offset: int = 0) -> tuple[torch.Tensor, int]:
    """Copy bytes to a fresh device buffer at `offset` bytes past a 256-byte
    aligned base; returns (holder, address)."""
    flat = np.ascontiguousarray(w, dtype=np.uint8).reshape(-1)
    holder = torch.zeros(flat.size + offset + 64, dtype=torch.uint8, device=dev())
    holder[offset:offset + flat.size] = torch.from_numpy(flat).to(dev())
    return holder, holder.data_ptr() + offset


def to_dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev())


def canary(numel: int) -> torch.Tensor:
    return torch.full((numel,), float(CANARY), dtype=torch.float32, device=dev())


def run_matvec(w: np.ndarray, wt, n: int, k: int, batch: int, x: np.ndarray, m: int, xrs: int, xbs: int,
               yrs: int, ybs: int, ylen: int, split: int = 0, rows_per_cta: int = 0, w_offset: int = 0,
               use_ex: bool = True) -> np.ndarray:
    """y as a flat f32 host array of ylen elements (canary where unwritten)."""
    wh, wp = to_dev_bytes(w, w_offset)
    xd = to_dev_f32(x)
    yd = canary(ylen)
    if use_ex:
        rc = rem.rem_matvec_ex(wp, wt, n, k, batch, xd, m, xrs, xbs, yd, yrs, ybs, split, rows_per_cta)
    else:
        rc = rem.rem_matvec(wp, wt, n, k, batch, xd, m, xbs, yd, ybs)
    rem.check(rc)
    torch.cuda.synchronize()
    out = yd.cpu().numpy()
    del wh
    return out


def run_sched(w: np.ndarray, wt, n: int, k: int, batch: int, x: np.ndarray, m: int, xrs: int, xbs: int,
              yrs: int, ybs: int, ylen: int, sched=None, w_offset: int = 0, tail: int = 0) -> np.ndarray:
    """y through rem_matvec_sched as a flat f32 host array of ylen + tail
    elements; everything the call does not write (strided gaps and the
    `tail` elements past the last output) keeps the canary."""
    wh, wp = to_dev_bytes(w, w_offset)
    xd = to_dev_f32(x)
    yd = canary(ylen + tail)
    rem.check(rem.rem_matvec_sched(wp, wt, n, k, batch, xd, m, xrs, xbs, yd, yrs, ybs, sched))
    torch.cuda.synchronize()
    out = yd.cpu().numpy()
    del wh
    return out


def gather_y(yflat: np.ndarray, batch: int, m: int, n: int, yrs: int, ybs: int) -> np.ndarray:
    """[batch, m, n] view of a strided flat output."""
    b = np.arange(batch)[:, None, None] * ybs
    j = np.arange(m)[None, :, None] * yrs
    i = np.arange(n)[None, None, :]
    return yflat[b + j + i]


def contiguous(wt, n: int, k: int, m: int, seed_w: int, seed_x: int, rows_scale=None):
    from quantized_few_row_gb300 import inputs
    wf = inputs.weights(n, k, seed_w)
    if rows_scale is not None:
        wf = wf * np.float32(rows_scale)
    w = oracle.quantize(wf, wt)
    x = inputs.activations(m, k, seed_x)
    return w, x


def assert_close_to_oracle(y_gpu: np.ndarray, y_ref: np.ndarray, a_ref: np.ndarray, what: str = ""):
    ok = oracle.within_tolerance(y_gpu, y_ref, a_ref)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        detail = [(tuple(int(t) for t in b), float(y_gpu[tuple(b)]), float(y_ref[tuple(b)]),
                   float(a_ref[tuple(b)])) for b in bad]
        raise AssertionError(f"{what}: {int((~ok).sum())} outputs outside 1e-4*A + 1e-7, e.g. {detail}")


def adversarial_blocks(fmt, rows, k, seed):
    """Random bytes with finite fp16 scale fields (normal and subnormal)."""
    rb = oracle.row_bytes(fmt, k)
    b = _inputs().uniform_bytes(rows * rb, seed).reshape(rows, rb)
    if fmt == "f16":
        h = b.view(np.uint16)
        h[(h & 0x7C00) == 0x7C00] &= 0x3FFF   # no inf / NaN
        return b
    if fmt == "bf16":
        h = b.view(np.uint16)
        h[(h & 0x7F80) == 0x7F80] &= 0xBFFF   # no inf / NaN
        return b
    if fmt == "f32":
        u = b.view(np.uint32)
        u[(u & 0x7F800000) == 0x7F800000] &= 0xBFFFFFFF
        return b
    g = np.random.Generator(np.random.PCG64(seed + 1))
    bb = oracle.block_bytes(fmt)
    nb = rb // bb
    blocks = b.reshape(rows, nb, bb)
    fields = {"q8_0": [0], "q5_0": [0], "q4_K": [0, 2], "q6_K": [208]}[fmt]
    for off in fields:
        h = g.integers(0, 0x7C00, size=(rows, nb)).astype(np.uint16)   # finite, positive
        h |= (g.integers(0, 2, size=(rows, nb)) << 15).astype(np.uint16)
        h[:, ::7] &= 0x03FF                                            # some subnormal scales
        blocks[:, :, off:off + 2] = h.view(np.uint8).reshape(rows, nb, 2)
    return b


def _inputs():
    from quantized_few_row_gb300 import inputs
    return inputs
