"""Seeded synthetic inputs for the attention workloads.

This module is shared by the oracle side and the CUDA side of every parity
check, so it holds none of the attention arithmetic: it only draws random
numbers, shapes them and rounds them to the working dtype.  Each input is rounded
once; the CUDA path receives that tensor and the oracle receives the same values
widened exactly to fp64.

Recipe (one ``numpy.random.Generator(PCG64(seed))`` per workload, platform
independent, drawn in the order Q, K, V, dO, then the block mask):

* i.i.d. tensors: ``standard_normal`` in fp32, multiplied by ``qkv_scale``
  (Q, K, V only), then rounded to the dtype (round to nearest even).
* AR(1) tensors: per (batch, head, feature) an independent series along the
  sequence with x_0 ~ N(0,1) and x_t = rho x_{t-1} + sqrt(1 - rho^2) e_t,
  e_t ~ N(0,1), in fp64, then rounded to the dtype (unit marginal variance).
* block mask: uint8 [T, T] with T = ceil(N / mask_block), diagonal entries 1,
  off-diagonal entries 1 with probability ``mask_p``; one mask shared by every
  batch and head.

* outliers (``outlier_p``): after the i.i.d. draw, each entry of Q, K and V is
  replaced, with probability ``outlier_p``, by ``outlier_sd`` * N(0, 1) (one
  ``random`` draw for the choice, then one ``standard_normal`` for the value,
  per tensor) -- heavy coordinates of the kind that ruin naive FP8 attention.
* rotation signs: ``rotation_signs(d, seed)``, d values in {-1, +1} from their own
  generator (PCG64(seed)), the random diagonal the FP8 path rotates with.

The five named workloads stand in for the pages' workloads (a trading day of
23,400 one-second steps with 12 heads, the 8192-token fp16 single-head case, a
block-sparse long sequence); no dataset is read.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str               # "f32" | "f16" | "bf16"
    seed: int
    causal: tuple = (False,)  # the causal settings the workload runs
    backward: bool = True
    qkv_scale: float = 1.0
    ar1_rho: Optional[float] = None
    mask_p: Optional[float] = None
    mask_block: int = 128

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


WORKLOADS = {
    # forward only, fp32, the small case the oracle finishes in well under a second
    "fp32_n256": Workload("fp32_n256", 1, 1, 256, 64, "f32", 0, backward=False),
    # B=4 H=12 N=2048 d=64 bf16, non-causal and causal, forward + backward
    "bf16_b4h12_n2048": Workload("bf16_b4h12_n2048", 4, 12, 2048, 64, "bf16", 2,
                                 causal=(False, True)),
    # one layer, one head, N=8192 fp16: the unfused score matrix would be 128 MiB
    "fp16_n8192": Workload("fp16_n8192", 1, 1, 8192, 64, "f16", 3, qkv_scale=0.5),
    # a trading day at one-second resolution, 12 heads, causal, AR(1) inputs
    "bf16_day_n23400": Workload("bf16_day_n23400", 1, 12, 23400, 64, "bf16", 4,
                                causal=(True,), ar1_rho=0.9),
    # block-sparse: 128x128 block mask, diagonal kept, off-diagonal kept with p=0.25
    "bf16_sparse_n16384": Workload("bf16_sparse_n16384", 2, 16, 16384, 128, "bf16", 5,
                                   mask_p=0.25),
}


def _iid(rng: np.random.Generator, shape, mult: float) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if mult != 1.0:
        x = x * np.float32(mult)
    return x


def _ar1(rng: np.random.Generator, shape, rho: float) -> np.ndarray:
    B, H, N, d = shape
    e = rng.standard_normal(shape)  # fp64
    x = np.empty(shape, dtype=np.float64)
    c = math.sqrt(1.0 - rho * rho)
    x[:, :, 0, :] = e[:, :, 0, :]
    for t in range(1, N):
        x[:, :, t, :] = rho * x[:, :, t - 1, :] + c * e[:, :, t, :]
    return x


def block_mask(rng: np.random.Generator, N: int, mask_block: int, p: float) -> np.ndarray:
    T = (N + mask_block - 1) // mask_block
    m = (rng.random((T, T)) < p).astype(np.uint8)
    np.fill_diagonal(m, 1)
    return m


def rotation_signs(d: int, seed: int) -> torch.Tensor:
    """d random signs (fp32 tensor of -1.0 / +1.0) from PCG64(seed)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return torch.from_numpy(np.where(rng.random(d) < 0.5, -1.0, 1.0).astype(np.float32))


def make_inputs(B: int, H: int, N: int, d: int, dtype: str, seed: int, *,
                qkv_scale: float = 1.0, ar1_rho: Optional[float] = None,
                mask_p: Optional[float] = None, mask_block: int = 128,
                backward: bool = True, outlier_p: float = 0.0,
                outlier_sd: float = 10.0) -> dict:
    """Draw Q, K, V (and dO, and a block mask when mask_p is set) as CPU tensors.

    Returns a dict with torch tensors ``q, k, v`` (and ``do``) in the dtype,
    shape [B, H, N, d], and ``mask`` (uint8 numpy [T, T]) or None.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    shape = (B, H, N, d)
    td = _DT[dtype]
    out = {}
    for name in ("q", "k", "v"):
        if ar1_rho is not None:
            x = _ar1(rng, shape, ar1_rho)
        else:
            x = _iid(rng, shape, qkv_scale)
        if outlier_p > 0.0:
            hit = rng.random(shape) < outlier_p
            x = np.where(hit, np.float32(outlier_sd) * rng.standard_normal(shape, dtype=np.float32),
                         x)
        out[name] = torch.from_numpy(x).to(td).contiguous()
    if backward:
        out["do"] = torch.from_numpy(_iid(rng, shape, 1.0)).to(td).contiguous()
    out["mask"] = block_mask(rng, N, mask_block, mask_p) if mask_p is not None else None
    return out


def workload_inputs(w: Workload) -> dict:
    """Inputs of a named workload (see ``WORKLOADS``)."""
    return make_inputs(w.B, w.H, w.N, w.d, w.dtype, w.seed, qkv_scale=w.qkv_scale,
                       ar1_rho=w.ar1_rho, mask_p=w.mask_p, mask_block=w.mask_block,
                       backward=w.backward)


def torch_dtype(name: str) -> torch.dtype:
    return _DT[name]
