"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI,
run the fp64 oracle on the same (dtype-rounded) inputs, compare.

Tolerances (stated for the workloads; derived where the statement is silent):
  fp32 inputs:       max |O - O_ref| <= 1e-5, max |LSE - LSE_ref| <= 1e-5
  fp16/bf16 inputs:  max |O - O_ref| <= 1e-2 + half an output ulp of O_ref
                     (O is stored in the 16-bit type; for |O| >= 4 half a bf16
                     ulp alone exceeds 1e-2), max |LSE - LSE_ref| <= 1e-3,
                     ||g - g_ref||_F / ||g_ref||_F <= 2e-2 for g in dQ, dK, dV.
"""
from __future__ import annotations

import numpy as np
import torch

import exact_io_aware_26_gb300 as fa
import oracle

TOL = {
    "f32": dict(o=1e-5, lse=1e-5),
    "f16": dict(o=1e-2, lse=1e-3, grad=2e-2),
    "bf16": dict(o=1e-2, lse=1e-3, grad=2e-2),
}
DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def dtype_name(t: torch.dtype) -> str:
    return {v: k for k, v in DTYPES.items()}[t]


def half_ulp(ref: np.ndarray, dtype: str) -> np.ndarray:
    """Half a unit in the last place of the output type at |ref|."""
    if dtype == "f32":
        return np.zeros_like(ref)
    mant = 7 if dtype == "bf16" else 10
    a = np.maximum(np.abs(ref), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(a)) - mant) / 2


def guarded(shape, dtype, device="cuda", guard=4096, fill=0x5A):
    """Tensor view inside a larger byte buffer whose guard bands hold `fill`."""
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    raw = torch.full((n + 2 * guard,), fill, dtype=torch.uint8, device=device)
    view = raw[guard:guard + n].view(dtype).view(shape)
    return raw, view


def guards_intact(raw, guard=4096, fill=0x5A) -> bool:
    return bool((raw[:guard] == fill).all()) and bool((raw[-guard:] == fill).all())


def to_np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def check_fwd(O, LSE, O_ref, L_ref, dtype, rows_mask=None):
    """Assert the forward outputs against the oracle; returns (max O err, max LSE err)."""
    tol = TOL[dtype]
    O = to_np64(O)
    L = to_np64(LSE)
    err_o = np.abs(O - O_ref)
    bound = tol["o"] + half_ulp(O_ref, dtype)
    fin = np.isfinite(L_ref)
    assert np.array_equal(np.isfinite(L), fin), "LSE finiteness differs"
    assert np.all(L[~fin] == L_ref[~fin]), "hidden rows must have LSE = -inf"
    err_l = np.abs(L[fin] - L_ref[fin]) if fin.any() else np.zeros(1)
    assert np.all(err_o <= bound), f"O max err {err_o.max():.3e} (worst excess {(err_o - bound).max():.3e})"
    assert err_l.max() <= tol["lse"], f"LSE max err {err_l.max():.3e}"
    return float(err_o.max()), float(err_l.max())


def rel_fro(a: np.ndarray, b: np.ndarray) -> float:
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def check_grads(got, ref, dtype):
    tol = TOL[dtype]["grad"]
    errs = []
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        e = rel_fro(to_np64(g) if isinstance(g, torch.Tensor) else g, r)
        assert np.all(np.isfinite(to_np64(g) if isinstance(g, torch.Tensor) else g)), name
        assert e <= tol, f"{name} relative Frobenius error {e:.3e} > {tol}"
        errs.append(e)
    return errs


def oracle_inputs(inp):
    return {k: (to_np64(v) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
