"""GB300 exact tiled attention: the Python binding of ``libfa.so``.

This module only marshals arguments: it turns torch tensors into the pointers,
sizes and stream handle of the C ABI declared in ``include/fa.h`` and raises
``FaError`` on a non-OK status.  Every step of the attention runs in the CUDA
kernels of ``libfa.so``; there is no fallback of any kind, and the calls fail
loudly when the library has not been built.

    import exact_io_aware_26_gb300 as fa
    o, lse = fa.attention_fwd(q, k, v, causal=True)           # q, k, v: [B,H,N,d] cuda
    dq, dk, dv = fa.attention_bwd(q, k, v, o, do, lse, causal=True)
"""
from __future__ import annotations

import ctypes
import math
import os
import re
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfa.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "fa.h")

FA_OK = 0
FA_ERR_INVALID = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_CUDA = -3
FA_ERR_TIMEOUT = -4
FA_ERR_WORKSPACE = -5
FA_ERR_DEVICE = -6
FA_ERR_BOUNDS = -7
FA_F32, FA_F16, FA_BF16 = 0, 1, 2


class FaError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: status {status}: {detail}")
        self.status = status


class FaParams(ctypes.Structure):
    """Mirror of ``fa_params``."""
    _fields_ = [
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int), ("d", ctypes.c_int),
        ("dtype", ctypes.c_int), ("scale", ctypes.c_float), ("causal", ctypes.c_int),
        ("block_mask", ctypes.c_void_p), ("mask_block", ctypes.c_int),
        ("mask_stride_b", ctypes.c_longlong), ("mask_stride_h", ctypes.c_longlong),
        ("dropout_p", ctypes.c_float), ("dropout_seed", ctypes.c_ulonglong),
        ("dropout_offset", ctypes.c_uint),
    ]


_lib = None


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile libfa.so (debug=True: libfa_debug.so, whose kernels check their indices
    and report FA_ERR_BOUNDS through get_status()); returns the library's path."""
    from . import _builder as _b
    return _b.build(force=force, verbose=verbose, debug=debug)


def use_library(path: str) -> str:
    """Make the calls of this module go to the library at `path` (e.g. the debug
    build) from the next call on; returns the path in use before."""
    global LIB_PATH, _lib
    old = LIB_PATH
    LIB_PATH = path
    _lib = None
    return old


def load() -> ctypes.CDLL:
    """Load libfa.so (built in place by ``build()``); raises when it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise FileNotFoundError(
            f"{LIB_PATH} is missing: run exact_io_aware_26_gb300.build() (nvcc, sm_103a) first")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    PP = ctypes.POINTER(FaParams)
    sigs = {
        "fa_check": (I, [PP, I]),
        "fa_fwd": (I, [PP, P, P, P, P, P, P]),
        "fa_fwd_split": (I, [PP, P, P, P, P, P, I, P]),
        "fa_fwd_num_splits": (I, [PP, I]),
        "fa_bwd_workspace_size": (S, [PP]),
        "fa_bwd": (I, [PP, P, P, P, P, P, P, P, P, P, P, S, P]),
        "fa_bwd_preprocess": (I, [PP, P, P, P, S, P]),
        "fa_bwd_main": (I, [PP, P, P, P, P, P, P, P, P, S, P]),
        "fa_bwd_finalize": (I, [PP, P, P, P, P, S, P]),
        "fa_set_bwd_ctas": (I, [I]),
        "fa_get_status": (I, [P]),
        "fa_set_wait_limit_ns": (ctypes.c_ulonglong, [ctypes.c_ulonglong]),
        "fa_selftest_timeout": (I, [P]),
        "fa_status_string": (ctypes.c_char_p, [I]),
        "fa_last_error": (ctypes.c_char_p, []),
        "fa_version": (I, []),
        "fa_fp8_vt_cols": (I, [I]),
        "fa_fp8_quantize": (I, [PP, P, P, P, P, P, P, P, P, P, P, P]),
        "fa_fwd_fp8": (I, [PP, P, P, P, P, P, P, P, P, P]),
    }
    for name, (res, args) in sigs.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    _lib = lib
    return lib


def header_functions() -> list[str]:
    """Names of the functions ``include/fa.h`` declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def _check(status: int, where: str) -> None:
    if status != FA_OK:
        lib = load()
        raise FaError(status, where, (lib.fa_last_error() or b"").decode() or
                      lib.fa_status_string(status).decode())


def _dtype_code(t) -> int:
    import torch
    m = {torch.float32: FA_F32, torch.float16: FA_F16, torch.bfloat16: FA_BF16}
    if t.dtype not in m:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return m[t.dtype]


def make_params(q, scale: Optional[float] = None, causal: bool = False, block_mask=None,
                mask_block: int = 128, dropout_p: float = 0.0, seed: int = 0,
                offset: int = 0) -> tuple[FaParams, object]:
    """fa_params for [B,H,N,d] tensors; returns (params, mask tensor kept alive)."""
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    p = FaParams(B, H, N, d, _dtype_code(q), float(scale), int(bool(causal)), None,
                 int(mask_block), 0, 0, float(dropout_p), int(seed) & 0xFFFFFFFFFFFFFFFF,
                 int(offset) & 0xFFFFFFFF)
    keep = None
    if block_mask is not None:
        import torch
        m = block_mask
        if not (m.is_cuda and m.dtype == torch.uint8):
            raise TypeError("block_mask must be a cuda uint8 tensor")
        T = (N + mask_block - 1) // mask_block
        if m.dim() == 2:
            m = m.reshape(1, 1, T, T)
        if tuple(m.shape[-2:]) != (T, T) or m.stride(-1) != 1 or m.stride(-2) != T:
            raise ValueError(f"block_mask must end in a contiguous [{T}, {T}] matrix")
        p.block_mask = m.data_ptr()
        p.mask_stride_b = 0 if m.shape[0] == 1 else m.stride(0)
        p.mask_stride_h = 0 if m.shape[1] == 1 else m.stride(1)
        keep = m
    return p, keep


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check_tensor(t, name, like):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous cuda tensor")
    if like is not None and (t.shape != like.shape or t.dtype != like.dtype):
        raise ValueError(f"{name} must match q's shape and dtype")


def attention_fwd(q, k, v, scale=None, causal=False, block_mask=None, mask_block=128,
                  out=None, lse=None, stream=None, dropout_p=0.0, seed=0, offset=0):
    """O, LSE = fa_fwd(Q, K, V); tensors [B,H,N,d] on the current device."""
    import torch
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(t, n, q)
    p, keep = make_params(q, scale, causal, block_mask, mask_block, dropout_p, seed, offset)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    _check(load().fa_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                         _stream(stream)), "fa_fwd")
    return out, lse


def fp8_vt_cols(N: int) -> int:
    """fa_fp8_vt_cols: row length of the transposed V codes (N rounded up to 16)."""
    return int(load().fa_fp8_vt_cols(int(N)))


def fp8_quantize(q, k, v, signs=None, stream=None, out=None) -> dict:
    """fa_fp8_quantize: rotation (``signs``: d floats of +-1 on the device, or None) and
    block quantisation of [B,H,N,d] Q, K, V.  Returns q8, k8 [B,H,N,d] and vt8
    [B,H,d,fp8_vt_cols(N)] (uint8 e4m3 codes) and sq, sk, sv [B,H,ceil(N/128)] (fp32),
    written into ``out`` (a dict of such tensors) when given."""
    import torch
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(t, n, q)
    B, H, N, d = q.shape
    if signs is not None and not (signs.is_cuda and signs.dtype == torch.float32
                                  and signs.is_contiguous() and signs.numel() == d):
        raise ValueError(f"signs must be a contiguous cuda float32 tensor of {d} values")
    T = (N + 127) // 128
    u8 = dict(dtype=torch.uint8, device=q.device)
    f32 = dict(dtype=torch.float32, device=q.device)
    shapes = {"q8": (B, H, N, d), "k8": (B, H, N, d), "vt8": (B, H, d, fp8_vt_cols(N)),
              "sq": (B, H, T), "sk": (B, H, T), "sv": (B, H, T)}
    if out is None:
        t = {n: torch.empty(shp, **(u8 if n.endswith("8") else f32)) for n, shp in shapes.items()}
    else:
        t = out
        for n, shp in shapes.items():
            want = torch.uint8 if n.endswith("8") else torch.float32
            x = t[n]
            if not (x.is_cuda and x.is_contiguous() and x.dtype == want and tuple(x.shape) == shp):
                raise ValueError(f"out[{n!r}] must be a contiguous cuda {want} tensor of shape {shp}")
    p, _ = make_params(q)
    _check(load().fa_fp8_quantize(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(signs),
                                  _ptr(t["q8"]), _ptr(t["k8"]), _ptr(t["vt8"]), _ptr(t["sq"]),
                                  _ptr(t["sk"]), _ptr(t["sv"]), _stream(stream)),
           "fa_fp8_quantize")
    return t


def attention_fwd_fp8_codes(t: dict, scale, causal=False, block_mask=None, mask_block=128,
                            dtype=None, out=None, lse=None, stream=None):
    """O, LSE = fa_fwd_fp8 on the codes and scales of ``fp8_quantize`` (same keys and
    layout); O in ``dtype`` (default bf16)."""
    import torch
    q8 = t["q8"]
    B, H, N, d = q8.shape
    T = (N + 127) // 128
    shapes = {"q8": (B, H, N, d), "k8": (B, H, N, d), "vt8": (B, H, d, fp8_vt_cols(N)),
              "sq": (B, H, T), "sk": (B, H, T), "sv": (B, H, T)}
    for n, shp in shapes.items():
        x = t[n]
        want = torch.uint8 if n.endswith("8") else torch.float32
        if not (x.is_cuda and x.is_contiguous() and x.dtype == want and tuple(x.shape) == shp):
            raise ValueError(f"{n} must be a contiguous cuda {want} tensor of shape {shp}")
    dtype = torch.bfloat16 if dtype is None else dtype
    p, keep = make_params(torch.empty((B, H, N, d), dtype=dtype, device="meta"), scale, causal,
                          block_mask, mask_block)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=dtype, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    _check(load().fa_fwd_fp8(ctypes.byref(p), _ptr(t["q8"]), _ptr(t["k8"]), _ptr(t["vt8"]),
                             _ptr(t["sq"]), _ptr(t["sk"]), _ptr(t["sv"]), _ptr(out), _ptr(lse),
                             _stream(stream)), "fa_fwd_fp8")
    return out, lse


def attention_fwd_fp8(q, k, v, signs=None, scale=None, causal=False, block_mask=None,
                      mask_block=128, stream=None):
    """O, LSE of the FP8 forward: fa_fp8_quantize then fa_fwd_fp8 (O in q's dtype)."""
    t = fp8_quantize(q, k, v, signs, stream)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    return attention_fwd_fp8_codes(t, scale, causal, block_mask, mask_block, q.dtype,
                                   stream=stream)


def num_splits(p: FaParams, num_sms: int = 0) -> int:
    """fa_fwd_num_splits: split count for fa_fwd_split (num_sms <= 0 asks the device)."""
    return int(load().fa_fwd_num_splits(ctypes.byref(p), int(num_sms)))


def attention_fwd_split(q, k, v, scale=None, causal=False, block_mask=None, mask_block=128,
                        splits=None, out=None, lse=None, stream=None,
                        dropout_p=0.0, seed=0, offset=0):
    """O, LSE = fa_fwd_split(Q, K, V): the key range cut into ``splits`` slices
    (None: fa_fwd_num_splits for the current device)."""
    import torch
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(t, n, q)
    p, keep = make_params(q, scale, causal, block_mask, mask_block, dropout_p, seed, offset)
    lib = load()
    if splits is None:
        splits = int(lib.fa_fwd_num_splits(ctypes.byref(p), 0))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    _check(lib.fa_fwd_split(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                            int(splits), _stream(stream)),
           "fa_fwd_split")
    return out, lse


def fwd_split_raw(p: FaParams, q, k, v, o, lse, splits, stream=None):
    _check(load().fa_fwd_split(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                               int(splits), _stream(stream)),
           "fa_fwd_split")


def workspace_bytes(q, scale=None, causal=False, block_mask=None, mask_block=128) -> int:
    p, _ = make_params(q, scale, causal, block_mask, mask_block)
    return int(load().fa_bwd_workspace_size(ctypes.byref(p)))


def attention_bwd(q, k, v, o, do, lse, scale=None, causal=False, block_mask=None,
                  mask_block=128, dq=None, dk=None, dv=None, workspace=None, stream=None,
                  dropout_p=0.0, seed=0, offset=0):
    """dQ, dK, dV = fa_bwd(Q, K, V, O, dO, LSE); with dropout, the same dropout_p, seed
    and offset as the forward call that produced O."""
    import torch
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _check_tensor(t, n, q)
    p, keep = make_params(q, scale, causal, block_mask, mask_block, dropout_p, seed, offset)
    lib = load()
    nbytes = int(lib.fa_bwd_workspace_size(ctypes.byref(p)))
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    _check(lib.fa_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                      _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(),
                      _stream(stream)), "fa_bwd")
    return dq, dk, dv


def bwd_preprocess(p: FaParams, o, do, workspace, stream=None):
    _check(load().fa_bwd_preprocess(ctypes.byref(p), _ptr(o), _ptr(do), _ptr(workspace),
                                    workspace.numel(), _stream(stream)), "fa_bwd_preprocess")


def bwd_main(p: FaParams, q, k, v, do, lse, dk, dv, workspace, stream=None):
    _check(load().fa_bwd_main(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse),
                              _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(),
                              _stream(stream)), "fa_bwd_main")


def bwd_finalize(p: FaParams, dq, dk, dv, workspace, stream=None):
    _check(load().fa_bwd_finalize(ctypes.byref(p), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                  workspace.numel(), _stream(stream)), "fa_bwd_finalize")


def set_bwd_ctas(n: int) -> int:
    """fa_set_bwd_ctas: the CTAs per wave the backward plans its slices for (0 = one per SM)."""
    return int(load().fa_set_bwd_ctas(int(n)))


def fwd_raw(p: FaParams, q, k, v, o, lse, stream=None):
    _check(load().fa_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                         _stream(stream)), "fa_fwd")


def get_status(stream=None) -> int:
    """Device-side status since the last call (syncs the stream, clears it)."""
    return int(load().fa_get_status(_stream(stream)))


def set_wait_limit_ns(ns: int) -> int:
    return int(load().fa_set_wait_limit_ns(int(ns)))


def selftest_timeout(stream=None) -> None:
    _check(load().fa_selftest_timeout(_stream(stream)), "fa_selftest_timeout")


def check_params(p: FaParams, for_backward: bool = False) -> int:
    return int(load().fa_check(ctypes.byref(p), int(bool(for_backward))))
