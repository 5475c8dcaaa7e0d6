"""fp64 CPU oracle for exact scaled-dot-product attention (test infrastructure).

This package is the oracle that the CUDA kernels are checked against.  Only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import it; the product path never does.  It shares no code with the CUDA
library: the arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over
rows), and this module only marshals numpy arrays into it.

Functions and the passages they follow:

* ``attention_fwd`` -- the direct two-pass softmax(scale * Q K^T) V with the
  per-row log-sum-exp ("Pourquoi l'attention est liée à la mémoire",
  marketmaker.cc; "Problema e motivação", FlashAttention reading guide).
* ``attention_fwd_blockwise`` -- the tiled online-softmax recurrence in the
  pages' order ("L'algorithme Flash Attention", marketmaker.cc; "Método" and
  "Rastreamento Incremental do Softmax", reading guide), with the output either
  renormalised per step or divided by the running sum at the end (the deferred
  form of "FA2 : parallélisme" and of the loop on the Ultralytics page).
* ``attention_bwd`` / ``attention_bwd_rows`` -- gradients from the derivative of
  the definition ("Passe arrière : recalculer au lieu de stocker" only says that
  P is recomputed from the saved statistics; the formulas are calculus).

* ``philox4x32_10`` / ``dropout_keep`` -- the counter-based generator that
  decides which attention weights dropout keeps (Salmon et al., SC 2011; the
  pages fuse dropout into the kernel -- "Fusão de Kernels", reading guide -- and
  pass ``dropout_p`` to the attention call -- "L'intégration est de huit
  lignes", marketmaker.cc -- but name no generator).

Dropout (``dropout_p`` > 0): weight P_ij of head bh = b * H + h is kept when
the 16-bit half (low for even j, high for odd j) of word (j mod 8) // 2 of
Philox4x32-10 with counter (j // 8, i, bh, offset) and key (seed mod 2^32,
seed // 2^32) is at least t = floor(p * 2^16), else set to 0; kept weights are
scaled by 2^16 / (2^16 - t) (``dropout_scale``), the inverse of the keep
probability.  m, l and LSE stay those of the undropped softmax.

* ``e4m3_encode`` / ``e4m3_decode`` / ``fp8_block_scale`` / ``hadamard_rotate`` /
  ``fp8_quantize`` / ``fp8_attention_fwd`` -- the FP8 forward with incoherent
  processing ("Trois idées pour FA3", marketmaker.cc, point 3: a random rotation
  of the query and key vectors before block quantisation spreads outliers over the
  coordinates); ``fp8_oracle.c`` states the readings taken where the page is silent
  (randomised Sylvester-Hadamard rotation, power-of-two scale per 128-row block,
  e4m3 round-to-nearest-even, P~ quantised as e4m3(256 P~) in the online loop).

Masks: ``mask`` is a uint8 array of shape [T, T] (shared by every batch and
head) or [B, H, T, T], with T = ceil(N / mask_block); entry [i // mb, j // mb]
keeps (1) or hides (0) the pair (query i, key j) ("Extensão: Block-Sparse
FlashAttention", reading guide).  Causal hides keys j > i.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_SRCS = (_SRC, os.path.join(_HERE, "fp8_oracle.c"))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` and ``fp8_oracle.c`` into ``liboracle.so`` next to them
    (gcc, OpenMP)."""
    if force or not os.path.exists(_SO) or any(os.path.getmtime(_SO) < os.path.getmtime(f)
                                               for f in _SRCS):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=gnu11", "-fopenmp", "-fPIC", "-shared",
               "-ffp-contract=off", "-o", tmp, *_SRCS, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_SO)
    P = ctypes.c_void_p
    I = ctypes.c_int
    LL = ctypes.c_longlong
    Dd = ctypes.c_double
    F = ctypes.c_float
    lib.orc_num_threads.restype = I
    U64 = ctypes.c_ulonglong
    U32 = ctypes.c_uint
    lib.orc_fwd.argtypes = [I, I, I, I, P, P, P, Dd, I, P, I, LL, LL, P, P, Dd, U64, U32]
    lib.orc_fwd_rows.argtypes = [I, I, P, P, P, Dd, I, P, I, I, P, P, P, Dd, U64, U32, I]
    lib.orc_fwd_blockwise_f64.argtypes = [I, I, I, I, P, P, P, Dd, I, P, I, LL, LL,
                                          I, I, I, P, P]
    lib.orc_fwd_blockwise_f32.argtypes = [I, I, I, I, P, P, P, F, I, P, I, LL, LL,
                                          I, I, I, P, P]
    lib.orc_bwd.argtypes = [I, I, I, I, P, P, P, P, Dd, I, P, I, LL, LL, P, P, P, Dd, U64, U32]
    lib.orc_bwd_rows.argtypes = [I, I, P, P, P, P, Dd, I, P, I, I, P, P, I, P, P, P, Dd, U64,
                                 U32, I]
    lib.orc_philox4x32_10.argtypes = [P, P, P]
    lib.orc_dropout_keep.argtypes = [I, I, I, Dd, U64, U32, P]
    lib.orc_e4m3_encode.argtypes = [LL, P, P]
    lib.orc_e4m3_decode.argtypes = [LL, P, P]
    lib.orc_fp8_block_scale.argtypes = [Dd]
    lib.orc_fp8_block_scale.restype = Dd
    lib.orc_hadamard_rotate.argtypes = [LL, I, P, P, Dd, P]
    lib.orc_fp8_quantize.argtypes = [I, I, I, P, P, P, P, I, LL, P, P, P, P, P, P]
    lib.orc_fp8_fwd.argtypes = [I, I, I, P, P, P, LL, P, P, P, I, Dd, I, P, I, P, P]
    for f in ("orc_e4m3_encode", "orc_e4m3_decode", "orc_hadamard_rotate", "orc_fp8_quantize",
              "orc_fp8_fwd"):
        getattr(lib, f).restype = None
    for f in ("orc_fwd", "orc_fwd_rows", "orc_fwd_blockwise_f64",
              "orc_fwd_blockwise_f32", "orc_bwd", "orc_bwd_rows", "orc_philox4x32_10",
              "orc_dropout_keep"):
        getattr(lib, f).restype = None
    _lib = lib
    return lib


def num_threads() -> int:
    """OpenMP threads the oracle runs on."""
    return int(_load().orc_num_threads())


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _mask_args(mask, B, H, N, mask_block):
    """(pointer, kept array, batch stride, head stride) for the C side."""
    if mask is None:
        return None, None, 0, 0
    m = np.ascontiguousarray(np.asarray(mask, dtype=np.uint8))
    T = (N + mask_block - 1) // mask_block
    if m.ndim == 2:
        if m.shape != (T, T):
            raise ValueError(f"mask shape {m.shape} != {(T, T)}")
        return _ptr(m), m, 0, 0
    if m.ndim == 4 and m.shape[2:] == (T, T):
        if m.shape[0] not in (1, B) or m.shape[1] not in (1, H):
            raise ValueError(f"mask shape {m.shape} does not broadcast to B={B}, H={H}")
        sh = T * T if m.shape[1] > 1 else 0
        sb = m.shape[1] * T * T if m.shape[0] > 1 else 0
        return _ptr(m), m, sb, sh
    raise ValueError(f"mask shape {m.shape} is neither [T,T] nor [B,H,T,T] with T={T}")


def _head_mask(mask, b, h, N, mask_block):
    if mask is None:
        return None
    m = np.asarray(mask, dtype=np.uint8)
    if m.ndim == 4:
        m = m[b if m.shape[0] > 1 else 0, h if m.shape[1] > 1 else 0]
    return np.ascontiguousarray(m)


def _drop(dropout_p, seed, offset):
    p = float(dropout_p)
    if not 0.0 <= p < 1.0:
        raise ValueError(f"dropout_p {p} is not in [0, 1)")
    return p, int(seed) & 0xFFFFFFFFFFFFFFFF, int(offset) & 0xFFFFFFFF


def philox4x32_10(counter, key) -> np.ndarray:
    """Philox4x32-10 of one counter (4 uint32) under one key (2 uint32) -> 4 uint32."""
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint32).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
    out = np.zeros(4, dtype=np.uint32)
    _load().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def dropout_scale(dropout_p) -> float:
    """The factor kept weights are multiplied by: 2^16 / (2^16 - floor(p * 2^16))."""
    t = min(int(np.floor(float(dropout_p) * 65536.0)), 65535)
    return 65536.0 / (65536.0 - t) if dropout_p > 0 else 1.0


def dropout_keep(B, H, N, dropout_p, seed=0, offset=0) -> np.ndarray:
    """Dropout's keep decisions [B,H,N,N] (uint8, 1 = kept) for every (query, key)."""
    p, seed, offset = _drop(dropout_p, seed, offset)
    keep = np.zeros((B, H, N, N), dtype=np.uint8)
    _load().orc_dropout_keep(B, H, N, p, seed, offset, _ptr(keep))
    return keep


def attention_fwd(q, k, v, scale, causal=False, mask=None, mask_block=128, dropout_p=0.0,
                  seed=0, offset=0):
    """Direct forward over whole [B,H,N,d] tensors -> (O [B,H,N,d], LSE [B,H,N]), fp64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    O = np.zeros_like(q)
    LSE = np.zeros((B, H, N), dtype=np.float64)
    mp, keep, sb, sh = _mask_args(mask, B, H, N, mask_block)
    _load().orc_fwd(B, H, N, d, _ptr(q), _ptr(k), _ptr(v), float(scale), int(bool(causal)),
                    mp, int(mask_block), sb, sh, _ptr(O), _ptr(LSE),
                    *_drop(dropout_p, seed, offset))
    return O, LSE


def attention_fwd_rows(qh, kh, vh, rows, scale, causal=False, mask_h=None, mask_block=128,
                       dropout_p=0.0, seed=0, offset=0, bh=0):
    """Direct forward of selected query rows of one head ([N,d] tensors; bh = b * H + h
    is the head's index, which dropout's counter uses).

    Returns (O_rows [len(rows), d], LSE_rows [len(rows)]).
    """
    qh, kh, vh = _f64(qh), _f64(kh), _f64(vh)
    N, d = qh.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    O = np.zeros((len(rows), d), dtype=np.float64)
    L = np.zeros(len(rows), dtype=np.float64)
    m = None if mask_h is None else np.ascontiguousarray(np.asarray(mask_h, dtype=np.uint8))
    _load().orc_fwd_rows(N, d, _ptr(qh), _ptr(kh), _ptr(vh), float(scale), int(bool(causal)),
                         None if m is None else _ptr(m), int(mask_block), len(rows),
                         _ptr(rows), _ptr(O), _ptr(L), *_drop(dropout_p, seed, offset), int(bh))
    return O, L


def attention_fwd_blockwise(q, k, v, scale, Br, Bc, causal=False, mask=None, mask_block=128,
                            precision="f64", norm_at_end=False):
    """Blockwise online-softmax forward -> (O, LSE) in the requested precision."""
    dt = np.float64 if precision == "f64" else np.float32
    q = np.ascontiguousarray(np.asarray(q, dtype=dt))
    k = np.ascontiguousarray(np.asarray(k, dtype=dt))
    v = np.ascontiguousarray(np.asarray(v, dtype=dt))
    B, H, N, d = q.shape
    O = np.zeros_like(q)
    LSE = np.zeros((B, H, N), dtype=dt)
    mp, keep, sb, sh = _mask_args(mask, B, H, N, mask_block)
    fn = _load().orc_fwd_blockwise_f64 if precision == "f64" else _load().orc_fwd_blockwise_f32
    fn(B, H, N, d, _ptr(q), _ptr(k), _ptr(v), float(scale), int(bool(causal)), mp,
       int(mask_block), sb, sh, int(Br), int(Bc), int(bool(norm_at_end)), _ptr(O), _ptr(LSE))
    return O, LSE


def attention_bwd(q, k, v, do, scale, causal=False, mask=None, mask_block=128, dropout_p=0.0,
                  seed=0, offset=0):
    """Gradients (dQ, dK, dV) of sum(dO * O) over whole [B,H,N,d] tensors, fp64."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, d = q.shape
    dQ, dK, dV = np.zeros_like(q), np.zeros_like(q), np.zeros_like(q)
    mp, keep, sb, sh = _mask_args(mask, B, H, N, mask_block)
    _load().orc_bwd(B, H, N, d, _ptr(q), _ptr(k), _ptr(v), _ptr(do), float(scale),
                    int(bool(causal)), mp, int(mask_block), sb, sh,
                    _ptr(dQ), _ptr(dK), _ptr(dV), *_drop(dropout_p, seed, offset))
    return dQ, dK, dV


def attention_bwd_rows(qh, kh, vh, doh, qrows, krows, scale, causal=False, mask_h=None,
                       mask_block=128, dropout_p=0.0, seed=0, offset=0, bh=0):
    """Gradients of selected rows of one head: dQ[qrows], dK[krows], dV[krows]."""
    qh, kh, vh, doh = _f64(qh), _f64(kh), _f64(vh), _f64(doh)
    N, d = qh.shape
    qr = np.ascontiguousarray(np.asarray(qrows, dtype=np.int32))
    kr = np.ascontiguousarray(np.asarray(krows, dtype=np.int32))
    dQ = np.zeros((len(qr), d))
    dK = np.zeros((len(kr), d))
    dV = np.zeros((len(kr), d))
    m = None if mask_h is None else np.ascontiguousarray(np.asarray(mask_h, dtype=np.uint8))
    _load().orc_bwd_rows(N, d, _ptr(qh), _ptr(kh), _ptr(vh), _ptr(doh), float(scale),
                         int(bool(causal)), None if m is None else _ptr(m), int(mask_block),
                         len(qr), _ptr(qr), _ptr(dQ), len(kr), _ptr(kr), _ptr(dK), _ptr(dV),
                         *_drop(dropout_p, seed, offset), int(bh))
    return dQ, dK, dV


def head_mask(mask, b, h, N, mask_block=128):
    """The [T,T] mask matrix that applies to head (b, h), or None."""
    return _head_mask(mask, b, h, N, mask_block)


# ---------------------------------------------------------------------------
# FP8 forward with incoherent processing (fp8_oracle.c)
# ---------------------------------------------------------------------------

def e4m3_encode(x) -> np.ndarray:
    """e4m3 codes (uint8) of x: round to nearest, ties to even, saturating at +-448."""
    a = _f64(x)
    out = np.zeros(a.shape, dtype=np.uint8)
    _load().orc_e4m3_encode(a.size, _ptr(a), _ptr(out))
    return out


def e4m3_decode(codes) -> np.ndarray:
    """Values (fp64) of e4m3 codes."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.zeros(c.shape, dtype=np.float64)
    _load().orc_e4m3_decode(c.size, _ptr(c), _ptr(out))
    return out


def fp8_block_scale(amax: float) -> float:
    """Smallest power of two sigma with amax / sigma <= 448 (1 for amax = 0)."""
    return float(_load().orc_fp8_block_scale(float(amax)))


def hadamard_rotate(x, signs, post=1.0) -> np.ndarray:
    """Rows of x times diag(signs) H_d times post (H_d the Sylvester Hadamard matrix)."""
    a = _f64(x)
    d = a.shape[-1]
    sg = _f64(signs).reshape(d)
    out = np.zeros_like(a)
    _load().orc_hadamard_rotate(a.size // d, d, _ptr(a), _ptr(sg), float(post), _ptr(out))
    return out


def fp8_vt_cols(N: int) -> int:
    """Row length of the transposed V codes: N rounded up to a multiple of 16."""
    return (N + 15) // 16 * 16


def fp8_quantize(q, k, v, signs=None, block=128):
    """Rotation (signs given) and block quantisation of [B,H,N,d] Q, K, V.

    Returns a dict with q8, k8 [B,H,N,d] and vt8 [B,H,d,fp8_vt_cols(N)] (uint8 e4m3
    codes; vt8 is V transposed, zero past N) and sq, sk, sv [B,H,ceil(N/block)] (fp64
    powers of two), the layout the CUDA library's FP8 forward takes."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    T = (N + block - 1) // block
    ld = fp8_vt_cols(N)
    r = {"q8": np.zeros((B, H, N, d), np.uint8), "k8": np.zeros((B, H, N, d), np.uint8),
         "vt8": np.zeros((B, H, d, ld), np.uint8), "sq": np.zeros((B, H, T)),
         "sk": np.zeros((B, H, T)), "sv": np.zeros((B, H, T))}
    sg = None if signs is None else _f64(signs).reshape(d)
    _load().orc_fp8_quantize(B * H, N, d, _ptr(q), _ptr(k), _ptr(v),
                             None if sg is None else _ptr(sg), int(block), ld,
                             _ptr(r["q8"]), _ptr(r["k8"]), _ptr(r["vt8"]), _ptr(r["sq"]),
                             _ptr(r["sk"]), _ptr(r["sv"]))
    return r


def fp8_attention_fwd(t, scale, causal=False, mask=None, mask_block=128, block=128):
    """The FP8 forward on the codes and scales of ``fp8_quantize`` -> (O, LSE), fp64."""
    q8, k8, vt8 = (np.ascontiguousarray(t[n], dtype=np.uint8) for n in ("q8", "k8", "vt8"))
    sq, sk, sv = (_f64(t[n]) for n in ("sq", "sk", "sv"))
    B, H, N, d = q8.shape
    O = np.zeros((B, H, N, d))
    LSE = np.zeros((B, H, N))
    m = None
    if mask is not None:
        m = np.ascontiguousarray(np.asarray(mask, dtype=np.uint8))
        T = (N + mask_block - 1) // mask_block
        if m.shape != (T, T):
            raise ValueError(f"mask shape {m.shape} != {(T, T)}")
    _load().orc_fp8_fwd(B * H, N, d, _ptr(q8), _ptr(k8), _ptr(vt8), vt8.shape[-1], _ptr(sq),
                        _ptr(sk), _ptr(sv), int(block), float(scale), int(bool(causal)),
                        None if m is None else _ptr(m), int(mask_block), _ptr(O), _ptr(LSE))
    return O, LSE
