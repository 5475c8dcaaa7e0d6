"""The FP8 forward with incoherent processing on the GPU against the FP8 oracle
("Trois idées pour FA3", marketmaker.cc, point 3).

Two stages, each checked on its own:

* fa_fp8_quantize against ``oracle.fp8_quantize``: the block scales are equal, the
  codes of V are equal, and a code of Q^ or K^ may differ only where the rotated
  value (formed in fp32 by a butterfly on the GPU, by a matrix product in fp64 in
  the oracle) lies within 1e-5 (relative) of the midpoint between two neighbouring
  e4m3 values, and then by one step.
* fa_fwd_fp8, fed the ORACLE's codes and scales, against ``oracle.fp8_attention_fwd``
  on the same codes, within the 16-bit tolerances (max |O - O_ref| <= 1e-2 + half an
  output ulp, max |LSE - LSE_ref| <= 1e-3).  Both sides quantise P~ from its fp32
  value; a weight whose fp32 value differs by an ulp across a rounding midpoint
  moves one code, which is far inside the bound; the mean error is also asserted.

End to end (quantise + forward on the GPU) the error against the exact fp64 result
must match the oracle's FP8 error, and rotation must lower it on inputs with
outliers.  The full-size case runs the bench's workload (B=4, H=12, N=2048, d=64,
bf16) and compares two whole heads with the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import check_fwd, to_np64

import exact_io_aware_26_gb300 as fa

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f16": torch.float16}
E4M3 = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))


def _inputs(B, H, N, d, dtype, seed, outlier_p=0.0):
    x = synth.make_inputs(B, H, N, d, dtype, seed, backward=False, outlier_p=outlier_p)
    gpu = {n: x[n].cuda() for n in ("q", "k", "v")}
    ref = {n: x[n].double().numpy() for n in ("q", "k", "v")}
    return gpu, ref


def _signs(d, seed, rot):
    if not rot:
        return None, None
    s = synth.rotation_signs(d, seed)
    return s.cuda(), s.double().numpy()


def _to_gpu(t):
    return {n: torch.from_numpy(np.ascontiguousarray(t[n])).to(
        "cuda", torch.uint8 if n.endswith("8") else torch.float32) for n in t}


def _near_boundary(amax, rel=1e-5):
    """amax within `rel` of 1.75 * 2^k, where the block scale changes."""
    k = np.floor(np.log2(amax / 1.75))
    return np.abs(amax / (1.75 * 2.0 ** k) - 1) < rel or np.abs(amax / (1.75 * 2.0 ** (k + 1)) - 1) < rel


def _check_codes(got, want, exact, sigma, name):
    """Codes agree in value (+0 and -0 alike); a difference is allowed only where
    the oracle's exact value / sigma lies within 1e-5 of the midpoint of the two
    values, which must be neighbours.  Returns the number of such differences."""
    g, w = E4M3[got], E4M3[want]
    diff = g != w
    if not diff.any():
        return 0
    x = (exact / sigma)[diff]
    lo, hi = np.minimum(g[diff], w[diff]), np.maximum(g[diff], w[diff])
    mid = (lo + hi) / 2
    finite = np.sort(np.unique(E4M3[np.isfinite(E4M3)]))
    pos_lo = np.searchsorted(finite, lo)
    neighbours = finite[np.minimum(pos_lo + 1, len(finite) - 1)] == hi
    assert np.all(neighbours), f"{name}: codes differ by more than one step"
    assert np.all(np.abs(x - mid) <= 1e-5 * np.abs(mid)), f"{name}: a code differs away from a midpoint"
    assert diff.mean() < 1e-3, f"{name}: {diff.sum()} codes differ"
    return int(diff.sum())


def _compare_quantized(t_gpu, t_ref, ref, signs64, N, d):
    got = {n: t_gpu[n].cpu().numpy() for n in t_gpu}
    T = (N + 127) // 128
    # scales: V exactly; Q^ and K^ exactly unless the rotated amax sits on a boundary
    assert np.array_equal(got["sv"].astype(np.float64), t_ref["sv"])
    qr = oracle.hadamard_rotate(ref["q"], signs64, 1.0 / d) if signs64 is not None else ref["q"]
    kr = oracle.hadamard_rotate(ref["k"], signs64) if signs64 is not None else ref["k"]
    for sname, xr in (("sq", qr), ("sk", kr)):
        bad = np.argwhere(got[sname].astype(np.float64) != t_ref[sname])
        for b, h, t in bad:
            amax = np.abs(xr[b, h, t * 128:(t + 1) * 128]).max()
            assert _near_boundary(amax), f"{sname}[{b},{h},{t}] differs"
    # codes
    assert np.all(got["vt8"][..., N:] == 0)
    assert np.array_equal(E4M3[got["vt8"]], E4M3[t_ref["vt8"]])
    for cname, sname, xr in (("q8", "sq", qr), ("k8", "sk", kr)):
        sig = np.repeat(t_ref[sname], 128, axis=-1)[..., :N, None]
        _check_codes(got[cname], t_ref[cname], xr, sig, cname)


QUANT_CASES = [
    (1, 2, 300, 64, "bf16", True, 0.01),
    (2, 1, 77, 64, "f16", True, 0.0),
    (1, 2, 256, 128, "bf16", True, 0.01),
    (1, 1, 1000, 128, "f16", False, 0.0),
    (1, 3, 129, 64, "bf16", False, 0.001),
    (1, 1, 1, 64, "bf16", True, 0.0),
]


@pytest.mark.parametrize("B,H,N,d,dtype,rot,outliers", QUANT_CASES)
def test_quantize_matches_oracle(cuda_lib, B, H, N, d, dtype, rot, outliers):
    gpu, ref = _inputs(B, H, N, d, dtype, 40 + N, outliers)
    sg, sg64 = _signs(d, N, rot)
    t_gpu = fa.fp8_quantize(gpu["q"], gpu["k"], gpu["v"], sg)
    torch.cuda.synchronize()
    assert fa.get_status() == fa.FA_OK
    t_ref = oracle.fp8_quantize(ref["q"], ref["k"], ref["v"], sg64)
    _compare_quantized(t_gpu, t_ref, ref, sg64, N, d)


FWD_CASES = [
    (1, 2, 300, 64, "bf16", False, False),
    (1, 2, 300, 64, "bf16", True, False),
    (2, 1, 517, 128, "f16", False, True),
    (1, 2, 256, 128, "bf16", True, False),
    (1, 1, 1000, 64, "f16", True, True),
    (1, 3, 128, 64, "bf16", False, False),
    (1, 1, 1, 64, "bf16", False, False),
    (1, 1, 130, 128, "bf16", True, False),
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal,masked", FWD_CASES)
def test_forward_on_oracle_codes_matches_oracle(cuda_lib, B, H, N, d, dtype, causal, masked):
    gpu, ref = _inputs(B, H, N, d, dtype, 7 + N, 0.001)
    _, sg64 = _signs(d, 5, True)
    t_ref = oracle.fp8_quantize(ref["q"], ref["k"], ref["v"], sg64)
    mask = None
    if masked:
        T = (N + 127) // 128
        mask = synth.block_mask(np.random.Generator(np.random.PCG64(N)), N, 128, 0.4)
    scale = 1.0 / math.sqrt(d)
    O, L = fa.attention_fwd_fp8_codes(_to_gpu(t_ref), scale, causal=causal,
                                      block_mask=None if mask is None else torch.from_numpy(mask).cuda(),
                                      dtype=DT[dtype])
    torch.cuda.synchronize()
    assert fa.get_status() == fa.FA_OK
    O_ref, L_ref = oracle.fp8_attention_fwd(t_ref, scale, causal=causal, mask=mask)
    check_fwd(O, L, O_ref, L_ref, dtype)
    assert np.abs(to_np64(O) - O_ref).mean() < 2e-3


def _rmse(a, b):
    return float(np.sqrt(np.mean((a - b) ** 2)))


@pytest.mark.parametrize("d,causal", [(64, False), (128, True)])
def test_end_to_end_error_matches_the_oracle_fp8_error(cuda_lib, d, causal):
    B, H, N = 1, 4, 512
    gpu, ref = _inputs(B, H, N, d, "bf16", 9, 0.001)
    scale = 1.0 / math.sqrt(d)
    O_exact, _ = oracle.attention_fwd(ref["q"], ref["k"], ref["v"], scale, causal=causal)
    err = {}
    for rot in (True, False):
        sg, sg64 = _signs(d, 9, rot)
        O, _ = fa.attention_fwd_fp8(gpu["q"], gpu["k"], gpu["v"], sg, scale, causal=causal)
        torch.cuda.synchronize()
        assert fa.get_status() == fa.FA_OK
        O_emul, _ = oracle.fp8_attention_fwd(oracle.fp8_quantize(ref["q"], ref["k"], ref["v"], sg64),
                                             scale, causal=causal)
        e_gpu, e_emul = _rmse(to_np64(O), O_exact), _rmse(O_emul, O_exact)
        assert e_gpu <= 1.05 * e_emul + 2e-4, (rot, e_gpu, e_emul)
        err[rot] = e_gpu
    assert err[True] * 1.2 < err[False], err


@pytest.mark.parametrize("causal", [False, True])
def test_full_size_workload_two_heads(cuda_lib, causal):
    """B=4 H=12 N=2048 d=64 bf16 (the bench's workload): whole-tensor quantise and
    forward on the GPU; heads (0, 0) and (3, 11) against the oracle, codes and O."""
    w = synth.WORKLOADS["bf16_b4h12_n2048"]
    x = synth.workload_inputs(w)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    sg = synth.rotation_signs(w.d, 1)
    t = fa.fp8_quantize(q, k, v, sg.cuda())
    O, L = fa.attention_fwd_fp8_codes(t, w.scale, causal=causal, dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert fa.get_status() == fa.FA_OK
    sg64 = sg.double().numpy()
    for b, h in ((0, 0), (3, 11)):
        ref = {n: x[n][b:b + 1, h:h + 1].double().numpy() for n in ("q", "k", "v")}
        t_ref = oracle.fp8_quantize(ref["q"], ref["k"], ref["v"], sg64)
        t_head = {n: t[n][b:b + 1, h:h + 1].contiguous() for n in t}
        _compare_quantized(t_head, t_ref, ref, sg64, w.N, w.d)
        O_ref, L_ref = oracle.fp8_attention_fwd(t_ref, w.scale, causal=causal)
        check_fwd(O[b:b + 1, h:h + 1], L[b:b + 1, h:h + 1], O_ref, L_ref, "bf16")


@pytest.mark.parametrize("causal,masked", [(True, False), (False, True)])
def test_head_order_of_a_problem_larger_than_l2(cuda_lib, causal, masked):
    """B2 H16 N16384 d128 (the block-sparse workload's shape): its FP8 K and V (134 MB)
    exceed three quarters of L2, so the launch runs head by head (causal: its last heads
    as one more group).  Every (query tile, head) must be computed once, with its own
    coordinates: O and LSE equal, bit for bit, those of the same kernel run one head at a
    time (whose K, V fit)."""
    B, H, N, d = 2, 16, 16384, 128
    g = torch.Generator().manual_seed(2024)
    q, k, v = (torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).cuda() for _ in range(3))
    t = fa.fp8_quantize(q, k, v, synth.rotation_signs(d, 3).cuda())
    m = None
    if masked:
        m = torch.from_numpy(synth.block_mask(np.random.Generator(np.random.PCG64(5)), N, 128, 0.25)).cuda()
    scale = 1.0 / math.sqrt(d)
    O, L = fa.attention_fwd_fp8_codes(t, scale, causal=causal, block_mask=m, dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert fa.get_status() == fa.FA_OK
    for b, h in ((0, 0), (0, 9), (1, 4), (1, 15)):
        th = {n: t[n][b:b + 1, h:h + 1].contiguous() for n in t}
        Oh, Lh = fa.attention_fwd_fp8_codes(th, scale, causal=causal, block_mask=m, dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert fa.get_status() == fa.FA_OK
        assert torch.equal(O[b, h], Oh[0, 0]) and torch.equal(L[b, h], Lh[0, 0]), (b, h)
