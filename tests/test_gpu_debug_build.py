"""The debug build of the library (FA_DEBUG, libfa_debug.so): its kernels check the
tile coordinates they copy from, the schedule's slices and the rows they store to,
and record FA_ERR_BOUNDS instead of trapping when a check fails.  On a sweep of small
shapes that reaches every launch kind (ragged tails, both head sizes, causal and not,
block masks, split-KV, whole and sliced key tiles in the backward) every check must
pass (status FA_OK), and the results must be those of the release build and agree with
the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import check_fwd, check_grads, oracle_inputs

import exact_io_aware_26_gb300 as fa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib(cuda_lib):
    path = fa.build(debug=True)
    old = fa.use_library(path)
    lib = fa.load()
    yield lib
    fa.use_library(old)
    fa.load()


def _ref(inp, causal, mask=None, mb=128):
    o = oracle_inputs(inp)
    scale = 1.0 / math.sqrt(o["q"].shape[-1])
    O, L = oracle.attention_fwd(o["q"], o["k"], o["v"], scale, causal=causal, mask=mask, mask_block=mb)
    g = oracle.attention_bwd(o["q"], o["k"], o["v"], o["do"], scale, causal=causal, mask=mask,
                             mask_block=mb)
    return O, L, g


CASES = [
    # B, H, N, d, causal, mask_p, bwd CTA cap (0: default), forward splits
    (1, 1, 1, 64, True, None, 0, 1),
    (2, 3, 63, 64, False, None, 0, 1),
    (1, 2, 129, 128, True, None, 0, 1),
    (2, 2, 777, 64, True, None, 50, 1),     # every key tile cut into query slices
    (2, 2, 777, 128, False, None, 9, 1),
    (1, 1, 1000, 64, False, None, 0, 3),    # sliced backward (8 key tiles), split-KV forward
    (1, 2, 900, 64, True, 0.4, 0, 1),       # block mask
    (1, 1, 1300, 128, False, 0.5, 0, 4),
]


@pytest.mark.parametrize("B,H,N,d,causal,mask_p,cap,splits", CASES)
def test_debug_build_checks_pass_and_results_match(debug_lib, B, H, N, d, causal, mask_p, cap, splits):
    inp = synth.make_inputs(B, H, N, d, "bf16", seed=7100 + N + d, mask_p=mask_p)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    m = None if inp["mask"] is None else torch.as_tensor(inp["mask"]).cuda()
    old = fa.set_bwd_ctas(cap)
    try:
        if splits > 1:
            o, lse = fa.attention_fwd_split(q, k, v, causal=causal, block_mask=m, splits=splits)
        else:
            o, lse = fa.attention_fwd(q, k, v, causal=causal, block_mask=m)
        grads = fa.attention_bwd(q, k, v, o, do, lse, causal=causal, block_mask=m)
    finally:
        fa.set_bwd_ctas(old)
    st = fa.get_status()
    assert st == fa.FA_OK, fa.load().fa_status_string(st)
    O, L, g = _ref(inp, causal, inp["mask"])
    check_fwd(o, lse, O, L, "bf16")
    check_grads(grads, g, "bf16")


@pytest.mark.parametrize("d,causal,mask_p", [(64, True, None), (128, False, 0.4)])
def test_debug_build_fp8_forward(debug_lib, d, causal, mask_p):
    """The FP8 quantiser and forward (head order, block-mask bitmask) under the debug
    build: every check passes and the result agrees with the oracle's FP8 forward on
    the oracle's own codes."""
    B, H, N = 1, 2, 700
    inp = synth.make_inputs(B, H, N, d, "bf16", seed=7300 + d, mask_p=mask_p, backward=False)
    o = oracle_inputs(inp)
    signs = synth.rotation_signs(d, 4)
    t_ref = oracle.fp8_quantize(o["q"], o["k"], o["v"], signs.double().numpy())
    t = {n: torch.from_numpy(np.ascontiguousarray(t_ref[n])).cuda() for n in ("q8", "k8", "vt8")}
    t.update({n: torch.from_numpy(np.ascontiguousarray(t_ref[n])).to("cuda", torch.float32)
              for n in ("sq", "sk", "sv")})
    m = None if inp["mask"] is None else torch.as_tensor(inp["mask"]).cuda()
    scale = 1.0 / math.sqrt(d)
    O, L = fa.attention_fwd_fp8_codes(t, scale, causal=causal, block_mask=m, dtype=torch.bfloat16)
    st = fa.get_status()
    assert st == fa.FA_OK, fa.load().fa_status_string(st)
    O_ref, L_ref = oracle.fp8_attention_fwd(t_ref, scale, causal=causal, mask=inp["mask"])
    check_fwd(O, L, O_ref, L_ref, "bf16")


def test_debug_build_reports_its_status_code(debug_lib):
    assert debug_lib.fa_status_string(fa.FA_ERR_BOUNDS) == b"index check failed in a kernel (debug build)"
