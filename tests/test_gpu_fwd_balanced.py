"""Balanced forward on the GPU (fa_fwd_balanced): persistent CTAs with equal
shares of the (query tile, key tile) iterations, query tiles split between
CTAs merged by log-sum-exp.  Checked against the fp64 oracle on the same
seeded inputs, and against fa_fwd."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import check_fwd, guarded, guards_intact, oracle_inputs

import exact_io_aware_26_gb300 as fa

pytestmark = pytest.mark.gpu


def _run(inp, causal=False, ctas=0, scale=None):
    q, k, v = (inp[n].cuda() for n in "qkv")
    p, _ = fa.make_params(q, scale, causal)
    nbytes = fa.balanced_workspace_bytes(p)
    # the workspace's contents on entry must not matter: fill it with NaN bytes
    ws = torch.full((max(nbytes, 1),), 0xFF, dtype=torch.uint8, device="cuda")
    old = fa.set_fwd_ctas(ctas)
    try:
        O, L = fa.attention_fwd_balanced(q, k, v, scale=scale, causal=causal, workspace=ws)
    finally:
        fa.set_fwd_ctas(old)
    assert fa.get_status() == fa.FA_OK
    return O, L


def _ref(inp, causal=False, scale=None):
    o = oracle_inputs(inp)
    d = o["q"].shape[-1]
    return oracle.attention_fwd(o["q"], o["k"], o["v"], scale or 1.0 / math.sqrt(d), causal=causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 300, 1000, 2047])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_balanced_fwd_small(cuda_lib, dtype, d, N, causal):
    inp = synth.make_inputs(2, 3, N, d, dtype, seed=6000 + N + d, backward=False)
    O, L = _run(inp, causal)
    check_fwd(O, L, *_ref(inp, causal), dtype)


@pytest.mark.parametrize("ctas", [1, 2, 3, 7, 50])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_balanced_fwd_few_ctas_share_query_tiles(cuda_lib, d, causal, ctas):
    """A cap on the CTAs makes each walk several query tiles, most of them split."""
    inp = synth.make_inputs(2, 2, 777, d, "bf16", seed=6100 + ctas + d, backward=False)
    O, L = _run(inp, causal, ctas)
    check_fwd(O, L, *_ref(inp, causal), "bf16")


def test_balanced_fwd_matches_fa_fwd(cuda_lib):
    inp = synth.make_inputs(1, 4, 1536, 64, "bf16", seed=6200, backward=False)
    q, k, v = (inp[n].cuda() for n in "qkv")
    for causal in (False, True):
        O1, L1 = fa.attention_fwd(q, k, v, causal=causal)
        for ctas in (0, 5, 37):
            O, L = _run(inp, causal, ctas)
            assert (O.float() - O1.float()).abs().max().item() <= 2e-2
            assert (L - L1).abs().max().item() <= 1e-4


def test_balanced_fwd_with_block_mask_is_fa_fwd(cuda_lib):
    inp = synth.make_inputs(1, 2, 700, 64, "bf16", seed=6300, mask_p=0.4, backward=False)
    q, k, v = (inp[n].cuda() for n in "qkv")
    m = torch.as_tensor(inp["mask"], dtype=torch.uint8).cuda()
    O1, L1 = fa.attention_fwd(q, k, v, block_mask=m)
    O, L = fa.attention_fwd_balanced(q, k, v, block_mask=m)
    assert torch.equal(O, O1) and torch.equal(L, L1)


def test_balanced_fwd_outputs_stay_inside_their_buffers(cuda_lib):
    B, H, N, d = 1, 2, 383, 128
    inp = synth.make_inputs(B, H, N, d, "f16", seed=6400, backward=False)
    q, k, v = (inp[n].cuda() for n in "qkv")
    p, _ = fa.make_params(q, causal=True)
    raw_w, ws = guarded((fa.balanced_workspace_bytes(p),), torch.uint8)
    raw_o, O = guarded((B, H, N, d), torch.float16)
    raw_l, L = guarded((B, H, N), torch.float32)
    old = fa.set_fwd_ctas(4)
    try:
        fa.attention_fwd_balanced(q, k, v, causal=True, out=O, lse=L, workspace=ws)
    finally:
        fa.set_fwd_ctas(old)
    assert fa.get_status() == fa.FA_OK
    torch.cuda.synchronize()
    assert guards_intact(raw_o) and guards_intact(raw_l) and guards_intact(raw_w)
    check_fwd(O, L, *_ref(inp, True), "f16")


@pytest.mark.parametrize("causal", [False, True])
def test_balanced_fwd_workload_b4h12_n2048_full(cuda_lib, causal):
    w = synth.WORKLOADS["bf16_b4h12_n2048"]
    inp = synth.workload_inputs(w)
    O, L = _run(inp, causal)
    check_fwd(O, L, *_ref(inp, causal), "bf16")


def test_balanced_fwd_workload_trading_day_sampled(cuda_lib):
    w = synth.WORKLOADS["bf16_day_n23400"]
    inp = synth.workload_inputs(w)
    O, L = _run(inp, True)
    rng = np.random.default_rng(7)
    for h in (0, 11):
        rows = np.unique(np.concatenate([[0, 1, 127, 128, w.N - 1], rng.integers(0, w.N, 400)]))
        rows = rows.astype(np.int32)
        o = oracle_inputs({n: inp[n][0, h] for n in "qkv"})
        O_ref, L_ref = oracle.attention_fwd_rows(o["q"], o["k"], o["v"], rows, w.scale, causal=True)
        check_fwd(O[0, h, rows], L[0, h, rows], O_ref, L_ref, w.dtype)
