"""Split-KV forward on the GPU (fa_fwd_split): every query tile's key range cut
into slices run by the CTAs of one cluster and merged by their running
statistics in shared memory.  Checked against the fp64 oracle on the same seeded
inputs, and against the unsplit forward."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import check_fwd, check_grads, guarded, guards_intact, oracle_inputs

import exact_io_aware_26_gb300 as fa

pytestmark = pytest.mark.gpu


def _run(inp, splits, causal=False, mask=None, mask_block=128, scale=None):
    q, k, v = (inp[n].cuda() for n in "qkv")
    m = None if mask is None else torch.as_tensor(mask, dtype=torch.uint8).cuda()
    # the outputs' contents on entry must not matter: fill them with NaN bytes
    O = torch.full(q.shape, float("nan"), dtype=q.dtype, device="cuda")
    L = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    fa.attention_fwd_split(q, k, v, scale=scale, causal=causal, block_mask=m, mask_block=mask_block,
                           splits=splits, out=O, lse=L)
    assert fa.get_status() == fa.FA_OK
    return O, L


def _ref(inp, causal=False, mask=None, mask_block=128, scale=None):
    o = oracle_inputs(inp)
    d = o["q"].shape[-1]
    return oracle.attention_fwd(o["q"], o["k"], o["v"], scale or 1.0 / math.sqrt(d), causal=causal,
                                mask=mask, mask_block=mask_block)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,splits", [(129, 2), (300, 3), (1000, 2), (1000, 5), (1000, 8),
                                      (1000, 7), (2047, 6), (2047, 8)])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_split_fwd_small(cuda_lib, dtype, d, N, splits, causal):
    inp = synth.make_inputs(2, 3, N, d, dtype, seed=5000 + N + d + splits, backward=False)
    O, L = _run(inp, splits, causal)
    check_fwd(O, L, *_ref(inp, causal), dtype)


@pytest.mark.parametrize("causal", [False, True])
def test_split_fwd_block_mask_and_hidden_rows(cuda_lib, causal):
    B, H, N, d, mb = 2, 3, 1024, 64, 128
    inp = synth.make_inputs(B, H, N, d, "bf16", seed=5100, backward=False)
    rng = np.random.default_rng(5101)
    m = (rng.random((B, H, 8, 8)) < 0.4).astype(np.uint8)
    m[0, 1, 5, :] = 0   # every key of query block 5 hidden in head (0, 1)
    m[1, 2, :, :] = 0   # a head with nothing visible
    m[0, 0, :, 4:] = 0  # whole slices hidden for every query block of head (0, 0)
    O, L = _run(inp, 4, causal, m, mb)
    O_ref, L_ref = _ref(inp, causal, m, mb)
    check_fwd(O, L, O_ref, L_ref, "bf16")
    assert torch.all(O[0, 1, 640:768] == 0) and torch.all(torch.isneginf(L[0, 1, 640:768]))
    assert torch.all(O[1, 2] == 0) and torch.all(torch.isneginf(L[1, 2]))


def test_split_fwd_matches_unsplit(cuda_lib):
    """Same O and LSE as fa_fwd up to rounding order, for every split count."""
    inp = synth.make_inputs(1, 4, 1536, 64, "bf16", seed=5200, backward=False)
    q, k, v = (inp[n].cuda() for n in "qkv")
    O1, L1 = fa.attention_fwd(q, k, v, causal=True)
    for s in (1, 2, 3, 4, 6, 7, 8):
        O, L = _run(inp, s, True)
        assert (O.float() - O1.float()).abs().max().item() <= 2e-2
        assert (L - L1).abs().max().item() <= 1e-4
    O, L = _run(inp, 1, True)
    assert torch.equal(O, O1) and torch.equal(L, L1)  # one slice is fa_fwd itself


def test_split_fwd_outputs_stay_inside_their_buffers(cuda_lib):
    B, H, N, d = 1, 2, 383, 128
    inp = synth.make_inputs(B, H, N, d, "f16", seed=5300, backward=False)
    q, k, v = (inp[n].cuda() for n in "qkv")
    raw_o, O = guarded((B, H, N, d), torch.float16)
    raw_l, L = guarded((B, H, N), torch.float32)
    fa.attention_fwd_split(q, k, v, causal=True, splits=3, out=O, lse=L)
    assert fa.get_status() == fa.FA_OK
    torch.cuda.synchronize()
    assert guards_intact(raw_o) and guards_intact(raw_l)
    check_fwd(O, L, *_ref(inp, True), "f16")


def test_split_fwd_lse_drives_the_backward(cuda_lib):
    """The merged LSE is the one the backward recomputes P from."""
    inp = synth.make_inputs(1, 2, 700, 64, "bf16", seed=5400)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    O, L = fa.attention_fwd_split(q, k, v, causal=True, splits=3)
    dq, dk, dv = fa.attention_bwd(q, k, v, O, do, L, causal=True)
    assert fa.get_status() == fa.FA_OK
    o = oracle_inputs(inp)
    ref = oracle.attention_bwd(o["q"], o["k"], o["v"], o["do"], 0.125, causal=True)
    check_grads((dq, dk, dv), ref, "bf16")


def test_split_count_on_this_device(cuda_lib):
    w = synth.WORKLOADS["fp16_n8192"]
    q = torch.empty((w.B, w.H, w.N, w.d), dtype=torch.float16, device="cuda")
    p, _ = fa.make_params(q)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert fa.num_splits(p) == fa.num_splits(p, sms) > 1


def test_split_fwd_workload_fp16_n8192_full(cuda_lib):
    """One head, N = 8192: 64 query tiles, split to fill the GPU."""
    w = synth.WORKLOADS["fp16_n8192"]
    inp = synth.workload_inputs(w)
    q = inp["q"].cuda()
    p, _ = fa.make_params(q)
    s = fa.num_splits(p)
    assert s > 1
    O, L = _run(inp, s)
    check_fwd(O, L, *_ref(inp), "f16")


def test_split_fwd_workload_trading_day_sampled(cuda_lib):
    """Causal N = 23400 with 8 slices: sampled rows against the oracle."""
    w = synth.WORKLOADS["bf16_day_n23400"]
    inp = synth.workload_inputs(w)
    O, L = _run(inp, 8, True)
    rng = np.random.default_rng(6)
    for h in (0, 7):
        rows = np.unique(np.concatenate([[0, 1, 127, 128, w.N - 1], rng.integers(0, w.N, 400)]))
        rows = rows.astype(np.int32)
        o = oracle_inputs({n: inp[n][0, h] for n in "qkv"})
        O_ref, L_ref = oracle.attention_fwd_rows(o["q"], o["k"], o["v"], rows, w.scale, causal=True)
        check_fwd(O[0, h, rows], L[0, h, rows], O_ref, L_ref, w.dtype)


@pytest.mark.parametrize("causal", [False, True])
def test_split_fwd_d128_block_mask(cuda_lib, causal):
    """d = 128 with a block mask and 3 slices per query tile: the slices' cluster merge
    against the oracle."""
    inp = synth.make_inputs(1, 3, 1100, 128, "bf16", seed=5600, mask_p=0.5, backward=False)
    O, L = _run(inp, 3, causal, inp["mask"], 128)
    check_fwd(O, L, *_ref(inp, causal, inp["mask"], 128), "bf16")


def test_split_fwd_concurrent_streams(cuda_lib):
    """Two split forwards (different problems, different slice counts) on two streams
    at once give the results they give one after the other."""
    a = synth.make_inputs(1, 2, 2000, 64, "bf16", seed=5700, backward=False)
    b = synth.make_inputs(2, 1, 1500, 128, "f16", seed=5701, backward=False)
    ta = [a[n].cuda() for n in "qkv"]
    tb = [b[n].cuda() for n in "qkv"]
    Oa, La = fa.attention_fwd_split(*ta, causal=True, splits=5)
    Ob, Lb = fa.attention_fwd_split(*tb, causal=False, splits=3)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(3):
        with torch.cuda.stream(s1):
            oa, la = fa.attention_fwd_split(*ta, causal=True, splits=5, stream=s1)
        with torch.cuda.stream(s2):
            ob, lb = fa.attention_fwd_split(*tb, causal=False, splits=3, stream=s2)
        outs.append((oa, la, ob, lb))
    torch.cuda.synchronize()
    assert fa.get_status() == fa.FA_OK
    for oa, la, ob, lb in outs:
        assert torch.equal(oa, Oa) and torch.equal(la, La)
        assert torch.equal(ob, Ob) and torch.equal(lb, Lb)
