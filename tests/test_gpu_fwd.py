"""Forward parity on the GPU: the CUDA path (through the C ABI) against the fp64
oracle on the same seeded, dtype-rounded inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import DTYPES, check_fwd, guarded, guards_intact, oracle_inputs, to_np64

import exact_io_aware_26_gb300 as fa

pytestmark = pytest.mark.gpu


def _run(inp, causal=False, mask=None, mask_block=128, scale=None):
    q, k, v = (inp[n].cuda() for n in "qkv")
    m = None if mask is None else torch.as_tensor(mask, dtype=torch.uint8).cuda()
    O, L = fa.attention_fwd(q, k, v, scale=scale, causal=causal, block_mask=m, mask_block=mask_block)
    assert fa.get_status() == fa.FA_OK
    return O, L


def _ref(inp, causal=False, mask=None, mask_block=128, scale=None):
    o = oracle_inputs(inp)
    d = o["q"].shape[-1]
    return oracle.attention_fwd(o["q"], o["k"], o["v"], scale or 1.0 / math.sqrt(d), causal=causal,
                                mask=mask, mask_block=mask_block)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 63, 127, 128, 129, 255, 1000])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_fwd_tensor_core_small(cuda_lib, dtype, d, N, causal):
    inp = synth.make_inputs(2, 3, N, d, dtype, seed=1000 + N + d, backward=False)
    O, L = _run(inp, causal)
    check_fwd(O, L, *_ref(inp, causal), dtype)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 63, 256, 300])
@pytest.mark.parametrize("d", [64, 128])
def test_fwd_fp32_small(cuda_lib, d, N, causal):
    inp = synth.make_inputs(1, 2, N, d, "f32", seed=2000 + N + d, backward=False)
    O, L = _run(inp, causal)
    check_fwd(O, L, *_ref(inp, causal), "f32")


def test_fwd_fp32_workload_n256(cuda_lib):
    w = synth.WORKLOADS["fp32_n256"]
    inp = synth.workload_inputs(w)
    O, L = _run(inp)
    eo, el = check_fwd(O, L, *_ref(inp), "f32")
    assert eo <= 1e-5 and el <= 1e-5


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("mask_block", [128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_block_mask(cuda_lib, dtype, mask_block, causal):
    N, d = 700, 64
    inp = synth.make_inputs(1, 2, N, d, dtype, seed=3000 + mask_block, mask_p=0.4,
                            mask_block=mask_block, backward=False)
    O, L = _run(inp, causal, inp["mask"], mask_block)
    check_fwd(O, L, *_ref(inp, causal, inp["mask"], mask_block), dtype)


def test_fwd_per_head_masks_and_hidden_rows(cuda_lib):
    B, H, N, d, mb = 2, 3, 512, 128, 128
    inp = synth.make_inputs(B, H, N, d, "bf16", seed=3100, backward=False)
    rng = np.random.default_rng(3101)
    m = (rng.random((B, H, 4, 4)) < 0.5).astype(np.uint8)
    m[0, 1, 2, :] = 0  # every key of query block 2 hidden in head (0, 1)
    m[1, 2, :, :] = 0  # a head with nothing visible
    O, L = _run(inp, False, m, mb)
    O_ref, L_ref = _ref(inp, False, m, mb)
    check_fwd(O, L, O_ref, L_ref, "bf16")
    assert torch.all(O[0, 1, 256:384] == 0) and torch.all(torch.isneginf(L[0, 1, 256:384]))
    assert torch.all(O[1, 2] == 0)


def test_fwd_scale_other_than_inverse_sqrt_d(cuda_lib):
    inp = synth.make_inputs(1, 2, 333, 64, "bf16", seed=3200, backward=False)
    O, L = _run(inp, True, scale=0.05)
    check_fwd(O, L, *_ref(inp, True, scale=0.05), "bf16")


def test_fwd_shift_invariance_on_gpu(cuda_lib):
    """Adding u to every key row leaves O unchanged and moves LSE_i by scale * q_i . u."""
    inp = synth.make_inputs(1, 1, 640, 64, "f32", seed=3300, backward=False)
    u = torch.randn(64, generator=torch.Generator().manual_seed(3))
    inp2 = dict(inp, k=(inp["k"] + u).contiguous())
    O1, L1 = _run(inp, True)
    O2, L2 = _run(inp2, True)
    assert (O1 - O2).abs().max().item() <= 1e-5
    shift = 0.125 * (inp["q"].double() @ u.double()).cuda()
    assert ((L2.double() - L1.double()) - shift).abs().max().item() <= 1e-4


def test_fwd_outputs_stay_inside_their_buffers(cuda_lib):
    B, H, N, d = 1, 2, 383, 128
    inp = synth.make_inputs(B, H, N, d, "bf16", seed=3400, backward=False)
    q, k, v = (inp[n].cuda() for n in "qkv")
    raw_o, O = guarded((B, H, N, d), torch.bfloat16)
    raw_l, L = guarded((B, H, N), torch.float32)
    fa.attention_fwd(q, k, v, causal=True, out=O, lse=L)
    assert fa.get_status() == fa.FA_OK
    torch.cuda.synchronize()
    assert guards_intact(raw_o) and guards_intact(raw_l)
    check_fwd(O, L, *_ref(inp, True), "bf16")


# ------------------------------------------------------------------ workloads at full size


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_workload_b4h12_n2048_full(cuda_lib, causal):
    w = synth.WORKLOADS["bf16_b4h12_n2048"]
    inp = synth.workload_inputs(w)
    O, L = _run(inp, causal)
    check_fwd(O, L, *_ref(inp, causal), "bf16")


def test_fwd_workload_fp16_n8192_full_and_no_score_matrix(cuda_lib):
    w = synth.WORKLOADS["fp16_n8192"]
    inp = synth.workload_inputs(w)
    q, k, v = (inp[n].cuda() for n in "qkv")
    O = torch.empty_like(q)
    L = torch.empty(q.shape[:3], device="cuda", dtype=torch.float32)
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    fa.attention_fwd(q, k, v, out=O, lse=L)
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated() - base
    assert peak <= 1 << 20, f"forward allocated {peak} bytes; the score matrix would be {8192 * 8192 * 2}"
    assert fa.get_status() == fa.FA_OK
    check_fwd(O, L, *_ref(inp), "f16")


def _sampled_rows(w, heads, rows_per_head, seed, always=()):
    inp = synth.workload_inputs(w)
    causal = w.causal[0]
    O, L = _run(inp, causal, inp["mask"], w.mask_block)
    rng = np.random.default_rng(seed)
    for (b, h) in heads:
        rows = np.unique(np.concatenate([
            [0, 1, w.N - 1, w.N - 2], np.asarray(list(always), dtype=np.int64),
            rng.integers(0, w.N, rows_per_head)])).astype(np.int32)
        o = oracle_inputs({n: inp[n][b, h] for n in "qkv"})
        mh = oracle.head_mask(inp["mask"], b, h, w.N, w.mask_block)
        O_ref, L_ref = oracle.attention_fwd_rows(o["q"], o["k"], o["v"], rows, w.scale,
                                                 causal=causal, mask_h=mh,
                                                 mask_block=w.mask_block)
        check_fwd(O[b, h, rows], L[b, h, rows], O_ref, L_ref, w.dtype)


def test_fwd_workload_trading_day_n23400_sampled(cuda_lib):
    """First, a middle and the last head; every row of the last, partial 104-row tile."""
    w = synth.WORKLOADS["bf16_day_n23400"]
    _sampled_rows(w, [(0, 0), (0, 5), (0, 11)], 600, 4, always=range(23296, 23400))


def test_fwd_workload_block_sparse_n16384_sampled(cuda_lib):
    w = synth.WORKLOADS["bf16_sparse_n16384"]
    _sampled_rows(w, [(0, 0), (1, 3), (1, 15)], 400, 5, always=range(w.N - 128, w.N))


# ------------------------------------------------------------------ failure detection


def test_barrier_timeout_is_reported_without_faulting(cuda_lib):
    old = fa.set_wait_limit_ns(20_000_000)  # 20 ms
    try:
        fa.selftest_timeout()
        assert fa.get_status() == fa.FA_ERR_TIMEOUT
        assert fa.get_status() == fa.FA_OK  # read-and-clear
    finally:
        fa.set_wait_limit_ns(old)
    # the context is still usable
    inp = synth.make_inputs(1, 1, 200, 64, "bf16", seed=3500, backward=False)
    O, L = _run(inp, True)
    check_fwd(O, L, *_ref(inp, True), "bf16")
