"""Backward parity on the GPU: dQ, dK, dV from the CUDA path (C ABI) against the
fp64 oracle's gradients of sum(dO * O) on the same seeded, rounded inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import check_grads, guarded, guards_intact, oracle_inputs, rel_fro, to_np64

import exact_io_aware_26_gb300 as fa

pytestmark = pytest.mark.gpu


def _run(inp, causal=False, mask=None, mask_block=128, scale=None, guard=False):
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    m = None if mask is None else torch.as_tensor(mask, dtype=torch.uint8).cuda()
    o, lse = fa.attention_fwd(q, k, v, scale=scale, causal=causal, block_mask=m,
                              mask_block=mask_block)
    raws = None
    if guard:
        raws, views = zip(*(guarded(tuple(q.shape), q.dtype) for _ in range(3)))
        dq, dk, dv = fa.attention_bwd(q, k, v, o, do, lse, scale=scale, causal=causal,
                                      block_mask=m, mask_block=mask_block, dq=views[0],
                                      dk=views[1], dv=views[2])
    else:
        dq, dk, dv = fa.attention_bwd(q, k, v, o, do, lse, scale=scale, causal=causal,
                                      block_mask=m, mask_block=mask_block)
    assert fa.get_status() == fa.FA_OK
    if guard:
        torch.cuda.synchronize()
        assert all(guards_intact(r) for r in raws)
    return dq, dk, dv


def _ref(inp, causal=False, mask=None, mask_block=128, scale=None):
    o = oracle_inputs(inp)
    d = o["q"].shape[-1]
    return oracle.attention_bwd(o["q"], o["k"], o["v"], o["do"], scale or 1.0 / math.sqrt(d),
                                causal=causal, mask=mask, mask_block=mask_block)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 63, 127, 128, 129, 255, 1000])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_bwd_small(cuda_lib, dtype, d, N, causal):
    inp = synth.make_inputs(2, 3, N, d, dtype, seed=4000 + N + d)
    got = _run(inp, causal)
    check_grads(got, _ref(inp, causal), dtype)


@pytest.mark.parametrize("ctas", [1, 3, 5, 9, 50])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_bwd_sliced_key_tiles(cuda_lib, d, causal, ctas):
    """28 key tiles (B=2, H=2, N=777) planned for `ctas` CTAs per wave: 50 cuts
    every key tile into query slices that fill one wave; 3, 5 and 9 (non-causal)
    run most key tiles one CTA each and cut those of the last, partly filled
    wave; 1 runs one CTA per key tile.  Key tiles of several slices get their
    dK, dV from the finalize stage."""
    inp = synth.make_inputs(2, 2, 777, d, "bf16", seed=4200 + ctas + d)
    old = fa.set_bwd_ctas(ctas)
    try:
        got = _run(inp, causal, guard=True)
    finally:
        fa.set_bwd_ctas(old)
    check_grads(got, _ref(inp, causal), "bf16")


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_sliced_and_whole_key_tile_paths_agree(cuda_lib, causal):
    """The same gradients (up to summation order) whatever the CTA count."""
    inp = synth.make_inputs(1, 3, 1100, 64, "f16", seed=4300)  # 27 key tiles
    outs = []
    for ctas in (0, 1, 5, 23, 40):
        old = fa.set_bwd_ctas(ctas)
        try:
            outs.append([to_np64(g) for g in _run(inp, causal)])
        finally:
            fa.set_bwd_ctas(old)
    for o in outs[1:]:
        for g, g0 in zip(o, outs[0]):
            assert rel_fro(g, g0) <= 2e-3


@pytest.mark.parametrize("d,n_tiles,extra", [(64, 16, 8), (64, 16, 24), (64, 16, 72), (64, 8, 8), (64, 5, 3),
                                             (64, 16, 100), (128, 16, 8), (128, 6, 20)])
def test_bwd_last_partial_wave_split(cuda_lib, d, n_tiles, extra):
    """Non-causal grids of SMs + `extra` key tiles (one partly filled last wave): the
    leftover key tiles are split over the idle SMs (2 to 8 slices of their query
    tiles, fp32 partial dK, dV added up by the finalize stage; with 100 left over no
    split fits).  The last query tile is ragged."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H = -(-(sms + extra) // n_tiles)  # key tiles = H * n_tiles, just past sms + extra
    N = 128 * n_tiles - 37
    inp = synth.make_inputs(1, H, N, d, "bf16", seed=4500 + n_tiles + extra + d)
    got = _run(inp, False, guard=True)
    check_grads(got, _ref(inp, False), "bf16")


@pytest.mark.parametrize("mask_block", [128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_block_mask(cuda_lib, mask_block, causal):
    inp = synth.make_inputs(1, 2, 900, 64, "bf16", seed=4100 + mask_block, mask_p=0.4,
                            mask_block=mask_block)
    got = _run(inp, causal, inp["mask"], mask_block)
    check_grads(got, _ref(inp, causal, inp["mask"], mask_block), "bf16")


def test_bwd_per_head_masks_and_hidden_rows(cuda_lib):
    B, H, N, d, mb = 2, 2, 512, 128, 128
    inp = synth.make_inputs(B, H, N, d, "bf16", seed=4200)
    rng = np.random.default_rng(4201)
    m = (rng.random((B, H, 4, 4)) < 0.5).astype(np.uint8)
    m[0, 1, 2, :] = 0   # query block 2 of head (0,1) sees nothing
    m[1, 0, :, 3] = 0   # key block 3 of head (1,0) is seen by nobody
    got = _run(inp, False, m, mb)
    ref = _ref(inp, False, m, mb)
    check_grads(got, ref, "bf16")
    dq, dk, dv = got
    assert torch.all(dq[0, 1, 256:384] == 0)
    assert torch.all(dk[1, 0, 384:] == 0) and torch.all(dv[1, 0, 384:] == 0)


def test_bwd_outputs_stay_inside_their_buffers(cuda_lib):
    inp = synth.make_inputs(1, 2, 397, 64, "f16", seed=4300)
    got = _run(inp, True, guard=True)
    check_grads(got, _ref(inp, True), "f16")


def test_bwd_gradient_identities_on_gpu(cuda_lib):
    """sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i, per head."""
    inp = synth.make_inputs(1, 4, 1536, 64, "bf16", seed=4400)
    dq, dk, dv = _run(inp, True)
    do = inp["do"].double()
    assert (dk.double().sum(2)).abs().max().item() <= 0.02 * dk.double().abs().sum(2).max().item() + 1e-3
    np.testing.assert_allclose(to_np64(dv.sum(2)), to_np64(do.sum(2)), rtol=0,
                               atol=0.02 * float(do.abs().sum(2).max()))


# ------------------------------------------------------------------ workloads at full size


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_workload_b4h12_n2048_full(cuda_lib, causal):
    w = synth.WORKLOADS["bf16_b4h12_n2048"]
    inp = synth.workload_inputs(w)
    check_grads(_run(inp, causal), _ref(inp, causal), "bf16")


def test_bwd_workload_fp16_n8192_full_and_no_score_matrix(cuda_lib):
    w = synth.WORKLOADS["fp16_n8192"]
    inp = synth.workload_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.attention_fwd(q, k, v)
    ws = torch.empty(fa.workspace_bytes(q), dtype=torch.uint8, device="cuda")
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    fa.attention_bwd(q, k, v, o, do, lse, dq=dq, dk=dk, dv=dv, workspace=ws)
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated() - base
    assert peak <= 1 << 20, f"backward allocated {peak} bytes"
    # linear in N (D and the dQ accumulator) plus the slices' partial-sum slots,
    # whose size does not depend on N; the score matrix would be N^2 * 2 bytes
    linear = 8192 * 4 + 8192 * 64 * 4
    slots = 160 * 2 * 128 * 64 * 4
    assert ws.numel() <= linear + slots + 3 * 256
    assert ws.numel() < 8192 * 8192 * 2 // 4
    assert fa.get_status() == fa.FA_OK
    check_grads((dq, dk, dv), _ref(inp), "f16")


def _sampled(w, heads, nq, nk, seed, always=()):
    """Gradients of whole workloads at full size against the oracle on sampled rows of
    the listed heads: nq random query rows and nk random key rows, plus rows 0 and N - 1
    and every row in `always` (as query and as key rows)."""
    inp = synth.workload_inputs(w)
    causal = w.causal[0]
    dq, dk, dv = _run(inp, causal, inp["mask"], w.mask_block)
    rng = np.random.default_rng(seed)
    fixed = np.asarray([0, w.N - 1, *always], dtype=np.int64)
    for (b, h) in heads:
        qr = np.unique(np.concatenate([fixed, rng.integers(0, w.N, nq)])).astype(np.int32)
        kr = np.unique(np.concatenate([fixed, rng.integers(0, w.N, nk)])).astype(np.int32)
        o = oracle_inputs({n: inp[n][b, h] for n in ("q", "k", "v", "do")})
        mh = oracle.head_mask(inp["mask"], b, h, w.N, w.mask_block)
        rq, rk, rv = oracle.attention_bwd_rows(o["q"], o["k"], o["v"], o["do"], qr, kr, w.scale,
                                               causal=causal, mask_h=mh, mask_block=w.mask_block)
        for name, got, ref in (("dQ", dq[b, h, qr], rq), ("dK", dk[b, h, kr], rk),
                               ("dV", dv[b, h, kr], rv)):
            e = rel_fro(to_np64(got), ref)
            assert e <= 2e-2, (name, b, h, e)


def test_bwd_workload_trading_day_n23400_sampled(cuda_lib):
    """First, a middle and the last head; every row of the last, partial 104-row tile
    (rows 23296-23399) as query and as key rows."""
    w = synth.WORKLOADS["bf16_day_n23400"]
    _sampled(w, [(0, 0), (0, 5), (0, 11)], 256, 256, 44, always=range(23296, 23400))


def test_bwd_workload_block_sparse_n16384_sampled(cuda_lib):
    """First, a middle and the last head (of 32); the first and last 128-row tiles in full."""
    w = synth.WORKLOADS["bf16_sparse_n16384"]
    _sampled(w, [(0, 0), (1, 3), (1, 15)], 256, 256, 55,
             always=[*range(0, 128), *range(w.N - 128, w.N)])


def test_bwd_concurrent_streams(cuda_lib):
    """Two backward passes (one sliced, one with whole key tiles; separate workspaces) on
    two streams at once give the gradients they give one after the other, up to the
    order of the dQ accumulator's additions."""
    a = synth.make_inputs(1, 2, 1500, 64, "bf16", seed=4700)   # 24 key tiles: sliced
    b = synth.make_inputs(2, 12, 1024, 64, "bf16", seed=4701)  # 192 key tiles: whole
    probs = []
    for inp, causal in ((a, False), (b, True)):
        q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
        o, lse = fa.attention_fwd(q, k, v, causal=causal)
        probs.append((q, k, v, do, o, lse, causal))
    ref = [fa.attention_bwd(q, k, v, o, do, lse, causal=c) for q, k, v, do, o, lse, c in probs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    got = []
    for _ in range(3):
        for (q, k, v, do, o, lse, c), st in zip(probs, streams):
            with torch.cuda.stream(st):
                got.append(fa.attention_bwd(q, k, v, o, do, lse, causal=c, stream=st))
    torch.cuda.synchronize()
    assert fa.get_status() == fa.FA_OK
    for i, g in enumerate(got):
        for x, x0 in zip(g, ref[i % 2]):
            assert rel_fro(to_np64(x), to_np64(x0)) <= 1e-3
