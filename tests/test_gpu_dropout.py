"""Dropout on the GPU: the kernels regenerate the oracle's keep decisions
(Philox4x32-10 with counter (key / 4, query, b*H + h, offset)) bit for bit, and
their outputs and gradients match the fp64 oracle with the same dropout_p, seed
and offset.

Keep decisions are read back exactly: with Q = 0 every allowed weight of row i
is 1 / |A_i|, so with V holding an identity block over d keys, O[i, c] is
z_ij / |A_i| for key j of that block (0 exactly when dropped); with dO holding
an identity block over d queries, dV[j, c] is P_ij z_ij for query i of that
block."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import check_fwd, check_grads, oracle_inputs

import exact_io_aware_26_gb300 as fa

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def _allowed(N, causal):
    a = np.ones((N, N), dtype=bool)
    return np.tril(a) if causal else a


def _fwd_keep(B, H, N, d, dtype, causal, p, seed, offset, splits=None):
    """Keep decisions [B,H,N,N] as the forward kernel applied them."""
    t = DT[dtype]
    q = torch.zeros((B, H, N, d), dtype=t, device="cuda")
    k = torch.randn((B, H, N, d), dtype=torch.float32, device="cuda").to(t)
    keep = np.zeros((B, H, N, N), dtype=np.uint8)
    for j0 in range(0, N, d):
        v = torch.zeros((B, H, N, d), dtype=t, device="cuda")
        n = min(d, N - j0)
        v[:, :, j0:j0 + n, :n] = torch.eye(n, dtype=t, device="cuda")
        if splits is None:
            O, _ = fa.attention_fwd(q, k, v, causal=causal, dropout_p=p, seed=seed, offset=offset)
        else:
            O, _ = fa.attention_fwd_split(q, k, v, causal=causal, splits=splits, dropout_p=p,
                                          seed=seed, offset=offset)
        assert fa.get_status() == fa.FA_OK
        keep[:, :, :, j0:j0 + n] = (O[:, :, :, :n].float() > 0).cpu().numpy()
    return keep


def _bwd_keep(B, H, N, d, dtype, causal, p, seed, offset):
    """Keep decisions [B,H,N,N] as the backward kernel applied them (from dV)."""
    t = DT[dtype]
    q = torch.zeros((B, H, N, d), dtype=t, device="cuda")
    k = torch.randn((B, H, N, d), dtype=torch.float32, device="cuda").to(t)
    v = torch.randn((B, H, N, d), dtype=torch.float32, device="cuda").to(t)
    o, lse = fa.attention_fwd(q, k, v, causal=causal, dropout_p=p, seed=seed, offset=offset)
    keep = np.zeros((B, H, N, N), dtype=np.uint8)
    for i0 in range(0, N, d):
        do = torch.zeros((B, H, N, d), dtype=t, device="cuda")
        n = min(d, N - i0)
        do[:, :, i0:i0 + n, :n] = torch.eye(n, dtype=t, device="cuda")
        _, _, dv = fa.attention_bwd(q, k, v, o, do, lse, causal=causal, dropout_p=p, seed=seed,
                                    offset=offset)
        assert fa.get_status() == fa.FA_OK
        # dV[j, c] = P_{i0+c, j} z_{i0+c, j}
        keep[:, :, i0:i0 + n, :] = (dv[:, :, :, :n].float() > 0).permute(0, 1, 3, 2).cpu().numpy()
    return keep


def _expect_keep(B, H, N, causal, p, seed, offset):
    return oracle.dropout_keep(B, H, N, p, seed, offset) & _allowed(N, causal)[None, None]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,dtype", [(64, "f16"), (128, "bf16"), (64, "f32")])
def test_forward_applies_the_oracle_keep_decisions(cuda_lib, d, dtype, causal):
    B, H, N, p, seed, off = 2, 3, 300, 0.4, 0xDEADBEEF12345, 3
    got = _fwd_keep(B, H, N, d, dtype, causal, p, seed, off)
    assert np.array_equal(got, _expect_keep(B, H, N, causal, p, seed, off))


def test_split_forward_applies_the_oracle_keep_decisions(cuda_lib):
    B, H, N, p, seed, off = 1, 2, 640, 0.3, 77, 0
    got = _fwd_keep(B, H, N, 128, "f16", False, p, seed, off, splits=3)
    assert np.array_equal(got, _expect_keep(B, H, N, False, p, seed, off))


@pytest.mark.parametrize("ctas", [0, 1])  # 0: key tiles cut into query slices (few key tiles); 1: whole
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,dtype", [(64, "f16"), (128, "bf16")])
def test_backward_regenerates_the_oracle_keep_decisions(cuda_lib, d, dtype, causal, ctas):
    B, H, N, p, seed, off = 1, 2, 300, 0.45, 2 ** 40 + 9, 11
    old = fa.set_bwd_ctas(ctas)
    try:
        got = _bwd_keep(B, H, N, d, dtype, causal, p, seed, off)
    finally:
        fa.set_bwd_ctas(old)
    assert np.array_equal(got, _expect_keep(B, H, N, causal, p, seed, off))


def _ref_fwd(inp, causal, p, seed, off):
    o = oracle_inputs(inp)
    d = o["q"].shape[-1]
    return oracle.attention_fwd(o["q"], o["k"], o["v"], 1.0 / math.sqrt(d), causal=causal,
                                dropout_p=p, seed=seed, offset=off)


@pytest.mark.parametrize("p", [0.1, 0.5])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 300, 1000])
@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (64, "f16"), (128, "bf16")])
def test_dropout_forward_matches_oracle(cuda_lib, d, dtype, N, causal, p):
    inp = synth.make_inputs(2, 3, N, d, dtype, seed=9000 + N + d, backward=False)
    q, k, v = (inp[n].cuda() for n in "qkv")
    O, L = fa.attention_fwd(q, k, v, causal=causal, dropout_p=p, seed=1234, offset=5)
    assert fa.get_status() == fa.FA_OK
    check_fwd(O, L, *_ref_fwd(inp, causal, p, 1234, 5), dtype)


def test_dropout_fp32_forward_matches_oracle(cuda_lib):
    inp = synth.make_inputs(1, 2, 257, 64, "f32", seed=9100, backward=False)
    q, k, v = (inp[n].cuda() for n in "qkv")
    for causal in (False, True):
        O, L = fa.attention_fwd(q, k, v, causal=causal, dropout_p=0.2, seed=8, offset=1)
        assert fa.get_status() == fa.FA_OK
        check_fwd(O, L, *_ref_fwd(inp, causal, 0.2, 8, 1), "f32")


def test_dropout_split_forward_matches_oracle(cuda_lib):
    inp = synth.make_inputs(1, 2, 1500, 64, "bf16", seed=9200, backward=False)
    q, k, v = (inp[n].cuda() for n in "qkv")
    O, L = fa.attention_fwd_split(q, k, v, causal=True, splits=4, dropout_p=0.25, seed=3,
                                  offset=0)
    assert fa.get_status() == fa.FA_OK
    check_fwd(O, L, *_ref_fwd(inp, True, 0.25, 3, 0), "bf16")


@pytest.mark.parametrize("ctas", [0, 1, 5])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (64, "f16"), (128, "bf16")])
def test_dropout_backward_matches_oracle(cuda_lib, d, dtype, causal, ctas):
    B, H, N, p, seed, off = 2, 2, 777, 0.2, 31337, 2
    inp = synth.make_inputs(B, H, N, d, dtype, seed=9300 + d + ctas)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    old = fa.set_bwd_ctas(ctas)
    try:
        O, L = fa.attention_fwd(q, k, v, causal=causal, dropout_p=p, seed=seed, offset=off)
        got = fa.attention_bwd(q, k, v, O, do, L, causal=causal, dropout_p=p, seed=seed,
                               offset=off)
        assert fa.get_status() == fa.FA_OK
    finally:
        fa.set_bwd_ctas(old)
    o = oracle_inputs(inp)
    ref = oracle.attention_bwd(o["q"], o["k"], o["v"], o["do"], 1.0 / math.sqrt(d),
                               causal=causal, dropout_p=p, seed=seed, offset=off)
    check_grads(got, ref, dtype)


def test_dropout_is_deterministic_and_follows_seed_and_offset(cuda_lib):
    inp = synth.make_inputs(1, 2, 512, 64, "bf16", seed=9400)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    runs = {}
    for key in ((5, 0), (5, 0), (6, 0), (5, 1)):
        O, L = fa.attention_fwd(q, k, v, dropout_p=0.3, seed=key[0], offset=key[1])
        g = fa.attention_bwd(q, k, v, O, do, L, dropout_p=0.3, seed=key[0], offset=key[1])
        runs.setdefault(key, []).append((O, L) + tuple(g))
    a, b = runs[(5, 0)]
    assert all(torch.equal(x, y) for x, y in zip(a[:2], b[:2]))  # the forward is deterministic
    assert torch.equal(a[4], b[4]) and torch.equal(a[3], b[3])   # dK, dV too (no atomics)
    assert not torch.equal(a[0], runs[(6, 0)][0][0])
    assert not torch.equal(a[0], runs[(5, 1)][0][0])
    assert torch.equal(a[1], runs[(6, 0)][0][1])  # LSE does not depend on the dropout draw


def test_dropout_workload_b4h12_n2048_sampled(cuda_lib):
    """The full headline shape with p = 0.1: sampled rows against the oracle."""
    w = synth.WORKLOADS["bf16_b4h12_n2048"]
    inp = synth.workload_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    p, seed, off = 0.1, 20260101, 7
    O, L = fa.attention_fwd(q, k, v, causal=True, dropout_p=p, seed=seed, offset=off)
    dq, dk, dv = fa.attention_bwd(q, k, v, O, do, L, causal=True, dropout_p=p, seed=seed, offset=off)
    assert fa.get_status() == fa.FA_OK
    rng = np.random.default_rng(12)
    for (b, h) in ((0, 0), (3, 11)):
        bh = b * w.H + h
        rows = np.unique(np.concatenate([[0, 127, 128, w.N - 1], rng.integers(0, w.N, 60)]))
        rows = rows.astype(np.int32)
        o = oracle_inputs({n: inp[n][b, h] for n in ("q", "k", "v", "do")})
        O_ref, L_ref = oracle.attention_fwd_rows(o["q"], o["k"], o["v"], rows, w.scale, causal=True,
                                                 dropout_p=p, seed=seed, offset=off, bh=bh)
        check_fwd(O[b, h, rows], L[b, h, rows], O_ref, L_ref, w.dtype)
        a, b_, c = oracle.attention_bwd_rows(o["q"], o["k"], o["v"], o["do"], rows, rows, w.scale,
                                             causal=True, dropout_p=p, seed=seed, offset=off, bh=bh)
        check_grads((dq[b, h, rows], dk[b, h, rows], dv[b, h, rows]), (a, b_, c), w.dtype)
