"""Pins of the fp64 CPU oracle to facts that do not come from the oracle itself.

Each test ties one part of the oracle to something the pages or the mathematics
fix: a library routine that computes the same special case, a closed form, an
invariant, a value the pages print, or brute-force finite differences.  Together
they are chosen so that a dropped term, a wrong sign, a transposed operand, a
misplaced scale or a mis-indexed mask fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _torch_attention(q, k, v, scale, causal=False, dense_mask=None):
    """softmax(scale * Q K^T) V in torch fp64 with explicit masking (library route)."""
    q, k, v = (torch.tensor(x, dtype=torch.float64) for x in (q, k, v))
    s = scale * q @ k.transpose(-1, -2)
    N = q.shape[-2]
    hide = torch.zeros(N, N, dtype=torch.bool)
    if causal:
        hide |= torch.triu(torch.ones(N, N, dtype=torch.bool), diagonal=1)
    if dense_mask is not None:
        hide = hide | ~torch.as_tensor(dense_mask, dtype=torch.bool)
    s = s.masked_fill(hide, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return (torch.softmax(s, dim=-1) @ v).numpy(), lse.numpy()


def _expand_mask(m, N, mb):
    idx = np.arange(N) // mb
    return m[np.ix_(idx, idx)]


# ---------------------------------------------------------------- forward


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 8), (37, 16), (130, 64)])
def test_fwd_equals_library_softmax(causal, N, d):
    q, k, v = (_rand((2, 3, N, d), s) for s in (1, 2, 3))
    scale = 1.0 / math.sqrt(d)
    O, L = oracle.attention_fwd(q, k, v, scale, causal=causal)
    Ot, Lt = _torch_attention(q, k, v, scale, causal)
    assert np.abs(O - Ot).max() <= 1e-12
    assert np.abs(L - Lt).max() <= 1e-12
    sd = torch.nn.functional.scaled_dot_product_attention(
        *(torch.tensor(x) for x in (q, k, v)), is_causal=causal, scale=scale).numpy()
    assert np.abs(O - sd).max() <= 1e-12


def test_single_key_gives_v_and_scaled_logit():
    q, k, v = (_rand((1, 2, 1, 32), s) for s in (4, 5, 6))
    O, L = oracle.attention_fwd(q, k, v, 0.3)
    np.testing.assert_allclose(O, v, rtol=0, atol=1e-15)
    np.testing.assert_allclose(L[..., 0], 0.3 * np.sum(q[..., 0, :] * k[..., 0, :], -1),
                               rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_allowed_values(causal):
    N, d = 50, 8
    q, v = _rand((1, 1, N, d), 7), _rand((1, 1, N, d), 8)
    krow = _rand((d,), 9)
    k = np.broadcast_to(krow, (1, 1, N, d)).copy()
    O, L = oracle.attention_fwd(q, k, v, 0.125, causal=causal)
    for i in range(N):
        n_allowed = i + 1 if causal else N
        np.testing.assert_allclose(O[0, 0, i], v[0, 0, :n_allowed].mean(0), rtol=0, atol=1e-13)
        expect = 0.125 * q[0, 0, i] @ krow + math.log(n_allowed)
        assert abs(L[0, 0, i] - expect) <= 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_shift_of_keys_leaves_output_and_moves_lse(causal):
    N, d = 40, 16
    q, k, v = (_rand((1, 2, N, d), s) for s in (10, 11, 12))
    u = _rand((d,), 13)
    O, L = oracle.attention_fwd(q, k, v, 0.25, causal=causal)
    O2, L2 = oracle.attention_fwd(q, k + u, v, 0.25, causal=causal)
    assert np.abs(O - O2).max() <= 1e-12
    np.testing.assert_allclose(L2 - L, 0.25 * (q @ u), rtol=0, atol=1e-12)


def test_rows_sum_to_one_and_linearity_in_v():
    N, d = 33, 8
    q, k, v = (_rand((1, 1, N, d), s) for s in (14, 15, 16))
    O1, _ = oracle.attention_fwd(q, k, np.ones_like(v), 0.5, causal=True)
    assert np.abs(O1 - 1.0).max() <= 1e-13
    O, _ = oracle.attention_fwd(q, k, v, 0.5)
    Oa, _ = oracle.attention_fwd(q, k, 3.0 * v - 2.0, 0.5)
    np.testing.assert_allclose(Oa, 3.0 * O - 2.0, rtol=0, atol=1e-12)


def test_causal_first_row_sees_only_itself():
    q, k, v = (_rand((1, 1, 20, 8), s) for s in (17, 18, 19))
    O, L = oracle.attention_fwd(q, k, v, 0.7, causal=True)
    np.testing.assert_allclose(O[0, 0, 0], v[0, 0, 0], rtol=0, atol=1e-15)
    assert abs(L[0, 0, 0] - 0.7 * q[0, 0, 0] @ k[0, 0, 0]) <= 1e-13


def test_all_ones_mask_equals_dense_and_asymmetric_mask_equals_explicit():
    N, d, mb = 100, 8, 16
    T = (N + mb - 1) // mb
    q, k, v = (_rand((1, 1, N, d), s) for s in (20, 21, 22))
    O, L = oracle.attention_fwd(q, k, v, 0.35)
    Om, Lm = oracle.attention_fwd(q, k, v, 0.35, mask=np.ones((T, T), np.uint8), mask_block=mb)
    assert np.abs(O - Om).max() == 0 and np.abs(L - Lm).max() == 0
    # strictly lower block triangle plus the diagonal plus one upper block: not symmetric
    m = np.tril(np.ones((T, T), np.uint8))
    m[1, 4] = 1
    m[5, 2] = 0
    Om, Lm = oracle.attention_fwd(q, k, v, 0.35, mask=m, mask_block=mb)
    Ot, Lt = _torch_attention(q, k, v, 0.35, dense_mask=_expand_mask(m, N, mb))
    assert np.abs(Om - Ot).max() <= 1e-12 and np.abs(Lm - Lt).max() <= 1e-12


def test_block_diagonal_mask_is_independent_attentions():
    N, d, mb = 96, 8, 32
    q, k, v = (_rand((1, 1, N, d), s) for s in (23, 24, 25))
    m = np.eye(N // mb, dtype=np.uint8)
    O, L = oracle.attention_fwd(q, k, v, 0.4, mask=m, mask_block=mb, causal=True)
    for t in range(N // mb):
        sl = slice(t * mb, (t + 1) * mb)
        Ot, Lt = oracle.attention_fwd(q[:, :, sl], k[:, :, sl], v[:, :, sl], 0.4, causal=True)
        assert np.abs(O[:, :, sl] - Ot).max() <= 1e-14
        assert np.abs(L[:, :, sl] - Lt).max() <= 1e-14


def test_per_head_masks_follow_strides():
    B, H, N, d, mb = 2, 3, 64, 4, 16
    T = N // mb
    q, k, v = (_rand((B, H, N, d), s) for s in (26, 27, 28))
    rng = np.random.default_rng(29)
    m = (rng.random((B, H, T, T)) < 0.5).astype(np.uint8)
    for b in range(B):
        for h in range(H):
            np.fill_diagonal(m[b, h], 1)
    O, L = oracle.attention_fwd(q, k, v, 0.5, mask=m, mask_block=mb)
    for b in range(B):
        for h in range(H):
            Ot, Lt = _torch_attention(q[b, h], k[b, h], v[b, h], 0.5,
                                      dense_mask=_expand_mask(m[b, h], N, mb))
            assert np.abs(O[b, h] - Ot).max() <= 1e-12 and np.abs(L[b, h] - Lt).max() <= 1e-12


def test_fully_hidden_row_is_zero_with_minus_inf_lse():
    N, d, mb = 64, 4, 16
    q, k, v = (_rand((1, 1, N, d), s) for s in (30, 31, 32))
    m = np.ones((4, 4), np.uint8)
    m[2, :] = 0
    O, L = oracle.attention_fwd(q, k, v, 0.5, mask=m, mask_block=mb)
    assert np.all(O[0, 0, 32:48] == 0) and np.all(np.isneginf(L[0, 0, 32:48]))
    do = _rand((1, 1, N, d), 33)
    dQ, dK, dV = oracle.attention_bwd(q, k, v, do, 0.5, mask=m, mask_block=mb)
    assert np.all(dQ[0, 0, 32:48] == 0)
    m2 = m.copy()
    Ok, _ = oracle.attention_fwd(q, k, v, 0.5, mask=m2, mask_block=mb)
    # the hidden rows' dO must not reach any key: changing it changes nothing
    do2 = do.copy()
    do2[0, 0, 32:48] += 5.0
    _, dK2, dV2 = oracle.attention_bwd(q, k, v, do2, 0.5, mask=m, mask_block=mb)
    assert np.abs(dK - dK2).max() == 0 and np.abs(dV - dV2).max() == 0


def test_rows_entry_matches_whole_tensor():
    N, d = 77, 16
    q, k, v = (_rand((1, 1, N, d), s) for s in (34, 35, 36))
    O, L = oracle.attention_fwd(q, k, v, 0.25, causal=True)
    rows = [0, 5, 76, 40]
    Or, Lr = oracle.attention_fwd_rows(q[0, 0], k[0, 0], v[0, 0], rows, 0.25, causal=True)
    assert np.abs(Or - O[0, 0, rows]).max() == 0 and np.abs(Lr - L[0, 0, rows]).max() == 0


# ---------------------------------------------------------------- blockwise online recurrence


@pytest.mark.parametrize("norm_at_end", [False, True])
@pytest.mark.parametrize("Br,Bc", [(1, 1), (16, 16), (7, 13), (64, 300)])
@pytest.mark.parametrize("causal", [False, True])
def test_blockwise_online_equals_direct_fp64(norm_at_end, Br, Bc, causal):
    N, d = 101, 16
    q, k, v = (_rand((1, 2, N, d), s, 2.0) for s in (37, 38, 39))
    O, L = oracle.attention_fwd(q, k, v, 0.25, causal=causal)
    Ob, Lb = oracle.attention_fwd_blockwise(q, k, v, 0.25, Br, Bc, causal=causal,
                                            norm_at_end=norm_at_end)
    assert np.abs(O - Ob).max() <= 1e-12
    assert np.abs(L - Lb).max() <= 1e-12


def test_blockwise_with_block_mask_equals_direct():
    N, d, mb = 96, 8, 32
    q, k, v = (_rand((1, 1, N, d), s) for s in (40, 41, 42))
    m = np.array([[1, 0, 0], [1, 1, 0], [0, 1, 1]], np.uint8)
    O, L = oracle.attention_fwd(q, k, v, 0.3, mask=m, mask_block=mb)
    Ob, Lb = oracle.attention_fwd_blockwise(q, k, v, 0.3, 10, 24, mask=m, mask_block=mb)
    assert np.abs(O - Ob).max() <= 1e-13 and np.abs(L - Lb).max() <= 1e-13


def test_printed_fp32_online_softmax_example():
    """The Ultralytics page runs its blockwise loop in fp32 and prints the max difference."""
    with open(os.path.join(GOLDEN, "online_softmax_fp32_example.json")) as f:
        g = json.load(f)
    n, d, block = g["n"], g["d"], g["block"]
    torch.manual_seed(g["torch_seed"])
    q, k, v = torch.randn(3, n, d).unbind(0)
    standard = (torch.softmax(q @ k.T / d ** 0.5, dim=-1) @ v).numpy()
    Ob, _ = oracle.attention_fwd_blockwise(q[None, None].numpy(), k[None, None].numpy(),
                                           v[None, None].numpy(), 1.0 / math.sqrt(d), n, block,
                                           precision="f32", norm_at_end=True)
    diff = np.abs(Ob[0, 0] - standard).max()
    printed = g["printed_max_abs_diff_fp32"]
    assert printed / 4 <= diff <= printed * 2.5, diff
    assert (n, block) == tuple(g["printed_largest_score_tile"])
    # against the exact result the fp32 loop is still at fp32 rounding level
    O64, _ = oracle.attention_fwd(q[None, None].numpy(), k[None, None].numpy(),
                                  v[None, None].numpy(), 1.0 / math.sqrt(d))
    assert np.abs(Ob[0, 0] - O64[0, 0]).max() <= 1e-6


# ---------------------------------------------------------------- backward


def _loss(q, k, v, do, scale, causal, mask=None, mb=128):
    O, _ = oracle.attention_fwd(q, k, v, scale, causal=causal, mask=mask, mask_block=mb)
    return float(np.sum(O * do))


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_central_differences(causal):
    N, d = 7, 4
    q, k, v, do = (_rand((1, 1, N, d), s) for s in (43, 44, 45, 46))
    scale = 0.6
    dQ, dK, dV = oracle.attention_bwd(q, k, v, do, scale, causal=causal)
    h = 1e-5
    for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (_loss(args_p["q"], args_p["k"], args_p["v"], do, scale, causal)
                        - _loss(args_m["q"], args_m["k"], args_m["v"], do, scale, causal)) / (2 * h)
        err = np.linalg.norm(num - g) / np.linalg.norm(g)
        assert err <= 1e-6, (name, err)


def test_gradients_with_block_mask_match_central_differences():
    N, d, mb = 8, 3, 2
    q, k, v, do = (_rand((1, 1, N, d), s) for s in (47, 48, 49, 50))
    m = np.array([[1, 0, 1, 0], [1, 1, 0, 0], [0, 1, 1, 1], [1, 0, 0, 1]], np.uint8)
    dQ, dK, dV = oracle.attention_bwd(q, k, v, do, 0.9, mask=m, mask_block=mb)
    h = 1e-5
    for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            a = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
            b = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
            a[name][idx] += h
            b[name][idx] -= h
            num[idx] = (_loss(a["q"], a["k"], a["v"], do, 0.9, False, m, mb)
                        - _loss(b["q"], b["k"], b["v"], do, 0.9, False, m, mb)) / (2 * h)
        assert np.linalg.norm(num - g) / np.linalg.norm(g) <= 1e-6, name


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_torch_autograd(causal):
    B, H, N, d = 2, 2, 45, 16
    q, k, v, do = (_rand((B, H, N, d), s) for s in (51, 52, 53, 54))
    scale = 0.25
    dQ, dK, dV = oracle.attention_bwd(q, k, v, do, scale, causal=causal)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    s = scale * tq @ tk.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
    out = torch.softmax(s, -1) @ tv
    out.backward(torch.tensor(do))
    for mine, ref in ((dQ, tq.grad), (dK, tk.grad), (dV, tv.grad)):
        assert np.abs(mine - ref.numpy()).max() <= 1e-11


def test_gradient_identities():
    """sum_j dK_j = 0 (rows of dS sum to zero) and sum_j dV_j = sum_i dO_i."""
    N, d = 60, 8
    q, k, v, do = (_rand((1, 1, N, d), s) for s in (55, 56, 57, 58))
    for causal in (False, True):
        dQ, dK, dV = oracle.attention_bwd(q, k, v, do, 0.3, causal=causal)
        assert np.abs(dK.sum(2)).max() <= 1e-11
        np.testing.assert_allclose(dV.sum(2), do.sum(2), rtol=0, atol=1e-11)


def test_bwd_rows_entry_matches_whole_tensor():
    N, d, mb = 64, 8, 16
    q, k, v, do = (_rand((1, 1, N, d), s) for s in (59, 60, 61, 62))
    m = np.tril(np.ones((4, 4), np.uint8))
    m[0, 3] = 1
    dQ, dK, dV = oracle.attention_bwd(q, k, v, do, 0.3, causal=True, mask=m, mask_block=mb)
    qr, kr = [0, 13, 63], [1, 40, 63, 17]
    a, b, c = oracle.attention_bwd_rows(q[0, 0], k[0, 0], v[0, 0], do[0, 0], qr, kr, 0.3,
                                        causal=True, mask_h=m, mask_block=mb)
    assert np.abs(a - dQ[0, 0, qr]).max() <= 1e-14
    assert np.abs(b - dK[0, 0, kr]).max() <= 1e-14
    assert np.abs(c - dV[0, 0, kr]).max() <= 1e-14
