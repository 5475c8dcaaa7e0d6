"""Pins of the oracle's dropout (CPU, no GPU).

The pages fuse dropout into the attention kernel ("Fusão de Kernels" among the
"Ideias centrais" of the FlashAttention reading guide) and pass ``dropout_p`` to
the attention call ("L'intégration est de huit lignes", marketmaker.cc); they
name no generator.  The oracle draws the keep decisions from Philox4x32-10
(Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3",
SC 2011).  Pinned here by: the generator's published known-answer vectors; p = 0
reducing to plain attention; the keep fraction and the unbiasedness of the
scaled weights (statistics over many draws); and, for a fixed mask, the
gradients against central differences and against torch autograd of the same
masked product.
"""
import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# Known-answer vectors of Philox4x32-10 published with the generator (counter,
# key -> output), 32-bit words.
PHILOX_KAT = [
    ([0x00000000, 0x00000000, 0x00000000, 0x00000000], [0x00000000, 0x00000000],
     [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]),
    ([0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF], [0xFFFFFFFF, 0xFFFFFFFF],
     [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]),
    ([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0],
     [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]),
]


@pytest.mark.parametrize("ctr,key,expect", PHILOX_KAT)
def test_philox_known_answer_vectors(ctr, key, expect):
    assert list(oracle.philox4x32_10(ctr, key)) == expect


def test_keep_decisions_follow_the_documented_counter_layout():
    """Half j mod 2 of word (j mod 8) // 2 of the counter (j // 8, i, bh, offset) under
    key (seed lo, seed hi), against floor(p 2^16)."""
    B, H, N, p, seed, off = 2, 3, 37, 0.35, 0x123456789ABCDEF0, 77
    keep = oracle.dropout_keep(B, H, N, p, seed, off)
    t = int(np.floor(p * 2.0 ** 16))
    key = [seed & 0xFFFFFFFF, seed >> 32]
    rng = np.random.default_rng(0)
    for _ in range(200):
        b, h, i, j = (int(rng.integers(0, n)) for n in (B, H, N, N))
        w = int(oracle.philox4x32_10([j // 8, i, b * H + h, off], key)[(j % 8) // 2])
        half = (w >> 16) if j % 2 else (w & 0xFFFF)
        assert keep[b, h, i, j] == (1 if half >= t else 0)
    assert oracle.dropout_scale(p) == 65536.0 / (65536.0 - t)


def test_p0_is_plain_attention():
    q, k, v, do = (_rand((2, 2, 50, 8), s) for s in (1, 2, 3, 4))
    O0, L0 = oracle.attention_fwd(q, k, v, 0.3, causal=True)
    g0 = oracle.attention_bwd(q, k, v, do, 0.3, causal=True)
    for seed in (0, 5, 2 ** 40 + 3):
        O, L = oracle.attention_fwd(q, k, v, 0.3, causal=True, dropout_p=0.0, seed=seed, offset=9)
        g = oracle.attention_bwd(q, k, v, do, 0.3, causal=True, dropout_p=0.0, seed=seed)
        assert np.array_equal(O, O0) and np.array_equal(L, L0)
        for a, b in zip(g, g0):
            assert np.array_equal(a, b)
    assert oracle.dropout_keep(1, 1, 16, 0.0).all()


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_keep_fraction_is_one_minus_p(p):
    B, H, N = 2, 3, 256
    keep = oracle.dropout_keep(B, H, N, p, seed=11, offset=3)
    n = keep.size
    frac = keep.mean()
    q = 1.0 / oracle.dropout_scale(p)  # the keep probability, 1 - p to within 2^-16
    assert abs(q - (1 - p)) <= 2.0 ** -16
    sigma = np.sqrt(q * (1 - q) / n)
    assert abs(frac - q) <= 5 * sigma, (frac, q, sigma)


def test_masks_differ_across_seeds_offsets_and_heads_and_repeat_for_equal_ones():
    a = oracle.dropout_keep(1, 2, 64, 0.5, seed=1, offset=0)
    assert np.array_equal(a, oracle.dropout_keep(1, 2, 64, 0.5, seed=1, offset=0))
    assert not np.array_equal(a, oracle.dropout_keep(1, 2, 64, 0.5, seed=2, offset=0))
    assert not np.array_equal(a, oracle.dropout_keep(1, 2, 64, 0.5, seed=1, offset=1))
    assert not np.array_equal(a[0, 0], a[0, 1])


def test_scaled_weights_are_unbiased_over_draws():
    """E[O_drop] = O: the mean over many seeds lies within 5 standard errors."""
    N, d, p = 6, 3, 0.3
    q, k, v = (_rand((1, 1, N, d), s) for s in (5, 6, 7))
    O, _ = oracle.attention_fwd(q, k, v, 0.7)
    draws = np.stack([oracle.attention_fwd(q, k, v, 0.7, dropout_p=p, seed=s)[0]
                      for s in range(3000)])
    mean, se = draws.mean(0), draws.std(0, ddof=1) / np.sqrt(len(draws))
    assert np.all(np.abs(mean - O) <= 5 * se + 1e-12)
    # and a generator that kept with probability p instead of 1 - p would be biased
    assert np.abs(mean - O).max() < 0.1 * np.abs(O).max()


def _torch_dropout_attention(q, k, v, do, scale, causal, z):
    """(softmax(scale Q K^T) * Z) V and its gradients in torch fp64 (library route)."""
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    s = scale * tq @ tk.transpose(-1, -2)
    N = q.shape[-2]
    if causal:
        s = s.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
    out = (torch.softmax(s, -1) * torch.tensor(z)) @ tv
    out.backward(torch.tensor(do))
    return out.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
def test_forward_and_gradients_match_torch_with_the_same_mask(causal):
    B, H, N, d, p, seed, off = 2, 2, 45, 16, 0.25, 99, 4
    q, k, v, do = (_rand((B, H, N, d), s) for s in (11, 12, 13, 14))
    z = oracle.dropout_keep(B, H, N, p, seed, off).astype(np.float64) * oracle.dropout_scale(p)
    O_t, dq_t, dk_t, dv_t = _torch_dropout_attention(q, k, v, do, 0.25, causal, z)
    O, L = oracle.attention_fwd(q, k, v, 0.25, causal=causal, dropout_p=p, seed=seed, offset=off)
    O_plain, L_plain = oracle.attention_fwd(q, k, v, 0.25, causal=causal)
    assert np.abs(O - O_t).max() <= 1e-12
    assert np.array_equal(L, L_plain)  # the statistics are those of the undropped softmax
    dQ, dK, dV = oracle.attention_bwd(q, k, v, do, 0.25, causal=causal, dropout_p=p, seed=seed,
                                      offset=off)
    for mine, ref in ((dQ, dq_t), (dK, dk_t), (dV, dv_t)):
        assert np.abs(mine - ref).max() <= 1e-11


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_gradients_match_central_differences(causal):
    N, d, p, seed = 7, 4, 0.3, 123
    q, k, v, do = (_rand((1, 1, N, d), s) for s in (21, 22, 23, 24))
    dQ, dK, dV = oracle.attention_bwd(q, k, v, do, 0.6, causal=causal, dropout_p=p, seed=seed)

    def loss(a):
        O, _ = oracle.attention_fwd(a["q"], a["k"], a["v"], 0.6, causal=causal, dropout_p=p,
                                    seed=seed)
        return float(np.sum(O * do))

    h = 1e-5
    for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            a = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
            b = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
            a[name][idx] += h
            b[name][idx] -= h
            num[idx] = (loss(a) - loss(b)) / (2 * h)
        assert np.linalg.norm(num - g) / np.linalg.norm(g) <= 1e-6, name


def test_dropout_rows_entries_match_whole_tensor():
    B, H, N, d, p, seed, off = 1, 3, 64, 8, 0.2, 7, 2
    q, k, v, do = (_rand((B, H, N, d), s) for s in (31, 32, 33, 34))
    O, L = oracle.attention_fwd(q, k, v, 0.3, causal=True, dropout_p=p, seed=seed, offset=off)
    dQ, dK, dV = oracle.attention_bwd(q, k, v, do, 0.3, causal=True, dropout_p=p, seed=seed,
                                      offset=off)
    h = 2
    rows = [0, 5, 63]
    o, l = oracle.attention_fwd_rows(q[0, h], k[0, h], v[0, h], rows, 0.3, causal=True,
                                     dropout_p=p, seed=seed, offset=off, bh=h)
    assert np.abs(o - O[0, h, rows]).max() <= 1e-14 and np.abs(l - L[0, h, rows]).max() <= 1e-14
    a, b, c = oracle.attention_bwd_rows(q[0, h], k[0, h], v[0, h], do[0, h], rows, [1, 40], 0.3,
                                        causal=True, dropout_p=p, seed=seed, offset=off, bh=h)
    assert np.abs(a - dQ[0, h, rows]).max() <= 1e-14
    assert np.abs(b - dK[0, h, [1, 40]]).max() <= 1e-14
    assert np.abs(c - dV[0, h, [1, 40]]).max() <= 1e-14
