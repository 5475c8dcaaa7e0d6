"""The largest problem fa_check accepts: B*H*N*d just under 2^31 elements
(16383 heads of N = 2048, d = 64, bf16; 4.3 GB per tensor, about 45 GB in all),
forward and backward, both causal settings (the causal one with dropout, whose
counter carries the head index).  Rows of the first, a middle and the last head
are checked against the fp64 oracle, so an index that overflowed 32 bits
anywhere on the path would show up."""
import math

import numpy as np
import pytest
import torch

import oracle
from _parity import check_fwd, check_grads, to_np64

import exact_io_aware_26_gb300 as fa

pytestmark = pytest.mark.gpu

B, H, N, D = 1, 16383, 2048, 64


def test_largest_accepted_problem(cuda_lib):
    assert B * H * N * D < 2 ** 31
    free, _ = torch.cuda.mem_get_info()
    if free < 60 * 2 ** 30:
        pytest.skip(f"needs about 45 GB of free device memory, {free / 2 ** 30:.0f} GB free")
    p, _ = fa.make_params(torch.empty((B, H, N, D), dtype=torch.bfloat16, device="meta"))
    assert fa.check_params(p) == fa.FA_OK
    g = torch.Generator(device="cuda")
    g.manual_seed(31)
    shape = (B, H, N, D)
    q, k, v, do = (torch.randn(shape, generator=g, device="cuda", dtype=torch.float32)
                   .to(torch.bfloat16) for _ in range(4))
    scale = 1.0 / math.sqrt(D)
    heads = (0, H // 2, H - 1)
    rng = np.random.default_rng(3)
    for causal, drop in ((False, 0.0), (True, 0.15)):
        O, L = fa.attention_fwd(q, k, v, causal=causal, dropout_p=drop, seed=99, offset=1)
        dq, dk, dv = fa.attention_bwd(q, k, v, O, do, L, causal=causal, dropout_p=drop, seed=99,
                                      offset=1)
        assert fa.get_status() == fa.FA_OK
        for h in heads:
            rows = np.unique(np.concatenate([[0, 127, 128, N - 1], rng.integers(0, N, 28)]))
            rows = rows.astype(np.int32)
            x = {n: to_np64(t[0, h]) for n, t in (("q", q), ("k", k), ("v", v), ("do", do))}
            O_ref, L_ref = oracle.attention_fwd_rows(x["q"], x["k"], x["v"], rows, scale,
                                                     causal=causal, dropout_p=drop, seed=99,
                                                     offset=1, bh=h)
            check_fwd(O[0, h, rows], L[0, h, rows], O_ref, L_ref, "bf16")
            ref = oracle.attention_bwd_rows(x["q"], x["k"], x["v"], x["do"], rows, rows, scale,
                                            causal=causal, dropout_p=drop, seed=99, offset=1, bh=h)
            check_grads((dq[0, h, rows], dk[0, h, rows], dv[0, h, rows]), ref, "bf16")
        del O, L, dq, dk, dv
        torch.cuda.empty_cache()
