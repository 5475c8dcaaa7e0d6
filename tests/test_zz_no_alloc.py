"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Some callers run the backward pass where they may not allocate: a plugin that its
host application gives a fixed memory budget, an engine that plans every buffer
ahead of time, or code that must not enter the CUDA allocator while other work
holds it.  fa_bwd_noalloc serves them from a fixed scratch array inside the
library.  This file checks it through the C ABI against fa_bwd (the entry point
that takes a caller workspace) and against the fp64 oracle, on calls in a row with
different inputs, so that anything one call leaves in the shared array would show up
in the next: causal and not, a problem whose scratch reaches near the array's end, and
a block-masked problem.  It sorts last so that a run stopping at its first failure has already
run every other test.
"""
import ctypes

import pytest
import torch

import synth
from _parity import TOL, rel_fro, to_np64

import exact_io_aware_26_gb300 as fa

pytestmark = pytest.mark.gpu


def _noalloc(lib):
    f = lib.fa_bwd_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(fa.FaParams)] + [ctypes.c_void_p] * 10
    return f


def _call(noalloc, lib, inp, causal, mask=None, mask_block=128):
    """fa_bwd_noalloc and fa_bwd on the same problem; returns both gradient triples."""
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    m = None if mask is None else torch.as_tensor(mask, dtype=torch.uint8).cuda()
    o, lse = fa.attention_fwd(q, k, v, causal=causal, block_mask=m, mask_block=mask_block)
    ref = fa.attention_bwd(q, k, v, o, do, lse, causal=causal, block_mask=m,
                           mask_block=mask_block)
    p, _ = fa.make_params(q, None, causal, m, mask_block)
    assert lib.fa_bwd_workspace_size(ctypes.byref(p)) <= (64 << 20)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    st = noalloc(ctypes.byref(p), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                 do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                 torch.cuda.current_stream().cuda_stream)
    assert st == fa.FA_OK, lib.fa_last_error()
    assert fa.get_status() == fa.FA_OK
    return (dq, dk, dv), ref


def _check(got, ref, oracle_ref, tag):
    for i, name in enumerate(("dQ", "dK", "dV")):
        assert torch.isfinite(got[i]).all(), (tag, name)
        e = rel_fro(to_np64(got[i]), to_np64(ref[i]))
        assert e <= TOL["bf16"]["grad"], (tag, name, "vs fa_bwd", e)
        if oracle_ref is not None:
            e = rel_fro(to_np64(got[i]), oracle_ref[i])
            assert e <= TOL["bf16"]["grad"], (tag, name, "vs oracle", e)


def _oracle(inp, causal, mask=None, mask_block=128):
    import math
    import oracle
    o = {n: to_np64(inp[n]) for n in ("q", "k", "v", "do")}
    return oracle.attention_bwd(o["q"], o["k"], o["v"], o["do"], 1.0 / math.sqrt(o["q"].shape[-1]),
                                causal=causal, mask=mask, mask_block=mask_block)


def test_bwd_noalloc_matches_bwd_on_two_calls_in_a_row(cuda_lib):
    """Two calls with different inputs (causal, then not): each against fa_bwd and the
    fp64 oracle."""
    lib = fa.load()
    noalloc = _noalloc(lib)
    for call, seed in enumerate((101, 202)):
        inp = synth.make_inputs(2, 3, 700, 64, "bf16", seed=seed)
        causal = call == 0
        got, ref = _call(noalloc, lib, inp, causal)
        _check(got, ref, _oracle(inp, causal), call)


def test_bwd_noalloc_near_the_array_end_and_with_a_block_mask(cuda_lib):
    """A problem whose workspace (B=4, H=12, N=3600, d=64: about 53 MiB) reaches near the
    array's end, then a block-masked one (which takes no partial-sum slots) right after."""
    lib = fa.load()
    noalloc = _noalloc(lib)
    inp = synth.make_inputs(4, 12, 3600, 64, "bf16", seed=404)
    p, _ = fa.make_params(inp["q"], None, False)
    assert (48 << 20) < lib.fa_bwd_workspace_size(ctypes.byref(p)) <= (64 << 20)
    got, ref = _call(noalloc, lib, inp, False)
    _check(got, ref, None, "large")
    inp = synth.make_inputs(1, 2, 900, 64, "bf16", seed=303, mask_p=0.4)
    got, ref = _call(noalloc, lib, inp, True, inp["mask"])
    _check(got, ref, _oracle(inp, True, inp["mask"]), "mask")


def test_bwd_noalloc_rejects_problems_larger_than_its_array(cuda_lib):
    lib = fa.load()
    noalloc = _noalloc(lib)
    # B*H*N*(d+1)*4 bytes > 64 MiB: rejected on the host, nothing is launched
    p = fa.FaParams(1, 12, 23400, 64, fa.FA_BF16, 0.125, 1, None, 128, 0, 0)
    assert lib.fa_bwd_workspace_size(ctypes.byref(p)) > (64 << 20)
    st = noalloc(ctypes.byref(p), *([1 << 20] * 9), None)
    assert st == fa.FA_ERR_WORKSPACE
    assert b"scratch" in lib.fa_last_error()
