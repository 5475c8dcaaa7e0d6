"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Some callers run the backward pass where they may not allocate: a plugin that its
host application gives a fixed memory budget, an engine that plans every buffer
ahead of time, or code that must not enter the CUDA allocator while other work
holds it.  fa_bwd_noalloc serves them from a fixed scratch array inside the
library.  This file checks it through the C ABI against fa_bwd (the entry point
that takes a caller workspace) on two calls in a row with different inputs, so
that anything the first call leaves in the shared array would show up in the
second.  It sorts last so that a run stopping at its first failure has already
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


def test_bwd_noalloc_matches_bwd_on_two_calls_in_a_row(cuda_lib):
    lib = fa.load()
    noalloc = _noalloc(lib)
    stream = torch.cuda.current_stream().cuda_stream
    for call, seed in enumerate((101, 202)):
        inp = synth.make_inputs(2, 3, 700, 64, "bf16", seed=seed)
        q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
        causal = call == 0
        o, lse = fa.attention_fwd(q, k, v, causal=causal)
        ref = fa.attention_bwd(q, k, v, o, do, lse, causal=causal)
        p, _ = fa.make_params(q, None, causal)
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        st = noalloc(ctypes.byref(p), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                     do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                     stream)
        assert st == fa.FA_OK, lib.fa_last_error()
        assert fa.get_status() == fa.FA_OK
        for name, got, want in (("dQ", dq, ref[0]), ("dK", dk, ref[1]), ("dV", dv, ref[2])):
            assert torch.isfinite(got).all(), (call, name)
            e = rel_fro(to_np64(got), to_np64(want))
            assert e <= TOL["bf16"]["grad"], (call, name, e)


def test_bwd_noalloc_rejects_problems_larger_than_its_array(cuda_lib):
    lib = fa.load()
    noalloc = _noalloc(lib)
    # B*H*N*(d+1)*4 bytes > 64 MiB: rejected on the host, nothing is launched
    p = fa.FaParams(1, 12, 23400, 64, fa.FA_BF16, 0.125, 1, None, 128, 0, 0)
    assert lib.fa_bwd_workspace_size(ctypes.byref(p)) > (64 << 20)
    st = noalloc(ctypes.byref(p), *([1 << 20] * 9), None)
    assert st == fa.FA_ERR_WORKSPACE
    assert b"scratch" in lib.fa_last_error()
