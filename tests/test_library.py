"""Host-only checks of libfa.so: it builds, loads without a GPU, exports every
function include/fa.h declares, and rejects bad arguments before any CUDA call."""
import ctypes
import os

import pytest

import exact_io_aware_26_gb300 as fa


@pytest.fixture(scope="module")
def lib():
    fa.build()
    return fa.load()


def test_every_declared_function_is_exported(lib):
    names = fa.header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert lib.fa_version() >= 100
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.fa_status_string(code)


def _p(**kw):
    base = dict(B=1, H=1, N=128, d=64, dtype=fa.FA_BF16, scale=0.125, causal=0,
                block_mask=None, mask_block=128, mask_stride_b=0, mask_stride_h=0)
    base.update(kw)
    return fa.FaParams(**base)


@pytest.mark.parametrize("kw,expect", [
    ({}, fa.FA_OK),
    ({"dtype": fa.FA_F32}, fa.FA_OK),
    ({"N": 1}, fa.FA_OK),
    ({"N": 23400, "H": 12}, fa.FA_OK),
    ({"d": 128}, fa.FA_OK),
    ({"B": 0}, fa.FA_ERR_INVALID),
    ({"N": 0}, fa.FA_ERR_INVALID),
    ({"d": 32}, fa.FA_ERR_UNSUPPORTED),
    ({"d": 96}, fa.FA_ERR_UNSUPPORTED),
    ({"dtype": 7}, fa.FA_ERR_INVALID),
    ({"scale": 0.0}, fa.FA_ERR_INVALID),
    ({"scale": -1.0}, fa.FA_ERR_INVALID),
    ({"scale": float("inf")}, fa.FA_ERR_INVALID),
    ({"scale": float("nan")}, fa.FA_ERR_INVALID),
    ({"B": 64, "H": 64, "N": 65536}, fa.FA_ERR_UNSUPPORTED),
    ({"block_mask": 4096, "mask_block": 64}, fa.FA_ERR_UNSUPPORTED),
    ({"block_mask": 4096, "mask_block": 0}, fa.FA_ERR_INVALID),
    ({"block_mask": 4096, "mask_block": 256}, fa.FA_OK),
    ({"block_mask": 4096, "mask_stride_h": -1}, fa.FA_ERR_INVALID),
    ({"dropout_p": 0.1, "dropout_seed": 2 ** 63 + 5, "dropout_offset": 7}, fa.FA_OK),
    ({"dropout_p": 0.999}, fa.FA_OK),
    ({"dropout_p": 1.0}, fa.FA_ERR_INVALID),
    ({"dropout_p": -0.1}, fa.FA_ERR_INVALID),
    ({"dropout_p": float("nan")}, fa.FA_ERR_INVALID),
])
def test_check_params(lib, kw, expect):
    assert fa.check_params(_p(**kw)) == expect


def test_backward_limits(lib):
    assert fa.check_params(_p(dtype=fa.FA_F32), for_backward=True) == fa.FA_ERR_UNSUPPORTED
    assert fa.check_params(_p(dtype=fa.FA_F16), for_backward=True) == fa.FA_OK
    assert lib.fa_check(None, 0) == fa.FA_ERR_INVALID


def test_workspace_size(lib):
    up = lambda x: (x + 255) // 256 * 256
    # D, the dQ accumulator and, without a block mask, one [dV | dK] fp32 slot
    # of 128 x d per slice CTA (at most 160, at most one per visited tile pair)
    slots = lambda ctas, d: up(ctas * 2 * 128 * d * 4)
    p = _p(B=4, H=12, N=2048, d=64)
    rows = 4 * 12 * 2048
    assert lib.fa_bwd_workspace_size(ctypes.byref(p)) == up(rows * 4) + up(rows * 64 * 4) + slots(160, 64)
    p = _p(N=23400, H=12, d=64, causal=1)
    rows = 12 * 23400
    assert lib.fa_bwd_workspace_size(ctypes.byref(p)) == up(rows * 4) + up(rows * 64 * 4) + slots(160, 64)
    p = _p(N=300, H=1, d=128, causal=1)  # 3 tiles: 6 causal tile pairs, so 6 slices at most
    assert lib.fa_bwd_workspace_size(ctypes.byref(p)) == up(300 * 4) + up(300 * 128 * 4) + slots(6, 128)
    p = _p(B=2, H=3, N=700, d=64, block_mask=4096)  # one CTA per key tile: no slots
    rows = 2 * 3 * 700
    assert lib.fa_bwd_workspace_size(ctypes.byref(p)) == up(rows * 4) + up(rows * 64 * 4)
    assert lib.fa_bwd_workspace_size(ctypes.byref(_p(d=32))) == 0


def test_bwd_cta_cap_setter(lib):
    old = fa.set_bwd_ctas(7)
    assert fa.set_bwd_ctas(-3) == 7   # negative clamps to 0 (one CTA per SM per wave)
    assert fa.set_bwd_ctas(old) == 0


def test_invalid_calls_return_before_any_launch(lib):
    """Null or misaligned pointers and a short workspace fail on the host."""
    p = _p()
    ok_ptr = 1 << 20  # never dereferenced: every call below fails validation first
    assert lib.fa_fwd(ctypes.byref(p), None, ok_ptr, ok_ptr, ok_ptr, ok_ptr, None) == fa.FA_ERR_INVALID
    assert lib.fa_fwd(ctypes.byref(p), ok_ptr + 2, ok_ptr, ok_ptr, ok_ptr, ok_ptr, None) == fa.FA_ERR_INVALID
    assert lib.fa_fwd(ctypes.byref(p), ok_ptr, ok_ptr, ok_ptr, ok_ptr, None, None) == fa.FA_ERR_INVALID
    assert lib.fa_fwd(ctypes.byref(_p(d=32)), ok_ptr, ok_ptr, ok_ptr, ok_ptr, ok_ptr, None) == fa.FA_ERR_UNSUPPORTED
    need = lib.fa_bwd_workspace_size(ctypes.byref(p))
    args = [ok_ptr] * 9
    assert lib.fa_bwd(ctypes.byref(p), *args, ok_ptr, need - 1, None) == fa.FA_ERR_WORKSPACE
    assert lib.fa_bwd(ctypes.byref(p), *args, None, need, None) == fa.FA_ERR_WORKSPACE
    assert lib.fa_bwd(ctypes.byref(p), *args, ok_ptr + 16, need, None) == fa.FA_ERR_WORKSPACE
    assert lib.fa_bwd(ctypes.byref(_p(dtype=fa.FA_F32)), *args, ok_ptr, need, None) == fa.FA_ERR_UNSUPPORTED
    assert b"workspace" in lib.fa_last_error() or b"fp16" in lib.fa_last_error()


def test_library_links_no_cuda_driver_at_load_time():
    """libfa.so must load on a machine without the driver: no libcuda dependency."""
    import subprocess
    out = subprocess.run(["ldd", fa.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out


def test_split_count_model(lib):
    """fa_fwd_num_splits with an explicit SM count is host arithmetic: few query
    tiles get split, a full grid does not, and the count always divides the key
    tiles into non-empty slices."""
    one_head = _p(B=1, H=1, N=8192, d=64, dtype=fa.FA_F16)
    s = fa.num_splits(one_head, 152)
    assert s > 1
    per = -(-64 // s)
    assert -(-64 // per) == s
    assert fa.num_splits(_p(B=4, H=12, N=2048), 152) == 1
    assert fa.num_splits(_p(N=23400, H=12), 152) == 1
    assert fa.num_splits(_p(N=128), 152) == 1          # one key tile: nothing to split
    assert fa.num_splits(_p(N=8192, dtype=fa.FA_F32), 152) == 1
    assert fa.num_splits(_p(d=32), 152) == 0
    for n in (256, 1000, 4096, 65536):
        s = fa.num_splits(_p(N=n), 152)
        t = -(-n // 128)
        assert 1 <= s <= min(t, 64)
        per = -(-t // s)
        assert -(-t // per) == s


def test_split_invalid_calls_return_before_any_launch(lib):
    ok_ptr = 1 << 20  # never dereferenced: every call below fails validation first
    args = [ok_ptr] * 5
    call = lambda q, s: lib.fa_fwd_split(ctypes.byref(q), *args, s, None)
    assert call(_p(N=1024), 0) == fa.FA_ERR_INVALID
    assert call(_p(N=1024), 9) == fa.FA_ERR_INVALID       # 8 key tiles
    assert call(_p(N=2048), 9) == fa.FA_ERR_INVALID       # above FA_MAX_SPLITS = 8
    assert call(_p(N=300), 4) == fa.FA_ERR_INVALID        # more slices than key tiles
    assert call(_p(N=1024, dtype=fa.FA_F32), 4) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd_split(ctypes.byref(_p(N=1024)), ok_ptr + 2, ok_ptr, ok_ptr, ok_ptr, ok_ptr, 4,
                            None) == fa.FA_ERR_INVALID


def test_fp8_calls_validate_before_any_launch(lib):
    """The FP8 calls reject unsupported settings and bad pointers on the host."""
    ok = 1 << 20  # never dereferenced
    assert [lib.fa_fp8_vt_cols(n) for n in (0, 1, 16, 17, 2048, 23400)] == [0, 16, 16, 32, 2048, 23408]
    q_args = [ok] * 3 + [None] + [ok] * 6 + [None]  # Q K V signs q8 k8 vt8 sq sk sv stream
    f_args = [ok] * 8 + [None]                       # q8 k8 vt8 sq sk sv O LSE stream
    for bad, code in (({"dtype": fa.FA_F32}, fa.FA_ERR_UNSUPPORTED), ({"d": 96}, fa.FA_ERR_UNSUPPORTED),
                      ({"dropout_p": 0.1}, fa.FA_ERR_UNSUPPORTED), ({"N": 0}, fa.FA_ERR_INVALID)):
        p = _p(**bad)
        assert lib.fa_fp8_quantize(ctypes.byref(p), *q_args) == code
        assert lib.fa_fwd_fp8(ctypes.byref(p), *f_args) == code
    p = _p()
    for i in range(3):  # q8, k8, vt8 null or misaligned
        for v in (None, ok + 8):
            a = list(f_args)
            a[i] = v
            assert lib.fa_fwd_fp8(ctypes.byref(p), *a) == fa.FA_ERR_INVALID
    a = list(f_args)
    a[3] = ok + 2  # a scale array off its 4-byte alignment
    assert lib.fa_fwd_fp8(ctypes.byref(p), *a) == fa.FA_ERR_INVALID
    a = list(q_args)
    a[0] = None
    assert lib.fa_fp8_quantize(ctypes.byref(p), *a) == fa.FA_ERR_INVALID


def test_fp8_binding_rejects_bad_tensors_before_the_library():
    """The FP8 binding's checks run on the host: CPU tensors, wrong shapes or dtypes and
    a malformed code dict raise before any library call."""
    import torch
    q = torch.zeros(1, 1, 130, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fp8_quantize(q, q, q)  # not cuda
    T = 2
    good = {"q8": torch.zeros(1, 1, 130, 64, dtype=torch.uint8),
            "k8": torch.zeros(1, 1, 130, 64, dtype=torch.uint8),
            "vt8": torch.zeros(1, 1, 64, 144, dtype=torch.uint8),
            "sq": torch.ones(1, 1, T), "sk": torch.ones(1, 1, T), "sv": torch.ones(1, 1, T)}
    with pytest.raises(ValueError):
        fa.attention_fwd_fp8_codes(good, 0.125)  # not cuda
    assert fa.fp8_vt_cols(130) == 144
