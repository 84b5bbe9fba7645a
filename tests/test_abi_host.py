"""Host-side checks of the C ABI: the library loads, exports what the header declares, and
rejects bad arguments before launching anything (these run without a GPU)."""

import ctypes
import os
import re

import pytest

import scaled_dot_product_vt_gb300 as vt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vt_attn.h")


@pytest.fixture(scope="module")
def lib():
    vt.build()
    return vt.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vt_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(vt.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_debug_library_exports_every_declared_symbol(lib):
    dbg = vt.load_debug()
    for name in declared_functions():
        assert hasattr(dbg, name), name
    # host-side checks are shared: the same argument error before any launch
    assert dbg.vt_attn_fwd(1 << 20, 2 << 20, 3 << 20, 4 << 20, 1, 1, 4, 0, 8, 8, 0.5, 0, vt.VT_BF16, None) == 1


def test_status_strings(lib):
    for code, name in vt.STATUS.items():
        assert vt.vt_status_str(code).startswith(name)
    assert vt.vt_status_str(99) == "unknown vt_status"


A = 1 << 20  # fake, 16-byte aligned, distinct "device" addresses: never dereferenced on these paths


def call(B=1, H=1, S_q=4, S_k=4, D_qk=8, D_v=8, scale=0.5, causal=0, dtype=vt.VT_BF16,
         ptrs=(A, 2 * A, 3 * A, 4 * A)):
    return vt.vt_attn_fwd(*ptrs, B, H, S_q, S_k, D_qk, D_v, scale, causal, dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(S_k=0), 1), (dict(D_qk=0), 1), (dict(D_v=0), 1),
    (dict(B=-1), 1), (dict(H=-2), 1), (dict(S_q=-1), 1), (dict(S_k=-5), 1),
    (dict(dtype=7), 1), (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(D_qk=129), 2), (dict(D_v=256), 2), (dict(S_q=1 << 31), 2),
    (dict(S_q=(1 << 30) + 1), 2), (dict(S_k=(1 << 30) + 1), 2), (dict(B=1 << 31), 2), (dict(H=1 << 31), 2),
    (dict(ptrs=(A, 2 * A, 3 * A, 0)), 1), (dict(ptrs=(0, 2 * A, 3 * A, 4 * A)), 1),
    (dict(ptrs=(A + 8, 2 * A, 3 * A, 4 * A)), 3), (dict(ptrs=(A, 2 * A, 3 * A, 4 * A + 2)), 3),
    (dict(D_qk=4, dtype=vt.VT_BF16), 3),        # row pitch 8 bytes: not a TMA stride
    (dict(D_v=20, dtype=vt.VT_BF16), 3),        # 40-byte rows
    (dict(ptrs=(A, 2 * A, 3 * A, A + 32)), 1),  # O overlaps Q
])
def test_argument_errors(lib, kw, code):
    assert call(**kw) == code


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0), dict(S_q=0), dict(B=0, ptrs=(0, 0, 0, 0))])
def test_empty_problems_are_ok_without_launch(lib, kw):
    assert call(**kw) == 0


def test_strided_errors(lib):
    good = (32, 32, 8)
    assert vt.vt_attn_fwd_strided(A, good, 2 * A, good, 3 * A, good, 4 * A, (32, 32, 0),
                                  1, 1, 4, 4, 8, 8, 0.5, 0, vt.VT_BF16, None) == 1
    assert vt.vt_attn_fwd_strided(A, good, 2 * A, good, 3 * A, (32, 32, 12), 4 * A, good,
                                  1, 1, 4, 4, 8, 8, 0.5, 0, vt.VT_BF16, None) == 3
    # strided O whose rows interleave with V's span
    assert vt.vt_attn_fwd_strided(A, good, 2 * A, good, 3 * A, good, 3 * A + 16, (64, 64, 16),
                                  1, 1, 4, 4, 8, 8, 0.5, 0, vt.VT_BF16, None) == 1


def test_valid_call_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    assert call() == 4
    assert vt.vt_last_device_status(0) == 4


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="no fallback"):
        vt.load(str(tmp_path / "libvt_attn.so"))


# ---------------------------------------------------------------- split-KV entry points

def test_huge_strides_and_spans_are_rejected_before_launch(lib):
    # a stride of 2^40 bytes or more is beyond a TMA tensor map
    big = (1 << 40) // 2
    st = (big, 64, 8)
    assert vt.vt_attn_fwd_strided(A, st, 2 * A, (64, 64, 8), 3 * A, (64, 64, 8), 4 * A, (64, 64, 8),
                                  2, 1, 4, 4, 8, 8, 0.5, 0, vt.VT_BF16, None) == 2
    # strides just below that limit whose byte span overflows 64 bits: no such tensor fits in memory
    st = (big - 8, 64, 8)
    assert vt.vt_attn_fwd_strided(A, st, 2 * A, (64, 64, 8), 3 * A, (64, 64, 8), 4 * A, (64, 64, 8),
                                  1 << 30, 1, 4, 4, 8, 8, 0.5, 0, vt.VT_BF16, None) == 1
    # a workspace size that cannot exist is reported as 0
    assert vt.vt_attn_splitkv_workspace_size(1 << 31, 1 << 31, 1 << 30, 128, 64) == 0


def test_splitkv_workspace_size(lib):
    assert vt.vt_attn_splitkv_workspace_size(2, 3, 5, 8, 1) == 0
    assert vt.vt_attn_splitkv_workspace_size(2, 3, 5, 8, 0) == 0
    assert vt.vt_attn_splitkv_workspace_size(0, 3, 5, 8, 4) == 0
    up = lambda x: (x + 255) // 256 * 256
    rows = 2 * 3 * 5
    expect = up(4 * rows * 8 * 4) + 3 * up(4 * rows * 4)  # O, then m, l and the row-sum correction
    assert vt.vt_attn_splitkv_workspace_size(2, 3, 5, 8, 4) == expect


def split_call(n_split=2, dtype=vt.VT_BF16, ws=8 * A, ws_bytes=1 << 24, D_v=8):
    st = (32, 32, 8)
    so = (32, 32, D_v)
    return vt.vt_attn_fwd_splitkv(A, st, 2 * A, st, 3 * A, (32, 32, D_v), 4 * A, so, 1, 1, 4, 4, 8, D_v,
                                  0.5, 0, dtype, n_split, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(n_split=0), 1), (dict(n_split=-3), 1), (dict(n_split=65), 2),
    (dict(ws=None), 1), (dict(ws_bytes=64), 1),       # missing or too small workspace
    (dict(dtype=vt.VT_F32, ws_bytes=64), 1),          # fp32 partials need more workspace too
    (dict(ws=8 * A + 16), 3),                         # workspace not 256-byte aligned
    (dict(ws=A), 1),                                  # workspace overlaps Q
])
def test_splitkv_argument_errors(lib, kw, code):
    assert split_call(**kw) == code


def test_splitkv_choose_without_gpu(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    # no device to query: falls back to no split
    assert vt.vt_attn_splitkv_choose(1, 8, 256, 32768, 0, vt.VT_BF16) == 1
    assert vt.vt_attn_splitkv_choose(1, 8, 256, 32768, 0, vt.VT_F32) == 1


# ---------------------------------------------------------------- the general entry point

def general_call(H=4, H_kv=2, kind=0, offset=0, window=0, reserved=0, lse=None, n_split=1, ws=None, ws_bytes=0,
                 dtype=vt.VT_BF16, mask=True):
    st = (H * 32, 32, 8)
    skv = (H_kv * 32, 32, 8) if H_kv > 0 else st
    m = vt.vt_attn_mask(kind, reserved, offset, window) if mask else None
    return vt.vt_attn_fwd_general(A, st, 2 * A, skv, 3 * A, skv, 4 * A, st, lse, 1, H, H_kv, 4, 4, 8, 8, 0.5, dtype,
                                  m, n_split, ws, ws_bytes, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(H_kv=0), 1), (dict(H_kv=-1), 1), (dict(H_kv=3), 1),       # H must be a multiple of H_kv
    (dict(kind=4), 1), (dict(kind=-1), 1), (dict(reserved=1), 1),
    (dict(kind=1, offset=-1), 1),
    (dict(kind=2, window=0), 1), (dict(kind=3, window=-4), 1),
    (dict(kind=1, offset=(1 << 40) + 1), 2), (dict(kind=2, window=(1 << 40) + 1), 2),
    (dict(lse=8 * A + 2), 1),                                       # lse not 4-byte aligned
    (dict(lse=A + 16), 1),                                          # lse overlaps Q
    (dict(n_split=0), 1), (dict(n_split=65), 2),
    (dict(n_split=2), 1),                                           # no workspace
    (dict(n_split=2, ws=8 * A, ws_bytes=1 << 24, lse=8 * A + 64), 1),  # lse inside the workspace
])
def test_general_argument_errors(lib, kw, code):
    assert general_call(**kw) == code


def test_general_empty_problem_and_null_mask(lib):
    st = (32, 32, 8)
    assert vt.vt_attn_fwd_general(A, st, 2 * A, st, 3 * A, st, 4 * A, st, None, 1, 0, 1, 4, 4, 8, 8, 0.5,
                                  vt.VT_BF16, None, 1, None, 0, None, None) == 0
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    # a valid call with mask NULL reaches the launch, which reports the missing GPU
    assert general_call(mask=False) == 4
    assert general_call(kind=3, offset=2, window=5, lse=16 * A) == 4
    # fp32 I/O with split-KV passes every argument check and reaches the launch
    assert general_call(n_split=2, ws=8 * A, ws_bytes=1 << 24, dtype=vt.VT_F32) == 4
    assert split_call(dtype=vt.VT_F32) == 4
    assert vt.vt_last_device_status(0) == 4


# ---------------------------------------------------------------- extents whose packed size overflows

def test_packed_strides_that_overflow_are_rejected(lib):
    # every extent is within the limits, but H * S * D of the packed layout does not fit in 64 bits
    H, S = (1 << 31) - 1, 1 << 30
    assert vt.vt_attn_fwd(A, 2 * A, 3 * A, 4 * A, 1, H, S, S, 128, 128, 0.5, 0, vt.VT_BF16, None) == 1
    assert vt.vt_attn_fwd(A, 2 * A, 3 * A, 4 * A, 1, H, S, S, 128, 128, 0.5, 1, vt.VT_F32, None) == 1
    # shape errors keep their own codes and precedence
    assert vt.vt_attn_fwd(A, 2 * A, 3 * A, 4 * A, 1, H, S, S, 129, 128, 0.5, 0, vt.VT_BF16, None) == 2
    assert vt.vt_attn_fwd(A, 2 * A, 3 * A, 4 * A, -1, H, S, S, 128, 128, 0.5, 0, vt.VT_BF16, None) == 1
    assert vt.vt_attn_fwd(A, 2 * A, 3 * A, 4 * A, 0, H, S, S, 128, 128, 0.5, 0, vt.VT_BF16, None) == 0


# ---------------------------------------------------------------- output elements must not share addresses

@pytest.mark.parametrize("o_stride,H,S_q,dtype", [
    ((64, 64, 4), 1, 4, vt.VT_F32),    # rows 4 elements apart, 8 wide
    ((256, 8, 8), 2, 4, vt.VT_BF16),   # heads and rows on the same stride
    ((16, 64, 8), 2, 4, vt.VT_BF16),   # batches 16 elements apart, inside the 32 elements of a head's rows
])
def test_self_overlapping_output_is_rejected(lib, o_stride, H, S_q, dtype):
    B = 2
    sq = (H * S_q * 8, S_q * 8, 8)
    skv = (H * 4 * 8, 4 * 8, 8)
    assert vt.vt_attn_fwd_strided(A, sq, 2 * A, skv, 3 * A, skv, 8 * A, o_stride, B, H, S_q, 4, 8, 8, 0.5, 0,
                                  dtype, None) == 1


def test_other_output_nestings_pass_the_checks(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: a valid call would launch on these fake addresses")
    # [B, S, H, D] output (heads interleaved within each row block) and a padded one reach the launch
    B, H, S_q, D = 2, 2, 4, 8
    sq = (H * S_q * D, S_q * D, D)
    skv = (H * 4 * D, 4 * D, D)
    for o_stride in ((S_q * H * D, D, H * D), (H * S_q * 24, S_q * 24, 24)):
        assert vt.vt_attn_fwd_strided(A, sq, 2 * A, skv, 3 * A, skv, 8 * A, o_stride, B, H, S_q, 4, D, D, 0.5, 0,
                                      vt.VT_BF16, None) == 4
