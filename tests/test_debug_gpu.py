"""The debug library (libvt_attn_debug.so, built with VT_DEBUG): device index checks.

Its kernels check their index invariants (decoded work units, key-tile ranges, ring slots) before
the accesses they guard.  On valid calls every check passes and the outputs are bit-identical to the
release library's.  VT_OPT_TEST_BOUNDS makes the first producer check report a failure: the call
then records VT_ERR_DEVICE_BOUNDS, leaves O untouched and the context stays usable.  The release
library ignores that flag.
"""

from __future__ import annotations

import ctypes
import math

import numpy as np
import pytest

import synth
from gpu_util import to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import scaled_dot_product_vt_gb300 as vt  # noqa: E402


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return vt.load(), vt.load_debug()


def _st(t):
    return (ctypes.c_int64 * 3)(*[int(x) for x in t.stride()[:3]])


def _general(lib, Q, K, V, O, lse, scale, mask, offset, window, n_split, ws, flags=0):
    B, H, S_q, D_qk = Q.shape
    H_kv, S_k, D_v = K.shape[1], K.shape[2], V.shape[3]
    m = vt.vt_attn_mask(vt.MASKS[mask], 0, offset, window)
    opts = vt.vt_attn_opts(0, flags, 0)
    code = vt.VT_BF16 if Q.dtype == torch.bfloat16 else vt.VT_F32
    return lib.vt_attn_fwd_general(Q.data_ptr(), _st(Q), K.data_ptr(), _st(K), V.data_ptr(), _st(V), O.data_ptr(),
                                   _st(O), lse.data_ptr() if lse is not None else None, B, H, H_kv, S_q, S_k, D_qk,
                                   D_v, scale, code, ctypes.byref(m), n_split,
                                   ws.data_ptr() if ws is not None else None,
                                   ws.numel() if ws is not None else 0, ctypes.byref(opts),
                                   torch.cuda.current_stream().cuda_stream)


# name: dtype, B, H, H_kv, S_q, S_k, D_qk, D_v, mask, offset, window, n_split
CASES = {
    "bf16_causal": ("bf16", 2, 4, 4, 700, 700, 128, 128, "causal", 0, 0, 1),
    "bf16_ragged_noncausal": ("bf16", 1, 3, 3, 333, 1000, 96, 64, "none", 0, 0, 1),
    "bf16_split_offset": ("bf16", 1, 2, 2, 300, 3000, 128, 128, "causal", 2700, 0, 4),
    "bf16_gqa_window": ("bf16", 2, 8, 2, 900, 900, 64, 64, "window", 0, 200, 1),
    "bf16_complement_split": ("bf16", 1, 4, 4, 600, 1500, 128, 128, "window_complement", 900, 300, 3),
    "f32_causal": ("f32", 2, 2, 2, 300, 300, 72, 72, "causal", 0, 0, 1),
    "f32_split_window": ("f32", 1, 2, 1, 200, 900, 64, 40, "window", 700, 250, 2),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_debug_checks_pass_and_match_release(libs, name):
    rel, dbg = libs
    dtype, B, H, H_kv, S_q, S_k, D_qk, D_v, mask, offset, window, n_split = CASES[name]
    q, k, v = synth.make_qkv(B, H, S_q, S_k, D_qk, D_v, dtype, seed=500 + sorted(CASES).index(name), H_kv=H_kv,
                             dist="uniform" if dtype == "f32" else "normal")
    Q, K, V = to_device(q), to_device(k), to_device(v)
    scale = float(np.float32(1.0 / math.sqrt(D_qk)))
    ws = None
    if n_split > 1:
        ws = torch.empty(vt.vt_attn_splitkv_workspace_size(B, H, S_q, D_v, n_split), dtype=torch.uint8, device="cuda")
    outs = []
    for lib in (rel, dbg):
        O = torch.empty((B, H, S_q, D_v), dtype=Q.dtype, device="cuda")
        lse = torch.empty((B, H, S_q), dtype=torch.float32, device="cuda")
        assert _general(lib, Q, K, V, O, lse, scale, mask, offset, window, n_split, ws) == 0
        assert lib.vt_last_device_status(torch.cuda.current_stream().cuda_stream) == 0, name
        outs.append((O, lse))
    assert torch.equal(outs[0][0], outs[1][0]), f"{name}: debug output differs from release"
    assert torch.equal(outs[0][1], outs[1][1]), f"{name}: debug LSE differs from release"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_forced_check_failure_reports_bounds_and_context_survives(libs, dtype):
    rel, dbg = libs
    B, H, S, D = 1, 2, 300, 64
    q, k, v = synth.make_qkv(B, H, S, S, D, D, dtype, seed=520)
    Q, K, V = to_device(q), to_device(k), to_device(v)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    sentinel = 1234.5
    stream = torch.cuda.current_stream().cuda_stream
    O = torch.full((B, H, S, D), sentinel, dtype=Q.dtype, device="cuda")
    assert _general(dbg, Q, K, V, O, None, scale, "causal", 0, 0, 1, None, flags=vt.VT_OPT_TEST_BOUNDS) == 0
    assert dbg.vt_last_device_status(stream) == 6  # VT_ERR_DEVICE_BOUNDS
    assert bool((O == sentinel).all()), "the stopped call wrote O"
    # the context is intact: a normal call works and its status is clean
    assert _general(dbg, Q, K, V, O, None, scale, "causal", 0, 0, 1, None) == 0
    assert dbg.vt_last_device_status(stream) == 0
    ref = torch.empty_like(O)
    assert _general(rel, Q, K, V, ref, None, scale, "causal", 0, 0, 1, None) == 0
    assert torch.equal(O, ref)
    # the release library ignores the flag
    O2 = torch.full_like(O, sentinel)
    assert _general(rel, Q, K, V, O2, None, scale, "causal", 0, 0, 1, None, flags=vt.VT_OPT_TEST_BOUNDS) == 0
    assert rel.vt_last_device_status(stream) == 0
    assert torch.equal(O2, ref)
