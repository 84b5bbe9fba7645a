"""vt_attn_fwd_splitkv_noalloc: the split-KV forward for callers that cannot allocate device memory.

Some callers may not call cudaMalloc at all: a plugin inside a host framework that owns every byte
of device memory, or a latency-critical service that must not allocate after start-up because an
allocation can block and synchronise the device.  This entry point keeps the shares' partial
results in the library's fixed 32 MiB device array instead of a caller workspace.  The GPU test
checks it against the workspace-taking entry point and against the fp64 oracle on calls in a row
(each later call finds the earlier calls' data still in the shared array), for both element types;
the host tests check the size limit.
"""

from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import synth
from gpu_util import check, to_device, to_host64

import scaled_dot_product_vt_gb300 as vt

LIMIT = 32 << 20  # bytes of the library's fixed scratch array
A = 1 << 20       # fake, aligned, distinct "device" addresses: never dereferenced on host-checked paths


def _strides(t):
    return (t.stride(0), t.stride(1), t.stride(2))


def test_rejects_problems_beyond_the_fixed_scratch():
    vt.build()
    # B=1, H=32, S_q=4096, D_v=128 with 2 shares needs about 68 MB of partial results
    B, H, S_q, S_k, D = 1, 32, 4096, 4096, 128
    assert vt.vt_attn_splitkv_workspace_size(B, H, S_q, D, 2) > LIMIT
    st = (H * S_q * D, S_q * D, D)
    rc = vt.vt_attn_fwd_splitkv_noalloc(A, st, A * 256, st, A * 512, st, A * 768, st, B, H, S_q, S_k, D, D,
                                        0.125, 0, vt.VT_BF16, 2, None)
    assert rc == 2  # VT_ERR_UNSUPPORTED, before anything runs
    assert vt.vt_attn_fwd_splitkv_noalloc(A, st, A * 256, st, A * 512, st, A * 768, st, B, H, S_q, S_k, D, D,
                                          0.125, 0, vt.VT_BF16, 0, None) == 1  # VT_ERR_INVALID_ARG


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    vt.load()
    stream = torch.cuda.current_stream().cuda_stream
    calls = [
        # B, H, S_q, S_k, D_qk, D_v, causal, n_split, dtype
        (1, 4, 200, 4096, 128, 128, False, 6, "bf16"),
        (2, 2, 64, 3000, 64, 64, True, 4, "bf16"),
        (1, 2, 100, 2000, 72, 72, False, 3, "f32"),
    ]
    for i, (B, H, S_q, S_k, D_qk, D_v, causal, n_split, dtype) in enumerate(calls):
        assert vt.vt_attn_splitkv_workspace_size(B, H, S_q, D_v, n_split) <= LIMIT
        q, k, v = synth.make_qkv(B, H, S_q, S_k, D_qk, D_v, dtype, seed=50 + i)
        scale = float(np.float32(1.0 / math.sqrt(D_qk)))
        Q, K, V = to_device(q), to_device(k), to_device(v)
        O_ref = vt.attn_fwd_splitkv(Q, K, V, scale=scale, causal=causal, n_split=n_split)
        O = torch.empty_like(O_ref)
        code = vt.VT_BF16 if dtype == "bf16" else vt.VT_F32
        rc = vt.vt_attn_fwd_splitkv_noalloc(Q.data_ptr(), _strides(Q), K.data_ptr(), _strides(K), V.data_ptr(),
                                            _strides(V), O.data_ptr(), _strides(O), B, H, S_q, S_k, D_qk, D_v,
                                            scale, causal, code, n_split, stream)
        assert rc == 0
        assert vt.vt_last_device_status(stream) == 0
        got = to_host64(O)
        check(got, to_host64(O_ref), dtype, f"no-alloc call {i + 1} vs the workspace entry point")
        check(got, oracle.attn_fwd(q, k, v, scale, causal), dtype, f"no-alloc call {i + 1} vs the oracle")
