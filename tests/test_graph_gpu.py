"""CUDA graph capture of the library's calls.

A forward captured once replays with new contents in its input tensors and gives the same bytes as
an eager call on the same inputs: the plain causal form, split-KV with a caller workspace, the
general form with grouped heads, a window and the LSE, and split-KV on the library's static scratch.  Replays reuse the captured launch
parameters (tensor maps, work-unit counter slot), so they skip the host-side work of a call.
"""

from __future__ import annotations

import math

import numpy as np
import pytest

import synth
from gpu_util import to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import scaled_dot_product_vt_gb300 as vt  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    vt.load()


def _replay_matches_eager(run, shapes, seeds):
    """Capture run(Q, K, V) -> list of output tensors on static inputs, then for each seed load new
    inputs into the static tensors, replay, and compare every output with an eager run."""
    static = [to_device(a) for a in synth.make_qkv(*shapes[0], seed=seeds[0], **shapes[1])]
    run(*static)  # per-device state and kernel attributes are set up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        outs = run(*static)
    for seed in seeds:
        fresh = [to_device(a) for a in synth.make_qkv(*shapes[0], seed=seed, **shapes[1])]
        for dst, src in zip(static, fresh):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        ref = run(*fresh)
        torch.cuda.synchronize()
        for got, want in zip(outs, ref):
            assert torch.equal(got, want), f"replay with inputs of seed {seed} differs from the eager call"
    assert vt.vt_last_device_status() == 0


def test_plain_causal_forward_in_a_graph():
    B, H, S_q, S_k, D = 2, 4, 700, 900, 128
    scale = float(np.float32(1.0 / math.sqrt(D)))

    def run(Q, K, V):
        o = torch.empty((B, H, S_q, D), dtype=torch.bfloat16, device="cuda")
        vt.attn_fwd(Q, K, V, scale=scale, causal=True, out=o)
        return [o]

    _replay_matches_eager(run, ((B, H, S_q, S_k, D, D, "bf16"), {}), seeds=(400, 401, 402))


def test_split_kv_forward_in_a_graph():
    B, H, S_q, S_k, D, n_split = 1, 2, 300, 4000, 128, 4
    scale = float(np.float32(1.0 / math.sqrt(D)))
    ws = torch.empty(vt.vt_attn_splitkv_workspace_size(B, H, S_q, D, n_split), dtype=torch.uint8, device="cuda")

    def run(Q, K, V):
        o = torch.empty((B, H, S_q, D), dtype=torch.bfloat16, device="cuda")
        vt.attn_fwd_general(Q, K, V, scale=scale, mask="causal", offset=S_k - S_q, n_split=n_split, out=o,
                            workspace=ws)
        return [o]

    _replay_matches_eager(run, ((B, H, S_q, S_k, D, D, "bf16"), {}), seeds=(410, 411))


def test_general_window_lse_forward_in_a_graph():
    B, H, H_kv, S, D = 2, 8, 2, 1500, 64
    scale = float(np.float32(1.0 / math.sqrt(D)))

    def run(Q, K, V):
        o = torch.empty((B, H, S, D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
        vt.attn_fwd_general(Q, K, V, scale=scale, mask="window", window=300, return_lse=True, out=o, lse=lse)
        return [o, lse]

    _replay_matches_eager(run, ((B, H, S, S, D, D, "bf16"), {"H_kv": H_kv}), seeds=(420, 421))


def test_noalloc_split_forward_in_a_graph():
    B, H, S_q, S_k, D = 1, 4, 256, 3000, 128
    scale = float(np.float32(1.0 / math.sqrt(D)))

    def run(Q, K, V):
        o = torch.empty((B, H, S_q, D), dtype=torch.bfloat16, device="cuda")
        rc = vt.vt_attn_fwd_splitkv_noalloc(Q.data_ptr(), [int(x) for x in Q.stride()[:3]], K.data_ptr(), [int(x) for x in K.stride()[:3]],
                                            V.data_ptr(), [int(x) for x in V.stride()[:3]], o.data_ptr(),
                                            [int(x) for x in o.stride()[:3]], B, H, S_q, S_k, D, D, scale, 0,
                                            vt.VT_BF16, 3, torch.cuda.current_stream().cuda_stream)
        assert rc == 0, vt.vt_status_str(rc)
        return [o]

    _replay_matches_eager(run, ((B, H, S_q, S_k, D, D, "bf16"), {}), seeds=(430, 431))
