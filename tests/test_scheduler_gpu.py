"""The persistent bf16 kernel's scheduling: correct across many launches, concurrent streams and graphs.

A launch has one CTA per work unit; running CTAs take over the units of CTAs that have not started
(cluster launch control), so no device state is shared between launches.  These tests check that the
outputs stay bit-identical to a single reference launch over (a) 1100 launches in a row, (b) launches on
two streams that run at the same time and (c) two captured CUDA graphs replayed on two streams at once.
"""

from __future__ import annotations

import math

import numpy as np
import pytest

import synth
from gpu_util import check, to_device, to_host64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import scaled_dot_product_vt_gb300 as vt  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    vt.load()


def _inputs(seed, B=1, H=4, S=600):
    q, k, v = synth.make_qkv(B, H, S, S, 64, 64, "bf16", seed=seed)
    return q, k, v, float(np.float32(1.0 / math.sqrt(64)))


def test_many_launches_in_a_row():
    """1100 launches in a row, all equal to the first."""
    q, k, v, scale = _inputs(90)
    Q, K, V = to_device(q), to_device(k), to_device(v)
    ref = vt.attn_fwd(Q, K, V, scale=scale, causal=True)
    torch.cuda.synchronize()
    check(to_host64(ref), oracle.attn_fwd(q, k, v, scale, True), "bf16", "reference launch")
    out = torch.empty_like(ref)
    mismatches = torch.zeros((), dtype=torch.int64, device="cuda")
    for _ in range(1100):
        vt.attn_fwd(Q, K, V, scale=scale, causal=True, out=out)
        mismatches += (out != ref).sum()
    assert vt.vt_last_device_status() == 0
    assert int(mismatches) == 0


def test_concurrent_streams():
    """Launches on two streams overlap in time and still give the single-stream results."""
    q1, k1, v1, scale = _inputs(91, B=2, H=8, S=1500)
    q2, k2, v2, _ = _inputs(92, B=2, H=8, S=1500)
    Q1, K1, V1 = to_device(q1), to_device(k1), to_device(v1)
    Q2, K2, V2 = to_device(q2), to_device(k2), to_device(v2)
    ref1 = vt.attn_fwd(Q1, K1, V1, scale=scale, causal=False)
    ref2 = vt.attn_fwd(Q2, K2, V2, scale=scale, causal=True)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs1 = [torch.empty_like(ref1) for _ in range(20)]
    outs2 = [torch.empty_like(ref2) for _ in range(20)]
    for i in range(20):
        vt.attn_fwd(Q1, K1, V1, scale=scale, causal=False, out=outs1[i], stream=s1)
        vt.attn_fwd(Q2, K2, V2, scale=scale, causal=True, out=outs2[i], stream=s2)
    torch.cuda.synchronize()
    assert vt.vt_last_device_status(s1) == 0 and vt.vt_last_device_status(s2) == 0
    for i in range(20):
        assert torch.equal(outs1[i], ref1), f"stream 1 launch {i}"
        assert torch.equal(outs2[i], ref2), f"stream 2 launch {i}"


def test_graphs_replayed_on_two_streams_at_once():
    """Two captured forwards replayed concurrently on two streams, many times, give the eager results."""
    q1, k1, v1, scale = _inputs(93, B=2, H=8, S=1200)
    q2, k2, v2, _ = _inputs(94, B=2, H=8, S=1200)
    Q1, K1, V1 = to_device(q1), to_device(k1), to_device(v1)
    Q2, K2, V2 = to_device(q2), to_device(k2), to_device(v2)
    ref1 = vt.attn_fwd(Q1, K1, V1, scale=scale, causal=True)
    ref2 = vt.attn_fwd(Q2, K2, V2, scale=scale, causal=False)
    torch.cuda.synchronize()
    o1, o2 = torch.empty_like(ref1), torch.empty_like(ref2)
    g1, g2 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1):
        vt.attn_fwd(Q1, K1, V1, scale=scale, causal=True, out=o1)
    with torch.cuda.graph(g2):
        vt.attn_fwd(Q2, K2, V2, scale=scale, causal=False, out=o2)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    bad1 = torch.zeros((), dtype=torch.int64, device="cuda")
    bad2 = torch.zeros((), dtype=torch.int64, device="cuda")
    for _ in range(50):
        o1.zero_()
        o2.zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(s1):
            g1.replay()
        with torch.cuda.stream(s2):
            g2.replay()
        torch.cuda.synchronize()
        bad1 += (o1 != ref1).sum()
        bad2 += (o2 != ref2).sum()
    assert vt.vt_last_device_status() == 0
    assert int(bad1) == 0 and int(bad2) == 0
