"""The persistent bf16 kernel's work-unit counter: correct across many launches and concurrent streams.

Each launch draws its units from one slot of a static array of 1024 counters (launch sequence
number mod 1024) and its last CTA resets the slot.  These tests check that the outputs stay
bit-identical to a single reference launch when (a) more than 1024 launches wrap the slots
around and (b) launches on two streams run at the same time (each on its own slot).
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


def test_slots_wrap_around():
    """1100 launches (more than the 1024 counter slots) in a row, all equal to the first."""
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
