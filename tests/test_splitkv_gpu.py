"""GPU parity of the split-KV forward (shares of the key range + merge) against the fp64 oracle."""

from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import synth
from gpu_util import check, to_device, to_host64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import scaled_dot_product_vt_gb300 as vt  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    vt.load()


CASES = [
    # B, H, S_q, S_k, D_qk, D_v, causal, n_split
    (1, 2, 64, 4096, 128, 128, False, 8),
    (1, 2, 300, 2000, 64, 64, True, 4),      # early rows have no key in the later shares
    (2, 3, 129, 1000, 96, 64, False, 3),     # uneven shares, D_qk != D_v
    (1, 1, 1, 513, 128, 128, False, 5),      # one query row, ragged key tail
    (1, 1, 256, 256, 128, 128, True, 4),     # more shares than key tiles: empty shares
    (2, 1, 77, 8191, 32, 48, False, 64),     # the largest share count
    (1, 4, 200, 3000, 128, 128, True, 2),
]


@pytest.mark.parametrize("case", CASES, ids=str)
def test_splitkv_matches_oracle(case):
    B, H, S_q, S_k, D_qk, D_v, causal, n_split = case
    q, k, v = synth.make_qkv(B, H, S_q, S_k, D_qk, D_v, "bf16", seed=(hash(case) & 0xFFFF) + 3)
    scale = float(np.float32(1.0 / math.sqrt(D_qk)))
    Q, K, V = to_device(q), to_device(k), to_device(v)
    got = to_host64(vt.attn_fwd_splitkv(Q, K, V, scale=scale, causal=causal, n_split=n_split))
    assert vt.vt_last_device_status() == 0
    ref = oracle.attn_fwd(q, k, v, scale, causal)
    check(got, ref, "bf16", f"split-KV {case}")
    plain = to_host64(vt.attn_fwd(Q, K, V, scale=scale, causal=causal))
    assert np.abs(got - plain).max() <= 2e-2


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("scale", [-0.2, 0.0])
def test_splitkv_non_positive_scale(dtype, scale):
    """Split-KV shares with a scale that cannot fold into the exponent (the partial-output and merge path of
    the kernel variants that scale the scores first)."""
    B, H, S_q, S_k, D = 1, 2, 300, 1500, (128 if dtype == "bf16" else 72)
    q, k, v = synth.make_qkv(B, H, S_q, S_k, D, D, dtype, seed=29)
    Q, K, V = to_device(q), to_device(k), to_device(v)
    got = to_host64(vt.attn_fwd_splitkv(Q, K, V, scale=scale, causal=True, n_split=3))
    assert vt.vt_last_device_status() == 0
    check(got, oracle.attn_fwd(q, k, v, scale, True), dtype, f"split-KV scale={scale}")


CASES_F32 = [
    # B, H, S_q, S_k, D_qk, D_v, causal, n_split (fp32 I/O, TF32 path; 64-key tiles)
    (2, 4, 1000, 1000, 72, 72, True, 2),    # the mid fp32 workload's shape
    (1, 2, 200, 3000, 64, 48, False, 5),
    (1, 1, 100, 130, 20, 20, False, 3),     # three key tiles, one per share
    (1, 2, 130, 1000, 128, 128, True, 4),   # early rows have no key in the later shares
    (1, 1, 64, 256, 32, 32, True, 8),       # more shares than key tiles: empty shares
]


@pytest.mark.parametrize("case", CASES_F32, ids=str)
def test_splitkv_fp32_matches_oracle(case):
    B, H, S_q, S_k, D_qk, D_v, causal, n_split = case
    q, k, v = synth.make_qkv(B, H, S_q, S_k, D_qk, D_v, "f32", dist="uniform", seed=(hash(case) & 0xFFFF) + 5)
    scale = float(np.float32(1.0 / math.sqrt(D_qk)))
    Q, K, V = to_device(q), to_device(k), to_device(v)
    got = to_host64(vt.attn_fwd_splitkv(Q, K, V, scale=scale, causal=causal, n_split=n_split))
    assert vt.vt_last_device_status() == 0
    check(got, oracle.attn_fwd(q, k, v, scale, causal), "f32", f"fp32 split-KV {case}")


def test_splitkv_workspace_reuse_and_auto_choice():
    """One workspace serves calls with different share counts; the library's choice is used when none is given."""
    B, H, S_q, S_k, D = 1, 4, 128, 16384, 128
    q, k, v = synth.make_qkv(B, H, S_q, S_k, D, D, "bf16", seed=41)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    Q, K, V = to_device(q), to_device(k), to_device(v)
    n_auto = vt.vt_attn_splitkv_choose(B, H, S_q, S_k, False, vt.VT_BF16)
    assert n_auto > 1  # 4 work items on a GPU with many more SMs
    need = max(vt.vt_attn_splitkv_workspace_size(B, H, S_q, D, n) for n in (2, 7, n_auto))
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device="cuda")
    ref = oracle.attn_fwd(q, k, v, scale, False)
    for n in (7, 2, n_auto):
        got = to_host64(vt.attn_fwd_splitkv(Q, K, V, scale=scale, n_split=n, workspace=ws))
        assert vt.vt_last_device_status() == 0
        check(got, ref, "bf16", f"n_split={n}")
    got = to_host64(vt.attn_fwd_splitkv(Q, K, V, scale=scale))
    check(got, ref, "bf16", "auto split")


@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_write_set_guard_bands(causal):
    """The merge writes only O's logical elements: padding columns, rows and canaries stay bit-exact."""
    B, H, S_q, S_k, D_qk, D_v = 2, 2, 150, 1500, 64, 24
    q, k, v = synth.make_qkv(B, H, S_q, S_k, D_qk, D_v, "bf16", seed=43)
    row = D_v + 8
    o_strides = (H * (S_q + 3) * row, (S_q + 3) * row, row, 1)
    canary = 2048
    total = canary + B * o_strides[0] + canary
    sentinel = 0xDEAD - (1 << 16)
    buf = torch.full((total,), sentinel, dtype=torch.int16, device="cuda")
    O = torch.as_strided(buf.view(torch.bfloat16), (B, H, S_q, D_v), o_strides, canary + row)
    Q, K, V = to_device(q), to_device(k), to_device(v)
    vt.attn_fwd_splitkv(Q, K, V, scale=0.125, causal=causal, n_split=5, out=O)
    assert vt.vt_last_device_status() == 0
    host = buf.cpu().numpy()
    mask = np.ones(total, bool)
    idx = (canary + row + np.arange(B)[:, None, None, None] * o_strides[0] + np.arange(H)[None, :, None, None] * o_strides[1]
           + np.arange(S_q)[None, None, :, None] * o_strides[2] + np.arange(D_v)[None, None, None, :])
    mask[idx.ravel()] = False
    assert np.all(host[mask] == sentinel)
    check(to_host64(O), oracle.attn_fwd(q, k, v, 0.125, causal), "bf16", "strided split-KV")
