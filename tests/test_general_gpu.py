"""GPU parity of the general entry point: grouped key/value heads, the offset causal mask, the
sliding window and its complement, and the per-row log-sum-exp, against the fp64 oracle.

Tolerances.  O: the same bars as the plain forward (bf16 max abs 2e-2 and relative Frobenius 1e-2;
fp32 I/O max abs 5e-3).  LSE: bf16 inputs make every product exact in the fp32 accumulator, so the
scores are off by a few fp32 ulps of sum |scale q_d k_d| (~1e-5 here) and the exp2/log2 hardware
approximations add ~1e-6 relative; 1e-3 absolute leaves a wide margin.  TF32 operands keep 10
mantissa bits, so an fp32-I/O score can be off by ~2^-11 sum |scale q_d k_d| (~1e-3 for these
shapes); 1e-2 absolute.  Rows with no allowed key must be exactly 0 with LSE = -inf.
"""

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

TOL_LSE = {"bf16": 1e-3, "f32": 1e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    vt.load()


def inputs(dtype, B, H, H_kv, S_q, S_k, D_qk, D_v, seed, dist="normal"):
    return synth.make_qkv(B, H, S_q, S_k, D_qk, D_v, dtype, dist=dist, seed=seed, H_kv=H_kv)


def run_general(q, k, v, scale, mask, offset=0, window=0, n_split=1):
    Q, K, V = to_device(q), to_device(k), to_device(v)
    O, L = vt.attn_fwd_general(Q, K, V, scale=scale, mask=mask, offset=offset, window=window, return_lse=True,
                               n_split=n_split)
    assert vt.vt_last_device_status() == 0
    return to_host64(O), L.double().cpu().numpy()


def check_lse(got, ref, dtype, what):
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), f"{what}: empty rows differ"
    fin = np.isfinite(ref)
    assert np.all(np.isfinite(got[fin])), f"{what}: non-finite LSE"
    err = float(np.abs(got[fin] - ref[fin]).max(initial=0.0))
    assert err <= TOL_LSE[dtype], f"{what}: LSE max abs error {err:.3e} > {TOL_LSE[dtype]}"


# name: dtype, B, H, H_kv, S_q, S_k, D_qk, D_v, mask, offset, window, n_split
CASES = {
    "offset_bottom_right": ("bf16", 1, 2, 2, 300, 1000, 128, 128, "causal", 700, 0, 1),
    "offset_37_ragged": ("bf16", 2, 2, 2, 517, 530, 64, 64, "causal", 37, 0, 1),
    "offset_past_all_keys": ("bf16", 1, 2, 2, 260, 300, 64, 64, "causal", 5000, 0, 1),
    "gqa_causal": ("bf16", 2, 8, 2, 520, 520, 128, 128, "causal", 0, 0, 1),
    "mqa_none": ("bf16", 1, 6, 1, 300, 777, 96, 64, "none", 0, 0, 1),
    "window_200": ("bf16", 1, 4, 2, 1100, 1100, 128, 128, "window", 0, 200, 1),
    "window_1": ("bf16", 1, 2, 2, 300, 300, 64, 64, "window", 0, 1, 1),
    "window_129_offset_5": ("bf16", 1, 2, 1, 700, 705, 128, 128, "window", 5, 129, 1),
    "window_decode": ("bf16", 1, 2, 2, 300, 1000, 128, 128, "window", 700, 256, 1),
    "window_past_keys": ("bf16", 1, 2, 2, 600, 300, 64, 64, "window", 0, 64, 1),
    "complement_256": ("bf16", 1, 2, 2, 700, 700, 128, 128, "window_complement", 0, 256, 1),
    "complement_all_empty": ("bf16", 1, 1, 1, 200, 200, 64, 64, "window_complement", 0, 1000, 1),
    "complement_offset": ("bf16", 1, 2, 2, 400, 900, 96, 96, "window_complement", 300, 100, 1),
    "f32_offset": ("f32", 1, 2, 2, 200, 450, 72, 72, "causal", 250, 0, 1),
    "f32_gqa_window": ("f32", 2, 4, 2, 333, 333, 64, 48, "window", 3, 70, 1),
    "f32_complement_empty_block": ("f32", 1, 2, 1, 300, 300, 32, 32, "window_complement", 0, 130, 1),
    "f32_mqa_none": ("f32", 1, 4, 1, 130, 200, 20, 20, "none", 0, 0, 1),
    "split_window": ("bf16", 1, 2, 2, 256, 4096, 128, 128, "window", 3840, 1500, 4),
    "split_gqa_offset": ("bf16", 1, 8, 2, 200, 3000, 128, 128, "causal", 2800, 0, 5),
    "split_complement": ("bf16", 1, 2, 2, 300, 2000, 64, 64, "window_complement", 1700, 500, 3),
    "split_window_empty_shares": ("bf16", 1, 2, 1, 300, 4000, 64, 64, "window", 0, 100, 8),
    "f32_split_window": ("f32", 1, 2, 2, 300, 2000, 64, 64, "window", 1700, 500, 3),
    "f32_split_gqa_complement": ("f32", 1, 4, 1, 256, 1500, 32, 32, "window_complement", 1200, 300, 4),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_general_case(name):
    dtype, B, H, H_kv, S_q, S_k, D_qk, D_v, mask, offset, window, n_split = CASES[name]
    dist = "uniform" if dtype == "f32" else "normal"
    q, k, v = inputs(dtype, B, H, H_kv, S_q, S_k, D_qk, D_v, seed=100 + sorted(CASES).index(name), dist=dist)
    scale = float(np.float32(1.0 / math.sqrt(D_qk)))
    got, lse = run_general(q, k, v, scale, mask, offset, window, n_split)
    ref, ref_lse = oracle.attn_general(q, k, v, scale, mask, offset, window, with_lse=True)
    check(got, ref, dtype, name)
    check_lse(lse, ref_lse, dtype, name)
    empty = np.isneginf(ref_lse)
    assert np.all(got[empty] == 0.0), f"{name}: a row with no allowed key is not 0"


def test_lse_merges_window_and_complement_into_causal():
    """Two calls over disjoint key sets (a window and its complement) merged through their GPU
    log-sum-exps reproduce the causal output (the continuation identity)."""
    B, H, S, D, w, o = 1, 4, 900, 128, 160, 40
    q, k, v = inputs("bf16", B, H, H, S, S + o, D, D, seed=71)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    Ow, Lw = run_general(q, k, v, scale, "window", o, w)
    Oc, Lc = run_general(q, k, v, scale, "window_complement", o, w)
    M = np.maximum(Lw, Lc)
    ww, wc = np.exp(Lw - M), np.exp(Lc - M)
    merged = (ww[..., None] * Ow + wc[..., None] * Oc) / (ww + wc)[..., None]
    ref = oracle.attn_general(q, k, v, scale, "causal", o)
    check(merged, ref, "bf16", "window + complement merged")


def test_gqa_equals_repeated_heads_on_gpu():
    """Grouped heads give bit-identical results to plain multi-head attention on repeated K/V."""
    B, H, H_kv, S, D = 2, 8, 2, 300, 64
    q, k, v = inputs("bf16", B, H, H_kv, S, S, D, D, seed=72)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    got, _ = run_general(q, k, v, scale, "causal")
    rep = H // H_kv
    kx, vx = np.repeat(k, rep, axis=1), np.repeat(v, rep, axis=1)
    O = vt.attn_fwd(to_device(q), to_device(kx), to_device(vx), scale=scale, causal=True)
    assert np.array_equal(got, to_host64(O))


def test_general_plain_masks_match_plain_entry_point():
    """mask none / causal with offset 0 and H_kv = H give bit-identical results to vt_attn_fwd."""
    q, k, v = inputs("bf16", 2, 3, 3, 333, 333, 96, 64, seed=73)
    for causal in (False, True):
        got, _ = run_general(q, k, v, 0.1, "causal" if causal else "none")
        O = vt.attn_fwd(to_device(q), to_device(k), to_device(v), scale=0.1, causal=causal)
        assert np.array_equal(got, to_host64(O))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_empty_rows_written_and_guard_bands_kept(dtype):
    """A row with no allowed key is written as 0; padding around a strided O stays untouched."""
    B, H, S_q, S_k, D_qk, D_v = 1, 2, 300, 300, 64, 40
    q, k, v = inputs(dtype, B, H, H, S_q, S_k, D_qk, D_v, seed=74)
    elt = 2 if dtype == "bf16" else 4
    row = D_v + 8
    o_strides = (H * (S_q + 2) * row, (S_q + 2) * row, row)
    canary = 4096 // elt
    total = canary + B * o_strides[0] + canary
    tdt = torch.int16 if dtype == "bf16" else torch.int32
    sentinel = 0xDEAD - (1 << 16) if dtype == "bf16" else 0x7FC0DEAD
    buf = torch.full((total,), sentinel, dtype=tdt, device="cuda")
    view_dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    O = torch.as_strided(buf.view(view_dt), (B, H, S_q, D_v), o_strides + (1,), canary + row)
    vt.attn_fwd_general(to_device(q), to_device(k), to_device(v), scale=0.125, mask="window_complement", window=150,
                        out=O)
    assert vt.vt_last_device_status() == 0
    host = buf.cpu().numpy()
    keep = np.ones(total, bool)
    idx = (canary + row + np.arange(B)[:, None, None, None] * o_strides[0] + np.arange(H)[None, :, None, None] * o_strides[1]
           + np.arange(S_q)[None, None, :, None] * o_strides[2] + np.arange(D_v)[None, None, None, :])
    keep[idx.ravel()] = False
    assert np.all(host[keep] == sentinel), "a position outside O's logical elements was written"
    got = to_host64(O)
    assert np.all(got[:, :, :150] == 0.0), "rows with no allowed key must be 0"
    check(got, oracle.attn_general(q, k, v, 0.125, "window_complement", 0, 150), dtype, "complement, strided O")


# ---------------------------------------------------------------- full-size shapes, sampled rows

SAMPLED = {
    # name: B, H, H_kv, S_q, S_k, D, mask, offset, window, n_split (0: the library's choice)
    "gqa_causal_4k": (8, 32, 8, 4096, 4096, 128, "causal", 0, 0, 1),
    "prefill_on_cache_8k": (8, 16, 16, 1024, 8192, 128, "causal", 7168, 0, 1),
    "window_1024_8k": (4, 16, 16, 8192, 8192, 128, "window", 0, 1024, 1),
    "complement_1024_8k": (2, 16, 4, 8192, 8192, 128, "window_complement", 0, 1024, 1),
    # the 32k-cache chunk workload, with the library's share count (4 on 152 SMs) and without shares
    "chunk_on_cache_32k_split": (2, 16, 16, 256, 32768, 128, "causal", 32512, 0, 0),
    "chunk_on_cache_32k_one": (2, 16, 16, 256, 32768, 128, "causal", 32512, 0, 1),
    # long and wide extremes: 2^20 keys (8192 key tiles; 38 shares on 152 SMs), and 4096 heads
    "long_cache_1m_split": (1, 2, 2, 300, 1 << 20, 128, "causal", (1 << 20) - 300, 0, 0),
    "many_heads_4096": (64, 64, 16, 256, 256, 64, "none", 0, 0, 1),
}


@pytest.mark.parametrize("name", sorted(SAMPLED))
def test_full_size_sampled(name):
    B, H, H_kv, S_q, S_k, D, mask, offset, window, n_split = SAMPLED[name]
    if n_split == 0:
        n_split = vt.vt_attn_splitkv_choose(B, H, S_q, S_k, 1, vt.VT_BF16)
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        items = B * H * ((S_q + 255) // 256)
        assert n_split == max(1, min(sms // items if items < sms else 1, (S_k + 127) // 128 // 4, 64))
    q, k, v = inputs("bf16", B, H, H_kv, S_q, S_k, D, D, seed=80 + len(name))
    scale = float(np.float32(1.0 / math.sqrt(D)))
    got, lse = run_general(q, k, v, scale, mask, offset, window, n_split)
    rng = np.random.default_rng(81)
    edges = [e for e in (0, 1, 127, 128, 255, 256, S_q // 2, S_q - 129, S_q - 1) if 0 <= e < S_q]
    rows = sorted({(int(b), int(h), int(i)) for b, h in [(0, 0), (B - 1, H - 1), (B // 2, H // 3)]
                   for i in edges + [int(x) for x in rng.integers(0, S_q, size=24)]})
    rows = np.array(rows, dtype=np.int64)
    ref, ref_lse = oracle.attn_general(q, k, v, scale, mask, offset, window, rows=rows, with_lse=True)
    g = got[rows[:, 0], rows[:, 1], rows[:, 2]]
    check(g, ref, "bf16", name)
    check_lse(lse[rows[:, 0], rows[:, 1], rows[:, 2]], ref_lse, "bf16", name)
