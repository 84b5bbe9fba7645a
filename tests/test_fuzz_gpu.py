"""Seeded random configurations of the general entry point against the fp64 oracle.

Each case draws an element type, batch, heads, grouped key/value heads, sequence lengths, head
dimensions (row pitch a multiple of 16 bytes, as the TMA requires), a mask kind with its offset and
window, a split-KV share count and whether the log-sum-exp is returned.  Sizes stay small enough
for the oracle to finish in well under a second per case, while still spanning several tiles and
ragged tails.  The tolerances are those of the other parity tests.
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
N_CASES = 96


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    vt.load()


def draw_case(i: int):
    rng = np.random.default_rng(1000 + i)
    dtype = "bf16" if rng.random() < 0.6 else "f32"
    step = 8 if dtype == "bf16" else 4          # head dims whose row pitch is a multiple of 16 bytes
    H_kv = int(rng.integers(1, 4))
    H = H_kv * int(rng.integers(1, 4))
    B = int(rng.integers(1, 3))
    S_q = int(rng.integers(1, 700))
    S_k = int(rng.integers(1, 1300))
    D_qk = int(step * rng.integers(1, 128 // step + 1))
    D_v = int(step * rng.integers(1, 128 // step + 1))
    mask = str(rng.choice(list(oracle.MASKS)))
    offset = int(rng.integers(0, 2 * S_k + 2)) if rng.random() < 0.7 else 0
    window = int(rng.integers(1, S_k + 200))
    n_split = int(rng.choice([1, 1, 2, 3, 5]))
    return dtype, B, H, H_kv, S_q, S_k, D_qk, D_v, mask, offset, window, n_split


@pytest.mark.parametrize("i", range(N_CASES))
def test_fuzz_case(i):
    dtype, B, H, H_kv, S_q, S_k, D_qk, D_v, mask, offset, window, n_split = draw_case(i)
    what = (f"case {i}: {dtype} B={B} H={H} H_kv={H_kv} S_q={S_q} S_k={S_k} D={D_qk}/{D_v} {mask} "
            f"offset={offset} window={window} n_split={n_split}")
    dist = "uniform" if dtype == "f32" else "normal"
    q, k, v = synth.make_qkv(B, H, S_q, S_k, D_qk, D_v, dtype, dist=dist, seed=2000 + i, H_kv=H_kv)
    scale = float(np.float32(1.0 / math.sqrt(D_qk)))
    Q, K, V = to_device(q), to_device(k), to_device(v)
    O, L = vt.attn_fwd_general(Q, K, V, scale=scale, mask=mask, offset=offset, window=window, return_lse=True,
                               n_split=n_split)
    assert vt.vt_last_device_status() == 0, what
    got, lse = to_host64(O), L.double().cpu().numpy()
    ref, ref_lse = oracle.attn_general(q, k, v, scale, mask, offset, window, with_lse=True)
    check(got, ref, dtype, what)
    empty = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: empty rows differ"
    assert np.all(got[empty] == 0.0), f"{what}: a row with no allowed key is not 0"
    fin = ~empty
    err = float(np.abs(lse[fin] - ref_lse[fin]).max(initial=0.0))
    assert err <= TOL_LSE[dtype], f"{what}: LSE max abs error {err:.3e}"
