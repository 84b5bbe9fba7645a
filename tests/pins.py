"""Pins for the attention oracle: facts fixed by the definition, not by the oracle's code.

Each pin takes a loaded oracle library (the real one, or a deliberately broken
copy built by the mutation test) and raises AssertionError when the fact fails.
The definition pinned is the naive reference of the VeriTile page
"VeriTile.Examples.FlashAttention1.NaiveRefinement" (fa1NaiveReference4D and the
causal form, key j <= query i) and the accy page's CPU routine `expectedOutput`;
the general form's extras (grouped key/value heads, the offset causal mask, the
sliding window and its complement, the per-row log-sum-exp) are pinned against
the plain non-causal definition on truncated or repeated inputs and against
closed forms.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle
from synth import make_qkv, to_bf16_bits, element_counts

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rand(shape, seed, sigma=1.0):
    r = np.random.default_rng(seed)
    return (r.standard_normal(shape) * sigma).astype(np.float32)


def _O(lib, Q, K, V, scale, causal):
    return oracle.attn_fwd(Q, K, V, scale, causal, nthreads=2, lib=lib)


def pin_ones_value(lib):
    """V == 1 everywhere gives O == 1 (weights sum to one), both modes."""
    Q, K = _rand((2, 3, 7, 5), 1), _rand((2, 3, 9, 5), 2)
    V = np.ones((2, 3, 9, 4), np.float32)
    for causal in (False, True):
        O = _O(lib, Q, K, V, 0.7, causal)
        assert np.allclose(O, 1.0, atol=1e-13), "V==1 must give O==1"


def pin_identical_keys_mean(lib):
    """All key rows equal: every weight is equal, so O is the mean of V over the allowed keys."""
    Q = _rand((1, 2, 6, 3), 3)
    K = np.broadcast_to(_rand((1, 2, 1, 3), 4), (1, 2, 8, 3)).copy()
    V = _rand((1, 2, 8, 5), 5)
    O = _O(lib, Q, K, V, 0.9, False)
    assert np.allclose(O, V.astype(np.float64).mean(axis=2, keepdims=True), atol=1e-12)
    Oc = _O(lib, Q, K, V, 0.9, True)
    cum = np.cumsum(V.astype(np.float64), axis=2) / np.arange(1, 9)[None, None, :, None]
    assert np.allclose(Oc, cum[:, :, :6, :], atol=1e-12), "causal: mean of V[0..i]"


def pin_scale_zero_mean(lib):
    """scale = 0 makes every score 0: O is the plain mean of V over the allowed keys."""
    Q, K, V = _rand((1, 1, 5, 4), 6), _rand((1, 1, 5, 4), 7), _rand((1, 1, 5, 3), 8)
    O = _O(lib, Q, K, V, 0.0, False)
    assert np.allclose(O, V.astype(np.float64).mean(axis=2, keepdims=True), atol=1e-13)


def pin_key_permutation(lib):
    """Non-causal O is unchanged when one permutation is applied to the rows of K and V."""
    Q, K, V = _rand((2, 2, 5, 6), 9), _rand((2, 2, 11, 6), 10), _rand((2, 2, 11, 3), 11)
    perm = np.random.default_rng(12).permutation(11)
    O1 = _O(lib, Q, K, V, 0.4, False)
    O2 = _O(lib, Q, K[:, :, perm], V[:, :, perm], 0.4, False)
    assert np.allclose(O1, O2, atol=1e-12)


def pin_causal_row0_and_prefix(lib):
    """Causal row 0 is V[0] exactly; causal row i equals the non-causal output over keys 0..i."""
    Q, K, V = _rand((1, 2, 6, 4), 13), _rand((1, 2, 6, 4), 14), _rand((1, 2, 6, 3), 15)
    Oc = _O(lib, Q, K, V, 0.8, True)
    assert np.array_equal(Oc[:, :, 0, :], V[:, :, 0, :].astype(np.float64)), "causal row 0 == V[0]"
    for i in range(6):
        On = _O(lib, Q[:, :, i:i + 1], K[:, :, :i + 1], V[:, :, :i + 1], 0.8, False)
        assert np.allclose(Oc[:, :, i:i + 1], On, atol=1e-13), f"causal row {i} == prefix"


def pin_single_key(lib):
    """S_k = 1: the only weight is 1, so every row is V[0]."""
    Q, K, V = _rand((2, 1, 4, 3), 16), _rand((2, 1, 1, 3), 17), _rand((2, 1, 1, 5), 18)
    for causal in (False, True):
        O = _O(lib, Q, K, V, 1.3, causal)
        assert np.allclose(O, np.broadcast_to(V.astype(np.float64), O.shape), atol=0)


def pin_logistic(lib):
    """D_qk = 1, S_k = 2: weight of key 0 is the logistic sigma(scale*q*(k0-k1)) (textbook softmax of two)."""
    q = np.array([0.5, -1.25, 2.0, 0.0, 3.5], np.float32).reshape(1, 1, 5, 1)
    k = np.array([0.75, -0.5], np.float32).reshape(1, 1, 2, 1)
    v = np.array([[1.0, -2.0, 0.5], [3.0, 4.0, -1.5]], np.float32).reshape(1, 1, 2, 3)
    scale = float(np.float32(0.625))
    O = _O(lib, q, k, v, scale, False)
    for i in range(5):
        w0 = 1.0 / (1.0 + math.exp(-scale * float(q[0, 0, i, 0]) * (0.75 - (-0.5))))
        expect = w0 * v[0, 0, 0].astype(np.float64) + (1.0 - w0) * v[0, 0, 1].astype(np.float64)
        assert np.allclose(O[0, 0, i], expect, atol=1e-14), f"row {i}"


def pin_hand_rows(lib):
    """Two rows of the accy worked example, derived by hand from the definition.

    Batch 0, query 0: q = (1, 0); keys (1,0), (0,1), (1,1) give dots 1, 0, 1, so with
    c = scale the weights are e^c, 1, e^c over 2e^c + 1 and, with V rows (1,0), (0,2),
    (3,1), O = (4 e^c, 2 + e^c) / (2 e^c + 1).
    Batch 1, query 0: q = (1, 1); keys (0.5,-1), (1,2), (-1,1) give dots -0.5, 3, 0;
    V rows (-1,1), (2,0), (0,4): O = (-e^{-c/2} + 2 e^{3c}, e^{-c/2} + 4) / (e^{-c/2} + e^{3c} + 1).
    """
    ex = _worked_example()
    Q, K, V, c = ex["Q"], ex["K"], ex["V"], ex["scale"]
    O = _O(lib, Q, K, V, c, False)
    e = math.exp(c)
    assert np.allclose(O[0, 0, 0], [4 * e / (2 * e + 1), (2 + e) / (2 * e + 1)], atol=1e-14)
    a, b = math.exp(-c / 2), math.exp(3 * c)
    den = a + b + 1
    assert np.allclose(O[1, 0, 0], [(-a + 2 * b) / den, (a + 4) / den], atol=1e-14)


def pin_shift_invariance(lib):
    """Adding the same constant to every score of a row leaves O unchanged.

    Realised by appending one feature: Q gets a per-row value t_i, K gets the
    constant 1, so row i's scores all move by scale * t_i.
    """
    Q, K, V = _rand((1, 2, 5, 4), 19), _rand((1, 2, 7, 4), 20), _rand((1, 2, 7, 3), 21)
    t = _rand((1, 2, 5, 1), 22, sigma=3.0)
    Q2 = np.concatenate([Q, t], axis=3)
    K2 = np.concatenate([K, np.ones((1, 2, 7, 1), np.float32)], axis=3)
    for causal in (False, True):
        assert np.allclose(_O(lib, Q, K, V, 0.6, causal), _O(lib, Q2, K2, V, 0.6, causal), atol=1e-12)


def pin_peaky(lib):
    """One key's score above all others by >= 60 gives that key's V row (to e^-60); large scores stay finite."""
    S = 6
    K = np.eye(S, dtype=np.float32).reshape(1, 1, S, S)
    V = _rand((1, 1, S, 3), 23)
    sel = np.array([3, 0, 5, 1, 4, 2])
    Q = np.zeros((1, 1, S, S), np.float32)
    Q[0, 0, np.arange(S), sel] = 100.0          # score 100*scale on the selected key, 0 elsewhere
    O = _O(lib, Q, K, V, 1.0, False)
    assert np.allclose(O[0, 0], V[0, 0, sel].astype(np.float64), atol=1e-12), "selector rows"
    Q[0, 0, np.arange(S), sel] = 3000.0          # exp(3000) overflows without the max shift
    O = _O(lib, Q, K, V, 1.0, False)
    assert np.all(np.isfinite(O)) and np.allclose(O[0, 0], V[0, 0, sel].astype(np.float64), atol=1e-12)


def pin_convexity(lib):
    """Each O[i, e] lies within [min_j V[j, e], max_j V[j, e]] over the allowed keys."""
    Q, K, V = _rand((1, 3, 9, 4), 24, 3.0), _rand((1, 3, 9, 4), 25), _rand((1, 3, 9, 5), 26)
    for causal in (False, True):
        O = _O(lib, Q, K, V, 1.0, causal)
        for i in range(9):
            n = i + 1 if causal else 9
            lo = V[:, :, :n].min(axis=2).astype(np.float64) - 1e-12
            hi = V[:, :, :n].max(axis=2).astype(np.float64) + 1e-12
            assert np.all(O[:, :, i] >= lo) and np.all(O[:, :, i] <= hi), f"row {i}"


def pin_selector_unequal_dims(lib):
    """D_qk != D_v and S_q != S_k: a one-hot query row picks exactly one key's V row.

    Catches a transposed Q/K operand or a V indexed by anything but (key, e).
    """
    S_q, S_k, D_qk, D_v = 4, 6, 6, 3
    K = np.eye(S_k, D_qk, dtype=np.float32)[None, None]
    V = _rand((1, 1, S_k, D_v), 27)
    sel = np.array([5, 2, 0, 3])
    Q = np.zeros((1, 1, S_q, D_qk), np.float32)
    Q[0, 0, np.arange(S_q), sel] = 80.0
    O = _O(lib, Q, K, V, 1.0, False)
    assert np.allclose(O[0, 0], V[0, 0, sel].astype(np.float64), atol=1e-12)


def pin_heads_independent(lib):
    """Each (b, h) slice only sees its own K and V: changing one head's K/V changes only that head."""
    Q, K, V = _rand((2, 3, 4, 3), 28), _rand((2, 3, 5, 3), 29), _rand((2, 3, 5, 2), 30)
    O1 = _O(lib, Q, K, V, 0.5, False)
    K2, V2 = K.copy(), V.copy()
    K2[1, 2] += 1.5
    V2[1, 2] -= 2.0
    O2 = _O(lib, Q, K2, V2, 0.5, False)
    changed = np.abs(O1 - O2).max(axis=(2, 3)) > 1e-9
    expect = np.zeros((2, 3), bool)
    expect[1, 2] = True
    assert np.array_equal(changed, expect)
    # and a head computed alone equals the same head inside the batch
    Oh = _O(lib, Q[1:2, 2:3], K[1:2, 2:3], V[1:2, 2:3], 0.5, False)
    assert np.array_equal(Oh[0, 0], O1[1, 2])


def pin_bf16_widening(lib):
    """bf16 inputs are widened exactly: the bf16 run equals the f32 run on the same (bf16-exact) values."""
    Q, K, V = _rand((1, 2, 5, 4), 31), _rand((1, 2, 6, 4), 32), _rand((1, 2, 6, 3), 33)
    qb, kb, vb = (to_bf16_bits(x) for x in (Q, K, V))
    widen = lambda b: (b.astype(np.uint32) << 16).view(np.float32)
    O16 = _O(lib, qb, kb, vb, 0.5, True)
    O32 = _O(lib, widen(qb), widen(kb), widen(vb), 0.5, True)
    assert np.array_equal(O16, O32)


def pin_longdouble(lib):
    """fp64 oracle agrees with the long-double brute force (no max shift) to 1e-12 on tiny random inputs."""
    rng = np.random.default_rng(34)
    for t in range(12):
        B, H = rng.integers(1, 3, size=2)
        S_q, S_k, D_qk, D_v = rng.integers(1, 9, size=4)
        causal = bool(t % 2)
        Q, K, V = make_qkv(int(B), int(H), int(S_q), int(S_k), int(D_qk), int(D_v), "f32", seed=100 + t)
        scale = float(np.float32(1.0 / math.sqrt(D_qk)))
        O = _O(lib, Q, K, V, scale, causal)
        L = oracle.attn_fwd_longdouble(Q, K, V, scale, causal, lib=lib).astype(np.float64)
        assert np.abs(O - L).max() <= 1e-12, f"case {t}"


def _worked_example():
    with open(os.path.join(GOLDEN, "accy_worked_example.json")) as f:
        g = json.load(f)
    B, S_q, S_k, D, Dv = g["batch"], g["queries"], g["keys"], g["qk"], g["value"]
    Q = np.array(g["query"], np.float32).reshape(B, 1, S_q, D)
    K = np.array(g["key"], np.float32).reshape(B, 1, S_k, D)
    V = np.array(g["value_rows"], np.float32).reshape(B, 1, S_k, Dv)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    return {"Q": Q, "K": K, "V": V, "scale": scale, "tol": g["tolerance_abs"]}


def _page_cpu_routine_f32(Q, K, V, scale):
    """The accy page's CPU check routine, restated in f32 numpy: scores, max from -inf, exp-sum, weighted sum."""
    B, _, S_q, D = Q.shape
    S_k, Dv = V.shape[2], V.shape[3]
    out = np.zeros((B, 1, S_q, Dv), np.float32)
    s32 = np.float32(scale)
    for b in range(B):
        for i in range(S_q):
            scores = np.zeros(S_k, np.float32)
            mx = np.float32(-np.inf)
            for j in range(S_k):
                dot = np.float32(0)
                for d in range(D):
                    dot = np.float32(dot + Q[b, 0, i, d] * K[b, 0, j, d])
                scores[j] = np.float32(dot * s32)
                mx = max(mx, scores[j])
            den = np.float32(0)
            for j in range(S_k):
                den = np.float32(den + np.exp(np.float32(scores[j] - mx)))
            for e in range(Dv):
                acc = np.float32(0)
                for j in range(S_k):
                    w = np.float32(np.exp(np.float32(scores[j] - mx)) / den)
                    acc = np.float32(acc + w * V[b, 0, j, e])
                out[b, 0, i, e] = acc
    return out


def pin_worked_example(lib):
    """accy worked example (B=2, S_q=2, S_k=3, D=2): oracle vs the page's f32 CPU routine within the page's 1e-4."""
    ex = _worked_example()
    O = _O(lib, ex["Q"], ex["K"], ex["V"], ex["scale"], False)
    ref = _page_cpu_routine_f32(ex["Q"], ex["K"], ex["V"], ex["scale"])
    assert np.abs(O - ref).max() <= ex["tol"]


def pin_rows_match_full(lib):
    """The sampled-rows entry point returns exactly the rows of the full computation."""
    Q, K, V = make_qkv(2, 3, 9, 7, 5, 4, "bf16", seed=35)
    full = _O(lib, Q, K, V, 0.3, True)
    rows = np.array([[0, 0, 0], [1, 2, 8], [0, 1, 4], [1, 0, 3]])
    got = oracle.attn_rows(Q, K, V, 0.3, True, rows, nthreads=2, lib=lib)
    assert np.array_equal(got, full[rows[:, 0], rows[:, 1], rows[:, 2]])


def pin_shape_convention():
    """accy page, specialization test for 3x2x4x5x3: element counts Q 30, K 60, V 36, O 18 (H = 1)."""
    assert element_counts(3, 1, 2, 4, 5, 3) == (30, 60, 36, 18)


# ---- the general form: grouped heads, offset causal, windows, log-sum-exp ---------------------

def _G(lib, Q, K, V, scale, mask="none", offset=0, window=0, lse=False):
    return oracle.attn_general(Q, K, V, scale, mask, offset, window, with_lse=lse, nthreads=2, lib=lib)


def _plain_rows(lib, Q, K, V, scale, i, lo, hi):
    """Non-causal softmax of query row i over keys lo..hi (inclusive), every (b, h)."""
    return _O(lib, Q[:, :, i:i + 1], K[:, :, lo:hi + 1], V[:, :, lo:hi + 1], scale, False)


def pin_offset_causal_prefix(lib):
    """Offset causal: query i at key position i + o sees keys 0..min(i + o, S_k - 1).

    The VeriTile coverage table's attention_llama causal row gives query block p the key span
    (p + 1) BLOCK_N + start_position: query i reaches key i + start_position.  o = S_k - S_q is
    the bottom-right alignment (the last query sees every key); o >= S_k - 1 allows every key.
    """
    S_q, S_k = 5, 9
    Q, K, V = _rand((1, 2, S_q, 4), 40), _rand((1, 2, S_k, 4), 41), _rand((1, 2, S_k, 3), 42)
    for o in (0, 1, 3, S_k - S_q, 8, 20):
        O = _G(lib, Q, K, V, 0.7, "causal", o)
        for i in range(S_q):
            ref = _plain_rows(lib, Q, K, V, 0.7, i, 0, min(i + o, S_k - 1))
            assert np.allclose(O[:, :, i:i + 1], ref, atol=1e-13), f"offset {o} row {i}"
    assert np.allclose(_G(lib, Q, K, V, 0.7, "causal", S_k - 1), _O(lib, Q, K, V, 0.7, False), atol=1e-13)


def pin_window_recent_keys(lib):
    """Sliding window w, offset o: row i sees keys max(0, i+o-w+1)..min(i+o, S_k-1), the w most recent.

    w = 1 returns V[i + o] exactly; a row whose window lies past the last key has no key and is 0.
    """
    S_q, S_k = 6, 10
    Q, K, V = _rand((1, 2, S_q, 3), 43, 2.0), _rand((1, 2, S_k, 3), 44), _rand((1, 2, S_k, 4), 45)
    for o, w in ((0, 1), (0, 3), (2, 2), (4, 5), (3, 40), (8, 2)):
        O = _G(lib, Q, K, V, 0.9, "window", o, w)
        for i in range(S_q):
            lo, hi = max(0, i + o - w + 1), min(i + o, S_k - 1)
            if lo > hi:
                assert np.all(O[:, :, i] == 0.0), f"window {w} offset {o}: row {i} has no key"
                continue
            ref = _plain_rows(lib, Q, K, V, 0.9, i, lo, hi)
            assert np.allclose(O[:, :, i:i + 1], ref, atol=1e-13), f"window {w} offset {o} row {i}"
            if w == 1:
                assert np.array_equal(O[:, :, i], V[:, :, i + o].astype(np.float64))


def pin_window_complement(lib):
    """Complement of the window: row i sees keys 0..min(i+o-w, S_k-1); rows with i + o < w have none
    (O = 0, LSE = -inf)."""
    S_q, S_k = 7, 8
    Q, K, V = _rand((2, 1, S_q, 3), 46, 2.0), _rand((2, 1, S_k, 3), 47), _rand((2, 1, S_k, 2), 48)
    for o, w in ((0, 1), (0, 3), (1, 4), (5, 2), (0, 9)):
        O, L = _G(lib, Q, K, V, 1.1, "window_complement", o, w, lse=True)
        for i in range(S_q):
            hi = min(i + o - w, S_k - 1)
            if hi < 0:
                assert np.all(O[:, :, i] == 0.0) and np.all(L[:, :, i] == -np.inf), f"row {i} is empty"
                continue
            ref = _plain_rows(lib, Q, K, V, 1.1, i, 0, hi)
            assert np.allclose(O[:, :, i:i + 1], ref, atol=1e-13), f"complement {w} offset {o} row {i}"


def pin_window_split_merges_to_causal(lib):
    """Window and complement split each causal key set in two.  Merging their outputs with their
    log-sum-exps, O = sum_k e^{LSE_k} O_k / sum_k e^{LSE_k} (the continuation case of the
    attention_fwd_triton3 row), gives the offset causal output and LSE = log(e^{LSE_w} + e^{LSE_c})."""
    S = 9
    Q, K, V = _rand((1, 2, S, 4), 49, 2.0), _rand((1, 2, S + 3, 4), 50), _rand((1, 2, S + 3, 3), 51)
    for o, w in ((0, 3), (3, 1), (2, 6), (0, 20)):
        Ow, Lw = _G(lib, Q, K, V, 0.8, "window", o, w, lse=True)
        Oc, Lc = _G(lib, Q, K, V, 0.8, "window_complement", o, w, lse=True)
        M = np.maximum(Lw, Lc)
        ww, wc = np.exp(Lw - M), np.exp(Lc - M)
        Om = (ww[..., None] * Ow + wc[..., None] * Oc) / (ww + wc)[..., None]
        for i in range(S):
            ref = _plain_rows(lib, Q, K, V, 0.8, i, 0, min(i + o, S + 2))
            assert np.allclose(Om[:, :, i:i + 1], ref, atol=1e-12), f"window {w} offset {o} row {i}"
        Lf = np.log(np.exp(Lw - M) + np.exp(Lc - M)) + M
        _, Lcausal = _G(lib, Q, K, V, 0.8, "causal", o, lse=True)
        assert np.allclose(Lf, Lcausal, atol=1e-12)


def pin_lse_closed_forms(lib):
    """LSE_i = log sum_{j in A_i} exp(s_j): scale 0 gives log |A_i|; one key gives its score;
    D_qk = 1, S_k = 2 gives log(e^a + e^b)."""
    Q, K, V = _rand((1, 2, 6, 3), 52), _rand((1, 2, 6, 3), 53), _rand((1, 2, 6, 2), 54)
    _, L = _G(lib, Q, K, V, 0.0, "none", lse=True)
    assert np.allclose(L, math.log(6), atol=1e-14)
    _, L = _G(lib, Q, K, V, 0.0, "causal", lse=True)
    assert np.allclose(L, np.log(np.arange(1, 7))[None, None, :], atol=1e-14)
    _, L = _G(lib, Q, K, V, 0.0, "window", 0, 2, lse=True)
    assert np.allclose(L, np.log(np.minimum(np.arange(1, 7), 2))[None, None, :], atol=1e-14)
    q = np.array([0.5, -1.25, 2.0, 0.0, 3.5], np.float32).reshape(1, 1, 5, 1)
    k = np.array([0.75, -0.5], np.float32).reshape(1, 1, 2, 1)
    v = np.ones((1, 1, 2, 1), np.float32)
    _, L = _G(lib, q, k[:, :, :1], v[:, :, :1], 0.625, "none", lse=True)
    assert np.allclose(L[0, 0], 0.625 * q[0, 0, :, 0].astype(np.float64) * 0.75, atol=1e-14)
    _, L = _G(lib, q, k, v, 0.625, "none", lse=True)
    a, b = 0.625 * q[0, 0, :, 0].astype(np.float64) * 0.75, 0.625 * q[0, 0, :, 0].astype(np.float64) * -0.5
    assert np.allclose(L[0, 0], np.log(np.exp(a) + np.exp(b)), atol=1e-14)


def pin_grouped_heads_expand(lib):
    """H_kv < H: the result equals multi-head attention with each key/value head repeated for its
    H / H_kv query heads (query head h reads head h // (H / H_kv)); H_kv = 1 is multi-query."""
    Q = _rand((2, 6, 5, 4), 55)
    for H_kv in (3, 2, 1):
        K, V = _rand((2, H_kv, 7, 4), 56 + H_kv), _rand((2, H_kv, 7, 3), 60 + H_kv)
        rep = 6 // H_kv
        Kx, Vx = np.repeat(K, rep, axis=1), np.repeat(V, rep, axis=1)
        for mask in ("none", "causal"):
            O = _G(lib, Q, K, V, 0.6, mask)
            assert np.allclose(O, _O(lib, Q, Kx, Vx, 0.6, mask == "causal"), atol=1e-13), f"H_kv {H_kv} {mask}"


def pin_general_rows_match_full(lib):
    """The general form's sampled rows equal the same rows of its full result (grouped heads, window)."""
    Q, K, V = make_qkv(2, 4, 9, 11, 5, 4, "bf16", seed=64)
    K, V = K[:, :2].copy(), V[:, :2].copy()
    full, L = _G(lib, Q, K, V, 0.3, "window", 2, 4, lse=True)
    rows = np.array([[0, 0, 0], [1, 3, 8], [0, 1, 4], [1, 2, 3]])
    got, Lr = oracle.attn_general(Q, K, V, 0.3, "window", 2, 4, rows=rows, with_lse=True, nthreads=2, lib=lib)
    assert np.array_equal(got, full[rows[:, 0], rows[:, 1], rows[:, 2]])
    assert np.array_equal(Lr, L[rows[:, 0], rows[:, 1], rows[:, 2]])


def pin_general_longdouble(lib):
    """The general form agrees with its long-double brute force (no max shift) on random tiny cases,
    O to 1e-12 and LSE to 1e-12 (empty rows: both 0 and -inf)."""
    rng = np.random.default_rng(65)
    masks = list(oracle.MASKS)
    for t in range(24):
        B = int(rng.integers(1, 3))
        H_kv = int(rng.integers(1, 3))
        H = H_kv * int(rng.integers(1, 4))
        S_q, S_k, D_qk, D_v = (int(x) for x in rng.integers(1, 9, size=4))
        mask = masks[t % 4]
        offset, window = int(rng.integers(0, 6)), int(rng.integers(1, 6))
        Q, _, _ = make_qkv(B, H, S_q, S_k, D_qk, D_v, "f32", seed=200 + t)
        _, K, V = make_qkv(B, H_kv, S_q, S_k, D_qk, D_v, "f32", seed=300 + t)
        scale = float(np.float32(1.0 / math.sqrt(D_qk)))
        O, L = _G(lib, Q, K, V, scale, mask, offset, window, lse=True)
        Ol, Ll = oracle.attn_general_longdouble(Q, K, V, scale, mask, offset, window, lib=lib)
        assert np.abs(O - Ol.astype(np.float64)).max() <= 1e-12, f"case {t}"
        Ll = Ll.astype(np.float64)
        assert np.array_equal(np.isinf(L), np.isinf(Ll)), f"case {t}: empty rows"
        fin = np.isfinite(L)
        assert np.abs(L[fin] - Ll[fin]).max(initial=0.0) <= 1e-12, f"case {t}"


# Pins that do not compare the oracle with its own long-double brute force.
INDEPENDENT_PINS = [
    pin_ones_value, pin_identical_keys_mean, pin_scale_zero_mean, pin_key_permutation,
    pin_causal_row0_and_prefix, pin_single_key, pin_logistic, pin_hand_rows, pin_shift_invariance,
    pin_peaky, pin_convexity, pin_selector_unequal_dims, pin_heads_independent, pin_bf16_widening,
    pin_worked_example, pin_rows_match_full,
    pin_offset_causal_prefix, pin_window_recent_keys, pin_window_complement, pin_window_split_merges_to_causal,
    pin_lse_closed_forms, pin_grouped_heads_expand, pin_general_rows_match_full,
]
ALL_PINS = INDEPENDENT_PINS + [pin_longdouble, pin_general_longdouble]
