"""Host logic of bench.py on CPU: flop counts, the L2-flush decision and the parity report of the
CPU-baseline sample (the oracle's own output must pass, a perturbed one must fail)."""

from __future__ import annotations

import dataclasses

import numpy as np

import bench
import oracle
import synth


def test_flop_counts_follow_the_metric_and_the_kept_pairs():
    w = synth.WORKLOADS["bf16_causal_8k_peaky"]
    assert bench.workload_flops(w, True) == 4.0 * 8 * 16 * 8192 * 8192 * 128 / 2
    assert bench.workload_flops(w, False) == 4.0 * 8 * 16 * 8192 * 8192 * 128
    m = dataclasses.replace(synth.WORKLOADS["bf16_window_1k_8k"], B=1, H=1, S_q=40, S_k=50, D_qk=8, D_v=4,
                            window=7, offset=3)
    pairs = sum(1 for i in range(40) for j in range(50) if i + 3 - 7 < j <= i + 3)
    assert bench.workload_flops(m, True) == 2.0 * pairs * (8 + 4)


def test_l2_flush_decision():
    l2 = 126 << 20
    assert bench.needs_l2_flush(100 << 20, 33 << 20, l2)          # 2k causal: flushed
    assert not bench.needs_l2_flush(805 << 20, 268 << 20, l2)     # 8k causal: inputs larger than L2
    assert not bench.needs_l2_flush(2 * l2, 0, l2)


def _small():
    w = dataclasses.replace(synth.WORKLOADS["bf16_causal_2k"], B=1, H=2, S_q=192, S_k=192, name="small")
    return w, synth.make_workload(w)


def _oracle_slice(w, q, k, v):
    def get(b, h):
        rows = np.stack([np.full(w.S_q, b), np.full(w.S_q, h), np.arange(w.S_q)], axis=1)
        return np.asarray(oracle.attn_rows(q, k, v, w.scale, True, rows), dtype=np.float64).reshape(w.S_q, w.D_v)
    return get


def test_parity_report_passes_the_exact_output():
    w, (q, k, v) = _small()
    r = bench.cpu_oracle_sample(w, q, k, v, True, target_s=0.2, max_slices=2, gpu_slice=_oracle_slice(w, q, k, v))
    par = r["parity"]
    assert par["pass"] and par["max_abs"] == 0.0 and par["rel_fro"] == 0.0 and par["slices"] >= 1
    assert r["kind"] == "oracle" and r["cores"] >= 1


def test_parity_report_fails_a_perturbed_output():
    w, (q, k, v) = _small()
    exact = _oracle_slice(w, q, k, v)
    r = bench.cpu_oracle_sample(w, q, k, v, True, target_s=0.2, max_slices=2,
                                gpu_slice=lambda b, h: exact(b, h) + 0.03)
    par = r["parity"]
    assert not par["pass"] and abs(par["max_abs"] - 0.03) < 1e-12
