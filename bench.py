#!/usr/bin/env python
"""Benchmark of the attention forward on GB300: one JSON line on stdout (rank 0).

A step is one vt_attn_fwd call over the whole workload (default: B=8, H=16,
S_q=S_k=8192, D=128, bf16, causal, Q ~ N(0, 4^2), K, V ~ N(0, 1), seed 4).  The masked and
grouped-head workloads (--workload bf16_gqa_causal_8k, bf16_prefill_on_cache_8k,
bf16_window_1k_8k, bf16_chunk_on_cache_32k) call vt_attn_fwd_general instead and count
2*(D_qk+D_v) flops per (query, key) pair their mask keeps.  Split-KV shares are the library's
choice (vt_attn_splitkv_choose; --split N overrides): 1 for the default workload, more where
the query blocks do not fill the SMs, in which case a step also runs the merge kernel.

  value        TFLOP/s over the timed steps, inputs resident in HBM (flops = 4*B*H*S_q*S_k*D,
               halved for causal; 2*B*H*S_q*S_k*(D_qk+D_v) in general), CUDA events on the
               launching stream, max over ranks; inputs (805 MB) are larger than L2.  A
               workload whose inputs and output are under twice the L2 size gets an L2 flush
               before every timed step (outside the step's events) and is timed from the
               per-step events; config.l2 says which.
  e2e          the same metric with every step's host->device copies of Q, K, V from pinned
               memory and its device->host copy of O inside the timed region (steps pipelined
               over copy-in / compute / copy-out streams with double-buffered device tensors).
  roofline     the kernel against the measured dense bf16 (or derived tf32) tensor peak.
  cpu_baseline the fp64 CPU oracle on a bounded sample of the same workload (rank 0 only).

--impl reference times that oracle as the reference arm.  Under torchrun each rank
runs its own copy of the workload on its own GPU (replicas, weak scaling; no
collective on the data path).
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "attention fwd TFLOP/s (causal-adjusted) and % of GB300 dense tensor peak"
DEFAULT_WORKLOAD = "bf16_causal_8k_peaky"
# device code of the bf16 kernel the default workload runs (its traffic figure is tied to these)
KERNEL_SOURCES = [os.path.join(ROOT, "scaled_dot_product_vt_gb300", "csrc", f)
                  for f in ("vt_attn_bf16_2q.cuh", "vt_attn_common.cuh", "vt_ptx.cuh")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_fwd_traffic.json")
# nominal dense tf32 : bf16 tensor ratio (1.1 : 2.25 PFLOP/s), applied to the measured bf16 peak; the issue-rate
# probe of tcgen05.mma measured kind::tf32 at exactly half of kind::f16 per clock (4096 vs 8192 flop/clk/SM at
# every N), which the line reports beside it as peak_probe_ratio
TF32_OVER_BF16 = 1.1 / 2.25
TF32_OVER_BF16_PROBE = 0.5


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"bf16": float(p["bf16_tflops"]), "bf16_sustained": float(p["bf16_tflops_sustained"]),
                "hbm": float(p["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


def load_traffic(workload: str):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on the current kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("kernel_source_hash") != kernel_source_hash() or t.get("workload") != workload:
        return None
    return t.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None
        self.first = threading.Event()

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())
            self.first.set()
        self.first.set()

    def wait_first(self, timeout: float = 15.0):
        """Block until nvidia-smi has printed its first sample: its start-up (NVML initialisation)
        can hold driver locks for seconds, which must not fall inside a timed region."""
        if self.proc is not None:
            self.first.wait(timeout)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def workload_flops(w, causal: bool) -> float:
    """Flops of one step: the metric's convention for plain workloads, kept pairs for masked ones."""
    return w.flops_masked() if w.mask else w.flops(causal)


def mode_of(w, causal: bool) -> str:
    if not w.mask:
        return f"causal={causal}"
    extra = f", offset {w.offset}" if w.offset else ""
    extra += f", window {w.window}" if w.mask.startswith("window") else ""
    heads = f", H_kv {w.kv_heads}" if w.kv_heads != w.H else ""
    return f"mask {w.mask}{extra}{heads}"


def needs_l2_flush(in_bytes: int, out_bytes: int, l2_bytes: int) -> bool:
    """True when a step's inputs and output could stay in L2 between timed steps (under twice its size)."""
    return in_bytes + out_bytes < 2 * l2_bytes


# parity bars of the element types: (max abs, relative Frobenius or None)
TOLERANCE = {"bf16": (2e-2, 1e-2), "f32": (5e-3, None)}


def cpu_oracle_sample(w, q, k, v, causal: bool, target_s: float = 12.0, max_slices: int = 32, gpu_slice=None):
    """Time the fp64 oracle on whole (b, h) slices of the workload until ~target_s seconds have passed.
    With gpu_slice(b, h) -> the GPU's output of that slice (fp64), also return the parity of the sampled
    slices (compared outside the timed part)."""
    import oracle
    nthreads = oracle.default_threads()
    rows_per_slice = w.S_q
    done_flops, t_total, slices = 0.0, 0.0, 0
    max_abs, err2, ref2 = 0.0, 0.0, 0.0
    for s in range(max_slices):
        b, h = divmod(s, w.H)
        b %= w.B
        rows = np.stack([np.full(rows_per_slice, b), np.full(rows_per_slice, h), np.arange(rows_per_slice)], axis=1)
        t0 = time.perf_counter()
        if w.mask:
            ref = oracle.attn_general(q, k, v, w.scale, w.mask, w.offset, w.window, rows=rows, nthreads=nthreads)
        else:
            ref = oracle.attn_rows(q, k, v, w.scale, causal, rows, nthreads=nthreads)
        t_total += time.perf_counter() - t0
        if gpu_slice is not None:
            d = gpu_slice(b, h) - np.asarray(ref, dtype=np.float64).reshape(w.S_q, w.D_v)
            max_abs = max(max_abs, float(np.abs(d).max()))
            err2 += float((d * d).sum())
            ref2 += float((np.asarray(ref, dtype=np.float64) ** 2).sum())
        done_flops += workload_flops(w, causal) / (w.B * w.H)
        slices += 1
        if t_total >= target_s:
            break
    out = {"value": done_flops / t_total / 1e12, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
           "sample": f"{slices} whole (b,h) slice(s) of {w.name} ({w.S_q} rows each, {mode_of(w, causal)}), "
                     f"{t_total:.1f} s fp64 on {nthreads} host threads"}
    if gpu_slice is not None:
        tol_abs, tol_rel = TOLERANCE[w.dtype]
        rel = math.sqrt(err2 / ref2) if ref2 > 0 else 0.0
        out["parity"] = {"slices": slices, "max_abs": max_abs, "rel_fro": rel, "tol_max_abs": tol_abs,
                         "tol_rel_fro": tol_rel,
                         "pass": max_abs <= tol_abs and (tol_rel is None or rel <= tol_rel)}
    return out


def run_reference(args, w, causal):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    q, k, v = synth.make_workload(w)
    import oracle
    nthreads = oracle.default_threads()
    rows_per_step = max(1, min(w.S_q, int(args.ref_rows)))
    # each step: the oracle over `rows_per_step` rows spread over one (b, h) slice
    step_rows = np.linspace(0, w.S_q - 1, rows_per_step).astype(np.int64)
    if w.mask:
        step_flops = float(w.keys_per_row()[step_rows].sum()) * 2.0 * (w.D_qk + w.D_v)
    elif causal:
        step_flops = float(sum(2.0 * (i + 1) * (w.D_qk + w.D_v) for i in step_rows))
    else:
        step_flops = 2.0 * rows_per_step * w.S_k * (w.D_qk + w.D_v)
    times = []
    for it in range(args.warmup + args.steps):
        b, h = divmod(it % (w.B * w.H), w.H)
        rows = np.stack([np.full(len(step_rows), b), np.full(len(step_rows), h), step_rows], axis=1)
        t0 = time.perf_counter()
        if w.mask:
            oracle.attn_general(q, k, v, w.scale, w.mask, w.offset, w.window, rows=rows, nthreads=nthreads)
        else:
            oracle.attn_rows(q, k, v, w.scale, causal, rows, nthreads=nthreads)
        dt = time.perf_counter() - t0
        if it >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = step_flops * len(times) / total / 1e12
    sample = (f"{rows_per_step} query rows evenly spread over one (b,h) slice of {w.name} per step "
              f"({mode_of(w, causal)}), fp64 on {nthreads} host threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / len(times) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "S_q": w.S_q, "S_k": w.S_k, "D_qk": w.D_qk,
                   "D_v": w.D_v, "causal": causal, "io_dtype": w.dtype, "mode": mode_of(w, causal)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main() -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--causal", type=int, default=None, help="override the workload's mode (0/1)")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's B (smaller profiling cases)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-rows", type=int, default=512, help="reference arm: query rows per step")
    ap.add_argument("--split", default="auto",
                    help="split-KV shares: 'auto' (the library's vt_attn_splitkv_choose) or a count")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")

    w = synth.WORKLOADS[args.workload]
    if args.batch is not None:
        w = dataclasses.replace(w, B=args.batch, name=f"{w.name}_B{args.batch}")
    causal = bool(w.causal[-1] if args.causal is None else args.causal)
    if args.impl == "reference":
        return run_reference(args, w, causal)

    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import scaled_dot_product_vt_gb300 as vt
    vt.load()
    vt_dtype = vt.VT_BF16 if w.dtype == "bf16" else vt.VT_F32
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    q, k, v = synth.make_workload(w)

    def pinned(a):
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).pin_memory()
        return t.view(tdt) if a.dtype == np.uint16 else t

    hq, hk, hv = pinned(q), pinned(k), pinned(v)
    Q, K, V = (t.to(dev) for t in (hq, hk, hv))
    O = torch.empty((w.B, w.H, w.S_q, w.D_v), dtype=tdt, device=dev)
    hO = torch.empty(O.shape, dtype=tdt).pin_memory()
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    flops = workload_flops(w, causal)
    mask = vt.vt_attn_mask(vt.MASKS[w.mask], 0, w.offset, w.window) if w.mask else None
    n_split = (vt.vt_attn_splitkv_choose(w.B, w.H, w.S_q, w.S_k, int(causal), vt_dtype) if args.split == "auto"
               else int(args.split))
    workspace, ws_bytes = None, 0
    if n_split > 1:
        ws_bytes = vt.vt_attn_splitkv_workspace_size(w.B, w.H, w.S_q, w.D_v, n_split)
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        if mask is None:
            mask = vt.vt_attn_mask(vt.MASKS["causal" if causal else "none"], 0, 0, 0)

    def call(q_, k_, v_, o_, stream_handle):
        """One forward through the C ABI: vt_attn_fwd, or the general entry point for masked,
        grouped-head or split-KV runs (its launches run on one stream, so one workspace serves)."""
        if mask is None:
            return vt.vt_attn_fwd(q_.data_ptr(), k_.data_ptr(), v_.data_ptr(), o_.data_ptr(), w.B, w.H, w.S_q,
                                  w.S_k, w.D_qk, w.D_v, w.scale, int(causal), vt_dtype, stream_handle)
        return vt.vt_attn_fwd_general(q_.data_ptr(), q_.stride()[:3], k_.data_ptr(), k_.stride()[:3],
                                      v_.data_ptr(), v_.stride()[:3], o_.data_ptr(), o_.stride()[:3], None, w.B,
                                      w.H, w.kv_heads, w.S_q, w.S_k, w.D_qk, w.D_v, w.scale, vt_dtype, mask, n_split,
                                      workspace.data_ptr() if workspace is not None else None, ws_bytes, None,
                                      stream_handle)

    def step():
        rc = call(Q, K, V, O, sh)
        if rc != 0:
            raise RuntimeError(f"vt_attn_fwd: {vt.vt_status_str(rc)}")

    # A working set that L2 could hold between steps is flushed before every timed step (a write of
    # twice the L2 size, outside the step's events), and such a run is timed from the per-step events.
    in_bytes = hq.numel() * hq.element_size() + hk.numel() * hk.element_size() + hv.numel() * hv.element_size()
    out_bytes = hO.numel() * hO.element_size()
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (129 << 20))
    flush_buf = torch.empty(2 * l2_bytes // 4, dtype=torch.int32, device=dev) if needs_l2_flush(
        in_bytes, out_bytes, l2_bytes) else None

    for _ in range(args.warmup):
        step()
    st = vt.vt_last_device_status(sh)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {vt.vt_status_str(st)}")

    # ---- kernel-only timed region: inputs resident in HBM
    clocks = ClockSampler(torch.cuda.current_device() if world == 1 else local)
    clocks.start()
    clocks.wait_first()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        if flush_buf is not None:
            flush_buf.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    st = vt.vt_last_device_status(sh)
    if st != 0:
        raise RuntimeError(f"device status after timed steps: {vt.vt_status_str(st)}")
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = t_start.elapsed_time(t_end) if flush_buf is None else sum(launch_ms)
    total_ms = max_over_ranks(total_ms, world, dev)

    # ---- end to end through the public API: every step copies its own inputs from pinned host
    # memory to the device, runs the forward and reads its result back.  Steps are pipelined over
    # three streams (copy in, compute, copy out) with double-buffered device tensors, so step i's
    # copies overlap the kernels of its neighbours; every copy stays inside the timed region.
    dev_sets = [(Q, K, V, O), tuple(torch.empty_like(t) for t in (Q, K, V, O))]
    host_out = [hO, torch.empty(O.shape, dtype=tdt).pin_memory()]
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        b = i % 2
        q_, k_, v_, o_ = dev_sets[b]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_cmp[b])  # buffer set b is free once step i-2's kernel is done
            q_.copy_(hq, non_blocking=True)
            k_.copy_(hk, non_blocking=True)
            v_.copy_(hv, non_blocking=True)
            ev_in[b].record(s_in)
        s_cmp.wait_event(ev_in[b])
        if i >= 2:
            s_cmp.wait_event(ev_out[b])  # O_b is free once step i-2's result has been read back
        rc = call(q_, k_, v_, o_, s_cmp.cuda_stream)
        if rc != 0:
            raise RuntimeError(f"vt_attn_fwd: {vt.vt_status_str(rc)}")
        ev_cmp[b].record(s_cmp)
        s_out.wait_event(ev_cmp[b])
        with torch.cuda.stream(s_out):
            host_out[b].copy_(o_, non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(2):  # untimed: warm the streams and the second buffer set
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e2e_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    barrier(world)
    torch.cuda.synchronize(dev)
    e2e_ev[0].record(s_in)
    for i in range(args.steps):
        e2e_step(i)
    e2e_ev[1].record(s_out)  # after the last read-back, which follows every earlier operation
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(e2e_ev[0].elapsed_time(e2e_ev[1]), world, dev)
    for b in range(2):
        st = vt.vt_last_device_status(s_cmp.cuda_stream)
        if st != 0:
            raise RuntimeError(f"device status after e2e steps: {vt.vt_status_str(st)}")

    peaks = load_peaks()
    peak = peaks["bf16"] if w.dtype == "bf16" else peaks["bf16"] * TF32_OVER_BF16
    value = world * flops * args.steps / (total_ms * 1e-3) / 1e12
    per_launch_ms = statistics.mean(launch_ms)
    achieved = flops / (per_launch_ms * 1e-3) / 1e12
    line = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            # O holds the result of the timed steps (the end-to-end steps rewrote it from the same inputs)
            cpu = cpu_oracle_sample(w, q, k, v, causal, target_s=args.cpu_seconds,
                                    gpu_slice=lambda b, h: O[b, h].double().cpu().numpy())
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "S_q": w.S_q, "S_k": w.S_k, "D_qk": w.D_qk,
                       "D_v": w.D_v, "causal": causal, "mode": mode_of(w, causal), "H_kv": w.kv_heads,
                       "n_split": n_split,
                       "flops_per_step": flops,
                       "l2": (f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB read per step)" if flush_buf is None
                              else f"L2 flushed before every timed step ({in_bytes / 1e6:.0f} MB of inputs, "
                                   f"{l2_bytes / 1e6:.0f} MB L2); value from the per-step events"),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "peak_frac": value / world / peak,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": load_traffic(w.name),
                         "peak_source": (f"{peaks['source']} bf16 burst" if w.dtype == "bf16"
                                         else f"{peaks['source']} bf16 burst x nominal tf32/bf16 ratio"),
                         "kernel": "vt::attn_fwd_bf16_2q_kernel" if w.dtype == "bf16" else "vt::attn_fwd_f32_2q_kernel",
                         "peak_probe_ratio": None if w.dtype == "bf16" else peaks["bf16"] * TF32_OVER_BF16_PROBE,
                         "launch_ms": per_launch_ms,  # one call: the attention kernel (+ the merge if split)
                         "merge_kernel": "vt::attn_merge_kernel" if n_split > 1 else None},
            "cpu_baseline": cpu,
            "e2e": {"value": world * flops * args.steps / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
                    "ms_per_step": e2e_ms / args.steps, "pipelined": True},
            # kernel-only timed region: per step and rank one attention launch, plus the merge when split
            "gpu_launches": world * args.steps * (2 if n_split > 1 else 1),
            "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"]},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
