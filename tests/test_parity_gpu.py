"""GPU parity: vt_attn_fwd (through the C ABI) against the fp64 oracle on the same seeded inputs."""

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


def run(q, k, v, scale, causal):
    Q, K, V = to_device(q), to_device(k), to_device(v)
    O = vt.attn_fwd(Q, K, V, scale=scale, causal=causal)
    assert vt.vt_last_device_status() == 0
    return to_host64(O)


# ---------------------------------------------------------------- the five workloads

@pytest.mark.parametrize("name,causal", [
    ("tiny_f32", False), ("mid_f32", False), ("mid_f32", True), ("bf16_causal_2k", True), ("bf16_ragged", False),
])
def test_workload_full(name, causal):
    w = synth.WORKLOADS[name]
    q, k, v = synth.make_workload(w)
    got = run(q, k, v, w.scale, causal)
    ref = oracle.attn_fwd(q, k, v, w.scale, causal)
    check(got, ref, w.dtype, f"{name} causal={causal}")


def sample_rows(w, rng, n_random=48, n_bh=8):
    """Rows at tile edges and ragged ends plus random ones, over a spread of (b, h)."""
    edges = sorted({0, 1, 63, 64, 127, 128, 129, 255, 256, w.S_q // 2, w.S_q - 129, w.S_q - 128, w.S_q - 2,
                    w.S_q - 1})
    rows = []
    bhs = [(0, 0), (w.B - 1, w.H - 1)] + [(int(rng.integers(w.B)), int(rng.integers(w.H))) for _ in range(n_bh - 2)]
    for b, h in bhs:
        for i in edges + [int(x) for x in rng.integers(0, w.S_q, size=n_random)]:
            if 0 <= i < w.S_q:
                rows.append((b, h, i))
    return np.array(sorted(set(rows)), dtype=np.int64)


def test_workload_8k_peaky_sampled():
    """The largest workload at full size, in the bench's launch configuration; sampled rows vs the oracle."""
    w = synth.WORKLOADS["bf16_causal_8k_peaky"]
    q, k, v = synth.make_workload(w)
    got = run(q, k, v, w.scale, True)
    assert np.all(np.isfinite(got))
    rows = sample_rows(w, np.random.default_rng(0))
    ref = oracle.attn_rows(q, k, v, w.scale, True, rows)
    check(got[rows[:, 0], rows[:, 1], rows[:, 2]], ref, "bf16", "8k peaky sampled rows")
    # causal row 0 is V[0] exactly in every head
    assert np.array_equal(got[:, :, 0, :], synth.bf16_bits_to_fp32(v[:, :, 0, :]).astype(np.float64))


def test_workload_8k_peaky_whole_output():
    """The largest workload at full size, every one of its 1.07e9 outputs against the oracle (all 128 (b, h)
    slices; about a minute of the multithreaded fp64 oracle).  Sampled rows once missed 9 values over the
    max abs bar, all in rows that one key dominates."""
    w = synth.WORKLOADS["bf16_causal_8k_peaky"]
    q, k, v = synth.make_workload(w)
    O = vt.attn_fwd(to_device(q), to_device(k), to_device(v), scale=w.scale, causal=True)
    assert vt.vt_last_device_status() == 0
    worst, err2, ref2 = 0.0, 0.0, 0.0
    for b in range(w.B):
        for h in range(w.H):
            rows = np.stack([np.full(w.S_q, b), np.full(w.S_q, h), np.arange(w.S_q)], axis=1)
            ref = np.asarray(oracle.attn_rows(q, k, v, w.scale, True, rows), dtype=np.float64).reshape(w.S_q, w.D_v)
            d = O[b, h].double().cpu().numpy() - ref
            worst = max(worst, float(np.abs(d).max()))
            err2 += float((d * d).sum())
            ref2 += float((ref * ref).sum())
    rel = math.sqrt(err2 / ref2)
    assert worst <= 2e-2, f"max abs error {worst:.4g} over the whole output"
    assert rel <= 1e-2, f"relative Frobenius error {rel:.4g}"


# ---------------------------------------------------------------- edge shapes

EDGE = [
    # B, H, S_q, S_k, D_qk, D_v, causal
    (1, 1, 1, 1, 8, 8, False), (1, 1, 1, 1, 8, 8, True),
    (1, 2, 7, 13, 16, 32, False), (2, 1, 129, 129, 64, 64, True),
    (1, 1, 128, 128, 128, 128, True), (1, 1, 300, 257, 72, 40, False), (1, 1, 300, 257, 72, 40, True),
    (1, 1, 200, 100, 128, 128, True), (1, 1, 100, 300, 32, 48, True), (3, 2, 255, 383, 96, 64, False),
    (1, 1, 129, 1000, 128, 8, False), (1, 1, 5, 130, 120, 128, True), (2, 3, 64, 64, 16, 16, True),
]
EDGE_F32 = [
    (1, 1, 65, 70, 20, 12, False), (1, 1, 65, 70, 20, 12, True), (1, 3, 130, 64, 4, 4, False),
    (1, 1, 37, 37, 20, 20, True), (2, 1, 200, 333, 72, 72, True), (1, 1, 1, 1, 4, 4, False),
    (1, 2, 129, 65, 128, 128, False), (1, 1, 100, 100, 36, 100, True),
]


@pytest.mark.parametrize("shape", EDGE, ids=str)
def test_edge_bf16(shape):
    B, H, S_q, S_k, D_qk, D_v, causal = shape
    q, k, v = synth.make_qkv(B, H, S_q, S_k, D_qk, D_v, "bf16", seed=hash(shape) & 0xFFFF)
    scale = float(np.float32(1 / math.sqrt(D_qk)))
    check(run(q, k, v, scale, causal), oracle.attn_fwd(q, k, v, scale, causal), "bf16", str(shape))


@pytest.mark.parametrize("shape", EDGE_F32, ids=str)
def test_edge_f32(shape):
    B, H, S_q, S_k, D_qk, D_v, causal = shape
    q, k, v = synth.make_qkv(B, H, S_q, S_k, D_qk, D_v, "f32", seed=hash(shape) & 0xFFFF)
    scale = float(np.float32(1 / math.sqrt(D_qk)))
    check(run(q, k, v, scale, causal), oracle.attn_fwd(q, k, v, scale, causal), "f32", str(shape))


@pytest.mark.parametrize("scale", [0.0, -0.3, 2.5])
@pytest.mark.parametrize("D", [64, 128])
def test_unusual_scales(scale, D):
    """Zero and negative scales take the kernel variants that scale the scores before the exponent;
    D = 64 runs the score-ring kernel, D = 128 the two-tile kernel."""
    q, k, v = synth.make_qkv(1, 2, 150, 140, D, D, "bf16", seed=11)
    for causal in (False, True):
        check(run(q, k, v, scale, causal), oracle.attn_fwd(q, k, v, scale, causal), "bf16", f"scale={scale} D={D}")


def _tf32_exact(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the 10-bit mantissa the TF32 tensor path reads (nearest, ties away)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
def test_rescale_path(dtype, causal):
    """Key norms grow along the sequence, so each row's running max keeps jumping by more than the
    lazy-rescale threshold: the O-rescale path runs on most key tiles.  Inputs are exactly
    representable in the tensor path's input precision (bf16, or TF32 for fp32 I/O), so the
    comparison checks the rescale logic rather than input rounding at these very large scores."""
    B, H, S_q, S_k, D = 1, 2, 300, 700, 64
    q, k, v = synth.make_qkv(B, H, S_q, S_k, D, D, "f32", sigma_q=3.0, seed=17)
    growth = (1.0 + np.arange(S_k, dtype=np.float32) / 16.0)[None, None, :, None]
    k = (k * growth).astype(np.float32)
    if dtype == "bf16":
        q, k, v = (synth.to_bf16_bits(x) for x in (q, k, v))
    else:
        q, k, v = (_tf32_exact(x) for x in (q, k, v))
    scale = float(np.float32(0.125))  # a power of two: exact in any precision
    check(run(q, k, v, scale, causal), oracle.attn_fwd(q, k, v, scale, causal), dtype, "rescale path")


# ---------------------------------------------------------------- invariants on the GPU

def test_gpu_ones_value_and_causal_row0():
    q, k, _ = synth.make_qkv(2, 2, 300, 300, 64, 64, "bf16", seed=12)
    ones = synth.to_bf16_bits(np.ones((2, 2, 300, 64), np.float32))
    for causal in (False, True):
        got = run(q, k, ones, 0.125, causal)
        assert np.abs(got - 1.0).max() <= 1e-2
    _, _, v = synth.make_qkv(2, 2, 300, 300, 64, 64, "bf16", seed=13)
    got = run(q, k, v, 0.125, True)
    assert np.array_equal(got[:, :, 0, :], synth.bf16_bits_to_fp32(v[:, :, 0, :]).astype(np.float64))


# ---------------------------------------------------------------- write set and strided views

SENT16 = 0xDEAD
SENT32 = 0x7FC0DEAD


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shift", [0, 16])
@pytest.mark.parametrize("D_v", [24, 128])
def test_write_set_guard_bands(dtype, causal, shift, D_v):
    """Only O[b,h,i<S_q,e<D_v] is written: padding columns, padding rows and 4 KiB canaries stay bit-exact.
    shift = 16 starts O 16 bytes past a 32-byte boundary (the bf16 epilogue then stores 16 bytes at a time);
    D_v = 128 with shift 0 takes the bf16 two-tile kernel's short epilogue (32-byte rows, whole 16-column groups)."""
    B, H, S_q, S_k, D_qk = 2, 3, 201, 150, 40
    q, k, v = synth.make_qkv(B, H, S_q, S_k, D_qk, D_v, dtype, seed=14)
    elt = 2 if dtype == "bf16" else 4
    pad_d, pad_s = (8 if D_v == 24 else 32), 3
    row = D_v + pad_d
    o_strides = (H * (S_q + pad_s) * row, (S_q + pad_s) * row, row)
    canary = 4096 // elt
    total = canary + B * o_strides[0] + canary + 16
    tdt = torch.int16 if dtype == "bf16" else torch.int32
    sentinel = SENT16 - (1 << 16) if dtype == "bf16" else SENT32
    buf = torch.full((total,), sentinel, dtype=tdt, device="cuda")
    view_dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    o0 = canary + row + shift // elt  # after one pad row
    O = torch.as_strided(buf.view(view_dt), (B, H, S_q, D_v), o_strides + (1,), o0)
    Q, K, V = to_device(q), to_device(k), to_device(v)
    vt.attn_fwd(Q, K, V, scale=0.2, causal=causal, out=O)
    assert vt.vt_last_device_status() == 0
    host = buf.cpu().numpy()
    mask = np.ones(total, bool)
    idx = (o0 + np.arange(B)[:, None, None, None] * o_strides[0] + np.arange(H)[None, :, None, None] * o_strides[1]
           + np.arange(S_q)[None, None, :, None] * o_strides[2] + np.arange(D_v)[None, None, None, :])
    mask[idx.ravel()] = False
    assert np.all(host[mask] == sentinel), "a position outside O's logical elements was written"
    check(to_host64(O), oracle.attn_fwd(q, k, v, 0.2, causal), dtype, "strided O")


def test_strided_inputs():
    """Q, K, V given as [B, S, H, D] memory viewed as [B, H, S, D] (non-packed strides)."""
    B, H, S_q, S_k, D_qk, D_v = 2, 3, 130, 190, 64, 32
    q, k, v = synth.make_qkv(B, H, S_q, S_k, D_qk, D_v, "bf16", seed=15)
    Qs = to_device(np.ascontiguousarray(q.transpose(0, 2, 1, 3))).permute(0, 2, 1, 3)
    Ks = to_device(np.ascontiguousarray(k.transpose(0, 2, 1, 3))).permute(0, 2, 1, 3)
    Vs = to_device(np.ascontiguousarray(v.transpose(0, 2, 1, 3))).permute(0, 2, 1, 3)
    assert not Qs.is_contiguous()
    O = vt.attn_fwd(Qs, Ks, Vs, scale=0.125, causal=True)
    assert vt.vt_last_device_status() == 0
    check(to_host64(O), oracle.attn_fwd(q, k, v, 0.125, True), "bf16", "strided inputs")


def test_empty_problem_writes_nothing():
    O = torch.full((1, 1, 4, 8), 3.0, dtype=torch.bfloat16, device="cuda")
    Q = torch.zeros((0, 1, 4, 8), dtype=torch.bfloat16, device="cuda")
    rc = vt.vt_attn_fwd(Q.data_ptr(), Q.data_ptr(), Q.data_ptr(), O.data_ptr(), 0, 1, 4, 4, 8, 8, 1.0, 0,
                        vt.VT_BF16, torch.cuda.current_stream().cuda_stream)
    assert rc == 0 and torch.all(O == 3.0)


# ---------------------------------------------------------------- bounded waits

def test_stalled_pipeline_reports_timeout_and_context_survives():
    """A wait on a barrier nobody signals gives up after its limit: status VT_ERR_DEVICE_TIMEOUT, no hang."""
    q, k, v = synth.make_qkv(1, 2, 256, 256, 64, 64, "bf16", seed=16)
    Q, K, V = to_device(q), to_device(k), to_device(v)
    opts = vt.vt_attn_opts(wait_timeout_ns=20_000_000, flags=vt.VT_OPT_TEST_STALL)
    vt.attn_fwd(Q, K, V, scale=0.125, opts=opts)
    assert vt.vt_last_device_status() == 5
    assert vt.vt_last_device_status() == 0  # cleared
    got = to_host64(vt.attn_fwd(Q, K, V, scale=0.125))
    assert vt.vt_last_device_status() == 0
    check(got, oracle.attn_fwd(q, k, v, 0.125, False), "bf16", "after timeout")


def test_device_status_is_kept_per_stream():
    """A time-out on one stream is reported to that stream only: a caller polling another stream sees VT_OK
    and does not clear it.  Both element types' kernels, each on its own pair of streams."""
    for dtype, seed in (("bf16", 17), ("f32", 18)):
        q, k, v = synth.make_qkv(1, 2, 256, 256, 64, 64, dtype, seed=seed)
        Q, K, V = to_device(q), to_device(k), to_device(v)
        stalled, healthy = torch.cuda.Stream(), torch.cuda.Stream()
        opts = vt.vt_attn_opts(wait_timeout_ns=20_000_000, flags=vt.VT_OPT_TEST_STALL)
        vt.attn_fwd(Q, K, V, scale=0.125, opts=opts, stream=stalled)
        out = vt.attn_fwd(Q, K, V, scale=0.125, stream=healthy)
        assert vt.vt_last_device_status(healthy) == 0
        assert vt.vt_last_device_status(stalled) == 5  # still there after the other stream's poll
        assert vt.vt_last_device_status(stalled) == 0  # cleared by its own poll
        healthy.synchronize()
        check(to_host64(out), oracle.attn_fwd(q, k, v, 0.125, False), dtype, f"{dtype} beside a stalled stream")


def test_rows_dominated_by_one_key_reproduce_its_value_row():
    """Where one key carries all but ~1e-4 of a row's weight, the output must round to that key's V values:
    P V multiplies the dominant P rounded to bf16, and the row sum has to weigh it the same way (a mismatch
    of up to 2^-9 moves the result by up to half a bf16 step).  Checked on every element whose exact value
    lies within a quarter bf16 step of the dominant key's value."""
    B, H, S, D = 1, 4, 1024, 128
    q, k, v = synth.make_qkv(B, H, S, S, D, D, "bf16", sigma_q=40.0, seed=77)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    got = vt.attn_fwd(to_device(q), to_device(k), to_device(v), scale=scale, causal=False)
    assert vt.vt_last_device_status() == 0
    got = got.double().cpu().numpy()
    qf, kf, vf = (synth.bf16_bits_to_fp32(a).astype(np.float64) for a in (q, k, v))
    checked = 0
    for h in range(H):
        s = scale * qf[0, h] @ kf[0, h].T
        w = np.exp(s - s.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        exact = w @ vf[0, h]
        top = w.argmax(axis=1)
        vtop = vf[0, h][top]
        step = np.ldexp(1.0, np.frexp(vtop)[1] - 8)  # bf16 spacing at |vtop|
        sel = ((w[np.arange(S), top] > 1.0 - 1e-4)[:, None] & (np.abs(vtop) >= 1e-2)
               & (np.abs(exact - vtop) <= 0.25 * step))
        checked += int(sel.sum())
        bad = np.nonzero(sel & (got[0, h] != vtop))
        assert bad[0].size == 0, f"head {h}: {bad[0].size} elements of dominated rows are off their key's value"
    assert checked > B * H * S * D // 4, f"only {checked} elements checked"
