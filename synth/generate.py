"""Counter-based SplitMix64 inputs for the attention workloads.

Generator (defined here, used by both the oracle's and the CUDA path's tests):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014; the 64-bit finaliser of Vigna's public
  ``splitmix64.c``), used in counter form: draw ``n`` of seed ``s`` is
  ``mix(s + (n + 1) * 0x9E3779B97F4A7C15)`` with the wrapping 64-bit arithmetic of
  the stateful version, so any slice of the stream is computed without the ones
  before it.
* Uniform in [0, 1): the top 53 bits of a draw times 2**-53.
* Normal: Box-Muller on consecutive draw pairs (2k, 2k+1):
  ``r = sqrt(-2 ln(1 - u0))``, ``t = 2 pi u1``, elements 2k and 2k+1 are
  ``r cos t`` and ``r sin t``, then multiplied by sigma.
* Uniform(-1, 1): ``2 u - 1``, one draw per element.
* Q, K and V come from one stream of the workload's seed, in that order, each in
  row-major [B, H, S, D] order; a normal tensor of n elements consumes
  ``2 * ceil(n / 2)`` draws, a uniform one ``n``.
* Values are produced in fp64, rounded to fp32 with round-to-nearest-even and,
  for bf16 I/O, from fp32 to bf16 with round-to-nearest-even.  bf16 tensors are
  returned as their uint16 bit patterns.
"""

from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of the SplitMix64 stream of ``seed`` (uint64)."""
    n = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + n * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, start: int, count: int) -> np.ndarray:
    """Uniforms in [0, 1) (fp64) from draws ``start ..``."""
    z = splitmix64(seed, start, count)
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal(seed: int, start: int, count: int, sigma: float = 1.0) -> np.ndarray:
    """``count`` N(0, sigma^2) values (fp64) by Box-Muller from draws ``start ..``.

    ``count`` must be even when this is called on a slice of a longer tensor; the
    caller rounds the pair boundary.
    """
    npairs = (count + 1) // 2
    u = uniform01(seed, start, 2 * npairs).reshape(npairs, 2)
    r = np.sqrt(-2.0 * np.log1p(-u[:, 0]))
    t = (2.0 * math.pi) * u[:, 1]
    out = np.empty((npairs, 2), dtype=np.float64)
    out[:, 0] = r * np.cos(t)
    out[:, 1] = r * np.sin(t)
    return out.reshape(-1)[:count] * sigma


def to_fp32(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp32, round to nearest even."""
    return x.astype(np.float32)


def to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    with np.errstate(over="ignore"):
        r = (u + bias) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_fp32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact fp32 values."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _fill(seed: int, start: int, n: int, dist: str, sigma: float, dtype: str) -> tuple[np.ndarray, int]:
    """One tensor of ``n`` elements from draw ``start``; returns (array, draws consumed).

    Chunks are independent slices of the counter-based stream, so they are filled
    by a thread pool (numpy releases the GIL); the result does not depend on it.
    """
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)
    if dist == "normal":
        used = 2 * ((n + 1) // 2)
    elif dist == "uniform":
        used = n
    else:
        raise ValueError(dist)

    def chunk(pos: int) -> None:
        m = min(_CHUNK, n - pos)
        if dist == "normal":
            # pos and _CHUNK are even, so each chunk starts on a pair boundary
            vals = normal(seed, start + pos, m, sigma)
        else:
            vals = 2.0 * uniform01(seed, start + pos, m) - 1.0
        v32 = to_fp32(vals)
        out[pos:pos + m] = to_bf16_bits(v32) if dtype == "bf16" else v32

    starts = list(range(0, n, _CHUNK))
    if len(starts) <= 1:
        for p in starts:
            chunk(p)
    else:
        workers = min(len(starts), os.cpu_count() or 1, 32)
        with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(chunk, starts))
    return out, used


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S_q: int
    S_k: int
    D_qk: int
    D_v: int
    dtype: str            # "f32" (TF32 tensor path) or "bf16"
    causal: tuple         # modes exercised: (False,), (True,) or (False, True)
    dist: str             # "normal" or "uniform"
    sigma_q: float
    sigma_kv: float
    seed: int
    # Variants beyond plain/causal attention (empty mask: the modes in `causal` above).
    H_kv: int = 0         # key/value heads (0: H)
    mask: str = ""        # "none", "causal", "window" or "window_complement"
    offset: int = 0
    window: int = 0

    @property
    def kv_heads(self) -> int:
        return self.H_kv or self.H

    def allowed_pairs(self) -> int:
        """Number of (query, key) pairs the mask keeps in one (b, h) slice (mask set)."""
        return int(self.keys_per_row().sum())

    def keys_per_row(self) -> np.ndarray:
        """|A_i| for every query row i of one (b, h) slice (mask set)."""
        i = np.arange(self.S_q, dtype=np.int64)
        hi = np.minimum(i + self.offset, self.S_k - 1)            # last key (causal kinds)
        if self.mask == "none":
            n = np.full(self.S_q, self.S_k, dtype=np.int64)
        elif self.mask == "causal":
            n = hi + 1
        elif self.mask == "window":
            lo = np.maximum(i + self.offset - self.window + 1, 0)
            n = np.maximum(hi - lo + 1, 0)
        elif self.mask == "window_complement":
            n = np.maximum(np.minimum(i + self.offset - self.window, self.S_k - 1) + 1, 0)
        else:
            raise ValueError(f"unknown mask {self.mask!r}")
        return n

    def flops_masked(self) -> float:
        """Algorithmic flops of a masked workload: 2*(D_qk+D_v) per kept (query, key) pair."""
        return 2.0 * self.B * self.H * self.allowed_pairs() * (self.D_qk + self.D_v)

    @property
    def scale(self) -> float:
        """1/sqrt(D_qk) rounded to fp32 (the value passed to both sides)."""
        return float(np.float32(1.0 / math.sqrt(self.D_qk)))

    def flops(self, causal: bool) -> float:
        """Algorithmic flops: 2*B*H*S_q*S_k*(D_qk+D_v), halved for causal."""
        f = 2.0 * self.B * self.H * self.S_q * self.S_k * (self.D_qk + self.D_v)
        return f / 2.0 if causal else f

    def bytes(self) -> int:
        """Algorithmic bytes: Q, K, V read once and O written once."""
        elt = 2 if self.dtype == "bf16" else 4
        return self.B * (self.H * self.S_q * (self.D_qk + self.D_v)
                         + self.kv_heads * self.S_k * (self.D_qk + self.D_v)) * elt


# The five attention workloads: shapes, value distributions and seeds.
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 1, 37, 37, 20, 20, "f32", (False,), "normal", 1.0, 1.0, 0),
    "mid_f32": Workload("mid_f32", 2, 4, 1000, 1000, 72, 72, "f32", (False, True), "uniform", 1.0, 1.0, 1),
    "bf16_causal_2k": Workload("bf16_causal_2k", 4, 16, 2048, 2048, 128, 128, "bf16", (True,), "normal", 1.0, 1.0, 2),
    "bf16_ragged": Workload("bf16_ragged", 2, 32, 333, 8191, 96, 64, "bf16", (False,), "normal", 1.0, 1.0, 3),
    "bf16_causal_8k_peaky": Workload("bf16_causal_8k_peaky", 8, 16, 8192, 8192, 128, 128, "bf16", (True,), "normal", 4.0, 1.0, 4),
    # masked and grouped-head variants (flops count the kept (query, key) pairs exactly)
    "bf16_gqa_causal_8k": Workload("bf16_gqa_causal_8k", 4, 32, 8192, 8192, 128, 128, "bf16", (True,), "normal",
                                   1.0, 1.0, 5, H_kv=8, mask="causal"),
    "bf16_prefill_on_cache_8k": Workload("bf16_prefill_on_cache_8k", 8, 16, 1024, 8192, 128, 128, "bf16", (True,),
                                         "normal", 1.0, 1.0, 6, mask="causal", offset=7168),
    "bf16_window_1k_8k": Workload("bf16_window_1k_8k", 8, 16, 8192, 8192, 128, 128, "bf16", (True,), "normal",
                                  1.0, 1.0, 7, mask="window", window=1024),
    # a 256-query chunk at the end of a 32k-key cache: 32 query blocks for the whole GPU (split-KV's case)
    "bf16_chunk_on_cache_32k": Workload("bf16_chunk_on_cache_32k", 2, 16, 256, 32768, 128, 128, "bf16", (True,),
                                        "normal", 1.0, 1.0, 8, mask="causal", offset=32512),
}


def tensor_shapes(B, H, S_q, S_k, D_qk, D_v):
    """Logical shapes of Q, K, V and O: [B,H,S_q,D_qk], [B,H,S_k,D_qk], [B,H,S_k,D_v], [B,H,S_q,D_v]."""
    return (B, H, S_q, D_qk), (B, H, S_k, D_qk), (B, H, S_k, D_v), (B, H, S_q, D_v)


def element_counts(B, H, S_q, S_k, D_qk, D_v):
    return tuple(int(np.prod(s)) for s in tensor_shapes(B, H, S_q, S_k, D_qk, D_v))


def make_qkv(B, H, S_q, S_k, D_qk, D_v, dtype="bf16", dist="normal", sigma_q=1.0, sigma_kv=1.0, seed=0, H_kv=None):
    """Q, K, V as numpy arrays of shape [B,H,S,D] (bf16 as uint16 bits, f32 as float32); with H_kv, K and V
    have H_kv heads.  Filled in the order Q, K, V from one stream."""
    sq, _, _, _ = tensor_shapes(B, H, S_q, S_k, D_qk, D_v)
    _, sk, sv, _ = tensor_shapes(B, H_kv or H, S_q, S_k, D_qk, D_v)
    pos = 0
    out = []
    for shape, sigma in ((sq, sigma_q), (sk, sigma_kv), (sv, sigma_kv)):
        n = int(np.prod(shape))
        arr, used = _fill(seed, pos, n, dist, sigma, dtype)
        pos += used
        out.append(arr.reshape(shape))
    return tuple(out)


def make_workload(w: Workload):
    return make_qkv(w.B, w.H, w.S_q, w.S_k, w.D_qk, w.D_v, w.dtype, w.dist, w.sigma_q, w.sigma_kv, w.seed,
                    H_kv=w.kv_heads)
