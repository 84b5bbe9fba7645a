"""CPU oracle for the scaled dot-product attention forward (fp64, plus a long-double brute force).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the bench's
CPU-baseline leg are the only callers.  The CUDA library never imports, links or
calls this; it shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain C, compiled with gcc by
``build()``); this module only marshals numpy arrays through ctypes.  What it
computes follows the naive reference of the VeriTile page
"VeriTile.Examples.FlashAttention1.NaiveRefinement" (fa1NaiveReference4D and its
causal twin) and the CPU routine ``expectedOutput`` of the accy page
"tiny.accy.kernel.library.attention": per (b, h, i), scores over the allowed keys,
their max, the shifted exp-sum and the value-weighted sum, in fp64.

Pins: every function here is checked in ``tests/test_oracle_pins.py`` against
closed forms, invariants, a long-double brute force and the accy page's worked
example; none is "parity unpinned" except the causal alignment for S_q != S_k
beyond j <= i (see the design notes).
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

F32, BF16 = 0, 1
MASKS = {"none": 0, "causal": 1, "window": 2, "window_complement": 3}


def build(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile the oracle with gcc into a shared library; returns its path."""
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", *extra_flags, "-o", out, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    return out


def _needs_build() -> bool:
    return not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)


def load(path: str | None = None):
    """Load (building if needed) the oracle library; ``path`` loads another build of it."""
    global _lib
    if path is None:
        if _lib is not None:
            return _lib
        if _needs_build():
            build()
        path = _LIB
    lib = ctypes.CDLL(path)
    i64, vp, d, i = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double, ctypes.c_int
    lib.oracle_attn_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, d, i, i, i]
    lib.oracle_attn_fwd.restype = i
    lib.oracle_attn_rows.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, d, i, i, vp, i64, i]
    lib.oracle_attn_rows.restype = i
    lib.oracle_attn_fwd_ld.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, d, i, i]
    lib.oracle_attn_fwd_ld.restype = i
    lib.oracle_attn_general.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, d, i, i64, i64, i,
                                        vp, i64, i]
    lib.oracle_attn_general.restype = i
    lib.oracle_attn_general_ld.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, d, i, i64, i64, i]
    lib.oracle_attn_general_ld.restype = i
    if path == _LIB:
        _lib = lib
    return lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle inputs are float32 or bf16 bit patterns (uint16), got {a.dtype}")


def _prep(Q, K, V):
    Q, K, V = (np.ascontiguousarray(x) for x in (Q, K, V))
    code = _dtype_code(Q)
    if _dtype_code(K) != code or _dtype_code(V) != code:
        raise TypeError("Q, K and V must share one dtype")
    B, H, S_q, D_qk = Q.shape
    B2, H2, S_k, D_qk2 = K.shape
    B3, H3, S_k3, D_v = V.shape
    if (B, H, D_qk) != (B2, H2, D_qk2) or (B, H, S_k) != (B3, H3, S_k3):
        raise ValueError("shape mismatch between Q, K and V")
    return Q, K, V, code, (B, H, S_q, S_k, D_qk, D_v)


def default_threads() -> int:
    return os.cpu_count() or 1


def attn_fwd(Q, K, V, scale: float, causal: bool, nthreads: int | None = None, lib=None) -> np.ndarray:
    """O[B,H,S_q,D_v] (float64).  ``scale`` is widened from the fp32 value passed here."""
    lib = lib or load()
    Q, K, V, code, (B, H, S_q, S_k, D_qk, D_v) = _prep(Q, K, V)
    O = np.empty((B, H, S_q, D_v), dtype=np.float64)
    rc = lib.oracle_attn_fwd(Q.ctypes.data, K.ctypes.data, V.ctypes.data, O.ctypes.data,
                             B, H, S_q, S_k, D_qk, D_v, float(np.float32(scale)), int(causal), code,
                             nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd failed with code {rc}")
    return O


def attn_rows(Q, K, V, scale: float, causal: bool, rows, nthreads: int | None = None, lib=None) -> np.ndarray:
    """Selected rows: ``rows`` is an (n, 3) array of (b, h, i); returns (n, D_v) float64."""
    lib = lib or load()
    Q, K, V, code, (B, H, S_q, S_k, D_qk, D_v) = _prep(Q, K, V)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    O = np.empty((rows.shape[0], D_v), dtype=np.float64)
    rc = lib.oracle_attn_rows(Q.ctypes.data, K.ctypes.data, V.ctypes.data, O.ctypes.data,
                              B, H, S_q, S_k, D_qk, D_v, float(np.float32(scale)), int(causal), code,
                              rows.ctypes.data, rows.shape[0], nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attn_rows failed with code {rc}")
    return O


def attn_fwd_longdouble(Q, K, V, scale: float, causal: bool, lib=None) -> np.ndarray:
    """Brute force in long double (tiny inputs only); returned as numpy longdouble."""
    lib = lib or load()
    Q, K, V, code, (B, H, S_q, S_k, D_qk, D_v) = _prep(Q, K, V)
    O = np.empty((B, H, S_q, D_v), dtype=np.longdouble)
    if ctypes.sizeof(ctypes.c_longdouble) != O.itemsize:
        raise RuntimeError("numpy longdouble does not match C long double on this host")
    rc = lib.oracle_attn_fwd_ld(Q.ctypes.data, K.ctypes.data, V.ctypes.data, O.ctypes.data,
                                B, H, S_q, S_k, D_qk, D_v, float(np.float32(scale)), int(causal), code)
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd_ld failed with code {rc}")
    return O


def _prep_general(Q, K, V):
    Q, K, V = (np.ascontiguousarray(x) for x in (Q, K, V))
    code = _dtype_code(Q)
    if _dtype_code(K) != code or _dtype_code(V) != code:
        raise TypeError("Q, K and V must share one dtype")
    B, H, S_q, D_qk = Q.shape
    B2, H_kv, S_k, D_qk2 = K.shape
    B3, H_kv3, S_k3, D_v = V.shape
    if (B, D_qk) != (B2, D_qk2) or (B, H_kv, S_k) != (B3, H_kv3, S_k3):
        raise ValueError("shape mismatch between Q, K and V")
    return Q, K, V, code, (B, H, H_kv, S_q, S_k, D_qk, D_v)


def attn_general(Q, K, V, scale: float, mask: str = "none", offset: int = 0, window: int = 0, rows=None,
                 with_lse: bool = False, nthreads: int | None = None, lib=None):
    """General form: Q [B,H,S_q,D_qk], K [B,H_kv,S_k,D_qk], V [B,H_kv,S_k,D_v] (H a multiple of H_kv).

    ``mask`` is one of ``MASKS``; ``offset`` >= 0 and ``window`` >= 1 as in attn_oracle.c.  Returns
    O (float64, [B,H,S_q,D_v], or (n, D_v) for ``rows`` = (n, 3) triples (b, h, i)), and with
    ``with_lse`` also the natural-log LSE per row ([B,H,S_q] or (n,)).
    """
    lib = lib or load()
    Q, K, V, code, (B, H, H_kv, S_q, S_k, D_qk, D_v) = _prep_general(Q, K, V)
    if rows is None:
        O = np.empty((B, H, S_q, D_v), dtype=np.float64)
        L = np.empty((B, H, S_q), dtype=np.float64) if with_lse else None
        rp, nr = None, 0
    else:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
        O = np.empty((rows.shape[0], D_v), dtype=np.float64)
        L = np.empty((rows.shape[0],), dtype=np.float64) if with_lse else None
        rp, nr = rows.ctypes.data, rows.shape[0]
    rc = lib.oracle_attn_general(Q.ctypes.data, K.ctypes.data, V.ctypes.data, O.ctypes.data,
                                 L.ctypes.data if L is not None else None, B, H, H_kv, S_q, S_k, D_qk, D_v,
                                 float(np.float32(scale)), MASKS[mask], int(offset), int(window), code, rp, nr,
                                 nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attn_general failed with code {rc}")
    return (O, L) if with_lse else O


def attn_general_longdouble(Q, K, V, scale: float, mask: str = "none", offset: int = 0, window: int = 0,
                            lib=None):
    """Long-double brute force of the general form (tiny inputs): returns (O, LSE) as numpy longdouble."""
    lib = lib or load()
    Q, K, V, code, (B, H, H_kv, S_q, S_k, D_qk, D_v) = _prep_general(Q, K, V)
    O = np.empty((B, H, S_q, D_v), dtype=np.longdouble)
    L = np.empty((B, H, S_q), dtype=np.longdouble)
    if ctypes.sizeof(ctypes.c_longdouble) != O.itemsize:
        raise RuntimeError("numpy longdouble does not match C long double on this host")
    rc = lib.oracle_attn_general_ld(Q.ctypes.data, K.ctypes.data, V.ctypes.data, O.ctypes.data, L.ctypes.data,
                                    B, H, H_kv, S_q, S_k, D_qk, D_v, float(np.float32(scale)), MASKS[mask],
                                    int(offset), int(window), code)
    if rc != 0:
        raise ValueError(f"oracle_attn_general_ld failed with code {rc}")
    return O, L
