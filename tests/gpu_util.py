"""Shared helpers for the GPU tests: numpy <-> torch transfer, tolerances, error metrics."""

from __future__ import annotations

import numpy as np

# Tolerances against the fp64 oracle (BF16: fp32 accumulation; F32: TF32 tensor path).
TOL_F32_MAX_ABS = 5e-3
TOL_BF16_MAX_ABS = 2e-2
TOL_BF16_REL_FRO = 1e-2


def to_device(a: np.ndarray):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host64(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def errors(got: np.ndarray, ref: np.ndarray):
    d = got.astype(np.float64) - ref
    max_abs = float(np.abs(d).max()) if d.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(d) / den) if den > 0 else float(np.linalg.norm(d))
    return max_abs, rel


def check(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    max_abs, rel = errors(got, ref)
    if dtype == "f32":
        ok = max_abs <= TOL_F32_MAX_ABS
        lim = f"max_abs<={TOL_F32_MAX_ABS}"
    else:
        ok = max_abs <= TOL_BF16_MAX_ABS and rel <= TOL_BF16_REL_FRO
        lim = f"max_abs<={TOL_BF16_MAX_ABS}, rel_fro<={TOL_BF16_REL_FRO}"
    if not ok:
        d = np.abs(got.astype(np.float64) - ref)
        idx = np.unravel_index(np.argmax(d), d.shape)
        bad = np.argwhere(d > (TOL_F32_MAX_ABS if dtype == "f32" else TOL_BF16_MAX_ABS))
        raise AssertionError(f"{what}: max_abs={max_abs:.3e} rel_fro={rel:.3e} (need {lim}); worst at {idx} "
                             f"got={got[idx]} ref={ref[idx]}; {len(bad)} bad elements, first {bad[:8].tolist()}")
    return max_abs, rel
