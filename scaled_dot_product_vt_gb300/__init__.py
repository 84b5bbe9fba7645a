"""Python binding of the vt_attn C ABI (include/vt_attn.h): argument marshalling only.

Every step of the attention forward runs in the CUDA kernels of ``libvt_attn.so``;
this module only converts arguments and calls the C entry points through ctypes.
There is no fallback: if the library is missing or cannot be loaded, every call
raises.  PyTorch is used for device memory and the current stream.
"""

from __future__ import annotations

import ctypes
import os

from ._build import LIB, LIB_DEBUG, build  # noqa: F401

VT_F32, VT_BF16 = 0, 1
VT_OPT_TEST_STALL = 1
VT_OPT_TEST_BOUNDS = 2
VT_MASK_NONE, VT_MASK_CAUSAL, VT_MASK_WINDOW, VT_MASK_WINDOW_COMPLEMENT = 0, 1, 2, 3
MASKS = {"none": VT_MASK_NONE, "causal": VT_MASK_CAUSAL, "window": VT_MASK_WINDOW,
         "window_complement": VT_MASK_WINDOW_COMPLEMENT}

STATUS = {
    0: "VT_OK", 1: "VT_ERR_INVALID_ARG", 2: "VT_ERR_UNSUPPORTED", 3: "VT_ERR_MISALIGNED",
    4: "VT_ERR_CUDA", 5: "VT_ERR_DEVICE_TIMEOUT", 6: "VT_ERR_DEVICE_BOUNDS",
}

# Every symbol the header declares.
EXPORTS = ("vt_attn_fwd", "vt_attn_fwd_strided", "vt_attn_fwd_ex", "vt_attn_fwd_splitkv",
           "vt_attn_splitkv_workspace_size", "vt_attn_splitkv_choose", "vt_attn_fwd_splitkv_noalloc",
           "vt_attn_fwd_general", "vt_status_str", "vt_last_device_status")


class VtError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


class vt_attn_opts(ctypes.Structure):
    _fields_ = [("wait_timeout_ns", ctypes.c_uint64), ("flags", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


class vt_attn_mask(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("reserved", ctypes.c_int32), ("offset", ctypes.c_int64),
                ("window", ctypes.c_int64)]


_lib = None


def load(path: str | None = None):
    """Load libvt_attn.so (it must have been built; see ``build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: run scaled_dot_product_vt_gb300.build() (the CUDA path has no fallback)")
    lib = ctypes.CDLL(p)
    i64, vp, f, i, u = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int, ctypes.c_uint
    st3 = ctypes.POINTER(ctypes.c_int64)
    lib.vt_attn_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f, i, i, vp]
    lib.vt_attn_fwd.restype = i
    lib.vt_attn_fwd_strided.argtypes = [vp, st3, vp, st3, vp, st3, vp, st3, i64, i64, i64, i64, i64, i64, f, i, i, vp]
    lib.vt_attn_fwd_strided.restype = i
    lib.vt_attn_fwd_ex.argtypes = [vp, st3, vp, st3, vp, st3, vp, st3, i64, i64, i64, i64, i64, i64, f, i, i,
                                   ctypes.POINTER(vt_attn_opts), vp]
    lib.vt_attn_fwd_ex.restype = i
    sz = ctypes.c_size_t
    lib.vt_attn_fwd_splitkv.argtypes = [vp, st3, vp, st3, vp, st3, vp, st3, i64, i64, i64, i64, i64, i64, f, i, i,
                                        i, vp, sz, vp]
    lib.vt_attn_fwd_splitkv.restype = i
    lib.vt_attn_splitkv_workspace_size.argtypes = [i64, i64, i64, i64, i]
    lib.vt_attn_splitkv_workspace_size.restype = sz
    lib.vt_attn_splitkv_choose.argtypes = [i64, i64, i64, i64, i, i]
    lib.vt_attn_splitkv_choose.restype = i
    lib.vt_attn_fwd_splitkv_noalloc.argtypes = [vp, st3, vp, st3, vp, st3, vp, st3, i64, i64, i64, i64, i64, i64,
                                                f, i, i, i, vp]
    lib.vt_attn_fwd_splitkv_noalloc.restype = i
    lib.vt_attn_fwd_general.argtypes = [vp, st3, vp, st3, vp, st3, vp, st3, vp, i64, i64, i64, i64, i64, i64, i64, f,
                                        i, ctypes.POINTER(vt_attn_mask), i, vp, sz, ctypes.POINTER(vt_attn_opts), vp]
    lib.vt_attn_fwd_general.restype = i
    lib.vt_status_str.argtypes = [i]
    lib.vt_status_str.restype = ctypes.c_char_p
    lib.vt_last_device_status.argtypes = [vp]
    lib.vt_last_device_status.restype = i
    if path is None:
        _lib = lib
    return lib


def load_debug():
    """Load libvt_attn_debug.so: the same entry points, with device index checks (VT_DEBUG) that report
    VT_ERR_DEVICE_BOUNDS.  Returns a separate handle; the module-level wrappers keep using the release
    library."""
    return load(LIB_DEBUG)


def _stride3(s):
    if s is None:
        return None
    return (ctypes.c_int64 * 3)(*[int(x) for x in s])


def vt_attn_fwd(Q, K, V, O, B, H, S_q, S_k, D_qk, D_v, scale, causal, dtype, stream) -> int:
    """The C entry point with raw device addresses (ints); returns the vt_status code."""
    return load().vt_attn_fwd(Q, K, V, O, B, H, S_q, S_k, D_qk, D_v, scale, int(causal), dtype, stream)


def vt_attn_fwd_strided(Q, q_stride, K, k_stride, V, v_stride, O, o_stride,
                        B, H, S_q, S_k, D_qk, D_v, scale, causal, dtype, stream) -> int:
    return load().vt_attn_fwd_strided(Q, _stride3(q_stride), K, _stride3(k_stride), V, _stride3(v_stride),
                                      O, _stride3(o_stride), B, H, S_q, S_k, D_qk, D_v, scale, int(causal),
                                      dtype, stream)


def vt_attn_fwd_ex(Q, q_stride, K, k_stride, V, v_stride, O, o_stride,
                   B, H, S_q, S_k, D_qk, D_v, scale, causal, dtype, opts, stream) -> int:
    return load().vt_attn_fwd_ex(Q, _stride3(q_stride), K, _stride3(k_stride), V, _stride3(v_stride),
                                 O, _stride3(o_stride), B, H, S_q, S_k, D_qk, D_v, scale, int(causal), dtype,
                                 ctypes.byref(opts) if opts is not None else None, stream)


def vt_attn_fwd_splitkv(Q, q_stride, K, k_stride, V, v_stride, O, o_stride, B, H, S_q, S_k, D_qk, D_v,
                        scale, causal, dtype, n_split, workspace, workspace_bytes, stream) -> int:
    return load().vt_attn_fwd_splitkv(Q, _stride3(q_stride), K, _stride3(k_stride), V, _stride3(v_stride),
                                      O, _stride3(o_stride), B, H, S_q, S_k, D_qk, D_v, scale, int(causal), dtype,
                                      int(n_split), workspace, int(workspace_bytes), stream)


def vt_attn_splitkv_workspace_size(B, H, S_q, D_v, n_split) -> int:
    return int(load().vt_attn_splitkv_workspace_size(B, H, S_q, D_v, int(n_split)))


def vt_attn_splitkv_choose(B, H, S_q, S_k, causal, dtype) -> int:
    return int(load().vt_attn_splitkv_choose(B, H, S_q, S_k, int(causal), dtype))


def vt_attn_fwd_splitkv_noalloc(Q, q_stride, K, k_stride, V, v_stride, O, o_stride, B, H, S_q, S_k, D_qk, D_v,
                                scale, causal, dtype, n_split, stream) -> int:
    """Split-KV forward whose scratch is the library's fixed 32 MiB device array: for callers that
    may not allocate device memory.  Raw device addresses (ints); returns the vt_status code."""
    return load().vt_attn_fwd_splitkv_noalloc(Q, _stride3(q_stride), K, _stride3(k_stride), V, _stride3(v_stride),
                                              O, _stride3(o_stride), B, H, S_q, S_k, D_qk, D_v, scale, int(causal),
                                              dtype, int(n_split), stream)


def vt_attn_fwd_general(Q, q_stride, K, k_stride, V, v_stride, O, o_stride, lse, B, H, H_kv, S_q, S_k, D_qk, D_v,
                        scale, dtype, mask, n_split, workspace, workspace_bytes, opts, stream) -> int:
    """The general C entry point with raw device addresses (ints; lse and workspace may be None);
    ``mask`` is a vt_attn_mask or None.  Returns the vt_status code."""
    return load().vt_attn_fwd_general(Q, _stride3(q_stride), K, _stride3(k_stride), V, _stride3(v_stride), O,
                                      _stride3(o_stride), lse, B, H, H_kv, S_q, S_k, D_qk, D_v, scale, dtype,
                                      ctypes.byref(mask) if mask is not None else None, int(n_split), workspace,
                                      int(workspace_bytes), ctypes.byref(opts) if opts is not None else None, stream)


def vt_status_str(code: int) -> str:
    return load().vt_status_str(code).decode()


def vt_last_device_status(stream=None) -> int:
    return load().vt_last_device_status(_stream_handle(stream))


# ---------------------------------------------------------------- torch conveniences

def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return VT_BF16
    if t.dtype == torch.float32:
        return VT_F32
    raise TypeError(f"vt_attn supports bfloat16 and float32 tensors, got {t.dtype}")


def _bhs_strides(t):
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError("tensors are [B, H, S, D] with the last dimension contiguous")
    return (t.stride(0), t.stride(1), t.stride(2))


def attn_fwd(q, k, v, scale: float | None = None, causal: bool = False, out=None, stream=None, opts=None):
    """O = softmax(scale * q k^T) v for CUDA tensors q [B,H,S_q,D_qk], k [B,H,S_k,D_qk], v [B,H,S_k,D_v].

    Strided inputs are passed as they are (last dimension contiguous).  ``out`` may be a
    preallocated (possibly strided) [B,H,S_q,D_v] tensor; otherwise one is allocated.
    """
    import torch
    B, H, S_q, D_qk = q.shape
    S_k, D_v = k.shape[2], v.shape[3]
    if k.shape != (B, H, S_k, D_qk) or v.shape != (B, H, S_k, D_v):
        raise ValueError("shape mismatch between q, k and v")
    code = _dtype_code(q)
    if _dtype_code(k) != code or _dtype_code(v) != code:
        raise TypeError("q, k and v must share one dtype")
    if scale is None:
        scale = float(D_qk) ** -0.5
    if out is None:
        out = torch.empty((B, H, S_q, D_v), dtype=q.dtype, device=q.device)
    rc = vt_attn_fwd_ex(q.data_ptr(), _bhs_strides(q), k.data_ptr(), _bhs_strides(k), v.data_ptr(),
                        _bhs_strides(v), out.data_ptr(), _bhs_strides(out), B, H, S_q, S_k, D_qk, D_v,
                        float(scale), causal, code, opts, _stream_handle(stream))
    if rc != 0:
        raise VtError(rc, "vt_attn_fwd")
    return out


def attn_fwd_splitkv(q, k, v, scale: float | None = None, causal: bool = False, n_split: int | None = None,
                     out=None, workspace=None, stream=None):
    """Split-KV forward for CUDA tensors (bf16 or fp32).  ``n_split=None`` uses the
    library's choice; ``workspace`` may be a preallocated uint8 CUDA tensor of at least
    ``vt_attn_splitkv_workspace_size`` bytes (allocated here otherwise)."""
    import torch
    B, H, S_q, D_qk = q.shape
    S_k, D_v = k.shape[2], v.shape[3]
    if k.shape != (B, H, S_k, D_qk) or v.shape != (B, H, S_k, D_v):
        raise ValueError("shape mismatch between q, k and v")
    code = _dtype_code(q)
    if _dtype_code(k) != code or _dtype_code(v) != code:
        raise TypeError("q, k and v must share one dtype")
    if scale is None:
        scale = float(D_qk) ** -0.5
    if n_split is None:
        n_split = vt_attn_splitkv_choose(B, H, S_q, S_k, causal, code)
    if out is None:
        out = torch.empty((B, H, S_q, D_v), dtype=q.dtype, device=q.device)
    need = vt_attn_splitkv_workspace_size(B, H, S_q, D_v, n_split)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = vt_attn_fwd_splitkv(q.data_ptr(), _bhs_strides(q), k.data_ptr(), _bhs_strides(k), v.data_ptr(),
                             _bhs_strides(v), out.data_ptr(), _bhs_strides(out), B, H, S_q, S_k, D_qk, D_v,
                             float(scale), causal, code, n_split, ws_ptr, ws_bytes, _stream_handle(stream))
    if rc != 0:
        raise VtError(rc, "vt_attn_fwd_splitkv")
    return out


def attn_fwd_general(q, k, v, scale: float | None = None, mask: str = "none", offset: int = 0, window: int = 0,
                     return_lse: bool = False, n_split: int = 1, out=None, lse=None, workspace=None, stream=None,
                     opts=None):
    """General forward for CUDA tensors: q [B,H,S_q,D_qk], k [B,H_kv,S_k,D_qk], v [B,H_kv,S_k,D_v] with H a
    multiple of H_kv (grouped heads), ``mask`` one of ``MASKS`` with ``offset`` and ``window`` (see
    include/vt_attn.h).  Returns O, or (O, LSE) with ``return_lse`` (LSE: float32 [B,H,S_q], natural log).
    ``n_split`` > 1 runs the split-KV form; its workspace is allocated here unless given."""
    import torch
    B, H, S_q, D_qk = q.shape
    H_kv, S_k, D_v = k.shape[1], k.shape[2], v.shape[3]
    if k.shape != (B, H_kv, S_k, D_qk) or v.shape != (B, H_kv, S_k, D_v):
        raise ValueError("shape mismatch between q, k and v")
    code = _dtype_code(q)
    if _dtype_code(k) != code or _dtype_code(v) != code:
        raise TypeError("q, k and v must share one dtype")
    if scale is None:
        scale = float(D_qk) ** -0.5
    if out is None:
        out = torch.empty((B, H, S_q, D_v), dtype=q.dtype, device=q.device)
    if return_lse and lse is None:
        lse = torch.empty((B, H, S_q), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous() or lse.numel() != B * H * S_q):
        raise ValueError("lse must be a contiguous float32 tensor of B*H*S_q elements")
    need = vt_attn_splitkv_workspace_size(B, H, S_q, D_v, n_split)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    m = vt_attn_mask(MASKS[mask], 0, int(offset), int(window))
    rc = vt_attn_fwd_general(q.data_ptr(), _bhs_strides(q), k.data_ptr(), _bhs_strides(k), v.data_ptr(),
                             _bhs_strides(v), out.data_ptr(), _bhs_strides(out),
                             lse.data_ptr() if lse is not None else None, B, H, H_kv, S_q, S_k, D_qk, D_v,
                             float(scale), code, m, n_split, ws_ptr, ws_bytes, opts, _stream_handle(stream))
    if rc != 0:
        raise VtError(rc, "vt_attn_fwd_general")
    return (out, lse) if return_lse else out
