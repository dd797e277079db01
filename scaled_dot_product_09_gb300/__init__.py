"""GB300 (sm_103a) fused scaled-dot-product attention forward.

Thin Python binding over the C ABI of ``libsdpa09.so`` (declared in
``include/sdpa09.h``): it only marshals torch tensors into pointers and
sizes.  Every step of the computation runs in the library's CUDA kernels;
there is no CPU or PyTorch fallback -- a missing or unbuildable library
raises.

    O = softmax(scale * Q.K^T + bias) . V

with bias one of: none (diffusion UNet self/cross attention), Swin's
relative-position table plus shifted-window mask, or SAM's decomposed
relative position ("视觉大模型训练和推理加速" section 一; "Accelerated
Diffusers with PyTorch 2.0" section 加速 Transformer 块; SAM rewrite,
section Bfloat16 半精度).
"""
from __future__ import annotations

import array
import ctypes
import math
import os
import threading

__all__ = ["attn_fwd", "attn_fwd_train", "attn_fwd_varlen", "attn_bwd", "attn_bwd_workspace_size", "attn_bwd_noalloc", "attn_debug_bias", "attn_device_status", "selftest_wait_timeout", "SwinBias", "SamBias",
           "load_library", "AttnError", "ATTN_OK", "ATTN_ERR_ARG", "ATTN_ERR_UNSUPPORTED",
           "ATTN_ERR_CUDA", "ATTN_ERR_DEVICE_TIMEOUT", "HEADER_SYMBOLS"]

ATTN_OK, ATTN_ERR_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_DEVICE_TIMEOUT = 0, -1, -2, -3, -4
ATTN_BF16, ATTN_FP16 = 0, 1
ATTN_BIAS_NONE, ATTN_BIAS_SWIN, ATTN_BIAS_SAM_RELPOS = 0, 1, 2
ATTN_SWIN_WINDOWS, ATTN_SWIN_IMAGE = 0, 1

# Every extern "C" function include/sdpa09.h declares.
HEADER_SYMBOLS = ("attn_fwd", "attn_fwd_train", "attn_fwd_varlen", "attn_bwd", "attn_bwd_workspace_size",
                  "attn_bwd_noalloc",
                  "attn_debug_bias", "attn_device_status",
                  "attn_selftest_wait_timeout", "attn_last_error", "attn_abi_version")
ATTN_VARLEN_MAX_SEQ = 128

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"sdpa09 error {code}: {msg}")
        self.code = code


class _SwinArgs(ctypes.Structure):
    _fields_ = [("table", ctypes.c_void_p), ("win", ctypes.c_int), ("grid_h", ctypes.c_int),
                ("grid_w", ctypes.c_int), ("shift", ctypes.c_int), ("layout", ctypes.c_int)]


class _SamArgs(ctypes.Structure):
    _fields_ = [("rel_h", ctypes.c_void_p), ("rel_w", ctypes.c_void_p), ("q_h", ctypes.c_int),
                ("q_w", ctypes.c_int), ("k_h", ctypes.c_int), ("k_w", ctypes.c_int),
                ("rel_h_len", ctypes.c_int), ("rel_w_len", ctypes.c_int)]


class SwinBias:
    """Swin relative-position bias + shifted-window mask.
    table: device fp32 [(2*win-1)^2, H]; grid_h/grid_w: tokens per image side.
    layout "windows": q/k/v/out are [B windows, H, win*win, d], already shifted
    and partitioned; layout "image": they are [images, grid_h, grid_w, H, d]
    and the kernel applies the shift and partition (and their inverse on the
    output) itself."""

    def __init__(self, table, win, grid_h, grid_w, shift, layout="windows"):
        if layout not in ("windows", "image"):
            raise ValueError(f"layout must be 'windows' or 'image', not {layout!r}")
        self.table, self.win, self.grid_h, self.grid_w, self.shift = table, win, grid_h, grid_w, shift
        self.layout = layout

    def _c(self):
        return _SwinArgs(_ptr(self.table), self.win, self.grid_h, self.grid_w, self.shift,
                         ATTN_SWIN_IMAGE if self.layout == "image" else ATTN_SWIN_WINDOWS)


class SamBias:
    """SAM decomposed relative position.  rel_h [L_h, d], rel_w [L_w, d] on
    the device in the Q dtype; query grid q_h x q_w, key grid k_h x k_w
    (default: the query grid).  Tables whose length is not 2*max(q, k) - 1
    are resampled linearly in the kernel; unequal grids index them through
    the coordinate scalers."""

    def __init__(self, rel_h, rel_w, q_h, q_w, k_h=None, k_w=None):
        self.rel_h, self.rel_w, self.q_h, self.q_w = rel_h, rel_w, q_h, q_w
        self.k_h = q_h if k_h is None else k_h
        self.k_w = q_w if k_w is None else k_w

    def _c(self):
        return _SamArgs(_ptr(self.rel_h), _ptr(self.rel_w), self.q_h, self.q_w, self.k_h, self.k_w,
                        int(self.rel_h.shape[0]), int(self.rel_w.shape[0]))


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def load_library(build: bool = True):
    """Load libsdpa09.so (building it first when missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        from . import _build
        path = _build.build() if build else _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libsdpa09.so not found at {path}; run the build first")
        lib = ctypes.CDLL(path)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, vp]
        lib.attn_fwd.restype = i
        lib.attn_fwd_train.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, vp]
        lib.attn_fwd_train.restype = i
        ip = ctypes.POINTER(ctypes.c_int)
        lib.attn_fwd_varlen.argtypes = [vp, vp, vp, vp, ip, ip, i, i, i, f, i, vp]
        lib.attn_fwd_varlen.restype = i
        sz = ctypes.c_size_t
        lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, vp, vp, sz, vp]
        lib.attn_bwd.restype = i
        lib.attn_bwd_workspace_size.argtypes = [i, i, i, i, i, i, vp]
        lib.attn_bwd_workspace_size.restype = sz
        lib.attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        lib.attn_bwd_noalloc.restype = i
        lib.attn_debug_bias.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, vp]
        lib.attn_debug_bias.restype = i
        lib.attn_device_status.argtypes = [vp]
        lib.attn_device_status.restype = i
        lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
        lib.attn_selftest_wait_timeout.restype = i
        lib.attn_last_error.argtypes = []
        lib.attn_last_error.restype = ctypes.c_char_p
        lib.attn_abi_version.argtypes = []
        lib.attn_abi_version.restype = i
        _lib = lib
        return lib


def _check(lib, rc):
    if rc != ATTN_OK:
        raise AttnError(rc, lib.attn_last_error().decode(errors="replace"))


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float16:
        return ATTN_FP16
    raise AttnError(ATTN_ERR_ARG, f"unsupported dtype {t.dtype}")


def _bias_args(bias):
    if bias is None:
        return ATTN_BIAS_NONE, None, None
    c = bias._c()
    kind = ATTN_BIAS_SWIN if isinstance(bias, SwinBias) else ATTN_BIAS_SAM_RELPOS
    return kind, c, ctypes.byref(c)


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _is_image(bias):
    return isinstance(bias, SwinBias) and bias.layout == "image"


def _shape_image(q, k, v, bias):
    if q.dim() != 5 or q.shape != k.shape or q.shape != v.shape:
        raise AttnError(ATTN_ERR_ARG, "image layout needs q, k, v of one shape [images, grid_h, grid_w, H, d]")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise AttnError(ATTN_ERR_ARG, "q, k, v must be contiguous")
    n_img, gh, gw, H, d = q.shape
    if (gh, gw) != (bias.grid_h, bias.grid_w) or gh % bias.win or gw % bias.win:
        raise AttnError(ATTN_ERR_ARG, "image grid does not match the Swin arguments")
    n = bias.win * bias.win
    return n_img * (gh // bias.win) * (gw // bias.win), H, n, n, d


def _shape(q, k, v):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise AttnError(ATTN_ERR_ARG, "q, k, v must be [B, H, N, d]")
    B, H, Nq, d = q.shape
    if k.shape[:2] != (B, H) or v.shape != k.shape or k.shape[3] != d:
        raise AttnError(ATTN_ERR_ARG, "k, v must be [B, H, Nk, d] matching q")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise AttnError(ATTN_ERR_ARG, "tensors must be contiguous")
    return B, H, Nq, k.shape[2], d


def attn_fwd(q, k, v, out=None, scale=None, bias=None, stream=None):
    """O = softmax(scale*Q.K^T + bias).V on the GPU.  q [B,H,Nq,d], k/v
    [B,H,Nk,d] contiguous bf16/fp16 CUDA tensors; returns out [B,H,Nq,d].
    With SwinBias(layout="image") q/k/v/out are [images, grid_h, grid_w, H, d]
    instead (B then counts windows)."""
    import torch
    lib = load_library()
    B, H, Nq, Nk, d = _shape_image(q, k, v, bias) if _is_image(bias) else _shape(q, k, v)
    if out is None:
        out = torch.empty_like(q)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kind, _keep, args = _bias_args(bias)
    rc = lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H, Nq, Nk, d, scale,
                      _dtype_code(q), kind, args, _stream_ptr(stream))
    _check(lib, rc)
    return out


def attn_fwd_train(q, k, v, out=None, lse=None, scale=None, bias=None, stream=None):
    """attn_fwd that also returns each query row's natural-log log-sum-exp,
    fp32 [B, H, Nq] (the statistic attn_bwd needs): returns (out, lse)."""
    import torch
    lib = load_library()
    B, H, Nq, Nk, d = _shape_image(q, k, v, bias) if _is_image(bias) else _shape(q, k, v)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if lse.dtype != torch.float32 or not lse.is_contiguous() or lse.numel() != B * H * Nq:
        raise AttnError(ATTN_ERR_ARG, "lse must be a contiguous fp32 tensor of B * H * Nq values")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kind, _keep, args = _bias_args(bias)
    rc = lib.attn_fwd_train(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq, Nk, d, scale,
                            _dtype_code(q), kind, args, _stream_ptr(stream))
    _check(lib, rc)
    return out, lse


def _cu_array(cu):
    """Host token offsets (list, tuple, numpy array or tensor) as an int32
    array and a ctypes view of it (built without a Python int per element:
    this runs on every call)."""
    if hasattr(cu, "detach"):  # a tensor
        cu = cu.detach().cpu()
    if hasattr(cu, "numpy") or hasattr(cu, "dtype"):
        import numpy as np
        a = np.asarray(cu)
        if a.size and (int(a.max()) > 0x7FFFFFFF or int(a.min()) < -0x80000000):
            raise OverflowError("token offsets must fit in int32")
        vals = array.array("i", np.ascontiguousarray(a, dtype=np.int32).tobytes())
    else:
        vals = array.array("i", cu)
    return (ctypes.c_int * len(vals)).from_buffer(vals), vals


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, H, out=None, scale=None, stream=None):
    """Attention over a nested batch of sequences of different lengths,
    each attending only to itself (no bias).  q/out hold the concatenation
    over sequences s of [H][Lq_s][d], k/v of [H][Lk_s][d], as contiguous
    bf16/fp16 CUDA tensors whose last dim is d (e.g. [H * total, d]);
    cu_seqlens_q/k are the host token offsets [n_seq + 1] (list, numpy or CPU
    tensor).  Returns out."""
    import torch
    lib = load_library()
    cq, vq = _cu_array(cu_seqlens_q)
    ck, vk = _cu_array(cu_seqlens_k)
    if len(vq) != len(vk) or len(vq) < 2:
        raise AttnError(ATTN_ERR_ARG, "cu_seqlens_q and cu_seqlens_k need the same n_seq + 1 >= 2 entries")
    d = q.shape[-1]
    for t, tot in ((q, vq[-1]), (k, vk[-1]), (v, vk[-1])):
        if not t.is_contiguous() or t.shape[-1] != d or t.numel() != H * tot * d:
            raise AttnError(ATTN_ERR_ARG, "q, k, v must be contiguous with H * total tokens rows of d")
    if out is None:
        out = torch.empty_like(q)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rc = lib.attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), cq, ck, len(vq) - 1, H, d, scale,
                             _dtype_code(q), _stream_ptr(stream))
    _check(lib, rc)
    return out


def attn_bwd_workspace_size(B, H, Nq, Nk, d, bias=None):
    """Bytes of device scratch attn_bwd needs for these sizes (0: none)."""
    lib = load_library()
    kind, _keep, args = _bias_args(bias)
    return int(lib.attn_bwd_workspace_size(B, H, Nq, Nk, d, kind, args))


def attn_bwd(q, k, v, out, dout, lse=None, scale=None, bias=None, stream=None, grads=None, workspace=None):
    """Gradients of attn_fwd: q/k/v/out/dout [B,H,N,d] contiguous bf16/fp16
    CUDA tensors (out: the forward's output, dout: the gradient with respect
    to it; with SwinBias(layout="image") all of them and the returned dq, dk,
    dv are [images, grid_h, grid_w, H, d]), lse: the fp32 [B,H,Nq] row
    log-sum-exp from attn_fwd_train (may be None when Nq, Nk <= 128 without
    SAM).  Returns (dq, dk, dv, d_bias) with
    d_bias the fp32 gradient of a SwinBias table, the pair (d_rel_h, d_rel_w)
    of a SamBias, else None.  grads: the four buffers to use instead (d_bias is
    added to; for SAM one fp32 [L_h + L_w, d] tensor); workspace: a uint8 CUDA
    tensor of at least attn_bwd_workspace_size bytes (allocated here when
    None)."""
    import torch
    lib = load_library()
    B, H, Nq, Nk, d = _shape_image(q, k, v, bias) if _is_image(bias) else _shape(q, k, v)
    for t in (out, dout):
        if t.shape != q.shape or not t.is_contiguous():
            raise AttnError(ATTN_ERR_ARG, "out and dout must be contiguous and shaped like q")
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous() or lse.numel() != B * H * Nq):
        raise AttnError(ATTN_ERR_ARG, "lse must be a contiguous fp32 tensor of B * H * Nq values")
    if grads is not None:
        dq, dk, dv, d_bias = grads
    else:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        if isinstance(bias, SwinBias):
            d_bias = torch.zeros_like(bias.table)
        elif isinstance(bias, SamBias):
            d_bias = torch.zeros((bias.rel_h.shape[0] + bias.rel_w.shape[0], d), dtype=torch.float32, device=q.device)
        else:
            d_bias = None
    kind, _keep, args = _bias_args(bias)
    need = int(lib.attn_bwd_workspace_size(B, H, Nq, Nk, d, kind, args))
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                      B, H, Nq, Nk, d, scale, _dtype_code(q), kind, args,
                      _ptr(d_bias) if d_bias is not None else None,
                      _ptr(workspace) if workspace is not None else None, ws_bytes, _stream_ptr(stream))
    _check(lib, rc)
    if isinstance(bias, SamBias) and d_bias is not None:
        n_h = bias.rel_h.shape[0]
        return dq, dk, dv, (d_bias[:n_h], d_bias[n_h:])
    return dq, dk, dv, d_bias


def attn_bwd_noalloc(q, k, v, out, dout, lse=None, scale=None, stream=None, grads=None):
    """attn_bwd without a bias, for callers that may not allocate device memory
    while they run it: the library's own fixed scratch (at most 2^20 query
    rows B * H * Nq) stands in for the workspace.  grads: (dq, dk, dv) buffers
    to write (allocated here when None).  Calls that overlap on the GPU race on
    that scratch; returns (dq, dk, dv)."""
    import torch
    lib = load_library()
    B, H, Nq, Nk, d = _shape(q, k, v)
    for t in (out, dout):
        if t.shape != q.shape or not t.is_contiguous():
            raise AttnError(ATTN_ERR_ARG, "out and dout must be contiguous and shaped like q")
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous() or lse.numel() != B * H * Nq):
        raise AttnError(ATTN_ERR_ARG, "lse must be a contiguous fp32 tensor of B * H * Nq values")
    dq, dk, dv = grads if grads is not None else (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rc = lib.attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                              _ptr(dv), B, H, Nq, Nk, d, scale, _dtype_code(q), _stream_ptr(stream))
    _check(lib, rc)
    return dq, dk, dv


def attn_debug_bias(q, k, v, scale=None, bias=None, stream=None):
    """The bias the in-kernel builder adds, as fp32 [B,H,Nq,Nk] (test hook)."""
    import torch
    lib = load_library()
    B, H, Nq, Nk, d = _shape(q, k, v)
    dbg = torch.zeros((B, H, Nq, Nk), dtype=torch.float32, device=q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kind, _keep, args = _bias_args(bias)
    rc = lib.attn_debug_bias(_ptr(q), _ptr(k), _ptr(v), _ptr(dbg), B, H, Nq, Nk, d, scale,
                             _dtype_code(q), kind, args, _stream_ptr(stream))
    _check(lib, rc)
    return dbg


def selftest_wait_timeout(limit_us: int, stream=None):
    """Launch the bounded-wait self-test (a wait that runs out after
    `limit_us`); read the outcome with attn_device_status."""
    lib = load_library()
    rc = lib.attn_selftest_wait_timeout(int(limit_us), _stream_ptr(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, lib.attn_last_error().decode(errors="replace"))


def attn_device_status(stream=None):
    """Synchronise the stream and return the library's device status code."""
    lib = load_library()
    return lib.attn_device_status(_stream_ptr(stream))
