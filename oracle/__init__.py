"""fp64 CPU oracle for the fused scaled-dot-product attention forward pass.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  Nothing here is used
by, or shares code with, the CUDA path in ``scaled_dot_product_09_gb300``.

The arithmetic lives in ``sdpa_oracle.c`` (plain C, fp64, OpenMP over rows);
this module compiles it on first use with gcc and wraps it with ctypes.  Its
inputs are float64 numpy arrays converted exactly from the half-precision
tensors by the caller.

Definition followed (per slice): S = scale*Q.K^T + bias, P = softmax_rows(S),
O = P.V -- "视觉大模型训练和推理加速" section 一 (attention map from query and
key with softmax, weighting the values) and "Accelerated Diffusers with
PyTorch 2.0" section 加速 Transformer 块 (all SDPA backends compute the same
function; the native C++ one is the high-precision path).  Variable-length
batches (``attn_varlen``) apply that definition to each sequence of the
batch on its own.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdpa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libsdpa_oracle.so")
_lock = threading.Lock()
_lib = None

BIAS_NONE, BIAS_SWIN, BIAS_SAM = 0, 1, 2


class _Bias(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int),
        ("table", ctypes.c_void_p),
        ("win", ctypes.c_int),
        ("grid_h", ctypes.c_int),
        ("grid_w", ctypes.c_int),
        ("shift", ctypes.c_int),
        ("rel_h", ctypes.c_void_p),
        ("rel_w", ctypes.c_void_p),
        ("s_h", ctypes.c_int),
        ("s_w", ctypes.c_int),
        ("k_h", ctypes.c_int),
        ("k_w", ctypes.c_int),
        ("idx_h", ctypes.c_void_p),
        ("idx_w", ctypes.c_void_p),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, -O2, OpenMP) if stale."""
    with _lock:
        fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
        if fresh and not force:
            return _LIB_PATH
        os.makedirs(_OUT_DIR, exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = build()
    lib = ctypes.CDLL(path)
    dp = ctypes.c_void_p
    i = ctypes.c_int
    lib.oracle_swin_index.argtypes = [i, i, i, i, i]
    lib.oracle_swin_index.restype = i
    lib.oracle_swin_mask.argtypes = [i, i, i, i, i, i, i]
    lib.oracle_swin_mask.restype = ctypes.c_double
    lib.oracle_bias_matrix.argtypes = [dp, i, i, i, i, i, ctypes.POINTER(_Bias), dp]
    lib.oracle_bias_matrix.restype = i
    lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, i, i, i, i, i, ctypes.c_double,
                                    ctypes.POINTER(_Bias), i]
    lib.oracle_attn_fwd.restype = i
    lib.oracle_attn_rows.argtypes = [dp, dp, dp, dp, i, i, i, i, i, ctypes.c_double,
                                     ctypes.POINTER(_Bias), dp, ctypes.c_int64, i]
    lib.oracle_attn_rows.restype = i
    lib.oracle_attn_probs.argtypes = [dp, dp, dp, i, i, i, i, i, ctypes.c_double,
                                      ctypes.POINTER(_Bias), i, dp, dp]
    lib.oracle_attn_probs.restype = i
    _lib = lib
    return lib


def _f64(a):
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


class Bias:
    """Bias description in fp64.  kind: 'none' | 'swin' | 'sam'.

    swin: table [(2M-1)^2, H], win=M, grid_h, grid_w, shift.
    sam:  rel_h [L_h, d], rel_w [L_w, d] as the model holds them, query grid
          s_h x s_w, key grid k_h x k_w (default: the query grid).  Tables
          whose length is not 2*max(query, key) - 1 are resized
          (``sam_resize``) and rows are picked by ``sam_rel_index``.
    """

    def __init__(self, kind="none", table=None, win=0, grid_h=0, grid_w=0, shift=0,
                 rel_h=None, rel_w=None, s_h=0, s_w=0, k_h=0, k_w=0):
        self.kind = kind
        self.table = None if table is None else _f64(table)
        self.rel_h = None if rel_h is None else _f64(rel_h)
        self.rel_w = None if rel_w is None else _f64(rel_w)
        self.win, self.grid_h, self.grid_w, self.shift = win, grid_h, grid_w, shift
        self.s_h, self.s_w = s_h, s_w
        self.k_h, self.k_w = (k_h or s_h), (k_w or s_w)
        if kind == "sam":
            self._rh = _f64(sam_resize(self.rel_h, 2 * max(s_h, self.k_h) - 1))
            self._rw = _f64(sam_resize(self.rel_w, 2 * max(s_w, self.k_w) - 1))
            self._ih = np.ascontiguousarray(sam_rel_index(s_h, self.k_h), dtype=np.int32)
            self._iw = np.ascontiguousarray(sam_rel_index(s_w, self.k_w), dtype=np.int32)

    def _c(self):
        k = {"none": BIAS_NONE, "swin": BIAS_SWIN, "sam": BIAS_SAM}[self.kind]
        if self.kind != "sam":
            return _Bias(k, _ptr(self.table), self.win, self.grid_h, self.grid_w, self.shift)
        return _Bias(k, None, 0, 0, 0, 0, _ptr(self._rh), _ptr(self._rw), self.s_h, self.s_w,
                     self.k_h, self.k_w, _ptr(self._ih), _ptr(self._iw))


def sam_rel_index(q_size: int, k_size: int):
    """Table row for each (query, key) coordinate pair along one axis of
    SAM's decomposed relative position ("Accelerating Generative AI (part 1),
    Segment Anything", section Bfloat16 半精度: q_coords and k_coords are
    coordinate scalers indexing rel_pos_resized).  Published definition:
    query coordinates scaled by max(k/q, 1), key coordinates by max(q/k, 1),
    offset by (k-1) * max(q/k, 1); evaluated in float32 as the published code
    does, then truncated.  Equal sizes give q_i - k_j + q - 1.  Returns
    [q_size, k_size] int64."""
    qs = np.float32(max(k_size / q_size, 1.0))
    ks = np.float32(max(q_size / k_size, 1.0))
    qc = np.arange(q_size, dtype=np.float32)[:, None] * qs
    kc = np.arange(k_size, dtype=np.float32)[None, :] * ks
    rel = (qc - kc) + np.float32((k_size - 1) * max(q_size / k_size, 1.0))
    return rel.astype(np.int64)


def sam_resize(table, L_out: int):
    """rel_pos_resized: the table linearly resampled to L_out rows when its
    length differs (half-pixel centres, source position clamped at 0, the
    upper neighbour clamped to the last row -- 1-D linear interpolation
    without corner alignment).  fp64; a table of the right length is
    returned as is."""
    t = np.asarray(table, dtype=np.float64)
    L_in = t.shape[0]
    if L_in == L_out:
        return t
    out = np.empty((L_out, t.shape[1]), dtype=np.float64)
    scale = L_in / L_out
    for m in range(L_out):
        src = max(scale * (m + 0.5) - 0.5, 0.0)
        i0 = int(src)
        i1 = min(i0 + 1, L_in - 1)
        w1 = src - i0
        out[m] = (1.0 - w1) * t[i0] + w1 * t[i1]
    return out


def _shape(q, k):
    BH, Nq, d = q.shape
    assert k.shape[0] == BH and k.shape[2] == d
    return BH, Nq, k.shape[1], d


def attn_fwd(q, k, v, H, scale, bias: Bias | None = None, nthreads: int = 0):
    """O for every row.  q [BH, Nq, d], k/v [BH, Nk, d] (any float dtype,
    converted to fp64).  Returns (out [BH, Nq, d] float64, threads used)."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    BH, Nq, Nk, d = _shape(q, k)
    out = np.empty((BH, Nq, d), dtype=np.float64)
    b = (bias or Bias())._c()
    used = lib.oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), BH, H, Nq, Nk, d,
                               float(scale), ctypes.byref(b), int(nthreads))
    if used < 0:
        raise ValueError("oracle_attn_fwd: invalid arguments")
    return out, used


def attn_rows(q, k, v, H, scale, row_ids, bias: Bias | None = None, nthreads: int = 0):
    """O for selected rows only; row_ids[t] = slice*Nq + i.  Returns
    (out [n, d] float64, threads used)."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    BH, Nq, Nk, d = _shape(q, k)
    ids = np.ascontiguousarray(row_ids, dtype=np.int64)
    out = np.empty((ids.size, d), dtype=np.float64)
    b = (bias or Bias())._c()
    used = lib.oracle_attn_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(out), BH, H, Nq, Nk, d,
                                float(scale), ctypes.byref(b), _ptr(ids), ids.size, int(nthreads))
    if used < 0:
        raise ValueError("oracle_attn_rows: invalid arguments")
    return out, used


def attn_probs(q, k, v, H, scale, slice_index, bias: Bias | None = None):
    """(P [Nq, Nk], O [Nq, d]) of one slice, fp64."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    BH, Nq, Nk, d = _shape(q, k)
    probs = np.empty((Nq, Nk), dtype=np.float64)
    out = np.empty((Nq, d), dtype=np.float64)
    b = (bias or Bias())._c()
    rc = lib.oracle_attn_probs(_ptr(q), _ptr(k), _ptr(v), BH, H, Nq, Nk, d, float(scale),
                               ctypes.byref(b), int(slice_index), _ptr(probs), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_attn_probs: invalid arguments")
    return probs, out


def attn_lse(q, k, H, scale, bias: Bias | None = None):
    """Row log-sum-exp of the scores, lse_i = log sum_j exp(scale Q_i.K_j +
    bias_ij) (natural log, fp64), the statistic a training step keeps from
    the forward pass so that P = exp(S - lse) (the Swin talk, section 二:
    forward and backward computations of the attention operators).  Plain
    definition: the explicit score matrix of each slice with the largest
    score taken out.  q [BH, Nq, d], k [BH, Nk, d]; returns [BH, Nq]."""
    q, k = _f64(q), _f64(k)
    BH, Nq, Nk, d = _shape(q, k)
    out = np.empty((BH, Nq), dtype=np.float64)
    for s in range(BH):
        S = scale * (q[s] @ k[s].T)
        if bias is not None and bias.kind != "none":
            S = S + bias_matrix(q, H, s, Nk, bias)
        m = S.max(axis=1, keepdims=True)
        out[s] = (m + np.log(np.exp(S - m).sum(axis=1, keepdims=True)))[:, 0]
    return out


def bias_matrix(q, H, slice_index, Nk, bias: Bias):
    """The bias of one slice as an explicit Nq x Nk matrix (fp64)."""
    lib = _load()
    q = _f64(q)
    BH, Nq, d = q.shape
    out = np.empty((Nq, Nk), dtype=np.float64)
    b = bias._c()
    rc = lib.oracle_bias_matrix(_ptr(q), H, int(slice_index), Nq, Nk, d, ctypes.byref(b), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_bias_matrix: invalid arguments")
    return out


def swin_index(M, ri, ci, rj, cj) -> int:
    return _load().oracle_swin_index(M, ri, ci, rj, cj)


def swin_mask(M, grid_h, grid_w, shift, window, ti, tj) -> float:
    return _load().oracle_swin_mask(M, grid_h, grid_w, shift, window, ti, tj)


def swin_partition(x, win: int, shift: int):
    """Cyclic shift then window partition of image-layout tokens, the plain
    definition ("视觉大模型训练和推理加速" section 一: attention inside windows
    of the shifted feature map; section 二: both steps are index mapping).

    x: [B_img, G_h, G_w, H, d] -> [B_img * nW, H, win * win, d], windows
    row-major over the image, tokens row-major inside a window.  Token (r, c)
    of window (wr, wc) is the image token at ((wr*win + r + shift) mod G_h,
    (wc*win + c + shift) mod G_w)."""
    x = np.roll(np.asarray(x), shift=(-shift, -shift), axis=(1, 2))
    B, Gh, Gw, H, d = x.shape
    x = x.reshape(B, Gh // win, win, Gw // win, win, H, d).transpose(0, 1, 3, 5, 2, 4, 6)
    return np.ascontiguousarray(x.reshape(B * (Gh // win) * (Gw // win), H, win * win, d))


def swin_unpartition(xw, B_img: int, G_h: int, G_w: int, win: int, shift: int):
    """Inverse of swin_partition: windows back to the image, then the
    cyclic shift undone.  xw: [B_img * nW, H, win * win, d]."""
    xw = np.asarray(xw)
    H, d = xw.shape[1], xw.shape[3]
    x = xw.reshape(B_img, G_h // win, G_w // win, H, win, win, d).transpose(0, 1, 4, 2, 5, 3, 6)
    x = x.reshape(B_img, G_h, G_w, H, d)
    return np.ascontiguousarray(np.roll(x, shift=(shift, shift), axis=(1, 2)))


def attn_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, H, scale, nthreads: int = 0):
    """Attention over a batch of sequences of different lengths, each
    attending only to itself, no bias -- a nested tensor ("PyTorch团队重写
    「分割一切」模型", Nested Tensor: data of non-uniform size, such as images
    of different sizes, batched in one tensor as {tensor, mask}).

    q [H * sum(Lq), d] is the concatenation over sequences s of [H][Lq_s][d]
    (Lq_s = cu_seqlens_q[s+1] - cu_seqlens_q[s]); k, v likewise with Lk_s.
    Each sequence is one call of ``attn_fwd`` with H slices.  Returns out
    [H * sum(Lq), d] float64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    d = q.shape[-1]
    out = np.zeros((q.shape[0], d), dtype=np.float64)
    for s in range(len(cu_seqlens_q) - 1):
        lq = cu_seqlens_q[s + 1] - cu_seqlens_q[s]
        lk = cu_seqlens_k[s + 1] - cu_seqlens_k[s]
        if lq == 0:
            continue
        if lk == 0:
            raise ValueError(f"sequence {s} has queries but no keys")
        q0, k0 = H * cu_seqlens_q[s], H * cu_seqlens_k[s]
        qs = q[q0:q0 + H * lq].reshape(H, lq, d)
        ks = k[k0:k0 + H * lk].reshape(H, lk, d)
        vs = v[k0:k0 + H * lk].reshape(H, lk, d)
        o, _ = attn_fwd(qs, ks, vs, H, scale, None, nthreads)
        out[q0:q0 + H * lq] = o.reshape(H * lq, d)
    return out


def attn_bwd(q, k, v, dout, H, scale, bias: Bias | None = None, out=None):
    """Gradients of the forward pass for training (the Swin talk, "视觉大模型训练和
    推理加速" section 二, treats the forward and the backward computation of its
    custom operators alike).  Per slice, with P and O from the forward
    definition and dO the gradient of the loss with respect to O:

        dV = P^T dO,   dP = dO V^T,   D_i = sum_c dO[i,c] O[i,c]  (= sum_j P dP),
        dS = P * (dP - D),   dQ = scale dS K,   dK = scale dS^T Q,

    and dS is the gradient of every additive bias entry.  Swin: the table row
    of each (query, key) pair of head h collects dS (the mask is constant).
    SAM: bias[i,j] = Q_i . (R_h'[ih] + R_w'[iw]) adds sum_j dS[i,j] (R_h'[ih] +
    R_w'[iw]) to dQ_i and dS[i,j] Q_i to rows ih / iw of the resampled
    tables, which the transposed resampling returns to the tables as given.

    q [BH, Nq, d], k/v [BH, Nk, d], dout [BH, Nq, d]; out, when given, is the
    forward output the caller holds (e.g. rounded to 16 bits) and D is taken
    from it, as a training step does; by default the exact O.  Returns a dict with
    dq, dk, dv and, per bias kind, d_table [(2M-1)^2, H] or d_rel_h, d_rel_w
    (fp64)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    out = None if out is None else _f64(out)
    BH, Nq, Nk, d = _shape(q, k)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    kind = bias.kind if bias is not None else "none"
    res = {}
    if kind == "swin":
        M = bias.win
        t = np.arange(M * M)
        idx = np.array([[swin_index(M, i // M, i % M, j // M, j % M) for j in t] for i in t])
        d_table = np.zeros_like(bias.table)
    elif kind == "sam":
        i_q, i_k = np.arange(Nq), np.arange(Nk)
        IH = bias._ih[(i_q // bias.s_w)[:, None], (i_k // bias.k_w)[None, :]]
        IW = bias._iw[(i_q % bias.s_w)[:, None], (i_k % bias.k_w)[None, :]]
        d_rh, d_rw = np.zeros_like(bias._rh), np.zeros_like(bias._rw)
    for s in range(BH):
        P, O = attn_probs(q, k, v, H, scale, s, bias)
        if out is not None:
            O = out[s]
        dO = dout[s]
        dv[s] = P.T @ dO
        dP = dO @ v[s].T
        D = np.sum(dO * O, axis=1, keepdims=True)
        dS = P * (dP - D)
        dq[s] = scale * (dS @ k[s])
        dk[s] = scale * (dS.T @ q[s])
        if kind == "swin":
            np.add.at(d_table[:, s % H], idx.ravel(), dS.ravel())
        elif kind == "sam":
            # the same sums a block of query rows at a time, so that the
            # [rows, Nk, d] gathers stay small on long sequences
            for i0 in range(0, Nq, 64):
                i1 = min(Nq, i0 + 64)
                dq[s, i0:i1] += np.einsum("ij,ijc->ic", dS[i0:i1], bias._rh[IH[i0:i1]] + bias._rw[IW[i0:i1]])
                contrib = (dS[i0:i1, :, None] * q[s][i0:i1, None, :]).reshape(-1, d)
                np.add.at(d_rh, IH[i0:i1].ravel(), contrib)
                np.add.at(d_rw, IW[i0:i1].ravel(), contrib)
    res.update(dq=dq, dk=dk, dv=dv)
    if kind == "swin":
        res["d_table"] = d_table
    elif kind == "sam":
        # the resampling is linear (R' = W R): its transpose carries the gradient back
        W_h = sam_resize(np.eye(bias.rel_h.shape[0]), bias._rh.shape[0])
        W_w = sam_resize(np.eye(bias.rel_w.shape[0]), bias._rw.shape[0])
        res["d_rel_h"] = W_h.T @ d_rh
        res["d_rel_w"] = W_w.T @ d_rw
    return res
