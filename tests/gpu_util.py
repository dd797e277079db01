"""Helpers shared by the GPU tests: run the CUDA path through the C ABI and
the fp64 oracle on the same seeded inputs, and compare."""
import numpy as np
import torch

import oracle
import scaled_dot_product_09_gb300 as sdpa
from scaled_dot_product_09_gb300.workloads import Inputs, Workload, make_inputs

# Tolerance stated for bf16/fp16 outputs against the fp64 oracle.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def require_gpu():
    if not torch.cuda.is_available():
        raise RuntimeError("GPU test selected but no CUDA device is visible")


def gpu_bias(w: Workload, inp: Inputs, dev="cuda"):
    if w.bias == "swin":
        return sdpa.SwinBias(inp.table.to(dev), w.win, w.grid_h, w.grid_w, w.shift)
    if w.bias == "sam":
        return sdpa.SamBias(inp.rel_h.to(dev), inp.rel_w.to(dev), w.s_h, w.s_w)
    return None


def oracle_bias(w: Workload, inp: Inputs):
    if w.bias == "swin":
        return oracle.Bias("swin", table=inp.table.double().numpy(), win=w.win, grid_h=w.grid_h,
                           grid_w=w.grid_w, shift=w.shift)
    if w.bias == "sam":
        return oracle.Bias("sam", rel_h=inp.rel_h.double().numpy(), rel_w=inp.rel_w.double().numpy(),
                           s_h=w.s_h, s_w=w.s_w)
    return None


def flat64(t):
    B, H, N, d = t.shape
    return t.double().reshape(B * H, N, d).numpy()


def run_gpu(w: Workload, inp: Inputs, scale=None):
    require_gpu()
    q, k, v = (x.cuda() for x in (inp.q, inp.k, inp.v))
    out = sdpa.attn_fwd(q, k, v, scale=w.scale if scale is None else scale, bias=gpu_bias(w, inp))
    torch.cuda.synchronize()
    assert sdpa.attn_device_status() == sdpa.ATTN_OK
    return out.cpu()


def compare(got, want, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    err = np.abs(got - want)
    mx, mn = float(err.max()), float(err.mean())
    assert mx <= max_abs and mn <= mean_abs, f"{what}: max|err| {mx:.3e} mean|err| {mn:.3e}"
    return mx, mn


def full_parity(w: Workload, seed=None):
    inp = make_inputs(w, seed)
    got = run_gpu(w, inp)
    want, _ = oracle.attn_fwd(flat64(inp.q), flat64(inp.k), flat64(inp.v), w.H, w.scale,
                              oracle_bias(w, inp))
    return compare(flat64(got), want, what=w.name)


def sampled_parity(w: Workload, n_rows=96, seed=None):
    """Full-size run; the oracle computes a deterministic sample of rows one
    by one (first and last rows of the first and last slices, plus random)."""
    inp = make_inputs(w, seed)
    got = run_gpu(w, inp)
    BH = w.B * w.H
    rng = np.random.default_rng(12345)
    fixed = [0, w.Nq - 1, (BH - 1) * w.Nq, BH * w.Nq - 1]
    ids = np.unique(np.concatenate([fixed, rng.integers(0, BH * w.Nq, n_rows)]))
    want, _ = oracle.attn_rows(flat64(inp.q), flat64(inp.k), flat64(inp.v), w.H, w.scale, ids,
                               oracle_bias(w, inp))
    got_rows = flat64(got).reshape(BH * w.Nq, w.d)[ids]
    return compare(got_rows, want, what=w.name + " (sampled)")
