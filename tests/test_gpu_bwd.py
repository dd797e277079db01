"""GPU parity of the backward pass (windows, long sequences, the Swin and SAM
biases) against the fp64 oracle's attn_bwd on the same seeded inputs,
through the C ABI.

Tolerance: dQ, dK and dV are 16-bit outputs and are held to the bound
stated for every 16-bit output against the fp64 oracle, max |err| <= 2e-2
and mean |err| <= 2e-3 over each tensor.  The fp32 table gradient sums many
dS terms, each off by fp32 rounding only (the oracle takes D from the same
16-bit O): |err| <= 1e-3 + 1e-3 |want| per element; the SAM table
gradients (fp32 sums of fp32 row sums of dS) are held to the same bound."""
import numpy as np
import pytest
import torch

import oracle
import scaled_dot_product_09_gb300 as sdpa
from scaled_dot_product_09_gb300.workloads import WORKLOADS, Workload, make_inputs

from gpu_util import compare, flat64, gpu_bias, oracle_bias, require_gpu

pytestmark = pytest.mark.gpu

W = WORKLOADS


def _check_table(got, want, what, atol=1e-3, rtol=1e-3):
    """fp32 bias gradients: |err| <= atol * max(1, max |want|) + rtol * |want|
    per element.  Each entry is a sum over every query row of a slice batch;
    the rounding of its terms (fp32 sums, the 16-bit P in dS, the fp16 bias
    terms) follows the size of the summands, i.e. the gradient's overall
    scale, so the absolute floor scales with the largest entry."""
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - want)
    bad = err > atol * max(1.0, float(np.abs(want).max())) + rtol * np.abs(want)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off, max |err| {err.max():.3e}"


def _sam_resized_rounded(w: Workload, inp):
    """SAM tables of another length than 2 * side - 1, read as the kernels
    read them: resampled (the oracle's rel_pos_resized) and rounded to the
    model dtype, as the model's resized tensor is.  Returns the oracle bias on
    those tables and, per table, the resampling matrix A [2S-1][L] (A applied
    to the unit rows), whose transpose returns a gradient to the table."""
    L = 2 * w.s_h - 1
    rz = [torch.from_numpy(oracle.sam_resize(t.double().numpy(), L)).to(t.dtype).double().numpy()
          for t in (inp.rel_h, inp.rel_w)]
    A = [oracle.sam_resize(np.eye(t.shape[0]), L) for t in (inp.rel_h, inp.rel_w)]
    return oracle.Bias("sam", rel_h=rz[0], rel_w=rz[1], s_h=w.s_h, s_w=w.s_w), A


def _bwd_case(w: Workload, seed=None, use_lse=False):
    require_gpu()
    inp = make_inputs(w, seed)
    g = torch.Generator().manual_seed(w.seed + 1000)
    dout = torch.randn(inp.q.shape, generator=g).to(inp.q.dtype)
    q, k, v, do = (x.cuda() for x in (inp.q, inp.k, inp.v, dout))
    bias = gpu_bias(w, inp)
    out, lse = sdpa.attn_fwd_train(q, k, v, scale=w.scale, bias=bias)
    dq, dk, dv, dtab = sdpa.attn_bwd(q, k, v, out, do, lse=lse if use_lse or w.Nq > 128 or w.Nk > 128 else None,
                                     scale=w.scale, bias=bias)
    torch.cuda.synchronize()
    assert sdpa.attn_device_status() == sdpa.ATTN_OK
    resized = w.bias == "sam" and w.rel_len and w.rel_len != 2 * w.s_h - 1
    ob, A = _sam_resized_rounded(w, inp) if resized else (oracle_bias(w, inp), None)
    # D = rowsum(dO * O) from the 16-bit O the kernel was given
    want = oracle.attn_bwd(flat64(inp.q), flat64(inp.k), flat64(inp.v), flat64(dout), w.H, w.scale,
                           ob, out=flat64(out.cpu()))
    if resized:
        want["d_rel_h"], want["d_rel_w"] = A[0].T @ want["d_rel_h"], A[1].T @ want["d_rel_w"]
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        compare(flat64(t.cpu()), want[name], what=f"{w.name} {name}")
    if w.bias == "swin":
        _check_table(dtab.cpu().double().numpy(), want["d_table"], f"{w.name} d_table")
    if w.bias == "sam":
        _check_table(dtab[0].cpu().double().numpy(), want["d_rel_h"], f"{w.name} d_rel_h")
        _check_table(dtab[1].cpu().double().numpy(), want["d_rel_w"], f"{w.name} d_rel_w")


def test_bwd_no_bias_short():
    _bwd_case(Workload("bwd_none", B=2, H=3, Nq=49, Nk=77, d=32, dtype="bf16", bias="none", seed=80))


@pytest.mark.parametrize("nq,nk,d", [(1, 1, 8), (128, 128, 64), (100, 30, 40), (17, 128, 16)])
def test_bwd_no_bias_shapes(nq, nk, d):
    _bwd_case(Workload("bwd_shape", B=1, H=2, Nq=nq, Nk=nk, d=d, dtype="fp16", bias="none", seed=81 + nq))


def test_bwd_swin_reduced():
    # 2 images x 64 windows of 7x7, 3 heads, shift 3
    _bwd_case(W["swin_t_stage1"].with_(B=2 * 64, seed=82))


def test_bwd_swin_small_window_and_ragged_grid():
    _bwd_case(W["swin_t_stage1"].with_(B=2 * 16, win=4, Nq=16, Nk=16, grid_h=16, grid_w=16, shift=2, seed=83))
    _bwd_case(W["swin_t_stage1"].with_(B=9, grid_h=21, grid_w=21, dtype="bf16", seed=84))


def test_bwd_swin_full_size():
    """Swin-T stage 1, all 32 images: every gradient against the oracle."""
    _bwd_case(W["swin_t_stage1"])


# --------------------------------------------------------- long sequences --
# Two tensor-core passes (key blocks: dK, dV; query blocks: dQ) from the
# forward's row log-sum-exp.

@pytest.mark.parametrize("nq,nk,d,dtype", [(300, 300, 64, "bf16"), (200, 513, 40, "fp16"), (257, 129, 80, "bf16"),
                                           (129, 40, 32, "fp16"), (60, 700, 16, "bf16")])
def test_bwd_long_no_bias(nq, nk, d, dtype):
    _bwd_case(Workload("bwd_long", B=1, H=2, Nq=nq, Nk=nk, d=d, dtype=dtype, bias="none", seed=90 + nq + nk))


def test_bwd_long_windows_path_with_lse():
    # a short sequence with d > 64 takes the long path too
    _bwd_case(Workload("bwd_d80", B=2, H=2, Nq=100, Nk=77, d=80, dtype="bf16", bias="none", seed=95), use_lse=True)


def test_bwd_long_sd_self_4096():
    """Stable Diffusion self-attention rows (4096 tokens, d = 40) on two
    slices: every gradient against the oracle."""
    _bwd_case(W["sd_unet_self"].with_(B=1, H=2, seed=96))


# ------------------------------------------------------------- SAM rel-pos --
# dQ, dK, dV and the gradients of both rel-pos tables (d_rel_h, d_rel_w).

def test_bwd_sam_window_14x14():
    """SAM windowed attention (14 x 14 windows, 196 tokens, d = 80)."""
    _bwd_case(W["sam_vith_window"].with_(B=2, H=2, seed=97), use_lse=True)


def test_bwd_sam_global_64x64():
    """SAM global attention on the 64 x 64 grid (4096 tokens, d = 80), one slice."""
    _bwd_case(W["sam_vith_global"].with_(B=1, H=1, seed=98), use_lse=True)


@pytest.mark.parametrize("case", ["48x48_tables127", "14x14_tables31_fp16", "64x64_tables95"])
def test_bwd_sam_48_and_resampled_tables(case):
    """The 48 x 48 grid (a 768-pixel input) with the 1024-pixel model's
    127-row tables, and 14 x 14 / 64 x 64 grids with tables of another length:
    the backward runs on the tables resampled to 2 * side - 1 rows as the
    forward does, and returns their gradients through the transposed
    resampling; every gradient against the oracle."""
    w = {"48x48_tables127": W["sam_vith_global_768"].with_(B=1, H=1, seed=103),
         "14x14_tables31_fp16": W["sam_vith_window"].with_(B=1, H=2, rel_len=31, dtype="fp16", seed=104),
         "64x64_tables95": W["sam_vith_global"].with_(B=1, H=1, rel_len=95, seed=105)}[case]
    _bwd_case(w, use_lse=True)


@pytest.mark.parametrize("case", ["14x14_d56_fp16", "64x64_d64_bf16"])
def test_bwd_sam_narrow_heads(case):
    """Head dims padded to 64 (d = 56: a partial 16-column block; d = 64),
    fp16 and bf16: the rel pre-pass and both passes in their 64-column
    instantiations."""
    w = {"14x14_d56_fp16": W["sam_vith_window"].with_(B=1, H=3, d=56, dtype="fp16", seed=101),
         "64x64_d64_bf16": W["sam_vith_global"].with_(B=1, H=1, d=64, seed=102)}[case]
    _bwd_case(w, use_lse=True)


# ------------------------------------------------- Swin image token layout --
def _images(w):
    return w.B // ((w.grid_h // w.win) * (w.grid_w // w.win))


def _to_image(t, w):
    """[B windows, H, win^2, d] -> [images, grid_h, grid_w, H, d], bit-exact."""
    raw = t.reshape(w.B, w.H, w.Nq, w.d).view(torch.int16).numpy()
    return torch.from_numpy(oracle.swin_unpartition(raw, _images(w), w.grid_h, w.grid_w, w.win, w.shift)).view(t.dtype)


@pytest.mark.parametrize("case", ["swin_t_stage1_2img", "ragged_grid_21"])
def test_bwd_swin_image_layout_matches_windows_layout(case):
    """The image-layout backward (the kernel gathers each window's rows and
    writes the gradients back to their image positions) returns, bit for
    bit, the windows-layout backward's gradients mapped back to the image,
    and the same table gradient (the windows layout is checked against the
    oracle above)."""
    require_gpu()
    w = {"swin_t_stage1_2img": W["swin_t_stage1"].with_(B=2 * 64, seed=91),
         "ragged_grid_21": W["swin_t_stage1"].with_(B=9, grid_h=21, grid_w=21, seed=92)}[case]
    inp = make_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 1000)
    dout = torch.randn(inp.q.shape, generator=g).to(inp.q.dtype)
    qw, kw, vw, dow = (x.cuda() for x in (inp.q, inp.k, inp.v, dout))
    bw = gpu_bias(w, inp)
    ow, lse = sdpa.attn_fwd_train(qw, kw, vw, scale=w.scale, bias=bw)
    want = sdpa.attn_bwd(qw, kw, vw, ow, dow, scale=w.scale, bias=bw)
    bi = sdpa.SwinBias(inp.table.cuda(), w.win, w.grid_h, w.grid_w, w.shift, layout="image")
    qi, ki, vi, oi, doi = (_to_image(x.cpu(), w).cuda() for x in (qw, kw, vw, ow, dow))
    got = sdpa.attn_bwd(qi, ki, vi, oi, doi, scale=w.scale, bias=bi)
    torch.cuda.synchronize()
    assert sdpa.attn_device_status() == sdpa.ATTN_OK
    for name, a, b in zip(("dq", "dk", "dv"), got[:3], want[:3]):
        assert a.shape == (_images(w), w.grid_h, w.grid_w, w.H, w.d), name
        assert torch.equal(a.cpu().view(torch.int16), _to_image(b.cpu(), w).view(torch.int16)), name
    # the table gradient sums the same fp32 terms; the CTAs add their sums to
    # the table with atomics, in an order that varies from call to call
    np.testing.assert_allclose(got[3].cpu().numpy(), want[3].cpu().numpy(), rtol=1e-4, atol=1e-5)
