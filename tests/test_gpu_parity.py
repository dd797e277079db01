"""GPU parity: the CUDA path, called through the C ABI, against the fp64
oracle on the same seeded inputs.  Tolerance: max |err| <= 2e-2 and mean
|err| <= 2e-3 on the bf16/fp16 outputs; bias indexing bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import scaled_dot_product_09_gb300 as sdpa
from scaled_dot_product_09_gb300.workloads import WORKLOADS, Workload, make_inputs

from gpu_util import (compare, flat64, full_parity, gpu_bias, oracle_bias, require_gpu, run_gpu,
                      sampled_parity)

pytestmark = pytest.mark.gpu

W = WORKLOADS


# ----------------------------------------------------- workloads, reduced --

def test_toy_full():
    full_parity(W["toy"])


def test_swin_reduced_full():
    # 2 images x 64 windows x 3 heads
    full_parity(W["swin_t_stage1"].with_(B=2 * 64))


def test_swin_ragged_tail():
    # one 21x21 image: 9 windows x 3 heads = 27 slices -> last tile holds one window
    full_parity(W["swin_t_stage1"].with_(B=9, grid_h=21, grid_w=21, seed=11))


def test_swin_no_shift():
    full_parity(W["swin_t_stage1"].with_(B=64, shift=0, seed=12))


def test_swin_many_heads():
    # Swin-T stage 2 shape (28x28 tokens, 16 windows, 6 heads): the per-head
    # bias rows exceed their shared-memory area, the bias goes through MMAs
    full_parity(W["swin_t_stage1"].with_(B=2 * 16, H=6, grid_h=28, grid_w=28, seed=13))


def test_swin_small_window():
    # 4x4 windows (16 tokens, 32-row slots), shift 2
    full_parity(W["swin_t_stage1"].with_(B=2 * 16, H=3, win=4, Nq=16, Nk=16, grid_h=16, grid_w=16,
                                          shift=2, seed=14))


def test_swin_large_window():
    # 10x10 windows (100 tokens, one slice per 128-row tile), shift 5
    full_parity(W["swin_t_stage1"].with_(B=2 * 4, H=1, win=10, Nq=100, Nk=100, grid_h=20, grid_w=20,
                                          shift=5, seed=15))


def test_sam_window_reduced_full():
    full_parity(W["sam_vith_window"].with_(B=3))


def test_sam_global_reduced_grid():
    # 16x16 grid: 256 tokens, two query and two key tiles
    full_parity(W["sam_vith_global"].with_(B=1, H=3, Nq=256, Nk=256, s_h=16, s_w=16, seed=21))


def test_sam_global_nonsquare_ragged():
    # 12x20 grid: 240 tokens, ragged last tiles, height != width
    full_parity(W["sam_vith_global"].with_(B=1, H=2, Nq=240, Nk=240, s_h=12, s_w=20, seed=22))


def test_sd_self_reduced_ragged():
    full_parity(W["sd_unet_self"].with_(B=1, H=2, Nq=1000, Nk=1000, seed=31))


def test_sd_cross_reduced():
    full_parity(W["sd_unet_cross"].with_(B=2, H=3, Nq=700))


# ------------------------------------------------------ workloads, full size --

@pytest.mark.parametrize("name", ["swin_t_stage1", "sam_vith_window", "sam_vith_global",
                                  "sam_vith_global_768", "sd_unet_self", "sd_unet_cross"])
def test_full_size_sampled(name):
    sampled_parity(W[name])


# ------------------------------------------------------------- edge shapes --

@pytest.mark.parametrize("d", [8, 16, 24, 40, 56, 64, 80, 96, 112, 128])
def test_head_dims(d):
    w = Workload("edge_d", B=1, H=2, Nq=150, Nk=200, d=d, dtype="bf16", bias="none", seed=40 + d)
    full_parity(w)


@pytest.mark.parametrize("nq,nk", [(1, 1), (1, 300), (300, 1), (128, 128), (129, 129),
                                   (64, 64), (7, 9), (33, 100), (200, 50)])
def test_lengths(nq, nk):
    w = Workload("edge_n", B=2, H=3, Nq=nq, Nk=nk, d=32, dtype="fp16", bias="none", seed=nq * 7 + nk)
    full_parity(w)


@pytest.mark.parametrize("d,nk", [(16, 77), (32, 1), (40, 77), (48, 80), (40, 33)])
def test_one_key_tile_pipeline(d, nk):
    """At most 80 keys and head dims up to 48: jobs of one score tile, the
    next job's S issued early and each output written during the next job;
    256 jobs over the CTAs, so CTAs run several in a row."""
    w = Workload("cross", B=4, H=8, Nq=2000, Nk=nk, d=d, dtype="fp16", bias="none", seed=60 + d + nk)
    full_parity(w)


def test_single_slice():
    full_parity(Workload("bh1", B=1, H=1, Nq=77, Nk=333, d=40, dtype="fp16", bias="none", seed=5))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_dtypes(dtype):
    full_parity(Workload("dt", B=2, H=2, Nq=256, Nk=256, d=64, dtype=dtype, bias="none", seed=9))


def test_large_scores_stay_finite():
    """Scores of a few hundred: the online softmax must rescale, not overflow."""
    w = Workload("big", B=1, H=1, Nq=256, Nk=512, d=64, dtype="bf16", bias="none", seed=3)
    inp = make_inputs(w)
    inp.q = (inp.q.float() * 4).to(torch.bfloat16)
    got = run_gpu(w, inp, scale=1.0)
    want, _ = oracle.attn_fwd(flat64(inp.q), flat64(inp.k), flat64(inp.v), 1, 1.0)
    compare(flat64(got), want, what="large scores")


NONPOS_SCALE_CASES = {
    "none_shared_ragged": Workload("np1", B=1, H=2, Nq=300, Nk=333, d=64, dtype="bf16", bias="none", seed=11),
    "none_packed": Workload("np2", B=3, H=2, Nq=49, Nk=40, d=32, dtype="fp16", bias="none", seed=12),
    "none_one_tile": Workload("np3", B=2, H=2, Nq=300, Nk=77, d=40, dtype="fp16", bias="none", seed=13),
    "swin_rows": W["swin_t_stage1"].with_(B=64, seed=14),
    "sam_64x64": W["sam_vith_global"].with_(B=1, H=2, seed=15),
    "sam_14x14": W["sam_vith_window"].with_(B=2, H=2, seed=16),
}


@pytest.mark.parametrize("scale", [0.0, -0.3])
@pytest.mark.parametrize("case", sorted(NONPOS_SCALE_CASES))
def test_nonpositive_scale(case, scale):
    """scale = 0 (every key weighted by its bias alone: the mean of V without
    bias) and a negative scale (the score order flips), against the oracle;
    masked key padding must stay at weight zero either way."""
    w = NONPOS_SCALE_CASES[case]
    inp = make_inputs(w)
    got = run_gpu(w, inp, scale=scale)
    want, _ = oracle.attn_fwd(flat64(inp.q), flat64(inp.k), flat64(inp.v), w.H, scale, oracle_bias(w, inp))
    compare(flat64(got), want, what=f"{case} scale {scale}")


def test_output_not_aliasing_and_repeatable():
    w = W["toy"]
    inp = make_inputs(w)
    a = run_gpu(w, inp)
    b = run_gpu(w, inp)
    assert torch.equal(a, b)


# ------------------------------------------------------- bias bit-exactness --

SWIN_BIAS_CASES = {
    "rows": dict(B=64),
    "mma_many_heads": dict(B=16, H=6, grid_h=28, grid_w=28),
    "rows_small_window": dict(B=16, win=4, Nq=16, Nk=16, grid_h=16, grid_w=16, shift=2),
    "mma_large_window": dict(B=4, H=1, win=10, Nq=100, Nk=100, grid_h=20, grid_w=20, shift=5),
}


@pytest.mark.parametrize("case", sorted(SWIN_BIAS_CASES))
def test_swin_bias_indexing_bit_exact(case):
    """table[r, h] = r + 256*h is exact in fp32 (and in fp16 up to 2048): the
    in-kernel gather must return index + 256*h (+ -100 across regions)
    exactly, for the bias added by the softmax and by MMAs."""
    require_gpu()
    w = W["swin_t_stage1"].with_(**SWIN_BIAS_CASES[case])
    M, H = w.win, w.H
    table = torch.tensor([[r + 256.0 * h for h in range(H)] for r in range((2 * M - 1) ** 2)])
    inp = make_inputs(w)
    inp.table = table
    q, k, v = (x.cuda() for x in (inp.q, inp.k, inp.v))
    got = sdpa.attn_debug_bias(q, k, v, scale=w.scale, bias=gpu_bias(w, inp)).cpu().double()
    b = oracle_bias(w, inp)
    for s in range(0, w.B * H, 7):
        want = oracle.bias_matrix(flat64(inp.q), H, s, w.Nk, b)
        np.testing.assert_array_equal(got.reshape(-1, w.Nq, w.Nk)[s].numpy(), want)


def test_sam_bias_indexing_bit_exact():
    """Integer tables R_h[r,0] = r, R_w[r,1] = r and Q = 128*e0 + e1 make
    the decomposed term 128*(qh-kh+S_h-1) + (qw-kw+S_w-1), exact in bf16
    operands with fp32 accumulation."""
    require_gpu()
    w = W["sam_vith_global"].with_(B=1, H=2, Nq=240, Nk=240, s_h=12, s_w=20)
    inp = make_inputs(w)
    Rh = torch.zeros(2 * w.s_h - 1, w.d)
    Rh[:, 0] = torch.arange(2 * w.s_h - 1)
    Rw = torch.zeros(2 * w.s_w - 1, w.d)
    Rw[:, 1] = torch.arange(2 * w.s_w - 1)
    inp.rel_h, inp.rel_w = Rh.to(torch.bfloat16), Rw.to(torch.bfloat16)
    qq = torch.zeros_like(inp.q, dtype=torch.float32)
    qq[..., 0], qq[..., 1] = 128.0, 1.0
    inp.q = qq.to(torch.bfloat16)
    q, k, v = (x.cuda() for x in (inp.q, inp.k, inp.v))
    got = sdpa.attn_debug_bias(q, k, v, scale=w.scale, bias=gpu_bias(w, inp)).cpu().double()
    b = oracle_bias(w, inp)
    for s in range(w.B * w.H):
        want = oracle.bias_matrix(flat64(inp.q), w.H, s, w.Nk, b)
        np.testing.assert_array_equal(got.reshape(-1, w.Nq, w.Nk)[s].numpy(), want)


def test_sam_window_bias_indexing_bit_exact():
    _sam_bias_bit_exact(W["sam_vith_window"].with_(B=2, H=2))


def test_sam_global_64x64_bias_indexing_bit_exact():
    # the kernel specialised for 64x64 grids (6-bit G-row shifts, 2-row key tiles)
    _sam_bias_bit_exact(W["sam_vith_global"].with_(B=1, H=2), slices=(0, 1), rows=range(0, 4096, 37))


def test_sam_global_48x48_bias_indexing_bit_exact():
    # the kernel specialised for 48x48 grids (48-key tiles of one grid row, two score buffers)
    _sam_bias_bit_exact(W["sam_vith_global_768"].with_(B=1, H=2, rel_len=0), slices=(0, 1),
                        rows=range(0, 2304, 23))


def test_sam_resampled_tables_48x48_full():
    # 127-row tables resampled to 95 rows in the 48x48 kernel (768-pixel input)
    full_parity(W["sam_vith_global_768"].with_(B=1, H=2, seed=72))


def _sam_bias_bit_exact(w, slices=None, rows=None):
    require_gpu()
    inp = make_inputs(w)
    Rh = torch.zeros(2 * w.s_h - 1, w.d)
    Rh[:, 0] = torch.arange(2 * w.s_h - 1)
    Rw = torch.zeros(2 * w.s_w - 1, w.d)
    Rw[:, 1] = torch.arange(2 * w.s_w - 1)
    inp.rel_h, inp.rel_w = Rh.to(torch.bfloat16), Rw.to(torch.bfloat16)
    qq = torch.zeros_like(inp.q, dtype=torch.float32)
    qq[..., 0], qq[..., 1] = 128.0, 1.0
    inp.q = qq.to(torch.bfloat16)
    q, k, v = (x.cuda() for x in (inp.q, inp.k, inp.v))
    got = sdpa.attn_debug_bias(q, k, v, scale=w.scale, bias=gpu_bias(w, inp)).cpu().double()
    got = got.reshape(-1, w.Nq, w.Nk)
    b = oracle_bias(w, inp)
    for s in (slices if slices is not None else range(w.B * w.H)):
        want = oracle.bias_matrix(flat64(inp.q), w.H, s, w.Nk, b)
        r = list(rows) if rows is not None else slice(None)
        np.testing.assert_array_equal(got[s].numpy()[r], want[r])


# ------------------------------------------- SAM on unequal grids, resampled --
# Query grid != key grid (coordinate scalers) and tables of another length
# than 2*max(q, k)-1 (linear resampling, which the kernel applies to G = Q.R).

SAM_GENERAL_CASES = {
    # name: (query grid, key grid, rel_h rows, rel_w rows)
    "keys_coarser": ((12, 12), (6, 6), 23, 23),
    "keys_finer": ((6, 8), (12, 16), 23, 31),
    "aspect": ((20, 10), (5, 40), 39, 79),
    "resample_down": ((14, 14), (14, 14), 40, 40),
    "resample_up": ((16, 16), (16, 16), 9, 13),
    "both": ((10, 12), (7, 9), 30, 11),
}


def _sam_general_inputs(qg, kg, lh, lw, H=2, d=80, seed=70):
    g = torch.Generator().manual_seed(seed)
    Nq, Nk = qg[0] * qg[1], kg[0] * kg[1]
    q = torch.randn(1, H, Nq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(1, H, Nk, d, generator=g).to(torch.bfloat16)
    v = torch.randn(1, H, Nk, d, generator=g).to(torch.bfloat16)
    rh = (torch.randn(lh, d, generator=g) * 0.05).to(torch.bfloat16)
    rw = (torch.randn(lw, d, generator=g) * 0.05).to(torch.bfloat16)
    return q, k, v, rh, rw


@pytest.mark.parametrize("case", sorted(SAM_GENERAL_CASES))
def test_sam_general_full(case):
    require_gpu()
    qg, kg, lh, lw = SAM_GENERAL_CASES[case]
    q, k, v, rh, rw = _sam_general_inputs(qg, kg, lh, lw)
    H, d = q.shape[1], q.shape[3]
    scale = d ** -0.5
    out = sdpa.attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale,
                        bias=sdpa.SamBias(rh.cuda(), rw.cuda(), qg[0], qg[1], kg[0], kg[1]))
    torch.cuda.synchronize()
    assert sdpa.attn_device_status() == sdpa.ATTN_OK
    b = oracle.Bias("sam", rel_h=rh.double().numpy(), rel_w=rw.double().numpy(), s_h=qg[0], s_w=qg[1],
                    k_h=kg[0], k_w=kg[1])
    want, _ = oracle.attn_fwd(flat64(q), flat64(k), flat64(v), H, scale, b)
    compare(flat64(out.cpu()), want, what=f"sam general {case}")


@pytest.mark.parametrize("qg,kg", [((12, 12), (6, 6)), ((6, 8), (12, 16)), ((20, 10), (5, 40))])
def test_sam_unequal_grids_bias_indexing_bit_exact(qg, kg):
    """Integer tables (R_h[r,0] = r, R_w[r,1] = r) of the addressed length and
    Q = 128*e0 + e1: the bias is 128*ih + iw exactly, so every float32
    coordinate-scaler index must match the oracle's."""
    require_gpu()
    lh, lw = 2 * max(qg[0], kg[0]) - 1, 2 * max(qg[1], kg[1]) - 1
    q, k, v, _, _ = _sam_general_inputs(qg, kg, lh, lw, seed=71)
    d = q.shape[3]
    rh = torch.zeros(lh, d)
    rh[:, 0] = torch.arange(lh)
    rw = torch.zeros(lw, d)
    rw[:, 1] = torch.arange(lw)
    rh, rw = rh.to(torch.bfloat16), rw.to(torch.bfloat16)
    qq = torch.zeros_like(q, dtype=torch.float32)
    qq[..., 0], qq[..., 1] = 128.0, 1.0
    q = qq.to(torch.bfloat16)
    got = sdpa.attn_debug_bias(q.cuda(), k.cuda(), v.cuda(), scale=d ** -0.5,
                               bias=sdpa.SamBias(rh.cuda(), rw.cuda(), qg[0], qg[1], kg[0], kg[1]))
    got = got.cpu().double().reshape(-1, qg[0] * qg[1], kg[0] * kg[1])
    b = oracle.Bias("sam", rel_h=rh.double().numpy(), rel_w=rw.double().numpy(), s_h=qg[0], s_w=qg[1],
                    k_h=kg[0], k_w=kg[1])
    for s_ in range(got.shape[0]):
        want = oracle.bias_matrix(flat64(q), q.shape[1], s_, kg[0] * kg[1], b)
        np.testing.assert_array_equal(got[s_].numpy(), want)


# ----------------------------------------------- Swin image token layout --
# q/k/v/out as [images, grid_h, grid_w, H, d]: the kernel folds the cyclic
# shift and the window partition into its row gathers and their inverse into
# its stores.  Image inputs are the windows-layout inputs mapped back through
# the oracle's inverse partition (an exact index permutation); the expected
# output is the oracle's window attention mapped the same way.

SWIN_IMAGE_CASES = {
    "stage1": dict(B=2 * 64),
    "no_shift": dict(B=64, shift=0, seed=12),
    "ragged_tail": dict(B=9, grid_h=21, grid_w=21, seed=11),
    "mma_many_heads": dict(B=2 * 16, H=6, grid_h=28, grid_w=28, seed=13),
    "small_window": dict(B=2 * 16, win=4, Nq=16, Nk=16, grid_h=16, grid_w=16, shift=2, seed=14),
    "large_window": dict(B=2 * 4, H=1, win=10, Nq=100, Nk=100, grid_h=20, grid_w=20, shift=5, seed=15),
    # rings of 2..5 stages, each with enough jobs that CTAs wrap their ring
    # (the gather keeps fewer tiles in flight on shorter rings):
    # d=64 with bias MMAs: 2 stages, 192 jobs
    "ring2_d64_mma": dict(B=32 * 4, H=6, d=64, grid_h=14, grid_w=14, seed=16),
    # d=64 with bias rows: 3 stages, 192 jobs
    "ring3_d64_rows": dict(B=4 * 64, d=64, seed=18),
    # d=48 with bias rows: 4 stages, 384 jobs
    "ring4_d48_rows": dict(B=8 * 64, d=48, seed=19),
    # 6 heads, bias MMAs: 5 stages, 384 jobs
    "ring5_mma_many_heads": dict(B=16 * 16, H=6, grid_h=28, grid_w=28, seed=20),
    "bf16": dict(B=64, dtype="bf16", seed=17),
    # d not a multiple of 16: zero column padding written by the gathers
    "d40_gathered": dict(B=2 * 64, d=40, seed=21),
}


def _images(w):
    return w.B // ((w.grid_h // w.win) * (w.grid_w // w.win))


def _to_image(t, w):
    """[B windows, H, win^2, d] -> [images, grid_h, grid_w, H, d], bit-exact."""
    raw = t.view(torch.int16).numpy()
    img = oracle.swin_unpartition(raw, _images(w), w.grid_h, w.grid_w, w.win, w.shift)
    return torch.from_numpy(img).view(t.dtype)


def _image_bias(w, inp):
    return sdpa.SwinBias(inp.table.cuda(), w.win, w.grid_h, w.grid_w, w.shift, layout="image")


@pytest.mark.parametrize("case", sorted(SWIN_IMAGE_CASES))
def test_swin_image_layout_full(case):
    require_gpu()
    w = W["swin_t_stage1"].with_(**SWIN_IMAGE_CASES[case])
    inp = make_inputs(w)
    q, k, v = (_to_image(x, w).cuda() for x in (inp.q, inp.k, inp.v))
    out = sdpa.attn_fwd(q, k, v, scale=w.scale, bias=_image_bias(w, inp))
    torch.cuda.synchronize()
    assert sdpa.attn_device_status() == sdpa.ATTN_OK
    assert out.shape == (_images(w), w.grid_h, w.grid_w, w.H, w.d)
    want, _ = oracle.attn_fwd(flat64(inp.q), flat64(inp.k), flat64(inp.v), w.H, w.scale, oracle_bias(w, inp))
    want = oracle.swin_unpartition(want.reshape(w.B, w.H, w.Nq, w.d), _images(w), w.grid_h, w.grid_w,
                                   w.win, w.shift)
    compare(out.cpu().double().numpy(), want, what=f"swin image {case}")
    # same smem tiles as the windows-layout path: identical bits
    win_out = run_gpu(w, inp)
    assert torch.equal(out.cpu().view(torch.int16), _to_image(win_out, w).view(torch.int16))


def test_swin_image_layout_full_size_matches_windows_layout():
    """Full Swin-T stage-1 batch: the image-layout call returns, bit for bit,
    the windows-layout result mapped back to the image (the windows layout is
    itself checked against the oracle at this size)."""
    require_gpu()
    w = W["swin_t_stage1"]
    inp = make_inputs(w)
    win_out = run_gpu(w, inp)
    q, k, v = (_to_image(x, w).cuda() for x in (inp.q, inp.k, inp.v))
    out = sdpa.attn_fwd(q, k, v, scale=w.scale, bias=_image_bias(w, inp))
    torch.cuda.synchronize()
    assert sdpa.attn_device_status() == sdpa.ATTN_OK
    assert torch.equal(out.cpu().view(torch.int16), _to_image(win_out, w).view(torch.int16))


# ------------------------------------------------------ bounded-wait failure --

def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait that nothing completes gives up after its limit, the status word
    carries its code, and the next attention call on the same context works."""
    require_gpu()
    assert sdpa.attn_device_status() == sdpa.ATTN_OK
    sdpa.selftest_wait_timeout(20000)  # 20 ms
    assert sdpa.attn_device_status() == sdpa.ATTN_ERR_DEVICE_TIMEOUT
    assert b"code 9" in sdpa.load_library().attn_last_error()
    assert sdpa.attn_device_status() == sdpa.ATTN_OK  # read and cleared
    full_parity(W["toy"])
    assert sdpa.attn_device_status() == sdpa.ATTN_OK
