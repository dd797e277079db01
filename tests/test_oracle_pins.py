"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these compares the oracle with a retyped copy of itself: each pin is
a hand-enumerated fixture, a closed form, an invariant, a brute-force
geometric characterisation, or an independent library routine
(torch's CPU scaled_dot_product_attention, the pages' "native C++"
backend -- "Accelerated Diffusers with PyTorch 2.0", section 加速 Transformer 块).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from scaled_dot_product_09_gb300.workloads import WORKLOADS, make_inputs


def _rand(shape, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * scale


def _read_golden(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


# ------------------------------------------------------------------ softmax --

@pytest.mark.parametrize("kind", ["none", "swin", "sam"])
def test_p1_rows_sum_to_one(kind):
    """P1: every probability row sums to 1 (softmax definition)."""
    H, d = 2, 8
    if kind == "swin":
        M = 3
        N = M * M
        bias = oracle.Bias("swin", table=_rand(((2 * M - 1) ** 2, H), 7, 0.5), win=M,
                           grid_h=6, grid_w=6, shift=1)
        BH = 4 * H
    elif kind == "sam":
        sh, sw = 3, 4
        N = sh * sw
        bias = oracle.Bias("sam", rel_h=_rand((2 * sh - 1, d), 8, 0.3),
                           rel_w=_rand((2 * sw - 1, d), 9, 0.3), s_h=sh, s_w=sw)
        BH = 2 * H
    else:
        N, bias, BH = 13, None, 2 * H
    q, k, v = (_rand((BH, N, d), s) for s in (1, 2, 3))
    for s in range(BH):
        P, _ = oracle.attn_probs(q, k, v, H, 0.37, s, bias)
        assert np.all(P >= 0)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)


def test_p2_uniform_scores_give_mean_of_v():
    """P2: Q = 0 makes every score equal, so O is the column mean of V."""
    BH, H, N, d = 3, 3, 17, 8
    q = np.zeros((BH, N, d))
    k, v = _rand((BH, N, d), 4), _rand((BH, N, d), 5)
    out, _ = oracle.attn_fwd(q, k, v, H, 0.25)
    want = np.broadcast_to(v.mean(axis=1, keepdims=True), out.shape)
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-14)


def test_single_key_returns_that_value():
    """Nk = 1: the only key gets probability 1, O = V[0] exactly."""
    q, k, v = _rand((2, 5, 8), 1), _rand((2, 1, 8), 2), _rand((2, 1, 8), 3)
    out, _ = oracle.attn_fwd(q, k, v, 1, 1.0)
    np.testing.assert_array_equal(out, np.broadcast_to(v, out.shape))


def test_large_scores_are_stable_and_pick_the_argmax():
    """A key whose score dominates by >> 40 gets all the weight; no overflow."""
    d = 4
    q = np.array([[[1.0, 0, 0, 0]]])
    k = np.array([[[1000.0, 0, 0, 0], [900.0, 0, 0, 0], [-1000.0, 0, 0, 0]]])
    v = np.array([[[1.0, 2, 3, 4], [5.0, 6, 7, 8], [9.0, 9, 9, 9]]])
    out, _ = oracle.attn_fwd(q, k, v, 1, 1.0)
    np.testing.assert_array_equal(out[0, 0], v[0, 0])


def test_p9_matches_torch_sdpa_fp64():
    """P9: no-bias attention equals torch's CPU SDPA math backend in fp64."""
    B, H, Nq, Nk, d = 2, 3, 19, 23, 16
    q, k, v = _rand((B * H, Nq, d), 1), _rand((B * H, Nk, d), 2), _rand((B * H, Nk, d), 3)
    scale = 1 / math.sqrt(d)
    out, _ = oracle.attn_fwd(q, k, v, H, scale)
    t = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), scale=scale)
    np.testing.assert_allclose(out, t.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("kind", ["swin", "sam"])
def test_p9_biased_matches_torch_sdpa_with_explicit_mask(kind):
    """The attention half of the biased path equals torch SDPA given the
    oracle's explicit bias matrix as an additive float mask."""
    H, d = 2, 8
    if kind == "swin":
        M = 3
        N = M * M
        bias = oracle.Bias("swin", table=_rand(((2 * M - 1) ** 2, H), 7), win=M,
                           grid_h=6, grid_w=9, shift=1)
        BH = 6 * H
    else:
        sh, sw = 3, 5
        N = sh * sw
        bias = oracle.Bias("sam", rel_h=_rand((2 * sh - 1, d), 8), rel_w=_rand((2 * sw - 1, d), 9),
                           s_h=sh, s_w=sw)
        BH = 2 * H
    q, k, v = (_rand((BH, N, d), s) for s in (1, 2, 3))
    out, _ = oracle.attn_fwd(q, k, v, H, 0.3, bias)
    for s in range(BH):
        Bm = oracle.bias_matrix(q, H, s, N, bias)
        t = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[s:s + 1]), torch.from_numpy(k[s:s + 1]),
            torch.from_numpy(v[s:s + 1]), attn_mask=torch.from_numpy(Bm)[None], scale=0.3)
        np.testing.assert_allclose(out[s], t[0].numpy(), rtol=0, atol=1e-12)


def test_rows_entry_equals_full_entry():
    BH, H, N, d = 4, 2, 11, 8
    q, k, v = (_rand((BH, N, d), s) for s in (1, 2, 3))
    full, _ = oracle.attn_fwd(q, k, v, H, 0.5)
    ids = np.array([0, 5, 12, 43, 21])
    rows, _ = oracle.attn_rows(q, k, v, H, 0.5, ids)
    np.testing.assert_array_equal(rows, full.reshape(-1, d)[ids])


# --------------------------------------------------------------------- Swin --

def test_p5_swin_index_2x2_golden(golden_dir):
    """P5: the hand-enumerated index matrix of one 2x2 window."""
    want = np.array(_read_golden(os.path.join(golden_dir, "swin_index_M2.txt")), dtype=int)
    got = np.array([[oracle.swin_index(2, i // 2, i % 2, j // 2, j % 2) for j in range(4)]
                    for i in range(4)])
    np.testing.assert_array_equal(got, want)


def test_p4_swin_index_invariants():
    """P4: idx(i,i) = 2M(M-1) (84 for M=7); idx(i,j)+idx(j,i) = 2*idx(i,i);
    range [0, (2M-1)^2); for a fixed query all keys get distinct indices."""
    M = 7
    N = M * M
    idx = np.array([[oracle.swin_index(M, i // M, i % M, j // M, j % M) for j in range(N)]
                    for i in range(N)])
    assert np.all(np.diag(idx) == 84)
    assert np.all(idx + idx.T == 168)
    assert idx.min() == 0 and idx.max() == 168
    for i in range(N):
        assert len(set(idx[i])) == N


def _brute_force_allowed(G_h, G_w, M, s):
    """Geometric characterisation of the shifted-window mask, independent of
    the strip rule: roll the map of original coordinates by -s (torch.roll),
    partition into windows, and allow a pair iff the two tokens were within
    one window size of each other in the ORIGINAL image (a pair that wrapped
    around the border is > G-M apart)."""
    ys, xs = torch.meshgrid(torch.arange(G_h), torch.arange(G_w), indexing="ij")
    ys = torch.roll(ys, shifts=(-s, -s), dims=(0, 1))
    xs = torch.roll(xs, shifts=(-s, -s), dims=(0, 1))
    res = []
    for wr in range(G_h // M):
        for wc in range(G_w // M):
            oy = ys[wr * M:(wr + 1) * M, wc * M:(wc + 1) * M].reshape(-1)
            ox = xs[wr * M:(wr + 1) * M, wc * M:(wc + 1) * M].reshape(-1)
            near = ((oy[:, None] - oy[None, :]).abs() < M) & ((ox[:, None] - ox[None, :]).abs() < M)
            res.append(near.numpy())
    return res


@pytest.mark.parametrize("geom", [(56, 56, 7, 3), (4, 4, 2, 1), (14, 21, 7, 3), (12, 8, 4, 2)])
def test_p3_swin_mask_matches_geometric_brute_force(geom):
    G_h, G_w, M, s = geom
    allowed = _brute_force_allowed(G_h, G_w, M, s)
    for w, want in enumerate(allowed):
        got = np.array([[oracle.swin_mask(M, G_h, G_w, s, w, i, j) for j in range(M * M)]
                        for i in range(M * M)])
        assert set(np.unique(got)) <= {0.0, -100.0}
        np.testing.assert_array_equal(got == 0.0, want)


def test_p3_swin_mask_counts_golden(golden_dir):
    """P3: allowed pair counts per window and per image (hand-enumerated)."""
    rows = _read_golden(os.path.join(golden_dir, "swin_mask_counts.txt"))
    cache = {}
    for gh, gw, M, s, w, cnt in rows:
        gh, gw, M, s, cnt = int(gh), int(gw), int(M), int(s), int(cnt)
        key = (gh, gw, M, s)
        if key not in cache:
            nW = (gh // M) * (gw // M)
            cache[key] = [sum(oracle.swin_mask(M, gh, gw, s, win, i, j) == 0.0
                              for i in range(M * M) for j in range(M * M)) for win in range(nW)]
        counts = cache[key]
        if w == "total":
            assert sum(counts) == cnt
        else:
            assert counts[int(w)] == cnt


def test_swin_no_shift_means_no_mask():
    for w in range(16):
        for i in range(0, 49, 5):
            for j in range(0, 49, 3):
                assert oracle.swin_mask(7, 28, 28, 0, w, i, j) == 0.0


def test_swin_bias_is_table_gather_plus_mask():
    """bias = table[idx, h] + mask, read back through an integer-valued table
    (value = index + 256*h, exact in fp64/fp32)."""
    M, H = 2, 3
    table = np.array([[r + 256.0 * h for h in range(H)] for r in range((2 * M - 1) ** 2)])
    b = oracle.Bias("swin", table=table, win=M, grid_h=4, grid_w=4, shift=1)
    q = np.zeros((4 * H, M * M, 4))
    golden = np.array([[4, 3, 1, 0], [5, 4, 2, 1], [7, 6, 4, 3], [8, 7, 5, 4]])
    for s in range(4 * H):
        w, h = (s // H) % 4, s % H
        Bm = oracle.bias_matrix(q, H, s, M * M, b)
        mask = np.array([[oracle.swin_mask(M, 4, 4, 1, w, i, j) for j in range(4)] for i in range(4)])
        np.testing.assert_array_equal(Bm, golden + 256.0 * h + mask)


def test_swin_2x2_window_softmax_brute_force():
    """Q = K = 0 leaves only the bias; with V = I the output row is the
    softmax of the bias row, computed here by hand with math.exp over the
    golden index matrix and table value 0.1*index."""
    M, H = 2, 1
    table = np.arange(9, dtype=float)[:, None] * 0.1
    b = oracle.Bias("swin", table=table, win=M, grid_h=2, grid_w=2, shift=0)
    q = np.zeros((1, 4, 4))
    k = np.zeros((1, 4, 4))
    v = np.eye(4)[None]
    out, _ = oracle.attn_fwd(q, k, v, H, 1.0, b)
    golden = [[4, 3, 1, 0], [5, 4, 2, 1], [7, 6, 4, 3], [8, 7, 5, 4]]
    for i in range(4):
        e = [math.exp(0.1 * golden[i][j]) for j in range(4)]
        want = [x / sum(e) for x in e]
        np.testing.assert_allclose(out[0, i], want, rtol=0, atol=1e-15)


def test_swin_mask_is_finite_minus_100():
    """Masked pairs keep a weight of about e^-100 (finite mask), not 0."""
    M, H = 2, 1
    b = oracle.Bias("swin", table=np.zeros((9, 1)), win=M, grid_h=4, grid_w=4, shift=1)
    q = np.zeros((4, 4, 4))
    P, _ = oracle.attn_probs(q, q, np.ones((4, 4, 4)), H, 1.0, 3, b)
    # window 3: four singleton regions -> diagonal weight 1/(1+3e^-100)
    off = P[~np.eye(4, dtype=bool)]
    assert np.all(off > 0)
    np.testing.assert_allclose(off, math.exp(-100) / (1 + 3 * math.exp(-100)), rtol=1e-12)


def test_p7_swin_table_column_shift_invariance():
    """P7: adding a constant to one head's whole table column shifts every
    score row of that head by the same amount; O is unchanged."""
    M, H, d = 3, 2, 8
    table = _rand(((2 * M - 1) ** 2, H), 3)
    b1 = oracle.Bias("swin", table=table, win=M, grid_h=6, grid_w=6, shift=1)
    t2 = table.copy()
    t2[:, 1] += 5.0
    b2 = oracle.Bias("swin", table=t2, win=M, grid_h=6, grid_w=6, shift=1)
    q, k, v = (_rand((4 * H, M * M, d), s) for s in (1, 2, 3))
    o1, _ = oracle.attn_fwd(q, k, v, H, 0.4, b1)
    o2, _ = oracle.attn_fwd(q, k, v, H, 0.4, b2)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)


# ---------------------------------------------------------------------- SAM --

@pytest.mark.parametrize("grid", [(2, 2), (3, 5), (5, 3), (14, 14)])
def test_p6_p8_sam_relpos_closed_form(grid):
    """P6/P8: with R_h[r] = r*u and R_w[r] = r*w the decomposed term is
    (qh-kh+S_h-1)*(Q.u) + (qw-kw+S_w-1)*(Q.w) for tokens i=(qh,qw), j=(kh,kw).
    Non-square grids catch a swapped height/width; the sign of the offsets
    and the S-1 shift are fixed by the closed form."""
    sh, sw = grid
    d = 6
    u, w = _rand(d, 11), _rand(d, 12)
    Rh = np.arange(2 * sh - 1)[:, None] * u[None]
    Rw = np.arange(2 * sw - 1)[:, None] * w[None]
    b = oracle.Bias("sam", rel_h=Rh, rel_w=Rw, s_h=sh, s_w=sw)
    N = sh * sw
    q = _rand((1, N, d), 13)
    Bm = oracle.bias_matrix(q, 1, 0, N, b)
    for i in range(N):
        qh, qw = divmod(i, sw)
        for j in range(N):
            kh, kw = divmod(j, sw)
            want = (qh - kh + sh - 1) * (q[0, i] @ u) + (qw - kw + sw - 1) * (q[0, i] @ w)
            assert abs(Bm[i, j] - want) < 1e-12 * (1 + abs(want))


def test_p8_sam_integer_tables_exact():
    """P8: integer-valued tables and Q = 128*e0 + e1 give the exact index
    pair 128*(qh-kh+S_h-1) + (qw-kw+S_w-1), the fixture of the bit-exact
    kernel test."""
    sh, sw, d = 3, 4, 16
    Rh = np.zeros((2 * sh - 1, d))
    Rh[:, 0] = np.arange(2 * sh - 1)
    Rw = np.zeros((2 * sw - 1, d))
    Rw[:, 1] = np.arange(2 * sw - 1)
    N = sh * sw
    q = np.zeros((1, N, d))
    q[..., 0] = 128.0
    q[..., 1] = 1.0
    b = oracle.Bias("sam", rel_h=Rh, rel_w=Rw, s_h=sh, s_w=sw)
    Bm = oracle.bias_matrix(q, 1, 0, N, b)
    for i in range(N):
        for j in range(N):
            want = 128 * (i // sw - j // sw + sh - 1) + (i % sw - j % sw + sw - 1)
            assert Bm[i, j] == want


def test_p7_sam_constant_table_shift_invariance():
    """P7: adding the same vector c to every row of R_h adds Q_i.c to the
    whole score row i; the softmax output is unchanged."""
    sh, sw, d = 3, 4, 8
    Rh, Rw = _rand((2 * sh - 1, d), 1), _rand((2 * sw - 1, d), 2)
    c = _rand(d, 3)
    q, k, v = (_rand((2, sh * sw, d), s) for s in (4, 5, 6))
    o1, _ = oracle.attn_fwd(q, k, v, 1, 0.5, oracle.Bias("sam", rel_h=Rh, rel_w=Rw, s_h=sh, s_w=sw))
    o2, _ = oracle.attn_fwd(q, k, v, 1, 0.5,
                            oracle.Bias("sam", rel_h=Rh + c, rel_w=Rw, s_h=sh, s_w=sw))
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)


def test_sam_bias_uses_unscaled_q():
    """The decomposed term does not depend on the softmax scale: zero K makes
    the scores bias-only, and changing scale must leave O unchanged."""
    sh, sw, d = 2, 3, 4
    Rh, Rw = _rand((2 * sh - 1, d), 1), _rand((2 * sw - 1, d), 2)
    b = oracle.Bias("sam", rel_h=Rh, rel_w=Rw, s_h=sh, s_w=sw)
    q, v = _rand((1, 6, d), 3), _rand((1, 6, d), 4)
    k = np.zeros_like(q)
    o1, _ = oracle.attn_fwd(q, k, v, 1, 0.1, b)
    o2, _ = oracle.attn_fwd(q, k, v, 1, 7.0, b)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-14)


# --------------------------------------------------------------- arguments --

def test_oracle_rejects_bad_shapes():
    q = np.zeros((2, 9, 4))
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, q, q, 3, 1.0)  # BH not a multiple of H
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, q, q, 1, 1.0, oracle.Bias("swin", table=np.zeros((25, 1)), win=2,
                                                     grid_h=4, grid_w=4))  # N != M*M
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, q, q, 1, 1.0, oracle.Bias("sam", rel_h=np.zeros((3, 4)),
                                                     rel_w=np.zeros((3, 4)), s_h=2, s_w=2))


def test_workload_inputs_are_seeded_and_shaped():
    w = WORKLOADS["toy"]
    a, b = make_inputs(w), make_inputs(w)
    assert torch.equal(a.q, b.q) and a.q.shape == (1, 2, 64, 32) and a.q.dtype == torch.bfloat16
    sw = WORKLOADS["swin_t_stage1"].with_(B=64)
    i = make_inputs(sw)
    assert i.table.shape == (169, 3) and i.table.dtype == torch.float32
    sm = WORKLOADS["sam_vith_window"].with_(B=2)
    i = make_inputs(sm)
    assert i.rel_h.shape == (27, 80) and i.rel_h.dtype == torch.bfloat16


# ------------------------------------------- Swin shift + window partition --

def test_swin_partition_matches_index_definition_by_brute_force():
    rng = np.random.default_rng(7)
    B, Gh, Gw, H, d, M, s = 2, 4, 6, 2, 3, 2, 1
    x = rng.standard_normal((B, Gh, Gw, H, d))
    xw = oracle.swin_partition(x, M, s)
    nwh, nww = Gh // M, Gw // M
    assert xw.shape == (B * nwh * nww, H, M * M, d)
    for b in range(B):
        for wr in range(nwh):
            for wc in range(nww):
                for h in range(H):
                    for r in range(M):
                        for c in range(M):
                            want = x[b, (wr * M + r + s) % Gh, (wc * M + c + s) % Gw, h]
                            got = xw[(b * nwh + wr) * nww + wc, h, r * M + c]
                            np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("shift", [0, 1, 3])
def test_swin_unpartition_inverts_partition(shift):
    rng = np.random.default_rng(8)
    x = rng.standard_normal((2, 14, 21, 3, 4))
    back = oracle.swin_unpartition(oracle.swin_partition(x, 7, shift), 2, 14, 21, 7, shift)
    np.testing.assert_array_equal(back, x)


def test_swin_partition_without_shift_is_a_reshape():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((1, 3, 3, 2, 5))  # one 3x3 window
    xw = oracle.swin_partition(x, 3, 0)
    np.testing.assert_array_equal(xw[0], x[0].reshape(9, 2, 5).transpose(1, 0, 2))


# --------------------------------------------------- variable-length batch --
# A nested tensor packs {tensor, mask}: the packed-batch attention must equal
# attention over the zero-padded batch whose padded keys are masked out.

def _packed_to_padded(x, cu, H, fill):
    """[H * sum(L), d] packed as [H][L_s][d] per sequence -> [n, H, max L, d]."""
    n, d = len(cu) - 1, x.shape[-1]
    L = max(cu[s + 1] - cu[s] for s in range(n))
    out = fill((n, H, L, d))
    for s in range(n):
        ls = cu[s + 1] - cu[s]
        out[s, :, :ls] = x[H * cu[s]:H * cu[s + 1]].reshape(H, ls, d)
    return out


def test_varlen_equals_padded_batch_with_key_mask():
    rng = np.random.default_rng(21)
    H, d = 3, 8
    lq = [5, 0, 17, 1, 9]
    lk = [7, 4, 17, 1, 3]   # cross lengths, an empty query set, single tokens
    cu_q = [0] + list(np.cumsum(lq))
    cu_k = [0] + list(np.cumsum(lk))
    q = rng.standard_normal((H * cu_q[-1], d))
    k = rng.standard_normal((H * cu_k[-1], d))
    v = rng.standard_normal((H * cu_k[-1], d))
    scale = 0.37
    got = oracle.attn_varlen(q, k, v, cu_q, cu_k, H, scale)
    # padded rows and keys hold junk, not zeros, so a missing mask shows
    junk = lambda shape: rng.standard_normal(shape) * 5.0  # noqa: E731
    Qp = torch.from_numpy(_packed_to_padded(q, cu_q, H, junk))
    Kp = torch.from_numpy(_packed_to_padded(k, cu_k, H, junk))
    Vp = torch.from_numpy(_packed_to_padded(v, cu_k, H, junk))
    mask = torch.zeros((len(lq), 1, Qp.shape[2], Kp.shape[2]), dtype=torch.bool)
    for s, n in enumerate(lk):
        mask[s, :, :, :n] = True
    want = torch.nn.functional.scaled_dot_product_attention(Qp, Kp, Vp, attn_mask=mask, scale=scale).numpy()
    for s in range(len(lq)):
        if lq[s] == 0:
            continue
        blk = got[H * cu_q[s]:H * cu_q[s + 1]].reshape(H, lq[s], d)
        np.testing.assert_allclose(blk, want[s, :, :lq[s]], rtol=0, atol=1e-12)


def test_varlen_sequence_order_does_not_matter():
    rng = np.random.default_rng(22)
    H, d = 2, 4
    lens = [6, 2, 11]
    blocks_q = [rng.standard_normal((H * n, d)) for n in lens]
    blocks_k = [rng.standard_normal((H * n, d)) for n in lens]
    blocks_v = [rng.standard_normal((H * n, d)) for n in lens]
    cu = [0] + list(np.cumsum(lens))
    fwd = oracle.attn_varlen(np.concatenate(blocks_q), np.concatenate(blocks_k), np.concatenate(blocks_v),
                             cu, cu, H, 0.5)
    rl = lens[::-1]
    rcu = [0] + list(np.cumsum(rl))
    rev = oracle.attn_varlen(np.concatenate(blocks_q[::-1]), np.concatenate(blocks_k[::-1]),
                             np.concatenate(blocks_v[::-1]), rcu, rcu, H, 0.5)
    for s, n in enumerate(lens):
        r = len(lens) - 1 - s
        np.testing.assert_array_equal(fwd[H * cu[s]:H * cu[s + 1]], rev[H * rcu[r]:H * rcu[r + 1]])


def test_varlen_single_key_returns_its_value():
    rng = np.random.default_rng(23)
    H, d = 2, 5
    cu_q, cu_k = [0, 4, 7], [0, 1, 2]
    q = rng.standard_normal((H * 7, d))
    k = rng.standard_normal((H * 2, d))
    v = rng.standard_normal((H * 2, d))
    out = oracle.attn_varlen(q, k, v, cu_q, cu_k, H, 1.0)
    for s in range(2):
        lq = cu_q[s + 1] - cu_q[s]
        blk = out[H * cu_q[s]:H * cu_q[s + 1]].reshape(H, lq, d)
        for h in range(H):
            np.testing.assert_array_equal(blk[h], np.broadcast_to(v[H * cu_k[s] + h], (lq, d)))


# ------------------------------------- SAM rel-pos on unequal query/key grids --
# Published definition: coordinates scaled by max(k/q, 1) (queries) and
# max(q/k, 1) (keys), offset (k-1)*max(q/k, 1), evaluated in float32 and
# truncated; tables whose length is not 2*max(q, k)-1 are resampled linearly.

def test_sam_rel_index_hand_computed():
    # q=2, k=4: 2i - j + 3
    np.testing.assert_array_equal(oracle.sam_rel_index(2, 4), [[3, 2, 1, 0], [5, 4, 3, 2]])
    # q=4, k=2: i - 2j + 2
    np.testing.assert_array_equal(oracle.sam_rel_index(4, 2), [[2, 0], [3, 1], [4, 2], [5, 3]])
    # q=2, k=3: 1.5i - j + 2, truncated: 3.5 -> 3, 2.5 -> 2, 1.5 -> 1
    np.testing.assert_array_equal(oracle.sam_rel_index(2, 3), [[2, 1, 0], [3, 2, 1]])
    # equal sizes: i - j + q - 1
    np.testing.assert_array_equal(oracle.sam_rel_index(3, 3), [[2, 1, 0], [3, 2, 1], [4, 3, 2]])


@pytest.mark.parametrize("q,k", [(14, 64), (64, 14), (5, 7), (7, 5), (64, 64), (3, 40)])
def test_sam_rel_index_in_float32_like_torch(q, k):
    """torch evaluates the scaled coordinates of an int arange in float32."""
    qc = torch.arange(q)[:, None] * max(k / q, 1.0)
    kc = torch.arange(k)[None, :] * max(q / k, 1.0)
    want = ((qc - kc) + (k - 1) * max(q / k, 1.0)).long().numpy()
    got = oracle.sam_rel_index(q, k)
    np.testing.assert_array_equal(got, want)
    assert got.min() >= 0 and got.max() <= 2 * max(q, k) - 2


@pytest.mark.parametrize("L_in,L_out", [(27, 127), (127, 27), (10, 13), (13, 10), (9, 9)])
def test_sam_resize_is_linear_interpolation(L_in, L_out):
    rng = np.random.default_rng(L_in * 131 + L_out)
    t = rng.standard_normal((L_in, 6))
    want = torch.nn.functional.interpolate(torch.from_numpy(t).T[None], size=L_out, mode="linear",
                                           align_corners=False)[0].T.numpy()
    np.testing.assert_allclose(oracle.sam_resize(t, L_out), want, rtol=0, atol=1e-12)


def _sam_bias_brute(q, qg, kg, Rh, Rw):
    """Bias of every (query, key) pair from torch-resized tables and torch's
    float32 coordinate scaling."""
    (qh_n, qw_n), (kh_n, kw_n) = qg, kg

    def rows(R, a, b):
        L = 2 * max(a, b) - 1
        Rt = torch.from_numpy(R)
        if R.shape[0] != L:
            Rt = torch.nn.functional.interpolate(Rt.T[None], size=L, mode="linear", align_corners=False)[0].T
        qc = torch.arange(a)[:, None] * max(b / a, 1.0)
        kc = torch.arange(b)[None, :] * max(a / b, 1.0)
        return Rt.numpy(), ((qc - kc) + (b - 1) * max(a / b, 1.0)).long().numpy()

    Rh_r, ih = rows(Rh, qh_n, kh_n)
    Rw_r, iw = rows(Rw, qw_n, kw_n)
    out = np.empty((qh_n * qw_n, kh_n * kw_n))
    for i in range(qh_n * qw_n):
        for j in range(kh_n * kw_n):
            a, b = divmod(i, qw_n)
            c, e = divmod(j, kw_n)
            out[i, j] = q[i] @ Rh_r[ih[a, c]] + q[i] @ Rw_r[iw[b, e]]
    return out


def test_sam_unequal_grids_bias_by_brute_force():
    rng = np.random.default_rng(51)
    qg, kg, d = (3, 4), (5, 2), 6
    Rh = rng.standard_normal((7, d))    # 2*max(3,5)-1 = 9 rows needed: upsampled
    Rw = rng.standard_normal((11, d))   # 2*max(4,2)-1 = 7 rows needed: downsampled
    q = rng.standard_normal((1, 12, d))
    b = oracle.Bias("sam", rel_h=Rh, rel_w=Rw, s_h=3, s_w=4, k_h=5, k_w=2)
    got = oracle.bias_matrix(q, 1, 0, 10, b)
    np.testing.assert_allclose(got, _sam_bias_brute(q[0], qg, kg, Rh, Rw), rtol=0, atol=1e-12)


def test_sam_unequal_grids_attention_matches_torch_sdpa():
    rng = np.random.default_rng(52)
    qg, kg, d, H = (4, 3), (2, 5), 8, 2
    Nq, Nk = 12, 10
    Rh = rng.standard_normal((5, d)) * 0.3
    Rw = rng.standard_normal((9, d)) * 0.3
    q = rng.standard_normal((H, Nq, d))
    k = rng.standard_normal((H, Nk, d))
    v = rng.standard_normal((H, Nk, d))
    b = oracle.Bias("sam", rel_h=Rh, rel_w=Rw, s_h=4, s_w=3, k_h=2, k_w=5)
    got, _ = oracle.attn_fwd(q, k, v, H, 0.4, b)
    for h in range(H):
        bias = torch.from_numpy(_sam_bias_brute(q[h], qg, kg, Rh, Rw))
        want = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[h])[None], torch.from_numpy(k[h])[None], torch.from_numpy(v[h])[None],
            attn_mask=bias[None], scale=0.4)[0].numpy()
        np.testing.assert_allclose(got[h], want, rtol=0, atol=1e-12)


# ------------------------------------------------------------- backward pass --
# attn_bwd against torch fp64 autograd of the forward definition (a separate
# differentiation) and against central finite differences of the oracle's
# own forward pass.

def _torch_attn(q, k, v, scale, bias):
    s = scale * q @ k.transpose(-1, -2) + bias
    return torch.softmax(s, dim=-1) @ v


def _grads(out, dout, *xs):
    return torch.autograd.grad(out, xs, grad_outputs=dout)


def test_bwd_no_bias_matches_autograd():
    rng = np.random.default_rng(60)
    BH, Nq, Nk, d, H = 4, 9, 13, 6, 2
    q, k, v = (rng.standard_normal((BH, n, d)) for n in (Nq, Nk, Nk))
    dout = rng.standard_normal((BH, Nq, d))
    got = oracle.attn_bwd(q, k, v, dout, H, 0.3)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    want = _grads(_torch_attn(tq, tk, tv, 0.3, 0.0), torch.tensor(dout), tq, tk, tv)
    for name, w in zip(("dq", "dk", "dv"), want):
        np.testing.assert_allclose(got[name], w.numpy(), rtol=0, atol=1e-11)


def test_bwd_swin_matches_autograd():
    rng = np.random.default_rng(61)
    M, G, s_, H, d = 3, 6, 1, 2, 5
    nW = (G // M) ** 2
    BH, N = nW * H, M * M
    table = rng.standard_normal(((2 * M - 1) ** 2, H)) * 0.3
    q, k, v, dout = (rng.standard_normal((BH, N, d)) for _ in range(4))
    b = oracle.Bias("swin", table=table, win=M, grid_h=G, grid_w=G, shift=s_)
    got = oracle.attn_bwd(q, k, v, dout, H, 0.4, b)
    # torch: the table gathered by relative offset (requires grad), plus the
    # constant mask taken from a zero table
    r, c = np.arange(N) // M, np.arange(N) % M
    idx = torch.tensor((r[:, None] - r[None, :] + M - 1) * (2 * M - 1) + (c[:, None] - c[None, :] + M - 1))
    zero = oracle.Bias("swin", table=np.zeros_like(table), win=M, grid_h=G, grid_w=G, shift=s_)
    mask = torch.tensor(np.stack([oracle.bias_matrix(q, H, i, N, zero) for i in range(BH)]))
    tt = torch.tensor(table, requires_grad=True)
    heads = torch.tensor([i % H for i in range(BH)])
    bias = tt[idx][:, :, heads].permute(2, 0, 1) + mask
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    want = _grads(_torch_attn(tq, tk, tv, 0.4, bias), torch.tensor(dout), tq, tk, tv, tt)
    for name, w in zip(("dq", "dk", "dv", "d_table"), want):
        np.testing.assert_allclose(got[name], w.numpy(), rtol=0, atol=1e-11)


def test_bwd_sam_unequal_resampled_matches_autograd():
    rng = np.random.default_rng(62)
    (qh, qw), (kh, kw), d, H = (3, 4), (2, 5), 6, 2
    Nq, Nk = qh * qw, kh * kw
    Rh = rng.standard_normal((4, d)) * 0.3    # 2*max(3,2)-1 = 5 rows addressed: upsampled
    Rw = rng.standard_normal((12, d)) * 0.3   # 2*max(4,5)-1 = 9 rows addressed: downsampled
    q, dout = (rng.standard_normal((H, Nq, d)) for _ in range(2))
    k, v = (rng.standard_normal((H, Nk, d)) for _ in range(2))
    b = oracle.Bias("sam", rel_h=Rh, rel_w=Rw, s_h=qh, s_w=qw, k_h=kh, k_w=kw)
    got = oracle.attn_bwd(q, k, v, dout, H, 0.35, b)

    def rows(R, a, bb):
        L = 2 * max(a, bb) - 1
        Rr = torch.nn.functional.interpolate(R.T[None], size=L, mode="linear", align_corners=False)[0].T
        qc = torch.arange(a)[:, None] * max(bb / a, 1.0)
        kc = torch.arange(bb)[None, :] * max(a / bb, 1.0)
        return Rr, ((qc - kc) + (bb - 1) * max(a / bb, 1.0)).long()

    tRh, tRw = torch.tensor(Rh, requires_grad=True), torch.tensor(Rw, requires_grad=True)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    Rh_r, ih = rows(tRh, qh, kh)
    Rw_r, iw = rows(tRw, qw, kw)
    i, j = torch.arange(Nq), torch.arange(Nk)
    IH = ih[(i // qw)[:, None], (j // kw)[None, :]]
    IW = iw[(i % qw)[:, None], (j % kw)[None, :]]
    bias = torch.einsum("hic,ijc->hij", tq, Rh_r[IH] + Rw_r[IW])
    want = _grads(_torch_attn(tq, tk, tv, 0.35, bias), torch.tensor(dout), tq, tk, tv, tRh, tRw)
    for name, w in zip(("dq", "dk", "dv", "d_rel_h", "d_rel_w"), want):
        np.testing.assert_allclose(got[name], w.numpy(), rtol=0, atol=1e-11)


def test_bwd_finite_differences():
    """Central differences of L = sum(dO * O) through the oracle's forward."""
    rng = np.random.default_rng(63)
    M, G, H, d = 2, 4, 1, 3
    BH, N = (G // M) ** 2 * H, M * M
    table = rng.standard_normal(((2 * M - 1) ** 2, H)) * 0.5
    q, k, v, dout = (rng.standard_normal((BH, N, d)) for _ in range(4))

    def loss(q_, k_, v_, t_):
        b_ = oracle.Bias("swin", table=t_, win=M, grid_h=G, grid_w=G, shift=1)
        o, _ = oracle.attn_fwd(q_, k_, v_, H, 0.6, b_)
        return float(np.sum(o * dout))

    got = oracle.attn_bwd(q, k, v, dout, H, 0.6, oracle.Bias("swin", table=table, win=M, grid_h=G, grid_w=G, shift=1))
    eps = 1e-6
    for name, x, pos in (("dq", q, (1, 2, 0)), ("dk", k, (3, 0, 2)), ("dv", v, (0, 3, 1)), ("d_table", table, (4, 0))):
        xp, xm = x.copy(), x.copy()
        xp[pos] += eps
        xm[pos] -= eps
        args_p = [xp if a is x else a for a in (q, k, v, table)]
        args_m = [xm if a is x else a for a in (q, k, v, table)]
        fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        assert abs(fd - got[name][pos]) < 1e-7, (name, fd, got[name][pos])


def test_bwd_out_given_as_exact_o_equals_default():
    """attn_bwd(out=O) with O the forward's exact output reproduces the
    default call, which takes O from the forward definition itself."""
    rng = np.random.default_rng(64)
    M, G, s_, H, d = 3, 6, 1, 2, 5
    BH, N = (G // M) ** 2 * H, M * M
    table = rng.standard_normal(((2 * M - 1) ** 2, H)) * 0.3
    q, k, v, dout = (rng.standard_normal((BH, N, d)) for _ in range(4))
    for b in (None, oracle.Bias("swin", table=table, win=M, grid_h=G, grid_w=G, shift=s_)):
        o, _ = oracle.attn_fwd(q, k, v, H, 0.45, b)
        base = oracle.attn_bwd(q, k, v, dout, H, 0.45, b)
        given = oracle.attn_bwd(q, k, v, dout, H, 0.45, b, out=o)
        for name in base:
            np.testing.assert_allclose(given[name], base[name], rtol=0, atol=1e-14)


def test_bwd_out_perturbed_follows_the_rowsum_formula():
    """With out = O + E the oracle takes D' = rowsum(dO * (O + E)) in place of
    the exact D.  dS then moves by P * (D - D'), which is the gradient of
    sum_i (D_i - D'_i) * logsumexp_j S_ij: torch fp64 autograd of
    L = sum(dO * O) + sum_i c_i logsumexp(S_i), c = D - D' held constant,
    must give the same dQ, dK, dV (dV unchanged) and table gradient."""
    rng = np.random.default_rng(65)
    M, G, s_, H, d = 3, 6, 1, 2, 5
    BH, N = (G // M) ** 2 * H, M * M
    table = rng.standard_normal(((2 * M - 1) ** 2, H)) * 0.3
    q, k, v, dout = (rng.standard_normal((BH, N, d)) for _ in range(4))
    b = oracle.Bias("swin", table=table, win=M, grid_h=G, grid_w=G, shift=s_)
    o, _ = oracle.attn_fwd(q, k, v, H, 0.45, b)
    o_given = o + rng.standard_normal(o.shape) * 0.05
    got = oracle.attn_bwd(q, k, v, dout, H, 0.45, b, out=o_given)
    c = torch.tensor(np.sum(dout * o, axis=2) - np.sum(dout * o_given, axis=2))  # D - D'
    r, cc = np.arange(N) // M, np.arange(N) % M
    idx = torch.tensor((r[:, None] - r[None, :] + M - 1) * (2 * M - 1) + (cc[:, None] - cc[None, :] + M - 1))
    zero = oracle.Bias("swin", table=np.zeros_like(table), win=M, grid_h=G, grid_w=G, shift=s_)
    mask = torch.tensor(np.stack([oracle.bias_matrix(q, H, i, N, zero) for i in range(BH)]))
    tt = torch.tensor(table, requires_grad=True)
    heads = torch.tensor([i % H for i in range(BH)])
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    s = 0.45 * tq @ tk.transpose(-1, -2) + tt[idx][:, :, heads].permute(2, 0, 1) + mask
    out = torch.softmax(s, dim=-1) @ tv
    loss = torch.sum(torch.tensor(dout) * out) + torch.sum(c * torch.logsumexp(s, dim=-1))
    want = torch.autograd.grad(loss, (tq, tk, tv, tt))
    for name, w in zip(("dq", "dk", "dv", "d_table"), want):
        np.testing.assert_allclose(got[name], w.numpy(), rtol=0, atol=1e-11)
    # and the perturbation is not a no-op: dQ moved
    base = oracle.attn_bwd(q, k, v, dout, H, 0.45, b)
    assert np.abs(got["dq"] - base["dq"]).max() > 1e-3


# ------------------------------------------------------------ log-sum-exp --

def test_lse_closed_form_uniform_scores():
    """Q = 0 and no bias: every score is 0, so lse = log(Nk) exactly."""
    rng = np.random.default_rng(66)
    q = np.zeros((3, 5, 4))
    k = rng.standard_normal((3, 7, 4))
    np.testing.assert_allclose(oracle.attn_lse(q, k, 1, 0.7), np.log(7.0), rtol=0, atol=1e-15)


def test_lse_gives_the_c_oracle_probabilities():
    """exp(S - lse) equals the probabilities the C oracle computes (a
    separate implementation of the softmax), with and without a bias."""
    rng = np.random.default_rng(67)
    M, G, H, d = 3, 6, 2, 5
    BH, N = (G // M) ** 2 * H, M * M
    table = rng.standard_normal(((2 * M - 1) ** 2, H)) * 0.3
    q, k, v = (rng.standard_normal((BH, N, d)) for _ in range(3))
    for b in (None, oracle.Bias("swin", table=table, win=M, grid_h=G, grid_w=G, shift=1)):
        lse = oracle.attn_lse(q, k, H, 0.4, b)
        for s in range(BH):
            P, _ = oracle.attn_probs(q, k, v, H, 0.4, s, b)
            S = 0.4 * q[s] @ k[s].T + (oracle.bias_matrix(q, H, s, N, b) if b is not None else 0.0)
            np.testing.assert_allclose(np.exp(S - lse[s][:, None]), P, rtol=0, atol=1e-13)
