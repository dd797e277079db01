"""GPU parity of the variable-length (nested) batch: each sequence of a packed
[H][L_s][d] batch attends only to itself.  The CUDA path, through the C ABI,
against the fp64 oracle on the same seeded inputs; tolerance as for attn_fwd
(max |err| <= 2e-2, mean |err| <= 2e-3)."""
import numpy as np
import pytest
import torch

import oracle
import scaled_dot_product_09_gb300 as sdpa
from scaled_dot_product_09_gb300.workloads import WORKLOADS, Workload, make_inputs

from gpu_util import compare, require_gpu

pytestmark = pytest.mark.gpu


def _varlen_workload(lq, lk, H=4, d=64, dtype="fp16", seed=30):
    return Workload("varlen_case", B=len(lq), H=H, Nq=max(lq), Nk=max(lk), d=d, dtype=dtype, bias="none",
                    seed=seed, seqlens_q=tuple(lq), seqlens_k=tuple(lk))


def _run(w, inp):
    require_gpu()
    q, k, v = (x.cuda() for x in (inp.q, inp.k, inp.v))
    out = sdpa.attn_fwd_varlen(q, k, v, w.cu_seqlens_q, w.cu_seqlens_k, w.H, scale=w.scale)
    torch.cuda.synchronize()
    assert sdpa.attn_device_status() == sdpa.ATTN_OK
    return out.cpu()


def _full(w):
    inp = make_inputs(w)
    got = _run(w, inp).double().numpy()
    want = oracle.attn_varlen(inp.q.double().numpy(), inp.k.double().numpy(), inp.v.double().numpy(),
                              w.cu_seqlens_q, w.cu_seqlens_k, w.H, w.scale)
    # rows of sequences without queries do not exist; every row of q is some sequence's
    return compare(got, want, what=w.name)


def test_varlen_mixed_lengths():
    # tile-edge lengths (255/256/257), one token, an empty sequence, long ones
    lens = [300, 1, 0, 257, 1000, 77, 256, 513, 255]
    _full(_varlen_workload(lens, lens))


def test_varlen_cross_lengths():
    # queries and keys of different lengths per sequence (one key; many keys)
    _full(_varlen_workload([129, 7, 600, 64], [1, 300, 129, 1100], seed=31))


def test_varlen_bf16_partial_column_block():
    # d = 40: two full 16-column blocks and a partial one
    lens = [200, 450, 31]
    _full(_varlen_workload(lens, lens, H=8, d=40, dtype="bf16", seed=32))


@pytest.mark.parametrize("d", [32, 80, 128])
def test_varlen_head_dims(d):
    lens = [130, 390]
    _full(_varlen_workload(lens, lens, H=2, d=d, seed=33 + d))


def test_varlen_many_sequences():
    # the most sequences one call takes, lengths 1..300
    rng = np.random.default_rng(40)
    lens = [int(x) for x in rng.integers(1, 301, sdpa.ATTN_VARLEN_MAX_SEQ)]
    _full(_varlen_workload(lens, lens, H=2, d=32, seed=41))


def test_varlen_no_queries_is_a_no_op():
    require_gpu()
    k = torch.randn(2 * 5, 32, dtype=torch.float16, device="cuda")
    q = torch.empty(0, 32, dtype=torch.float16, device="cuda")
    out = sdpa.attn_fwd_varlen(q, k, k, [0, 0, 0], [0, 2, 5], H=2)
    assert out.numel() == 0


def test_varlen_single_sequence_matches_attn_fwd_bit_for_bit():
    """One sequence's [H][L][d] block is attn_fwd's [1][H][L][d] layout; both
    run the shared tiling with 128-key tiles, so the bits agree (rows and keys
    past the sequence are weighted by exact zeros in either)."""
    w = _varlen_workload([1000], [1000], H=2, d=64, seed=42)
    inp = make_inputs(w)
    got = _run(w, inp)
    q, k, v = (x.reshape(1, w.H, 1000, w.d).cuda() for x in (inp.q, inp.k, inp.v))
    ref = sdpa.attn_fwd(q, k, v, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.cpu().reshape(-1, w.d).view(torch.int16))


def test_varlen_full_size_sampled():
    """The ragged Stable Diffusion batch at full size; the oracle computes a
    sample of rows one by one (first, last and random rows of every sequence
    and head)."""
    w = WORKLOADS["sd_unet_self_varlen"]
    inp = make_inputs(w)
    got = _run(w, inp).double().numpy()
    rng = np.random.default_rng(43)
    q, k, v = (x.double().numpy() for x in (inp.q, inp.k, inp.v))
    cq, ck, H, d = w.cu_seqlens_q, w.cu_seqlens_k, w.H, w.d
    for s in range(w.B):
        lq, lk = cq[s + 1] - cq[s], ck[s + 1] - ck[s]
        qs = q[H * cq[s]:H * cq[s + 1]].reshape(H, lq, d)
        ks = k[H * ck[s]:H * ck[s + 1]].reshape(H, lk, d)
        vs = v[H * ck[s]:H * ck[s + 1]].reshape(H, lk, d)
        ids = np.unique(np.concatenate([[0, lq - 1, H * lq - 1], rng.integers(0, H * lq, 6)]))
        want, _ = oracle.attn_rows(qs, ks, vs, H, w.scale, ids)
        compare(got[H * cq[s] + ids], want, what=f"{w.name} sequence {s} (sampled)")


def test_varlen_sequences_do_not_interact():
    """Non-finite values in one sequence leave every other sequence's output
    unchanged: a tile that runs past its sequence reads the next one's rows,
    which must be masked (keys) and cleared (values), never weighted by zero
    (0 * inf = NaN).  Sequence 1 is poisoned with inf in V and K and NaN in
    Q; sequences 0 and 2 must still match the oracle on the clean data."""
    lens = [200, 150, 130]
    w = _varlen_workload(lens, lens, H=2, d=64, seed=44)
    inp = make_inputs(w)
    cq, H = w.cu_seqlens_q, w.H
    poisoned = [x.clone() for x in (inp.q, inp.k, inp.v)]
    rows = slice(H * cq[1], H * cq[2])
    poisoned[0][rows] = float("nan")
    poisoned[1][rows] = float("inf")
    poisoned[2][rows] = float("inf")
    got = _run(w, type(inp)(*poisoned)).double().numpy()
    want = oracle.attn_varlen(inp.q.double().numpy(), inp.k.double().numpy(), inp.v.double().numpy(),
                              w.cu_seqlens_q, w.cu_seqlens_k, w.H, w.scale)
    for s in (0, 2):
        r = slice(H * cq[s], H * cq[s + 1])
        compare(got[r], want[r], what=f"sequence {s} next to a poisoned sequence")


# ------------------------------------------------ packed short sequences
# Sequences of at most 32 (64) query and key tokens with d <= 64 share
# 128-row tiles, four (two) (sequence, head) slices per tile.

@pytest.mark.parametrize("lq,lk,H,d,dtype", [
    # slices of 32 rows: one token, tile-edge lengths, an odd slice count
    ([1, 7, 32, 20, 31, 16, 2], None, 3, 32, "fp16"),
    # slices of 64 rows, d = 40 (a partial 16-column block), bf16
    ([33, 64, 50, 40, 63], None, 4, 40, "bf16"),
    # queries and keys of different lengths (the longer decides the slice)
    ([3, 60, 10, 32, 1], [64, 2, 33, 1, 32], 2, 64, "fp16"),
    # d = 48 and d = 16 (one data chunk of a 32-column block), one head
    ([5, 17, 29, 64, 45, 12], None, 1, 48, "bf16"),
    ([9, 30, 57, 3], None, 5, 16, "fp16"),
])
def test_varlen_packed_short(lq, lk, H, d, dtype):
    lk = lq if lk is None else lk
    _full(_varlen_workload(lq, lk, H=H, d=d, dtype=dtype, seed=50 + H + d))


def test_varlen_packed_mixed_with_long():
    # three launches: the shared tiling (300, 129) and both packed slice sizes
    lens = [5, 300, 64, 33, 1, 129, 17, 0, 65]
    _full(_varlen_workload(lens, lens, H=2, d=64, seed=60))


def test_varlen_packed_many_sequences():
    rng = np.random.default_rng(61)
    lens = [int(x) for x in rng.integers(1, 65, sdpa.ATTN_VARLEN_MAX_SEQ)]
    _full(_varlen_workload(lens, lens, H=3, d=32, dtype="bf16", seed=62))


@pytest.mark.parametrize("lens", [[20, 30, 25, 10], [40, 50, 60]])
def test_varlen_packed_sequences_do_not_interact(lens):
    """With one head, consecutive sequences share a packed tile (four slices
    of 32 rows, or two of 64).  Sequence 1 is poisoned with NaN in Q and inf
    in K and V; every other sequence must still match the oracle on the clean
    data, although its tile's P.V also holds sequence 1's values."""
    w = _varlen_workload(lens, lens, H=1, d=32, seed=63)
    inp = make_inputs(w)
    cq, H = w.cu_seqlens_q, w.H
    poisoned = [x.clone() for x in (inp.q, inp.k, inp.v)]
    rows = slice(H * cq[1], H * cq[2])
    poisoned[0][rows] = float("nan")
    poisoned[1][rows] = float("inf")
    poisoned[2][rows] = float("inf")
    got = _run(w, type(inp)(*poisoned)).double().numpy()
    want = oracle.attn_varlen(inp.q.double().numpy(), inp.k.double().numpy(), inp.v.double().numpy(),
                              w.cu_seqlens_q, w.cu_seqlens_k, w.H, w.scale)
    for s in range(len(lens)):
        if s == 1:
            continue
        r = slice(H * cq[s], H * cq[s + 1])
        compare(got[r], want[r], what=f"packed sequence {s} next to a poisoned sequence")


@pytest.mark.parametrize("scale,d", [(-0.3, 8), (0.0, 64), (2.5, 24)])
def test_varlen_packed_scales_and_narrow_heads(scale, d):
    """Packed slices with a negative, a zero and a large scale (the softmax
    scales before its maximum when scale <= 0), and head dims 8 and 24 (one
    and three data chunks of a 32-column block)."""
    lens = [3, 40, 17, 64, 1, 32]
    w = _varlen_workload(lens, lens, H=3, d=d, dtype="bf16", seed=70 + d)
    inp = make_inputs(w)
    require_gpu()
    q, k, v = (x.cuda() for x in (inp.q, inp.k, inp.v))
    got = sdpa.attn_fwd_varlen(q, k, v, w.cu_seqlens_q, w.cu_seqlens_k, w.H, scale=scale)
    torch.cuda.synchronize()
    assert sdpa.attn_device_status() == sdpa.ATTN_OK
    want = oracle.attn_varlen(inp.q.double().numpy(), inp.k.double().numpy(), inp.v.double().numpy(),
                              w.cu_seqlens_q, w.cu_seqlens_k, w.H, scale)
    compare(got.double().cpu().numpy(), want, what=f"packed, scale {scale}, d {d}")
