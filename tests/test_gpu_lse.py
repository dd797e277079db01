"""GPU: attn_fwd_train writes each row's log-sum-exp (natural log, fp32) next
to the output attn_fwd writes, on every tiling of the forward kernel,
against the oracle's attn_lse on the same seeded inputs.

Tolerance: the GPU sums fp32 exponentials of fp32 scores (ex2.approx,
relative error about 2^-22 per term); the bias terms it adds are held in 16
bits on some paths (SAM rel_w in fp16: 2^-11 of a term of about 0.5; the
Swin MMA variant's table / scale in the operand type: 2^-9 of about 0.2).
|err| <= 2e-3 on every row covers those with a wide margin, while any wrong
or missing score term moves lse by far more."""
import numpy as np
import pytest
import torch

import oracle
import scaled_dot_product_09_gb300 as sdpa
from scaled_dot_product_09_gb300.workloads import WORKLOADS, Workload, make_inputs

from gpu_util import flat64, gpu_bias, oracle_bias, require_gpu

pytestmark = pytest.mark.gpu
W = WORKLOADS

CASES = {
    "packed_none": Workload("l1", B=3, H=2, Nq=49, Nk=40, d=32, dtype="fp16", bias="none", seed=90),
    "packed_swin_rows": W["swin_t_stage1"].with_(B=64, seed=91),
    "packed_swin_mma": W["swin_t_stage1"].with_(B=4, H=1, win=10, Nq=100, Nk=100, grid_h=20, grid_w=20,
                                               shift=5, seed=92),
    "shared_ragged": Workload("l2", B=1, H=2, Nq=300, Nk=333, d=64, dtype="bf16", bias="none", seed=93),
    "one_tile_cross": Workload("l3", B=2, H=2, Nq=600, Nk=77, d=40, dtype="fp16", bias="none", seed=94),
    "sam_14x14": W["sam_vith_window"].with_(B=2, H=2, seed=95),
    "sam_64x64": W["sam_vith_global"].with_(B=1, H=2, seed=96),
    "sam_16x16": W["sam_vith_global"].with_(B=1, H=3, Nq=256, Nk=256, s_h=16, s_w=16, seed=97),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_lse_matches_oracle(case):
    require_gpu()
    w = CASES[case]
    inp = make_inputs(w)
    q, k, v = (x.cuda() for x in (inp.q, inp.k, inp.v))
    bias = gpu_bias(w, inp)
    out, lse = sdpa.attn_fwd_train(q, k, v, scale=w.scale, bias=bias)
    ref = sdpa.attn_fwd(q, k, v, scale=w.scale, bias=bias)
    torch.cuda.synchronize()
    assert sdpa.attn_device_status() == sdpa.ATTN_OK
    # the output is the forward's, bit for bit
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    want = oracle.attn_lse(flat64(inp.q), flat64(inp.k), w.H, w.scale, oracle_bias(w, inp))
    got = lse.double().cpu().numpy().reshape(want.shape)
    err = np.abs(got - want)
    assert np.isfinite(got).all() and err.max() <= 2e-3, f"{case}: max |err| {err.max():.3e}"
