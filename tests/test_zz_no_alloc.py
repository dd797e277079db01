"""attn_bwd_noalloc: the backward without a caller workspace, for callers
that cannot allocate device memory when they run it.  Its fixed scratch
replaces the workspace attn_bwd takes, so on the same inputs the two entry
points must give the same gradients; checked through the C ABI on two calls
in a row (the scratch keeps the first call's contents, which the second must
not depend on).  This file is collected last: run alone in a fresh process it
also covers the first call's look-up of the scratch address."""

import pytest
import torch

import scaled_dot_product_09_gb300 as sdpa
from scaled_dot_product_09_gb300.workloads import Workload, make_inputs

from gpu_util import compare, flat64, require_gpu

FAKE = 0x10000


def test_noalloc_rejects_more_rows_than_its_scratch():
    # 2^20 + 1 query rows: refused before any CUDA call, with a clear message
    lib = sdpa.load_library()
    rc = lib.attn_bwd_noalloc(FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288, FAKE + 16384, FAKE + 20480,
                              FAKE + 24576, FAKE + 28672, FAKE + 32768, 1, 1, (1 << 20) + 1, 300, 64, 0.125, 0,
                              None)
    assert rc == sdpa.ATTN_ERR_UNSUPPORTED
    assert b"2^20" in lib.attn_last_error() or b"1048576" in lib.attn_last_error()


@pytest.mark.gpu
def test_noalloc_matches_attn_bwd_on_two_calls():
    require_gpu()
    shapes = [Workload("na1", B=1, H=2, Nq=300, Nk=333, d=64, dtype="bf16", bias="none", seed=201),
              Workload("na2", B=2, H=3, Nq=257, Nk=129, d=40, dtype="fp16", bias="none", seed=202)]
    for w in shapes:  # two calls in a row, the second on other shapes and data
        inp = make_inputs(w)
        g = torch.Generator().manual_seed(w.seed + 7)
        dout = torch.randn(inp.q.shape, generator=g).to(inp.q.dtype)
        q, k, v, do = (x.cuda() for x in (inp.q, inp.k, inp.v, dout))
        out, lse = sdpa.attn_fwd_train(q, k, v, scale=w.scale)
        ref = sdpa.attn_bwd(q, k, v, out, do, lse=lse, scale=w.scale)[:3]
        got = sdpa.attn_bwd_noalloc(q, k, v, out, do, lse=lse, scale=w.scale)
        torch.cuda.synchronize()
        assert sdpa.attn_device_status() == sdpa.ATTN_OK
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            compare(flat64(a.cpu()), flat64(b.cpu()), what=f"{w.name} {name}")
