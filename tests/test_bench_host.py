"""Host-side logic of bench.py that needs no GPU: the multi-rank timing
reduction (max over ranks) and barrier on a two-rank gloo group, the
reference arm's rank handling, the oracle sample sizing, and the rule that
recorded DRAM traffic is reported only for the kernel sources it was
measured on."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from scaled_dot_product_09_gb300.workloads import WORKLOADS, make_inputs  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank "timed" a different duration: every rank must see the max
        t = 1.5 if rank == 0 else 2.5
        m = bench._max_over_ranks(t, world, torch.device("cpu"))
        bench._barrier(world)
        w, r, _ = bench._dist()
        with open(f"{out_path}.{rank}", "w") as f:
            json.dump({"max": m, "world": w, "rank": r}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    port = _free_port()
    out = str(tmp_path / "rank")
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    for rank in range(2):
        with open(f"{out}.{rank}") as f:
            got = json.load(f)
        assert got == {"max": 2.5, "world": 2, "rank": rank}


def test_max_over_ranks_single_process_is_identity():
    assert bench._max_over_ranks(3.25, 1, torch.device("cpu")) == 3.25


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class Args:
        steps, warmup, gpus = 1, 0, 2
        metric = "m"

    assert bench.run_reference(Args(), WORKLOADS["toy"], world=2, rank=1) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line(capsys):
    class Args:
        steps, warmup, gpus = 2, 1, 1
        metric = "attention fwd TFLOP/s"

    assert bench.run_reference(Args(), WORKLOADS["toy"], world=1, rank=0) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "toy"


def test_oracle_sample_repeats_whole_passes_for_short_workloads():
    w = WORKLOADS["toy"]
    tf, sec, rows, used = bench._oracle_sample(w, make_inputs(w), budget_s=0.2)
    total = w.B * w.H * w.Nq
    assert rows >= total and rows % total == 0  # whole passes over every row
    assert sec > 0 and tf > 0 and used >= 1


def test_traffic_only_for_matching_sources(tmp_path, monkeypatch):
    rec = {"toy": {"dram_bytes_per_launch": 123, "kernel_sources_sha256": bench._kernel_sources_hash()}}
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the hash is computed from the real sources, the record from the temp dir
    monkeypatch.setattr(bench, "_kernel_sources_hash", lambda: rec["toy"]["kernel_sources_sha256"])
    assert bench._traffic("toy") == 123
    assert bench._traffic("swin_t_stage1") is None
    monkeypatch.setattr(bench, "_kernel_sources_hash", lambda: "0" * 64)
    assert bench._traffic("toy") is None


def test_bound_classification():
    assert bench._bound(WORKLOADS["swin_t_stage1"]) == "hbm"
    assert bench._bound(WORKLOADS["sd_unet_cross"]) == "hbm"
    assert bench._bound(WORKLOADS["sd_unet_self"]) == "tensor"
    assert bench._bound(WORKLOADS["sam_vith_global"]) == "tensor"


def test_sources_hash_ignores_comments_not_code():
    a = 'int f(int x) {  // twice\n  return 2 * x; /* doubled */ }\nconst char* s = "//not a comment";'
    b = 'int f(int x) {\n    return 2 * x; }\nconst char* s = "//not a comment"; // note'
    c = 'int f(int x) { return 3 * x; }\nconst char* s = "//not a comment";'
    assert bench._code_tokens(a) == bench._code_tokens(b)
    assert bench._code_tokens(a) != bench._code_tokens(c)
    assert '"//not a comment"' in bench._code_tokens(a)


def test_torch_cpu_context_sample():
    w = WORKLOADS["toy"]
    tf, sec, slices, threads = bench._torch_cpu_sample(w, make_inputs(w), budget_s=0.05)
    assert tf > 0 and sec > 0 and 1 <= slices <= w.B * w.H and threads >= 1
