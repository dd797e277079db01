"""Benchmark of the fused SDPA forward on one GB300 (or N replicas).

Default workload: SAM ViT-H global encoder attention (8 images, 16 heads,
4096 x 4096 tokens of the 64 x 64 grid, d=80, bf16, decomposed relative
position with 127-row tables) -- the largest configuration, the one the
tensor-core metric is about.  One step = one attn_fwd over that whole batch
with the inputs resident in HBM.  The metric is attention forward TFLOP/s
counted as 4*B*H*Nq*Nk*d with the true head dim, and its fraction of the
measured dense bf16 peak.  The other workloads are timed the same way under
``suite``.

Timing: the K timed steps run as CUDA-graph replays of back-to-back
launches on one stream, bracketed by CUDA events, after W warm-up steps;
input sets rotate so their total exceeds 3x the L2 size (no L2 reuse
between consecutive steps).  SM clocks are sampled with nvidia-smi during
the timed region.  ``e2e`` repeats the measurement through the same C-ABI
call with pinned host buffers: each step copies Q, K, V host->device, runs
the kernel and copies O device->host, all inside the timed region; steps
are pipelined over two device buffer sets, so the copies of one step overlap
the kernel of another.

``--impl reference`` times the fp64 CPU oracle (test infrastructure, as it
stands) on the host cores on a bounded sample of the same workload.

Multi-GPU: the path has no exchange step; with torchrun each rank runs an
independent replica of the workload (weak scaling) and rank 0 reports the
aggregate over the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from scaled_dot_product_09_gb300.workloads import WORKLOADS, Workload, make_inputs  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
GRAPH_CHUNK = 100


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def _code_tokens(text: str) -> str:
    """C/C++/CUDA source without comments, whitespace runs collapsed: what
    the compiler sees (string and character literals kept as written)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def _kernel_sources_hash() -> str:
    """sha256 over the code (comments and whitespace left out) of the sources
    the forward kernel is compiled from -- its header, the PTX wrappers, the
    launchers and the per-(head dim, bias) instantiation units -- to tell
    whether recorded ncu counters of attn_fwd_kernel still describe the
    kernel being run (the backward's files and the host code do not enter)."""
    import hashlib
    d = os.path.join(ROOT, "scaled_dot_product_09_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(d)):
        fwd = name in ("attn_fwd_kernel.cuh", "sm103_ptx.cuh", "attn_launch.cuh") or (
            name.startswith("attn_d") and name.endswith(".cu"))
        if fwd:
            with open(os.path.join(d, name), encoding="utf-8") as f:
                h.update(name.encode() + b"\0" + _code_tokens(f.read()).encode())
    return h.hexdigest()


def _traffic(workload: str):
    """DRAM bytes (read + write) per launch from the recorded ncu capture of
    this workload, or None when there is none for the current sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(workload)
    except Exception:
        return None
    if not rec or rec.get("kernel_sources_sha256") != _kernel_sources_hash():
        return None
    return rec.get("dram_bytes_per_launch")


def _bound(w: Workload) -> str:
    # arithmetic intensity vs the machine balance (~300 flop/B for bf16 on GB300)
    return "tensor" if w.flops / w.io_bytes > 300 else "hbm"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except Exception:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _barrier(world):
    if world > 1:
        torch.distributed.barrier()


def _max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _gpu_bias(w, inp, dev, image=False):
    import scaled_dot_product_09_gb300 as sdpa
    if w.bias == "swin":
        return sdpa.SwinBias(inp.table.to(dev), w.win, w.grid_h, w.grid_w, w.shift,
                             layout="image" if image else "windows")
    if w.bias == "sam":
        return sdpa.SamBias(inp.rel_h.to(dev), inp.rel_w.to(dev), w.s_h, w.s_w)
    return None


class DeviceSets:
    """Rotating input sets resident in HBM, totalling > 3x L2.  image=True
    (Swin) views the same random tokens as [images, grid_h, grid_w, H, d]
    feature maps, which the kernel shifts and partitions itself."""

    def __init__(self, w: Workload, inp, dev, image=False):
        per = w.io_bytes
        self.n = max(2, math.ceil(3 * L2_BYTES / per) + 1)

        def put(t):
            if image:
                t = t.reshape(w.B // ((w.grid_h // w.win) * (w.grid_w // w.win)), w.grid_h, w.grid_w, w.H, w.d)
            return t.to(dev)

        self.q = [put(inp.q) for _ in range(self.n)]
        self.k = [put(inp.k) for _ in range(self.n)]
        self.v = [put(inp.v) for _ in range(self.n)]
        self.o = [torch.empty_like(self.q[0]) for _ in range(self.n)]
        self.bias = _gpu_bias(w, inp, dev, image)


def _time_bwd(w: Workload, stream, dev, steps: int):
    """Seconds per attn_bwd call (gradients of the whole workload) over
    rotating input sets, CUDA-graph replays like the forward."""
    import scaled_dot_product_09_gb300 as sdpa
    inp = make_inputs(w)
    n = max(2, math.ceil(3 * L2_BYTES / (2 * w.io_bytes)) + 1)
    g = torch.Generator().manual_seed(w.seed + 1000)
    dout = torch.randn(inp.q.shape, generator=g).to(inp.q.dtype)
    bias = _gpu_bias(w, inp, dev)
    sets = []
    need = sdpa.attn_bwd_workspace_size(w.B, w.H, w.Nq, w.Nk, w.d, bias)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    for _ in range(n):
        q, k, v, do = (x.to(dev) for x in (inp.q, inp.k, inp.v, dout))
        o, lse = sdpa.attn_fwd_train(q, k, v, scale=w.scale, bias=bias, stream=stream)
        if isinstance(bias, sdpa.SwinBias):
            d_bias = torch.zeros_like(bias.table)
        elif isinstance(bias, sdpa.SamBias):
            d_bias = torch.zeros((bias.rel_h.shape[0] + bias.rel_w.shape[0], w.d), dtype=torch.float32, device=dev)
        else:
            d_bias = None
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), d_bias)
        sets.append((q, k, v, o, lse, do, grads))
    torch.cuda.synchronize()

    def step(i):
        q, k, v, o, lse, do, grads = sets[i % n]
        sdpa.attn_bwd(q, k, v, o, do, lse=lse, scale=w.scale, bias=bias, stream=stream, grads=grads, workspace=ws)

    with torch.cuda.stream(stream):
        for i in range(3):
            step(i)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(steps):
            step(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        graph.replay()
        start.record(stream)
        graph.replay()
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3 / steps


def _attn(w: Workload, q, k, v, out, bias, stream):
    """One step through the public API: attn_fwd, or attn_fwd_varlen for a
    nested batch."""
    import scaled_dot_product_09_gb300 as sdpa
    if w.varlen:
        sdpa.attn_fwd_varlen(q, k, v, w.cu_seqlens_q, w.cu_seqlens_k, w.H, out=out, scale=w.scale, stream=stream)
    else:
        sdpa.attn_fwd(q, k, v, out=out, scale=w.scale, bias=bias, stream=stream)


def _time_device(w: Workload, sets: DeviceSets, steps: int, warmup: int, stream):
    """Returns (total seconds of the K timed steps, number of launches, launches
    per captured graph)."""
    import scaled_dot_product_09_gb300 as sdpa

    def step(i):
        j = i % sets.n
        _attn(w, sets.q[j], sets.k[j], sets.v[j], sets.o[j], sets.bias, stream)

    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):
            step(i)
    torch.cuda.synchronize()
    chunk = min(GRAPH_CHUNK, max(1, steps))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(chunk):
            step(i)
    torch.cuda.synchronize()
    full, rest = divmod(steps, chunk)
    rest_graph = None
    if rest:
        rest_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(rest_graph, stream=stream):
            for i in range(rest):
                step(i)
    with torch.cuda.stream(stream):
        graph.replay()  # one warm replay of the captured sequence
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(full):
            graph.replay()
        if rest_graph is not None:
            rest_graph.replay()
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3, steps, chunk


def _time_e2e(w: Workload, inp, steps: int, warmup: int, stream, dev, depth: int = 2):
    """Pinned host buffers; every step copies its Q, K, V host->device, runs
    attn_fwd and copies O device->host.  Steps are pipelined over `depth`
    device buffer sets with one stream per copy direction, so one step's
    copies overlap another step's kernel; events keep
    each set's copy-in, kernel and copy-out in order.  Returns the seconds,
    H2D bytes and D2H bytes per step."""
    import scaled_dot_product_09_gb300 as sdpa
    hq, hk, hv = (x.pin_memory() for x in (inp.q, inp.k, inp.v))
    hos = [torch.empty_like(hq).pin_memory() for _ in range(depth)]
    sets = [tuple(torch.empty_like(x, device=dev) for x in (hq, hk, hv, hq)) for _ in range(depth)]
    bias = _gpu_bias(w, inp, dev)
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(depth)]    # set j's inputs landed
    ev_run = [torch.cuda.Event() for _ in range(depth)]   # set j's kernel finished
    ev_out = [torch.cuda.Event() for _ in range(depth)]   # set j's output copied back

    def step(i):
        j = i % depth
        dq, dk, dv, do = sets[j]
        s_in.wait_event(ev_run[j])  # the set's previous kernel has read its inputs
        with torch.cuda.stream(s_in):
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
        ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        stream.wait_event(ev_out[j])  # the set's previous output has been copied back
        _attn(w, dq, dk, dv, do, bias, stream)
        ev_run[j].record(stream)
        s_out.wait_event(ev_run[j])
        with torch.cuda.stream(s_out):
            hos[j].copy_(do, non_blocking=True)
        ev_out[j].record(s_out)

    n = max(depth, min(steps, 200))
    for i in range(max(warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for i in range(n):
        step(i)
    end.record(s_out)  # after the last copy-out, which follows every earlier step
    end.synchronize()
    torch.cuda.synchronize()
    sec = start.elapsed_time(end) / 1e3 / n
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
    d2h = hos[0].numel() * hos[0].element_size()
    return sec, h2d, d2h


def _suite(stream, dev, peaks, names):
    """Quick device-only numbers for the other workloads (same method).  A
    name ending in "@image" times that Swin workload in the image layout."""
    out = {}
    for name in names:
        base, _, layout = name.partition("@")
        w = WORKLOADS[base]
        if layout == "bwd":
            # backward (attn_bwd, tensor cores): algorithmic work 10*B*H*Nq*Nk*d, the
            # five products S, dP, dV, dK, dQ (the kernels recompute S and dP in
            # both passes of the long-sequence path, which is not counted)
            t = _time_bwd(w, stream, dev, 20 if w.flops > 1e11 else 50)
            tf = 2.5 * w.flops / t / 1e12
            out[name] = {"us_per_step": round(t * 1e6, 2), "tflops": round(tf, 2), "bound": "tensor",
                         "frac": round(tf / peaks["bf16_tflops"], 4)}
            torch.cuda.empty_cache()
            continue
        inp = make_inputs(w)
        sets = DeviceSets(w, inp, dev, image=layout == "image")
        steps = max(20, min(2000, int(0.3 / max(w.flops / 1e15, 1e-6))))
        sec, _, _ = _time_device(w, sets, steps, 3, stream)
        t = sec / steps
        tf = w.flops / t / 1e12
        gbs = w.io_bytes / t / 1e9
        bound = _bound(w)
        frac = tf / peaks["bf16_tflops"] if bound == "tensor" else gbs / peaks["hbm_gbs"]
        out[name] = {"us_per_step": round(t * 1e6, 2), "tflops": round(tf, 2), "gbs": round(gbs, 1),
                     "bound": bound, "frac": round(frac, 4)}
        del sets
        torch.cuda.empty_cache()
    return out


def _oracle_sample(w: Workload, inp, budget_s: float, nthreads: int = 0):
    """Time the oracle on whole rows until ~budget_s; returns (TFLOP/s,
    seconds, rows, threads).  A nested batch is sampled on its first
    sequence."""
    import oracle
    if w.varlen:
        lq, lk = w.seqlens_q[0], w.seqlens_k[0]
        q = inp.q[:w.H * lq].double().reshape(w.H, lq, w.d).numpy()
        k = inp.k[:w.H * lk].double().reshape(w.H, lk, w.d).numpy()
        v = inp.v[:w.H * lk].double().reshape(w.H, lk, w.d).numpy()
        w = w.with_(B=1, Nq=lq, Nk=lk, seqlens_q=(), seqlens_k=())
    else:
        q = inp.q.double().reshape(w.B * w.H, w.Nq, w.d).numpy()
        k = inp.k.double().reshape(w.B * w.H, w.Nk, w.d).numpy()
        v = inp.v.double().reshape(w.B * w.H, w.Nk, w.d).numpy()
    BH = w.B * w.H
    if w.bias == "swin":
        b = oracle.Bias("swin", table=inp.table.double().numpy(), win=w.win, grid_h=w.grid_h,
                        grid_w=w.grid_w, shift=w.shift)
    elif w.bias == "sam":
        b = oracle.Bias("sam", rel_h=inp.rel_h.double().numpy(), rel_w=inp.rel_w.double().numpy(),
                        s_h=w.s_h, s_w=w.s_w)
    else:
        b = None
    # calibrate on a few rows, then size the sample to the budget: a prefix of
    # the workload's rows, or whole passes over it when one pass is shorter
    probe_rows = min(w.Nq, 64)
    t0 = time.perf_counter()
    _, used = oracle.attn_rows(q, k, v, w.H, w.scale, list(range(probe_rows)), b, nthreads)
    per_row = max((time.perf_counter() - t0) / probe_rows, 1e-9)
    total = BH * w.Nq
    rows = int(min(total, max(w.Nq, budget_s / per_row)))
    ids = list(range(rows))
    rows_done, sec = 0, 0.0
    while True:
        t0 = time.perf_counter()
        _, used = oracle.attn_rows(q, k, v, w.H, w.scale, ids, b, nthreads)
        sec += time.perf_counter() - t0
        rows_done += rows
        if rows < total or sec >= budget_s:
            break
    flops = 4.0 * rows_done * w.Nk * w.d
    return flops / sec / 1e12, sec, rows_done, used


def _torch_cpu_sample(w: Workload, inp, budget_s: float):
    """Context for the no-bias workloads: torch's CPU scaled_dot_product_attention
    in fp32 (the "native C++" backend of the Diffusers page, section 加速
    Transformer 块) on whole slices until ~budget_s.  Returns (TFLOP/s,
    seconds, slices, threads)."""
    BH = w.B * w.H
    q = inp.q.float().reshape(BH, w.Nq, w.d)
    k = inp.k.float().reshape(BH, w.Nk, w.d)
    v = inp.v.float().reshape(BH, w.Nk, w.d)
    done, sec = 0, 0.0
    while done < BH and sec < budget_s:
        t0 = time.perf_counter()
        torch.nn.functional.scaled_dot_product_attention(q[done:done + 1], k[done:done + 1], v[done:done + 1],
                                                         scale=w.scale)
        sec += time.perf_counter() - t0
        done += 1
    return 4.0 * done * w.Nq * w.Nk * w.d / sec / 1e12, sec, done, torch.get_num_threads()


def run_reference(args, w: Workload, world, rank):
    if rank != 0:
        return 0
    inp = make_inputs(w)
    steps, warmup = args.steps, args.warmup
    per_step_budget = max(0.05, min(5.0, 60.0 / max(1, steps + warmup)))
    for _ in range(warmup):
        _oracle_sample(w, inp, per_step_budget)
    flops, secs, rows_total, used = 0.0, 0.0, 0, 0
    for _ in range(steps):
        tf, sec, rows, used = _oracle_sample(w, inp, per_step_budget)
        flops += tf * 1e12 * sec
        secs += sec
        rows_total += rows
    value = flops / secs / 1e12
    total = w.H * w.seqlens_q[0] if w.varlen else w.B * w.H * w.Nq
    of_seq = " of the first sequence" if w.varlen else ""
    rows_step = rows_total // steps
    per = (f"{rows_step} of {total} query rows{of_seq}" if rows_step <= total
           else f"{rows_step // total} whole passes over the {total} query rows{of_seq}")
    line = {
        "impl": "reference", "metric": args.metric, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": warmup,
        "ms_per_step": secs / steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                   "bias": w.bias, "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": used, "kind": "oracle",
                         "sample": f"{per} per step (whole rows, fp64 oracle, OpenMP over rows)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="sam_vith_global", choices=sorted(WORKLOADS))
    ap.add_argument("--no-suite", action="store_true", help="skip the other workloads' numbers")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--batch", type=int, default=0,
                    help="profiling aid: run the workload with this B (a smaller case of the same kernels)")
    ap.add_argument("--bwd-only", action="store_true",
                    help="profiling aid: time only attn_bwd on the workload and print its numbers")
    args = ap.parse_args(argv)
    args.metric = "attention fwd TFLOP/s (4*B*H*Nq*Nk*d)"
    world, rank, local = _dist()
    w = WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(B=args.batch)

    if args.impl == "reference":
        return run_reference(args, w, world, rank)

    if world > 1:
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import scaled_dot_product_09_gb300 as sdpa
    sdpa.load_library()
    peaks = _peaks()
    stream = torch.cuda.Stream(device=dev)
    if args.bwd_only:
        t = _time_bwd(w, stream, dev, max(1, args.steps))
        if rank == 0:
            print(json.dumps({"bwd_only": w.name, "B": w.B, "us_per_step": t * 1e6,
                              "tflops": 2.5 * w.flops / t / 1e12}))
        return 0

    # CPU baseline first (host only), before any GPU timing.
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        inp_cpu = make_inputs(w)
        tf, sec, rows, used = _oracle_sample(w, inp_cpu, 15.0)
        total = w.H * w.seqlens_q[0] if w.varlen else w.B * w.H * w.Nq
        what = (f"{rows} of {total} query rows" if rows <= total
                else f"{rows // total} whole passes over all {total} query rows")
        if w.varlen:
            what += " of the first sequence"
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": used, "kind": "oracle",
               "sample": f"{what} ({sec:.1f} s, fp64, OpenMP over rows)"}
        if w.bias == "none" and not w.varlen:
            ttf, tsec, tsl, tth = _torch_cpu_sample(w, inp_cpu, 5.0)
            cpu["torch_cpu_sdpa_fp32"] = {"value": ttf, "unit": "TFLOP/s", "threads": tth,
                                          "sample": f"{tsl} of {w.B * w.H} slices ({tsec:.1f} s)"}

    inp = make_inputs(w)
    sets = DeviceSets(w, inp, dev)
    n_sets = sets.n
    _barrier(world)
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    sec, launches, chunk = _time_device(w, sets, args.steps, args.warmup, stream)
    clocks = sampler.stop()
    torch.cuda.synchronize()
    _barrier(world)
    sec = _max_over_ranks(sec, world, dev)

    t_step = sec / args.steps
    value = world * w.flops / t_step / 1e12
    bound = _bound(w)
    if bound == "hbm":
        achieved = w.io_bytes / t_step / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": _traffic(w.name),
                "peak_source": peaks["source"], "bytes_per_launch": w.io_bytes}
    else:
        achieved = w.flops / t_step / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "traffic": _traffic(w.name),
                "peak_source": peaks["source"], "flops_per_launch": w.flops}

    e2e_sec, h2d, d2h = _time_e2e(w, inp, args.steps, args.warmup, stream, dev)
    e2e_sec = _max_over_ranks(e2e_sec, world, dev)
    suite = None
    if rank == 0 and not args.no_suite:
        del sets
        torch.cuda.empty_cache()
        suite = _suite(stream, dev, peaks, [n for n in ("swin_t_stage1", "swin_t_stage1@image", "swin_t_stage1@bwd",
                                                        "sam_vith_window", "sam_vith_window@bwd", "sam_vith_global",
                                                        "sam_vith_global@bwd", "sam_vith_global_768", "sam_vith_global_768@bwd", "sd_unet_self",
                                                        "sd_unet_self@bwd", "sd_unet_cross", "sd_unet_self_varlen")
                                            if n != w.name])
    if rank == 0:
        line = {
            "metric": args.metric, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                       "bias": w.bias, "global_batch": w.B * world, "parallelism": f"replicas{world}",
                       "l2": f"{n_sets} rotating input sets, {n_sets * w.io_bytes / 2**20:.0f} MiB > 3x L2",
                       "launch": f"CUDA graphs of {chunk} back-to-back "
                                 f"{'attn_fwd_varlen' if w.varlen else 'attn_fwd'} launches"},
            "roofline": roof,
            "gpu_launches": launches,
            "clocks": clocks,
            "e2e": {"value": world * w.flops / e2e_sec / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "cpu_baseline": cpu,
        }
        if suite is not None:
            line["suite"] = suite
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
