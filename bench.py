"""Benchmark of paged-attention decode on GB300.

One step = one decode call for each workload of the chosen group (default:
the long-context split-KV group, batch in {1, 4} x context in {8192, 32768,
131072}, 32 query / 8 kv heads, head_dim 128, block_size 16, bf16), each
through ``pa_decode_splitkv`` with the automatic partition choice (which runs
the single pass when one partition suffices).  Inputs rotate among enough
independent seeded sets that every step reads from HBM, not L2.  The step is
captured once per input set as a CUDA graph and replayed, so host launch
overhead does not pace the GPU.  Multi-token workloads (``--workload multi``:
q_len > 1 query tokens per sequence, causal over the new tokens) run through
``pa_decode_multi`` instead.

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
on the same workload instead.  Under torchrun each rank runs an independent
replica on its own GPU (the decode step has no cross-GPU exchange).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_attention_08_gb300 import workloads  # noqa: E402

METRIC = "paged decode µs/step and achieved HBM GB/s (fraction of GB300 roofline)"
FALLBACK_HBM_GBS = 6800.0
DTYPE_NAME = {torch.float16: "f16", torch.bfloat16: "bf16", torch.float32: "f32"}


# ---------------------------------------------------------------------------
# bytes
# ---------------------------------------------------------------------------
def algorithmic_bytes(x: workloads.Inputs, out_elem: int = 4) -> int:
    """Bytes one decode call must move at least once: K and V of every attended
    token for each kv head, q, the output, the block table and the lengths.
    (With several query tokens the last one attends every cached token.)"""
    B, D = x.q.shape[0], x.q.shape[-1]
    _, bs, Hkv, _ = x.k_cache.shape
    e = x.q.element_size()
    mb = x.block_tables.shape[1]
    tokens = sum(min(max(t, 0), mb * bs) for t in x.lens_host)
    return (tokens * Hkv * D * 2 * e + x.q.numel() * e + x.q.numel() * out_elem
            + B * mb * 4 + B * 4)


def algorithmic_flops(x: workloads.Inputs) -> int:
    """Multiply-adds x 2 of one call: S = q.K and O = P.V over every attended
    token of every query row (with several query tokens, token i of a sequence
    attends its causal prefix of T - Q + i + 1 tokens)."""
    D = x.q.shape[-1]
    H = x.q.shape[-2]
    _, bs, _, _ = x.k_cache.shape
    cap = x.block_tables.shape[1] * bs
    Q = x.q.shape[1] if x.q.dim() == 4 else 1
    rows_tokens = 0
    for t in x.lens_host:
        t = max(t, 0)
        for i in range(Q):
            rows_tokens += max(0, min(t - Q + i + 1, cap))
    return 4 * rows_tokens * H * D


def decode_call(pa, out, q, k_cache, v_cache, block_tables, context_lens, scale, max_context_len,
                partition_tokens, workspace, stream):
    """One decode call through the public API: one query token per sequence
    (q [B, H, D]) or several (q [B, Q, H, D])."""
    fn = pa.decode_multi if q.dim() == 4 else pa.decode_splitkv
    fn(out, q, k_cache, v_cache, block_tables, context_lens, scale, max_context_len,
       partition_tokens, workspace=workspace, stream=stream)


def workspace_bytes(pa, x, partition_tokens) -> int:
    fn = pa.workspace_size_multi if x.q.dim() == 4 else pa.workspace_size
    return fn(x.q, x.k_cache, x.block_tables, torch.float32, x.max_context_len, partition_tokens)


def oracle_rows(oracle, h, rows, token=None):
    """fp64 oracle output of (b, h) rows; for several query tokens, those of
    query token `token` (the one-token decode of its causal prefix)."""
    if h.q.dim() == 3:
        return oracle.decode_rows(h.q, h.k_cache, h.v_cache, h.block_tables, h.context_lens,
                                  h.scale, rows)
    Q = h.q.shape[1]
    prefix = torch.clamp(h.context_lens - Q + token + 1, min=0)
    return oracle.decode_rows(h.q[:, token].contiguous(), h.k_cache, h.v_cache, h.block_tables,
                              prefix, h.scale, rows)


def input_bytes(x: workloads.Inputs) -> int:
    return sum(t.numel() * t.element_size()
               for t in (x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens))


# ---------------------------------------------------------------------------
# distributed helpers (replicas: no data-path collective)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, device) -> float:
    """Max over ranks (identity for one process)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_max_list(values, device):
    """Element-wise max over ranks of a list of floats (identity for one process)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return list(values)
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def reduce_sum(value: float, device) -> float:
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while active."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="pa_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["active_mask", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names[1:], r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# peaks
# ---------------------------------------------------------------------------
def tensor_peak():
    """Dense bf16 (= fp16) tensor peak in TFLOP/s for a kernel timed alone."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(path))["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e, nominal (context beside the measured peak)


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        v = float(json.load(open(path))["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch recorded from an ncu capture (profiles/), or None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    try:
        for line in open(path):
            if line.startswith("dram_bytes_per_launch_full_size:"):
                return int(float(line.split(":", 1)[1]))
    except OSError:
        pass
    return None


def dominant_traffic(plan: dict, workload: str):
    """DRAM bytes per launch of the kernel the plan picked for `workload`: the
    tile kernel's summaries are profiles/pa_tile_<workload>.txt, the warp-level
    kernel's pa_attn_<workload>.txt (an HBM-bound call may run on either)."""
    return ncu_traffic("pa_tile" if "tile" in plan["kernel"] else "pa_attn", workload)


# ---------------------------------------------------------------------------
# CPU oracle arm
# ---------------------------------------------------------------------------
def oracle_step(sets_host, threads=1):
    """One whole step through the oracle; with threads > 1 its independent
    (sequence, head) rows -- sequences for several query tokens -- run on that
    many host threads.  Returns the most threads a call used."""
    import oracle
    used = 1
    for x in sets_host:
        args = (x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale)
        if threads <= 1:
            (oracle.decode_multi if x.q.dim() == 4 else oracle.decode)(*args)
        else:
            fn = oracle.decode_multi_mt if x.q.dim() == 4 else oracle.decode_mt
            used = max(used, fn(*args, threads=threads)[1])
    return used


def time_oracle(sets_host, min_s=10.0, max_steps=None, threads=1):
    """Whole oracle steps until ``min_s`` elapse; (seconds/step, steps, threads used)."""
    n, used, t0 = 0, 1, time.perf_counter()
    while True:
        used = max(used, oracle_step(sets_host, threads))
        n += 1
        el = time.perf_counter() - t0
        if el >= min_s or (max_steps and n >= max_steps):
            return el / n, n, used


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------
def describe(group):
    specs = [workloads.SPECS[n] for n in workloads.GROUPS[group]]

    def shape(s):
        return (f"H{s.num_heads}/Hkv{s.num_kv_heads}, D{s.head_dim}, bs{s.block_size}, "
                f"{DTYPE_NAME[s.dtype]} K/V")

    def case(s):
        return f"({s.batch},{s.lens}" + (f",{s.q_len})" if s.q_len > 1 else ")")

    head = f"(batch, ctx{', q_len' if any(s.q_len > 1 for s in specs) else ''})"
    if len({shape(s) for s in specs}) == 1:
        return (f"{group}: {head} in {{{', '.join(case(s) for s in specs)}}}, "
                f"{shape(specs[0])}, fp32 out")
    return f"{group}: {head}: " + "; ".join(f"{case(s)} {shape(s)}" for s in specs) + "; fp32 out"


def bench_config(args):
    """The ``config`` object of the JSON line, identical for both arms: what
    workload is measured, with which split, and how L2 is kept out."""
    pt = args.partition_tokens
    return {"workload": describe(args.workload),
            "partition_tokens": ("balanced split" if getattr(args, "balanced", False) else
                                 "automatic" if pt == 0 else
                                 "each workload's own" if pt < 0 else pt),
            "l2": "inputs rotate over independent seeded sets totalling more than 3x L2, "
                  "so every step reads HBM"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    names = workloads.GROUPS[args.workload]
    sets = [workloads.make(n, seed=0, device="cpu") for n in names]
    step_bytes = sum(algorithmic_bytes(x) for x in sets)
    threads = oracle.host_threads()
    used = 1
    for _ in range(args.warmup):
        used = max(used, oracle_step(sets, threads))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        used = max(used, oracle_step(sets, threads))
    sec = (time.perf_counter() - t0) / max(1, args.steps)
    gbs = step_bytes / sec / 1e9
    sample = (f"{args.steps} whole steps of the {args.workload} group (every sequence, every "
              f"head), fp64 oracle on {used} host threads of {oracle.cpu_model()}")
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": bench_config(args),
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": used, "kind": "oracle",
                             "sample": sample, "cpu_model": oracle.cpu_model()},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(workloads.GROUPS), default="long")
    ap.add_argument("--partition-tokens", default="0",
                    help="split-KV partition size in tokens; 0 = the library's automatic choice; "
                         "-1 = each workload's own (512 tokens for the long group); "
                         "'balanced' = the balanced split")
    ap.add_argument("--regions", type=int, default=7,
                    help="timed regions of --steps steps each; the line reports their median")
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of graph replay")
    ap.add_argument("--graph-per-step", action="store_true",
                    help="replay one graph per step instead of one per loop over the input sets")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--with-append", action="store_true",
                    help="each call first appends the step's new token (the last of every "
                         "context) with pa_append_kv, as a full decode iteration does "
                         "(one-token workloads only)")
    ap.add_argument("--min-warmup-s", type=float, default=1.0,
                    help="keep warming up (graph replays) at least this long")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    args.balanced = args.partition_tokens == "balanced"
    args.partition_tokens = 0 if args.balanced else int(args.partition_tokens)

    if args.impl == "reference":
        return run_reference(args)

    import paged_kv_attention_08_gb300 as pa
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    names = workloads.GROUPS[args.workload]
    specs = [workloads.SPECS[n] for n in names]
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    set0 = [workloads.make(n, seed=0, device=dev) for n in names]
    set_bytes = sum(input_bytes(x) for x in set0)
    nsets = max(1, min(64, math.ceil(3 * l2 / set_bytes) + 1))
    sets = [set0] + [[workloads.make(n, seed=100 * r + rank, device=dev) for n in names]
                     for r in range(1, nsets)]
    pts = [pa.PARTITION_BALANCED if args.balanced else
           s.partition_tokens if args.partition_tokens < 0 else args.partition_tokens for s in specs]
    if args.with_append and any(s.q_len > 1 for s in specs):
        print(json.dumps({"metric": METRIC, "error": "--with-append needs one-token workloads"}))
        return 1

    outs = [[torch.empty(x.q.shape, dtype=torch.float32, device=dev) for x in st] for st in sets]
    ws = []
    for i in range(len(set0)):
        # every rotated set has its own longest context, hence its own plan
        need = max(workspace_bytes(pa, st[i], pts[i]) for st in sets)
        ws.append(torch.empty(max(need, 16), dtype=torch.uint8, device=dev))
    sms = props.multi_processor_count
    # the library's own description of each call's plan on this device
    plans = {names[i]: pa.plan_info(x.q, x.k_cache, x.block_tables, x.max_context_len, pts[i])
             for i, x in enumerate(set0)}
    # kernels per call: the attention kernel, plus the combine kernel when the
    # partials go through the workspace
    launches_per_step = sum(2 if p["reduce"] in ("workspace+combine kernel", "balanced split")
                            else 1 for p in plans.values()) + (len(set0) if args.with_append else 0)

    stream = torch.cuda.Stream(device=dev)

    new_kv = {}
    if args.with_append:
        for si, st_ in enumerate(sets):
            for i, x in enumerate(st_):
                B, _, D = x.q.shape
                Hkv = x.k_cache.shape[2]
                gk = torch.Generator(device=dev).manual_seed(1000 + si * 10 + i)
                kn = torch.randn(B, Hkv, D, generator=gk, device=dev).to(x.q.dtype)
                vn = torch.randn(B, Hkv, D, generator=gk, device=dev).to(x.q.dtype)
                new_kv[(si, i)] = (kn, vn, (x.context_lens - 1).clamp(min=-1).contiguous())

    def call(si, i, st):
        x = sets[si][i]
        if args.with_append:
            kn, vn, pos = new_kv[(si, i)]
            pa.append_kv(x.k_cache, x.v_cache, kn, vn, x.block_tables, pos, stream=st)
        decode_call(pa, outs[si][i], x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens,
                    x.scale, x.max_context_len, pts[i], ws[i], st)

    # ---- parity before timing (sampled rows against the fp64 oracle) ----
    import oracle
    with torch.cuda.stream(stream):
        for i in range(len(set0)):
            call(0, i, stream)
    stream.synchronize()
    max_err = 0.0
    if rank == 0:
        for i, x in enumerate(set0):
            g = np.random.default_rng(i)
            B, H = x.q.shape[0], x.q.shape[-2]
            rows = np.stack([g.integers(0, B, 16), g.integers(0, H, 16)], 1).astype(np.int32)
            h = x.to("cpu")
            tokens = [None] if x.q.dim() == 3 else sorted({0, x.q.shape[1] - 1})
            for tok in tokens:
                want = oracle_rows(oracle, h, rows, tok)
                o = outs[0][i] if tok is None else outs[0][i][:, tok]
                got = o[rows[:, 0], rows[:, 1]].double().cpu().numpy()
                max_err = max(max_err, float(np.abs(got - want).max()))
        if not max_err <= 2e-3:
            print(json.dumps({"metric": METRIC, "error": f"parity failed: max_err {max_err}"}))
            return 1

    # ---- graphs: one step per input set, and a loop graph that runs every
    # set's step in turn (nsets steps per replay: programmatic dependent launch
    # then links every call, step boundaries included, instead of one graph
    # launch per step) ----
    graphs = []
    loop_graph = None
    if not args.no_graph:
        with torch.cuda.stream(stream):
            for si in range(nsets):               # warm every set once before capture
                for i in range(len(set0)):
                    call(si, i, stream)
        stream.synchronize()
        for si in range(nsets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(len(set0)):
                    call(si, i, torch.cuda.current_stream())
            graphs.append(g)
        if nsets > 1 and not args.graph_per_step:
            loop_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(loop_graph, stream=stream):
                for si in range(nsets):
                    for i in range(len(set0)):
                        call(si, i, torch.cuda.current_stream())
    torch.cuda.synchronize()

    def step(k, st):
        si = k % nsets
        if graphs:
            graphs[si].replay()
        else:
            for i in range(len(set0)):
                call(si, i, st)

    step_bytes = sum(algorithmic_bytes(x) for x in set0)
    with ClockSampler(local) as clocks:
        with torch.cuda.stream(stream):
            t_warm = time.perf_counter()
            k = 0
            while k < args.warmup or time.perf_counter() - t_warm < args.min_warmup_s:
                step(k, stream)
                k += 1
                if k % 256 == 0:
                    stream.synchronize()
            if loop_graph is not None:
                for _ in range(3):
                    loop_graph.replay()
            stream.synchronize()
            # --regions timed regions of exactly --steps steps each, every one
            # bracketed by a barrier and a device synchronize; the line reports
            # the median region (max over ranks per region)
            region_ms = []
            for _ in range(max(1, args.regions)):
                barrier()
                torch.cuda.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                k = 0
                if loop_graph is not None:      # whole loops of the nsets steps
                    while k + nsets <= args.steps:
                        loop_graph.replay()
                        k += nsets
                while k < args.steps:           # the rest, one step graph each
                    step(k, stream)
                    k += 1
                e1.record(stream)
                e1.synchronize()
                torch.cuda.synchronize()
                barrier()
                region_ms.append(e0.elapsed_time(e1))

            # per-call durations: one graph per workload that runs its call on the
            # input sets in turn, at least 8 calls back to back (the sets together
            # exceed 3x L2, so every call reads HBM); replay time / calls = the
            # call's device time (attention kernel plus, when it splits, combine)
            per_call = [[] for _ in set0]
            call_graphs = []
            calls_per_graph = nsets * max(1, math.ceil(8 / nsets))   # at least 8 calls
            for i in range(len(set0)):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for k in range(calls_per_graph):
                        call(k % nsets, i, torch.cuda.current_stream())
                call_graphs.append(g)
            # hot: the same call on input set 0 only, so its inputs stay in L2
            # when they fit (reported beside the cold figures, not the metric)
            per_call_hot = [[] for _ in set0]
            hot_graphs = []
            for i in range(len(set0)):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for k in range(calls_per_graph):
                        call(0, i, torch.cuda.current_stream())
                hot_graphs.append(g)
            reps = max(3, min(args.steps // 10, 50))
            for _ in range(reps):
                for graphs_, acc in ((call_graphs, per_call), (hot_graphs, per_call_hot)):
                    for i, g in enumerate(graphs_):
                        a = torch.cuda.Event(enable_timing=True)
                        b = torch.cuda.Event(enable_timing=True)
                        a.record(stream)
                        g.replay()
                        b.record(stream)
                        b.synchronize()
                        acc[i].append(a.elapsed_time(b) / calls_per_graph)
    clk = clocks.summary() if rank == 0 else None

    region_ms = reduce_max_list(region_ms, dev)
    ms_step = statistics.median(region_ms) / args.steps
    total_bytes = reduce_sum(float(step_bytes), dev)
    value = total_bytes / (ms_step * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()

    # dominant call: largest share of time; its achieved bytes / its own duration
    call_us = [statistics.median(v) * 1e3 for v in per_call]
    dom = int(np.argmax(call_us))
    dom_bytes = algorithmic_bytes(set0[dom])
    dom_gbs = dom_bytes / (call_us[dom] * 1e-6) / 1e9
    dom_name = names[dom]
    # the bound of the dominant call: its FLOPs per byte against the ridge of
    # the measured peaks (a multi-token call with many query rows is a
    # contraction, a decode call streams K and V)
    tpeak, tpeak_kind = tensor_peak()
    dom_flops = algorithmic_flops(set0[dom])
    dom_tflops = dom_flops / (call_us[dom] * 1e-6) / 1e12
    tensor_bound = dom_flops / dom_bytes > tpeak * 1e12 / (peak * 1e9)
    per_call_rates = {n: {"GB/s": round(algorithmic_bytes(x) / (u * 1e-6) / 1e9, 1),
                          "frac_of_measured_hbm": round(algorithmic_bytes(x) / (u * 1e-6) / 1e9
                                                        / peak, 4),
                          "TFLOP/s": round(algorithmic_flops(x) / (u * 1e-6) / 1e12, 2)}
                      for n, x, u in zip(names, set0, call_us)}

    # ---- end to end: host buffers, copies inside the timed region ----
    # A decode step as a serving loop runs it: the paged K/V cache is state
    # resident on the device (filled once, before timing); each step's inputs
    # -- the query, the new token's key and value, the block tables and the
    # context lengths of every workload -- sit in one pinned host buffer and
    # are copied to the device in one transfer; the step appends the new
    # token to the cache (pa_append_kv), runs the decode calls through the
    # public API, and copies the outputs back to pinned host memory.  Steps
    # are double-buffered: a step's input copy (its own stream) overlaps the
    # previous step's kernels.  Multi-token workloads append nothing (their
    # new tokens are already in the cache).
    e2e = None
    if not args.no_e2e:
        host = [x.to("cpu") for x in set0]
        fields = []      # (workload, name, host tensor)
        for i, (h, x) in enumerate(zip(host, set0)):
            fields.append((i, "q", h.q))
            if h.q.dim() == 3:
                B, _, D = h.q.shape
                Hkv = h.k_cache.shape[2]
                gk = torch.Generator().manual_seed(2000 + i)
                fields.append((i, "k_new", torch.randn(B, Hkv, D, generator=gk).to(h.q.dtype)))
                fields.append((i, "v_new", torch.randn(B, Hkv, D, generator=gk).to(h.q.dtype)))
                fields.append((i, "positions", (h.context_lens - 1).clamp(min=-1).contiguous()))
            fields.append((i, "block_tables", h.block_tables))
            fields.append((i, "context_lens", h.context_lens))
        offs, total = [], 0
        for _, _, t in fields:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        pin_in = torch.empty(total, dtype=torch.uint8).pin_memory()
        for (_, _, t), o in zip(fields, offs):
            n = t.numel() * t.element_size()
            pin_in[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
        # the resident caches: copies of input set 0's, so that the timed
        # region's appends leave the other measurements' inputs untouched
        caches = [(x.k_cache.clone(), x.v_cache.clone()) for x in set0]
        out_elems = [x.q.numel() for x in set0]
        out_offs = [sum(out_elems[:i]) for i in range(len(out_elems))]
        nbuf = 2
        dev_in = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(nbuf)]
        dev_out = [torch.empty(sum(out_elems), dtype=torch.float32, device=dev) for _ in range(nbuf)]
        pin_out = [torch.empty(sum(out_elems), dtype=torch.float32).pin_memory() for _ in range(nbuf)]
        views = [[dict() for _ in host] for _ in range(nbuf)]
        for k in range(nbuf):
            for (i, name, t), o in zip(fields, offs):
                n = t.numel() * t.element_size()
                views[k][i][name] = dev_in[k][o:o + n].view(t.dtype).view(t.shape)
        ws2 = [[torch.empty_like(w) for w in ws] for _ in range(nbuf)]
        h2d, d2h = total, pin_out[0].numel() * 4
        e2e_steps = max(4, min(args.steps, 50))
        copy_stream = torch.cuda.Stream(device=dev)
        copied = [torch.cuda.Event() for _ in range(nbuf)]
        consumed = [torch.cuda.Event() for _ in range(nbuf)]

        def e2e_step(k):
            buf = k % nbuf
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(consumed[buf])          # step k-2's kernels are done
                dev_in[buf].copy_(pin_in, non_blocking=True)
                copied[buf].record(copy_stream)
            stream.wait_event(copied[buf])
            with torch.cuda.stream(stream):
                for i, x in enumerate(set0):
                    v = views[buf][i]
                    kc, vc = caches[i]
                    if "k_new" in v:
                        pa.append_kv(kc, vc, v["k_new"], v["v_new"], v["block_tables"],
                                     v["positions"], stream=stream)
                    o = dev_out[buf][out_offs[i]:out_offs[i] + out_elems[i]].view(x.q.shape)
                    decode_call(pa, o, v["q"], kc, vc, v["block_tables"], v["context_lens"],
                                x.scale, x.max_context_len, pts[i], ws2[buf][i], stream)
                pin_out[buf].copy_(dev_out[buf], non_blocking=True)
                consumed[buf].record(stream)

        for k in range(nbuf):
            consumed[k].record(stream)
        for k in range(3):
            e2e_step(k)
        torch.cuda.synchronize()
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        copy_stream.wait_event(a)
        for k in range(e2e_steps):
            e2e_step(k)
        b.record(stream)
        b.synchronize()
        ms_e2e = reduce_max(a.elapsed_time(b), dev) / e2e_steps
        e2e = {"value": total_bytes / (ms_e2e * 1e-3) / 1e9, "unit": "GB/s",
               "ms_per_step": ms_e2e, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": e2e_steps,
               "step": "H2D of q, the new token's K/V, block tables and lengths (pinned); "
                       "pa_append_kv + decode per workload, eager; D2H of the outputs; "
                       "K/V cache resident on the device",
               "pipeline": "2 buffers; step k+1 H2D (copy stream) overlaps step k kernels"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # whole steps of the group on all host threads for >= 10 s; one thread
        # on a bounded sample: the group's smallest call, repeated for >= 5 s
        import oracle
        host = [x.to("cpu") for x in set0]
        sec, n, used = time_oracle(host, min_s=10.0, threads=oracle.host_threads())
        small = min(range(len(host)), key=lambda i: algorithmic_bytes(host[i]))
        sec1, n1, _ = time_oracle([host[small]], min_s=5.0, threads=1)
        cpu = {"value": step_bytes / sec / 1e9, "unit": "GB/s", "cores": used, "kind": "oracle",
               "sample": f"{n} whole steps of the {args.workload} group (input set 0), "
                         f"fp64 oracle on {used} host threads, {sec * 1e3:.1f} ms/step",
               "cpu_model": oracle.cpu_model(),
               "single_thread": {"value": algorithmic_bytes(host[small]) / sec1 / 1e9,
                                 "unit": "GB/s", "ms_per_call": sec1 * 1e3, "calls": n1,
                                 "sample": f"the {names[small]} call, whole"}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": bench_config(args),
            "detail": {
                "us_per_step": ms_step * 1e3,
                "region_us_per_step": [round(r / args.steps * 1e3, 3) for r in region_ms],
                "gpu_launches_per_step": launches_per_step,
                "per_call_us": {n: round(u, 3) for n, u in zip(names, call_us)},
                "per_call_us_hot": {n: round(statistics.median(v) * 1e3, 3)
                                    for n, v in zip(names, per_call_hot)},
                "per_call_rate": per_call_rates,
                "algorithmic_bytes_per_step": step_bytes,
                "partition_tokens": {n: ("balanced" if p == pa.PARTITION_BALANCED else p if p else "auto")
                                     for n, p in zip(names, pts)},
                "plan": plans,
                "l2": f"rotating {nsets} input sets of {set_bytes / 1e6:.1f} MB "
                      f"({nsets * set_bytes / 1e6:.0f} MB > 3x L2 {l2 / 1e6:.0f} MB)",
                "launch": (f"CUDA graph of {nsets} steps (one per input set) per replay, "
                           "programmatic dependent launch between all calls"
                           if loop_graph is not None else
                           "CUDA graph replay per step" if graphs else "eager"),
                "append": ("each call appends the new token first (pa_append_kv); bytes "
                           "counted are the decode's only") if args.with_append else None,
                "parallelism": f"replicas x{world}",
                "parity_max_abs_err": max_err,
            },
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps * len(region_ms),
            "roofline": ({"bound": "tensor", "achieved": dom_tflops, "peak": tpeak,
                          "unit": "TFLOP/s", "frac": dom_tflops / tpeak, "peak_kind": tpeak_kind,
                          "flops_per_launch": dom_flops}
                         if tensor_bound else
                         {"bound": "hbm", "achieved": dom_gbs, "peak": peak, "unit": "GB/s",
                          "frac": dom_gbs / peak, "peak_kind": peak_kind,
                          "step_frac": value / world / peak,
                          "frac_of_nominal": dom_gbs / NOMINAL_HBM_GBS}) | {
                "kernel": f"decode call on {dom_name} ({plans[dom_name]['kernel']} kernel, "
                          f"{plans[dom_name]['partitions']} partition(s), reduce: "
                          f"{plans[dom_name]['reduce']})",
                "bytes_per_launch": dom_bytes,
                "traffic": dominant_traffic(plans[dom_name], dom_name)},
            "cpu_baseline": cpu,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
