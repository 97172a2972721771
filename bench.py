#!/usr/bin/env python3
"""Dispatch + combine throughput on one GB300 (tokens/s and achieved HBM GB/s).

One step = one pass of the whole hot path over one batch: the layout (counts,
prefix sums, positions), the permute into the fixed-stride receive buffer and
the score-weighted combine back to token order. The expert between dispatch
and combine is the identity (y = recv_x) and is not timed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload deepseek|mixtral|prefill32k|ragged|tiny]

Prints ONE JSON line (rank 0). Under torchrun (N > 1) each rank runs an
independent replica on its own GPU (the path has no exchange step: logical
ranks are partitions of one GPU's buffer), the timed region is bracketed by a
barrier and synchronisation, and the slowest rank's time is used.

--impl reference times the CPU oracle (single-threaded C, the correctness
reference) on one host core, on the same step: its dispatch and combine of the
same call(s) with the same inputs (about 2 s per DeepSeek-shaped step; 5 steps
by default). The GPU arm's `cpu_baseline` is the median of 3 such runs.

Other modes: --mode ceilings (the HBM ceiling of each access pattern the step
uses), --mode dedup / backward, --gemm DOUT (the expert grouped GEMM);
--graph [--fresh-routing] replays each step from a CUDA graph (with a fresh
routing copied into the captured inputs before every replay).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "dispatch+combine tokens/s & achieved HBM GB/s vs GB300 peak (bf16, 1 GPU)"
FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.txt")
KERNEL_SOURCES = [os.path.join(ROOT, "combine_topk_ids_expert_gb300", "csrc", f)
                  for f in ("layout.cu", "permute.cu", "combine.cu", "ep_kernels.cuh",
                            "ep_device.cuh")]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 2000 on the GPU, 5 for the oracle arm)")
    ap.add_argument("--warmup", type=int, default=None,
                    help="untimed warm-up steps (default: 20 on the GPU, 1 for the oracle arm)")
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default="deepseek", choices=sorted(W.WORKLOADS))
    ap.add_argument("--permute", choices=["default", "vec", "bulk"], default="default")
    ap.add_argument("--num-sms", type=int, default=0)
    ap.add_argument("--tokens", type=int, default=0,
                    help="override T (and N) of the workload: smaller cases for profiling")
    ap.add_argument("--graph", action="store_true", help="replay each step from a CUDA graph")
    ap.add_argument("--fresh-routing", action="store_true",
                    help="with --graph: write a fresh routing (ids and scores) into the captured "
                         "input buffers before every replay, outside the timed events")
    ap.add_argument("--flush", choices=["read", "memset"], default="read",
                    help="L2 flush between timed steps: read: a read-only sweep over 4x L2 (every "
                         "dirty line is written back before the step starts); memset: a write of "
                         "2x L2 (leaves ~L2-size dirty lines that the step then writes back)")
    ap.add_argument("--gemm", type=int, default=0, metavar="DOUT",
                    help="instead: time the expert grouped GEMM (D -> DOUT) on the receive rows")
    ap.add_argument("--mode", choices=["step", "dedup", "backward", "ceilings"], default="step",
                    help="step: layout+dispatch+combine (the benchmark); dedup: the per-rank "
                         "dedupe dispatch alone; backward: combine and dispatch backward; "
                         "ceilings: the HBM ceiling of each access pattern the step uses")
    ap.add_argument("--seed", type=int, default=None,
                    help="routing and hidden-state seed (default: the workload's own)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph-leg", action="store_true",
                    help="skip the extra captured-graph timing of the same step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-repeats", type=int, default=3,
                    help="oracle runs of the benched step for the CPU baseline (median taken)")
    args = ap.parse_args()
    # The oracle takes about 2 s per DeepSeek-shaped step on one host core: its
    # defaults keep an unflagged run within a minute or so.
    ref = args.impl == "reference"
    if args.steps is None:
        args.steps = 5 if ref else 2000
    if args.warmup is None:
        args.warmup = 1 if ref else 20
    return args


# ---------------------------------------------------------------------------
# workload description and algorithmic bytes
# ---------------------------------------------------------------------------

def workload_desc(w: W.Workload, T: int, N: int) -> dict:
    return {
        "workload": (f"{w.name}: T={T} D={w.D} {w.dtype} E={w.E} K={w.K} R={w.R} "
                     f"num_tokens_per_rank={N} num_max_tokens_per_rank={w.N_max} "
                     f"ids={w.ids} scores={w.scores}"),
        "T": T, "D": w.D, "E": w.E, "K": w.K, "R": w.R, "num_tokens_per_rank": N,
        "num_max_tokens_per_rank": w.N_max,
    }


def step_config(args, w: W.Workload, inps: list[dict], N: int) -> dict:
    """The `config` both arms print: the workload of one benched step."""
    cfg = workload_desc(w, sum(c["T"] for c in inps), N)
    if len(inps) > 1:
        cfg["workload"] += f" ({len(inps)} calls per step: T = {[c['T'] for c in inps]})"
    if args.fresh_routing:
        cfg["workload"] += ", fresh routing per step"
    return cfg


def workload_tokens(args, w: W.Workload) -> tuple[int, int]:
    """(T, N) of the benched call: the workload's own, or --tokens for both."""
    if args.tokens > 0:
        return args.tokens, args.tokens
    if w.T is None:   # ragged: source rank 0, padded to the group max of the 8 counts
        counts = W.ragged_counts(w)
        return counts[0], max(counts)
    return w.T, w.N


def algorithmic_bytes(T: int, K: int, D: int, b: int, pairs: int) -> dict:
    """Bytes the method must move per call (pairs = routed (t, k) pairs)."""
    row = D * b
    layout = T * K * 4 + pairs * 4                # ids read once, pos written
    permute = T * row + pairs * row + pairs * (4 + 4) + pairs * (4 + 4)
    #          x read    rows written  pos+score read   recv_scores+recv_src written
    combine = pairs * row + T * row + T * K * (4 + 4)
    #          rows read    out written  pos+score read
    return {"layout": layout, "permute": permute, "combine": combine,
            "step": layout + permute + combine}


def quantile(xs, q: float) -> float:
    """q-quantile of xs by linear interpolation between order statistics."""
    v = sorted(xs)
    if not v:
        return float("nan")
    f = q * (len(v) - 1)
    i = int(f)
    j = min(i + 1, len(v) - 1)
    return v[i] + (v[j] - v[i]) * (f - i)


def measured_peak_hbm() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; otherwise None."""
    try:
        lines = open(PROFILE_TRAFFIC).read().splitlines()
    except OSError:
        return None
    src = kernel_source_hash()
    for ln in lines:
        if ln.lstrip().startswith("#"):
            continue
        parts = ln.split()
        if len(parts) == 4 and parts[0] == kernel and parts[1] == workload and parts[3] == src:
            return float(parts[2])
    return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        for ln in open(self.path):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]),
                             "power": float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else 0.0,
                             "hw": parts[5], "hw_thermal": parts[6], "sw_thermal": parts[7],
                             "sw_power": parts[8]})
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        loaded = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"),
                              ("sw_power", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len(loaded)}


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline and --impl reference)
# ---------------------------------------------------------------------------

def oracle_step_seconds(w: W.Workload, inps: list[dict], N: int) -> float:
    """Seconds the oracle, as it stands (single-threaded C), takes for one
    benched step: its dispatch and combine of every call of the step, on the
    step's own inputs (the same T, N and routing the GPU arm times)."""
    import oracle
    o = oracle.get()
    t0 = time.perf_counter()
    for c in inps:
        d = o.dispatch(c["x"], c["scores"], c["ids"], N, w.E, w.R)
        o.combine(d["recv_x"], c["scores"], d["pos"], d["rank_prefix"], d["S"], w.R)
        del d
    return time.perf_counter() - t0


def oracle_baseline(w: W.Workload, inps: list[dict], N: int, repeats: int) -> dict:
    """The oracle on the benched step, `repeats` times; the median is reported."""
    secs = [oracle_step_seconds(w, inps, N) for _ in range(max(1, repeats))]
    T_step = sum(c["T"] for c in inps)
    med = statistics.median(secs)
    return {"value": T_step / med, "unit": "tokens/s", "cores": 1,
            "host_cores": os.cpu_count(), "kind": "oracle",
            "sample": (f"the whole benched step ({len(inps)} call(s), {T_step} tokens, the same "
                       f"inputs as the GPU arm), {len(secs)} runs on one host thread, median "
                       f"{med:.2f} s (runs: {', '.join(f'{x:.2f}' for x in secs)} s)")}


# ---------------------------------------------------------------------------
# distributed helpers (replicas)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(v: float, world: int) -> float:
    """The slowest rank's value (all ranks call it). NCCL reduces a CUDA
    tensor; other backends (gloo, used by the CPU tests) a host tensor."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(tokens_per_rank_step: int, steps: int, rank_ms: float, world: int) -> float:
    """Whole-job tokens/s of `world` independent replicas: all ranks' tokens
    over the slowest rank's time (weak scaling)."""
    slowest = max_over_ranks(rank_ms, world)
    return world * tokens_per_rank_step * steps / (slowest / 1e3)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def make_l2_flush(args, dev):
    """The L2 flush run before every timed step, outside its events. read: a
    read-only sweep over 4x L2 (a sum), after which L2 holds only clean lines,
    so the step pays for no earlier write-back; memset: a 2x L2 memset, which
    leaves about L2's size of dirty lines for the step to write back."""
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    if args.flush == "read":
        # fp32 so that the sum reads the buffer in place (an integer sum would
        # first write a widened copy)
        buf = torch.zeros(max(4 * l2, 512 << 20) // 4, dtype=torch.float32, device=dev)
        return lambda: buf.sum()
    buf = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    return lambda: buf.zero_()


def _routing_job(job):
    name, rank, T, seed, replay = job
    inp = W.make(name, rank=rank, T=T, seed=seed, replay=replay, with_x=False)
    return inp["ids"], inp["scores"]


def fresh_routings(args, w: W.Workload, Ts: list[int]) -> list:
    """Pinned host copies of a fresh routing (ids, scores) per call for up to
    100 replays (replay i of the workload's graph schedule), drawn in a pool
    of spawned processes."""
    import multiprocessing as mp

    import torch
    n = max(1, min(args.steps, 100))
    jobs = [(args.workload, c, T, args.seed, i) for i in range(n) for c, T in enumerate(Ts)]
    with mp.get_context("spawn").Pool(min(16, os.cpu_count() or 1)) as pool:
        flat = pool.map(_routing_job, jobs)
    out = []
    for i in range(n):
        calls = flat[i * len(Ts):(i + 1) * len(Ts)]
        out.append([(torch.from_numpy(a).pin_memory(), torch.from_numpy(b).pin_memory())
                    for a, b in calls])
    return out


def step_calls(args, w: W.Workload) -> tuple[list[dict], int]:
    """The dispatch+combine calls of one step and their shared N: one call, or
    one per source rank of the ragged workload (padded to the group max)."""
    if args.tokens > 0 or w.T is not None:
        T, N = workload_tokens(args, w)
        return [W.make(args.workload, rank=0, T=T, seed=args.seed)], N
    counts = W.ragged_counts(w)
    return [W.make(args.workload, rank=r, seed=args.seed) for r in range(w.ragged_ranks)], max(counts)


def run_gb300(args) -> dict | None:
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)          # before NCCL, so its communicator binds this GPU
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)

    import combine_topk_ids_expert_gb300 as ep
    from combine_topk_ids_expert_gb300.build import build as build_lib
    if rank == 0:
        build_lib()
    barrier(world)

    w = W.WORKLOADS[args.workload]
    inps, N = step_calls(args, w)
    Ts = [c["T"] for c in inps]
    T_step = sum(Ts)
    n_calls = len(inps)
    b = w.elem_bytes
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    raw = torch.int16 if tdt == torch.bfloat16 else tdt

    def host(a: np.ndarray):
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        return t.pin_memory()

    xh = [host(c["x"]) for c in inps]
    idh = [host(c["ids"]) for c in inps]
    sch = [host(c["scores"]) for c in inps]
    xs = [t.to(dev).view(tdt) if tdt == torch.bfloat16 else t.to(dev) for t in xh]
    idss = [t.to(dev) for t in idh]
    scs = [t.to(dev) for t in sch]
    outs = [torch.empty((T, w.D), dtype=tdt, device=dev) for T in Ts]
    impl = {"default": ep.EP_PERMUTE_DEFAULT, "vec": ep.EP_PERMUTE_VEC,
            "bulk": ep.EP_PERMUTE_BULK}[args.permute]
    n_max = args.tokens if args.tokens > 0 else w.N_max   # smaller workspace when profiling
    buf = ep.Buffer(n_max, w.D, w.E, w.R, w.K, dtype=tdt, num_sms=args.num_sms,
                    permute_impl=impl, device=dev)
    h = buf.handle
    out_code = ep.EP_BF16 if tdt == torch.bfloat16 else ep.EP_F32
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream

    # One untimed pass: routed pairs per call, launches per step, reference outputs.
    n_launch0 = buf.info()["kernel_launches"]
    pairs = []
    recv_x = None
    for i in range(n_calls):
        d = buf.dispatch(xs[i], scs[i], idss[i], N)
        recv_x = d.recv_x
        buf.combine(recv_x, scs[i], out=outs[i])
        pairs.append(int(d.layout.tokens_per_expert.sum().item()))
    per_step_launches = buf.info()["kernel_launches"] - n_launch0
    torch.cuda.synchronize(dev)
    assert buf.device_error() == 0
    ref_outs = [o.clone() for o in outs]

    l2_flush = make_l2_flush(args, dev)
    routes = fresh_routings(args, w, Ts) if args.fresh_routing else None

    def step_kernels(stream_ptr):
        for i in range(n_calls):
            ep.ep_dispatch(h, xs[i], scs[i], idss[i], Ts[i], N, stream_ptr)
            ep.ep_combine(h, recv_x, scs[i], Ts[i], outs[i], out_code, stream_ptr)

    def capture():
        step_kernels(sptr)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(dev)
        s.wait_stream(stream)
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                step_kernels(s.cuda_stream)
        stream.wait_stream(s)
        torch.cuda.synchronize(dev)
        return g

    graph = capture() if args.graph else None

    for _ in range(args.warmup):
        l2_flush()
        if graph is not None:
            graph.replay()
        else:
            step_kernels(sptr)
    torch.cuda.synchronize(dev)

    K = args.steps
    # events per step: start, then after each call's dispatch and combine
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(1 + 2 * n_calls)]
          for _ in range(K)]
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    launches0 = buf.info()["kernel_launches"]
    barrier(world)
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for it in range(K):
        if routes is not None:              # fresh routing into the captured inputs
            r = routes[it % len(routes)]
            for i in range(n_calls):
                idss[i].copy_(r[i][0], non_blocking=True)
                scs[i].copy_(r[i][1], non_blocking=True)
        l2_flush()                          # L2 flush, outside the events
        e = ev[it]
        e[0].record(stream)
        if graph is not None:
            graph.replay()
            e[-1].record(stream)
        else:
            for i in range(n_calls):
                ep.ep_dispatch(h, xs[i], scs[i], idss[i], Ts[i], N, sptr)
                e[1 + 2 * i].record(stream)
                ep.ep_combine(h, recv_x, scs[i], Ts[i], outs[i], out_code, sptr)
                e[2 + 2 * i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    wall = time.perf_counter() - wall0
    clk = clocks.stop() if rank == 0 else None
    launches = buf.info()["kernel_launches"] - launches0
    if graph is not None:
        launches = K * per_step_launches
    assert buf.device_error() == 0
    if routes is None:
        for o, r in zip(outs, ref_outs):
            assert torch.equal(o.view(raw), r.view(raw)), "timed steps changed the output"
    else:
        # the last replay's outputs against an eager step on the same routing
        last = [o.clone() for o in outs]
        step_kernels(sptr)
        torch.cuda.synchronize(dev)
        assert buf.device_error() == 0
        for o, r in zip(outs, last):
            assert torch.equal(o.view(raw), r.view(raw)), "replay differs from an eager step"
        for i in range(n_calls):            # back to the first routing for the legs below
            idss[i].copy_(idh[i])
            scs[i].copy_(sch[i])
        step_kernels(sptr)
        torch.cuda.synchronize(dev)

    step_ms = [e[0].elapsed_time(e[-1]) for e in ev]
    total_ms = sum(step_ms)
    total_ms_max = max_over_ranks(total_ms, world)
    ms_per_step = total_ms_max / K
    tok_s = replica_throughput(T_step, K, total_ms, world)
    nb = [algorithmic_bytes(T, w.K, w.D, b, p) for T, p in zip(Ts, pairs)]
    nbytes = {k: sum(x[k] for x in nb) for k in nb[0]}
    peak, peak_src = measured_peak_hbm()
    res = {"ms_per_step": ms_per_step, "value": tok_s,
           "step_ms_median": statistics.median(step_ms),
           "step_ms_p10": quantile(step_ms, 0.10), "step_ms_p90": quantile(step_ms, 0.90),
           "hbm_gbs_step": nbytes["step"] / (ms_per_step / 1e3) / 1e9,
           "wall_s": wall, "launches": launches, "clocks": clk, "T_step": T_step,
           "calls_per_step": n_calls}
    if graph is None:
        dis, com = [], []
        for e in ev:
            prev = e[0]
            d_ms = c_ms = 0.0
            for i in range(n_calls):
                d_ms += prev.elapsed_time(e[1 + 2 * i])
                c_ms += e[1 + 2 * i].elapsed_time(e[2 + 2 * i])
                prev = e[2 + 2 * i]
            dis.append(d_ms)
            com.append(c_ms)
        kern = {}
        for name, arr, nbk in (("dispatch", dis, nbytes["layout"] + nbytes["permute"]),
                               ("combine", com, nbytes["combine"])):
            avg = sum(arr) / len(arr)
            kern[name] = {"avg_us": avg * 1e3, "median_us": statistics.median(arr) * 1e3,
                          "algorithmic_bytes": nbk, "achieved_gbs": nbk / (avg / 1e3) / 1e9}
        for k in kern.values():   # each kernel against the same measured peak
            k["frac_of_peak"] = round(k["achieved_gbs"] / peak, 4)
        dom = "dispatch" if kern["dispatch"]["avg_us"] >= kern["combine"]["avg_us"] else "combine"
        ach = kern[dom]["achieved_gbs"]
        impl_name = {1: "vec", 2: "bulk"}[buf.info()["permute_impl"]]
        kname = {"dispatch": f"dispatch_{impl_name}", "combine": "combine"}[dom]
        res["kernels"] = kern
        res["roofline"] = {"bound": "hbm", "kernel": kname, "achieved": round(ach, 1),
                           "peak": peak, "unit": "GB/s", "frac": round(ach / peak, 4),
                           "peak_source": peak_src,
                           "traffic": profiled_traffic(kname, args.workload),
                           "algorithmic_bytes_per_launch": kern[dom]["algorithmic_bytes"]}
    if routes is not None:
        res["fresh_routing"] = {"routings": len(routes), "replays": K,
                                "copied_per_replay_bytes": sum(8 * T * w.K for T in Ts)}
    res["bytes"] = nbytes
    res["pairs"] = sum(pairs)
    res["info"] = buf.info()
    props = torch.cuda.get_device_properties(dev)
    res["device"] = {"name": props.name, "sms": props.multi_processor_count,
                     "l2_bytes": props.L2_cache_size, "dispatch_ctas": buf.info()["permute_grid"]}

    # The same step replayed from a captured CUDA graph (events around each
    # replay, L2 flushed before each), reported beside the eager timing.
    if graph is None and not args.no_graph_leg:
        g = capture()
        for _ in range(3):
            l2_flush()
            g.replay()
        Kg = max(3, min(K, 300))
        evg = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(Kg)]
        barrier(world)
        torch.cuda.synchronize(dev)
        for a, c in evg:
            l2_flush()
            a.record(stream)
            g.replay()
            c.record(stream)
        torch.cuda.synchronize(dev)
        assert buf.device_error() == 0
        for o, r in zip(outs, ref_outs):
            assert torch.equal(o.view(raw), r.view(raw)), "graph replays changed the output"
        gms = [a.elapsed_time(c) for a, c in evg]
        g_ms = max_over_ranks(sum(gms), world) / Kg
        res["graph_replay"] = {"steps": Kg, "ms_per_step": g_ms,
                               "value": replica_throughput(T_step, Kg, sum(gms), world),
                               "unit": "tokens/s", "median_ms": statistics.median(gms),
                               "p10_ms": quantile(gms, 0.10), "p90_ms": quantile(gms, 0.90)}
        del g

    # End to end through the public API with host buffers: every call copies its
    # inputs from pinned host memory and its output back, inside the timed region.
    # Calls are pipelined on three streams (H2D of call j+1, compute of call j,
    # D2H of call j-1) over double-buffered device inputs and outputs.
    if not args.no_e2e:
        Tm = max(Ts)
        dx = [torch.empty((Tm, w.D), dtype=tdt, device=dev) for _ in range(2)]
        did = [torch.empty((Tm, w.K), dtype=torch.int32, device=dev) for _ in range(2)]
        dsc = [torch.empty((Tm, w.K), dtype=torch.float32, device=dev) for _ in range(2)]
        dout = [torch.empty((Tm, w.D), dtype=tdt, device=dev) for _ in range(2)]
        hout = [torch.empty((Tm, w.D), dtype=raw).pin_memory() for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        s_cmp = stream

        def run_pipeline(n_units):
            ev_in = [torch.cuda.Event() for _ in range(n_units)]
            ev_cmp = [torch.cuda.Event() for _ in range(n_units)]
            ev_out = [torch.cuda.Event() for _ in range(n_units)]
            for j in range(n_units):
                i, bs = j % n_calls, j % 2
                T = Ts[i]
                with torch.cuda.stream(s_in):
                    if j >= 2:
                        s_in.wait_event(ev_cmp[j - 2])
                    dx[bs][:T].view(raw).copy_(xh[i], non_blocking=True)
                    did[bs][:T].copy_(idh[i], non_blocking=True)
                    dsc[bs][:T].copy_(sch[i], non_blocking=True)
                    ev_in[j].record(s_in)
                s_cmp.wait_event(ev_in[j])
                if j >= 2:
                    s_cmp.wait_event(ev_out[j - 2])
                ep.ep_dispatch(h, dx[bs][:T], dsc[bs][:T], did[bs][:T], T, N, s_cmp.cuda_stream)
                ep.ep_combine(h, recv_x, dsc[bs][:T], T, dout[bs][:T], out_code,
                              s_cmp.cuda_stream)
                ev_cmp[j].record(s_cmp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_cmp[j])
                    hout[bs][:T].copy_(dout[bs][:T].view(raw), non_blocking=True)
                    ev_out[j].record(s_out)
            return ev_out[n_units - 1]

        run_pipeline(2 * n_calls + 2)        # warm-up
        torch.cuda.synchronize(dev)
        Ke = max(3, min(K, 300))
        n_units = Ke * n_calls
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        s_cmp.wait_event(e0)
        s_out.wait_event(e0)
        last = run_pipeline(n_units)
        s_out.wait_event(last)
        e1.record(s_out)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
        jl = n_units - 1
        il, bl = jl % n_calls, jl % 2
        assert torch.equal(hout[bl][:Ts[il]], ref_outs[il].view(raw).cpu()), \
            "e2e output differs from the device path"
        h2d = sum(x.numel() * x.element_size() + a.numel() * 4 + c.numel() * 4
                  for x, a, c in zip(xh, idh, sch))
        d2h = sum(T * w.D * b for T in Ts)
        res["e2e"] = {"value": replica_throughput(T_step, Ke, e0.elapsed_time(e1), world),
                      "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "steps": Ke, "ms_per_step": e2e_ms / Ke,
                      "pipeline": "H2D(j+1) | dispatch+combine(j) | D2H(j-1), 3 streams"}
    buf.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return res if rank == 0 else None


def measured_peak_bf16(sustained: bool) -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    try:
        with open(p) as f:
            return float(json.load(f)[key]), f"measured (MEASURED_PEAKS.json {key})"
    except Exception:
        return (1700.0 if sustained else 1900.0), "fallback"


def run_gemm(args) -> None:
    """Times the expert consumer: y = x W_e^T over every expert's receive rows
    (bf16, fp32 accumulation on the tensor cores), after one dispatch."""
    import torch

    import combine_topk_ids_expert_gb300 as ep
    from combine_topk_ids_expert_gb300.build import build as build_lib
    build_lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = W.WORKLOADS[args.workload]
    inps, N = step_calls(args, w)
    inp = inps[0]
    T = inp["T"]
    x = torch.from_numpy(inp["x"].view(np.int16)).to(dev).view(torch.bfloat16)
    ids = torch.from_numpy(inp["ids"]).to(dev)
    sc = torch.from_numpy(inp["scores"]).to(dev)
    n_max = args.tokens if args.tokens > 0 else w.N_max
    buf = ep.Buffer(n_max, w.D, w.E, w.R, w.K, dtype=torch.bfloat16, device=dev)
    d = buf.dispatch(x, sc, ids, N)
    torch.cuda.synchronize(dev)
    pairs = int(d.layout.tokens_per_expert.sum().item())
    dout = args.gemm
    g = torch.Generator(device=dev).manual_seed(w.seed)
    wts = (torch.randn((w.E, dout, w.D), generator=g, device=dev, dtype=torch.float32) * 0.03
           ).to(torch.bfloat16)
    y = torch.empty(d.recv_x.shape[:-1] + (dout,), dtype=torch.bfloat16, device=dev)
    for _ in range(args.warmup):
        buf.expert_gemm(d.recv_x, wts, y_recv=y)
    torch.cuda.synchronize(dev)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    launches0 = buf.info()["kernel_launches"]
    clocks = ClockSampler(0)
    clocks.start()
    for e0, e1 in ev:
        e0.record()
        buf.expert_gemm(d.recv_x, wts, y_recv=y)
        e1.record()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    assert buf.device_error() == 0
    ms = [a.elapsed_time(b) for a, b in ev]
    avg = sum(ms) / K
    flops = 2.0 * pairs * w.D * dout
    tf = flops / (avg / 1e3) / 1e12
    peak, src = measured_peak_bf16(sustained=False)
    # Algorithmic HBM bytes: the weights of every expert that has rows (read at
    # least once), the routed rows in and their outputs out.
    used = int((d.layout.tokens_per_expert > 0).sum().item())
    nbytes = 2 * (used * dout * w.D + pairs * w.D + pairs * dout)
    bw_peak, bw_src = measured_peak_hbm()
    floor_tensor = flops / (peak * 1e12) * 1e3
    floor_hbm = nbytes / (bw_peak * 1e9) * 1e3
    if floor_tensor >= floor_hbm:
        roof = {"bound": "tensor", "achieved": round(tf, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(tf / peak, 4), "peak_source": src}
    else:
        gbs = nbytes / (avg / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": bw_peak, "unit": "GB/s",
                "frac": round(gbs / bw_peak, 4), "peak_source": bw_src,
                "algorithmic_bytes_per_launch": nbytes}
    roof["floors_ms"] = {"tensor": round(floor_tensor, 4), "hbm": round(floor_hbm, 4)}
    info = buf.info()
    line = {"metric": "expert grouped GEMM TFLOP/s (bf16 in, fp32 accumulate, tcgen05)",
            "value": tf, "unit": "TFLOP/s", "n_gpus": 1, "steps": K, "warmup": args.warmup,
            "ms_per_step": avg, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{w.name} receive rows ({pairs} routed pairs) x "
                                   f"W[{w.E}, {dout}, {w.D}]",
                       "rows": pairs, "din": w.D, "dout": dout, "experts": w.E,
                       "l2": "inputs larger than L2 (weights + rows), no flush"},
            "roofline": roof,
            "kernel": {1: "single-CTA 128-row tiles", 2: "two-SM 256-row tiles"}.get(
                info["gemm_kernel"]),
            "grid": info["gemm_grid"],
            "gpu_launches": info["kernel_launches"] - launches0, "clocks": clk}
    buf.close()
    print(json.dumps(line))


def run_aux(args) -> None:
    """Times a NEXT-row operation (dedupe dispatch, or the backward pass) on the
    workload's first call, L2 flushed between steps, and prints one JSON line."""
    import torch

    import combine_topk_ids_expert_gb300 as ep
    from combine_topk_ids_expert_gb300.build import build as build_lib
    build_lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = W.WORKLOADS[args.workload]
    inps, N = step_calls(args, w)
    inp = inps[0]
    T, D, K, b = inp["T"], w.D, w.K, w.elem_bytes
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    x = torch.from_numpy(inp["x"].view(np.int16) if w.dtype == "bf16" else inp["x"]).to(dev)
    x = x.view(tdt)
    ids = torch.from_numpy(inp["ids"]).to(dev)
    sc = torch.from_numpy(inp["scores"]).to(dev)
    n_max = args.tokens if args.tokens > 0 else w.N_max
    buf = ep.Buffer(n_max, D, w.E, w.R, K, dtype=tdt, device=dev)
    h = buf.handle
    row = D * b
    if args.mode == "dedup":
        d = buf.dispatch_dedup(x, sc, ids, N)
        torch.cuda.synchronize(dev)
        rows = int(d.layout.tokens_in_rank.sum().item())
        nbytes = T * row + rows * row + T * K * 8 + rows * (4 + 8 * K) + T * w.R * 4
        metric = "per-rank dedupe dispatch tokens/s (layout + one row per distinct (token, rank))"

        def op():
            ep.ep_dispatch_dedup(h, x, sc, ids, T, N)
        extra = {"dedupe_rows": rows, "per_expert_rows": T * K}
    else:
        d = buf.dispatch(x, sc, ids, N)
        g = torch.randn((T, D), device=dev, dtype=torch.float32).to(tdt)
        gy = torch.empty_like(d.recv_x)
        gx = torch.empty((T, D), dtype=tdt, device=dev)
        gs = torch.empty((T, K), dtype=torch.float32, device=dev)
        torch.cuda.synchronize(dev)
        pairs = int(d.layout.tokens_per_expert.sum().item())
        nbytes = (T * row + 2 * pairs * row + T * K * 12) + (pairs * row + T * row + T * K * 4)
        metric = "combine + dispatch backward tokens/s (grad_y, grad_scores, grad_x)"
        code = ep.EP_BF16 if tdt == torch.bfloat16 else ep.EP_F32

        def op():
            ep.ep_combine_backward(h, g, d.recv_x, sc, T, gy, gs)
            ep.ep_dispatch_backward(h, gy, None, T, gx, code)
        extra = {"pairs": pairs}
    l2_flush = make_l2_flush(args, dev)
    for _ in range(args.warmup):
        l2_flush()
        op()
    torch.cuda.synchronize(dev)
    Ks = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(Ks)]
    clocks = ClockSampler(0)
    clocks.start()
    launches0 = buf.info()["kernel_launches"]
    for e0, e1 in ev:
        l2_flush()
        e0.record()
        op()
        e1.record()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    assert buf.device_error() == 0
    avg = sum(a.elapsed_time(c) for a, c in ev) / Ks
    peak, src = measured_peak_hbm()
    gbs = nbytes / (avg / 1e3) / 1e9
    line = {"metric": metric, "value": T / (avg / 1e3), "unit": "tokens/s", "n_gpus": 1,
            "steps": Ks, "warmup": args.warmup, "ms_per_step": avg, "higher_is_better": True,
            "dtype": w.dtype, "data": "synthetic", "config": workload_desc(w, T, N),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "peak_source": src,
                         "algorithmic_bytes_per_launch": nbytes},
            "gpu_launches": buf.info()["kernel_launches"] - launches0, "clocks": clk}
    line.update(extra)
    buf.close()
    print(json.dumps(line))


def run_ceilings(args) -> None:
    """The HBM ceiling of each access pattern the step uses, on the workload's
    row size: ep_pattern_probe moves the rows of one call (T tokens, K = fan)
    in each shape alone in a kernel, L2 flushed before every launch, CUDA
    events around it; bytes are the rows read plus the rows written."""
    import torch

    import combine_topk_ids_expert_gb300 as ep
    from combine_topk_ids_expert_gb300.build import build as build_lib
    build_lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = W.WORKLOADS[args.workload]
    T, _ = workload_tokens(args, w)
    row, fan = w.D * w.elem_bytes, w.K
    src = torch.zeros(T * fan * row // 4, dtype=torch.int32, device=dev)
    dst = torch.zeros(T * fan * row // 4, dtype=torch.int32, device=dev)
    shapes = {   # name: (pattern, rows, bytes moved)
        "read": (ep._abi.EP_PATTERN_READ, T * fan, T * fan * (row + 16)),
        "write": (ep._abi.EP_PATTERN_WRITE, T * fan, T * fan * row),
        "copy": (ep._abi.EP_PATTERN_COPY, T * fan, 2 * T * fan * row),
        f"fanout_1to{fan}": (ep._abi.EP_PATTERN_FANOUT, T, (1 + fan) * T * row),
        f"gather_{fan}to1": (ep._abi.EP_PATTERN_GATHER, T, (1 + fan) * T * row),
    }
    l2_flush = make_l2_flush(args, dev)
    peak, src_name = measured_peak_hbm()
    steps = max(3, min(args.steps, 200))
    clocks = ClockSampler(0)
    clocks.start()
    out = {}
    for name, (pat, rows, nbytes) in shapes.items():
        def op():
            ep.ep_pattern_probe(pat, src, dst, rows, row, fan)
        for _ in range(max(3, args.warmup)):
            l2_flush()
            op()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for a, b in ev:
            l2_flush()
            a.record()
            op()
            b.record()
        torch.cuda.synchronize(dev)
        us = [a.elapsed_time(b) * 1e3 for a, b in ev]
        avg = sum(us) / len(us)
        gbs = nbytes / (avg / 1e6) / 1e9
        out[name] = {"bytes": nbytes, "avg_us": round(avg, 2),
                     "median_us": round(statistics.median(us), 2), "gbs": round(gbs, 1),
                     "frac_of_peak": round(gbs / peak, 4)}
    clk = clocks.stop()
    line = {"metric": "HBM ceiling of each access pattern of the step (GB/s)", "unit": "GB/s",
            "n_gpus": 1, "steps": steps, "warmup": args.warmup, "higher_is_better": True,
            "data": "synthetic", "row_bytes": row, "fan": fan, "rows": T,
            "workload": w.name, "patterns": out, "peak": peak, "peak_source": src_name,
            "l2": f"flushed before every launch ({args.flush})", "clocks": clk}
    print(json.dumps(line))


def main():
    args = parse_args()
    if args.mode == "ceilings":
        run_ceilings(args)
        return
    if args.gemm and args.impl == "gb300":
        run_gemm(args)
        return
    if args.mode != "step" and args.impl == "gb300":
        run_aux(args)
        return
    world, rank, _ = dist_env()
    w = W.WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return
        inps, N = step_calls(args, w)
        T_step = sum(c["T"] for c in inps)
        for _ in range(args.warmup):
            oracle_step_seconds(w, inps, N)
        secs = [oracle_step_seconds(w, inps, N) for _ in range(args.steps)]
        v = T_step * len(secs) / sum(secs)
        sample = (f"each step the oracle's dispatch+combine of the whole benched step "
                  f"({len(inps)} call(s), {T_step} tokens: the GPU arm's workload and inputs), "
                  f"one host thread")
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": sum(secs) / len(secs) * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
                "config": step_config(args, w, inps, N),
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1,
                                 "host_cores": os.cpu_count(), "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                "gpu_launches": 0}
        print(json.dumps(line))
        return

    res = run_gb300(args)
    if rank != 0:
        return
    inps, N = step_calls(args, w)
    cfg = step_config(args, w, inps, N)
    setup = {"calls_per_step": res.get("calls_per_step", 1),
             "l2": {"read": "flushed before every timed step by a read-only sweep over 4x L2 "
                            "(every dirty line written back before the step starts)",
                    "memset": "flushed before every timed step by a memset of 2x L2 (its dirty "
                              "lines are written back inside the step)"}[args.flush],
             "expert": "identity (y = recv_x), not timed",
             "permute_impl": {1: "vec", 2: "bulk"}.get(res["info"]["permute_impl"]),
             "timing": ("CUDA graph replay" if args.graph else "eager, per-kernel CUDA events")
             + (", fresh routing copied in before every replay (outside the events)"
                if args.fresh_routing else ""),
             "parallelism": f"replicas x{args.gpus}",
             "device": res.get("device")}
    line = {"metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic", "config": cfg, "setup": setup,
            "achieved_hbm_gbs": round(res["hbm_gbs_step"], 1),
            "hbm_frac_step": round(res["hbm_gbs_step"] / measured_peak_hbm()[0], 4),
            "step_ms": {"median": res["step_ms_median"], "p10": res["step_ms_p10"],
                        "p90": res["step_ms_p90"]}}
    for key in ("roofline", "kernels", "e2e", "graph_replay", "fresh_routing"):
        if key in res:
            line[key] = res[key]
    line["gpu_launches"] = res["launches"]
    line["clocks"] = res["clocks"]
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(w, inps, N, args.cpu_repeats)
    print(json.dumps(line))


if __name__ == "__main__":
    main()
