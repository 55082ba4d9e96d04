#!/usr/bin/env python3
"""Benchmark of the tree-verify step on GB300.

Default workload: the 8B-class dense decoder (36 layers, hidden 4096, SwiGLU
12288, 32/8 heads, vocab 151936, every linear weight W12-packed), one request,
a draft tree of M = 16 nodes (depth <= 8, copy-rule tokens with p = 0.7),
2048 cached positions.  A step is one sd_verify_step: tree bookkeeping,
forward over all nodes, fp32 argmax, greedy acceptance and commit.  Each
timed step starts from the same cache state (ctx_len is reset; the prefix is
never written by a step), so all steps do identical work.  The weights
(11.4 GB packed) are far larger than L2, so no flush is needed.

Prints one JSON line (rank 0).  --impl reference times the oracle (the plain
CPU implementation the tests compare against) on this machine's host cores
on a bounded sample of the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_BW_GBS = 8000.0       # the metric's "fraction of 8 TB/s"
# DRAM bytes (read + write) per launch of the dominant kernel, from ncu
# captures of the current kernels (profiles/), keyed by (model, rows, kernel
# group): the gate/up GEMM of the 8B-class model at 16 rows (warp-level
# kernel: 151.70 MB read + 4.04 MB written, captured on the same shape through
# sd_w12_linear, whose plain store writes 0.4 MB more than the SiLU epilogue)
# and at 256 rows (tcgen05 kernel: 165.84 + 18.66 MB); none for the streamed
# launch
STREAM_TRAFFIC = {("8b", 16, "gemm_gate_up"): 155.74e6, ("8b", 256, "gemm_gate_up"): 184.51e6}


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return PEAKS_FALLBACK, "fallback"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="sdv", choices=["sdv", "reference"])
    ap.add_argument("--workload", default="8b_m16")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--timeline", action="store_true", help="print the per-kernel breakdown to stderr")
    ap.add_argument("--no-strip", action="store_true",
                    help="skinny O / down launches on the warp-level split-K kernel instead of the strip-parallel one")
    ap.add_argument("--deferred-finish", action="store_true",
                    help="split row blocks finished by a separate kernel after the GEMM")
    ap.add_argument("--cluster-finish", action="store_true",
                    help="finish split row blocks through thread-block clusters instead of workspace partials")
    ap.add_argument("--fused", action="store_true",
                    help="skinny steps: the linears between two attention kernels as one launch")
    ap.add_argument("--nvtx", action="store_true", help="wrap the timed steps in the NVTX range 'sdv_step'")
    ap.add_argument("--probe", default=None, metavar="N,K,M",
                    help="time the fused W12 linear alone on an N x K tensor with M rows")
    ap.add_argument("--probe-weights", default="normal", choices=["normal", "scaled"],
                    help="--probe: i.i.d. N(0, 0.02) weights, or rows of different norms (wl.row_scaled)")
    ap.add_argument("--probe-format", default="tensor", choices=["tensor", "channel"],
                    help="--probe: per-tensor exponent table or per-channel bases (pack_channel)")
    ap.add_argument("--probe-kernel", default="gemm", choices=["gemm", "stream", "view8", "stream_view8"],
                    help="--probe: sd_w12_linear (warp-level / tcgen05), sd_w12_linear_stream, "
                         "sd_w12_linear_view8 (the nested 8-bit plane, 1 byte per weight), or the streaming "
                         "kernel over the plane")
    ap.add_argument("--gdn", default=None, metavar="R,nh,M",
                    help="time the gated-delta-rule tree kernel alone: R requests of M-node trees, nh heads")
    ap.add_argument("--tc-min-rows", type=int, default=0,
                    help="rows per launch from which GEMMs run on the tcgen05 kernel (0: the library default)")
    ap.add_argument("--select", default=None, metavar="R,n,budget,cap",
                    help="time the best-first node selection alone on R requests of n candidates")
    ap.add_argument("--attn-splits", type=int, default=0,
                    help="prefix key splits of the step's attention per kv head and row chunk (0: automatic)")
    return ap.parse_args()


def oracle_select_rate(c, budget: int, cap: int, reps: int = 3) -> dict:
    """The oracle's best-first selection on the same candidates, timed on
    the host (one Python thread): candidates per second, median of reps."""
    import oracle
    t = []
    for _ in range(max(1, reps)):
        t0 = time.perf_counter()
        oracle.best_first_select(c.parents, c.logprob, c.cu, budget, cap)
        t.append(time.perf_counter() - t0)
    s = statistics.median(t)
    n = int(c.cu[-1])
    return {"value": n / s, "unit": "candidates/s", "cores": 1, "kind": "oracle",
            "sample": f"the whole call ({n} candidates), median of {len(t)}", "s_per_call": s}


def select_arm(args):
    """Best-first node selection under a shared node budget alone
    (sd_best_first_select) on seeded synthetic candidate trees: per-call time
    with CUDA events over graph replays; candidates per second."""
    import numpy as np
    import torch
    from synthetic import workloads as wl
    from speculative_decoding_tree_bit_gb300 import _build
    from speculative_decoding_tree_bit_gb300 import model as Mdl
    _build.build()
    R, n, budget, cap = (int(v) for v in args.select.split(","))
    c = wl.candidates(args.seed, R, n, 8, 32000)
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a.astype(dt))).cuda()
    par, lp, cu, tok = dev(c.parents, np.int32), dev(c.logprob, np.float32), dev(c.cu, np.int32), dev(c.tokens, np.int32)
    sel = Mdl.Selector(int(c.cu[-1]), R)
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            sel(par, lp, cu, budget, cap, tokens=tok, stream=stream, clear_status=False)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(args.steps):
                sel(par, lp, cu, budget, cap, tokens=tok, stream=stream, clear_status=False)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    N = int(c.cu[-1])
    kept = int(sel.out_cu[R].item())
    status = int(sel.status.item())
    # algorithmic bytes: candidates read (parent, log-prob, token), kept nodes written (src, parent, token, score)
    nbytes = N * 12 + (R + 1) * 4 + kept * 16
    try:
        cpu = oracle_select_rate(c, budget, cap)
    except Exception as ex:  # the oracle leg must not cost the GPU figure
        cpu = {"error": str(ex)[:200]}
    return {"probe": "sd_best_first_select", "R": R, "n": n, "candidates": N, "budget": budget, "cap": cap,
            "kept": kept, "status": status, "us_per_call": us, "candidates_per_s": N / (us * 1e-6),
            "bound": "latency", "bytes": nbytes, "GBps": nbytes / (us * 1e-6) / 1e9,
            "launches_per_call": 2, "memsets_per_call": 1, "cpu_baseline": cpu}


def probe_arm(args):
    """The fused W12 GEMM alone (sd_w12_linear) on a seeded N x K tensor:
    per-launch time with CUDA events, algorithmic GB/s."""
    import numpy as np
    import torch
    import synthetic
    from speculative_decoding_tree_bit_gb300 import _build
    from speculative_decoding_tree_bit_gb300 import model as Mdl
    _build.build()
    tc_rows = Mdl.set_tc_min_rows(args.tc_min_rows)
    Mdl.set_cluster_finish(args.cluster_finish)
    Mdl.set_deferred_finish(args.deferred_finish)
    Mdl.set_strip(not args.no_strip)
    N, K, M = (int(v) for v in args.probe.split(","))
    from synthetic import workloads as wl
    w = (wl.row_scaled(args.seed + 4242, N, K) if args.probe_weights == "scaled" else
         synthetic.normal_bf16(synthetic.key(args.seed, 4242), N * K, 0.02).reshape(N, K))
    view8 = args.probe_kernel in ("view8", "stream_view8")
    p = (Mdl.pack_channel(Mdl.to_device_u16(w)) if args.probe_format == "channel" else
         Mdl.pack(Mdl.to_device_u16(w), view8=view8))
    del w
    wbytes = (p.plane8.numel() * p.plane8.element_size() + p.nbytes() - p.words.numel() * 4) if view8 else p.nbytes()
    # copies of the packed tensor that together exceed L2, cycled by the
    # launches, so that every launch streams its weights from HBM
    n_copies = max(1, -(-256 * 2 ** 20 // wbytes))
    packs = [p] + [p.copy() for _ in range(n_copies - 1)]
    x = Mdl.to_device_u16(synthetic.normal_bf16(synthetic.key(args.seed, 4243), M * K, 1.0).reshape(M, K))
    import speculative_decoding_tree_bit_gb300 as sdv
    kind = args.probe_kernel
    need = {"gemm": sdv.lib().sd_w12_linear_workspace, "view8": sdv.lib().sd_w12_linear_view8_workspace,
            "stream": sdv.lib().sd_w12_linear_stream_workspace,
            "stream_view8": sdv.lib().sd_w12_linear_stream_workspace}[kind](N, K, M)
    ws = Mdl.Workspace(int(need))
    if kind == "gemm":
        lin = lambda q, stream=None: Mdl.linear(q, x, ws, stream=stream)
    elif kind == "view8":
        lin = lambda q, stream=None: Mdl.linear_view8(q, x, q.plane8, ws=ws, stream=stream)
    else:
        lin = lambda q, stream=None: Mdl.linear_stream(q, x, q.plane8 if view8 else None, ws=ws, stream=stream)
    y = lin(p)
    stream = torch.cuda.Stream()
    # the launches are replayed from a CUDA graph: no host time between them
    g = torch.cuda.CUDAGraph()
    n_launch = args.steps * n_copies
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, n_copies)):
            lin(packs[i % n_copies], stream=stream)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_launch):
                lin(packs[i % n_copies], stream=stream)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / n_launch
    del y
    nbytes = wbytes + M * K * 2 + M * N * 2
    pk, src = peaks()
    name = {"gemm": "sd_w12_linear", "stream": "sd_w12_linear_stream", "view8": "sd_w12_linear_view8",
            "stream_view8": "sd_w12_linear_stream (8-bit view)"}
    return {"probe": name[args.probe_kernel], "N": N, "K": K, "M": M,
            "tc_min_rows": tc_rows, "us_per_launch": us,
            "GBps": nbytes / (us * 1e-6) / 1e9, "frac_of_peak": nbytes / (us * 1e-6) / 1e9 / pk["hbm_gbs"],
            "peak_source": src, "bytes": nbytes, "escapes": p.n_escapes, "weights": args.probe_weights,
            "format": args.probe_format,
            "l2": f"{n_copies} copies of the packed tensor cycled ({n_copies * wbytes / 2**20:.0f} MiB)"}


def gdn_arm(args):
    """The gated-delta-rule tree kernel (sd_gdn_tree_verify) alone, then with
    the commit (sd_gdn_commit): per-launch time with CUDA events over graph
    replays, against the bytes it must move - each request's fp32 state S0
    [nh][128][128] read once (and written once by the commit), q/k/v in,
    o out, alpha/beta - as a fraction of the measured copy bandwidth."""
    import numpy as np
    import torch
    from speculative_decoding_tree_bit_gb300 import _build
    from speculative_decoding_tree_bit_gb300 import model as Mdl
    from synthetic import workloads as wl
    _build.build()
    R, nh, M = (int(v) for v in args.gdn.split(","))
    # several input sets whose states together exceed L2, cycled by the replays
    per_set = R * nh * 128 * 128 * 4
    n_sets = max(1, -(-256 * 2 ** 20 // per_set))
    sets = []
    for i in range(n_sets):
        g = wl.gdn_inputs(args.seed + i, [M] * R, 8, nh)
        dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a).view(dt)).cuda()
        sets.append(dict(q=dev(g.q, np.int16), k=dev(g.k, np.int16), v=dev(g.v, np.int16),
                         alpha=torch.from_numpy(g.alpha).cuda(), beta=torch.from_numpy(g.beta).cuda(),
                         par=torch.from_numpy(g.parents.astype(np.int32)).cuda(), cu=g.cu,
                         cu_dev=torch.from_numpy(g.cu.astype(np.int32)).cuda(),
                         S=torch.from_numpy(g.S).cuda(), last=torch.full((R,), M - 1, dtype=torch.int32).cuda()))
    layer = Mdl.GdnLayer(R * M, nh)
    rows = R * M
    io_bytes = rows * nh * 128 * 2 * 4 + rows * nh * 4 * 2 + rows * 4
    res = {"probe": "gdn_tree", "R": R, "nh": nh, "M": M, "l2": f"{n_sets} input sets cycled ({n_sets * per_set / 2**20:.0f} MiB of states)"}
    pk, src = peaks()
    for with_commit in (False, True):
        stream = torch.cuda.Stream()
        g_ = torch.cuda.CUDAGraph()

        def one(i):
            d = sets[i % n_sets]
            layer.verify(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["par"], d["cu"], d["S"], stream=stream,
                         cu_dev=d["cu_dev"])
            if with_commit:
                layer.commit(d["last"], d["S"], stream=stream)
        with torch.cuda.stream(stream):
            for i in range(max(args.warmup, n_sets)):
                one(i)
            stream.synchronize()
            with torch.cuda.graph(g_, stream=stream):
                for i in range(args.steps * n_sets):
                    one(i)
        torch.cuda.synchronize()
        g_.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g_.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (args.steps * n_sets)
        nbytes = per_set * (2 if with_commit else 1) + io_bytes
        key = "verify_commit" if with_commit else "verify"
        res[key] = {"us_per_call": us, "bytes": nbytes, "GBps": nbytes / (us * 1e-6) / 1e9,
                    "frac_of_peak": nbytes / (us * 1e-6) / 1e9 / pk["hbm_gbs"]}
    res["status"] = int(layer.status.item())
    res["peak_source"] = src
    return res


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.p:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except Exception:
                self.p.kill()

    def summary(self):
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sms.append(float(r[1]))
                mx = float(r[2])
                for nm, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(nm)
            except Exception:
                continue
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms)}


# ------------------------------------------------------------ CPU oracle --

def oracle_sample(shape, seed, M, ctx, parents, tokens, n_layers=1, reps=1):
    """Time the oracle on a bounded sample: the first n_layers layers plus the
    final norm, lm_head and argmax; returns (per-layer s, lm_head s, threads)."""
    import numpy as np
    import oracle
    from synthetic import workloads as wl
    W = wl.SyntheticWeights(shape, seed, cache=True)
    for l in range(n_layers):
        for nm in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down"):
            W.layer(l, nm)
    W.lm_head()
    layers = []
    for l in range(n_layers):
        k, v = wl.kv_prefix(shape, seed, 0, l, ctx, ctx + M)
        layers.append(oracle.LayerState(k=k, v=v))
    req = oracle.Request(np.asarray(tokens, np.int32), np.asarray(parents, np.int32), ctx, layers)
    t_full = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle.forward(shape, W, [req], n_layers=n_layers)
        t_full.append(time.perf_counter() - t0)
    x = oracle.bf16_to_f64(W.embed_rows(tokens))
    t0 = time.perf_counter()
    oracle.linear(x, W.lm_head())
    t_lm = time.perf_counter() - t0
    per_layer = max(1e-9, (statistics.median(t_full) - t_lm) / n_layers)
    return per_layer, t_lm, oracle_threads()


def oracle_threads() -> int:
    """Threads the oracle's OpenMP loops use: OMP_NUM_THREADS when set (read
    when the library loads), else every host core."""
    try:
        n = int(os.environ.get("OMP_NUM_THREADS", "0").split(",")[0])
    except ValueError:
        n = 0
    return n if n > 0 else os.cpu_count()


def reference_arm(args):
    """The oracle as it stands, timed on the host cores (the reference arm)."""
    import numpy as np
    from synthetic import workloads as wl
    spec = wl.make(args.workload, args.seed)
    shape, M, ctx = spec.shape, spec.M, spec.ctx[0]
    td = spec.drafts[0]
    tokens = np.where(td.copy, 0, td.rand_tok).astype(np.int32)
    tokens[0] = td.root_token
    for _ in range(args.warmup):
        oracle_sample(shape, args.seed, M, ctx, td.parents, tokens, n_layers=1)
    per_layer, t_lm = [], []
    for _ in range(args.steps):
        a, b, thr = oracle_sample(shape, args.seed, M, ctx, td.parents, tokens, n_layers=1)
        per_layer.append(a)
        t_lm.append(b)
    step_s = statistics.median(per_layer) * shape.n_layers + statistics.median(t_lm)
    value = M / step_s
    sample = f"oracle forward of layer 0 + lm_head/argmax per step, M={M}, ctx={ctx}; step = layer x {shape.n_layers} + lm_head"
    return {"metric": "tree_tokens_per_s", "value": value, "unit": "tree tokens/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "M": M, "ctx": ctx, "layers": shape.n_layers},
            "cpu_baseline": {"value": value, "unit": "tree tokens/s", "cores": thr, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tree tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# --------------------------------------------------------------- GPU arm --

def kv_bytes_per_step(shape, ctx, M):
    """Algorithmic cache bytes of one step: every attention layer reads the
    K/V prefix and writes the tree's K/V; every recurrent layer reads its
    state and commits it."""
    hd = 128
    attn = shape.n_attn * shape.Hkv * (ctx + M) * hd * 2 * 2
    nh = shape.H // hd
    rec = shape.n_rec * nh * (hd * hd + hd) * 4 * 2
    return attn + rec


def step_distribution(times_ms) -> dict:
    """Median, 10th / 90th percentiles and a 95% confidence interval of the
    mean (normal approximation) of individually timed steps."""
    import numpy as np
    a = np.asarray(times_ms, dtype=np.float64)
    n = int(a.size)
    mean = float(a.mean())
    half = 1.96 * float(a.std(ddof=1)) / math.sqrt(n) if n > 1 else 0.0
    return {"n": n, "median_ms": float(np.median(a)), "p10_ms": float(np.percentile(a, 10)),
            "p90_ms": float(np.percentile(a, 90)), "mean_ms": mean, "ci95_ms": [mean - half, mean + half]}


def overhead_factor(step_ms: float, timeline) -> tuple:
    """Step time over the sum of its kernels' serialised, event-timed
    durations: below 1 where programmatic dependent launch overlaps kernels."""
    total = sum(t for _, t, _ in timeline)
    return (step_ms / total if total > 0 else None), total


def slowest_rank(ms: float, ms_e2e: float, dist, device) -> tuple:
    """The step times of the slowest replica (max over ranks): the job moves
    at the pace of its slowest rank.  dist None: one process."""
    if dist is None:
        return ms, ms_e2e
    import torch
    t = torch.tensor([ms, ms_e2e], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0]), float(t[1])


def job_throughput(world: int, rows_per_rank: int, ms: float) -> float:
    """Tree tokens per second of the whole job: every rank verifies its own
    rows each step (independent replicas, weak scaling)."""
    return world * rows_per_rank / (ms * 1e-3)


def gpu_arm(args, rank, world, dist):
    import numpy as np
    import torch
    from speculative_decoding_tree_bit_gb300 import _build
    from speculative_decoding_tree_bit_gb300 import model as Mdl
    from synthetic import workloads as wl

    _build.build()
    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    tc_rows = Mdl.set_tc_min_rows(args.tc_min_rows)
    Mdl.set_cluster_finish(args.cluster_finish)
    Mdl.set_deferred_finish(args.deferred_finish)
    Mdl.set_strip(not args.no_strip)
    attn_splits = Mdl.set_attn_splits(args.attn_splits)
    spec = wl.make(args.workload, args.seed)
    shape, R = spec.shape, spec.R
    ctx = max(spec.ctx)
    t0 = time.time()
    W = wl.SyntheticWeights(shape, args.seed)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    if R == 1:
        M = spec.M
        model = Mdl.Model(shape, W, max_rows=M, max_requests=1, max_positions=ctx + M + 64)
        model.set_fused(args.fused)
        kv = Mdl.KVCache(shape, ctx + M + 16).fill(args.seed, ctx)
        log(f"[rank {rank}] model built in {time.time() - t0:.1f}s, packed {model.packed_bytes / 1e9:.2f} GB")
        td = spec.drafts[0]

        def am_fn(tok, par):
            _, am = model.forward(tok, par, kv, logits=False)
            return am.cpu().numpy()

        tokens = wl.copy_rule_tokens(td, am_fn, full_tree=True)
        parents = np.asarray(td.parents, np.int32)
        tok_d = torch.from_numpy(tokens).to(dev)
        par_d = torch.from_numpy(parents).to(dev)
        out = model.outputs(M)
        ctx0 = kv.ctx_len.clone()
        # a recurrent layer's commit replaces its state in place: each step
        # restores it (device copies inside the timed region) so that every
        # step verifies the same tree from the same root state
        S0 = kv.S.clone() if shape.n_rec else None
        z0 = kv.z.clone() if shape.n_rec else None
        restore_bytes = 0 if S0 is None else 2 * (S0.numel() * 4 + z0.numel() * 4)

        def step():
            kv.ctx_len.copy_(ctx0, non_blocking=True)
            if S0 is not None:
                kv.S.copy_(S0, non_blocking=True)
                kv.z.copy_(z0, non_blocking=True)
            model.verify(tok_d, par_d, kv, out=out, stream=stream)
    else:
        # R requests over a paged cache, one batched verify per step
        Mr = spec.M
        M = R * Mr
        model = Mdl.Model(shape, W, max_rows=M, max_requests=R, max_positions=ctx + Mr + 64)
        model.set_fused(args.fused)
        table, n_pages = wl.page_tables(args.seed, spec.ctx, Mr, spec.page_size)
        kv = Mdl.PagedKVCache(shape, table, n_pages, spec.page_size).fill(args.seed, spec.ctx)
        log(f"[rank {rank}] model built in {time.time() - t0:.1f}s, packed {model.packed_bytes / 1e9:.2f} GB")
        cu = np.cumsum([0] + [Mr] * R).astype(np.int32)
        parents = np.concatenate([np.asarray(d.parents, np.int32) for d in spec.drafts])
        par_d = torch.from_numpy(parents).to(dev)
        ctx0 = kv.ctx_len.clone()
        S0 = kv.S.clone() if shape.n_rec else None  # as above: each step from the same root states
        z0 = kv.z.clone() if shape.n_rec else None
        restore_bytes = 0 if S0 is None else 2 * (S0.numel() * 4 + z0.numel() * 4)
        # copy-rule tokens by depth waves over the whole batch (a node's argmax
        # depends on its root path only, final once its ancestors are)
        tokens = np.concatenate([np.where(np.arange(Mr) == 0, d.root_token, d.rand_tok).astype(np.int32)
                                 for d in spec.drafts])
        dep = np.concatenate([wl.depths(np.asarray(d.parents)) for d in spec.drafts])
        cop = np.concatenate([np.asarray(d.copy) for d in spec.drafts])
        rnd = np.concatenate([np.asarray(d.rand_tok) for d in spec.drafts])
        for wave in range(1, int(dep.max()) + 1):
            kv.ctx_len.copy_(ctx0)
            if S0 is not None:
                kv.S.copy_(S0)
                kv.z.copy_(z0)
            o = model.verify_batch(tokens, parents, cu, kv)
            am = o["argmax"].cpu().numpy()
            for r in range(R):
                for i in range(1, Mr):
                    g = cu[r] + i
                    if dep[g] == wave:
                        tokens[g] = am[cu[r] + parents[g]] if cop[g] else rnd[g]
        tok_d = torch.from_numpy(tokens).to(dev)
        out = model.outputs(M, R=R)

        def step():
            kv.ctx_len.copy_(ctx0, non_blocking=True)
            if S0 is not None:
                kv.S.copy_(S0, non_blocking=True)
                kv.z.copy_(z0, non_blocking=True)
            model.verify_batch(tok_d, par_d, cu, kv, out=out, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    st = model.status()
    if st != 0:
        raise SystemExit(f"device status {st} after warm-up")
    acc_len = float(out["accepted_len"].float().mean())
    launches = model.last_launches()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- device-resident timed region
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        if args.nvtx:
            torch.cuda.nvtx.range_push("sdv_step")
        t_host = time.perf_counter()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps):
                step()
            e1.record(stream)
        t_host = (time.perf_counter() - t_host) / args.steps
        if args.nvtx:
            torch.cuda.nvtx.range_pop()
        barrier()
    ms = e0.elapsed_time(e1) / args.steps
    clocks = clk.summary()

    # ---- end to end through the public API with host buffers
    tok_h = torch.from_numpy(tokens).pin_memory()
    par_h = torch.from_numpy(parents).pin_memory()
    res_h = {k: torch.empty_like(out[k], device="cpu").pin_memory() for k in ("accepted_len", "accepted_tokens",
                                                                                 "bonus")}

    def e2e_step():
        tok_d.copy_(tok_h, non_blocking=True)
        par_d.copy_(par_h, non_blocking=True)
        step()
        for k, h in res_h.items():
            h.copy_(out[k], non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            e2e_step()
        barrier()
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
    barrier()
    ms_e2e = e0.elapsed_time(e1) / args.steps

    # ---- per-step distribution: each step between its own pair of events
    # (after the timed region above; diagnostics only, never the value)
    try:
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(max(args.steps, 50))]
        with torch.cuda.stream(stream):
            for a, b in pairs:
                a.record(stream)
                step()
                b.record(stream)
        torch.cuda.synchronize()
        step_stats = step_distribution([a.elapsed_time(b) for a, b in pairs])
    except Exception as ex:  # a failure here must not cost the bench line
        step_stats = {"error": str(ex)[:200]}
    h2d = tok_h.numel() * 4 + par_h.numel() * 4 + 4
    d2h = sum(h.numel() * 4 for h in res_h.values())

    # ---- per-kernel timing pass (events around each kernel group)
    model.set_timing(True)
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    tl = model.timeline()
    model.set_timing(False)

    ms, ms_e2e = slowest_rank(ms, ms_e2e, dist, dev)

    pk, pk_src = peaks()
    gemm = [(k, t, b) for k, t, b in tl if k.startswith("gemm")]  # streamed launches or single GEMMs
    g_ms = sum(t for _, t, _ in gemm)
    g_bytes = sum(b for _, _, b in gemm)
    all_gemm_gbs = g_bytes / (g_ms * 1e-3) / 1e9 if g_ms > 0 else None
    # the dominant kernel: a layer's streamed launch (O, gate/up, down and the
    # next q/k/v: the weights of a whole layer), or, on the tcgen05 path, the
    # gate/up GEMM; algorithmic bytes per launch / its mean event-timed launch
    dom_kind = "gemm_stream" if any(k == "gemm_stream" for k, _, _ in tl) else "gemm_gate_up"
    dom = [(t, b) for k, t, b in tl if k == dom_kind]
    if dom_kind == "gemm_stream":
        # the per-layer launches (the first launch holds layer 0's q/k/v only)
        big = max(b for _, b in dom)
        dom = [(t, b) for t, b in dom if b > 0.5 * big]
    dom_ms = sum(t for t, _ in dom) / len(dom) if dom else None
    dom_bytes = sum(b for _, b in dom) / len(dom) if dom else None
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9 if dom else all_gemm_gbs
    traffic = STREAM_TRAFFIC.get((shape.name, M, dom_kind))
    peak = pk["hbm_gbs"]
    ctx_sum = int(sum(spec.ctx))  # every request's prefix
    step_bytes = model.packed_bytes + kv_bytes_per_step(shape, ctx_sum, M)
    # the pages' per-kernel lower bound: max(FLOPs at 60% of dense peak, bytes at 90% of bandwidth)
    flops = 2.0 * M * (shape.n_weights())
    P = pk["bf16_tflops"] * 1e12
    bound_s = sum(max(2.0 * M * (b / 1.5) / (0.6 * P), b / (0.9 * NOMINAL_BW_GBS * 1e9)) for _, _, b in gemm)
    bound_s += kv_bytes_per_step(shape, ctx_sum, M) / (0.9 * NOMINAL_BW_GBS * 1e9)
    by_kind = {}
    for k, t, b in tl:
        a = by_kind.setdefault(k, [0, 0.0, 0.0])
        a[0] += 1
        a[1] += t
        a[2] += b
    if args.timeline:
        log(json.dumps({k: {"launches": v[0], "ms": round(v[1], 4), "GB/s": round(v[2] / v[1] / 1e6, 1) if v[2] else None}
                        for k, v in by_kind.items()}))
    value = job_throughput(world, M, ms)
    ovh, kernel_sum = overhead_factor(ms, tl)
    res = {
        "metric": "tree_tokens_per_s", "value": value, "unit": "tree tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "verify_step_us": ms * 1e3, "host_submit_us_per_step": t_host * 1e6, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "model": shape.name, "layers": shape.n_layers, "M": M,
                   "requests": R, "tc_min_rows": tc_rows,
                   "attn_splits": attn_splits or "auto", "schedule": "fused" if args.fused else "per-linear",
                   "strip_kernel": not args.no_strip,
                   "split_finish": ("cluster" if args.cluster_finish else
                                    "deferred kernel" if args.deferred_finish else "workspace"),
                   "max_depth": spec.max_depth, "ctx": ctx, "p_copy": spec.p, "accepted_len": acc_len,
                   "state_restore_bytes_per_step": restore_bytes,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2 (packed weights %.1f GB)" % (model.packed_bytes / 1e9)},
        "hbm_gbs": step_bytes / (ms * 1e-3) / 1e9,
        "hbm_frac_of_8tbs": step_bytes / (ms * 1e-3) / 1e9 / NOMINAL_BW_GBS,
        "step_bytes": step_bytes, "step_flops": flops,
        "step_lower_bound_us": bound_s * 1e6,
        "frac_of_step_lower_bound": bound_s / (ms * 1e-3),
        "step_stats": step_stats,
        "kernel_sum_ms": kernel_sum, "overhead_factor": ovh,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak if achieved else None, "traffic": traffic,
                     "kernel": ("k_w12_stream, the per-layer launches (O, gate/up, down, next q/k/v): algorithmic "
                                "bytes per launch / mean event-timed launch" if dom_kind == "gemm_stream" else
                                "%s, gate/up launches (algorithmic bytes per launch / mean event-timed launch)" %
                                ("k_w12_stream" if args.fused else "k_w12_gemm") if M <= 64 and M < tc_rows else
                                "k_w12_gemm_tc"),
                     "algorithmic_bytes_per_launch": dom_bytes, "launch_ms": dom_ms,
                     "all_gemm_launches_gbs": all_gemm_gbs,
                     "peak_source": pk_src},
        "kernels": {k: {"launches": v[0], "ms": v[1]} for k, v in by_kind.items()},
        "e2e": {"value": job_throughput(world, M, ms_e2e), "unit": "tree tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and R == 1:
        per_layer, t_lm, thr = oracle_sample(shape, args.seed, M, ctx, parents, tokens, n_layers=1)
        est = per_layer * shape.n_layers + t_lm
        res["cpu_baseline"] = {"value": M / est, "unit": "tree tokens/s", "cores": thr, "kind": "oracle",
                               "sample": f"oracle forward of layer 0 + lm_head/argmax (M={M}, ctx={ctx}); "
                                         f"step estimated as layer x {shape.n_layers} + lm_head"}
    model.close()
    return res


def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    dist = None
    if args.select:
        print(json.dumps(select_arm(args)), flush=True)
        return
    if args.probe:
        print(json.dumps(probe_arm(args)), flush=True)
        return
    if args.gdn:
        print(json.dumps(gdn_arm(args)), flush=True)
        return
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist_mod
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    res = gpu_arm(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
