#!/usr/bin/env python
"""Benchmark of the fused MoE layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Default workload: the 8-expert top-2 decode sweep (H=4096, I=14336, E=8, k=2,
FP8 E4M3 weights with per-expert scales, dynamic per-tensor FP8 activations,
T in {1,2,4,8,16,32,64}).  One step = one moe_fused_forward call per T of the
sweep (127 tokens).  Inputs are synthetic (seeded); the weights are larger
than L2 and two copies alternate call to call, so every call streams its
experts' weights from HBM.

Prints one JSON line: tokens/s over the timed steps (max over ranks), per-T
microseconds per call, the dominant kernel's roofline (HBM bytes of the
touched experts' weights per launch / its CUDA-event duration), an end-to-end
number through the same API with host buffers, SM clocks sampled during the
timed region, and (rank 0, one GPU) the CPU oracle timed on this host.

--impl reference times the CPU oracle (the plain fp64 implementation the GPU
path is checked against) on the same workload; under torchrun only rank 0
runs it.  N > 1 GPUs run independent replicas (the layer needs no exchange).
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused-MoE layer tokens/s & µs/call; % of HBM BW (decode) or FP8 TC peak"
STEP_NAMES = ["route", "align", "gather_quant_x", "gemm1_swiglu", "quant_h", "gemm2_combine",
              "finalize"]
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 2.0  # nominal dense FP8 / bf16 tensor rate


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode_e8_top2")
    ap.add_argument("--tokens", default="", help="comma list overriding the workload's T sweep")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--shape-sweep", action="store_true",
                    help="first-call vs steady-state time for every T in 1..--max-tokens "
                         "in one process, plus CUDA-graph capture per T bucket")
    ap.add_argument("--max-tokens", type=int, default=8192)
    ap.add_argument("--tp-sweep", action="store_true",
                    help="per-rank device time of the layer sharded over the intermediate "
                         "size for W = 1..8 ranks, the shards run one after another on this "
                         "GPU (tensor-parallel row; the all-reduce itself is not timed)")
    ap.add_argument("--cta-trace", action="store_true",
                    help="per-CTA timeline of the two expert GEMMs (MOE_DEBUG_TRACE stamps: "
                         "entry, inputs ready, first stage landed, exit) for the workload's T "
                         "values, weights cold; prints one JSON line")
    ap.add_argument("--rope", action="store_true",
                    help="time the inverse rotary embedding + per-head FP8 quantisation "
                         "kernel (32 heads of 128, T in 1..8192) instead of the layer")
    ap.add_argument("--placement", default="auto", choices=["auto", "weights", "tokens"],
                    help="MMA operand placement of both expert GEMMs: weight rows in M (the "
                         "swap), tokens in M (ablation), or the library's default choice")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload sweep of every measured configuration")
    ap.add_argument("--config-calls", type=int, default=50,
                    help="blocks of back-to-back calls per T in the per-workload sweep (at "
                         "least 50)")
    ap.add_argument("--one-kernel", action="store_true",
                    help="small batches as one cooperative kernel (MOE_FLAG_ONE_KERNEL)")
    ap.add_argument("--no-sm-pairs", action="store_true",
                    help="ablation: wide FP8 gate/up tiles on one SM each instead of SM pairs "
                         "(tcgen05 cta_group::2)")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def measured_peaks():
    """(HBM GB/s, bf16 dense TFLOP/s burst, 'measured' | 'fallback')."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return (float(d.get("hbm_gbs", FALLBACK_HBM_GBS)),
                float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), "measured")
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "mixture_experts_layer_align_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, Ts):
    """DRAM bytes per launch of the gate/up GEMM from the committed ncu summary,
    averaged over the T values of one step (one launch each), if it was taken
    on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", f"gemm1_swiglu_{workload}_traffic.txt")
    if not os.path.exists(p):
        return None
    kv = {}
    with open(p) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.split("=", 1)
                kv[k.strip()] = v.strip()
    if kv.get("kernel_source_hash") != kernel_source_hash():
        return None
    try:
        return sum(float(kv[f"dram_bytes_T{T}"]) for T in Ts) / len(Ts)
    except (KeyError, ValueError):
        return None


def max_over_ranks(ms: float, dist=None, device="cpu") -> float:
    """The slowest rank's time (each rank runs one independent replica)."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_step: int, steps: int, ms: float) -> float:
    """Whole-job throughput: every replica processed steps x tokens_per_step."""
    return world * tokens_per_step * steps / (ms * 1e-3)


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.5)  # let the sampler start before the timed region
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def mark(self, begin: bool):
        import datetime
        if begin:
            self.t0 = datetime.datetime.now()
        else:
            self.t1 = datetime.datetime.now()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.tmp is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.tmp.flush()
        with open(self.tmp.name) as f:
            rows = [r.split(", ") for r in f.read().strip().splitlines() if r.strip()]
        os.unlink(self.tmp.name)
        import datetime
        uuids = {r[1].strip() for r in rows if len(r) >= 10}
        use_uuid = self.uuid if self.uuid in uuids else None
        stamped = []
        for r in rows:
            if len(r) < 10 or (use_uuid and r[1].strip() != use_uuid):
                continue
            try:
                stamped.append((datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f"),
                                r[1:]))
            except ValueError:
                continue
        t0, t1 = getattr(self, "t0", None), getattr(self, "t1", None)
        window = "timed region"
        mine = [r for ts, r in stamped if t0 is None or t1 is None or t0 <= ts <= t1]
        if not mine and t0 is not None and t1 is not None:
            # a timed region shorter than the sampling period: the samples
            # taken within 100 ms of it
            pad = datetime.timedelta(milliseconds=100)
            mine = [r for ts, r in stamped if t0 - pad <= ts <= t1 + pad]
            window = "within 100 ms of the timed region"
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in mine:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
               "samples": len(sm)}
        if window != "timed region":
            out["window"] = window
        return out


def tokens_list(args, cfg):
    if args.tokens:
        return [int(t) for t in args.tokens.split(",")]
    return list(cfg["T"])


def workload_config(name, cfg, Ts):
    """The `config` object of the JSON line: the workload by name and its
    sizes.  Both arms (ours and the reference arm) print exactly this dict."""
    fp8 = cfg["dtype"] == "fp8"
    return {"workload": name, "tokens": list(Ts), "H": cfg["H"], "I": cfg["I"], "E": cfg["E"],
            "top_k": cfg["top_k"], "renormalize": True, "routing": cfg["routing"],
            "weights": "e4m3 per-expert scale" if fp8 else "bf16",
            "activations": "dynamic per-tensor e4m3" if fp8 else "bf16"}


def layer_work(touched, T, H, I, E, k, fp8):
    """Algorithmic bytes and FLOPs of one layer call (the touched experts'
    weights, logits, x in, out; 2 x routed pairs x weight rows x K)."""
    esize = 1 if fp8 else 2
    nbytes = touched * 3 * H * I * esize + (8 * E if fp8 else 0) + T * E * 4 + 2 * T * H * 2
    flops = 6.0 * T * k * H * I
    return nbytes, flops


def roofline_fractions(us, nbytes, flops, hbm_gbs, tc_tflops):
    """(binding limit, fraction of it, HBM fraction, tensor fraction)."""
    t = us * 1e-6
    hbm = nbytes / t / 1e9 / hbm_gbs
    tc = flops / t / 1e12 / tc_tflops
    t_hbm = nbytes / (hbm_gbs * 1e9)
    t_tc = flops / (tc_tflops * 1e12)
    return ("hbm", hbm, hbm, tc) if t_hbm >= t_tc else ("tensor", tc, hbm, tc)


def percentile(v, q):
    v = sorted(v)
    return v[min(len(v) - 1, max(0, int(round(q * (len(v) - 1)))))]


CALL_BLOCK = 5


def time_calls(call, n, block=CALL_BLOCK, warm=10):
    """Device time per call, us, of each of n blocks of `block` back-to-back
    calls: CUDA events on the current stream between blocks, none between the
    calls of a block (an event between two calls keeps the next call's first
    kernel from overlapping the previous call's last one, which back-to-back
    calls otherwise do) and none inside a call."""
    import torch
    for i in range(warm):
        call(i)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    torch.cuda.synchronize()
    ev[0].record()
    for b in range(n):
        for j in range(block):
            call(b * block + j)
        ev[b + 1].record()
    torch.cuda.synchronize()
    return [ev[b].elapsed_time(ev[b + 1]) * 1e3 / block for b in range(n)]


def graph_call_us(call, n=20, reps=5):
    """Device time per call when n back-to-back calls (cycling the same
    inputs and weight copies as `call`) are captured once in a CUDA graph and
    the graph is replayed: the launch path a serving loop would use.  Not the
    headline `value` (that is eager calls), reported beside it."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(0)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(n):
            call(i)
    graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (n * reps)


L2_BYTES = 129 * 2 ** 20


def weight_copies(w, touched_bytes_min, inputs):
    """Enough copies of the weights that consecutive calls, cycling through
    them, never find their experts' weights in L2: >= 2 x L2 of distinct
    weight bytes between two uses of one copy."""
    n = min(512, max(2, -(-2 * L2_BYTES // max(touched_bytes_min, 1))))
    out = [w]
    for _ in range(n - 1):
        out.append(inputs.Weights(w.w13.clone(), w.w2.clone(), w.w13_scale, w.w2_scale, w.dtype,
                                  w.H, w.I, w.E))
    return out


def oracle_sample(cfg, Ts, w, acts):
    """One oracle call per T (the prefill workloads: the smallest T only):
    tokens/s of the fp64 CPU oracle on this host."""
    import oracle
    wc = [t.cpu() if t is not None else None for t in (w.w13, w.w2, w.w13_scale, w.w2_scale)]
    sample_T = [min(Ts)] if min(Ts) >= 2048 else list(Ts)
    el, tokens = 0.0, 0
    for T in sample_T:
        a = acts[T]
        x, lg = a.x.cpu(), a.logits.cpu()
        t0 = time.perf_counter()
        oracle.moe_forward(x, lg, wc[0], wc[1], wc[2], wc[3], cfg["top_k"], True)
        el += time.perf_counter() - t0
        tokens += T
    cores = oracle.max_threads()
    return {"value": round(tokens / el, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"one fp64 oracle call per T in {sample_T} ({tokens} tokens, {el:.1f} s)"}


CONFIG_NAMES = ["tiny_bf16", "decode_e8_top2", "finegrained_e128", "skewed_e256",
                "prefill_e128_uniform", "prefill_e128_zipf"]


def config_sweep(moe, inputs, dev, hbm_peak, fp8_peak, bf16_peak, n_calls, with_cpu, flags=0):
    """Every measured workload: per-T device time of a call (median, p10,
    p90 over n_calls blocks of back-to-back calls, weights cold in L2),
    tokens/s, and the fraction of the binding roofline (HBM bytes or tensor
    FLOPs)."""
    import torch
    out = {}
    for name in CONFIG_NAMES:
        cfg = inputs.workload(name)
        H, I, E, k = cfg["H"], cfg["I"], cfg["E"], cfg["top_k"]
        fp8 = cfg["dtype"] == "fp8"
        dtype = moe.MOE_DT_FP8_E4M3 if fp8 else moe.MOE_DT_BF16
        tc_peak = fp8_peak if fp8 else bf16_peak
        Ts = list(cfg["T"])
        w = inputs.make_weights(H, I, E, cfg["dtype"], seed=0, device=dev)
        acts = {T: inputs.make_activations(T, H, E, cfg["routing"], seed=0, device=dev) for T in Ts}
        outs = {T: torch.empty(T, H, dtype=torch.bfloat16, device=dev) for T in Ts}
        wss = {T: moe.alloc_workspace(T, H, I, E, k, dtype, dev) for T in Ts}
        touched = {}
        for T in Ts:
            cnt = torch.empty(E, dtype=torch.int32, device=dev)
            a = acts[T]
            moe.moe_fused_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, k, True,
                                  out=outs[T], workspace=wss[T], counts_out=cnt, debug_flags=flags)
            st = moe.moe_check_status(wss[T])
            if st != 0:
                raise RuntimeError(f"{name} T={T}: device status {moe.status_string(st)}")
            touched[T] = int((cnt > 0).sum())
        esize = 1 if fp8 else 2
        copies = weight_copies(w, min(touched.values()) * 3 * H * I * esize, inputs)
        rows = []
        for T in Ts:
            a = acts[T]

            def call(i, T=T, a=a):
                ww = copies[i % len(copies)]
                moe.moe_fused_forward(a.x, a.logits, ww.w13, ww.w2, ww.w13_scale, ww.w2_scale, k,
                                      True, out=outs[T], workspace=wss[T], debug_flags=flags)

            us = time_calls(call, n_calls)
            st = moe.moe_check_status(wss[T])
            if st != 0:
                raise RuntimeError(f"{name} T={T}: device status {moe.status_string(st)}")
            med = statistics.median(us)
            nbytes, flops = layer_work(touched[T], T, H, I, E, k, fp8)
            bound, frac, hfrac, tfrac = roofline_fractions(med, nbytes, flops, hbm_peak, tc_peak)
            rows.append({"T": T, "us_median": round(med, 2), "us_p10": round(percentile(us, 0.1), 2),
                         "us_p90": round(percentile(us, 0.9), 2), "calls": len(us) * CALL_BLOCK,
                         "tokens_per_s": round(T / (med * 1e-6), 1), "touched_experts": touched[T],
                         "layer_bytes": nbytes, "layer_flops": flops, "bound": bound,
                         "frac": round(frac, 4), "hbm_frac": round(hfrac, 4),
                         "tensor_frac": round(tfrac, 4)})
        entry = {"config": workload_config(name, cfg, Ts), "weight_copies": len(copies),
                 "per_T": rows,
                 "tokens_per_s": round(sum(Ts) / (sum(r["us_median"] for r in rows) * 1e-6), 1)}
        if with_cpu:
            entry["cpu_baseline"] = oracle_sample(cfg, Ts, w, acts)
        out[name] = entry
        del w, copies, acts, outs, wss
        torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------------- CPU oracle
def time_oracle(cfg, Ts, weights_cpu, acts_cpu, min_seconds=10.0, max_passes=8):
    """Wall time of the CPU oracle over the T sweep; repeats whole passes
    until `min_seconds` elapsed (at most `max_passes`)."""
    import oracle
    w = weights_cpu
    passes, t0 = 0, time.perf_counter()
    while True:
        for T in Ts:
            a = acts_cpu[T]
            oracle.moe_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale,
                               cfg["top_k"], True)
        passes += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or passes >= max_passes:
            return el, passes, oracle.max_threads()


def run_reference(args, rank, world):
    if rank != 0:
        return
    import torch
    from mixture_experts_layer_align_gb300 import inputs
    cfg = inputs.workload(args.workload)
    Ts = tokens_list(args, cfg)
    w = inputs.make_weights(cfg["H"], cfg["I"], cfg["E"], cfg["dtype"], seed=0,
                            device="cuda" if torch.cuda.is_available() else "cpu")
    w = inputs.Weights(w.w13.cpu(), w.w2.cpu(), None if w.w13_scale is None else w.w13_scale.cpu(),
                       None if w.w2_scale is None else w.w2_scale.cpu(), w.dtype, w.H, w.I, w.E)
    acts = {T: inputs.make_activations(T, cfg["H"], cfg["E"], cfg["routing"], seed=0) for T in Ts}
    import oracle

    # One step = one oracle call, on the sweep's T values in turn: a bounded
    # sample of the workload (the oracle's cost per routed pair hardly depends
    # on T), so that K steps of the slow fp64 program still end within minutes.
    def call(i):
        T = Ts[i % len(Ts)]
        a = acts[T]
        t0 = time.perf_counter()
        oracle.moe_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, cfg["top_k"],
                           True)
        return time.perf_counter() - t0, T

    for i in range(args.warmup):
        call(i)
    el, tokens = 0.0, 0
    for i in range(args.steps):
        e, T = call(i)
        el += e
        tokens += T
    value = tokens / el
    cores = oracle.max_threads()
    sample = (f"{args.workload}: one oracle call per step, T cycling through {Ts} "
              f"({tokens} tokens over {args.steps} steps), fp64, {cores} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload, cfg, Ts),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU path
def run_ours(args, rank, local_rank, world):
    import torch
    import mixture_experts_layer_align_gb300 as moe
    from mixture_experts_layer_align_gb300 import inputs

    moe.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    cfg = inputs.workload(args.workload)
    Ts = tokens_list(args, cfg)
    H, I, E, k = cfg["H"], cfg["I"], cfg["E"], cfg["top_k"]
    fp8 = cfg["dtype"] == "fp8"
    dtype = moe.MOE_DT_FP8_E4M3 if fp8 else moe.MOE_DT_BF16
    flags = {"auto": 0, "weights": moe.MOE_FLAG_WEIGHTS_IN_M,
             "tokens": moe.MOE_FLAG_TOKENS_IN_M}[args.placement]
    if args.no_sm_pairs:
        flags |= moe.MOE_FLAG_NO_SM_PAIRS
    if args.one_kernel:
        flags |= moe.MOE_FLAG_ONE_KERNEL
    w = inputs.make_weights(H, I, E, cfg["dtype"], seed=0, device=dev)
    acts = {T: inputs.make_activations(T, H, E, cfg["routing"], seed=0, device=dev) for T in Ts}
    outs = {T: torch.empty(T, H, dtype=torch.bfloat16, device=dev) for T in Ts}
    wss = {T: moe.alloc_workspace(T, H, I, E, k, dtype, dev) for T in Ts}

    # routing statistics per T (touched experts -> algorithmic bytes)
    stats = {}
    esize = 1 if fp8 else 2
    for T in Ts:
        counts = torch.empty(E, dtype=torch.int32, device=dev)
        a = acts[T]
        moe.moe_fused_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, k, True,
                              out=outs[T], workspace=wss[T], counts_out=counts, debug_flags=flags)
        st = moe.moe_check_status(wss[T])
        if st != 0:
            raise RuntimeError(f"device status {moe.status_string(st)}")
        c = counts.cpu()
        touched = int((c > 0).sum())
        P = T * k
        stats[T] = dict(
            touched=touched, max_rows=int(c.max()),
            gemm1_bytes=touched * 2 * I * H * esize + P * H * esize + P * I * (4 if fp8 else 2),
            gemm2_bytes=touched * H * I * esize + P * I * esize + P * H * 4,
            gemm1_flops=2.0 * P * 2 * I * H, gemm2_flops=2.0 * P * H * I,
            layer_bytes=touched * 3 * H * I * esize + 8 * E + T * E * 4 + 2 * T * H * 2)

    # copies of the weights in other buffers, cycled call to call, so that no
    # call finds its experts' weights in L2
    copies = weight_copies(w, min(stats[T]["touched"] for T in Ts) * 3 * I * H * esize, inputs)
    n_copies = len(copies)
    calls_per_step = len(Ts)
    def launches(T):
        # the single cooperative kernel replaces the sequence where it applies
        if args.one_kernel and T * k <= 2048 and E <= 256 and T * k * H <= (8 << 20):
            return 1
        return moe.moe_fused_launch_count(T, H, I, E, k, dtype)

    launches_per_step = sum(launches(T) for T in Ts)

    def one_step(step_idx, events=None):
        for j, T in enumerate(Ts):
            ww = copies[(step_idx * calls_per_step + j) % len(copies)]
            a = acts[T]
            moe.moe_fused_forward(a.x, a.logits, ww.w13, ww.w2, ww.w13_scale, ww.w2_scale, k,
                                  True, out=outs[T], workspace=wss[T], debug_flags=flags,
                                  events=None if events is None else events[j])

    for i in range(max(args.warmup, 3)):
        one_step(i)
    torch.cuda.synchronize()

    K = args.steps
    ev = [[moe.make_step_events(8) for _ in Ts] for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if not uuid.startswith("GPU-"):
            uuid = "GPU-" + uuid
    except Exception:
        pass
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    # timed region: K steps through the plain API (kernels chained with
    # programmatic dependent launch), then the same K steps with CUDA events
    # recorded between the kernels of every call for the per-kernel durations
    # (an event between two kernels removes their launch overlap, so this
    # second pass is slightly slower and is not used for `value`)
    with ClockSampler(uuid) as clk:
        clk.mark(True)
        start.record()
        for s in range(K):
            one_step(s)
        stop.record()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        mid = torch.cuda.Event(enable_timing=True)
        end2 = torch.cuda.Event(enable_timing=True)
        mid.record()
        for s in range(K):
            one_step(s, ev[s])
        end2.record()
        torch.cuda.synchronize()
        clk.mark(False)
    if dist is not None:
        dist.barrier()
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), dist, dev)
    instrumented_ms = mid.elapsed_time(end2)
    clocks = clk.summary()

    # per-step (kernel) durations from the events inside the timed region
    per_T_call_us = {T: [] for T in Ts}
    step_ms = {n: 0.0 for n in STEP_NAMES}
    gemm1_ms = {T: [] for T in Ts}
    gemm2_ms = {T: [] for T in Ts}
    for s in range(K):
        for j, T in enumerate(Ts):
            e = ev[s][j]
            per_T_call_us[T].append(e[0].elapsed_time(e[7]) * 1e3)
            for i, n in enumerate(STEP_NAMES):
                step_ms[n] += e[i].elapsed_time(e[i + 1])
            gemm1_ms[T].append(e[3].elapsed_time(e[4]))
            gemm2_ms[T].append(e[5].elapsed_time(e[6]))
    total_kernel_ms = sum(step_ms.values())
    hbm_peak, bf16_peak, peak_kind = measured_peaks()
    tc_peak = bf16_peak * (FP8_OVER_BF16 if fp8 else 1.0)
    tc_kind = (f"{peak_kind} bf16_tflops x {FP8_OVER_BF16:g} (nominal FP8/bf16)" if fp8
               else f"{peak_kind} bf16_tflops")
    # roofline of the heavier expert GEMM over its launches, against the
    # binding limit: HBM bytes / bandwidth or FLOPs / tensor peak
    dominant = ("gemm2_combine" if step_ms["gemm2_combine"] > step_ms["gemm1_swiglu"]
                else "gemm1_swiglu")
    g = "gemm2" if dominant == "gemm2_combine" else "gemm1"
    dom_ms = sum(sum((gemm2_ms if g == "gemm2" else gemm1_ms)[T]) for T in Ts)
    dom_bytes = sum(stats[T][f"{g}_bytes"] for T in Ts) * K
    dom_flops = sum(stats[T][f"{g}_flops"] for T in Ts) * K
    tensor_bound = dom_flops / (tc_peak * 1e12) > dom_bytes / (hbm_peak * 1e9)
    achieved_gbs = dom_bytes / (dom_ms * 1e-3) / 1e9
    achieved_tfs = dom_flops / (dom_ms * 1e-3) / 1e12
    traffic = recorded_traffic(args.workload, Ts) if dominant == "gemm1_swiglu" else None
    if tensor_bound:
        roofline = {"kernel": dominant, "bound": "tensor", "achieved": round(achieved_tfs, 1),
                    "peak": round(tc_peak, 1), "peak_kind": tc_kind, "unit": "TFLOP/s",
                    "frac": round(achieved_tfs / tc_peak, 4), "traffic": traffic,
                    "algorithmic_flops": "2 x routed pairs x weight rows x K, per launch",
                    "hbm_frac": round(achieved_gbs / hbm_peak, 4)}
    else:
        roofline = {"kernel": dominant, "bound": "hbm", "achieved": round(achieved_gbs, 1),
                    "peak": hbm_peak, "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s",
                    "frac": round(achieved_gbs / hbm_peak, 4), "traffic": traffic,
                    "algorithmic_bytes": "touched experts' weight bytes + routed activation "
                                         "rows in + h out, per launch",
                    "tensor_frac": round(achieved_tfs / tc_peak, 4)}

    one_kernel_Ts = [T for T in Ts if launches(T) == 1]
    if one_kernel_Ts:
        # the whole layer runs as one kernel there, so the events between the
        # steps of a call do not bracket the GEMMs: report that kernel against
        # the layer's algorithmic bytes over the call time instead
        ok_us = sum(sum(per_T_call_us[T]) for T in one_kernel_Ts)
        ok_bytes = sum(stats[T]["layer_bytes"] for T in one_kernel_Ts) * K
        ok_gbs = ok_bytes / (ok_us * 1e-6) / 1e9
        roofline = {"kernel": "moe_fused_small_kernel (whole layer, one cooperative kernel)",
                    "bound": "hbm", "achieved": round(ok_gbs, 1), "peak": hbm_peak,
                    "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s",
                    "frac": round(ok_gbs / hbm_peak, 4), "traffic": None,
                    "algorithmic_bytes": "touched experts' weight bytes + scales + logits + x "
                                         "in + out, per call",
                    "calls": f"T in {one_kernel_Ts}"}

    tokens_per_step = sum(Ts)
    value = job_tokens_per_s(world, tokens_per_step, K, elapsed_ms)
    # per-T device time of a call without events inside it (events between
    # blocks of back-to-back calls), median / p10 / p90 over >= 50 blocks
    sweep = []
    for T in Ts:
        a = acts[T]

        def call(i, T=T, a=a):
            ww = copies[i % len(copies)]
            moe.moe_fused_forward(a.x, a.logits, ww.w13, ww.w2, ww.w13_scale, ww.w2_scale, k,
                                  True, out=outs[T], workspace=wss[T], debug_flags=flags)

        us_all = time_calls(call, max(50, K))
        us = statistics.median(us_all)
        graph_us = graph_call_us(call)
        nbytes, flops = layer_work(stats[T]["touched"], T, H, I, E, k, fp8)
        bound, frac, hfrac, tfrac = roofline_fractions(us, nbytes, flops, hbm_peak, tc_peak)
        sweep.append({
            "T": T, "us_median": round(us, 2), "us_p10": round(percentile(us_all, 0.1), 2),
            "us_p90": round(percentile(us_all, 0.9), 2), "calls": len(us_all) * CALL_BLOCK,
            "tokens_per_s": round(T / (us * 1e-6), 1),
            "touched_experts": stats[T]["touched"], "max_rows_per_expert": stats[T]["max_rows"],
            "layer_bytes": nbytes, "bound": bound, "frac": round(frac, 4),
            "hbm_frac": round(hfrac, 4), "tensor_frac": round(tfrac, 4),
            "gemm1_us_events": round(statistics.median(gemm1_ms[T]) * 1e3, 2),
            "gemm2_us_events": round(statistics.median(gemm2_ms[T]) * 1e3, 2),
            "graph_us_per_call": round(graph_us, 2),
            "graph_frac": round(roofline_fractions(graph_us, nbytes, flops, hbm_peak,
                                                   tc_peak)[1], 4)})

    # end to end through the same API: pinned host inputs -> device -> host output
    e2e = None
    if not args.no_e2e:
        host = {T: (acts[T].x.cpu().pin_memory(), acts[T].logits.cpu().pin_memory(),
                    torch.empty(T, H, dtype=torch.bfloat16).pin_memory()) for T in Ts}
        h2d = sum(T * H * 2 + T * E * 4 for T in Ts)
        d2h = sum(T * H * 2 for T in Ts)

        # Copies run on two side streams, as a serving loop would issue them:
        # two sets of device buffers alternate step to step, the next step's
        # inputs go up while this step runs, and the step's results come back
        # once its calls are done.  The compute stream waits twice per step (its
        # inputs are up; the results last held in this set have left) and
        # records one event, so that nothing between two calls of a step keeps
        # one call's first kernel from overlapping the previous call's last.
        compute = torch.cuda.current_stream(dev)
        up = torch.cuda.Stream(device=dev)
        down = torch.cuda.Stream(device=dev)
        dx = [{T: torch.empty_like(acts[T].x) for T in Ts} for _ in range(2)]
        dl = [{T: torch.empty_like(acts[T].logits) for T in Ts} for _ in range(2)]
        do = [{T: torch.empty(T, H, dtype=torch.bfloat16, device=dev) for T in Ts}
              for _ in range(2)]
        inputs_up = [torch.cuda.Event() for _ in range(2)]
        step_done = [torch.cuda.Event() for _ in range(2)]
        results_down = [torch.cuda.Event() for _ in range(2)]
        for b in range(2):
            step_done[b].record(compute)
            results_down[b].record(compute)

        def e2e_step(s):
            b = s % 2
            with torch.cuda.stream(up):
                up.wait_event(step_done[b])  # the step that last used this set has run
                for T in Ts:
                    hx, hl, _ = host[T]
                    dx[b][T].copy_(hx, non_blocking=True)
                    dl[b][T].copy_(hl, non_blocking=True)
                inputs_up[b].record(up)
            compute.wait_event(inputs_up[b])
            compute.wait_event(results_down[b])
            for j, T in enumerate(Ts):
                ww = copies[(s * calls_per_step + j) % len(copies)]
                moe.moe_fused_forward(dx[b][T], dl[b][T], ww.w13, ww.w2, ww.w13_scale,
                                      ww.w2_scale, k, True, out=do[b][T], workspace=wss[T],
                                      debug_flags=flags)
            step_done[b].record(compute)
            with torch.cuda.stream(down):
                down.wait_event(step_done[b])
                for T in Ts:
                    host[T][2].copy_(do[b][T], non_blocking=True)
                results_down[b].record(down)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record()
        up.wait_stream(compute)  # the first step's uploads start inside the timed region
        for s in range(K):
            e2e_step(s)
        compute.wait_stream(down)  # the last results have reached the host
        s1.record()
        torch.cuda.synchronize()
        e_ms = max_over_ranks(s0.elapsed_time(s1), dist, dev)
        e2e = {"value": job_tokens_per_s(world, tokens_per_step, K, e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        wc = inputs.Weights(w.w13.cpu(), w.w2.cpu(),
                            None if w.w13_scale is None else w.w13_scale.cpu(),
                            None if w.w2_scale is None else w.w2_scale.cpu(), w.dtype, H, I, E)
        ac = {T: inputs.Activations(acts[T].x.cpu(), acts[T].logits.cpu(), T) for T in Ts}
        el, passes, cores = time_oracle(cfg, Ts, wc, ac)
        cpu = {"value": passes * tokens_per_step / el, "unit": "tokens/s", "cores": cores,
               "kind": "oracle",
               "sample": f"{passes} pass(es) of the T sweep {Ts} ({passes * tokens_per_step} "
                         f"tokens), fp64 oracle, {el:.1f} s"}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    configs = None
    if rank == 0 and world == 1 and not args.no_configs:
        del copies
        torch.cuda.empty_cache()
        with ClockSampler(uuid) as clk2:
            clk2.mark(True)
            configs = config_sweep(moe, inputs, dev, hbm_peak, bf16_peak * FP8_OVER_BF16,
                                   bf16_peak, max(50, args.config_calls),
                                   not args.no_cpu_baseline, flags)
            clk2.mark(False)
        configs_clocks = clk2.summary()
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if fp8 else "bf16",
        "data": "synthetic",
        "config": workload_config(args.workload, cfg, Ts),
        "setup": {
            "step": f"one moe_fused_forward per T ({calls_per_step} calls, {tokens_per_step} "
                    "tokens)",
            "l2": f"inputs larger than L2: {n_copies} copies of the "
                  f"{(w.w13.numel() + w.w2.numel()) * esize / 1e9:.2f} GB weights, cycled call "
                  "to call",
            "parallelism": f"replicas x{world}",
            "placement": {"auto": "gate/up: weights in the MMA M slot; down: weights in M "
                                   "if I > 2048 else tokens in M",
                           "weights": "weights in the MMA M slot for both GEMMs (swap-AB)",
                           "tokens": "tokens in the MMA M slot for both GEMMs (no swap)"}[
                              args.placement] + (
                              "; wide gate/up tiles on one SM each" if args.no_sm_pairs
                              else "") + ("; small batches as one cooperative kernel"
                                          if args.one_kernel else "")},
        "sweep": sweep,
        "sweep_timing": f"per call: CUDA events between blocks of {CALL_BLOCK} back-to-back "
                        "calls (none between the calls of a block, none inside a call); "
                        "median / p10 / p90 over the blocks' per-call times; weights cold "
                        "in L2; graph_us_per_call: 20 of the same calls captured in one "
                        "CUDA graph and replayed (reported beside, not in value)",
        "kernel_share": {n: round(step_ms[n] / total_kernel_ms, 4) for n in STEP_NAMES},
        "kernel_timing": "CUDA events between the kernels of every call, second pass of the "
                         f"same {K} steps ({instrumented_ms / K:.3f} ms/step with events)",
        "roofline": roofline,
        "clocks": clocks,
        "gpu_launches": K * launches_per_step,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if configs is not None:
        line["configs"] = configs
        line["configs_timing"] = ("every measured workload: device time per call from CUDA "
                                  f"events between blocks of {CALL_BLOCK} back-to-back calls "
                                  "(median, p10, p90 over the blocks), "
                                  "weights cycled through enough copies to stay out of L2; "
                                  "frac = fraction of the binding roofline (HBM bytes of the "
                                  "touched experts + x/logits/out against measured hbm_gbs, or "
                                  "6 x pairs x H x I FLOPs against the tensor peak)")
        line["configs_clocks"] = configs_clocks
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# --------------------------------------------------------------------------- shapes
def run_shape_sweep(args, rank, local_rank):
    """Every T in 1..max_tokens (shuffled) through one process: the first call
    at each T against the median of three more.  There is no per-shape
    compilation or plan, so a first call costs what a later one does.  Then one
    CUDA graph per power-of-two T bucket is captured, replayed on new inputs
    written into its static buffers, and checked against an eager call."""
    import random

    import torch
    import mixture_experts_layer_align_gb300 as moe
    from mixture_experts_layer_align_gb300 import inputs

    if rank != 0:
        return
    moe.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = args.workload if args.workload != "decode_e8_top2" else "finegrained_e128"
    cfg = inputs.workload(wl)
    H, I, E, k = cfg["H"], cfg["I"], cfg["E"], cfg["top_k"]
    fp8 = cfg["dtype"] == "fp8"
    dtype = moe.MOE_DT_FP8_E4M3 if fp8 else moe.MOE_DT_BF16
    Tmax = args.max_tokens
    w = inputs.make_weights(H, I, E, cfg["dtype"], seed=0, device=dev)
    a = inputs.make_activations(Tmax, H, E, cfg["routing"], seed=0, device=dev)
    out = torch.empty(Tmax, H, dtype=torch.bfloat16, device=dev)
    ws = moe.alloc_workspace(Tmax, H, I, E, k, dtype, dev)

    def call(T, o=None, x=None, lg=None):
        moe.moe_fused_forward(a.x[:T] if x is None else x, a.logits[:T] if lg is None else lg,
                              w.w13, w.w2, w.w13_scale, w.w2_scale, k, True,
                              out=out[:T] if o is None else o, workspace=ws)

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ev[0].record()
    call(1)
    ev[1].record()
    torch.cuda.synchronize()
    process_first = {"host_us": (time.perf_counter() - t0) * 1e6,
                     "device_us": ev[0].elapsed_time(ev[1]) * 1e3}

    # Each first call is enqueued behind the previous T's calls, so the GPU is
    # busy while the host prepares it (as in steady use); results are read
    # after every chunk of T values.
    Ts = list(range(2, Tmax + 1))
    random.Random(0).shuffle(Ts)
    rows = []
    chunk = 64
    prev = 1
    for c0 in range(0, len(Ts), chunk):
        part = Ts[c0:c0 + chunk]
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in part]
        host = []
        call(prev)  # keeps the GPU busy while the first measured call is enqueued
        for T, e in zip(part, evs):
            h0 = time.perf_counter()
            e[0].record()
            call(T)
            e[1].record()
            host.append((time.perf_counter() - h0) * 1e6)
            for i in range(3):
                call(T)
                e[2 + i].record()
        torch.cuda.synchronize()
        for T, e, h in zip(part, evs, host):
            first = e[0].elapsed_time(e[1]) * 1e3
            steady = sorted([e[1].elapsed_time(e[2]), e[2].elapsed_time(e[3]),
                             e[3].elapsed_time(e[4])])[1] * 1e3
            rows.append((T, first, steady, h))
        prev = part[-1]
    st = moe.moe_check_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {moe.status_string(st)}")
    ratios = sorted(r[1] / r[2] for r in rows)
    host = sorted(r[3] for r in rows)
    rows.sort()
    pick = {1 << i for i in range(14)} | {3, 37, 100, 1000, 3000, 5000, 7777}
    per_T = [{"T": T, "first_us": round(f, 1), "steady_us": round(s_, 1),
              "host_first_us": round(h, 1)} for T, f, s_, h in rows if T in pick]

    # one CUDA graph per bucket: capture, replay on fresh inputs, compare
    graphs = []
    for T in [1 << i for i in range(14) if (1 << i) <= Tmax]:
        gx = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        gl = torch.empty(T, E, dtype=torch.float32, device=dev)
        go = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        gx.copy_(a.x[:T])
        gl.copy_(a.logits[:T])
        s_ = torch.cuda.Stream(device=dev)
        s_.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s_):
            call(T, go, gx, gl)  # eager call on the capture stream first
        torch.cuda.current_stream().wait_stream(s_)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s_):
            call(T, go, gx, gl)
        fresh = inputs.make_activations(T, H, E, cfg["routing"], seed=T + 1, device=dev)
        gx.copy_(fresh.x)
        gl.copy_(fresh.logits)
        g.replay()
        ref = torch.empty_like(go)
        call(T, ref, fresh.x, fresh.logits)
        torch.cuda.synchronize()
        err = ((go.float() - ref.float()).abs().max() /
               ref.float().abs().max().clamp_min(1e-30)).item()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record()
        for _ in range(20):
            g.replay()
        g1.record()
        torch.cuda.synchronize()
        graphs.append({"T": T, "replay_us": round(g0.elapsed_time(g1) * 1e3 / 20, 1),
                       "max_rel_diff_vs_eager": err})
        del g
    line = {
        "metric": "first-call vs steady-state us per moe_fused_forward, every T in 1..%d" % Tmax,
        "workload": f"{wl}: H={H}, I={I}, E={E}, top_k={k}, {cfg['routing']} routing, "
                    f"{'FP8 E4M3' if fp8 else 'bf16'}",
        "order": "T = 2..%d in seeded random order after the process's first call (T=1)" % Tmax,
        "process_first_call": {k_: round(v, 1) for k_, v in process_first.items()},
        "first_over_steady": {"median": round(statistics.median(ratios), 3),
                              "p99": round(ratios[int(0.99 * (len(ratios) - 1))], 3),
                              "max": round(ratios[-1], 3)},
        "host_us_per_first_call": {"median": round(statistics.median(host), 1),
                                   "max": round(host[-1], 1)},
        "per_T": per_T,
        "cuda_graphs": graphs,
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- inverse RoPE
def run_rope(args, rank, local_rank):
    """Inverse rotary embedding + per-head E4M3 quantisation of [T, 32, 128]
    head vectors (max position 8192).  Four copies of the inputs rotate call
    to call, so the 64 MB inputs of T=8192 do not stay in L2."""
    import torch
    import mixture_experts_layer_align_gb300 as moe
    from mixture_experts_layer_align_gb300 import inputs

    if rank != 0:
        return
    moe.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    NH, D, max_pos = 32, 128, 8192
    hbm_peak, _, peak_kind = measured_peaks()
    K = max(args.steps // 10, 20)
    sweep = []
    for T in (1, 64, 1024, 8192):
        cps = [inputs.make_rope_inputs(T, NH, D, max_pos, seed=c, device=dev) for c in range(4)]
        codes = torch.empty(T, NH, D, dtype=torch.uint8, device=dev)
        scales = torch.empty(NH, dtype=torch.float32, device=dev)
        scratch = torch.empty(moe.moe_inv_rope_scratch_size(T, NH, D), dtype=torch.uint8,
                              device=dev)

        def call(i):
            r = cps[i % 4]
            moe.moe_inv_rope_quant_per_head(r.x, r.positions, r.cos, r.sin, codes, scales,
                                            scratch)

        for i in range(max(args.warmup, 3)):
            call(i)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        # eager: K back-to-back calls from Python (small T: paced by the host)
        e0.record()
        for i in range(K):
            call(i)
        e1.record()
        torch.cuda.synchronize()
        eager_us = e0.elapsed_time(e1) * 1e3 / K
        # device time: the same K calls captured once in a CUDA graph, replayed
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            call(0)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(K):
                call(i)
        graph.replay()
        torch.cuda.synchronize()
        reps = 3
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        if moe.moe_check_status(scratch) != 0:
            raise RuntimeError("device status")
        us = e0.elapsed_time(e1) * 1e3 / (K * reps)
        # algorithmic bytes: x once, codes, positions, the cos/sin rows used, scales
        nbytes = T * NH * D * 2 + T * NH * D + T * 4 + T * D * 4 + NH * 4
        sweep.append({"T": T, "us_per_call": round(us, 2), "eager_us_per_call": round(eager_us, 2),
                      "tokens_per_s": round(T / (us * 1e-6), 1),
                      "algorithmic_bytes": nbytes,
                      "hbm_frac": round(nbytes / (us * 1e-6) / 1e9 / hbm_peak, 4)})
    big = sweep[-1]
    line = {"metric": "inverse-RoPE + per-head FP8 quant tokens/s (32 heads x 128)",
            "value": big["tokens_per_s"], "unit": "tokens/s", "steps": K, "warmup": args.warmup,
            "config": {"workload": "x bf16 [T, 32, 128], positions < 8192, fp32 cos/sin tables; "
                                   "one cooperative kernel up to 1216 tokens, else two "
                                   "launches (per-head amax; scale fold + quantise)",
                       "l2": "four input copies rotate call to call",
                       "timing": "us_per_call: K calls captured in one CUDA graph, replayed "
                                 "(device time); eager_us_per_call: the same calls launched "
                                 "from Python one by one"},
            "sweep": sweep,
            "roofline": {"bound": "hbm", "achieved": round(big["algorithmic_bytes"] /
                                                           (big["us_per_call"] * 1e-6) / 1e9, 1),
                         "peak": hbm_peak, "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s",
                         "frac": big["hbm_frac"],
                         "note": "x is read twice (amax pass, quantise pass); the algorithmic "
                                 "bytes count it once"}}
    print(json.dumps(line), flush=True)


def run_tp_sweep(args, rank, local_rank):
    """Tensor-parallel shards over the intermediate size, timed on one GPU.

    For W ranks every rank holds I/W of each expert's gate, up and down
    weights and runs the layer as two library calls with an all-reduce (MAX)
    of one fp32 word between them and an all-reduce (SUM) of the output after.
    Here the W shards run one after another on this GPU: the W gate/up calls
    back to back, the MAX over the W words (not timed), the W down calls back
    to back.  us_per_rank = device time of the two timed phases / W, i.e. what
    one GPU of the W-way group spends in the layer without the collectives.
    Two copies of every shard alternate so that no call finds its weights in
    L2 from the previous one."""
    import torch
    import mixture_experts_layer_align_gb300 as moe
    from mixture_experts_layer_align_gb300 import inputs
    from mixture_experts_layer_align_gb300 import tp

    if rank != 0:
        return
    moe.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    plan = [("decode_e8_top2", (1, 8, 64), (1, 2, 4, 8)),
            ("skewed_e256", (8, 128), (1, 2, 4, 8)),
            ("prefill_e128_uniform", (2048, 8192), (1, 2, 3, 6))]
    if args.workload != "decode_e8_top2":
        plan = [p for p in plan if p[0] == args.workload] or plan
    reps = max(5, min(args.steps, 20))
    rows = []
    for wl, Ts, Ws in plan:
        cfg = inputs.workload(wl)
        H, I, E, k = cfg["H"], cfg["I"], cfg["E"], cfg["top_k"]
        w = inputs.make_weights(H, I, E, cfg["dtype"], seed=0, device=dev)
        for W in Ws:
            if (I // W) % 128 != 0 or I % W != 0:
                continue
            shards = [[tp.shard_weights(w.w13, w.w2, r, W) for r in range(W)] for _ in range(2)]
            for T in Ts:
                a = inputs.make_activations(T, H, E, cfg["routing"], seed=0, device=dev)
                outs = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(W)]
                wss = [moe.alloc_workspace(T, H, I // W, E, k, moe.MOE_DT_FP8_E4M3, dev)
                       for _ in range(W)]
                words = [moe.h_amax_view(ws_) for ws_ in wss]
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
                per = []
                for it in range(reps + 3):
                    sh = shards[it % 2]
                    # hold the GPU for ~1 ms so that the host has enqueued the
                    # phase's calls before its first kernel may start: the
                    # events then see device time, not the host's enqueue rate
                    torch.cuda._sleep(2_000_000)
                    ev[0].record()
                    for r in range(W):
                        moe.moe_fused_forward_gate_up(a.x, a.logits, sh[r][0], sh[r][1],
                                                      w.w13_scale, w.w2_scale, k, True,
                                                      outs[r], wss[r])
                    ev[1].record()
                    m = torch.stack(words).amax()  # the all-reduce (MAX), not timed
                    for wd in words:
                        wd.copy_(m.reshape(1))
                    torch.cuda._sleep(2_000_000)
                    ev[2].record()
                    for r in range(W):
                        moe.moe_fused_forward_down(a.x, a.logits, sh[r][0], sh[r][1],
                                                   w.w13_scale, w.w2_scale, k, True,
                                                   outs[r], wss[r])
                    ev[3].record()
                    torch.cuda.synchronize()
                    if it >= 3:
                        per.append((ev[0].elapsed_time(ev[1]) + ev[2].elapsed_time(ev[3])) * 1e3 / W)
                for ws_ in wss:
                    if moe.moe_check_status(ws_) != 0:
                        raise RuntimeError("device status")
                per.sort()
                row = {"workload": wl, "T": T, "W": W, "I_per_rank": I // W,
                       "us_per_rank": round(per[len(per) // 2], 2)}
                if W == 1:
                    # the same layer as one call (no split, no collectives)
                    ws1 = moe.alloc_workspace(T, H, I, E, k, moe.MOE_DT_FP8_E4M3, dev)
                    out1 = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
                    ws_w = [w, inputs.Weights(w.w13.clone(), w.w2.clone(), w.w13_scale,
                                              w.w2_scale, w.dtype, H, I, E)]

                    def one(i):
                        ww = ws_w[i % 2]
                        moe.moe_fused_forward(a.x, a.logits, ww.w13, ww.w2, ww.w13_scale,
                                              ww.w2_scale, k, True, out=out1, workspace=ws1)
                    us1 = sorted(time_calls(one, 20))
                    row["one_call_us"] = round(us1[len(us1) // 2], 2)
                    del ws_w
                rows.append(row)
            del shards
            torch.cuda.empty_cache()
        del w
        torch.cuda.empty_cache()
    for r_ in rows:
        base = next(x["us_per_rank"] for x in rows
                    if x["workload"] == r_["workload"] and x["T"] == r_["T"] and x["W"] == 1)
        r_["vs_one_rank"] = round(base / r_["us_per_rank"], 3)
        r_["of_ideal"] = round(base / r_["W"] / r_["us_per_rank"], 3)
    print(json.dumps({"metric": "per-rank layer device time, tensor-parallel shards over I "
                                "(ranks run one after another on one GPU)",
                      "unit": "us", "timing": "CUDA events around the W gate/up calls and "
                      "around the W down calls, each phase enqueued behind a ~1 ms GPU sleep "
                      "(the MAX of the h scale word between them and the output all-reduce "
                      "are not timed), median over %d layers; one_call_us: the unsharded "
                      "layer as one call, blocks of back-to-back calls" % reps,
                      "rows": rows}), flush=True)


def run_cta_trace(args, rank, local_rank):
    """Per-CTA %globaltimer stamps of the two expert GEMMs of one call per T,
    relative to the kernel's first CTA entry (us): min/median/max of the
    stamps and the CTAs' exit spread.  Diagnostic only (not a bench line)."""
    if rank != 0:
        return
    import numpy as np
    import torch
    import mixture_experts_layer_align_gb300 as moe
    from mixture_experts_layer_align_gb300 import inputs
    moe.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = inputs.workload(args.workload)
    H, I, E, k = cfg["H"], cfg["I"], cfg["E"], cfg["top_k"]
    dtype = moe.MOE_DT_FP8_E4M3 if cfg["dtype"] == "fp8" else moe.MOE_DT_BF16
    w = inputs.make_weights(H, I, E, cfg["dtype"], seed=0, device=dev)
    w_alt = inputs.Weights(w.w13.clone(), w.w2.clone(), w.w13_scale, w.w2_scale, w.dtype, H, I, E)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {"metric": "per-CTA timeline of the expert GEMMs (us from the kernel's first CTA)",
           "workload": args.workload, "per_T": []}
    for T in tokens_list(args, cfg):
        a = inputs.make_activations(T, H, E, cfg["routing"], seed=0, device=dev)
        ws = moe.alloc_workspace(T, H, I, E, k, dtype, dev)
        ws.zero_()  # trace rows of CTAs that are not launched keep their contents
        for it in range(6):  # the two weight copies alternate: the last call is cold
            ww = w if it % 2 == 0 else w_alt
            moe.moe_fused_forward(a.x, a.logits, ww.w13, ww.w2, ww.w13_scale, ww.w2_scale, k, True,
                                  workspace=ws, debug_flags=moe.MOE_DEBUG_TRACE)
        torch.cuda.synchronize()
        tr = moe.read_trace(ws, T, H, I, E, k, dtype).numpy()
        row = {"T": T}
        for g, name in enumerate(("gate_up", "down")):
            t = tr[g][:min(n_sm, tr.shape[1])].astype(np.float64)
            t = t[t[:, 0] > 0]
            if len(t) == 0:
                continue
            rel = (t - t[:, 0].min()) / 1e3
            row[name] = {"ctas": int(len(t)),
                         "entry_max": round(float(rel[:, 0].max()), 2),
                         "ready_max": round(float(rel[:, 1].max()), 2),
                         "first_median": round(float(np.median(rel[:, 2])), 2),
                         "exit_min_median_max": [round(float(rel[:, 3].min()), 2),
                                                 round(float(np.median(rel[:, 3])), 2),
                                                 round(float(rel[:, 3].max()), 2)]}
        out["per_T"].append(row)
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    rank, local_rank, world = dist_env()
    if args.cta_trace:
        run_cta_trace(args, rank, local_rank)
        return
    if args.rope:
        run_rope(args, rank, local_rank)
        return
    if args.shape_sweep:
        run_shape_sweep(args, rank, local_rank)
        return
    if args.tp_sweep:
        run_tp_sweep(args, rank, local_rank)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, local_rank, world)


if __name__ == "__main__":
    main()
