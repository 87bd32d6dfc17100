#!/usr/bin/env python
"""Benchmark of the fused two-stage MoE expert computation on GB300.

Workload (default): Kimi-K3 TP8-shard decode, a16w4 -- hidden 3584, inter 384,
896 experts, top-16 uniform routing, SiTUv2 (beta 4, linear beta 25), bf16
activations and output, MXFP4 weights ~N(0, 1/sqrt(fan_in)), seed 123.
A step is one moe_forward (sort -> activation encode -> stage 1 -> stage 2 ->
combine) over one batch of T tokens; the headline is T = 64 and the line also
carries the sweep T = 1, 4, 16, 64. Metric: microseconds per call (lower is
better) and the fraction of the HBM roofline.

--impl reference times the CPU fp64 oracle (the correctness reference) on the
host cores on a bounded sample of the same workload.
Replicas only across GPUs: each rank runs its own copy, no collective on the
data path; the timing is the max over ranks.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np
import torch

from quantized_moe_expert_sort_gb300 import inputs

CFG = inputs.CONFIGS["tp8_decode"]
H, I, E, K = CFG.hidden, CFG.inter, CFG.experts, CFG.topk
SEED = CFG.seed
HEAD_T = 64
SWEEP_T = [1, 4, 16, 64]
# MI355X isolated stage1+stage2 us (aiter PR 4463, Performance), TP8 shape, per activation dtype
PAGE_US = {"bf16": {1: 28.3, 4: 42.7, 16: 107.3, 64: 260.6, 256: 374.7, 1024: 422.5, 2048: 651.3, 4096: 1087.3,
                    8192: 1994.4, 16384: 3600.3},
           "fp8": {1: 20.1, 4: 33.7, 16: 93.0, 64: 229.1, 256: 329.8, 1024: 365.7, 2048: 475.8, 4096: 774.4,
                   8192: 1249.4, 16384: 2074.8},
           "fp4": {1: 20.0, 4: 32.9, 16: 91.2, 64: 225.9, 256: 325.3, 1024: 349.9, 2048: 428.2, 4096: 653.2,
                   8192: 1020.3, 16384: 1716.5}}
L2_FLUSH_BYTES = 256 << 20


def select_config(name):
    """Point the module-level workload constants at one of the named configs."""
    global CFG, H, I, E, K, SEED, SWEEP_T, HEAD_T
    CFG = inputs.CONFIGS[name]
    H, I, E, K, SEED = CFG.hidden, CFG.inter, CFG.experts, CFG.topk, CFG.seed
    SWEEP_T = list(CFG.tokens)
    HEAD_T = 64 if name == "tp8_decode" else CFG.tokens[-1]


def workload_text(T):
    c = CFG
    act = "SiTUv2 beta 4 / linear beta 25" if "situv2" in c.acts else "SiLU"
    return ("%s: hidden %d, inter %d, %d experts, top-%d %s routing, %s, a_dtype %s, bf16 out, seed %d, T=%d"
            % (c.notes, c.hidden, c.inter, c.experts, c.topk, c.routing, act, c.a_dtype, c.seed, T))


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, v, device):
    if pg is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job(pg, step_ms, world, device):
    """Replicas: every rank runs the same calls on its own GPU, no collective on the
    data path. Returns (the slowest rank's ms per step, us per call of the whole job =
    that time over the calls all ranks made in it)."""
    ms = max_over_ranks(pg, step_ms, device)
    return ms, ms * 1000.0 / world


def relaunch_as_replicas(n):
    """`--gpus N` without a launcher: run N replicas of this command under torchrun (one
    process per GPU, rendezvous on 127.0.0.1)."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=%d" % n,
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    os.execv(sys.executable, cmd)


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.lines = []
        self.err = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception as e:  # no nvidia-smi
            self.err = str(e)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            if not (t0 - 0.25 <= ts <= t1 + 0.25):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append(dict(sm=float(parts[0]), smax=float(parts[1]), power=float(parts[2]),
                                 hw=parts[4], hwt=parts[5], swt=parts[6], pcap=parts[7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": self.err or "no nvidia-smi samples in the timed window"}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------
def device_weights(device, seed=None, chunk=32):
    """MXFP4 weights of all experts, drawn on the device (seeded per expert) and
    quantised by the library's own GPU quantiser."""
    import quantized_moe_expert_sort_gb300 as moe
    seed = SEED if seed is None else seed
    w13 = torch.empty((E, 2 * I, H // 2), dtype=torch.uint8, device=device)
    w13s = torch.empty((E, 2 * I, H // 32), dtype=torch.uint8, device=device)
    w2 = torch.empty((E, H, I // 2), dtype=torch.uint8, device=device)
    w2s = torch.empty((E, H, I // 32), dtype=torch.uint8, device=device)
    for e in range(E):
        a = inputs.expert_w13(e, H, I, seed, device=device)
        w13[e], w13s[e] = moe.quantize_mxfp4(a)
        b = inputs.expert_w2(e, H, I, seed, device=device)
        w2[e], w2s[e] = moe.quantize_mxfp4(b)
    torch.cuda.synchronize(device)
    return w13, w13s, w2, w2s


def batch(T, device, seed=None):
    seed = SEED if seed is None else seed
    x = inputs.make_x(T, H, seed)
    ids, w = inputs.make_routing(T, E, K, CFG.routing, seed, CFG.zipf_s)
    return x, ids, w, x.to(device), ids.to(device), w.to(device)


def algo_bytes(T, n_active, n_pairs, a_bytes=None):
    """Algorithmic bytes: active experts' weights (fp4 + e8m0), x once, the
    intermediate written and read once, out once (bf16)."""
    if a_bytes is None:
        a_bytes = {"bf16": 2.0, "fp8": 1.0 + 1 / 32, "fp4": 0.5 + 1 / 32}[CFG.a_dtype]
    w13 = n_active * 2 * I * (H // 2 + H // 32)
    w2 = n_active * H * (I // 2 + I // 32)
    x = T * H * 2
    inter = int(n_pairs * I * a_bytes)
    out = T * H * 2
    return dict(stage1=w13 + x + inter, stage2=w2 + inter + out, call=w13 + w2 + x + 2 * inter + out)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# Dense tensor rate of the MMA kind each activation dtype runs on, relative to bf16
# (nominal GB300 dense figures: bf16 2.25, fp8 4.5, fp4 13.5 PFLOP/s). bf16
# activations run kind::mxf4 on six e2m1 code terms: 6 / 6 of the bf16 rate for
# the algorithmic FLOPs.
TENSOR_RATIO = {"bf16": 6.0 / 6.0, "fp8": 2.0, "fp4": 6.0}


def tensor_peak_tflops(a_dtype):
    """(peak TFLOP/s for the algorithmic FLOPs of a_dtype's MMA kind, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops"]) * TENSOR_RATIO[a_dtype], "measured bf16 burst x nominal kind ratio"
    return 1900.0 * TENSOR_RATIO[a_dtype], "fallback bf16 burst x nominal kind ratio"


def kernel_roofline(nbytes, nflops, t_ms, peak_gbs, peak_src, tpeak_tflops, tpeak_src):
    """A kernel against its governing bound: the slower of its algorithmic bytes at the
    HBM peak and its algorithmic FLOPs at the tensor peak of its MMA kind."""
    t = t_ms * 1e-3
    if nflops / (tpeak_tflops * 1e12) > nbytes / (peak_gbs * 1e9):
        achieved, kpeak, unit, src, bound = nflops / t / 1e12, tpeak_tflops, "TFLOP/s", tpeak_src, "tensor"
    else:
        achieved, kpeak, unit, src, bound = nbytes / t / 1e9, peak_gbs, "GB/s", peak_src, "hbm"
    return {"bound": bound, "achieved": round(achieved, 1), "peak": round(kpeak, 1), "peak_source": src,
            "unit": unit, "frac": round(achieved / kpeak, 4)}


def call_roofline(nbytes, nflops, t_ms, peak_gbs, tpeak_tflops):
    """(governing bound, fraction) of a whole call: its roofline time over its measured time."""
    t_bytes, t_flops = nbytes / (peak_gbs * 1e9), nflops / (tpeak_tflops * 1e12)
    return ("tensor" if t_flops > t_bytes else "hbm"), round(max(t_bytes, t_flops) / (t_ms * 1e-3), 4)


def stored_traffic(config, kernel_name, T):
    """DRAM bytes per launch from a committed ncu summary, if it is current."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        ent = d.get("%s_%s_T%d" % (config, kernel_name, T))
        if not ent:
            return None
        import hashlib
        src = os.path.join(ROOT, "quantized_moe_expert_sort_gb300", "csrc", ent["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        return ent["dram_bytes"] if h == ent["source_sha"] else None
    except Exception:
        return None


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args, world, rank, local, pg):
    import quantized_moe_expert_sort_gb300 as moe
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    t_setup = time.time()
    w13, w13s, w2, w2s = device_weights(device)
    ctx = moe.MoE(H, I, E, K, max(SWEEP_T + [args.tokens]) if not args.no_sweep else args.tokens, device=local)
    if args.prepack:  # load-time repack of the stage-2 weights (few-rows path)
        ctx.prepack(w2, w2s, CFG.a_dtype)
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    clean_buf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    class _Flush:
        """Evict L2 between steps: write a buffer larger than L2, then read another one so
        that the write-back of the dirty lines happens here and not inside the next step."""

        @staticmethod
        def zero_():
            flush_buf.zero_()
            clean_buf.sum()

    flush = _Flush()
    stream = torch.cuda.current_stream(device)
    log("setup %.1fs" % (time.time() - t_setup))

    ACT = args.act or CFG.acts[-1]

    def fwd(xd, idd, wd, out):
        ctx.forward(xd, idd, wd, w13, w13s, w2, w2s, ACT, 4.0, 25.0, CFG.a_dtype, out=out)

    def timed_loop(T, steps, warmup):
        x, ids, w, xd, idd, wd = batch(T, device)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        for _ in range(warmup):
            flush.zero_()
            fwd(xd, idd, wd, out)
        torch.cuda.synchronize(device)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        barrier(pg)
        torch.cuda.synchronize(device)
        for i in range(steps):
            flush.zero_()
            starts[i].record(stream)
            fwd(xd, idd, wd, out)
            ends[i].record(stream)
        torch.cuda.synchronize(device)
        barrier(pg)
        ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        return ms, out

    # --- clocks: sampled over a soak + the timed region + a soak
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.5)
    t_soak = time.time()
    soak_until = t_soak + args.soak
    xs_, ids_, ws_, xd_, idd_, wd_ = batch(args.tokens, device)
    out_soak = torch.empty((args.tokens, H), dtype=torch.bfloat16, device=device)
    while time.time() < soak_until:
        for _ in range(20):
            fwd(xd_, idd_, wd_, out_soak)
        torch.cuda.synchronize(device)

    t0 = time.time()
    ms, _ = timed_loop(args.tokens, args.steps, args.warmup)
    t1 = time.time()
    soak_until = time.time() + args.soak
    while time.time() < soak_until:
        for _ in range(20):
            fwd(xd_, idd_, wd_, out_soak)
        torch.cuda.synchronize(device)
    t2 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_soak, t2)

    step_ms_max, value_us = whole_job(pg, statistics.mean(ms), world, device)
    step_ms = statistics.mean(ms)

    # --- per-kernel breakdown (separate, profiled pass)
    ctx.set_profiling(True)
    x, ids, w, xd, idd, wd = batch(args.tokens, device)
    out = torch.empty((args.tokens, H), dtype=torch.bfloat16, device=device)
    per = {}
    for i in range(args.warmup + args.steps):
        flush.zero_()
        fwd(xd, idd, wd, out)
        prof = ctx.read_profile()
        if i >= args.warmup:
            for name, t in prof:
                per.setdefault(name, []).append(t)
    ctx.set_profiling(False)
    per_avg = {k: statistics.mean(v) for k, v in per.items()}
    tile_m = ctx.last_sort()["tile_m"]
    srt = ctx.last_sort()
    n_active = srt["num_active"]
    n_pairs = int((srt["sorted_ids"] < args.tokens * K).sum().item())
    ab = algo_bytes(args.tokens, n_active, n_pairs)
    dominant = max(("stage1", "stage2"), key=lambda k: per_avg.get(k, 0.0))
    peak, peak_kind = measured_peaks()
    tpeak, tpeak_kind = tensor_peak_tflops(CFG.a_dtype)
    flops = 6.0 * n_pairs * H * I
    kflops = {"stage1": 4.0 * n_pairs * H * I, "stage2": 2.0 * n_pairs * H * I, "call": flops}
    # the governing bound of a kernel: the slower of its bytes at the HBM peak and its
    # FLOPs at the tensor peak of the MMA kind it runs
    roof = kernel_roofline(ab[dominant], kflops[dominant], per_avg[dominant], peak, peak_kind, tpeak, tpeak_kind)
    call_bound, call_frac = call_roofline(ab["call"], flops, step_ms, peak, tpeak)
    traffic = stored_traffic(args.config, dominant, args.tokens)

    # --- sweep over the decode token tiers
    sweep = {}
    for T in ([] if args.no_sweep else SWEEP_T):
        ms_t, _ = timed_loop(T, max(10, args.steps // 2), 3)
        sweep[str(T)] = round(statistics.mean(ms_t) * 1000.0, 2)

    # --- end to end through the host-buffer API (pinned host memory)
    x_h = x.pin_memory()
    ids_h = ids.pin_memory()
    w_h = w.pin_memory()
    out_h = torch.empty((args.tokens, H), dtype=torch.bfloat16).pin_memory()
    for _ in range(args.warmup):
        ctx.forward_host(x_h, ids_h, w_h, w13, w13s, w2, w2s, ACT, 4.0, 25.0, CFG.a_dtype, out=out_h)
    e2e = []
    for _ in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize(device)
        ts = time.perf_counter()
        ctx.forward_host(x_h, ids_h, w_h, w13, w13s, w2, w2s, ACT, 4.0, 25.0, CFG.a_dtype, out=out_h)
        e2e.append((time.perf_counter() - ts) * 1e6)
    e2e_us = max_over_ranks(pg, statistics.mean(e2e), device) / world
    st, flags = ctx.get_error()
    if st != 0:
        log("device error flags: %d" % flags)

    result = {
        "metric": "fused-MoE us/call and % roofline vs tokens (3584x384, 896 experts, top-16)",
        "value": round(value_us, 3),
        "unit": "us/call",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms_max, 5),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": (round(value_us / PAGE_US[CFG.a_dtype][args.tokens], 4)
                        if (I == 384 and E == 896 and args.tokens in PAGE_US[CFG.a_dtype]) else None),
        "dtype": {"bf16": "e2m1 x bf16 (bf16 carried as six 1x32-scaled e2m1 terms), fp32 accumulate",
                  "fp8": "e2m1 x e4m3 block-scaled (1x32 e8m0), fp32 accumulate",
                  "fp4": "e2m1 x e2m1 block-scaled (1x32 e8m0), fp32 accumulate"}[CFG.a_dtype],
        "data": "synthetic (seeded; weights drawn on the GPU and MXFP4-quantised by the library)",
        "config": {"workload": workload_text(args.tokens), "name": args.config,
                   "tokens": args.tokens, "a_dtype": CFG.a_dtype, "act": ACT, "path_tile_m": tile_m,
                   "tflops": round(flops / (step_ms * 1e-3) / 1e12, 2),
                   "l2": "flushed before every timed step (256 MB memset, then a 256 MB read so that no dirty "
                         "line is written back inside the step; both outside the events)",
                   "active_experts": n_active, "routed_pairs": n_pairs,
                   "w2_prepacked": bool(args.prepack),
                   "sweep_us_per_call": sweep, "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": dict(roof, kernel=dominant, traffic=traffic, algo_bytes_per_launch=ab[dominant],
                         algo_flops_per_launch=kflops[dominant], call_bound=call_bound, call_frac=call_frac,
                         kernel_ms={k: round(v, 5) for k, v in per_avg.items()}),
        # launches per call, from the launch groups the library recorded (the
        # stand-alone sort is three kernels above 8192 pairs), times the timed calls
        "gpu_launches": sum(3 if name == "sort" and args.tokens * K > 8192 else 1 for name in per_avg) * args.steps,
        "clocks": clocks,
        "e2e": {"value": round(e2e_us, 3), "unit": "us/call",
                "h2d_bytes_per_step": args.tokens * H * 2 + args.tokens * K * 8,
                "d2h_bytes_per_step": args.tokens * H * 2,
                "transfer": "moe_forward_host on pinned host tensors: the kernels read x, ids and weights "
                            "and write out across the host link (no staging copies)"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.tokens, args.cpu_sample)
    tables = [t for t in args.tables.split(",") if t] if args.config == "tp8_decode" else []
    if tables:
        del ctx, w13, w13s, w2, w2s
        torch.cuda.empty_cache()
    if "router" in tables:
        result["router"] = router_row(device, flush, pg, world)
    if "ep" in tables:
        result["ep_emulation"] = ep_rows(device, flush, pg, world)
        select_config(args.config)
    if "prefill" in tables:
        result["prefill"] = prefill_table(device, flush, pg, world)
        select_config(args.config)
    return result


ROUTER_SHAPE = (32768, 896, 16)  # tokens, router logits per token (experts), top-k


def router_row(device, flush, pg, world, steps=10, warmup=3):
    """The top-k softmax router on a prefill-sized batch: us/call and its fraction of
    HBM (logits read once, ids and weights written once), L2 flushed before every call."""
    import quantized_moe_expert_sort_gb300 as moe
    T, Er, Kr = ROUTER_SHAPE
    logits = inputs.make_router_logits(T, Er, SEED).to(device)
    ms = []
    for i in range(warmup + steps):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        moe.route(logits, Kr)
        e.record()
        torch.cuda.synchronize(device)
        if i >= warmup:
            ms.append(s.elapsed_time(e))
    us = max_over_ranks(pg, statistics.mean(ms), device) * 1000.0 / world
    nbytes = T * Er * 4 + T * Kr * 8
    peak, _ = measured_peaks()
    log("router T=%d E=%d K=%d: %.1f us" % (T, Er, Kr, us))
    return {"tokens": T, "experts": Er, "topk": Kr, "us_per_call": round(us, 1), "bound": "hbm",
            "achieved_gbs": round(nbytes / (us * 1e-6) / 1e9, 1), "frac": round(nbytes / (us * 1e-6) / 1e9 / peak, 4)}


EP_RANKS, EP_LOCAL_EXPERTS, EP_TOKENS = 8, 112, (128, 1024)


def ep_rows(device, flush, pg, world, steps=5, warmup=3):
    """Expert-parallel forward of the wide shape (8 ranks x 112 experts, inter 3072, a8 SiTUv2)
    emulated on this GPU: us/call and the whole-call HBM fraction (the active experts'
    weights of all ranks, x, the intermediate, out and the fp8 combine wire)."""
    import quantized_moe_expert_sort_gb300 as moe
    global E
    select_config("ep_wide")
    E = EP_RANKS * EP_LOCAL_EXPERTS
    w13, w13s, w2, w2s = device_weights(device)
    ep = moe.MoEEP(H, I, EP_LOCAL_EXPERTS, EP_RANKS, K, max(EP_TOKENS), device=device.index or 0)
    rows = {}
    peak, _ = measured_peaks()
    for T in EP_TOKENS:
        x = inputs.make_x(T, H, SEED).to(device)
        ids, w = inputs.make_routing(T, E, K, "uniform", SEED)
        ids, w = ids.to(device), w.to(device)
        ms = []
        for i in range(warmup + steps):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            ep.forward(x, ids, w, w13, w13s, w2, w2s, "situv2", 4.0, 25.0, "fp8")
            e.record()
            torch.cuda.synchronize(device)
            if i >= warmup:
                ms.append(s.elapsed_time(e))
        us = max_over_ranks(pg, statistics.mean(ms), device) * 1000.0 / world
        n_active = int(torch.unique(ids).numel())
        ab = algo_bytes(T, n_active, T * K)["call"] + EP_RANKS * T * H * (1 + 1 / 32)  # + the fp8 wire
        rows["T%d" % T] = {"us_per_call": round(us, 1), "bound": "hbm", "call_frac": round(ab / (peak * 1e9) / (us * 1e-6), 4),
                           "active_experts": n_active, "ranks": EP_RANKS}
        log("EP emulation T=%d: %.1f us" % (T, us))
    del ep, w13, w13s, w2, w2s
    torch.cuda.empty_cache()
    return rows


PREFILL_ROWS = [("tp8_a8", 4096, "situv2"), ("ep_wide", 8192, "situv2"), ("tp8_a4_zipf", 32768, "situv2")]


def prefill_table(device, flush, pg, world, steps=5, warmup=3):
    """The prefill workloads: us/call, governing bound and call fraction of the
    roofline (whole call; the slower of its bytes at HBM and its FLOPs at the
    tensor peak of its MMA kind), L2 flushed before every timed call."""
    import quantized_moe_expert_sort_gb300 as moe
    rows = {}
    for name, T, act in PREFILL_ROWS:
        select_config(name)
        w13, w13s, w2, w2s = device_weights(device)
        ctx = moe.MoE(H, I, E, K, T, device=device.index or 0)
        x, ids, w, xd, idd, wd = batch(T, device)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        ms = []
        for i in range(warmup + steps):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            ctx.forward(xd, idd, wd, w13, w13s, w2, w2s, act, 4.0, 25.0, CFG.a_dtype, out=out)
            e.record()
            torch.cuda.synchronize(device)
            if i >= warmup:
                ms.append(s.elapsed_time(e))
        us = max_over_ranks(pg, statistics.mean(ms), device) * 1000.0 / world
        srt = ctx.last_sort()
        n_pairs = int((srt["sorted_ids"] < T * K).sum().item())
        ab = algo_bytes(T, srt["num_active"], n_pairs)
        peak, _ = measured_peaks()
        tpeak, _ = tensor_peak_tflops(CFG.a_dtype)
        t_bytes, t_flops = ab["call"] / (peak * 1e9), 6.0 * n_pairs * H * I / (tpeak * 1e12)
        rows["%s_T%d" % (name, T)] = {"us_per_call": round(us, 1), "bound": "tensor" if t_flops > t_bytes else "hbm",
                                      "call_frac": round(max(t_bytes, t_flops) / (us * 1e-6), 4),
                                      "a_dtype": CFG.a_dtype, "act": act, "path_tile_m": srt["tile_m"]}
        log("prefill %s T=%d: %.1f us" % (name, T, us))
        del ctx, w13, w13s, w2, w2s, out
        torch.cuda.empty_cache()
    return rows


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------
def _oracle_inputs(T, sample):
    import oracle
    x = inputs.make_x(T, H, SEED)
    ids, w = inputs.make_routing(T, E, K, CFG.routing, SEED, CFG.zipf_s)
    sub = np.arange(min(sample, T), dtype=np.int32)
    experts = np.unique(ids.numpy()[sub])
    w13 = np.zeros((E, 2 * I, H // 2), np.uint8)
    w13s = np.zeros((E, 2 * I, H // 32), np.uint8)
    w2 = np.zeros((E, H, I // 2), np.uint8)
    w2s = np.zeros((E, H, I // 32), np.uint8)
    for e in experts:
        w13[e], w13s[e] = oracle.quantize_weights(inputs.expert_w13(int(e), H, I, SEED).numpy())
        w2[e], w2s[e] = oracle.quantize_weights(inputs.expert_w2(int(e), H, I, SEED).numpy())
    xb = x.view(torch.int16).numpy().astype(np.uint16)
    return xb, ids.numpy(), w.numpy(), w13, w13s, w2, w2s, sub


def _oracle_step(args_in):
    import oracle
    xb, ids, w, w13, w13s, w2, w2s, sub = args_in
    t = time.perf_counter()
    oracle.moe_forward(xb, ids, w, w13, w13s, w2, w2s, CFG.acts[-1], 4.0, 25.0, CFG.a_dtype, subset=sub)
    return time.perf_counter() - t


def cpu_baseline(T, sample):
    import oracle
    data = _oracle_inputs(T, sample)
    dt = _oracle_step(data)
    n = len(data[-1])
    return {"value": round(dt / n * T * 1e6, 1), "unit": "us/call", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "%d of the %d tokens of the T=%d batch (all their %d routed pairs), one timed oracle call, "
                      "scaled by T/%d" % (n, T, T, n * K, n)}


def run_reference(args, world, rank, local, pg):
    import oracle
    if rank != 0:
        return None
    data = _oracle_inputs(args.tokens, args.ref_sample)
    n = len(data[-1])
    for _ in range(args.warmup):
        _oracle_step(data)
    ts = [_oracle_step(data) for _ in range(args.steps)]
    us = statistics.mean(ts) / n * args.tokens * 1e6
    sample = ("%d of the %d tokens per step (all their routed pairs), scaled by T/%d; fp64 CPU oracle"
              % (n, args.tokens, n))
    return {
        "impl": "reference",
        "metric": "fused-MoE us/call and % roofline vs tokens (3584x384, 896 experts, top-16)",
        "value": round(us, 1), "unit": "us/call", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(us / 1000.0, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; weights quantised by the oracle)",
        "config": {"workload": workload_text(args.tokens), "name": args.config, "tokens": args.tokens},
        "cpu_baseline": {"value": round(us, 1), "unit": "us/call", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(us, 1), "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="tp8_decode", choices=sorted(inputs.CONFIGS))
    ap.add_argument("--tokens", type=int, default=None)
    ap.add_argument("--act", default=None, choices=["silu", "situv2"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of untimed steps around the timed region")
    ap.add_argument("--cpu-sample", type=int, default=16)
    ap.add_argument("--ref-sample", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prepack", action="store_true", help="stage 2 reads a prepacked copy of w2 (moe_prepack)")
    ap.add_argument("--tables", default="router,ep,prefill",
                    help="extra rows of the default workload's line: router, ep (expert-parallel emulation), "
                         "prefill; empty for none")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    select_config(args.config)
    if args.tokens is None:
        args.tokens = HEAD_T
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        relaunch_as_replicas(args.gpus)
    world, rank, local, pg = dist_setup()
    if world != args.gpus:
        ap.error("--gpus %d but %d ranks were launched" % (args.gpus, world))
    if args.impl == "reference":
        res = run_reference(args, world, rank, local, pg)
    else:
        res = run_ours(args, world, rank, local, pg)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
