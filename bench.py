"""Benchmark of the GB300 quantized MoE layer.

Default workload: the GLM-5.2-shaped decode layer (hidden 6144, expert FFN
2048, 256 routed experts top-8 + 1 shared expert, int4 experts all resident in
HBM), one token per forward, fresh N(0,1) activations every forward.  One
"step" is one full layer forward (quantise, route, dispatch, gate/up, down,
combine).  L2 is flushed (a 512 MiB write) between timed steps, outside the
timed region, so the shared expert and router weights are re-read from HBM
like in a real multi-layer decode.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode|verify|prefill|sweep]
                  [--path auto|gemv|gemm] [--sub verify,prefill,sweep|none]
  python bench.py --impl reference ...   # the CPU oracle as the reference arm

The default decode run also measures, in the same process and printed as
sub-records of the one JSON line: "verify" (4 correlated tokens per forward on
the same resident weights), "prefill" (2048 tokens, Zipf-skewed routing, the
same weights) and "sweep" (8 stacked layers at batches 1, 8, 32 and 128).
Each sub-record carries its own roofline, clocks, e2e and cpu_baseline.

The 2048-token prefill workload runs the grouped tensor-core GEMM (auto path);
its roofline line is the gate/up GEMM's FLOP/s against the measured bf16 dense
peak (int4 and int8 codes are exact in bf16), and "tops_layer" is the whole
layer's integer multiply-add rate (2 ops per MAC).

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE layer tok/s"
EXPERT_BYTES_PER = None  # filled per workload: int4 bytes + row scales of one expert


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# dominant kernels, from the ncu captures summarised under profiles/.  A value
# applies only while the kernel's sources hash to the same SHA-256 as when it
# was captured, and only to the workloads whose launches move the same bytes
# as the captured one; otherwise the roofline's traffic is null.
CSRC = os.path.join(ROOT, "int4_routed_expert_f32_gb300", "csrc")
TRAFFIC = {
    "k_experts": {
        "sources": ["k_experts.cu", "coli_common.cuh", "tma.cuh", "coli_internal.h"],
        "sha256": "c074085f2c6edf20921080096aa39e35c1d4c78b0e6aec9036e00b4fa596fbc1",
        "bytes_per_launch": 171017472,   # the median of three launches: 170.97 MB read + 0.05 MB written
        # a decode forward streams 8 routed + 1 shared expert; the capture ran
        # the decode workload itself
        "workloads": ("decode", "profile"),
        "capture": "profiles/decode_layer_launches.md",
    },
    "k_gemm_gateup": {
        "sources": ["k_gemm.cu", "coli_common.cuh", "tma.cuh", "coli_internal.h"],
        "sha256": "37a282ced7fc5c0eb9521ca1ba4e922b36949240e2499bc3a5b3829b9671a378",
        "bytes_per_launch": 3655883264,  # the median of three launches: 3541.60 MB read + 114.28 MB written
        "workloads": ("prefill",),
        "capture": "profiles/prefill_layer_launches.md",
    },
}


def kernel_traffic(kernel: str, workload: str):
    t = TRAFFIC.get(kernel)
    if t is None or workload not in t["workloads"]:
        return None
    import hashlib
    h = hashlib.sha256()
    for f in t["sources"]:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return t["bytes_per_launch"] if h.hexdigest() == t["sha256"] else None


def max_over_ranks(value: float, world: int, device: str = "cuda") -> float:
    """The slowest rank's figure: whole-job timings take the max over ranks
    (each rank times its own replica of the workload)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1910.0)), "measured"
    return 6800.0, 1900.0, "fallback"


def expert_bytes(wl, wbits=4):
    """Algorithmic bytes of one expert: its weight container (3*F*H*wbits/8)
    plus its F32 row scales."""
    return 3 * wl.ffn * wl.hidden * wbits // 8 + 4 * wl.expert_scales


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"coli_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            # nvidia-smi's start-up (NVML initialisation) can hold up
            # CUDA calls of this process for seconds: let it finish, i.e. wait
            # for its first sample, before the timed region begins
            t0 = time.perf_counter()
            while time.perf_counter() - t0 < 15.0 and self.proc.poll() is None:
                if os.path.getsize(self.path) > 0:
                    break
                time.sleep(0.05)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- #
def oracle_baseline(wl, n_forwards: int, seed_base: int = 900000, max_tokens: int = 0,
                    min_seconds: float = 0.0, threads: int = 0, wbits: int = 4):
    """Time the CPU oracle on a bounded sample of the workload (forwards of the
    same shape, or the first `max_tokens` tokens of each when that is set: the
    oracle's cost is per token and expert, so a token subset keeps its rate);
    the timed loop cycles over the sample's inputs until at least `min_seconds`
    have passed; returns (tok/s, threads, sample description)."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from helpers import OracleLayer
    oracle.build()
    oracle.set_threads(threads)
    try:
        return _oracle_baseline(oracle, OracleLayer, wl, n_forwards, seed_base, max_tokens, min_seconds, wbits)
    finally:
        oracle.set_threads(0)


def _oracle_baseline(oracle, OracleLayer, wl, n_forwards, seed_base, max_tokens, min_seconds, wbits=4):
    xs = [synth.activations(wl, seed_base + i) for i in range(n_forwards)]
    if max_tokens > 0:
        xs = [x[:max_tokens] for x in xs]
    if wl.layers > 1:
        # the stacked layers: x <- x + layer_l(x); experts are packed lazily
        # inside the timed loop's first pass, so time a second pass
        refs = [OracleLayer(wl, layer=l) for l in range(wl.layers)]

        def stack(x):
            for r in refs:
                x = (x + r.forward(oracle.rmsnorm(x))).astype(np.float32)
            return x

        for x in xs:
            stack(x)
        t0 = time.perf_counter()
        for x in xs:
            stack(x)
        dt = time.perf_counter() - t0
        toks = n_forwards * xs[0].shape[0]
        return toks / dt, oracle.num_threads(), (f"{n_forwards} passes x {xs[0].shape[0]} token(s) through the "
                                                 f"{wl.layers}-layer {wl.name} stack ({dt:.1f} s)")
    ref = OracleLayer(wl, wbits=wbits)
    # pack the experts the sample touches before timing (the oracle's converter)
    for x in xs:
        idx, _ = oracle.route(x, ref.W, ref.b, wl.top_k, wl.routed_scale)
        for e in set(int(v) for v in idx.ravel()):
            ref.expert(e)
    t0 = time.perf_counter()
    done = 0
    while True:
        ref.forward(xs[done % len(xs)])
        done += 1
        dt = time.perf_counter() - t0
        if done >= n_forwards and dt >= min_seconds:
            break
    n_forwards = done
    toks = n_forwards * xs[0].shape[0]
    sub = f" (first {xs[0].shape[0]} of {wl.n_tok} tokens)" if xs[0].shape[0] < wl.n_tok else ""
    return toks / dt, oracle.num_threads(), (f"{n_forwards} forwards x {xs[0].shape[0]} tokens of the {wl.name} "
                                             f"workload{sub} ({dt:.1f} s)")


CPU_SAMPLE_TOKENS = {"prefill": 24, "sweep": 1}   # bounded oracle sample per forward (tokens)


def cpu_baseline_line(wl, n_forwards: int, min_seconds: float, single_thread: bool = True, wbits: int = 4):
    """The oracle on all of the host's cores, plus (optionally) a shorter
    single-thread sample, with the host's machine type."""
    import platform
    mt = CPU_SAMPLE_TOKENS.get(wl.name, 0)
    tps, cores, sample = oracle_baseline(wl, n_forwards, max_tokens=mt, min_seconds=min_seconds, wbits=wbits)
    rec = {"value": tps, "unit": "tok/s", "cores": cores, "kind": "oracle", "sample": sample,
           "machine": platform.machine()}
    if single_thread:
        st_tps, _, st_sample = oracle_baseline(wl, max(1, n_forwards // 4), max_tokens=mt,
                                               min_seconds=min_seconds / 3.0, threads=1)
        rec["single_thread"] = {"value": st_tps, "unit": "tok/s", "sample": st_sample}
    return rec


def run_reference(args):
    """Reference arm: the CPU oracle (plain C, OpenMP over independent outputs)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = synth.WORKLOADS[args.workload]
    n = max(1, args.steps if args.steps <= 50 else 20)
    if wl.n_tok > 64:
        n = min(n, 3)
    mt = CPU_SAMPLE_TOKENS.get(wl.name, 0)
    for _ in range(min(args.warmup, 1)):
        oracle_baseline(wl, 1, seed_base=800000, max_tokens=mt)
    tps, cores, sample = oracle_baseline(wl, n, max_tokens=mt)
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tok/s", "n_gpus": args.gpus,
        "steps": n, "warmup": args.warmup,
        "ms_per_step": 1000.0 * (wl.batches[0] if wl.layers > 1 else wl.n_tok) / tps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int4xint8->f32",
        "data": "synthetic", "config": workload_config(wl),
        "cpu_baseline": {"value": tps, "unit": "tok/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": tps, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(wl, wbits=4):
    if wl.layers > 1:
        return {"workload": f"{wl.name}: {wl.layers} stacked GLM-5.2-shaped MoE layers (hidden {wl.hidden}, "
                            f"expert FFN {wl.ffn}, {wl.n_experts} experts top-{wl.top_k} + 1 shared), residual "
                            f"add between layers, batches {list(wl.batches)}; value = tokens/s through the "
                            f"stack at batch {wl.batches[0]}",
                "layers": wl.layers, "batches": list(wl.batches), "hidden": wl.hidden, "ffn": wl.ffn,
                "n_experts": wl.n_experts, "top_k": wl.top_k,
                "weights": f"int4 + F32 row scales, {wl.layers} x {wl.n_experts + 1} experts resident in HBM",
                "l2": "flushed between timed steps (512 MiB write, outside the timed region)"}
    return {"workload": f"{wl.name}: GLM-5.2-shaped MoE layer, hidden {wl.hidden}, expert FFN {wl.ffn}, "
                        f"{wl.n_experts} routed experts top-{wl.top_k} + 1 shared, {wl.n_tok} token(s) per forward",
            "hidden": wl.hidden, "ffn": wl.ffn, "n_experts": wl.n_experts, "top_k": wl.top_k,
            "tokens_per_forward": wl.n_tok,
            "weights": f"int{wbits} + F32 row scales, all experts resident in HBM",
            "l2": "flushed between timed steps (512 MiB write, outside the timed region)"}


def _setup(args):
    """Build the library, set the device and (torchrun) the process group."""
    import torch
    import torch.distributed as dist

    import __graft_entry__
    __graft_entry__._builder().build()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    return world, rank, local


def measure_layer(args, wl, L, router_b, world, rank, local, cpu_seconds, single_thread_cpu=True, wbits=4):
    """One layer workload on resident weights L (router bias `router_b`;
    weight container `wbits`): the timed forwards, the dominant kernel timed
    alone, the end-to-end host-I/O forwards and the CPU oracle sample;
    returns the record."""
    import torch

    import int4_routed_expert_f32_gb300 as coli

    T = wl.n_tok
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, T)
    coli.set_weight_bits(wbits)
    path = {"auto": coli.PATH_AUTO, "gemv": coli.PATH_GEMV, "gemm": coli.PATH_GEMM}[args.path]
    coli.set_path(path)
    use_gemm = path == coli.PATH_GEMM or (path == coli.PATH_AUTO and
                                          coli.auto_uses_gemm(T, wl.top_k, wl.n_experts))
    n_total = args.warmup + args.steps
    # distinct inputs per step (cycled for large batches to bound host time and memory)
    n_in = n_total if T <= 64 else min(n_total, 8)
    xs = torch.from_numpy(np.stack([synth.activations(wl, 10_000 + rank * 100_000 + i)
                                    for i in range(n_in)])).cuda()
    out = torch.empty((T, wl.hidden), dtype=torch.float32, device="cuda")
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()

    # union of routed experts per step (bookkeeping for weight bytes; not timed)
    unions = []
    for i in range(n_total):
        idx, _ = coli.dbg_route(xs[i % n_in], L["router_w"], router_b, wl.top_k)
        unions.append(len(set(idx.cpu().numpy().ravel().tolist())))
    torch.cuda.synchronize()

    def fwd(i):
        coli.layer_forward(xs[i % n_in], L["router_w"], router_b, L["expert_w4"], L["expert_rs"],
                           L["shared_w4"], L["shared_rs"], out=out)

    for i in range(args.warmup):
        flush.zero_()
        fwd(i)
    torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    coli.launch_count()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for s in range(args.steps):
            flush.zero_()
            ev[s][0].record(st)
            fwd(args.warmup + s)
            ev[s][1].record(st)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches = coli.launch_count()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(float(sum(step_ms)), world)

    # dominant-kernel timing: the library records events around the expert
    # kernel; they serialise it behind routing, so this is a separate pass over
    # the same inputs
    coli.timing_read()
    coli.timing_enable(True)
    for s in range(args.steps):
        flush.zero_()
        fwd(args.warmup + s)
    torch.cuda.synchronize()
    coli.timing_enable(False)
    k_ms, k_n = coli.timing_read()
    status = coli.get_device_status()

    # end to end through the host-I/O entry point: pinned host x in, host out
    n_h = args.steps if T <= 64 else min(args.steps, 4)
    xh = torch.from_numpy(np.stack([synth.activations(wl, 20_000 + i) for i in range(n_h)]))
    xh = xh.pin_memory()
    oh = torch.empty((T, wl.hidden), dtype=torch.float32).pin_memory()
    # the public call a serving loop makes: a layer prepared once, then one
    # host-I/O forward per step
    layer = coli.PreparedLayer(L["router_w"], router_b, L["expert_w4"], L["expert_rs"], L["shared_w4"],
                               L["shared_rs"])
    xh_steps = [xh[i] for i in range(n_h)]
    for i in range(min(args.warmup, 5)):
        layer.forward_hostio(xh_steps[i % n_h], oh)
    e2e_s = 0.0
    gc.disable()      # no collector pause inside the host-timed steps
    for s in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        layer.forward_hostio(xh_steps[s % n_h], oh)
        e2e_s += time.perf_counter() - t0
    gc.enable()
    e2e_s = max_over_ranks(e2e_s, world)
    coli.set_path(coli.PATH_AUTO)
    coli.set_weight_bits(4)

    hbm_peak, bf16_peak, peak_kind = peaks()
    ub = np.array(unions[args.warmup:], dtype=np.float64)
    bytes_per_fwd = float(np.mean((ub + 1) * expert_bytes(wl, wbits)))
    k_avg_ms = k_ms / max(k_n, 1)
    value = world * args.steps * T / (total_ms * 1e-3)
    # multiply-adds of one forward: (T*k routed + T shared) rows x (2F*H + H*F)
    macs_gu = (T * wl.top_k + T) * 2 * wl.ffn * wl.hidden
    macs_layer = (T * wl.top_k + T) * 3 * wl.ffn * wl.hidden
    if use_gemm:
        achieved = 2.0 * macs_gu / (k_avg_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
                    "frac": achieved / bf16_peak, "traffic": kernel_traffic("k_gemm_gateup", wl.name),
                    "traffic_unit": "DRAM bytes per launch",
                    "kernel": "k_gemm<gate/up> (tcgen05 bf16 on exact int codes, SiLU*up + Q8_0 of h fused), "
                              "timed alone",
                    "algorithmic_flops_per_launch": 2.0 * macs_gu,
                    "avg_launch_ms": k_avg_ms, "peak_kind": f"{peak_kind} bf16_tflops (burst)"}
    else:
        achieved = bytes_per_fwd / (k_avg_ms * 1e-3) / 1e9
        traffic = kernel_traffic("k_experts", wl.name) if wbits == 4 else None
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved / hbm_peak, "traffic": traffic, "traffic_unit": "bytes per launch",
                    "kernel": "k_experts (gate/up + SiLU*up requant + down + combine), timed alone",
                    "algorithmic_bytes_per_launch": bytes_per_fwd,
                    "avg_launch_ms": k_avg_ms, "peak_kind": f"{peak_kind} hbm_gbs"}
    step_s = total_ms / args.steps * 1e-3
    rec = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": f"int{wbits}xint8->f32", "data": "synthetic",
        "config": workload_config(wl, wbits),
        "roofline": roofline,
        "expert_path": "gemm" if use_gemm else "gemv",
        "weight_gbs_layer": bytes_per_fwd / step_s / 1e9,
        "tops_layer": 2.0 * macs_layer / step_s / 1e12,
        # whole-layer bound: max(weight bytes / HBM peak, ops / bf16 peak) over the step time
        "layer_roofline_frac": max(bytes_per_fwd / (hbm_peak * 1e9), 2.0 * macs_layer / (bf16_peak * 1e12))
                               / step_s,
        "union_mean": float(np.mean(ub)),
        "e2e": {"value": world * args.steps * T / e2e_s, "unit": "tok/s",
                "h2d_bytes_per_step": T * wl.hidden * 4, "d2h_bytes_per_step": T * wl.hidden * 4},
        "gpu_launches": launches,
        "clocks": clocks.summary(),
        "device_status": status,
        "step_ms_p10_p50_p90": [float(np.percentile(step_ms, q)) for q in (10, 50, 90)],
    }
    if use_gemm:
        rec["layer_roofline_terms_ms"] = {"weights_at_hbm_peak": bytes_per_fwd / (hbm_peak * 1e9) * 1e3,
                                          "ops_at_bf16_peak": 2.0 * macs_layer / (bf16_peak * 1e12) * 1e3}
    else:
        # reference for the expert kernel: one bare read of the same number of
        # bytes in one launch (coli_moe_dbg_stream_read: bulk copies into the
        # same per-block rings, no arithmetic), L2 flushed before each pass,
        # i.e. what a single read of that much data reaches on this GPU, ramp
        # and tail included
        nb = int(bytes_per_fwd) // 16 * 16
        buf = torch.ones(nb // 4, dtype=torch.int32, device="cuda")
        sink = torch.empty(1, dtype=torch.int64, device="cuda")
        fl = []
        for i in range(25):
            flush.zero_()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(st)
            coli.dbg_stream_read(buf, sum_out=sink)
            b_.record(st)
            fl.append((a_, b_))
        torch.cuda.synchronize()
        fms = float(np.mean([a_.elapsed_time(b_) for a_, b_ in fl[5:]]))
        rec["stream_floor"] = {"bytes": nb, "ms": fms, "gbs": nb / (fms * 1e-3) / 1e9,
                               "frac_of_hbm": nb / (fms * 1e-3) / 1e9 / hbm_peak,
                               "expert_kernel_vs_floor": fms / k_avg_ms,
                               "what": "coli_moe_dbg_stream_read: one launch reading the forward's algorithmic "
                                       "bytes through bulk copies into per-block shared-memory rings, no "
                                       "arithmetic, L2 flushed, mean of 20"}
        del buf, sink
    if rank == 0 and not args.no_cpu_baseline:
        nf = args.cpu_forwards if T <= 64 else 1
        rec["cpu_baseline"] = cpu_baseline_line(wl, nf, cpu_seconds, single_thread=single_thread_cpu, wbits=wbits)
    del xs, out, flush
    return rec


def measure_tier(args, wl, L, router_b, world, rank, local, n_slots=64):
    """The decode layer with its routed experts in host memory (page-locked)
    and an LRU cache of n_slots experts in HBM (coli_moe_tier_forward): every
    step routes, copies in the experts it misses and runs the expert kernel on
    the slots.  Reports tok/s, the hit rate and the host-to-HBM copy rate."""
    import torch

    import int4_routed_expert_f32_gb300 as coli

    T = wl.n_tok
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, T)
    hw = L["expert_w4"].cpu().pin_memory()
    hrs = L["expert_rs"].cpu().pin_memory()
    coli.tier_configure(n_slots)
    # every step synchronises the host once, so a single host stall weighs on
    # a short run: time at least 200 steps (and at least 20 warm-up steps, so
    # that the cache is full)
    steps = max(args.steps, 200)
    warm = max(args.warmup, 20)
    n_total = warm + steps
    xs = torch.from_numpy(np.stack([synth.activations(wl, 50_000 + rank * 100_000 + i)
                                    for i in range(n_total)])).cuda()
    out = torch.empty((T, wl.hidden), dtype=torch.float32, device="cuda")
    for i in range(warm):
        coli.tier_forward(xs[i], L["router_w"], router_b, hw, hrs, L["shared_w4"], L["shared_rs"], out=out)
    torch.cuda.synchronize()
    h0, m0, b0, _ = coli.tier_stats()
    step_s = []
    with ClockSampler(local) as clocks:
        t0 = time.perf_counter()
        for s_ in range(steps):
            t1 = time.perf_counter()
            coli.tier_forward(xs[warm + s_], L["router_w"], router_b, hw, hrs, L["shared_w4"],
                              L["shared_rs"], out=out)
            torch.cuda.synchronize()
            step_s.append(time.perf_counter() - t1)
        dt = max_over_ranks(time.perf_counter() - t0, world)
    h1, m1, b1, res = coli.tier_stats()
    status = coli.get_device_status()
    coli.tier_release()
    hits, misses, nbytes = h1 - h0, m1 - m0, b1 - b0
    return {"value": world * steps * T / dt, "unit": "tok/s", "steps": steps, "warmup": warm,
            "ms_per_step": dt / steps * 1e3,
            "step_ms_p10_p50_p90": [float(np.percentile(step_s, q)) * 1e3 for q in (10, 50, 90)],
            "config": {"workload": f"decode layer (hidden {wl.hidden}, expert FFN {wl.ffn}, {wl.n_experts} experts "
                                   f"top-{wl.top_k} + 1 shared), routed experts in page-locked host memory, "
                                   f"LRU cache of {n_slots} experts in HBM, 1 token per forward, fresh activations",
                       "hbm_slots": n_slots, "host_expert_bytes": int(hw.numel())},
            "hit_rate": hits / max(hits + misses, 1), "misses_per_step": misses / steps,
            "h2d_gbs": nbytes / dt / 1e9, "h2d_bytes_per_step": nbytes / steps,
            "resident_experts": res, "clocks": clocks.summary(), "device_status": status,
            "timing": "host wall clock around the steps (each step synchronises once, after routing)"}


# sub-records of the default decode run: the verify batch and the prefill on
# the same resident weights, the decode layer with int8-container experts, the
# decode layer with its experts in host memory, and the stacked-layer sweep
SUB_WORKLOADS = ("verify", "prefill", "decode_int8", "tier", "stream", "sweep")


def measure_stream(n_bytes: int, big_bytes: int = 1200 << 20):
    """The single-launch read rate of this GPU: coli_moe_dbg_stream_read over
    n_bytes (the decode forward's algorithmic bytes) for a grid of copy
    sizes, ring depths and blocks per SM, and over big_bytes for a few, each
    the median of 5 launches (after 2) with L2 flushed before each.  The best
    single-launch read of n_bytes is the ceiling of any one-launch kernel that
    reads them; the large read shows the per-launch cost that sets it."""
    import torch

    import int4_routed_expert_f32_gb300 as coli

    hbm_peak, _, peak_kind = peaks()
    smem_sm = torch.cuda.get_device_properties(0).shared_memory_per_multiprocessor
    buf = torch.ones(big_bytes // 4, dtype=torch.int32, device="cuda")
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    sink = torch.empty(1, dtype=torch.int64, device="cuda")
    st = torch.cuda.current_stream()

    def timed(nb, chunk, stages, bps):
        ts = []
        for i in range(12):
            flush.zero_()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(st)
            coli.dbg_stream_read(buf, n_bytes=nb, sum_out=sink, chunk=chunk, stages=stages, blocks_per_sm=bps)
            b_.record(st)
            ts.append((a_, b_))
        torch.cuda.synchronize()
        # the mean: this GPU's event timestamps step by about 2 us, so a
        # median of a few launches lands on one of those steps
        ms = float(np.mean([a_.elapsed_time(b_) for a_, b_ in ts[2:]]))
        gbs = nb / (ms * 1e-3) / 1e9
        return {"chunk": chunk, "stages": stages, "blocks_per_sm": bps, "us": round(ms * 1e3, 2),
                "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_peak, 4)}

    nb = n_bytes // 16 * 16
    grid = []
    for chunk in (8192, 16384, 32768):
        for stages in (2, 3, 4, 6):
            for bps in (1, 2, 3, 4, 6):
                if bps * (chunk * stages + 2048) > smem_sm or chunk * stages > 200 * 1024:
                    continue
                grid.append(timed(nb, chunk, stages, bps))
    best = max(grid, key=lambda r: r["gbs"])
    default = next(r for r in grid if (r["chunk"], r["stages"], r["blocks_per_sm"]) == (16384, 3, 4))
    big = [timed(big_bytes, c, s_, b) for c, s_, b in ((16384, 3, 4), (32768, 2, 3), (32768, 3, 2))]
    del buf, flush, sink
    torch.cuda.empty_cache()
    return {"bytes": nb, "peak": hbm_peak, "peak_kind": f"{peak_kind} hbm_gbs", "best": best,
            "expert_kernel_arrangement": default, "configs": grid,
            "large_read": {"bytes": big_bytes, "configs": big},
            "what": "coli_moe_dbg_stream_read: one launch, bulk copies into per-block shared-memory rings, no "
                    "arithmetic; CUDA events around the launch, L2 flushed before each, mean of 10"}


def run(args):
    import torch

    from synth.device import build_device_layer

    world, rank, local = _setup(args)
    wl = synth.WORKLOADS[args.workload]
    t_build = time.perf_counter()
    L = build_device_layer(wl)
    t_build = time.perf_counter() - t_build
    _, b = synth.router(wl)
    line = measure_layer(args, wl, L, torch.from_numpy(b).cuda(), world, rank, local, args.cpu_seconds)
    line["setup_s"] = round(t_build, 1)
    subs = [w for w in args.sub.split(",") if w] if args.sub != "none" else []
    bad = [w for w in subs if w not in SUB_WORKLOADS]
    if bad:
        raise SystemExit(f"unknown sub-record(s) {bad}; choose from {SUB_WORKLOADS}")
    subs = sorted(set(subs), key=SUB_WORKLOADS.index)     # the sweep (which frees L) last
    if subs and wl.name == "decode":
        for name in subs:
            t0 = time.perf_counter()
            if name == "sweep":
                del L
                torch.cuda.empty_cache()
                rec = measure_sweep(args, world, rank, local, args.cpu_seconds / 2)
            elif name == "stream":
                rec = measure_stream(int(line["roofline"]["algorithmic_bytes_per_launch"]))
            elif name == "tier":
                rec = measure_tier(args, wl, L, torch.from_numpy(b).cuda(), world, rank, local)
            elif name == "decode_int8":
                L8 = build_device_layer(wl, wbits=8)
                rec = measure_layer(args, wl, L8, torch.from_numpy(b).cuda(), world, rank, local,
                                    args.cpu_seconds / 2, single_thread_cpu=False, wbits=8)
                del L8
                torch.cuda.empty_cache()
            else:
                swl = synth.WORKLOADS[name]
                _, sb = synth.router(swl)          # same weights; prefill's bias is Zipf-skewed
                rec = measure_layer(args, swl, L, torch.from_numpy(sb).cuda(), world, rank, local,
                                    args.cpu_seconds / 2, single_thread_cpu=False)
            for k in ("metric", "n_gpus", "higher_is_better", "scaling", "vs_baseline", "dtype", "data",
                      "warmup"):
                rec.pop(k, None)
            rec["wall_s"] = round(time.perf_counter() - t0, 1)
            line[name] = rec
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def measure_sweep(args, world, rank, local, cpu_seconds):
    """Multi-layer decode sweep: the stacked layers (residual add fused into
    each layer's combine) at each batch size; one step = one pass through all
    layers.  `value` is tokens/s through the stack at batch 1; the per-batch
    figures are in "sweep"; the roofline is the expert kernel's weight
    stream at batch 1 (every layer's launch, timed alone)."""
    import torch

    import int4_routed_expert_f32_gb300 as coli
    from synth.device import build_device_layer

    wl = synth.WORKLOADS["sweep"]
    t_build = time.perf_counter()
    layers = [build_device_layer(wl, layer=l) for l in range(wl.layers)]
    t_build = time.perf_counter() - t_build
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, max(wl.batches))
    coli.set_path(coli.PATH_AUTO)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()
    hbm_peak, _, peak_kind = peaks()
    per_b = []
    launches_total = 0
    kernel_b1 = None
    with ClockSampler(local) as clocks:
        for B in wl.batches:
            n_in = 4
            xs = [torch.from_numpy(synth.activations(wl, 30_000 + rank * 100 + i, n_tok=B)).cuda()
                  for i in range(n_in)]
            bufs = [torch.empty((B, wl.hidden), dtype=torch.float32, device="cuda") for _ in range(2)]

            def stack(x0, record_unions=None, record_idx=None, prefetch=True):
                x = x0
                for l, L in enumerate(layers):
                    if record_unions is not None:
                        xn = coli.dbg_rmsnorm(x)    # the layer routes its normalised input
                        idx, _ = coli.dbg_route(xn, L["router_w"], L["router_b"], wl.top_k)
                        idx = idx.cpu().numpy()
                        record_unions.append(len(set(idx.ravel().tolist())))
                        if record_idx is not None:
                            record_idx.append(idx)
                    out = bufs[l & 1]
                    nxt = layers[l + 1] if prefetch and l + 1 < len(layers) else None
                    if nxt is not None:
                        # layer-ahead L2 prefetch of the next layer's router and shared expert
                        coli.layer_forward_residual_prefetch(x, L["router_w"], L["router_b"], L["expert_w4"],
                                                             L["expert_rs"], L["shared_w4"], L["shared_rs"],
                                                             nxt["router_w"], nxt["shared_w4"], out=out)
                    else:
                        coli.layer_forward_residual(x, L["router_w"], L["router_b"], L["expert_w4"],
                                                    L["expert_rs"], L["shared_w4"], L["shared_rs"], out=out)
                    x = out
                return x

            unions = {}
            overlaps = []
            for i in range(n_in):
                u, ids = [], []
                stack(xs[i], u, ids)
                unions[i] = u
                for l in range(1, len(ids)):
                    overlaps.append(np.mean([len(set(ids[l][t]) & set(ids[l - 1][t])) / wl.top_k
                                             for t in range(B)]))
            for i in range(args.warmup):
                flush.zero_()
                stack(xs[i % n_in])
            torch.cuda.synchronize()
            coli.launch_count()
            if world > 1:
                import torch.distributed as dist
                dist.barrier()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            for k in range(args.steps):
                flush.zero_()
                ev[k][0].record(st)
                stack(xs[k % n_in])
                ev[k][1].record(st)
            torch.cuda.synchronize()
            launches_total += coli.launch_count()
            ms = [a.elapsed_time(b) for a, b in ev]
            t = max_over_ranks(float(np.mean(ms)), world)
            ub = [unions[k % n_in] for k in range(args.steps)]
            bytes_step = float(np.mean([sum(u_ + 1 for u_ in uu) for uu in ub])) * expert_bytes(wl)
            gbs = bytes_step / (t * 1e-3) / 1e9
            # the expert kernel of every layer, timed alone (a second pass)
            coli.timing_read()
            coli.timing_enable(True)
            for k in range(args.steps):
                flush.zero_()
                stack(xs[k % n_in])
            torch.cuda.synchronize()
            coli.timing_enable(False)
            k_ms, k_n = coli.timing_read()
            k_gbs = bytes_step / (k_ms * 1e-3 / max(args.steps, 1)) / 1e9
            # the same stack without the layer-ahead prefetch, for comparison
            ev0 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            for k in range(args.steps):
                flush.zero_()
                ev0[k][0].record(st)
                stack(xs[k % n_in], prefetch=False)
                ev0[k][1].record(st)
            torch.cuda.synchronize()
            t0 = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in ev0])), world)
            per_b.append({"batch": B, "ms_per_step": t, "tok_s": world * B / (t * 1e-3),
                          "tok_s_without_layer_prefetch": world * B / (t0 * 1e-3),
                          "weight_gbs_per_gpu": gbs, "weight_frac_of_hbm": gbs / hbm_peak,
                          "expert_kernel_gbs": k_gbs, "expert_kernel_frac_of_hbm": k_gbs / hbm_peak,
                          "union_mean": float(np.mean([np.mean(uu) for uu in ub])),
                          "routing_overlap_prev_layer": float(np.mean(overlaps)),
                          "step_ms_p10_p50_p90": [float(np.percentile(ms, q)) for q in (10, 50, 90)]})
            if B == wl.batches[0]:
                kernel_b1 = {"bound": "hbm", "achieved": k_gbs, "peak": hbm_peak, "unit": "GB/s",
                             "frac": k_gbs / hbm_peak, "traffic": None, "traffic_unit": "bytes per launch",
                             "kernel": f"k_experts of each of the {wl.layers} layers at batch {B}, timed alone",
                             "algorithmic_bytes_per_launch": bytes_step / wl.layers,
                             "avg_launch_ms": k_ms / max(k_n, 1), "peak_kind": f"{peak_kind} hbm_gbs"}
    status = coli.get_device_status()
    # end to end at batch 1: pinned host x in, the stack, host out
    B = wl.batches[0]
    xh = torch.from_numpy(synth.activations(wl, 40_000, n_tok=B)).pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    x_dev = torch.empty((B, wl.hidden), dtype=torch.float32, device="cuda")
    bufs = [torch.empty((B, wl.hidden), dtype=torch.float32, device="cuda") for _ in range(2)]

    def e2e_once():
        x_dev.copy_(xh, non_blocking=True)
        x = x_dev
        for l, L in enumerate(layers):
            out = bufs[l & 1]
            nxt = layers[l + 1] if l + 1 < len(layers) else None
            if nxt is not None:
                coli.layer_forward_residual_prefetch(x, L["router_w"], L["router_b"], L["expert_w4"],
                                                     L["expert_rs"], L["shared_w4"], L["shared_rs"],
                                                     nxt["router_w"], nxt["shared_w4"], out=out)
            else:
                coli.layer_forward_residual(x, L["router_w"], L["router_b"], L["expert_w4"], L["expert_rs"],
                                            L["shared_w4"], L["shared_rs"], out=out)
            x = out
        oh.copy_(x, non_blocking=True)
        torch.cuda.synchronize()

    for _ in range(3):
        e2e_once()
    e2e_s = 0.0
    n_e2e = min(args.steps, 50)
    gc.disable()
    for _ in range(n_e2e):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_once()
        e2e_s += time.perf_counter() - t0
    gc.enable()
    e2e_s = max_over_ranks(e2e_s, world)
    b1 = per_b[0]
    rec = {
        "metric": METRIC, "value": b1["tok_s"], "unit": "tok/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": b1["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int4xint8->f32",
        "data": "synthetic",
        "config": workload_config(wl),
        "roofline": kernel_b1,
        "sweep": per_b,
        "e2e": {"value": world * n_e2e * B / e2e_s, "unit": "tok/s", "h2d_bytes_per_step": B * wl.hidden * 4,
                "d2h_bytes_per_step": B * wl.hidden * 4},
        "gpu_launches": launches_total,
        "clocks": clocks.summary(),
        "device_status": status,
        "setup_s": round(t_build, 1),
        "peak_kind": f"{peak_kind} hbm_gbs",
    }
    if rank == 0 and not args.no_cpu_baseline:
        rec["cpu_baseline"] = cpu_baseline_line(wl, 2, cpu_seconds, single_thread=False)
    del layers, flush
    torch.cuda.empty_cache()
    return rec


def run_sweep(args):
    world, rank, local = _setup(args)
    line = measure_sweep(args, world, rank, local, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--path", default="auto", choices=["auto", "gemv", "gemm"])
    ap.add_argument("--workload", default="decode", choices=["tiny", "decode", "verify", "prefill", "profile",
                                                          "route_profile", "prefill_profile", "verify_profile", "batch_profile",
                                                          "sweep"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-forwards", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="minimum oracle time of the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sub", default=",".join(SUB_WORKLOADS),
                    help="with the decode workload: comma-separated sub-records measured in the same run "
                         f"({', '.join(SUB_WORKLOADS)}), or 'none'")
    args = ap.parse_args()
    big = synth.WORKLOADS[args.workload].n_tok > 64
    if args.steps is None:
        args.steps = 30 if big else 1000
        if args.workload == "sweep":
            args.steps = 100
    if args.warmup is None:
        args.warmup = 5 if big else 20
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "sweep":
        run_sweep(args)
    else:
        run(args)


if __name__ == "__main__":
    main()
