"""Timeline of one layer forward on the streaming (decode) path, from the
library's event log (``coli_moe_trace_enable`` / ``coli_moe_trace_read``).

    python -m int4_routed_expert_f32_gb300.trace_report [workload] [reps]
    python -m int4_routed_expert_f32_gb300.trace_report --gemm [workload]

Builds the workload's layer on the current CUDA device, runs a few untraced
forwards (L2 flushed before each, as in the benchmark), then traces ``reps``
forwards and prints, relative to the first expert-kernel consumer start:

* the routing launch's phase stamps (its last block's tail);
* when expert-kernel blocks start and exit;
* per unit kind (gate/up, down): counts, start / end times, durations and the
  time spent staging activation codes;
* the consumers' time waiting for weight stages and the producers' time
  waiting for free ring slots;
* when the 64-row output chunks were combined.

With ``--gemm`` (the grouped tensor-core path, default workload
prefill_profile) it prints, for a few blocks of the gate/up GEMM, the median
stage interval, the TMA latency (stage issued to stage landed), the weight
conversion time per stage, the drain time per accumulator block and the
interval between drained blocks, from the GEMM's stage log (per block four
sub-logs: producer code 11 stage issued; first converter warp 14 landed,
15 converted; first drain warp 16 accumulator ready, 17 folded; entry 0 of a
sub-log counts its events; a steady-state window of stages is logged).

Event codes written by the expert kernel (per block, slot 0 counts events):
1 consumer start, 2 unit start (first stage arrived), 3 activations staged,
4 unit done, 5 combine done, 6 consumer exit, 7 consumer waiting time (ns, in
the unit field); the producer's waiting time is code 8 in the block's last
slot.  The routing tail stamps phases 0..8 (16: the first block's logits done)
into the last block region's first slots.
"""
from __future__ import annotations

import sys

import numpy as np
import torch

import int4_routed_expert_f32_gb300 as coli

_MASK56 = (1 << 56) - 1   # stamps carry the timer shifted left by 8 bits


def _pct(x, q):
    return float(np.percentile(x, q)) if len(x) else float("nan")


def report(name: str = "decode", reps: int = 3, events_per_block: int = 128) -> None:
    import synth
    from synth.device import build_device_layer

    wl = synth.WORKLOADS[name]
    T = wl.n_tok
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, T)
    L = build_device_layer(wl)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    xs = [torch.from_numpy(synth.activations(wl, 5000 + i)).cuda() for i in range(5 + reps)]
    out = torch.empty((T, wl.hidden), dtype=torch.float32, device="cuda")

    def fwd(i):
        coli.layer_forward(xs[i], L["router_w"], L["router_b"], L["expert_w4"], L["expert_rs"],
                           L["shared_w4"], L["shared_rs"], out=out)

    for i in range(5):
        flush.zero_()
        fwd(i)
    torch.cuda.synchronize()
    G, CH = wl.ffn // 32, wl.hidden // 64
    coli.trace_enable(events_per_block)
    try:
        for rep in range(reps):
            flush.zero_()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fwd(5 + rep)
            e1.record()
            torch.cuda.synchronize()
            ev, nb, ne = coli.trace_read()
            _print_rep(rep, e0.elapsed_time(e1), ev, nb, ne, G, CH)
    finally:
        coli.trace_enable(0)


def _print_rep(rep, fwd_ms, ev, nb, ne, G, CH):
    recs = []
    producer_wait = []
    for blk in range(nb - 1):
        last = int(ev[blk, ne - 1, 0])
        if (last & 255) == 8:
            producer_wait.append((last >> 8) / 1000.0)
        for i in range(1, int(ev[blk, 0, 0]) + 1):
            w, u = int(ev[blk, i, 0]), int(np.int64(ev[blk, i, 1]))
            recs.append((w >> 8, w & 255, u))
    recs = np.array(recs, dtype=np.int64)
    code, unit = recs[:, 1], recs[:, 2]
    t0 = recs[code == 1, 0].min()
    t = (recs[:, 0] - t0) / 1000.0
    route = ev[nb - 1].reshape(-1)[:17].astype(np.int64)

    def rt(i):
        return (((int(route[i]) & _MASK56) - int(t0)) / 1000.0) if route[i] else float("nan")

    print(f"--- forward {rep}: {fwd_ms * 1000:.1f} us (events around the traced forward)")
    print("  routing (us before the expert consumers start): first block's logits %.2f, "
          "tail start %.2f, keys %.2f, top-k %.2f, phases 2..6: %s"
          % (rt(16), rt(1), rt(7), rt(8), " ".join("%.2f" % rt(i) for i in range(2, 7))))
    for c, nm in ((1, "start"), (6, "exit")):
        x = t[code == c]
        print(f"  block {nm:5s} n={len(x):4d}  min {x.min():6.2f}  p50 {np.median(x):6.2f}  "
              f"p90 {_pct(x, 90):6.2f}  max {x.max():6.2f} us")
    starts, staged, done = {}, {}, {}
    for ti, c, u in zip(t, code, unit):
        if c == 2:
            starts[u] = ti
        elif c == 3:
            staged[u] = ti
        elif c == 4:
            done[u] = ti
    ids = np.array(sorted(starts))
    n_tiles = int(round(len(ids) / (G + CH)))      # every tile has G gate/up and CH down units
    n_gu = n_tiles * G
    for nm, sel in (("gate/up", ids < n_gu), ("down", ids >= n_gu)):
        uu = ids[sel]
        st = np.array([starts[u] for u in uu])
        en = np.array([done.get(u, np.nan) for u in uu])
        sg = np.array([staged.get(u, starts[u]) for u in uu]) - st
        print(f"  {nm:7s} units {len(uu):4d}  start p0/p50/p100 {st.min():5.1f} {np.median(st):5.1f} "
              f"{st.max():5.1f}  end p50/p100 {np.nanmedian(en):5.1f} {np.nanmax(en):5.1f}  "
              f"duration p50 {np.nanmedian(en - st):5.2f}  staging p50 {np.median(sg):4.2f} max {sg.max():4.2f} us")
    cw = unit[code == 7] / 1000.0
    print(f"  consumers waiting for stages: p10 {_pct(cw, 10):.1f}  p50 {_pct(cw, 50):.1f}  p90 {_pct(cw, 90):.1f} us")
    if producer_wait:
        pw = np.array(producer_wait)
        print(f"  producers waiting for free slots: p10 {_pct(pw, 10):.1f}  p50 {_pct(pw, 50):.1f}  "
              f"p90 {_pct(pw, 90):.1f} us")
    cb = t[code == 5]
    if len(cb):
        print(f"  chunks combined: {len(cb)}, first {cb.min():.1f}, last {cb.max():.1f} us")
    print(f"  tiles {n_tiles}")


def gemm_sublog(ev_block: np.ndarray, role: int, quarter: int):
    """Events (time_ns, code, value) of one role's sub-log of a GEMM block."""
    n = int(ev_block[role * quarter, 0])
    out = []
    for i in range(1, min(n, quarter - 1) + 1):
        w, v = int(ev_block[role * quarter + i, 0]), int(np.int64(ev_block[role * quarter + i, 1]))
        out.append((w >> 8, w & 255, v))
    return out


def gemm_stage_stats(ev_block: np.ndarray) -> dict:
    """Medians (us) of one gate/up GEMM block's stage log; NaN where a role
    logged nothing."""
    q = ev_block.shape[0] // 4
    prod, conv, drain = gemm_sublog(ev_block, 0, q), gemm_sublog(ev_block, 2, q), gemm_sublog(ev_block, 3, q)
    issue = {v: t / 1000.0 for t, c, v in prod if c == 11}
    landed = {v: t / 1000.0 for t, c, v in conv if c == 14}
    converted = {v: t / 1000.0 for t, c, v in conv if c == 15}
    ready = {v: t / 1000.0 for t, c, v in drain if c == 16}
    folded = {v: t / 1000.0 for t, c, v in drain if c == 17}
    nan = float("nan")
    st = sorted(issue)
    iss = np.array([issue[k] for k in st])
    land = np.array([landed.get(k, np.nan) for k in st])
    cv = np.array([converted.get(k, np.nan) for k in st])
    bl = sorted(folded)
    dd = np.array([folded[b] - ready[b] for b in bl if b in ready])
    fo = np.array([folded[b] for b in bl])
    return {
        "stages": len(st),
        "stage_interval_us": float(np.median(np.diff(iss))) if len(iss) > 1 else nan,
        "issue_to_landed_us": float(np.nanmedian(land - iss)) if len(st) else nan,
        "convert_us": float(np.nanmedian(cv - land)) if len(st) else nan,
        "drain_per_block_us": float(np.median(dd)) if len(dd) else nan,
        "drained_interval_us": float(np.median(np.diff(fo))) if len(fo) > 1 else nan,
    }


def report_gemm(name: str = "prefill_profile", blocks=(0, 1, 77), events_per_block: int = 2048) -> None:
    import synth
    from synth.device import build_device_layer

    wl = synth.WORKLOADS[name]
    T = wl.n_tok
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, T)
    coli.set_path(coli.PATH_GEMM)
    try:
        L = build_device_layer(wl)
        flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
        x = torch.from_numpy(synth.activations(wl, 5000)).cuda()
        out = torch.empty((T, wl.hidden), dtype=torch.float32, device="cuda")

        def fwd():
            coli.layer_forward(x, L["router_w"], L["router_b"], L["expert_w4"], L["expert_rs"],
                               L["shared_w4"], L["shared_rs"], out=out)

        for _ in range(3):
            flush.zero_()
            fwd()
        torch.cuda.synchronize()
        coli.trace_enable(events_per_block)
        try:
            flush.zero_()
            torch.cuda.synchronize()
            fwd()
            torch.cuda.synchronize()
            ev, nb, ne = coli.trace_read()
        finally:
            coli.trace_enable(0)
    finally:
        coli.set_path(coli.PATH_AUTO)
    for blk in blocks:
        if blk >= nb:
            continue
        st = gemm_stage_stats(ev[blk])
        print(f"block {blk}: {st['stages']} stages logged; stage interval {st['stage_interval_us']:.3f} us, "
              f"issue->landed {st['issue_to_landed_us']:.3f}, convert {st['convert_us']:.3f}, "
              f"drain per block {st['drain_per_block_us']:.3f}, drained-block interval "
              f"{st['drained_interval_us']:.3f}")


if __name__ == "__main__":
    if len(sys.argv) > 1 and sys.argv[1] == "--gemm":
        report_gemm(sys.argv[2] if len(sys.argv) > 2 else "prefill_profile")
    else:
        report(sys.argv[1] if len(sys.argv) > 1 else "decode", int(sys.argv[2]) if len(sys.argv) > 2 else 3)
