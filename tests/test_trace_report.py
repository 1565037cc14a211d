"""The GEMM stage-log reader of trace_report on a synthetic log with known
timings (CPU): a wrong sub-log offset, code or unit fails it."""
import numpy as np


def _entry(t_ns, code, value):
    return ((t_ns << 8) | code, value)


def test_gemm_stage_stats_on_a_known_log():
    from int4_routed_expert_f32_gb300.trace_report import gemm_stage_stats
    cap, q = 64, 16
    ev = np.zeros((cap, 2), np.uint64)

    def sublog(role, entries):
        ev[role * q, 0] = len(entries)
        for i, (w, v) in enumerate(entries, start=1):
            ev[role * q + i] = (w, v)

    base = 10_000_000
    stages = range(10, 15)
    issue = {s: base + 1000 * (s - 10) for s in stages}                 # 1.0 us apart
    sublog(0, [_entry(issue[s], 11, s) for s in stages])
    conv = []
    for s in stages:
        conv.append(_entry(issue[s] + 500, 14, s))                      # landed 0.5 us after issue
        conv.append(_entry(issue[s] + 800, 15, s))                      # converted 0.3 us later
    sublog(2, conv)
    drain = []
    for i, b in enumerate(range(20, 27)):
        r = base + 5000 + 500 * i                                       # blocks 0.5 us apart
        drain.append(_entry(r, 16, b))
        drain.append(_entry(r + 200, 17, b))                            # 0.2 us per block
    sublog(3, drain)
    st = gemm_stage_stats(ev)
    assert st["stages"] == 5
    assert abs(st["stage_interval_us"] - 1.0) < 1e-9
    assert abs(st["issue_to_landed_us"] - 0.5) < 1e-9
    assert abs(st["convert_us"] - 0.3) < 1e-9
    assert abs(st["drain_per_block_us"] - 0.2) < 1e-9
    assert abs(st["drained_interval_us"] - 0.5) < 1e-9
