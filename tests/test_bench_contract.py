"""bench.py's command line and JSON line, checked on CPU through the
reference arm (the oracle timed on the host cores), which needs no GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, timeout=600):
    env = dict(os.environ, OMP_NUM_THREADS="2")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=timeout, env=env)


def test_reference_line_carries_every_contract_key():
    r = _run("--impl", "reference", "--steps", "2", "--warmup", "3", "--workload", "tiny")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == "MoE layer tok/s" and d["unit"] == "tok/s"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["vs_baseline"] is None
    assert isinstance(d["dtype"], str) and d["data"] == "synthetic"
    assert isinstance(d["config"], dict) and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert isinstance(cb["sample"], str) and cb["unit"] == "tok/s"
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == "tok/s"
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_fewer_than_three_warmup_steps_are_rejected():
    r = _run("--impl", "reference", "--steps", "1", "--warmup", "2", "--workload", "tiny", timeout=120)
    assert r.returncode != 0
    assert "warmup" in r.stderr


def _bench_module():
    import importlib
    return importlib.import_module("bench")


def test_traffic_entries_apply_to_the_sources_in_the_tree():
    """Every captured DRAM-traffic figure applies to the kernel sources as they
    are: the bench line carries it for the captured workloads (a stale hash
    would silently leave the roofline's traffic null), and for no other."""
    b = _bench_module()
    for kernel, t in b.TRAFFIC.items():
        for wl in t["workloads"]:
            assert b.kernel_traffic(kernel, wl) == t["bytes_per_launch"], kernel
        assert b.kernel_traffic(kernel, "tiny") is None


def test_traffic_is_dropped_once_a_kernel_source_changes(tmp_path, monkeypatch):
    """A captured figure describes one version of the kernel: after any change
    to one of its sources the bench line reports traffic as null."""
    import shutil
    b = _bench_module()
    for f in {f for t in b.TRAFFIC.values() for f in t["sources"]}:
        shutil.copy(os.path.join(b.CSRC, f), tmp_path / f)
    monkeypatch.setattr(b, "CSRC", str(tmp_path))
    for kernel, t in b.TRAFFIC.items():
        wl = t["workloads"][0]
        assert b.kernel_traffic(kernel, wl) == t["bytes_per_launch"]
        src = tmp_path / t["sources"][0]
        original = src.read_bytes()
        src.write_bytes(original + b"\n// changed\n")
        assert b.kernel_traffic(kernel, wl) is None
        src.write_bytes(original)
