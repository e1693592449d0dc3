"""bench.py and __graft_entry__.py import cleanly, their host-side tables are well formed, and
the bench's reporting logic (roofline bound and fraction, clock summary) computes what its JSON
line claims (no GPU needed)."""

import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _load(name):
    spec = importlib.util.spec_from_file_location(name, os.path.join(ROOT, name + ".py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_bench_imports_and_traffic_table():
    bench = _load("bench")
    assert set(bench.NCU_TRAFFIC) <= {"tiny", "global", "local", "long", "short"}
    for name, (sha, nbytes) in bench.NCU_TRAFFIC.items():
        assert len(sha) == 40 and int(sha, 16) >= 0, name
        assert isinstance(nbytes, int) and nbytes > 0, name
    assert len(bench.kernel_source_hash()) == 40


def test_traffic_records_name_no_other_kernel():
    # a recorded capture is keyed by the source hash of the kernel that workload runs by default
    # (windows 1..16: the narrow-window kernel; otherwise the paired tensor-core kernel, 16-bit
    # inputs): it must not be the hash of another kernel's sources
    import synth

    bench = _load("bench")
    for name, (sha, _) in bench.NCU_TRAFFIC.items():
        w = synth.make_config("tiny").window if name == "tiny" else {"global": 0, "local": 64, "long": 0, "short": 4}[name]
        own = 0 if 1 <= w <= 16 else 2
        others = {bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES
                  if bench.KERNEL_SOURCES[k] != bench.KERNEL_SOURCES[own]}
        assert sha not in others, f"{name}: traffic recorded under another kernel's source hash"


def test_graft_entry_imports():
    entry = _load("__graft_entry__")
    assert callable(entry.build) and callable(entry.smoke)


def test_roofline_bound_and_fraction():
    import synth

    bench = _load("bench")
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0}
    # many short sequences: bytes dominate -> HBM bound
    short = synth.make_lens_workload("probe_short", [8] * 64, "bf16", H=2, window=0)
    r = bench.roofline(short, 0.01, peaks, "measured")
    flops, nbytes = bench.work(short)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - nbytes / 1e-5 / 1e9) < 1e-9 * r["achieved"]
    assert abs(r["frac"] - r["achieved"] / 6000.0) < 1e-12
    assert r["traffic"] is None  # no ncu counters recorded for this workload
    # one long sequence: flops dominate -> tensor bound
    long = synth.make_lens_workload("probe_long", [4096], "bf16", H=2, window=0)
    r = bench.roofline(long, 1.0, peaks, "fallback")
    flops, nbytes = bench.work(long)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak_source"] == "fallback"
    assert abs(r["achieved"] - flops / 1e-3 / 1e12) < 1e-9 * r["achieved"]
    assert abs(r["t_roof_us"] - flops / 2000e12 * 1e6) < 1e-9


def test_clock_summary():
    bench = _load("bench")
    c = bench.ClockSampler(0)
    c.lines = [
        "0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 345, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active",  # idle sample
        "garbage",
    ]
    s = c.summary()
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3
    c.lines = []
    assert c.summary() is None


def test_kernel_tables_cover_every_forward_kernel():
    """Every forward kernel id has a name and a source file in the bench's tables (the roofline's
    traffic record is keyed by that source's hash)."""
    bench = _load("bench")
    assert set(bench.KERNEL_NAMES) == set(bench.KERNEL_SOURCES) == set(range(6))
    for k, src in bench.KERNEL_SOURCES.items():
        assert os.path.exists(os.path.join(ROOT, "rope_cu_tile_gb300", "csrc", src)), (k, src)
        assert len(bench.kernel_source_hash(k)) == 40
