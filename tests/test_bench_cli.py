"""bench.py and __graft_entry__.py import cleanly and their host-side tables are well formed
(no GPU needed)."""

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


def test_graft_entry_imports():
    entry = _load("__graft_entry__")
    assert callable(entry.build) and callable(entry.smoke)
