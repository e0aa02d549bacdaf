"""bench.py rejects bad options before it touches a GPU (CPU test)."""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          timeout=300)


def test_unknown_workload_section_is_rejected():
    r = _run("--workloads", "dgrad,bogus")
    assert r.returncode == 2 and "unknown workload sections: ['bogus']" in r.stderr


def test_moe_sizes_are_checked():
    r = _run("--moe-experts", "4")
    assert r.returncode == 2 and "--moe-experts must be at least 8" in r.stderr
    r = _run("--moe-tokens", "0")
    assert r.returncode == 2
