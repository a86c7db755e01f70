"""bench.py's command line on a machine without a GPU: the reference arms of
the producer, consumer and block-scorer modes print one JSON line and exit 0 (their oracle
timing lives in the GPU arm's cpu_baseline), and every mode is listed."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    return r.returncode, r.stdout


def test_reference_arms_of_the_neighbouring_steps():
    for op in ("produce", "attend", "blocks"):
        rc, out = _run("--op", op, "--impl", "reference")
        assert rc == 0
        line = json.loads(out.strip().splitlines()[-1])
        assert line["impl"] == "reference" and "unavailable" in line


def test_help_lists_every_mode():
    rc, out = _run("--help")
    assert rc == 0
    for word in ("select", "produce", "attend", "blocks", "--producer-workload", "--window"):
        assert word in out
