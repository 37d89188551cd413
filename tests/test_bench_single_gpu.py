"""bench.py runs on one GPU only: the grouped GEMM's cluster-multicast loads
are kept to one-GPU runs, so with --gpus > 1, or as a rank of a multi-rank
launch (WORLD_SIZE > 1), it prints one JSON line marked "unavailable" and
exits 0 without building or loading libdwdp.so.  Checked on CPU, with the
environment a torchrun launch of two ranks would give."""
import json
import os
import subprocess
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parents[1]

# runs bench.main() in a fresh interpreter, then reports whether the
# library's binding was imported or its .so mapped into the process
PROBE = """
import sys, runpy
sys.argv = ["bench.py"] + sys.argv[1:]
try:
    runpy.run_path("bench.py", run_name="__main__")
finally:
    maps = open("/proc/self/maps").read()
    print("LOADED", "libdwdp" in maps or "moe_expert_grouped_split_gb300.binding" in sys.modules)
"""


def _run(args, env_extra):
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, "-c", PROBE, *args], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    return r.stdout.splitlines()


def test_gpus_flag_above_one_is_refused_without_loading_the_library():
    out = _run(["--gpus", "2"], {})
    line = json.loads(out[0])
    assert line["n_gpus"] == 2 and "single-GPU" in line["unavailable"] and "value" not in line
    assert out[-1] == "LOADED False"


def test_two_rank_launch_prints_once_and_loads_nothing():
    env = {"WORLD_SIZE": "2", "LOCAL_RANK": "0", "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": "29555"}
    out0 = _run(["--gpus", "2"], dict(env, RANK="0"))
    out1 = _run(["--gpus", "2"], dict(env, RANK="1", LOCAL_RANK="1"))
    assert json.loads(out0[0])["unavailable"]
    assert out1 == ["LOADED False"]          # rank 1 prints nothing
    assert out0[-1] == "LOADED False"
