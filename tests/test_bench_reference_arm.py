"""`bench.py --impl reference` (the fp64 oracle timed on the host cores) keeps
the bench's JSON contract; it needs no GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "0",
                          "--steps", "2", "--warmup", "1", "--ref-budget", "0.3"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny_fp32"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert abs(d["ms_per_step"] - 256 / d["value"] * 1e3) < 1e-6 * d["ms_per_step"]


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, "-c",
                          "import sys, bench; sys.argv = ['bench.py', '--impl', 'reference', '--workload', '0',"
                          " '--steps', '1', '--warmup', '0', '--ref-budget', '0.2'];"
                          " import types; a = types.SimpleNamespace(steps=1, warmup=0, ref_budget=0.2);"
                          " bench.run_reference(a, bench.ssd_synth.WORKLOADS[0], 1, 2)"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr[-2000:]
    assert not [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
