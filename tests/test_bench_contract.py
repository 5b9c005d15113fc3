"""The bench's JSON line, checked on the CPU through its reference arm (the fp64 oracle
timed on the host cores): one line on stdout with the keys, types and config the
driver-side comparison reads, the same workload config as the GPU arm, and an e2e
object without host<->device traffic."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_reference(*extra):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "0", "--budget-s", "0.3", *extra], capture_output=True, text=True, cwd=ROOT,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_line_keys_and_types():
    d = run_reference()
    for key, typ in (("metric", str), ("value", float), ("unit", str), ("n_gpus", int), ("steps", int),
                     ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool), ("scaling", str),
                     ("dtype", str), ("data", str), ("config", dict), ("cpu_baseline", dict), ("e2e", dict)):
        assert isinstance(d[key], typ), (key, d[key])
    assert d["impl"] == "reference"
    assert d["steps"] == 2 and d["warmup"] == 0
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["vs_baseline"] is None
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_config_is_the_gpu_arms_workload():
    import bench
    d = run_reference("--workload", "sink_window_dit_bf16_b2h12d128")
    w = bench.WORKLOADS["sink_window_dit_bf16_b2h12d128"]
    shape = bench.workload_config(w)
    assert {k: d["config"][k] for k in shape} == json.loads(json.dumps(shape))
    # 4 x B x H x n_q x kv x D per attend: chunks 1..7 fill the window, 8..10 see all of it
    kvs = [min((c + 1) * w.chunk, w.window) for c in range(w.n_chunks)]
    flops = sum(4 * w.batch * w.heads * w.chunk * kv * w.head_dim for kv in kvs) * w.rewrites
    assert abs(d["config"]["tflop_per_step"] - flops / 1e12) < 1e-9
    assert abs(flops / 1e12 - 52.7507914752) < 1e-9          # the DiT run's 52.75 TFLOP
