"""The benchmark's reference arm (the CPU oracle timed on the host) prints one JSON line
with the contract's keys; runs on CPU in a few seconds on the tiny workload."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    # at least three warm-up steps are always run (and reported): the request of one is raised
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 3
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert "workload" in d["config"]


def test_reference_arm_follows_the_dispatch_fake_quant_option():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "1", "--dispatch-fq"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert d["config"]["dispatch"].startswith("E4M3 fake-quant") and d["value"] > 0
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "1", "--dispatch-fq", "nvfp4"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert d["config"]["dispatch"].startswith("NVFP4 fake-quant")


def test_oracle_step_with_dispatch_fake_quant_changes_the_routed_input_only():
    """The bench's oracle sample with --dispatch-fq feeds the routed experts the
    fake-quantised rows (at the oracle's own 448 / max|x| scale): its output differs from
    the plain sample's, and equals the oracle layer called with that scale directly."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    from combine_moe_route_softmax_gb300 import synth
    from oracle import moe_ref as ref
    w = synth.WORKLOADS["tiny"]
    sample = bench.oracle_sample(w, 4)
    plain = bench.oracle_step(w, sample)
    dq = bench.oracle_step(w, sample, None, "e4m3")
    logits, xb, w13, w2, shared = sample
    idx, wt = ref.route_topk(logits, w.K)
    want = ref.layer_reference(xb, idx, wt, w13, w2, shared=shared,
                               dispatch_scale=ref.fq_scale_from_amax(ref.tensor_amax(xb)))
    assert np.array_equal(dq, want)
    assert not np.array_equal(dq, plain)
