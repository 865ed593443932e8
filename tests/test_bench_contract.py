"""The benchmark's reference arm on CPU: one JSON line with the keys the driver reads, printed by
rank 0 only (the oracle timed on the host cores; no GPU involved)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                          capture_output=True, text=True, cwd=ROOT, env=env, timeout=600)


def test_reference_arm_json_line():
    r = _run({"WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "TFLOP/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] >= 3      # warm-up is raised to 3
    assert d["ms_per_step"] > 0 and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["data"] == "synthetic" and d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_print_nothing():
    r = _run({"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def test_long_context_flops_match_the_workloads():
    """The long-context legs count 2*D*H_q*[S(S+1)/2 + (S-w)(S-w+1)/2] per layer, the same
    algorithmic flops as the workload definitions (2.81e14 and 1.405e14)."""
    sys.path.insert(0, ROOT)
    import bench
    import kvp_inputs
    for w, want in ((kvp_inputs.LLAMA31_8B_32L, 2.809e14), (kvp_inputs.QWEN3_8B_131K, 1.405e14)):
        f = bench.long_context_flops(w)
        assert f == w.attn_mass_flops()
        assert abs(f - want) / want < 1e-3
