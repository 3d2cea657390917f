"""bench.py's reference arm (the float64 oracle timed on host cores) keeps the JSON
contract; runs on the CPU with the 1,024-row attention workload and a short-prefix shape."""
import importlib.util
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "attn_tiny_1024", "--steps", "1", "--warmup", "0"],
                         check=True, capture_output=True, text=True, cwd=ROOT).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    for k in ("metric", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "scaling",
              "vs_baseline", "dtype", "data", "config"):
        assert k in d, k
    assert d["config"]["workload"] == "attn_tiny_1024"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["unit"] == d["unit"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_oracle_sample_with_a_prefix_shorter_than_a_chunk():
    sys.path.insert(0, ROOT)
    import synthetic as S
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    s = S.BlockShape(36, 0, 256, hidden=256, heads=2, head_dim=64, mlp_width=512, topk=2)
    t, desc = bench.oracle_block_sample(s)
    assert t > 0 and "prefix chunks" in desc
