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


def _bench():
    sys.path.insert(0, ROOT)
    spec = importlib.util.spec_from_file_location("bench_mod2", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    return bench


def test_attention_flops_equal_the_pairs_the_method_attends():
    # the roofline counts 4 d flops per (query, key) pair the method attends; with full
    # 64-row tiles the formula is exact: count the pairs from the oracle's own key sets
    import numpy as np
    import oracle as O
    import synthetic as S
    bench = _bench()
    for shp in (S.BlockShape(128, 64, 6 * 64, hidden=256, heads=2, head_dim=64,
                             mlp_width=1024, topk=2),
                S.BlockShape(0, 64, 5 * 64, hidden=256, heads=1, head_dim=128,
                             mlp_width=1024, topk=5)):
        inp = S.attention_inputs(shp, 5, structured=0.5)
        q, k = (S.bf16_bits_to_f64(inp[n]) for n in ("q", "k"))
        sets = O.shape_tiles(shp)
        idx = O.topk_select(O.tile_scores(O.tile_means(q, shp.n_prefix, shp.n_video, 64, sets),
                                          O.tile_means(k, shp.n_prefix, shp.n_video, 64, sets)),
                            shp.topk)
        pairs = 0
        for h in range(shp.heads):
            pairs += shp.n_prefix * shp.n_rows
            for i, rows in enumerate(sets):
                keys = shp.n_prefix + sum(len(sets[j]) for j in idx[h, i])
                pairs += len(rows) * keys
        _, attn = bench.block_flops(shp)
        assert attn == 4.0 * shp.head_dim * pairs


def test_block_flops_of_the_15435_row_block():
    # 26 N D^2 for the four projections of the 4x GELU block, and the attention the method
    # does at k = 16 of 218 tiles: 10,520 and ~1,214 GFLOP (1,214 counts 64 rows per kept
    # tile; the mean tile holds 13,899 / 218 = 63.76 rows, which gives 1,213.1)
    import synthetic as S
    bench = _bench()
    s = S.BLOCK_15K.shape
    gemm, attn = bench.block_flops(s)
    assert gemm == 26.0 * s.n_rows * s.hidden ** 2
    assert round(gemm / 1e9) == 10520 and 1213.0 < attn / 1e9 < 1214.0
