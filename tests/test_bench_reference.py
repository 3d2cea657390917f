"""bench.py's reference arm (the float32 C oracle timed on host cores) keeps the JSON
contract; runs on the CPU with the 1,024-row attention workload and a small block shape.
Also the host-side pieces of the GPU line: the near-tie audit and the flop accounting."""
import importlib.util
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "routed_attention_1024", "--steps", "2", "--warmup", "1"],
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
    assert cb["kind"].startswith("oracle") and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["unit"] == d["unit"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    # the value is the rows of the measured steps over their measured time
    assert abs(d["value"] - 1024 / (d["ms_per_step"] / 1e3)) < 1e-6 * d["value"]


def test_reference_block_steps_are_measured_samples():
    """A block step of the reference arm is a uniform sample of the block; its time is
    measured, and the value is the rows the sample processed per second."""
    bench = _bench()
    import synthetic as S
    s = S.BlockShape(36, 64, 7 * 64 + 5, hidden=256, heads=2, head_dim=64, mlp_width=512,
                     topk=2)
    blk, x, s2 = bench.cpu_block(s)
    assert s2 is s
    for sample in (1, 3):
        t = bench.time_cpu_block(blk, x, sample)
        assert t > 0
    assert bench.sampled_rows(s.n_rows, 1) == s.n_rows
    assert bench.sampled_rows(s.n_rows, 3) == 64 * len(range(0, -(-s.n_rows // 64), 3)) - (
        64 - s.n_rows % 64 if (s.n_rows // 64) % 3 == 0 else 0)
    cb = bench.cpu_baseline(s, budget_s=30.0)
    assert cb["kind"] == "oracle fp32, measured full block" and cb["value"] > 0
    assert cb["s_per_block"] == cb["seconds_timed"]


def test_near_tie_audit_counts_gaps_and_checks_selections():
    bench = _bench()
    just_above_4 = np.nextafter(np.float32(4.0), np.float32(5.0))
    sc = np.array([[[5.0, 4.0, just_above_4, 1.0], [1.0, 2.0, 3.0, np.nan]]], np.float32)
    idx = np.array([[[0, 1], [1, 2]]], np.int32)
    a = bench.near_tie_audit(sc, idx, 2)
    assert a["pairs"] == 2 and a["near_ties"] == 1  # 4 vs 4 + 1 ulp is a near-tie; 2 vs 1 not
    assert a["selections_are_topk_of_scores"] is False  # row 0: the top-2 is {0, 2}
    idx = np.array([[[0, 2], [1, 2]]], np.int32)
    assert bench.near_tie_audit(sc, idx, 2)["selections_are_topk_of_scores"] is True
    # every tile selected: no (k+1)-th score, no near-tie
    assert bench.near_tie_audit(sc, np.array([[[0, 1, 2, 3]] * 2], np.int32), 4)["near_ties"] == 0


def test_per_clock_peak():
    bench = _bench()
    assert bench.per_clock_peak(152, 2070.0) == 8192 * 152 * 2070e6 / 1e12
    assert bench.per_clock_peak(152, None) is None


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
