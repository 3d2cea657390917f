"""The float32 timing baseline (oracle/h3time.c) against the float64 oracle.

bench.py times h3time.c on the host's cores as the CPU baseline; these tests tie it
to the float64 oracle (itself pinned in test_oracle_pins.py) on small seeded blocks:
the same top-k selections (apart from near-ties), the residual rows and the block's
own update within float32-vs-float64 rounding, and a sampled call that does the
stated fraction of the work on the sampled rows only.
"""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from helpers import NEAR_TIE, rel_l2, cosine
from oracle import ctime

CASES = [
    ("gelu_prefix", S.BlockShape(64, 64, 5 * 64 + 17, hidden=256, heads=2, head_dim=128,
                                 mlp_width=1024, topk=2)),
    ("swiglu_prefix_table_d64", S.BlockShape(0, 128, 6 * 64, hidden=512, heads=4, head_dim=64,
                                             mlp_width=384, topk=3, mlp="swiglu",
                                             prefix_mod=True)),
    ("dense_no_pool", S.BlockShape(64, 0, 256, hidden=256, heads=2, head_dim=128,
                                   mlp_width=512, topk=8, pooled=False)),
]


def _f64(w):
    return {n: (S.bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64))
            for n, a in w.items()}


@pytest.mark.parametrize("name,shp", CASES, ids=[c[0] for c in CASES])
def test_float32_block_matches_float64_oracle(name, shp):
    w = _f64(S.block_weights(shp, 41))
    x0 = S.bf16_bits_to_f64(S.hidden_rows(shp, 41))
    ref = O.block_forward(x0, w, shp, p_bf16=True)
    blk = ctime.Block(shp, ctime.input_major(w))
    x = x0.astype(np.float32)
    idx = blk.run(x, want_idx=True)
    diff = np.any(idx != ref["idx"], axis=-1)
    for h, i in zip(*np.nonzero(diff)):  # fp32 tile means may flip a near-tie only
        assert ref["gap"][h, i] < NEAR_TIE, (name, h, i)
    got = x.astype(np.float64)
    assert rel_l2(got, ref["x2"]) < 2e-3 and cosine(got, ref["x2"]) > 0.99999
    if not diff.any():
        assert rel_l2(got - x0, ref["x2"] - x0) < 2e-2
        assert cosine(got - x0, ref["x2"] - x0) > 0.998
    # every value is a bf16 value (the residual stream is stored in bf16)
    assert np.array_equal(O.bf16(got), got)


def test_sampled_call_touches_only_sampled_rows():
    shp = CASES[0][1]
    w = ctime.input_major(_f64(S.block_weights(shp, 42)))
    x0 = S.bf16_bits_to_f64(S.hidden_rows(shp, 42)).astype(np.float32)
    blk = ctime.Block(shp, w)
    x = x0.copy()
    blk.run(x, sample=3)
    rows = np.arange(shp.n_rows)
    on = (rows // 64) % 3 == 0
    assert np.array_equal(x[~on], x0[~on])
    assert not np.array_equal(x[on], x0[on])
    assert ctime.threads() >= 1


@pytest.mark.parametrize("structured,topk", [(0.5, 4), (0.0, 16)])
def test_float32_attention_matches_float64_oracle(structured, topk):
    """The attention-only entry (router, routed and dense attention, pooled mix) on the
    1,024-row, 4 x 64 shape, k = 4 and k = 16 (every tile: dense attention)."""
    shp = S.ATTN_TINY.shape.with_(topk=topk)
    inp = S.attention_inputs(shp, 43, structured=structured)
    q, k, v, g = (S.bf16_bits_to_f64(inp[n]) for n in ("q", "k", "v", "gate"))
    ref = O.attention_layer(q, k, v, g, shp.n_prefix, shp.n_video, shp.topk, p_bf16=True)
    att = ctime.Attention(shp, q, k, v, g)
    out, idx = att.run(want_idx=True)
    assert np.array_equal(idx, ref["idx"])
    got = out.astype(np.float64)
    assert rel_l2(got, ref["o_f64"]) < 3e-3 and cosine(got, ref["o_f64"]) > 0.99999
    assert np.mean(got == ref["o"]) > 0.99
