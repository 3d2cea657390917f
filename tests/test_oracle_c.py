"""The plain C reference block (oracle/h3ref.c) against the numpy oracle, and pins of its own.

Two restatements of the pages' block, written separately (float64 C loops and
numpy), must agree on the same tiny seeded inputs: the tile sets and top-k
selections exactly, the attention layer's float64 outputs to rounding, and the
block's bf16 outputs except where float64 rounding order tips a bf16 rounding
(then by one bf16 step).  The C side is also pinned directly: every tile
selected equals dense softmax attention done by brute force, and bf16 rounding
against torch's conversion.  No GPU is needed.
"""
import math

import numpy as np
import pytest

import oracle as O
import synthetic as S
from oracle import cref

rng = np.random.default_rng(4321)


def _weights(shape, seed=7):
    w = S.block_weights(shape, seed)
    return {k: (S.bf16_bits_to_f64(v) if v.dtype == np.uint16 else v.astype(np.float64))
            for k, v in w.items()}


def _attn_inputs(shape, seed, structured):
    inp = S.attention_inputs(shape, seed, structured=structured)
    return [S.bf16_bits_to_f64(inp[n]) for n in ("q", "k", "v", "gate")]


def _bf16_close(a, b, min_equal=0.99):
    """bf16 arrays equal except at rounding ties tipped by float64 summation order."""
    a, b = np.asarray(a), np.asarray(b)
    assert np.all(np.abs(a - b) <= np.abs(b) * 2.0 ** -7 + 1e-30)
    assert np.mean(a == b) >= min_equal


SHAPES = {
    "slices_prefix_ragged": S.BlockShape(64, 64, 150, hidden=64, heads=2, head_dim=32,
                                         mlp_width=256, topk=2),
    "slices_video_only_k_all": S.BlockShape(0, 0, 200, hidden=64, heads=2, head_dim=32,
                                            mlp_width=256, topk=8),
    "cubes_3d_rope_prefix_450": S.BlockShape(36, 414, 5 * 6 * 7, hidden=64, heads=2,
                                             head_dim=48, mlp_width=256, topk=3,
                                             video_grid=(5, 6, 7)),
    "swiglu_prefix_table": S.BlockShape(64, 64, 150, hidden=64, heads=2, head_dim=32,
                                        mlp_width=128, topk=2, mlp="swiglu", prefix_mod=True),
    "no_norm_no_rope_no_pool": S.BlockShape(64, 0, 190, hidden=64, heads=1, head_dim=64,
                                            mlp_width=256, topk=2, qk_norm=False, rope=False,
                                            pooled=False),
}


def test_bf16_rounding_against_torch():
    torch = pytest.importorskip("torch")
    x = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-40, 38, 4000),
                        [0.0, -0.0, 1.0, 3.3895313892515355e38, 3.4e38, 1e-39, -2.5e-40]])
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    got = np.array([cref.bf16(v) for v in x.astype(np.float32).astype(np.float64)])
    assert np.array_equal(got, want)
    # ties go to even: 1 + 2^-8 sits halfway between 1 and 1 + 2^-7
    assert cref.bf16(1.0 + 2.0 ** -8) == 1.0
    assert cref.bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_tiles_match_numpy_oracle(name):
    s = SHAPES[name]
    got = cref.tiles(s)
    want = O.shape_tiles(s)
    assert len(got) == len(want) == s.n_video_tiles
    for a, b in zip(got, want):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("structured", [0.0, 0.5])
@pytest.mark.parametrize("name", sorted(SHAPES))
def test_attention_layer_matches_numpy_oracle(name, structured):
    s = SHAPES[name]
    Q, K, V, G = _attn_inputs(s, 11, structured)
    for p_bf16 in (False, True):
        c = cref.attention_layer(s, Q, K, V, G, p_bf16)
        n = O.attention_layer(Q, K, V, G, s.n_prefix, s.n_video, s.topk, s.tile, s.pooled,
                              p_bf16, O.shape_tiles(s))
        assert np.array_equal(c["idx"], n["idx"])
        assert np.allclose(c["scores"], n["scores"], rtol=1e-12, atol=1e-12)
        if s.pooled:
            assert np.allclose(c["pooled"], n["pooled"], rtol=1e-12, atol=1e-12)
        assert np.allclose(c["o_f64"], n["o_f64"], rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_block_matches_numpy_oracle(name):
    s = SHAPES[name]
    w = _weights(s, 17)
    x = S.bf16_bits_to_f64(S.hidden_rows(s, 5))
    c = cref.block_forward(x, w, s)
    n = O.block_forward(x, w, s)
    _bf16_close(c["o"], n["o"])
    _bf16_close(c["x1"], n["x1"])
    _bf16_close(c["x2"], n["x2"])


def test_c_routed_attention_all_tiles_is_dense_brute_force():
    # every tile selected and no pooled term: the layer is dense softmax attention,
    # done here by brute force with math.exp over every key
    s = S.BlockShape(64, 0, 130, hidden=64, heads=1, head_dim=16, mlp_width=256, topk=3,
                     pooled=False)
    Q, K, V, G = _attn_inputs(s, 3, 0.0)
    c = cref.attention_layer(s, Q, K, V, G)
    N, d = s.n_rows, s.head_dim
    for r in (0, 63, 64, 100, 193):
        sc = [sum(Q[0, r, e] * K[0, j, e] for e in range(d)) / math.sqrt(d) for j in range(N)]
        m = max(sc)
        p = [math.exp(v - m) for v in sc]
        want = [sum(p[j] * V[0, j, e] for j in range(N)) / sum(p) for e in range(d)]
        assert np.allclose(c["o_f64"][r], want, rtol=1e-12, atol=1e-13)


def test_c_topk_rules():
    # planted ties and NaN on a tiny layer: a copy of a key tile ties with it and the
    # lower index wins the last place; a NaN mean ranks last
    def layer(K, k):
        s = S.BlockShape(0, 0, 4 * 64, hidden=64, heads=1, head_dim=8, mlp_width=256,
                         topk=k, pooled=False)
        return cref.attention_layer(s, np.ones((1, 256, 8)), K, V, None)["idx"][0].tolist()
    V = rng.standard_normal((1, 256, 8))
    K = np.zeros((1, 256, 8))
    K[0, 0:64] = 2.0      # tile 0
    K[0, 128:192] = 2.0   # tile 2 equals tile 0
    K[0, 64:128] = 1.0    # tile 1
    assert layer(K, 1) == [[0]] * 4
    assert layer(K, 2) == [[0, 2]] * 4
    K[0, 192:256] = 1.0   # tile 3 equals tile 1: the third place goes to tile 1
    assert layer(K, 3) == [[0, 1, 2]] * 4
    K[0, 0:64] = np.nan
    assert layer(K, 1) == [[2]] * 4
    assert layer(K, 3) == [[1, 2, 3]] * 4


# --------------------------------------------------------------------------- denoiser and ends
def test_euler_and_extrapolation_match_numpy_oracle():
    N, D, P = 40, 24, 9
    z = rng.standard_normal((N, D)).astype(np.float32).astype(np.float64)
    v = O.bf16(rng.standard_normal((N, D)))
    for dt, dtp in ((-0.125, None), (-0.05, -0.3)):
        assert np.array_equal(cref.euler(z, v, dt, dtp, P), O.euler_update(z, v, dt, dtp, P))
    va, vb = rng.standard_normal((2, N, D))
    sv, sp = (0.4, 0.5, 0.65), (0.3, 0.45, 0.5)
    assert np.array_equal(cref.extrapolate(va, vb, sv, sp, P),
                          O.extrapolate(va, vb, *sv, sp, P))


def test_both_ends_match_numpy_oracle():
    z = rng.standard_normal((37, 96))
    w_in = rng.standard_normal((96, 256)) * 0.1
    b_in = rng.standard_normal(256) * 0.02
    _bf16_close(cref.patch_in(z, w_in, b_in), O.patch_in(z, w_in, b_in), min_equal=0.999)
    x = O.bf16(rng.standard_normal((37, 256)))
    mod2 = rng.standard_normal((2, 256)) * 0.1
    w_out = O.bf16(rng.standard_normal((32, 256)) * 0.02)
    b_out = O.bf16(rng.standard_normal(32) * 0.02)
    a, b = cref.output_head(x, mod2, w_out, b_out), O.output_head(x, mod2, w_out, b_out)
    assert np.all(np.abs(a - b) <= np.abs(b) * 2.0 ** -22 + 1e-30)  # fp32 rounding order


@pytest.mark.parametrize("grid", [(3, 4, 7), (2, 3, 8), (1, 1, 1)])
def test_token_pool_and_restore_match_numpy_oracle(grid):
    s = S.BlockShape(8, 24, int(np.prod(grid)), hidden=16, heads=2, head_dim=8, mlp_width=64,
                     topk=2, video_grid=grid, token_reduction=True)
    x = O.bf16(rng.standard_normal((s.n_rows, 16)))
    xr_c, base_c = cref.token_pool(x, s)
    xr_n, base_n = O.token_pool(x, s)
    assert np.array_equal(xr_c, xr_n) and np.array_equal(base_c, base_n)
    y = O.bf16(xr_n + rng.standard_normal(xr_n.shape) * 0.1)  # the reduced rows after blocks
    assert np.array_equal(cref.token_restore(x, y, base_n, s), O.token_restore(x, y, base_n, s))


def test_thin_layers_matches_numpy_oracle():
    mods = rng.standard_normal((12, 6, 32))
    mods[4] = mods[7]  # a planted tie: the higher index is dropped first
    for keep in (2, 5, 9, 11, 12):
        assert cref.thin_layers(mods, keep) == O.thin_layers(mods, keep)
