"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test ties one oracle function to a closed form, an invariant, a brute
force on a tiny input, an independent library routine, or a value printed on
the pages (tests/golden/).  None of them needs a GPU.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle as O
import synthetic as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# --------------------------------------------------------------------------- bf16
def test_bf16_against_torch_conversion():
    torch = pytest.importorskip("torch")
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        [0.0, -0.0, 1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 3.3895e38, -1e-39]])
    x32 = x.astype(np.float32).astype(np.float64)  # torch converts from fp32
    want = torch.tensor(x32, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16(x32)
    fin = np.isfinite(want)
    assert np.array_equal(got[fin], want[fin])
    assert np.array_equal(np.isinf(got), np.isinf(want))


def test_bf16_hand_values():
    assert O.bf16(1.0) == 1.0
    assert O.bf16(1.0 + 2 ** -8) == 1.0                 # tie -> even
    assert O.bf16(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6    # tie -> even (up)
    assert O.bf16(1.0 + 2 ** -8 + 2 ** -30) == 1.0 + 2 ** -7
    assert np.isnan(O.bf16(np.nan))
    assert O.bf16(1e39) == np.inf


def test_bf16_matches_generator_storage():
    x = rng.standard_normal(5000).astype(np.float32).astype(np.float64)
    bits = S.to_bf16_bits(x)
    assert np.array_equal(S.bf16_bits_to_f64(bits), O.bf16(x))


# --------------------------------------------------------------------------- rows
def test_rms_modulate_closed_forms():
    eps = 1e-6
    c = 0.75
    x = np.full((1, 64), c)
    h = O.rms_modulate(x, np.zeros(64), np.zeros(64), eps)
    assert np.all(h == O.bf16(c / math.sqrt(c * c + eps)))
    a = 2.0
    x = np.tile([a, -a], (3, 32))
    shift = np.full(64, 0.25)
    scale = np.full(64, 1.0)
    h = O.rms_modulate(x, shift, scale, eps)
    r = a / math.sqrt(a * a + eps)
    assert np.all(h[:, 0::2] == O.bf16(2 * r + 0.25))
    assert np.all(h[:, 1::2] == O.bf16(-2 * r + 0.25))
    # scale = -1 removes the row: h = shift exactly
    h = O.rms_modulate(rng.standard_normal((4, 64)), shift, -np.ones(64), eps)
    assert np.all(h == 0.25)


def test_modulate_rows_picks_each_rows_table():
    # scale = -1 on both tables makes every modulated row equal to its own table's shift
    # exactly (the closed form above), so each row shows which table it took: packed
    # indices below n_prefix the prefix table, the rest the main one, also for a row subset
    D, P, eps = 64, 3, 1e-6
    x = rng.standard_normal((7, D))
    mod = np.zeros((6, D))
    modp = np.zeros((6, D))
    mod[1], modp[1] = -1.0, -1.0
    mod[0], modp[0] = 0.5, -0.25
    h = O.modulate_rows(x, mod, modp, P, 0, 1, eps)
    assert np.all(h[:P] == -0.25) and np.all(h[P:] == 0.5)
    rows = np.array([5, 0, 2, 3])
    h = O.modulate_rows(x[:4], mod, modp, P, 0, 1, eps, rows=rows)
    assert np.all(h[[1, 2]] == -0.25) and np.all(h[[0, 3]] == 0.5)
    # without a prefix table every row takes the main table
    assert np.all(O.modulate_rows(x, mod, None, P, 0, 1, eps) == 0.5)


def test_gate_rows_picks_each_rows_table():
    D, P = 8, 2
    mod = np.arange(6 * D, dtype=np.float64).reshape(6, D)
    modp = -mod - 1.0
    g = O.gate_rows(mod, modp, P, 2, np.array([0, 1, 2, 5]))
    assert np.array_equal(g, np.stack([modp[2], modp[2], mod[2], mod[2]]))
    assert np.array_equal(O.gate_rows(mod, None, P, 5, np.array([0, 3])), mod[5])


def test_linear_small_integers_exact():
    a = rng.integers(-8, 9, (37, 96))
    w = rng.integers(-8, 9, (53, 96))
    b = rng.integers(-8, 9, 53)
    want = a.astype(np.int64) @ w.astype(np.int64).T + b
    assert np.array_equal(O.linear(a, w, b), want.astype(np.float64))


def test_gelu_closed_forms():
    assert O.gelu_erf(0.0) == 0.0
    x = rng.standard_normal(1000) * 3
    assert np.allclose(O.gelu_erf(x) - O.gelu_erf(-x), x, rtol=0, atol=1e-14)
    # GELU(1) = Phi(1), the standard normal CDF at 1 (table value 0.841344746068543)
    assert abs(float(O.gelu_erf(1.0)) - 0.841344746068543) < 1e-15
    assert abs(float(O.gelu_erf(-10.0))) < 1e-20
    assert float(O.gelu_erf(10.0)) == 10.0


def test_head_rms_norm_unit_rms():
    x = rng.standard_normal((3, 10, 128)) * 5
    y = O.head_rms_norm(x, np.ones(128), 0.0)
    assert np.allclose(np.mean(y * y, axis=-1), 1.0, atol=1e-13)
    w = rng.standard_normal(128)
    assert np.allclose(O.head_rms_norm(x, w, 0.0), y * w, atol=1e-14)


def test_rope_closed_form_and_relative_position():
    # d = 2: one pair, frequency theta^0 = 1, so the angle is the position itself
    x = np.array([[1.0, 0.0], [0.3, -0.7]])
    p = np.array([0.0, 2.5])
    y = O.rope(x, p)
    assert np.allclose(y[0], [1.0, 0.0])
    c, s = math.cos(2.5), math.sin(2.5)
    assert np.allclose(y[1], [0.3 * c + 0.7 * s, -0.7 * c + 0.3 * s])
    # norm per pair preserved; dot products depend only on the position difference
    d = 128
    q = rng.standard_normal((1, d))
    k = rng.standard_normal((1, d))
    a = O.rope(q, np.array([17.0]))[0] @ O.rope(k, np.array([5.0]))[0]
    b = O.rope(q, np.array([1017.0]))[0] @ O.rope(k, np.array([1005.0]))[0]
    assert abs(a - b) < 1e-9
    z = O.rope(q, np.array([123.0]))
    assert abs(np.linalg.norm(z) - np.linalg.norm(q)) < 1e-12
    # pair c uses frequency theta^(-2c/d): pair 1 of d=4 at position 100 rotates by 100/100
    x4 = np.array([[0.0, 1.0, 0.0, 0.0]])
    y4 = O.rope(x4, np.array([100.0]), theta=10000.0)
    assert np.allclose(y4[0], [0.0, math.cos(1.0), 0.0, math.sin(1.0)])


# --------------------------------------------------------------------------- router
def test_tile_means_brute_force_and_partial_tile():
    H, P, Vn, d = 2, 64, 150, 8
    X = rng.standard_normal((H, P + Vn, d))
    m = O.tile_means(X, P, Vn, 64)
    assert m.shape == (H, 3, d)
    for h in range(H):
        for t in range(3):
            rows = [r for r in range(P + 64 * t, min(P + 64 * t + 64, P + Vn))]
            want = [sum(X[h, r, c] for r in rows) / len(rows) for c in range(d)]
            assert np.allclose(m[h, t], want, atol=1e-14)
    assert len(O.video_tiles(P, Vn, 64)) == 3 and O.video_tiles(P, Vn, 64)[-1] == (P + 128, 22)


def test_tile_scores_brute_force():
    mq = rng.standard_normal((2, 5, 7))
    mk = rng.standard_normal((2, 5, 7))
    s = O.tile_scores(mq, mk)
    for h, i, j in itertools.product(range(2), range(5), range(5)):
        assert abs(s[h, i, j] - sum(mq[h, i, c] * mk[h, j, c] for c in range(7))) < 1e-13


def _brute_topk(row, k):
    """The unique k-subset C with: for i in C, j not in C, s_i > s_j or (s_i == s_j and i < j)."""
    s = [(-math.inf if math.isnan(v) else v) for v in row]
    T = len(s)
    found = []
    for C in itertools.combinations(range(T), k):
        ok = all(s[i] > s[j] or (s[i] == s[j] and i < j)
                 for i in C for j in range(T) if j not in C)
        if ok:
            found.append(C)
    assert len(found) == 1
    return list(found[0])


@pytest.mark.parametrize("T,k", [(6, 1), (6, 3), (7, 4), (8, 2), (8, 7)])
def test_topk_brute_force_with_ties_and_nans(T, k):
    for trial in range(20):
        row = rng.integers(-3, 4, T).astype(np.float64)  # many exact ties
        if trial % 3 == 0:
            row[rng.integers(0, T, 2)] = np.nan
        if trial % 5 == 0:
            row[rng.integers(0, T)] = -np.inf
        got = O.topk_select(row[None, None, :], k)[0, 0]
        assert got.tolist() == _brute_topk(row.tolist(), k)


def test_topk_nan_regression_exact_k():
    # A NaN must never let a row keep more than k tiles (TensorFold #949 kernel-contract finding).
    row = np.array([np.nan, 1.0, np.nan, 2.0, np.nan])
    got = O.topk_select(row[None, None, :], 2)[0, 0]
    assert got.tolist() == [1, 3]
    got = O.topk_select(row[None, None, :], 4)[0, 0]
    assert got.tolist() == [0, 1, 2, 3]  # NaNs rank as -inf; ties among them go to the lower index


def test_topk_all_and_gap():
    s = rng.standard_normal((2, 3, 5))
    assert np.array_equal(O.topk_select(s, 5)[0, 0], np.arange(5))
    assert np.array_equal(O.topk_select(s, 9)[1, 2], np.arange(5))
    assert np.all(np.isinf(O.topk_gap(s, 5)))
    t = np.array([[[3.0, 1.0, 2.0, 2.0 + 1e-9]]])
    assert O.topk_gap(t, 2)[0, 0] < 1e-5
    assert O.topk_set_valid(t[0, 0], [0, 2]) and O.topk_set_valid(t[0, 0], [0, 3])
    assert not O.topk_set_valid(t[0, 0], [0, 1])


# --------------------------------------------------------------------------- attention
def _brute_attention(q, K, V, scale):
    out = []
    for qi in q:
        s = [sum(qi[c] * kj[c] for c in range(len(qi))) * scale for kj in K]
        m = max(s)
        w = [math.exp(v - m) for v in s]
        z = sum(w)
        out.append([sum(w[j] * V[j][c] for j in range(len(K))) / z for c in range(V.shape[1])])
    return np.array(out)


@pytest.mark.parametrize("P", [0, 64])
def test_routed_all_tiles_equals_dense_brute_force(P):
    H, Vn, d = 2, 150, 8
    N = P + Vn
    Q, K, V = (rng.standard_normal((H, N, d)) for _ in range(3))
    tv = len(O.video_tiles(P, Vn))
    idx = O.topk_select(O.tile_scores(O.tile_means(Q, P, Vn), O.tile_means(K, P, Vn)), tv)
    out = O.routed_attention(Q, K, V, P, Vn, idx)
    for h in range(H):
        want = _brute_attention(Q[h], K[h], V[h], 1.0 / math.sqrt(d))
        assert np.allclose(out[h], want, atol=1e-12)


def test_attend_bf16_weights_streamed_in_octaves():
    """The bf16-weight reading: weights rounded against a whole-octave maximum give the
    same result however the keys are streamed, as long as each running maximum is a
    whole octave (a power-of-two rescale commutes with the bf16 rounding).  A streaming
    softmax over random key chunks, written here with its own running maximum, must
    reproduce the one-shot result; for positive values the rounding moves the output
    by at most 2^-9 relative."""
    d, nq, nk = 16, 5, 300
    q = rng.standard_normal((nq, d)) * 2.0
    k = rng.standard_normal((nk, d))
    v = rng.standard_normal((nk, d))
    scale = 1.0 / math.sqrt(d)
    want = O.attend(q, k, v, scale, p_bf16=True)
    for trial in range(4):
        cuts = np.sort(rng.choice(np.arange(1, nk), size=5 + trial, replace=False))
        chunks = np.split(np.arange(nk), cuts)
        for r in range(nq):
            m, l, acc = -np.inf, 0.0, np.zeros(d)
            for ch in chunks:
                z = (k[ch] @ q[r]) * scale / math.log(2.0)
                if z.max() > m:
                    m_new = math.ceil(z.max())
                    f = 0.0 if m == -np.inf else 2.0 ** (m - m_new)
                    l, acc, m = l * f, acc * f, m_new
                w = 2.0 ** (z - m)
                l += w.sum()
                acc += O.bf16(w) @ v[ch]
            assert np.allclose(acc / l, want[r], rtol=0, atol=1e-13)
    vp = np.abs(v) + 0.5
    exact = O.attend(q, k, vp, scale)
    rounded = O.attend(q, k, vp, scale, p_bf16=True)
    assert np.all(np.abs(rounded - exact) <= 2.0 ** -9 * exact + 1e-15)
    assert not np.array_equal(rounded, exact)


def test_routed_keyset_brute_force():
    # every video query row attends to the prefix plus exactly its selected tiles
    H, P, Vn, d, k = 1, 64, 256, 8, 2
    N = P + Vn
    Q, K, V = (rng.standard_normal((H, N, d)) for _ in range(3))
    idx = np.array([[[0, 3], [1, 2], [0, 1], [2, 3]]], dtype=np.int32)
    out = O.routed_attention(Q, K, V, P, Vn, idx)
    scale = 1.0 / math.sqrt(d)
    for i in range(4):
        keys = list(range(P)) + [P + 64 * j + r for j in idx[0, i] for r in range(64)]
        rows = range(P + 64 * i, P + 64 * i + 64)
        for r in list(rows)[:3]:
            want = _brute_attention(Q[0, [r]], K[0, keys], V[0, keys], scale)
            assert np.allclose(out[0, r], want[0], atol=1e-12)


def test_attention_row_stochastic_and_zero_query():
    H, P, Vn, d = 2, 64, 200, 16
    N = P + Vn
    Q = rng.standard_normal((H, N, d))
    K = rng.standard_normal((H, N, d))
    V = np.broadcast_to(rng.standard_normal((H, 1, d)), (H, N, d)).copy()
    idx = O.topk_select(O.tile_scores(O.tile_means(Q, P, Vn), O.tile_means(K, P, Vn)), 2)
    out = O.routed_attention(Q, K, V, P, Vn, idx)
    assert np.allclose(out, V, atol=1e-14)  # weights sum to one
    V = rng.standard_normal((H, N, d))
    out = O.routed_attention(np.zeros_like(Q), K, V, P, Vn, idx)
    assert np.allclose(out[:, :P], V.mean(axis=1, keepdims=True).repeat(P, 1), atol=1e-13)
    for h in range(H):
        for i, (r0, nv) in enumerate(O.video_tiles(P, Vn)):
            kr = list(range(P)) + [r for j in idx[h, i] for r in range(
                O.video_tiles(P, Vn)[j][0], O.video_tiles(P, Vn)[j][0] + O.video_tiles(P, Vn)[j][1])]
            assert np.allclose(out[h, r0:r0 + nv], V[h, kr].mean(axis=0), atol=1e-13)


def test_attention_layer_given_selections():
    """Selections passed in replace the router's in the attention only: the router's own
    set reproduces the plain call, and another set gives the attention of that set's key
    rows (brute force) while the reported selections and scores stay the router's."""
    H, P, Vn, d, k = 2, 64, 64 * 5, 8, 2
    N = P + Vn
    Q, K, V = (rng.standard_normal((H, N, d)) for _ in range(3))
    G = rng.standard_normal((N, H * d))
    base = O.attention_layer(Q, K, V, G, P, Vn, k)
    same = O.attention_layer(Q, K, V, G, P, Vn, k, idx=base["idx"])
    assert np.array_equal(same["o_f64"], base["o_f64"])
    other = base["idx"].copy()
    other[1, 3] = [0, 4] if list(base["idx"][1, 3]) != [0, 4] else [1, 2]
    alt = O.attention_layer(Q, K, V, G, P, Vn, k, idx=other)
    assert np.array_equal(alt["idx"], base["idx"]) and np.array_equal(alt["scores"],
                                                                     base["scores"])
    rows = range(P + 3 * 64, P + 4 * 64)
    keys = list(range(P)) + [P + 64 * j + r for j in other[1, 3] for r in range(64)]
    for r in list(rows)[:4]:
        want = _brute_attention(Q[1, [r]], K[1, keys], V[1, keys], 1.0 / math.sqrt(d))[0]
        got = alt["o_f64"][r, d:2 * d] - G[r, d:2 * d] * alt["pooled"][1, 3]
        assert np.allclose(got, want, atol=1e-12)
    untouched = [r for r in range(N) if not (P + 3 * 64 <= r < P + 4 * 64)]
    assert np.array_equal(alt["o_f64"][untouched, d:2 * d], base["o_f64"][untouched, d:2 * d])


def test_router_tile_permutation_equivariance():
    H, Vn, d, k = 2, 64 * 6, 16, 3
    Q, K, V = (rng.standard_normal((H, Vn, d)) for _ in range(3))
    perm = rng.permutation(6)  # new tile t holds old tile perm[t]
    rows = np.concatenate([np.arange(64 * p, 64 * p + 64) for p in perm])
    a = O.attention_layer(Q, K, V, None, 0, Vn, k, pooled=False)
    b = O.attention_layer(Q[:, rows], K[:, rows], V[:, rows], None, 0, Vn, k, pooled=False)
    inv = np.argsort(perm)
    for h in range(H):
        for t in range(6):
            assert sorted(perm[b["idx"][h, t]].tolist()) == a["idx"][h, perm[t]].tolist()
    assert np.allclose(b["o_f64"], a["o_f64"][rows], atol=1e-12)
    # permuting rows inside a tile leaves the means and the selections unchanged
    inner = np.arange(Vn).reshape(6, 64)
    inner = np.concatenate([rng.permutation(r) for r in inner])
    c = O.attention_layer(Q[:, inner], K[:, inner], V[:, inner], None, 0, Vn, k, pooled=False)
    assert np.array_equal(c["idx"], a["idx"])
    assert np.allclose(c["mq"], a["mq"], atol=1e-14)
    assert np.allclose(c["o_f64"], a["o_f64"][inner], atol=1e-12)
    del inv


def test_planted_tie_lower_tile_wins():
    H, Vn, d = 1, 64 * 4, 8
    Q, K, V = (rng.standard_normal((H, Vn, d)) for _ in range(3))
    K[:, 128:192] = K[:, 64:128]  # tiles 1 and 2 identical -> equal scores for every query
    mq = O.tile_means(Q, 0, Vn)
    mk = O.tile_means(K, 0, Vn)
    S_ = O.tile_scores(mq, mk)
    idx = O.topk_select(S_, 1)
    for i in range(4):
        if np.argmax(S_[0, i]) in (1, 2):
            assert idx[0, i, 0] == 1


def test_pooled_closed_forms():
    mv = rng.standard_normal((2, 1, 8))
    S_ = rng.standard_normal((2, 1, 1))
    assert np.allclose(O.pooled_branch(S_, mv, 8), mv, atol=1e-15)
    mv = np.broadcast_to(rng.standard_normal((2, 1, 8)), (2, 5, 8))
    S_ = rng.standard_normal((2, 5, 5))
    assert np.allclose(O.pooled_branch(S_, mv, 8), mv, atol=1e-14)
    S_ = rng.standard_normal((1, 3, 4))
    mv = rng.standard_normal((1, 4, 2))
    got = O.pooled_branch(S_, mv, 16)
    for i in range(3):
        w = [math.exp(S_[0, i, j] / 4.0) for j in range(4)]
        want = [sum(w[j] * mv[0, j, c] for j in range(4)) / sum(w) for c in range(2)]
        assert np.allclose(got[0, i], want, atol=1e-14)


def test_gate_mix_brute_force():
    H, P, Vn, d = 2, 64, 100, 4
    N = P + Vn
    Ov = rng.standard_normal((H, N, d))
    G = rng.standard_normal((N, H * d))
    pb = rng.standard_normal((H, 2, d))
    out = O.gate_mix(Ov, G, pb, P, Vn)
    for r in range(N):
        for h in range(H):
            for c in range(d):
                want = Ov[h, r, c] + (G[r, h * d + c] * pb[h, (r - P) // 64, c] if r >= P else 0.0)
                assert abs(out[r, h * d + c] - want) < 1e-14


# --------------------------------------------------------------------------- cubes, 3-D rotary
def test_cube_tiles_receipt_golden():
    with open(os.path.join(GOLDEN, "receipt_tiles.txt")) as f:
        rows = [list(map(int, ln.split())) for ln in f if ln.strip() and not ln.startswith("#")]
    for nt, na, nv, T, Hg, Wg, total, pre, kept in rows:
        assert T * Hg * Wg == nv and nt + na + nv == 15435
        tiles = O.cube_tiles(nt + na, (T, Hg, Wg))
        assert -(-(nt + na) // 64) == pre
        assert len(tiles) + pre == total
        assert kept < len(tiles)


@pytest.mark.parametrize("grid,cube", [((37, 15, 27), (4, 4, 4)), ((5, 6, 7), (4, 4, 4)),
                                       ((1, 1, 1), (4, 4, 4)), ((8, 8, 8), (4, 4, 4)),
                                       ((3, 9, 10), (2, 8, 4))])
def test_cube_tiles_partition_by_membership(grid, cube):
    # every video row lies in exactly one tile, namely the cube containing its (t, h, w),
    # and each tile lists its rows in raster order
    P = 7
    T, Hg, Wg = grid
    tiles = O.cube_tiles(P, grid, cube)
    allrows = np.concatenate(tiles)
    assert np.array_equal(np.sort(allrows), P + np.arange(T * Hg * Wg))
    nh, nw = -(-Hg // cube[1]), -(-Wg // cube[2])
    for i, tr in enumerate(tiles):
        assert np.all(np.diff(tr) > 0) and 1 <= len(tr) <= cube[0] * cube[1] * cube[2]
        for r in tr:
            t, h, w = (r - P) // (Hg * Wg), (r - P) // Wg % Hg, (r - P) % Wg
            assert ((t // cube[0]) * nh + h // cube[1]) * nw + w // cube[2] == i


def test_rope_axis_split_values():
    # the common video-DiT split: 44 / 42 / 42 dims at d = 128, 24 / 20 / 20 at d = 64
    assert O.rope_axis_split(128) == (22, 21, 21)
    assert O.rope_axis_split(64) == (12, 10, 10)


def test_rope_3d_brute_force_complex():
    d, N = 64, 9
    x = rng.standard_normal((2, N, d))
    coords = rng.integers(0, 40, (N, 3))
    got = O.rope_3d(x, coords, 10000.0)
    mt, mh, mw = 12, 10, 10
    for h in range(2):
        for n in range(N):
            for c in range(d // 2):
                if c < mt:
                    a, j, m = 0, c, mt
                elif c < mt + mh:
                    a, j, m = 1, c - mt, mh
                else:
                    a, j, m = 2, c - mt - mh, mw
                z = complex(x[h, n, c], x[h, n, c + d // 2]) * \
                    np.exp(1j * coords[n, a] * 10000.0 ** (-j / m))
                assert abs(got[h, n, c] - z.real) < 1e-12
                assert abs(got[h, n, c + d // 2] - z.imag) < 1e-12


def test_rope_3d_relative_per_axis_and_isolation():
    d = 128
    q, k = rng.standard_normal((1, 1, d)), rng.standard_normal((1, 1, d))
    a, b = np.array([[3, 5, 7]]), np.array([[11, 2, 9]])
    base = float(O.rope_3d(q, a)[0, 0] @ O.rope_3d(k, b)[0, 0])
    for delta in ([4, 0, 0], [0, 6, 0], [0, 0, 13], [2, 3, 5]):
        dd = np.array([delta])
        moved = float(O.rope_3d(q, a + dd)[0, 0] @ O.rope_3d(k, b + dd)[0, 0])
        assert abs(moved - base) < 1e-10
    # a width-only move turns only the width pairs (the last 21 of 64)
    r0 = O.rope_3d(q, a)[0, 0]
    r1 = O.rope_3d(q, a + np.array([[0, 0, 1]]))[0, 0]
    same = np.isclose(r0, r1, rtol=0, atol=1e-15)
    pair_same = same[:64] & same[64:]
    assert pair_same[:43].all() and not pair_same[43:].any()
    assert np.allclose(O.rope_3d(q, np.zeros((1, 3))), q)


def test_rope_coords_raster():
    c = O.rope_coords(5, 3 * 4 * 6, (3, 4, 6))
    assert np.array_equal(c[:5], np.repeat(np.arange(5)[:, None], 3, axis=1))
    assert np.array_equal(c[5 + (2 * 4 + 1) * 6 + 5], [2, 1, 5])


def test_cube_block_equals_permuted_slices_when_dense():
    # with every tile selected and no pooled term the tiling does not matter: the cube
    # shape equals the 1-D shape on the same rows (up to the rotary, disabled here)
    base = dict(n_text=36, n_audio=64, n_video=5 * 6 * 7, hidden=64, heads=2, head_dim=32,
                mlp_width=256, topk=64, rope=False, pooled=False)
    s1 = S.BlockShape(**base)
    s3 = S.BlockShape(**base, video_grid=(5, 6, 7))
    w = _weights(s1)
    x = S.bf16_bits_to_f64(S.hidden_rows(s1, 8))
    a = O.block_forward(x, w, s1)["x2"]
    b = O.block_forward(x, w, s3)["x2"]
    assert np.array_equal(a, b)


# --------------------------------------------------------------------------- block
def _tiny_shape(**kw):
    base = dict(n_text=64, n_audio=64, n_video=150, hidden=64, heads=2, head_dim=32,
                mlp_width=256, topk=2)
    base.update(kw)
    return S.BlockShape(**base)


def _weights(shape, seed=7):
    w = S.block_weights(shape, seed)
    return {k: (S.bf16_bits_to_f64(v) if v.dtype == np.uint16 else v.astype(np.float64))
            for k, v in w.items()}


def test_block_closed_form_constant_rows():
    # scale1 = -1 makes every modulated row equal to shift1; without rotary, all q, k, v rows
    # are then equal, so attention returns that v row and the pooled branch returns it too.
    shape = _tiny_shape(rope=False)
    w = _weights(shape)
    w["mod"][1] = -1.0
    x = S.bf16_bits_to_f64(S.hidden_rows(shape, 3))
    out = O.block_forward(x, w, shape)
    hrow = O.bf16(w["mod"][0])
    qkvg = O.bf16(O.linear(hrow[None, :], w["w_qkvg"], w["b_qkvg"]))[0]
    A = shape.attn_width
    vrow, grow = qkvg[2 * A:3 * A], qkvg[3 * A:]
    o = np.tile(vrow, (shape.n_rows, 1))
    o[shape.n_prefix:] += grow * vrow
    assert np.allclose(out["o_f64"], o, atol=1e-12)
    x1 = O.bf16(x + w["mod"][2] * O.linear(O.bf16(o), w["w_o"], w["b_o"]))
    assert np.array_equal(out["x1"], x1)


def test_block_zero_gates_pass_residual():
    shape = _tiny_shape()
    w = _weights(shape)
    w["mod"][2] = 0.0
    w["mod"][5] = 0.0
    x = S.bf16_bits_to_f64(S.hidden_rows(shape, 3))
    out = O.block_forward(x, w, shape)
    assert np.array_equal(out["x1"], x) and np.array_equal(out["x2"], x)


def test_block_all_tiles_equals_dense():
    shape = _tiny_shape(topk=3, pooled=False)
    w = _weights(shape)
    x = S.bf16_bits_to_f64(S.hidden_rows(shape, 3))
    out = O.block_forward(x, w, shape)
    H, d = shape.heads, shape.head_dim
    dense = np.stack([O.attend(out["q"][h], out["k"][h], out["v"][h], 1 / math.sqrt(d))
                      for h in range(H)])
    assert np.allclose(out["O"], dense, atol=1e-12)


def test_block_prefix_table_zero_gates_split_by_modality():
    # zero gates on one table leave exactly that modality's rows untouched
    shape = _tiny_shape(prefix_mod=True)
    x = S.bf16_bits_to_f64(S.hidden_rows(shape, 3))
    P = shape.n_prefix
    for zeroed, same, moved in (("mod_prefix", slice(0, P), slice(P, None)),
                                ("mod", slice(P, None), slice(0, P))):
        w = _weights(shape)
        w[zeroed][2] = 0.0
        w[zeroed][5] = 0.0
        out = O.block_forward(x, w, shape)
        assert np.array_equal(out["x2"][same], x[same])
        assert not np.array_equal(out["x2"][moved], x[moved])


def test_block_prefix_table_norm_applies_to_its_rows():
    # scale1 = -1 on one table makes that modality's modulated rows all equal to its shift1;
    # with no rotary and every tile selected (dense), those rows' queries are equal, so
    # their attention outputs are equal too, while the other modality's are not
    for table, rows, other in (("mod_prefix", slice(0, 128), slice(128, None)),
                               ("mod", slice(128, None), slice(0, 128))):
        shape = _tiny_shape(rope=False, pooled=False, topk=3, prefix_mod=True)
        w = _weights(shape)
        w[table][1] = -1.0
        x = S.bf16_bits_to_f64(S.hidden_rows(shape, 5))
        o = O.block_forward(x, w, shape)["o_f64"]
        assert np.allclose(o[rows], o[rows][:1], atol=1e-12, rtol=0)
        assert np.abs(o[other] - o[other][:1]).max() > 1e-3


def test_block_prefix_table_equal_to_shared_table():
    shape = _tiny_shape(prefix_mod=True)
    w = _weights(shape)
    w["mod_prefix"] = w["mod"].copy()
    x = S.bf16_bits_to_f64(S.hidden_rows(shape, 6))
    a = O.block_forward(x, w, shape)["x2"]
    w.pop("mod_prefix")
    assert np.array_equal(a, O.block_forward(x, w, shape)["x2"])


def test_block_rows_equals_full_block_with_prefix_table():
    shape = _tiny_shape(prefix_mod=True, mlp="swiglu")
    w = _weights(shape)
    x = S.bf16_bits_to_f64(S.hidden_rows(shape, 4))
    full = O.block_forward(x, w, shape)
    rows = [0, 64, 127, 128, 200, shape.n_rows - 1]
    part = O.block_forward_rows(x, w, shape, rows)
    ref = full["x2"][rows]
    assert np.all(np.abs(part["x2"] - ref) <= np.abs(ref) * 2.0 ** -7)
    assert np.mean(part["x2"] == ref) > 0.99


# --------------------------------------------------------------------------- denoiser
def test_euler_power_of_two_exact():
    z = rng.standard_normal(1000).astype(np.float32)
    v = O.bf16(rng.standard_normal(1000))
    got = O.euler_update(z, v, -0.125)
    want = (z.astype(np.float32) + np.float32(-0.125) * v.astype(np.float32))  # exact product
    assert np.array_equal(got, want.astype(np.float64))


def test_extrapolation_exact_for_linear_velocity():
    a, b = rng.standard_normal(50), rng.standard_normal(50)
    v = lambda s: a + b * s  # noqa: E731
    got = O.extrapolate(v(0.7), v(0.8), 0.65, 0.7, 0.8)
    assert np.allclose(got, v(0.65), atol=1e-13)


def test_euler_and_extrapolation_per_modality_rows():
    P = 3
    z = np.zeros((7, 4))
    got = O.euler_update(z, np.ones((7, 4)), -0.25, -0.5, P)
    assert np.all(got[:P] == -0.5) and np.all(got[P:] == -0.25)
    # velocities linear in each modality's own sigma are extrapolated exactly
    a, b = rng.standard_normal((7, 4)), rng.standard_normal((7, 4))
    sv, sp = (0.65, 0.7, 0.8), (0.5, 0.55, 0.7)
    va = np.where(np.arange(7)[:, None] < P, a + b * sp[1], a + b * sv[1])
    vb = np.where(np.arange(7)[:, None] < P, a + b * sp[2], a + b * sv[2])
    got = O.extrapolate(va, vb, *sv, prefix=sp, n_prefix=P)
    assert np.allclose(got[:P], (a + b * sp[0])[:P], atol=1e-13)
    assert np.allclose(got[P:], (a + b * sv[0])[P:], atol=1e-13)


def test_sigma_schedule_shift_endpoints_and_composition():
    for n in (1, 4, 30):
        for s in (1.0, 0.5, 3.0, 5.0):
            sig = O.sigma_schedule(n, s)
            assert sig[0] == 1.0 and sig[-1] == 0.0 and np.all(np.diff(sig) < 0)
    assert np.array_equal(O.sigma_schedule(8), 1 - np.arange(9) / 8)
    # a larger shift keeps more of the run at high noise: every interior sigma rises
    assert np.all(O.sigma_schedule(10, 3.0)[1:-1] > O.sigma_schedule(10)[1:-1])
    # the map t -> s t / (1 + (s - 1) t) composes multiplicatively in s (a Moebius family)
    t = O.sigma_schedule(12)
    f = lambda s, u: s * u / (1 + (s - 1) * u)  # noqa: E731
    assert np.allclose(f(2.0, f(1.5, t)), O.sigma_schedule(12, 3.0), atol=1e-15)
    assert np.allclose(O.sigma_schedule(12, 0.25), f(0.5, f(0.5, t)), atol=1e-15)


def test_denoise_loop_per_modality_without_blocks():
    # with no blocks v = bf16(z) and the rows are independent: each modality follows the
    # Euler product prod(1 + dt_i) of its own schedule up to bf16/fp32 rounding
    class Shp:
        n_prefix = 5
    n = 6
    z0 = rng.standard_normal((12, 8)).astype(np.float32).astype(np.float64)
    sv, sp = O.sigma_schedule(n), O.sigma_schedule(n, 3.0)
    out = O.denoise_loop(z0, [], Shp, n, 1, [], sig_video=sv, sig_prefix=sp)
    for rows, sig in ((slice(0, 5), sp), (slice(5, None), sv)):
        want = z0[rows] * np.prod(1 + np.diff(sig))
        assert np.allclose(out["z"][rows], want, rtol=n * 2.0 ** -8, atol=0)
    # reuse 2: the video rows do not depend on the prefix schedule, and equal sigmas give
    # the default run
    a = O.denoise_loop(z0, [], Shp, n, 2, [], sig_video=sv, sig_prefix=sp)
    b = O.denoise_loop(z0, [], Shp, n, 2, [], sig_video=sv, sig_prefix=sv)
    c = O.denoise_loop(z0, [], Shp, n, 2, [])
    assert np.array_equal(a["z"][5:], b["z"][5:]) and np.array_equal(b["z"], c["z"])
    assert not np.array_equal(a["z"][:5], b["z"][:5])


def test_fresh_step_counts_golden():
    with open(os.path.join(GOLDEN, "reuse_fresh_counts.txt")) as f:
        rows = [list(map(int, ln.split())) for ln in f if ln.strip() and not ln.startswith("#")]
    assert rows
    for n, r, want in rows:
        steps = O.fresh_steps(n, r)
        assert len(steps) == want and steps[0] == 0 and steps[-1] == n - 1


def test_thin_layers_hand_example():
    D = 4
    g = [5.0, 1.0, 3.0, 1.0, 0.5, 9.0]  # block 4 smallest, blocks 1 and 3 tie
    mods = []
    for s in g:
        m = np.zeros((6, D))
        m[2, 0] = s
        mods.append(m)
    assert O.thin_layers(mods, 6) == [0, 1, 2, 3, 4, 5]
    assert O.thin_layers(mods, 5) == [0, 1, 2, 3, 5]
    assert O.thin_layers(mods, 4) == [0, 1, 2, 5]      # tie 1 vs 3: the higher (3) goes first
    assert O.thin_layers(mods, 3) == [0, 2, 5]
    assert O.thin_layers(mods, 2) == [0, 5]


def test_block_rows_equals_full_block():
    # the sampled evaluation must reproduce the full evaluation on the sampled rows exactly
    shape = _tiny_shape()
    w = _weights(shape)
    x = S.bf16_bits_to_f64(S.hidden_rows(shape, 4))
    full = O.block_forward(x, w, shape)
    rows = [0, 63, 64, 127, 128, 200, shape.n_rows - 1]
    part = O.block_forward_rows(x, w, shape, rows)
    # the same arithmetic; only BLAS blocking of a 1-row vs a 64-row product may differ
    # in the last float64 bit, which can move a bf16 rounding by one ulp
    ref = full["x2"][rows]
    ulp = np.abs(ref) * 2.0 ** -7
    assert np.all(np.abs(part["x2"] - ref) <= ulp)
    assert np.mean(part["x2"] == ref) > 0.99
    assert np.array_equal(part["idx"], full["idx"])
    # the same with the softmax weights rounded to bf16
    full = O.block_forward(x, w, shape, p_bf16=True)
    part = O.block_forward_rows(x, w, shape, rows, p_bf16=True)
    ref = full["x2"][rows]
    assert np.all(np.abs(part["x2"] - ref) <= np.abs(ref) * 2.0 ** -7)
    assert np.mean(part["x2"] == ref) > 0.99


def test_denoise_loop_orchestration_without_blocks():
    # with no blocks the velocity is bf16(z): check which velocities and sigmas the loop
    # combines, step by step, against a hand-written schedule for n = 8, reuse = 2
    z0 = rng.standard_normal(64).astype(np.float32).astype(np.float64)
    out = O.denoise_loop(z0, [], None, 8, 2, [])
    assert out["fresh"] == [0, 2, 4, 6, 7]
    z = z0.copy()
    sig = [1 - i / 8 for i in range(9)]
    hist = []
    for i in range(8):
        if i in (0, 2, 4, 6, 7):
            v = O.bf16(z)
            hist.append((sig[i], v))
        else:
            (sa, va), (sb, vb) = hist[-1], (hist[-2] if len(hist) > 1 else hist[-1])
            v = va if len(hist) == 1 else va + (va - vb) * (sig[i] - sa) / (sa - sb)
        z = (z + (-0.125) * v).astype(np.float32).astype(np.float64)
    assert np.array_equal(out["z"], z)
    # step 1 holds the single fresh velocity; step 3 extrapolates from passes 2 and 0
    assert abs((sig[3] - sig[2]) / (sig[2] - sig[0]) - 0.5) < 1e-15  # v = v2 + 0.5 (v2 - v0)


# --------------------------------------------------------------------------- both ends
def test_patch_in_small_integers_brute_force():
    z = rng.integers(-4, 5, (5, 32)).astype(np.float64)
    w = rng.integers(-4, 5, (32, 16)).astype(np.float64)
    b = rng.integers(-4, 5, 16).astype(np.float64)
    got = O.patch_in(z, w, b)
    for r in range(5):
        for c in range(16):
            acc = b[c]
            for j in range(32):
                acc += z[r, j] * w[j, c]  # input-major weights: w[j, c]
            assert got[r, c] == O.bf16(acc)


def test_output_head_constant_rows():
    # scale = -1 turns every normalised row into the shift, so every velocity row is
    # W_out bf16(shift) + b
    x = rng.standard_normal((6, 16))
    mod2 = np.stack([rng.standard_normal(16), -np.ones(16)])
    w = O.bf16(rng.standard_normal((4, 16)))
    b = O.bf16(rng.standard_normal(4))
    v = O.output_head(x, mod2, w, b)
    want = O.f32(w @ O.bf16(mod2[0]) + b)
    assert np.array_equal(v, np.tile(want, (6, 1)))


def _ends_case(blocks=2):
    shape = _tiny_shape(n_text=8, n_audio=56, hidden=64, prefix_mod=True)
    ends = S.ends_weights(shape, 5, c_video=32, c_audio=32)
    ends = {k: (S.bf16_bits_to_f64(v) if isinstance(v, np.ndarray) and v.dtype == np.uint16
                else v) for k, v in ends.items()}
    zv, za = S.modality_latents(shape, 6, 32, 32)
    return shape, ends, [_weights(shape, 10 + i) for i in range(blocks)], zv, za


def test_core_reuse_reproduces_the_fresh_velocity():
    # the held residual applied to the same x_0 gives back x_L exactly, so the velocity
    # and the step are the fresh pass's
    shape, ends, blocks, zv, za = _ends_case()
    f = O.sample_step(zv, za, ends, blocks, shape, "fresh", -0.125, -0.25)
    c = O.sample_step(zv, za, ends, blocks, shape, "core", -0.125, -0.25, residual=f["residual"])
    assert np.array_equal(c["xL"], f["xL"])
    for k in ("v_video", "v_audio", "z_video", "z_audio"):
        assert np.array_equal(c[k], f[k])
    assert not np.array_equal(f["xL"], f["x0"])


def test_sample_loop_core_reuse_without_blocks_equals_every_pass_fresh():
    shape, ends, _, zv, za = _ends_case()
    a = O.sample_loop(zv, za, ends, [], shape, 6, core_reuse=3)
    b = O.sample_loop(zv, za, ends, [], shape, 6)
    assert a["fresh"] == [0, 3, 5]
    assert np.array_equal(a["z_video"], b["z_video"]) and np.array_equal(a["z_audio"], b["z_audio"])


def test_sample_step_without_blocks_is_the_heads_of_the_patches():
    # no blocks: x_L = x_0, so each modality's velocity is its head over its own patch rows
    shape, ends, _, zv, za = _ends_case()
    r = O.sample_step(zv, za, ends, [], shape, "fresh", -0.125, -0.25)
    xv = O.patch_in(zv, ends["w_in_video"], ends["b_in_video"])
    xa = O.patch_in(za, ends["w_in_audio"], ends["b_in_audio"])
    assert np.array_equal(r["v_video"], O.output_head(xv, ends["mod_out_video"],
                                                      ends["w_out_video"], ends["b_out_video"]))
    assert np.array_equal(r["v_audio"], O.output_head(xa, ends["mod_out_audio"],
                                                      ends["w_out_audio"], ends["b_out_audio"]))
    assert np.array_equal(r["z_video"], (zv + np.float32(-0.125) * r["v_video"].astype(np.float32)))


# --------------------------------------------------------------------------- token reduction
def _tr_shape(grid=(3, 4, 7)):
    return S.BlockShape(8, 24, int(np.prod(grid)), hidden=16, heads=2, head_dim=8,
                        mlp_width=64, topk=2, video_grid=grid, token_reduction=True)


@pytest.mark.parametrize("grid", [(3, 4, 7), (2, 3, 8), (1, 1, 1), (2, 2, 3)])
def test_token_pool_brute_force_pairs(grid):
    shape = _tr_shape(grid)
    T, Hg, Wg = grid
    P = shape.n_prefix
    x = O.bf16(rng.standard_normal((shape.n_rows, 16)))
    xr, base = O.token_pool(x, shape)
    Wr = (Wg + 1) // 2
    assert xr.shape[0] == P + T * Hg * Wr and np.array_equal(xr[:P], x[:P])
    for t in range(T):
        for h in range(Hg):
            for j in range(Wr):
                a = x[P + (t * Hg + h) * Wg + 2 * j]
                want = a if 2 * j + 1 == Wg else O.bf16(
                    O.f32(a + x[P + (t * Hg + h) * Wg + 2 * j + 1]) * 0.5)
                assert np.array_equal(xr[P + (t * Hg + h) * Wr + j], want)
    assert np.array_equal(base, xr[P:])


def test_token_restore_identity_and_pair_update():
    shape = _tr_shape()
    P = shape.n_prefix
    x = O.bf16(rng.standard_normal((shape.n_rows, 16)))
    xr, base = O.token_pool(x, shape)
    assert np.array_equal(O.token_restore(x, xr, base, shape), x)  # nothing learned
    # a pair's update reaches both of its tokens; text/audio rows come from the reduced rows
    y = xr.copy()
    y[:P] += 1.0
    y[P + 5] += 0.25  # reduced row 5 = (t 0, h 1, j 1): full columns 2 and 3 of row (0, 1)
    out = O.token_restore(x, y, base, shape)
    assert np.array_equal(out[:P], y[:P])
    changed = np.nonzero(np.any(out[P:] != x[P:], axis=1))[0]
    assert changed.tolist() == [7 + 2, 7 + 3]
    assert np.allclose(out[P + 9], O.bf16(x[P + 9] + 0.25), atol=0)


def test_rope_coords_pooled_positions():
    c = O.rope_coords_pooled(4, (2, 3, 4), 7)
    assert np.array_equal(c[4:8, 2], [0.5, 2.5, 4.5, 6.0])  # last column of width 7 is alone
    assert np.array_equal(c[4 + 12 + 4 * 2 + 1], [1, 2, 2.5])


def test_run_blocks_reduction_boundaries():
    # first == last is no reduction; an identity block (zero gates) between pool and
    # restore gives back the unreduced run exactly
    shape = _tr_shape()
    blocks = [_weights(shape, 20 + i) for i in range(3)]
    x = S.bf16_bits_to_f64(S.hidden_rows(shape, 3))
    plain = O.run_blocks(x, blocks, shape)
    assert np.array_equal(O.run_blocks(x, blocks, shape, reduction=(1, 1)), plain)
    ident = dict(blocks[1])
    ident["mod"] = ident["mod"].copy()
    ident["mod"][2] = 0.0
    ident["mod"][5] = 0.0
    three = [blocks[0], ident, blocks[2]]
    a = O.run_blocks(x, three, shape, reduction=(1, 2))
    b = O.run_blocks(x, [blocks[0], blocks[2]], shape)
    assert np.array_equal(a, b)
    c = O.run_blocks(x, blocks, shape, reduction=(1, 2))
    assert not np.array_equal(c, plain)


def test_silu_closed_forms():
    assert O.silu(0.0) == 0.0
    x = rng.standard_normal(1000) * 4
    assert np.allclose(O.silu(x) - O.silu(-x), x, rtol=0, atol=1e-13)  # sigmoid(x)+sigmoid(-x)=1
    assert abs(float(O.silu(1.0)) - 0.7310585786300049) < 1e-15  # 1 / (1 + e^-1)
    assert float(O.silu(-800.0)) == 0.0


def test_swiglu_split_layout_and_block():
    F, D = 256, 8
    gate = rng.standard_normal((F, D))
    up = rng.standard_normal((F, D))
    w1 = np.empty((2 * F, D))
    for j in range(F // 128):  # the storage convention written out by loops
        w1[256 * j:256 * j + 128] = gate[128 * j:128 * j + 128]
        w1[256 * j + 128:256 * j + 256] = up[128 * j:128 * j + 128]
    bg, bu = rng.standard_normal(F), rng.standard_normal(F)
    b1 = np.concatenate([np.concatenate([bg[128 * j:128 * j + 128], bu[128 * j:128 * j + 128]])
                         for j in range(F // 128)])
    wg, bg2, wu, bu2 = O.swiglu_split(w1, b1)
    assert np.array_equal(wg, gate) and np.array_equal(wu, up)
    assert np.array_equal(bg2, bg) and np.array_equal(bu2, bu)
    h = rng.standard_normal((3, D))
    u = O.mlp_inner(h, {"w1": w1, "b1": b1}, "swiglu")
    for r in range(3):
        for c in range(0, F, 37):
            a = h[r] @ gate[c] + bg[c]
            b = h[r] @ up[c] + bu[c]
            assert u[r, c] == O.bf16(a / (1 + math.exp(-a)) * b)


# --------------------------------------------------------------------------- added pins
def test_qkv_heads_layout_by_loops():
    # projection columns [Q | K | V | G], each H*d wide and head-major inside: head h of row
    # n is columns h*d .. h*d+d-1 of its slab; q and k are RMS-normed over d, scaled by the
    # learned weight, then turned pair (c, c + d/2) by n * theta^(-2c/d) as a complex product
    H, d, N, eps, theta = 3, 8, 5, 1e-6, 10000.0
    A = H * d
    qkvg = O.bf16(rng.standard_normal((N, 4 * A)))
    wq = 1.0 + 0.1 * rng.standard_normal(d)
    wk = 1.0 + 0.1 * rng.standard_normal(d)
    Q, K, V, G = O.qkv_heads(qkvg, H, d, wq, wk, eps, theta)
    assert Q.shape == K.shape == V.shape == (H, N, d) and G.shape == (N, A)
    for h in range(H):
        for n in range(N):
            for slab, w, got in ((0, wq, Q), (1, wk, K)):
                x = [float(t) for t in qkvg[n, slab * A + h * d:slab * A + (h + 1) * d]]
                inv = 1.0 / math.sqrt(sum(t * t for t in x) / d + eps)
                y = [t * inv * float(wi) for t, wi in zip(x, w)]
                zs = [complex(y[c], y[c + d // 2]) * complex(math.cos(n * theta ** (-2 * c / d)),
                                                             math.sin(n * theta ** (-2 * c / d)))
                      for c in range(d // 2)]
                want = O.bf16(np.array([z.real for z in zs] + [z.imag for z in zs]))
                assert np.allclose(got[h, n], want, rtol=2.0 ** -8, atol=0)
            for c in range(d):
                assert V[h, n, c] == qkvg[n, 2 * A + h * d + c]
                assert G[n, h * d + c] == qkvg[n, 3 * A + h * d + c]
    # no norm weights and no rotary: plain head-major slices
    Q0, K0, _, _ = O.qkv_heads(qkvg, H, d, None, None, eps, theta, use_rope=False)
    for h in range(H):
        assert np.array_equal(Q0[h], qkvg[:, h * d:(h + 1) * d])
        assert np.array_equal(K0[h], qkvg[:, A + h * d:A + (h + 1) * d])


def _mlp_row_by_loops(h2row, w, mlp):
    # the MLP of one row written out: fc1 (+ bias), activation, bf16 mid, fc2 (+ bias)
    D = len(h2row)
    w1, b1, w2, b2 = w["w1"], w["b1"], w["w2"], w["b2"]
    F = w2.shape[1]

    def fc1(r):
        return float(b1[r]) + sum(float(w1[r, c]) * float(h2row[c]) for c in range(D))
    u = []
    for j in range(F):
        if mlp == "swiglu":  # gate row 256*(j//128) + j%128, its up row 128 further on
            rg = 256 * (j // 128) + j % 128
            a, b = fc1(rg), fc1(rg + 128)
            u.append(a / (1.0 + math.exp(-a)) * b)
        else:
            a = fc1(j)
            u.append(0.5 * a * (1.0 + math.erf(a / math.sqrt(2.0))))
    u = O.bf16(np.array(u))
    return np.array([float(b2[o]) + sum(float(w2[o, j]) * float(u[j]) for j in range(F))
                     for o in range(w2.shape[0])])


@pytest.mark.parametrize("mlp", ["gelu", "swiglu"])
def test_block_mlp_half_closed_form(mlp):
    # gate1 = 0 leaves x1 = x; scale2 = -1 makes every h2 row bf16(shift2), so every row
    # gets the same MLP output m and x2 = bf16(x + gate2 * m): pins the second norm's table
    # rows, the MLP's biases, activation and bf16 mid, and the second gated residual
    shape = _tiny_shape(hidden=64, mlp_width=128, mlp=mlp)
    w = _weights(shape, 21)
    w["mod"][2] = 0.0
    w["mod"][4] = -1.0
    x = S.bf16_bits_to_f64(S.hidden_rows(shape, 9))
    out = O.block_forward(x, w, shape)
    assert np.array_equal(out["x1"], x)
    m = _mlp_row_by_loops(O.bf16(w["mod"][3]), w, mlp)
    want = O.bf16(x + w["mod"][5] * m[None, :])
    got = out["x2"]
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -8)
    assert np.mean(got == want) > 0.99


def test_denoise_forward_closed_forms():
    # blocks with zero gates are the identity on bf16 rows, so v = bf16(z) and
    # z' = fp32(z + dt v); with dt = -1/8 the product is exact
    shape = _tiny_shape()
    z = rng.standard_normal((shape.n_rows, shape.hidden)).astype(np.float32).astype(np.float64)
    blocks = []
    for i in range(3):
        w = _weights(shape, 30 + i)
        w["mod"][2] = 0.0
        w["mod"][5] = 0.0
        blocks.append(w)
    want_v = O.bf16(z)
    want_z = (z.astype(np.float32) + np.float32(-0.125) * want_v.astype(np.float32))
    for blks, ids in (([], None), (blocks, None), (blocks, [2, 0])):
        r = O.denoise_forward(z, blks, shape, -0.125, ids)
        assert np.array_equal(r["v"], want_v)
        assert np.array_equal(r["z"], want_z.astype(np.float64))
    # the text/audio rows step by their own dt
    r = O.denoise_forward(z, [], shape, -0.125, None, dt_prefix=-0.5)
    P = shape.n_prefix
    assert np.array_equal(r["z"][:P], (z[:P].astype(np.float32)
                                       + np.float32(-0.5) * want_v[:P].astype(np.float32)))
    assert np.array_equal(r["z"][P:], want_z[P:])


def test_tile_sets_slices_and_cubes():
    # without a grid: consecutive 64-row slices of the video rows, the last one partial
    sets = O.tile_sets(100, 150, 64)
    assert [list(s) for s in sets] == [list(range(100, 164)), list(range(164, 228)),
                                       list(range(228, 250))]
    # with a grid: the cubes, and shape_tiles picks by the shape's grid field
    shape = S.BlockShape(4, 0, 2 * 3 * 5, hidden=64, heads=1, head_dim=64, mlp_width=256,
                         topk=1, video_grid=(2, 3, 5))
    cubes = O.shape_tiles(shape)
    assert [list(s) for s in cubes] == [list(s) for s in O.cube_tiles(4, (2, 3, 5))]
    assert len(cubes) == 2  # 1 x 1 x 2 cubes of 4 x 4 x 4: w splits into 4 + 1
    assert sorted(np.concatenate(cubes).tolist()) == list(range(4, 34))
    plain = O.shape_tiles(shape.with_(video_grid=None))
    assert [list(s) for s in plain] == [list(range(4, 34))]


def test_reduced_shape_hand_values():
    shape = _tr_shape((3, 2, 5))
    r = O.reduced_shape(shape)
    assert r.video_grid == (3, 2, 3) and r.n_video == 18 and r.pair_w == 5
    assert not r.token_reduction and r.n_prefix == shape.n_prefix
    r2 = O.reduced_shape(_tr_shape((2, 3, 8)))
    assert r2.video_grid == (2, 3, 4) and r2.n_video == 24 and r2.pair_w == 8


def test_pin_table_covers_every_oracle_function():
    # the oracle's header names the pins of every public function; each must exist here
    doc = O.h3block.__doc__
    body = doc[doc.index("PIN TABLE"):doc.index("END PIN TABLE")].splitlines()[1:]
    table, last = {}, None
    for line in body:
        if not line.strip():
            continue
        if line.startswith("    "):  # continuation of the previous entry
            table[last] += [t.strip() for t in line.split(",") if t.strip()]
            continue
        name, tests = line.strip().split(":", 1)
        last = name
        table[name] = [t.strip() for t in tests.split(",") if t.strip()]
    assert set(table) == set(O.h3block.__all__)
    here = globals()
    for name, tests in table.items():
        assert tests, name
        for t in tests:
            assert callable(here.get("test_" + t)), f"{name}: no pin test_{t}"
