"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bars: top-k index sets bit-exact except near-ties (relative gap < 1e-5),
outputs within relative L2 2e-2 and cosine 0.998 of the float64 oracle (plus
tighter per-stage bounds where the arithmetic allows), exact results where the
float arithmetic is exact, and two runs byte-identical.
"""
import numpy as np
import pytest

import oracle
import synthetic as S
from helpers import (assert_close, check_bf16_stage, check_close, compare_topk, dev_bf16,
                     dev_f32, host_f64, log, router_on_gpu_inputs, same_fraction, weights_to_device, weights_to_f64,
                     workspace_views)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def h3():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    import audio_diffusion_transformer_gb300 as pkg
    return pkg


def empty_bf16(*shape):
    return torch.empty(*shape, dtype=torch.bfloat16, device="cuda")


# ----------------------------------------------------------------------------- GEMM
@pytest.mark.parametrize("M,N,K", [(300, 512, 320), (128, 256, 64), (1, 256, 128), (515, 768, 1024)])
def test_linear_small_integers_bit_exact(h3, M, N, K):
    rng = np.random.default_rng(M + N + K)
    a = rng.integers(-8, 9, (M, K)).astype(np.float32)
    w = rng.integers(-8, 9, (N, K)).astype(np.float32)
    b = rng.integers(-8, 9, N).astype(np.float32)
    ad, wd, bd = (dev_bf16(S.to_bf16_bits(x)) for x in (a, w, b))
    y = empty_bf16(M, N)
    h3.linear(ad, wd, bd, y)
    torch.cuda.synchronize()
    want = oracle.bf16(oracle.linear(a, w, b))  # fp32 sums of small integers are exact
    assert np.array_equal(host_f64(y), want)
    y2 = empty_bf16(M, N)
    h3.linear(ad, wd, None, y2)
    assert np.array_equal(host_f64(y2), oracle.bf16(oracle.linear(a, w)))


def test_linear_pair_tiles_bit_exact(h3):
    """Rows enough for 256-row pair tiles (38 bands at 152 SMs), the 128-row tiles after
    them and a ragged last block: exact on small integers."""
    M, N, K = 15360 + 37, 1024, 192
    rng = np.random.default_rng(7)
    a = rng.integers(-8, 9, (M, K)).astype(np.float32)
    w = rng.integers(-8, 9, (N, K)).astype(np.float32)
    ad, wd = (dev_bf16(S.to_bf16_bits(x)) for x in (a, w))
    y = empty_bf16(M, N)
    h3.linear(ad, wd, None, y)
    torch.cuda.synchronize()
    assert np.array_equal(host_f64(y), oracle.bf16(oracle.linear(a, w)))


def test_linear_random_close(h3):
    M, N, K = 1000, 1024, 3072
    a = S.normal_bf16(5, "a", (M, K))
    w = S.normal_bf16(5, "w", (N, K), std=0.02)
    y = empty_bf16(M, N)
    h3.linear(dev_bf16(a), dev_bf16(w), None, y)
    torch.cuda.synchronize()
    ref = oracle.linear(S.bf16_bits_to_f64(a), S.bf16_bits_to_f64(w))
    got = host_f64(y)
    assert_close(got, ref, "linear", rel=4e-3, cos=0.99999)
    # within one bf16 ulp of the exact value almost everywhere
    ulp = np.abs(ref) * 2.0 ** -8 + 1e-30
    assert np.mean(np.abs(got - ref) <= ulp) > 0.999


@pytest.mark.parametrize("M,N,K", [(1, 256, 64), (255, 512, 192), (15435, 768, 320),
                                   (4097, 1024, 1280), (515, 512, 5120),
                                   # 1,220 tiles: a short last round on 76 SM pairs
                                   (15435, 5120, 512), (15435, 5120, 4608)])
def test_linear_cta_pairs_equal_one_sm_kernel(h3, M, N, K):
    """The cluster-pair GEMM (256 x 256 tiles over two SMs; eight epilogue warps for
    K <= 4,096, four above) and the one-SM kernel sum in the same order: byte-identical
    outputs on random inputs, ragged rows included."""
    a = S.normal_bf16(M + K, "a", (M, K))
    w = S.normal_bf16(M + K, "w", (N, K), std=0.02)
    b = S.normal_bf16(M + K, "b", (N,), std=0.02)
    ad, wd, bd = dev_bf16(a), dev_bf16(w), dev_bf16(b)
    outs = []
    prev = h3.gemm_cta_pairs(-1)
    try:
        for pairs in (1, 0):
            h3.gemm_cta_pairs(pairs)
            y = empty_bf16(M, N)
            h3.linear(ad, wd, bd, y)
            torch.cuda.synchronize()
            outs.append(y.view(torch.int16).clone())
    finally:
        h3.gemm_cta_pairs(prev)
    assert torch.equal(outs[0], outs[1])


# ----------------------------------------------------------------------------- attention
def run_attention(h3, shp, inp, with_gate=True, flags=None):
    cs = h3.attn_shape(shp, flags)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    q, k, v = (dev_bf16(inp[n]) for n in ("q", "k", "v"))
    g = dev_bf16(inp["gate"]) if with_gate else None
    tv, ks = shp.n_video_tiles, min(shp.topk, shp.n_video_tiles)
    out = empty_bf16(shp.n_rows, shp.attn_width)
    idx = torch.empty(shp.heads, tv, ks, dtype=torch.int32, device="cuda")
    sc = torch.empty(shp.heads, tv, tv, dtype=torch.float32, device="cuda")
    pooled = torch.empty(shp.heads, tv, shp.head_dim, dtype=torch.float32, device="cuda")
    h3.routed_attention(cs, q, k, v, g, out, ws, pooled=pooled, idx=idx, scores=sc)
    torch.cuda.synchronize()
    assert h3.sync_status(ws) == 0
    return {"o": host_f64(out), "idx": idx.cpu().numpy(), "scores": sc.cpu().double().numpy(),
            "pooled": pooled.cpu().double().numpy(), "out_t": out}


def oracle_attention(shp, inp, with_gate=True, pooled=True, p_bf16=False):
    q, k, v = (S.bf16_bits_to_f64(inp[n]) for n in ("q", "k", "v"))
    g = S.bf16_bits_to_f64(inp["gate"]) if with_gate else None
    return oracle.attention_layer(q, k, v, g, shp.n_prefix, shp.n_video, shp.topk, shp.tile,
                                  pooled, p_bf16)


ATTN_CASES = [
    # (name, shape, structured)
    ("tiny_k4", S.ATTN_TINY.shape, 0.0),
    ("tiny_k4_structured", S.ATTN_TINY.shape, 0.5),
    ("tiny_k16_dense", S.ATTN_TINY.shape.with_(topk=16), 0.0),
    ("prefix_ragged_d128", S.BlockShape(64, 64, 300, hidden=256, heads=2, head_dim=128,
                                        mlp_width=1024, topk=2), 0.3),
    ("prefix_odd_tiles_d64", S.BlockShape(128, 64, 5 * 64 + 1, hidden=256, heads=3, head_dim=64,
                                          mlp_width=1024, topk=3), 0.3),
]


@pytest.mark.parametrize("name,shp,structured", ATTN_CASES, ids=[c[0] for c in ATTN_CASES])
def test_routed_attention_matches_oracle(h3, name, shp, structured):
    inp = S.attention_inputs(shp, 0x48334455, structured=structured)
    got = run_attention(h3, shp, inp)
    ref = oracle_attention(shp, inp)
    ks = min(shp.topk, shp.n_video_tiles)
    assert np.allclose(got["scores"], ref["scores"], rtol=1e-4, atol=1e-6)
    n_tie = compare_topk(got["idx"], ref["idx"], ref["scores"], ks)
    if n_tie:  # recompute the oracle with the GPU's selections where near-ties differ
        q, k, v = (S.bf16_bits_to_f64(inp[n]) for n in ("q", "k", "v"))
        O = oracle.routed_attention(q, k, v, shp.n_prefix, shp.n_video, got["idx"], shp.tile)
        ref["o_f64"] = oracle.gate_mix(O, S.bf16_bits_to_f64(inp["gate"]), ref["pooled"],
                                       shp.n_prefix, shp.n_video, shp.tile)
    assert np.allclose(got["pooled"], ref["pooled"], rtol=1e-4, atol=1e-6)
    check_close(got["o"], ref["o_f64"], name)
    # tighter: against the oracle that also rounds the softmax weights to bf16 (in whole
    # octaves, as the kernel does), which leaves only fp32 sums and the output rounding
    refp = oracle_attention(shp, inp, p_bf16=True)
    if not n_tie:
        check_close(got["o"], refp["o_f64"], name + " (bf16 P)", rel=2e-3, cos=0.999998)
        log(f"{name} (bf16 P): identical bf16 outputs {same_fraction(got['o'], refp['o']):.5f}")


def test_routed_all_tiles_equals_dense_attention(h3):
    shp = S.ATTN_TINY.shape.with_(topk=16)
    inp = S.attention_inputs(shp, 77)
    got = run_attention(h3, shp, inp, with_gate=False)
    q, k, v = (S.bf16_bits_to_f64(inp[n]) for n in ("q", "k", "v"))
    d = shp.head_dim
    dense = np.stack([oracle.attend(q[h], k[h], v[h], 1 / np.sqrt(d)) for h in range(shp.heads)])
    dense = dense.transpose(1, 0, 2).reshape(shp.n_rows, -1)
    assert_close(got["o"], dense, "dense", rel=5e-3, cos=0.99995)


def test_attention_constant_v_and_row_stochastic(h3):
    shp = S.BlockShape(64, 0, 256 + 40, hidden=256, heads=2, head_dim=128, mlp_width=1024, topk=2)
    inp = S.attention_inputs(shp, 9, with_gate=False)
    vrow = S.normal_bf16(9, "vrow", (shp.heads, 1, shp.head_dim))
    inp["v"] = np.ascontiguousarray(np.broadcast_to(vrow, (shp.heads, shp.n_rows, shp.head_dim)))
    got = run_attention(h3, shp, inp, with_gate=False)
    want = np.broadcast_to(S.bf16_bits_to_f64(vrow).transpose(1, 0, 2).reshape(1, -1),
                           got["o"].shape)
    # P rounded to bf16 but l from unrounded P: |o - v| <= 2^-8 |v| per element
    assert np.all(np.abs(got["o"] - want) <= 2.0 ** -8 * np.abs(want) + 1e-6)


def test_attention_running_max_past_2_32(h3):
    # Hand-built scores, in octaves (s / ln 2): every video query tile sees the prefix keys
    # at 0 first.  Query tiles 0 and 2 (direction A) select key tiles 0 and 1, met at ~20
    # and then ~60 octaves: the running maximum must move, O rescaled by 2^-61 between the
    # steps.  Query tiles 1 and 3 (direction B) select key tiles 2 and 3, at ~28 and ~31
    # octaves: the sums of their 64 weights pass 2^32 although no single weight does, and
    # the maximum stays.  Neighbouring tiles select disjoint pairs, so both are routed steps.
    d = 64
    shp = S.BlockShape(64, 0, 256, hidden=256, heads=1, head_dim=d, mlp_width=1024, topk=2)
    N, P = shp.n_rows, shp.n_prefix
    q, k = np.zeros((1, N, d)), np.zeros((1, N, d))
    e_a, e_b = np.zeros(d), np.zeros(d)
    e_a[:16], e_b[16:32] = 1.0, 1.0
    amp = 4.0
    per_unit = amp * 16 / np.sqrt(d) / np.log(2)  # octaves per unit of key amplitude
    for t, e in enumerate((e_a, e_b, e_a, e_b)):
        q[0, P + 64 * t:P + 64 * (t + 1)] = amp * e
    for t, (e, z) in enumerate(((e_a, 20.0), (e_a, 60.0), (e_b, 28.0), (e_b, 31.0))):
        k[0, P + 64 * t:P + 64 * (t + 1)] = (z / per_unit) * e
    v = S.normal(5, "v", (1, N, d))
    inp = {"q": S.to_bf16_bits(q), "k": S.to_bf16_bits(k), "v": S.to_bf16_bits(v)}
    got = run_attention(h3, shp, inp, with_gate=False)
    ref = oracle_attention(shp, inp, with_gate=False, pooled=False)
    assert np.array_equal(got["idx"][0], [[0, 1], [2, 3], [0, 1], [2, 3]])
    assert np.array_equal(ref["idx"], got["idx"])
    assert np.all(np.isfinite(got["o"]))
    check_close(got["o"], ref["o_f64"], "running max past 2^32")
    refp = oracle_attention(shp, inp, with_gate=False, pooled=False, p_bf16=True)
    check_close(got["o"], refp["o_f64"], "running max past 2^32 (bf16 P)", rel=2e-3,
                cos=0.999998)


def test_topk_nan_and_tie_rule(h3):
    # identical K tiles 1 and 2 give equal scores for every query: the lower tile must win
    shp = S.BlockShape(0, 0, 64 * 6, hidden=256, heads=1, head_dim=64, mlp_width=1024, topk=2)
    inp = S.attention_inputs(shp, 3, structured=0.5, with_gate=False)
    k = inp["k"].copy()
    k[:, 128:192] = k[:, 64:128]
    inp["k"] = k
    got = run_attention(h3, shp, inp, with_gate=False)
    ref = oracle_attention(shp, inp, with_gate=False, pooled=False)
    assert np.array_equal(got["idx"], ref["idx"])
    # NaN rows: a NaN in K's tile mean ranks as -inf and never adds a tile
    k[:, 64 * 3 + 5, 7] = np.uint16(0x7FC0)
    inp["k"] = k
    got = run_attention(h3, shp, inp, with_gate=False)
    ref = oracle_attention(shp, inp, with_gate=False, pooled=False)
    assert np.array_equal(got["idx"], ref["idx"])
    assert not np.any(got["idx"] == 3)


def test_attention_deterministic(h3):
    shp = ATTN_CASES[3][1]
    inp = S.attention_inputs(shp, 21, structured=0.3)
    a = run_attention(h3, shp, inp)["out_t"]
    b = run_attention(h3, shp, inp)["out_t"]
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ----------------------------------------------------------------------------- block
def run_block(h3, shp, seed, x_bits=None, wts=None, keep=False):
    w = wts if wts is not None else S.block_weights(shp, seed)
    xb = x_bits if x_bits is not None else S.hidden_rows(shp, seed)
    cs = h3.make_shape(shp)
    if keep:
        cs = h3.make_shape(shp, cs.flags | h3.H3DIT_KEEP_INTERMEDIATES)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    x = dev_bf16(xb)
    h3.block_forward(cs, weights_to_device(w), x, ws)
    torch.cuda.synchronize()
    assert h3.sync_status(ws) == 0
    if keep:
        return x, w, xb, workspace_views(h3, cs, shp, ws)
    return x, w, xb


def check_block(h3, shp, seed, name, intermediates=True):
    """One block with its intermediates kept, against the oracle that rounds the softmax
    weights to bf16 (TensorFold #949 "Precision").

    * Router on identical inputs: the oracle's selections from the GPU's own q and k
      must equal the GPU's except near-ties.  (The GPU's q and k differ from the
      oracle's own in about 0.1% of their bf16 roundings, which can move selections
      whose scores are close; the whole-block oracle therefore attends over the GPU's
      selections, the comparison rule for differing selections.)
    * The chain: x2 overall, and the block's own updates x1 - x and x2 - x at the
      required bar (rel L2 2e-2, cos 0.998); q, k, v, g, the attention output o, h2 and
      u element by element.
    * Each stage given the GPU's own input to it: attention from the GPU's q, k, v, g;
      the out projection's x1 from the GPU's o; h2 and u from the GPU's x1; x2 from the
      GPU's x1 and u -- these leave only fp32-vs-fp64 sums: at least 99.5% of the bf16
      outputs identical to the oracle's, every one within one bf16 spacing (plus 2^-12
      of the tensor's RMS where a sum cancels to near zero).
    Keeping the intermediates must not change x2."""
    import oracle.h3block as OB
    x, w, xb, it = run_block(h3, shp, seed, keep=True)
    x0 = S.bf16_bits_to_f64(xb)
    wo = weights_to_f64(w)
    n_tie = router_on_gpu_inputs(it["q"], it["k"], shp, it["idx"])
    ref = oracle.block_forward(x0, wo, shp, p_bf16=True, idx=it["idx"])
    n_own = int(np.any(it["idx"] != ref["idx"], axis=-1).sum())
    log(f"{name}: selections differing from the oracle's own q/k: {n_own}; "
        f"near-ties differing on the GPU's q/k: {n_tie}")
    got = host_f64(x)
    check_close(got, ref["x2"], name + " x2", rel=2e-3, cos=0.99999)
    check_close(it["x1"] - x0, ref["x1"] - x0, name + " x1 - x", rel=2e-2, cos=0.998)
    check_close(got - x0, ref["x2"] - x0, name + " x2 - x", rel=2e-2, cos=0.998)
    if intermediates:
        for n in ("q", "k", "v", "g", "o", "h2", "u"):
            check_close(it[n], ref[n], f"{name} {n}", rel=3e-3, cos=0.99999)
            log(f"{name} {n}: identical bf16 values {same_fraction(it[n], ref[n]):.5f}")
    # stage by stage, from the GPU's own input to each stage
    rows = np.arange(shp.n_rows)
    P = shp.n_prefix
    att = oracle.attention_layer(it["q"], it["k"], it["v"], it["g"] if shp.pooled else None,
                                 P, shp.n_video, shp.topk, shp.tile, shp.pooled, True,
                                 oracle.shape_tiles(shp), it["idx"])
    check_close(it["o"], att["o_f64"], name + " o given q, k, v, g", rel=2e-3, cos=0.999998)
    x1 = oracle.bf16(x0 + OB.gate_rows(wo["mod"], wo.get("mod_prefix"), P, 2, rows)
                     * oracle.linear(it["o"], wo["w_o"], wo["b_o"]))
    check_bf16_stage(it["x1"], x1, name + " x1 given o")
    h2 = OB.modulate_rows(it["x1"], wo["mod"], wo.get("mod_prefix"), P, 3, 4, shp.rms_eps)
    check_bf16_stage(it["h2"], h2, name + " h2 given x1")
    u = oracle.mlp_inner(it["h2"], wo, shp.mlp)
    check_bf16_stage(it["u"], u, name + " u given h2")
    x2 = oracle.bf16(it["x1"] + OB.gate_rows(wo["mod"], wo.get("mod_prefix"), P, 5, rows)
                     * oracle.linear(it["u"], wo["w2"], wo["b2"]))
    check_bf16_stage(got, x2, name + " x2 given x1, u")
    plain = run_block(h3, shp, seed, wts=w)[0]
    assert torch.equal(plain.view(torch.int16), x.view(torch.int16)), "keep mode changed x2"
    return got, ref, x0


BLOCK_CASES = [
    ("tiny_d128", S.BlockShape(64, 64, 192 + 17, hidden=256, heads=2, head_dim=128,
                               mlp_width=1024, topk=2)),
    ("tiny_d64_norope", S.BlockShape(0, 128, 300, hidden=512, heads=4, head_dim=64,
                                     mlp_width=1024, topk=3, rope=False)),
    ("tiny_dense_nopool", S.BlockShape(64, 0, 256, hidden=256, heads=2, head_dim=128,
                                       mlp_width=512, topk=8, pooled=False)),
]


@pytest.mark.parametrize("name,shp", BLOCK_CASES, ids=[c[0] for c in BLOCK_CASES])
def test_block_forward_small(h3, name, shp):
    got, _, x0 = check_block(h3, shp, 31, name)
    # against the exact-weight oracle the required bar still holds
    ref = oracle.block_forward(x0, weights_to_f64(S.block_weights(shp, 31)), shp)
    check_close(got - x0, ref["x2"] - x0, name + " x2 - x (exact weights)", rel=3e-2, cos=0.999)


def test_block_forward_4096_rows(h3):
    wl = S.BLOCK_4K
    check_block(h3, wl.shape, wl.seed, "block 4096")


@pytest.mark.parametrize("case", ["gelu_d128", "norope_d64", "swiglu_prefix_table", "block_4096"])
def test_block_cta_pairs_equal_one_sm_kernel(h3, case):
    """Every epilogue of the block (q/k norm + rotary + head layout for d 64 and 128,
    GELU, SwiGLU, gated residual with a prefix table) gives the same bytes on the
    cluster-pair GEMM as on the one-SM kernel, from tiny shapes to the 4,096-row block."""
    shp = {"gelu_d128": BLOCK_CASES[0][1], "norope_d64": BLOCK_CASES[1][1],
           "swiglu_prefix_table": SWIGLU_CASES[0][1].with_(prefix_mod=True),
           "block_4096": S.BLOCK_4K.shape}[case]
    w = S.block_weights(shp, 91)
    outs = []
    prev = h3.gemm_cta_pairs(-1)
    try:
        for pairs in (1, 0):
            h3.gemm_cta_pairs(pairs)
            outs.append(run_block(h3, shp, 91, wts=w)[0].view(torch.int16).clone())
    finally:
        h3.gemm_cta_pairs(prev)
    assert torch.equal(outs[0], outs[1])


def test_block_forward_deterministic(h3):
    shp = BLOCK_CASES[0][1]
    a = run_block(h3, shp, 5)[0]
    b = run_block(h3, shp, 5)[0]
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_block_work_counters_need_no_zeroed_workspace(h3):
    """The kernels' work counters in the workspace's status block (the attention unit
    counter and the projection GEMMs' tile counters) are zeroed by the block's own
    kernels and reset by the last CTA pair of every GEMM launch: a workspace whose
    status block holds garbage (status word aside) gives the same bytes as a zeroed one,
    and repeated calls on one workspace give the same bytes each time.  The 4,096-row
    block's projections have 192-768 tiles on at most 76 SM pairs, so the counter hands
    out most of them."""
    shp = S.BLOCK_4K.shape
    seed = 9
    w = weights_to_device(S.block_weights(shp, seed))
    xb = S.hidden_rows(shp, seed)
    cs = h3.make_shape(shp)
    nbytes = h3.workspace_bytes(cs)
    status_at = h3.workspace_layout(cs)["status"]

    def run(ws):
        x = dev_bf16(xb)
        h3.block_forward(cs, w, x, ws)
        torch.cuda.synchronize()
        assert h3.sync_status(ws) == 0
        return x.view(torch.int16).clone()

    ref = run(torch.zeros(nbytes, dtype=torch.uint8, device="cuda"))
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    words = ws[status_at:status_at + 256].view(torch.int32)
    words[1:] = torch.tensor(0x3FFFFFFF, dtype=torch.int32)  # every counter word
    for _ in range(3):
        assert torch.equal(run(ws), ref)


# ----------------------------------------------------------------------------- denoiser
def test_denoise_fresh_and_extrapolated_steps(h3):
    shp = BLOCK_CASES[0][1]
    blocks = [S.block_weights(shp, 100 + b) for b in range(3)]
    dblocks = [weights_to_device(b) for b in blocks]
    z0 = S.latents(shp, 7)
    z = dev_f32(z0)
    ring = torch.zeros(2, shp.n_rows, shp.hidden, dtype=torch.float32, device="cuda")
    cs = h3.make_shape(shp)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    ids = [0, 2]
    sig = oracle.sigma_schedule(4)
    dt = -0.25
    # step 0 fresh, step 1 fresh, step 2 skipped (extrapolated), step 3 fresh
    wo = [weights_to_f64(b) for b in blocks]
    zr = z0.astype(np.float64)
    vs = []
    n_fresh = 0
    for i, fresh in enumerate([True, True, False, True]):
        if fresh:
            h3.denoise_step(cs, dblocks, ids, z, ring, True, (sig[i], 0, 0, dt), n_fresh, ws)
            r = oracle.denoise_forward(zr, wo, shp, dt, ids)
            vs.append((sig[i], r["v"]))
            zr = r["z"]
            n_fresh += 1
        else:
            h3.denoise_step(cs, dblocks, ids, z, ring, False, (sig[i], vs[-1][0], vs[-2][0], dt),
                            n_fresh, ws)
            vh = oracle.extrapolate(vs[-1][1], vs[-2][1], sig[i], vs[-1][0], vs[-2][0])
            zr = oracle.euler_update(zr, vh, dt)
        torch.cuda.synchronize()
        assert h3.sync_status(ws) == 0
        got = z.cpu().double().numpy()
        assert_close(got, zr, f"z after step {i}", rel=2e-3, cos=0.99999)
        # the ring holds the most recent fresh velocity exactly as fp32 of the bf16 rows
        slot = (n_fresh - 1) % 2
        vring = ring[slot].cpu().double().numpy()
        assert_close(vring, vs[-1][1], f"v ring step {i}", rel=2e-2, cos=0.998)


def test_euler_step_bit_exact_given_velocity(h3):
    # with zero blocks the velocity is bf16(z) itself, and z + (-1/8) v is exact in fp32
    shp = BLOCK_CASES[0][1]
    z0 = S.latents(shp, 8)
    z = dev_f32(z0)
    ring = torch.zeros(2, shp.n_rows, shp.hidden, dtype=torch.float32, device="cuda")
    cs = h3.make_shape(shp)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    h3.denoise_step(cs, [], [], z, ring, True, (1.0, 0, 0, -0.125), 0, ws)
    torch.cuda.synchronize()
    want = oracle.euler_update(z0, oracle.bf16(z0.astype(np.float64)), -0.125)
    assert np.array_equal(z.cpu().double().numpy(), want)


def test_denoise_loop_reuse_and_layer_thinning(h3):
    """Six Euler steps with reuse 2 (fresh passes 0, 2, 4, 5) over 3 of 4 blocks chosen
    by layer thinning, driven through h3dit_denoise_step, against the oracle's loop."""
    shp = BLOCK_CASES[0][1]
    blocks = [S.block_weights(shp, 300 + b) for b in range(4)]
    ids = h3.select_blocks(np.stack([b["mod"] for b in blocks]), 3)
    assert ids == oracle.thin_layers([b["mod"] for b in blocks], 3)
    z0 = S.latents(shp, 17)
    z = dev_f32(z0)
    ring = torch.zeros(2, shp.n_rows, shp.hidden, dtype=torch.float32, device="cuda")
    cs = h3.make_shape(shp)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    dblocks = [weights_to_device(b) for b in blocks]
    n_steps, reuse = 6, 2
    sig = oracle.sigma_schedule(n_steps)
    fresh = oracle.fresh_steps(n_steps, reuse)
    assert fresh == [0, 2, 4, 5]
    nf, fs = 0, []
    for i in range(n_steps):
        if i in fresh:
            h3.denoise_step(cs, dblocks, ids, z, ring, True, (sig[i], 0, 0, -1 / n_steps), nf, ws)
            nf += 1
            fs.append(sig[i])
        else:
            h3.denoise_step(cs, dblocks, ids, z, ring, False,
                            (sig[i], fs[-1], fs[-2] if len(fs) > 1 else fs[-1], -1 / n_steps),
                            nf, ws)
    torch.cuda.synchronize()
    assert h3.sync_status(ws) == 0
    ref = oracle.denoise_loop(z0, [weights_to_f64(b) for b in blocks], shp, n_steps, reuse, ids)
    assert_close(z.cpu().double().numpy(), ref["z"], "z after the loop", rel=2e-3, cos=0.99999)


SWIGLU_CASES = [
    ("swiglu_attn_wider_than_hidden", S.BlockShape(64, 64, 200, hidden=256, heads=4, head_dim=128,
                                                   mlp_width=384, topk=2, mlp="swiglu")),
    ("swiglu_d64", S.BlockShape(0, 128, 130, hidden=512, heads=4, head_dim=64, mlp_width=256,
                                topk=1, mlp="swiglu")),
]


@pytest.mark.parametrize("name,shp", SWIGLU_CASES, ids=[c[0] for c in SWIGLU_CASES])
def test_block_forward_swiglu_small(h3, name, shp):
    assert shp.attn_width != shp.hidden or shp.head_dim == 64
    check_block(h3, shp, 61, name)


# ----------------------------------------------------------------------------- per-modality
PREFIX_MOD_CASES = [
    ("prefix_table_gelu", BLOCK_CASES[0][1].with_(prefix_mod=True)),
    ("prefix_table_swiglu", SWIGLU_CASES[0][1].with_(prefix_mod=True)),
]


@pytest.mark.parametrize("name,shp", PREFIX_MOD_CASES, ids=[c[0] for c in PREFIX_MOD_CASES])
def test_block_forward_prefix_table(h3, name, shp):
    """Text and audio rows on their own modulation table (norm shift/scale and gates)."""
    assert "mod_prefix" in S.block_weights(shp, 71)
    got, ref, x0 = check_block(h3, shp, 71, name)
    P = shp.n_prefix
    for part, sl in (("prefix", slice(0, P)), ("video", slice(P, None))):
        check_close(got[sl] - x0[sl], ref["x2"][sl] - x0[sl], f"{name} {part} x2 - x",
                    rel=2e-2, cos=0.998)



def test_block_prefix_table_zero_gates_leave_prefix_rows(h3):
    shp = PREFIX_MOD_CASES[0][1]
    w = S.block_weights(shp, 72)
    w["mod_prefix"][2] = 0.0
    w["mod_prefix"][5] = 0.0
    x, _, xb = run_block(h3, shp, 72, wts=w)
    got = x.view(torch.int16).cpu().numpy()
    P = shp.n_prefix
    assert np.array_equal(got[:P], xb[:P].view(np.int16))
    assert not np.array_equal(got[P:], xb[P:].view(np.int16))


def test_denoise_loop_per_modality_schedules(h3):
    """Video rows on the uniform schedule, text/audio rows on a shifted one (shift 3),
    reuse 2 over 5 steps, both modulation tables, against the oracle's loop."""
    shp = PREFIX_MOD_CASES[0][1]
    blocks = [S.block_weights(shp, 400 + b) for b in range(2)]
    ids = [0, 1]
    z0 = S.latents(shp, 19)
    z = dev_f32(z0)
    ring = torch.zeros(2, shp.n_rows, shp.hidden, dtype=torch.float32, device="cuda")
    cs = h3.make_shape(shp)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    dblocks = [weights_to_device(b) for b in blocks]
    n_steps, reuse = 5, 2
    sv, sp = oracle.sigma_schedule(n_steps), oracle.sigma_schedule(n_steps, 3.0)
    fresh = oracle.fresh_steps(n_steps, reuse)
    hist = []
    for i in range(n_steps):
        dv, dp = sv[i + 1] - sv[i], sp[i + 1] - sp[i]
        if i in fresh:
            h3.denoise_step(cs, dblocks, ids, z, ring, True, (sv[i], 0, 0, dv), len(hist), ws,
                            prefix=(sp[i], 0, 0, dp))
            hist.append(i)
        else:
            a, b = hist[-1], hist[-2] if len(hist) > 1 else hist[-1]
            h3.denoise_step(cs, dblocks, ids, z, ring, False, (sv[i], sv[a], sv[b], dv),
                            len(hist), ws, prefix=(sp[i], sp[a], sp[b], dp))
    torch.cuda.synchronize()
    assert h3.sync_status(ws) == 0
    ref = oracle.denoise_loop(z0, [weights_to_f64(b) for b in blocks], shp, n_steps, reuse, ids,
                              sig_video=sv, sig_prefix=sp)
    got = z.cpu().double().numpy()
    P = shp.n_prefix
    assert_close(got[:P], ref["z"][:P], "prefix rows after the loop", rel=2e-3, cos=0.99999)
    assert_close(got[P:], ref["z"][P:], "video rows after the loop", rel=2e-3, cos=0.99999)


def test_euler_per_modality_bit_exact_given_velocity(h3):
    # zero blocks: v = bf16(z); prefix rows step by -1/4, video rows by -1/8, both exact
    shp = BLOCK_CASES[0][1]
    z0 = S.latents(shp, 9)
    z = dev_f32(z0)
    ring = torch.zeros(2, shp.n_rows, shp.hidden, dtype=torch.float32, device="cuda")
    cs = h3.make_shape(shp)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    h3.denoise_step(cs, [], [], z, ring, True, (1.0, 0, 0, -0.125), 0, ws,
                    prefix=(1.0, 0, 0, -0.25))
    torch.cuda.synchronize()
    want = oracle.euler_update(z0, oracle.bf16(z0.astype(np.float64)), -0.125, -0.25,
                               shp.n_prefix)
    assert np.array_equal(z.cpu().double().numpy(), want)
