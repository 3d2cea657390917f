"""Full-size GPU parity at the 15,435-row shape (hidden 5,120, 40 heads x 128,
top-k 16 of 218 video tiles, last video tile 11 rows), in the launch
configuration bench.py times.  The oracle computes sampled outputs one by one
(sampled query tiles and rows); routing is compared over every (head, tile)."""
import time

import numpy as np
import pytest

import oracle
import synthetic as S
from helpers import assert_close, check_bf16_stage, check_close, compare_topk, dev_bf16, dev_f32, host_f64, log, \
    router_on_gpu_inputs, weights_to_device, weights_to_f64, workspace_views

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

WL = S.workload_by_name("block_15435_d5120")
SHAPE = WL.shape


@pytest.fixture(scope="module")
def h3():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    import audio_diffusion_transformer_gb300 as pkg
    return pkg


_log = log


def sample_rows(shp):
    P, N = shp.n_prefix, shp.n_rows
    rows = {0, 1, shp.n_text - 1, shp.n_text, P - 1, P, P + 63, P + 64, N // 2, N - 12, N - 11,
            N - 1}
    return sorted(r for r in rows if 0 <= r < N)


def test_routed_attention_fullsize(h3):
    shp = SHAPE
    t0 = time.time()
    inp = S.attention_inputs(shp, WL.seed)
    q64, k64, v64, g64 = (S.bf16_bits_to_f64(inp[n]) for n in ("q", "k", "v", "gate"))
    _log(f"attention inputs {time.time() - t0:.1f}s")
    cs = h3.attn_shape(shp)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    tv = shp.n_video_tiles
    out = torch.empty(shp.n_rows, shp.attn_width, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(shp.heads, tv, shp.topk, dtype=torch.int32, device="cuda")
    sc = torch.empty(shp.heads, tv, tv, dtype=torch.float32, device="cuda")
    pooled = torch.empty(shp.heads, tv, shp.head_dim, dtype=torch.float32, device="cuda")
    h3.routed_attention(cs, *(dev_bf16(inp[n]) for n in ("q", "k", "v", "gate")), out, ws,
                        pooled=pooled, idx=idx, scores=sc)
    torch.cuda.synchronize()
    assert h3.sync_status(ws) == 0
    t0 = time.time()
    P, Vn = shp.n_prefix, shp.n_video
    mq, mk, mv = (oracle.tile_means(a, P, Vn) for a in (q64, k64, v64))
    Sref = oracle.tile_scores(mq, mk)
    idx_ref = oracle.topk_select(Sref, shp.topk)
    gi = idx.cpu().numpy()
    n_tie = compare_topk(gi, idx_ref, Sref, shp.topk)
    _log(f"router oracle {time.time() - t0:.1f}s, near-tie rows that differ: {n_tie} "
         f"of {shp.heads * tv}")
    assert np.allclose(sc.cpu().numpy(), Sref, rtol=1e-4, atol=1e-6)
    pref = oracle.pooled_branch(Sref, mv, shp.head_dim)
    assert np.allclose(pooled.cpu().double().numpy(), pref, rtol=1e-4, atol=1e-6)
    # sampled outputs: one video query tile of every head (spread over the tile range)
    # plus the partial last tile, using the GPU's selections (identical to the oracle's
    # except counted near-ties); against exact weights at the required bar, and against
    # the oracle that rounds the weights to bf16 in whole octaves, as the kernel does
    tiles = [(h, (37 * h + 11) % tv) for h in range(shp.heads)] + [(39, tv - 1), (20, tv - 2)]
    O = oracle.routed_attention(q64, k64, v64, P, Vn, gi, tiles=tiles)
    Op = oracle.routed_attention(q64, k64, v64, P, Vn, gi, p_bf16=True, tiles=tiles)
    got = host_f64(out)
    worst = 0.0
    d = shp.head_dim
    for h, i in tiles:
        r0, nv = oracle.video_tiles(P, Vn)[i]
        gm = g64[r0:r0 + nv, h * d:(h + 1) * d] * pref[h, i]
        sl = got[r0:r0 + nv, h * d:(h + 1) * d]
        assert_close(sl, O[h, r0:r0 + nv] + gm, f"video tile ({h},{i})")
        r, _ = assert_close(sl, Op[h, r0:r0 + nv] + gm, f"video tile ({h},{i}) bf16 P",
                            rel=2e-3, cos=0.999998)
        worst = max(worst, r)
    _log(f"attention 15,435 rows: {len(tiles)} sampled video tiles over all {shp.heads} heads, "
         f"worst rel L2 against the bf16-weight oracle {worst:.3e}")
    # sampled dense prefix rows
    for r in (0, shp.n_text, P - 1):
        for h in (0, 19, 39):
            d = shp.head_dim
            want = oracle.attend(q64[h, [r]], k64[h], v64[h], 1 / np.sqrt(d))[0]
            assert_close(got[r, h * d:(h + 1) * d], want, f"prefix row {r} head {h}")
    _log(f"attention sampled oracle {time.time() - t0:.1f}s")


def block_sampled(h3, shp, seed, name, rows, perm=None):
    """One block on the device with its intermediates kept, checked on sampled rows
    against the oracle that rounds the softmax weights to bf16: the router against the
    oracle's on the GPU's own q and k (all heads and tiles; equal except near-ties);
    then, with the oracle attending over the GPU's selections, x2 and the block's own
    updates x1 - x and x2 - x at the required bar (rel L2 2e-2, cos 0.998), and the out
    projection given the GPU's attention output.  ``perm`` (cube layouts) maps library
    rows to the oracle's raster rows."""
    import oracle.h3block as OB
    t0 = time.time()
    w = S.block_weights(shp, seed)
    xb = S.hidden_rows(shp, seed)
    _log(f"{name} inputs {time.time() - t0:.1f}s")
    cs = h3.make_shape(shp)
    cs = h3.make_shape(shp, cs.flags | h3.H3DIT_KEEP_INTERMEDIATES)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    x = dev_bf16(xb if perm is None else xb[perm])
    h3.block_forward(cs, weights_to_device(w), x, ws)
    torch.cuda.synchronize()
    assert h3.sync_status(ws) == 0
    lib = workspace_views(h3, cs, shp, ws, ["q", "k", "o", "x1", "idx"])
    del ws
    got = host_f64(x)
    it = dict(lib)
    if perm is not None:
        got = np.empty_like(got)
        got[perm] = host_f64(x)
        for n in ("q", "k"):
            it[n] = np.empty_like(lib[n])
            it[n][:, perm] = lib[n]
        for n in ("o", "x1"):
            it[n] = np.empty_like(lib[n])
            it[n][perm] = lib[n]
    assert np.all(np.isfinite(got))
    t0 = time.time()
    n_tie = router_on_gpu_inputs(it["q"], it["k"], shp, it["idx"])
    x64, wo = S.bf16_bits_to_f64(xb), weights_to_f64(w)
    ref = oracle.block_forward_rows(x64, wo, shp, rows, p_bf16=True, idx=it["idx"])
    n_own = int(np.any(it["idx"] != ref["idx"], axis=-1).sum())
    _log(f"{name} sampled oracle {time.time() - t0:.1f}s; of {shp.heads * shp.n_video_tiles} "
         f"(head, tile) pairs: near-ties differing on the GPU's q/k {n_tie}, selections "
         f"differing from the oracle's own q/k {n_own}")
    r = ref["rows"]
    x0 = x64[r]
    check_close(got[r], ref["x2"], f"{name} x2 (sampled rows)", rel=2e-3, cos=0.99999)
    check_close(it["x1"][r] - x0, ref["x1"] - x0, f"{name} x1 - x (sampled rows)", rel=2e-2,
                cos=0.998)
    check_close(got[r] - x0, ref["x2"] - x0, f"{name} x2 - x (sampled rows)", rel=2e-2,
                cos=0.998)
    x1 = oracle.bf16(x0 + OB.gate_rows(wo["mod"], wo.get("mod_prefix"), shp.n_prefix, 2, r)
                     * oracle.linear(it["o"][r], wo["w_o"], wo["b_o"]))
    check_bf16_stage(it["x1"][r], x1, f"{name} x1 given o (sampled rows)")


def test_block_forward_fullsize_sampled(h3):
    block_sampled(h3, SHAPE, WL.seed, "block 15,435", sample_rows(SHAPE))


def test_block_forward_fullsize_deterministic(h3):
    shp = SHAPE
    w = weights_to_device(S.block_weights(shp, WL.seed + 1))
    xb = S.hidden_rows(shp, WL.seed + 1)
    cs = h3.make_shape(shp)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        x = dev_bf16(xb)
        h3.block_forward(cs, w, x, ws)
        torch.cuda.synchronize()
        outs.append(x.view(torch.int16).clone())
    assert torch.equal(outs[0], outs[1])


def test_denoise_two_blocks_fullsize(h3):
    """The 50-block forward's velocity path, checked on its first 2 blocks:
    v = x_2 after two blocks of bf16(z), then z' = z - v/8 (bit-exact given v)."""
    shp = SHAPE
    blocks = [S.block_weights(shp, WL.seed + 10 + b) for b in range(2)]
    z0 = S.latents(shp, WL.seed)
    cs = h3.make_shape(shp)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    z = dev_f32(z0)
    ring = torch.zeros(2, shp.n_rows, shp.hidden, dtype=torch.float32, device="cuda")
    h3.denoise_step(cs, [weights_to_device(b) for b in blocks], [0, 1], z, ring, True,
                    (1.0, 0.0, 0.0, -0.125), 0, ws)
    torch.cuda.synchronize()
    assert h3.sync_status(ws) == 0
    v_gpu = ring[0].cpu().double().numpy()
    z_gpu = z.cpu().double().numpy()
    # Euler step exact given the GPU's own velocity
    assert np.array_equal(z_gpu, oracle.euler_update(z0, v_gpu, -0.125))
    # velocity against the oracle: block 0 in full, block 1 on sampled rows
    t0 = time.time()
    wo = [weights_to_f64(b) for b in blocks]
    x1 = oracle.block_forward(oracle.bf16(z0.astype(np.float64)), wo[0], shp, p_bf16=True)["x2"]
    _log(f"denoise block0 full oracle {time.time() - t0:.1f}s")
    rows = sample_rows(shp)
    ref = oracle.block_forward_rows(x1, wo[1], shp, rows, p_bf16=True)
    _log(f"denoise block1 sampled oracle {time.time() - t0:.1f}s")
    assert_close(v_gpu[rows], ref["x2"], "velocity after 2 blocks (sampled rows)")


def test_pages_shape_block_sampled(h3):
    """The pages' own block shape at 15,435 rows: hidden 5,376, attention width 7,168
    (56 x 128), SwiGLU 14,336, checked on sampled rows."""
    wl = S.workload_by_name("block_15435_d5376_swiglu")
    block_sampled(h3, wl.shape, wl.seed, "pages-shape block", sample_rows(wl.shape))


def test_receipt_cubes_block_sampled(h3):
    """The pages' receipt sequence on the pages' block shape: 36 text + 414 audio rows
    (a prefix of 450, not a multiple of 64) and 14,985 video rows on a 37 x 15 x 27 grid
    in 280 clipped 4x4x4 cubes, top-k 56, 3-D rotary; sampled rows against the oracle
    (video rows in raster order there, cube order on the device)."""
    wl = S.workload_by_name("block_15435_cubes_d5376_swiglu")
    shp = wl.shape
    assert shp.n_video_tiles == 280
    perm = np.concatenate([np.arange(shp.n_prefix)] + oracle.shape_tiles(shp))
    P, N = shp.n_prefix, shp.n_rows
    T, Hg, Wg = shp.video_grid
    rr = lambda t, h, w: P + (t * Hg + h) * Wg + w  # noqa: E731  raster row of a token
    rows = [0, 35, 36, 448, 449, rr(0, 0, 0), rr(0, 3, 3), rr(3, 3, 4), rr(17, 7, 13),
            rr(36, 14, 26), rr(36, 0, 0), rr(35, 12, 24), N - 1]
    block_sampled(h3, shp, wl.seed, "receipt cube block", rows, perm=perm)


def test_receipt_attention_repeat_identical_and_sampled(h3):
    """Routed attention alone on the receipt sequence (56 heads, 280 cubes, k = 56: long key
    lists, 64+ steps per unit) three times: byte-identical outputs (a race between the
    softmax warps and the MMA issuer would show here), and one query tile of every head
    and sampled prefix rows against the oracle."""
    wl = S.workload_by_name("block_15435_cubes_d5376_swiglu")
    shp = wl.shape
    t0 = time.time()
    inp = S.attention_inputs(shp, wl.seed + 3, structured=0.3)
    perm = np.concatenate([np.arange(shp.n_prefix)] + oracle.shape_tiles(shp))
    _log(f"receipt attention inputs {time.time() - t0:.1f}s")
    cs = h3.attn_shape(shp)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    q, k, v = (dev_bf16(inp[n][:, perm]) for n in ("q", "k", "v"))
    g = dev_bf16(inp["gate"][perm])
    tv = shp.n_video_tiles
    idx = torch.empty(shp.heads, tv, shp.topk, dtype=torch.int32, device="cuda")
    pooled = torch.empty(shp.heads, tv, shp.head_dim, dtype=torch.float32, device="cuda")
    outs = []
    for _ in range(3):
        out = torch.empty(shp.n_rows, shp.attn_width, dtype=torch.bfloat16, device="cuda")
        h3.routed_attention(cs, q, k, v, g, out, ws, pooled=pooled, idx=idx)
        torch.cuda.synchronize()
        assert h3.sync_status(ws) == 0
        outs.append(out.view(torch.int16).clone())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    got = np.empty((shp.n_rows, shp.attn_width))
    got[perm] = outs[0].view(torch.bfloat16).float().cpu().double().numpy()
    q64, k64, v64, g64 = (S.bf16_bits_to_f64(inp[n]) for n in ("q", "k", "v", "gate"))
    sets = oracle.shape_tiles(shp)
    gi = idx.cpu().numpy()
    pb = pooled.cpu().double().numpy()
    # one query tile of every head, plus the first and the last tile
    tiles = [(h, (41 * h + 7) % tv) for h in range(shp.heads)] + [(0, 0), (55, tv - 1)]
    O = oracle.routed_attention(q64, k64, v64, shp.n_prefix, shp.n_video, gi, tiles=tiles,
                                sets=sets)
    d = shp.head_dim
    for h, i in tiles:
        rows = sets[i]
        want = O[h, rows] + g64[rows, h * d:(h + 1) * d] * pb[h, i]
        assert_close(got[rows, h * d:(h + 1) * d], want, f"receipt video tile ({h},{i})")
    for r in (0, 35, 36, shp.n_prefix - 1):
        for h in (0, 30, 55):
            want = oracle.attend(q64[h, [r]], k64[h], v64[h], 1 / np.sqrt(d))[0]
            assert_close(got[r, h * d:(h + 1) * d], want, f"receipt prefix row {r} head {h}")
    _log(f"receipt attention repeat + sampled oracle {time.time() - t0:.1f}s")


def _device_block(shp, g, zero_gates=False):
    """One block of random weights of ``shp`` made on the device (no host generation)."""
    D, A, F, d = shp.hidden, shp.attn_width, shp.mlp_width, shp.head_dim
    F1 = 2 * F if shp.mlp == "swiglu" else F

    def rn(*sz, std=0.02, mean=0.0, dtype=torch.bfloat16):
        return (torch.randn(*sz, generator=g, device="cuda") * std + mean).to(dtype)

    w = {"w_qkvg": rn(4 * A, D), "b_qkvg": rn(4 * A), "w_o": rn(D, A), "b_o": rn(D),
         "w1": rn(F1, D), "b1": rn(F1), "w2": rn(D, F), "b2": rn(D),
         "mod": rn(6, D, std=0.1, dtype=torch.float32), "qnorm_w": rn(d, mean=1.0),
         "knorm_w": rn(d, mean=1.0), "mod_prefix": rn(6, D, std=0.1, dtype=torch.float32)}
    if zero_gates:
        for t in ("mod", "mod_prefix"):
            w[t][2].zero_()
            w[t][5].zero_()
    return w


def _device_ends(shp, g, cv=96, ca=32):
    D = shp.hidden

    def rn(*sz, std=1.0, dtype=torch.float32):
        return (torch.randn(*sz, generator=g, device="cuda") * std).to(dtype)

    e = {"c_video": cv, "c_audio": ca, "text": rn(shp.n_text, D, dtype=torch.bfloat16)}
    for m, c in (("video", cv), ("audio", ca)):
        e.update({f"w_in_{m}": rn(c, D, std=0.1), f"b_in_{m}": rn(D, std=0.02),
                  f"w_out_{m}": rn(c, D, std=0.02, dtype=torch.bfloat16),
                  f"b_out_{m}": rn(c, std=0.02, dtype=torch.bfloat16),
                  f"mod_out_{m}": rn(2, D, std=0.1)})
    return e


def test_receipt_sampler_exact_properties_fullsize(h3):
    """The sampler at the receipt size (pages' shape, 280 cubes, k = 56), exact properties
    that hold at any size: (1) a core-reuse pass at the same latents gives the fresh
    pass's latents bit for bit; (2) token reduction around a block with zero gates gives
    the run without that block bit for bit (each token = bypass + a zero update)."""
    shp = S.workload_by_name("sample50_15435_cubes_d5376_swiglu_tokred").shape
    g = torch.Generator(device="cuda")
    g.manual_seed(2024)
    blocks = [_device_block(shp, g), _device_block(shp, g, zero_gates=True), _device_block(shp, g)]
    ends = _device_ends(shp, g)
    zv0 = torch.randn(shp.n_video, 96, generator=g, device="cuda")
    za0 = torch.randn(shp.n_audio, 32, generator=g, device="cuda")
    cs = h3.make_shape(shp)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    rv = torch.zeros(2, shp.n_video, 96, device="cuda")
    ra = torch.zeros(2, shp.n_audio, 32, device="cuda")
    res = torch.zeros(shp.n_rows, shp.hidden, device="cuda")
    sched = (1.0, 0.0, 0.0, -0.125)

    def run(ids, kind, reduction=None, residual=None):
        zv, za = zv0.clone(), za0.clone()
        h3.sample_step(cs, ends, blocks, ids, zv, za, rv, ra, residual, kind, sched, sched, 1,
                       ws, reduction=reduction)
        torch.cuda.synchronize()
        assert h3.sync_status(ws) == 0
        return zv, za

    fresh = run([0, 2], h3.H3DIT_PASS_FRESH, residual=res)
    core = run([], h3.H3DIT_PASS_CORE_REUSE, residual=res)
    assert torch.equal(fresh[0], core[0]) and torch.equal(fresh[1], core[1])
    assert not torch.equal(fresh[0], zv0)
    reduced = run([0, 1, 2], h3.H3DIT_PASS_FRESH, reduction=(1, 2))
    assert torch.equal(fresh[0], reduced[0]) and torch.equal(fresh[1], reduced[1])
