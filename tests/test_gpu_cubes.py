"""GPU parity for 4 x 4 x 4 cube tiling with the 3-D rotary and a prefix that is not
a multiple of 64 rows.

The oracle works on video rows in raster (t, h, w) order with each tile a set of
rows (a clipped cube); the library keeps the video rows in cube order.  The tests
move rows between the two orders with the permutation built from the oracle's
own tiles (prefix rows first, then the tiles' rows one tile after the other), so
the library's layout is checked against the oracle's definition, not against
itself.
"""
import numpy as np
import pytest

import oracle
import synthetic as S
from helpers import (assert_close, check_close, compare_topk, dev_bf16, dev_f32, host_f64, log,
                     router_on_gpu_inputs, weights_to_device, weights_to_f64, workspace_views)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def h3():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    import audio_diffusion_transformer_gb300 as pkg
    return pkg


def cube_perm(shp):
    """lib_row -> raster row: prefix rows, then every oracle tile's rows in tile order."""
    return np.concatenate([np.arange(shp.n_prefix)] + oracle.shape_tiles(shp))


ATTN_CUBE_CASES = [
    # (name, shape, structured)
    ("cubes_5x6x7_d128_k3", S.BlockShape(36, 64, 5 * 6 * 7, hidden=256, heads=2, head_dim=128,
                                         mlp_width=1024, topk=3, qk_norm=False, rope=False,
                                         video_grid=(5, 6, 7)), 0.4),
    ("cubes_9x10x11_d64_k5_prefix450", S.BlockShape(36, 414, 9 * 10 * 11, hidden=256, heads=3,
                                                    head_dim=64, mlp_width=1024, topk=5,
                                                    qk_norm=False, rope=False,
                                                    video_grid=(9, 10, 11)), 0.4),
    ("cubes_dense_all_tiles", S.BlockShape(0, 64, 6 * 5 * 9, hidden=256, heads=2, head_dim=128,
                                           mlp_width=1024, topk=64, qk_norm=False, rope=False,
                                           video_grid=(6, 5, 9)), 0.0),
    ("cubes_flat_tiles_2x8x4", S.BlockShape(20, 0, 7 * 16 * 9, hidden=256, heads=2,
                                            head_dim=128, mlp_width=1024, topk=4, qk_norm=False,
                                            rope=False, video_grid=(7, 16, 9), cube=(2, 8, 4)),
     0.4),
]


@pytest.mark.parametrize("name,shp,structured", ATTN_CUBE_CASES,
                         ids=[c[0] for c in ATTN_CUBE_CASES])
def test_routed_attention_cubes(h3, name, shp, structured):
    inp = S.attention_inputs(shp, 0x48334460, structured=structured)
    perm = cube_perm(shp)
    # library order on the device
    q, k, v = (dev_bf16(inp[n][:, perm]) for n in ("q", "k", "v"))
    g = dev_bf16(inp["gate"][perm])
    cs = h3.attn_shape(shp)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    tv, ks = shp.n_video_tiles, min(shp.topk, shp.n_video_tiles)
    out = torch.empty(shp.n_rows, shp.attn_width, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(shp.heads, tv, ks, dtype=torch.int32, device="cuda")
    sc = torch.empty(shp.heads, tv, tv, dtype=torch.float32, device="cuda")
    pooled = torch.empty(shp.heads, tv, shp.head_dim, dtype=torch.float32, device="cuda")
    h3.routed_attention(cs, q, k, v, g, out, ws, pooled=pooled, idx=idx, scores=sc)
    torch.cuda.synchronize()
    assert h3.sync_status(ws) == 0
    # oracle in raster order
    q64, k64, v64, g64 = (S.bf16_bits_to_f64(inp[n]) for n in ("q", "k", "v", "gate"))
    sets = oracle.shape_tiles(shp)
    ref = oracle.attention_layer(q64, k64, v64, g64, shp.n_prefix, shp.n_video, shp.topk,
                                 shp.tile, True, False, sets)
    assert np.allclose(sc.cpu().double().numpy(), ref["scores"], rtol=1e-4, atol=1e-6)
    gi = idx.cpu().numpy()
    compare_topk(gi, ref["idx"], ref["scores"], shp.topk)
    assert np.allclose(pooled.cpu().double().numpy(), ref["pooled"], rtol=1e-4, atol=1e-6)
    # outputs: recompute with the GPU's selections (identical except counted near-ties)
    O = oracle.routed_attention(q64, k64, v64, shp.n_prefix, shp.n_video, gi, sets=sets)
    want = oracle.gate_mix(O, g64, ref["pooled"], shp.n_prefix, shp.n_video, sets=sets)
    got = np.empty_like(want)
    got[perm] = host_f64(out)
    assert_close(got, want, name, rel=1e-2, cos=0.9999)
    if shp.topk >= tv:  # every tile selected: dense attention over all rows for every row
        H, d = shp.heads, shp.head_dim
        dense = np.stack([oracle.attend(q64[h], k64[h], v64[h], 1 / np.sqrt(d))
                          for h in range(H)])
        assert_close(got, oracle.gate_mix(dense, g64, ref["pooled"], shp.n_prefix, shp.n_video,
                                          sets=sets), name + " dense", rel=1e-2, cos=0.9999)


BLOCK_CUBE_CASES = [
    ("block_cubes_rope3d_gelu", S.BlockShape(36, 92, 5 * 6 * 7, hidden=256, heads=2, head_dim=128,
                                             mlp_width=1024, topk=3, video_grid=(5, 6, 7))),
    ("block_cubes_rope3d_swiglu_prefix_table",
     S.BlockShape(36, 414, 6 * 7 * 9, hidden=256, heads=4, head_dim=64, mlp_width=384, topk=4,
                  mlp="swiglu", prefix_mod=True, video_grid=(6, 7, 9))),
]


def run_block_cubes(h3, shp, seed, keep=False):
    w = S.block_weights(shp, seed)
    xb = S.hidden_rows(shp, seed)  # raster order
    perm = cube_perm(shp)
    cs = h3.make_shape(shp)
    if keep:
        cs = h3.make_shape(shp, cs.flags | h3.H3DIT_KEEP_INTERMEDIATES)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    x = dev_bf16(xb[perm])
    h3.block_forward(cs, weights_to_device(w), x, ws)
    torch.cuda.synchronize()
    assert h3.sync_status(ws) == 0
    got = np.empty((shp.n_rows, shp.hidden))
    got[perm] = host_f64(x)
    if not keep:
        return got, w, xb
    lib = workspace_views(h3, cs, shp, ws, ["q", "k", "x1", "idx"])
    it = {"idx": lib["idx"]}  # cube tiles are numbered alike on both sides
    for n in ("q", "k"):
        it[n] = np.empty_like(lib[n])
        it[n][:, perm] = lib[n]
    it["x1"] = np.empty_like(lib["x1"])
    it["x1"][perm] = lib["x1"]
    return got, w, xb, it


@pytest.mark.parametrize("name,shp", BLOCK_CUBE_CASES, ids=[c[0] for c in BLOCK_CUBE_CASES])
def test_block_forward_cubes(h3, name, shp):
    """The block's updates x1 - x and x2 - x against the oracle that rounds the softmax
    weights to bf16, rows moved between the two orders; the router checked against the
    oracle's on the GPU's own q and k, and the oracle attending over the GPU's selections."""
    got, w, xb, it = run_block_cubes(h3, shp, 81, keep=True)
    x0 = S.bf16_bits_to_f64(xb)
    n_tie = router_on_gpu_inputs(it["q"], it["k"], shp, it["idx"])
    ref = oracle.block_forward(x0, weights_to_f64(w), shp, p_bf16=True, idx=it["idx"])
    log(f"{name}: near-ties differing on the GPU's q/k: {n_tie}; selections differing from "
        f"the oracle's own: {int(np.any(it['idx'] != ref['idx'], axis=-1).sum())}")
    check_close(got, ref["x2"], name + " x2", rel=2e-3, cos=0.99999)
    check_close(it["x1"] - x0, ref["x1"] - x0, name + " x1 - x", rel=2e-2, cos=0.998)
    check_close(got - x0, ref["x2"] - x0, name + " x2 - x", rel=2e-2, cos=0.998)
    assert np.array_equal(run_block_cubes(h3, shp, 81)[0], got)  # keeping changes nothing


def test_block_cubes_rotary_is_3d(h3):
    """The same rows and weights with the grid described as 1-D slices give a different
    result: the 3-D rotary and the cube tiles are in effect (guards against a silent
    fallback to the 1-D layout)."""
    shp = BLOCK_CUBE_CASES[0][1]
    got, w, xb = run_block_cubes(h3, shp, 82)
    flat = shp.with_(video_grid=None)
    ref_flat = oracle.block_forward(S.bf16_bits_to_f64(xb), weights_to_f64(w), flat)["x2"]
    ref_cube = oracle.block_forward(S.bf16_bits_to_f64(xb), weights_to_f64(w), shp)["x2"]
    x0 = S.bf16_bits_to_f64(xb)
    from helpers import rel_l2
    assert rel_l2(got - x0, ref_cube - x0) < 0.5 * rel_l2(got - x0, ref_flat - x0)


def test_denoise_step_cubes(h3):
    """denoise_step builds its own rotary table once per step: one fresh step over two
    cube-layout blocks against the oracle (rows moved between the two orders)."""
    shp = BLOCK_CUBE_CASES[1][1]
    blocks = [S.block_weights(shp, 500 + b) for b in range(2)]
    perm = cube_perm(shp)
    z0 = S.latents(shp, 23)
    z = dev_f32(z0[perm])
    ring = torch.zeros(2, shp.n_rows, shp.hidden, dtype=torch.float32, device="cuda")
    cs = h3.make_shape(shp)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    h3.denoise_step(cs, [weights_to_device(b) for b in blocks], [0, 1], z, ring, True,
                    (1.0, 0, 0, -0.125), 0, ws, prefix=(0.5, 0, 0, -0.25))
    torch.cuda.synchronize()
    assert h3.sync_status(ws) == 0
    ref = oracle.denoise_forward(z0, [weights_to_f64(b) for b in blocks], shp, -0.125, [0, 1],
                                 dt_prefix=-0.25)
    got = np.empty_like(ref["z"])
    got[perm] = z.cpu().double().numpy()
    v = np.empty_like(ref["v"])
    v[perm] = ring[0].cpu().double().numpy()
    assert_close(v, ref["v"], "velocity", rel=2e-2, cos=0.998)
    assert np.array_equal(got, oracle.euler_update(z0, v, -0.125, -0.25, shp.n_prefix))
