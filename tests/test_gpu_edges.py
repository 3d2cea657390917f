"""Edge cases of the CUDA path through the C ABI: degenerate tile counts, a
single partial tile, the maximum row count the attention accepts, all-equal
scores (every selection decided by the tie rule), k = 1, and the device-side
failure path (a bounded wait that runs out and reports a status)."""
import numpy as np
import pytest

import oracle
import synthetic as S
from helpers import assert_close, compare_topk, dev_bf16, host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def h3():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    import audio_diffusion_transformer_gb300 as pkg
    return pkg


def run(h3, shp, inp, with_gate=True):
    cs = h3.attn_shape(shp)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    tv, ks = shp.n_video_tiles, min(shp.topk, shp.n_video_tiles)
    out = torch.empty(shp.n_rows, shp.attn_width, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(shp.heads, tv, ks, dtype=torch.int32, device="cuda")
    sc = torch.empty(shp.heads, tv, tv, dtype=torch.float32, device="cuda")
    g = dev_bf16(inp["gate"]) if with_gate else None
    h3.routed_attention(cs, *(dev_bf16(inp[n]) for n in ("q", "k", "v")), g, out, ws, idx=idx,
                        scores=sc)
    torch.cuda.synchronize()
    assert h3.sync_status(ws) == 0
    return host_f64(out), idx.cpu().numpy(), sc.cpu().double().numpy()


def oracle_layer(shp, inp, with_gate=True):
    q, k, v = (S.bf16_bits_to_f64(inp[n]) for n in ("q", "k", "v"))
    g = S.bf16_bits_to_f64(inp["gate"]) if with_gate else None
    return oracle.attention_layer(q, k, v, g, shp.n_prefix, shp.n_video, shp.topk)


@pytest.mark.parametrize("shp", [
    S.BlockShape(0, 0, 10, hidden=256, heads=2, head_dim=64, mlp_width=1024, topk=1),
    S.BlockShape(64, 0, 37, hidden=256, heads=2, head_dim=128, mlp_width=1024, topk=3),
    S.BlockShape(128, 128, 64, hidden=256, heads=1, head_dim=128, mlp_width=1024, topk=1),
], ids=["one_partial_tile", "prefix_plus_partial_tile", "one_full_tile"])
def test_single_video_tile(h3, shp):
    inp = S.attention_inputs(shp, 41)
    got, idx, _ = run(h3, shp, inp)
    ref = oracle_layer(shp, inp)
    assert np.array_equal(idx, ref["idx"])
    assert_close(got, ref["o_f64"], "single tile", rel=5e-3, cos=0.99995)


def test_k1_many_tiles(h3):
    shp = S.BlockShape(64, 64, 64 * 40 + 5, hidden=256, heads=2, head_dim=128, mlp_width=1024,
                       topk=1)
    inp = S.attention_inputs(shp, 43, structured=0.3)
    got, idx, sc = run(h3, shp, inp)
    ref = oracle_layer(shp, inp)
    compare_topk(idx, ref["idx"], ref["scores"], 1)
    assert_close(got, ref["o_f64"], "k = 1")


def test_all_scores_equal_tie_rule(h3):
    # every row of q and k equal: all tile means equal, every score ties, so each query
    # tile must keep tiles 0..k-1 (ties go to the lower tile)
    shp = S.BlockShape(0, 0, 64 * 9 + 20, hidden=256, heads=2, head_dim=64, mlp_width=1024,
                       topk=4)
    inp = S.attention_inputs(shp, 47, with_gate=False)
    for n in ("q", "k"):
        row = inp[n][:, :1, :]
        inp[n] = np.ascontiguousarray(np.broadcast_to(row, inp[n].shape))
    got, idx, sc = run(h3, shp, inp, with_gate=False)
    assert np.all(idx == np.arange(4)[None, None, :])
    ref = oracle_layer(shp, inp, with_gate=False)
    assert np.array_equal(idx, ref["idx"])
    assert_close(got, ref["o_f64"], "equal scores", rel=5e-3, cos=0.99995)


def test_maximum_rows(h3):
    # the largest accepted sequence: 65,408 rows (1,022 tiles)
    shp = S.BlockShape(0, 0, 1022 * 64, hidden=256, heads=1, head_dim=64, mlp_width=1024,
                       topk=8)
    inp = S.attention_inputs(shp, 53, structured=0.3, with_gate=False)
    got, idx, sc = run(h3, shp, inp, with_gate=False)
    q, k, v = (S.bf16_bits_to_f64(inp[n]) for n in ("q", "k", "v"))
    mq, mk = oracle.tile_means(q, 0, shp.n_video), oracle.tile_means(k, 0, shp.n_video)
    Sref = oracle.tile_scores(mq, mk)
    compare_topk(idx, oracle.topk_select(Sref, 8), Sref, 8)
    tiles = [(0, 0), (0, 511), (0, 1021)]
    O = oracle.routed_attention(q, k, v, 0, shp.n_video, idx, tiles=tiles)
    for _, i in tiles:
        r = slice(64 * i, 64 * i + 64)
        assert_close(got[r], O[0, r], f"tile {i}", rel=5e-3, cos=0.99995)


def test_shape_beyond_maximum_is_refused(h3):
    shp = S.BlockShape(0, 0, 1023 * 64, hidden=256, heads=1, head_dim=64, mlp_width=1024, topk=8)
    with pytest.raises(h3.H3DitError):
        h3.workspace_bytes(h3.attn_shape(shp))


def test_bounded_wait_reports_timeout_and_context_survives(h3):
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    h3.selftest_timeout(ws, limit_ms=200)
    assert h3.sync_status(ws) == 6  # H3DIT_ERR_TIMEOUT
    assert h3.sync_status(ws) == 0  # read-and-clear
    # the context is still usable: a GEMM runs and is exact on small integers
    a = torch.randint(-4, 5, (256, 128), device="cuda").to(torch.bfloat16)
    w = torch.randint(-4, 5, (256, 128), device="cuda").to(torch.bfloat16)
    y = torch.empty(256, 256, dtype=torch.bfloat16, device="cuda")
    h3.linear(a, w, None, y)
    torch.cuda.synchronize()
    ref = a.double().cpu().numpy() @ w.double().cpu().numpy().T
    assert np.array_equal(y.double().cpu().numpy(), oracle.bf16(ref))
