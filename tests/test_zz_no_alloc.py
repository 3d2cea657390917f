"""The allocation-free routed-attention entry point against the workspace one.

h3dit_routed_attention_static serves callers that cannot call cudaMalloc
(code inside a framework that owns all device memory, or under a fixed memory
budget): it runs the same router and attention kernels on a scratch array
compiled into the library.  Both paths run the same deterministic kernels on
the same inputs, so their outputs must be byte-identical, call after call, even
though every static call reuses the array that the previous call left behind
(a larger shape first, then smaller ones whose regions sit inside its stale
tails).  This file is collected last so that a run stopping at its first
failure has already run every other test.
"""
import ctypes

import pytest

import synthetic as S
from helpers import dev_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def h3():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    import audio_diffusion_transformer_gb300 as pkg
    return pkg


def _outputs(shp):
    tv, ks = shp.n_video_tiles, min(shp.topk, shp.n_video_tiles)
    return (torch.empty(shp.n_rows, shp.attn_width, dtype=torch.bfloat16, device="cuda"),
            torch.empty(shp.heads, tv, shp.head_dim, dtype=torch.float32, device="cuda"),
            torch.empty(shp.heads, tv, ks, dtype=torch.int32, device="cuda"),
            torch.empty(shp.heads, tv, tv, dtype=torch.float32, device="cuda"))


# larger router scratch first, so the later calls meet its leftovers
SEQUENCE = [
    ("block4k_d128", S.BLOCK_4K.shape, 0.5),                     # 4,096 rows, 24 x 128, 56 tiles
    ("video_only_d64", S.ATTN_TINY.shape, 0.0),                 # 1,024 rows, 4 x 64, k 4
    ("prefix_ragged_d128", S.BlockShape(128, 64, 300, hidden=256, heads=2, head_dim=128,
                                        mlp_width=1024, topk=2), 0.3),
    ("video_only_d64_again", S.ATTN_TINY.shape, 0.5),
]


def test_static_scratch_matches_workspace_entry(h3):
    for call, (name, shp, structured) in enumerate(SEQUENCE):
        cs = h3.attn_shape(shp)
        inp = S.attention_inputs(shp, 101 + call, structured=structured)
        q, k, v, g = (dev_bf16(inp[n]) for n in ("q", "k", "v", "gate"))
        ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
        out_w, pooled_w, idx_w, sc_w = _outputs(shp)
        h3.routed_attention(cs, q, k, v, g, out_w, ws, pooled=pooled_w, idx=idx_w, scores=sc_w)
        out_s, pooled_s, idx_s, sc_s = _outputs(shp)
        h3.routed_attention_static(cs, q, k, v, g, out_s, pooled=pooled_s, idx=idx_s, scores=sc_s)
        assert h3.routed_attention_static_status() == 0, f"{name}: static status"
        torch.cuda.synchronize()
        assert h3.sync_status(ws) == 0
        assert torch.equal(idx_s, idx_w), f"call {call} ({name}): selected tiles differ"
        assert torch.equal(out_s.view(torch.int16), out_w.view(torch.int16)), \
            f"call {call} ({name}): outputs differ"
        assert torch.equal(pooled_s, pooled_w), f"call {call} ({name}): pooled branch differs"
        assert torch.equal(sc_s, sc_w), f"call {call} ({name}): tile scores differ"


def test_static_scratch_rejects_oversized_shape(h3):
    big = S.BLOCK_15K.shape  # 15,435 rows x 40 heads x 128, 218 tiles: 26 MB of router scratch
    cs = h3.attn_shape(big)
    assert h3.workspace_bytes(cs) > 4 << 20
    lib = h3.lib()
    dummy = ctypes.c_void_p(16)  # never dereferenced: the size check comes first
    rc = lib.h3dit_routed_attention_static(ctypes.byref(cs), dummy, dummy, dummy, None, dummy,
                                           None, None, None, None)
    assert rc == 4  # H3DIT_ERR_WORKSPACE
