"""The allocation-free routed-attention entry point against the workspace one.

h3dit_routed_attention_static serves callers that cannot call cudaMalloc
(code inside a framework that owns all device memory, or under a fixed memory
budget): it runs the same router and attention kernels on a scratch array
compiled into the library.  Its results must equal those of
h3dit_routed_attention with a caller workspace, call after call, even though
every call reuses the same array.  This file is collected last so that a run
stopping at its first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import synthetic as S
from helpers import assert_close, dev_bf16, host_f64

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


CASES = [
    ("video_only_d64", S.ATTN_TINY.shape),                       # 1,024 rows, 4 x 64, k 4
    ("prefix_ragged_d128", S.BlockShape(128, 64, 300, hidden=256, heads=2, head_dim=128,
                                        mlp_width=1024, topk=2)),  # text + audio + ragged video
]


@pytest.mark.parametrize("name,shp", CASES, ids=[c[0] for c in CASES])
def test_static_scratch_matches_workspace_entry(h3, name, shp):
    cs = h3.attn_shape(shp)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    # two calls in a row with different inputs: the second must not see the first's leftovers
    for call, (seed, structured) in enumerate([(101, 0.0), (202, 0.5)]):
        inp = S.attention_inputs(shp, seed, structured=structured)
        q, k, v, g = (dev_bf16(inp[n]) for n in ("q", "k", "v", "gate"))
        out_w, pooled_w, idx_w, sc_w = _outputs(shp)
        h3.routed_attention(cs, q, k, v, g, out_w, ws, pooled=pooled_w, idx=idx_w, scores=sc_w)
        out_s, pooled_s, idx_s, sc_s = _outputs(shp)
        h3.routed_attention_static(cs, q, k, v, g, out_s, pooled=pooled_s, idx=idx_s, scores=sc_s)
        torch.cuda.synchronize()
        assert torch.equal(idx_s, idx_w), f"{name} call {call}: selected tiles differ"
        assert_close(host_f64(out_s), host_f64(out_w), f"{name} call {call} output")
        assert_close(pooled_s.double().cpu().numpy(), pooled_w.double().cpu().numpy(),
                     f"{name} call {call} pooled")
        assert np.allclose(sc_s.cpu().numpy(), sc_w.cpu().numpy(), rtol=0, atol=0)


def test_static_scratch_rejects_oversized_shape(h3):
    big = S.BLOCK_4K.shape  # 4,096 rows x 24 heads x 128 needs more than the fixed scratch
    cs = h3.attn_shape(big)
    assert h3.workspace_bytes(cs) > 4 << 20
    lib = h3.lib()
    dummy = ctypes.c_void_p(16)  # never dereferenced: the size check comes first
    rc = lib.h3dit_routed_attention_static(ctypes.byref(cs), dummy, dummy, dummy, None, dummy,
                                           None, None, None, None)
    assert rc == 4  # H3DIT_ERR_WORKSPACE
