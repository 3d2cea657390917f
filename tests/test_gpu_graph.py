"""The library's calls can be captured into a CUDA graph and replayed: every call only
enqueues work on the given stream (kernel launches, device-to-device copies), so a
captured denoiser step or sampler step replays to the same bytes as eager calls."""
import numpy as np
import pytest

import synthetic as S
from helpers import dev_f32, weights_to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def h3():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    import audio_diffusion_transformer_gb300 as pkg
    return pkg


SHAPE = S.BlockShape(36, 92, 5 * 6 * 7, hidden=256, heads=2, head_dim=128, mlp_width=512,
                     topk=3, mlp="swiglu", prefix_mod=True, video_grid=(5, 6, 7),
                     token_reduction=True)


def test_denoise_loop_graph_replay_matches_eager(h3):
    shp = SHAPE
    blocks = [weights_to_device(S.block_weights(shp, 1100 + b)) for b in range(3)]
    z0 = dev_f32(S.latents(shp, 31))
    cs = h3.make_shape(shp)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    ring = torch.zeros(2, shp.n_rows, shp.hidden, device="cuda")
    z = torch.empty_like(z0)

    def loop(stream):
        z.copy_(z0)
        h3.denoise_step(cs, blocks, [0, 1, 2], z, ring, True, (1.0, 0, 0, -0.25), 0, ws,
                        stream=stream)
        h3.denoise_step(cs, blocks, [0, 1, 2], z, ring, True, (0.75, 0, 0, -0.25), 1, ws,
                        stream=stream)
        h3.denoise_step(cs, blocks, [0, 2], z, ring, False, (0.5, 0.75, 1.0, -0.25), 2, ws,
                        stream=stream)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        loop(side.cuda_stream)  # eager, and the warm-up torch asks for before capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = z.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        loop(torch.cuda.current_stream().cuda_stream)
    z.zero_()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert h3.sync_status(ws) == 0
    assert torch.equal(z, eager)


def test_sampler_step_with_token_reduction_graph_replay_matches_eager(h3):
    shp = SHAPE
    e = S.ends_weights(shp, 33)
    ends = {k: (torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16)
                .cuda() if isinstance(v, np.ndarray) and v.dtype == np.uint16 else
                (dev_f32(v) if isinstance(v, np.ndarray) else v)) for k, v in e.items()}
    blocks = [weights_to_device(S.block_weights(shp, 1200 + b)) for b in range(3)]
    zv0, za0 = (dev_f32(a) for a in S.modality_latents(shp, 34))
    cs = h3.make_shape(shp)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device="cuda")
    rv = torch.zeros(2, shp.n_video, 96, device="cuda")
    ra = torch.zeros(2, shp.n_audio, 32, device="cuda")
    res = torch.zeros(shp.n_rows, shp.hidden, device="cuda")
    zv, za = torch.empty_like(zv0), torch.empty_like(za0)

    def step(stream):
        zv.copy_(zv0)
        za.copy_(za0)
        h3.sample_step(cs, ends, blocks, [0, 1, 2], zv, za, rv, ra, res, h3.H3DIT_PASS_FRESH,
                       (1.0, 0, 0, -0.125), (1.0, 0, 0, -0.25), 0, ws, stream=stream,
                       reduction=(1, 3))
        h3.sample_step(cs, ends, [], [], zv, za, rv, ra, res, h3.H3DIT_PASS_CORE_REUSE,
                       (0.875, 0, 0, -0.125), (0.75, 0, 0, -0.25), 1, ws, stream=stream)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(side.cuda_stream)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = (zv.clone(), za.clone())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream().cuda_stream)
    zv.zero_()
    za.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert h3.sync_status(ws) == 0
    assert torch.equal(zv, eager[0]) and torch.equal(za, eager[1])
