"""GPU parity of both ends of the denoiser through h3dit_sample_step: the fp32 patch
projections, the final per-modality AdaLN and narrow output heads with the Euler
update fused into the head GEMM, whole-velocity reuse per modality and core
(residual) reuse, against the oracle."""
import numpy as np
import pytest

import oracle
import synthetic as S
from helpers import assert_close, dev_bf16, dev_f32, weights_to_device, weights_to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

FRESH, EXTRAP, CORE = 0, 1, 2


@pytest.fixture(scope="module")
def h3():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    import audio_diffusion_transformer_gb300 as pkg
    return pkg


def ends_device(e):
    out = {}
    for k, v in e.items():
        if isinstance(v, np.ndarray):
            out[k] = dev_bf16(v) if v.dtype == np.uint16 else dev_f32(v)
        else:
            out[k] = v
    return out


def ends_f64(e):
    return {k: (S.bf16_bits_to_f64(v) if isinstance(v, np.ndarray) and v.dtype == np.uint16
                else v) for k, v in e.items()}


def video_perm(shp):
    """Library video row i holds raster video row perm[i]."""
    if shp.video_grid is None:
        return np.arange(shp.n_video)
    return np.concatenate(oracle.shape_tiles(shp)) - shp.n_prefix


class Run:
    """Device state of one sampler run (latents, rings, residual, workspace)."""

    def __init__(self, h3, shp, ends, zv, za):
        self.h3, self.shp = h3, shp
        self.perm = video_perm(shp)
        self.cs = h3.make_shape(shp)
        self.ws = torch.zeros(h3.workspace_bytes(self.cs), dtype=torch.uint8, device="cuda")
        self.ends = ends_device(ends)
        self.zv = dev_f32(zv[self.perm])
        self.za = dev_f32(za)
        cv, ca = ends["c_video"], ends["c_audio"]
        self.rv = torch.zeros(2, shp.n_video, cv, dtype=torch.float32, device="cuda")
        self.ra = torch.zeros(2, shp.n_audio, ca, dtype=torch.float32, device="cuda")
        self.res = torch.zeros(shp.n_rows, shp.hidden, dtype=torch.float32, device="cuda")

    def step(self, blocks, ids, kind, video, audio, nf, reduction=None):
        self.h3.sample_step(self.cs, self.ends, blocks, ids, self.zv, self.za, self.rv, self.ra,
                            self.res, kind, video, audio, nf, self.ws, reduction=reduction)

    def z(self):
        torch.cuda.synchronize()
        assert self.h3.sync_status(self.ws) == 0
        zv = np.empty((self.shp.n_video, self.zv.shape[1]))
        zv[self.perm] = self.zv.cpu().double().numpy()
        return zv, self.za.cpu().double().numpy()


FLAT = S.BlockShape(64, 64, 256 + 40, hidden=256, heads=2, head_dim=128, mlp_width=1024, topk=2)
CUBES = S.BlockShape(36, 92, 5 * 6 * 7, hidden=256, heads=2, head_dim=128, mlp_width=512,
                     topk=3, mlp="swiglu", prefix_mod=True, video_grid=(5, 6, 7))


@pytest.mark.parametrize("cv,ca", [(96, 32), (128, 64)])
def test_heads_and_patches_bit_exact_small_integers(h3, cv, ca):
    """No blocks and scale = -1 in the final AdaLN: every row's head input is
    bf16(shift), so v = W_out shift + b; with small-integer weights and a power-of-two
    step the fp32 results are exact, pinning the narrow head GEMM (N = 96 / 32 / 128 /
    64 tiles), its fused Euler update and the ring store."""
    shp = FLAT
    rng = np.random.default_rng(cv + ca)
    e = S.ends_weights(shp, 3, cv, ca)
    for m, c in (("video", cv), ("audio", ca)):
        mod = np.zeros((2, shp.hidden), np.float32)
        mod[0] = rng.integers(-3, 4, shp.hidden)
        mod[1] = -1.0
        e[f"mod_out_{m}"] = mod
        e[f"w_out_{m}"] = S.to_bf16_bits(rng.integers(-3, 4, (c, shp.hidden)).astype(np.float32))
        e[f"b_out_{m}"] = S.to_bf16_bits(rng.integers(-3, 4, c).astype(np.float32))
    zv, za = S.modality_latents(shp, 4, cv, ca)
    r = Run(h3, shp, e, zv, za)
    r.step([], [], FRESH, (1.0, 0, 0, -0.125), (1.0, 0, 0, -0.25), 0)
    gv, ga = r.z()
    ref = oracle.sample_step(zv, za, ends_f64(e), [], shp, "fresh", -0.125, -0.25)
    assert np.array_equal(gv, ref["z_video"]) and np.array_equal(ga, ref["z_audio"])
    assert np.array_equal(r.rv[0].cpu().double().numpy(), ref["v_video"])
    assert np.array_equal(r.ra[0].cpu().double().numpy(), ref["v_audio"])


@pytest.mark.parametrize("shp", [FLAT, CUBES], ids=["flat", "cubes"])
def test_sample_fresh_step_matches_oracle(h3, shp):
    e = S.ends_weights(shp, 7)
    blocks = [S.block_weights(shp, 600 + b) for b in range(2)]
    zv, za = S.modality_latents(shp, 8)
    r = Run(h3, shp, e, zv, za)
    r.step([weights_to_device(b) for b in blocks], [0, 1], FRESH, (1.0, 0, 0, -0.125),
           (0.8, 0, 0, -0.2), 0)
    gv, ga = r.z()
    ref = oracle.sample_step(zv, za, ends_f64(e), [weights_to_f64(b) for b in blocks], shp,
                             "fresh", -0.125, -0.2)
    vv = np.empty_like(ref["v_video"])
    vv[r.perm] = r.rv[0].cpu().double().numpy()
    assert_close(vv, ref["v_video"], "video velocity")
    assert_close(r.ra[0].cpu().double().numpy(), ref["v_audio"], "audio velocity")
    assert_close(gv - zv, ref["z_video"] - zv, "video step", rel=2e-2, cos=0.998)
    assert_close(ga - za, ref["z_audio"] - za, "audio step", rel=2e-2, cos=0.998)
    # the held residual is x_L - x_0 of the fresh pass
    res = r.res.cpu().double().numpy()
    full_perm = np.concatenate([np.arange(shp.n_prefix), shp.n_prefix + r.perm])
    want = np.empty_like(res)
    want[:] = ref["residual"][full_perm]
    assert_close(res, want, "core residual", rel=3e-2, cos=0.999)


def test_core_reuse_at_the_same_latents_is_bit_identical_to_fresh(h3):
    shp = CUBES
    e = S.ends_weights(shp, 9)
    blocks = [weights_to_device(S.block_weights(shp, 700 + b)) for b in range(2)]
    zv, za = S.modality_latents(shp, 10)
    a = Run(h3, shp, e, zv, za)
    a.step(blocks, [0, 1], FRESH, (1.0, 0, 0, -0.125), (1.0, 0, 0, -0.25), 0)
    b = Run(h3, shp, e, zv, za)
    b.res.copy_(a.res)
    b.step([], [], CORE, (1.0, 0, 0, -0.125), (1.0, 0, 0, -0.25), 1)
    av, aa = a.z()
    bv, ba = b.z()
    assert np.array_equal(av, bv) and np.array_equal(aa, ba)
    assert not np.array_equal(av, zv.astype(np.float64))


@pytest.mark.parametrize("mode", ["velocity_reuse", "core_reuse"])
def test_sample_loop_matches_oracle(h3, mode):
    """Five steps, passes 0, 2 and 4 run the blocks; in between either whole-velocity
    reuse (each modality extrapolated on its own schedule: video uniform, audio shifted
    by 3) or core reuse (held residual, fresh patch projections and heads)."""
    shp = CUBES
    e = S.ends_weights(shp, 11)
    bw = [S.block_weights(shp, 800 + b) for b in range(2)]
    blocks = [weights_to_device(b) for b in bw]
    zv, za = S.modality_latents(shp, 12)
    n, r_ = 5, 2
    sv, sa = oracle.sigma_schedule(n), oracle.sigma_schedule(n, 3.0)
    fresh = oracle.fresh_steps(n, r_)
    run = Run(h3, shp, e, zv, za)
    hist = []
    for i in range(n):
        dv, da = sv[i + 1] - sv[i], sa[i + 1] - sa[i]
        if i in fresh:
            run.step(blocks, [0, 1], FRESH, (sv[i], 0, 0, dv), (sa[i], 0, 0, da), len(hist))
            hist.append(i)
        elif mode == "core_reuse":
            run.step([], [], CORE, (sv[i], 0, 0, dv), (sa[i], 0, 0, da), len(hist))
        else:
            ia, ib = hist[-1], hist[-2] if len(hist) > 1 else hist[-1]
            run.step([], [], EXTRAP, (sv[i], sv[ia], sv[ib], dv), (sa[i], sa[ia], sa[ib], da),
                     len(hist))
    gv, ga = run.z()
    kw = {"reuse": r_} if mode == "velocity_reuse" else {"core_reuse": r_}
    ref = oracle.sample_loop(zv, za, ends_f64(e), [weights_to_f64(b) for b in bw], shp, n,
                             block_ids=[0, 1], sig_video=sv, sig_audio=sa, **kw)
    assert_close(gv - zv, ref["z_video"] - zv, f"{mode}: video change", rel=2e-2, cos=0.998)
    assert_close(ga - za, ref["z_audio"] - za, f"{mode}: audio change", rel=2e-2, cos=0.998)


# ----------------------------------------------------------------------------- token reduction
TR = CUBES.with_(token_reduction=True)  # 5 x 6 x 7 grid: the odd width leaves lone tokens


def test_token_reduction_around_an_identity_block_is_exact(h3):
    """Pool before block 1, restore before block 2, block 1 with zero gates: each token
    comes back as its bypass value plus a zero update, so the run equals blocks 0 and 2
    without reduction, bit for bit."""
    e = S.ends_weights(TR, 13)
    bw = [S.block_weights(TR, 900 + b) for b in range(3)]
    bw[1]["mod"][2] = 0.0
    bw[1]["mod"][5] = 0.0
    bw[1]["mod_prefix"][2] = 0.0
    bw[1]["mod_prefix"][5] = 0.0
    blocks = [weights_to_device(b) for b in bw]
    zv, za = S.modality_latents(TR, 14)
    a = Run(h3, TR, e, zv, za)
    a.step(blocks, [0, 1, 2], FRESH, (1.0, 0, 0, -0.125), (1.0, 0, 0, -0.25), 0, reduction=(1, 2))
    b = Run(h3, TR, e, zv, za)
    b.step(blocks, [0, 2], FRESH, (1.0, 0, 0, -0.125), (1.0, 0, 0, -0.25), 0)
    av, aa = a.z()
    bv, ba = b.z()
    assert np.array_equal(av, bv) and np.array_equal(aa, ba)


@pytest.mark.parametrize("reduction", [(1, 2), (1, 3), (0, 2)])
def test_token_reduction_matches_oracle(h3, reduction):
    e = S.ends_weights(TR, 15)
    bw = [S.block_weights(TR, 950 + b) for b in range(3)]
    zv, za = S.modality_latents(TR, 16)
    r = Run(h3, TR, e, zv, za)
    r.step([weights_to_device(b) for b in bw], [0, 1, 2], FRESH, (1.0, 0, 0, -0.125),
           (1.0, 0, 0, -0.25), 0, reduction=reduction)
    gv, ga = r.z()
    ref = oracle.sample_step(zv, za, ends_f64(e), [weights_to_f64(b) for b in bw], TR, "fresh",
                             -0.125, -0.25, reduction=reduction)
    plain = oracle.sample_step(zv, za, ends_f64(e), [weights_to_f64(b) for b in bw], TR,
                               "fresh", -0.125, -0.25)
    vv = np.empty_like(ref["v_video"])
    vv[r.perm] = r.rv[0].cpu().double().numpy()
    assert_close(vv, ref["v_video"], f"video velocity {reduction}")
    assert_close(r.ra[0].cpu().double().numpy(), ref["v_audio"], f"audio velocity {reduction}")
    from helpers import rel_l2
    # the reduction changes the result (it is an approximation); the GPU follows the oracle's
    assert rel_l2(vv, ref["v_video"]) < 0.25 * rel_l2(plain["v_video"], ref["v_video"])


def test_sample_step_video_only_without_text_or_audio(h3):
    """No text and no audio rows (prefix of 0): the audio latents, heads and schedule are
    absent (null pointers) and the video path alone runs, against the oracle."""
    shp = S.BlockShape(0, 0, 6 * 5 * 7, hidden=256, heads=2, head_dim=128, mlp_width=1024,
                       topk=3, video_grid=(6, 5, 7))
    e = S.ends_weights(shp, 21, 96, 32)
    for n in ("w_in_audio", "b_in_audio", "w_out_audio", "b_out_audio", "mod_out_audio", "text"):
        e.pop(n)
    e["c_audio"] = 0
    bw = [S.block_weights(shp, 1000 + b) for b in range(2)]
    zv, _ = S.modality_latents(shp, 22, 96, 32)
    za = np.zeros((0, 32), np.float32)
    r = Run(h3, shp, dict(e, c_audio=32), zv, za)
    r.ends = ends_device(e)
    r.step([weights_to_device(b) for b in bw], [0, 1], FRESH, (1.0, 0, 0, -0.125),
           (1.0, 0, 0, -0.125), 0)
    gv, _ = r.z()
    ref = oracle.sample_step(zv, za, ends_f64(dict(e, text=np.zeros((0, shp.hidden)))),
                             [weights_to_f64(b) for b in bw], shp, "fresh", -0.125, -0.125)
    vv = np.empty_like(ref["v_video"])
    vv[r.perm] = r.rv[0].cpu().double().numpy()
    assert_close(vv, ref["v_video"], "video velocity (no prefix)")
