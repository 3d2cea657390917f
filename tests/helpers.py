"""Shared test helpers: device upload of seeded inputs and the comparison metrics."""
from __future__ import annotations

import os

import numpy as np

import synthetic as S

REL_L2_TOL = 2e-2    # relative L2 error bound against the oracle
COS_TOL = 0.998      # cosine similarity bound against the oracle
NEAR_TIE = 1e-5      # relative top-k score gap below which two selections may differ


def dev_bf16(bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def dev_f32(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def host_f64(t):
    return t.float().cpu().double().numpy()


def weights_to_device(w: dict, device="cuda") -> dict:
    return {n: (dev_bf16(a, device) if a.dtype == np.uint16 else dev_f32(a, device))
            for n, a in w.items()}


def weights_to_f64(w: dict) -> dict:
    return {n: (S.bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64))
            for n, a in w.items()}


def rel_l2(got, ref) -> float:
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def cosine(got, ref) -> float:
    a, b = got.ravel(), ref.ravel()
    return float(a @ b / max(np.linalg.norm(a) * np.linalg.norm(b), 1e-300))


def assert_close(got, ref, what="", rel=REL_L2_TOL, cos=COS_TOL):
    r, c = rel_l2(got, ref), cosine(got, ref)
    assert r <= rel and c >= cos, f"{what}: rel L2 {r:.3e} (<= {rel}), cos {c:.6f} (>= {cos})"
    return r, c


def compare_topk(gpu_idx, ref_idx, ref_scores, k):
    """Index sets must match exactly except at near-ties, where the GPU's set must
    still be a valid top-k of the oracle's float64 scores.  Returns the number of
    near-tie rows whose selections differ."""
    import oracle
    gap = oracle.topk_gap(ref_scores, k)
    diff = np.any(gpu_idx != ref_idx, axis=-1)
    bad = []
    for h, i in zip(*np.nonzero(diff)):
        ok = gap[h, i] < NEAR_TIE and oracle.topk_set_valid(ref_scores[h, i], gpu_idx[h, i],
                                                            NEAR_TIE)
        if not ok:
            bad.append((int(h), int(i), gpu_idx[h, i].tolist(), ref_idx[h, i].tolist(),
                        float(gap[h, i])))
    assert not bad, f"top-k mismatches beyond near-ties: {bad[:5]} (total {len(bad)})"
    return int(diff.sum())


def log(msg: str):
    """Measured figures of a test (oracle timings, errors against the oracle): printed
    (pytest -s shows them) and appended to the file named by H3DIT_TEST_LOG when set."""
    print(msg)
    path = os.environ.get("H3DIT_TEST_LOG")
    if path:
        with open(path, "a") as f:
            f.write(msg + "\n")


def check_close(got, ref, what="", rel=REL_L2_TOL, cos=COS_TOL):
    """assert_close that also logs the measured relative L2 error and cosine."""
    r, c = rel_l2(got, ref), cosine(got, ref)
    log(f"{what}: rel L2 {r:.3e} (bar {rel:g}), cos {c:.7f} (bar {cos})")
    assert r <= rel and c >= cos, f"{what}: rel L2 {r:.3e} (<= {rel}), cos {c:.6f} (>= {cos})"
    return r, c


def same_fraction(got, ref) -> float:
    """Fraction of elements with identical values (bf16 results against bf16 mids)."""
    return float(np.mean(np.asarray(got) == np.asarray(ref)))


def workspace_views(h3, cs, shp, ws, names=None) -> dict:
    """Host copies of a block's intermediates from a workspace laid out with
    H3DIT_KEEP_INTERMEDIATES (library row order): q, k, v [H, N, d]; g, o [N, A];
    x1, h2 [N, D]; u [N, F] (float64 values of the bf16 data); idx [H, Tv, k] int32.
    ``names`` restricts the copy (full-size shapes)."""
    import torch
    lay = h3.workspace_layout(cs)
    N, H, d, A, D, F = (shp.n_rows, shp.heads, shp.head_dim, shp.attn_width, shp.hidden,
                        shp.mlp_width)
    tv, ks = shp.n_video_tiles, min(shp.topk, shp.n_video_tiles)
    spec = {"q": ("q", (H, N, d)), "k": ("k", (H, N, d)), "v": ("v", (H, N, d)),
            "g": ("g", (N, A)), "o": ("o", (N, A)), "x1": ("x1", (N, D)), "h2": ("h", (N, D)),
            "u": ("u", (N, F))}
    out = {}
    for n in (names or list(spec) + ["idx"]):
        if n == "idx":
            off, size = lay["idx"], H * tv * ks * 4
            out[n] = ws[off:off + size].view(torch.int32).view(H, tv, ks).cpu().numpy()
            continue
        region, shape = spec[n]
        off = lay[region]
        assert off is not None, region
        size = int(np.prod(shape)) * 2
        out[n] = host_f64(ws[off:off + size].view(torch.bfloat16).view(*shape))
    return out


def router_on_gpu_inputs(q, k, shp, idx, sets=None):
    """The router's selections against the oracle's on the GPU's own q and k (raster row
    order, float64 values of the bf16 data): index sets must be equal except near-ties.
    Returns the number of near-tied (head, tile) pairs that differ."""
    import oracle
    P, V = shp.n_prefix, shp.n_video
    sets = oracle.shape_tiles(shp) if sets is None else sets
    S = oracle.tile_scores(oracle.tile_means(q, P, V, shp.tile, sets),
                           oracle.tile_means(k, P, V, shp.tile, sets))
    ks = min(shp.topk, shp.n_video_tiles)
    return compare_topk(idx, oracle.topk_select(S, ks), S, ks)


def check_bf16_stage(got, ref, what, min_same=0.995):
    """A stage's bf16 output against the oracle's rounding of the SAME inputs: only
    fp32-vs-float64 sums separate the two.  Nearly every value identical, and every
    value within one bf16 spacing plus 2^-12 of the tensor's RMS (a sum that cancels to
    near zero carries the fp32 error of its much larger terms, which one spacing of the
    small result does not cover)."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    same = same_fraction(got, ref)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    tol = np.maximum(np.abs(got), np.abs(ref)) * 2.0 ** -7 + 2.0 ** -12 * rms + 1e-30
    worst = float(np.max(np.abs(got - ref) / tol)) if got.size else 0.0
    log(f"{what}: identical {same:.6f} (bar {min_same}), largest difference {worst:.3f} of "
        f"(1 bf16 spacing + 2^-12 RMS) (bar 1)")
    assert worst <= 1.0 and same >= min_same, f"{what}: identical {same}, worst {worst}"
