"""Float64 CPU oracle of one routed-attention DiT block and the denoiser step.

Test infrastructure only (see the package docstring): nothing in the product
library imports or calls this module.

Sources, cited by page title and section:

* "TensorFold #949" = the page "ashhart/TensorFold pull request #949"
  (MiniMax H3 / FastH3 denoiser on Metal): the "Precision" list, the
  "What it adds" file list (block.zig, h3_routing.metal, h3_attention.metal),
  the "Receipts" tile counts and the "Kernel contract" rules.
* "h3.c README" = the page "Antirez/h3.c: MiniMax H3 inference engine for Mac
  computers": the sampler/reuse paragraph, the layer-thinning paragraph, the
  fused gated-AdaLN paragraph and the Q/K RMS + RoPE paragraph.
* "H3-metal (zh)" = the page "H3-metal：Apple Silicon上的MiniMax-H3原生推理",
  control table (whole-denoiser reuse row).

Readings taken where the pages leave a step open are marked "Reading:".
Array conventions: activations are [rows, features]; head-major tensors are
[H, N, d]; linear weights are [out, in] and ``linear`` computes h @ W^T + b.

Pins.  Every public function below is tied, by the tests named beside it in
tests/test_oracle_pins.py, to something other than itself: a closed form, an
invariant, a brute force on a tiny input, an independent library routine or a
value printed on the pages (tests/golden/).  The pages print no worked example
of a whole block or denoiser step, so the composed functions (block_forward,
denoise_forward, sample_step and the loops) are pinned through closed-form
special cases of each of their stages rather than by value on general inputs.

PIN TABLE (function: pin tests, without their "test_" prefix)
  bf16: bf16_against_torch_conversion, bf16_hand_values
  f32: output_head_constant_rows, token_pool_brute_force_pairs
  rms_modulate: rms_modulate_closed_forms
  modulate_rows: modulate_rows_picks_each_rows_table, block_prefix_table_norm_applies_to_its_rows
  gate_rows: gate_rows_picks_each_rows_table, block_prefix_table_zero_gates_split_by_modality
  linear: linear_small_integers_exact
  gelu_erf: gelu_closed_forms
  silu: silu_closed_forms
  swiglu_split: swiglu_split_layout_and_block
  mlp_inner: swiglu_split_layout_and_block, block_mlp_half_closed_form
  head_rms_norm: head_rms_norm_unit_rms
  rope: rope_closed_form_and_relative_position
  rope_axis_split: rope_axis_split_values
  rope_3d: rope_3d_brute_force_complex, rope_3d_relative_per_axis_and_isolation
  rope_coords: rope_coords_raster
  rope_coords_pooled: rope_coords_pooled_positions
  video_tiles: tile_means_brute_force_and_partial_tile, tile_sets_slices_and_cubes
  cube_tiles: cube_tiles_receipt_golden, cube_tiles_partition_by_membership
  tile_sets: tile_sets_slices_and_cubes
  shape_tiles: tile_sets_slices_and_cubes
  tile_means: tile_means_brute_force_and_partial_tile
  tile_scores: tile_scores_brute_force
  topk_select: topk_brute_force_with_ties_and_nans, topk_nan_regression_exact_k
  topk_gap: topk_all_and_gap
  topk_set_valid: topk_all_and_gap
  attend: routed_all_tiles_equals_dense_brute_force, block_all_tiles_equals_dense,
    attend_bf16_weights_streamed_in_octaves
  routed_attention: routed_all_tiles_equals_dense_brute_force, routed_keyset_brute_force,
    attention_row_stochastic_and_zero_query
  pooled_branch: pooled_closed_forms
  gate_mix: gate_mix_brute_force
  attention_layer: router_tile_permutation_equivariance, block_closed_form_constant_rows,
    attention_layer_given_selections
  qkv_heads: qkv_heads_layout_by_loops
  block_forward: block_closed_form_constant_rows, block_mlp_half_closed_form,
    block_zero_gates_pass_residual, block_all_tiles_equals_dense,
    block_prefix_table_zero_gates_split_by_modality
  block_forward_rows: block_rows_equals_full_block
  euler_update: euler_power_of_two_exact, euler_and_extrapolation_per_modality_rows
  extrapolate: extrapolation_exact_for_linear_velocity
  fresh_steps: fresh_step_counts_golden
  sigma_schedule: sigma_schedule_shift_endpoints_and_composition
  denoise_forward: denoise_forward_closed_forms
  denoise_loop: denoise_loop_orchestration_without_blocks,
    denoise_loop_per_modality_without_blocks
  thin_layers: thin_layers_hand_example
  patch_in: patch_in_small_integers_brute_force
  output_head: output_head_constant_rows
  sample_x0: sample_step_without_blocks_is_the_heads_of_the_patches
  sample_heads: sample_step_without_blocks_is_the_heads_of_the_patches
  sample_step: sample_step_without_blocks_is_the_heads_of_the_patches,
    core_reuse_reproduces_the_fresh_velocity
  sample_loop: sample_loop_core_reuse_without_blocks_equals_every_pass_fresh
  reduced_shape: reduced_shape_hand_values
  token_pool: token_pool_brute_force_pairs
  token_restore: token_restore_identity_and_pair_update
  run_blocks: run_blocks_reduction_boundaries
END PIN TABLE
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf as _erf

__all__ = [
    "bf16", "f32", "rms_modulate", "linear", "gelu_erf", "silu", "swiglu_split", "mlp_inner",
    "head_rms_norm", "rope", "rope_axis_split", "rope_3d", "rope_coords",
    "video_tiles", "cube_tiles", "tile_sets", "shape_tiles", "tile_means", "tile_scores", "topk_select", "topk_gap",
    "topk_set_valid", "attend", "routed_attention", "pooled_branch", "gate_mix",
    "attention_layer", "qkv_heads", "block_forward", "block_forward_rows", "euler_update",
    "extrapolate",
    "fresh_steps", "sigma_schedule", "denoise_forward", "denoise_loop", "thin_layers",
    "patch_in", "output_head", "sample_x0", "sample_heads", "sample_step", "sample_loop",
    "rope_coords_pooled", "reduced_shape", "token_pool", "token_restore", "run_blocks",
    "modulate_rows", "gate_rows",
]


# ---------------------------------------------------------------------------
# Storage roundings ("mids")
# ---------------------------------------------------------------------------

def bf16(a) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even), returned as float64.

    bf16 = 1 sign, 8 exponent, 7 mantissa bits (the storage type of weights and
    activations, TensorFold #949 "Precision").  Done directly on the float64
    bits: drop the low 45 mantissa bits with round-to-nearest-even; values at
    or above 2^128 become inf; below 2^-126 (bf16 subnormals) the value is
    rounded to a multiple of 2^-133.
    """
    a = np.asarray(a, dtype=np.float64)
    u = np.ascontiguousarray(a).view(np.uint64)
    low = np.uint64((1 << 45) - 1)
    lsb = (u >> np.uint64(45)) & np.uint64(1)
    with np.errstate(over="ignore"):
        r = (u + np.uint64((1 << 44) - 1) + lsb) & ~low
    out = r.view(np.float64).reshape(a.shape).copy()
    big = np.abs(out) >= 2.0 ** 128
    out[big] = np.copysign(np.inf, a[big])
    small = np.abs(a) < 2.0 ** -126
    if np.any(small):
        out[small] = np.round(a[small] * 2.0 ** 133) / 2.0 ** 133
    nan = np.isnan(a)
    out[nan] = np.nan
    return out


def f32(a) -> np.ndarray:
    """Round to float32 (nearest even) and return as float64."""
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Row operations
# ---------------------------------------------------------------------------

def rms_modulate(x, shift, scale, eps: float = 1e-6) -> np.ndarray:
    """Modulated norm: bf16( x / sqrt(mean(x^2) + eps) * (1 + scale) + shift ).

    TensorFold #949 "What it adds" (block.zig: "modulated norm"); the h3.c
    README's fused gated-AdaLN paragraph names an RMS over each row.
    Reading: no learned weight, eps = 1e-6, the adaLN form (1 + scale).
    Output is a bf16 mid (the projection input is bf16).
    """
    x = np.asarray(x, dtype=np.float64)
    inv = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return bf16(x * inv * (1.0 + np.asarray(scale, np.float64)) + np.asarray(shift, np.float64))


def linear(h, w, b=None) -> np.ndarray:
    """h @ w^T + b with float64 sums of the (bf16) operands, no rounding.

    TensorFold #949 "Precision": bf16 weights and activations, fp32 sums.
    The oracle sums in float64; the bf16 result rounding is applied by the
    caller where the method stores bf16.
    """
    y = np.asarray(h, np.float64) @ np.asarray(w, np.float64).T
    if b is not None:
        y = y + np.asarray(b, np.float64)
    return y


def gelu_erf(x) -> np.ndarray:
    """GELU(x) = 0.5 x (1 + erf(x / sqrt 2)).

    Reading: the 4x-GELU MLP of the synthetic block shapes; the pages' own
    checkpoint uses SwiGLU, and no GELU form is printed, so the exact erf form
    is taken.
    """
    x = np.asarray(x, np.float64)
    return 0.5 * x * (1.0 + _erf(x / math.sqrt(2.0)))


def silu(x) -> np.ndarray:
    """SiLU(x) = x / (1 + exp(-x)), the activation of the SwiGLU gate."""
    x = np.asarray(x, np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def swiglu_split(w1, b1):
    """Gate and up halves of a SwiGLU fc1 stored [2F, D] with gate/up rows interleaved in
    groups of 128 (the library's storage convention): returns (Wg, bg, Wu, bu), [F, D] / [F]."""
    w1 = np.asarray(w1, np.float64)
    b1 = np.asarray(b1, np.float64)
    F2, D = w1.shape
    g = w1.reshape(F2 // 256, 2, 128, D)
    bb = b1.reshape(F2 // 256, 2, 128)
    return (g[:, 0].reshape(-1, D), bb[:, 0].reshape(-1), g[:, 1].reshape(-1, D),
            bb[:, 1].reshape(-1))


def mlp_inner(h2, wts: dict, mlp: str = "gelu") -> np.ndarray:
    """The MLP's inner activations u, rounded to bf16.

    "gelu": u = GELU(h2 W1^T + b1) (the synthetic 4x shapes).
    "swiglu": u = SiLU(h2 Wg^T + bg) * (h2 Wu^T + bu), the pages' MLP (h3.c README:
    the FC1 gate/up products feed SwiGLU and only the activated intermediate is
    written; TensorFold #949 "What it adds": h3_swiglu).  No rounding between the
    two products and the activation.
    """
    if mlp == "swiglu":
        wg, bg, wu, bu = swiglu_split(wts["w1"], wts["b1"])
        return bf16(silu(linear(h2, wg, bg)) * linear(h2, wu, bu))
    return bf16(gelu_erf(linear(h2, wts["w1"], wts["b1"])))


def head_rms_norm(x, w, eps: float = 1e-6) -> np.ndarray:
    """Per-head RMS norm over the last axis (d) times a learned weight w [d].

    h3.c README, Q/K RMS normalization + RoPE paragraph; TensorFold #949
    "What it adds" (h3_routing.metal: head layout with q/k norm and rotary).
    """
    x = np.asarray(x, np.float64)
    inv = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x * inv * np.asarray(w, np.float64)


def _rotate_half(x, ang) -> np.ndarray:
    """Turn pairs (c, c + d/2) of the last axis by ang[..., row, c]."""
    x = np.asarray(x, np.float64)
    half = x.shape[-1] // 2
    cos, sin = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., :half], x[..., half:]
    out = np.empty_like(x)
    out[..., :half] = x0 * cos - x1 * sin
    out[..., half:] = x1 * cos + x0 * sin
    return out


def rope(x, positions, theta: float = 10000.0) -> np.ndarray:
    """Rotary embedding, rotate-half pairing, over the last axis.

    Pairs (c, c + d/2) for c < d/2 are rotated by angle p * theta^(-2c/d),
    p = the packed row index.  Reading: the pages name "q/k norm and rotary"
    but give no axes or base; a 1-D rotary over the packed row index with
    theta = 10,000 is taken when no video grid is given.
    """
    d = np.shape(x)[-1]
    c = np.arange(d // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * c / d)
    ang = np.asarray(positions, np.float64)[:, None] * inv_freq[None, :]  # [N, half]
    return _rotate_half(x, ang)


def rope_axis_split(d: int):
    """Rotary pairs per axis (time, height, width) for head width d.

    Reading: the pages speak of spatial and temporal rotary coordinates (the h3.c
    README halves the spatial ones at 256 square) without the split; the common
    video-DiT split gives height and width floor(d/6) pairs each and time the rest.
    """
    half = d // 2
    ms = half // 3
    return half - 2 * ms, ms, ms


def rope_3d(x, coords, theta: float = 10000.0) -> np.ndarray:
    """3-D rotary: pair c of axis a (local index j of m_a pairs) turns by
    coords[row, a] * theta^(-j / m_a); axes in the order time, height, width over
    consecutive pair ranges."""
    d = np.shape(x)[-1]
    coords = np.asarray(coords, np.float64)
    ang = np.empty((coords.shape[0], d // 2))
    c0 = 0
    for a, m in enumerate(rope_axis_split(d)):
        j = np.arange(m, dtype=np.float64)
        ang[:, c0:c0 + m] = coords[:, a:a + 1] * theta ** (-j / m)[None, :]
        c0 += m
    return _rotate_half(x, ang)


def rope_coords(n_prefix: int, n_video: int, grid) -> np.ndarray:
    """Per packed row (t, h, w) for the 3-D rotary: text/audio row p -> (p, p, p)
    (reading: the pages give the prefix rows no grid), video row in raster order
    v = (t * H + h) * W + w -> (t, h, w)."""
    T, Hg, Wg = grid
    out = np.empty((n_prefix + n_video, 3), np.int64)
    p = np.arange(n_prefix)
    out[:n_prefix] = p[:, None]
    v = np.arange(n_video)
    out[n_prefix:, 0] = v // (Hg * Wg)
    out[n_prefix:, 1] = (v // Wg) % Hg
    out[n_prefix:, 2] = v % Wg
    return out


def rope_coords_pooled(n_prefix: int, grid, pair_w: int) -> np.ndarray:
    """``rope_coords`` of a token-reduced grid (T, H, ceil(W/2)): the row for column j
    pools full columns 2j and 2j + 1 and sits at their mean, 2j + 0.5; a lone last
    column of an odd width stays at 2j.  Reading: the pages do not give the pooled
    rows' rotary positions."""
    out = rope_coords(n_prefix, int(np.prod(grid)), grid).astype(np.float64)
    j = out[n_prefix:, 2]
    out[n_prefix:, 2] = np.where(2 * j + 1 < pair_w, 2 * j + 0.5, 2 * j)
    return out


# ---------------------------------------------------------------------------
# Router: tile means, tile scores, top-k   (TensorFold #949 "What it adds":
# h3_routing.metal tile means / tile scores / top-k; "Precision": fp32 tile
# means, scores and top-k; "Kernel contract": NaN ranks as -inf, ties go to
# the lower tile)
# ---------------------------------------------------------------------------

def video_tiles(n_prefix: int, n_video: int, tile: int = 64):
    """[(first_row, n_valid)] for each video tile; the last may be partial.

    Reading: video rows [P, N) are cut into contiguous 64-row tiles in packed
    order; the pages' 4x4x4 cube map is a fixed row permutation applied before
    this step and is not part of these shapes.
    """
    return [(n_prefix + t * tile, min(tile, n_video - t * tile))
            for t in range((n_video + tile - 1) // tile)]


def cube_tiles(n_prefix: int, grid, cube=(4, 4, 4)) -> list:
    """Packed row indices of each video tile when the video rows are the latent grid
    T x H x W in raster order, cut into ct x ch x cw cubes (edge cubes clipped).

    TensorFold #949 "Receipts": 4 x 4 x 4 cubes give 280 video tiles at 864 x 480 x 124
    (a 37 x 15 x 27 grid).  Reading: cubes numbered in raster (cube t, h, w) order;
    the rows of a cube listed in raster (t, h, w) order.
    """
    T, Hg, Wg = grid
    ct, ch, cw = cube
    tiles = []
    for a in range(0, T, ct):
        for b in range(0, Hg, ch):
            for c in range(0, Wg, cw):
                rows = [n_prefix + (t * Hg + h) * Wg + w
                        for t in range(a, min(T, a + ct))
                        for h in range(b, min(Hg, b + ch))
                        for w in range(c, min(Wg, c + cw))]
                tiles.append(np.array(rows, dtype=np.int64))
    return tiles


def tile_sets(n_prefix: int, n_video: int, tile: int = 64, grid=None, cube=(4, 4, 4)) -> list:
    """Packed row indices of each video tile: contiguous slices, or cubes of ``grid``."""
    if grid is None:
        return [np.arange(r0, r0 + nv) for r0, nv in video_tiles(n_prefix, n_video, tile)]
    return cube_tiles(n_prefix, grid, cube)


def shape_tiles(shape) -> list:
    return tile_sets(shape.n_prefix, shape.n_video, shape.tile,
                     getattr(shape, "video_grid", None), getattr(shape, "cube", (4, 4, 4)))


def tile_means(X, n_prefix: int, n_video: int, tile: int = 64, sets=None) -> np.ndarray:
    """Mean over the rows of each video tile: [H, N, d] -> [H, Tv, d] (float64).
    ``sets``: the tiles' row indices (default: contiguous 64-row slices)."""
    X = np.asarray(X, np.float64)
    sets = tile_sets(n_prefix, n_video, tile) if sets is None else sets
    out = np.empty((X.shape[0], len(sets), X.shape[2]))
    for t, rows in enumerate(sets):
        out[:, t, :] = X[:, rows, :].sum(axis=1) / len(rows)
    return out


def tile_scores(mq, mk) -> np.ndarray:
    """S[h, i, j] = mq[h, i] . mk[h, j], unscaled (float64).

    Reading: the pages do not say whether tile scores carry 1/sqrt(d); the
    scale does not change the order, so S is unscaled here and the pooled
    branch applies 1/sqrt(d).
    """
    return np.einsum("hid,hjd->hij", np.asarray(mq, np.float64), np.asarray(mk, np.float64))


def topk_select(scores, k: int) -> np.ndarray:
    """Top-k tiles per (h, i) taken on fp32 scores: [H, Tq, T] -> int32 [H, Tq, min(k, T)].

    Rule (TensorFold #949 "Kernel contract"): a NaN score ranks as -inf; among
    equal scores the lower tile index wins.  The decision is made on scores
    rounded to fp32 (the routing precision on the pages).  Output indices are
    sorted ascending.
    """
    s = f32(scores)
    s = np.where(np.isnan(s), -np.inf, s)
    H, Tq, T = s.shape
    kk = min(k, T)
    out = np.empty((H, Tq, kk), dtype=np.int32)
    j = np.arange(T)
    for h in range(H):
        for i in range(Tq):
            order = np.lexsort((j, -s[h, i]))  # by score descending, then index ascending
            out[h, i] = np.sort(order[:kk])
    return out


def topk_gap(scores, k: int) -> np.ndarray:
    """Relative float64 gap between the k-th and (k+1)-th largest score per (h, i).

    Used to classify near-ties (gap < 1e-5): where two correct implementations
    may choose different tiles.  Returns +inf where k >= T.
    """
    s = np.asarray(scores, np.float64)
    s = np.where(np.isnan(s), -np.inf, s)
    T = s.shape[-1]
    if k >= T:
        return np.full(s.shape[:-1], np.inf)
    srt = -np.sort(-s, axis=-1)
    a, b = srt[..., k - 1], srt[..., k]
    with np.errstate(invalid="ignore"):
        gap = (a - b) / np.maximum(np.abs(a), 1e-30)
    return np.where(np.isfinite(gap), gap, np.inf)


def topk_set_valid(scores_row, chosen, tol: float = 1e-5) -> bool:
    """True if ``chosen`` is a top-k set of ``scores_row`` up to a relative tolerance."""
    s = np.where(np.isnan(scores_row), -np.inf, np.asarray(scores_row, np.float64))
    chosen = np.asarray(chosen)
    mask = np.zeros(s.shape[0], bool)
    mask[chosen] = True
    if mask.all() or len(set(chosen.tolist())) != len(chosen):
        return bool(mask.all() and len(set(chosen.tolist())) == len(chosen))
    lo = s[mask].min()
    hi = s[~mask].max()
    return bool(lo >= hi - tol * max(abs(lo), abs(hi), 1e-30))


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def attend(q, k, v, scale: float, p_bf16: bool = False) -> np.ndarray:
    """softmax(q k^T * scale) v for one head; bidirectional, no mask.

    With ``p_bf16`` the unnormalised weights are rounded to bf16 before the
    value product, as TensorFold #949 "Precision" states for the routed
    attention; the row sum l uses the unrounded weights (reading: the pages do
    not say which).  The pages do not say against which maximum the
    unnormalised weights are taken, and a bf16 rounding depends on it.
    Reading: against a whole power of two, p_j = 2^(z_j - M) with
    z_j = s_j log2(e) and M = ceil(max_j z_j).  Scaling by a power of two
    commutes with the rounding, so the result is the same for every integer M
    (any maximum a streaming softmax meets on the way, if it keeps its maximum
    in whole octaves); without rounding it is the exact softmax.
    Default: exact float64.
    """
    s = (np.asarray(q, np.float64) @ np.asarray(k, np.float64).T) * scale
    if p_bf16:
        z = s * (1.0 / math.log(2.0))
        M = np.ceil(z.max(axis=1, keepdims=True))
        p = np.exp2(z - M)
        l = p.sum(axis=1, keepdims=True)
        return (bf16(p) @ np.asarray(v, np.float64)) / l
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    return (p @ np.asarray(v, np.float64)) / l


def routed_attention(Q, K, V, n_prefix: int, n_video: int, idx, tile: int = 64,
                     p_bf16: bool = False, tiles=None, sets=None) -> np.ndarray:
    """Tile-routed attention, [H, N, d] each -> O [H, N, d] (float64).

    TensorFold #949 "What it adds" (h3_attention.metal: tile-routed attention
    with fp32 scores and online softmax) and "Receipts" (the tile count puts 8
    prefix tiles beside the 56 video tiles each query keeps: prefix tiles are
    kept for every query).
    * prefix (text + audio) query rows attend densely to all N rows;
    * a video query row in tile i attends to every prefix row plus the valid
      rows of the tiles idx[h, i].
    Scale 1/sqrt(d).  ``tiles`` optionally restricts the work to a list of
    (h, i) video query tiles (rows elsewhere are left zero); ``sets`` are the
    tiles' row indices (default: contiguous 64-row slices).
    """
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    H, N, d = Q.shape
    scale = 1.0 / math.sqrt(d)
    O = np.zeros_like(Q)
    vt = tile_sets(n_prefix, n_video, tile) if sets is None else sets
    if tiles is None:
        for h in range(H):
            if n_prefix:
                O[h, :n_prefix] = attend(Q[h, :n_prefix], K[h], V[h], scale, p_bf16)
        tiles = [(h, i) for h in range(H) for i in range(len(vt))]
    pre = np.arange(n_prefix)
    for h, i in tiles:
        qr = vt[i]
        kr = np.concatenate([pre] + [vt[j] for j in idx[h, i]])
        O[h, qr] = attend(Q[h, qr], K[h, kr], V[h, kr], scale, p_bf16)
    return O


def pooled_branch(S, mv, head_dim: int) -> np.ndarray:
    """Pooled branch: op[h, i] = sum_j softmax_j(S[h, i, j] / sqrt(d)) mv[h, j].

    TensorFold #949 "What it adds" ("the pooled branch", h3_routing.metal).
    Reading: attention of each video query tile's mean over all video tile
    means, reusing the tile scores (the coarse half of a coarse + fine sparse
    attention).
    """
    z = np.asarray(S, np.float64) / math.sqrt(head_dim)
    z = z - z.max(axis=-1, keepdims=True)
    w = np.exp(z)
    w = w / w.sum(axis=-1, keepdims=True)
    return w @ np.asarray(mv, np.float64)


def gate_mix(O, G, pooled, n_prefix: int, n_video: int, tile: int = 64, sets=None) -> np.ndarray:
    """o[r, h*d:(h+1)*d] = O[h, r] + G[r, h*d:(h+1)*d] * pooled[h, tile(r)] for video rows.

    TensorFold #949 "What it adds" ("the routing gate", h3_gate_mix).
    Reading: the gate is a linear (unsquashed) full-width product; prefix rows
    get no pooled term.  Returns [N, H*d] float64, not rounded.
    """
    O = np.asarray(O, np.float64)
    H, N, d = O.shape
    out = O.transpose(1, 0, 2).reshape(N, H * d).copy()
    if pooled is None or G is None or n_video == 0:
        return out
    G = np.asarray(G, np.float64)
    sets = tile_sets(n_prefix, n_video, tile) if sets is None else sets
    pb = np.asarray(pooled, np.float64)
    for i, rows in enumerate(sets):
        out[rows] += G[rows] * pb[:, i, :].reshape(H * d)[None, :]
    return out


def attention_layer(Q, K, V, G, n_prefix: int, n_video: int, topk: int, tile: int = 64,
                    pooled: bool = True, p_bf16: bool = False, sets=None, idx=None) -> dict:
    """Router + routed/dense attention + pooled branch + gate mix.

    Inputs are the bf16 values of Q, K, V [H, N, d] and G [N, H*d] (or None).
    Returns the intermediates and ``o`` = bf16(mixed output) [N, H*d].  ``idx``
    [H, Tv, k], when given, replaces the router's selections in the attention
    (the comparison rule for near-tied selections recomputes the outputs with
    the other implementation's tiles); the returned "idx" stays the router's.
    """
    Q = np.asarray(Q, np.float64)
    d = Q.shape[2]
    sets = tile_sets(n_prefix, n_video, tile) if sets is None else sets
    mq = tile_means(Q, n_prefix, n_video, tile, sets)
    mk = tile_means(K, n_prefix, n_video, tile, sets)
    mv = tile_means(V, n_prefix, n_video, tile, sets)
    S = tile_scores(mq, mk)
    idx_r = topk_select(S, topk)
    gap = topk_gap(S, topk)
    idx = idx_r if idx is None else np.asarray(idx)
    O = routed_attention(Q, K, V, n_prefix, n_video, idx, tile, p_bf16, sets=sets)
    pb = pooled_branch(S, mv, d) if pooled else None
    mixed = gate_mix(O, G, pb, n_prefix, n_video, tile, sets)
    return {"mq": mq, "mk": mk, "mv": mv, "scores": S, "idx": idx_r, "gap": gap,
            "O": O, "pooled": pb, "o_f64": mixed, "o": bf16(mixed)}


# ---------------------------------------------------------------------------
# Block
# ---------------------------------------------------------------------------

def qkv_heads(qkvg, heads: int, head_dim: int, qnorm_w=None, knorm_w=None,
              eps: float = 1e-6, theta: float = 10000.0, use_rope: bool = True, coords=None):
    """Split [N, 4A] projection rows into head-major Q, K, V [H, N, d] and G [N, A].

    q and k get the per-head RMS norm (learned weight) and the rotary, then are
    rounded to bf16; v and g are the projection's bf16 values.  ``coords`` [N, 3]
    selects the 3-D rotary.  Column order of
    the projection: [Q | K | V | G], each A = H*d wide, head-major inside.
    TensorFold #949 "What it adds" (block.zig "q/k/v and the routing gate,
    head layout"); h3.c README Q/K RMS + RoPE paragraph.
    """
    qkvg = np.asarray(qkvg, np.float64)
    N = qkvg.shape[0]
    A = heads * head_dim
    parts = [qkvg[:, s * A:(s + 1) * A].reshape(N, heads, head_dim).transpose(1, 0, 2)
             for s in range(3)]
    q, k, v = parts
    pos = np.arange(N)
    if qnorm_w is not None:
        q = head_rms_norm(q, qnorm_w, eps)
    if knorm_w is not None:
        k = head_rms_norm(k, knorm_w, eps)
    if use_rope and coords is not None:  # 3-D rotary over (t, h, w)
        q = rope_3d(q, coords, theta)
        k = rope_3d(k, coords, theta)
    elif use_rope:
        q = rope(q, pos, theta)
        k = rope(k, pos, theta)
    return bf16(q), bf16(k), v.copy(), qkvg[:, 3 * A:4 * A].copy()


def modulate_rows(x, mod, mod_prefix, n_prefix: int, k_shift: int, k_scale: int,
                  eps: float = 1e-6, rows=None) -> np.ndarray:
    """``rms_modulate`` with the text and audio rows (packed index < n_prefix) on their
    own table when ``mod_prefix`` is given (independent audio conditioning; reading:
    text rows share the audio rows' table).  ``rows`` are the packed indices of x."""
    mod = np.asarray(mod, np.float64)
    if mod_prefix is None:
        return rms_modulate(x, mod[k_shift], mod[k_scale], eps)
    modp = np.asarray(mod_prefix, np.float64)
    r = np.arange(np.shape(x)[0]) if rows is None else np.asarray(rows)
    pre = r < n_prefix
    out = np.empty(np.shape(x))
    if pre.any():
        out[pre] = rms_modulate(np.asarray(x)[pre], modp[k_shift], modp[k_scale], eps)
    if (~pre).any():
        out[~pre] = rms_modulate(np.asarray(x)[~pre], mod[k_shift], mod[k_scale], eps)
    return out


def gate_rows(mod, mod_prefix, n_prefix: int, k: int, rows) -> np.ndarray:
    """Gate row k of the modulation for each packed row index in ``rows``: [R, D] or [D]."""
    mod = np.asarray(mod, np.float64)
    if mod_prefix is None:
        return mod[k]
    pre = (np.asarray(rows) < n_prefix)[:, None]
    return np.where(pre, np.asarray(mod_prefix, np.float64)[k], mod[k])


def _coords(shape):
    grid = getattr(shape, "video_grid", None)
    if grid is None:
        return None
    if getattr(shape, "pair_w", 0):
        return rope_coords_pooled(shape.n_prefix, grid, shape.pair_w)
    return rope_coords(shape.n_prefix, shape.n_video, grid)


# ---------------------------------------------------------------------------
# Token reduction (h3.c README, token-reduction paragraph: horizontally adjacent
# video tokens run as one row through the middle blocks, text and audio exact, a
# full-resolution bypass kept, each token restored as its original value plus the
# update its pair received)
# ---------------------------------------------------------------------------

def reduced_shape(shape):
    """The reduced section's shape: video grid T x H x ceil(W/2), rotary at pair means."""
    T, Hg, Wg = shape.video_grid
    Wr = (Wg + 1) // 2
    return shape.with_(n_video=T * Hg * Wr, video_grid=(T, Hg, Wr), pair_w=Wg,
                       token_reduction=False)


def token_pool(x, shape):
    """(x_r, baseline): prefix rows as they are, then per (t, h, j) the mean of video
    tokens (t, h, 2j) and (t, h, 2j + 1) (fp32 sum, halved, rounded to bf16; a lone last
    token of an odd row passes as it is), rows in raster order of the reduced grid.
    Reading: "pairs" is taken as the mean."""
    T, Hg, Wg = shape.video_grid
    P = shape.n_prefix
    x = np.asarray(x, np.float64)
    v = x[P:].reshape(T, Hg, Wg, -1)
    pooled = v[:, :, 0::2].copy()
    npair = Wg // 2
    pooled[:, :, :npair] = bf16(f32(v[:, :, 0:2 * npair:2] + v[:, :, 1:2 * npair:2]) * 0.5)
    base = pooled.reshape(-1, x.shape[1])
    return np.concatenate([x[:P], base], axis=0), base


def token_restore(bypass, x_r, base, shape) -> np.ndarray:
    """Full rows again: prefix rows from x_r; video token (t, h, w) =
    bf16(bypass + (x_r - base) of its pair (t, h, w // 2)), in fp32 arithmetic."""
    T, Hg, Wg = shape.video_grid
    P = shape.n_prefix
    Wr = (Wg + 1) // 2
    D = np.shape(bypass)[1]
    d = f32(np.asarray(x_r, np.float64)[P:] - np.asarray(base, np.float64)).reshape(T, Hg, Wr, D)
    dfull = np.repeat(d, 2, axis=2)[:, :, :Wg].reshape(-1, D)
    out = np.array(bypass, np.float64)
    out[:P] = np.asarray(x_r, np.float64)[:P]
    out[P:] = bf16(f32(out[P:] + dfull))
    return out


def run_blocks(x, blocks: list, shape, block_ids=None, reduction=None) -> np.ndarray:
    """Run the blocks ``block_ids`` on x, with token reduction over the block positions
    [first, last) when ``reduction`` = (first, last) is given (first < last)."""
    ids = list(range(len(blocks))) if block_ids is None else list(block_ids)
    first, last = reduction if reduction is not None else (-1, -1)
    on = reduction is not None and 0 <= first < last and first < len(ids)
    rs = reduced_shape(shape) if on else None
    bypass = base = None
    for pos, b in enumerate(ids):
        if on and pos == first:
            bypass = x
            x, base = token_pool(x, shape)
        if on and pos == last:
            x = token_restore(bypass, x, base, shape)
        s = rs if on and first <= pos < last else shape
        x = block_forward(x, blocks[b], s)["x2"]
    if on and last >= len(ids):
        x = token_restore(bypass, x, base, shape)
    return x


def block_forward(x, wts: dict, shape, p_bf16: bool = False, idx=None) -> dict:
    """One DiT block on the packed rows x (bf16 values, [N, D]).

    TensorFold #949 "What it adds" (block.zig: modulated norm, q/k/v and the
    routing gate, head layout, routing, attention, the pooled branch, the out
    projection and the MLP) and h3.c README (gated residual adds and AdaLN).
    Reading: the MLP is 4x GELU for the synthetic shapes and SwiGLU for the
    pages' own shape; gated residuals are x + gate * branch with shift/scale/gate
    rows of the [6, D] table.
    ``wts`` holds float64 values of the bf16 weights and the fp32 table.
    ``p_bf16`` and ``idx`` as in ``attention_layer``.
    """
    s = shape
    mod = np.asarray(wts["mod"], np.float64)
    modp = wts.get("mod_prefix")
    P = s.n_prefix
    x = np.asarray(x, np.float64)
    allr = np.arange(x.shape[0])
    h = modulate_rows(x, mod, modp, P, 0, 1, s.rms_eps)
    qkvg = bf16(linear(h, wts["w_qkvg"], wts["b_qkvg"]))
    q, k, v, g = qkv_heads(qkvg, s.heads, s.head_dim,
                           wts.get("qnorm_w") if s.qk_norm else None,
                           wts.get("knorm_w") if s.qk_norm else None,
                           s.rms_eps, s.rope_theta, s.rope, _coords(s))
    att = attention_layer(q, k, v, g if s.pooled else None, s.n_prefix, s.n_video,
                          s.topk, s.tile, s.pooled, p_bf16, shape_tiles(s), idx)
    x1 = bf16(x + gate_rows(mod, modp, P, 2, allr) * linear(att["o"], wts["w_o"], wts["b_o"]))
    h2 = modulate_rows(x1, mod, modp, P, 3, 4, s.rms_eps)
    u = mlp_inner(h2, wts, getattr(s, "mlp", "gelu"))
    x2 = bf16(x1 + gate_rows(mod, modp, P, 5, allr) * linear(u, wts["w2"], wts["b2"]))
    out = dict(att)
    out.update({"h": h, "qkvg": qkvg, "q": q, "k": k, "v": v, "g": g,
                "x1": x1, "h2": h2, "u": u, "x2": x2})
    return out


def block_forward_rows(x, wts: dict, shape, rows, p_bf16: bool = False, idx=None) -> dict:
    """``block_forward`` evaluated for a subset of output rows (for full-size checks).

    The same steps in the same order as ``block_forward``; only the work that
    the requested rows depend on is done: the projection of every row (keys,
    values and the video query rows that feed the tile means), the router over
    all tiles, attention for the requested rows' query rows / tiles, and the
    out projection and MLP for the requested rows.  ``p_bf16`` and ``idx`` as in
    ``block_forward``.
    """
    s = shape
    mod = np.asarray(wts["mod"], np.float64)
    modp = wts.get("mod_prefix")
    x = np.asarray(x, np.float64)
    rows = np.array(sorted(set(int(r) for r in rows)))
    h = modulate_rows(x, mod, modp, s.n_prefix, 0, 1, s.rms_eps)
    qkvg = bf16(linear(h, wts["w_qkvg"], wts["b_qkvg"]))
    q, k, v, g = qkv_heads(qkvg, s.heads, s.head_dim,
                           wts.get("qnorm_w") if s.qk_norm else None,
                           wts.get("knorm_w") if s.qk_norm else None,
                           s.rms_eps, s.rope_theta, s.rope, _coords(s))
    del qkvg
    P, Vn, tile, d = s.n_prefix, s.n_video, s.tile, s.head_dim
    vt = shape_tiles(s)
    tile_of = np.empty(s.n_rows, np.int64)
    for i, tr in enumerate(vt):
        tile_of[tr] = i
    mq = tile_means(q, P, Vn, tile, vt)
    mk = tile_means(k, P, Vn, tile, vt)
    mv = tile_means(v, P, Vn, tile, vt)
    S = tile_scores(mq, mk)
    idx_r = topk_select(S, s.topk)
    idx = idx_r if idx is None else np.asarray(idx)
    H = s.heads
    O = np.zeros((H, len(rows), d))
    scale = 1.0 / math.sqrt(d)
    for n, r in enumerate(rows):
        for hh in range(H):
            if r < P:
                keys = np.arange(s.n_rows)
            else:
                keys = np.concatenate([np.arange(P)] + [vt[j] for j in idx[hh, tile_of[r]]])
            O[hh, n] = attend(q[hh, [r]], k[hh, keys], v[hh, keys], scale, p_bf16)[0]
    o = O.transpose(1, 0, 2).reshape(len(rows), H * d)
    if s.pooled:
        pb = pooled_branch(S, mv, d)
        for n, r in enumerate(rows):
            if r >= P:
                o[n] += g[r] * pb[:, tile_of[r], :].reshape(H * d)
    o = bf16(o)
    x1 = bf16(x[rows] + gate_rows(mod, modp, s.n_prefix, 2, rows) *
              linear(o, wts["w_o"], wts["b_o"]))
    h2 = modulate_rows(x1, mod, modp, s.n_prefix, 3, 4, s.rms_eps, rows)
    u = mlp_inner(h2, wts, getattr(s, "mlp", "gelu"))
    x2 = bf16(x1 + gate_rows(mod, modp, s.n_prefix, 5, rows) * linear(u, wts["w2"], wts["b2"]))
    return {"rows": rows, "x1": x1, "x2": x2, "idx": idx_r, "scores": S, "o": o}


# ---------------------------------------------------------------------------
# Denoiser step (h3.c README sampler paragraph: first and last passes plus
# every r-th pass run the model, skipped velocities are extrapolated;
# H3-metal (zh) control table: 20 steps give 20 / 11 / 8 fresh evaluations
# at reuse 1 / 2 / 3)
# ---------------------------------------------------------------------------

def _per_row(value_v, value_p, n_rows: int, n_prefix: int):
    """A per-row column of a schedule value: value_p for the first n_prefix rows."""
    if value_p is None or n_prefix == 0:
        return value_v
    return np.where((np.arange(n_rows) < n_prefix)[:, None], value_p, value_v)


def euler_update(z, v, dt: float, dt_prefix=None, n_prefix: int = 0) -> np.ndarray:
    """z + dt * v, computed in float64 and stored as fp32 (the latent type); the text and
    audio rows (index < n_prefix) step by ``dt_prefix`` when given (their own schedule)."""
    z = np.asarray(z, np.float64)
    dtr = _per_row(dt, dt_prefix, z.shape[0], n_prefix) if z.ndim == 2 else dt
    return f32(z + dtr * np.asarray(v, np.float64))


def extrapolate(v_a, v_b, sigma_i: float, sigma_a: float, sigma_b: float,
                prefix=None, n_prefix: int = 0) -> np.ndarray:
    """Linear extrapolation in sigma from the last two fresh velocities.

    v_hat = v_a + (v_a - v_b) * (sigma_i - sigma_a) / (sigma_a - sigma_b).
    Reading: "extrapolates skipped ... velocities" with the variable taken as
    sigma; ``prefix`` = (sigma_i, sigma_a, sigma_b) of the text/audio rows' own
    schedule.  With no second fresh velocity the caller holds v_a.
    """
    v_a = np.asarray(v_a, np.float64)
    v_b = np.asarray(v_b, np.float64)
    c = (sigma_i - sigma_a) / (sigma_a - sigma_b)
    cp = None if prefix is None else (prefix[0] - prefix[1]) / (prefix[1] - prefix[2])
    coef = _per_row(c, cp, v_a.shape[0], n_prefix) if v_a.ndim == 2 else c
    return v_a + (v_a - v_b) * coef


def fresh_steps(n_steps: int, reuse: int) -> list:
    """Steps that run the model: i % reuse == 0, plus the last step."""
    return [i for i in range(n_steps) if i % reuse == 0 or i == n_steps - 1]


def sigma_schedule(n_steps: int, shift: float = 1.0) -> np.ndarray:
    """sigma_i for i = 0..n: uniform 1 - i/n, then the time shift s*t / (1 + (s-1)*t).

    Reading: the pages speak of a released shifted video/audio schedule without
    its formula or values; shift = 1 gives the uniform grid.
    """
    t = 1.0 - np.arange(n_steps + 1, dtype=np.float64) / n_steps
    return shift * t / (1.0 + (shift - 1.0) * t)


def denoise_forward(z, blocks: list, shape, dt: float, block_ids=None, dt_prefix=None) -> dict:
    """One fresh step: x0 = bf16(z); run the kept blocks; v = x_L; z' = z + dt v.

    Reading: the synthetic workload has no patch or output layers, so the last
    hidden rows are the velocity.
    """
    ids = list(range(len(blocks))) if block_ids is None else list(block_ids)
    x = bf16(z)
    for b in ids:
        x = block_forward(x, blocks[b], shape)["x2"]
    v = f32(x)
    P = shape.n_prefix if shape is not None else 0
    return {"v": v, "z": euler_update(z, v, dt, dt_prefix, P)}


def denoise_loop(z, blocks: list, shape, n_steps: int, reuse: int, block_ids=None,
                 sig_video=None, sig_prefix=None) -> dict:
    """A whole sampler run: n_steps Euler steps, fresh velocities on
    ``fresh_steps(n_steps, reuse)``, linear extrapolation in sigma otherwise (holding
    the only fresh velocity while there is one).  ``sig_video`` / ``sig_prefix`` are the
    n_steps + 1 sigmas of the video rows and of the text/audio rows (default: uniform;
    the prefix defaults to the video schedule); dt_i = sigma_{i+1} - sigma_i.
    Returns the final latents and the fresh-step indices.
    """
    sv = sigma_schedule(n_steps) if sig_video is None else np.asarray(sig_video, np.float64)
    sp = sv if sig_prefix is None else np.asarray(sig_prefix, np.float64)
    P = shape.n_prefix if shape is not None else 0
    fresh = set(fresh_steps(n_steps, reuse))
    z = np.asarray(z, np.float64)
    hist = []  # (index, v) of fresh steps, most recent last
    for i in range(n_steps):
        dtv, dtp = sv[i + 1] - sv[i], sp[i + 1] - sp[i]
        if i in fresh:
            r = denoise_forward(z, blocks, shape, dtv, block_ids, dtp)
            hist.append((i, r["v"]))
            z = r["z"]
        else:
            (ia, va) = hist[-1]
            if len(hist) > 1:
                (ib, vb) = hist[-2]
                v = extrapolate(va, vb, sv[i], sv[ia], sv[ib], (sp[i], sp[ia], sp[ib]), P)
            else:
                v = va
            z = euler_update(z, v, dtv, dtp, P)
    return {"z": z, "fresh": sorted(fresh)}


# ---------------------------------------------------------------------------
# Both ends of the denoiser (h3.c README: fp32 96 -> 5,376 video and 32 -> 5,376
# audio patch projections rounded to bf16; final audio / video AdaLN on their
# slices of the residual stream; narrow bf16 output heads; core reuse holds the
# transformer residual while the patch projection and the head are refreshed)
# ---------------------------------------------------------------------------

def patch_in(z, w_in, b_in) -> np.ndarray:
    """x = bf16(z w_in + b_in): w_in input-major [c, D] (fp32 on the pages; exact sums
    here), the result rounded to bf16 as it enters the hidden rows."""
    return bf16(np.asarray(z, np.float64) @ np.asarray(w_in, np.float64)
                + np.asarray(b_in, np.float64))


def output_head(x_rows, mod2, w_out, b_out, eps: float = 1e-6) -> np.ndarray:
    """Final AdaLN then the narrow head: v = bf16(rms(x)(1 + scale) + shift) W_out^T + b,
    returned as fp32 (the latents' type).  Reading: the final AdaLN has the block
    norms' form with its own (shift, scale) table per modality."""
    mod2 = np.asarray(mod2, np.float64)
    h = rms_modulate(x_rows, mod2[0], mod2[1], eps)
    return f32(linear(h, w_out, b_out))


def sample_x0(z_video, z_audio, ends: dict, shape) -> np.ndarray:
    """Packed rows x_0 = [text; patch_in(audio); patch_in(video)] (video rows in the
    order of z_video)."""
    parts = [np.asarray(ends["text"], np.float64).reshape(shape.n_text, shape.hidden)]
    if shape.n_audio:
        parts.append(patch_in(z_audio, ends["w_in_audio"], ends["b_in_audio"]))
    parts.append(patch_in(z_video, ends["w_in_video"], ends["b_in_video"]))
    return np.concatenate(parts, axis=0)


def sample_heads(xL, ends: dict, shape) -> tuple:
    """(v_video, v_audio) from the last hidden rows."""
    P, T = shape.n_prefix, shape.n_text
    vv = output_head(xL[P:], ends["mod_out_video"], ends["w_out_video"], ends["b_out_video"],
                     shape.rms_eps)
    va = (output_head(xL[T:P], ends["mod_out_audio"], ends["w_out_audio"], ends["b_out_audio"],
                      shape.rms_eps) if shape.n_audio else np.zeros((0, 0)))
    return vv, va


def sample_step(z_video, z_audio, ends: dict, blocks: list, shape, kind: str, dt_video: float,
                dt_audio: float, block_ids=None, residual=None, reduction=None) -> dict:
    """One sampler step on the modality latents.  kind "fresh": x_L = blocks(x_0) and the
    residual x_L - x_0 (fp32) is returned; kind "core": x_L = bf16(x_0 + residual).
    Then per modality v = head(x_L rows), z' = fp32(z + dt v)."""
    x0 = sample_x0(z_video, z_audio, ends, shape)
    if kind == "fresh":
        x = run_blocks(x0, blocks, shape, block_ids, reduction)
        res = f32(x - x0)
    elif kind == "core":
        res = residual
        x = bf16(f32(x0 + np.asarray(residual, np.float64)))
    else:
        raise ValueError(kind)
    vv, va = sample_heads(x, ends, shape)
    zv = f32(np.asarray(z_video, np.float64) + dt_video * vv)
    za = f32(np.asarray(z_audio, np.float64) + dt_audio * va) if shape.n_audio else z_audio
    return {"z_video": zv, "z_audio": za, "v_video": vv, "v_audio": va, "residual": res,
            "x0": x0, "xL": x}


def sample_loop(z_video, z_audio, ends: dict, blocks: list, shape, n_steps: int,
                reuse: int = 1, core_reuse: int = 1, block_ids=None, sig_video=None,
                sig_audio=None) -> dict:
    """A sampler run on the modality latents.  Passes that run the blocks follow
    ``fresh_steps`` of whichever reuse is on; between them whole-velocity reuse
    extrapolates each modality on its own schedule, and core reuse applies the held
    residual with fresh patch projections and heads.  The two reuse modes exclude each
    other (h3.c README)."""
    assert reuse == 1 or core_reuse == 1, "whole-velocity and core reuse exclude each other"
    sv = sigma_schedule(n_steps) if sig_video is None else np.asarray(sig_video, np.float64)
    sa = sv if sig_audio is None else np.asarray(sig_audio, np.float64)
    fresh = set(fresh_steps(n_steps, max(reuse, core_reuse)))
    zv, za = np.asarray(z_video, np.float64), np.asarray(z_audio, np.float64)
    hist, res = [], None
    for i in range(n_steps):
        dv, da = sv[i + 1] - sv[i], sa[i + 1] - sa[i]
        if i in fresh:
            r = sample_step(zv, za, ends, blocks, shape, "fresh", dv, da, block_ids)
            hist.append((i, r["v_video"], r["v_audio"]))
            res = r["residual"]
            zv, za = r["z_video"], r["z_audio"]
        elif core_reuse > 1:
            r = sample_step(zv, za, ends, blocks, shape, "core", dv, da, block_ids, res)
            zv, za = r["z_video"], r["z_audio"]
        else:
            ia, vva, vaa = hist[-1]
            if len(hist) > 1:
                ib, vvb, vab = hist[-2]
                vv = extrapolate(vva, vvb, sv[i], sv[ia], sv[ib])
                va = extrapolate(vaa, vab, sa[i], sa[ia], sa[ib]) if shape.n_audio else vaa
            else:
                vv, va = vva, vaa
            zv = f32(zv + dv * np.asarray(vv, np.float64))
            if shape.n_audio:
                za = f32(za + da * np.asarray(va, np.float64))
    return {"z_video": zv, "z_audio": za, "fresh": sorted(fresh)}


def thin_layers(mods, keep: int) -> list:
    """Block ids kept when thinning to ``keep`` of L blocks.

    h3.c README layer-thinning paragraph: rank the AdaLN gates, protect the
    first and last blocks.  Reading: score_b = ||gate1_b||_2 + ||gate2_b||_2
    (rows 2 and 5 of the table), computed in float64; the smallest scores are
    dropped, ties drop the higher index first.
    """
    mods = [np.asarray(m, np.float64) for m in mods]
    L = len(mods)
    if keep >= L:
        return list(range(L))
    if keep < 2:
        raise ValueError("keep must be >= 2 (first and last blocks are protected)")
    score = {b: float(np.linalg.norm(mods[b][2]) + np.linalg.norm(mods[b][5]))
             for b in range(1, L - 1)}
    order = sorted(score, key=lambda b: (score[b], -b))  # drop order
    dropped = set(order[:L - keep])
    return [b for b in range(L) if b not in dropped]
