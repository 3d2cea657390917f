"""Seeded synthetic inputs for the routed-attention DiT block.

This module is the one piece of code that both the CUDA path's harness and the
CPU oracle use.  It draws numbers and packs them into storage formats; it holds
none of the block's arithmetic.

Generator (counter based, so any element can be drawn on its own):

* SplitMix64 finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom
  number generators", OOPSLA 2014): ``mix(z)`` below.
* Stream key: ``key = mix(seed + fnv1a64(name))`` with 64-bit wrap-around,
  where ``name`` labels the tensor ("blk0.w_qkvg", "x", ...).
* Raw draw ``i`` of a stream: ``u64_i = mix(key + (i + 1) * 0x9E3779B97F4A7C15)``.
* Uniform on (0, 1]: ``u = ((u64 >> 11) + 1) * 2**-53``.
* Normal (Box and Muller 1958), element ``2i`` and ``2i + 1`` from the uniform
  pair ``(u_{2i}, u_{2i+1})``: ``r = sqrt(-2 ln u_{2i})``,
  ``z_{2i} = r cos(2 pi u_{2i+1})``, ``z_{2i+1} = r sin(2 pi u_{2i+1})``.

Storage: bf16 tensors are produced as uint16 bit patterns by round-to-nearest-
even of the float32 value; the float64 view of those bits is exact.
"""
from __future__ import annotations

import numpy as np

from .configs import (  # noqa: F401
    ATTN_TINY, BLOCK_4K, BLOCK_15K, BLOCK_PAGES, BLOCK_RECEIPT, FORWARD_50, FORWARD_PAGES,
    FORWARD_RECEIPT, LOOP_4K, SAMPLE_RECEIPT, SAMPLE_RECEIPT_TR, WORKLOADS, BlockShape,
    Workload, workload_by_name)

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
BASE_SEED = 0x48334454  # "H3DT"


def fnv1a64(name: str) -> int:
    h = 0xCBF29CE484222325
    for byte in name.encode("utf-8"):
        h ^= byte
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, name: str) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([(seed + fnv1a64(name)) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return _mix(s)[0]


def raw_u64(seed: int, name: str, start: int, count: int) -> np.ndarray:
    key = stream_key(seed, name)
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
        return _mix(key + i * _GOLDEN)


def uniform(seed: int, name: str, count: int, start: int = 0) -> np.ndarray:
    """Uniform draws on (0, 1], float64."""
    bits = raw_u64(seed, name, start, count)
    return ((bits >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


_CHUNK = 1 << 18  # pairs per chunk: temporaries stay small and are reused


def normal(seed: int, name: str, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """Standard-normal draws (Box-Muller on the uniform stream), float64.

    Drawn in fixed-size chunks of uniform pairs; the values do not depend on
    the chunking (every draw is addressed by its counter).
    """
    n = int(np.prod(shape)) if len(tuple(np.atleast_1d(shape))) else 1
    pairs = (n + 1) // 2
    z = np.empty(2 * pairs, dtype=np.float64)
    for p0 in range(0, pairs, _CHUNK):
        p1 = min(pairs, p0 + _CHUNK)
        u = uniform(seed, name, 2 * (p1 - p0), start=2 * p0)
        r = np.sqrt(-2.0 * np.log(u[0::2]))
        t = 2.0 * np.pi * u[1::2]
        z[2 * p0:2 * p1:2] = r * np.cos(t)
        z[2 * p0 + 1:2 * p1:2] = r * np.sin(t)
    out = z[:n]
    if std != 1.0:
        out *= std
    if mean != 0.0:
        out += mean
    return out.reshape(shape)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float -> bf16 storage bits (uint16), round to nearest even via float32."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32)
    nan = np.isnan(f)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    out = r.astype(np.uint16)
    out[nan] = np.uint16(0x7FC0)
    return out.reshape(np.shape(a))


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact float64 value of bf16 storage bits."""
    u = np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def normal_bf16(seed: int, name: str, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """bf16 bits of ``normal(seed, name, shape, mean, std)``, drawn chunk by chunk."""
    n = int(np.prod(shape)) if len(tuple(np.atleast_1d(shape))) else 1
    out = np.empty(n, dtype=np.uint16)
    step = 2 * _CHUNK
    for e0 in range(0, n, step):
        e1 = min(n, e0 + step)
        # draws e0..e1-1 of the stream: pairs e0/2 .. ceil(e1/2)
        p0, p1 = e0 // 2, (e1 + 1) // 2
        u = uniform(seed, name, 2 * (p1 - p0), start=2 * p0)
        r = np.sqrt(-2.0 * np.log(u[0::2]))
        t = 2.0 * np.pi * u[1::2]
        z = np.empty(2 * (p1 - p0))
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        z = z[:e1 - e0]
        if std != 1.0:
            z *= std
        if mean != 0.0:
            z += mean
        out[e0:e1] = to_bf16_bits(z)
    return out.reshape(shape)


# ---------------------------------------------------------------------------
# Workload builders.  Each returns bf16 tensors as uint16 bit arrays and fp32
# tensors as float32 arrays, with the distributions stated beside them.
# ---------------------------------------------------------------------------

def attention_inputs(shape: BlockShape, seed: int, structured: float = 0.0,
                     with_gate: bool = True) -> dict:
    """Q, K, V bf16 [H, N, d] ~ N(0,1); gate bf16 [N, H*d] ~ N(0,1).

    ``structured`` > 0 adds a per-(head, video block) offset vector ~ N(0, s^2)
    to every row of that block in Q and K (blocks: 64-row slices, or cubes of the
    latent grid with the video rows in raster order), so that tile means separate
    and routing is decisive; 0 gives the flat i.i.d. regime.
    """
    H, N, d = shape.heads, shape.n_rows, shape.head_dim
    q = normal(seed, "q", (H, N, d))
    k = normal(seed, "k", (H, N, d))
    v = normal(seed, "v", (H, N, d))
    if structured > 0.0:
        P, tile = shape.n_prefix, shape.tile
        rows = np.arange(shape.n_video)
        if shape.video_grid is None:
            t_of = rows // tile  # one offset per 64-row slice
        else:  # one offset per block of the latent grid, rows in raster (t, h, w) order
            T, Hg, Wg = shape.video_grid
            ct, ch, cw = shape.cube
            nh, nw = -(-Hg // ch), -(-Wg // cw)
            t_of = ((rows // (Hg * Wg)) // ct * nh + (rows // Wg % Hg) // ch) * nw \
                + (rows % Wg) // cw
        tv = int(t_of.max()) + 1
        cq = normal(seed, "q.tile_offset", (H, tv, d), std=structured)
        ck = normal(seed, "k.tile_offset", (H, tv, d), std=structured)
        q[:, P:, :] += cq[:, t_of, :]
        k[:, P:, :] += ck[:, t_of, :]
    out = {"q": to_bf16_bits(q), "k": to_bf16_bits(k), "v": to_bf16_bits(v)}
    if with_gate:
        out["gate"] = normal_bf16(seed, "gate", (N, H * d))
    return out


def block_weights(shape: BlockShape, seed: int, block: int = 0) -> dict:
    """One block's synthetic parameters.

    Linear weights are stored [out, in] (row-major, the input dimension
    contiguous).  With a SwiGLU MLP, fc1 holds 2F rows: the gate and up rows of
    each group of 128 outputs, one after the other.  Weights and biases bf16
    ~ N(0, 0.02); modulation table fp32 [6, D] ~ N(0, 0.1^2) in the order shift1,
    scale1, gate1, shift2, scale2, gate2; with ``prefix_mod`` the text and audio
    rows get their own table "mod_prefix" of the same kind; q/k norm weights bf16
    = 1 + N(0, 0.02).
    """
    D, A, F = shape.hidden, shape.attn_width, shape.mlp_width
    F1 = 2 * F if shape.mlp == "swiglu" else F  # fc1 rows: gate/up interleaved by 128
    p = f"blk{block}."
    out = {
        "w_qkvg": normal_bf16(seed, p + "w_qkvg", (4 * A, D), std=0.02),
        "b_qkvg": normal_bf16(seed, p + "b_qkvg", (4 * A,), std=0.02),
        "w_o": normal_bf16(seed, p + "w_o", (D, A), std=0.02),
        "b_o": normal_bf16(seed, p + "b_o", (D,), std=0.02),
        "w1": normal_bf16(seed, p + "w1", (F1, D), std=0.02),
        "b1": normal_bf16(seed, p + "b1", (F1,), std=0.02),
        "w2": normal_bf16(seed, p + "w2", (D, F), std=0.02),
        "b2": normal_bf16(seed, p + "b2", (D,), std=0.02),
        "mod": normal(seed, p + "mod", (6, D), std=0.1).astype(np.float32),
        "qnorm_w": normal_bf16(seed, p + "qnorm_w", (shape.head_dim,), mean=1.0, std=0.02),
        "knorm_w": normal_bf16(seed, p + "knorm_w", (shape.head_dim,), mean=1.0, std=0.02),
    }
    if shape.prefix_mod:  # the text/audio rows' own modulation table, same distribution
        out["mod_prefix"] = normal(seed, p + "mod_prefix", (6, D), std=0.1).astype(np.float32)
    return out


def hidden_rows(shape: BlockShape, seed: int) -> np.ndarray:
    """Block input x, bf16 [N, D] ~ N(0, 1)."""
    return normal_bf16(seed, "x", (shape.n_rows, shape.hidden))


def latents(shape: BlockShape, seed: int) -> np.ndarray:
    """Denoiser latents z, fp32 [N, D] ~ N(0, 1)."""
    return normal(seed, "z", (shape.n_rows, shape.hidden)).astype(np.float32)


def ends_weights(shape: BlockShape, seed: int, c_video: int = 96, c_audio: int = 32) -> dict:
    """Both ends of the denoiser for ``shape``: patch projections (fp32, input-major
    [c, D], weights ~ N(0, 0.1^2), biases ~ N(0, 0.02^2)), final AdaLN tables (fp32
    [2, D] ~ N(0, 0.1^2): shift, scale), output heads (bf16 [c, D] and [c], ~ N(0, 0.02^2))
    and the text rows (bf16 [n_text, D] ~ N(0, 1)).  96 and 32 are the pages' video and
    audio latent widths."""
    D = shape.hidden
    out = {"c_video": c_video, "c_audio": c_audio}
    for m, c in (("video", c_video), ("audio", c_audio)):
        out[f"w_in_{m}"] = normal(seed, f"ends.w_in_{m}", (c, D), std=0.1).astype(np.float32)
        out[f"b_in_{m}"] = normal(seed, f"ends.b_in_{m}", (D,), std=0.02).astype(np.float32)
        out[f"w_out_{m}"] = normal_bf16(seed, f"ends.w_out_{m}", (c, D), std=0.02)
        out[f"b_out_{m}"] = normal_bf16(seed, f"ends.b_out_{m}", (c,), std=0.02)
        out[f"mod_out_{m}"] = normal(seed, f"ends.mod_out_{m}", (2, D), std=0.1).astype(np.float32)
    out["text"] = normal_bf16(seed, "ends.text", (shape.n_text, D))
    return out


def modality_latents(shape: BlockShape, seed: int, c_video: int = 96, c_audio: int = 32):
    """Latents of the two modalities, fp32 ~ N(0, 1): video [n_video, c_video] (raster
    row order), audio [n_audio, c_audio]."""
    zv = normal(seed, "z.video", (shape.n_video, c_video)).astype(np.float32)
    za = normal(seed, "z.audio", (shape.n_audio, c_audio)).astype(np.float32)
    return zv, za
