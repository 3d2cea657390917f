"""Workload shapes.

The packed sequence holds text rows first, then audio rows, then video rows.
Text and audio rows form the prefix; video rows are cut into tiles of at most 64
rows that the router selects among: contiguous 64-row slices, or, with a video
grid, 4 x 4 x 4 cubes of the latent grid (edge cubes clipped).  Row order here is
raster (t, h, w) for video rows.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class BlockShape:
    n_text: int
    n_audio: int
    n_video: int
    hidden: int
    heads: int
    head_dim: int
    mlp_width: int
    topk: int
    tile: int = 64
    rms_eps: float = 1e-6
    rope_theta: float = 10000.0
    qk_norm: bool = True
    rope: bool = True
    pooled: bool = True
    attn_width_override: int = 0
    mlp: str = "gelu"  # "gelu": fc1 [F, D]; "swiglu": fc1 [2F, D] gate/up interleaved by 128 rows
    prefix_mod: bool = False  # text/audio rows modulated by their own [6, D] table
    # video latent grid (T, H, W) cut into cubes; None = contiguous 64-row tiles
    video_grid: tuple | None = None
    cube: tuple = (4, 4, 4)
    # token reduction: reserve its buffers (the pass chooses the blocks it spans)
    token_reduction: bool = False
    # set on the reduced section's shape: the full width whose column pairs were pooled
    pair_w: int = 0

    @property
    def n_rows(self) -> int:
        return self.n_text + self.n_audio + self.n_video

    @property
    def n_prefix(self) -> int:
        return self.n_text + self.n_audio

    @property
    def attn_width(self) -> int:
        return self.attn_width_override or self.heads * self.head_dim

    @property
    def n_video_tiles(self) -> int:
        if self.video_grid is None:
            return (self.n_video + self.tile - 1) // self.tile
        n = 1
        for g, c in zip(self.video_grid, self.cube):
            n *= (g + c - 1) // c
        return n

    def with_(self, **kw) -> "BlockShape":
        return replace(self, **kw)


@dataclass(frozen=True)
class Workload:
    name: str
    seed_id: int  # seed = 0x48334454 + seed_id
    shape: BlockShape
    description: str
    n_blocks: int = 1
    extra: dict = field(default_factory=dict)

    @property
    def seed(self) -> int:
        return 0x48334454 + self.seed_id


# routed attention alone, 1,024 video rows, 4 heads x 64, top-k 4 of 16.
ATTN_TINY = Workload(
    "attn_tiny_1024", 1,
    BlockShape(0, 0, 1024, hidden=256, heads=4, head_dim=64, mlp_width=1024, topk=4,
               qk_norm=False, rope=False),
    "routed attention only: 1,024 rows, 4 heads x 64, 16 tiles of 64, top-k 4 + pooled",
)

# one block shaped like a 512x512 video: 4,096 rows, D = 3,072, 24 x 128.
BLOCK_4K = Workload(
    "block_4096_d3072", 2,
    BlockShape(256, 256, 3584, hidden=3072, heads=24, head_dim=128, mlp_width=4 * 3072, topk=8),
    "one block: 4,096 rows (256 text, 256 audio, 3,584 video), hidden 3,072, 24 x 128, "
    "MLP 4x GELU, top-k 8 of 56",
)

# one block at the long-sequence shape: 15,435 rows, D = 5,120, 40 x 128.
BLOCK_15K = Workload(
    "block_15435_d5120", 3,
    BlockShape(512, 1024, 13899, hidden=5120, heads=40, head_dim=128, mlp_width=4 * 5120, topk=16),
    "one block: 15,435 rows (512 text, 1,024 audio, 13,899 video), hidden 5,120, 40 x 128, "
    "MLP 4x GELU, top-k 16 of 218 + pooled",
)

# 50 blocks of the 15,435-row shape, then one Euler step dt = -1/8.
FORWARD_50 = Workload(
    "forward50_15435_d5120", 4, BLOCK_15K.shape,
    "50-block denoising forward at 15,435 rows (hidden 5,120 block shape), "
    "then z <- z + dt v with dt = -1/8",
    n_blocks=50, extra={"dt": -0.125, "forward": True},
)

# 20-step denoising loop at 4,096 rows, 45 of 50 blocks, reuse 2.
LOOP_4K = Workload(
    "loop20_4096_d3072", 5, BLOCK_4K.shape,
    "20 Euler steps, 45 of 50 blocks, velocity reuse 2 (11 fresh), top-k sweep {4,8,16,32,56}",
    n_blocks=50, extra={"steps": 20, "reuse": 2, "keep": 45, "topk_sweep": [4, 8, 16, 32, 56]},
)

# The pages' own block shape: hidden 5,376, attention width 7,168 (56 x 128), SwiGLU MLP
# 14,336 wide; 50 such blocks hold 21.2 B parameters (42 GB bf16).
PAGES_SHAPE = BlockShape(512, 1024, 13899, hidden=5376, heads=56, head_dim=128,
                         mlp_width=14336, topk=16, mlp="swiglu", prefix_mod=True)
BLOCK_PAGES = Workload(
    "block_15435_d5376_swiglu", 6, PAGES_SHAPE,
    "one block of the pages' shape: 15,435 rows, hidden 5,376, 56 x 128 heads (attention "
    "width 7,168), SwiGLU MLP 14,336, top-k 16 + pooled",
)
FORWARD_PAGES = Workload(
    "forward50_15435_d5376_swiglu", 7, PAGES_SHAPE,
    "50-block denoising forward of the pages' shape (21.2 B parameters, 42 GB bf16) at "
    "15,435 rows, then z <- z + dt v with dt = -1/8",
    n_blocks=50, extra={"dt": -0.125, "forward": True},
)

# The pages' receipt sequence: 864 x 480, 124 frames -> 15,435 rows (36 text, 414 audio,
# 14,985 video = a 37 x 15 x 27 latent grid), 4 x 4 x 4 cubes -> 280 video tiles beside
# 8 prefix tiles, 56 video tiles kept per query tile, on the pages' block shape.
RECEIPT_SHAPE = PAGES_SHAPE.with_(n_text=36, n_audio=414, n_video=14985, topk=56,
                                  video_grid=(37, 15, 27))
BLOCK_RECEIPT = Workload(
    "block_15435_cubes_d5376_swiglu", 8, RECEIPT_SHAPE,
    "one block of the pages' shape on the receipt sequence: 15,435 rows (36 text, 414 audio, "
    "14,985 video on a 37 x 15 x 27 grid), 280 4x4x4 video tiles, top-k 56 + pooled, 3-D rotary",
)
FORWARD_RECEIPT = Workload(
    "forward50_15435_cubes_d5376_swiglu", 9, RECEIPT_SHAPE,
    "50-block denoising forward of the pages' shape on the receipt sequence (280 cube tiles, "
    "top-k 56), then z <- z + dt v with dt = -1/8",
    n_blocks=50, extra={"dt": -0.125, "forward": True},
)

SAMPLE_RECEIPT = Workload(
    "sample50_15435_cubes_d5376_swiglu", 10, RECEIPT_SHAPE,
    "one fresh sampler step on the modality latents of the receipt sequence: fp32 patch "
    "projections (96 -> 5,376 video, 32 -> 5,376 audio), 50 blocks of the pages' shape, "
    "final AdaLN and output heads with the Euler update, dt = -1/8",
    n_blocks=50, extra={"dt": -0.125, "forward": True, "ends": True, "c_video": 96,
                        "c_audio": 32},
)

SAMPLE_RECEIPT_TR = Workload(
    "sample50_15435_cubes_d5376_swiglu_tokred", 11, RECEIPT_SHAPE.with_(token_reduction=True),
    "the sampler step of the receipt sequence with token reduction: horizontal video token "
    "pairs pooled after block 3 and restored before block 40 (an early, noisy evaluation)",
    n_blocks=50, extra={"dt": -0.125, "forward": True, "ends": True, "c_video": 96,
                        "c_audio": 32, "reduction": (3, 40)},
)

WORKLOADS = [ATTN_TINY, BLOCK_4K, BLOCK_15K, FORWARD_50, LOOP_4K, BLOCK_PAGES, FORWARD_PAGES,
             BLOCK_RECEIPT, FORWARD_RECEIPT, SAMPLE_RECEIPT, SAMPLE_RECEIPT_TR]


def workload_by_name(name: str) -> Workload:
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)
