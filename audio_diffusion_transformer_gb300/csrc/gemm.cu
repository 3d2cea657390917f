// gemm.cu -- bf16 projection GEMM on tcgen05 tensor cores with fused epilogues.
//
// y[M, N] = a[M, K] * w[N, K]^T with fp32 accumulation in TMEM (TensorFold
// #949 "Precision": bf16 weights and activations, fp32 sums).  The 256-wide projections
// of the block (and h3dit_linear) run on SM pairs: 256 x 256 tiles on clusters of two
// CTAs with cta_group::2 MMAs (the CTA-pair kernel below, with every epilogue); where a
// device cannot host such clusters, and for the narrow output heads, one SM per tile.
// One-SM kernel: one persistent CTA per SM walks the output tiles in a grouped order
// (8 or 16 row-blocks per group, so a wave of tiles shares A and B panels in L2).  Two
// tilings:
//   128 x 256 tiles (every epilogue of the block: GELU, SwiGLU, q/k norm + rotary,
//   gated residual; the output heads):
//     warp 0      TMA producer: 64-wide K slices of A (128 rows) and W (256 rows)
//                 into a 4-stage shared-memory ring (128-byte swizzle)
//     warp 1      tcgen05.mma issuer (one thread), M=128 N=256 K=16 per op, into
//                 one of two 256-column TMEM accumulators, so the epilogue of tile i
//                 overlaps the K loop of tile i+1
//     warps 2..5  epilogue: TMEM -> registers (warp w reads lanes 32*(w%4)..)
//   256 x 256 tiles ("pair" tiles: plain stores, h3dit_linear): two M=128 MMAs per K
//   step share the W slice, so each stage's 64 KB (3 stages) feeds twice the tensor
//   work of a 128-row stage; the two 256-column accumulators fill TMEM, so the epilogue
//   (warps 2..9, one half each) runs between tiles while the producer prefills the ring.
//   The first bands of 256 rows are pair tiles and the remaining rows 128 x 256 tiles on
//   the same accumulator, in a number that balances the last wave across the SMs.  An
//   epilogue that reads memory (the gated residual) stays on the double accumulator:
//   between pair tiles it cannot hide behind the next K loop.
// No split-K and no atomics: results are deterministic.
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace h3 {

namespace {

#ifndef H3_GEMM_STAGES
#define H3_GEMM_STAGES 4  // 128 x 256 tiles: a 4-stage ring of 48 KB stages
#endif

constexpr int BM = 128, BK = 64;
constexpr int BN_WIDE = 256;  // output tile width of the projections

// Per tile width BN and tiling: shared-memory ring, threads and TMEM accumulators.
template <int BN, bool PAIR>
struct Tile {
  static constexpr int A_ROWS = PAIR ? 2 * BM : BM;  // A rows per stage
  static constexpr int A_BYTES = A_ROWS * BK * 2;    // 16 KB, or 32 KB for pair tiles
  static constexpr int B_BYTES = BN * BK * 2;        // 32 KB at BN = 256
  static constexpr int STAGES = PAIR ? 3 : H3_GEMM_STAGES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
  static constexpr int EPI_WARPS = PAIR ? 8 : 4;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int NACC = PAIR ? 1 : 2;  // accumulators (a pair tile's two halves fill TMEM)
  static constexpr uint32_t TMEM_COLS =
      PAIR ? 512 : (2 * BN <= 64 ? 64 : (2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512)));
  // accumulator b (or, for pair tiles, row half b) starts at column b * ACC_STRIDE
  static constexpr uint32_t ACC_STRIDE = PAIR ? 256 : TMEM_COLS / 2;
};

struct Params {
  int M, N, K;
  int group;  // row-blocks per raster group
  int pairs;  // pair tiling: bands of 256 rows taken as pair tiles (rows beyond: 128-row tiles)
  const __nv_bfloat16* bias;
  __nv_bfloat16* y;
  const float* gate;
  const float* gate_prefix;  // rows < n_prefix use this gate when set
  int n_prefix;
  int heads, head_dim, attn_width;
  __nv_bfloat16 *q, *k, *v, *g;
  const __nv_bfloat16 *qnorm_w, *knorm_w;
  const float2* rope_cs;
  float eps;
  float* v_out;  // head epilogue: fp32 velocity [M, N] or null
  float* z;      // head epilogue: fp32 latents [M, N], z += dt * v
  float dt;
  int* status;
  int* tile_counter;  // CTA-pair kernel: [0] tiles fetched, [1] clusters done; or null
};

__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int group,
                                            int& m_blk, int& n_blk) {
  const int g = tile / (group * num_n);
  const int first = g * group;
  const int gm = min(num_m - first, group);
  const int in_group = tile - g * group * num_n;
  m_blk = first + in_group % gm;
  n_blk = in_group / gm;
}

__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* p, float* out) {
  const uint4* v = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u = __ldg(v + i);
    out[8 * i + 0] = bf16_lo(u.x);
    out[8 * i + 1] = bf16_hi(u.x);
    out[8 * i + 2] = bf16_lo(u.y);
    out[8 * i + 3] = bf16_hi(u.y);
    out[8 * i + 4] = bf16_lo(u.z);
    out[8 * i + 5] = bf16_hi(u.z);
    out[8 * i + 6] = bf16_lo(u.w);
    out[8 * i + 7] = bf16_hi(u.w);
  }
}

// Plain (not read-only-cache) load, for data this kernel may also write.
__device__ __forceinline__ void load_bf16x32_rw(const __nv_bfloat16* p, float* out) {
  const uint4* v = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u = v[i];
    out[8 * i + 0] = bf16_lo(u.x);
    out[8 * i + 1] = bf16_hi(u.x);
    out[8 * i + 2] = bf16_lo(u.y);
    out[8 * i + 3] = bf16_hi(u.y);
    out[8 * i + 4] = bf16_lo(u.z);
    out[8 * i + 5] = bf16_hi(u.z);
    out[8 * i + 6] = bf16_lo(u.w);
    out[8 * i + 7] = bf16_hi(u.w);
  }
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* p, const float* v) {
  uint4* d = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
    u.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
    u.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
    u.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
    d[i] = u;
  }
}

// Tile t of the pair tiling: first pairs x num_n tiles of 256 rows, then 128-row tiles for
// the rest; each region in grouped raster order.  two = true for a 256-row tile.
__device__ __forceinline__ void pair_tile(const Params& p, int tile, int num_n, int& m0,
                                          bool& two, int& n_blk) {
  const int big = p.pairs * num_n;
  int mb;
  if (tile < big) {
    tile_coords(tile, p.pairs, num_n, p.group > 1 ? p.group / 2 : 1, mb, n_blk);
    m0 = mb * 2 * BM;
    two = true;
  } else {
    const int rest = (p.M + BM - 1) / BM - 2 * p.pairs;
    tile_coords(tile - big, rest, num_n, p.group, mb, n_blk);
    m0 = (2 * p.pairs + mb) * BM;
    two = false;
  }
}

// GELU, 0.5 x (1 + erf(x / sqrt 2)), with erf from Abramowitz & Stegun, Handbook of
// Mathematical Functions, formula 7.1.26: for z >= 0,
// erfc(z) = t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2) + e, t = 1 / (1 + p z),
// |e| <= 1.5e-7 (far below the bf16 spacing of the stored activations).  1 + erf(x / sqrt 2)
// = 2 - erfc(z) for x >= 0 and erfc(z) for x < 0 (z = |x| / sqrt 2), which avoids
// cancellation for negative x.  About 2.5% faster per fc1 launch than erff.
__device__ __forceinline__ float gelu_erf(float x) {
  const float z = fabsf(x) * 0.70710678118654752f;
  float t;  // 1 / (1 + p z), approximate reciprocal (relative error ~2^-23)
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(fmaf(0.3275911f, z, 1.0f)));
  float q = fmaf(t, 1.061405429f, -1.453152027f);
  q = fmaf(t, q, 1.421413741f);
  q = fmaf(t, q, -0.284496736f);
  q = fmaf(t, q, 0.254829592f);
  const float erfc_z = t * q * ex2_approx(-z * z * 1.4426950408889634f);
  const float one_plus_erf = x >= 0.0f ? 2.0f - erfc_z : erfc_z;
  return 0.5f * x * one_plus_erf;
}

// Epilogue of an output head: v = acc + b (fp32); v -> the velocity ring, z += dt * v.
template <int BN>
__device__ __forceinline__ void epilogue_head(const Params& p, uint32_t t_row, int row, int n0) {
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    float v[32];
    tmem_ld32(t_row + c * 32, v);
    if (row < p.M) {
      const int col0 = n0 + c * 32;
      float b[32];
      load_bf16x32(p.bias + col0, b);
      const size_t off = (size_t)row * p.N + col0;
      float4* z4 = reinterpret_cast<float4*>(p.z + off);
      float4* v4 = p.v_out ? reinterpret_cast<float4*>(p.v_out + off) : nullptr;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 vv = make_float4(v[4 * j] + b[4 * j], v[4 * j + 1] + b[4 * j + 1],
                                      v[4 * j + 2] + b[4 * j + 2], v[4 * j + 3] + b[4 * j + 3]);
        float4 zz = z4[j];
        zz.x = fmaf(p.dt, vv.x, zz.x);
        zz.y = fmaf(p.dt, vv.y, zz.y);
        zz.z = fmaf(p.dt, vv.z, zz.z);
        zz.w = fmaf(p.dt, vv.w, zz.w);
        z4[j] = zz;
        if (v4) v4[j] = vv;
      }
    }
  }
}

// Epilogue of a plain / GELU / residual tile: BN / 32 chunks of 32 columns.
template <int EPI, int BN>
__device__ __forceinline__ void epilogue_rows(const Params& p, uint32_t t_row, int row, int n0) {
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    float v[32];
    tmem_ld32(t_row + c * 32, v);
    if (row < p.M) {
      const int col0 = n0 + c * 32;
      if (p.bias) {
        float b[32];
        load_bf16x32(p.bias + col0, b);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += b[j];
      }
      __nv_bfloat16* dst = p.y + (size_t)row * p.N + col0;
      if (EPI == kEpiGelu) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = gelu_erf(v[j]);
      } else if (EPI == kEpiResid) {
        float r[32];
        load_bf16x32_rw(dst, r);
        const float* gsel = (p.gate_prefix != nullptr && row < p.n_prefix) ? p.gate_prefix : p.gate;
        const float4* g4 = reinterpret_cast<const float4*>(gsel + col0);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 g = __ldg(g4 + j);
          v[4 * j + 0] = fmaf(g.x, v[4 * j + 0], r[4 * j + 0]);
          v[4 * j + 1] = fmaf(g.y, v[4 * j + 1], r[4 * j + 1]);
          v[4 * j + 2] = fmaf(g.z, v[4 * j + 2], r[4 * j + 2]);
          v[4 * j + 3] = fmaf(g.w, v[4 * j + 3], r[4 * j + 3]);
        }
      }
      store_bf16x32(dst, v);
    }
  }
}

__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }

// Epilogue of the SwiGLU fc1: tile columns 0..127 are gate, 128..255 up, for the 128
// activated outputs 128 * (n0 / 256) ..; y has N / 2 columns.
// Chunks [c0, c1) of the tile's four 32-output chunks.
__device__ __forceinline__ void epilogue_swiglu(const Params& p, uint32_t t_row, int row, int n0,
                                                int c0 = 0, int c1 = 4) {
  const int F = p.N / 2;
  const int out0 = n0 / 2;
#pragma unroll 1
  for (int c = c0; c < c1; ++c) {
    float g[32], u[32];
    tmem_ld32(t_row + c * 32, g);
    tmem_ld32(t_row + 128 + c * 32, u);
    if (row < p.M) {
      float bg[32], bu[32];
      load_bf16x32(p.bias + n0 + c * 32, bg);
      load_bf16x32(p.bias + n0 + 128 + c * 32, bu);
#pragma unroll
      for (int j = 0; j < 32; ++j) g[j] = silu(g[j] + bg[j]) * (u[j] + bu[j]);
      store_bf16x32(p.y + (size_t)row * F + out0 + c * 32, g);
    }
  }
}

// Epilogue of the fused q/k/v/gate projection: one head (HD columns) at a time.
template <int HD, int BN>
__device__ __forceinline__ void epilogue_qkvg(const Params& p, uint32_t t_row, int row, int n0) {
  const int A = p.attn_width;
  const int slab = n0 / A;  // 0 q, 1 k, 2 v, 3 g  (A is a multiple of BN)
  const int col_in_slab = n0 - slab * A;
#pragma unroll 1
  for (int hh = 0; hh < BN / HD; ++hh) {
    float v[HD];
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) tmem_ld32(t_row + hh * HD + c * 32, v + c * 32);
    if (row >= p.M) continue;
    const int head = (col_in_slab + hh * HD) / HD;
    const int col0 = n0 + hh * HD;
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
      float b[32];
      load_bf16x32(p.bias + col0 + c * 32, b);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[c * 32 + j] = bf16_round(v[c * 32 + j] + b[j]);
    }
    if (slab <= 1) {
      const __nv_bfloat16* nw = slab == 0 ? p.qnorm_w : p.knorm_w;
      if (nw) {
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < HD; ++j) ss = fmaf(v[j], v[j], ss);
        const float inv = 1.0f / sqrtf(ss / (float)HD + p.eps);
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          float w[32];
          load_bf16x32(nw + c * 32, w);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[c * 32 + j] = v[c * 32 + j] * inv * w[j];
        }
      }
      if (p.rope_cs) {
        const float4* cs = reinterpret_cast<const float4*>(p.rope_cs + (size_t)row * (HD / 2));
#pragma unroll
        for (int j = 0; j < HD / 4; ++j) {
          const float4 t = __ldg(cs + j);  // (cos, sin) of pairs 2j and 2j+1
          const float x0 = v[2 * j], y0 = v[2 * j + HD / 2];
          const float x1 = v[2 * j + 1], y1 = v[2 * j + 1 + HD / 2];
          v[2 * j] = x0 * t.x - y0 * t.y;
          v[2 * j + HD / 2] = y0 * t.x + x0 * t.y;
          v[2 * j + 1] = x1 * t.z - y1 * t.w;
          v[2 * j + 1 + HD / 2] = y1 * t.z + x1 * t.w;
        }
      }
    }
    __nv_bfloat16* dst;
    if (slab == 3) {
      dst = p.g + (size_t)row * A + head * HD;
    } else {
      __nv_bfloat16* base = slab == 0 ? p.q : (slab == 1 ? p.k : p.v);
      dst = base + ((size_t)head * p.M + row) * HD;
    }
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) store_bf16x32(dst + c * 32, v + c * 32);
  }
}

template <int EPI, int HD, int BN, bool PAIR>
__global__ void __launch_bounds__(Tile<BN, PAIR>::THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA1,
                const __grid_constant__ CUtensorMap tmB, const Params p) {
  // tmA: A with boxes of A_ROWS rows; tmA1 (pair tiling): boxes of 128 rows
  using T = Tile<BN, PAIR>;
  constexpr int A_BYTES = T::A_BYTES;
  constexpr int B_BYTES = T::B_BYTES;
  constexpr int STAGES = T::STAGES;
  constexpr int STAGE_BYTES = T::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_m = (p.M + BM - 1) / BM;
  const int num_n = p.N / BN;
  const int num_tiles = PAIR ? (num_m - p.pairs) * num_n : num_m * num_n;
  const int num_k = p.K / BK;
  // tile -> first row, whether it is a 256-row pair tile, column block
  auto coords = [&](int tile, int& m0, bool& two, int& n_blk) {
    if constexpr (PAIR) {
      pair_tile(p, tile, num_n, m0, two, n_blk);
    } else {
      int m_blk;
      tile_coords(tile, num_m, num_n, p.group, m_blk, n_blk);
      m0 = m_blk * BM;
      two = false;
    }
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], T::EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, T::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    if (PAIR) prefetch_tmap(&tmA1);
    prefetch_tmap(&tmB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        int m0, n_blk;
        bool two;
        coords(tile, m0, two, n_blk);
        // a 128-row tile of the pair tiling loads half an A stage
        const uint32_t bytes = (PAIR && !two) ? STAGE_BYTES - A_BYTES / 2 : STAGE_BYTES;
        for (int kb = 0; kb < num_k; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], bytes);
          tma_load_2d(sA + stage * A_BYTES, (PAIR && !two) ? &tmA1 : &tmA, &full[stage], kb * BK,
                      m0);
          tma_load_2d(sB + stage * B_BYTES, &tmB, &full[stage], kb * BK, n_blk * BN);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BM, BN, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        int m0, n_blk;
        bool two;
        coords(tile, m0, two, n_blk);
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * T::ACC_STRIDE;
        for (int kb = 0; kb < num_k; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t bd = sdesc_sw128(b0 + k * 32, 16, 1024);
            const uint32_t accum = (kb | k) != 0 ? 1u : 0u;
            umma_bf16(d_tmem, sdesc_sw128(a0 + k * 32, 16, 1024), bd, idesc, accum);
            // rows 128..255 of a pair tile (16 KB into the stage) into the second half
            if (PAIR && two)
              umma_bf16(d_tmem + T::ACC_STRIDE, sdesc_sw128(a0 + BM * 128 + k * 32, 16, 1024), bd,
                        idesc, accum);
          }
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&acc_full[acc]);
        if (++acc == T::NACC) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // every MMA this thread issued has completed before TMEM is released
      umma_commit(drain);
      mbar_drain(drain, 0);
    }
  } else {
    const int quad = warp & 3;
    const int half = PAIR ? (warp - 2) / 4 : 0;  // pair tiling: warps 6..9 take rows 128..255
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      int m0, n_blk;
      bool two;
      coords(tile, m0, two, n_blk);
      if (!mbar_wait(&acc_full[acc], acc_phase, abort_flag, p.status)) break;
      tc_fence_after();
      if (half == 0 || two) {
        const int row = m0 + half * BM + quad * 32 + lane;
        const uint32_t t_row =
            tmem + ((uint32_t)(quad * 32) << 16) + (acc + half) * T::ACC_STRIDE;
        if (EPI == kEpiQkvg)
          epilogue_qkvg<HD, BN>(p, t_row, row, n_blk * BN);
        else if (EPI == kEpiSwiglu)
          epilogue_swiglu(p, t_row, row, n_blk * BN);
        else if (EPI == kEpiHeadEuler)
          epilogue_head<BN>(p, t_row, row, n_blk * BN);
        else
          epilogue_rows<EPI, BN>(p, t_row, row, n_blk * BN);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      if (++acc == T::NACC) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, T::TMEM_COLS);
  }
}

template <int EPI, int HD, int BN = BN_WIDE, bool PAIR = false>
cudaError_t launch_one(const GemmArgs& g, const CUtensorMap& tb, Params p, cudaStream_t stream) {
  using T = Tile<BN, PAIR>;
  CUtensorMap ta, ta1;
  if (!make_tmap_2d(&ta, g.a, g.M, g.K, T::A_ROWS)) return cudaErrorInvalidValue;
  ta1 = ta;
  if (PAIR && !make_tmap_2d(&ta1, g.a, g.M, g.K, BM)) return cudaErrorInvalidValue;
  auto kern = gemm_kernel<EPI, HD, BN, PAIR>;
  constexpr int smem = T::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int sms = num_sms();
  const int num_m = (p.M + BM - 1) / BM, num_n = p.N / BN;
  p.pairs = 0;
  if (PAIR) {
    // as many bands of 256 rows as fill whole waves while leaving about two 128-row tiles
    // per SM for the last wave, which the round-robin then balances to within one tile
    const double per_sm = (double)num_m * num_n / sms;
    const int big = per_sm > 1.0 ? sms * (int)((per_sm - 1.0) / 2.0) : 0;
    p.pairs = big / num_n < num_m / 2 ? big / num_n : num_m / 2;
  }
  const int tiles = (num_m - p.pairs) * num_n;
  const int grid = tiles < sms ? tiles : sms;
  kern<<<grid, T::THREADS, smem, stream>>>(ta, ta1, tb, p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ CTA-pair kernel
// 256 x 256 output tiles on a cluster of two CTAs (two SMs) with cta_group::2 MMAs: each
// CTA loads its own 128 rows of A and its own 128 rows of the W tile (no multicast), and
// rank 0's MMA thread issues M = 256, N = 256, K = 16 MMAs that read both CTAs' shared
// memory and write 128 x 256 fp32 accumulators into each CTA's TMEM.  Per SM and K step
// that is 32 KB of operands written and read through shared memory for 1,024 MMA cycles
// of tensor work, against 48 KB per 512 cycles for the one-SM 128 x 256 tile, and each
// CTA keeps two 256-column accumulators, so the epilogue of one tile overlaps the K loop
// of the next.
//   warp 0      TMA producer (both CTAs): A rows and W rows of this CTA's half into a
//               6-stage ring; the bytes of both halves are counted on rank 0's barrier.
//               Rank 0's producer also decides the cluster's next tile and publishes it
//               in a 4-slot queue in both CTAs' shared memory, read by every role.
//   warp 1      rank 0: the MMA issuer; both ranks: TMEM allocation for the pair
//   warps 2..5  epilogue (both CTAs): this CTA's 128 rows; accumulator release counted
//               on rank 0's barrier (eight warps)
// Tiles: cluster c starts with tile c; with a tile counter, a cluster that finishes takes
// the next unstarted tile from it (atomicAdd), so the tiles in flight stay a window of
// consecutive numbers in the grouped raster order and share their A and W panels in L2
// (clusters dealt tiles round-robin drift apart over a launch: the 20,480-deep fc2 at
// 15,435 rows read 4.4-6.7 GB from DRAM that way, 3.6 GB with tiles taken in order).
// The last cluster to finish resets the counter for the next launch.
constexpr int P_STAGES = 6;
constexpr int P_TQ = 4;  // tile queue slots
constexpr int P_A_BYTES = BM * BK * 2;           // 16 KB: this CTA's 128 rows of A
constexpr int P_B_BYTES = (BN_WIDE / 2) * BK * 2;  // 16 KB: this CTA's 128 rows of W
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
constexpr int P_SMEM_BYTES = P_STAGES * P_STAGE_BYTES + 1024 + 256;
// Epilogue warps EW: 4 (one per SM sub-partition) or 8 (two, each taking half of the
// tile's columns).  Eight pay where the K loop is short (K <= 4,096: the 4,096-row block's
// fc1 took 16% less time with them) and cost 2-3% where it is long (K = 5,120 and 20,480 at
// 15,435 rows); the q/k/v/gate epilogue's per-head registers allow only four.
__host__ __device__ constexpr int pair_threads(int ew) { return 64 + 32 * ew; }
constexpr uint32_t P_TMEM_COLS = 512;  // two 256-column accumulators per CTA

template <int EPI, int HD, int EW>
__global__ void __launch_bounds__(pair_threads(EW), 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + P_STAGES * P_A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P_STAGES * P_STAGE_BYTES);
  uint64_t* full = bars;                  // [P_STAGES] rank 0: both halves landed
  uint64_t* empty = bars + P_STAGES;      // [P_STAGES] the stage's MMAs completed
  uint64_t* acc_full = bars + 2 * P_STAGES;  // [2] accumulator ready (both CTAs)
  uint64_t* acc_empty = acc_full + 2;     // [2] rank 0: both CTAs' epilogues read it
  uint64_t* drain = acc_empty + 2;        // rank 0: every MMA completed
  uint64_t* tq_full = drain + 1;          // [P_TQ] tile number published (each CTA)
  uint64_t* tq_empty = tq_full + P_TQ;    // [P_TQ] rank 0: every reader has taken it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tq_empty + P_TQ);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* tq = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [P_TQ] tile numbers

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int cluster = blockIdx.x >> 1;
  const int n_clusters = gridDim.x >> 1;
  const int num_m = (p.M + 2 * BM - 1) / (2 * BM);  // 256-row tiles
  const int num_n = p.N / BN_WIDE;
  const int num_tiles = num_m * num_n;
  const int num_k = p.K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 2 * EW);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < P_TQ; ++i) {
      mbar_init(&tq_full[i], 1);
      // readers: rank 1's producer, the MMA issuer, the epilogue warps of both CTAs
      mbar_init(&tq_empty[i], 2 + 2 * EW);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  // Reads the next tile number from the queue (every reader but rank 0's producer) and
  // releases the slot on rank 0; num_tiles marks the end, -1 an abort.
  const uint32_t tq_empty0 = rank == 0 ? smem_u32(tq_empty) : mapa_shared(smem_u32(tq_empty), 0);
  auto take_tile = [&](int& slot, uint32_t& ph, bool whole_warp) -> int {
    if (!mbar_wait<true>(&tq_full[slot], ph, abort_flag, p.status)) return -1;
    const int t = tq[slot];
    if (whole_warp) __syncwarp();
    if (!whole_warp || lane == 0) {
      if (rank == 0)
        mbar_arrive(&tq_empty[slot]);
      else
        mbar_arrive_cluster(tq_empty0 + slot * 8);
    }
    if (++slot == P_TQ) {
      slot = 0;
      ph ^= 1;
    }
    return t;
  };
  // both CTAs are running and their barriers initialised before any remote access
  cluster_sync();
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, P_TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the pair's TMEM is allocated in both CTAs before rank 0 issues MMAs
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // completion of both CTAs' loads is counted on rank 0's full barriers
      const uint32_t full0 = rank == 0 ? smem_u32(full) : mapa_shared(smem_u32(full), 0);
      const uint32_t tq1 = rank == 0 ? mapa_shared(smem_u32((const void*)tq), 1) : 0u;
      const uint32_t tq_full1 = rank == 0 ? mapa_shared(smem_u32(tq_full), 1) : 0u;
      int stage = 0;
      uint32_t phase = 0;
      int slot = 0;
      uint32_t qph = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        int tile;
        if (rank == 0) {
          // the slot of the tile P_TQ back has been read by everyone
          if (!mbar_wait<true>(&tq_empty[slot], qph ^ 1, abort_flag, p.status)) break;
          if (i == 0)
            tile = cluster;
          else if (p.tile_counter != nullptr)
            tile = n_clusters + atomicAdd(p.tile_counter, 1);
          else
            tile = cluster + i * n_clusters;
          tile = min(tile, num_tiles);
          tq[slot] = tile;
          st_cluster_u32(tq1 + slot * 4, (uint32_t)tile);
          mbar_arrive(&tq_full[slot]);
          mbar_arrive_cluster(tq_full1 + slot * 8);  // orders the store above before it
          if (++slot == P_TQ) {
            slot = 0;
            qph ^= 1;
          }
        } else {
          tile = take_tile(slot, qph, false);
        }
        if (tile < 0 || tile >= num_tiles) break;
        int m_blk, n_blk;
        tile_coords(tile, num_m, num_n, p.group, m_blk, n_blk);
        const int arow = m_blk * 2 * BM + (int)rank * BM;
        const int brow = n_blk * BN_WIDE + (int)rank * (BN_WIDE / 2);
        for (int kb = 0; kb < num_k; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * P_STAGE_BYTES);
          const uint32_t fb = full0 + stage * 8;
          tma_load_2d_pair(sA + stage * P_A_BYTES, &tmA, fb, kb * BK, arow);
          tma_load_2d_pair(sB + stage * P_B_BYTES, &tmB, fb, kb * BK, brow);
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (rank == 0 && p.tile_counter != nullptr) {
        // this cluster takes no more tiles; the last one to finish resets the counters
        __threadfence();
        if (atomicAdd(p.tile_counter + 1, 1) == n_clusters - 1) {
          __threadfence();
          atomicExch(p.tile_counter, 0);
          atomicExch(p.tile_counter + 1, 0);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16(2 * BM, BN_WIDE, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int slot = 0;
      uint32_t qph = 0;
      bool ok = true;
      while (ok) {
        const int tile = take_tile(slot, qph, false);
        if (tile < 0 || tile >= num_tiles) break;
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * 256;
        for (int kb = 0; kb < num_k; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * P_A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * P_B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16_pair(d_tmem, sdesc_sw128(a0 + k * 32, 16, 1024),
                           sdesc_sw128(b0 + k * 32, 16, 1024), idesc, (kb | k) != 0 ? 1u : 0u);
          umma_commit_pair(&empty[stage], 0x3);
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit_pair(&acc_full[acc], 0x3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // every MMA this thread issued has completed before either CTA releases TMEM
      umma_commit_pair(drain, 0x1);
      mbar_drain(drain, 0);
    }
  } else {
    const int quad = warp & 3;
    const int half = EW == 8 ? (warp - 2) >> 2 : 0;  // eight warps: the tile's column half
    const uint32_t rel0 = smem_u32(acc_empty);
    const uint32_t rel0_remote = rank == 0 ? 0u : mapa_shared(rel0, 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    int slot = 0;
    uint32_t qph = 0;
    while (true) {
      const int tile = take_tile(slot, qph, true);
      if (tile < 0 || tile >= num_tiles) break;
      int m_blk, n_blk;
      tile_coords(tile, num_m, num_n, p.group, m_blk, n_blk);
      if (!mbar_wait(&acc_full[acc], acc_phase, abort_flag, p.status)) break;
      tc_fence_after();
      const int row = m_blk * 2 * BM + (int)rank * BM + quad * 32 + lane;
      const uint32_t t_row = tmem + ((uint32_t)(quad * 32) << 16) + acc * 256;
      if (EPI == kEpiQkvg)
        epilogue_qkvg<HD, BN_WIDE>(p, t_row, row, n_blk * BN_WIDE);
      else if (EPI == kEpiSwiglu && EW == 8)
        epilogue_swiglu(p, t_row, row, n_blk * BN_WIDE, 2 * half, 2 * half + 2);
      else if (EPI == kEpiSwiglu)
        epilogue_swiglu(p, t_row, row, n_blk * BN_WIDE);
      else if (EW == 8)
        epilogue_rows<EPI, BN_WIDE / 2>(p, t_row + half * (BN_WIDE / 2), row,
                                        n_blk * BN_WIDE + half * (BN_WIDE / 2));
      else
        epilogue_rows<EPI, BN_WIDE>(p, t_row, row, n_blk * BN_WIDE);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(&acc_empty[acc]);
        else
          mbar_arrive_cluster(rel0_remote + acc * 8);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // rank 0's MMAs have drained and both epilogues are done with TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, P_TMEM_COLS);
  }
}

// Clusters of two that can be resident at once for this kernel (0: none / unsupported).
template <int EPI, int HD, int EW>
int pair_capacity() {
  static int cap = -1;
  if (cap >= 0) return cap;
  auto kern = gemm_pair_kernel<EPI, HD, EW>;
  cap = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM_BYTES) !=
      cudaSuccess)
    return cap;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
  cfg.blockDim = dim3(pair_threads(EW), 1, 1);
  cfg.dynamicSmemBytes = P_SMEM_BYTES;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) cap = n;
  cudaGetLastError();  // a refused query leaves no sticky error behind
  return cap;
}

// Launches the pair kernel; cudaErrorNotSupported when clusters of two cannot run here.
template <int EPI, int HD, int EW>
cudaError_t launch_pair(const GemmArgs& g, Params p, cudaStream_t stream) {
  const int cap = pair_capacity<EPI, HD, EW>();
  if (cap < 1) return cudaErrorNotSupported;
  CUtensorMap ta, tb;
  if (!make_tmap_2d(&ta, g.a, g.M, g.K, BM) || !make_tmap_2d(&tb, g.w, g.N, g.K, BN_WIDE / 2))
    return cudaErrorInvalidValue;
  // raster groups of 256-row tiles (tiles taken in order from the counter): 16 for the
  // 20,480- and 28,672-wide projections, 8 otherwise (measured at 15,435 rows: 0.5-1.5%
  // over 8 and 4 respectively; 16 made the 20,480-deep fc2 slower)
  p.group = g.N >= 16384 ? 16 : 8;
  p.pairs = 0;
  const int tiles = ((g.M + 2 * BM - 1) / (2 * BM)) * (g.N / BN_WIDE);
  const int clusters = tiles < cap ? tiles : cap;
  p.tile_counter = g.tile_counter;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(pair_threads(EW), 1, 1);
  cfg.dynamicSmemBytes = P_SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<EPI, HD, EW>, ta, tb, p);
}

bool g_use_pairs = true;  // h3dit_gemm_cta_pairs

}  // namespace

bool gemm_cta_pairs(int enable) {
  const bool prev = g_use_pairs;
  if (enable >= 0) g_use_pairs = enable != 0;
  return prev;
}

cudaError_t launch_gemm(int epi, const GemmArgs& g, cudaStream_t stream) {
  // the output heads use one tile of exactly N columns; everything else 256-wide tiles
  const bool head = epi == kEpiHeadEuler;
  const int bn = head ? g.N : BN_WIDE;
  if (head && (g.N % 32 != 0 || g.N > 128 || !g.z || !g.bias)) return cudaErrorInvalidValue;
  if (g.M <= 0 || g.N <= 0 || g.N % bn != 0 || g.K % BK != 0 || g.K <= 0)
    return cudaErrorInvalidValue;
  CUtensorMap tb;
  if (!make_tmap_2d(&tb, g.w, g.N, g.K, bn)) return cudaErrorInvalidValue;
  Params p;
  // raster group: 16 row-blocks when N or K is long (the measured best at 15,435 rows:
  // N = 20,480 and K = 20,480), else 8 (N = K = 5,120)
  p.group = (g.N >= 16384 || g.K >= 16384) ? 16 : 8;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.bias = g.bias;
  p.y = g.y;
  p.gate = g.gate;
  p.gate_prefix = g.gate_prefix;
  p.n_prefix = g.n_prefix;
  p.heads = g.heads;
  p.head_dim = g.head_dim;
  p.attn_width = g.attn_width;
  p.q = g.q;
  p.k = g.k;
  p.v = g.v;
  p.g = g.g;
  p.qnorm_w = g.qnorm_w;
  p.knorm_w = g.knorm_w;
  p.rope_cs = g.rope_cs;
  p.eps = g.eps;
  p.v_out = g.v_out;
  p.z = g.z;
  p.dt = g.dt;
  p.status = g.status;
  p.tile_counter = nullptr;  // the one-SM kernel deals tiles round-robin
  if (g_use_pairs && epi != kEpiHeadEuler && !(epi == kEpiSwiglu && !g.bias) &&
      (epi != kEpiQkvg || g.head_dim == 64 || g.head_dim == 128)) {
    cudaError_t e = cudaErrorNotSupported;
    const bool short_k = g.K <= 4096;  // eight epilogue warps
    switch (epi) {
      case kEpiStore:
        e = short_k ? launch_pair<kEpiStore, 128, 8>(g, p, stream)
                    : launch_pair<kEpiStore, 128, 4>(g, p, stream);
        break;
      case kEpiGelu:
        e = short_k ? launch_pair<kEpiGelu, 128, 8>(g, p, stream)
                    : launch_pair<kEpiGelu, 128, 4>(g, p, stream);
        break;
      case kEpiResid:
        e = short_k ? launch_pair<kEpiResid, 128, 8>(g, p, stream)
                    : launch_pair<kEpiResid, 128, 4>(g, p, stream);
        break;
      case kEpiSwiglu:
        e = short_k ? launch_pair<kEpiSwiglu, 128, 8>(g, p, stream)
                    : launch_pair<kEpiSwiglu, 128, 4>(g, p, stream);
        break;
      case kEpiQkvg:
        e = g.head_dim == 128 ? launch_pair<kEpiQkvg, 128, 4>(g, p, stream)
                              : launch_pair<kEpiQkvg, 64, 4>(g, p, stream);
        break;
      default: break;
    }
    if (e != cudaErrorNotSupported) return e;  // launched (or failed for another reason)
  }
  switch (epi) {
    // plain stores: pair tiles; the rest 128 x 256
    case kEpiStore:
      return launch_one<kEpiStore, 128, BN_WIDE, true>(g, tb, p, stream);
    case kEpiGelu:
      return launch_one<kEpiGelu, 128>(g, tb, p, stream);
    case kEpiResid:
      return launch_one<kEpiResid, 128>(g, tb, p, stream);
    case kEpiSwiglu:
      if (!g.bias) return cudaErrorInvalidValue;
      return launch_one<kEpiSwiglu, 128>(g, tb, p, stream);
    case kEpiQkvg:
      if (g.head_dim == 128) return launch_one<kEpiQkvg, 128>(g, tb, p, stream);
      if (g.head_dim == 64) return launch_one<kEpiQkvg, 64>(g, tb, p, stream);
      return cudaErrorInvalidValue;
    case kEpiHeadEuler:
      if (g.N == 32) return launch_one<kEpiHeadEuler, 128, 32>(g, tb, p, stream);
      if (g.N == 64) return launch_one<kEpiHeadEuler, 128, 64>(g, tb, p, stream);
      if (g.N == 96) return launch_one<kEpiHeadEuler, 128, 96>(g, tb, p, stream);
      if (g.N == 128) return launch_one<kEpiHeadEuler, 128, 128>(g, tb, p, stream);
      return cudaErrorInvalidValue;
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace h3
