// attention.cu -- tile-routed attention on tcgen05 tensor cores.
//
// TensorFold #949, "What it adds" (h3_attention.metal: tile-routed attention
// with fp32 scores and an online softmax) and "Precision" (softmax weights
// rounded to bf16 before the value product).
//
// One CTA owns 128 query rows of one head:
//   * a prefix unit: 128 text/audio rows, attending to all N rows;
//   * a video unit: two video query tiles (2u, 2u+1) of up to 64 rows each (a
//     64-row slice or a clipped 4x4x4 cube, contiguous in the library's row
//     order), attending to all prefix rows plus the union of the two tiles'
//     selected key tiles; a key tile with fewer than 64 rows masks the rest.  Each
//     key tile carries a 2-bit mask saying which of the two query tiles chose
//     it; scores of the other half are masked to -inf, so every row sees
//     exactly its own key set.
// CTAs run the long prefix units first (all heads), then the video units
// head-major, so a wave of video CTAs shares one or two heads' K/V in L2 and no
// long unit starts at the end of the grid.  The KV loop walks the key-tile
// list one 64-row tile per step.  K and V tiles arrive by TMA (one box per
// 64 x 64 piece, 128-byte swizzle, no multicast) into 2-stage K and V rings; a
// K stage is released as soon as its S MMA completes, a V stage as soon as its
// PV MMA completes, and each ring has its own producer warp, so a key tile is
// requested two steps before its S MMA.  A CTA needs ~101 KB of shared memory
// and 256 TMEM columns, so two CTAs share an SM and each hides the other's
// latencies.
//   warp 0      TMA producer: Q once, then the K ring
//   warp 6      TMA producer: the V ring
//   warp 1      MMA issuer: S = Q K^T (M=128, N=64, fp32 in TMEM, double
//               buffered) and O += P V (M=128, N=d, K=64) with P read from TMEM
//               and V from shared memory as an MN-major operand
//   warps 2..5  softmax, thread = query row (TMEM lane): one 64-column TMEM read
//               of S per step, row max on the raw scores, P = exp2(s*scale*log2e
//               - m) rounded to bf16 and stored back over the step's S columns
//               (two bf16 per 32-bit column), l summing the unrounded weights;
//               O is rescaled in TMEM only when the max grows by more than 2^8, and
//               only then does a step wait for the previous step's PV to finish, so
//               the softmax of step t overlaps the PV of step t - 1.
//               Epilogue: O / l, + gate * pooled for video rows, bf16 store.
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace h3 {

namespace {

constexpr int THREADS = 224;  // 7 warps: K/Q producer, MMA, 4 softmax, V producer
constexpr int MAX_TILES = 1024;  // key tiles per unit: N <= 65,536 rows
constexpr float kRescaleLog2 = 8.0f;

template <int HD>
struct Layout {
  static constexpr int QCHUNK = 128 * 128;       // 128 query rows x 64 dims (bf16)
  static constexpr int KCHUNK = 64 * 128;        // 64 keys x 64 dims (bf16)
  static constexpr int Q_BYTES = 128 * HD * 2;
  static constexpr int KV_BYTES = 64 * HD * 2;   // one 64-row key tile
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF0 = Q_OFF + Q_BYTES;          // K stage s at K_OFF0 + s * KV_BYTES
  static constexpr int V_OFF0 = K_OFF0 + 2 * KV_BYTES;    // V stage s at V_OFF0 + s * KV_BYTES
  static constexpr int TILES_OFF = V_OFF0 + 2 * KV_BYTES;
  static constexpr int BAR_OFF = TILES_OFF + MAX_TILES * 4;
  static constexpr int USED = BAR_OFF + 256;
  // + alignment slack; at least 80 KB so that no more than two CTAs (the TMEM
  // budget: 2 x 256 columns) are resident on an SM
  static constexpr int SMEM = (USED + 1024) > 80 * 1024 ? (USED + 1024) : 80 * 1024;
  static constexpr uint32_t S_COL = 0;                    // two 64-column score buffers
  static constexpr uint32_t O_COL = 128;                  // HD-column accumulator
  static constexpr uint32_t TMEM_COLS = 256;
};

struct Params {
  int N, H, n_prefix, n_video, Tv, ksel;
  int n_pre_units;
  TileGeom geom;
  const int* idx;
  const __nv_bfloat16* gate;
  const float* pooled;
  __nv_bfloat16* out;
  float scale_log2;
  int* status;
};

// max of three fp32 values in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <int HD>
__device__ __forceinline__ void rescale_rows(uint32_t taddr, float alpha) {
#pragma unroll 1
  for (int c = 0; c < HD / 32; ++c) {
    float o[32];
    tmem_ld32(taddr + c * 32, o);
#pragma unroll
    for (int j = 0; j < 32; ++j) o[j] *= alpha;
    tmem_st32(taddr + c * 32, o);
  }
}

template <int HD>
__global__ void __launch_bounds__(THREADS, 2)
    attention_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const Params p) {
  using L = Layout<HD>;
  static_assert(L::SMEM <= 113 * 1024, "two CTAs must fit on one SM");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + L::Q_OFF;
  int* tiles = reinterpret_cast<int*>(smem + L::TILES_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [2]
  uint64_t* v_full = bars + 3;    // [2]
  // s_done[st]: S of the step in stage st is in TMEM and its K stage is free (one commit,
  // waited by the softmax warps and the K producer); pv_done[st]: the step's PV completed,
  // so its V stage is free and O is stable (waited by the V producer and the softmax)
  uint64_t* s_done = bars + 5;    // [2]
  uint64_t* pv_done = bars + 7;   // [2]
  uint64_t* p_full = bars + 11;   // [2] by step parity: no waiter can fall two phases behind
  uint64_t* drain = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
  int* n_steps_s = reinterpret_cast<int*>(tmem_slot + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // longest work first: all prefix units (each walks every key tile), head-major, then all
  // video units, head-major (a wave of video CTAs shares one or two heads' K/V in L2)
  const int n_vid_units = (p.Tv + 1) / 2;
  const int n_pre_ctas = p.n_pre_units * p.H;
  int h, unit;
  if ((int)blockIdx.x < n_pre_ctas) {
    h = blockIdx.x / p.n_pre_units;
    unit = blockIdx.x % p.n_pre_units;
  } else {
    const int b = blockIdx.x - n_pre_ctas;
    h = b / n_vid_units;
    unit = p.n_pre_units + b % n_vid_units;
  }
  const bool is_prefix = unit < p.n_pre_units;
  const int vu = unit - p.n_pre_units;
  const int ta = 2 * vu, tb = 2 * vu + 1;  // video query tiles of a video unit

  if (threadIdx.x == 0) {
    // key-tile list: entry = first_row << 9 | rows << 2 | mask (rows: 1..64 keys from
    // first_row; mask bit 0: query rows 0-63 use it, bit 1: query rows 64-127)
    int nt = 0;
    if (is_prefix) {
      for (int r0 = 0; r0 < p.N && nt < MAX_TILES; r0 += 64)
        tiles[nt++] = (r0 << 9) | (min(64, p.N - r0) << 2) | 3;
    } else {
      for (int r0 = 0; r0 < p.n_prefix && nt < MAX_TILES; r0 += 64)
        tiles[nt++] = (r0 << 9) | (min(64, p.n_prefix - r0) << 2) | 3;
      const int* ia = p.idx + ((size_t)h * p.Tv + ta) * p.ksel;
      const int* ib = p.idx + ((size_t)h * p.Tv + tb) * p.ksel;
      const int na = p.ksel, nb = tb < p.Tv ? p.ksel : 0;
      int i = 0, j = 0;
      while ((i < na || j < nb) && nt < MAX_TILES) {
        int t, m;
        if (j >= nb || (i < na && ia[i] < ib[j])) {
          t = ia[i++];
          m = 1;
        } else if (i >= na || ib[j] < ia[i]) {
          t = ib[j++];
          m = 2;
        } else {
          t = ia[i++];
          ++j;
          m = 3;
        }
        t = min(max(t, 0), p.Tv - 1);  // indices come from the router; clamp defensively
        int f, c;
        tile_span(p.geom, t, &f, &c);
        tiles[nt++] = (f << 9) | (c << 2) | m;
      }
    }
    *n_steps_s = nt;
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&s_done[s], 1);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(&p_full[0], 4);
    mbar_init(&p_full[1], 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_steps = *n_steps_s;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      int qrow0, qrow1;
      if (is_prefix) {
        qrow0 = unit * 128;
        qrow1 = unit * 128 + 64;
      } else {
        int c;
        tile_span(p.geom, ta, &qrow0, &c);
        qrow1 = qrow0;  // an odd tile count leaves the second half without a tile
        if (tb < p.Tv) tile_span(p.geom, tb, &qrow1, &c);
      }
      mbar_arrive_expect_tx(q_full, L::Q_BYTES);
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) {
        tma_load_3d(sQ + c * L::QCHUNK, &tmQ, q_full, 64 * c, qrow0, h);
        tma_load_3d(sQ + c * L::QCHUNK + 8192, &tmQ, q_full, 64 * c, qrow1, h);
      }
      // K ring: a stage is refilled as soon as its S MMA completes (V has its own producer)
      for (int t = 0; t < n_steps; ++t) {
        const int st = t & 1;
        if (!mbar_wait(&s_done[st], ((t >> 1) & 1) ^ 1, abort_flag, p.status)) break;
        uint8_t* sK = smem + L::K_OFF0 + st * L::KV_BYTES;
        const int r0 = tiles[t] >> 9;
        mbar_arrive_expect_tx(&k_full[st], L::KV_BYTES);
#pragma unroll
        for (int c = 0; c < HD / 64; ++c)
          tma_load_3d(sK + c * L::KCHUNK, &tmK, &k_full[st], 64 * c, r0, h);
      }
    }
  } else if (warp == 6) {
    if (lane == 0) {
      // V ring: a stage is refilled as soon as its PV MMA completes
      for (int t = 0; t < n_steps; ++t) {
        const int st = t & 1;
        if (!mbar_wait(&pv_done[st], ((t >> 1) & 1) ^ 1, abort_flag, p.status)) break;
        uint8_t* sV = smem + L::V_OFF0 + st * L::KV_BYTES;
        const int r0 = tiles[t] >> 9;
        mbar_arrive_expect_tx(&v_full[st], L::KV_BYTES);
#pragma unroll
        for (int c = 0; c < HD / 64; ++c)
          tma_load_3d(sV + c * L::KCHUNK, &tmV, &v_full[st], 64 * c, r0, h);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 64, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(128, HD, false, true);
      const uint32_t q0 = smem_u32(sQ);
      auto issue_s = [&](int t) {
        const int st = t & 1;
        const uint32_t k0 = smem_u32(smem + L::K_OFF0 + st * L::KV_BYTES);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t qoff = (ks >> 2) * L::QCHUNK + (ks & 3) * 32;
          const uint32_t koff = (ks >> 2) * L::KCHUNK + (ks & 3) * 32;
          umma_bf16(tmem + L::S_COL + st * 64, sdesc_sw128(q0 + qoff, 16, 1024),
                    sdesc_sw128(k0 + koff, 16, 1024), idesc_s, ks > 0 ? 1u : 0u);
        }
        umma_commit(&s_done[st]);
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status);
      if (ok && n_steps > 0) ok = mbar_wait(&k_full[0], 0, abort_flag, p.status);
      if (ok && n_steps > 0) {
        tc_fence_after();
        issue_s(0);
      }
      for (int t = 0; ok && t < n_steps; ++t) {
        const int st = t & 1;
        if (t + 1 < n_steps) {
          if (!mbar_wait(&k_full[(t + 1) & 1], ((t + 1) >> 1) & 1, abort_flag, p.status)) break;
          tc_fence_after();
          issue_s(t + 1);
        }
        if (!mbar_wait(&p_full[st], (t >> 1) & 1, abort_flag, p.status)) break;
        if (!mbar_wait(&v_full[st], (t >> 1) & 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t v0 = smem_u32(smem + L::V_OFF0 + st * L::KV_BYTES);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          // P: keys 16ks..16ks+15 are TMEM columns 8ks..8ks+7 of the step's S buffer;
          // V: MN-major, LBO = next 64-dim column block, SBO = next 8 keys
          umma_bf16_ts(tmem + L::O_COL, tmem + L::S_COL + st * 64 + ks * 8,
                       sdesc_sw128(v0 + ks * 2048, L::KCHUNK, 1024), idesc_pv,
                       (t > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(&pv_done[st]);
      }
      umma_commit(drain);
      mbar_drain(drain, 0);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ---------------------------------------------------------------- softmax
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int half = row >> 6;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY;
    float l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < n_steps; ++t) {
      const int sb = t & 1;
      if (!mbar_wait(&s_done[sb], (t >> 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int e = tiles[t];
      const int nv = ((e >> half) & 1) ? ((e >> 2) & 127) : 0;
      const uint32_t s_addr = t_lane + L::S_COL + sb * 64;
      float sv[64];
      tmem_ld64(s_addr, sv);
      // row max, two new scores per three-input max
      float mx4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) mx4[u] = -INFINITY;
      if (nv < 64) {  // warp-uniform: mask the keys of this tile that the row does not see
#pragma unroll
        for (int j = 0; j < 64; ++j) sv[j] = j < nv ? sv[j] : -INFINITY;
      }
#pragma unroll
      for (int j = 0; j < 64; j += 2) mx4[(j >> 1) & 3] = fmax3(mx4[(j >> 1) & 3], sv[j], sv[j + 1]);
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * sl2;
      const bool need = mx > m_run + kRescaleLog2;
      const float m_new = need ? mx : m_run;
      const float alpha = need ? ex2_approx(m_run - m_new) : 1.0f;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      // P = exp2(s * scale - m) rounded to bf16; l sums the unrounded weights.  The
      // scale-and-shift and the sums run two lanes of fp32 per instruction.
      uint32_t pk[32];
      const float2 sc2 = make_float2(sl2, sl2), nm2 = make_float2(-m_use, -m_use);
      float2 ls2[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) ls2[u] = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 64; j += 2) {
        const float2 x = __ffma2_rn(make_float2(sv[j], sv[j + 1]), sc2, nm2);
        const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        ls2[(j >> 1) & 3] = __fadd2_rn(ls2[(j >> 1) & 3], e);
        pk[j >> 1] = pack_bf16x2(e.x, e.y);
      }
      const float lsum = ((ls2[0].x + ls2[0].y) + (ls2[1].x + ls2[1].y)) +
                         ((ls2[2].x + ls2[2].y) + (ls2[3].x + ls2[3].y));
      // P over the first 32 columns of this step's S buffer (already read above)
      tmem_st32_u(s_addr, pk);
      if (t > 0 && __any_sync(0xffffffffu, need)) {
        // O must not change under a rescale while the previous step's PV runs
        if (!mbar_wait(&pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        rescale_rows<HD>(t_lane + L::O_COL, alpha);
      }
      l_run = fmaf(l_run, alpha, lsum);
      m_run = m_new;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
    }
    if (ok && n_steps > 0 &&
        mbar_wait(&pv_done[(n_steps - 1) & 1], ((n_steps - 1) >> 1) & 1, abort_flag, p.status)) {
      tc_fence_after();
      int grow, tile = -1;
      bool store;
      if (is_prefix) {
        grow = unit * 128 + row;
        store = grow < p.n_prefix;
      } else {
        tile = half ? tb : ta;
        int f = 0, c = 0;
        if (tile < p.Tv) tile_span(p.geom, tile, &f, &c);
        grow = f + (row & 63);
        store = (row & 63) < c;
      }
      const float inv_l = l_run > 0.f ? 1.0f / l_run : 0.f;
      const int A = p.H * HD;
      const bool mix = !is_prefix && p.gate != nullptr && p.pooled != nullptr;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        float o[32];
        tmem_ld32(t_lane + L::O_COL + c * 32, o);
        if (store) {
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] *= inv_l;
          if (mix) {
            const uint4* g4 =
                reinterpret_cast<const uint4*>(p.gate + (size_t)grow * A + h * HD + c * 32);
            const float4* pb4 = reinterpret_cast<const float4*>(
                p.pooled + ((size_t)h * p.Tv + tile) * HD + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 g = __ldg(g4 + i);
              const float4 b0 = __ldg(pb4 + 2 * i), b1 = __ldg(pb4 + 2 * i + 1);
              o[8 * i + 0] = fmaf(bf16_lo(g.x), b0.x, o[8 * i + 0]);
              o[8 * i + 1] = fmaf(bf16_hi(g.x), b0.y, o[8 * i + 1]);
              o[8 * i + 2] = fmaf(bf16_lo(g.y), b0.z, o[8 * i + 2]);
              o[8 * i + 3] = fmaf(bf16_hi(g.y), b0.w, o[8 * i + 3]);
              o[8 * i + 4] = fmaf(bf16_lo(g.z), b1.x, o[8 * i + 4]);
              o[8 * i + 5] = fmaf(bf16_hi(g.z), b1.y, o[8 * i + 5]);
              o[8 * i + 6] = fmaf(bf16_lo(g.w), b1.z, o[8 * i + 6]);
              o[8 * i + 7] = fmaf(bf16_hi(g.w), b1.w, o[8 * i + 7]);
            }
          }
          uint4* dst = reinterpret_cast<uint4*>(p.out + (size_t)grow * A + h * HD + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            dst[i] = make_uint4(pack_bf16x2(o[8 * i + 0], o[8 * i + 1]),
                                pack_bf16x2(o[8 * i + 2], o[8 * i + 3]),
                                pack_bf16x2(o[8 * i + 4], o[8 * i + 5]),
                                pack_bf16x2(o[8 * i + 6], o[8 * i + 7]));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int HD>
cudaError_t launch_hd(const AttnArgs& a, cudaStream_t stream) {
  using L = Layout<HD>;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_3d(&tq, a.q, a.H, a.N, HD) || !make_tmap_3d(&tk, a.k, a.H, a.N, HD) ||
      !make_tmap_3d(&tv, a.v, a.H, a.N, HD))
    return cudaErrorInvalidValue;
  Params p;
  p.N = a.N;
  p.H = a.H;
  p.n_prefix = a.n_prefix;
  p.n_video = a.n_video;
  p.Tv = a.Tv;
  p.ksel = a.ksel;
  p.n_pre_units = (a.n_prefix + 127) / 128;
  p.geom = a.geom;
  p.idx = a.idx;
  p.gate = a.gate;
  p.pooled = a.pooled;
  p.out = a.out;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)HD));
  p.status = a.status;
  const int n_units = p.n_pre_units + (a.Tv + 1) / 2;
  auto kern = attention_kernel<HD>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<n_units * a.H, THREADS, L::SMEM, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream) {
  if (a.N <= 0 || a.H <= 0 || a.N > MAX_TILES * 64) return cudaErrorInvalidValue;
  if (a.d == 128) return launch_hd<128>(a, stream);
  if (a.d == 64) return launch_hd<64>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace h3
