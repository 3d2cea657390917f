// attention.cu -- tile-routed attention on tcgen05 tensor cores.
//
// TensorFold #949, "What it adds" (h3_attention.metal: tile-routed attention
// with fp32 scores and an online softmax) and "Precision" (softmax weights
// rounded to bf16 before the value product).
//
// One CTA owns 128 query rows of one head:
//   * a prefix unit: 128 text/audio rows, attending to all N rows;
//   * a video unit: two 64-row video query tiles (2u, 2u+1), attending to all
//     prefix rows plus the union of the two tiles' selected key tiles.  Each
//     key tile carries a 2-bit mask saying which of the two query tiles chose
//     it; scores of the other half are masked to -inf, so every row sees
//     exactly its own key set.
// CTAs are ordered head-major (all units of head 0, then head 1, ...), so a
// wave of CTAs shares one head's K/V in L2.  The KV loop walks the key-tile
// list two 64-row tiles ("slots" 0 and 1, 128 keys) per step.  K and V tiles
// are gathered per step with one TMA box per 64 x 64 piece into 2-stage K and V
// rings (128-byte swizzle, no multicast); a K stage is released as soon as its
// S MMA completes and the producer loads K one step ahead of V, so the next
// step's keys arrive while the current step's softmax runs.
//   warp 0      TMA producer (Q once, then K and V per step)
//   warp 1      MMA issuer: S = Q K^T (M=128, N=128, fp32 in TMEM, double
//               buffered); O_c += P[:, slot c] V[slot c] for c = 0, 1 (two
//               fp32 TMEM accumulators, V read as an MN-major operand)
//   warps 2..9  softmax, two warps per TMEM lane quarter: warp (q, c) owns rows
//               32q..32q+31 and key slot c.  Each runs its own online softmax
//               over the keys of its slot (split-K): one 64-column TMEM read of
//               S per step, row max on the raw scores, P = exp2(s*scale*log2e -
//               m) rounded to bf16 into the swizzled K-major P tile in shared
//               memory, l summing the unrounded weights, O_c rescaled in TMEM
//               only when the max grows by more than 2^8.  The epilogue merges
//               the two slots' (m, l, O) per row, divides, adds gate * pooled
//               for video rows and stores bf16; each warp of a pair writes half
//               of the head dimensions.
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace h3 {

namespace {

constexpr int THREADS = 320;
constexpr int MAX_TILES = 1024;  // key tiles per unit: N <= 65,536 rows
constexpr float kRescaleLog2 = 8.0f;

template <int HD>
struct Layout {
  static constexpr int CHUNK = 128 * 128;        // 128 rows x 64 bf16 (one swizzle column)
  static constexpr int Q_BYTES = 128 * HD * 2;   // 128 query rows
  static constexpr int KV_BYTES = 128 * HD * 2;  // 128 keys
  static constexpr int P_BYTES = 128 * 128 * 2;  // 128 rows x 128 keys
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF0 = Q_OFF + Q_BYTES;
  static constexpr int V_OFF0 = K_OFF0 + KV_BYTES;
  static constexpr int STAGE_STRIDE = 2 * KV_BYTES;
  static constexpr int P_OFF = K_OFF0 + 2 * STAGE_STRIDE;
  static constexpr int TILES_OFF = P_OFF + P_BYTES;
  static constexpr int MERGE_OFF = TILES_OFF + MAX_TILES * 4;  // float2 [2][128]
  static constexpr int BAR_OFF = MERGE_OFF + 2 * 128 * 8;
  static constexpr int USED = BAR_OFF + 256;
  // keep one CTA per SM (the kernel allocates 512 TMEM columns)
  static constexpr int SMEM = (USED + 1024) > 120 * 1024 ? (USED + 1024) : 120 * 1024;
  static constexpr uint32_t S_COL = 0;          // two 128-column score buffers
  static constexpr uint32_t O_COL0 = 256;       // slot-0 accumulator
  static constexpr uint32_t O_COL1 = 256 + HD;  // slot-1 accumulator
};

struct Params {
  int N, H, n_prefix, n_video, Tv, ksel;
  int n_pre_units;
  const int* idx;
  const __nv_bfloat16* gate;
  const float* pooled;
  __nv_bfloat16* out;
  float scale_log2;
  int* status;
};

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
__global__ void __launch_bounds__(THREADS, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const Params p) {
  using L = Layout<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + L::Q_OFF;
  uint8_t* sP = smem + L::P_OFF;
  int* tiles = reinterpret_cast<int*>(smem + L::TILES_OFF);
  float2* merge_ml = reinterpret_cast<float2*>(smem + L::MERGE_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [2]
  uint64_t* v_full = bars + 3;    // [2]
  uint64_t* k_empty = bars + 5;   // [2] K stage free: its S MMA completed
  uint64_t* s_full = bars + 7;    // [2]
  uint64_t* p_full = bars + 9;
  uint64_t* pv_done = bars + 10;
  uint64_t* drain = bars + 11;
  uint64_t* merge_bar = bars + 12;
  uint64_t* v_empty = bars + 13;  // [2] V stage free: its PV MMA completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 15);
  int* n_steps_s = reinterpret_cast<int*>(tmem_slot + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // head-major order: a wave of CTAs works on one or two heads, so their K/V stay in L2
  const int n_units = p.n_pre_units + (p.Tv + 1) / 2;
  const int h = blockIdx.x / n_units;
  const int unit = blockIdx.x % n_units;
  const bool is_prefix = unit < p.n_pre_units;
  const int vu = unit - p.n_pre_units;
  const int ta = 2 * vu, tb = 2 * vu + 1;  // video query tiles of a video unit

  if (threadIdx.x == 0) {
    // key-tile list: entry = first_row << 2 | mask (bit 0: rows 0-63 use it, bit 1: rows 64-127)
    int nt = 0;
    if (is_prefix) {
      for (int r0 = 0; r0 < p.N && nt < MAX_TILES - 1; r0 += 64) tiles[nt++] = (r0 << 2) | 3;
    } else {
      for (int r0 = 0; r0 < p.n_prefix && nt < MAX_TILES - 1; r0 += 64)
        tiles[nt++] = (r0 << 2) | 3;
      const int* ia = p.idx + ((size_t)h * p.Tv + ta) * p.ksel;
      const int* ib = p.idx + ((size_t)h * p.Tv + tb) * p.ksel;
      const int na = p.ksel, nb = tb < p.Tv ? p.ksel : 0;
      int i = 0, j = 0;
      while ((i < na || j < nb) && nt < MAX_TILES - 1) {
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
        tiles[nt++] = ((p.n_prefix + 64 * t) << 2) | m;
      }
    }
    if (nt & 1) {  // pad to whole steps with a masked copy of the last tile
      tiles[nt] = tiles[nt - 1] & ~3;
      ++nt;
    }
    *n_steps_s = nt / 2;
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&s_full[s], 1);
    }
    mbar_init(p_full, 8);
    mbar_init(pv_done, 1);
    mbar_init(drain, 1);
    mbar_init(merge_bar, 8);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
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
        qrow0 = p.n_prefix + 64 * ta;
        qrow1 = p.n_prefix + 64 * tb;
      }
      mbar_arrive_expect_tx(q_full, L::Q_BYTES);
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) {
        tma_load_3d(sQ + c * L::CHUNK, &tmQ, q_full, 64 * c, qrow0, h);
        tma_load_3d(sQ + c * L::CHUNK + 8192, &tmQ, q_full, 64 * c, qrow1, h);
      }
      // K runs one step ahead of V: K_t is needed for S_t, V_t only after softmax(t)
      auto load_k = [&](int t) {
        const int st = t & 1;
        uint8_t* sK = smem + L::K_OFF0 + st * L::STAGE_STRIDE;
        const int r0 = tiles[2 * t] >> 2, r1 = tiles[2 * t + 1] >> 2;
        mbar_arrive_expect_tx(&k_full[st], L::KV_BYTES);
#pragma unroll
        for (int c = 0; c < HD / 64; ++c) {
          tma_load_3d(sK + c * L::CHUNK, &tmK, &k_full[st], 64 * c, r0, h);
          tma_load_3d(sK + c * L::CHUNK + 8192, &tmK, &k_full[st], 64 * c, r1, h);
        }
      };
      auto load_v = [&](int t) {
        const int st = t & 1;
        uint8_t* sV = smem + L::V_OFF0 + st * L::STAGE_STRIDE;
        const int r0 = tiles[2 * t] >> 2, r1 = tiles[2 * t + 1] >> 2;
        mbar_arrive_expect_tx(&v_full[st], L::KV_BYTES);
#pragma unroll
        for (int c = 0; c < HD / 64; ++c) {
          tma_load_3d(sV + c * L::CHUNK, &tmV, &v_full[st], 64 * c, r0, h);
          tma_load_3d(sV + c * L::CHUNK + 8192, &tmV, &v_full[st], 64 * c, r1, h);
        }
      };
      for (int t = 0; t <= n_steps; ++t) {
        if (t < n_steps) {
          if (!mbar_wait(&k_empty[t & 1], ((t >> 1) & 1) ^ 1, abort_flag, p.status)) break;
          load_k(t);
        }
        if (t >= 1) {
          const int tv = t - 1;
          if (!mbar_wait(&v_empty[tv & 1], ((tv >> 1) & 1) ^ 1, abort_flag, p.status)) break;
          load_v(tv);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(128, HD, false, true);
      const uint32_t q0 = smem_u32(sQ);
      const uint32_t p0 = smem_u32(sP);
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status);
      if (ok) ok = mbar_wait(&k_full[0], 0, abort_flag, p.status);
      if (ok) {
        tc_fence_after();
        const uint32_t k0 = smem_u32(smem + L::K_OFF0);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * L::CHUNK + (ks & 3) * 32;
          umma_bf16(tmem + L::S_COL, sdesc_sw128(q0 + off, 16, 1024),
                    sdesc_sw128(k0 + off, 16, 1024), idesc_s, ks > 0 ? 1u : 0u);
        }
        umma_commit(&k_empty[0]);
        umma_commit(&s_full[0]);
      }
      for (int t = 0; ok && t < n_steps; ++t) {
        const int st = t & 1;
        if (t + 1 < n_steps) {
          const int sn = (t + 1) & 1;
          if (!mbar_wait(&k_full[sn], ((t + 1) >> 1) & 1, abort_flag, p.status)) break;
          tc_fence_after();
          const uint32_t k0 = smem_u32(smem + L::K_OFF0 + sn * L::STAGE_STRIDE);
#pragma unroll
          for (int ks = 0; ks < HD / 16; ++ks) {
            const uint32_t off = (ks >> 2) * L::CHUNK + (ks & 3) * 32;
            umma_bf16(tmem + L::S_COL + sn * 128, sdesc_sw128(q0 + off, 16, 1024),
                      sdesc_sw128(k0 + off, 16, 1024), idesc_s, ks > 0 ? 1u : 0u);
          }
          umma_commit(&k_empty[sn]);
          umma_commit(&s_full[sn]);
        }
        if (!mbar_wait(p_full, t & 1, abort_flag, p.status)) break;
        if (!mbar_wait(&v_full[st], (t >> 1) & 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t v0 = smem_u32(smem + L::V_OFF0 + st * L::STAGE_STRIDE);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          // keys 16ks..16ks+15: slot ks/4 -> accumulator O_(ks/4)
          const uint32_t aoff = (ks >> 2) * L::CHUNK + (ks & 3) * 32;
          const uint32_t obuf = tmem + (ks < 4 ? L::O_COL0 : L::O_COL1);
          // V: MN-major; LBO = next 64-dim column block, SBO = next 8 keys
          umma_bf16(obuf, sdesc_sw128(p0 + aoff, 16, 1024),
                    sdesc_sw128(v0 + ks * 2048, L::CHUNK, 1024), idesc_pv,
                    (t > 0 || (ks & 3) > 0) ? 1u : 0u);
        }
        umma_commit(&v_empty[st]);
        umma_commit(pv_done);
      }
      umma_commit(drain);
      mbar_drain(drain, 0);
    }
  } else {
    // ---------------------------------------------------------------- softmax
    const int quad = warp & 3;
    const int slot = (warp - 2) >> 2;  // warps 2..5 -> slot 0, warps 6..9 -> slot 1
    const int row = quad * 32 + lane;
    const int half = row >> 6;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t o_mine = t_lane + (slot ? L::O_COL1 : L::O_COL0);
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY;
    float l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < n_steps; ++t) {
      const int sb = t & 1;
      if (!mbar_wait(&s_full[sb], (t >> 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int e = tiles[2 * t + slot];
      const int nv = ((e >> half) & 1) ? min(64, p.N - (e >> 2)) : 0;
      // this slot's 64 raw scores; max on the raw values (the scale is positive)
      float sv[64];
      tmem_ld64(t_lane + L::S_COL + sb * 128 + slot * 64, sv);
      float mx8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx8[u] = -INFINITY;
      if (nv == 64) {  // warp-uniform: every key of the slot is visible to these rows
#pragma unroll
        for (int j = 0; j < 64; ++j) mx8[j & 7] = fmaxf(mx8[j & 7], sv[j]);
      } else {
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          sv[j] = j < nv ? sv[j] : -INFINITY;
          mx8[j & 7] = fmaxf(mx8[j & 7], sv[j]);
        }
      }
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * sl2;
      const bool need = mx > m_run + kRescaleLog2;
      const float m_new = need ? mx : m_run;
      const float alpha = need ? ex2_approx(m_run - m_new) : 1.0f;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      // P = exp2(s * scale - m) rounded to bf16; l sums the unrounded weights
      uint32_t pk[32];
      float ls8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) ls8[u] = 0.f;
#pragma unroll
      for (int j = 0; j < 64; j += 2) {
        const float e0 = ex2_approx(fmaf(sv[j], sl2, -m_use));
        const float e1 = ex2_approx(fmaf(sv[j + 1], sl2, -m_use));
        ls8[(j >> 1) & 7] += e0;
        ls8[(j >> 1) & 7] += e1;
        pk[j >> 1] = pack_bf16x2(e0, e1);
      }
      const float lsum = ((ls8[0] + ls8[1]) + (ls8[2] + ls8[3])) +
                         ((ls8[4] + ls8[5]) + (ls8[6] + ls8[7]));
      if (t > 0) {
        // the previous step's PV reads the single P tile and updates O: wait for it
        if (!mbar_wait(pv_done, (t - 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, need)) rescale_rows<HD>(o_mine, alpha);
      }
      l_run = fmaf(l_run, alpha, lsum);
      m_run = m_new;
      // keys of this slot -> column block `slot`; 16-byte unit u holds keys 8u..8u+7
      uint8_t* rowp = sP + slot * L::CHUNK + row * 128;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        *reinterpret_cast<uint4*>(rowp + ((u ^ (row & 7)) << 4)) =
            make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok && n_steps > 0) {
      bool done = mbar_wait(pv_done, (n_steps - 1) & 1, abort_flag, p.status);
      if (done) {
        // merge the two slots' online-softmax states of each row
        merge_ml[slot * 128 + row] = make_float2(m_run, l_run);
        __syncwarp();
        if (lane == 0) mbar_arrive(merge_bar);
        done = mbar_wait(merge_bar, 0, abort_flag, p.status);
      }
      if (done) {
        tc_fence_after();
        const float2 a = merge_ml[row], b = merge_ml[128 + row];
        const float m = fmaxf(a.x, b.x);
        const float sa = (a.x == -INFINITY) ? 0.f : ex2_approx(a.x - m);
        const float sbb = (b.x == -INFINITY) ? 0.f : ex2_approx(b.x - m);
        const float l = fmaf(a.y, sa, b.y * sbb);
        const float inv_l = l > 0.f ? 1.0f / l : 0.f;
        int grow, tile = -1;
        bool store;
        if (is_prefix) {
          grow = unit * 128 + row;
          store = grow < p.n_prefix;
        } else {
          tile = half ? tb : ta;
          grow = p.n_prefix + 64 * tile + (row & 63);
          store = tile < p.Tv && grow < p.N;
        }
        const int A = p.H * HD;
        const bool mix = !is_prefix && p.gate != nullptr && p.pooled != nullptr;
        // this warp writes head dims [slot * HD/2, (slot + 1) * HD/2)
#pragma unroll 1
        for (int c = 0; c < HD / 64; ++c) {
          const int d0 = slot * (HD / 2) + c * 32;
          float o0[32], o1[32];
          tmem_ld32(t_lane + L::O_COL0 + d0, o0);
          tmem_ld32(t_lane + L::O_COL1 + d0, o1);
          if (store) {
            float o[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = fmaf(o0[j], sa, o1[j] * sbb) * inv_l;
            if (mix) {
              const uint4* g4 =
                  reinterpret_cast<const uint4*>(p.gate + (size_t)grow * A + h * HD + d0);
              const float4* pb4 = reinterpret_cast<const float4*>(
                  p.pooled + ((size_t)h * p.Tv + tile) * HD + d0);
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
            uint4* dst = reinterpret_cast<uint4*>(p.out + (size_t)grow * A + h * HD + d0);
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
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
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
  if (a.N <= 0 || a.H <= 0 || a.N > (MAX_TILES - 2) * 64) return cudaErrorInvalidValue;
  if (a.d == 128) return launch_hd<128>(a, stream);
  if (a.d == 64) return launch_hd<64>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace h3
