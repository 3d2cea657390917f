// attention.cu -- tile-routed attention on tcgen05 tensor cores.
//
// TensorFold #949, "What it adds" (h3_attention.metal: tile-routed attention
// with fp32 scores and an online softmax) and "Precision" (softmax weights
// rounded to bf16 before the value product).
//
// Work unit: 128 query rows of one head.
//   * a prefix unit: 128 text/audio rows, attending to all N rows;
//   * a video unit: two video query tiles a = 2u and b = 2u + 1 (up to 64 rows each, a
//     64-row slice or a clipped 4x4x4 cube, contiguous in the library's row order) as
//     rows 0-63 and 64-127, attending to all prefix rows plus each tile's own k
//     selected key tiles.
// A step feeds 128 keys to the tensor cores as two 64-row key blocks, X and Y:
//   * dense step (the prefix keys of a video unit, every key of a prefix unit): X and
//     Y are consecutive 64-row chunks and every query row uses both;
//   * routed step i (video units): X is the i-th key tile selected by tile a, Y the
//     i-th selected by tile b.  The score MMA computes all four 64 x 64 products
//     (N = 128); rows of a read only the X columns, rows of b only the Y columns, and
//     the softmax writes P block-diagonally (zeros in the other block), so the PV MMA
//     (K = 128) adds each row's own keys and nothing else.
//   Key tiles that both query tiles selected go two to a dense step (no discarded
//   blocks), and the routed steps pair the tiles only a selected with those only b
//   selected: a video unit with s tiles in common takes ceil(P / 128) + ceil(s / 2) +
//   (k - s) steps, and a row's softmax sees 64 scores per routed step.  A key block with
//   fewer than 64 rows (a clipped cube, the end of a range) masks the rest.
//
// Persistent: one CTA per SM.  A CTA takes units blockIdx.x and gridDim.x + blockIdx.x,
// then fetches further units from a counter in the workspace (zeroed by the router,
// which runs first), so that the long prefix units spread evenly; units are numbered
// prefix units first (head-major), then video units head-major, so the CTAs in flight
// share one or two heads' K/V in L2.  The pipelines run across unit boundaries.
// Tensor memory (512 columns): three 128-column score buffers and the O accumulator.
// The kernel's time is set by each step's S -> softmax -> PV chain (mostly the softmax's
// work on its TMEM lane quarter), not by memory bandwidth: step g + 3's score MMAs wait
// for step g's PV to free their buffer, so a third buffer gives the chain a step more of
// slack than two (attention 5% faster on the default block, 9% on the receipt).  Q therefore
// lives in shared memory (one buffer, the score MMA reading both operands there), beside
// a three-stage K ring and a two-stage V ring (32 KB stages; 192 KB in all).
//   warp 0       TMA: the K ring (a stage = X + Y, 128 keys), and the unit's Q (rows
//                0-63 and 64-127 as X and Y) once the previous unit's score MMAs are done
//   warp 1       S issuer: S = Q [K_X; K_Y]^T (M = 128, N = 128, fp32) into the step's
//                score buffer once the PV three steps back has read it
//   warp 11      PV issuer: O += P [V_X; V_Y] (K = 128, P from tensor memory, V
//                MN-major).  Two issuing threads keep the tensor pipe fed: the S
//                MMAs of later steps queue while the PV issuer waits for a softmax.
//   warps 2..5   softmax, thread = query row (TMEM lane): P = exp2(s * scale * log2e
//                - m) rounded to bf16 over the step's S columns (two per 32-bit
//                column), l summing the unrounded weights; the running max m is kept
//                in whole octaves (rounded up to an integer in the log2 domain), so a
//                weight's bf16 rounding does not depend on which max the row had met
//                (a power-of-two scale commutes with it); O is rescaled in TMEM, by an
//                exact power of two, only when the row max grows by more than 2^32
//                (weights up to 2^32 keep l and O finite for |v| < 2^80 over 65,536
//                keys), and only then does a step wait for the previous PV
//   warp 6       TMA: the V ring
//   warps 7..10  per unit: O / l, + gate * pooled for video rows, bf16 store; warp 7
//                also fetches units and writes their step lists
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace h3 {

namespace {

constexpr int THREADS = 384;     // 12 warps
constexpr int MAX_STEPS = 512;   // steps per unit (a prefix unit walks N / 128 steps)
constexpr int NSK = 3;           // stages of the K ring
constexpr int NSV = 2;           // stages of the V ring
constexpr int NSB = 3;           // score buffers in tensor memory
constexpr float kRescaleLog2 = 32.0f;

template <int HD>
struct Layout {
  static constexpr int KCHUNK = 64 * 128;  // 64 keys x 64 dims (bf16, 128-byte rows)
  static constexpr int BLK = 64 * HD * 2;  // one 64-row key block
  // A K or V stage holds X and Y interleaved per 64-dim chunk: chunk c of X at
  // 2c * KCHUNK, chunk c of Y right after it, so each chunk is one 128-row operand.
  static constexpr int STAGE = 2 * BLK;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + NSK * STAGE;
  // Q of the unit: rows 0-63 and 64-127 as X and Y of a stage (one 128-row operand per
  // 64-dim chunk), the score MMA's A operand
  static constexpr int Q_OFF = V_OFF + NSV * STAGE;
  static constexpr int LIST_OFF = Q_OFF + STAGE;                 // two step lists (int2)
  static constexpr int LBUF_OFF = LIST_OFF + 2 * MAX_STEPS * 8;  // 128 row sums
  static constexpr int UNIT_OFF = LBUF_OFF + 128 * 4;            // unit numbers, step counts
  static constexpr int MASK_OFF = UNIT_OFF + 16;                 // list builder's tile masks
  static constexpr int BAR_OFF = MASK_OFF + 2 * 32 * 4;
  static constexpr int USED = BAR_OFF + 256;
  static constexpr int SMEM = USED + 1024;                       // + alignment slack
  static constexpr uint32_t S_COL = 0;    // three 128-column score buffers
  static constexpr uint32_t O_COL = 384;  // the accumulator, HD columns
  static constexpr uint32_t TMEM_COLS = 512;
};

struct Params {
  int N, H, n_prefix, Tv, ksel;
  int n_pre_units, n_vid_units, total;  // units per head (prefix, video); all units
  int steps_all, steps_pre;             // ceil(N / 128), ceil(n_prefix / 128)
  TileGeom geom;
  const __nv_bfloat16* q;
  const int* idx;
  const __nv_bfloat16* gate;
  const float* pooled;
  __nv_bfloat16* out;
  float scale_log2;
  int* status;
  int* counter;
};

struct Unit {
  int h, unit, ta, tb;
  bool prefix;
};

__device__ __forceinline__ Unit unit_of(const Params& p, int w) {
  Unit u;
  const int n_pre = p.n_pre_units * p.H;
  if (w < n_pre) {
    u.h = w / p.n_pre_units;
    u.unit = w % p.n_pre_units;
  } else {
    const int b = w - n_pre;
    u.h = b / p.n_vid_units;
    u.unit = p.n_pre_units + b % p.n_vid_units;
  }
  u.prefix = u.unit < p.n_pre_units;
  u.ta = 2 * (u.unit - p.n_pre_units);
  u.tb = u.ta + 1;
  return u;
}

// key block entry: first_row << 9 | rows << 2 | dense (rows 0..64 from first_row)
__device__ __forceinline__ int chunk_entry(int r0, int limit) {
  return (r0 << 9) | (max(0, min(64, limit - r0)) << 2) | 1;
}

// Step list of unit u, written by one warp; returns the unit's step count.
//   prefix unit: ceil(N / 128) dense steps over consecutive 128-row chunks;
//   video unit: ceil(P / 128) dense steps over the prefix rows, then the key tiles both
//   query tiles selected, two to a dense step, then routed steps pairing the tiles only
//   tile a selected with those only tile b selected (ascending tile order throughout).
// The selections become bitmasks over the (at most 1,024) video tiles in masks[0..63]:
// lane i owns the words for tiles 32i..32i+31, so ascending order is lane order.
__device__ int build_list(const Params& p, const Unit& u, int2* list, uint32_t* masks,
                          int lane) {
  const int limit = u.prefix ? p.N : p.n_prefix;
  const int n_dense = u.prefix ? p.steps_all : p.steps_pre;
  for (int s = lane; s < n_dense; s += 32)
    list[s] = make_int2(chunk_entry(128 * s, limit), chunk_entry(128 * s + 64, limit));
  if (u.prefix) return n_dense;
  uint32_t* ma = masks;
  uint32_t* mb = masks + 32;
  ma[lane] = 0u;
  mb[lane] = 0u;
  __syncwarp();
  const int* ia = p.idx + ((size_t)u.h * p.Tv + u.ta) * p.ksel;
  // an odd tile count leaves the last unit's second half without a tile: it repeats a
  const int* ib = u.tb < p.Tv ? p.idx + ((size_t)u.h * p.Tv + u.tb) * p.ksel : ia;
  for (int i = lane; i < p.ksel; i += 32) {
    // indices come from the router; clamp defensively
    const int a = min(max(__ldg(ia + i), 0), p.Tv - 1);
    const int b = min(max(__ldg(ib + i), 0), p.Tv - 1);
    atomicOr(&ma[a >> 5], 1u << (a & 31));
    atomicOr(&mb[b >> 5], 1u << (b & 31));
  }
  __syncwarp();
  const uint32_t A = ma[lane], B = mb[lane];
  const uint32_t m_sh = A & B, m_ao = A & ~B, m_bo = B & ~A;
  // exclusive prefix counts over the lanes (tiles below this lane's 32)
  int e_sh = __popc(m_sh), e_ao = __popc(m_ao), e_bo = __popc(m_bo);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, e_sh, o);
    const int y = __shfl_up_sync(0xffffffffu, e_ao, o);
    const int z = __shfl_up_sync(0xffffffffu, e_bo, o);
    if (lane >= o) {
      e_sh += x;
      e_ao += y;
      e_bo += z;
    }
  }
  const int n_sh = __shfl_sync(0xffffffffu, e_sh, 31);
  const int n_ao = __shfl_sync(0xffffffffu, e_ao, 31);
  const int n_bo = __shfl_sync(0xffffffffu, e_bo, 31);
  e_sh -= __popc(m_sh);
  e_ao -= __popc(m_ao);
  e_bo -= __popc(m_bo);
  const int n_shared = (n_sh + 1) / 2;
  const int n_routed = max(n_ao, n_bo);  // equal unless the router repeated an index
  const int base_r = n_dense + n_shared;
  // empty halves (entry 0: row 0, no keys): the Y of an odd last shared step, and routed
  // halves without a partner
  if (lane == 0 && (n_sh & 1)) list[base_r - 1].y = 0;
  for (int i = lane; i < n_routed; i += 32) list[base_r + i] = make_int2(0, 0);
  __syncwarp();
  int* words = reinterpret_cast<int*>(list);
  auto put = [&](uint32_t m, int k, int at, int stride, int flag) {
    while (m) {
      const int t = lane * 32 + __ffs(m) - 1;
      m &= m - 1;
      int f, c;
      tile_span(p.geom, t, &f, &c);
      words[at + k * stride] = (f << 9) | (c << 2) | flag;
      ++k;
    }
  };
  put(m_sh, e_sh, 2 * n_dense, 1, 1);     // shared k -> step n_dense + k/2, X or Y
  put(m_ao, e_ao, 2 * base_r, 2, 0);      // only a: X of routed step k
  put(m_bo, e_bo, 2 * base_r + 1, 2, 0);  // only b: Y of routed step k
  return base_r + n_routed;
}

// 2^e for a whole number e <= 0 (or -inf), exactly: the rescale factor between two
// running maxima that are both whole octaves; 0 below the normal range.
__device__ __forceinline__ float octave(float e) {
  return e < -126.0f ? 0.0f : __int_as_float((127 + (int)e) << 23);
}

// max of three fp32 values in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 32 lanes x 32 columns of TMEM <- 0 (no wait; the P store that follows waits for both)
__device__ __forceinline__ void tmem_zero32(uint32_t taddr) {
  const uint32_t z = 0;
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,"
      "%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1};" ::"r"(taddr),
      "r"(z)
      : "memory");
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

// Masks scores j >= c (warp-uniform c) and returns the max of the 64 values.
__device__ __forceinline__ float masked_max64(float* sv, int c) {
  if (c < 64) {
#pragma unroll
    for (int j = 0; j < 64; ++j) sv[j] = j < c ? sv[j] : -INFINITY;
  }
  float mx4[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) mx4[u] = -INFINITY;
#pragma unroll
  for (int j = 0; j < 64; j += 2) mx4[(j >> 1) & 3] = fmax3(mx4[(j >> 1) & 3], sv[j], sv[j + 1]);
  return fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
}

// P = exp2(s * scale - m) for 64 scores: bf16 pairs into pk, returns the unrounded sum.
// The scale-and-shift and the sums run two lanes of fp32 per instruction.
__device__ __forceinline__ float exp_pack64(const float* sv, float sl2, float m_use,
                                            uint32_t* pk) {
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
  return ((ls2[0].x + ls2[0].y) + (ls2[1].x + ls2[1].y)) +
         ((ls2[2].x + ls2[2].y) + (ls2[3].x + ls2[3].y));
}

template <int HD>
__global__ void __launch_bounds__(THREADS, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmQ, const Params p) {
  using L = Layout<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int2* lists = reinterpret_cast<int2*>(smem + L::LIST_OFF);
  float* lbuf = reinterpret_cast<float*>(smem + L::LBUF_OFF);
  volatile int* unit_w = reinterpret_cast<volatile int*>(smem + L::UNIT_OFF);
  volatile int* unit_n = unit_w + 2;  // step counts of the units on list buffers 0 and 1
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* k_full = bars + 0;      // [NSK] K stage landed
  uint64_t* k_free = bars + 3;      // [NSK] the stage's S MMAs completed
  uint64_t* v_full = bars + 6;      // [NSV] V stage landed
  uint64_t* v_free = bars + 8;      // [NSV] the stage's PV MMAs completed (O stable)
  uint64_t* s_done = bars + 10;     // [NSB] S of the step is in its buffer
  uint64_t* p_full = bars + 13;     // [NSB] P of the step written (four softmax warps)
  uint64_t* s_free = bars + 16;     // [NSB] the step's PV completed: its score buffer is free
  uint64_t* list_full = bars + 19;  // [2] unit number and step list written
  uint64_t* o_full = bars + 21;     // the unit's last PV completed
  uint64_t* o_free = bars + 22;     // O and the row sums read (four epilogue warps)
  uint64_t* l_ready = bars + 23;    // the row sums are in lbuf (four softmax warps)
  uint64_t* q_full = bars + 24;     // the unit's Q landed in shared memory
  uint64_t* q_free = bars + 25;     // the unit's S MMAs completed: Q may be overwritten
  uint64_t* drain = bars + 26;      // [2] per issuing thread
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 28);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int b = 0; b < NSK; ++b) {
      mbar_init(&k_full[b], 1);
      mbar_init(&k_free[b], 1);
    }
    for (int b = 0; b < NSV; ++b) {
      mbar_init(&v_full[b], 1);
      mbar_init(&v_free[b], 1);
    }
    for (int b = 0; b < NSB; ++b) {
      mbar_init(&s_done[b], 1);
      mbar_init(&p_full[b], 4);
      mbar_init(&s_free[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&drain[b], 1);
      mbar_init(&list_full[b], 1);
    }
    mbar_init(o_full, 1);
    mbar_init(o_free, 4);
    mbar_init(l_ready, 4);
    mbar_init(q_full, 1);
    mbar_init(q_free, 1);
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

  if (warp == 0 || warp == 6) {
    // ------------------------------------------------------------ TMA producers
    if (lane == 0) {
      const bool is_k = warp == 0;
      const CUtensorMap* tm = is_k ? &tmK : &tmV;
      prefetch_tmap(tm);
      if (is_k) prefetch_tmap(&tmQ);
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* freed = is_k ? k_free : v_free;
      uint8_t* ring = smem + (is_k ? L::K_OFF : L::V_OFF);
      const int nst = is_k ? NSK : NSV;
      int st = 0;        // ring stage and phase of the next load
      uint32_t ph = 0;
      int issued = 0;
      int q_loads = 0;   // (K producer) Q loads issued
      bool ok = true;
      for (int lj = 0; ok; ++lj) {
        const int lb = lj & 1;
        if (!mbar_wait(&list_full[lb], (lj >> 1) & 1, abort_flag, p.status)) break;
        const int w = unit_w[lb];
        if (w >= p.total) break;
        const Unit u = unit_of(p, w);
        const int2* list = lists + lb * MAX_STEPS;
        const int n = unit_n[lb];
        // (K producer) the unit's Q goes into the one Q buffer once the previous unit's
        // score MMAs have completed; until then the unit's K loads go ahead, and every
        // wait below polls for that moment
        bool q_pending = is_k;
        auto try_q = [&]() {
          if (!q_pending) return;
          if (lj > 0 && !mbar_try_wait(smem_u32(q_free), (uint32_t)(lj - 1) & 1u)) return;
          int rx, ry;  // first rows of the unit's two 64-row query blocks
          if (u.prefix) {
            rx = u.unit * 128;
            ry = rx + 64;
          } else {
            int c;
            tile_span(p.geom, u.ta, &rx, &c);
            // an odd tile count leaves the last unit's second half without a tile: it
            // repeats a
            if (u.tb < p.Tv)
              tile_span(p.geom, u.tb, &ry, &c);
            else
              ry = rx;
          }
          uint8_t* qs = smem + L::Q_OFF;
          mbar_arrive_expect_tx(q_full, L::STAGE);
#pragma unroll
          for (int ch = 0; ch < HD / 64; ++ch) {
            tma_load_3d(qs + 2 * ch * L::KCHUNK, &tmQ, q_full, 64 * ch, rx, u.h);
            tma_load_3d(qs + (2 * ch + 1) * L::KCHUNK, &tmQ, q_full, 64 * ch, ry, u.h);
          }
          ++q_loads;
          q_pending = false;
        };
        for (int t = 0; t < n; ++t) {
          // wait for the stage to be free (bounded), polling for the Q buffer meanwhile
          const uint32_t fa = smem_u32(&freed[st]);
          if (!mbar_try_wait(fa, ph ^ 1)) {
            const unsigned long long t0 = global_ns();
            while (true) {
              try_q();
              bool done = false;
              for (int i = 0; i < 64 && !done; ++i) done = mbar_try_wait(fa, ph ^ 1);
              if (done) break;
              if (*abort_flag || global_ns() - t0 > kWaitLimitNs) {
                if (!*abort_flag) {
                  *abort_flag = 1;
                  if (p.status) atomicExch(p.status, kStatusTimeout);
                }
                ok = false;
                break;
              }
            }
            if (!ok) break;
          }
          try_q();
          const int2 e = list[t];
          uint8_t* s = ring + st * L::STAGE;
          mbar_arrive_expect_tx(&full[st], L::STAGE);
#pragma unroll
          for (int ch = 0; ch < HD / 64; ++ch) {
            tma_load_3d(s + 2 * ch * L::KCHUNK, tm, &full[st], 64 * ch, e.x >> 9, u.h);
            tma_load_3d(s + (2 * ch + 1) * L::KCHUNK, tm, &full[st], 64 * ch, e.y >> 9, u.h);
          }
          ++issued;
          if (++st == nst) {
            st = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        // a unit whose K loads all went ahead still needs its Q
        if (q_pending) {
          if (lj > 0 && !mbar_wait(q_free, (uint32_t)(lj - 1) & 1u, abort_flag, p.status)) break;
          try_q();
        }
      }
      // wait (bounded) for the last load into each stage, and the last Q load, before the
      // CTA exits (already complete unless the CTA is aborting)
      for (int i = issued > nst ? issued - nst : 0; i < issued; ++i)
        mbar_drain(&full[i % nst], (i / nst) & 1);
      if (q_loads > 0) mbar_drain(q_full, (uint32_t)(q_loads - 1) & 1u);
    }
  } else if (warp == 1 || warp == 11) {
    // ------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      const bool is_s = warp == 1;
      const int nst = is_s ? NSK : NSV;
      uint32_t g = 0;  // steps issued, across units
      int sb = 0;      // score buffer of step g (g mod NSB) and its use count parity
      uint32_t sph = 0;
      int st = 0;      // K (S issuer) or V (PV issuer) ring stage and phase
      uint32_t ph = 0;
      bool ok = true;
      for (int lj = 0; ok; ++lj) {
        const int lb = lj & 1;
        if (!mbar_wait(&list_full[lb], (lj >> 1) & 1, abort_flag, p.status)) break;
        const int w = unit_w[lb];
        if (w >= p.total) break;
        const int n = unit_n[lb];
        for (int t = 0; t < n; ++t, ++g) {
          if (is_s) {
            // S of step g: Q of the unit, K of the step, and a score buffer the PV of step
            // g - 3 has finished reading
            if (t == 0 && !mbar_wait(q_full, (uint32_t)lj & 1u, abort_flag, p.status)) {
              ok = false;
              break;
            }
            if (!mbar_wait(&k_full[st], ph, abort_flag, p.status) ||
                !mbar_wait(&s_free[sb], sph ^ 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
            const uint64_t kd =
                sdesc_sw128(smem_u32(smem + L::K_OFF + st * L::STAGE), 16, 1024);
            const uint64_t qd = sdesc_sw128(smem_u32(smem + L::Q_OFF), 16, 1024);
#pragma unroll
            for (int ks = 0; ks < HD / 16; ++ks) {
              // dims 16ks..16ks+15: 32-byte step within a 64-dim chunk of Q and of K
              const uint32_t koff = (ks >> 2) * 2 * L::KCHUNK + (ks & 3) * 32;
              umma_bf16(tmem + L::S_COL + sb * 128, qd + (koff >> 4), kd + (koff >> 4), idesc_s,
                        ks > 0 ? 1u : 0u);
            }
            umma_commit(&s_done[sb]);
            umma_commit(&k_free[st]);
            if (t == n - 1) umma_commit(q_free);  // the unit's last read of Q
          } else {
            // PV of step g: O read out of the previous unit, P of the step, V of the step
            if (t == 0 && !mbar_wait(o_free, (lj & 1) ^ 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            if (!mbar_wait(&p_full[sb], sph, abort_flag, p.status) ||
                !mbar_wait(&v_full[st], ph, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            constexpr uint32_t idesc_pv = idesc_bf16(128, HD, false, true);
            const uint64_t vd =
                sdesc_sw128(smem_u32(smem + L::V_OFF + st * L::STAGE), 2 * L::KCHUNK, 1024);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              // P: keys 16ks..16ks+15 of the step are columns 8ks..8ks+7 of its S buffer;
              // V: block ks / 4 (X or Y), MN-major, LBO = next 64-dim chunk, SBO = next 8 keys
              const uint32_t voff = (ks >> 2) * L::KCHUNK + (ks & 3) * 2048;
              umma_bf16_ts(tmem + L::O_COL, tmem + L::S_COL + sb * 128 + ks * 8, vd + (voff >> 4),
                           idesc_pv, (t > 0 || ks > 0) ? 1u : 0u);
            }
            umma_commit(&s_free[sb]);
            umma_commit(&v_free[st]);
            if (t == n - 1) umma_commit(o_full);
          }
          if (++st == nst) {
            st = 0;
            ph ^= 1;
          }
          if (++sb == NSB) {
            sb = 0;
            sph ^= 1;
          }
        }
      }
      umma_commit(&drain[is_s ? 0 : 1]);
      mbar_drain(&drain[is_s ? 0 : 1], 0);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int half = row >> 6;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t o_addr = t_lane + L::O_COL;
    const float sl2 = p.scale_log2;
    uint32_t g = 0;
    int sb = 0;    // score buffer of step g (g mod NSB) and its use count parity
    uint32_t sph = 0;
    int v_st = 0;  // V stage and phase of step g (the rescale waits on step g - 1's PV)
    uint32_t v_ph = 0;
    int pv_st = 0;
    uint32_t pv_ph = 0;
    bool ok = true;
    for (int lj = 0; ok; ++lj) {
      const int lb = lj & 1;
      if (!mbar_wait(&list_full[lb], (lj >> 1) & 1, abort_flag, p.status)) break;
      const int w = unit_w[lb];
      if (w >= p.total) break;
      const int n = unit_n[lb];
      const int2* list = lists + lb * MAX_STEPS;
      float m_run = -INFINITY;
      float l_run = 0.f;
      for (int t = 0; t < n; ++t, ++g) {
        if (!mbar_wait(&s_done[sb], sph, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int2 e = list[t];
        const uint32_t s_addr = t_lane + L::S_COL + sb * 128;
        float sv[128];
        uint32_t pk[32];
        float mx, lsum, alpha;
        bool need;
        if (e.x & 1) {
          // dense: every row uses X (columns 0-63) and Y (64-127), read in one load
          const int cx = (e.x >> 2) & 127, cy = (e.y >> 2) & 127;
          float my = -INFINITY;
          if (cy > 0) {
            tmem_ld128(s_addr, sv);
            my = masked_max64(sv + 64, cy);
          } else {
            tmem_ld64(s_addr, sv);
          }
          mx = fmaxf(masked_max64(sv, cx), my) * sl2;
          need = mx > m_run + kRescaleLog2;
          const float m_new = need ? ceilf(mx) : m_run;
          alpha = need ? octave(m_run - m_new) : 1.0f;
          const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
          m_run = m_new;
          lsum = exp_pack64(sv, sl2, m_use, pk);
          if (cy == 0) tmem_zero32(s_addr + 32);  // no Y keys
          tmem_st32_u(s_addr, pk);  // P_X over S columns 0-31 (already read)
          if (cy > 0) {
            lsum += exp_pack64(sv + 64, sl2, m_use, pk);  // masked scores are -inf
            tmem_st32_u(s_addr + 32, pk);  // P_Y over S columns 32-63 (already read)
          }
        } else {
          // routed: rows 0-63 use X (columns 0-63), rows 64-127 use Y (64-127)
          const int c = ((half ? e.y : e.x) >> 2) & 127;
          tmem_ld64(s_addr + half * 64, sv);
          mx = masked_max64(sv, c) * sl2;
          need = mx > m_run + kRescaleLog2;
          const float m_new = need ? ceilf(mx) : m_run;
          alpha = need ? octave(m_run - m_new) : 1.0f;
          const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
          m_run = m_new;
          lsum = exp_pack64(sv, sl2, m_use, pk);
          tmem_zero32(s_addr + (half ^ 1) * 32);  // the other block's keys
          tmem_st32_u(s_addr + half * 32, pk);
        }
        if (t > 0 && __any_sync(0xffffffffu, need)) {
          // O must not change under a rescale while the previous step's PV runs
          if (!mbar_wait(&v_free[pv_st], pv_ph, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          rescale_rows<HD>(o_addr, alpha);
        }
        l_run = fmaf(l_run, alpha, lsum);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[sb]);
        pv_st = v_st;
        pv_ph = v_ph;
        if (++v_st == NSV) {
          v_st = 0;
          v_ph ^= 1;
        }
        if (++sb == NSB) {
          sb = 0;
          sph ^= 1;
        }
      }
      if (!ok) break;
      // hand the row sums over once the epilogue has read the previous unit's
      if (!mbar_wait(o_free, (lj & 1) ^ 1, abort_flag, p.status)) break;
      lbuf[row] = l_run;
      __syncwarp();
      if (lane == 0) mbar_arrive(l_ready);
    }
  } else if (warp >= 7 && warp <= 10) {
    // ------------------------------------------------------------ epilogue, scheduler
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int half = row >> 6;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    const bool sched = warp == 7;
    bool ended = false;  // (warp 7) the end of the unit sequence has been published
    uint32_t* masks = reinterpret_cast<uint32_t*>(smem + L::MASK_OFF);
    auto publish = [&](int buf, int w) {
      const int n =
          w < p.total ? build_list(p, unit_of(p, w), lists + buf * MAX_STEPS, masks, lane) : 0;
      if (lane == 0) {
        unit_w[buf] = w;
        unit_n[buf] = n;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&list_full[buf]);
      if (w >= p.total) ended = true;
    };
    int end_at = 1 << 30;  // first unit index known to be past the end
    int wc0 = 0, wc1 = 0;  // units on list buffers 0 and 1
    bool ok = true;
    if (sched) {
      publish(0, blockIdx.x);
      if (!ended) publish(1, gridDim.x + blockIdx.x);
    }
    for (int b = 0; b < 2 && ok; ++b) {
      if (!mbar_wait(&list_full[b], 0, abort_flag, p.status)) {
        ok = false;
        break;
      }
      const int w = unit_w[b];
      if (b) wc1 = w; else wc0 = w;
      if (w >= p.total) {
        end_at = b;
        break;
      }
    }
    const int A = p.H * HD;
    for (int lj = 0; ok && lj < end_at; ++lj) {
      const int ob = lj & 1;
      const Unit u = unit_of(p, ob ? wc1 : wc0);
      if (!mbar_wait(o_full, lj & 1, abort_flag, p.status)) break;
      if (!mbar_wait(l_ready, lj & 1, abort_flag, p.status)) break;
      tc_fence_after();
      const float l = lbuf[row];
      float o[HD];
      if constexpr (HD == 128)
        tmem_ld128(t_lane + L::O_COL, o);
      else
        tmem_ld64(t_lane + L::O_COL, o);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);  // O and lbuf may take the next unit
      int grow, tile = -1;
      bool store;
      if (u.prefix) {
        grow = u.unit * 128 + row;
        store = grow < p.n_prefix;
      } else {
        tile = half ? u.tb : u.ta;
        int f = 0, c = 0;
        if (tile < p.Tv) tile_span(p.geom, tile, &f, &c);
        grow = f + (row & 63);
        store = (row & 63) < c;
      }
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      const bool mix = !u.prefix && p.gate != nullptr && p.pooled != nullptr;
      if (store) {
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          float* oc = o + 32 * c;
#pragma unroll
          for (int j = 0; j < 32; ++j) oc[j] *= inv_l;
          if (mix) {
            const uint4* g4 =
                reinterpret_cast<const uint4*>(p.gate + (size_t)grow * A + u.h * HD + c * 32);
            const float4* pb4 = reinterpret_cast<const float4*>(
                p.pooled + ((size_t)u.h * p.Tv + tile) * HD + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 gv = __ldg(g4 + i);
              const float4 b0 = __ldg(pb4 + 2 * i), b1 = __ldg(pb4 + 2 * i + 1);
              oc[8 * i + 0] = fmaf(bf16_lo(gv.x), b0.x, oc[8 * i + 0]);
              oc[8 * i + 1] = fmaf(bf16_hi(gv.x), b0.y, oc[8 * i + 1]);
              oc[8 * i + 2] = fmaf(bf16_lo(gv.y), b0.z, oc[8 * i + 2]);
              oc[8 * i + 3] = fmaf(bf16_hi(gv.y), b0.w, oc[8 * i + 3]);
              oc[8 * i + 4] = fmaf(bf16_lo(gv.z), b1.x, oc[8 * i + 4]);
              oc[8 * i + 5] = fmaf(bf16_hi(gv.z), b1.y, oc[8 * i + 5]);
              oc[8 * i + 6] = fmaf(bf16_lo(gv.w), b1.z, oc[8 * i + 6]);
              oc[8 * i + 7] = fmaf(bf16_hi(gv.w), b1.w, oc[8 * i + 7]);
            }
          }
          uint4* dst = reinterpret_cast<uint4*>(p.out + (size_t)grow * A + u.h * HD + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            dst[i] = make_uint4(pack_bf16x2(oc[8 * i + 0], oc[8 * i + 1]),
                                pack_bf16x2(oc[8 * i + 2], oc[8 * i + 3]),
                                pack_bf16x2(oc[8 * i + 4], oc[8 * i + 5]),
                                pack_bf16x2(oc[8 * i + 6], oc[8 * i + 7]));
          }
        }
      }
      // unit lj + 2 takes this list buffer once all four warps are done with unit lj
      // (every reader of its list finished before o_full)
      if (sched && !ended) {
        if (!mbar_wait(o_free, lj & 1, abort_flag, p.status)) break;
        int w2 = 0;
        if (lane == 0) w2 = 2 * (int)gridDim.x + atomicAdd(p.counter, 1);
        publish(ob, __shfl_sync(0xffffffffu, w2, 0));
      }
      if (lj + 1 < end_at) {  // unit lj + 1 exists, so unit lj + 2 (or the end) is published
        if (!mbar_wait(&list_full[ob], ((lj + 2) >> 1) & 1, abort_flag, p.status)) break;
        const int w2 = unit_w[ob];
        if (ob) wc1 = w2; else wc0 = w2;
        if (w2 >= p.total) end_at = lj + 2;
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
  CUtensorMap tk, tv, tq;
  if (!make_tmap_3d(&tk, a.k, a.H, a.N, HD) || !make_tmap_3d(&tv, a.v, a.H, a.N, HD) ||
      !make_tmap_3d(&tq, a.q, a.H, a.N, HD))
    return cudaErrorInvalidValue;
  Params p;
  p.N = a.N;
  p.H = a.H;
  p.n_prefix = a.n_prefix;
  p.Tv = a.Tv;
  p.ksel = a.ksel;
  p.n_pre_units = (a.n_prefix + 127) / 128;
  p.n_vid_units = (a.Tv + 1) / 2;
  p.total = (p.n_pre_units + p.n_vid_units) * a.H;
  p.steps_all = (a.N + 127) / 128;
  p.steps_pre = (a.n_prefix + 127) / 128;
  if (p.steps_all > MAX_STEPS || p.steps_pre + a.ksel > MAX_STEPS) return cudaErrorInvalidValue;
  p.geom = a.geom;
  p.q = a.q;
  p.idx = a.idx;
  p.gate = a.gate;
  p.pooled = a.pooled;
  p.out = a.out;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)HD));
  p.status = a.status;
  p.counter = a.counter;
  auto kern = attention_kernel<HD>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  const int grid = p.total < num_sms() ? p.total : num_sms();
  kern<<<grid, THREADS, L::SMEM, stream>>>(tk, tv, tq, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream) {
  if (a.N <= 0 || a.H <= 0 || a.N > MAX_STEPS * 128 || a.counter == nullptr)
    return cudaErrorInvalidValue;
  if (a.d == 128) return launch_hd<128>(a, stream);
  if (a.d == 64) return launch_hd<64>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace h3
