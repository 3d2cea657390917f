// router.cu -- tile means, tile scores, top-k selection and the pooled branch.
//
// TensorFold #949, "What it adds" (h3_routing.metal: tile means, tile scores,
// top-k and the pooled branch), "Precision" (fp32 tile means, scores, top-k and
// pooled branch) and "Kernel contract" (a NaN score ranks as -inf; ties go to
// the lower tile; a row never keeps more than k tiles).
//
// Kernel 1 (tile_means): one CTA per (video tile, head, tensor of q/k/v); four
//   warps sum 16-row blocks of the tile's rows (a contiguous run of at most 64
//   rows: a 64-row slice, or a clipped 4x4x4 cube) in row order, the block sums
//   are added in order and divided by the tile's row count.  Reads each
//   video row of q, k, v once (HBM-bound).
// Kernel 2 (route): one CTA per (head h, 32 query tiles), four query tiles per
//   warp; the head's key / value tile means pass through shared memory once
//   per CTA in chunks of 32 tiles, and each staged mean a lane reads serves the
//   warp's four query tiles (the kernel is bound by shared-memory bandwidth):
//   S[h,i,j] = sum_c mq[h,i,c] mk[h,j,c]: one lane per key tile, four
//   interleaved partial sums over c (c mod 4) added as ((p0 + p1) + (p2 + p3)),
//   operands read from shared memory 16 bytes at a time;
//   top-k under the total order (score descending, tile index ascending), NaN
//   ranking as -inf: the k-th largest order key found bit by bit with warp
//   reductions, then every larger key and the lowest-index equal keys -- the same
//   set as "rank_j < k" with rank_j = #{j' : s_j' > s_j or (s_j' == s_j and j' < j)};
//   kept tiles are written ascending (ballots);
//   pooled[h,i,:] = sum_j softmax_j(S[h,i,j] / sqrt(d)) mv[h,j,:]: max and
//   denominator by fixed warp reductions, the weighted sum in j order.
// Every reduction has a fixed order, so results are deterministic.
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace h3 {

namespace {

constexpr int ROUTE_THREADS = 256;

// One CTA (4 warps) per (video tile, head, tensor); warp w sums rows 16w..16w+15
// of the tile in row order, lane l holding columns l*D/32 .. (l+1)*D/32 - 1;
// the four partial sums are added in warp order.
template <int D>
__global__ void __launch_bounds__(128)
    tile_means_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                      const __nv_bfloat16* __restrict__ v, float* __restrict__ means, int N, int H,
                      const TileGeom geom, int Tv, int* __restrict__ counter) {
  constexpr int CPL = D / 32;  // columns per lane: 4 (d = 128) or 2 (d = 64)
  __shared__ float part[4][D];
  const int t = blockIdx.x, h = blockIdx.y, which = blockIdx.z;
  // the attention kernel, which runs after the router, fetches work units from this counter
  if ((t | h | which | threadIdx.x) == 0 && counter != nullptr) *counter = 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const __nv_bfloat16* X = which == 0 ? q : (which == 1 ? k : v);
  int r0, nv;
  tile_span(geom, t, &r0, &nv);
  const int ra = warp * 16, rb = min(nv, ra + 16);
  float acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
  const __nv_bfloat16* src = X + ((size_t)h * N + r0) * D + lane * CPL;
  int r = ra;
  for (; r + 4 <= rb; r += 4) {  // four rows in flight, summed in row order
    uint32_t w[4][CPL / 2];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (CPL == 4) {
        const uint2 x = __ldg(reinterpret_cast<const uint2*>(src + (size_t)(r + u) * D));
        w[u][0] = x.x;
        w[u][CPL / 2 - 1] = x.y;
      } else {
        w[u][0] = __ldg(reinterpret_cast<const unsigned int*>(src + (size_t)(r + u) * D));
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll
      for (int c = 0; c < CPL / 2; ++c) {
        acc[2 * c] += bf16_lo(w[u][c]);
        acc[2 * c + 1] += bf16_hi(w[u][c]);
      }
    }
  }
  for (; r < rb; ++r) {
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] += __bfloat162float(src[(size_t)r * D + c]);
  }
#pragma unroll
  for (int c = 0; c < CPL; ++c) part[warp][lane * CPL + c] = acc[c];
  __syncthreads();
  for (int c = threadIdx.x; c < D; c += 128) {
    const float tot = ((part[0][c] + part[1][c]) + part[2][c]) + part[3][c];
    means[(((size_t)which * H + h) * Tv + t) * D + c] = tot / (float)nv;
  }
}

constexpr int TILES_PER_WARP = 4;  // query tiles per warp: each staged mean read serves 4
constexpr int TILES_PER_CTA = ROUTE_THREADS / 32 * TILES_PER_WARP;
constexpr int KCHUNK = 32;  // key-tile means staged per round
constexpr int SPAD = 4;  // staged row padding (floats): conflict-free 16-byte column reads

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Order key of a score for the top-k: a larger key ranks first; NaN ranks as -inf and
// -0 equals +0 (the float comparison's view), so equal keys are exactly the ties.
__device__ __forceinline__ uint32_t order_key(float x) {
  float v = isnan(x) ? -INFINITY : x;
  if (v == 0.f) v = 0.f;
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Top-k of one query tile's scores s[0, Tv) by one warp; lane l owns tiles l + 32m, m < NM,
// and gets bit m of `taken` set for each of its selected tiles.  T = the ksel-th largest
// order key, found bit by bit (the largest T with #{key >= T} >= ksel); every tile with a
// key above T is selected, then those equal to T in ascending tile order until ksel --
// the ksel first tiles of the total order (score descending, tile ascending).
template <int NM>
__device__ __forceinline__ unsigned select_topk(const float* s, int Tv, int ksel, int lane) {
  uint32_t u[NM];
  unsigned valid = 0u;
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    const int j = lane + 32 * m;
    u[m] = j < Tv ? order_key(s[j]) : 0u;
    if (j < Tv) valid |= 1u << m;
  }
  uint32_t T = 0u;
#pragma unroll 1
  for (int b = 31; b >= 0; --b) {
    const uint32_t cand = T | (1u << b);
    int c = 0;
#pragma unroll
    for (int m = 0; m < NM; ++m) c += (((valid >> m) & 1u) && u[m] >= cand) ? 1 : 0;
    if (__reduce_add_sync(0xffffffffu, c) >= ksel) T = cand;
  }
  unsigned taken = 0u;
  int gt = 0;
#pragma unroll
  for (int m = 0; m < NM; ++m)
    if (((valid >> m) & 1u) && u[m] > T) {
      taken |= 1u << m;
      ++gt;
    }
  int need = ksel - __reduce_add_sync(0xffffffffu, gt);
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    if (need <= 0) break;  // warp-uniform
    const bool eq = ((valid >> m) & 1u) && u[m] == T;
    const unsigned bal = __ballot_sync(0xffffffffu, eq);
    if (eq && __popc(bal & ((1u << lane) - 1u)) < need) taken |= 1u << m;
    need -= __popc(bal);
  }
  return taken;
}

// One CTA per (head h, block of 32 query tiles); warp w owns query tiles
// i = 32 * blockIdx.x + 4 * w + r, r < 4.  The head's key and value tile means are
// staged through shared memory once per CTA; every staged mean a lane reads serves the
// warp's four query tiles (shared-memory bandwidth is what bounds this kernel).
// NM: 32-tile groups per lane in the top-k (Tv <= 32 * NM).
template <int D, int NM>
__global__ void __launch_bounds__(ROUTE_THREADS)
    route_kernel(const float* __restrict__ means, float* __restrict__ scores,
                 int* __restrict__ idx, float* __restrict__ pooled, int H, int Tv, int ksel) {
  constexpr int R = TILES_PER_WARP;
  extern __shared__ __align__(16) float sh[];
  float* stage = sh;                                  // [KCHUNK][D + SPAD] staged means
  float* qrow = stage + KCHUNK * (D + SPAD);          // [32][D] query means, 4 rows per warp
  float* srow = qrow + TILES_PER_CTA * D;             // [32][Tv4] scores, then pooled weights
  const int Tv4 = (Tv + 3) & ~3;                      // row stride: 16-byte aligned rows
  const int h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i0 = blockIdx.x * TILES_PER_CTA + warp * R;  // the warp's first query tile
  const float* mQ = means + ((size_t)0 * H + h) * Tv * D;
  const float* mK = means + ((size_t)1 * H + h) * Tv * D;
  const float* mV = means + ((size_t)2 * H + h) * Tv * D;
  constexpr int D4 = D / 4;  // float4 lanes per row (<= 32)
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float* mq = qrow + (warp * R + r) * D;
    for (int c = lane; c < D; c += 32) mq[c] = i0 + r < Tv ? mQ[(size_t)(i0 + r) * D + c] : 0.f;
  }
  // scores: stage 32 key means (row stride D + 4 floats: 16-byte column reads are
  // conflict-free), then lane l of each warp computes the whole dot product of key tile
  // j0 + l with each of its four query tiles, four interleaved partial sums over the
  // dimensions (c mod 4) per product, added as ((p0 + p1) + (p2 + p3)); the key mean is
  // read once per 16-byte step for the four products, the query means by broadcast
  for (int j0 = 0; j0 < Tv; j0 += KCHUNK) {
    const int nj = min(KCHUNK, Tv - j0);
    __syncthreads();
    for (int e = threadIdx.x; e < nj * D4; e += ROUTE_THREADS)
      reinterpret_cast<float4*>(stage + (e / D4) * (D + SPAD))[e % D4] =
          __ldg(reinterpret_cast<const float4*>(mK + (size_t)j0 * D) + e);
    __syncthreads();
    if (i0 < Tv && lane < nj) {
      const float4* kr = reinterpret_cast<const float4*>(stage + lane * (D + SPAD));
      const float4* q4 = reinterpret_cast<const float4*>(qrow + warp * R * D);
      float a[R][4];
#pragma unroll
      for (int r = 0; r < R; ++r) a[r][0] = a[r][1] = a[r][2] = a[r][3] = 0.f;
#pragma unroll 4
      for (int c = 0; c < D4; ++c) {
        const float4 y = kr[c];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float4 x = q4[r * D4 + c];
          a[r][0] = fmaf(x.x, y.x, a[r][0]);
          a[r][1] = fmaf(x.y, y.y, a[r][1]);
          a[r][2] = fmaf(x.z, y.z, a[r][2]);
          a[r][3] = fmaf(x.w, y.w, a[r][3]);
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r)
        srow[(warp * R + r) * Tv4 + j0 + lane] = (a[r][0] + a[r][1]) + (a[r][2] + a[r][3]);
    }
  }
  __syncwarp();
  // top-k of each of the warp's query tiles under the total order (score desc, index asc),
  // NaN ranking as -inf; selected tiles are then written in ascending order via ballots
  for (int r = 0; r < R; ++r) {
    const int i = i0 + r;
    if (i >= Tv) break;  // warp-uniform
    const float* s = srow + (warp * R + r) * Tv4;
    float* srow_out = scores + ((size_t)h * Tv + i) * Tv;
    for (int j = lane; j < Tv; j += 32) srow_out[j] = s[j];
    int* out = idx + ((size_t)h * Tv + i) * ksel;
    unsigned taken = 0u;
    if (ksel >= Tv) {
      for (int m = 0; lane + 32 * m < Tv; ++m) taken |= 1u << m;
    } else {
      taken = select_topk<NM>(s, Tv, ksel, lane);
    }
    int base = 0;
    for (int m = 0; 32 * m < Tv; ++m) {
      const bool keep = (taken >> m) & 1u;
      const unsigned bal = __ballot_sync(0xffffffffu, keep);
      const int pos = base + __popc(bal & ((1u << lane) - 1u));
      if (keep && pos < ksel) out[pos] = lane + 32 * m;
      base += __popc(bal);
    }
  }
  if (!pooled) return;
  // pooled branch: softmax over all video tiles of S / sqrt(D), then weights . mean(v)
  float inv_sum[R];
  const float sc = 1.0f / sqrtf((float)D);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    inv_sum[r] = 0.f;
    if (i0 + r < Tv) {
      float* s = srow + (warp * R + r) * Tv4;
      float mx = -INFINITY;
      for (int j = lane; j < Tv; j += 32) mx = fmaxf(mx, s[j] * sc);
      mx = warp_max(mx);
      float sum = 0.f;
      for (int j = lane; j < Tv; j += 32) {
        const float e = expf(s[j] * sc - mx);
        s[j] = e;  // the scores row becomes the weights row
        sum += e;
      }
      inv_sum[r] = 1.0f / warp_sum(sum);
    }
  }
  __syncwarp();
  float4 acc[R];
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* wrow = srow + warp * R * Tv4;
  for (int j0 = 0; j0 < Tv; j0 += KCHUNK) {
    const int nj = min(KCHUNK, Tv - j0);
    __syncthreads();
    for (int e = threadIdx.x; e < nj * D4; e += ROUTE_THREADS)
      reinterpret_cast<float4*>(stage)[e] = __ldg(reinterpret_cast<const float4*>(mV + (size_t)j0 * D) + e);
    __syncthreads();
    if (i0 < Tv && lane < D4) {
      int jj = 0;
      for (; jj + 4 <= nj; jj += 4) {  // j order; four weights per 16-byte read
        float w[R][4];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float4 w4 = *reinterpret_cast<const float4*>(wrow + r * Tv4 + j0 + jj);
          w[r][0] = w4.x;
          w[r][1] = w4.y;
          w[r][2] = w4.z;
          w[r][3] = w4.w;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float4 v = reinterpret_cast<const float4*>(stage + (jj + u) * D)[lane];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            acc[r].x = fmaf(w[r][u], v.x, acc[r].x);
            acc[r].y = fmaf(w[r][u], v.y, acc[r].y);
            acc[r].z = fmaf(w[r][u], v.z, acc[r].z);
            acc[r].w = fmaf(w[r][u], v.w, acc[r].w);
          }
        }
      }
      for (; jj < nj; ++jj) {
        const float4 v = reinterpret_cast<const float4*>(stage + jj * D)[lane];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float w = wrow[r * Tv4 + j0 + jj];
          acc[r].x = fmaf(w, v.x, acc[r].x);
          acc[r].y = fmaf(w, v.y, acc[r].y);
          acc[r].z = fmaf(w, v.z, acc[r].z);
          acc[r].w = fmaf(w, v.w, acc[r].w);
        }
      }
    }
  }
  if (lane < D4) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (i0 + r < Tv)
        reinterpret_cast<float4*>(pooled + ((size_t)h * Tv + i0 + r) * D)[lane] =
            make_float4(acc[r].x * inv_sum[r], acc[r].y * inv_sum[r], acc[r].z * inv_sum[r],
                        acc[r].w * inv_sum[r]);
    }
  }
}

}  // namespace

cudaError_t launch_router(const RouterArgs& a, cudaStream_t stream) {
  // the top-k keeps one bit per tile in a 32-bit mask per lane: at most 1,024 video tiles
  if (a.Tv <= 0 || a.Tv > 1024 || (a.d != 64 && a.d != 128) || a.ksel <= 0)
    return cudaErrorInvalidValue;
  dim3 g1(a.Tv, a.H, 3);
  if (a.d == 128)
    tile_means_kernel<128><<<g1, 128, 0, stream>>>(a.q, a.k, a.v, a.means, a.N, a.H, a.geom,
                                                   a.Tv, a.counter);
  else
    tile_means_kernel<64><<<g1, 128, 0, stream>>>(a.q, a.k, a.v, a.means, a.N, a.H, a.geom,
                                                  a.Tv, a.counter);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t shm =
      (size_t)(KCHUNK * (a.d + SPAD) + TILES_PER_CTA * (a.d + ((a.Tv + 3) & ~3))) * 4;
  if (shm > 200 * 1024) return cudaErrorInvalidValue;
  const int nm = (a.Tv + 31) / 32;
  auto kern = a.d == 128 ? (nm <= 8 ? route_kernel<128, 8>
                                    : (nm <= 16 ? route_kernel<128, 16> : route_kernel<128, 32>))
                         : (nm <= 8 ? route_kernel<64, 8>
                                    : (nm <= 16 ? route_kernel<64, 16> : route_kernel<64, 32>));
  if (shm > 48 * 1024) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)shm);
    if (e != cudaSuccess) return e;
  }
  dim3 g2((a.Tv + TILES_PER_CTA - 1) / TILES_PER_CTA, a.H);
  kern<<<g2, ROUTE_THREADS, shm, stream>>>(a.means, a.scores, a.idx, a.pooled, a.H, a.Tv,
                                           a.ksel);
  return cudaGetLastError();
}

}  // namespace h3
