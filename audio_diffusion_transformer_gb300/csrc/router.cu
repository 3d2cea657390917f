// router.cu -- tile means, tile scores, top-k selection and the pooled branch.
//
// TensorFold #949, "What it adds" (h3_routing.metal: tile means, tile scores,
// top-k and the pooled branch), "Precision" (fp32 tile means, scores, top-k and
// pooled branch) and "Kernel contract" (a NaN score ranks as -inf; ties go to
// the lower tile; a row never keeps more than k tiles).
//
// Kernel 1 (tile_means): one CTA per (video tile, head, tensor of q/k/v),
//   thread c sums column c over the tile's valid rows in row order and divides
//   by the valid-row count.  Reads each video row of q, k, v once (HBM-bound).
// Kernel 2 (route): one CTA (8 warps) per (query tile i, head h):
//   S[h,i,j] = sum_c mq[h,i,c] mk[h,j,c]: one warp per j (four j's in flight), lane l sums dims
//   4l..4l+3 in order, then a fixed xor-shuffle tree across the lanes;
//   rank_j = #{j' : s_j' > s_j or (s_j' == s_j and j' < j)} with NaN -> -inf;
//   tile j is kept iff rank_j < k; kept tiles are written ascending;
//   pooled[h,i,:] = sum_j softmax_j(S[h,i,j] / sqrt(d)) mv[h,j,:]: max and
//   denominator by fixed block reductions, the weighted sum in j order over
//   contiguous j ranges whose partial sums are added in range order.
// Every reduction has a fixed order, so results are deterministic.
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace h3 {

namespace {

constexpr int ROUTE_THREADS = 256;

__global__ void tile_means_kernel(const __nv_bfloat16* __restrict__ q,
                                  const __nv_bfloat16* __restrict__ k,
                                  const __nv_bfloat16* __restrict__ v, float* __restrict__ means,
                                  int N, int H, int d, int n_prefix, int n_video, int Tv) {
  const int t = blockIdx.x, h = blockIdx.y, which = blockIdx.z;
  const int c = threadIdx.x;
  if (c >= d) return;
  const __nv_bfloat16* X = which == 0 ? q : (which == 1 ? k : v);
  const int r0 = n_prefix + 64 * t;
  const int nv = min(64, n_video - 64 * t);
  const __nv_bfloat16* src = X + ((size_t)h * N + r0) * d + c;
  float s = 0.f;
  int r = 0;
  for (; r + 8 <= nv; r += 8) {  // eight rows in flight, summed in row order
    float x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) x[u] = __bfloat162float(src[(size_t)(r + u) * d]);
#pragma unroll
    for (int u = 0; u < 8; ++u) s += x[u];
  }
  for (; r < nv; ++r) s += __bfloat162float(src[(size_t)r * d]);
  means[(((size_t)which * H + h) * Tv + t) * d + c] = s / (float)nv;
}

__device__ __forceinline__ float rank_key(float s) { return isnan(s) ? -INFINITY : s; }

// Fixed-order block reductions over ROUTE_THREADS threads (8 warps).
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < ROUTE_THREADS / 32; ++w) r = fmaxf(r, red[w]);
  __syncthreads();
  return r;
}

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < ROUTE_THREADS / 32; ++w) r += red[w];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(ROUTE_THREADS)
    route_kernel(const float* __restrict__ means, float* __restrict__ scores,
                 int* __restrict__ idx, float* __restrict__ pooled, int H, int d, int Tv,
                 int ksel) {
  extern __shared__ float sh[];
  float* s = sh;                               // [Tv] scores
  float* w = s + Tv;                           // [Tv] pooled weights
  int* keep = reinterpret_cast<int*>(w + Tv);  // [Tv]
  float* part = reinterpret_cast<float*>(keep + Tv);  // [ROUTE_THREADS] pooled partials
  __shared__ float red[ROUTE_THREADS / 32];
  const int i = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* mQ = means + ((size_t)0 * H + h) * Tv * d;
  const float* mK = means + ((size_t)1 * H + h) * Tv * d;
  const float* mV = means + ((size_t)2 * H + h) * Tv * d;
  // scores: one warp per key tile j; lane l holds dims 4l..4l+3 (+128 per round), then a
  // fixed xor-tree across lanes
  const int d4 = d >> 2;
  const float4* q4 = reinterpret_cast<const float4*>(mQ + (size_t)i * d);
  float4 qa = lane < d4 ? __ldg(q4 + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int NW = ROUTE_THREADS / 32;
  constexpr int U = 4;  // key tiles in flight per warp (independent loads before the reductions)
  for (int jb = warp * U; jb < Tv; jb += NW * U) {
    float acc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = jb + u;
      acc[u] = 0.f;
      if (j < Tv && lane < d4) {
        const float4 kb = __ldg(reinterpret_cast<const float4*>(mK + (size_t)j * d) + lane);
        acc[u] = fmaf(qa.x, kb.x, acc[u]);
        acc[u] = fmaf(qa.y, kb.y, acc[u]);
        acc[u] = fmaf(qa.z, kb.z, acc[u]);
        acc[u] = fmaf(qa.w, kb.w, acc[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], o);
    }
    if (lane == 0) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = jb + u;
        if (j < Tv) {
          s[j] = acc[u];
          scores[((size_t)h * Tv + i) * Tv + j] = acc[u];
        }
      }
    }
  }
  __syncthreads();
  // top-k by rank: rank_j = #{j' : s_j' > s_j or (s_j' == s_j and j' < j)}, NaN as -inf
  for (int j = threadIdx.x; j < Tv; j += ROUTE_THREADS) {
    const float sj = rank_key(s[j]);
    int rank = 0;
    for (int j2 = 0; j2 < Tv; ++j2) {
      const float s2 = rank_key(s[j2]);
      rank += (s2 > sj || (s2 == sj && j2 < j)) ? 1 : 0;
    }
    keep[j] = rank < ksel ? 1 : 0;
  }
  __syncthreads();
  // ascending compaction: a kept tile's slot is the number of kept tiles before it
  int* out = idx + ((size_t)h * Tv + i) * ksel;
  for (int j = threadIdx.x; j < Tv; j += ROUTE_THREADS) {
    if (keep[j]) {
      int pos = 0;
      for (int j2 = 0; j2 < j; ++j2) pos += keep[j2];
      if (pos < ksel) out[pos] = j;
    }
  }
  if (!pooled) return;
  // pooled branch: softmax over all video tiles of S / sqrt(d), then weights . mean(v)
  const float sc = 1.0f / sqrtf((float)d);
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < Tv; j += ROUTE_THREADS) mx = fmaxf(mx, s[j] * sc);
  mx = block_max(mx, red);
  float sum = 0.f;
  for (int j = threadIdx.x; j < Tv; j += ROUTE_THREADS) {
    const float e = expf(s[j] * sc - mx);
    w[j] = e;
    sum += e;
  }
  sum = block_sum(sum, red);  // ends with __syncthreads: w[] complete
  // two halves of the key tiles per column, summed in j order, combined in a fixed order
  const int c = threadIdx.x % d;
  const int half = threadIdx.x / d;  // d = 64: 4 quarters; d = 128: 2 halves
  const int parts = ROUTE_THREADS / d;
  const int per = (Tv + parts - 1) / parts;
  const int j0 = half * per, j1 = min(Tv, j0 + per);
  float acc = 0.f;
  int j = j0;
  for (; j + 8 <= j1; j += 8) {  // eight loads in flight, then the sums in j order
    float m[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) m[u] = __ldg(mV + (size_t)(j + u) * d + c);
#pragma unroll
    for (int u = 0; u < 8; ++u) acc = fmaf(w[j + u], m[u], acc);
  }
  for (; j < j1; ++j) acc = fmaf(w[j], __ldg(mV + (size_t)j * d + c), acc);
  part[half * d + c] = acc;
  __syncthreads();
  if (threadIdx.x < d) {
    float tot = 0.f;
    for (int p = 0; p < parts; ++p) tot += part[p * d + threadIdx.x];
    pooled[((size_t)h * Tv + i) * d + threadIdx.x] = tot / sum;
  }
}

}  // namespace

cudaError_t launch_router(const RouterArgs& a, cudaStream_t stream) {
  if (a.Tv <= 0 || (a.d != 64 && a.d != 128) || a.ksel <= 0) return cudaErrorInvalidValue;
  dim3 g1(a.Tv, a.H, 3);
  tile_means_kernel<<<g1, a.d, 0, stream>>>(a.q, a.k, a.v, a.means, a.N, a.H, a.d, a.n_prefix,
                                            a.n_video, a.Tv);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t shm = (size_t)(3 * a.Tv + 4 * a.d) * 4;
  if (shm > 200 * 1024) return cudaErrorInvalidValue;
  if (shm > 48 * 1024) {
    e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)shm);
    if (e != cudaSuccess) return e;
  }
  dim3 g2(a.Tv, a.H);
  route_kernel<<<g2, ROUTE_THREADS, shm, stream>>>(a.means, a.scores, a.idx, a.pooled, a.H,
                                                    a.d, a.Tv, a.ksel);
  return cudaGetLastError();
}

}  // namespace h3
