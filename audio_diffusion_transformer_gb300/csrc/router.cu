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
// Kernel 2 (route): one CTA per (query tile i, head h):
//   S[h,i,j] = sum_c mq[h,i,c] mk[h,j,c] (fp32 FMA chain, c ascending);
//   rank_j = #{j' : s_j' > s_j or (s_j' == s_j and j' < j)} with NaN -> -inf;
//   tile j is kept iff rank_j < k; kept tiles are written ascending;
//   pooled[h,i,:] = sum_j softmax_j(S[h,i,j] / sqrt(d)) mv[h,j,:] (sums in j order).
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
  for (int r = 0; r < nv; ++r) s += __bfloat162float(src[(size_t)r * d]);
  means[(((size_t)which * H + h) * Tv + t) * d + c] = s / (float)nv;
}

__device__ __forceinline__ float rank_key(float s) { return isnan(s) ? -INFINITY : s; }

__global__ void __launch_bounds__(ROUTE_THREADS)
    route_kernel(const float* __restrict__ means, float* __restrict__ scores,
                 int* __restrict__ idx, float* __restrict__ pooled, int H, int d, int Tv,
                 int ksel) {
  extern __shared__ float sh[];
  float* mq = sh;         // [d]
  float* s = sh + d;      // [Tv]
  float* w = s + Tv;      // [Tv]
  int* keep = reinterpret_cast<int*>(w + Tv);  // [Tv]
  __shared__ float red[2];
  const int i = blockIdx.x, h = blockIdx.y;
  const float* mQ = means + ((size_t)0 * H + h) * Tv * d;
  const float* mK = means + ((size_t)1 * H + h) * Tv * d;
  const float* mV = means + ((size_t)2 * H + h) * Tv * d;
  for (int c = threadIdx.x; c < d; c += blockDim.x) mq[c] = mQ[(size_t)i * d + c];
  __syncthreads();
  for (int j = threadIdx.x; j < Tv; j += blockDim.x) {
    const float* kr = mK + (size_t)j * d;
    float acc = 0.f;
    for (int c = 0; c < d; ++c) acc = fmaf(mq[c], kr[c], acc);
    s[j] = acc;
    scores[((size_t)h * Tv + i) * Tv + j] = acc;
  }
  __syncthreads();
  for (int j = threadIdx.x; j < Tv; j += blockDim.x) {
    const float sj = rank_key(s[j]);
    int rank = 0;
    for (int j2 = 0; j2 < Tv; ++j2) {
      const float s2 = rank_key(s[j2]);
      rank += (s2 > sj || (s2 == sj && j2 < j)) ? 1 : 0;
    }
    keep[j] = rank < ksel ? 1 : 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int n = 0;
    int* out = idx + ((size_t)h * Tv + i) * ksel;
    for (int j = 0; j < Tv && n < ksel; ++j)
      if (keep[j]) out[n++] = j;
    if (pooled) {
      const float sc = 1.0f / sqrtf((float)d);
      float mx = -INFINITY;
      for (int j = 0; j < Tv; ++j) mx = fmaxf(mx, s[j] * sc);
      float sum = 0.f;
      for (int j = 0; j < Tv; ++j) {
        const float e = expf(s[j] * sc - mx);
        w[j] = e;
        sum += e;
      }
      red[0] = sum;
    }
  }
  if (!pooled) return;
  __syncthreads();
  const float inv = 1.0f / red[0];
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < Tv; ++j) acc = fmaf(w[j], mV[(size_t)j * d + c], acc);
    pooled[((size_t)h * Tv + i) * d + c] = acc * inv;
  }
}

}  // namespace

cudaError_t launch_router(const RouterArgs& a, cudaStream_t stream) {
  if (a.Tv <= 0 || a.d <= 0 || a.d > 1024 || a.ksel <= 0) return cudaErrorInvalidValue;
  dim3 g1(a.Tv, a.H, 3);
  tile_means_kernel<<<g1, a.d, 0, stream>>>(a.q, a.k, a.v, a.means, a.N, a.H, a.d, a.n_prefix,
                                            a.n_video, a.Tv);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t shm = (size_t)(a.d + 3 * a.Tv) * 4;
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
