// rows.cu -- HBM-bound row and elementwise kernels of the block and the sampler.
//
//  * rms_modulate: h = bf16(x / sqrt(mean(x^2) + eps) * (1 + scale) + shift), with
//    the prefix (text + audio) rows optionally on their own (shift, scale),
//    one 128-thread CTA per row, 16-byte loads kept in registers between the
//    reduction and the write (TensorFold #949 "What it adds": modulated norm;
//    h3.c README fused gated-AdaLN paragraph: a per-row RMS).
//  * rope_table: (cos, sin) per packed row and rotary pair, evaluated in double
//    precision and stored fp32 for the projection epilogue: p * theta^(-2c/d)
//    over the packed index p, or with a video grid a 3-D rotary whose pairs are
//    split into time, height and width groups, each with its own frequency
//    ladder, at the row's latent (t, h, w) (text and audio rows: (p, p, p)).
//  * f32_to_bf16: the sampler's latents -> the bf16 residual stream.
//  * patch_in: a modality's fp32 patch projection into its bf16 hidden rows (h3.c
//    README: fp32 weights, inputs and sums, the result rounded to bf16).
//  * token_pool / token_restore: token reduction (h3.c README): adjacent horizontal
//    video tokens pooled into one row with a full-resolution bypass, and each token
//    restored as its bypass value plus the update its pair received.
//  * core_residual: the blocks' residual x_L - x_0 kept in fp32, and x_L =
//    bf16(x_0 + residual) on a core-reuse pass.
//  * euler_fresh / euler_extrap: v = fp32(x_L), ring store, z += dt * v; or the
//    linear extrapolation of the last two fresh velocities (h3.c README sampler
//    paragraph); prefix rows and video rows each on their own schedule.
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace h3 {

namespace {

constexpr int ROW_THREADS = 128;
constexpr int MAXV = 8;  // 16-byte vectors per thread: D <= 8 * 8 * 128 = 8192

__global__ void __launch_bounds__(ROW_THREADS)
    rms_modulate_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ shift_v,
                        const float* __restrict__ scale_v, const float* __restrict__ shift_p,
                        const float* __restrict__ scale_p, int n_prefix,
                        __nv_bfloat16* __restrict__ h, int D, float eps, int* zero2) {
  __shared__ float wsum[ROW_THREADS / 32];
  const int row = blockIdx.x;
  // the tile counters of the projection GEMMs that follow start from zero
  if (zero2 != nullptr && row == 0 && threadIdx.x < 2) zero2[threadIdx.x] = 0;
  const bool pre = shift_p != nullptr && row < n_prefix;
  const float* shift = pre ? shift_p : shift_v;
  const float* scale = pre ? scale_p : scale_v;
  const int nvec = D / 8;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)row * D);
  uint4 xv[MAXV];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int v = threadIdx.x + i * ROW_THREADS;
    if (v < nvec) {
      xv[i] = src[v];
      const uint32_t w[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a = bf16_lo(w[e]), b = bf16_hi(w[e]);
        ss = fmaf(a, a, ss);
        ss = fmaf(b, b, ss);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < ROW_THREADS / 32; ++w) tot += wsum[w];
  const float inv = 1.0f / sqrtf(tot / (float)D + eps);
  uint4* dst = reinterpret_cast<uint4*>(h + (size_t)row * D);
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int v = threadIdx.x + i * ROW_THREADS;
    if (v < nvec) {
      const float4 s0 = reinterpret_cast<const float4*>(scale)[2 * v];
      const float4 s1 = reinterpret_cast<const float4*>(scale)[2 * v + 1];
      const float4 b0 = reinterpret_cast<const float4*>(shift)[2 * v];
      const float4 b1 = reinterpret_cast<const float4*>(shift)[2 * v + 1];
      const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
      const float sh[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
      const uint32_t w[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a = fmaf(bf16_lo(w[e]) * inv, 1.0f + sc[2 * e], sh[2 * e]);
        const float b = fmaf(bf16_hi(w[e]) * inv, 1.0f + sc[2 * e + 1], sh[2 * e + 1]);
        o[e] = pack_bf16x2(a, b);
      }
      dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

__global__ void rope_table_kernel(float2* cs, int rows, int half, int d, double log_theta,
                                  const TileGeom g) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)rows * half) return;
  const int p = (int)(i / half), c = (int)(i % half);
  double pos, expo;
  if (g.gt == 0) {  // 1-D: pair c turns by p * theta^(-2c/d)
    pos = (double)p;
    expo = 2.0 * (double)c / (double)d;
  } else {  // 3-D: pairs [0, mt) time, [mt, mt + ms) height, the rest width
    const int ms = half / 3, mt = half - 2 * ms;
    int tt = p, hh = p, ww = p;  // text and audio rows: the packed index on every axis
    double wpos = (double)p;
    if (p >= g.P) {
      video_coord(g, p - g.P, &tt, &hh, &ww);
      wpos = (double)ww;
      // a pooled pair of full-width tokens sits at their mean column
      if (g.gw_full > 0) wpos = 2 * ww + 1 < g.gw_full ? 2.0 * ww + 0.5 : 2.0 * ww;
    }
    int j, m;
    if (c < mt) {
      pos = (double)tt, j = c, m = mt;
    } else if (c < mt + ms) {
      pos = (double)hh, j = c - mt, m = ms;
    } else {
      pos = wpos, j = c - mt - ms, m = ms;
    }
    expo = (double)j / (double)m;
  }
  double sn, cn;
  sincos(pos * exp(-expo * log_theta), &sn, &cn);
  cs[i] = make_float2((float)cn, (float)sn);
}

__global__ void f32_to_bf16_kernel(const float4* __restrict__ z, uint2* __restrict__ x, size_t n4) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = z[i];
    x[i] = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
  }
}

__global__ void euler_fresh_kernel(const uint2* __restrict__ x, float4* __restrict__ z,
                                   float4* __restrict__ v_slot, float dt_v, float dt_p,
                                   size_t n4_pre, size_t n4) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const float dt = i < n4_pre ? dt_p : dt_v;
    const uint2 u = x[i];
    const float4 v = make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
    float4 zz = z[i];
    zz.x = fmaf(dt, v.x, zz.x);
    zz.y = fmaf(dt, v.y, zz.y);
    zz.z = fmaf(dt, v.z, zz.z);
    zz.w = fmaf(dt, v.w, zz.w);
    v_slot[i] = v;
    z[i] = zz;
  }
}

__global__ void euler_extrap_kernel(float4* __restrict__ z, const float4* __restrict__ va,
                                    const float4* __restrict__ vb, float coef_v, float dt_v,
                                    float coef_p, float dt_p, size_t n4_pre, size_t n4) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const bool pre = i < n4_pre;
    const float coef = pre ? coef_p : coef_v;
    const float dt = pre ? dt_p : dt_v;
    const float4 a = va[i];
    float4 v = a;
    if (vb) {
      const float4 b = vb[i];
      v.x = fmaf(a.x - b.x, coef, a.x);
      v.y = fmaf(a.y - b.y, coef, a.y);
      v.z = fmaf(a.z - b.z, coef, a.z);
      v.w = fmaf(a.w - b.w, coef, a.w);
    }
    float4 zz = z[i];
    zz.x = fmaf(dt, v.x, zz.x);
    zz.y = fmaf(dt, v.y, zz.y);
    zz.z = fmaf(dt, v.z, zz.z);
    zz.w = fmaf(dt, v.w, zz.w);
    z[i] = zz;
  }
}

// Patch projection of one modality: x[r, :] = bf16(sum_j z[r, j] w[j, :] + b) with fp32
// weights, inputs and sums (j ascending), one CTA per 32 rows x 256 columns; thread
// (column group g, row group q) owns 8 rows x 4 columns.
__global__ void __launch_bounds__(256)
    patch_in_kernel(const float* __restrict__ z, const float* __restrict__ w,
                    const float* __restrict__ b, __nv_bfloat16* __restrict__ x, int R, int c,
                    int D) {
  __shared__ float4 ws4[32][64];  // 32 input channels x 256 columns of w
  __shared__ float zs[32][33];    // 32 rows x 32 input channels of z (padded)
  const int g = threadIdx.x & 63, q = threadIdx.x >> 6;
  const int row0 = blockIdx.x * 32, col0 = blockIdx.y * 256;
  float acc[8][4];
#pragma unroll
  for (int r = 0; r < 8; ++r) acc[r][0] = acc[r][1] = acc[r][2] = acc[r][3] = 0.f;
  for (int k0 = 0; k0 < c; k0 += 32) {
    __syncthreads();
    for (int i = threadIdx.x; i < 32 * 64; i += 256) {
      const int kk = i >> 6, gg = i & 63;
      ws4[kk][gg] = __ldg(reinterpret_cast<const float4*>(w + (size_t)(k0 + kk) * D + col0) + gg);
    }
    for (int i = threadIdx.x; i < 32 * 32; i += 256) {
      const int r = i >> 5, kk = i & 31;
      zs[r][kk] = row0 + r < R ? __ldg(z + (size_t)(row0 + r) * c + k0 + kk) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < 32; ++kk) {
      const float4 wv = ws4[kk][g];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float zv = zs[q * 8 + r][kk];
        acc[r][0] = fmaf(zv, wv.x, acc[r][0]);
        acc[r][1] = fmaf(zv, wv.y, acc[r][1]);
        acc[r][2] = fmaf(zv, wv.z, acc[r][2]);
        acc[r][3] = fmaf(zv, wv.w, acc[r][3]);
      }
    }
  }
  const float4 bv = __ldg(reinterpret_cast<const float4*>(b + col0) + g);
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int row = row0 + q * 8 + r;
    if (row < R) {
      *reinterpret_cast<uint2*>(x + (size_t)row * D + col0 + 4 * g) =
          make_uint2(pack_bf16x2(acc[r][0] + bv.x, acc[r][1] + bv.y),
                     pack_bf16x2(acc[r][2] + bv.z, acc[r][3] + bv.w));
    }
  }
}

// Core residual: mode 0 r = x; mode 1 r = x - r; mode 2 x = bf16(x + r)  (x bf16, r fp32)
__global__ void core_residual_kernel(uint2* __restrict__ x, float4* __restrict__ r, size_t n4,
                                     int mode) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const uint2 u = x[i];
    const float4 a = make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
    if (mode == 0) {
      r[i] = a;
    } else if (mode == 1) {
      const float4 b = r[i];
      r[i] = make_float4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w);
    } else {
      const float4 b = r[i];
      x[i] = make_uint2(pack_bf16x2(a.x + b.x, a.y + b.y), pack_bf16x2(a.z + b.z, a.w + b.w));
    }
  }
}

// Token reduction entry: reduced video row i (cube order of the reduced grid gr) is the
// mean of the full tokens (t, h, 2j) and (t, h, 2j + 1), or the lone last token of an odd
// row; written to xr row P + i and to the baseline row i.  One CTA per reduced row.
__global__ void __launch_bounds__(ROW_THREADS)
    token_pool_kernel(const __nv_bfloat16* __restrict__ full, __nv_bfloat16* __restrict__ xr,
                      __nv_bfloat16* __restrict__ base, const TileGeom gf, const TileGeom gr,
                      int D) {
  const int i = blockIdx.x;
  int t, h, j;
  video_coord(gr, i, &t, &h, &j);
  const bool pair = 2 * j + 1 < gf.gw;
  const int s0 = video_row_of(gf, t, h, 2 * j);
  const int s1 = pair ? video_row_of(gf, t, h, 2 * j + 1) : s0;
  const uint4* a = reinterpret_cast<const uint4*>(full + (size_t)(gf.P + s0) * D);
  const uint4* b = reinterpret_cast<const uint4*>(full + (size_t)(gf.P + s1) * D);
  uint4* o = reinterpret_cast<uint4*>(xr + (size_t)(gr.P + i) * D);
  uint4* q = reinterpret_cast<uint4*>(base + (size_t)i * D);
  for (int v = threadIdx.x; v < D / 8; v += ROW_THREADS) {
    const uint4 ua = a[v], ub = b[v];
    const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
    uint32_t r[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      r[e] = pack_bf16x2((bf16_lo(wa[e]) + bf16_lo(wb[e])) * 0.5f,
                         (bf16_hi(wa[e]) + bf16_hi(wb[e])) * 0.5f);
    const uint4 out = make_uint4(r[0], r[1], r[2], r[3]);
    o[v] = out;
    q[v] = out;
  }
}

// Token reduction exit: full video row k (cube order of gf) becomes
// bf16(bypass_k + (xr_i - baseline_i)) with i its pair's reduced row.  In place on the
// bypass.  One CTA per full video row.
__global__ void __launch_bounds__(ROW_THREADS)
    token_restore_kernel(__nv_bfloat16* __restrict__ full, const __nv_bfloat16* __restrict__ xr,
                         const __nv_bfloat16* __restrict__ base, const TileGeom gf,
                         const TileGeom gr, int D) {
  const int k = blockIdx.x;
  int t, h, w;
  video_coord(gf, k, &t, &h, &w);
  const int i = video_row_of(gr, t, h, w / 2);
  uint4* f = reinterpret_cast<uint4*>(full + (size_t)(gf.P + k) * D);
  const uint4* y = reinterpret_cast<const uint4*>(xr + (size_t)(gr.P + i) * D);
  const uint4* b0 = reinterpret_cast<const uint4*>(base + (size_t)i * D);
  for (int v = threadIdx.x; v < D / 8; v += ROW_THREADS) {
    const uint4 uf = f[v], uy = y[v], ub = b0[v];
    const uint32_t wf[4] = {uf.x, uf.y, uf.z, uf.w}, wy[4] = {uy.x, uy.y, uy.z, uy.w},
                   wb[4] = {ub.x, ub.y, ub.z, ub.w};
    uint32_t r[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      r[e] = pack_bf16x2(bf16_lo(wf[e]) + (bf16_lo(wy[e]) - bf16_lo(wb[e])),
                         bf16_hi(wf[e]) + (bf16_hi(wy[e]) - bf16_hi(wb[e])));
    f[v] = make_uint4(r[0], r[1], r[2], r[3]);
  }
}

int grid_for(size_t n, int threads) {
  size_t b = (n + threads - 1) / threads;
  const size_t cap = (size_t)num_sms() * 16;
  if (b > cap) b = cap;
  return b < 1 ? 1 : (int)b;
}

}  // namespace

cudaError_t launch_rms_modulate(const __nv_bfloat16* x, const float* shift, const float* scale,
                                const float* shift_p, const float* scale_p, int n_prefix,
                                __nv_bfloat16* h, int rows, int D, float eps, cudaStream_t s,
                                int* zero2) {
  if (rows <= 0 || D % 8 != 0 || D > 8 * MAXV * ROW_THREADS) return cudaErrorInvalidValue;
  rms_modulate_kernel<<<rows, ROW_THREADS, 0, s>>>(x, shift, scale, shift_p, scale_p, n_prefix, h,
                                                   D, eps, zero2);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(float2* cs, int rows, int d, float theta, const TileGeom& g,
                              cudaStream_t s) {
  const int half = d / 2;
  const size_t n = (size_t)rows * half;
  rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(cs, rows, half, d,
                                                                 log((double)theta), g);
  return cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float* z, __nv_bfloat16* x, size_t n, cudaStream_t s) {
  if (n % 4) return cudaErrorInvalidValue;
  f32_to_bf16_kernel<<<grid_for(n / 4, 256), 256, 0, s>>>(
      reinterpret_cast<const float4*>(z), reinterpret_cast<uint2*>(x), n / 4);
  return cudaGetLastError();
}

cudaError_t launch_patch_in(const float* z, const float* w, const float* b, __nv_bfloat16* x,
                            int rows, int c, int D, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (c <= 0 || c % 32 || D % 256) return cudaErrorInvalidValue;
  patch_in_kernel<<<dim3((rows + 31) / 32, D / 256), 256, 0, s>>>(z, w, b, x, rows, c, D);
  return cudaGetLastError();
}

cudaError_t launch_core_residual(__nv_bfloat16* x, float* r, size_t n, int mode, cudaStream_t s) {
  if (n % 4 || mode < 0 || mode > 2) return cudaErrorInvalidValue;
  core_residual_kernel<<<grid_for(n / 4, 256), 256, 0, s>>>(
      reinterpret_cast<uint2*>(x), reinterpret_cast<float4*>(r), n / 4, mode);
  return cudaGetLastError();
}

cudaError_t launch_token_pool(const __nv_bfloat16* full, __nv_bfloat16* xr, __nv_bfloat16* base,
                              const TileGeom& gf, const TileGeom& gr, int D, cudaStream_t s) {
  if (gr.V <= 0 || D % 8 || gf.gt == 0 || gr.gt == 0) return cudaErrorInvalidValue;
  token_pool_kernel<<<gr.V, ROW_THREADS, 0, s>>>(full, xr, base, gf, gr, D);
  return cudaGetLastError();
}

cudaError_t launch_token_restore(__nv_bfloat16* full, const __nv_bfloat16* xr,
                                 const __nv_bfloat16* base, const TileGeom& gf,
                                 const TileGeom& gr, int D, cudaStream_t s) {
  if (gf.V <= 0 || D % 8 || gf.gt == 0 || gr.gt == 0) return cudaErrorInvalidValue;
  token_restore_kernel<<<gf.V, ROW_THREADS, 0, s>>>(full, xr, base, gf, gr, D);
  return cudaGetLastError();
}

cudaError_t launch_euler_fresh(const __nv_bfloat16* x, float* z, float* v_slot, float dt,
                               float dt_p, size_t n_pre, size_t n, cudaStream_t s) {
  if (n % 4 || n_pre % 4) return cudaErrorInvalidValue;
  euler_fresh_kernel<<<grid_for(n / 4, 256), 256, 0, s>>>(
      reinterpret_cast<const uint2*>(x), reinterpret_cast<float4*>(z),
      reinterpret_cast<float4*>(v_slot), dt, dt_p, n_pre / 4, n / 4);
  return cudaGetLastError();
}

cudaError_t launch_euler_extrap(float* z, const float* v_a, const float* v_b, float coef,
                                float dt, float coef_p, float dt_p, size_t n_pre, size_t n,
                                cudaStream_t s) {
  if (n % 4 || n_pre % 4) return cudaErrorInvalidValue;
  euler_extrap_kernel<<<grid_for(n / 4, 256), 256, 0, s>>>(
      reinterpret_cast<float4*>(z), reinterpret_cast<const float4*>(v_a),
      reinterpret_cast<const float4*>(v_b), coef, dt, coef_p, dt_p, n_pre / 4, n / 4);
  return cudaGetLastError();
}

}  // namespace h3
