// internal.h -- declarations shared by the library's translation units (host side).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "h3dit.h"
#include "tiles.cuh"

namespace h3 {

// ---------------------------------------------------------------- GEMM
enum Epilogue : int {
  kEpiStore = 0,  // y = bf16(acc [+ bias])
  kEpiGelu = 1,   // y = bf16(gelu(acc + bias))
  kEpiResid = 2,  // y = bf16(y + gate * (acc + bias))   (y is the residual, in place)
  kEpiQkvg = 3,   // split into head-major q/k/v with q/k norm + rotary, and row-major g
  kEpiSwiglu = 4,   // y[:, 128j + c] = bf16(silu(acc_g + b_g) * (acc_u + b_u)), y is [M, N/2]
  kEpiHeadEuler = 5 // v = acc + bias (fp32) -> v_out; z += dt * v  (N in {32, 64, 96, 128})
};

struct GemmArgs {
  const __nv_bfloat16* a;  // [M, K]
  const __nv_bfloat16* w;  // [N, K]
  int M, N, K;
  const __nv_bfloat16* bias;  // [N] or null
  __nv_bfloat16* y;           // [M, N] (store / gelu / resid)
  const float* gate;          // [N] fp32 (resid)
  const float* gate_prefix;   // [N] fp32 for rows < n_prefix (resid), or null = gate
  int n_prefix;
  // qkvg epilogue
  int heads, head_dim, attn_width;
  __nv_bfloat16 *q, *k, *v, *g;            // q/k/v [H, M, d], g [M, A]
  const __nv_bfloat16 *qnorm_w, *knorm_w;  // [d] or null
  const float2* rope_cs;                   // [M, d/2] (cos, sin) or null
  float eps;
  // head epilogue
  float* v_out;  // fp32 [M, N] or null
  float* z;      // fp32 [M, N]
  float dt;
  int* status;
  // two ints, zero at launch: the CTA-pair kernel fetches tiles from the first and
  // counts finished clusters in the second (the last resets both); null: tiles are
  // dealt round-robin
  int* tile_counter;
};

cudaError_t launch_gemm(int epi, const GemmArgs& args, cudaStream_t stream);
// 1: the 256-wide projection GEMMs run on CTA pairs (clusters of two SMs, cta_group::2)
// where the device can host them; 0: one SM per tile; -1: query.  Returns the previous.
bool gemm_cta_pairs(int enable);

// ---------------------------------------------------------------- attention
struct AttnArgs {
  const __nv_bfloat16 *q, *k, *v;  // [H, N, d]
  int N, H, d, n_prefix, n_video, Tv, ksel;
  TileGeom geom;              // rows of each video tile
  const int* idx;             // [H, Tv, ksel]
  const __nv_bfloat16* gate;  // [N, A] or null
  const float* pooled;        // [H, Tv, d] or null
  __nv_bfloat16* out;         // [N, A]
  int* status;
  int* counter;  // unit counter of the persistent kernel; zero on entry (the router clears it)
};

cudaError_t launch_attention(const AttnArgs& args, cudaStream_t stream);

// ---------------------------------------------------------------- router
struct RouterArgs {
  const __nv_bfloat16 *q, *k, *v;  // [H, N, d]
  int N, H, d, n_prefix, n_video, Tv, ksel;
  TileGeom geom;  // rows of each video tile
  float* means;   // [3, H, Tv, d]
  float* scores;  // [H, Tv, Tv]
  int* idx;       // [H, Tv, ksel]
  float* pooled;  // [H, Tv, d] or null (skip)
  int* counter;   // set to zero for the attention kernel that follows
};

cudaError_t launch_router(const RouterArgs& args, cudaStream_t stream);

// ---------------------------------------------------------------- row kernels
// rows < n_prefix use (shift_p, scale_p) when shift_p is not null; zero2 (if set): two
// ints set to zero before any row is written (the GEMM tile counters)
cudaError_t launch_rms_modulate(const __nv_bfloat16* x, const float* shift, const float* scale,
                                const float* shift_p, const float* scale_p, int n_prefix,
                                __nv_bfloat16* h, int rows, int D, float eps, cudaStream_t s,
                                int* zero2 = nullptr);
// (cos, sin) per row and rotary pair: 1-D over the packed index, or 3-D (t, h, w) when
// the geometry has a video grid
cudaError_t launch_rope_table(float2* cs, int rows, int d, float theta, const TileGeom& g,
                              cudaStream_t s);
cudaError_t launch_f32_to_bf16(const float* z, __nv_bfloat16* x, size_t n, cudaStream_t s);
// x[r, :] = bf16(z[r, :] w + b), z fp32 [rows, c], w fp32 [c, D] (input-major), b fp32 [D]
cudaError_t launch_patch_in(const float* z, const float* w, const float* b, __nv_bfloat16* x,
                            int rows, int c, int D, cudaStream_t s);
// token reduction: pooled rows of the reduced grid gr from the full rows (grid gf) into
// xr (rows P..) and base; restore: full video rows += xr - base of their pair (in place)
cudaError_t launch_token_pool(const __nv_bfloat16* full, __nv_bfloat16* xr, __nv_bfloat16* base,
                              const TileGeom& gf, const TileGeom& gr, int D, cudaStream_t s);
cudaError_t launch_token_restore(__nv_bfloat16* full, const __nv_bfloat16* xr,
                                 const __nv_bfloat16* base, const TileGeom& gf,
                                 const TileGeom& gr, int D, cudaStream_t s);
// mode 0: r = x; 1: r = x - r; 2: x = bf16(x + r)   (n elements, x bf16, r fp32)
cudaError_t launch_core_residual(__nv_bfloat16* x, float* r, size_t n, int mode, cudaStream_t s);
// elements [0, n_pre) follow the prefix step dt_p (coef_p), the rest dt (coef)
cudaError_t launch_euler_fresh(const __nv_bfloat16* x, float* z, float* v_slot, float dt,
                               float dt_p, size_t n_pre, size_t n, cudaStream_t s);
cudaError_t launch_euler_extrap(float* z, const float* v_a, const float* v_b, float coef,
                                float dt, float coef_p, float dt_p, size_t n_pre, size_t n,
                                cudaStream_t s);

// ---------------------------------------------------------------- tensor maps
bool make_tmap_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                  uint32_t box_rows);
bool make_tmap_3d(CUtensorMap* map, const void* base, uint64_t heads, uint64_t rows,
                  uint64_t cols);

int num_sms();

}  // namespace h3
