// api.cu -- the exported C ABI: argument checks, workspace planning, tensor
// maps and the launch sequence of a block, an attention layer and a denoiser
// step.  Everything here runs on the host; all arithmetic is in the kernels.
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <atomic>
#include <vector>

#include "internal.h"

namespace h3 {

// ---------------------------------------------------------------- tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// bf16 row-major [rows, cols], box = 64 columns (128 bytes) x box_rows, 128-byte swizzle.
bool make_tmap_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                  uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [heads, rows, cols] (cols innermost), box = 64 x 64 x 1, 128-byte swizzle.
bool make_tmap_3d(CUtensorMap* map, const void* base, uint64_t heads, uint64_t rows,
                  uint64_t cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cols, rows, heads};
  cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
  cuuint32_t box[3] = {64, 64, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

namespace {

// ---------------------------------------------------------------- tracing
std::atomic<unsigned long long> g_launches{0};

struct Profiler {
  bool on = false;
  int max = 0, used = 0;
  std::vector<cudaEvent_t> ev;   // 2 per record
  std::vector<int> stage, nlaunch;
};
Profiler g_prof;

// Records an event pair around one stage when profiling is on.
struct StageScope {
  int rec = -1;
  unsigned long long l0;
  cudaStream_t st;
  StageScope(int id, cudaStream_t s) : st(s) {
    l0 = g_launches.load();
    if (g_prof.on && g_prof.used < g_prof.max) {
      rec = g_prof.used++;
      g_prof.stage[rec] = id;
      cudaEventRecord(g_prof.ev[2 * rec], st);
    }
  }
  ~StageScope() {
    if (rec >= 0) {
      cudaEventRecord(g_prof.ev[2 * rec + 1], st);
      g_prof.nlaunch[rec] = (int)(g_launches.load() - l0);
    }
  }
};

inline cudaError_t counted(cudaError_t e, int n) {
  if (e == cudaSuccess) g_launches += n;
  return e;
}

constexpr size_t kAlign = 256;
constexpr int kMaxRows = 1022 * 64;  // a prefix attention unit walks N / 128 <= 512 steps

inline size_t up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

struct Dims {
  int N, P, V, Tv, ksel, D, H, d, A, F;
  TileGeom geom;
  bool block;   // hidden / mlp widths given
  bool reduce;  // token-reduction buffers reserved
  bool keep;    // intermediates kept apart (H3DIT_KEEP_INTERMEDIATES)
};

#define H3_TRY_SHAPE(expr)                    \
  do {                                        \
    h3dit_status _st = (expr);                \
    if (_st != H3DIT_OK) return _st;          \
  } while (0)

// The video tile geometry of a shape; false if the grid or cube fields are inconsistent.
bool make_geom(const h3dit_shape* s, TileGeom* g) {
  memset(g, 0, sizeof(*g));
  g->P = s->n_text + s->n_audio;
  g->V = s->n_video;
  const int grid[3] = {s->video_t, s->video_h, s->video_w};
  const int cube[3] = {s->cube_t, s->cube_h, s->cube_w};
  bool any = false;
  for (int i = 0; i < 3; ++i) any = any || grid[i] != 0 || cube[i] != 0;
  if (!any) return true;
  for (int i = 0; i < 3; ++i)
    if (grid[i] < 1 || cube[i] < 1 || grid[i] > (1 << 20)) return false;
  if ((long long)grid[0] * grid[1] * grid[2] != s->n_video) return false;
  if (cube[0] * cube[1] * cube[2] != s->tile) return false;
  g->gt = grid[0];
  g->gh = grid[1];
  g->gw = grid[2];
  g->ct = cube[0];
  g->ch = cube[1];
  g->cw = cube[2];
  g->nt = (grid[0] + cube[0] - 1) / cube[0];
  g->nh = (grid[1] + cube[1] - 1) / cube[1];
  g->nw = (grid[2] + cube[2] - 1) / cube[2];
  return true;
}

h3dit_status check_attn(const h3dit_shape* s, Dims* o) {
  if (!s) return H3DIT_ERR_ARG;
  if (s->n_text < 0 || s->n_audio < 0 || s->n_video < 1) return H3DIT_ERR_SHAPE;
  if (s->tile != 64) return H3DIT_ERR_SHAPE;
  const long long N = (long long)s->n_text + s->n_audio + s->n_video;
  if (N > kMaxRows) return H3DIT_ERR_SHAPE;
  const int P = s->n_text + s->n_audio;
  if (s->head_dim != 64 && s->head_dim != 128) return H3DIT_ERR_SHAPE;
  if (s->heads < 1 || s->heads > 4096) return H3DIT_ERR_SHAPE;
  if (s->attn_width != s->heads * s->head_dim) return H3DIT_ERR_SHAPE;
  if (s->topk < 1) return H3DIT_ERR_ARG;
  if (!make_geom(s, &o->geom)) return H3DIT_ERR_SHAPE;
  const int Tv = tile_count_of(o->geom);
  if (Tv > 1024) return H3DIT_ERR_SHAPE;  // the router's top-k tracks at most 1,024 tiles
  if ((size_t)(s->head_dim + 3 * Tv) * 4 > 200 * 1024) return H3DIT_ERR_SHAPE;
  if (!(s->rms_eps >= 0.f)) return H3DIT_ERR_ARG;
  o->N = (int)N;
  o->P = P;
  o->V = s->n_video;
  o->Tv = Tv;
  o->ksel = s->topk < Tv ? s->topk : Tv;
  // a video unit's steps (128-row prefix chunks + one per selected tile) must fit the
  // attention kernel's 512-entry step lists
  if ((P + 127) / 128 + o->ksel > 512) return H3DIT_ERR_SHAPE;
  o->H = s->heads;
  o->d = s->head_dim;
  o->A = s->attn_width;
  o->D = s->hidden;
  o->F = s->mlp_width;
  o->block = false;
  o->reduce = false;
  o->keep = false;
  return H3DIT_OK;
}

h3dit_status check_block(const h3dit_shape* s, Dims* o) {
  h3dit_status st = check_attn(s, o);
  if (st != H3DIT_OK) return st;
  if (s->hidden < 256 || s->hidden % 256 || s->hidden > 8192) return H3DIT_ERR_SHAPE;
  if (s->attn_width % 256) return H3DIT_ERR_SHAPE;
  if (s->flags & H3DIT_SWIGLU) {
    if (s->mlp_width < 128 || s->mlp_width % 128) return H3DIT_ERR_SHAPE;  // fc1 N = 2F
    if (s->mlp_width % 64) return H3DIT_ERR_SHAPE;                         // fc2 K = F
  } else if (s->mlp_width < 256 || s->mlp_width % 256) {
    return H3DIT_ERR_SHAPE;
  }
  if ((s->flags & H3DIT_ROPE) && (s->rope_theta <= 1.0f)) return H3DIT_ERR_ARG;
  o->block = true;
  o->reduce = (s->flags & H3DIT_TOKEN_REDUCTION) != 0;
  o->keep = (s->flags & H3DIT_KEEP_INTERMEDIATES) != 0;
  if (o->reduce && (o->geom.gt == 0 || o->geom.gw < 2)) return H3DIT_ERR_SHAPE;
  return H3DIT_OK;
}

// The shape of the token-reduced section: the same rows but video t x h x ceil(w/2).
h3dit_status reduced_dims(const h3dit_shape* s, h3dit_shape* rs, Dims* rm) {
  *rs = *s;
  rs->video_w = (s->video_w + 1) / 2;
  rs->n_video = s->video_t * s->video_h * rs->video_w;
  rs->flags &= ~H3DIT_TOKEN_REDUCTION;
  H3_TRY_SHAPE(check_block(rs, rm));
  rm->geom.gw_full = s->video_w;
  return H3DIT_OK;
}

// Workspace layout (all offsets 256-byte aligned; kAbsent = region not reserved).
constexpr size_t kAbsent = H3DIT_WS_ABSENT;
struct Ws {
  size_t status, q, k, v, g, o, u, h, x, x1, rope, means, scores, idx, pooled, bypass, base,
      total;
};

Ws plan(const Dims& m) {
  Ws w;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off += up(bytes);
    return at;
  };
  const size_t NA = (size_t)m.N * m.A * 2;
  w.status = take(kAlign);
  // attention alone needs only the status word and the router's regions
  w.q = w.k = w.v = w.g = w.o = kAbsent;
  if (m.block) {
    w.q = take(NA);
    w.k = take(NA);
    w.v = take(NA);
    w.g = take(NA);
    w.o = take(NA);
  }
  w.means = take((size_t)3 * m.H * m.Tv * m.d * 4);
  w.scores = take((size_t)m.H * m.Tv * m.Tv * 4);
  w.idx = take((size_t)m.H * m.Tv * m.ksel * 4);
  w.pooled = take((size_t)m.H * m.Tv * m.d * 4);
  w.u = w.h = w.x = w.x1 = w.rope = kAbsent;
  if (m.block) {
    const size_t NF = (size_t)m.N * m.F * 2;
    // u (the MLP inner activations) reuses q..g, which are dead after attention, unless
    // the intermediates are kept for inspection
    w.u = (!m.keep && NF <= 4 * NA) ? w.q : take(NF);
    w.h = take((size_t)m.N * m.D * 2);
    w.x = take((size_t)m.N * m.D * 2);
    w.rope = take((size_t)m.N * (m.d / 2) * 8);
    if (m.keep) w.x1 = take((size_t)m.N * m.D * 2);
  }
  w.bypass = w.base = 0;
  if (m.reduce) {  // full-resolution bypass and the pooled rows' baselines
    w.bypass = take((size_t)m.N * m.D * 2);
    w.base = take((size_t)m.geom.gt * m.geom.gh * ((m.geom.gw + 1) / 2) * m.D * 2);
  }
  w.total = off;
  return w;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

h3dit_status device_ok() {
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return H3DIT_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return H3DIT_ERR_CUDA;
  return major == 10 ? H3DIT_OK : H3DIT_ERR_UNSUPPORTED;
}

inline h3dit_status cu(cudaError_t e) { return e == cudaSuccess ? H3DIT_OK : H3DIT_ERR_CUDA; }

#define H3_TRY(expr)                          \
  do {                                        \
    h3dit_status _st = (expr);                \
    if (_st != H3DIT_OK) return _st;          \
  } while (0)

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

h3dit_status run_attention(const h3dit_shape* s, const Dims& m, const Ws& w, void* ws,
                           const __nv_bfloat16* q, const __nv_bfloat16* k,
                           const __nv_bfloat16* v, const __nv_bfloat16* gate,
                           __nv_bfloat16* out, float* pooled, int* idx, float* scores,
                           cudaStream_t st) {
  const bool use_pool = (s->flags & H3DIT_POOLED) && gate != nullptr;
  RouterArgs r;
  r.q = q;
  r.k = k;
  r.v = v;
  r.N = m.N;
  r.H = m.H;
  r.d = m.d;
  r.n_prefix = m.P;
  r.n_video = m.V;
  r.Tv = m.Tv;
  r.geom = m.geom;
  r.ksel = m.ksel;
  r.means = at<float>(ws, w.means);
  r.scores = scores ? scores : at<float>(ws, w.scores);
  r.idx = idx ? idx : at<int>(ws, w.idx);
  r.pooled = use_pool || pooled ? (pooled ? pooled : at<float>(ws, w.pooled)) : nullptr;
  // the attention kernel's unit counter shares the status block (a separate 128-byte line)
  r.counter = at<int>(ws, w.status) + 32;
  {
    StageScope sc(H3DIT_STAGE_ROUTER, st);
    H3_TRY(cu(counted(launch_router(r, st), 2)));
  }
  AttnArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.N = m.N;
  a.H = m.H;
  a.d = m.d;
  a.n_prefix = m.P;
  a.n_video = m.V;
  a.Tv = m.Tv;
  a.geom = m.geom;
  a.ksel = m.ksel;
  a.idx = r.idx;
  a.gate = use_pool ? gate : nullptr;
  a.pooled = use_pool ? r.pooled : nullptr;
  a.out = out;
  a.status = at<int>(ws, w.status);
  a.counter = r.counter;
  StageScope sc(H3DIT_STAGE_ATTN, st);
  return cu(counted(launch_attention(a, st), 1));
}

h3dit_status run_block(const h3dit_shape* s, const Dims& m, const Ws& w, void* ws,
                       const h3dit_block_weights* wt, __nv_bfloat16* x, bool rope_ready,
                       cudaStream_t st) {
  const int N = m.N, D = m.D, A = m.A, F = m.F;
  int* status = at<int>(ws, w.status);
  // the projection GEMMs' tile counters share the status block (a separate 64-byte
  // sector from the status word and the attention unit counter); the norms zero them
  int* tiles = status + 48;
  __nv_bfloat16* h = at<__nv_bfloat16>(ws, w.h);
  __nv_bfloat16* q = at<__nv_bfloat16>(ws, w.q);
  __nv_bfloat16* k = at<__nv_bfloat16>(ws, w.k);
  __nv_bfloat16* v = at<__nv_bfloat16>(ws, w.v);
  __nv_bfloat16* g = at<__nv_bfloat16>(ws, w.g);
  __nv_bfloat16* o = at<__nv_bfloat16>(ws, w.o);
  __nv_bfloat16* u = at<__nv_bfloat16>(ws, w.u);
  float2* rope = at<float2>(ws, w.rope);
  const float* mod = wt->mod;
  const float* modp = wt->mod_prefix;  // null: every row uses mod
  const int P = m.P;
  const bool use_rope = (s->flags & H3DIT_ROPE) != 0;
  if (use_rope && !rope_ready) {
    StageScope sc(H3DIT_STAGE_SAMPLER, st);
    H3_TRY(cu(counted(launch_rope_table(rope, N, m.d, s->rope_theta, m.geom, st), 1)));
  }

  // a1: modulated norm 1
  {
    StageScope sc(H3DIT_STAGE_NORM1, st);
    H3_TRY(cu(counted(launch_rms_modulate(x, mod + 0 * D, mod + 1 * D, modp ? modp + 0 * D : nullptr,
                                          modp ? modp + 1 * D : nullptr, P, h, N, D, s->rms_eps,
                                          st, tiles), 1)));
  }
  // a2 + a3: q/k/v/gate projection with q/k norm, rotary and head-major layout
  GemmArgs ga;
  memset(&ga, 0, sizeof(ga));
  ga.a = h;
  ga.w = static_cast<const __nv_bfloat16*>(wt->w_qkvg);
  ga.M = N;
  ga.N = 4 * A;
  ga.K = D;
  ga.bias = static_cast<const __nv_bfloat16*>(wt->b_qkvg);
  ga.heads = m.H;
  ga.head_dim = m.d;
  ga.attn_width = A;
  ga.q = q;
  ga.k = k;
  ga.v = v;
  ga.g = g;
  if (s->flags & H3DIT_QK_NORM) {
    ga.qnorm_w = static_cast<const __nv_bfloat16*>(wt->qnorm_w);
    ga.knorm_w = static_cast<const __nv_bfloat16*>(wt->knorm_w);
  }
  ga.rope_cs = use_rope ? rope : nullptr;
  ga.eps = s->rms_eps;
  ga.status = status;
  ga.tile_counter = tiles;
  {
    StageScope sc(H3DIT_STAGE_QKVG, st);
    H3_TRY(cu(counted(launch_gemm(kEpiQkvg, ga, st), 1)));
  }
  // a4..a9: router, routed + dense attention, pooled branch and gate mix
  H3_TRY(run_attention(s, m, w, ws, q, k, v, g, o, nullptr, nullptr, nullptr, st));
  // a10: out projection + gated residual (in place on x)
  GemmArgs gb;
  memset(&gb, 0, sizeof(gb));
  gb.a = o;
  gb.w = static_cast<const __nv_bfloat16*>(wt->w_o);
  gb.M = N;
  gb.N = D;
  gb.K = A;
  gb.bias = static_cast<const __nv_bfloat16*>(wt->b_o);
  gb.y = x;
  gb.gate = mod + 2 * D;
  gb.gate_prefix = modp ? modp + 2 * D : nullptr;
  gb.n_prefix = P;
  gb.status = status;
  gb.tile_counter = tiles;
  {
    StageScope sc(H3DIT_STAGE_OUT, st);
    H3_TRY(cu(counted(launch_gemm(kEpiResid, gb, st), 1)));
  }
  if (w.x1 != kAbsent &&
      cudaMemcpyAsync(at<__nv_bfloat16>(ws, w.x1), x, (size_t)N * D * 2,
                      cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return H3DIT_ERR_CUDA;
  // a11: modulated norm 2
  {
    StageScope sc(H3DIT_STAGE_NORM2, st);
    H3_TRY(cu(counted(launch_rms_modulate(x, mod + 3 * D, mod + 4 * D, modp ? modp + 3 * D : nullptr,
                                          modp ? modp + 4 * D : nullptr, P, h, N, D, s->rms_eps,
                                          st, tiles), 1)));
  }
  // a12: fc1 + GELU, or the gate/up projection + SwiGLU
  const bool swiglu = (s->flags & H3DIT_SWIGLU) != 0;
  GemmArgs gc;
  memset(&gc, 0, sizeof(gc));
  gc.a = h;
  gc.w = static_cast<const __nv_bfloat16*>(wt->w1);
  gc.M = N;
  gc.N = swiglu ? 2 * F : F;
  gc.K = D;
  gc.bias = static_cast<const __nv_bfloat16*>(wt->b1);
  gc.y = u;
  gc.status = status;
  gc.tile_counter = tiles;
  {
    StageScope sc(H3DIT_STAGE_FC1, st);
    H3_TRY(cu(counted(launch_gemm(swiglu ? kEpiSwiglu : kEpiGelu, gc, st), 1)));
  }
  // a13: fc2 + gated residual (in place on x)
  GemmArgs gd;
  memset(&gd, 0, sizeof(gd));
  gd.a = u;
  gd.w = static_cast<const __nv_bfloat16*>(wt->w2);
  gd.M = N;
  gd.N = D;
  gd.K = F;
  gd.bias = static_cast<const __nv_bfloat16*>(wt->b2);
  gd.y = x;
  gd.gate = mod + 5 * D;
  gd.gate_prefix = modp ? modp + 5 * D : nullptr;
  gd.n_prefix = P;
  gd.status = status;
  gd.tile_counter = tiles;
  StageScope sc(H3DIT_STAGE_FC2, st);
  return cu(counted(launch_gemm(kEpiResid, gd, st), 1));
}

h3dit_status check_weights(const h3dit_shape* s, const h3dit_block_weights* w) {
  if (!w) return H3DIT_ERR_ARG;
  const void* req[] = {w->w_qkvg, w->b_qkvg, w->w_o, w->b_o, w->w1, w->b1, w->w2, w->b2, w->mod};
  for (const void* p : req) {
    if (!p) return H3DIT_ERR_ARG;
    if (!aligned16(p)) return H3DIT_ERR_ALIGN;
  }
  if (s->flags & H3DIT_QK_NORM) {
    if (!w->qnorm_w || !w->knorm_w) return H3DIT_ERR_ARG;
    if (!aligned16(w->qnorm_w) || !aligned16(w->knorm_w)) return H3DIT_ERR_ALIGN;
  }
  if (w->mod_prefix && !aligned16(w->mod_prefix)) return H3DIT_ERR_ALIGN;
  return H3DIT_OK;
}

// Checks the ends struct against a shape (host only).
h3dit_status check_ends(const h3dit_shape* s, const h3dit_ends* e) {
  if (!e) return H3DIT_ERR_ARG;
  auto ok_c = [](int c) { return c >= 32 && c <= 128 && c % 32 == 0; };
  if (!ok_c(e->c_video) || (s->n_audio > 0 && !ok_c(e->c_audio))) return H3DIT_ERR_SHAPE;
  const void* vid[] = {e->w_in_video, e->b_in_video, e->w_out_video, e->b_out_video,
                       e->mod_out_video};
  for (const void* p : vid) {
    if (!p) return H3DIT_ERR_ARG;
    if (!aligned16(p)) return H3DIT_ERR_ALIGN;
  }
  if (s->n_audio > 0) {
    const void* aud[] = {e->w_in_audio, e->b_in_audio, e->w_out_audio, e->b_out_audio,
                         e->mod_out_audio};
    for (const void* p : aud) {
      if (!p) return H3DIT_ERR_ARG;
      if (!aligned16(p)) return H3DIT_ERR_ALIGN;
    }
  }
  if (s->n_text > 0) {
    if (!e->text) return H3DIT_ERR_ARG;
    if (!aligned16(e->text)) return H3DIT_ERR_ALIGN;
  }
  return H3DIT_OK;
}

// x_0 rows from the text rows and the two modalities' patch projections.
h3dit_status build_x0(const h3dit_shape* s, const Dims& m, const h3dit_ends* e,
                      const float* z_video, const float* z_audio, __nv_bfloat16* x,
                      cudaStream_t st) {
  const int T = s->n_text, Aud = s->n_audio, D = m.D;
  if (T > 0 && cudaMemcpyAsync(x, e->text, (size_t)T * D * 2, cudaMemcpyDeviceToDevice, st) !=
                   cudaSuccess)
    return H3DIT_ERR_CUDA;
  if (Aud > 0)
    H3_TRY(cu(counted(launch_patch_in(z_audio, e->w_in_audio, e->b_in_audio, x + (size_t)T * D,
                                      Aud, e->c_audio, D, st), 1)));
  return cu(counted(launch_patch_in(z_video, e->w_in_video, e->b_in_video, x + (size_t)m.P * D,
                                    m.V, e->c_video, D, st), 1));
}

// Final AdaLN of one modality's rows [r0, r0 + rows) of x, then its output head with the
// Euler update fused: v = h W_out^T + b; v_out (if set) = v; z += dt v.
h3dit_status head_pass(const Dims& m, const Ws& w, void* ws, const __nv_bfloat16* x, int r0,
                       int rows, int c, const float* mod2, const void* w_out, const void* b_out,
                       float* z, float* v_out, float dt, float eps, cudaStream_t st) {
  if (rows <= 0) return H3DIT_OK;
  const int D = m.D;
  __nv_bfloat16* h = at<__nv_bfloat16>(ws, w.h) + (size_t)r0 * D;
  H3_TRY(cu(counted(launch_rms_modulate(x + (size_t)r0 * D, mod2, mod2 + D, nullptr, nullptr, 0,
                                        h, rows, D, eps, st), 1)));
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.a = h;
  g.w = static_cast<const __nv_bfloat16*>(w_out);
  g.M = rows;
  g.N = c;
  g.K = D;
  g.bias = static_cast<const __nv_bfloat16*>(b_out);
  g.z = z;
  g.v_out = v_out;
  g.dt = dt;
  g.status = at<int>(ws, w.status);
  return cu(counted(launch_gemm(kEpiHeadEuler, g, st), 1));
}

}  // namespace
}  // namespace h3

using namespace h3;

extern "C" {

const char* h3dit_version(void) { return "h3dit 0.1.0 sm_103a"; }

const char* h3dit_status_string(h3dit_status s) {
  switch (s) {
    case H3DIT_OK: return "ok";
    case H3DIT_ERR_ARG: return "invalid argument";
    case H3DIT_ERR_SHAPE: return "unsupported or inconsistent shape";
    case H3DIT_ERR_ALIGN: return "pointer not 16-byte aligned";
    case H3DIT_ERR_WORKSPACE: return "workspace missing or too small";
    case H3DIT_ERR_CUDA: return "CUDA call failed";
    case H3DIT_ERR_TIMEOUT: return "a kernel wait timed out";
    case H3DIT_ERR_UNSUPPORTED: return "unsupported device or feature";
  }
  return "unknown status";
}

h3dit_status h3dit_check_shape(const h3dit_shape* shape) {
  Dims m;
  return check_block(shape, &m);
}

size_t h3dit_workspace_bytes(const h3dit_shape* shape) {
  Dims m;
  if (!shape) return 0;
  if (shape->hidden == 0 && shape->mlp_width == 0) {
    if (check_attn(shape, &m) != H3DIT_OK) return 0;
  } else if (check_block(shape, &m) != H3DIT_OK) {
    return 0;
  }
  return plan(m).total;
}

h3dit_status h3dit_get_workspace_layout(const h3dit_shape* shape, h3dit_workspace_layout* out) {
  if (!shape || !out) return H3DIT_ERR_ARG;
  Dims m;
  if (shape->hidden == 0 && shape->mlp_width == 0)
    H3_TRY(check_attn(shape, &m));
  else
    H3_TRY(check_block(shape, &m));
  const Ws w = plan(m);
  out->status = w.status;
  out->q = w.q;
  out->k = w.k;
  out->v = w.v;
  out->g = w.g;
  out->o = w.o;
  out->u = w.u;
  out->h = w.h;
  out->x1 = w.x1;
  out->means = w.means;
  out->scores = w.scores;
  out->idx = w.idx;
  out->pooled = w.pooled;
  out->total = w.total;
  return H3DIT_OK;
}

h3dit_status h3dit_block_forward(const h3dit_shape* shape, const h3dit_block_weights* w,
                                 void* x_inout, void* workspace, size_t ws_bytes, void* stream) {
  Dims m;
  H3_TRY(check_block(shape, &m));
  H3_TRY(check_weights(shape, w));
  if (!x_inout || !workspace) return H3DIT_ERR_ARG;
  if (!aligned16(x_inout) || !aligned16(workspace)) return H3DIT_ERR_ALIGN;
  const Ws ws = plan(m);
  if (ws_bytes < ws.total) return H3DIT_ERR_WORKSPACE;
  H3_TRY(device_ok());
  return run_block(shape, m, ws, workspace, w, static_cast<__nv_bfloat16*>(x_inout), false,
                   static_cast<cudaStream_t>(stream));
}

h3dit_status h3dit_routed_attention(const h3dit_shape* shape, const void* q, const void* k,
                                    const void* v, const void* gate_or_null, void* out,
                                    float* pooled_out_or_null, int* topk_idx_out_or_null,
                                    float* tile_scores_out_or_null, void* workspace,
                                    size_t ws_bytes, void* stream) {
  Dims m;
  H3_TRY(check_attn(shape, &m));
  m.block = false;
  if (!q || !k || !v || !out || !workspace) return H3DIT_ERR_ARG;
  const void* ptrs[] = {q, k, v, out, workspace, gate_or_null, pooled_out_or_null,
                        topk_idx_out_or_null, tile_scores_out_or_null};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return H3DIT_ERR_ALIGN;
  const Ws ws = plan(m);
  if (ws_bytes < ws.total) return H3DIT_ERR_WORKSPACE;
  H3_TRY(device_ok());
  return run_attention(shape, m, ws, workspace, static_cast<const __nv_bfloat16*>(q),
                       static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v),
                       static_cast<const __nv_bfloat16*>(gate_or_null),
                       static_cast<__nv_bfloat16*>(out), pooled_out_or_null,
                       topk_idx_out_or_null, tile_scores_out_or_null,
                       static_cast<cudaStream_t>(stream));
}

h3dit_status h3dit_denoise_step(const h3dit_shape* shape, const h3dit_block_weights* blocks,
                                const int* block_ids, int n_blocks, float* z_inout,
                                float* v_ring, int fresh, const h3dit_schedule* video,
                                const h3dit_schedule* prefix_or_null, int n_fresh_so_far,
                                void* workspace, size_t ws_bytes, void* stream) {
  Dims m;
  H3_TRY(check_block(shape, &m));
  if (!z_inout || !v_ring || !workspace || !video) return H3DIT_ERR_ARG;
  if (!aligned16(z_inout) || !aligned16(v_ring) || !aligned16(workspace)) return H3DIT_ERR_ALIGN;
  if (n_fresh_so_far < 0) return H3DIT_ERR_ARG;
  const h3dit_schedule* pre = prefix_or_null ? prefix_or_null : video;
  const Ws ws = plan(m);
  if (ws_bytes < ws.total) return H3DIT_ERR_WORKSPACE;
  const size_t n = (size_t)m.N * m.D;
  const size_t n_pre = (size_t)m.P * m.D;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (fresh) {
    if (!blocks || (n_blocks > 0 && !block_ids) || n_blocks < 0) return H3DIT_ERR_ARG;
    for (int i = 0; i < n_blocks; ++i) {
      if (block_ids[i] < 0) return H3DIT_ERR_ARG;
      H3_TRY(check_weights(shape, &blocks[block_ids[i]]));
    }
    H3_TRY(device_ok());
    __nv_bfloat16* x = at<__nv_bfloat16>(workspace, ws.x);
    {
      StageScope sc(H3DIT_STAGE_SAMPLER, st);
      H3_TRY(cu(counted(launch_f32_to_bf16(z_inout, x, n, st), 1)));
      if (shape->flags & H3DIT_ROPE)
        H3_TRY(cu(counted(launch_rope_table(at<float2>(workspace, ws.rope), m.N, m.d,
                                            shape->rope_theta, m.geom, st), 1)));
    }
    for (int i = 0; i < n_blocks; ++i)
      H3_TRY(run_block(shape, m, ws, workspace, &blocks[block_ids[i]], x, true, st));
    float* slot = v_ring + (size_t)(n_fresh_so_far % 2) * n;
    StageScope sc(H3DIT_STAGE_SAMPLER, st);
    return cu(counted(launch_euler_fresh(x, z_inout, slot, video->dt, pre->dt, n_pre, n, st), 1));
  }
  if (n_fresh_so_far < 1) return H3DIT_ERR_ARG;  // nothing to extrapolate from
  const float* va = v_ring + (size_t)((n_fresh_so_far - 1) % 2) * n;
  const float* vb = n_fresh_so_far >= 2 ? v_ring + (size_t)(n_fresh_so_far % 2) * n : nullptr;
  float coef_v = 0.f, coef_p = 0.f;
  if (vb && (video->sigma_a == video->sigma_b || pre->sigma_a == pre->sigma_b))
    return H3DIT_ERR_ARG;  // no slope to extrapolate along
  H3_TRY(device_ok());
  if (vb) {
    coef_v = (float)(((double)video->sigma_i - video->sigma_a) /
                     ((double)video->sigma_a - video->sigma_b));
    coef_p = (float)(((double)pre->sigma_i - pre->sigma_a) / ((double)pre->sigma_a - pre->sigma_b));
  }
  StageScope sc(H3DIT_STAGE_SAMPLER, st);
  return cu(counted(launch_euler_extrap(z_inout, va, vb, coef_v, video->dt, coef_p, pre->dt, n_pre,
                                        n, st), 1));
}

h3dit_status h3dit_sample_step(const h3dit_shape* shape, const h3dit_ends* ends,
                               const h3dit_block_weights* blocks, const int* block_ids,
                               int n_blocks, float* z_video, float* z_audio,
                               float* v_ring_video, float* v_ring_audio, float* core_residual,
                               const h3dit_reduction* reduction, int pass,
                               const h3dit_schedule* video, const h3dit_schedule* audio,
                               int n_fresh_so_far, void* workspace, size_t ws_bytes,
                               void* stream) {
  Dims m;
  H3_TRY(check_block(shape, &m));
  H3_TRY(check_ends(shape, ends));
  const bool has_audio = shape->n_audio > 0;
  if (!video || (has_audio && !audio) || !workspace || !z_video) return H3DIT_ERR_ARG;
  if (has_audio && !z_audio) return H3DIT_ERR_ARG;
  if (pass != H3DIT_PASS_FRESH && pass != H3DIT_PASS_EXTRAPOLATE &&
      pass != H3DIT_PASS_CORE_REUSE)
    return H3DIT_ERR_ARG;
  if (n_fresh_so_far < 0) return H3DIT_ERR_ARG;
  const void* ptrs[] = {z_video, z_audio, v_ring_video, v_ring_audio, core_residual, workspace};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return H3DIT_ERR_ALIGN;
  if (pass != H3DIT_PASS_CORE_REUSE && (!v_ring_video || (has_audio && !v_ring_audio)))
    return H3DIT_ERR_ARG;
  if (pass == H3DIT_PASS_CORE_REUSE && !core_residual) return H3DIT_ERR_ARG;
  const Ws ws = plan(m);
  if (ws_bytes < ws.total) return H3DIT_ERR_WORKSPACE;
  const int cv = ends->c_video, ca = has_audio ? ends->c_audio : 0;
  const size_t nv = (size_t)m.V * cv, na = (size_t)shape->n_audio * ca;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  if (pass == H3DIT_PASS_EXTRAPOLATE) {
    if (n_fresh_so_far < 1) return H3DIT_ERR_ARG;  // nothing to extrapolate from
    const bool two = n_fresh_so_far >= 2;
    if (two && (video->sigma_a == video->sigma_b ||
                (has_audio && audio->sigma_a == audio->sigma_b)))
      return H3DIT_ERR_ARG;
    H3_TRY(device_ok());
    auto coef = [](const h3dit_schedule* sc) {
      return (float)(((double)sc->sigma_i - sc->sigma_a) / ((double)sc->sigma_a - sc->sigma_b));
    };
    const size_t sa = (size_t)((n_fresh_so_far - 1) % 2), sb = (size_t)(n_fresh_so_far % 2);
    StageScope sc(H3DIT_STAGE_SAMPLER, st);
    H3_TRY(cu(counted(launch_euler_extrap(z_video, v_ring_video + sa * nv,
                                          two ? v_ring_video + sb * nv : nullptr,
                                          two ? coef(video) : 0.f, video->dt, 0.f, 0.f, 0, nv,
                                          st), 1)));
    if (has_audio)
      H3_TRY(cu(counted(launch_euler_extrap(z_audio, v_ring_audio + sa * na,
                                            two ? v_ring_audio + sb * na : nullptr,
                                            two ? coef(audio) : 0.f, audio->dt, 0.f, 0.f, 0, na,
                                            st), 1)));
    return H3DIT_OK;
  }

  // token reduction over block positions [red_first, red_last)
  int red_first = -1, red_last = -1;
  h3dit_shape rshape;
  Dims rm;
  if (pass == H3DIT_PASS_FRESH && reduction && reduction->first >= 0 &&
      reduction->first < reduction->last && reduction->first < n_blocks) {
    if (!m.reduce) return H3DIT_ERR_SHAPE;  // buffers not reserved (H3DIT_TOKEN_REDUCTION)
    H3_TRY(reduced_dims(shape, &rshape, &rm));
    red_first = reduction->first;
    red_last = reduction->last < n_blocks ? reduction->last : n_blocks;
  }
  if (pass == H3DIT_PASS_FRESH) {
    if (!blocks || (n_blocks > 0 && !block_ids) || n_blocks < 0) return H3DIT_ERR_ARG;
    for (int i = 0; i < n_blocks; ++i) {
      if (block_ids[i] < 0) return H3DIT_ERR_ARG;
      H3_TRY(check_weights(shape, &blocks[block_ids[i]]));
    }
  }
  H3_TRY(device_ok());
  __nv_bfloat16* x = at<__nv_bfloat16>(workspace, ws.x);
  const size_t nd = (size_t)m.N * m.D;
  {
    StageScope sc(H3DIT_STAGE_SAMPLER, st);
    H3_TRY(build_x0(shape, m, ends, z_video, z_audio, x, st));
    if (pass == H3DIT_PASS_CORE_REUSE)
      H3_TRY(cu(counted(launch_core_residual(x, core_residual, nd, 2, st), 1)));
    if (pass == H3DIT_PASS_FRESH) {
      if (core_residual) H3_TRY(cu(counted(launch_core_residual(x, core_residual, nd, 0, st), 1)));
      if ((shape->flags & H3DIT_ROPE) && n_blocks > 0)
        H3_TRY(cu(counted(launch_rope_table(at<float2>(workspace, ws.rope), m.N, m.d,
                                            shape->rope_theta, m.geom, st), 1)));
    }
  }
  __nv_bfloat16* cur = x;  // the full-resolution rows (the bypass after a restore)
  if (pass == H3DIT_PASS_FRESH) {
    __nv_bfloat16* bypass = m.reduce ? at<__nv_bfloat16>(workspace, ws.bypass) : nullptr;
    __nv_bfloat16* base = m.reduce ? at<__nv_bfloat16>(workspace, ws.base) : nullptr;
    float2* rope = at<float2>(workspace, ws.rope);
    const bool use_rope = (shape->flags & H3DIT_ROPE) != 0;
    for (int i = 0; i < n_blocks; ++i) {
      if (i == red_first) {  // pool: bypass <- x; x <- [prefix rows; pooled video rows]
        StageScope sc(H3DIT_STAGE_SAMPLER, st);
        if (cudaMemcpyAsync(bypass, x, nd * 2, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
          return H3DIT_ERR_CUDA;
        H3_TRY(cu(counted(launch_token_pool(bypass, x, base, m.geom, rm.geom, m.D, st), 1)));
        if (use_rope)
          H3_TRY(cu(counted(launch_rope_table(rope, rm.N, rm.d, shape->rope_theta, rm.geom, st),
                            1)));
      }
      if (i == red_last) {  // restore into the bypass, which holds the full rows from here
        StageScope sc(H3DIT_STAGE_SAMPLER, st);
        if (cudaMemcpyAsync(bypass, x, (size_t)m.P * m.D * 2, cudaMemcpyDeviceToDevice, st) !=
            cudaSuccess)
          return H3DIT_ERR_CUDA;
        H3_TRY(cu(counted(launch_token_restore(bypass, x, base, m.geom, rm.geom, m.D, st), 1)));
        if (use_rope)
          H3_TRY(cu(counted(launch_rope_table(rope, m.N, m.d, shape->rope_theta, m.geom, st),
                            1)));
        cur = bypass;
      }
      const bool reduced = red_first >= 0 && i >= red_first && i < red_last;
      if (reduced)
        H3_TRY(run_block(&rshape, rm, ws, workspace, &blocks[block_ids[i]], x, true, st));
      else
        H3_TRY(run_block(shape, m, ws, workspace, &blocks[block_ids[i]], cur, true, st));
    }
    if (red_first >= 0 && red_last == n_blocks) {  // restore after the last block
      StageScope sc(H3DIT_STAGE_SAMPLER, st);
      if (cudaMemcpyAsync(bypass, x, (size_t)m.P * m.D * 2, cudaMemcpyDeviceToDevice, st) !=
          cudaSuccess)
        return H3DIT_ERR_CUDA;
      H3_TRY(cu(counted(launch_token_restore(bypass, x, base, m.geom, rm.geom, m.D, st), 1)));
      cur = bypass;
    }
    if (core_residual) {
      StageScope sc(H3DIT_STAGE_SAMPLER, st);
      H3_TRY(cu(counted(launch_core_residual(cur, core_residual, nd, 1, st), 1)));
    }
  }
  const bool fresh = pass == H3DIT_PASS_FRESH;
  const size_t slot = (size_t)(n_fresh_so_far % 2);
  StageScope sc(H3DIT_STAGE_SAMPLER, st);
  H3_TRY(head_pass(m, ws, workspace, cur, m.P, m.V, cv, ends->mod_out_video, ends->w_out_video,
                   ends->b_out_video, z_video, fresh ? v_ring_video + slot * nv : nullptr,
                   video->dt, shape->rms_eps, st));
  if (has_audio)
    H3_TRY(head_pass(m, ws, workspace, cur, shape->n_text, shape->n_audio, ca, ends->mod_out_audio,
                     ends->w_out_audio, ends->b_out_audio, z_audio,
                     fresh ? v_ring_audio + slot * na : nullptr, audio->dt, shape->rms_eps, st));
  return H3DIT_OK;
}

h3dit_status h3dit_select_blocks(const float* mods, int n_blocks, int hidden, int keep,
                                 int* kept_ids) {
  if (!mods || !kept_ids || n_blocks < 1 || hidden < 1 || keep < 1) return H3DIT_ERR_ARG;
  if (keep >= n_blocks) {
    for (int b = 0; b < n_blocks; ++b) kept_ids[b] = b;
    return H3DIT_OK;
  }
  if (keep < 2) return H3DIT_ERR_ARG;
  double* score = new double[n_blocks];
  char* dropped = new char[n_blocks];
  for (int b = 0; b < n_blocks; ++b) {
    const float* g1 = mods + ((size_t)b * 6 + 2) * hidden;
    const float* g2 = mods + ((size_t)b * 6 + 5) * hidden;
    double s1 = 0.0, s2 = 0.0;
    for (int c = 0; c < hidden; ++c) {
      s1 += (double)g1[c] * g1[c];
      s2 += (double)g2[c] * g2[c];
    }
    score[b] = sqrt(s1) + sqrt(s2);
    dropped[b] = 0;
  }
  for (int r = 0; r < n_blocks - keep; ++r) {
    int best = -1;
    for (int b = 1; b < n_blocks - 1; ++b) {
      if (dropped[b]) continue;
      if (best < 0 || score[b] < score[best] || (score[b] == score[best] && b > best)) best = b;
    }
    dropped[best] = 1;
  }
  int n = 0;
  for (int b = 0; b < n_blocks; ++b)
    if (!dropped[b]) kept_ids[n++] = b;
  delete[] score;
  delete[] dropped;
  return H3DIT_OK;
}

h3dit_status h3dit_tile_spans(const h3dit_shape* shape, int* first_row, int* n_rows,
                              int* n_tiles_inout) {
  if (!shape || !n_tiles_inout) return H3DIT_ERR_ARG;
  Dims m;
  H3_TRY(check_attn(shape, &m));
  const int cap = *n_tiles_inout;
  *n_tiles_inout = m.Tv;
  if (cap < m.Tv || !first_row || !n_rows) return H3DIT_ERR_ARG;
  for (int t = 0; t < m.Tv; ++t) tile_span(m.geom, t, &first_row[t], &n_rows[t]);
  return H3DIT_OK;
}

h3dit_status h3dit_video_order(const h3dit_shape* shape, int* raster_index) {
  if (!shape || !raster_index) return H3DIT_ERR_ARG;
  Dims m;
  H3_TRY(check_attn(shape, &m));
  const TileGeom& g = m.geom;
  for (int i = 0; i < m.V; ++i) {
    if (g.gt == 0) {
      raster_index[i] = i;
    } else {
      int t, h, w;
      video_coord(g, i, &t, &h, &w);
      raster_index[i] = (t * g.gh + h) * g.gw + w;
    }
  }
  return H3DIT_OK;
}

h3dit_status h3dit_linear(const void* a, const void* w, const void* b_or_null, void* y, int M,
                          int N, int K, void* stream) {
  if (!a || !w || !y) return H3DIT_ERR_ARG;
  if (M < 1 || N < 256 || N % 256 || K < 64 || K % 64) return H3DIT_ERR_SHAPE;
  if (!aligned16(a) || !aligned16(w) || !aligned16(y) || (b_or_null && !aligned16(b_or_null)))
    return H3DIT_ERR_ALIGN;
  H3_TRY(device_ok());
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.a = static_cast<const __nv_bfloat16*>(a);
  g.w = static_cast<const __nv_bfloat16*>(w);
  g.M = M;
  g.N = N;
  g.K = K;
  g.bias = static_cast<const __nv_bfloat16*>(b_or_null);
  g.y = static_cast<__nv_bfloat16*>(y);
  return cu(counted(launch_gemm(kEpiStore, g, static_cast<cudaStream_t>(stream)), 1));
}

unsigned long long h3dit_launch_count(void) { return g_launches.load(); }

int h3dit_gemm_cta_pairs(int enable) { return gemm_cta_pairs(enable) ? 1 : 0; }

h3dit_status h3dit_profile_begin(int max_records) {
  if (g_prof.on || max_records < 1 || max_records > (1 << 20)) return H3DIT_ERR_ARG;
  g_prof.ev.assign(2 * (size_t)max_records, nullptr);
  for (auto& e : g_prof.ev) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      for (auto& f : g_prof.ev)
        if (f) cudaEventDestroy(f);
      g_prof.ev.clear();
      return H3DIT_ERR_CUDA;
    }
  }
  g_prof.stage.assign(max_records, -1);
  g_prof.nlaunch.assign(max_records, 0);
  g_prof.max = max_records;
  g_prof.used = 0;
  g_prof.on = true;
  return H3DIT_OK;
}

h3dit_status h3dit_profile_end(float* stage_ms, int* stage_launches, int n_stages) {
  if (!g_prof.on) return H3DIT_ERR_ARG;
  g_prof.on = false;
  h3dit_status rc = H3DIT_OK;
  for (int i = 0; i < n_stages; ++i) {
    if (stage_ms) stage_ms[i] = 0.f;
    if (stage_launches) stage_launches[i] = 0;
  }
  for (int r = 0; r < g_prof.used; ++r) {
    float ms = 0.f;
    if (cudaEventSynchronize(g_prof.ev[2 * r + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_prof.ev[2 * r], g_prof.ev[2 * r + 1]) != cudaSuccess) {
      rc = H3DIT_ERR_CUDA;
      continue;
    }
    const int sidx = g_prof.stage[r];
    if (sidx >= 0 && sidx < n_stages) {
      if (stage_ms) stage_ms[sidx] += ms;
      if (stage_launches) stage_launches[sidx] += g_prof.nlaunch[r];
    }
  }
  for (auto& e : g_prof.ev) cudaEventDestroy(e);
  g_prof.ev.clear();
  g_prof.used = g_prof.max = 0;
  return rc;
}

h3dit_status h3dit_sync_status(void* workspace, size_t ws_bytes, void* stream) {
  if (!workspace || ws_bytes < sizeof(int)) return H3DIT_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return H3DIT_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return H3DIT_ERR_CUDA;
  if (v != 0 && cudaMemset(workspace, 0, sizeof(int)) != cudaSuccess) return H3DIT_ERR_CUDA;
  return v == 0 ? H3DIT_OK : static_cast<h3dit_status>(v);
}

}  // extern "C"
