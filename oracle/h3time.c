/*
 * h3time.c -- the CPU timing baseline: one routed-attention DiT block in float32.
 *
 * Test and measurement infrastructure only: bench.py times it on the host's cores
 * beside the GPU library, and tests/test_oracle_time.py checks it against the
 * float64 oracle (oracle/h3block.py); the product library never links, loads or
 * calls it, and it shares no code with the CUDA path or with the other oracles.
 *
 * It computes the same steps as the float64 oracle, in the same order, with the same
 * readings (listed there and in oracle/h3ref.c), but in float32 arithmetic, with the
 * linear weights stored input-major so that every inner loop is a contiguous
 * multiply-add the compiler can vectorise, and with OpenMP threads over rows, heads
 * and query tiles.  Sources (page title and section): "ashhart/TensorFold pull
 * request #949" -- "What it adds" (block.zig: modulated norm, q/k/v and the routing
 * gate, head layout, routing, attention, pooled branch, out projection, MLP;
 * h3_routing.metal: tile means, scores, top-k; h3_attention.metal: tile-routed
 * attention), "Precision" (bf16 weights and activations, fp32 sums and routing,
 * softmax weights rounded to bf16 before the value product), "Kernel contract"
 * (top-k: NaN ranks as -inf, ties go to the lower tile); "Antirez/h3.c: MiniMax H3
 * inference engine for Mac computers" -- the fused gated-AdaLN, Q/K RMS + RoPE and
 * SwiGLU paragraphs.  Video tiles are contiguous 64-row slices; rotary over the
 * packed row index.
 *
 * Sampling (for a bounded timing run): with sample = s > 1 only every s-th 64-row
 * chunk of rows runs the row-local stages (norms, projections, MLP), only every s-th
 * video query tile and every s-th prefix chunk of 64 query rows runs attention, and
 * the router runs over all tiles; the other rows keep whatever the scratch held.  The
 * work done is then about 1/s of a block (plus the router), for timing only: the
 * values of a sampled call are not a block's output.  sample = 1 is the whole block.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int n_text, n_audio, n_video;
  int hidden, heads, head_dim, mlp_width, topk;
  int qk_norm, rope, pooled, swiglu;
  float eps, theta;
} h3time_shape;

typedef struct {
  /* bf16 values held as float; linear weights INPUT-major: w_t[in][out] */
  const float *w_qkvg_t, *b_qkvg; /* [D][4A], [4A]: output columns q, k, v, g, head-major */
  const float *w_o_t, *b_o;       /* [A][D], [D] */
  const float *w1_t, *b1;         /* [D][F] (GELU) or [D][2F] (SwiGLU), bias likewise */
  const float *w2_t, *b2;         /* [F][D], [D] */
  const float *mod;               /* [6][D]: shift1, scale1, gate1, shift2, scale2, gate2 */
  const float *mod_prefix;        /* [6][D] for the text and audio rows, or NULL */
  const float *qnorm_w, *knorm_w; /* [d] */
} h3time_weights;

enum { TILE = 64, RB = 32, CB = 256, KB = 256 };

static float bf16f(float x) {
  /* nearest bf16, ties to even (the storage type of TensorFold #949 "Precision") */
  uint32_t u;
  memcpy(&u, &x, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) return x;
  u += 0x7fffu + ((u >> 16) & 1u);
  u &= 0xffff0000u;
  memcpy(&x, &u, 4);
  return x;
}

int h3time_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------ scratch layout */
typedef struct {
  size_t h, qkvg, q, k, kt, v, g, o, u, means, scores, pooled, idx, total;
} layout_t;

static layout_t plan(const h3time_shape* s) {
  const size_t N = (size_t)s->n_text + s->n_audio + s->n_video, D = s->hidden;
  const size_t H = s->heads, d = s->head_dim, A = H * d, F = s->mlp_width;
  const size_t Tv = (s->n_video + TILE - 1) / TILE, k = s->topk < (int)Tv ? s->topk : Tv;
  const size_t F1 = s->swiglu ? 2 * F : F;
  layout_t L;
  size_t off = 0;
#define TAKE(field, n) (L.field = off, off += (n))
  TAKE(h, N * D);
  TAKE(qkvg, N * (4 * A > F1 ? 4 * A : F1)); /* projection outputs, then fc1 outputs */
  TAKE(q, H * N * d);
  TAKE(k, H * N * d);
  TAKE(kt, H * d * N); /* k transposed per head: kt[h][c][n] */
  TAKE(v, H * N * d);
  TAKE(g, N * A);
  TAKE(o, N * A);
  TAKE(u, N * F);
  TAKE(means, 3 * H * Tv * d);
  TAKE(scores, H * Tv * Tv);
  TAKE(pooled, H * Tv * d);
  TAKE(idx, H * Tv * k); /* int32 stored in float-sized slots */
#undef TAKE
  L.total = off;
  return L;
}

size_t h3time_scratch_floats(const h3time_shape* s) { return plan(s).total; }

/* ------------------------------------------------------------------ row steps */

/* rows of the block that run the row-local stages (every sample-th 64-row chunk) */
static int active_rows(int N, int sample, int* rows) {
  int n = 0;
  for (int r = 0; r < N; ++r)
    if ((r / TILE) % sample == 0) rows[n++] = r;
  return n;
}

/* h = bf16(x / sqrt(mean(x^2) + eps) * (1 + scale) + shift) per row (TensorFold #949
 * "What it adds": modulated norm; h3.c README fused gated-AdaLN: per-row RMS). */
static void modulate(const float* x, float* h, const int* rows, int nr, int D, int P,
                     const float* mod, const float* modp, int i_shift, int i_scale, float eps) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < nr; ++t) {
    const int r = rows[t];
    const float* m = (modp && r < P) ? modp : mod;
    const float* xr = x + (size_t)r * D;
    float ss = 0.f;
    for (int c = 0; c < D; ++c) ss += xr[c] * xr[c];
    const float inv = 1.0f / sqrtf(ss / (float)D + eps);
    float* hr = h + (size_t)r * D;
    for (int c = 0; c < D; ++c)
      hr[c] = bf16f(xr[c] * inv * (1.0f + m[i_scale * D + c]) + m[i_shift * D + c]);
  }
}

/* C[r][:] = A[r][:] Bt + bias for the listed rows; Bt input-major [K][N]; fp32 sums. */
static void linear(const float* A, int K, const float* Bt, const float* bias, int N, float* C,
                   const int* rows, int nr) {
  const int nblk = (nr + RB - 1) / RB;
#pragma omp parallel for schedule(dynamic, 1)
  for (int b = 0; b < nblk; ++b) {
    const int t0 = b * RB, t1 = t0 + RB < nr ? t0 + RB : nr;
    float acc[RB][CB];
    for (int n0 = 0; n0 < N; n0 += CB) {
      const int nn = N - n0 < CB ? N - n0 : CB;
      for (int t = t0; t < t1; ++t)
        for (int j = 0; j < nn; ++j) acc[t - t0][j] = bias ? bias[n0 + j] : 0.f;
      for (int kk = 0; kk < K; ++kk) {
        const float* bk = Bt + (size_t)kk * N + n0;
        for (int t = t0; t < t1; ++t) {
          const float a = A[(size_t)rows[t] * K + kk];
          float* c = acc[t - t0];
          for (int j = 0; j < nn; ++j) c[j] += a * bk[j];
        }
      }
      for (int t = t0; t < t1; ++t) memcpy(C + (size_t)rows[t] * N + n0, acc[t - t0], nn * 4);
    }
  }
}

/* q, k: per-head RMS norm x learned weight, then rotate-half rotary over the packed index
 * (pairs (c, c + d/2), angle p theta^(-2c/d)); v, g: the projection's bf16 values. */
static void heads(const h3time_shape* s, const float* w_q, const float* w_k, const float* qkvg,
                  float* q, float* k, float* kt, float* v, float* g, const int* rows, int nr) {
  const int N = s->n_text + s->n_audio + s->n_video, H = s->heads, d = s->head_dim;
  const int A = H * d;
  /* rotary angles of pair c: theta^(-2c/d), turned by the row's packed index */
  double inv_freq[128];
  for (int c = 0; c < d / 2; ++c) inv_freq[c] = pow((double)s->theta, -2.0 * c / d);
#pragma omp parallel for schedule(static)
  for (int t = 0; t < nr; ++t) {
    const int r = rows[t];
    const float* row = qkvg + (size_t)r * 4 * A;
    float tmp[256], rc[128], rs[128];
    if (s->rope)
      for (int c = 0; c < d / 2; ++c) {
        rc[c] = (float)cos((double)r * inv_freq[c]);
        rs[c] = (float)sin((double)r * inv_freq[c]);
      }
    for (int hh = 0; hh < H; ++hh) {
      for (int slab = 0; slab < 2; ++slab) {
        const float* src = row + slab * A + hh * d;
        const float* nw = slab == 0 ? w_q : w_k;
        for (int c = 0; c < d; ++c) tmp[c] = src[c];
        if (s->qk_norm) {
          float ss = 0.f;
          for (int c = 0; c < d; ++c) ss += tmp[c] * tmp[c];
          const float inv = 1.0f / sqrtf(ss / (float)d + s->eps);
          for (int c = 0; c < d; ++c) tmp[c] = tmp[c] * inv * nw[c];
        }
        if (s->rope) {
          for (int c = 0; c < d / 2; ++c) {
            const float a = tmp[c], b = tmp[c + d / 2];
            tmp[c] = a * rc[c] - b * rs[c];
            tmp[c + d / 2] = b * rc[c] + a * rs[c];
          }
        }
        float* dst = (slab == 0 ? q : k) + ((size_t)hh * N + r) * d;
        for (int c = 0; c < d; ++c) dst[c] = bf16f(tmp[c]);
        if (slab == 1)
          for (int c = 0; c < d; ++c) kt[((size_t)hh * d + c) * N + r] = dst[c];
      }
      memcpy(v + ((size_t)hh * N + r) * d, row + 2 * A + hh * d, d * 4);
      memcpy(g + (size_t)r * A + hh * d, row + 3 * A + hh * d, d * 4);
    }
  }
}

/* ------------------------------------------------------------------ router */

/* fp32 means of every 64-row video tile (valid rows only), tile scores mq . mk (unscaled),
 * top-k under (score desc, index asc) with NaN as -inf, and the pooled branch
 * op_i = sum_j softmax_j(S_ij / sqrt(d)) mv_j (TensorFold #949 h3_routing.metal). */
static void router(const h3time_shape* s, const float* q, const float* k, const float* v,
                   float* means, float* scores, int* idx, float* pooled) {
  const int N = s->n_text + s->n_audio + s->n_video, P = s->n_text + s->n_audio;
  const int H = s->heads, d = s->head_dim, Tv = (s->n_video + TILE - 1) / TILE;
  const int kk = s->topk < Tv ? s->topk : Tv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int hh = 0; hh < H; ++hh) {
    for (int which = 0; which < 3; ++which) {
      const float* src = (which == 0 ? q : which == 1 ? k : v) + (size_t)hh * N * d;
      for (int t = 0; t < Tv; ++t) {
        float* m = means + (((size_t)which * H + hh) * Tv + t) * d;
        const int r0 = P + t * TILE, r1 = r0 + TILE < N ? r0 + TILE : N;
        for (int c = 0; c < d; ++c) m[c] = 0.f;
        for (int r = r0; r < r1; ++r)
          for (int c = 0; c < d; ++c) m[c] += src[(size_t)r * d + c];
        for (int c = 0; c < d; ++c) m[c] /= (float)(r1 - r0);
      }
    }
    const float* mq = means + ((size_t)0 * H + hh) * Tv * d;
    const float* mk = means + ((size_t)1 * H + hh) * Tv * d;
    const float* mv = means + ((size_t)2 * H + hh) * Tv * d;
    for (int i = 0; i < Tv; ++i) {
      float* srow = scores + ((size_t)hh * Tv + i) * Tv;
      for (int j = 0; j < Tv; ++j) {
        float acc = 0.f;
        for (int c = 0; c < d; ++c) acc += mq[(size_t)i * d + c] * mk[(size_t)j * d + c];
        srow[j] = acc;
      }
      int n = 0;
      for (int j = 0; j < Tv; ++j) {
        const float sj = isnan(srow[j]) ? -INFINITY : srow[j];
        int ahead = 0;
        for (int j2 = 0; j2 < Tv && ahead < kk; ++j2) {
          const float s2 = isnan(srow[j2]) ? -INFINITY : srow[j2];
          if (s2 > sj || (s2 == sj && j2 < j)) ++ahead;
        }
        if (ahead < kk) idx[((size_t)hh * Tv + i) * kk + n++] = j;
      }
      if (pooled) {
        const float sc = 1.0f / sqrtf((float)d);
        float mx = -INFINITY, l = 0.f;
        for (int j = 0; j < Tv; ++j) mx = fmaxf(mx, srow[j] * sc);
        float* op = pooled + ((size_t)hh * Tv + i) * d;
        for (int c = 0; c < d; ++c) op[c] = 0.f;
        for (int j = 0; j < Tv; ++j) {
          const float w = expf(srow[j] * sc - mx);
          l += w;
          for (int c = 0; c < d; ++c) op[c] += w * mv[(size_t)j * d + c];
        }
        for (int c = 0; c < d; ++c) op[c] /= l;
      }
    }
  }
}

/* ------------------------------------------------------------------ attention */

/* Attention of nq query rows against nk keys (kt [d][ldk] transposed keys, vv [nk][d]
 * values, both for this key set): scores in fp32, weights 2^(s log2 e - M) with M the
 * row's largest score rounded up to a whole number, rounded to bf16 before the value
 * product, the row sum from the unrounded weights.  sbuf holds nq x nk scores. */
static void attend(const float* qrows, int nq, const float* kt, int ldk, const float* vv,
                   int nk, int d, float* out, float* sbuf) {
  const float sl2 = (float)(1.4426950408889634 / sqrt((double)d));
  for (int j0 = 0; j0 < nk; j0 += KB) {
    const int nj = nk - j0 < KB ? nk - j0 : KB;
    for (int r = 0; r < nq; ++r) {
      float* srow = sbuf + (size_t)r * nk + j0;
      for (int j = 0; j < nj; ++j) srow[j] = 0.f;
      for (int c = 0; c < d; ++c) {
        const float a = qrows[(size_t)r * d + c];
        const float* kc = kt + (size_t)c * ldk + j0;
        for (int j = 0; j < nj; ++j) srow[j] += a * kc[j];
      }
    }
  }
  float lsum[TILE];
  for (int r = 0; r < nq; ++r) {
    float* srow = sbuf + (size_t)r * nk;
    float mx = -INFINITY;
    for (int j = 0; j < nk; ++j) {
      srow[j] *= sl2;
      mx = fmaxf(mx, srow[j]);
    }
    const float M = ceilf(mx);
    float l = 0.f;
    for (int j = 0; j < nk; ++j) {
      const float p = exp2f(srow[j] - M);
      l += p;
      srow[j] = bf16f(p);
    }
    lsum[r] = l;
    for (int c = 0; c < d; ++c) out[(size_t)r * d + c] = 0.f;
  }
  for (int j0 = 0; j0 < nk; j0 += KB) {
    const int nj = nk - j0 < KB ? nk - j0 : KB;
    for (int r = 0; r < nq; ++r) {
      float* o = out + (size_t)r * d;
      const float* p = sbuf + (size_t)r * nk + j0;
      for (int j = 0; j < nj; ++j) {
        const float w = p[j];
        const float* vj = vv + (size_t)(j0 + j) * d;
        for (int c = 0; c < d; ++c) o[c] += w * vj[c];
      }
    }
  }
  for (int r = 0; r < nq; ++r)
    for (int c = 0; c < d; ++c) out[(size_t)r * d + c] /= lsum[r];
}

/* Prefix rows attend to all N rows; a video row of tile i to the prefix rows plus the
 * rows of its selected tiles; video rows then add g * pooled of their tile. */
static void attention(const h3time_shape* s, const float* q, const float* kt, const float* v,
                      const float* k, const float* g, const int* idx, const float* pooled,
                      float* o, int sample) {
  const int N = s->n_text + s->n_audio + s->n_video, P = s->n_text + s->n_audio;
  const int H = s->heads, d = s->head_dim, A = H * d, Tv = (s->n_video + TILE - 1) / TILE;
  const int kk = s->topk < Tv ? s->topk : Tv;
  const int n_pre = (P + TILE - 1) / TILE;
  const int units = n_pre + Tv;
#pragma omp parallel
  {
    const int nk_max = N;
    float* sbuf = (float*)malloc((size_t)TILE * nk_max * sizeof(float));
    float* ksel = (float*)malloc((size_t)d * nk_max * sizeof(float));
    float* vsel = (float*)malloc((size_t)nk_max * d * sizeof(float));
    float* ob = (float*)malloc((size_t)TILE * d * sizeof(float));
    float* qb = (float*)malloc((size_t)TILE * d * sizeof(float));
#pragma omp for schedule(dynamic, 1)
    for (int w = 0; w < H * units; ++w) {
      const int hh = w / units, u = w % units;
      const int prefix = u < n_pre;
      const int chunk = prefix ? u : u - n_pre;
      if (chunk % sample) continue;
      const int r0 = prefix ? u * TILE : P + chunk * TILE;
      const int lim = prefix ? P : N;
      const int nq = lim - r0 < TILE ? lim - r0 : TILE;
      const float* qh = q + (size_t)hh * N * d;
      const float* kth = kt + (size_t)hh * d * N;
      const float* vh = v + (size_t)hh * N * d;
      memcpy(qb, qh + (size_t)r0 * d, (size_t)nq * d * 4);
      if (prefix) {
        attend(qb, nq, kth, N, vh, N, d, ob, sbuf);
      } else {
        /* key set: prefix rows, then the selected tiles' rows, gathered contiguously */
        int nk = 0;
        const int* sel = idx + ((size_t)hh * Tv + chunk) * kk;
        for (int seg = -1; seg < kk; ++seg) {
          const int a = seg < 0 ? 0 : P + sel[seg] * TILE;
          const int b = seg < 0 ? P : (a + TILE < N ? a + TILE : N);
          for (int c = 0; c < d; ++c) memcpy(ksel + (size_t)c * N + nk, kth + (size_t)c * N + a,
                                             (size_t)(b - a) * 4);
          memcpy(vsel + (size_t)nk * d, vh + (size_t)a * d, (size_t)(b - a) * d * 4);
          nk += b - a;
        }
        attend(qb, nq, ksel, N, vsel, nk, d, ob, sbuf);
      }
      for (int r = 0; r < nq; ++r) {
        float* dst = o + (size_t)(r0 + r) * A + hh * d;
        for (int c = 0; c < d; ++c) {
          float val = ob[(size_t)r * d + c];
          if (!prefix && pooled)
            val += g[(size_t)(r0 + r) * A + hh * d + c] *
                   pooled[((size_t)hh * Tv + chunk) * d + c];
          dst[c] = bf16f(val);
        }
      }
    }
    free(sbuf);
    free(ksel);
    free(vsel);
    free(ob);
    free(qb);
  }
  (void)k;
}

/* ------------------------------------------------------------------ block */

static float gelu(float x) { return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f)); }
static float silu(float x) { return x / (1.0f + expf(-x)); }

/* One block, in place on x (float values of bf16 rows [N][D]); returns 0 or -1.
 * idx_out (optional) receives the top-k selections [H][Tv][k]. */
int h3time_block(const h3time_shape* s, const h3time_weights* w, float* x, float* scratch,
                 int sample, int* idx_out) {
  if (!s || !w || !x || !scratch || sample < 1 || s->head_dim > 256) return -1;
  const int N = s->n_text + s->n_audio + s->n_video, P = s->n_text + s->n_audio;
  const int D = s->hidden, H = s->heads, d = s->head_dim, A = H * d, F = s->mlp_width;
  const int Tv = (s->n_video + TILE - 1) / TILE;
  const int kk = s->topk < Tv ? s->topk : Tv;
  const layout_t L = plan(s);
  float* h = scratch + L.h;
  float* qkvg = scratch + L.qkvg;
  int* idx = (int*)(scratch + L.idx);
  int* rows = (int*)malloc((size_t)N * sizeof(int));
  if (!rows) return -1;
  const int nr = active_rows(N, sample, rows);

  /* a1-a3: modulated norm, q/k/v/gate projection, heads */
  modulate(x, h, rows, nr, D, P, w->mod, w->mod_prefix, 0, 1, s->eps);
  linear(h, D, w->w_qkvg_t, w->b_qkvg, 4 * A, qkvg, rows, nr);
#pragma omp parallel for schedule(static)
  for (int t = 0; t < nr; ++t)
    for (int c = 0; c < 4 * A; ++c) qkvg[(size_t)rows[t] * 4 * A + c] =
        bf16f(qkvg[(size_t)rows[t] * 4 * A + c]);
  heads(s, w->qnorm_w, w->knorm_w, qkvg, scratch + L.q, scratch + L.k, scratch + L.kt,
        scratch + L.v, scratch + L.g, rows, nr);
  /* a4-a9: router, attention, pooled branch and gate mix */
  router(s, scratch + L.q, scratch + L.k, scratch + L.v, scratch + L.means, scratch + L.scores,
         idx, s->pooled ? scratch + L.pooled : NULL);
  attention(s, scratch + L.q, scratch + L.kt, scratch + L.v, scratch + L.k, scratch + L.g, idx,
            s->pooled ? scratch + L.pooled : NULL, scratch + L.o, sample);
  /* a10: x1 = bf16(x + gate1 * (o W_o + b_o)) */
  float* br = qkvg; /* the projection buffer is free again */
  linear(scratch + L.o, A, w->w_o_t, w->b_o, D, br, rows, nr);
#pragma omp parallel for schedule(static)
  for (int t = 0; t < nr; ++t) {
    const int r = rows[t];
    const float* m = (w->mod_prefix && r < P) ? w->mod_prefix : w->mod;
    for (int c = 0; c < D; ++c)
      x[(size_t)r * D + c] = bf16f(x[(size_t)r * D + c] + m[2 * D + c] * br[(size_t)r * D + c]);
  }
  /* a11-a13: modulated norm 2, fc1 + GELU (or SwiGLU), fc2 + gated residual */
  modulate(x, h, rows, nr, D, P, w->mod, w->mod_prefix, 3, 4, s->eps);
  const int F1 = s->swiglu ? 2 * F : F;
  linear(h, D, w->w1_t, w->b1, F1, qkvg, rows, nr);
  float* u = scratch + L.u;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < nr; ++t) {
    const int r = rows[t];
    const float* y = qkvg + (size_t)r * F1;
    float* ur = u + (size_t)r * F;
    if (s->swiglu) {
      /* gate and up columns in groups of 128: 256j.. gate, 256j+128.. up of 128j.. */
      for (int c = 0; c < F; ++c) {
        const int grp = c / 128, off = c % 128;
        ur[c] = bf16f(silu(y[256 * grp + off]) * y[256 * grp + 128 + off]);
      }
    } else {
      for (int c = 0; c < F; ++c) ur[c] = bf16f(gelu(y[c]));
    }
  }
  linear(u, F, w->w2_t, w->b2, D, br, rows, nr);
#pragma omp parallel for schedule(static)
  for (int t = 0; t < nr; ++t) {
    const int r = rows[t];
    const float* m = (w->mod_prefix && r < P) ? w->mod_prefix : w->mod;
    for (int c = 0; c < D; ++c)
      x[(size_t)r * D + c] = bf16f(x[(size_t)r * D + c] + m[5 * D + c] * br[(size_t)r * D + c]);
  }
  if (idx_out) memcpy(idx_out, idx, (size_t)H * Tv * kk * sizeof(int));
  free(rows);
  return 0;
}

/* Router + attention + pooled branch + gate mix alone (h3dit_routed_attention's work):
 * q, k, v float [H][N][d] (bf16 values), g float [N][A] or NULL, out float [N][A]
 * (bf16 values), idx_out [H][Tv][k] or NULL.  hidden and mlp_width are not used. */
int h3time_attention(const h3time_shape* s, const float* q, const float* k, const float* v,
                     const float* g, float* out, float* scratch, int* idx_out) {
  if (!s || !q || !k || !v || !out || !scratch) return -1;
  const int N = s->n_text + s->n_audio + s->n_video;
  const int H = s->heads, d = s->head_dim, Tv = (s->n_video + TILE - 1) / TILE;
  const int kk = s->topk < Tv ? s->topk : Tv;
  const layout_t L = plan(s);
  float* kt = scratch + L.kt;
  int* idx = (int*)(scratch + L.idx);
#pragma omp parallel for schedule(static)
  for (int hh = 0; hh < H; ++hh)
    for (int r = 0; r < N; ++r)
      for (int c = 0; c < d; ++c) kt[((size_t)hh * d + c) * N + r] = k[((size_t)hh * N + r) * d + c];
  const int pool = s->pooled && g != NULL;
  router(s, q, k, v, scratch + L.means, scratch + L.scores, idx, pool ? scratch + L.pooled : NULL);
  attention(s, q, kt, v, k, g, idx, pool ? scratch + L.pooled : NULL, out, 1);
  if (idx_out) memcpy(idx_out, idx, (size_t)H * Tv * kk * sizeof(int));
  return 0;
}
