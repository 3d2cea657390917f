/*
 * h3ref.c -- plain C reference of one routed-attention DiT block (float64).
 *
 * Test infrastructure only: the tests load it (through oracle/cref.py) to
 * cross-check the numpy oracle in oracle/h3block.py; the product library
 * never links, loads or calls it.  It shares no code with the CUDA path and
 * none with the numpy oracle: both restate the same steps from the pages.
 *
 * Sources (page title and section):
 *   "ashhart/TensorFold pull request #949" (FastH3 denoiser on Metal), cited
 *     as TensorFold #949: "What it adds" (block.zig: modulated norm, q/k/v and
 *     the routing gate, head layout, routing, attention, pooled branch, out
 *     projection, MLP; h3_routing.metal: tile means, tile scores, top-k;
 *     h3_attention.metal: tile-routed attention), "Precision" (bf16 weights
 *     and activations, fp32 sums and routing, softmax weights rounded to bf16
 *     before the value product), "Receipts" (prefix tiles kept for every
 *     query; 4 x 4 x 4 cubes) and "Kernel contract" (NaN ranks as -inf, ties
 *     go to the lower tile).
 *   "Antirez/h3.c: MiniMax H3 inference engine for Mac computers", cited as
 *     the h3.c README: the fused gated-AdaLN paragraph (per-row RMS, gated
 *     residual adds), the Q/K RMS normalisation + RoPE paragraph, the SwiGLU
 *     MLP paragraph.
 *
 * Arithmetic is float64 throughout; values are rounded to bf16 exactly where
 * the method stores bf16 (the modulated-norm outputs, the projection outputs,
 * q and k after norm and rotary, the attention output, the MLP activations and
 * the residual stream), and the top-k decision is taken on scores rounded to
 * float32.  Readings where the pages leave a step open (the same as the numpy
 * oracle's): RMS eps 1e-6 without a learned weight and the (1 + scale) form;
 * gated residual x + gate * branch; rotate-half rotary with theta 10,000 over
 * the packed row index, or 3-D over (t, h, w) with time / height / width pairs
 * d/2 - 2 floor(d/6), floor(d/6), floor(d/6); tile scores unscaled; the pooled
 * branch a softmax over all video tile means with scale 1/sqrt(d), added
 * through the linear gate g; exact erf GELU; SwiGLU fc1 rows stored gate / up
 * interleaved in groups of 128; with softmax weights rounded to bf16, the row
 * sum uses the unrounded weights.
 *
 * Everything is written as plain loops in the order the steps are listed; no
 * blocking, fusion or reordering.
 *
 * Pins (tests/test_oracle_c.py): bf16 rounding against torch's conversion; tile
 * sets, top-k selections, scores, pooled branch and attention outputs against the
 * numpy oracle on slices, clipped cubes with the 3-D rotary, a 450-row prefix and a
 * SwiGLU block with a prefix table; every tile selected against dense attention by
 * brute force; planted ties and NaN for the top-k rule; the Euler step, the
 * extrapolation, the patch projection, the output head, token pooling and restore and
 * layer thinning against the numpy oracle.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int n_text, n_audio, n_video;
  int hidden, heads, head_dim, mlp_width, topk;
  int qk_norm, rope, pooled, swiglu, p_bf16;
  int grid[3]; /* video latent grid (t, h, w); grid[0] == 0: contiguous 64-row slices */
  int cube[3]; /* cube shape when a grid is given */
  double eps, theta;
} h3ref_shape;

typedef struct {
  /* float64 values of the bf16 weights; linear weights stored [out, in] */
  const double *w_qkvg, *b_qkvg; /* [4A, D], [4A]: rows q, k, v, g, head-major */
  const double *w_o, *b_o;       /* [D, A], [D] */
  const double *w1, *b1;         /* [F, D] (GELU) or [2F, D] (SwiGLU), bias likewise */
  const double *w2, *b2;         /* [D, F], [D] */
  const double *mod;             /* [6, D]: shift1, scale1, gate1, shift2, scale2, gate2 */
  const double *mod_prefix;      /* [6, D] for the text and audio rows, or NULL */
  const double *qnorm_w, *knorm_w; /* [d] */
} h3ref_weights;

enum { TILE = 64 };

/* ------------------------------------------------------------------ roundings */

/* Nearest bf16 (8 significant bits, ties to even), returned as a double: the storage
 * type of weights and activations (TensorFold #949 "Precision"). */
static double bf16r(double x) {
  if (x != x || isinf(x) || x == 0.0) return x;
  const double a = fabs(x);
  int e;
  frexp(a, &e);                  /* a in [2^(e-1), 2^e) */
  int q = (e - 1) - 7;           /* spacing of bf16 values near a */
  if (q < -133) q = -133;        /* bf16 subnormals are multiples of 2^-133 */
  double r = ldexp(nearbyint(ldexp(a, -q)), q);
  if (r >= ldexp(1.0, 128)) r = INFINITY;
  return x < 0 ? -r : r;
}

static double f32r(double x) { return (double)(float)x; }

/* ------------------------------------------------------------------ tiles */

static int is_grid(const h3ref_shape* s) { return s->grid[0] > 0; }

/* Number of video tiles: 64-row slices, or clipped cubes of the grid. */
int h3ref_tile_count(const h3ref_shape* s) {
  if (!is_grid(s)) return (s->n_video + TILE - 1) / TILE;
  int n = 1;
  for (int a = 0; a < 3; ++a) n *= (s->grid[a] + s->cube[a] - 1) / s->cube[a];
  return n;
}

/* Packed row indices of every video tile, tile after tile: tile t holds
 * rows[start[t]] .. rows[start[t+1] - 1].  Video rows are in raster (t, h, w)
 * order after the prefix; cubes are numbered in raster (cube t, h, w) order and
 * a cube's rows listed in raster order (TensorFold #949 "Receipts": 4 x 4 x 4
 * cubes, edges clipped). */
int h3ref_tiles(const h3ref_shape* s, int* rows, int* start) {
  const int P = s->n_text + s->n_audio;
  int n = 0, t = 0;
  if (!is_grid(s)) {
    for (int r0 = 0; r0 < s->n_video; r0 += TILE, ++t) {
      start[t] = n;
      for (int r = r0; r < r0 + TILE && r < s->n_video; ++r) rows[n++] = P + r;
    }
    start[t] = n;
    return t;
  }
  const int T = s->grid[0], Hg = s->grid[1], W = s->grid[2];
  for (int a = 0; a < T; a += s->cube[0])
    for (int b = 0; b < Hg; b += s->cube[1])
      for (int c = 0; c < W; c += s->cube[2], ++t) {
        start[t] = n;
        for (int tt = a; tt < a + s->cube[0] && tt < T; ++tt)
          for (int hh = b; hh < b + s->cube[1] && hh < Hg; ++hh)
            for (int ww = c; ww < c + s->cube[2] && ww < W; ++ww)
              rows[n++] = P + (tt * Hg + hh) * W + ww;
      }
  start[t] = n;
  return t;
}

/* ------------------------------------------------------------------ row steps */

/* h = bf16(x / sqrt(mean(x^2) + eps) * (1 + scale) + shift) for one row (TensorFold #949
 * "What it adds": modulated norm; h3.c README fused gated-AdaLN paragraph: per-row RMS). */
static void modulated_norm(const double* x, int D, const double* shift, const double* scale,
                           double eps, double* h) {
  double ss = 0.0;
  for (int c = 0; c < D; ++c) ss += x[c] * x[c];
  const double inv = 1.0 / sqrt(ss / D + eps);
  for (int c = 0; c < D; ++c) h[c] = bf16r(x[c] * inv * (1.0 + scale[c]) + shift[c]);
}

/* y[r, o] = sum_i a[r, i] w[o, i] + b[o]  (w stored [out, in]; b may be NULL): the
 * projections, bf16 operands with wide sums (TensorFold #949 "Precision"). */
static void linear(const double* a, int M, int K, const double* w, const double* b, int Nout,
                   double* y) {
  for (int r = 0; r < M; ++r)
    for (int o = 0; o < Nout; ++o) {
      double acc = 0.0;
      for (int i = 0; i < K; ++i) acc += a[(size_t)r * K + i] * w[(size_t)o * K + i];
      y[(size_t)r * Nout + o] = acc + (b ? b[o] : 0.0);
    }
}

/* Per-head RMS norm over d with a learned weight (h3.c README, Q/K RMS norm). */
static void head_norm(double* v, int d, const double* w, double eps) {
  double ss = 0.0;
  for (int c = 0; c < d; ++c) ss += v[c] * v[c];
  const double inv = 1.0 / sqrt(ss / d + eps);
  for (int c = 0; c < d; ++c) v[c] = v[c] * inv * w[c];
}

/* Rotary angle of pair c (c < d/2) for packed row p (h3.c README, Q/K RMS + RoPE
 * paragraph: spatial and temporal rotary coordinates when a latent grid is given). */
static double rope_angle(const h3ref_shape* s, int p, int c) {
  const int d = s->head_dim, half = d / 2;
  if (!is_grid(s)) return (double)p * pow(s->theta, -2.0 * c / d);
  const int P = s->n_text + s->n_audio;
  int pos[3] = {p, p, p}; /* text and audio rows: the packed index on every axis */
  if (p >= P) {
    const int v = p - P, Hg = s->grid[1], W = s->grid[2];
    pos[0] = v / (Hg * W);
    pos[1] = (v / W) % Hg;
    pos[2] = v % W;
  }
  const int ms = half / 3, mt = half - 2 * ms;
  const int m[3] = {mt, ms, ms};
  int a = 0, j = c;
  while (j >= m[a]) j -= m[a++];
  return (double)pos[a] * pow(s->theta, -(double)j / m[a]);
}

/* Turn pairs (c, c + d/2) of one head vector by the row's angles. */
static void rotate(const h3ref_shape* s, int p, double* v) {
  const int half = s->head_dim / 2;
  for (int c = 0; c < half; ++c) {
    const double ang = rope_angle(s, p, c), co = cos(ang), si = sin(ang);
    const double x0 = v[c], x1 = v[c + half];
    v[c] = x0 * co - x1 * si;
    v[c + half] = x1 * co + x0 * si;
  }
}

/* ------------------------------------------------------------------ attention */

/* One query row against a key set: o = sum softmax(q k / sqrt(d)) v; with p_bf16 the
 * weights are rounded to bf16 before the value product and the row sum uses the
 * unrounded weights.  Reading (the pages do not fix the maximum the rounded weights
 * are taken against): with p_bf16 a weight is 2^(s log2(e) - M), M the smallest whole
 * number not below the largest s log2(e) of the row, so that the rounding does not
 * depend on which maximum a streaming softmax has met (whole octaves commute with it). */
static void attend_row(const double* q, const double* K, const double* V, const int* keys,
                       int nk, int d, int p_bf16, double* sbuf, double* o) {
  const double scale = 1.0 / sqrt((double)d);
  const double log2e = 1.0 / log(2.0);
  double m = -INFINITY;
  for (int j = 0; j < nk; ++j) {
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += q[c] * K[(size_t)keys[j] * d + c];
    sbuf[j] = acc * scale;
    if (p_bf16) sbuf[j] *= log2e;
    if (sbuf[j] > m) m = sbuf[j];
  }
  if (p_bf16) m = ceil(m);
  double l = 0.0;
  for (int c = 0; c < d; ++c) o[c] = 0.0;
  for (int j = 0; j < nk; ++j) {
    const double p = p_bf16 ? exp2(sbuf[j] - m) : exp(sbuf[j] - m);
    l += p;
    const double pv = p_bf16 ? bf16r(p) : p;
    for (int c = 0; c < d; ++c) o[c] += pv * V[(size_t)keys[j] * d + c];
  }
  for (int c = 0; c < d; ++c) o[c] /= l;
}

/* TensorFold #949 "Kernel contract" and "Precision" (fp32 routing).
 * Top-k of one query tile's scores under the total order (score descending, index
 * ascending) with NaN as -inf, decided on fp32 scores: tile j is kept when fewer than
 * k tiles rank ahead of it.  Kept tiles are written ascending. */
static void topk_row(const double* srow, int Tv, int k, int* out) {
  int n = 0;
  for (int j = 0; j < Tv; ++j) {
    double sj = f32r(srow[j]);
    if (sj != sj) sj = -INFINITY;
    int ahead = 0;
    for (int i = 0; i < Tv; ++i) {
      double si = f32r(srow[i]);
      if (si != si) si = -INFINITY;
      if (si > sj || (si == sj && i < j)) ++ahead;
    }
    if (ahead < k) out[n++] = j;
  }
}

/* TensorFold #949 "What it adds": h3_routing.metal (tile means, tile scores, top-k,
 * pooled branch), h3_attention.metal (tile-routed attention), h3_gate_mix.
 * Router + routed / dense attention + pooled branch + gate mix for one layer.
 * Q, K, V [H, N, d]; G [N, H*d] or NULL.  Outputs: o_mixed [N, H*d] (float64, not
 * rounded), idx [H, Tv, min(k, Tv)], scores [H, Tv, Tv], pooled [H, Tv, d] (any may
 * be NULL except o_mixed).  Returns 0, or -1 on a bad shape or allocation failure. */
int h3ref_attention_layer(const h3ref_shape* s, const double* Q, const double* K,
                          const double* V, const double* G, double* o_mixed, int* idx_out,
                          double* scores_out, double* pooled_out) {
  const int P = s->n_text + s->n_audio, N = P + s->n_video, H = s->heads, d = s->head_dim;
  const int A = H * d;
  if (N <= 0 || d <= 0 || H <= 0 || s->topk < 1) return -1;
  const int Tv = h3ref_tile_count(s);
  const int ksel = s->topk < Tv ? s->topk : Tv;
  int* rows = malloc(sizeof(int) * (s->n_video + 1));
  int* start = malloc(sizeof(int) * (Tv + 1));
  int* tile_of = malloc(sizeof(int) * N);
  double* mq = malloc(sizeof(double) * (size_t)Tv * d);
  double* mk = malloc(sizeof(double) * (size_t)Tv * d);
  double* mv = malloc(sizeof(double) * (size_t)Tv * d);
  double* S = malloc(sizeof(double) * (size_t)Tv * Tv);
  int* idx = malloc(sizeof(int) * (size_t)Tv * ksel);
  double* pooled = malloc(sizeof(double) * (size_t)Tv * d);
  int* keys = malloc(sizeof(int) * N);
  double* sbuf = malloc(sizeof(double) * N);
  double* o = malloc(sizeof(double) * d);
  int rc = 0;
  if (!rows || !start || !tile_of || !mq || !mk || !mv || !S || !idx || !pooled || !keys ||
      !sbuf || !o) {
    rc = -1;
    goto done;
  }
  h3ref_tiles(s, rows, start);
  for (int r = 0; r < N; ++r) tile_of[r] = -1;
  for (int t = 0; t < Tv; ++t)
    for (int e = start[t]; e < start[t + 1]; ++e) tile_of[rows[e]] = t;
  const double sc = 1.0 / sqrt((double)d);
  for (int h = 0; h < H; ++h) {
    const double* Qh = Q + (size_t)h * N * d;
    const double* Kh = K + (size_t)h * N * d;
    const double* Vh = V + (size_t)h * N * d;
    /* tile means over each tile's rows (TensorFold #949: h3_routing tile means) */
    for (int t = 0; t < Tv; ++t) {
      const int n = start[t + 1] - start[t];
      for (int c = 0; c < d; ++c) {
        double aq = 0.0, ak = 0.0, av = 0.0;
        for (int e = start[t]; e < start[t + 1]; ++e) {
          aq += Qh[(size_t)rows[e] * d + c];
          ak += Kh[(size_t)rows[e] * d + c];
          av += Vh[(size_t)rows[e] * d + c];
        }
        mq[(size_t)t * d + c] = aq / n;
        mk[(size_t)t * d + c] = ak / n;
        mv[(size_t)t * d + c] = av / n;
      }
    }
    /* tile scores, unscaled */
    for (int i = 0; i < Tv; ++i)
      for (int j = 0; j < Tv; ++j) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += mq[(size_t)i * d + c] * mk[(size_t)j * d + c];
        S[(size_t)i * Tv + j] = acc;
      }
    /* top-k per query tile */
    for (int i = 0; i < Tv; ++i) topk_row(S + (size_t)i * Tv, Tv, ksel, idx + (size_t)i * ksel);
    /* pooled branch: softmax over all video tiles of S / sqrt(d), weights . tile means of v */
    for (int i = 0; i < Tv; ++i) {
      double m = -INFINITY, l = 0.0;
      for (int j = 0; j < Tv; ++j) m = fmax(m, S[(size_t)i * Tv + j] * sc);
      for (int c = 0; c < d; ++c) pooled[(size_t)i * d + c] = 0.0;
      for (int j = 0; j < Tv; ++j) {
        const double w = exp(S[(size_t)i * Tv + j] * sc - m);
        l += w;
        for (int c = 0; c < d; ++c) pooled[(size_t)i * d + c] += w * mv[(size_t)j * d + c];
      }
      for (int c = 0; c < d; ++c) pooled[(size_t)i * d + c] /= l;
    }
    /* attention: prefix rows over all N rows; a video row of tile i over the prefix rows
     * and the rows of the tiles idx[i] (TensorFold #949 "Receipts": prefix tiles are
     * kept for every query) */
    for (int r = 0; r < N; ++r) {
      int nk = 0;
      if (r < P) {
        for (int j = 0; j < N; ++j) keys[nk++] = j;
      } else {
        const int i = tile_of[r];
        for (int j = 0; j < P; ++j) keys[nk++] = j;
        for (int u = 0; u < ksel; ++u) {
          const int t = idx[(size_t)i * ksel + u];
          for (int e = start[t]; e < start[t + 1]; ++e) keys[nk++] = rows[e];
        }
      }
      attend_row(Qh + (size_t)r * d, Kh, Vh, keys, nk, d, s->p_bf16, sbuf, o);
      for (int c = 0; c < d; ++c) {
        double v = o[c];
        /* gate mix: video rows add g * pooled of their tile (h3_gate_mix) */
        if (r >= P && s->pooled && G)
          v += G[(size_t)r * A + h * d + c] * pooled[(size_t)tile_of[r] * d + c];
        o_mixed[(size_t)r * A + h * d + c] = v;
      }
    }
    if (idx_out) memcpy(idx_out + (size_t)h * Tv * ksel, idx, sizeof(int) * (size_t)Tv * ksel);
    if (scores_out) memcpy(scores_out + (size_t)h * Tv * Tv, S, sizeof(double) * (size_t)Tv * Tv);
    if (pooled_out) memcpy(pooled_out + (size_t)h * Tv * d, pooled, sizeof(double) * (size_t)Tv * d);
  }
done:
  free(rows);
  free(start);
  free(tile_of);
  free(mq);
  free(mk);
  free(mv);
  free(S);
  free(idx);
  free(pooled);
  free(keys);
  free(sbuf);
  free(o);
  return rc;
}

/* ------------------------------------------------------------------ block */

static double gelu(double x) { return 0.5 * x * (1.0 + erf(x / sqrt(2.0))); }
static double silu(double x) { return x / (1.0 + exp(-x)); }

/* TensorFold #949 "What it adds" (block.zig, the block's steps in order); gated
 * residual adds as in the h3.c README's fused gated-AdaLN paragraph; SwiGLU MLP as in
 * its FC1 gate/up paragraph.
 * One DiT block on the packed rows x [N, D] (bf16 values).  Writes x1 and x2
 * (either may be NULL) and, when given, the bf16 attention output o [N, A].
 * Returns 0, or -1 on a bad shape or allocation failure. */
int h3ref_block_forward(const h3ref_shape* s, const h3ref_weights* w, const double* x,
                        double* x1_out, double* x2_out, double* o_out) {
  const int P = s->n_text + s->n_audio, N = P + s->n_video;
  const int D = s->hidden, H = s->heads, d = s->head_dim, A = H * d, F = s->mlp_width;
  const int F1 = s->swiglu ? 2 * F : F;
  if (N <= 0 || D <= 0 || F <= 0 || (s->swiglu && F % 128)) return -1;
  double* h = malloc(sizeof(double) * (size_t)N * D);
  double* qkvg = malloc(sizeof(double) * (size_t)N * 4 * A);
  double* Q = malloc(sizeof(double) * (size_t)H * N * d);
  double* Kt = malloc(sizeof(double) * (size_t)H * N * d);
  double* V = malloc(sizeof(double) * (size_t)H * N * d);
  double* G = malloc(sizeof(double) * (size_t)N * A);
  double* o = malloc(sizeof(double) * (size_t)N * A);
  double* br = malloc(sizeof(double) * (size_t)N * (D > F1 ? D : F1));
  double* x1 = malloc(sizeof(double) * (size_t)N * D);
  double* u = malloc(sizeof(double) * (size_t)N * F);
  int rc = 0;
  if (!h || !qkvg || !Q || !Kt || !V || !G || !o || !br || !x1 || !u) {
    rc = -1;
    goto done;
  }
  /* modulated norm 1: text and audio rows on their own table when one is given */
  for (int r = 0; r < N; ++r) {
    const double* mod = (w->mod_prefix && r < P) ? w->mod_prefix : w->mod;
    modulated_norm(x + (size_t)r * D, D, mod, mod + D, s->eps, h + (size_t)r * D);
  }
  /* q / k / v / gate projection, rounded to bf16 */
  linear(h, N, D, w->w_qkvg, w->b_qkvg, 4 * A, qkvg);
  for (size_t e = 0; e < (size_t)N * 4 * A; ++e) qkvg[e] = bf16r(qkvg[e]);
  /* head layout: q, k normed per head, turned by the rotary, rounded to bf16 */
  for (int r = 0; r < N; ++r)
    for (int hh = 0; hh < H; ++hh) {
      double* q = Q + ((size_t)hh * N + r) * d;
      double* k = Kt + ((size_t)hh * N + r) * d;
      double* v = V + ((size_t)hh * N + r) * d;
      for (int c = 0; c < d; ++c) {
        q[c] = qkvg[(size_t)r * 4 * A + 0 * A + hh * d + c];
        k[c] = qkvg[(size_t)r * 4 * A + 1 * A + hh * d + c];
        v[c] = qkvg[(size_t)r * 4 * A + 2 * A + hh * d + c];
        G[(size_t)r * A + hh * d + c] = qkvg[(size_t)r * 4 * A + 3 * A + hh * d + c];
      }
      if (s->qk_norm) {
        head_norm(q, d, w->qnorm_w, s->eps);
        head_norm(k, d, w->knorm_w, s->eps);
      }
      if (s->rope) {
        rotate(s, r, q);
        rotate(s, r, k);
      }
      for (int c = 0; c < d; ++c) {
        q[c] = bf16r(q[c]);
        k[c] = bf16r(k[c]);
      }
    }
  /* routing, attention, pooled branch and gate mix; the output is a bf16 mid */
  if (h3ref_attention_layer(s, Q, Kt, V, G, o, NULL, NULL, NULL) != 0) {
    rc = -1;
    goto done;
  }
  for (size_t e = 0; e < (size_t)N * A; ++e) o[e] = bf16r(o[e]);
  if (o_out) memcpy(o_out, o, sizeof(double) * (size_t)N * A);
  /* out projection + gated residual: x1 = bf16(x + gate1 * (o W_o^T + b_o)) */
  linear(o, N, A, w->w_o, w->b_o, D, br);
  for (int r = 0; r < N; ++r) {
    const double* mod = (w->mod_prefix && r < P) ? w->mod_prefix : w->mod;
    for (int c = 0; c < D; ++c)
      x1[(size_t)r * D + c] =
          bf16r(x[(size_t)r * D + c] + mod[2 * D + c] * br[(size_t)r * D + c]);
  }
  /* modulated norm 2 */
  for (int r = 0; r < N; ++r) {
    const double* mod = (w->mod_prefix && r < P) ? w->mod_prefix : w->mod;
    modulated_norm(x1 + (size_t)r * D, D, mod + 3 * D, mod + 4 * D, s->eps, h + (size_t)r * D);
  }
  /* MLP inner activations: GELU, or SwiGLU with gate / up rows interleaved by 128 */
  linear(h, N, D, w->w1, w->b1, F1, br);
  for (int r = 0; r < N; ++r)
    for (int j = 0; j < F; ++j) {
      double a;
      if (s->swiglu) {
        const int rg = 256 * (j / 128) + j % 128; /* gate row; its up row is 128 further */
        a = silu(br[(size_t)r * F1 + rg]) * br[(size_t)r * F1 + rg + 128];
      } else {
        a = gelu(br[(size_t)r * F1 + j]);
      }
      u[(size_t)r * F + j] = bf16r(a);
    }
  /* fc2 + gated residual: x2 = bf16(x1 + gate2 * (u W2^T + b2)) */
  linear(u, N, F, w->w2, w->b2, D, br);
  if (x1_out) memcpy(x1_out, x1, sizeof(double) * (size_t)N * D);
  if (x2_out) {
    for (int r = 0; r < N; ++r) {
      const double* mod = (w->mod_prefix && r < P) ? w->mod_prefix : w->mod;
      for (int c = 0; c < D; ++c)
        x2_out[(size_t)r * D + c] =
            bf16r(x1[(size_t)r * D + c] + mod[5 * D + c] * br[(size_t)r * D + c]);
    }
  }
done:
  free(h);
  free(qkvg);
  free(Q);
  free(Kt);
  free(V);
  free(G);
  free(o);
  free(br);
  free(x1);
  free(u);
  return rc;
}

/* ------------------------------------------------------------------ denoiser and ends */

/* h3.c README sampler paragraph: z' = fp32(z + dt v), the text and audio rows (index < P)
 * on their own step dt_prefix.  z, v, out [N, D]. */
void h3ref_euler(const double* z, const double* v, int N, int D, int P, double dt,
                 double dt_prefix, double* out) {
  for (int r = 0; r < N; ++r)
    for (int c = 0; c < D; ++c) {
      const double step = r < P ? dt_prefix : dt;
      out[(size_t)r * D + c] = f32r(z[(size_t)r * D + c] + step * v[(size_t)r * D + c]);
    }
}

/* h3.c README sampler paragraph: a skipped pass extrapolates linearly in sigma from the
 * last two fresh velocities, v = v_a + (v_a - v_b) (s_i - s_a) / (s_a - s_b), the text
 * and audio rows on their own sigmas sp[3] = (s_i, s_a, s_b). */
void h3ref_extrapolate(const double* va, const double* vb, int N, int D, int P,
                       const double* sv, const double* sp, double* out) {
  const double cv = (sv[0] - sv[1]) / (sv[1] - sv[2]);
  const double cp = (sp[0] - sp[1]) / (sp[1] - sp[2]);
  for (int r = 0; r < N; ++r)
    for (int c = 0; c < D; ++c) {
      const size_t e = (size_t)r * D + c;
      out[e] = va[e] + (va[e] - vb[e]) * (r < P ? cp : cv);
    }
}

/* h3.c README: a modality's patch projection, x = bf16(z w_in + b) with w_in stored
 * input-major [c, D] (fp32 weights and sums on the pages; float64 here). */
void h3ref_patch_in(const double* z, int rows, int c, const double* w_in, const double* b_in,
                    int D, double* x) {
  for (int r = 0; r < rows; ++r)
    for (int o = 0; o < D; ++o) {
      double acc = 0.0;
      for (int j = 0; j < c; ++j) acc += z[(size_t)r * c + j] * w_in[(size_t)j * D + o];
      x[(size_t)r * D + o] = bf16r(acc + b_in[o]);
    }
}

/* h3.c README: final AdaLN of a modality's rows (the block norms' form with its own
 * shift, scale [2, D]) and its narrow head: v = fp32(h W_out^T + b), W_out [c, D]. */
void h3ref_output_head(const double* x, int rows, int D, const double* mod2,
                       const double* w_out, const double* b_out, int c, double eps,
                       double* v) {
  double* h = malloc(sizeof(double) * (size_t)D);
  if (!h) return;
  for (int r = 0; r < rows; ++r) {
    modulated_norm(x + (size_t)r * D, D, mod2, mod2 + D, eps, h);
    for (int o = 0; o < c; ++o) {
      double acc = 0.0;
      for (int i = 0; i < D; ++i) acc += h[i] * w_out[(size_t)o * D + i];
      v[(size_t)r * c + o] = f32r(acc + b_out[o]);
    }
  }
  free(h);
}

/* h3.c README token-reduction paragraph: the prefix rows pass unchanged; each pair of
 * horizontally adjacent video tokens (t, h, 2j), (t, h, 2j + 1) becomes one row, their
 * mean (fp32 sum halved, rounded to bf16); a lone last token of an odd row passes as it
 * is.  Video rows of x are in raster order of the T x H x W grid; x_r [P + T H Wr, D] and
 * base [T H Wr, D] (the pooled rows as they were at pooling time), Wr = ceil(W / 2). */
void h3ref_token_pool(const double* x, int P, int T, int Hg, int W, int D, double* x_r,
                      double* base) {
  const int Wr = (W + 1) / 2;
  memcpy(x_r, x, sizeof(double) * (size_t)P * D);
  for (int tt = 0; tt < T; ++tt)
    for (int hh = 0; hh < Hg; ++hh)
      for (int j = 0; j < Wr; ++j) {
        const double* a = x + ((size_t)P + ((size_t)tt * Hg + hh) * W + 2 * j) * D;
        double* o = base + (((size_t)tt * Hg + hh) * Wr + j) * D;
        for (int c = 0; c < D; ++c)
          o[c] = (2 * j + 1 < W) ? bf16r(f32r(a[c] + a[D + c]) * 0.5) : a[c];
        memcpy(x_r + ((size_t)P + ((size_t)tt * Hg + hh) * Wr + j) * D, o, sizeof(double) * D);
      }
}

/* Restore: prefix rows from x_r; video token (t, h, w) = bf16(bypass + fp32(x_r - base)
 * of its pair row (t, h, w / 2)), in fp32 arithmetic.  out [P + T H W, D]. */
void h3ref_token_restore(const double* bypass, const double* x_r, const double* base, int P,
                         int T, int Hg, int W, int D, double* out) {
  const int Wr = (W + 1) / 2;
  memcpy(out, x_r, sizeof(double) * (size_t)P * D);
  for (int tt = 0; tt < T; ++tt)
    for (int hh = 0; hh < Hg; ++hh)
      for (int w = 0; w < W; ++w) {
        const size_t pr = ((size_t)tt * Hg + hh) * Wr + w / 2;
        const size_t full = (size_t)P + ((size_t)tt * Hg + hh) * W + w;
        for (int c = 0; c < D; ++c) {
          const double dlt = f32r(x_r[((size_t)P + pr) * D + c] - base[pr * D + c]);
          out[full * D + c] = bf16r(f32r(bypass[full * D + c] + dlt));
        }
      }
}

/* h3.c README layer-thinning paragraph: keep the first and last of L blocks, score the
 * others by ||gate1||_2 + ||gate2||_2 of their [6, D] tables (rows 2 and 5), drop the
 * lowest scores, ties dropping the higher index.  kept [keep] ascending; returns the
 * number kept, or -1 when keep < 2. */
int h3ref_thin_layers(const double* mods, int L, int D, int keep, int* kept) {
  if (keep >= L) {
    for (int b = 0; b < L; ++b) kept[b] = b;
    return L;
  }
  if (keep < 2) return -1;
  double* score = malloc(sizeof(double) * (size_t)L);
  char* drop = calloc((size_t)L, 1);
  if (!score || !drop) {
    free(score);
    free(drop);
    return -1;
  }
  for (int b = 1; b < L - 1; ++b) {
    double g1 = 0.0, g2 = 0.0;
    for (int c = 0; c < D; ++c) {
      const double a = mods[((size_t)b * 6 + 2) * D + c], e = mods[((size_t)b * 6 + 5) * D + c];
      g1 += a * a;
      g2 += e * e;
    }
    score[b] = sqrt(g1) + sqrt(g2);
  }
  /* drop L - keep blocks one at a time: the lowest score, the higher index among equals */
  for (int n = 0; n < L - keep; ++n) {
    int pick = -1;
    for (int b = 1; b < L - 1; ++b) {
      if (drop[b]) continue;
      if (pick < 0 || score[b] < score[pick] || (score[b] == score[pick] && b > pick)) pick = b;
    }
    drop[pick] = 1;
  }
  int n = 0;
  for (int b = 0; b < L; ++b)
    if (!drop[b]) kept[n++] = b;
  free(score);
  free(drop);
  return n;
}

/* Exported for the tests' rounding checks. */
double h3ref_bf16(double x) { return bf16r(x); }
