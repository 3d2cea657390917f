/*
 * h3dit.h -- C ABI of the GB300 (sm_103a) routed-attention DiT forward.
 *
 * The library runs the denoising forward of a joint video + audio diffusion
 * transformer of the MiniMax-H3 / FastH3 family: DiT blocks over one packed
 * sequence of text, audio and video rows, with tile-routed (block-sparse)
 * attention for the video rows.  Operations follow the pages
 *   "ashhart/TensorFold pull request #949" (FastH3 denoiser on Metal; cited
 *   below as TensorFold #949) and
 *   "Antirez/h3.c: MiniMax H3 inference engine for Mac computers" (cited as
 *   the h3.c README).
 *
 * Conventions shared by every entry point
 *   - Every data pointer is caller-owned DEVICE memory unless stated as host.
 *     The library allocates no device memory; scratch comes from the caller's
 *     workspace (size from h3dit_workspace_bytes).
 *   - Calls are asynchronous on the given stream: the status returned reports
 *     argument errors found on the host before any launch, and launch errors.
 *     Errors raised inside kernels (a bounded wait that ran out) are recorded
 *     in a status word inside the workspace; h3dit_sync_status() reads and
 *     clears it.
 *   - bf16 tensors are IEEE bfloat16 bit patterns (uint16).  Linear weights
 *     are stored [out, in] row-major (input features contiguous).
 *   - Row order of the packed sequence: text rows, then audio rows, then video
 *     rows.  The prefix (text + audio) may have any length (the pages' receipt
 *     has 36 + 414 rows); its keys are walked in 64-row chunks, the last one
 *     partial.  Video rows are cut into routing tiles of at most 64 rows:
 *     contiguous 64-row slices (the last may be partial), or clipped cubes of a
 *     latent grid (see h3dit_shape).
 *   - Results are deterministic: the same inputs give the same bytes.
 *   - Pointers must be 16-byte aligned; row pitches are dense.
 */
#ifndef H3DIT_H_
#define H3DIT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  H3DIT_OK = 0,
  H3DIT_ERR_ARG = 1,          /* null pointer or bad scalar argument            */
  H3DIT_ERR_SHAPE = 2,        /* unsupported or inconsistent shape              */
  H3DIT_ERR_ALIGN = 3,        /* pointer not 16-byte aligned                    */
  H3DIT_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required     */
  H3DIT_ERR_CUDA = 5,         /* a CUDA runtime / driver call failed            */
  H3DIT_ERR_TIMEOUT = 6,      /* a kernel's bounded wait ran out (device-side)  */
  H3DIT_ERR_UNSUPPORTED = 7   /* no sm_100-family GPU, or a feature not built   */
} h3dit_status;

/* Flags of h3dit_shape.flags */
#define H3DIT_QK_NORM 0x1u   /* per-head RMS norm of q and k with learned weights */
#define H3DIT_ROPE    0x2u   /* rotary on q and k: over the packed row index, or   */
                             /* 3-D (t, h, w) when a video grid is given below      */
#define H3DIT_POOLED  0x4u   /* pooled branch + gate mix for video rows            */
#define H3DIT_SWIGLU  0x8u   /* MLP u = silu(h W_gate^T + b_g) * (h W_up^T + b_u)   */
                             /* (else u = gelu(h W1^T + b1)); see w1 below          */
#define H3DIT_TOKEN_REDUCTION 0x10u /* reserve workspace for token reduction (needs a  */
                                    /* video grid at least 2 wide); see h3dit_sample_step */
#define H3DIT_KEEP_INTERMEDIATES 0x20u /* block forward keeps its intermediates in the    */
                                       /* workspace for inspection: see                   */
                                       /* h3dit_get_workspace_layout                      */

typedef struct {
  int n_text, n_audio, n_video; /* packed row counts, in this order               */
  int hidden;                   /* D: residual width (multiple of 256)            */
  int heads, head_dim;          /* H, d (d = 64 or 128)                           */
  int attn_width;               /* A = H * d (multiple of 256)                    */
  int mlp_width;                /* F: MLP inner width (multiple of 256)           */
  int tile;                     /* routing tile rows; must be 64                  */
  int topk;                     /* k video tiles kept per query tile (>= 1);      */
                                /* k >= number of video tiles means dense         */
  float rms_eps;                /* epsilon of every RMS norm (e.g. 1e-6)          */
  float rope_theta;             /* rotary base (e.g. 10000)                       */
  unsigned flags;               /* H3DIT_QK_NORM | H3DIT_ROPE | H3DIT_POOLED      */
  /* Video layout.  All zero: video rows form contiguous 64-row tiles in packed
   * order (the last may be partial).  Otherwise the video rows are the latent grid
   * video_t x video_h x video_w (n_video = t * h * w) cut into cubes of
   * cube_t x cube_h x cube_w = tile tokens, edge cubes clipped (TensorFold #949
   * "Receipts": 280 tiles from 4 x 4 x 4 cubes at 864 x 480 x 124), and every
   * buffer holds them in CUBE ORDER: cubes in raster (cube_t, cube_h, cube_w)
   * order, each cube's tokens in raster (t, h, w) order, so every tile is a
   * contiguous run of rows (h3dit_video_order gives the permutation).  With
   * H3DIT_ROPE the rotary is then 3-D: rotary pairs c < d/2 split into
   * m_t = d/2 - 2 m_s time pairs, then m_s height and m_s width pairs
   * (m_s = floor(d/6)); pair c of axis a with local index j turns by
   * pos_a * theta^(-j / m_a), pos = (t, h, w) for video rows and (p, p, p) for
   * a text or audio row at packed index p. */
  int video_t, video_h, video_w;
  int cube_t, cube_h, cube_w;
} h3dit_shape;

/* One block's parameters (device pointers, bf16 unless stated).
 *   w_qkvg [4A, D], b_qkvg [4A]: rows 0..A-1 -> q, A..2A-1 -> k, 2A..3A-1 -> v,
 *                                3A..4A-1 -> the routing gate g (head-major).
 *   w_o [D, A], b_o [D];  w1 [F, D], b1 [F];  w2 [D, F], b2 [D]
 *   with H3DIT_SWIGLU, w1 [2F, D] and b1 [2F] hold the gate and up projections
 *   interleaved in groups of 128 rows: rows 256j .. 256j+127 are the gate rows of
 *   outputs 128j .. 128j+127 and rows 256j+128 .. 256j+255 their up rows (F a
 *   multiple of 128); mlp_width is F, the activated width.
 *   mod  fp32 [6, D]: shift1, scale1, gate1, shift2, scale2, gate2
 *   qnorm_w, knorm_w [d]: per-head RMS-norm weights (used with H3DIT_QK_NORM)
 *   mod_prefix fp32 [6, D] or NULL: the modulation of the text and audio rows when
 *     they are conditioned on their own timestep (the h3.c README runs video and
 *     audio on independent schedules); NULL = every row uses mod */
typedef struct {
  const void *w_qkvg, *b_qkvg, *w_o, *b_o, *w1, *b1, *w2, *b2;
  const float *mod;
  const void *qnorm_w, *knorm_w;
  const float *mod_prefix;
} h3dit_block_weights;

/* One modality's position on its noise schedule for one sampler step. */
typedef struct {
  float sigma_i;  /* sigma of this step                                        */
  float sigma_a;  /* sigma of the most recent fresh step (extrapolation only)  */
  float sigma_b;  /* sigma of the fresh step before it (extrapolation only)    */
  float dt;       /* step: z <- z + dt * v                                     */
} h3dit_schedule;

/* Bytes of caller-allocated device workspace that h3dit_block_forward,
 * h3dit_routed_attention and h3dit_denoise_step need for this shape
 * (0 if the shape is invalid).  One workspace must not be shared by calls
 * that may run concurrently. */
size_t h3dit_workspace_bytes(const h3dit_shape* shape);

/* Checks a shape without touching the GPU. */
h3dit_status h3dit_check_shape(const h3dit_shape* shape);

/* Host-only switch of the projection GEMMs (no counterpart on the pages: a choice of
 * kernel).  1 (the default): the 256-wide projections run each 256 x 256 output tile
 * on a pair of SMs (a cluster of two CTAs issuing cta_group::2 tensor-core MMAs) when
 * the device can host such clusters, else on one SM; 0: one SM per 128 x 256 tile;
 * -1: query only.  Both kernels sum in the same order and give the same bytes.
 * Returns the previous setting (1 or 0).  Set it while no call is being made. */
int h3dit_gemm_cta_pairs(int enable);

/*
 * Byte offsets, from the start of the workspace, of the regions a call with this
 * shape uses (host only; no counterpart on the pages: a debugging aid).  A region
 * the shape does not reserve reads H3DIT_WS_ABSENT.
 *   status   256 bytes: the int32 device status word (h3dit_sync_status) and the
 *            kernels' work counters (reset by the kernels themselves)
 *   q, k, v  bf16 [H, N, d] after q/k norm and rotary        (block shapes only)
 *   g        bf16 [N, A] routing gate                          (block shapes only)
 *   o        bf16 [N, A] attention output after the gate mix (block shapes only)
 *   u        bf16 [N, F] MLP activations                       (block shapes only)
 *   h        bf16 [N, D] modulated-norm output (norm 2 after a block)
 *   x1       bf16 [N, D] residual rows after the attention half
 *                        (only with H3DIT_KEEP_INTERMEDIATES)
 *   means    fp32 [3, H, Tv, d] q, k, v tile means;  scores fp32 [H, Tv, Tv]
 *   idx      int32 [H, Tv, min(k, Tv)];             pooled fp32 [H, Tv, d]
 *   total    bytes the shape needs (= h3dit_workspace_bytes)
 * Without H3DIT_KEEP_INTERMEDIATES the MLP activations u reuse the q..g region (dead
 * once attention has run) and x1 is not kept, so after h3dit_block_forward only o,
 * h, u and the router regions hold that block's values.  With the flag u has its own
 * region and x1 is copied out after the out projection, so every region above holds
 * the block's values when its stream reaches the end of the call; attention-only
 * shapes (hidden = mlp_width = 0, h3dit_routed_attention) reserve only status and
 * the router regions.
 */
#define H3DIT_WS_ABSENT ((size_t)-1)
typedef struct {
  size_t status, q, k, v, g, o, u, h, x1, means, scores, idx, pooled, total;
} h3dit_workspace_layout;
h3dit_status h3dit_get_workspace_layout(const h3dit_shape* shape, h3dit_workspace_layout* out);

/*
 * h3dit_block_forward -- one DiT block, in place on the residual rows.
 *
 * TensorFold #949, "What it adds" (block.zig: modulated norm, q/k/v and the
 * routing gate, head layout, routing, attention, the pooled branch, the out
 * projection and the MLP) with the precision of its "Precision" list (bf16
 * weights and activations, fp32 sums, fp32 routing); gated residual adds as
 * in the h3.c README's fused gated-AdaLN paragraph.  Per block:
 *   h  = bf16(rms(x) * (1 + scale1) + shift1)
 *   [q|k|v|g] = bf16(h W_qkvg^T + b_qkvg); q, k <- bf16(rope(rms_d(.) * w))
 *   routed attention over video tiles (top-k of tile scores + prefix rows),
 *   dense attention for prefix rows, pooled branch mixed in through g
 *   x1 = bf16(x + gate1 * (o W_o^T + b_o))
 *   h2 = bf16(rms(x1) * (1 + scale2) + shift2)
 *   x2 = bf16(x1 + gate2 * (u W2^T + b2)),  u = bf16(gelu(h2 W1^T + b1)), or with
 *   H3DIT_SWIGLU u = bf16(silu(h2 Wg^T + bg) * (h2 Wu^T + bu)) (the pages' MLP:
 *   the h3.c README's FC1 gate/up + SwiGLU paragraph; TensorFold #949 h3_swiglu)
 * x_inout: bf16 [N, D], overwritten with x2.  Workspace as sized above.
 */
h3dit_status h3dit_block_forward(const h3dit_shape* shape, const h3dit_block_weights* w,
                                 void* x_inout, void* workspace, size_t ws_bytes,
                                 void* stream /* cudaStream_t; NULL = default */);

/*
 * h3dit_routed_attention -- router + routed/dense attention + pooled branch.
 *
 * TensorFold #949, "What it adds" (h3_routing.metal: tile means, tile scores,
 * top-k and the pooled branch; h3_attention.metal: tile-routed attention with
 * fp32 scores and an online softmax), "Precision" (softmax weights rounded to
 * bf16 before the value product) and "Kernel contract" (top-k: NaN ranks as
 * -inf, ties go to the lower tile).
 *   q, k, v       bf16 [H, N, d] head-major (row n of head h at (h*N + n)*d)
 *   gate_or_null  bf16 [N, A]: routing gate; NULL = no pooled mix
 *   out           bf16 [N, A]: out[n, h*d + c]
 *   pooled_out_or_null       fp32 [H, Tv, d]: pooled branch per video tile
 *   topk_idx_out_or_null     int32 [H, Tv, min(k, Tv)]: selected tiles, ascending
 *   tile_scores_out_or_null  fp32 [H, Tv, Tv]: unscaled tile-mean dot products
 * Text/audio (prefix) query rows attend to all N rows; a video row of tile i
 * attends to all prefix rows plus the rows of its selected tiles.  Scale 1/sqrt(d).
 * Tiles are 64-row slices or clipped cubes of the video grid (see h3dit_shape;
 * with a grid, every buffer holds the video rows in cube order); Tv is the number
 * of video tiles (h3dit_tile_spans), at most 1,024, the attention steps of a
 * video query tile, ceil(P / 128) + min(k, Tv), at most 512, and N at most 65,408
 * rows (a prefix query walks N / 128 key steps) -- larger shapes return
 * H3DIT_ERR_SHAPE.
 * The pooled branch and mix run when H3DIT_POOLED is set and gate is given.
 */
h3dit_status h3dit_routed_attention(const h3dit_shape* shape, const void* q, const void* k,
                                    const void* v, const void* gate_or_null, void* out,
                                    float* pooled_out_or_null, int* topk_idx_out_or_null,
                                    float* tile_scores_out_or_null, void* workspace,
                                    size_t ws_bytes, void* stream);

/*
 * h3dit_routed_attention_static -- h3dit_routed_attention without a workspace.
 *
 * No counterpart on the pages: this is a library convenience.  It is meant for
 * callers that cannot call cudaMalloc: code inside a framework that owns all
 * device memory, plugins that may not touch the host process's allocator, or
 * code under a fixed memory budget where an allocation would synchronise the
 * device.  Same arguments and results as h3dit_routed_attention, minus the
 * workspace: scratch comes from a 4 MiB array compiled into the library, which
 * every GPU that loads the library holds until the process exits.
 *   - Every argument is checked before the first CUDA call.  Returns
 *     H3DIT_ERR_WORKSPACE when the shape needs more than 4 MiB of scratch (the
 *     attention-only h3dit_workspace_bytes of the shape, i.e. with
 *     hidden = mlp_width = 0, must be <= 4 MiB: the status word and the router's
 *     tile means, scores, selections and pooled branch; for example 4,096 rows x
 *     24 heads x 128 with 56 video tiles needs 3.1 MB and fits, 15,435 rows x 40
 *     heads x 128 with 218 video tiles needs 26 MB and does not).
 *   - Each call looks up the array's device address with the caller's device
 *     current; the first call on a device may load the library's device code
 *     there, so make it before any stream capture.
 *   - Allocates nothing: no cudaMalloc, no cudaFree.
 *   - All calls share the array and it keeps the previous call's contents; the
 *     call clears the part that must start at zero (the device status word) on
 *     its stream.  Calls whose kernels overlap on the GPU (other streams, other
 *     host threads) race on the array: serialise them.
 *   - A device-side wait that runs out is recorded in the array's status word;
 *     h3dit_routed_attention_static_status reads it (the next call clears it).
 */
h3dit_status h3dit_routed_attention_static(const h3dit_shape* shape, const void* q,
                                           const void* k, const void* v,
                                           const void* gate_or_null, void* out,
                                           float* pooled_out_or_null,
                                           int* topk_idx_out_or_null,
                                           float* tile_scores_out_or_null, void* stream);

/* Synchronises the stream, then returns and clears the device status word of
 * h3dit_routed_attention_static's scratch array on the current device (H3DIT_OK
 * when the calls since the last query ran every wait to its end).  No
 * counterpart on the pages; allocates nothing. */
h3dit_status h3dit_routed_attention_static_status(void* stream);

/*
 * h3dit_denoise_step -- one Euler step of the denoiser, with velocity reuse.
 *
 * h3.c README sampler paragraph: passes that run the model produce a fresh
 * velocity; skipped passes extrapolate it, video and audio on their own
 * schedules; the latents stay on the device.
 *   fresh != 0: x = bf16(z); run blocks[block_ids[i]] for i < n_blocks
 *               (block_ids is a HOST array, blocks a HOST array of structs);
 *               v = fp32(x); v_ring[n_fresh_so_far % 2] = v
 *   fresh == 0: a = slot (n_fresh_so_far - 1) % 2, b = the other slot;
 *               v = v_a + (v_a - v_b) * (sigma_i - sigma_a) / (sigma_a - sigma_b)
 *               when n_fresh_so_far >= 2, else v = v_a
 *   then z <- z + dt * v (fp32).
 * video: the schedule of the video rows (HOST struct); prefix_or_null: the
 * schedule of the text and audio rows (NULL = the video schedule for all rows).
 * z_inout fp32 [N, D]; v_ring fp32 [2, N, D].
 */
h3dit_status h3dit_denoise_step(const h3dit_shape* shape, const h3dit_block_weights* blocks,
                                const int* block_ids, int n_blocks, float* z_inout,
                                float* v_ring, int fresh, const h3dit_schedule* video,
                                const h3dit_schedule* prefix_or_null, int n_fresh_so_far,
                                void* workspace, size_t ws_bytes, void* stream);

/*
 * Both ends of the denoiser: the modality patch projections into the packed
 * hidden rows and the final per-modality AdaLN + narrow output heads (h3.c
 * README: fp32 96 -> 5,376 video and 32 -> 5,376 audio patch projections with
 * fp32 sums rounded to bf16; final audio / video AdaLN on their slices of the
 * residual stream; narrow bf16 output heads).  D = shape->hidden.
 *   c_video, c_audio: latent channels per video / audio row (each a multiple of
 *     32, at most 128; the pages' model: 96 and 32)
 *   w_in_video fp32 [c_video, D] INPUT-major (row j: the weights of input
 *     channel j for every hidden column), b_in_video fp32 [D]; same for audio
 *   w_out_video bf16 [c_video, D] (output-major), b_out_video bf16 [c_video];
 *     same for audio
 *   mod_out_video, mod_out_audio fp32 [2, D]: shift, scale of the final AdaLN
 *   text bf16 [n_text, D]: the text rows (encoder output; constant over steps)
 * All device pointers, 16-byte aligned; audio pointers may be NULL when
 * n_audio == 0 and text when n_text == 0.
 */
typedef struct {
  int c_video, c_audio;
  const float *w_in_video, *b_in_video;
  const float *w_in_audio, *b_in_audio;
  const void *w_out_video, *b_out_video;
  const void *w_out_audio, *b_out_audio;
  const float *mod_out_video, *mod_out_audio;
  const void *text;
} h3dit_ends;

/*
 * Token reduction (h3.c README, token-reduction paragraph): from the block at
 * position `first` of block_ids up to the one before position `last`, each pair
 * of horizontally adjacent video tokens (t, h, 2j), (t, h, 2j + 1) runs as one
 * row, their mean (an odd row's last token runs alone); text and audio rows are
 * untouched.  The full-resolution rows are kept as a bypass, and before position
 * `last` every video token returns as its bypass value plus the update its pair's
 * row received since pooling.  The reduced rows use the grid t x h x ceil(w/2) in
 * cube order, with rotary width coordinate 2j + 0.5 (2j for a lone token).  The
 * pages pool after block 3 and restore before block 40 for the first ten noisy
 * evaluations, before block 30 after that.  Requires H3DIT_TOKEN_REDUCTION in the
 * shape's flags.
 */
typedef struct {
  int first, last;  /* block_ids positions; no reduction unless first < last, first < n */
} h3dit_reduction;

#define H3DIT_PASS_FRESH       0  /* run the blocks                                   */
#define H3DIT_PASS_EXTRAPOLATE 1  /* whole-velocity reuse: extrapolate, no model work */
#define H3DIT_PASS_CORE_REUSE  2  /* patch-in and heads fresh, the blocks' residual   */
                                  /* held from the last fresh pass                    */

/*
 * h3dit_sample_step -- one sampler step on the modality latents, both ends
 * included (h3.c README: sampler paragraph -- video and audio on independent
 * schedules, whole-velocity reuse; core reuse -- the transformer residual held
 * while the patch projection and the timestep-aware head are refreshed; the
 * two reuse modes exclude each other).
 *   z_video fp32 [n_video, c_video], z_audio fp32 [n_audio, c_audio]: latents,
 *     updated in place; video rows in the library's row order (see
 *     h3dit_video_order)
 *   v_ring_video fp32 [2, n_video, c_video], v_ring_audio fp32 [2, n_audio,
 *     c_audio]: the last two fresh velocities (ring slot n_fresh_so_far % 2)
 *   core_residual fp32 [N, D] or NULL: written by a FRESH pass (x_L - x_0),
 *     read by a CORE_REUSE pass
 *   reduction_or_null: token reduction of a FRESH pass (see h3dit_reduction)
 *   pass FRESH / CORE_REUSE:
 *     x_0 = [text; bf16(z_audio W_in_a + b); bf16(z_video W_in_v + b)]
 *     FRESH: x_L = blocks(x_0); residual <- x_L - x_0 when given
 *     CORE_REUSE: x_L = bf16(x_0 + residual)
 *     per modality m: h = bf16(rms(x_L rows of m)(1 + scale_m) + shift_m),
 *     v = h W_out_m^T + b (fp32 sums), z += dt_m v; FRESH also stores v in
 *     the ring
 *   pass EXTRAPOLATE: per modality as in h3dit_denoise_step (fresh == 0)
 *   video, audio: the two modalities' schedules (HOST structs).
 */
h3dit_status h3dit_sample_step(const h3dit_shape* shape, const h3dit_ends* ends,
                               const h3dit_block_weights* blocks, const int* block_ids,
                               int n_blocks, float* z_video, float* z_audio,
                               float* v_ring_video, float* v_ring_audio, float* core_residual,
                               const h3dit_reduction* reduction_or_null, int pass,
                               const h3dit_schedule* video, const h3dit_schedule* audio,
                               int n_fresh_so_far, void* workspace, size_t ws_bytes,
                               void* stream);

/*
 * h3dit_select_blocks -- layer thinning (host only, no GPU).
 * h3.c README layer-thinning paragraph: rank the blocks' AdaLN gates and keep
 * the first and last blocks.  score_b = ||gate1_b||_2 + ||gate2_b||_2 in
 * double precision; the lowest scores are dropped, ties drop the higher index.
 *   mods: HOST fp32 [n_blocks, 6, hidden]; keep: blocks to keep (>= 2)
 *   kept_ids: HOST int32 [keep], ascending.
 */
h3dit_status h3dit_select_blocks(const float* mods, int n_blocks, int hidden, int keep,
                                 int* kept_ids);

/*
 * h3dit_tile_spans -- the routing tiles of a shape (host only, no GPU).
 * first_row[t], n_rows[t] (HOST int32 [number of video tiles]): tile t is the
 * packed rows first_row[t] .. first_row[t] + n_rows[t] - 1.  n_tiles_inout: in,
 * the capacity of both arrays; out, the number of video tiles.
 */
h3dit_status h3dit_tile_spans(const h3dit_shape* shape, int* first_row, int* n_rows,
                              int* n_tiles_inout);

/*
 * h3dit_video_order -- the library's video row order (host only, no GPU).
 * raster_index (HOST int32 [n_video]): for the i-th video row as the library
 * stores it, the raster index (t * video_h + h) * video_w + w of its latent
 * token; the identity without a video grid.  A caller holding video rows in
 * raster order gathers row raster_index[i] into row i before the call and
 * scatters back after it.
 */
h3dit_status h3dit_video_order(const h3dit_shape* shape, int* raster_index);

/*
 * h3dit_linear -- plain bf16 GEMM on the tensor cores: y = bf16(a w^T [+ b]).
 * The projection primitive of the block (TensorFold #949 "Precision": bf16
 * operands, fp32 sums).  a bf16 [M, K], w bf16 [N, K], b bf16 [N] or NULL,
 * y bf16 [M, N].  K a multiple of 64, N a multiple of 256, M >= 1.
 */
h3dit_status h3dit_linear(const void* a, const void* w, const void* b_or_null, void* y, int M,
                          int N, int K, void* stream);

/*
 * Stage timing (tracing).  Between h3dit_profile_begin and h3dit_profile_end
 * the block, attention and denoiser entry points record a CUDA event pair on
 * the caller's stream around each stage below; h3dit_profile_end waits for
 * the recorded events, writes the summed milliseconds and the number of
 * kernel launches per stage, and releases the events.  Off by default; one
 * profiling session per process at a time (not thread-safe).
 */
#define H3DIT_N_STAGES 9
enum {
  H3DIT_STAGE_NORM1 = 0,   /* modulated norm before attention            */
  H3DIT_STAGE_QKVG = 1,    /* q/k/v/gate projection + heads epilogue      */
  H3DIT_STAGE_ROUTER = 2,  /* tile means, scores, top-k, pooled branch    */
  H3DIT_STAGE_ATTN = 3,    /* routed + dense attention + gate mix         */
  H3DIT_STAGE_OUT = 4,     /* out projection + gated residual             */
  H3DIT_STAGE_NORM2 = 5,   /* modulated norm before the MLP               */
  H3DIT_STAGE_FC1 = 6,     /* fc1 + GELU                                  */
  H3DIT_STAGE_FC2 = 7,     /* fc2 + gated residual                        */
  H3DIT_STAGE_SAMPLER = 8  /* rotary table, latent cast, Euler/extrapolate */
};
h3dit_status h3dit_profile_begin(int max_records);
h3dit_status h3dit_profile_end(float* stage_ms, int* stage_launches, int n_stages);

/* Number of kernels this library has launched in this process so far. */
unsigned long long h3dit_launch_count(void);

/*
 * h3dit_selftest_timeout -- checks the device-side failure path (diagnostics).
 * Launches one CTA that waits, through the same bounded mbarrier wait every
 * tensor-core kernel uses, on a barrier that nothing signals, with a limit of
 * limit_ms milliseconds (1..10000).  The wait runs out, the kernel records
 * H3DIT_ERR_TIMEOUT in the workspace status word and returns; read it with
 * h3dit_sync_status.  No fault or trap is raised: the context stays usable.
 * workspace: device memory of at least 256 bytes whose first int is the status.
 */
h3dit_status h3dit_selftest_timeout(void* workspace, size_t ws_bytes, int limit_ms,
                                    void* stream);

/* Synchronises the stream, reads the device status word of this workspace,
 * clears it and returns it (H3DIT_OK or H3DIT_ERR_TIMEOUT). */
h3dit_status h3dit_sync_status(void* workspace, size_t ws_bytes, void* stream);

const char* h3dit_status_string(h3dit_status s);

/* Library version, e.g. "h3dit 0.1.0 sm_103a". */
const char* h3dit_version(void);

#ifdef __cplusplus
}
#endif
#endif /* H3DIT_H_ */
