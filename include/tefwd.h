/*
 * tefwd - forward pass of a pre-norm transformer encoder block over a packed
 * batch of variable-length sequences, with int8 row-scaled (q8_row) weights,
 * for NVIDIA GB300 (sm_103a).
 *
 * Sources (the pages this library restates; each entry point cites its
 * section):
 *   [EG2]  "cortiq-engine 0.8.39 src/gpu_metal/egemma2.rs"  (EmbeddingGemma 2
 *          text/vision encoders on Metal: Prog::rms, Prog::add_norm,
 *          Prog::gelu, Prog::qkv, Prog::attention, att_plan,
 *          TextGpu::forward, VisionGpu::forward)
 *   [ZI]   "cortiq-engine 0.7.6 src/gpu_metal/zimage.rs"  (Z-Image DiT on
 *          Metal: module doc "The chain" / "Measured", Enc::gemm, Enc::rowop,
 *          Enc::block, bench_gemm, bench_flash)
 *   [VIT]  "cera 0.2.4 src/model/vision_encoder_gpu.rs"  (LFM2-VL ViT:
 *          trait VitGpuOps, encode_image_gpu)
 *
 * Conventions shared by every entry point
 *   - Memory is owned by the caller.  The library never allocates, frees or
 *     synchronises (te_check excepted); scratch is passed in as a workspace.
 *     The one exception is te_encoder_block_fwd_static, which uses a fixed
 *     array of the library's own (see its comment).
 *   - Device pointers are CUDA device addresses on the current device; host
 *     pointers (the *_host arguments and descriptors) are read during the
 *     call only.  Every device pointer must be 16-byte aligned and every
 *     leading dimension a multiple of 16 bytes.
 *   - Matrices are row-major.  "bf16" is IEEE bfloat16 stored as uint16,
 *     written with round-to-nearest-even.
 *   - All arguments are validated on the host before anything is launched;
 *     on any error no output is touched and a non-TE_OK status is returned,
 *     with a message in te_last_error() (thread-local).  Errors from earlier
 *     asynchronous work surface as TE_ECUDA from te_check().
 *   - Work is enqueued on `stream` (NULL = the legacy default stream); the
 *     calls return before it completes.  te_q8_linear, te_q8_gated_linear,
 *     te_attn_varlen_fwd,
 *     the row ops and te_encoder_block_fwd are capturable in a CUDA graph
 *     (no host synchronisation, no allocation).
 */
#ifndef TEFWD_H
#define TEFWD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *te_stream; /* the same handle as cudaStream_t */

typedef enum {
    TE_OK = 0,
    TE_EINVAL = 1,      /* a NULL pointer, a bad enum, or a bad cu_seqlens   */
    TE_ESHAPE = 2,      /* a size outside what the kernels support           */
    TE_EALIGN = 3,      /* a pointer or leading dimension not 16-byte aligned */
    TE_EWORKSPACE = 4,  /* workspace too small                              */
    TE_ECUDA = 5,       /* a CUDA runtime/driver call failed                 */
    TE_EDEVICE = 6      /* a kernel gave up a bounded wait (see te_check)    */
} te_status;

typedef enum { TE_F32 = 0, TE_BF16 = 1 } te_dtype;
typedef enum { TE_NORM_RMS = 0, TE_NORM_LN = 1 } te_norm_kind;
typedef enum { TE_ACT_GELU_TANH = 0, TE_ACT_SILU = 1 } te_act_kind;
typedef enum { TE_RESID_PLAIN = 0, TE_RESID_SANDWICH = 1 } te_resid_form;

/* One quantised weight.
 * q8_row ([ZI] module doc "The chain": the file's q8_row bytes, int8 tile
 * staged exactly, row scale applied in the f32 epilogue):
 *   q     int8 [n, k] row-major (device)        W[o, j] = scale[o] * q[o, j]
 *   scale f32 [n] (device)
 *   bias  f32 [n] (device) or NULL              ([VIT] bias_add of the linears)
 *   block_scale NULL
 * 32-element block formats (Q8_0, Q4_0 of [VIT]; unpacked by te_q8_0_unpack /
 * te_q4_0_unpack into q and block_scale):
 *   block_scale f16 bits [n, k/32] (device)    W[o, j] = scale[o] * bf16(q[o, j] * d[o, j/32])
 *   scale may be NULL (1).  The product q * d is exact in f32 and is rounded
 *   once, to the bf16 tensor-core operand.
 * q8_2f ([ZI] ensure_dev: q8_row plus a per-column f16 field):
 *   col f32 [k] (device) or NULL               W[o, j] = scale[o] * bf16(q[o, j] * col[j])
 *   ([ZI] folds the field into the activation's producer; here it is folded
 *   into the widened weight, rounded once to the bf16 operand.)  col and
 *   block_scale may not both be given.
 * Requirements: k % 64 == 0, n % 32 == 0, n >= 32; block_scale 4-byte and
 * col 16-byte aligned. */
typedef struct {
    const int8_t *q;
    const float *scale;
    const float *bias;
    int32_t n;
    int32_t k;
    const uint16_t *block_scale;
    const float *col;
} te_q8w;

/* Activation applied in a GEMM epilogue (TE_EPI_NONE: none). */
typedef enum { TE_EPI_NONE = 0, TE_EPI_GELU_TANH = 1, TE_EPI_SILU = 2 } te_epilogue;

/* Unpack the 32-element block formats of [VIT] (the test quantisers of
 * vision_encoder_gpu.rs; packed row-major, k/32 blocks per row):
 *   Q8_0: 34 bytes a block = f16 scale d (little-endian) + 32 int8 q
 *   Q4_0: 18 bytes a block = f16 scale d + 16 bytes; byte i holds element i
 *         in its low nibble and element i + 16 in its high nibble, each
 *         stored as q + 8 (q in [-8, 7])
 * into q int8 [n, k] and block_scale f16 bits [n, k/32] (bit-exact integer
 * work).  k % 32 == 0; q 16-byte aligned, block_scale 4-byte aligned. */
te_status te_q8_0_unpack(const void *packed, int32_t n, int32_t k, int8_t *q, uint16_t *block_scale,
                         te_stream stream);
te_status te_q4_0_unpack(const void *packed, int32_t n, int32_t k, int8_t *q, uint16_t *block_scale,
                         te_stream stream);

/* One item of a grouped q8 GEMM ([EG2] Prog::mm item table, one item per
 * grid z; [ZI] Enc::gemm, z <= 3).  All items share the activation x.
 *   y        [m, ldy] of y_dtype (TE_F32 or TE_BF16), device
 *   epilogue te_epilogue: y = act(bf16(s*acc + b)), the ungated MLP's
 *            activation folded into its producer ([VIT] encode_image_gpu
 *            "gelu" after the up projection); needs residual == NULL
 *   residual f32 [m, ldr] or NULL; y may alias residual (same pointer and
 *            leading dimension) for the in-place x += proj of the plain
 *            pre-norm block ([VIT] encode_image_gpu "add"). */
typedef struct {
    te_q8w w;
    void *y;
    int64_t ldy;
    int32_t y_dtype;
    int32_t epilogue;
    const float *residual;
    int64_t ldr;
} te_q8_item;

/* q8_linear: for each item i < z,
 *     y_i[t, o] = scale_i[o] * sum_j x[t, j] * q_i[o, j]  (+ bias_i[o])  (+ residual_i[t, o])
 * x: bf16 [m, k] with leading dimension ldx (elements), device.
 * f32 accumulation on the tensor cores; int8 widened to bf16 exactly.
 * Sizes: 1 <= m, k % 64 == 0 and every item's w.k == k, 1 <= z <= 4.
 * Cites [ZI] module doc ("Each GEMM stages the int8 tile as half (exact) and
 * applies the row scale in its f32 epilogue"), [EG2] Prog::mm. */
te_status te_q8_linear(const void *x, int64_t ldx, int32_t m, int32_t k,
                       const te_q8_item *items, int32_t z, te_stream stream);

/* q8_gated_linear: the gate|up projections and the gate in one pass,
 *     m[t, f] = act(bf16(g[t, f])) * bf16(u[t, f])   (stored bf16)
 *     g = s_g * (x . q_g^T) + b_g,   u = s_u * (x . q_u^T) + b_u
 * with act GELU-tanh or SiLU (te_act_kind).  The two products are rounded to
 * bf16 before the gate, exactly as storing g|u and then applying te_gate_act
 * would; the g|u panel itself is never written.
 * x: bf16 [m, k] (ldx); wg, wu: q8_row weights of equal shape [f, k]
 * (f % 32 == 0, k % 64 == 0); out: bf16 [m, ldm].
 * Cites [EG2] Prog::gelu (O = gelu_tanh(G) U over the gate|up GEMM's
 * output), [ZI] Enc::block SwiGLU (h = silu(w1 x) (w3 x)) and the module
 * doc's rule of folding a column-wise factor into the producer's epilogue. */
te_status te_q8_gated_linear(const void *x, int64_t ldx, int32_t m, int32_t k, const te_q8w *wg,
                             const te_q8w *wu, int32_t act, void *out, int64_t ldm,
                             te_stream stream);

/* attn_varlen_fwd: bidirectional multi-head attention over packed rows.
 * qkv: bf16 [T, ld] (device) holding q heads at columns q_off + h*hd, k and
 * v heads at k_off / v_off + g*hd, g = h / (nq_heads / nkv_heads).
 * Sequence s owns rows [cu[s], cu[s+1]); T = cu[nseq].  For a query row i
 * of sequence s the visible keys are the rows j of s with window == 0 or
 * |i - j| <= window.
 *     out[i, h*hd + c] = sum_j softmax_j(scale * q_i . k_j) v_j[c]   (bf16)
 * cu_host / cu_dev: the same int32 [nseq+1] offsets on the host (validated,
 * used to size the launch) and on the device (read by the kernel); cu[0] = 0,
 * strictly increasing.  hd in {64, 128}; nq_heads % nkv_heads == 0;
 * window >= 0; out bf16 [T, ldo], must not overlap qkv.
 * Cites [EG2] Prog::attention and att_plan (window span, "zeros outside the
 * window"), [ZI] module doc (flash attention, online softmax), [VIT]
 * VitGpuOps::attention. */
te_status te_attn_varlen_fwd(const void *qkv, int64_t ld, int32_t q_off, int32_t k_off,
                             int32_t v_off, const int32_t *cu_host, const int32_t *cu_dev,
                             int32_t nseq, int32_t nq_heads, int32_t nkv_heads, int32_t hd,
                             int32_t window, float scale, void *out, int64_t ldo,
                             te_stream stream);

/* attn_items_fwd: the same attention over two-range items ([ZI] PFa
 * {img_off, n_img, cap_off, n_cap}: the CFG program's image rows and caption
 * rows of one item attend as one sequence).  Item i is int32
 * [off1, len1, off2, len2]: its joint positions 0..len1-1 are the rows
 * off1.., positions len1..len1+len2-1 the rows off2..; the window applies to
 * joint positions; each query's output goes to its own row.
 * items_host / items_dev: the same int32 [nitems, 4] on the host (validated)
 * and on the device (16-byte aligned).  len1 >= 1, len2 >= 0, and when
 * len2 > 0, len1 % 32 == 0 (a key tile spanning both ranges is loaded in
 * 32-row pieces); every range inside rows [0, rows).  Otherwise as
 * te_attn_varlen_fwd (len2 = 0 for every item gives the same result). */
te_status te_attn_items_fwd(const void *qkv, int64_t ld, int32_t q_off, int32_t k_off,
                            int32_t v_off, const int32_t *items_host, const int32_t *items_dev,
                            int32_t nitems, int32_t rows, int32_t nq_heads, int32_t nkv_heads,
                            int32_t hd, int32_t window, float scale, void *out, int64_t ldo,
                            te_stream stream);

/* rownorm: y = Norm(pre * x) per row.
 *   RMS: v / sqrt(mean(v^2) + eps) * w            ([EG2] Prog::rms)
 *   LN : (v - mean) / sqrt(var + eps) * w + b      ([VIT] VitGpuOps::layernorm;
 *        biased variance, b may be NULL)
 * x [t, ldx] of xdt (f32/bf16), y [t, ldy] of ydt; may not overlap unless
 * identical with equal dtypes.  d % 8 == 0, 8 <= d <= 4096. */
te_status te_rownorm(const void *x, int32_t xdt, int64_t ldx, const float *w, const float *b,
                     int32_t kind, float eps, float pre, void *y, int32_t ydt, int64_t ldy,
                     int32_t t, int32_t d, te_stream stream);

/* add_norm: the residual add fused with the next pre-norm.
 *   h (f32 [rows, d], in place):
 *     w_post != NULL:  h = (h + RMS(t) * w_post) * post     ([EG2] Prog::add_norm,
 *                                                            [ZI] Enc::rowop post mode)
 *     w_post == NULL:  h = h + t      (t may be NULL: no add)
 *   then, when w_next != NULL:  a = Norm(h) * w_next (+ b_next), kind RMS/LN,
 *   stored as adt in a [rows, d].  d % 8 == 0, 8 <= d <= 4096. */
te_status te_add_norm(float *h, const float *t, const float *w_post, float post,
                      const float *w_next, const float *b_next, int32_t kind, float eps,
                      void *a, int32_t adt, int32_t rows, int32_t d, te_stream stream);

/* adaLN-modulated row ops of the DiT block ([ZI] Enc::block: per block the
 * vectors [s_msa | g_msa | s_mlp | g_mlp], a scale on each pre-norm and a gate
 * on each post-norm residual, Enc::rowop has_s / has_g; refine_caption: the
 * unmodulated block is s = 0, gate = 1).  The pages do not print the row
 * op's arithmetic; the reading taken is
 *   pre-norm:  a = (Norm(x) * w (+ b)) * (1 + s)          s: f32 [d]
 *   residual:  h = (h + g * RMS(t) * w_post) * post       g: f32 [d]
 * (w_post == NULL: h = h + g * t).  NULL s or g: unmodulated.  Otherwise as
 * te_rownorm / te_add_norm. */
te_status te_rownorm_mod(const void *x, int32_t xdt, int64_t ldx, const float *w, const float *b,
                         const float *mod_scale, int32_t kind, float eps, float pre, void *y,
                         int32_t ydt, int64_t ldy, int32_t t, int32_t d, te_stream stream);

te_status te_add_norm_mod(float *h, const float *t, const float *w_post, const float *gate,
                          float post, const float *w_next, const float *b_next,
                          const float *mod_scale, int32_t kind, float eps, void *a, int32_t adt,
                          int32_t rows, int32_t d, te_stream stream);

/* qk_prep_rope: in place on the bf16 q|k panel of qkv [rows, ld].
 * Per row and head: if qn/kn != NULL, x = x / sqrt(mean(x^2) + eps) * w
 * (w: f32 [hd], shared by all heads); then if sec > 0, rotate-half RoPE within
 * each section of sec channels: for section s and i < sec/2 the pair
 * (x[s*sec+i], x[s*sec+i+sec/2]) rotates by the angle whose cos/sin sit at
 * table column s*sec/2 + i of table row pos[row] (pos == NULL: the row index);
 * then q heads are multiplied by q_mul.  cos/sin: f32 [table_rows, hd/2].
 * sec in {0, hd, hd/2}; hd in {64, 128}.
 * Cites [EG2] Prog::qkv and EgQkv.sec (1-D sec = hd; vision 2-D sec = hd/2,
 * "the column half, then the row half"), [ZI] Enc::block (qk-norm + RoPE in
 * place, q pre-multiplied). */
te_status te_qk_prep_rope(void *qkv, int64_t ld, int32_t q_off, int32_t k_off, int32_t nq,
                          int32_t nkv, int32_t hd, const float *qn, const float *kn, float eps,
                          const float *cos, const float *sin, const int32_t *pos,
                          int32_t table_rows, int32_t sec, float q_mul, int32_t rows,
                          te_stream stream);

/* selftest_wait_timeout: launches one kernel whose mbarrier wait can never
 * complete, bounded like every pipeline wait of the library but after
 * limit_us microseconds (1..1e6).  The kernel then records the same error a
 * stuck pipeline records and returns: the next te_check reports TE_EDEVICE
 * (and clears it) and the context stays usable.  No fault is involved.  The
 * pages have no counterpart of this entry point. */
te_status te_selftest_wait_timeout(int32_t limit_us, te_stream stream);

/* mma_peak: the tensor-core ceiling of the q8 GEMM's own MMA form.  On every
 * SM pair of the current device, `stages` x 8 back-to-back 2-SM MMAs
 * (tcgen05 kind::f16, A in TMEM, B in shared memory, M = 256, N = bn,
 * K = 16, f32 accumulate) with no loads, no waits and no epilogue; *ms
 * receives the launch's device time (CUDA events on `stream`; the call
 * waits for it).  Work = (SMs / 2) x stages x 8 x 2 x 256 x bn x 16 flops.
 * bn in {64, 128, 192, 256}; 1 <= stages <= 2^22.  A measurement aid: the
 * counterpart of the [ZI] module doc's "Ceiling" item (a pure MMA loop with
 * no loads). */
te_status te_mma_peak(int32_t bn, int32_t stages, float *ms, te_stream stream);

/* cast_bf16: y = bf16(x) (round to nearest even) for x f32 [rows, d] (ldx),
 * y bf16 [rows, ldy]; d % 8 == 0.  The per-layer input path's GEMM reads the
 * residual stream this way. */
te_status te_cast_bf16(const float *x, int64_t ldx, void *y, int64_t ldy, int32_t rows, int32_t d,
                       te_stream stream);

/* qkv_prep_rope: qk_prep_rope, and with v_norm != 0 also the v heads (at
 * v_off + g*hd) RMS-normalised without a weight and without RoPE:
 * v = v / sqrt(mean(v^2) + eps) ([EG2] Prog::qkv "q/k norm + RoPE, v norm":
 * one pass over the nq + 2 nkv heads, weights for q and k only). */
te_status te_qkv_prep_rope(void *qkv, int64_t ld, int32_t q_off, int32_t k_off, int32_t v_off,
                           int32_t nq, int32_t nkv, int32_t hd, const float *qn, const float *kn,
                           int32_t v_norm, float eps, const float *cos, const float *sin,
                           const int32_t *pos, int32_t table_rows, int32_t sec, float q_mul,
                           int32_t rows, te_stream stream);

/* gate_act: m = act(g) * u with g = gu[:, 0:f], u = gu[:, u_off:u_off+f];
 * u_off < 0: ungated, m = act(g).  act: GELU-tanh
 * 0.5 g (1 + tanh(sqrt(2/pi)(g + 0.044715 g^3))) or SiLU g / (1 + e^-g).
 * gu bf16 [rows, ld], m bf16 [rows, ldm].  f % 8 == 0.
 * Cites [EG2] Prog::gelu, [ZI] Enc::block SwiGLU, [VIT] VitGpuOps::gelu. */
te_status te_gate_act(const void *gu, int64_t ld, int32_t u_off, int32_t act, void *m,
                      int64_t ldm, int32_t rows, int32_t f, te_stream stream);

/* pool_mean: out[s] = (1/len_s) sum_{r in s} RMS(x_r) * w_final
 * (w_final == NULL: the plain mean).  x f32 [T, d], out f32 [nseq, d].
 * Cites [EG2] TextGpu::forward (row_inv then pool: final-normed hidden
 * state mean-pooled per sequence).  d % 8 == 0, d <= 4096. */
te_status te_pool_mean(const float *x, int32_t d, const int32_t *cu_host,
                       const int32_t *cu_dev, int32_t nseq, const float *w_final, float eps,
                       float *out, te_stream stream);

/* One encoder block ([EG2] TextGpu::forward layer loop; [ZI] Enc::block;
 * [VIT] encode_image_gpu block loop). */
typedef struct {
    int32_t d, n_heads, n_kv_heads, head_dim, ffn;
    int32_t norm_kind;   /* te_norm_kind: the FFN pre-norm and the next norm      */
    int32_t resid_form;  /* te_resid_form                                          */
    int32_t act;         /* te_act_kind                                            */
    int32_t gated;       /* 1: gate|up pair (wg, wu), 0: single up (wg)            */
    int32_t window;      /* sliding window (0 = full attention)                    */
    float eps, attn_scale, post, q_mul;
    te_q8w wq, wk, wv, wo, wg, wu, wd;
    const float *ffn_norm_w, *ffn_norm_b;   /* FFN pre-norm (b: LN only, or NULL) */
    const float *post_attn_w, *post_ffn_w;  /* sandwich form only                 */
    const float *next_norm_w, *next_norm_b; /* next block's pre-norm, NULL = none */
    const float *q_norm, *k_norm;           /* [head_dim] or NULL                 */
    const float *rope_cos, *rope_sin;       /* [rope_rows, head_dim/2] or NULL    */
    const int32_t *rope_pos;                /* [T] table row per packed row, NULL = row index */
    int32_t rope_sec, rope_rows;
    /* adaLN modulation (sandwich form only; see te_add_norm_mod), or NULL:
     * mod = this block's f32 [4, d] = s_msa | g_msa | s_mlp | g_mlp (s_msa
     * scales this block's input a, which the caller's previous norm made);
     * next_mod_scale = the next block's s_msa, f32 [d], applied to a_out. */
    const float *mod, *next_mod_scale;
    int32_t v_norm;      /* 1: RMS-normalise the v heads too (te_qkv_prep_rope) */
    /* per-layer input path ([EG2] TextGpu::forward "per-layer input", LayerSpec
     * ple_in / ple_gate / ple_proj / ple_norm, TextSpec ple_scale / ple_norm;
     * sandwich form only), or ple_dim == 0.  After the FFN residual (then with
     * post 1 and no next norm):
     *   pin = RMS(ple_scale * (ple_x . W_in^T)) * ple_norm_w      [t, ple_dim]
     *   z   = gelu_tanh(bf16(bf16(x) . W_gate^T)) * pin           [t, ple_dim]
     *   x   = (x + RMS(z . W_proj^T) * ple_post_w) * post;  a = Norm_next(x)
     * ple_x: bf16 [t, d], the stack's input (the same for every layer). */
    int32_t ple_dim;
    float ple_scale;
    te_q8w ple_in, ple_gate, ple_proj;
    const float *ple_norm_w, *ple_post_w;
    const void *ple_x;
    /* two-range attention items ([ZI] module doc "The chain": the CFG pair is
     * one batch-2 program over rows [img0 | img1 | cap0 | cap1], every
     * row-local step runs once over all rows and attention runs per item over
     * its two row ranges; PFa {img_off, n_img, cap_off, n_cap}), or
     * n_attn_items == 0 (attention per cu_seqlens sequence).  With items the
     * attention step is te_attn_items_fwd over attn_items_host / _dev (int32
     * [n_attn_items, 4] = off1, len1, off2, len2; the same table on the host
     * and, 16-byte aligned, on the device); the items must cover every row of
     * [0, t) exactly once, and cu_seqlens then only gives t. */
    const int32_t *attn_items_host, *attn_items_dev;
    int32_t n_attn_items;
    /* per-step GPU timing (the pages' per-op-class profiling switch: [EG2]
     * the CMF_EGEMMA2_GPU_PROF recorder, one command buffer per op class;
     * [VIT] VitProfiler), or NULL.  TE_BLOCK_PROF_EVENTS events that the
     * caller created (cudaEvent_t with timing, owned by the caller); the
     * block records event k on its stream at step boundary k:
     *   0 before the q|k|v projection, 1 after it, 2 after the q/k norm and
     *   RoPE (right after 1 when the block has none), 3 after attention,
     *   4 after the O projection, 5 after the residual and FFN pre-norm,
     *   6 after gate|up, 7 after the down projection, 8 after the closing
     *   row ops (with the per-layer input path).
     * The time between events k and k+1 is step class k.  Only event records
     * are added: nothing synchronises.  Rejected (TE_EINVAL) while the stream
     * is being captured into a graph, where records give no timing. */
    void *const *prof_events;
} te_block_desc;

#define TE_BLOCK_PROF_EVENTS 9

/* Workspace bytes te_encoder_block_fwd needs for t packed rows. */
size_t te_encoder_block_workspace(const te_block_desc *desc, int32_t t);

/* encoder_block_fwd: one block, in place.
 *   x: f32 [t, d] residual stream (in/out).
 *   a: bf16 [t, d]; in: this block's normed input; out: Norm_next(x_out) when
 *      next_norm_w != NULL (otherwise left as the FFN's input).
 * Plain form ([VIT]):    x += Wo attn(qkv(a)) (+b); a = Norm2(x);
 *                        x += Wd act(Wg a, Wu a) (+b); a = Norm_next(x)
 * Sandwich form ([EG2], [ZI]): x = (x + RMS(Wo attn) w_pa) post; a = RMS(x) w_2;
 *                        x = (x + RMS(Wd act) w_pf) post; a = RMS(x) w_next
 * With adaLN modulation (mod != NULL, [ZI] Enc::block):
 *                        x = (x + g_msa RMS(Wo attn) w_pa) post; a = RMS(x) w_2 (1 + s_mlp);
 *                        x = (x + g_mlp RMS(Wd act) w_pf) post; a = RMS(x) w_next (1 + s_next)
 * t = cu_host[nseq]; workspace of te_encoder_block_workspace(desc, t) bytes,
 * 256-byte aligned. */
te_status te_encoder_block_fwd(const te_block_desc *desc, float *x, void *a,
                               const int32_t *cu_host, const int32_t *cu_dev, int32_t nseq,
                               void *workspace, size_t ws_bytes, te_stream stream);

/* Size of the fixed scratch array of te_encoder_block_fwd_static (bytes). */
#define TE_STATIC_SCRATCH_BYTES ((size_t)32 << 20)

/* te_encoder_block_fwd_static: the same block as te_encoder_block_fwd, with
 * the same arguments and results, for callers that cannot allocate device
 * memory - e.g. an application whose device memory is all handed to its own
 * allocator and which forbids libraries from calling cudaMalloc, or a
 * latency-critical loop where no allocation may happen.  Such a caller has
 * no workspace to pass, so this entry point takes none: its scratch is one
 * fixed array in device memory owned by the library
 * (TE_STATIC_SCRATCH_BYTES = 32 MiB, 256-byte aligned), which every GPU that
 * loads the library holds until the process exits.  Nothing is allocated or
 * freed by a call.
 *   - Limit: te_encoder_block_workspace(desc, t) must be at most
 *     TE_STATIC_SCRATCH_BYTES, i.e. t up to about TE_STATIC_SCRATCH_BYTES /
 *     te_encoder_block_workspace(desc, 1) packed rows (a d=512, F=2048 block
 *     needs 10,240 bytes a row: about 3,270 rows); larger t returns
 *     TE_EWORKSPACE before anything is launched.  The descriptor is
 *     validated first (TE_EINVAL / TE_ESHAPE / TE_EALIGN as for
 *     te_encoder_block_fwd).
 *   - The first call on each device (and the first after that device's
 *     context was destroyed and recreated, e.g. by cudaDeviceReset) looks up
 *     the array's device address with that device current; make that call
 *     before any stream capture.
 *   - Every call shares the one array, which keeps the last call's contents.
 *     No part of it needs to start at zero (each scratch region is written
 *     before it is read).  Calls that overlap on the GPU - on different
 *     streams or from different host threads - race on the array: issue them
 *     on one stream.
 * The pages have no counterpart of this entry point. */
te_status te_encoder_block_fwd_static(const te_block_desc *desc, float *x, void *a,
                                      const int32_t *cu_host, const int32_t *cu_dev,
                                      int32_t nseq, te_stream stream);

/* Synchronises `stream`; returns TE_ECUDA for a pending asynchronous CUDA
 * error, TE_EDEVICE if a kernel gave up a bounded wait since the last check
 * (the device-side word is then cleared), TE_OK otherwise. */
te_status te_check(te_stream stream);

/* Message of this thread's last non-OK status ("" if none). */
const char *te_last_error(void);

/* Library version string. */
const char *te_version(void);

/* Struct sizes as this library was compiled: sizes[0] = sizeof(te_q8w),
 * [1] = sizeof(te_q8_item), [2] = sizeof(te_block_desc), for a binding to
 * check its own mirror of them.  Writes min(n, 3) entries and returns 3;
 * sizes may be NULL when n == 0.  Host only. */
int32_t te_abi_sizes(size_t *sizes, int32_t n);

#ifdef __cplusplus
}
#endif

#endif /* TEFWD_H */
