/*
 * lca.h -- C ABI of the B300 (sm_103a) hybrid compressed attention library (liblca.so).
 *
 * The library implements the attention path of DeepSeek-V4 as described in the
 * web write-ups on the model:
 *   [P1] gxgjx.lffhtl.com/lxrt/355279.html, section "混肃穆力机制" (hybrid attention):
 *        CSA steps one to four (KV compression; lightning indexer + top-k; core
 *        Multi-Query Attention; grouped output projection), the HCA paragraph, and the
 *        tricks: Q/KV RMSNorm, partial RoPE with an output RoPE at -i, a sliding-window
 *        branch, and an attention sink.
 *   [P4] zhinnengdao.top, "DeepSeek-V4开源解读", section 3.1 "Hybrid Attention: CSA + HCA":
 *        m=4, 64 indexer heads of dim 128, top-k 512, m'=128, RoPE on the last 64 dims,
 *        one learnable sink logit per head, an SWA branch next to each attention.
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers to buffers the caller owns; the library
 *     allocates nothing and keeps no pointer after the call returns.
 *   - Work is enqueued on `stream` and runs asynchronously; results are ready when the
 *     stream reaches that point.
 *   - Arguments are validated on the host before anything is launched: a bad size,
 *     a NULL pointer, a pointer not aligned to 16 bytes, an unsupported shape or a
 *     workspace that is too small returns an error status and launches nothing.
 *     lca_last_error() then describes the problem (thread-local string).
 *   - Values that live on the device (positions, first entries, indices) are checked by
 *     the kernels: a violation skips the offending row and sets a bit in the device
 *     error word, which lca_device_error() reads and clears.
 *   - bf16 tensors are passed as raw 16-bit patterns (lca_bf16).  Row-major layouts;
 *     strides are in ELEMENTS.
 */
#ifndef LCA_H
#define LCA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Every declaration below is an exported symbol of liblca.so (built with hidden default
 * visibility; only this ABI is visible). */
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

typedef struct CUstream_st *cudaStream_t; /* the CUDA runtime's stream handle */
typedef uint16_t lca_bf16;                /* raw bfloat16 bit pattern */

typedef enum lca_status {
    LCA_OK = 0,
    LCA_ERR_INVALID_ARG = 1,  /* bad size, NULL or misaligned pointer */
    LCA_ERR_UNSUPPORTED = 2,  /* shape outside what the kernels are built for */
    LCA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than the *_workspace() size */
    LCA_ERR_CUDA = 4,         /* a CUDA runtime call or a launch failed */
    LCA_ERR_TIMEOUT = 5,      /* a kernel gave up on a bounded wait (device error word) */
    LCA_ERR_DEVICE = 6        /* a device-side check fired (device error word) */
} lca_status;

/* Bits of the device error word (see lca_device_error). */
#define LCA_DEVERR_MISSING_TOKEN  0x1u  /* compress: a window token outside the staging rows */
#define LCA_DEVERR_INDEX_RANGE    0x2u  /* attend: an index outside [0, cache_rows) (not -1) */
#define LCA_DEVERR_VISIBLE_RANGE  0x4u  /* visible entries exceed cache_rows; clamped */
#define LCA_DEVERR_NEGATIVE_POS   0x8u  /* a negative position */
#define LCA_DEVERR_FP16_RANGE     0x10u /* attend: a KV or window row element, or an element of
                                         * the normalised, rotated query, outside fp16's finite
                                         * range (|x| > 65504, inf, nan): the products saturate
                                         * there, so that call's outputs are not accurate */
#define LCA_DEVERR_SELECT         0x20u /* indexer with top-k: a candidate would not fit its
                                         * buffer and was dropped (a selection fault; the
                                         * query's list is then not exact) */
#define LCA_DEVERR_TIMEOUT        0x100u /* a bounded wait inside a kernel ran out */

/* Layer parameters (names follow the pages' notation). */
typedef struct lca_attn_params {
    int heads;           /* H: query heads sharing one KV (MQA); 1..64 */
    int head_dim;        /* c: width of a KV entry and of a head; 128, 256 or 512 */
    int rope_dims;       /* R: trailing dims rotated by RoPE; even, 0..c, R/2 <= 64 */
    float rope_base;     /* RoPE base; frequency of pair d is base^(-2d/R) */
    float rms_eps;       /* RMSNorm epsilon */
    float softmax_scale; /* logit scale; 0 selects 1/sqrt(c) */
    int window;          /* W: sliding-window tokens, the query's own token included */
    int ratio;           /* m (CSA) or m' (HCA): tokens per compressed entry */
    int topk;            /* k: entries selected per query (CSA) */
    int idx_heads;       /* H_I: indexer query heads */
    int idx_dim;         /* d_I: indexer head dim */
} lca_attn_params;

/* ---------------------------------------------------------------------------------
 * KV compression ([P1] CSA step one "KV 压缩" and the HCA paragraph; [P4] 3.1).
 *
 * For each sequence b and e < n_new, entry j = first_entry[b] + e pools the tokens
 *   CSA: t in [m(j-1), m(j+1)) clipped at 0   (windows of 2m, stride m, overlapping)
 *   HCA: t in [m'j, m'(j+1))                   (no overlap)
 * with softmax weights over (tok_z[t] + pos_bias[t - nominal window start]), then applies
 * RMSNorm with gamma (skipped when gamma == NULL) and, when apply_rope != 0, RoPE at the
 * entry's last token m(j+1)-1 to the trailing rope_dims dims, and stores the row in bf16
 * at cache[b*cache_batch_stride + j*width].
 *   width       row width: head_dim for the KV cache, idx_dim for the indexer keys;
 *               multiple of 8, at most 1024.
 *   tok_v       [batch][n_tok][width] bf16, token t of sequence b at local row
 *               t - tok_pos0[b]; tok_v_batch_stride elements between sequences.
 *   tok_z       [batch][n_tok] fp32 compressor logits, tok_z_batch_stride between sequences.
 *   tok_pos0    [batch] int32 (device): position of local row 0.
 *   pos_bias    [2m] (CSA) or [m'] (HCA) fp32 learned offset biases.
 *   gamma       [width] fp32 or NULL.
 *   first_entry [batch] int32 (device).
 *   cache_rows  rows available per sequence; j >= cache_rows is an error.
 * A window token outside the staging rows sets LCA_DEVERR_MISSING_TOKEN and skips the entry.
 * ------------------------------------------------------------------------------- */
lca_status csa_compress_kv(const lca_attn_params *p, int batch, int width,
                           const lca_bf16 *tok_v, int64_t tok_v_batch_stride, int n_tok,
                           const float *tok_z, int64_t tok_z_batch_stride,
                           const int32_t *tok_pos0, const float *pos_bias, const float *gamma,
                           int apply_rope, const int32_t *first_entry, int n_new,
                           lca_bf16 *cache, int64_t cache_batch_stride, int64_t cache_rows,
                           cudaStream_t stream);
lca_status hca_compress_kv(const lca_attn_params *p, int batch, int width,
                           const lca_bf16 *tok_v, int64_t tok_v_batch_stride, int n_tok,
                           const float *tok_z, int64_t tok_z_batch_stride,
                           const int32_t *tok_pos0, const float *pos_bias, const float *gamma,
                           int apply_rope, const int32_t *first_entry, int n_new,
                           lca_bf16 *cache, int64_t cache_batch_stride, int64_t cache_rows,
                           cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * Sliding-window rows ([P1] "Sliding window attention" branch: the last W uncompressed
 * tokens).  For each of the n_tok tokens of each sequence (position tok_pos0[b] + t),
 * writes RoPE(RMSNorm(v) * gamma, position) in bf16 to the ring row
 * (position mod win_cap) of win_kv[b*win_batch_stride ...].  Width is head_dim.
 * A ring of win_cap >= W rows serves decode; a prefill chunk of T tokens needs
 * win_cap >= T + W - 1 so that no row a query reads is overwritten.
 * ------------------------------------------------------------------------------- */
lca_status lca_window_update(const lca_attn_params *p, int batch,
                             const lca_bf16 *tok_v, int64_t tok_v_batch_stride, int n_tok,
                             const int32_t *tok_pos0, const float *gamma,
                             lca_bf16 *win_kv, int64_t win_batch_stride, int win_cap,
                             cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * Lightning indexer scores ([P1] CSA step two; [P4] 3.1: 64 heads x 128):
 *   s[b][i][j] = sum_h w[b][i][h] * ReLU(q[b][i][h] . k[b][j])   for j < n_vis(i),
 *   n_vis(i) = floor((q_pos[b][i] + 1) / m), entries j >= n_vis(i) set to -inf.
 *   q_idx   [batch][n_q][H_I][d_I] bf16;  w_idx [batch][n_q][H_I] fp32.
 *   k_cache [batch][cache_rows][d_I] bf16 (k_batch_stride between sequences).
 *   q_pos   [batch][n_q] int32 (device).
 *   scores  [batch][n_q][scores_stride] fp32, scores_stride >= cache_rows, multiple of 4.
 * Supported: d_I in {64, 128}, H_I in {16, 32, 64}; (d_I, H_I) = (32, 4) also accepted.
 * ------------------------------------------------------------------------------- */
lca_status csa_indexer_scores(const lca_attn_params *p, int batch, int n_q,
                              const lca_bf16 *q_idx, const float *w_idx,
                              const lca_bf16 *k_cache, int64_t k_batch_stride, int64_t cache_rows,
                              const int32_t *q_pos, float *scores, int64_t scores_stride,
                              cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * Top-k selection ([P1] CSA step two; [P4] 3.1 top-k): for each query, the first
 * min(k, n_vis) entries under (score descending, index ascending), written in ascending
 * index order to out_idx[b][i][0..k), the remainder set to -1.  Scores as produced by
 * csa_indexer_scores (only the first n_vis(i) entries of each row are read).
 * ------------------------------------------------------------------------------- */
lca_status lca_topk(const lca_attn_params *p, int batch, int n_q,
                    const float *scores, int64_t scores_stride, const int32_t *q_pos,
                    int64_t max_entries, int32_t *out_idx, cudaStream_t stream);

/* Indexer scores followed by top-k; the scores go to the workspace. */
size_t csa_indexer_workspace(const lca_attn_params *p, int batch, int n_q, int64_t cache_rows);
lca_status csa_indexer_topk(const lca_attn_params *p, int batch, int n_q,
                            const lca_bf16 *q_idx, const float *w_idx,
                            const lca_bf16 *k_cache, int64_t k_batch_stride, int64_t cache_rows,
                            const int32_t *q_pos, int32_t *out_idx,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * FP8 caches and the per-channel compressor: variants of the path.  The pages name FP8
 * storage only in passing ([P2] ynrysl.com, the paragraph on HCA) and call the compressor's
 * weighting "learned" without its shape ([P1] CSA step one); the readings taken are:
 *
 * e4m3 rows with one fp32 scale per row: the row's largest magnitude maps to 448 (the
 * largest finite e4m3 value),
 *     scale = amax / 448,   code_i = e4m3(x_i / scale),   read back as scale * value(code_i),
 * with IEEE fp32 divisions and round-to-nearest-even, saturating conversions; an all-zero
 * row gets scale 0 and zero codes.  e4m3: 1 sign, 4 exponent (bias 7), 3 mantissa bits,
 * no infinities.
 *
 * lca_quantize_rows_e4m3: rows x [rows][width] bf16 (16-byte aligned; width a multiple of
 * 8, at most 1024) to codes q [rows][width] (8-byte aligned) and scale [rows] fp32.  Caller
 * owns all buffers; no allocation.  Errors: LCA_ERR_INVALID_ARG for NULL or misaligned
 * pointers or a bad width.
 * ------------------------------------------------------------------------------- */
lca_status lca_quantize_rows_e4m3(const lca_bf16 *x, int64_t rows, int width, uint8_t *q, float *scale,
                                  cudaStream_t stream);

/* Options of *_compress_kv_ex (the arguments otherwise as *_compress_kv):
 *   per_channel  0: tok_z [batch][n_tok] and pos_bias [span] as in *_compress_kv.
 *                1: one logit per token and channel, tok_z [batch][n_tok][width] (16-byte
 *                   aligned, tok_z_batch_stride in floats, a multiple of 4), and one offset
 *                   bias per channel, pos_bias [span][width]; the softmax over the window is
 *                   taken per channel (span = 2m for CSA, m' for HCA).
 *   e4m3         0: cache is bf16 as in *_compress_kv.
 *                1: cache holds e4m3 codes (one byte per element, cache_batch_stride and
 *                   rows in elements; 8-byte aligned); the entry is RMS-normalised and
 *                   rotated, rounded to bf16, then quantised as by lca_quantize_rows_e4m3,
 *                   its scale going to cache_scale[b * scale_batch_stride + j]. */
typedef struct lca_compress_variant {
    int per_channel;
    int e4m3;
    float *cache_scale;
    int64_t scale_batch_stride;
} lca_compress_variant;

lca_status csa_compress_kv_ex(const lca_attn_params *p, const lca_compress_variant *variant, int batch, int width,
                              const lca_bf16 *tok_v, int64_t tok_v_batch_stride, int n_tok,
                              const float *tok_z, int64_t tok_z_batch_stride,
                              const int32_t *tok_pos0, const float *pos_bias, const float *gamma,
                              int apply_rope, const int32_t *first_entry, int n_new,
                              void *cache, int64_t cache_batch_stride, int64_t cache_rows,
                              cudaStream_t stream);
lca_status hca_compress_kv_ex(const lca_attn_params *p, const lca_compress_variant *variant, int batch, int width,
                              const lca_bf16 *tok_v, int64_t tok_v_batch_stride, int n_tok,
                              const float *tok_z, int64_t tok_z_batch_stride,
                              const int32_t *tok_pos0, const float *pos_bias, const float *gamma,
                              int apply_rope, const int32_t *first_entry, int n_new,
                              void *cache, int64_t cache_batch_stride, int64_t cache_rows,
                              cudaStream_t stream);

/* The lightning indexer over e4m3 rows: the score of csa_indexer_scores,
 *     s_j = sum_h w_h ReLU(q_h . k_j),
 * with q_h = q_scale[b][i][h] * value(q_idx8[b][i][h][.]) and
 *      k_j = k_scale[b * k_scale_batch_stride + j] * value(k_cache8[b * k_batch_stride + j * d_I + .]).
 * The products run on the tensor cores in e4m3 (kind::f8f6f4, K = 32) with fp32 accumulation;
 * since the scales are non-negative, q_scale is folded into the head weights and k_scale
 * multiplies the head sum.  Supported: d_I = 128 with 64 heads.  Buffers as in the bf16 calls
 * (codes 16-byte aligned), the workspace from csa_indexer_workspace. */
lca_status csa_indexer_scores_e4m3(const lca_attn_params *p, int batch, int n_q,
                                   const uint8_t *q_idx8, const float *q_scale, const float *w_idx,
                                   const uint8_t *k_cache8, int64_t k_batch_stride,
                                   const float *k_scale, int64_t k_scale_batch_stride, int64_t cache_rows,
                                   const int32_t *q_pos, float *scores, int64_t scores_stride,
                                   cudaStream_t stream);
lca_status csa_indexer_topk_e4m3(const lca_attn_params *p, int batch, int n_q,
                                 const uint8_t *q_idx8, const float *q_scale, const float *w_idx,
                                 const uint8_t *k_cache8, int64_t k_batch_stride,
                                 const float *k_scale, int64_t k_scale_batch_stride, int64_t cache_rows,
                                 const int32_t *q_pos, int32_t *out_idx,
                                 void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * Core attention ([P1] CSA step three, HCA dense attention and the tricks; [P4] 3.1).
 * For query i of sequence b at position pos = q_pos[b][i], per head h:
 *   q_h  = RoPE(RMSNorm(q[b][i][h]) * gamma_q, pos)
 *   rows = compressed rows (CSA: kv_cache[idx[b][i][r]] for idx >= 0, r < k;
 *                           HCA: kv_cache[0 .. floor((pos+1)/m')) )
 *          followed by the window rows of tokens max(0,pos-W+1)..pos, read from
 *          win_kv[b][t mod win_cap]; every row is both key and value (MQA);
 *   p_r  = exp(scale q_h.row_r) / (exp(sink[h]) + sum_r' exp(scale q_h.row_r'))
 *   out[b][i][h] = RoPE(sum_r p_r row_r, -pos)   (bf16)
 *   lse[b][i][h] = log(exp(sink[h]) + sum_r exp(scale q_h.row_r))   (fp32, optional)
 * q [batch][n_q][H][c] bf16; gamma_q [c] fp32; sink [H] fp32; out [batch][n_q][H][c] bf16.
 * Rows in the caches already carry RMSNorm and RoPE at their own positions.
 * Supported: c in {128, 256, 512}, H <= 64, W <= 4096.
 * Arithmetic: both products on the tensor cores in fp16 with fp32 accumulation (the rows are
 * re-encoded from bf16, exactly for magnitudes in [2^-14, 65504]; larger ones saturate; the
 * query carries about 22 bits as two fp16 parts), softmax in fp32.  Against an fp64
 * evaluation of the formulas above, max |error| <= 2e-2 x RMS of the output in the tests.
 * The workspace holds split-K partial results; its size comes from *_attend_workspace.
 * ------------------------------------------------------------------------------- */
size_t csa_attend_workspace(const lca_attn_params *p, int batch, int n_q);
size_t hca_attend_workspace(const lca_attn_params *p, int batch, int n_q, int64_t cache_rows);
lca_status csa_attend(const lca_attn_params *p, int batch, int n_q,
                      const lca_bf16 *q, const float *gamma_q, const int32_t *q_pos,
                      const lca_bf16 *kv_cache, int64_t kv_batch_stride, int64_t cache_rows,
                      const int32_t *idx,
                      const lca_bf16 *win_kv, int64_t win_batch_stride, int win_cap,
                      const float *sink, lca_bf16 *out, float *lse,
                      void *workspace, size_t workspace_bytes, cudaStream_t stream);
lca_status hca_attend(const lca_attn_params *p, int batch, int n_q,
                      const lca_bf16 *q, const float *gamma_q, const int32_t *q_pos,
                      const lca_bf16 *kv_cache, int64_t kv_batch_stride, int64_t cache_rows,
                      const lca_bf16 *win_kv, int64_t win_batch_stride, int win_cap,
                      const float *sink, lca_bf16 *out, float *lse,
                      void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* The attention over an e4m3 compressed cache (the FP8 variant; see the e4m3 reading above):
 * compressed row j of sequence b is kv_scale[b * kv_scale_batch_stride + j] *
 * value(kv_cache8[b * kv_batch_stride + j * c + .]) (kv_batch_stride in bytes = elements, a
 * multiple of 16; kv_cache8 16-byte aligned); the window rows stay bf16.  The rows are
 * re-encoded in the kernel as fp16(value) x fp16(scale), rounded to fp16 (about 2^-10 relative,
 * inside the codes' own 2^-4), so the products run as in the bf16 call; against an fp64
 * evaluation over the same decoded rows the error bound of the bf16 call holds.  A row whose
 * 448 x scale exceeds fp16's range, or a NaN code in a row that is read, sets
 * LCA_DEVERR_FP16_RANGE.  Supported: c = 512.  Workspaces from *_attend_workspace; errors as
 * the bf16 calls.  (No prepare/prepared halves for these calls.) */
lca_status csa_attend_e4m3(const lca_attn_params *p, int batch, int n_q,
                           const lca_bf16 *q, const float *gamma_q, const int32_t *q_pos,
                           const uint8_t *kv_cache8, int64_t kv_batch_stride,
                           const float *kv_scale, int64_t kv_scale_batch_stride, int64_t cache_rows,
                           const int32_t *idx,
                           const lca_bf16 *win_kv, int64_t win_batch_stride, int win_cap,
                           const float *sink, lca_bf16 *out, float *lse,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream);
lca_status hca_attend_e4m3(const lca_attn_params *p, int batch, int n_q,
                           const lca_bf16 *q, const float *gamma_q, const int32_t *q_pos,
                           const uint8_t *kv_cache8, int64_t kv_batch_stride,
                           const float *kv_scale, int64_t kv_scale_batch_stride, int64_t cache_rows,
                           const lca_bf16 *win_kv, int64_t win_batch_stride, int win_cap,
                           const float *sink, lca_bf16 *out, float *lse,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* The two halves of an attention call, for callers that overlap the query preparation with
 * other work (the selection, the cache updates) on another stream.  *_attend_prepare runs
 * only the query preparation (RMSNorm + RoPE(i) of q, fp16 hi/lo query images) into the workspace;
 * *_attend_prepared runs only the attention and the combine, reading those images.  Together,
 * with the same arguments and workspace, and the prepare ordered before the attention (same
 * stream, or an event), they compute exactly what *_attend computes.  The prepare reads q,
 * gamma_q and q_pos only; the attention reads the images instead of q and gamma_q. */
lca_status csa_attend_prepare(const lca_attn_params *p, int batch, int n_q,
                              const lca_bf16 *q, const float *gamma_q, const int32_t *q_pos,
                              const lca_bf16 *kv_cache, int64_t kv_batch_stride, int64_t cache_rows,
                              const int32_t *idx,
                              const lca_bf16 *win_kv, int64_t win_batch_stride, int win_cap,
                              const float *sink, lca_bf16 *out, float *lse,
                              void *workspace, size_t workspace_bytes, cudaStream_t stream);
lca_status csa_attend_prepared(const lca_attn_params *p, int batch, int n_q,
                               const lca_bf16 *q, const float *gamma_q, const int32_t *q_pos,
                               const lca_bf16 *kv_cache, int64_t kv_batch_stride, int64_t cache_rows,
                               const int32_t *idx,
                               const lca_bf16 *win_kv, int64_t win_batch_stride, int win_cap,
                               const float *sink, lca_bf16 *out, float *lse,
                               void *workspace, size_t workspace_bytes, cudaStream_t stream);
lca_status hca_attend_prepare(const lca_attn_params *p, int batch, int n_q,
                              const lca_bf16 *q, const float *gamma_q, const int32_t *q_pos,
                              const lca_bf16 *kv_cache, int64_t kv_batch_stride, int64_t cache_rows,
                              const lca_bf16 *win_kv, int64_t win_batch_stride, int win_cap,
                              const float *sink, lca_bf16 *out, float *lse,
                              void *workspace, size_t workspace_bytes, cudaStream_t stream);
lca_status hca_attend_prepared(const lca_attn_params *p, int batch, int n_q,
                               const lca_bf16 *q, const float *gamma_q, const int32_t *q_pos,
                               const lca_bf16 *kv_cache, int64_t kv_batch_stride, int64_t cache_rows,
                               const lca_bf16 *win_kv, int64_t win_batch_stride, int win_cap,
                               const float *sink, lca_bf16 *out, float *lse,
                               void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* hca_attend with no workspace argument and no allocation of any kind: the split-K
 * partials and query images go to a 32 MiB array that the library reserves in device
 * memory when its module loads (every device that loads the library holds it until the
 * process exits).  Same arguments, layout and result as hca_attend, bit for bit.
 * The paper has no counterpart; it serves callers that cannot allocate device memory: a
 * host program without a device allocator of its own, or a serving runtime that fixes its
 * device memory at start-up and may not allocate or free while it serves.
 *  - The array's address is looked up on every call, in the calling thread's current
 *    device and context (a context destroyed and created again, e.g. by cudaDeviceReset,
 *    may place the array elsewhere).  The first call on a device may load the library's
 *    module there: make that first call before capturing the stream into a graph.
 *  - A call whose scratch, hca_attend_workspace(p, batch, n_q, cache_rows), exceeds 32 MiB
 *    returns LCA_ERR_WORKSPACE and launches nothing; use hca_attend.  The size grows with
 *    batch * n_q * splits * H * c * 4 bytes, the split count being about the SM count
 *    divided by batch * n_q: on a 148-SM B300 at c = 512, H = 64, up to 127 queries fit.
 *  - Every call on a device shares the one array: calls that overlap in time on one
 *    device (two streams, two host threads) corrupt each other's results.  Serialise them.
 *  - Nothing in the array needs to start at zero. */
lca_status hca_attend_noalloc(const lca_attn_params *p, int batch, int n_q,
                              const lca_bf16 *q, const float *gamma_q, const int32_t *q_pos,
                              const lca_bf16 *kv_cache, int64_t kv_batch_stride, int64_t cache_rows,
                              const lca_bf16 *win_kv, int64_t win_batch_stride, int win_cap,
                              const float *sink, lca_bf16 *out, float *lse, cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * Grouped output projection ([P1] CSA step four): the H heads of each token are split
 * into `groups` groups of H/groups heads; group g is projected by Wg[g] (d_g rows of
 * (H/groups)*c) to d_g values, the groups' results are concatenated (bf16, in `mid`)
 * and projected by Wm (d_model rows of groups*d_g) to y.
 *   o   [batch][H*c] bf16;  Wg [groups*d_g][(H/groups)*c] bf16;  Wm [d_model][groups*d_g];
 *   mid [batch][groups*d_g] bf16 (caller-owned scratch);  y [batch][d_model] bf16.
 * Supported: batch <= 16, every row length a multiple of 8.
 * Wg and Wm are read from the moment the call's kernels start on the GPU, which may be
 * before kernels issued earlier on the stream have finished (o and mid are read only after
 * them): the weights must not be written by work still pending on the stream.
 * lca_gemm_bf16 is the plain product it is built from: C[M][N] = A[M][K] . B[N][K]^T
 * (fp32 accumulation, bf16 out, B the weight rows).  M <= 16 (decode activations) runs on
 * the CUDA cores, streaming B once; larger M (a prefill chunk's input projections) on the
 * tensor cores in 128 x 64/128/256 tiles.
 * lca_gemm_bf16_f32 is the tensor-core product with fp32 C, any M.  A and B rows are
 * 16-byte aligned with strides (elements) multiples of 8; K a multiple of 8.
 * ------------------------------------------------------------------------------- */
lca_status lca_grouped_oproj(int batch, int heads, int head_dim, int groups, int d_g, int d_model,
                             const lca_bf16 *o, const lca_bf16 *Wg, const lca_bf16 *Wm,
                             lca_bf16 *mid, lca_bf16 *y, cudaStream_t stream);
lca_status lca_gemm_bf16(int M, int N, int K, const lca_bf16 *A, int64_t lda,
                         const lca_bf16 *B, int64_t ldb, lca_bf16 *C, int64_t ldc,
                         cudaStream_t stream);
lca_status lca_gemm_bf16_f32(int M, int N, int K, const lca_bf16 *A, int64_t lda,
                             const lca_bf16 *B, int64_t ldb, float *C, int64_t ldc,
                             cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * Manifold-constrained hyper-connections ([P1] section "mHC", [P4] 3.2): the residual stream
 * is n parallel streams of width d.  Per token, the layer's coefficients are generated from
 * its input, z = flatten(x) . phi^T + bias (an input-dependent linear part and an input-
 * independent bias), read in the order a (n values), c (n values), B (n x n, row-major):
 *   a_i = sigmoid(z_i), c_i = sigmoid(z_{n+i}) (non-negative and bounded),
 *   B = Sinkhorn-Knopp(exp(z_B)): `iters` passes (20 on the page), each normalising the rows
 *       to sum 1 and then the columns, so B is doubly stochastic (columns exactly, rows to
 *       the iteration's convergence).
 * lca_mhc_pre writes the coefficients and the layer input h = sum_i a_i x[i]; after the layer
 * (output y), lca_mhc_post writes the new streams x_out[i] = sum_j B[i][j] x[j] + c_i y.
 *   x, x_out [T][n][d] bf16;  phi [2n + n^2][n d] bf16;  bias [2n + n^2] fp32;
 *   h, y [T][d] bf16;  a, c [T][n] fp32;  b_mix [T][n][n] fp32.
 * Supported: n in {1, 2, 4}, d a multiple of 8 up to 65536, iters in [1, 1000].  Arithmetic in
 * fp32 (z accumulated in fp32 on the tensor cores).  lca_mhc_workspace returns the workspace
 * lca_mhc_pre needs: 0 bytes in this version (z stays in tensor memory); the workspace
 * arguments are accepted for a later version that needs one.
 * ------------------------------------------------------------------------------- */
size_t lca_mhc_workspace(int T, int n);
lca_status lca_mhc_pre(int T, int n, int d, int iters, const lca_bf16 *x, const lca_bf16 *phi,
                       const float *bias, lca_bf16 *h, float *a, float *c, float *b_mix,
                       void *workspace, size_t workspace_bytes, cudaStream_t stream);
lca_status lca_mhc_post(int T, int n, int d, const lca_bf16 *x, const float *b_mix, const float *c,
                        const lca_bf16 *y, lca_bf16 *x_out, cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * Diagnostics.
 * ------------------------------------------------------------------------------- */
const char *lca_status_string(lca_status s);
/* Description of the last failure on the calling thread ("" if none). */
const char *lca_last_error(void);
/* Waits for `stream`, then reads and clears the device error word of the current device
 * into *word (LCA_DEVERR_* bits).  Returns LCA_ERR_TIMEOUT if a timeout bit is set,
 * LCA_ERR_DEVICE for any other bit, LCA_OK when the word is zero. */
lca_status lca_device_error(cudaStream_t stream, uint32_t *word);
/* For tests of the failure path only.  Sets, on the current device, the bound of every wait
 * inside the kernels (SM clock cycles; <= 0 restores the default of 2e9, about a second) and
 * a tile index (per CTA, counted from 0; 1 or later, 0 is rejected) whose rows the attention
 * kernel leaves unloaded (< 0: none), so that the waits on that tile run out: the kernel then stops, frees its
 * tensor memory, and lca_device_error reports LCA_ERR_TIMEOUT.  Affects every later launch
 * on the device until reset with lca_test_hooks(0, -1). */
lca_status lca_test_hooks(long long wait_limit_cycles, int attend_skip_tile);
/* Library version string. */
const char *lca_version(void);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif
#endif /* LCA_H */
