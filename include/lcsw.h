/*
 * lcsw.h -- C ABI of liblcsw.so: the global-retrieval half of a hybrid
 * long-context attention (pooled indexer keys -> indexer scores -> top-k
 * groups -> sparse attention over the selected tokens), for NVIDIA B300
 * (sm_103a).
 *
 * The operation chain is the DSA layer of the GLM-5.3-Flash release
 * ("G2C Brief -- GLM-5.3-Flash", section "DSA keeps selected global access in
 * eleven layers": full token history -> IndexPool -> learned sparse selection
 * (top 2048) -> attention over selected history; config index_kpool 4,
 * index_topk 2048).  IndexPool is described in the reading notes
 * "GLM-5.3-Flash: Hybrid Attention, IndexPool, and Vision-in-the-Loop",
 * section 2, sub-head "IndexPool".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers      Device pointers unless stated otherwise, owned by the caller;
 *               the library allocates and frees nothing.  Scratch space, when
 *               a call needs any, is a caller-provided workspace whose size a
 *               *_workspace_size query returns.
 * Types         lcsw_bf16 is the raw 16-bit pattern of a bfloat16 value.
 *               Weights, scores and lse are IEEE fp32; indices are int32.
 * Layouts       Row-major and contiguous, except that the batch dimension of
 *               per-token caches takes an explicit stride in ELEMENTS (so a
 *               cache may be allocated with more rows than it holds).
 * Alignment     Every bf16 tensor base and batch stride must give 16-byte
 *               aligned rows; fp32/int32 arrays must be 4-byte aligned.
 * Lengths       seq_len[b] (device int32, [B]) is the number of valid tokens
 *               of sequence b.  Group g of sequence b covers tokens
 *               [P*g, P*g+P); only complete groups (g < seq_len[b]/P) exist.
 * Asynchrony    Every call only enqueues work on `stream` and returns; it
 *               never synchronises the host (lcsw_get_status excepted).
 * Errors        Every call returns an lcsw_status; nothing aborts and no C++
 *               exception crosses the ABI.  On a nonzero status,
 *               lcsw_last_error() returns a message (thread-local).  Argument
 *               errors are detected on the host before anything is enqueued.
 *               Device-side failures (a bounded wait that ran out) are
 *               recorded in the workspace's status word and reported by
 *               lcsw_get_status().
 */
#ifndef LCSW_H
#define LCSW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t lcsw_bf16;
/* Same handle as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *lcsw_stream;

typedef enum {
    LCSW_OK = 0,
    LCSW_ERR_INVALID_ARG = 1,  /* null pointer, bad dimension, misalignment      */
    LCSW_ERR_CUDA = 2,         /* a CUDA runtime call or kernel launch failed     */
    LCSW_ERR_UNSUPPORTED = 3,  /* valid but not implemented shape/device          */
    LCSW_ERR_TIMEOUT = 4,      /* a device-side bounded wait ran out              */
    LCSW_ERR_WORKSPACE = 5     /* workspace missing, too small or misaligned      */
} lcsw_status;

/* Message describing the last failing call on this thread ("" if none). */
const char *lcsw_last_error(void);

/* Library version string. */
const char *lcsw_version(void);

/* ---------------------------------------------------------------------------
 * IndexPool (reading notes, section 2 "IndexPool": four indexer key vectors
 * become one by weighted pooling; index_kpool 4).
 *
 *   k_pooled[b][g][:] = bf16( sum_{j<P} pool_w[b][g][j] * k_idx[b][P*g+j][:] )
 *
 * The sum is formed exactly and rounded once to bf16 (nearest, ties to even).
 * Groups g in [g0_b, min(g0_b + g_span, seq_len[b]/P)) are written, where
 * g0_b = g_begin ? g_begin[b] : 0; every other row of k_pooled is untouched.
 *
 *   k_idx     [B][*][d_idx] bf16, batch stride sk_b elements (raw indexer keys)
 *   pool_w    [B][*][P] fp32, batch stride sw_b elements (pooling weights,
 *             used as given: no normalisation is applied)
 *   seq_len   [B] int32 device
 *   g_begin   [B] int32 device, or NULL for 0
 *   k_pooled  [B][*][d_idx] bf16, batch stride sp_b elements (output)
 *   P in {1, 2, 4, 8}; d_idx a multiple of 8; g_span >= 0.
 * ------------------------------------------------------------------------- */
lcsw_status lcsw_pool_keys(const lcsw_bf16 *k_idx, int64_t sk_b,
                           const float *pool_w, int64_t sw_b,
                           const int32_t *seq_len, const int32_t *g_begin,
                           int B, int g_span, int d_idx, int P,
                           lcsw_bf16 *k_pooled, int64_t sp_b, lcsw_stream stream);

/* ---------------------------------------------------------------------------
 * Indexer scores (reading notes, section 2: a lightweight indexer picks the
 * relevant slices; DSA-indexer form).
 *
 *   scores[b][t][g] = sum_h w_head[b][t][h] * max(0, q_idx[b][t][h][:] . k_pooled[b][g][:])
 *
 * for visible groups, -inf for the others (g < G_max).  Group g is visible to
 * query t of sequence b iff g < seq_len[b]/P and, when q_pos is given,
 * P*g + P - 1 <= q_pos[b][t] (causal at group granularity).  A score of -0 is
 * written as +0.  Products bf16 x bf16 are exact; sums are fp32 (tensor-core
 * accumulation), so results agree with an exact evaluation to about 1e-6
 * relative.
 *
 *   q_idx     [B][T][H_i][d_idx] bf16      w_head [B][T][H_i] fp32
 *   k_pooled  [B][*][d_idx] bf16, batch stride sp_b elements
 *   q_pos     [B][T] int32 device or NULL (decode: all complete groups visible)
 *   scores    [B][T][G_max] fp32 (output)
 *   d_idx == 64; 1 <= H_i <= 16; P in {1, 2, 4, 8}.
 * Query blocks of T >= 64 run as a tcgen05 GEMM fed by TMA when sp_b >=
 * 64 * G_max (it reads whole 128-group tiles up to G_max rows of every
 * sequence, so those rows must exist); otherwise the mma.sync kernel runs.
 * ------------------------------------------------------------------------- */
lcsw_status lcsw_index_scores(const lcsw_bf16 *q_idx, const float *w_head,
                              const lcsw_bf16 *k_pooled, int64_t sp_b,
                              const int32_t *seq_len, const int32_t *q_pos,
                              int B, int T, int H_i, int d_idx, int P, int G_max,
                              float *scores, lcsw_stream stream);

/* Visible group counts n_valid[b][t] (seq_len[b]/P, capped causally by q_pos
 * as above); the per-row valid prefix that lcsw_topk_groups takes. */
lcsw_status lcsw_visible_counts(const int32_t *seq_len, const int32_t *q_pos,
                                int B, int T, int P, int32_t *n_valid, lcsw_stream stream);

/* ---------------------------------------------------------------------------
 * Top-k groups ("learned sparse selection (top 2048)", index_topk 2048 read as
 * 512 groups of P = 4 tokens).
 *
 * For each row r: among groups [0, n_valid[r]) take the min(k, n_valid[r])
 * of largest score; equal scores (-0 equals +0) go to the lower index.  The
 * chosen indices are written in ascending order to idx[r][0..), and the
 * remaining entries are -1.  Scores must not be NaN.
 *
 *   scores [rows][G_max] fp32      n_valid [rows] int32 device
 *   idx    [rows][k] int32 (output)
 *   ws     device workspace of lcsw_topk_workspace_size(rows, G_max, k) bytes,
 *          256-byte aligned, no clearing needed (may be NULL when that size is
 *          0).  The size is nonzero for a few long rows (rows <= 32 and
 *          16384 <= G_max <= 524288), which are then spread over many blocks
 *          (a memset and three launches); with no or a smaller workspace those
 *          rows take one block each, with the same result.
 * ------------------------------------------------------------------------- */
size_t lcsw_topk_workspace_size(int64_t rows, int G_max, int k);
lcsw_status lcsw_topk_groups(const float *scores, const int32_t *n_valid,
                             int64_t rows, int G_max, int k, int32_t *idx,
                             void *ws, size_t ws_bytes, lcsw_stream stream);

/* ---------------------------------------------------------------------------
 * Sparse attention over the selected history ("attention over selected
 * history"; one shared K/V head serves every query head).
 *
 * For row (b, t) the token set is {P*g + i : g in idx[b][t][:], 0 <= g <
 * seq_len[b]/P, 0 <= i < P}; entries outside that range (e.g. -1 padding)
 * are skipped.  For each query head h:
 *   z_j = scale * q[b][t][h][:] . K[b][j][:],  p = softmax(z),
 *   out[b][t][h][:] = bf16( sum_j p_j V[b][j][:] ),
 *   lse[b][t][h] = ln sum_j exp(z_j).
 * An empty token set gives out = 0 and lse = -inf.  The token set is split
 * across thread blocks (split-K) and the partial softmax states are merged.
 *
 *   q    [B][T][H_q][d_qk] bf16
 *   K    [B][*][d_qk] bf16 (batch stride sK_b elements); V [B][*][d_v] (sV_b)
 *   idx  [B][T][k] int32 device
 *   out  [B][T][H_q][d_v] bf16 (output); lse [B][T][H_q] fp32 or NULL
 *   ws   device workspace of lcsw_sparse_attn_workspace_size(...) bytes
 *   H_q a multiple of 16, at most 128; d_qk in {64, 128, 192, 256};
 *   d_v in {64, 128}.
 * ------------------------------------------------------------------------- */
size_t lcsw_sparse_attn_workspace_size(int B, int T, int H_q, int d_v, int k, int P);
lcsw_status lcsw_sparse_attn(const lcsw_bf16 *q, const lcsw_bf16 *K, int64_t sK_b,
                             const lcsw_bf16 *V, int64_t sV_b, const int32_t *seq_len,
                             const int32_t *idx, int B, int T, int H_q, int d_qk, int d_v,
                             int P, int k, float scale, lcsw_bf16 *out, float *lse,
                             void *ws, size_t ws_bytes, lcsw_stream stream);

/* ---------------------------------------------------------------------------
 * FP8 (E4M3) K/V cache.  The serving stack of the reading notes quantizes
 * caches per tier to INT8, FP8 or BF16 ("The serving stack"); this is the FP8
 * tier for the attention cache, in the pooled keys' format: one fp32 scale
 * per token row (amax / 448), codes rounded exactly to nearest, ties to even.
 *
 * lcsw_quantize_rows_e4m3: rows [r0_b, r0_b + n_rows) of every sequence
 * (r0_b = row_begin[b], or 0 when row_begin is NULL) of a bf16 cache
 * x [B][*][width] (batch stride sx_b elements) -> codes [B][*][width] uint8
 * (batch stride sc_b bytes, a multiple of 16) and scales [B][*] fp32 (batch
 * stride ss_b elements).  width a multiple of 16.  Rows of other positions are
 * untouched, so a decode step quantizes just the newest token's row.
 *
 * lcsw_sparse_attn_kv8: lcsw_sparse_attn over such a cache,
 *
 *   z_j = scale * ks[b][j] * sum_i q_i e4m3(kc[b][j][i]),
 *   out = sum_j softmax_j(z) * vs[b][j] * e4m3(vc[b][j][:])
 *
 * with the same selection, masking and output rules; kc, vc 16-byte aligned
 * with strides (bytes) multiples of 16; ks, vs strides in elements.  The
 * workspace is lcsw_sparse_attn_kv8_workspace_size bytes, 16-byte aligned.
 * ------------------------------------------------------------------------- */
lcsw_status lcsw_quantize_rows_e4m3(const lcsw_bf16 *x, int64_t sx_b, const int32_t *row_begin,
                                    int B, int n_rows, int width, uint8_t *codes, int64_t sc_b,
                                    float *scales, int64_t ss_b, lcsw_stream stream);
size_t lcsw_sparse_attn_kv8_workspace_size(int B, int T, int H_q, int d_v, int k, int P);
lcsw_status lcsw_sparse_attn_kv8(const lcsw_bf16 *q, const uint8_t *kc, int64_t skc_b,
                                 const float *ks, int64_t sks_b, const uint8_t *vc,
                                 int64_t svc_b, const float *vs, int64_t svs_b,
                                 const int32_t *seq_len, const int32_t *idx, int B, int T,
                                 int H_q, int d_qk, int d_v, int P, int k, float scale,
                                 lcsw_bf16 *out, float *lse, void *ws, size_t ws_bytes,
                                 lcsw_stream stream);

/* ---------------------------------------------------------------------------
 * INT8 K/V cache: the INT8 tier of the same serving stack ("The serving
 * stack"; no format given).  Reading: symmetric codes in [-127, 127], one
 * fp32 scale per token row = amax / 127 (0 for an all-zero row, whose codes
 * are 0), code_i = the integer nearest to x_i / scale, ties to the even
 * integer; the rounding is exact.  Rows must be finite (a row holding an
 * infinity or a NaN gets unspecified codes).
 *
 * lcsw_quantize_rows_i8: as lcsw_quantize_rows_e4m3 (same row window, layout,
 * strides and alignment), int8 codes.
 *
 * lcsw_sparse_attn_kvi8: as lcsw_sparse_attn_kv8 with element values
 * kc[b][j][i] * ks[b][j] and vc[b][j][i] * vs[b][j]; the workspace is
 * lcsw_sparse_attn_kv8_workspace_size bytes, 16-byte aligned.
 * ------------------------------------------------------------------------- */
lcsw_status lcsw_quantize_rows_i8(const lcsw_bf16 *x, int64_t sx_b, const int32_t *row_begin,
                                  int B, int n_rows, int width, int8_t *codes, int64_t sc_b,
                                  float *scales, int64_t ss_b, lcsw_stream stream);
lcsw_status lcsw_sparse_attn_kvi8(const lcsw_bf16 *q, const int8_t *kc, int64_t skc_b,
                                  const float *ks, int64_t sks_b, const int8_t *vc,
                                  int64_t svc_b, const float *vs, int64_t svs_b,
                                  const int32_t *seq_len, const int32_t *idx, int B, int T,
                                  int H_q, int d_qk, int d_v, int P, int k, float scale,
                                  lcsw_bf16 *out, float *lse, void *ws, size_t ws_bytes,
                                  lcsw_stream stream);

/* ---------------------------------------------------------------------------
 * Sparse attention in the MLA latent geometry ("G2C Brief -- GLM-5.3-Flash":
 * MLA rank 512 per token, kv_lora_rank 512; the DSA diagram's "MLA latent
 * cache (rank 512 per token)").  One cached row per token, shared by every
 * query head, holds the rank-512 latent c and a rotary key part (64 wide; the
 * pages do not give that width): kv[b][j] = [c_j (512) | r_j (64)].  The
 * latent is both the key's first 512 dims and the value (the query is
 * absorbed into the latent space):
 *
 *   z_j = scale * q[b][t][h][:] . kv[b][j][:]                 (576 dims)
 *   out[b][t][h][:] = sum_j softmax_j(z) kv[b][j][0:512],  lse = log sum_j e^z_j
 *
 * over the tokens of groups idx[b][t][0..k) (entries outside [0, seq_len/P)
 * are skipped, as in lcsw_sparse_attn).
 *
 *   q    [B][T][H_q][576] bf16;  kv [B][*][576] bf16, batch stride skv_b
 *   idx  [B][T][k] int32;  out [B][T][H_q][512] bf16;  lse [B][T][H_q] or NULL
 *   ws   lcsw_sparse_attn_mla_workspace_size bytes (0: none needed), 16-byte
 *        aligned, no clearing needed
 * H_q a multiple of 16, B*T <= 65535.  lcsw_decode_fused and
 * lcsw_decode_reuse take the same geometry when d_qk = LCSW_MLA_DQK and
 * d_v = LCSW_MLA_DV, with V = NULL (or V = K, sV_b = sK_b).
 * ------------------------------------------------------------------------- */
#define LCSW_MLA_DQK 576
#define LCSW_MLA_DV 512
size_t lcsw_sparse_attn_mla_workspace_size(int B, int T, int H_q, int k, int P);
lcsw_status lcsw_sparse_attn_mla(const lcsw_bf16 *q, const lcsw_bf16 *kv, int64_t skv_b,
                                 const int32_t *seq_len, const int32_t *idx, int B, int T,
                                 int H_q, int P, int k, float scale, lcsw_bf16 *out, float *lse,
                                 void *ws, size_t ws_bytes, lcsw_stream stream);

/* ---------------------------------------------------------------------------
 * lcsw_sparse_attn without a caller workspace.  The pages have no counterpart
 * of this entry point: it serves callers that cannot allocate device memory
 * per call -- a plain-C host over this header with no device allocator of its
 * own, or a runtime whose device memory is budgeted up front -- and callers
 * that must not let a cudaMalloc/cudaFree synchronise the device mid-step.
 *
 * Arguments, results and errors are those of lcsw_sparse_attn, minus ws and
 * ws_bytes.  The split-K partial states go to a fixed scratch array of
 * LCSW_NOALLOC_SCRATCH_BYTES in the library's device memory, one per device.
 *   - Allocates nothing: no cudaMalloc/cudaFree and no allocating library call.
 *   - A shape whose lcsw_sparse_attn_workspace_size(...) exceeds
 *     LCSW_NOALLOC_SCRATCH_BYTES is rejected with LCSW_ERR_UNSUPPORTED (the
 *     message gives both sizes) before any device work.
 *   - Set-up: the first call on each device, with that device current, looks
 *     up the array's address (cudaGetSymbolAddress; a failure returns
 *     LCSW_ERR_CUDA).  That first call must come before any stream capture.
 *   - Nothing in the scratch has to start at zero: a call writes every partial
 *     state it reads.
 *   - One scratch per device: calls that overlap in time on the same device
 *     (two streams, or two host threads) race on it and give wrong results.
 *     Order them (one stream, or an event between them).
 * ------------------------------------------------------------------------- */
#define LCSW_NOALLOC_SCRATCH_BYTES (8u << 20) /* 8 MiB */
lcsw_status lcsw_sparse_attn_noalloc(const lcsw_bf16 *q, const lcsw_bf16 *K, int64_t sK_b,
                                     const lcsw_bf16 *V, int64_t sV_b, const int32_t *seq_len,
                                     const int32_t *idx, int B, int T, int H_q, int d_qk,
                                     int d_v, int P, int k, float scale, lcsw_bf16 *out,
                                     float *lse, lcsw_stream stream);

/* ---------------------------------------------------------------------------
 * Append of a decode step's new token.  The newest token of every sequence
 * (position seq_len[b] - 1, after the length has grown) is written into the
 * raw indexer-key cache, the K cache and the V cache from one packed staging
 * row per sequence, in one launch:
 *
 *   rows [B][*] bf16, batch stride s_rows elements:
 *        [k_idx row (d_idx) | K row (d_qk) | V row (d_v)]
 *   k_idx [B][*][d_idx], K [B][*][d_qk], V [B][*][d_v] bf16, batch strides in
 *        elements; V = NULL with d_v = 0 for the MLA geometry (the value is
 *        the latent part of K)
 *
 * Sequences with seq_len[b] <= 0 are skipped; nothing else is written.  The
 * decode step (lcsw_decode_fused with k_idx) then pools the group the new row
 * completes (IndexPool keeps its state per token: reading notes, section 2,
 * sub-head "IndexPool").  d_idx, d_qk, d_v multiples of 8; rows, caches and
 * strides 16-byte aligned.
 * ------------------------------------------------------------------------- */
lcsw_status lcsw_append_token(const lcsw_bf16 *rows, int64_t s_rows, const int32_t *seq_len,
                              int B, lcsw_bf16 *k_idx, int64_t sk_b, int d_idx, lcsw_bf16 *K,
                              int64_t sK_b, int d_qk, lcsw_bf16 *V, int64_t sV_b, int d_v,
                              lcsw_stream stream);

/* ---------------------------------------------------------------------------
 * One decode step of the whole retrieval path (one query token per sequence):
 * [append] -> scores -> top-k -> sparse attention, as one persistent kernel.
 *
 * Append: when k_idx is not NULL and seq_len[b] is a multiple of P, the group
 * that the newest token completes (g = seq_len[b]/P - 1) is pooled from
 * k_idx/pool_w into k_pooled before it is scored (same arithmetic as
 * lcsw_pool_keys).  Then every complete group is scored, the top k groups are
 * selected (rules of lcsw_topk_groups) and the query heads attend over their
 * tokens (rules of lcsw_sparse_attn).
 *
 * The workspace must be zero-filled once before its first use; the call
 * leaves it ready for the next call.  After LCSW_ERR_TIMEOUT from
 * lcsw_get_status it must be zero-filled again, and so before it serves
 * arguments of another shape (B, G_max, k, H_q, d_v): it carries state from
 * one call to the next.  Calls that share a workspace must not overlap on the
 * device.
 * ------------------------------------------------------------------------- */
typedef struct {
    const lcsw_bf16 *q_idx;    /* [B][H_i][d_idx]                              */
    const float *w_head;       /* [B][H_i]                                     */
    lcsw_bf16 *k_pooled;       /* [B][G_max][d_idx], batch stride sp_b; in/out:
                                  rows 0..G_max-1 of every sequence readable (the
                                  first copies go out before the lengths arrive) */
    int64_t sp_b;
    const lcsw_bf16 *k_idx;    /* [B][*][d_idx] raw keys (stride sk_b) or NULL */
    int64_t sk_b;
    const float *pool_w;       /* [B][*][P] (stride sw_b); needed with k_idx   */
    int64_t sw_b;
    const lcsw_bf16 *q;        /* [B][H_q][d_qk]                               */
    const lcsw_bf16 *K;        /* [B][*][d_qk], batch stride sK_b              */
    int64_t sK_b;
    const lcsw_bf16 *V;        /* [B][*][d_v], batch stride sV_b               */
    int64_t sV_b;
    const int32_t *seq_len;    /* [B]                                          */
    int B, G_max, H_i, d_idx, P, k, H_q, d_qk, d_v;
    float scale;
    lcsw_bf16 *out;            /* [B][H_q][d_v] output                         */
    float *lse;                /* [B][H_q] output or NULL                      */
    int32_t *idx_out;          /* [B][k] selected groups (ascending) or NULL   */
    float *scores_out;         /* [B][G_max] indexer scores or NULL            */
    int flags;                 /* 0, or LCSW_DECODE_* bits below (testing)     */
} lcsw_decode_args;

/* lcsw_decode_args.flags: alternative internal paths with identical results,
 * for tests.  FORCE_MULTIPASS_SELECT makes the persistent kernel take its
 * exact multi-pass selection (used when candidates overflow shared memory);
 * FORCE_MULTIKERNEL runs the step as separate kernels (score, top-k, attend). */
#define LCSW_DECODE_FORCE_MULTIPASS_SELECT 1
#define LCSW_DECODE_FORCE_MULTIKERNEL 2
/* Failure-detection test: the last block of each sequence returns before the
 * first cross-block barrier, so the others' bounded waits run out; the call
 * then reports LCSW_ERR_TIMEOUT through lcsw_get_status (workspace must be
 * zero-filled again afterwards). */
#define LCSW_DECODE_TEST_SKIP_ARRIVE 4

size_t lcsw_decode_workspace_size(const lcsw_decode_args *a);
/* Number of kernel launches one lcsw_decode_fused call with these arguments
 * enqueues (0 if the arguments are invalid). */
int lcsw_decode_launches(const lcsw_decode_args *a);
lcsw_status lcsw_decode_fused(const lcsw_decode_args *a, void *ws, size_t ws_bytes,
                              lcsw_stream stream);

/* ---------------------------------------------------------------------------
 * FP8 pooled indexer keys.  The serving stack of the reading notes (section
 * "The serving stack") quantizes caches per tier to INT8, FP8 or BF16 and
 * gives no format; the reading here: OCP E4M3 codes with one fp32 scale per
 * 64-value row,
 *
 *   scale = amax_i |x_i| / 448 (fp32),   code_i = nearest E4M3 of x_i / scale
 *
 * (ties to the even code, saturating at +-448; every code 0 when scale is 0).
 * The rounding is exact: the code is the nearest to the exact quotient.
 *
 * Cache layout kq, per sequence b (base kq + b * sq_b bytes): tiles of 16
 * groups, LCSW_E4M3_TILE_BYTES each -- 16 rows of 64 codes, then the 16 rows'
 * fp32 scales.  Group g: codes at tile g/16, byte (g%16)*64; scale at byte
 * 1024 + (g%16)*4 of the tile.  sq_b is a multiple of 16 and holds at least
 * ceil(G_max/16) tiles (the decode step reads whole tiles).
 *
 * lcsw_quantize_keys_e4m3 quantizes groups [0, n_groups) of every sequence's
 * bf16 pooled keys (k_pooled [B][*][64], batch stride sp_b elements).
 * ------------------------------------------------------------------------- */
#define LCSW_E4M3_TILE_BYTES 1088
lcsw_status lcsw_quantize_keys_e4m3(const lcsw_bf16 *k_pooled, int64_t sp_b, int B,
                                    int n_groups, uint8_t *kq, int64_t sq_b,
                                    lcsw_stream stream);

/* One decode step (as lcsw_decode_fused) whose indexer reads the FP8 cache kq
 * instead of bf16 pooled keys.  The indexer query q_idx (bf16) is quantized
 * per head in the same way inside the step, and
 *
 *   s[b][g] = sum_h w_head[b][h] * max(0, scale_q,h * scale_k,g * sum_i q_i k_i)
 *
 * over the codes' values; the selection and attention follow as in
 * lcsw_decode_fused.  Append: with k_idx and pool_w, the group the newest token
 * completes is pooled exactly (bf16, as lcsw_pool_keys) and quantized into kq
 * before it is scored; k_pooled is not read or written (it may be NULL).
 * Shapes outside the persistent kernel's envelope (lcsw_decode_launches(a)
 * != 1) return LCSW_ERR_UNSUPPORTED.  Workspace: lcsw_decode_workspace_size.
 * ------------------------------------------------------------------------- */
lcsw_status lcsw_decode_fused_e4m3(const lcsw_decode_args *a, uint8_t *kq, int64_t sq_b,
                                   void *ws, size_t ws_bytes, lcsw_stream stream);

/* ---------------------------------------------------------------------------
 * Cross-layer reuse of a selection (reading notes "GLM-5.3-Flash: Hybrid
 * Attention, IndexPool, and Vision-in-the-Loop", section 2, sub-head
 * "IndexPool": the cross-layer variant of the pooled-index idea is called
 * IndexCache; the pages say nothing more).  Reading: a later DSA layer of the
 * same decode step runs no indexer scores and no top-k of its own; it attends
 * over the groups an earlier layer selected, e.g. the idx_out of that layer's
 * lcsw_decode_fused call.
 *
 *   out[b][h][:], lse[b][h] = lcsw_sparse_attn of q over the groups
 *   idx_in[b][0..k) of K/V (entries outside [0, seq_len[b]/P), such as -1
 *   padding, are skipped; an empty set gives out = 0, lse = -inf).
 *
 * Reads q, K, sK_b, V, sV_b, seq_len, B, H_q, d_qk, d_v, P, k, scale, out and
 * lse of `a`; its indexer fields (q_idx, w_head, k_pooled, k_idx, pool_w,
 * H_i, d_idx), idx_out and scores_out are not used; G_max and flags are
 * read as below.
 *   idx_in  [B][k] int32 device
 *   ws      a decode workspace: lcsw_decode_workspace_size(a) bytes, 256-byte
 *           aligned, zero-filled before its first use like the workspace of
 *           lcsw_decode_fused (and left ready for the next call).  a->G_max
 *           only sizes it and may be 0.  It may be the workspace of the
 *           selecting layer's lcsw_decode_fused call (any G_max, H_q, d_v of
 *           that call), once that call has completed on the same stream.
 * Within the persistent kernel's envelope (2B <= SM count, k <= 2048, H_q a
 * multiple of 16 up to 64, and flags without LCSW_DECODE_FORCE_MULTIKERNEL):
 * one launch, whose blocks attend over slices of idx_in[b] and merge their
 * partial states; a bounded wait that runs out is reported through
 * lcsw_get_status.  Otherwise two launches: split-K partial states, then
 * their merge.
 * ------------------------------------------------------------------------- */
lcsw_status lcsw_decode_reuse(const lcsw_decode_args *a, const int32_t *idx_in, void *ws,
                              size_t ws_bytes, lcsw_stream stream);

/* ---------------------------------------------------------------------------
 * Chunked prefill: T new query tokens per sequence, the last T tokens of the
 * cache (positions seq_len[b]-T .. seq_len[b]-1), causal at group
 * granularity.  Pools the groups the chunk completes (from the group holding
 * token seq_len[b]-T onwards), scores every visible group for every query
 * with a tensor-core GEMM, selects the top k per query and attends.
 *
 * With H_i <= 8, T >= 64 and G_max <= 524288, the selection is fused with the
 * scoring: a sample of the groups sets each query's threshold, the GEMM keeps
 * only the groups at or above it, and the exact top k is taken from those.  A
 * query whose kept groups cannot be shown to hold its top k (too few, or more
 * than the per-row capacity) falls back to dense scores and the radix top-k,
 * decided on the device: the result is the same exact top k either way.
 * With at least 256 query rows (B*T), H_q <= 32 and d_qk = d_v = 128, the
 * attention runs on the tensor cores: a persistent kernel takes one query row
 * at a time per SM, without splitting its selected tokens.  Other shapes use
 * the split-K kernel of lcsw_sparse_attn.  Both give the same result within
 * the attention tolerance.
 * flags: LCSW_PREFILL_FORCE_FALLBACK sends every query through the fallback
 * (a test of that path).
 *
 * Workspace: lcsw_prefill_workspace_size(a) bytes, 256-byte aligned.  Its
 * first 256 bytes (the status word) must be zero before the first call;
 * lcsw_get_status clears the word, and no other region needs clearing (each
 * is written before it is read).  Calls sharing a workspace must not overlap.
 * ------------------------------------------------------------------------- */
#define LCSW_PREFILL_FORCE_FALLBACK 1
/* Failure-detection test: in the tensor-core attention (>= 256 query rows,
 * H_q <= 32, d_qk = d_v = 128) the first key chunk of every CTA is copied but
 * never handed over, so the MMA warp's bounded wait (about a second) runs out
 * and every role stops; the call reports LCSW_ERR_TIMEOUT through
 * lcsw_get_status and its output is not valid.  The context stays usable. */
#define LCSW_PREFILL_TEST_SKIP_GATHER 2
typedef struct {
    const lcsw_bf16 *q_idx;    /* [B][T][H_i][d_idx]                           */
    const float *w_head;       /* [B][T][H_i]                                  */
    lcsw_bf16 *k_pooled;       /* [B][*][d_idx] (stride sp_b); in/out          */
    int64_t sp_b;
    const lcsw_bf16 *k_idx;    /* [B][*][d_idx] raw keys (stride sk_b)         */
    int64_t sk_b;
    const float *pool_w;       /* [B][*][P] (stride sw_b)                      */
    int64_t sw_b;
    const lcsw_bf16 *q;        /* [B][T][H_q][d_qk]                            */
    const lcsw_bf16 *K;        /* [B][*][d_qk] (stride sK_b)                   */
    int64_t sK_b;
    const lcsw_bf16 *V;        /* [B][*][d_v] (stride sV_b)                    */
    int64_t sV_b;
    const int32_t *seq_len;    /* [B] tokens including the new chunk           */
    int B, T, G_max, H_i, d_idx, P, k, H_q, d_qk, d_v;
    float scale;
    lcsw_bf16 *out;            /* [B][T][H_q][d_v]                             */
    float *lse;                /* [B][T][H_q] or NULL                          */
    int32_t *idx_out;          /* [B][T][k] or NULL                            */
    int flags;                 /* LCSW_PREFILL_* bits, normally 0              */
} lcsw_prefill_args;

size_t lcsw_prefill_workspace_size(const lcsw_prefill_args *a);
lcsw_status lcsw_prefill(const lcsw_prefill_args *a, void *ws, size_t ws_bytes,
                         lcsw_stream stream);

/* ---------------------------------------------------------------------------
 * KDA step: the linear-attention half of the hybrid ("G2C Brief --
 * GLM-5.3-Flash", section "KDA carries fixed state through most layers":
 * Kimi Delta Attention is a gated delta-rule descendant of linear attention
 * that updates a fixed matrix state per head; a short convolution of kernel
 * size 4 and learned gates surround the recurrence; 64 heads of width 128).
 * The pages print no formula; the step computes, per sequence b, head h and
 * token t in order (S: the D x D state, key channels as rows):
 *
 *   a_c = SiLU(sum_{j<4} conv_w[c][j] * x_{t-3+j}[c])  for the head's q, k, v channels
 *         (x_{t'} = qkv[b][t'] for t' >= 0, conv_state[b][3+t'] for t' < 0)
 *   q   = a_q / sqrt(|a_q|^2 + 1e-6) / sqrt(D),   k = a_k / sqrt(|a_k|^2 + 1e-6),   v = a_v
 *   S   = (I - beta k k^T) Diag(exp(g)) S + beta k v^T,    out = S^T q
 *
 * with g = g[b][t][h][:] and beta = beta[b][t][h].  After the call state
 * holds S after the last token and conv_state the raw inputs of the last
 * three positions (oldest first).
 *
 *   qkv        [B][T][3*H*D] bf16: pre-convolution projections, q | k | v,
 *              each head-major (channel c of part p, head h: p*H*D + h*D + c)
 *   conv_w     [3*H*D][4] bf16: depthwise taps, tap 3 on the current token
 *   conv_state [B][3][3*H*D] bf16, read and written
 *   g          [B][T][H][D] fp32: log of the per-key-channel decay (<= 0)
 *   beta       [B][T][H] fp32: write strength
 *   state      [B][H][D][D] fp32, read and written; 16-byte aligned
 *   out        [B][T][H][D] bf16
 *
 * D must be 128 (LCSW_ERR_UNSUPPORTED otherwise); B = 0 or T = 0 is a no-op.
 * The output, gates and projections around the step (dense layers of the
 * model) are the caller's.  Work: one block per (head, sequence); the state
 * is read once and written once per call whatever T is.
 * ------------------------------------------------------------------------- */
lcsw_status lcsw_kda_step(const lcsw_bf16 *qkv, const lcsw_bf16 *conv_w, lcsw_bf16 *conv_state,
                          const float *g, const float *beta, float *state, lcsw_bf16 *out,
                          int B, int T, int H, int D, lcsw_stream stream);

/* ---------------------------------------------------------------------------
 * Device status word of a workspace (decode / prefill).  Synchronises
 * `stream`, then returns LCSW_OK, or LCSW_ERR_TIMEOUT if a bounded device
 * wait ran out during an earlier call on that workspace.  Clears the word.
 * ------------------------------------------------------------------------- */
lcsw_status lcsw_get_status(void *ws, lcsw_stream stream);

/* ---------------------------------------------------------------------------
 * Device-side bounds checks.  A library built with -DLCSW_CHECKS=1 checks the
 * data-dependent indices of its kernels (positions derived from candidate
 * counts, selections and lengths) against their extents; a failed check
 * records a nonzero code and skips the access (no trap, the context stays
 * usable).  lcsw_check_status synchronises the device and returns the first
 * code recorded since the last call (0: none; -1: the device could not be
 * read), clearing them.  lcsw_checks_enabled tells which build this is; in a
 * normal build lcsw_check_status always returns 0.
 * ------------------------------------------------------------------------- */
int lcsw_checks_enabled(void);
int lcsw_check_status(void);

#ifdef __cplusplus
}
#endif

#endif /* LCSW_H */
