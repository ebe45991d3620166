/*
 * si.h -- C ABI of libsi: indexer-driven Top-K sparse attention on GB300.
 *
 * The operation follows the page "Day0 Inference Support and Performance
 * Optimization for New Architecture LLMs" (Baidu Cloud):
 *   section 2.2  -- a lightweight indexer scores each query against all earlier
 *                   positions, the per-head scores are aggregated with head
 *                   weights, the Top-K positions are kept, and the sparse
 *                   attention core reads only the KV rows at those positions;
 *   section 4.1  -- scoring, head weighting and Top-K form one fused operator
 *                   that reads the paged K-cache directly and never stores the
 *                   full score matrix;
 *   section 4.2  -- the attention core gathers the selected rows from the main
 *                   KV cache by the position list the indexer produced.
 * The score of query row t against key position s is
 *   score(t,s) = k_scale[s] * sum_h w[t,h] * ReLU(q_idx[t,h,:] . k_idx[s,:])
 * (k_scale is the per-token FP8 dequantisation scale; it is positive, so
 * applying it after the ReLU equals scoring the dequantised key).
 *
 * Conventions for every entry point
 *   * All pointers named "device" are CUDA device pointers owned by the
 *     caller; the library never allocates, frees or retains them.
 *   * Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  A call that returns SI_OK has only enqueued work.
 *   * Host-side argument errors return a non-zero status before anything is
 *     launched.  A failed launch returns SI_ERR_CUDA.  si_last_error() gives
 *     a human-readable detail for the calling thread.
 *   * Device-side problems (a block-table entry or a selected index out of
 *     range, a bounded wait that gave up) never fault: the offending access is
 *     skipped and a bit is OR-ed into the sticky status word that lives in the
 *     first 16 bytes of the workspace.  Zero the workspace once after
 *     allocating it; read the word with si_workspace_status().
 *   * Apart from a diagnostic launch counter the library holds no global
 *     mutable state; calls from several host threads are safe as long as
 *     they use different workspaces.
 *
 * Paged caches: logical position s of sequence q is physical row
 *   block_table[q * max_blocks + s / page_size] * page_size + s % page_size
 * of a cache laid out [n_blocks, page_size, row_stride] (section 4.1's paged
 * K-cache).  The indexer-key cache and the KV cache share the block table.
 */
#ifndef SI_H_
#define SI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SI_VERSION 5

typedef enum si_status {
    SI_OK = 0,
    SI_ERR_INVALID_ARG = 1, /* null pointer, bad size or inconsistent shapes */
    SI_ERR_UNSUPPORTED = 2, /* valid request this build does not implement */
    SI_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or too small */
    SI_ERR_CUDA = 4,        /* a CUDA call or launch failed */
    SI_ERR_DEVICE = 5       /* si_workspace_status found device-side flags */
} si_status;

typedef enum si_dtype {
    SI_F32 = 0,  /* IEEE float32 */
    SI_BF16 = 1, /* bfloat16 */
    SI_E4M3 = 2, /* OCP FP8 e4m3 (finite, max 448) */
    SI_E2M1 = 3, /* OCP FP4 e2m1 (max 6), two per byte, even element in the low
                    nibble; attention caches only, with per-tile scales (the
                    NVFP4 KV format of the vLLM article on DeepSeek-V4.1 uses
                    blocks of 16 entries) */
    SI_MXE4M3 = 4 /* MXFP8 (OCP Microscaling v1.0), section 5.1's indexer
                     format: e4m3 codes in groups of 32 consecutive entries of
                     a row, each group with one E8M0 scale byte e meaning
                     2^(e - 127) (e = 255, NaN, is not allowed); entry =
                     2^(e - 127) * code.  Indexer query and keys only. */
} si_dtype;

/* Device status flags (sticky, OR-ed into the workspace status word). */
#define SI_DEVFLAG_BAD_BLOCK 0x1u /* block-table entry outside [0, n_blocks) */
#define SI_DEVFLAG_BAD_INDEX 0x2u /* selected index outside [0, pos] (not -1) */
#define SI_DEVFLAG_TIMEOUT 0x4u   /* a bounded on-chip wait gave up */
#define SI_DEVFLAG_RANGE 0x8u     /* a value met an f16 operand outside its range
                                     (|x| > 65504): the tensor-core attention
                                     multiplies the f16 softmax weights with
                                     f16 value entries, see si_sparse_attn */

/* Workspace must be at least this aligned. */
#define SI_WORKSPACE_ALIGN 256

/* Ragged batch of query rows over paged sequences (section 2.2: each query
 * looks at all of its sequence's earlier positions). */
typedef struct si_batch {
    const int32_t *block_table; /* device [n_seq, max_blocks] physical page ids */
    const int32_t *ctx_len;     /* device [n_seq] cached positions per sequence */
    const int32_t *q_seq;       /* device [n_q] sequence of each query row */
    const int32_t *q_pos;       /* device [n_q] absolute position of the row; it
                                   may look at key positions 0..q_pos inclusive.
                                   Requires q_pos < ctx_len[q_seq]. */
    int32_t n_seq;
    int32_t max_blocks;
    int32_t n_q;                /* number of query rows (0 is allowed: no-op) */
    int32_t page_size;          /* rows per page, 1..1024 */
    int32_t max_ctx;            /* host-known bound: q_pos + 1 <= max_ctx for all
                                   rows; sizes grids, scores and workspaces */
    int32_t n_blocks;           /* physical pages in each cache */
    const int32_t *host_q_seq;  /* optional HOST copy of q_seq [n_q], or NULL.  A
                                   serving scheduler knows its batch: with it the
                                   indexer sends each run of >= 64 consecutive
                                   rows of one sequence (a prefill chunk; section
                                   6.2) to the prefill kernel, whose key tiles
                                   serve several rows at once.  It must match
                                   q_seq; it is read on the host during the call. */
} si_batch;

/* One paged cache: [n_blocks, page_size, row_stride] elements of dtype.
 * Dequantised entry d of a row = code * scale, the scale taken per row or per
 * tile of `scale_tile` consecutive entries (section 5.2 stores the KV cache in
 * FP8 per token and tile of 128 entries).  row_dim and row_stride count
 * elements; an SI_E2M1 row of row_stride entries takes row_stride / 2 bytes
 * (row_stride even). */
typedef struct si_paged {
    const void *data;    /* device; 16-byte aligned */
    const void *scale;   /* device dequantisation scales, or NULL for 1.
                            float (> 0) for every dtype but SI_MXE4M3:
                            [n_blocks, page_size] when scale_tile == 0,
                            [n_blocks, page_size, ceil(row_stride / scale_tile)]
                            otherwise (entry d uses tile d / scale_tile; a
                            value cache that aliases the key rows shares their
                            scales).  SI_MXE4M3: required, E8M0 bytes
                            [n_blocks, page_size, row_stride / 32] with
                            scale_tile = 32 and row_stride a multiple of 32. */
    si_dtype dtype;
    int32_t row_dim;     /* elements used per row */
    int64_t row_stride;  /* elements between consecutive rows, >= row_dim */
    int32_t scale_tile;  /* 0: one scale per row; else entries per scale tile */
} si_paged;

/* Indexer operands (section 2.2: lightweight multi-head indexer; section 5.1
 * stores its keys in FP8). */
typedef struct si_indexer {
    const void *q;       /* device [n_q, n_heads, head_dim], SI_F32, SI_BF16,
                            SI_E4M3 or SI_MXE4M3 */
    si_dtype q_dtype;
    const void *q_scale; /* SI_E4M3 query: device float [n_q, n_heads], one
                            dequantisation scale (> 0) per (row, head) -- the
                            query stored quantised per group as in section
                            4.3's prolog, a group being one head.
                            SI_MXE4M3 query: device E8M0 bytes [n_q, n_heads,
                            head_dim / 32].  Required for those two dtypes,
                            ignored otherwise. */
    const float *w;      /* device [n_q, n_heads] head weights */
    int32_t n_heads;     /* 1..128 */
    int32_t head_dim;    /* 1..256 */
    si_paged k;          /* indexer keys: SI_F32, SI_BF16, SI_E4M3 (+ float
                            scale per row) or SI_MXE4M3.  MXFP8 keys (section
                            5.1) need head_dim a multiple of 32 and a query of
                            SI_MXE4M3, SI_BF16 or SI_F32; a bf16 or f32 query
                            is converted to MXFP8 on the device before scoring,
                            exactly as si_quant_mxfp8 converts it, and the
                            score is computed from the MXFP8 values:
                              score(t,s) = sum_h w[t,h] *
                                 ReLU(sum_d Xq[t,h,d/32] Pq[t,h,d] *
                                            Xk[s,d/32] Pk[s,d]),
                            fp32 accumulation of the exact group products. */
} si_indexer;

/* Sparse attention operands: one shared KV head (MQA / latent KV). */
typedef struct si_attention {
    const void *q;       /* device [n_q, n_heads, d_qk], SI_F32 or SI_BF16 */
    si_dtype q_dtype;
    int32_t n_heads;     /* query heads sharing each KV row, 1..256 */
    int32_t d_qk;        /* logit dims, 1..1024 */
    int32_t d_v;         /* value dims, 1..1024 */
    si_paged k;          /* key rows: row_dim >= d_qk; the dtype of q, or SI_E4M3
                            codes with scales (per row or per tile) for a bf16
                            or f32 q */
    si_paged v;          /* value rows: row_dim >= d_v, dtype as k; may alias k
                            (the value is then the first d_v entries of the key
                            row, with the key row's scales) */
    float softmax_scale; /* logits are softmax_scale * q . k */
} si_attention;

typedef enum si_op {
    SI_OP_INDEXER = 0,
    SI_OP_TOPK = 1,
    SI_OP_ATTN = 2,
    SI_OP_FUSED = 3,
    SI_OP_SELECT = 4  /* si_indexer_topk */
} si_op;

/* Bytes of workspace the operation `op` wants for this batch (the status
 * word included).  For SI_OP_FUSED this is the size that scores all rows in
 * one strip, capped at 64 MiB (a strip that stays in L2 between the indexer
 * and the Top-K); any workspace of at least
 * si_workspace_min(SI_OP_FUSED, ...) works, with fewer rows per strip.
 * Arguments not used by `op` may be NULL.  Returns 0 on invalid arguments. */
size_t si_workspace_size(si_op op, const si_batch *b, const si_indexer *ix,
                         const si_attention *at, int32_t k_top);
size_t si_workspace_min(si_op op, const si_batch *b, const si_indexer *ix,
                        const si_attention *at, int32_t k_top);

/* Indexer scores (section 2.2, first two bullets).
 * scores: device float [n_q, ld_scores], ld_scores >= max_ctx.  Row r gets
 * score(r, s) for s <= q_pos[r] and -inf for q_pos[r] < s < ld_scores. */
si_status si_indexer_scores(const si_batch *b, const si_indexer *ix, float *scores,
                            int64_t ld_scores, void *ws, size_t ws_bytes, void *stream);

/* Top-K selection (section 2.2, second bullet), never a full sort.
 * idx: device int32 [n_q, k_top].  Row r receives the k_top positions with
 * the largest scores among 0..q_pos[r] (equal scores: the lower position
 * wins; -0 equals +0), in ascending order; if q_pos[r] + 1 <= k_top it
 * receives all of them followed by -1 padding.  Scores must not be NaN. */
si_status si_topk(const si_batch *b, const float *scores, int64_t ld_scores, int32_t k_top,
                  int32_t *idx, void *ws, size_t ws_bytes, void *stream);

/* Sparse attention over selected rows (section 2.2 third bullet; 4.2).
 * idx: device int32 [n_q, k_top], entries -1 are skipped.
 * out: device [n_q, n_heads, d_v] of out_dtype (SI_F32 or SI_BF16),
 *   out[r,h] = sum_j softmax_j(softmax_scale * q[r,h] . k[idx_j]) * v[idx_j];
 *   a row with no valid index gets zeros.
 * lse: device float [n_q, n_heads] natural-log sum-exp of the logits, or NULL.
 * Arithmetic of the tensor-core kernel (128 heads, 576-entry latent rows,
 * V = the first 512 entries): logits from bf16 q and k with fp32
 * accumulation; softmax weights rounded to f16 and multiplied with the value
 * entries converted bf16 -> f16, accumulated in fp32.  Value entries (and,
 * with an FP8 cache, query entries and dequantised key entries) must lie in
 * the f16 range, |x| <= 65504: a larger one raises SI_DEVFLAG_RANGE and the
 * output of its row is then undefined.  Below 2^-14 the f16 form is
 * subnormal, an absolute error under 2^-25 per weighted entry. */
si_status si_sparse_attn(const si_batch *b, const si_attention *at, const int32_t *idx,
                         int32_t k_top, void *out, si_dtype out_dtype, float *lse, void *ws,
                         size_t ws_bytes, void *stream);

/* Section 4.1's fused indexer operator on its own (the last step of the
 * indexer prolog in section 4.3, one operator that scores, weights and
 * selects): scores, head weighting and Top-K for every query row, the scores
 * living only in the workspace, a strip of rows at a time, exactly as in
 * si_fused_decode.  idx receives what
 * si_indexer_scores followed by si_topk would give.  ws: at least
 * si_workspace_min(SI_OP_SELECT, ...) bytes (si_workspace_size(SI_OP_SELECT,
 * ...) scores every row in one strip, up to 64 MiB of scores). */
si_status si_indexer_topk(const si_batch *b, const si_indexer *ix, int32_t k_top, int32_t *idx,
                          void *ws, size_t ws_bytes, void *stream);

/* The whole path in one call (section 4.1 fused indexer + 4.2 gather
 * attention): scores -> Top-K -> attention for every query row.  Scores
 * live only in the workspace, a strip of rows at a time; idx receives the
 * selected positions exactly as si_topk would write them. */
si_status si_fused_decode(const si_batch *b, const si_indexer *ix, const si_attention *at,
                          int32_t k_top, int32_t *idx, void *out, si_dtype out_dtype,
                          float *lse, void *ws, size_t ws_bytes, void *stream);

/* Candidate-restricted selection (the vLLM article on DeepSeek-V4.1,
 * "Kernels": the sparse MQA indexer logits are computed over a fixed set of
 * candidate positions per query instead of the whole context; the selection
 * rule is that of section 2.2).
 * cand: device int32 [n_q, ld_cand], ld_cand >= n_cand >= 1.  Row r's
 *   candidates are its list entries s with 0 <= s <= q_pos[r]; they must come
 *   first and in strictly ascending order.  Entries after them that are -1 or
 *   above q_pos[r] are not candidates.  A candidate that does not follow a
 *   lower candidate raises SI_DEVFLAG_BAD_INDEX, and the row's result is then
 *   undefined.  A candidate whose page is invalid raises SI_DEVFLAG_BAD_BLOCK
 *   and is never selected; if the row has fewer than k_top valid candidates
 *   its output may then hold -1 before later positions.
 * idx: device int32 [n_q, k_top].  Row r receives the k_top candidates with the
 *   largest score(r, s) (equal scores: the lower position wins; -0 equals +0),
 *   in ascending order.  A row with fewer than k_top candidates receives all
 *   of them, followed by -1 padding.
 * scores: device float [n_q, ld_scores] with ld_scores >= n_cand, or NULL.
 *   Column j receives the score of list entry j, and -inf where that entry is
 *   not a candidate; columns n_cand..ld_scores-1 get -inf.
 * ws: at least si_workspace_size_cand(b, ix, n_cand) bytes.  It holds the
 *   gathered candidate key rows (n_q x n_cand rounded up to 128, key row
 *   stride bytes each), their scales, the scores when `scores` is NULL, and
 *   the status word.
 * Uses the same indexer operands and kernels as si_indexer_scores / si_topk. */
size_t si_workspace_size_cand(const si_batch *b, const si_indexer *ix, int32_t n_cand);
si_status si_indexer_topk_cand(const si_batch *b, const si_indexer *ix, const int32_t *cand,
                               int32_t n_cand, int64_t ld_cand, int32_t k_top, int32_t *idx,
                               float *scores, int64_t ld_scores, void *ws, size_t ws_bytes,
                               void *stream);

/* si_fused_decode without a workspace, for callers that cannot allocate
 * device memory (for instance code running inside an allocator's callbacks,
 * a process whose device memory another runtime has fully reserved, or a
 * plain C host without an allocator).  The pages describe no such call: it
 * is an interface convenience of this library and computes exactly what
 * si_fused_decode computes, with the same kernels.
 *
 * Scratch: a fixed array of SI_NOALLOC_SCRATCH_BYTES bytes inside the
 * library's device image (one per device) takes the workspace's place.  The
 * call allocates nothing -- no cudaMalloc, no cudaFree, no allocating library
 * routine.  Its first 256 bytes are the sticky status word, which must be
 * zero when the kernels start: the call enqueues a clear of those bytes on
 * `stream` before its kernels, so each call's flags are its own.  The rest is
 * the score strip and needs no initial value.
 * Limit: a request whose minimum fused workspace (si_workspace_min with
 *   SI_OP_FUSED, i.e. 256 + 4 * max_ctx bytes rounded up) exceeds the scratch
 *   -- max_ctx above about 2.09 million positions -- returns
 *   SI_ERR_WORKSPACE before any CUDA call; use si_fused_decode for those.
 * Set-up: the first successful call on each device (with that device
 *   current) looks up the scratch address (cudaGetSymbolAddress), which may
 *   load the library's device module; a failed lookup is retried by the
 *   next call.  Make that first call before any stream capture.
 * Concurrency: all calls on one device share the one scratch.  Calls issued
 *   in order on a single stream are fine; calls that overlap -- on different
 *   streams, or from several host threads without ordering -- race on the
 *   scratch and give undefined results.
 * scratch: if not NULL, *scratch receives the device address of the scratch
 *   when the call returns SI_OK (NULL otherwise), so
 *   si_workspace_status(*scratch, ...) reads the flags of the latest call. */
#define SI_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
si_status si_fused_decode_noalloc(const si_batch *b, const si_indexer *ix,
                                  const si_attention *at, int32_t k_top, int32_t *idx,
                                  void *out, si_dtype out_dtype, float *lse,
                                  const void **scratch, void *stream);

/* MXFP8 conversion (section 4.3's per-group quantisation of the query in
 * the indexer prolog, in section 5.1's format; the rule is the OCP MX
 * specification's, the pages give none of their own).  Per group of 32
 * consecutive entries of a row:
 *   E = floor(log2 max|x|) - 8, clamped to [-127, 127] (an all-zero group
 *       takes -127); scale byte = E + 127;
 *   code = e4m3(x / 2^E), round to nearest even, magnitudes above 448
 *       clamped to 448, the sign kept (-0 for a negative value that rounds
 *       to zero).
 * x: device [n_rows, dim] of x_dtype (SI_F32 or SI_BF16), finite values;
 *    a group holding an infinity or NaN gets scale byte 255 and NaN codes.
 * codes: device uint8 [n_rows, dim]; scales: device uint8 [n_rows, dim / 32].
 * dim: a multiple of 32, 32..65536.  x, codes and scales 16-byte aligned.
 * Needs no workspace; raises no device flag. */
si_status si_quant_mxfp8(const void *x, si_dtype x_dtype, int64_t n_rows, int32_t dim,
                         uint8_t *codes, uint8_t *scales, void *stream);

/* Synchronises `stream`, then reads the sticky device status word of `ws`
 * into *flags (SI_DEVFLAG_*).  Returns SI_ERR_DEVICE if any flag is set. */
si_status si_workspace_status(const void *ws, uint32_t *flags, void *stream);

/* Process-wide count of kernels this library has launched (diagnostic; the
 * only mutable state the library keeps, updated with an atomic add). */
uint64_t si_launch_count(void);

const char *si_status_string(si_status s);
const char *si_last_error(void);
int32_t si_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SI_H_ */
