// si_internal.h -- launchers shared between the libsi translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "si.h"

namespace si {

// Counts one kernel launch (process-wide diagnostic, see si_launch_count).
void count_launch(int n = 1);

// Records the calling thread's error detail (what si_last_error returns) and
// passes `s` through.
si_status set_error(si_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));

// Host validation of si_fused_decode's arguments other than the workspace
// (SI_OK for a valid or empty batch; records the error detail otherwise).
si_status check_fused_args(const si_batch *b, const si_indexer *ix, const si_attention *at,
                           int32_t k_top, const int32_t *idx, const void *out, si_dtype out_dtype);

// Generic CUDA-core kernels: any supported dtype and shape, fp32 arithmetic.
cudaError_t launch_indexer_generic(const si_batch &b, const si_indexer &ix, float *scores,
                                   int64_t ld, unsigned int *st, cudaStream_t s);
cudaError_t launch_attn_generic(const si_batch &b, const si_attention &at, const int32_t *idx,
                                int k_top, void *out, si_dtype out_dtype, float *lse,
                                unsigned int *st, cudaStream_t s);

// Tensor-core indexer: bf16 query, e4m3 keys, 64 heads x 128 dims.
bool indexer_tc_supported(const si_batch &b, const si_indexer &ix, int64_t ld);
cudaError_t launch_indexer_tc(const si_batch &b, const si_indexer &ix, float *scores, int64_t ld,
                              unsigned int *st, cudaStream_t s);
// The same kernel over candidate lists: tile t of row r is slots t*128 .. of
// cand + r * ld_cand (the first n_cand entries; entries -1 or past q_pos[r]
// score -inf); scores[r, j] is the score of slot j.  Same operand conditions.
cudaError_t launch_indexer_tc_cand(const si_batch &b, const si_indexer &ix, const int32_t *cand,
                                   int64_t ld_cand, int32_t n_cand, float *scores, int64_t ld,
                                   unsigned int *st, cudaStream_t s);

// Tensor-core indexer for query rows that all belong to one sequence (a
// causal prefill or a prefill chunk): blocks of four rows (bf16 or FP8 q) or
// three (MXFP8) share each key tile.  Same operand conditions as above; the caller
// guarantees the single sequence.  With fill_tail false the columns past each
// row's position are left unwritten (for a Top-K that reads 0..q_pos only).
// after_own_kernel: the previous kernel of the stream belongs to the same
// call (its inputs were complete before the call), so the launch may overlap
// that kernel's end; only the score stores wait for it.
cudaError_t launch_indexer_prefill(const si_batch &b, const si_indexer &ix, float *scores,
                                   int64_t ld, unsigned int *st, cudaStream_t s,
                                   bool fill_tail = true, bool after_own_kernel = false);

// Tensor-core sparse attention: bf16, 128 heads, 576-dim latent rows (V = first 512).
bool attn_tc_supported(const si_batch &b, const si_attention &at, int k_top);
// Splits of one row's key tiles over clusters for a batch of b.n_q rows on
// `sms` SMs, and the scratch their partial results need (0 when unsplit).
int attn_tc_split(const si_batch &b, int k_top, int sms);
size_t attn_tc_split_bytes(const si_batch &b, int n_split);
cudaError_t launch_attn_tc(const si_batch &b, const si_attention &at, const int32_t *idx,
                           int k_top, void *out, si_dtype out_dtype, float *lse, void *scratch,
                           size_t scratch_bytes, unsigned int *st, cudaStream_t s);

// Merges the split partial results of the tensor-core attention kernels:
// part_o [n_q * n_split * 128 heads, 512] unnormalised fp32 O and part_ml
// [n_q * n_split * 128, 2] (running maximum in log2 units, row sum).
cudaError_t launch_attn_combine(const si_batch &b, int n_split, const float *part_o,
                                const float *part_ml, void *out, si_dtype out_dtype, float *lse,
                                cudaStream_t s);

// Radix select of the k_top best scores per row: among positions 0..q_pos[r],
// or, with fixed_n > 0, among the first fixed_n entries of every row (q_pos
// is then not read).  With `cand`, entry p of row r is slot p of the
// candidate list cand + r * ld_cand, and a selected slot is written as the
// position it holds (-1 where its score is -inf).
cudaError_t launch_topk(const si_batch &b, const float *scores, int64_t ld, int k_top,
                        int32_t *idx, unsigned int *st, cudaStream_t s, int32_t fixed_n = 0,
                        const int32_t *cand = nullptr, int64_t ld_cand = 0);

// Candidate-restricted selection (si_cand.cu).  The candidates of query row r
// are gathered into a private sequence r of a workspace cache with pages of
// kCandPage rows; CandView holds that synthetic batch's device arrays and the
// gathered rows' geometry.
constexpr int32_t kCandPage = 128;
struct CandView {
    int32_t *block_table;     // [n_q, blocks_per_row]: identity
    int32_t *q_seq;           // [n_q]: r
    int32_t *q_pos;           // [n_q]: n_cand - 1
    int32_t *ctx_len;         // [n_q]: n_cand
    int32_t blocks_per_row;   // n_pad / kCandPage
    int32_t n_pad;            // slots per row: n_cand rounded up to kCandPage
    int64_t row_bytes;        // bytes per key row (row_stride x element size)
};
// Gathers the candidate key rows and scales (scale -1 for a slot without a
// candidate) and writes the synthetic batch's arrays.
cudaError_t launch_cand_gather(const si_batch &b, const int32_t *cand, int64_t ld_cand,
                               int32_t n_cand, const CandView &v, const si_paged &k,
                               uint8_t *keys, float *scales, unsigned int *st, cudaStream_t s);
// Sets -inf where a slot holds no candidate (for indexers that do not read
// the -1 scale as "no key").
cudaError_t launch_cand_mask(int32_t n_q, int32_t n_cand, const CandView &v, const float *scales,
                             float *scores, int64_t ld, cudaStream_t s);

}  // namespace si
