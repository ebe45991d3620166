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

// Tensor-core indexer for query rows that all belong to one sequence (a
// causal prefill or a prefill chunk): blocks of two (bf16 q) or four (FP8 q)
// rows share each key tile.  Same operand conditions as above; the caller
// guarantees the single sequence.
cudaError_t launch_indexer_prefill(const si_batch &b, const si_indexer &ix, float *scores,
                                   int64_t ld, unsigned int *st, cudaStream_t s);

// Tensor-core sparse attention: bf16, 128 heads, 576-dim latent rows (V = first 512).
bool attn_tc_supported(const si_batch &b, const si_attention &at, int k_top);
// Splits of one row's key tiles over clusters for a batch of b.n_q rows on
// `sms` SMs, and the scratch their partial results need (0 when unsplit).
int attn_tc_split(const si_batch &b, int k_top, int sms);
size_t attn_tc_split_bytes(const si_batch &b, int n_split);
cudaError_t launch_attn_tc(const si_batch &b, const si_attention &at, const int32_t *idx,
                           int k_top, void *out, si_dtype out_dtype, float *lse, void *scratch,
                           size_t scratch_bytes, unsigned int *st, cudaStream_t s);

// Radix select of the k_top best scores per row.
cudaError_t launch_topk(const si_batch &b, const float *scores, int64_t ld, int k_top,
                        int32_t *idx, unsigned int *st, cudaStream_t s);

}  // namespace si
