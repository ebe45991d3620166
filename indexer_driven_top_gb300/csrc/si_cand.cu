// si_cand.cu -- candidate-restricted selection: the indexer scores only a
// given list of candidate positions per query row instead of the whole
// context, and the Top-K is taken among them.
//
// The vLLM article on DeepSeek-V4.1 ("Kernels") computes the sparse MQA
// indexer logits over a fixed candidate set per query; at long contexts that
// replaces the full-context scoring.  The selection rule is that of "Day0
// Inference Support and Performance Optimization for New Architecture LLMs",
// section 2.2 (head-weighted ReLU scores, Top-K, ties to the lower position).
//
// GB300 mapping.  With the 64 x 128 FP8-key shapes, the tensor-core indexer
// gathers the candidate rows itself (k_indexer_tc<true>).  For other shapes,
// k_cand_gather copies each row's candidate key rows (and their scales) out
// of the paged cache into the workspace, laid out as one private sequence per
// query row with pages of 128 rows, so that candidate slot j of row r is
// position j of sequence r, and the CUDA-core indexer scores those sequences
// (k_cand_mask then sets -inf where a slot holds no candidate).  Either way
// the radix Top-K selects among the first n_cand slots of each row and
// writes each selected slot as the position it holds.  Candidate lists hold their
// candidates first and in strictly ascending order, so slot order is position
// order: the Top-K's tie rule and ascending output carry over unchanged.
#include <stdint.h>

#include <algorithm>

#include "si_common.cuh"
#include "si_internal.h"

namespace si {

namespace {

// Gathers candidate key rows.  A warp takes 32 consecutive slots of one row:
// lane l resolves slot l (list entry -> block table -> physical row) and
// writes its scale; then the warp copies the 32 rows in units of 16 bytes
// (1 byte when the row size is not a multiple of 16), each lane issuing up to
// eight independent loads before their stores, so that a warp has many row
// pieces in flight.  Also writes the synthetic batch (identity block table,
// one sequence per row).
__global__ void k_cand_gather(si_batch b, const int32_t *cand, int64_t ld_cand, int32_t n_cand,
                              CandView v, const uint8_t *kdata, const float *kscale,
                              uint8_t *keys, float *scales, unsigned int *st)
{
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nth = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = tid; i < (int64_t)b.n_q * v.blocks_per_row; i += nth)
        v.block_table[i] = (int32_t)i;
    for (int64_t r = tid; r < b.n_q; r += nth) {
        v.q_seq[r] = (int32_t)r;
        v.q_pos[r] = n_cand - 1;
        v.ctx_len[r] = n_cand;
    }
    const int lane = threadIdx.x & 31;
    const bool vec = v.row_bytes % 16 == 0;
    const int64_t units = vec ? v.row_bytes / 16 : v.row_bytes;  // per key row
    const int64_t groups = (int64_t)b.n_q * (v.n_pad / 32);       // n_pad is a multiple of 128
    for (int64_t gi = tid >> 5; gi < groups; gi += nth >> 5) {
        const int64_t slot0 = gi * 32;
        const int64_t slot = slot0 + lane;
        const int r = (int)(slot / v.n_pad), j = (int)(slot % v.n_pad);
        const int64_t cb = (int64_t)r * ld_cand;
        const int s = j < n_cand ? __ldg(cand + cb + j) : -1;
        const int pos = __ldg(b.q_pos + r), seq = __ldg(b.q_seq + r);
        int64_t prow = -1;
        if (s >= 0 && s <= pos) {
            // a candidate follows a candidate with a lower position
            if (j > 0) {
                const int sp = __ldg(cand + cb + j - 1);
                if (!(sp >= 0 && sp < s))
                    raise_flag(st, SI_DEVFLAG_BAD_INDEX);
            }
            const int lb = s / b.page_size;
            if ((unsigned)seq < (unsigned)b.n_seq && lb < b.max_blocks) {
                const int blk = __ldg(b.block_table + (int64_t)seq * b.max_blocks + lb);
                if ((unsigned)blk < (unsigned)b.n_blocks)
                    prow = (int64_t)blk * b.page_size + s % b.page_size;
            }
            if (prow < 0)
                raise_flag(st, SI_DEVFLAG_BAD_BLOCK);
        }
        scales[slot] = prow >= 0 ? (kscale ? __ldg(kscale + prow) : 1.f) : -1.f;
        // unit t of the group (t = k * 32 + lane) is unit t % units of slot t / units
        for (int64_t k0 = 0; k0 < units; k0 += 8) {
            if (vec) {
                uint4 x[8];
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    x[k] = make_uint4(0u, 0u, 0u, 0u);
                    if (k0 + k < units) {  // the same for every lane
                        const int64_t t = (k0 + k) * 32 + lane;
                        const int c = (int)(t / units);
                        const long long pr = __shfl_sync(0xffffffffu, (long long)prow, c);
                        if (pr >= 0)
                            x[k] = __ldg(reinterpret_cast<const uint4 *>(kdata + pr * v.row_bytes) +
                                         t % units);
                    }
                }
#pragma unroll
                for (int k = 0; k < 8; k++)
                    if (k0 + k < units) {
                        const int64_t t = (k0 + k) * 32 + lane;
                        reinterpret_cast<uint4 *>(keys + (slot0 + t / units) * v.row_bytes)[t % units] =
                            x[k];
                    }
            } else {
                for (int k = 0; k < 8 && k0 + k < units; k++) {
                    const int64_t t = (k0 + k) * 32 + lane;
                    const int c = (int)(t / units);
                    const long long pr = __shfl_sync(0xffffffffu, (long long)prow, c);
                    keys[(slot0 + c) * v.row_bytes + t % units] =
                        pr >= 0 ? __ldg(kdata + pr * v.row_bytes + t % units) : (uint8_t)0;
                }
            }
        }
    }
}

// -inf for the slots that hold no candidate (CUDA-core indexer path).
__global__ void k_cand_mask(int32_t n_q, int32_t n_cand, CandView v, const float *scales,
                            float *scores, int64_t ld)
{
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nth = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = tid; i < (int64_t)n_q * n_cand; i += nth) {
        const int64_t r = i / n_cand, j = i % n_cand;
        if (scales[r * v.n_pad + j] < 0.f)
            scores[r * ld + j] = -INFINITY;
    }
}

// One thread per work item: the gather's loads form a chain (list entry ->
// block table -> key row), so latency is hidden by many threads in flight,
// not by a grid-stride loop.
int grid_for(int64_t work, int threads)
{
    const int64_t want = (work + threads - 1) / threads;
    return (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)1 << 24));
}

}  // namespace

cudaError_t launch_cand_gather(const si_batch &b, const int32_t *cand, int64_t ld_cand,
                               int32_t n_cand, const CandView &v, const si_paged &k,
                               uint8_t *keys, float *scales, unsigned int *st, cudaStream_t s)
{
    // one warp per 32 slots
    const int grid = grid_for((int64_t)b.n_q * v.n_pad, 256);
    count_launch();
    k_cand_gather<<<grid, 256, 0, s>>>(b, cand, ld_cand, n_cand, v,
                                       static_cast<const uint8_t *>(k.data), fscale(k.scale), keys,
                                       scales, st);
    return cudaGetLastError();
}

cudaError_t launch_cand_mask(int32_t n_q, int32_t n_cand, const CandView &v, const float *scales,
                             float *scores, int64_t ld, cudaStream_t s)
{
    const int grid = grid_for((int64_t)n_q * n_cand, 256);
    count_launch();
    k_cand_mask<<<grid, 256, 0, s>>>(n_q, n_cand, v, scales, scores, ld);
    return cudaGetLastError();
}

}  // namespace si
