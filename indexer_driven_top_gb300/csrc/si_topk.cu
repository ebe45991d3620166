// si_topk.cu -- Top-K selection of indexer scores by radix select.
//
// "Day0 Inference Support and Performance Optimization for New Architecture
// LLMs", section 2.2: after head weighting, the Top-K most relevant
// historical positions are kept.  The selection here never sorts: it finds
// the exact K-th largest score by three histogram passes over an
// order-preserving 32-bit key (11 + 11 + 10 bits), then emits every position
// above that threshold plus the lowest-positioned ties, in ascending order.
#include "si_common.cuh"
#include "si_internal.h"

namespace si {

namespace {

constexpr int kTopkThreads = 1024;
constexpr int kRadixBins = 2048;

__global__ void __launch_bounds__(kTopkThreads)
k_topk_rows(si_batch b, const float *scores, int64_t ld, int k_top, int32_t *idx)
{
    __shared__ uint32_t hist[kRadixBins];
    __shared__ int sbuf[33];
    __shared__ uint32_t sh_digit;
    __shared__ int sh_rem;

    const int r = blockIdx.x, tid = threadIdx.x;
    int64_t n = (int64_t)b.q_pos[r] + 1;  // candidates 0..pos
    if (n > ld)
        n = ld;
    const float *row = scores + (int64_t)r * ld;
    int32_t *out = idx + (int64_t)r * k_top;

    if (n <= k_top) {  // everything is selected
        for (int i = tid; i < k_top; i += kTopkThreads)
            out[i] = i < n ? i : -1;
        return;
    }

    // ---- exact threshold: the k_top-th largest key
    uint32_t prefix = 0, mask = 0;
    int remaining = k_top;
    for (int pass = 0; pass < 3; pass++) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nbins = pass == 2 ? 1024 : 2048;
        for (int i = tid; i < nbins; i += kTopkThreads)
            hist[i] = 0;
        __syncthreads();
        for (int64_t i = tid; i < n; i += kTopkThreads) {
            const uint32_t key = order_key(__ldg(row + i));
            if ((key & mask) == prefix)
                atomicAdd(&hist[(key >> shift) & (nbins - 1)], 1u);
        }
        __syncthreads();
        // bins in descending order; thread t owns `per` consecutive of them
        const int per = nbins / kTopkThreads;
        int local = 0;
        for (int k = 0; k < per; k++)
            local += hist[nbins - 1 - (tid * per + k)];
        int total;
        int c = block_exclusive_scan(local, &total, sbuf);
        for (int k = 0; k < per; k++) {
            const int d = nbins - 1 - (tid * per + k);
            const int h = hist[d];
            if (c < remaining && c + h >= remaining) {
                sh_digit = (uint32_t)d;
                sh_rem = remaining - c;
            }
            c += h;
        }
        __syncthreads();
        prefix |= sh_digit << shift;
        mask |= (uint32_t)(nbins - 1) << shift;
        remaining = sh_rem;
        __syncthreads();
    }

    // ---- emit: keys above the threshold, then the first `remaining` ties
    const int64_t chunk = (n + kTopkThreads - 1) / kTopkThreads;
    const int64_t lo = min(n, (int64_t)tid * chunk), hi = min(n, lo + chunk);
    int gt = 0, eq = 0;
    for (int64_t i = lo; i < hi; i++) {
        const uint32_t key = order_key(__ldg(row + i));
        gt += key > prefix;
        eq += key == prefix;
    }
    int total;
    const int eq_before = block_exclusive_scan(eq, &total, sbuf);
    int take_eq = max(0, min(eq, remaining - eq_before));
    int o = block_exclusive_scan(gt + take_eq, &total, sbuf);
    for (int64_t i = lo; i < hi; i++) {
        const uint32_t key = order_key(__ldg(row + i));
        const bool take = key > prefix || (key == prefix && take_eq > 0);
        if (key == prefix && take)
            take_eq--;
        if (take && o < k_top)
            out[o++] = (int32_t)i;
    }
}

}  // namespace

cudaError_t launch_topk(const si_batch &b, const float *scores, int64_t ld, int k_top,
                        int32_t *idx, unsigned int *st, cudaStream_t s)
{
    (void)st;
    count_launch();
    k_topk_rows<<<b.n_q, kTopkThreads, 0, s>>>(b, scores, ld, k_top, idx);
    return cudaGetLastError();
}

}  // namespace si
