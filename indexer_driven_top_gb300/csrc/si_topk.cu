// si_topk.cu -- Top-K selection of indexer scores by radix select.
//
// "Day0 Inference Support and Performance Optimization for New Architecture
// LLMs", section 2.2: after head weighting, the Top-K most relevant
// historical positions are kept.  The selection here never sorts: it finds
// the exact K-th largest score by three histogram passes over an
// order-preserving 32-bit key (11 + 11 + 10 bits), then emits every position
// above that threshold plus the lowest-positioned ties, in ascending order.
//
// One 1024-thread CTA per query row.  Rows of up to 16384 candidates are read
// once into registers (thread t holds E consecutive positions) and every pass
// runs on the cached keys.  Rows of up to 8 x 16384 take a cluster of CTAs
// (one 16384-position segment each, histograms merged in distributed shared
// memory); longer rows stream from global memory per pass.
#include <algorithm>
#include <mutex>

#include "si_common.cuh"
#include "si_internal.h"
#include "si_sm100.cuh"

namespace si {

namespace {

using namespace sm100;

constexpr int kTopkThreads = 1024;
constexpr int kRadixBins = 2048;

// Candidate-restricted selection (si_indexer_topk_cand): the rows are the
// slots of per-row candidate lists, and a selected slot is written as the
// position it holds -- -1 for a slot without a candidate, whose score is
// -inf.  The lists hold their candidates first and ascending, so such slots
// sort after every candidate and the output stays ascending with -1 last.
struct SlotMap {
    const int32_t *cand;  // NULL: write the selected positions themselves
    int64_t ld;
};
constexpr uint32_t kNegInfKey = 0x007FFFFFu;  // order_key(-inf)

__device__ __forceinline__ int32_t out_value(const SlotMap &m, int r, int64_t p, uint32_t key)
{
    if (!m.cand)
        return (int32_t)p;
    return key == kNegInfKey ? -1 : __ldg(m.cand + (int64_t)r * m.ld + p);
}

// Finds, among the cached keys, the digit of the k-th largest key at `shift`
// (bins in descending order) and how many of the k fall in that digit's bin.
// Every thread returns the same (digit, remaining).
__device__ __forceinline__ void radix_step(uint32_t *hist, int *sbuf, uint32_t *sh_digit,
                                           int *sh_rem, int nbins, int &remaining)
{
    const int tid = threadIdx.x;
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
            *sh_digit = (uint32_t)d;
            *sh_rem = remaining - c;
        }
        c += h;
    }
    __syncthreads();
    remaining = *sh_rem;
}

// Row of n <= E * kTopkThreads candidates (n > k_top): keys cached in
// registers, thread t owning positions [t E, t E + E).
template <int E>
__device__ __forceinline__ void topk_cached(const SlotMap &m, int r, const float *row, int n,
                                            int k_top, int32_t *out,
                                            uint32_t *hist, int *sbuf, uint32_t *sh_digit,
                                            int *sh_rem)
{
    const int tid = threadIdx.x;
    const int p0 = tid * E;
    uint32_t key[E];
    uint32_t valid = 0;  // bit e: position p0 + e < n
    // vector loads need a 16-byte aligned row start (p0 is a multiple of 8)
    if (p0 + E <= n && (reinterpret_cast<uintptr_t>(row) & 15) == 0) {
#pragma unroll
        for (int e = 0; e < E; e += 4) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(row + p0 + e));
            key[e] = order_key(v.x);
            key[e + 1] = order_key(v.y);
            key[e + 2] = order_key(v.z);
            key[e + 3] = order_key(v.w);
        }
        valid = (E == 32) ? 0xffffffffu : ((1u << E) - 1);
    } else {
#pragma unroll
        for (int e = 0; e < E; e++) {
            const bool in = p0 + e < n;
            key[e] = in ? order_key(__ldg(row + p0 + e)) : 0u;
            valid |= (in ? 1u : 0u) << e;
        }
    }
    uint32_t prefix = 0, mask = 0;
    int remaining = k_top;
    for (int pass = 0; pass < 3; pass++) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nbins = pass == 2 ? 1024 : 2048;
        for (int i = tid; i < nbins; i += kTopkThreads)
            hist[i] = 0;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; e++)
            if (((valid >> e) & 1u) && (key[e] & mask) == prefix)
                atomicAdd(&hist[(key[e] >> shift) & (nbins - 1)], 1u);
        __syncthreads();
        radix_step(hist, sbuf, sh_digit, sh_rem, nbins, remaining);
        prefix |= *sh_digit << shift;
        mask |= (uint32_t)(nbins - 1) << shift;
        __syncthreads();
    }
    // emit: keys above the threshold, then the first `remaining` ties
    int gt = 0, eq = 0;
#pragma unroll
    for (int e = 0; e < E; e++) {
        const bool in = (valid >> e) & 1u;
        gt += in && key[e] > prefix;
        eq += in && key[e] == prefix;
    }
    int total;
    const int eq_before = block_exclusive_scan(eq, &total, sbuf);
    int take_eq = max(0, min(eq, remaining - eq_before));
    int o = block_exclusive_scan(gt + take_eq, &total, sbuf);
#pragma unroll
    for (int e = 0; e < E; e++) {
        const bool in = (valid >> e) & 1u;
        const bool tie = in && key[e] == prefix;
        const bool take = (in && key[e] > prefix) || (tie && take_eq > 0);
        if (tie && take)
            take_eq--;
        if (take && o < k_top)
            out[o++] = out_value(m, r, p0 + e, key[e]);
    }
}

__global__ void __launch_bounds__(kTopkThreads)
k_topk_rows(si_batch b, const float *scores, int64_t ld, int k_top, int32_t *idx, int32_t fixed_n,
            SlotMap m)
{
    __shared__ uint32_t hist[kRadixBins];
    __shared__ int sbuf[33];
    __shared__ uint32_t sh_digit;
    __shared__ int sh_rem;

    griddep_launch_dependents();  // the attention kernel may set itself up meanwhile
    const int r = blockIdx.x, tid = threadIdx.x;
    // candidates 0..pos, or the first fixed_n entries of every row
    int64_t n = fixed_n > 0 ? (int64_t)fixed_n : (int64_t)b.q_pos[r] + 1;
    if (n > ld)
        n = ld;
    const float *row = scores + (int64_t)r * ld;
    int32_t *out = idx + (int64_t)r * k_top;

    // The scores come from the previous kernel of the stream.  Every CTA
    // waits for it, so that this grid never completes before that one.
    griddep_wait();
    if (n <= k_top) {  // everything is selected
        for (int i = tid; i < k_top; i += kTopkThreads)
            out[i] = i < n ? out_value(m, r, i, m.cand ? order_key(__ldg(row + i)) : 0u) : -1;
        return;
    }
    if (n <= 8 * kTopkThreads) {
        topk_cached<8>(m, r, row, (int)n, k_top, out, hist, sbuf, &sh_digit, &sh_rem);
        return;
    }
    if (n <= 16 * kTopkThreads) {
        topk_cached<16>(m, r, row, (int)n, k_top, out, hist, sbuf, &sh_digit, &sh_rem);
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
            out[o++] = out_value(m, r, i, key);
    }
}

// Long rows (16384 < n <= 1024 E C): a cluster of C CTAs per row, CTA q
// caching positions [1024 E q, 1024 E (q + 1)) in shared memory (4 KB per
// key of a thread; thread t owns positions E t .. E t + E - 1, stored at
// e * 1024 + t so that a warp's accesses fall in distinct banks).  With
// E = 32 rows of 131072 take clusters of four: clusters of eight CTAs that
// each fill an SM do not all fit on the GPU at once, and the second wave
// starts only when the first has finished (clusters of eight with E = 16,
// two CTAs per SM, all fit but were not faster: 32.9 against 31.0 us on 16
// rows of 131072).  Each radix pass
// adds every CTA's histogram into a per-pass histogram in CTA 0's shared
// memory (distributed shared memory atomics), and every CTA then reads the
// merged counts and takes the same decision.  The emit pass orders the CTAs'
// selections by their segment: CTA q writes after the selections and the
// tie quota of CTAs 0..q-1, whose counts it reads from CTA 0.
// E keys per thread: 32 for the clusters of long rows; 16 (64 KB of keys, so
// that two 1024-thread CTAs share an SM) for batches of more rows than SMs
// whose rows of 8193..16384 fit one CTA (the register-cached row kernel holds
// an SM alone).
constexpr int kClusterE = 32;
constexpr int kSegment = kClusterE * kTopkThreads;  // positions per CTA
constexpr int kMaxCluster = 8;
constexpr int kClusterSmem = kSegment * 4;          // the CTA's keys (dynamic shared memory)
constexpr int kLeanE = 16;
constexpr int kLeanSmem = kLeanE * kTopkThreads * 4;

template <int E>
__global__ void __launch_bounds__(kTopkThreads)
k_topk_cluster(si_batch b, const float *scores, int64_t ld, int k_top, int32_t *idx,
               int32_t fixed_n, SlotMap m)
{
    constexpr int kSeg = E * kTopkThreads;      // positions per CTA
    extern __shared__ uint32_t ks[];             // [E][kTopkThreads] keys
    __shared__ uint32_t hist[kRadixBins];
    __shared__ uint32_t merged[3][kRadixBins];   // used in CTA 0: one histogram per pass
    __shared__ uint32_t counts[kMaxCluster][2];  // used in CTA 0: (above, ties) per CTA
    __shared__ int sbuf[33];
    __shared__ uint32_t sh_digit;
    __shared__ int sh_rem;

    griddep_launch_dependents();
    const uint32_t q = cluster_rank();
    uint32_t C;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(C));
    const int r = (int)(blockIdx.x / C), tid = threadIdx.x;
    int64_t n = fixed_n > 0 ? (int64_t)fixed_n : (int64_t)b.q_pos[r] + 1;
    if (n > ld)
        n = ld;
    const float *row = scores + (int64_t)r * ld;
    int32_t *out = idx + (int64_t)r * k_top;

    if (q == 0)
        for (int i = tid; i < 3 * kRadixBins; i += kTopkThreads)
            (&merged[0][0])[i] = 0;
    griddep_wait();  // the scores come from the previous kernel of the stream
    cluster_sync();  // CTA 0's merged histograms are zero before anyone adds

    if (n <= k_top) {  // everything is selected (the same on every CTA)
        if (q == 0)
            for (int i = tid; i < k_top; i += kTopkThreads)
                out[i] = i < n ? out_value(m, r, i, m.cand ? order_key(__ldg(row + i)) : 0u) : -1;
        cluster_sync();
        return;
    }
    const int64_t p0 = (int64_t)q * kSeg + (int64_t)tid * E;
    uint32_t valid = 0;  // bit e: position p0 + e < n
    if (p0 + E <= n && (reinterpret_cast<uintptr_t>(row) & 15) == 0) {
#pragma unroll
        for (int e = 0; e < E; e += 4) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(row + p0 + e));
            ks[(e + 0) * kTopkThreads + tid] = order_key(v.x);
            ks[(e + 1) * kTopkThreads + tid] = order_key(v.y);
            ks[(e + 2) * kTopkThreads + tid] = order_key(v.z);
            ks[(e + 3) * kTopkThreads + tid] = order_key(v.w);
        }
        valid = 0xffffffffu;
    } else {
#pragma unroll
        for (int e = 0; e < E; e++) {
            const bool in = p0 + e < n;
            ks[e * kTopkThreads + tid] = in ? order_key(__ldg(row + p0 + e)) : 0u;
            valid |= (in ? 1u : 0u) << e;
        }
    }
    const uint32_t merged0 = mapa_shared(smem_u32(&merged[0][0]), 0);
    const uint32_t counts0 = mapa_shared(smem_u32(&counts[0][0]), 0);
    uint32_t prefix = 0, mask = 0;
    int remaining = k_top;
    for (int pass = 0; pass < 3; pass++) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nbins = pass == 2 ? 1024 : 2048;
        for (int i = tid; i < nbins; i += kTopkThreads)
            hist[i] = 0;
        __syncthreads();
#pragma unroll 8
        for (int e = 0; e < E; e++) {
            const uint32_t key = ks[e * kTopkThreads + tid];
            if (((valid >> e) & 1u) && (key & mask) == prefix)
                atomicAdd(&hist[(key >> shift) & (nbins - 1)], 1u);
        }
        __syncthreads();
        for (int i = tid; i < nbins; i += kTopkThreads)
            if (hist[i])
                red_cluster_add_u32(merged0 + (uint32_t)(pass * kRadixBins + i) * 4u, hist[i]);
        cluster_sync();
        for (int i = tid; i < nbins; i += kTopkThreads)
            hist[i] = ld_cluster_u32(merged0 + (uint32_t)(pass * kRadixBins + i) * 4u);
        __syncthreads();
        radix_step(hist, sbuf, &sh_digit, &sh_rem, nbins, remaining);
        prefix |= sh_digit << shift;
        mask |= (uint32_t)(nbins - 1) << shift;
        __syncthreads();
    }
    // emit
    int gt = 0, eq = 0;
#pragma unroll 8
    for (int e = 0; e < E; e++) {
        const uint32_t key = ks[e * kTopkThreads + tid];
        const bool in = (valid >> e) & 1u;
        gt += in && key > prefix;
        eq += in && key == prefix;
    }
    int gt_total, eq_total;
    const int eq_before = block_exclusive_scan(eq, &eq_total, sbuf);
    block_exclusive_scan(gt, &gt_total, sbuf);
    if (tid == 0) {
        st_cluster_u32(counts0 + q * 8u, (uint32_t)gt_total);
        st_cluster_u32(counts0 + q * 8u + 4u, (uint32_t)eq_total);
    }
    cluster_sync();
    // selections and tie quota of the CTAs before this one
    int off = 0, eq_prev = 0;
    for (uint32_t c = 0; c < q; c++) {
        const int g = (int)ld_cluster_u32(counts0 + c * 8u);
        const int t = (int)ld_cluster_u32(counts0 + c * 8u + 4u);
        off += g + max(0, min(t, remaining - eq_prev));
        eq_prev += t;
    }
    int take_eq = max(0, min(eq, remaining - eq_prev - eq_before));
    int total;
    int o = off + block_exclusive_scan(gt + take_eq, &total, sbuf);
#pragma unroll 8
    for (int e = 0; e < E; e++) {
        const uint32_t key = ks[e * kTopkThreads + tid];
        const bool in = (valid >> e) & 1u;
        const bool tie = in && key == prefix;
        const bool take = (in && key > prefix) || (tie && take_eq > 0);
        if (tie && take)
            take_eq--;
        if (take && o < k_top)
            out[o++] = out_value(m, r, p0 + e, key);
    }
    cluster_sync();  // CTA 0's shared memory stays until every CTA has read it
}

}  // namespace

cudaError_t launch_topk(const si_batch &b, const float *scores, int64_t ld, int k_top,
                        int32_t *idx, unsigned int *st, cudaStream_t s, int32_t fixed_n,
                        const int32_t *cand, int64_t ld_cand)
{
    const SlotMap m{cand, ld_cand};
    (void)st;
    count_launch();
    // may overlap the tail of the kernel that wrote the scores (programmatic
    // dependent launch; the kernel waits for it before reading them)
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kTopkThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Rows longer than one CTA's register cache take a cluster of C CTAs per
    // row (b.max_ctx bounds every row's candidate count) when one CTA per row
    // would leave most of the GPU idle; a batch with many rows keeps one CTA
    // per row: with keys in shared memory (two CTAs per SM) when the rows fit
    // one CTA, outnumber the SMs and are longer than the 8-key register cache
    // (a late prefill strip; shorter rows are faster from registers), else
    // from registers or streaming.
    static int sms_of[kMaxDevices];
    static std::once_flag once[kMaxDevices];
    static cudaError_t err_of[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        dev = 0;
    std::call_once(once[dev], [dev] {
        err_of[dev] = cudaFuncSetAttribute(k_topk_cluster<kClusterE>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kClusterSmem);
        if (err_of[dev] == cudaSuccess)
            err_of[dev] = cudaFuncSetAttribute(k_topk_cluster<kLeanE>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kLeanSmem);
    });
    if (sms_of[dev] == 0 &&
        cudaDeviceGetAttribute(&sms_of[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms_of[dev] = 1;
    const int64_t longest = std::min<int64_t>(fixed_n > 0 ? fixed_n : b.max_ctx, ld);
    const int C = (int)((longest + kSegment - 1) / kSegment);
    if (longest > 16 * kTopkThreads && C <= kMaxCluster &&
        (int64_t)b.n_q * C <= 2 * (int64_t)sms_of[dev]) {
        if (err_of[dev] != cudaSuccess)
            return err_of[dev];
        cfg.gridDim = dim3((unsigned)(b.n_q * C));
        cfg.dynamicSmemBytes = kClusterSmem;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)C;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, k_topk_cluster<kClusterE>, b, scores, ld, k_top, idx,
                                  fixed_n, m);
    }
    cfg.gridDim = dim3((unsigned)b.n_q);
    if (longest > 8 * kTopkThreads && longest <= (int64_t)kLeanE * kTopkThreads &&
        b.n_q > sms_of[dev]) {
        if (err_of[dev] != cudaSuccess)
            return err_of[dev];
        cfg.dynamicSmemBytes = kLeanSmem;  // a cluster of one CTA per row
        return cudaLaunchKernelEx(&cfg, k_topk_cluster<kLeanE>, b, scores, ld, k_top, idx,
                                  fixed_n, m);
    }
    return cudaLaunchKernelEx(&cfg, k_topk_rows, b, scores, ld, k_top, idx, fixed_n, m);
}

}  // namespace si
