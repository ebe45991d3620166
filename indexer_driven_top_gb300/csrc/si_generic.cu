// si_generic.cu -- generic CUDA-core kernels of the indexer and the sparse
// attention core.  They accept every dtype and shape the ABI allows and
// compute in fp32; they are the exact path for fp32 workloads and the
// fallback for shapes the tensor-core kernels do not cover.
//
// Indexer: "Day0 Inference Support and Performance Optimization for New
// Architecture LLMs", section 2.2 (scores of each query against all earlier
// positions, aggregated with head weights) over the paged K-cache of 4.1.
// Attention: the same page, section 2.2 third bullet and section 4.2 (gather
// the selected KV rows, softmax-weighted sum).
#include <math.h>

#include "si_common.cuh"
#include "si_internal.h"

namespace si {

namespace {

constexpr int kIdxKeys = 64;  // keys per block of the generic indexer

// One block scores 64 consecutive key positions of one query row.
// Shared memory: q [H*D] | w [H] | keys transposed [D][64].
// MXFP8 keys (section 5.1): entries are code * 2^(e - 127) with the group's
// scale byte e; a bf16 / f32 query is first converted to MXFP8 per group of
// 32 (one warp per group), so both operands hold MXFP8 values.
__global__ void __launch_bounds__(kIdxKeys)
k_indexer_generic(si_batch b, si_indexer ix, float *scores, int64_t ld, unsigned int *st)
{
    extern __shared__ float sm[];
    const int H = ix.n_heads, D = ix.head_dim;
    float *q_s = sm;
    float *w_s = q_s + H * D;
    float *k_s = w_s + H;
    __shared__ int64_t rows[kIdxKeys];

    const int r = blockIdx.x;
    const int tid = threadIdx.x;
    const int64_t s0 = (int64_t)blockIdx.y * kIdxKeys;
    if (s0 >= ld)
        return;
    const int pos = b.q_pos[r];
    const int seq = b.q_seq[r];

    const bool mx = ix.k.dtype == SI_MXE4M3;
    for (int i = tid; i < H * D; i += kIdxKeys) {
        float x = load_elem(ix.q, ix.q_dtype, (int64_t)r * H * D + i);
        if (ix.q_dtype == SI_E4M3)
            x *= fscale(ix.q_scale)[(int64_t)r * H + i / D];
        else if (ix.q_dtype == SI_MXE4M3)  // D % 32 == 0: group (h, d / 32) is i / 32
            x *= mx_scale(__ldg(mxscale(ix.q_scale) + (int64_t)r * (H * D / 32) + i / 32));
        q_s[i] = x;
    }
    if (mx && ix.q_dtype != SI_MXE4M3) {
        __syncthreads();
        const int lane = tid & 31;
        for (int g = tid >> 5; g < H * D / 32; g += kIdxKeys / 32) {
            const float x = q_s[g * 32 + lane];
            const uint32_t b = mx_scale_byte(__reduce_max_sync(0xffffffffu, abs_bits(x)));
            __nv_fp8_e4m3 c;
            c.__x = (__nv_fp8_storage_t)(mx_codes2(x, 0.f, b) & 0xFFu);
            q_s[g * 32 + lane] = b == 255u ? __uint_as_float(0x7FC00000u) : float(c) * mx_scale(b);
        }
    }
    for (int i = tid; i < H; i += kIdxKeys)
        w_s[i] = ix.w[(int64_t)r * H + i];
    const int64_t s = s0 + tid;
    rows[tid] = (s <= pos) ? page_row(b, seq, s, st) : -1;
    __syncthreads();
    for (int i = tid; i < kIdxKeys * D; i += kIdxKeys) {
        const int j = i / D, d = i % D;
        const int64_t row = rows[j];
        float x = row >= 0 ? load_elem(ix.k.data, ix.k.dtype, row * ix.k.row_stride + d) : 0.f;
        if (mx && row >= 0)
            x *= mx_scale(__ldg(mxscale(ix.k.scale) + row * (ix.k.row_stride / 32) + d / 32));
        k_s[d * kIdxKeys + j] = x;
    }
    __syncthreads();
    if (s >= ld)
        return;
    float out = -INFINITY;
    const int64_t row = rows[tid];
    if (s <= pos && row >= 0) {
        float acc = 0.f;
        for (int h = 0; h < H; h++) {
            float dot = 0.f;
            for (int d = 0; d < D; d++)
                dot = fmaf(q_s[h * D + d], k_s[d * kIdxKeys + tid], dot);
            acc = fmaf(w_s[h], fmaxf(dot, 0.f), acc);  // head weight x ReLU
        }
        const float sc = (ix.k.scale && !mx) ? fscale(ix.k.scale)[row] : 1.f;
        out = acc * sc + 0.0f;
    }
    scores[(int64_t)r * ld + s] = out;
}

constexpr int kAttnThreads = 128;

// One block computes one (query row, head): logits over the selected rows,
// softmax, weighted sum of the value rows.
// Shared memory: physical rows [k_top] (int64) | q [d_qk] | z [k_top].
__global__ void __launch_bounds__(kAttnThreads)
k_attn_generic(si_batch b, si_attention at, const int32_t *idx, int k_top, void *out,
               si_dtype out_dtype, float *lse, unsigned int *st)
{
    extern __shared__ int64_t sm64[];
    int64_t *rows = sm64;
    float *q_s = reinterpret_cast<float *>(rows + k_top);
    float *z_s = q_s + at.d_qk;
    __shared__ float red[kAttnThreads / 32];
    __shared__ float bcast;

    const int r = blockIdx.x, h = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int pos = b.q_pos[r];
    const int seq = b.q_seq[r];
    const int64_t qoff = ((int64_t)r * at.n_heads + h) * at.d_qk;

    for (int d = tid; d < at.d_qk; d += kAttnThreads)
        q_s[d] = load_elem(at.q, at.q_dtype, qoff + d);
    for (int j = tid; j < k_top; j += kAttnThreads) {
        const int s = idx[(int64_t)r * k_top + j];
        int64_t row = -1;
        if (s >= 0 && s <= pos)
            row = page_row(b, seq, s, st);
        else if (s != -1)
            raise_flag(st, SI_DEVFLAG_BAD_INDEX);
        rows[j] = row;
    }
    __syncthreads();

    // logits, one warp per selected row
    for (int j = warp; j < k_top; j += kAttnThreads / 32) {
        const int64_t row = rows[j];
        float dot = 0.f;
        if (row >= 0)
            for (int d = lane; d < at.d_qk; d += 32)
                dot = fmaf(q_s[d], load_paged(at.k, row, d), dot);
        dot = warp_sum(dot);
        if (lane == 0)
            z_s[j] = row >= 0 ? dot * at.softmax_scale : -INFINITY;
    }
    __syncthreads();

    float m = -INFINITY;
    for (int j = tid; j < k_top; j += kAttnThreads)
        m = fmaxf(m, z_s[j]);
    m = warp_max(m);
    if (lane == 0)
        red[warp] = m;
    __syncthreads();
    if (tid == 0) {
        float t = red[0];
        for (int i = 1; i < kAttnThreads / 32; i++)
            t = fmaxf(t, red[i]);
        bcast = t;
    }
    __syncthreads();
    m = bcast;
    __syncthreads();
    float l = 0.f;
    for (int j = tid; j < k_top; j += kAttnThreads) {
        const float p = (rows[j] >= 0) ? expf(z_s[j] - m) : 0.f;
        z_s[j] = p;
        l += p;
    }
    l = warp_sum(l);
    if (lane == 0)
        red[warp] = l;
    __syncthreads();
    if (tid == 0) {
        float t = 0.f;
        for (int i = 0; i < kAttnThreads / 32; i++)
            t += red[i];
        bcast = t;
    }
    __syncthreads();
    l = bcast;
    const float inv = l > 0.f ? 1.f / l : 0.f;

    const int64_t ooff = ((int64_t)r * at.n_heads + h) * at.d_v;
    for (int d = tid; d < at.d_v; d += kAttnThreads) {
        float acc = 0.f;
        for (int j = 0; j < k_top; j++) {
            const int64_t row = rows[j];
            if (row >= 0)
                acc = fmaf(z_s[j], load_paged(at.v, row, d), acc);
        }
        acc *= inv;
        if (out_dtype == SI_F32)
            reinterpret_cast<float *>(out)[ooff + d] = acc;
        else
            reinterpret_cast<__nv_bfloat16 *>(out)[ooff + d] = __float2bfloat16_rn(acc);
    }
    if (lse && tid == 0)
        lse[(int64_t)r * at.n_heads + h] = l > 0.f ? m + logf(l) : -INFINITY;
}

}  // namespace

cudaError_t launch_indexer_generic(const si_batch &b, const si_indexer &ix, float *scores,
                                   int64_t ld, unsigned int *st, cudaStream_t s)
{
    const size_t smem = sizeof(float) * ((size_t)ix.n_heads * ix.head_dim + ix.n_heads +
                                         (size_t)ix.head_dim * kIdxKeys);
    cudaError_t e = cudaFuncSetAttribute(k_indexer_generic,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    dim3 grid((unsigned)b.n_q, (unsigned)((ld + kIdxKeys - 1) / kIdxKeys));
    count_launch();
    k_indexer_generic<<<grid, kIdxKeys, smem, s>>>(b, ix, scores, ld, st);
    return cudaGetLastError();
}

cudaError_t launch_attn_generic(const si_batch &b, const si_attention &at, const int32_t *idx,
                                int k_top, void *out, si_dtype out_dtype, float *lse,
                                unsigned int *st, cudaStream_t s)
{
    const size_t smem = sizeof(float) * ((size_t)at.d_qk + k_top) + sizeof(int64_t) * (size_t)k_top;
    cudaError_t e = cudaFuncSetAttribute(k_attn_generic,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    dim3 grid((unsigned)b.n_q, (unsigned)at.n_heads);
    count_launch();
    k_attn_generic<<<grid, kAttnThreads, smem, s>>>(b, at, idx, k_top, out, out_dtype, lse, st);
    return cudaGetLastError();
}

}  // namespace si
