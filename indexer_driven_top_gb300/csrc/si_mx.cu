// si_mx.cu -- MXFP8 conversion of rows (the per-group quantisation of the
// indexer query that the prolog in section 4.3 of "Day0 Inference Support
// and Performance Optimization for New Architecture LLMs" performs before
// scoring, in the indexer format of its section 5.1: groups of 32 entries,
// one E8M0 scale each).
//
// The pass is bound by HBM: 2 bytes read (bf16) and 1 + 1/32 written per
// entry.  Each thread converts 8 consecutive entries (one 16-byte load of
// bf16), four neighbouring lanes make up a group and agree on its maximum
// with two shuffles, and the codes leave as one 8-byte store per thread.
#include <cuda_fp8.h>

#include <algorithm>
#include <mutex>

#include "si_common.cuh"
#include "si_internal.h"

namespace si {

namespace {

constexpr int kQuantThreads = 256;

template <bool F32>
__global__ void __launch_bounds__(kQuantThreads)
k_quant_mxfp8(const void *x, int64_t n_units, uint8_t *codes, uint8_t *scales)
{
    const int lane = threadIdx.x & 31;
    const int64_t stride = (int64_t)gridDim.x * kQuantThreads;
    // u0 is warp-uniform, so every lane takes the same trips and the group
    // shuffles see whole quads; n_units is a multiple of 4, so a quad is
    // either wholly in range or wholly out.
    for (int64_t u0 = (int64_t)blockIdx.x * kQuantThreads + (threadIdx.x & ~31); u0 < n_units;
         u0 += stride) {
        const int64_t u = u0 + lane;  // unit u = entries 8u .. 8u + 7
        const bool in = u < n_units;
        float v[8];
        if (F32) {
            const float4 *p = reinterpret_cast<const float4 *>(x) + 2 * u;
            const float4 a = in ? __ldg(p) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 c = in ? __ldg(p + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
        } else {
            const uint4 w = in ? __ldg(reinterpret_cast<const uint4 *>(x) + u)
                               : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; i++) {
                v[2 * i] = __uint_as_float(ws[i] << 16);
                v[2 * i + 1] = __uint_as_float(ws[i] & 0xFFFF0000u);
            }
        }
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 8; i++)
            m = max(m, abs_bits(v[i]));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
        const uint32_t b = mx_scale_byte(m);
        uint2 c;
        c.x = mx_codes2(v[0], v[1], b) | (mx_codes2(v[2], v[3], b) << 16);
        c.y = mx_codes2(v[4], v[5], b) | (mx_codes2(v[6], v[7], b) << 16);
        if (in) {
            reinterpret_cast<uint2 *>(codes)[u] = c;
            if ((lane & 3) == 0)
                scales[u >> 2] = (uint8_t)b;
        }
    }
}

}  // namespace

}  // namespace si

extern "C" si_status si_quant_mxfp8(const void *x, si_dtype x_dtype, int64_t n_rows, int32_t dim,
                                    uint8_t *codes, uint8_t *scales, void *stream)
{
    if (n_rows < 0)
        return si::set_error(SI_ERR_INVALID_ARG, "n_rows %lld < 0", (long long)n_rows);
    if (dim < 32 || dim > 65536 || dim % 32 != 0)
        return si::set_error(SI_ERR_INVALID_ARG, "dim %d is not a multiple of 32 in 32..65536",
                             dim);
    if (x_dtype != SI_F32 && x_dtype != SI_BF16)
        return si::set_error(SI_ERR_INVALID_ARG, "x dtype must be f32 or bf16");
    if (n_rows > ((int64_t)1 << 40) / dim)
        return si::set_error(SI_ERR_INVALID_ARG, "n_rows x dim above 2^40");
    if (n_rows == 0)
        return SI_OK;
    if (!x || !codes || !scales)
        return si::set_error(SI_ERR_INVALID_ARG, "x, codes or scales is NULL");
    if (((uintptr_t)x | (uintptr_t)codes | (uintptr_t)scales) % 16 != 0)
        return si::set_error(SI_ERR_INVALID_ARG, "x, codes and scales must be 16-byte aligned");
    static std::once_flag once[si::kMaxDevices];
    static int sms_of[si::kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess && (dev < 0 || dev >= si::kMaxDevices))
        e = cudaErrorInvalidDevice;
    if (e == cudaSuccess) {
        std::call_once(once[dev], [dev] {
            if (cudaDeviceGetAttribute(&sms_of[dev], cudaDevAttrMultiProcessorCount, dev) !=
                cudaSuccess)
                sms_of[dev] = 0;
        });
        const int64_t n_units = n_rows * dim / 8;
        const int64_t want = (n_units + si::kQuantThreads - 1) / si::kQuantThreads;
        // up to 8 blocks of 256 threads per SM, the rest by the grid-stride loop
        const int64_t cap = std::max<int64_t>(1, (int64_t)sms_of[dev] * 8);
        const unsigned grid = (unsigned)std::min(want, cap);
        si::count_launch();
        if (x_dtype == SI_F32)
            si::k_quant_mxfp8<true><<<grid, si::kQuantThreads, 0, (cudaStream_t)stream>>>(
                x, n_units, codes, scales);
        else
            si::k_quant_mxfp8<false><<<grid, si::kQuantThreads, 0, (cudaStream_t)stream>>>(
                x, n_units, codes, scales);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess)
        return si::set_error(SI_ERR_CUDA, "MXFP8 conversion launch: %s", cudaGetErrorString(e));
    return SI_OK;
}
