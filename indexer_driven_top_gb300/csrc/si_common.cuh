// si_common.cuh -- device helpers shared by the libsi kernels: status flags,
// paged-cache address translation and scalar element loads.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "si.h"

namespace si {

// The first 16 bytes of every workspace hold the sticky device status word.
constexpr size_t kStatusBytes = 256;

// Launchers keep a few per-device facts (SM count, shared-memory opt-in).
constexpr int kMaxDevices = 64;

// A null status pointer means "do not report" (used by redundant lanes).
// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the previous kernel of its stream still runs;
// griddep_wait() returns once that kernel has completed and its writes are
// visible (at once when there is no such dependency).  griddep_launch_dependents()
// lets the next kernel of the stream start its own preamble early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void raise_flag(unsigned int *st, unsigned int f)
{
    if (st)
        atomicOr(st, f);
}

// Physical row of logical position s of sequence seq in a paged cache
// (paged K-cache of the fused indexer, "Overall Indexer Fusion"); -1 and a
// flag when the block-table entry points outside the cache.
__device__ __forceinline__ int64_t page_row(const si_batch &b, int seq, int64_t s,
                                            unsigned int *st)
{
    const int64_t lb = s / b.page_size;
    if ((unsigned)seq >= (unsigned)b.n_seq || s < 0 || lb >= b.max_blocks) {
        raise_flag(st, SI_DEVFLAG_BAD_BLOCK);
        return -1;
    }
    int blk = __ldg(b.block_table + (int64_t)seq * b.max_blocks + lb);
    if ((unsigned)blk >= (unsigned)b.n_blocks) {
        raise_flag(st, SI_DEVFLAG_BAD_BLOCK);
        return -1;
    }
    return (int64_t)blk * b.page_size + s % b.page_size;
}

// Float scales of a cache or query (every dtype but SI_MXE4M3).
__host__ __device__ __forceinline__ const float *fscale(const void *p)
{
    return static_cast<const float *>(p);
}

// E8M0 scale bytes of an MXFP8 buffer.
__host__ __device__ __forceinline__ const uint8_t *mxscale(const void *p)
{
    return static_cast<const uint8_t *>(p);
}

// ------------------------------------------------------------------ MXFP8
// Section 5.1's indexer format, OCP Microscaling: groups of 32 entries, e4m3
// codes, one E8M0 scale byte e = 2^(e - 127) per group.  Conversion rule (the
// MX specification's): E = floor(log2 max|x|) - 8 clamped to [-127, 127],
// code = e4m3(x / 2^E) with round-to-nearest-even and saturation at 448.
//
// |x| as bits: for non-negative floats the bit patterns order like the
// values, and NaN patterns sort above infinity, so the unsigned maximum of
// these over a group is the bits of max|x| (or marks a non-finite group).
__device__ __forceinline__ uint32_t abs_bits(float x) { return __float_as_uint(x) & 0x7FFFFFFFu; }

// Scale byte E + 127 of a group from the bits of its max|x|: for a normal
// max, floor(log2) + 127 is the exponent field be, so the byte is be - 8,
// and 0 (E = -127) when that is below zero (subnormal or zero max).  A group
// holding an infinity or NaN gets 255.
__device__ __forceinline__ uint32_t mx_scale_byte(uint32_t amax_bits)
{
    const uint32_t be = amax_bits >> 23;
    return be == 255u ? 255u : (be > 8u ? be - 8u : 0u);
}

// 2^-E = 2^(127 - b) for a scale byte b <= 246 (every finite float group):
// the exponent field 254 - b lies in [8, 254], a normal float.
__device__ __forceinline__ float mx_inv_scale(uint32_t b) { return __uint_as_float((254u - b) << 23); }

// 2^(b - 127) for a scale byte b < 255 (b = 0 is the subnormal 2^-127).
__device__ __forceinline__ float mx_scale(uint32_t b)
{
    return b > 0 ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}

// Codes of x0 (low byte) and x1 (high byte) in a group with scale byte b:
// the multiply by a power of two is exact, the conversion rounds to nearest
// even and saturates; a non-finite group gets NaN codes.
__device__ __forceinline__ uint32_t mx_codes2(float x0, float x1, uint32_t b)
{
    if (b == 255u)
        return 0x7F7Fu;
    const float m = mx_inv_scale(b);
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(x0 * m, x1 * m), __NV_SATFINITE,
                                              __NV_E4M3);
}

// OCP FP4 e2m1 code (low 4 bits): sign, 2 exponent bits with bias 1, 1
// mantissa bit; exponent field 0 is subnormal (0 or 0.5).
__device__ __forceinline__ float e2m1_to_float(unsigned c)
{
    const unsigned e = (c >> 1) & 3u, m = c & 1u;
    const float v = e == 0 ? 0.5f * (float)m : (1.f + 0.5f * (float)m) * (float)(1u << (e - 1));
    return (c & 8u) ? -v : v;
}

// Scalar load of element i of a buffer of type t, widened to float (e2m1:
// element i is the low nibble of byte i / 2 when i is even, the high one when
// it is odd).
__device__ __forceinline__ float load_elem(const void *p, si_dtype t, int64_t i)
{
    if (t == SI_F32)
        return __ldg(reinterpret_cast<const float *>(p) + i);
    if (t == SI_BF16) {
        unsigned short u = __ldg(reinterpret_cast<const unsigned short *>(p) + i);
        return __uint_as_float((unsigned)u << 16);
    }
    if (t == SI_E2M1) {
        const unsigned byte = __ldg(reinterpret_cast<const unsigned char *>(p) + (i >> 1));
        return e2m1_to_float((i & 1) ? byte >> 4 : byte & 15u);
    }
    __nv_fp8_e4m3 v;
    v.__x = __ldg(reinterpret_cast<const unsigned char *>(p) + i);
    return float(v);
}

// Dequantised entry d of physical row `row` of a paged cache: the stored
// element times its scale (per row, or per tile of scale_tile entries).
__device__ __forceinline__ float load_paged(const si_paged &p, int64_t row, int d)
{
    float x = load_elem(p.data, p.dtype, row * p.row_stride + d);
    if (p.dtype == SI_MXE4M3) {
        x *= mx_scale(__ldg(mxscale(p.scale) + row * (p.row_stride / 32) + d / 32));
    } else if (p.scale) {
        if (p.scale_tile > 0) {
            const int64_t nt = (p.row_stride + p.scale_tile - 1) / p.scale_tile;
            x *= fscale(p.scale)[row * nt + d / p.scale_tile];
        } else {
            x *= fscale(p.scale)[row];
        }
    }
    return x;
}

// Order-preserving map of a float score onto uint32 (larger score -> larger
// key); -0 is folded onto +0 so that the two compare equal.
__device__ __forceinline__ uint32_t order_key(float f)
{
    f = f + 0.0f;
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Exclusive prefix sum over the threads of a block (threads in order of
// threadIdx.x).  `sbuf` needs blockDim.x/32 + 1 ints.  All threads must call.
__device__ __forceinline__ int block_exclusive_scan(int v, int *total, int *sbuf)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        sbuf[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = lane < nwarps ? sbuf[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o)
                t += y;
        }
        if (lane < nwarps)
            sbuf[lane] = t;  // inclusive warp totals
        if (lane == 31)
            sbuf[32] = t;
    }
    __syncthreads();
    int before = (warp > 0 ? sbuf[warp - 1] : 0) + x - v;
    *total = sbuf[32];
    __syncthreads();
    return before;
}

}  // namespace si
