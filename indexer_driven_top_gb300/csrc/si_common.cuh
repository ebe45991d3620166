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
    if (p.scale) {
        if (p.scale_tile > 0) {
            const int64_t nt = (p.row_stride + p.scale_tile - 1) / p.scale_tile;
            x *= p.scale[row * nt + d / p.scale_tile];
        } else {
            x *= p.scale[row];
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
