// si_attn_tc.cu -- tensor-core sparse attention over selected latent KV rows.
//
// "Day0 Inference Support and Performance Optimization for New Architecture
// LLMs", section 2.2 third bullet and section 4.2: the attention core gathers
// only the KV rows at the selected positions from the main (paged) KV cache
// and returns the softmax-weighted sum of their values.  One shared latent
// KV row of 576 bf16 per position serves all 128 query heads (K = the whole
// row, V = its first 512 entries):
//     out[r,h] = sum_j softmax_j(scale * q[r,h] . k[idx_j]) * v[idx_j]
//
// GB300 mapping.  Each query row gets a cluster of two CTAs with different
// jobs, because one SM cannot hold the row's query (128 x 576 bf16, 147 KB of
// shared memory), its output accumulator (128 x 512 fp32, all 512 TMEM
// columns) and enough rows in flight at once:
//
//   score CTA (rank 0) -- keeps the whole query in shared memory (128-byte
//       swizzle) and streams the selected keys through a three-slot ring in
//       "dim chunks" of 128 keys x 64 dims (16 KB; the FP8 cache's variant
//       stages codes, below).  Nine chunks build the
//       tile's logits S = q . k^T (UMMA M = 128 heads, N = 128 keys) in TMEM
//       (double-buffered).  Eight softmax warps (two threads per head, each
//       taking half of the tile's keys) turn a tile into weights P (f16) and
//       stage them, with one rescale factor per head, in local shared memory;
//       one thread then hands the tile to the value CTA with two bulk copies
//       into its shared memory (the copy engine moves the 32.5 KB, the
//       softmax warps go on to the next tile).  A row warp resolves each
//       tile's selected
//       positions to physical rows (block table) and key-valid bits ahead of
//       the loaders and the softmax.
//   value CTA (rank 1) -- keeps O (128 heads x 512 value dims, fp32) in TMEM
//       and streams the same rows' first 512 entries through a five-slot ring
//       of 128-dim groups (32 KB).  Five warps rewrite each group from bf16 to
//       f16 in place (P.V needs one operand type), the MMA warp issues
//       O[:, group] += P . V_group (N = 128), and a warpgroup applies the
//       score CTA's rescale factors to O between tiles and normalises at the
//       end.
//
// Rows are gathered by eight loader warps per CTA with 16-byte cp.async
// copies straight into ring slots; the copies arrive on the slot's mbarrier
// when they land, so no thread stalls on them.  Lookups that feed the copies
// (index list, block table) are done by other warps or issued tiles ahead:
// a thread's plain loads complete behind its own copies in flight, and a
// release-ordered arrive waits for them.  Every wait is bounded.
//
// The query arrives by tensor copies; the output leaves by tensor stores of
// 128-byte column blocks staged in the idle value ring.  With few rows, each
// row's key tiles are split over up to eight clusters: a split writes its
// unnormalised O and (m, l) per head to scratch, and k_attn_combine merges
// the splits.
//
// Quantised caches (k_attn_tc<1>: section 5.2's FP8 codes with one scale per
// token and tile of 128 entries; k_attn_tc<2>: the NVFP4 latent cache of the
// vLLM article on DeepSeek-V4.1, e2m1 codes with one scale per 16-entry
// block): the score CTA converts the query to f16 once and dequantises key
// chunks to f16 (four warps gather codes -- and, for FP4, each chunk's block
// scales -- into staging slots, four dequantise them into the ring), the
// value CTA's converters dequantise staged value groups; per-tile or
// per-block fp32 scales do not fold into bf16 exactly, f16 keeps 11
// significant bits.
//
// Softmax: online in the log2 domain with fp32 state; the exponent reference
// is only raised when a tile's maximum exceeds it by more than 8, so most
// tiles leave O untouched.  P is rounded to f16 (11 significant bits) and the
// denominator sums the same rounded values.  Value rows are converted bf16 ->
// f16 (exact for 2^-14 <= |v| <= 65504).  Positions that are -1 or outside
// 0..pos get zero rows and zero weight.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include "si_common.cuh"
#include "si_internal.h"
#include "si_sm100.cuh"
#include "si_tmap.h"

namespace si {

namespace {

using namespace sm100;

constexpr int kHeads = 128;              // query heads = UMMA M
constexpr int kDqk = 576;                // logit dims
constexpr int kDv = 512;                 // value dims
constexpr int kTile = 128;               // selected keys per tile
constexpr int kQChunks = kDqk / 64;      // 9 score chunks per tile
constexpr int kVGroups = kDv / 128;      // 4 value groups per tile
constexpr uint32_t kChunk = 128 * 128;   // 16 KB: 128 rows x 128 bytes, SW128
constexpr uint32_t kGroup = 2 * kChunk;  // 32 KB: 128 keys x 128 value dims

constexpr int kLoaderWarps = 8;   // warps 0..7
constexpr int kLoaders = kLoaderWarps * 32;
constexpr int kRowsPerLoader = kTile / (kLoaders / 8);  // 4 rows x one 16-byte unit each
constexpr int kWarpSoft0 = 8;     // score CTA: softmax warps 8..15, two per TMEM lane quarter
constexpr int kSoftmax = 8 * 32;
constexpr int kWarpQuad = 8;      // value CTA: O rescale / epilogue warps 8..11
constexpr int kWarpMma = 16;
constexpr int kWarpRows = 17;     // score CTA: physical rows and key-valid bits of each tile
constexpr int kConverters = 5 * 32;  // value CTA: warps 12..15 and 17
constexpr int kThreads = 18 * 32;
constexpr float kRescaleThreshold = 8.f;  // log2 units
constexpr int kMaxSplit = 8;              // clusters per row at most

// score CTA layout
constexpr int kRingS = 3;
constexpr uint32_t kOffQ = 0;                                  // 9 x [128 heads x 64 dims]
constexpr uint32_t kOffRingS = kQChunks * kChunk;              // kRingS x [128 keys x 64 dims]
constexpr uint32_t kOffSP = kOffRingS + kRingS * kChunk;       // P staging: 2 x [128 heads x 64 keys]
constexpr uint32_t kOffSF = kOffSP + 2 * kChunk;               // rescale factor staging: 128 floats
constexpr int kRowSlots = 2;                                   // tiles of row tables in flight
constexpr uint32_t kOffRows = kOffSF + kHeads * 4;             // 2 x 128 physical rows (int32)
constexpr uint32_t kOffMask = kOffRows + kRowSlots * kTile * 4; // 2 x 4 key-valid words
// value CTA layout
constexpr int kPBufs = 2;                                      // P buffers (tiles) in flight
constexpr int kRingV = 5;
constexpr uint32_t kOffP = 0;                                  // kPBufs x (2 x [128 heads x 64 keys])
constexpr uint32_t kOffRingV = kPBufs * 2 * kChunk;            // kRingV x (2 x [128 keys x 64 dims])
constexpr uint32_t kOffF = kOffRingV + kRingV * kGroup;        // kPBufs x 128 floats
constexpr int kEpiBufs = 4;  // epilogue staging: 4 KB boxes per epilogue warp, in the value ring
static_assert(8 * kEpiBufs * 4096 <= kRingV * kGroup, "epilogue staging fits the value ring");
// FP8 KV cache (e4m3 rows of 576 codes, one fp32 scale per row and tile of
// 128 entries): the score CTA dequantises each gathered chunk into an f16
// ring slot itself, the value CTA's converters dequantise staged groups.
constexpr int kKvTiles = 5;                                    // scales per 576-entry row
// FP4 e2m1 cache: 288 bytes of codes per 576-entry row and one fp32 scale per
// 16-entry block (36 per row); its staging needs less room than the FP8
// cache's, in the same slots.
constexpr int kKvBlocks4 = 36;
constexpr int kRing8 = 3;                                      // score: f16 chunk slots
constexpr int kStg8 = 3;                                       // score: fp8 chunk staging slots
static_assert(kStg8 <= 5 && kRing8 <= 5, "barrier arrays");
constexpr uint32_t kStgBytes8 = kTile * 64;                    // 128 keys x 64 codes
constexpr uint32_t kOffRing8 = kQChunks * kChunk;
constexpr uint32_t kOffStg8 = kOffRing8 + kRing8 * kChunk;
constexpr uint32_t kOffScl8 = kOffStg8 + kStg8 * kStgBytes8;   // [row slot][tile][128] fp32
constexpr uint32_t kOffRows8 = kOffScl8 + kRowSlots * kKvTiles * kTile * 4;
constexpr uint32_t kOffMask8 = kOffRows8 + kRowSlots * kTile * 4;
constexpr int kVStg8 = 3;                                      // value: fp8 group staging slots
constexpr int kVRing8 = 3;                                     // value: f16 group slots
constexpr uint32_t kVStgBytes8 = kTile * 128 + kTile * 4;      // codes + one scale per key
constexpr uint32_t kOffVStg8 = kPBufs * 2 * kChunk;
constexpr uint32_t kOffVRing8 = (kOffVStg8 + kVStg8 * kVStgBytes8 + 1023u) & ~1023u;
constexpr uint32_t kOffF8 = kOffVRing8 + kVRing8 * kGroup;
static_assert(kOffVStg8 == kOffRingV && kOffF8 - kOffVStg8 >= 8 * kEpiBufs * 4096,
              "epilogue staging fits the FP8 value buffers");
static_assert(kTile * (32 + 16) <= kStgBytes8 && kTile * (64 + 32) <= kVStgBytes8,
              "FP4 codes and block scales fit the FP8 staging slots");
// both
constexpr uint32_t kOffBar = std::max(
    std::max(kOffF + kPBufs * kHeads * 4, kOffMask + kRowSlots * 16),
    std::max(kOffF8 + kPBufs * kHeads * 4, kOffMask8 + kRowSlots * 16));
constexpr uint32_t kBarArea = 416;                             // mbarriers + TMEM base word
constexpr uint32_t kSmemBytes = kOffBar + kBarArea + 1024;     // + alignment slack
static_assert(kOffMask + kRowSlots * 16 <= kOffBar, "score scratch overlaps the barriers");
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

// mbarriers: one array at kOffBar in both CTAs (a barrier that the other CTA
// arrives on lives at the same offset in both)
enum : int {
    B_FULL = 0,     // [ring] copies of a ring slot landed (cp.async arrivals)
    B_EMPTY = 5,    // [ring] ring slot consumed (MMA commit)
    B_CONV = 10,    // [ring] value: group converted to f16
    B_SFULL = 15,   // [2] score: S of a tile complete
    B_SEMPTY = 17,  // [2] score: softmax done with an S buffer
    B_MASK = 19,    // [2] score: row table and key-valid words of a tile written
    B_QREADY = 23,  // score: query resident
    B_PEMPTY = 24,  // [3] score: value CTA finished P.V from a P buffer (remote commit)
    B_PFULL = 27,   // [3] value: P and factors of a tile written (remote arrivals)
    B_OCORR = 30,   // value: O rescaled (if needed) for the next tile
    B_PVDONE = 31,  // value: P.V of a tile complete
    B_FINAL = 32,   // value: row sums l written (remote arrivals)
    B_MEMPTY = 33,  // [2] score: loaders and softmax done with a tile's row table / words
    B_QCONV = 35,   // score, FP8 cache: query converted to f16
    B_F16E = 36,    // [3] value, FP8 cache: f16 group slot consumed (MMA commit)
    B_STF8 = 39,    // [kStg8] score, FP8 cache: staging slot landed (cp.async arrivals)
    B_STE8 = 44,    // [kStg8] score, FP8 cache: staging slot dequantised
    B_SPFREE = 49,  // score, bf16 cache: P staging copied out (remote arrival per tile)
    B_COUNT = 50
};
constexpr uint32_t kTmemSlot = 8 * 50;  // byte offset of the TMEM base within the barrier area
static_assert(B_COUNT * 8 <= (int)kTmemSlot && kTmemSlot + 4 <= kBarArea, "barrier area");
static_assert(kRingS <= 5 && kRingV <= 5, "ring barrier arrays");
static_assert(kOffSP % 1024 == 0, "P staging keeps the 128-byte swizzle atoms of the P buffers");

// 2^x with the hardware approximation (ex2.approx: ~2 ulp, subnormal
// results flushed to zero), ample for a softmax whose weights are rounded to
// f16.
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// two bf16 (low, high) -> two f16
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w)
{
    return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// true when either f16 half is infinite or NaN (exponent field all ones): a
// value outside the f16 range met the conversion
__device__ __forceinline__ bool f16x2_nonfinite(uint32_t w)
{
    return (w & 0x7C00u) == 0x7C00u || (w & 0x7C000000u) == 0x7C000000u;
}

// Two e4m3 codes (low byte first) times a scale, as two f16 (low, high).
// The decode is exact; the product is rounded once to f16.
__device__ __forceinline__ uint32_t e4m3x2_scaled_f16x2(uint32_t codes2, float sc)
{
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)codes2, __NV_E4M3);
    return pack_f16x2(__half2float(__ushort_as_half(h.x)) * sc,
                      __half2float(__ushort_as_half(h.y)) * sc);
}

// 16 codes (one 16-byte unit) -> 16 f16 in two 16-byte units at dst0, dst1;
// returns true if a product left the f16 range.
__device__ __forceinline__ bool dequant16(uint4 c, float sc, uint32_t dst0, uint32_t dst1)
{
    const uint32_t a0 = e4m3x2_scaled_f16x2(c.x & 0xFFFFu, sc), a1 = e4m3x2_scaled_f16x2(c.x >> 16, sc),
                   a2 = e4m3x2_scaled_f16x2(c.y & 0xFFFFu, sc), a3 = e4m3x2_scaled_f16x2(c.y >> 16, sc),
                   b0 = e4m3x2_scaled_f16x2(c.z & 0xFFFFu, sc), b1 = e4m3x2_scaled_f16x2(c.z >> 16, sc),
                   b2 = e4m3x2_scaled_f16x2(c.w & 0xFFFFu, sc), b3 = e4m3x2_scaled_f16x2(c.w >> 16, sc);
    st_shared_v4(dst0, a0, a1, a2, a3);
    st_shared_v4(dst1, b0, b1, b2, b3);
    return f16x2_nonfinite(a0) | f16x2_nonfinite(a1) | f16x2_nonfinite(a2) |
           f16x2_nonfinite(a3) | f16x2_nonfinite(b0) | f16x2_nonfinite(b1) |
           f16x2_nonfinite(b2) | f16x2_nonfinite(b3);
}

__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
    return v;
}

// One byte of two e2m1 codes (even entry in the low nibble) times a block
// scale, as two f16 (low, high): the decode is exact, the product is rounded
// once to f16.
__device__ __forceinline__ uint32_t e2m1x2_scaled_f16x2(uint32_t byte, float sc)
{
    return pack_f16x2(e2m1_to_float(byte & 15u) * sc, e2m1_to_float((byte >> 4) & 15u) * sc);
}

// One byte of two e2m1 codes -> two f16 (exact), by the hardware conversion.
__device__ __forceinline__ __half2 e2m1x2_to_half2(uint32_t byte)
{
    const __half2_raw r = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)byte, __NV_E2M1);
    return *reinterpret_cast<const __half2 *>(&r);
}

// One 16-entry e2m1 block (8 bytes) times its scale -> 16 f16 in two 16-byte
// units at dst0, dst1; returns true if a product left the f16 range.  When
// the scale is an f16 value (an NVFP4 block scale is an e4m3 value, so it
// is), one packed f16 multiply rounds the exact product once -- the same
// result as the fp32 product rounded to f16.
__device__ __forceinline__ bool dequant16_e2m1(uint2 c, float sc, uint32_t dst0, uint32_t dst1)
{
    uint32_t w[8];
    const __half hs = __float2half_rn(sc);
    if (__half2float(hs) == sc) {
        const __half2 s2 = __half2half2(hs);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const __half2 a = __hmul2(e2m1x2_to_half2((c.x >> (8 * i)) & 0xFFu), s2);
            const __half2 b2 = __hmul2(e2m1x2_to_half2((c.y >> (8 * i)) & 0xFFu), s2);
            w[i] = *reinterpret_cast<const uint32_t *>(&a);
            w[4 + i] = *reinterpret_cast<const uint32_t *>(&b2);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            w[i] = e2m1x2_scaled_f16x2((c.x >> (8 * i)) & 0xFFu, sc);
            w[4 + i] = e2m1x2_scaled_f16x2((c.y >> (8 * i)) & 0xFFu, sc);
        }
    }
    st_shared_v4(dst0, w[0], w[1], w[2], w[3]);
    st_shared_v4(dst1, w[4], w[5], w[6], w[7]);
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 8; i++)
        bad |= f16x2_nonfinite(w[i]);
    return bad;
}

// 16 bytes of bf16 -> f16 in place.
__device__ __forceinline__ void to_f16_inplace(uint32_t a)
{
    const uint4 x = ld_shared_v4(a);
    st_shared_v4(a, bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y), bf16x2_to_f16x2(x.z),
                 bf16x2_to_f16x2(x.w));
}

// The same, folding the inputs' magnitude bits into `mag` (a per-half
// maximum), which bf16_beyond_f16 tests once at the end.
__device__ __forceinline__ void to_f16_inplace(uint32_t a, uint32_t &mag)
{
    const uint4 x = ld_shared_v4(a);
    st_shared_v4(a, bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y), bf16x2_to_f16x2(x.z),
                 bf16x2_to_f16x2(x.w));
    mag = __vmaxu2(mag, __vmaxu2(__vmaxu2(x.x & 0x7FFF7FFFu, x.y & 0x7FFF7FFFu),
                                 __vmaxu2(x.z & 0x7FFF7FFFu, x.w & 0x7FFF7FFFu)));
}

// A bf16 magnitude of 2^16 or more (bits 0x4780 and up, infinities and NaN
// included) has no f16 form; every smaller bf16 does (the largest bf16 below
// 2^16 is 65280 <= 65504).  `mag`: per-half maxima of magnitude bits.
__device__ __forceinline__ bool bf16_beyond_f16(uint32_t mag)
{
    return (mag & 0xFFFFu) >= 0x4780u || (mag >> 16) >= 0x4780u;
}

// 4-byte global -> shared copy, asynchronous like cp_async_16 (zeros when
// src_bytes = 0).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// 16-byte global -> shared copy that lands asynchronously; src_bytes = 0
// writes zeros without reading.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// The mbarrier receives one arrival once all of this thread's earlier
// cp.async copies have landed (its expected count includes these arrivals).
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Loader state of one thread: physical rows of its keys (kr0 + 16 i) for
// the even and the odd tile, and the lookahead: index-list values of tiles
// t+1 .. t+3 and block-table entries of tiles t+1, t+2.  The lookups are
// plain loads that complete behind the thread's in-flight copies, so they are
// issued two to three tiles before they are needed.
constexpr int kR = kRowsPerLoader;
struct LoaderState {
    int rb0[kR], rb1[kR];  // physical rows (< 2^31), -1 = zero row
    int sv1[kR], bk1[kR], sv2[kR], bk2[kR], sv3[kR];
    int have_tile;
};

__device__ __forceinline__ void load_idx(const int32_t *idx, int r, int k_top, int tile, int T,
                                         int n_valid, int kr0, int (&sv)[kR])
{
#pragma unroll
    for (int i = 0; i < kR; i++) {
        const int j = tile * kTile + kr0 + (kTile / kR) * i;
        sv[i] = (tile < T && j < n_valid) ? __ldg(idx + (int64_t)r * k_top + j) : -1;
    }
}

__device__ __forceinline__ void load_blk(const si_batch &b, int seq, int pos, const int (&sv)[kR],
                                         int (&bk)[kR])
{
#pragma unroll
    for (int i = 0; i < kR; i++) {
        bk[i] = -1;
        const int sp = sv[i];
        if (sp >= 0 && sp <= pos && (unsigned)seq < (unsigned)b.n_seq &&
            sp / b.page_size < b.max_blocks)
            bk[i] = __ldg(b.block_table + (int64_t)seq * b.max_blocks + sp / b.page_size);
    }
}

__device__ __forceinline__ void loader_init(LoaderState &ls, const si_batch &b, const int32_t *idx,
                                            int r, int k_top, int T, int n_valid, int seq, int pos,
                                            int kr0)
{
    ls.have_tile = -1;
    load_idx(idx, r, k_top, 0, T, n_valid, kr0, ls.sv1);
    load_idx(idx, r, k_top, 1, T, n_valid, kr0, ls.sv2);
    load_idx(idx, r, k_top, 2, T, n_valid, kr0, ls.sv3);
    load_blk(b, seq, pos, ls.sv1, ls.bk1);
    load_blk(b, seq, pos, ls.sv2, ls.bk2);
}

// Makes `tile` current: row offsets from the lookahead (-1: zero row).
__device__ __forceinline__ void activate_tile(LoaderState &ls, const si_batch &b, int pos, int u,
                                              unsigned int *st, int tile)
{
    ls.have_tile = tile;
#pragma unroll
    for (int i = 0; i < kR; i++) {
        const int sp = ls.sv1[i], bk = ls.bk1[i];
        bool ok = false;
        if (sp >= 0 && sp <= pos) {
            ok = (unsigned)bk < (unsigned)b.n_blocks;
            if (!ok && u == 0)
                raise_flag(st, SI_DEVFLAG_BAD_BLOCK);
        } else if (sp != -1 && u == 0) {
            raise_flag(st, SI_DEVFLAG_BAD_INDEX);
        }
        const int off = ok ? bk * b.page_size + sp % b.page_size : -1;
        if (tile & 1)
            ls.rb1[i] = off;
        else
            ls.rb0[i] = off;
    }
}

// Shifts the lookahead by one tile (issues the dependent lookups of the next
// tiles; they complete while this tile streams).
__device__ __forceinline__ void advance_lookahead(LoaderState &ls, const si_batch &b,
                                                  const int32_t *idx, int r, int k_top, int T,
                                                  int n_valid, int seq, int pos, int kr0, int tile)
{
#pragma unroll
    for (int i = 0; i < kR; i++) {
        ls.sv1[i] = ls.sv2[i];
        ls.bk1[i] = ls.bk2[i];
        ls.sv2[i] = ls.sv3[i];
    }
    load_blk(b, seq, pos, ls.sv2, ls.bk2);
    load_idx(idx, r, k_top, tile + 3, T, n_valid, kr0, ls.sv3);
}

// This thread's copies of dim chunk c (16-byte unit u of its key rows) of
// the current tile into the 16 KB chunk buffer at `dst`.
__device__ __forceinline__ void issue_chunk(const LoaderState &ls, uint32_t dst, const uint8_t *kv,
                                            int64_t row_bytes, int tile, int c, int kr0, int u)
{
    const bool odd = tile & 1;
#pragma unroll
    for (int i = 0; i < kR; i++) {
        const int row = odd ? ls.rb1[i] : ls.rb0[i];
        const uint8_t *src = row >= 0 ? kv + (int64_t)row * row_bytes + c * 128 + u * 16 : kv;
        cp_async_16(dst + sw128_offset(kr0 + (kTile / kR) * i, u), src, row >= 0 ? 16u : 0u);
    }
}

// KVT: the cache format -- 0 bf16 rows; 1 e4m3 codes with one fp32 scale
// per row and 128-entry tile; 2 e2m1 codes (two per byte) with one fp32 scale
// per row and 16-entry block.  The two quantised formats share the
// dequantising pipeline (KV8 below) and differ only in how a gathered piece
// of codes and scales becomes f16.
template <int KVT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
k_attn_tc(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
          si_batch b, si_attention at, const int32_t *idx, int k_top, si_dtype out_dtype,
          float *lse, int n_split, float *part_ml, unsigned int *st)
{
    constexpr bool KV8 = KVT != 0;  // a quantised cache, dequantised to f16
    constexpr bool KV4 = KVT == 2;  // ... from e2m1 codes
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - smem_u32(smem_raw));
    uint64_t *bars = reinterpret_cast<uint64_t *>(gbase + kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + kOffBar + kTmemSlot);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_rank();   // 0: score CTA, 1: value CTA
    const bool score_cta = rank == 0;
    // Cluster c handles row r = c / n_split and its key tiles
    // [t0, t1) of split sp = c % n_split (all of them when n_split is 1).
    const int cl = blockIdx.x >> 1;
    const int r = cl / n_split, sp = cl % n_split;
    const int pos = __ldg(b.q_pos + r), seq = __ldg(b.q_seq + r);
    const int n_row = max(0, min(k_top, pos + 1));
    const int T_row = (n_row + kTile - 1) / kTile;
    const int t0 = (int)((int64_t)T_row * sp / n_split);
    const int T = (int)((int64_t)T_row * (sp + 1) / n_split) - t0;  // key tiles of this split
    const int n_valid = max(0, min(n_row - t0 * kTile, T * kTile));
    const int32_t *idx_s = idx + (int64_t)r * k_top + (int64_t)t0 * kTile;
    const bool split = n_split > 1;

    if (tid == 0) {
        for (int i = 0; i < 5; i++) {
            // FP8 score ring slots are filled by the 128 dequantising threads
            mbar_init(bars + B_FULL + i, (KV8 && score_cta) ? kLoaders / 2 : kLoaders);
            // FP8 value staging is released by the converters, rings by the MMA
            mbar_init(bars + B_EMPTY + i, (KV8 && !score_cta) ? kConverters : 1);
            mbar_init(bars + B_CONV + i, kConverters);
        }
        for (int i = 0; i < kVRing8; i++)
            mbar_init(bars + B_F16E + i, 1);
        for (int i = 0; i < kStg8; i++) {
            mbar_init(bars + B_STF8 + i, kLoaders / 2);
            mbar_init(bars + B_STE8 + i, kLoaders / 2);
        }
        mbar_init(bars + B_QCONV, kSoftmax);
        for (int i = 0; i < 2; i++) {
            mbar_init(bars + B_SFULL + i, 1);
            mbar_init(bars + B_SEMPTY + i, kSoftmax);
        }
        for (int i = 0; i < kPBufs; i++) {
            mbar_init(bars + B_PEMPTY + i, 1);
            // bf16 cache: one arrival with the bytes of the bulk copies;
            // FP8 cache: remote arrivals of the softmax threads
            mbar_init(bars + B_PFULL + i, KV8 ? kSoftmax : 1);
        }
        for (int i = 0; i < kRowSlots; i++) {
            mbar_init(bars + B_MASK + i, 32);
            mbar_init(bars + B_MEMPTY + i, kSoftmax + kLoaders);
        }
        mbar_init(bars + B_QREADY, 1);
        mbar_init(bars + B_SPFREE, 1);
        mbar_init(bars + B_OCORR, kHeads);
        mbar_init(bars + B_PVDONE, 1);
        mbar_init(bars + B_FINAL, kHeads);
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(tmem_slot, 512u);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // both CTAs' barriers exist before any cross-CTA arrival
    const uint32_t tmem = *tmem_slot;
    if (score_cta && tid == 0) {
        // query: nine tensor copies of [128 heads x 64 dims], SW128 K-major
        mbar_arrive_expect_tx(bars + B_QREADY, kQChunks * kChunk);
        for (int c = 0; c < kQChunks; c++)
            tma_load_2d(base + kOffQ + c * kChunk, &qmap, c * 128, r * kHeads, bars + B_QREADY);
    }
    // The index list comes from the previous kernel of the stream (Top-K); all
    // set-up above overlaps its tail.
    griddep_wait();

    const uint8_t *kv = static_cast<const uint8_t *>(at.k.data);
    const int64_t row_bytes = KV4 ? at.k.row_stride / 2 : at.k.row_stride * (KV8 ? 1 : 2);
    // value-CTA buffers as seen from the score CTA
    const uint32_t peer_p = mapa_shared(base + kOffP, 1);
    const uint32_t peer_f = mapa_shared(base + kOffF, 1);
    const uint32_t peer_pfull = mapa_shared(smem_u32(bars + B_PFULL), 1);
    const uint32_t peer_final = mapa_shared(smem_u32(bars + B_FINAL), 1);
    // score-CTA barrier as seen from the value CTA
    const uint32_t peer_spfree = mapa_shared(smem_u32(bars + B_SPFREE), 0);

    if (warp < kLoaderWarps) {
        // -------------------------------------------------------------- loaders
        // Thread t owns 16-byte unit u = t & 7 of key rows (t >> 3) + 32 i.
        const int u = tid & 7, kr0 = tid >> 3;
        LoaderState ls;
        if (KV8 && score_cta) {
            // FP8 cache.  Warps 0..3 gather: per dim chunk, thread i copies the
            // 16-code parts (i & 3) of keys (i >> 2) + 32 m, m < 4, into an fp8
            // staging slot.  Warps 4..7 dequantise the same pieces of each
            // landed staging slot into the chunk's f16 ring slot.
            const int li = tid & 127, part = li & 3, k0 = li >> 2;
            const int *rows = reinterpret_cast<const int *>(gbase + kOffRows8);
            const float *scl = reinterpret_cast<const float *>(gbase + kOffScl8);
            const int n_chunks = kQChunks * T;
            if (warp < kLoaderWarps / 2) {
                int rw[4] = {-1, -1, -1, -1};
                int have_tile = -1;
                for (int g = 0; g < n_chunks; g++) {
                    const int tile = g / kQChunks, c = g % kQChunks, s8 = g % kStg8;
                    if (g >= kStg8 &&
                        !mbar_wait(bars + B_STE8 + s8, (uint32_t)((g / kStg8) - 1) & 1, st))
                        break;
                    if (tile > have_tile) {
                        const int rs = tile % kRowSlots;
                        if (!mbar_wait(bars + B_MASK + rs, (uint32_t)(tile / kRowSlots) & 1, st))
                            break;
                        have_tile = tile;
#pragma unroll
                        for (int m = 0; m < 4; m++)
                            rw[m] = rows[rs * kTile + k0 + 32 * m];
                        mbar_arrive(bars + B_MEMPTY + rs);
                    }
                    if constexpr (KV4) {
                        // per key: the chunk's 32 bytes of codes (units 0, 1)
                        // and its four 16-entry block scales (unit 2)
                        const uint32_t sc0 = base + kOffStg8 + s8 * kStgBytes8;
#pragma unroll
                        for (int m = 0; m < 4; m++) {
                            const int key = k0 + 32 * m, r = rw[m];
                            if (part < 2)
                                cp_async_16(sc0 + key * 32 + part * 16,
                                            r >= 0 ? kv + (int64_t)r * row_bytes + c * 32 + part * 16
                                                   : kv,
                                            r >= 0 ? 16u : 0u);
                            else if (part == 2)
                                cp_async_16(sc0 + kTile * 32 + key * 16,
                                            r >= 0 ? fscale(at.k.scale) + (int64_t)r * kKvBlocks4 + 4 * c
                                                   : fscale(at.k.scale),
                                            r >= 0 ? 16u : 0u);
                        }
                    } else {
                        const uint32_t sdst = base + kOffStg8 + s8 * kStgBytes8 + part * 16;
                        const int64_t col = c * 64 + part * 16;
#pragma unroll
                        for (int m = 0; m < 4; m++)
                            cp_async_16(sdst + (k0 + 32 * m) * 64,
                                        rw[m] >= 0 ? kv + (int64_t)rw[m] * row_bytes + col : kv,
                                        rw[m] >= 0 ? 16u : 0u);
                    }
                    cp_async_arrive(bars + B_STF8 + s8);
                }
            } else {
                bool range = false;
                for (int g = 0; g < n_chunks; g++) {
                    const int tile = g / kQChunks, c = g % kQChunks, rs = tile % kRowSlots;
                    const int s8 = g % kStg8, slot = g % kRing8;
                    // the tile's scales: its row-table phase (already complete, and
                    // not yet reusable before this group's MEMPTY arrival)
                    if ((c == 0 &&
                         !mbar_wait(bars + B_MASK + rs, (uint32_t)(tile / kRowSlots) & 1, st)) ||
                        !mbar_wait(bars + B_STF8 + s8, (uint32_t)(g / kStg8) & 1, st) ||
                        (g >= kRing8 &&
                         !mbar_wait(bars + B_EMPTY + slot, (uint32_t)((g / kRing8) - 1) & 1, st)))
                        break;
                    const uint32_t dst = base + kOffRing8 + slot * kChunk;
                    if constexpr (KV4) {
                        // one 16-entry block (8 bytes of codes) and its scale
                        const uint32_t sc0 = base + kOffStg8 + s8 * kStgBytes8;
                        const float *bsc = reinterpret_cast<const float *>(
                            gbase + kOffStg8 + s8 * kStgBytes8 + kTile * 32);
#pragma unroll
                        for (int m = 0; m < 4; m++) {
                            const int key = k0 + 32 * m;
                            range |= dequant16_e2m1(ld_shared_v2(sc0 + key * 32 + part * 8),
                                                    bsc[key * 4 + part],
                                                    dst + sw128_offset(key, 2 * part),
                                                    dst + sw128_offset(key, 2 * part + 1));
                        }
                    } else {
                        const uint32_t ssrc = base + kOffStg8 + s8 * kStgBytes8 + part * 16;
                        const float *sc_t = scl + (rs * kKvTiles + c / 2) * kTile;
#pragma unroll
                        for (int m = 0; m < 4; m++) {
                            const int key = k0 + 32 * m;
                            range |= dequant16(ld_shared_v4(ssrc + key * 64), sc_t[key],
                                               dst + sw128_offset(key, 2 * part),
                                               dst + sw128_offset(key, 2 * part + 1));
                        }
                    }
                    fence_async_smem();
                    mbar_arrive(bars + B_FULL + slot);
                    mbar_arrive(bars + B_STE8 + s8);
                    if (c == kQChunks - 1)
                        mbar_arrive(bars + B_MEMPTY + rs);  // done with the tile's scales
                }
                if (range)
                    raise_flag(st, SI_DEVFLAG_RANGE);
            }
        } else if (score_cta) {
            // physical rows come from the row table the row warp fills
            const int *rows = reinterpret_cast<const int *>(gbase + kOffRows);
            ls.have_tile = -1;
            const int n_chunks = kQChunks * T;
            for (int g = 0; g < n_chunks; g++) {
                const int slot = g % kRingS, tile = g / kQChunks, c = g % kQChunks;
                if (g >= kRingS &&
                    !mbar_wait(bars + B_EMPTY + slot, (uint32_t)((g / kRingS) - 1) & 1, st))
                    break;
                if (tile > ls.have_tile) {
                    const int rs = tile % kRowSlots;
                    if (!mbar_wait(bars + B_MASK + rs, (uint32_t)(tile / kRowSlots) & 1, st))
                        break;
                    ls.have_tile = tile;
#pragma unroll
                    for (int i = 0; i < kR; i++) {
                        const int row = rows[rs * kTile + kr0 + (kTile / kR) * i];
                        if (tile & 1)
                            ls.rb1[i] = row;
                        else
                            ls.rb0[i] = row;
                    }
                    mbar_arrive(bars + B_MEMPTY + rs);
                }
                issue_chunk(ls, base + kOffRingS + slot * kChunk, kv, row_bytes, tile, c, kr0, u);
                cp_async_arrive(bars + B_FULL + slot);
            }
        } else if (KV8) {
            // value CTA, FP8 cache: unit u of group j's 128 codes per key into
            // a staging slot; lane u == 0 also copies its keys' scales of tile j
            loader_init(ls, b, idx_s, 0, k_top, T, n_valid, seq, pos, kr0);
            const float *kscale = fscale(at.k.scale);
            const int n_groups = kVGroups * T;
            for (int g = 0; g < n_groups; g++) {
                const int slot = g % kVStg8, tile = g / kVGroups, j = g % kVGroups;
                if (g >= kVStg8 &&
                    !mbar_wait(bars + B_EMPTY + slot, (uint32_t)((g / kVStg8) - 1) & 1, st))
                    break;
                if (tile > ls.have_tile) {
                    activate_tile(ls, b, pos, u, st, tile);
                    advance_lookahead(ls, b, idx_s, 0, k_top, T, n_valid, seq, pos, kr0, tile);
                }
                const uint32_t dst = base + kOffVStg8 + slot * kVStgBytes8;
                const bool odd = tile & 1;
#pragma unroll
                for (int i = 0; i < kR; i++) {
                    const int key = kr0 + (kTile / kR) * i;
                    const int row = odd ? ls.rb1[i] : ls.rb0[i];
                    if constexpr (KV4) {
                        // per key: 64 bytes of codes (units 0..3) and the
                        // group's eight 16-entry block scales (units 4, 5)
                        if (u < 4)
                            cp_async_16(dst + key * 64 + u * 16,
                                        row >= 0 ? kv + (int64_t)row * row_bytes + j * 64 + u * 16
                                                 : kv,
                                        row >= 0 ? 16u : 0u);
                        else if (u < 6)
                            cp_async_16(dst + kTile * 64 + key * 32 + (u - 4) * 16,
                                        row >= 0 ? kscale + (int64_t)row * kKvBlocks4 + 8 * j +
                                                       4 * (u - 4)
                                                 : kscale,
                                        row >= 0 ? 16u : 0u);
                    } else {
                        cp_async_16(dst + key * 128 + u * 16,
                                    row >= 0 ? kv + (int64_t)row * row_bytes + j * 128 + u * 16
                                             : kv,
                                    row >= 0 ? 16u : 0u);
                        if (u == 0)
                            cp_async_4(dst + kTile * 128 + key * 4,
                                       row >= 0 ? kscale + (int64_t)row * kKvTiles + j : kscale,
                                       row >= 0 ? 4u : 0u);
                    }
                }
                cp_async_arrive(bars + B_FULL + slot);
            }
        } else {
            loader_init(ls, b, idx_s, 0, k_top, T, n_valid, seq, pos, kr0);
            const int n_groups = kVGroups * T;
            for (int g = 0; g < n_groups; g++) {
                const int slot = g % kRingV, tile = g / kVGroups, j = g % kVGroups;
                if (g >= kRingV &&
                    !mbar_wait(bars + B_EMPTY + slot, (uint32_t)((g / kRingV) - 1) & 1, st))
                    break;
                if (tile > ls.have_tile) {
                    activate_tile(ls, b, pos, u, st, tile);
                    advance_lookahead(ls, b, idx_s, 0, k_top, T, n_valid, seq, pos, kr0, tile);
                }
                const uint32_t dst = base + kOffRingV + slot * kGroup;
                issue_chunk(ls, dst, kv, row_bytes, tile, 2 * j, kr0, u);
                issue_chunk(ls, dst + kChunk, kv, row_bytes, tile, 2 * j + 1, kr0, u);
                cp_async_arrive(bars + B_FULL + slot);
            }
        }
        cp_async_wait_all();  // nothing may land after the block has moved on
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------------ MMA
        if (score_cta) {
            // bf16 (or, for an FP8 cache, f16 query and dequantised keys), K-major
            const uint32_t idesc = idesc_f16(kHeads, kTile, KV8 ? 0 : 1, 0, 0);
            constexpr int kSlots = KV8 ? kRing8 : kRingS;
            const uint32_t ring = base + (KV8 ? kOffRing8 : kOffRingS);
            bool ok = mbar_wait(bars + (KV8 ? B_QCONV : B_QREADY), 0, st);
            const int n_chunks = kQChunks * T;
            for (int g = 0; ok && g < n_chunks; g++) {
                const int slot = g % kSlots, tile = g / kQChunks, c = g % kQChunks;
                // S buffer of this tile must be free (softmax read S of tile - 2)
                if (c == 0 && tile >= 2 &&
                    !mbar_wait(bars + B_SEMPTY + (tile & 1), (uint32_t)((tile >> 1) - 1) & 1, st))
                    break;
                if (!mbar_wait(bars + B_FULL + slot, (uint32_t)(g / kSlots) & 1, st))
                    break;
                fence_async_smem();  // landed copies -> tensor core (async proxy)
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t d = tmem + (tile & 1) * kTile;
                    const uint32_t chunk = ring + slot * kChunk;
#pragma unroll
                    for (int kk = 0; kk < 4; kk++) {
                        const uint64_t ad =
                            smem_desc(base + kOffQ + c * kChunk + kk * 32, 16, 1024, kSwizzle128B);
                        const uint64_t bd = smem_desc(chunk + kk * 32, 16, 1024, kSwizzle128B);
                        umma_f16_ss(d, ad, bd, idesc, c > 0 || kk > 0);
                    }
                    umma_commit(bars + B_EMPTY + slot);
                    if (c == kQChunks - 1)
                        umma_commit(bars + B_SFULL + (tile & 1));
                }
                __syncwarp();
            }
        } else {
            // O[:, 128 j .. +128] += P[128 heads x 128 keys] . V_group j
            const uint32_t idesc = idesc_f16(kHeads, 128, 0, 0, 1);  // f16; B (V) MN-major
            bool ok = true;
            for (int t = 0; ok && t < T; t++) {
                const int pb = t % kPBufs;
                if (!mbar_wait_cluster(bars + B_PFULL + pb, (uint32_t)(t / kPBufs) & 1, st) ||
                    !mbar_wait(bars + B_OCORR, (uint32_t)t & 1, st))
                    break;
                fence_async_smem();  // P written by the score CTA -> tensor core
                for (int j = 0; j < kVGroups; j++) {
                    constexpr int kSlots = KV8 ? kVRing8 : kRingV;
                    const int g = t * kVGroups + j, slot = g % kSlots;
                    if (!mbar_wait(bars + B_CONV + slot, (uint32_t)(g / kSlots) & 1, st)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t grp = base + (KV8 ? kOffVRing8 : kOffRingV) + slot * kGroup;
#pragma unroll
                        for (int kk = 0; kk < kTile / 16; kk++) {
                            const uint64_t ad =
                                smem_desc(base + kOffP + pb * 2 * kChunk + (kk >> 2) * kChunk +
                                              (kk & 3) * 32,
                                          16, 1024, kSwizzle128B);
                            const uint64_t bd =
                                smem_desc(grp + kk * 2048, kChunk, 1024, kSwizzle128B);
                            umma_f16_ss(tmem + 128 * j, ad, bd, idesc, t > 0 || kk > 0);
                        }
                        umma_commit(bars + (KV8 ? B_F16E : B_EMPTY) + slot);
                    }
                    __syncwarp();
                }
                if (!ok)
                    break;
                if (lane == 0) {
                    umma_commit(bars + B_PVDONE);
                    umma_commit_multicast(bars + B_PEMPTY + pb, 0x1);  // P buffer free (score CTA)
                }
                __syncwarp();
            }
        }
    } else if (score_cta) {
        if (warp >= kWarpSoft0 && warp < kWarpSoft0 + 8) {
            // ---------------------------------------------------------- softmax
            // Two threads per head (TMEM lane): warps 4..7 take keys 0..63 of
            // each tile, warps 8..11 keys 64..127.  They share the tile
            // maximum through shared memory and keep partial row sums.
            const int quarter = warp & 3, kh = (warp - kWarpSoft0) >> 2;
            const int h = quarter * 32 + lane;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            if constexpr (KV8) {
                // FP8 cache: keys are dequantised to f16, so the query becomes
                // f16 too (one operand type per MMA; exact for |q| >= 2^-14)
                mbar_wait(bars + B_QREADY, 0, st);
                const int st_ = tid - kWarpSoft0 * 32;
                uint32_t mag = 0;
                for (int i = st_; i < (int)(kQChunks * kChunk / 16); i += kSoftmax)
                    to_f16_inplace(base + kOffQ + i * 16, mag);
                if (bf16_beyond_f16(mag))
                    raise_flag(st, SI_DEVFLAG_RANGE);
                fence_async_smem();
                mbar_arrive(bars + B_QCONV);
            }
            const float sl2 = at.softmax_scale * 1.4426950408889634f;  // scale * log2(e)
            const uint32_t *mask =
                reinterpret_cast<const uint32_t *>(gbase + (KV8 ? kOffMask8 : kOffMask));
            // the two threads of a head share TMEM lane h: column 256 + kh is
            // this thread's exchange cell
            const uint32_t xmine = tmem + 256 + kh + lane_off, xother = tmem + 257 - kh + lane_off;
            float m_used = -INFINITY;  // exponent reference (log2 units)
            float l = 0.f;             // this half's row sum
            bool ok = true;
            // FP8 cache: P goes to the value CTA as remote stores, announced
            // one step late (after the next tile's first pass), so that the
            // cluster-scope release does not wait on the stores' round trip.
            // bf16 cache: P is staged locally and handed over by bulk copies.
            const bool issuer = tid == kWarpSoft0 * 32;  // issues the bulk copies
            const uint32_t sp = base + kOffSP;
            int unpublished = -1;  // tile whose P is written but not yet announced
            auto publish = [&](int pt) {
                fence_async_cluster();
                mbar_arrive_remote(peer_pfull + (pt % kPBufs) * 8);
            };
            for (int t = 0; t < T; t++) {
                const int sb = t & 1;
                const int rs = t % kRowSlots;
                const bool got =
                    mbar_wait(bars + B_MASK + rs, (uint32_t)(t / kRowSlots) & 1, st) &&
                    mbar_wait(bars + B_SFULL + sb, (uint32_t)(t >> 1) & 1, st);
                // all 256 threads take the same branch (bar.red over the flag)
                if (bar_sync_or(1, kSoftmax, !got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t mw0 = mask[rs * 4 + 2 * kh], mw1 = mask[rs * 4 + 2 * kh + 1];
                mbar_arrive(bars + B_MEMPTY + rs);
                // pass 1: maximum of this half's valid logits, then of the tile
                float tmax = -INFINITY;
#pragma unroll 1
                for (int q = 0; q < 2; q++) {
                    uint32_t v[32];
                    tmem_ld32(tmem + sb * kTile + 64 * kh + lane_off + 32 * q, v);
                    tmem_wait_ld();
                    const uint32_t mwq = q ? mw1 : mw0;
#pragma unroll
                    for (int i = 0; i < 32; i++)
                        if (mwq & (1u << i))
                            tmax = fmaxf(tmax, __uint_as_float(v[i]) * sl2);
                }
                tmem_st1(xmine, __float_as_uint(tmax));
                tmem_wait_st();
                tc_fence_before();
                bar_sync_or(1, kSoftmax, false);
                tc_fence_after();
                tmax = fmaxf(tmax, __uint_as_float(tmem_ld1(xother)));
                tmem_wait_ld();
                float f = 1.f;  // factor the value CTA applies to O before this tile
                if (tmax > m_used + kRescaleThreshold) {
                    f = ex2(m_used - tmax);
                    l *= f;
                    m_used = tmax;
                }
                if (unpublished >= 0) {
                    publish(unpublished);
                    unpublished = -1;
                }
                // the value CTA's P buffer pb is free once its P.V of tile
                // t - kPBufs is done; the bf16 staging once the value CTA has
                // seen tile t - 1's copies land.  The bar.red also orders this
                // tile's reads of the exchange cell before the next tile's
                // writes.
                const int pb = t % kPBufs;
                bool free_ =
                    t < kPBufs ||
                    mbar_wait_cluster(bars + B_PEMPTY + pb, (uint32_t)((t / kPBufs) - 1) & 1, st);
                if (!KV8 && issuer && t >= 1)
                    free_ = free_ &&
                            mbar_wait_cluster(bars + B_SPFREE, (uint32_t)(t - 1) & 1, st);
                if (bar_sync_or(1, kSoftmax, !free_)) {
                    ok = false;
                    break;
                }
                // pass 2: p = 2^(x - m_used) as f16, chunk kh (this half's 64
                // keys) of the value CTA's P buffer pb (FP8 cache) or of the
                // local staging (bf16 cache)
                const uint32_t pc =
                    KV8 ? peer_p + pb * 2 * kChunk + kh * kChunk : sp + kh * kChunk;
#pragma unroll 1
                for (int q = 0; q < 2; q++) {
                    uint32_t v[32];
                    tmem_ld32(tmem + sb * kTile + 64 * kh + lane_off + 32 * q, v);
                    tmem_wait_ld();
                    if (q == 1) {
                        tc_fence_before();
                        mbar_arrive(bars + B_SEMPTY + sb);  // S buffer sb may be overwritten
                    }
                    const uint32_t mwq = q ? mw1 : mw0;
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float x0 = __uint_as_float(v[i]);
                        const float x1 = __uint_as_float(v[i + 1]);
                        const float p0 = (mwq & (1u << i)) ? ex2(x0 * sl2 - m_used) : 0.f;
                        const float p1 = (mwq & (1u << (i + 1))) ? ex2(x1 * sl2 - m_used) : 0.f;
                        pk[i >> 1] = pack_f16x2(p0, p1);
                        const __half2 pr = *reinterpret_cast<__half2 *>(&pk[i >> 1]);
                        l += __low2float(pr) + __high2float(pr);
                    }
#pragma unroll
                    for (int w = 0; w < 4; w++) {
                        if constexpr (KV8)
                            st_cluster_v4(pc + sw128_offset(h, q * 4 + w), pk[4 * w],
                                          pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
                        else
                            st_shared_v4(pc + sw128_offset(h, q * 4 + w), pk[4 * w],
                                         pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
                    }
                }
                if constexpr (KV8) {
                    if (kh == 0)
                        st_cluster_f32(peer_f + (pb * kHeads + h) * 4, f);
                    unpublished = t;
                } else {
                    // staged P and factors -> the value CTA's P buffer pb and
                    // factor slot pb; its barrier counts the bytes
                    if (kh == 0)
                        reinterpret_cast<float *>(gbase + kOffSF)[h] = f;
                    fence_async_smem();  // staging writes -> bulk copy engine
                    bar_sync_or(1, kSoftmax, false);
                    if (issuer) {
                        const uint32_t bar = peer_pfull + pb * 8;
                        mbar_arrive_expect_tx_remote(bar, 2 * kChunk + kHeads * 4);
                        bulk_s2cluster(peer_p + pb * 2 * kChunk, sp, 2 * kChunk, bar);
                        bulk_s2cluster(peer_f + pb * kHeads * 4, base + kOffSF, kHeads * 4, bar);
                    }
                }
            }
            if (unpublished >= 0)
                publish(unpublished);
            // Row sums: combine the halves.  Then wait until the value CTA's
            // P.V of the last (up to) kPBufs tiles is done -- so its commits
            // have landed here before this CTA ends, and F buffer T % kPBufs
            // is free -- and send l.
            tmem_st1(xmine, __float_as_uint(l));
            tmem_wait_st();
            tc_fence_before();
            bar_sync_or(1, kSoftmax, false);
            tc_fence_after();
            l += __uint_as_float(tmem_ld1(xother));
            tmem_wait_ld();
            if (kh == 0) {
                for (int tt = max(0, T - kPBufs); ok && tt < T; tt++)
                    if (!mbar_wait_cluster(bars + B_PEMPTY + tt % kPBufs,
                                           (uint32_t)(tt / kPBufs) & 1, st))
                        ok = false;
                st_cluster_f32(peer_f + ((T % kPBufs) * kHeads + h) * 4, ok ? l : 0.f);
                mbar_arrive_remote(peer_final);
                if (split) {
                    // this split's softmax state, for the combine kernel
                    float *ml = part_ml + ((int64_t)cl * kHeads + h) * 2;
                    ml[0] = (ok && l > 0.f) ? m_used : -INFINITY;
                    ml[1] = ok ? l : 0.f;
                } else if (lse) {
                    lse[(int64_t)r * kHeads + h] =
                        (ok && l > 0.f) ? (m_used + log2f(l)) * 0.6931471805599453f : -INFINITY;
                }
            }
        }
        if (warp == kWarpRows) {
            // ------------------------------------------------- row table, key-valid bits
            // For each tile: the physical row of every selected key (-1: none,
            // the loaders then write zeros) and bit i of word w set when key
            // 32 w + i is valid.  Up to two tiles ahead of its consumers.
            int *rows = reinterpret_cast<int *>(gbase + (KV8 ? kOffRows8 : kOffRows));
            uint32_t *mask = reinterpret_cast<uint32_t *>(gbase + (KV8 ? kOffMask8 : kOffMask));
            float *scl = reinterpret_cast<float *>(gbase + kOffScl8);  // FP8 cache: key scales
            for (int t = 0; t < T; t++) {
                const int rs = t % kRowSlots;
                if (t >= kRowSlots &&
                    !mbar_wait(bars + B_MEMPTY + rs, (uint32_t)((t / kRowSlots) - 1) & 1, st))
                    break;
                int sv[4], blk[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int j = t * kTile + 32 * i + lane;
                    sv[i] = j < n_valid ? __ldg(idx_s + j) : -1;
                }
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    blk[i] = -1;
                    if (sv[i] >= 0 && sv[i] <= pos && (unsigned)seq < (unsigned)b.n_seq &&
                        sv[i] / b.page_size < b.max_blocks)
                        blk[i] = __ldg(b.block_table + (int64_t)seq * b.max_blocks +
                                       sv[i] / b.page_size);
                }
                uint32_t word = 0;
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    bool ok = false;
                    if (sv[i] >= 0 && sv[i] <= pos) {
                        ok = (unsigned)blk[i] < (unsigned)b.n_blocks;
                        if (!ok)
                            raise_flag(st, SI_DEVFLAG_BAD_BLOCK);
                    } else if (sv[i] != -1) {
                        raise_flag(st, SI_DEVFLAG_BAD_INDEX);
                    }
                    const int prow = ok ? blk[i] * b.page_size + sv[i] % b.page_size : -1;
                    rows[rs * kTile + 32 * i + lane] = prow;
                    if constexpr (KV8 && !KV4) {
                        // the key's scales of every 128-entry tile (0 for no key)
#pragma unroll
                        for (int q5 = 0; q5 < kKvTiles; q5++)
                            scl[(rs * kKvTiles + q5) * kTile + 32 * i + lane] =
                                prow >= 0 ? __ldg(fscale(at.k.scale) + (int64_t)prow * kKvTiles + q5) : 0.f;
                    }
                    const uint32_t w = __ballot_sync(0xffffffffu, ok);
                    if (lane == i)
                        word = w;
                }
                if (lane < 4)
                    mask[rs * 4 + lane] = word;
                mbar_arrive(bars + B_MASK + rs);
            }
        }
    } else {
        // value CTA, warps 8..15 and 17
        bool ok = true;
        if (warp >= kWarpQuad + 4) {
            // ------------------------------------------------------- converters
            // Value groups feed the f16 P.V product: rewrite them bf16 -> f16
            // in place once their copies have landed (warps 12..15 and 17).
            const int ct = warp < kWarpMma ? tid - (kWarpQuad + 4) * 32 : 4 * 32 + lane;
            const int n_groups = kVGroups * T;
            bool range = false;  // a value beyond the f16 range met the conversion
            if constexpr (KV8) {
                // FP8 cache: staged codes times the key's scale into the f16
                // group slot (two chunks of [128 keys x 64 dims], SW128), then
                // the staging slot goes back to the loaders
                for (int g = 0; g < n_groups; g++) {
                    const int s8 = g % kVStg8, f = g % kVRing8;
                    if (!mbar_wait(bars + B_FULL + s8, (uint32_t)(g / kVStg8) & 1, st) ||
                        (g >= kVRing8 &&
                         !mbar_wait(bars + B_F16E + f, (uint32_t)((g / kVRing8) - 1) & 1, st)))
                        break;
                    const uint32_t src = base + kOffVStg8 + s8 * kVStgBytes8;
                    const float *ksc = reinterpret_cast<const float *>(
                        gbase + kOffVStg8 + s8 * kVStgBytes8 + kTile * (KV4 ? 64 : 128));
                    const uint32_t dst = base + kOffVRing8 + f * kGroup;
                    for (int i = ct; i < kTile * 8; i += kConverters) {
                        const int key = i >> 3, uu = i & 7;  // 16 codes: dims 16 uu .. 16 uu + 15
                        const uint32_t d0 = dst + (uu >> 2) * kChunk;
                        if constexpr (KV4)
                            range |= dequant16_e2m1(ld_shared_v2(src + key * 64 + uu * 8),
                                                    ksc[key * 8 + uu],
                                                    d0 + sw128_offset(key, 2 * (uu & 3)),
                                                    d0 + sw128_offset(key, 2 * (uu & 3) + 1));
                        else
                            range |= dequant16(ld_shared_v4(src + key * 128 + uu * 16), ksc[key],
                                               d0 + sw128_offset(key, 2 * (uu & 3)),
                                               d0 + sw128_offset(key, 2 * (uu & 3) + 1));
                    }
                    fence_async_smem();
                    mbar_arrive(bars + B_CONV + f);
                    mbar_arrive(bars + B_EMPTY + s8);
                }
            } else
            for (int g = 0; g < n_groups; g++) {
                const int slot = g % kRingV;
                if (!mbar_wait(bars + B_FULL + slot, (uint32_t)(g / kRingV) & 1, st))
                    break;
                const uint32_t src = base + kOffRingV + slot * kGroup;
                // (a value beyond the f16 range becomes inf here and makes O
                // non-finite; the epilogue checks O once per row)
                for (int i = ct; i < (int)(kGroup / 16); i += kConverters)
                    to_f16_inplace(src + i * 16);
                fence_async_smem();
                mbar_arrive(bars + B_CONV + slot);
            }
            if (range)
                raise_flag(st, SI_DEVFLAG_RANGE);
        } else {
            // ------------------------------------------------------ O rescale
            const int h = tid - kWarpQuad * 32;  // head = TMEM lane
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
            const float *fac = reinterpret_cast<const float *>(gbase + kOffF);
            for (int t = 0; t < T; t++) {
                const int pb = t % kPBufs;
                if (!mbar_wait_cluster(bars + B_PFULL + pb, (uint32_t)(t / kPBufs) & 1, st)) {
                    ok = false;
                    break;
                }
                // bf16 cache: tile t's copies have landed, so the score CTA may
                // restage P
                if (!KV8 && h == 0)
                    mbar_arrive_remote(peer_spfree);
                const float f = fac[pb * kHeads + h];
                // P.V of tile t - 1 must be complete before O is touched
                if (t >= 1 && !mbar_wait(bars + B_PVDONE, (uint32_t)(t - 1) & 1, st)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (t >= 1 && f != 1.f) {
#pragma unroll 1
                    for (int q = 0; q < kDv / 32; q++) {
                        uint32_t v[32];
                        tmem_ld32(tmem + lane_off + q * 32, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; i++)
                            v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
                        tmem_st32(tmem + lane_off + q * 32, v);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                mbar_arrive(bars + B_OCORR);
            }
            if (ok && T >= 1 && !mbar_wait(bars + B_PVDONE, (uint32_t)(T - 1) & 1, st))
                ok = false;
            if (!mbar_wait_cluster(bars + B_FINAL, 0, st))
                ok = false;
        }
        if (warp < kWarpMma) {
            // ------------------------------------------------------- epilogue
            // Warps 8..15 (two per TMEM lane quarter) write out = O / l: each
            // warp takes half of its 32 heads' columns, 128-byte column blocks
            // staged in the (now idle) value ring with the 128-byte swizzle and
            // stored by the tensor engine as [32 rows x 128 bytes] boxes.  The
            // bar.red gives every warp the same verdict on the waits above.
            const bool bad = bar_sync_or(2, 8 * 32, !ok);
            tc_fence_after();
            const int quarter = warp & 3, half = (warp - kWarpQuad) >> 2;
            const int h = quarter * 32 + lane;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            const float *fac = reinterpret_cast<const float *>(gbase + kOffF);
            const bool good = !bad && T > 0;
            const float lsum = fac[(T % kPBufs) * kHeads + h];
            // a split writes its unnormalised O (fp32); the combine divides
            const float inv = split ? 1.f : (good && lsum > 0.f) ? 1.f / lsum : 0.f;
            const uint32_t stage = base + kOffRingV + (uint32_t)(warp - kWarpQuad) * kEpiBufs * 4096u;
            const int orow = cl * kHeads + quarter * 32;
            const bool f32 = out_dtype == SI_F32;
            const int nblk = f32 ? 8 : 4;  // 32 fp32 or 64 bf16 columns per block
            // O is finite unless a value left the f16 range in the conversion
            // (inf times any weight, zero included, stays inf or becomes NaN):
            // the maximum of the magnitude bits of every O entry read
            uint32_t omag = 0;
#pragma unroll 1
            for (int k = 0; k < nblk; k++) {
                const uint32_t buf = stage + (uint32_t)(k % kEpiBufs) * 4096u;
                if (k >= kEpiBufs) {
                    if (lane == 0)
                        bulk_wait_read<kEpiBufs - 1>();  // buffer's previous store has read it
                    __syncwarp();
                }
                uint32_t w[32];
                int xbyte;
                if (f32) {
                    const int col0 = half * (kDv / 2) + k * 32;
                    if (good) {
                        tmem_ld32(tmem + lane_off + col0, w);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; i++)
                            omag = max(omag, w[i] & 0x7FFFFFFFu);
                    }
#pragma unroll
                    for (int i = 0; i < 32; i++)
                        w[i] = good ? __float_as_uint(__uint_as_float(w[i]) * inv) : 0u;
                    xbyte = col0 * 4;
                } else {
                    const int col0 = half * (kDv / 2) + k * 64;
#pragma unroll
                    for (int hh = 0; hh < 2; hh++) {
                        uint32_t v[32];
                        if (good) {
                            tmem_ld32(tmem + lane_off + col0 + 32 * hh, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; i++)
                                omag = max(omag, v[i] & 0x7FFFFFFFu);
                        }
#pragma unroll
                        for (int i = 0; i < 16; i++)
                            w[16 * hh + i] =
                                good ? pack_bf16x2(__uint_as_float(v[2 * i]) * inv,
                                                   __uint_as_float(v[2 * i + 1]) * inv)
                                     : 0u;
                    }
                    xbyte = col0 * 2;
                }
#pragma unroll
                for (int u = 0; u < 8; u++)
                    st_shared_v4(buf + sw128_offset(lane, u), w[4 * u], w[4 * u + 1], w[4 * u + 2],
                                 w[4 * u + 3]);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&omap, xbyte, orow, buf);
                    bulk_commit();
                }
                __syncwarp();
            }
            if (lane == 0)
                bulk_wait<0>();
            if (__any_sync(0xffffffffu, omag >= 0x7F800000u) && lane == 0)
                raise_flag(st, SI_DEVFLAG_RANGE);
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma)
        tmem_dealloc(tmem, 512u);
    cluster_sync();  // neither CTA leaves while the other may still write into it
}

// Merges the splits of each row: with per-split state (m_s, l_s) in log2
// units and unnormalised O_s, out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s
// with M = max m_s.  One warp per (row, head), 16 of the 512 dims per lane.
constexpr int kCombineHeads = 8;  // heads per 256-thread block

__global__ void __launch_bounds__(kCombineHeads * 32)
k_attn_combine(int n_split, const float *part_o, const float *part_ml, void *out,
               si_dtype out_dtype, float *lse)
{
    griddep_wait();  // the partial results come from the previous kernel
    const int r = blockIdx.x, h = blockIdx.y * kCombineHeads + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    float M = -INFINITY;
    for (int s = 0; s < n_split; s++) {
        const float *ml = part_ml + (((int64_t)r * n_split + s) * kHeads + h) * 2;
        if (ml[1] > 0.f)
            M = fmaxf(M, ml[0]);
    }
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; i++)
        acc[i] = 0.f;
    float L = 0.f;
    for (int s = 0; s < n_split; s++) {
        const float *ml = part_ml + (((int64_t)r * n_split + s) * kHeads + h) * 2;
        const float l = ml[1];
        if (!(l > 0.f))
            continue;
        const float wgt = exp2f(ml[0] - M);
        L += wgt * l;
        const float4 *o4 = reinterpret_cast<const float4 *>(
            part_o + (((int64_t)r * n_split + s) * kHeads + h) * kDv + lane * 16);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float4 v = o4[i];
            acc[4 * i] += wgt * v.x;
            acc[4 * i + 1] += wgt * v.y;
            acc[4 * i + 2] += wgt * v.z;
            acc[4 * i + 3] += wgt * v.w;
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int64_t obase = ((int64_t)r * kHeads + h) * kDv + lane * 16;
    if (out_dtype == SI_F32) {
        float4 *d = reinterpret_cast<float4 *>(static_cast<float *>(out) + obase);
#pragma unroll
        for (int i = 0; i < 4; i++)
            d[i] = make_float4(acc[4 * i] * inv, acc[4 * i + 1] * inv, acc[4 * i + 2] * inv,
                               acc[4 * i + 3] * inv);
    } else {
        uint4 *d = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(out) + obase);
#pragma unroll
        for (int i = 0; i < 2; i++)
            d[i] = make_uint4(pack_bf16x2(acc[8 * i] * inv, acc[8 * i + 1] * inv),
                              pack_bf16x2(acc[8 * i + 2] * inv, acc[8 * i + 3] * inv),
                              pack_bf16x2(acc[8 * i + 4] * inv, acc[8 * i + 5] * inv),
                              pack_bf16x2(acc[8 * i + 6] * inv, acc[8 * i + 7] * inv));
    }
    if (lse && lane == 0)
        lse[(int64_t)r * kHeads + h] =
            L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

}  // namespace

int attn_tc_split(const si_batch &b, int k_top, int sms)
{
    if (b.n_q <= 0 || sms <= 0)
        return 1;
    const int tiles = (k_top + kTile - 1) / kTile;
    const int s = sms / (2 * b.n_q);  // fill the GPU with clusters of two
    return std::max(1, std::min(std::min(s, tiles), kMaxSplit));
}

size_t attn_tc_split_bytes(const si_batch &b, int n_split)
{
    if (n_split <= 1)
        return 0;
    // unnormalised O (fp32 [128 x 512]) and (m, l) per head, per row and split
    return (size_t)b.n_q * n_split * ((size_t)kHeads * kDv * 4 + (size_t)kHeads * 8);
}

bool attn_tc_supported(const si_batch &b, const si_attention &at, int k_top)
{
    (void)b;
    (void)k_top;
    // one shared latent row per position: V is the first 512 entries of the
    // 576-entry key row (the same cache, same stride)
    const bool shape = at.q_dtype == SI_BF16 && at.n_heads == kHeads && at.d_qk == kDqk &&
                       at.d_v == kDv && at.v.data == at.k.data &&
                       at.v.row_stride == at.k.row_stride && ((uintptr_t)at.k.data % 16) == 0 &&
                       ((uintptr_t)at.q % 16) == 0;
    // bf16 latent rows, or FP8 rows of 576 codes with five 128-entry tile scales
    const bool bf16 = at.k.dtype == SI_BF16 && !at.k.scale && !at.v.scale &&
                      at.k.row_stride % 8 == 0;
    const bool fp8 = at.k.dtype == SI_E4M3 && at.v.dtype == SI_E4M3 && at.k.scale &&
                     at.v.scale == at.k.scale && at.k.scale_tile == 128 &&
                     at.v.scale_tile == 128 && at.k.row_stride == kDqk &&
                     ((uintptr_t)at.k.scale % 4) == 0;
    // e2m1 rows of 576 codes (288 bytes) with 36 block scales of 16 entries
    const bool fp4 = at.k.dtype == SI_E2M1 && at.v.dtype == SI_E2M1 && at.k.scale &&
                     at.v.scale == at.k.scale && at.k.scale_tile == 16 &&
                     at.v.scale_tile == 16 && at.k.row_stride == kDqk &&
                     ((uintptr_t)at.k.scale % 16) == 0;
    return shape && (bf16 || fp8 || fp4);
}

cudaError_t launch_attn_tc(const si_batch &b, const si_attention &at, const int32_t *idx,
                           int k_top, void *out, si_dtype out_dtype, float *lse, void *scratch,
                           size_t scratch_bytes, unsigned int *st, cudaStream_t s)
{
    static std::once_flag once[kMaxDevices];
    static cudaError_t err_of[kMaxDevices];
    static int sms_of[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::call_once(once[dev], [dev] {
        cudaError_t r = cudaDeviceGetAttribute(&sms_of[dev], cudaDevAttrMultiProcessorCount, dev);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(k_attn_tc<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBytes);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(k_attn_tc<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBytes);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(k_attn_tc<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBytes);
        err_of[dev] = r;
    });
    if (err_of[dev] != cudaSuccess)
        return err_of[dev];
    if (b.n_q <= 0)
        return cudaSuccess;
    // Few rows: each row's key tiles are split over several clusters (when the
    // scratch holds their partial results) and a combine kernel merges them.
    int n_split = attn_tc_split(b, k_top, sms_of[dev]);
    const size_t need = attn_tc_split_bytes(b, n_split);
    if (n_split > 1 && (!scratch || scratch_bytes < need || ((uintptr_t)scratch % 256) != 0))
        n_split = 1;
    float *part_o = static_cast<float *>(scratch);
    float *part_ml = n_split > 1 ? part_o + (size_t)b.n_q * n_split * kHeads * kDv : nullptr;
    // q [n_q * 128 rows x 1152 bytes] read as [128 x 128-byte] boxes; out (or
    // the splits' fp32 O) [rows x 512 elements] written as [32 x 128-byte] boxes
    CUtensorMap qmap, omap;
    const uint64_t rows = (uint64_t)b.n_q * kHeads;
    e = make_tmap_2d_u8_sw128(&qmap, at.q, kDqk * 2, rows, kDqk * 2, 128, kHeads);
    if (e != cudaSuccess)
        return e;
    const si_dtype kdt = n_split > 1 ? SI_F32 : out_dtype;
    const uint64_t orow_bytes = (uint64_t)kDv * (kdt == SI_F32 ? 4 : 2);
    e = make_tmap_2d_u8_sw128(&omap, n_split > 1 ? static_cast<void *>(part_o) : out, orow_bytes,
                              rows * n_split, orow_bytes, 128, 32);
    if (e != cudaSuccess)
        return e;
    count_launch();
    // may overlap the tail of the kernel that wrote idx (programmatic
    // dependent launch; the kernel waits for it before reading idx)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * b.n_q * n_split));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = at.k.dtype == SI_E4M3
            ? cudaLaunchKernelEx(&cfg, k_attn_tc<1>, qmap, omap, b, at, idx, k_top, kdt, lse,
                                 n_split, part_ml, st)
        : at.k.dtype == SI_E2M1
            ? cudaLaunchKernelEx(&cfg, k_attn_tc<2>, qmap, omap, b, at, idx, k_top, kdt, lse,
                                 n_split, part_ml, st)
            : cudaLaunchKernelEx(&cfg, k_attn_tc<0>, qmap, omap, b, at, idx, k_top, kdt, lse,
                                 n_split, part_ml, st);
    if (e != cudaSuccess || n_split == 1)
        return e;
    return launch_attn_combine(b, n_split, part_o, part_ml, out, out_dtype, lse, s);
}

cudaError_t launch_attn_combine(const si_batch &b, int n_split, const float *part_o,
                                const float *part_ml, void *out, si_dtype out_dtype, float *lse,
                                cudaStream_t s)
{
    count_launch();
    // a programmatic dependent of the attention kernel (it waits for it
    // before reading the partial results)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)b.n_q, kHeads / kCombineHeads);
    cfg.blockDim = dim3(kCombineHeads * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_attn_combine, n_split, part_o, part_ml, out, out_dtype, lse);
}

}  // namespace si
