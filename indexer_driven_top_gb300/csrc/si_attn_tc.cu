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
// GB300 mapping.  One CTA per (query row, half of the 512 value dims).  The
// 128 heads are the UMMA M dimension and stay resident in shared memory (the
// whole 128 x 576 query, 147 KB, 128-byte swizzle).  Selected keys are
// processed in tiles of 128 (UMMA N = 128).  A tile's key rows stream through
// shared memory as "dim chunks" of 128 keys x 64 dims (16 KB) in a three-slot
// ring: nine chunks build S = q . k^T in TMEM (fp32, double-buffered), four
// more (this CTA's 256 value dims) feed O += P . V.  Eight loader warps
// gather each chunk with 16-byte cp.async copies straight into its ring slot;
// the copies signal the slot's mbarrier when they land, so no thread waits
// on them and no register holds data in flight.  (Staging through registers
// caps the stream: the proxy fence and the release arrive each loader must
// issue per chunk also wait for that thread's outstanding loads, which
// serialises the chunks.)  Three converter warps rewrite the value chunks
// from bf16 to f16 in place.  The chunk sequence
// interleaves S of tile t with P.V of tile t-1, so the tensor core computes
// the next scores while the softmax warpgroup works on the current ones.
//
// Softmax: one thread per head, online in the log2 domain with fp32 state; the
// running maximum used for the exponent is only raised when a tile's maximum
// exceeds it by more than 8 (then O is rescaled in TMEM), so most tiles need
// no O traffic.  P is rounded to f16 (11 significant bits; bf16's 8 would
// cost up to ~2^-9 of the value spread when few keys dominate) and the
// denominator sums the same rounded values.  The P.V operands must share a
// type, so value chunks are converted from bf16 to f16 as they are stored
// (exact for 2^-14 <= |v| <= 65504).  Positions that are -1 or outside
// 0..pos get zero rows and zero weight.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include "si_common.cuh"
#include "si_internal.h"
#include "si_sm100.cuh"

namespace si {

namespace {

using namespace sm100;

constexpr int kHeads = 128;       // query heads = UMMA M
constexpr int kDqk = 576;         // logit dims
constexpr int kDv = 512;          // value dims
constexpr int kDvHalf = 256;      // value dims per CTA
constexpr int kTile = 128;        // selected keys per tile = UMMA N of S
constexpr int kQChunks = kDqk / 64;   // 9 dim chunks of 64
constexpr int kVChunks = kDvHalf / 64; // 4
constexpr int kChunksPerTile = kQChunks + kVChunks;  // 13
constexpr int kRing = 3;
constexpr int kLoaderWarps = 8;
constexpr int kLoaders = kLoaderWarps * 32;
constexpr int kWarpSoft0 = 8;     // softmax warps 8..11 (TMEM lanes by warp % 4)
constexpr int kWarpMma = 12;
constexpr int kWarpConv0 = 13;    // value-chunk converters: warps 13..15
constexpr int kConverters = 3 * 32;
constexpr int kThreads = 16 * 32;
constexpr float kRescaleThreshold = 8.f;  // log2 units

constexpr uint32_t kChunk = 128 * 128;           // 16 KB: 128 rows x 128 bytes, SW128
constexpr uint32_t kOffQ = 0;                      // kQChunks x [128 heads x 64 dims]
constexpr uint32_t kOffP = kOffQ + kQChunks * kChunk;   // 2 x [128 heads x 64 keys]
constexpr uint32_t kOffRing = kOffP + 2 * kChunk;       // kRing x [128 keys x 64 dims]
constexpr int kMaskSlots = 4;
constexpr uint32_t kOffMask = kOffRing + kRing * kChunk;  // kMaskSlots x 128 key-valid bytes
constexpr uint32_t kOffBar = kOffMask + kMaskSlots * kTile;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;   // + alignment slack

// TMEM columns: O (this CTA's 256 value dims) then two S buffers.
constexpr uint32_t kTmemO = 0, kTmemS = 256, kTmemCols = 512;

struct ChunkId {
    int tile;  // key tile
    int v;     // -1: score chunk, else value chunk 0..3
    int c;     // dim chunk index of the row (0..8)
};

// g-th chunk of the stream: S(0); then per t >= 1: S(t), V(t-1); finally V(T-1).
__device__ __forceinline__ ChunkId chunk_of(int g, int T, int half)
{
    ChunkId id;
    if (g < kQChunks) {
        id.tile = 0;
        id.v = -1;
        id.c = g;
        return id;
    }
    const int h = g - kQChunks;
    const int blk = h / kChunksPerTile + 1, o = h % kChunksPerTile;
    if (blk < T && o < kQChunks) {
        id.tile = blk;
        id.v = -1;
        id.c = o;
    } else {
        const int vv = blk < T ? o - kQChunks : o;
        id.tile = blk - 1;
        id.v = vv;
        id.c = half * kVChunks + vv;
    }
    return id;
}

// 2^x with the hardware approximation (ex2.approx: ~2 ulp), ample for a
// softmax whose weights are rounded to bf16.
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
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

// Loader state of one thread: physical row byte offsets of its four keys for
// the even and the odd tile in flight, and the two-tile lookahead (index list
// values of tile t+2, block-table entries of tile t+1).
struct LoaderState {
    int rb0[4], rb1[4];  // physical rows (< 2^31), -1 = zero row
    int sv1[4], bk1[4], sv2[4];
    int have_tile;
};

__device__ __forceinline__ void load_idx(const int32_t *idx, int r, int k_top, int tile, int T,
                                         int n_valid, int kr0, int (&sv)[4])
{
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int j = tile * kTile + kr0 + 32 * i;
        sv[i] = (tile < T && j < n_valid) ? __ldg(idx + (int64_t)r * k_top + j) : -1;
    }
}

__device__ __forceinline__ void load_blk(const si_batch &b, int seq, int pos, const int (&sv)[4],
                                         int (&bk)[4])
{
#pragma unroll
    for (int i = 0; i < 4; i++) {
        bk[i] = -1;
        const int sp = sv[i];
        if (sp >= 0 && sp <= pos && (unsigned)seq < (unsigned)b.n_seq &&
            sp / b.page_size < b.max_blocks)
            bk[i] = __ldg(b.block_table + (int64_t)seq * b.max_blocks + sp / b.page_size);
    }
}

// Makes `tile` current: row offsets and key-valid bytes from the lookahead,
// then shifts the lookahead by one tile.
__device__ __forceinline__ void start_tile(LoaderState &ls, const si_batch &b, const int32_t *idx,
                                           int r, int k_top, int T, int n_valid, int seq, int pos,
                                           int64_t row_bytes, int kr0, int u, uint8_t *mask_s,
                                           unsigned int *st, int tile)
{
    ls.have_tile = tile;
    uint8_t *mb = mask_s + (tile % kMaskSlots) * kTile;
#pragma unroll
    for (int i = 0; i < 4; i++) {
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
        if (u == 0)
            mb[kr0 + 32 * i] = ok ? 1 : 0;
    }
#pragma unroll
    for (int i = 0; i < 4; i++)
        ls.sv1[i] = ls.sv2[i];
    load_blk(b, seq, pos, ls.sv1, ls.bk1);
    load_idx(idx, r, k_top, tile + 2, T, n_valid, kr0, ls.sv2);
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

// Issues this thread's copies of chunk g (one 16-byte unit of four key rows)
// into the ring slot at `dst`.  The first chunk of a tile also publishes the
// tile's key-valid bytes.
__device__ __forceinline__ void issue_chunk(LoaderState &ls, uint32_t dst, const si_batch &b,
                                            const int32_t *idx, int r, int k_top, int T,
                                            int n_valid, int seq, int pos, int64_t row_bytes,
                                            int kr0, int u, uint8_t *mask_s, uint64_t *mask_bar,
                                            unsigned int *st, const uint8_t *kv, int half, int g)
{
    const ChunkId id = chunk_of(g, T, half);
    if (id.tile > ls.have_tile) {
        start_tile(ls, b, idx, r, k_top, T, n_valid, seq, pos, row_bytes, kr0, u, mask_s, st,
                   id.tile);
        mbar_arrive(mask_bar + (id.tile % kMaskSlots));
    }
    const bool odd = id.tile & 1;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int row = odd ? ls.rb1[i] : ls.rb0[i];
        const uint8_t *src = row >= 0 ? kv + (int64_t)row * row_bytes + id.c * 128 + u * 16 : kv;
        cp_async_16(dst + sw128_offset(kr0 + 32 * i, u), src, row >= 0 ? 16u : 0u);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
k_attn_tc(si_batch b, si_attention at, const int32_t *idx, int k_top, void *out,
          si_dtype out_dtype, float *lse, unsigned int *st)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - smem_u32(smem_raw));
    uint8_t *mask_s = gbase + kOffMask;                                     // [kMaskSlots][128]
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(gbase + kOffBar);    // [kRing] score chunks
    uint64_t *empty_bar = full_bar + kRing;                                 // [kRing]
    uint64_t *sfull_bar = empty_bar + kRing;                                // [2]
    uint64_t *sempty_bar = sfull_bar + 2;                                   // [2]
    uint64_t *mask_bar = sempty_bar + 2;                                    // [kMaskSlots]
    uint64_t *qready_bar = mask_bar + kMaskSlots;
    uint64_t *pfull_bar = qready_bar + 1;
    uint64_t *pvdone_bar = pfull_bar + 1;
    uint64_t *vfull_bar = pvdone_bar + 1;                                   // [kVChunks]
    uint64_t *conv_bar = vfull_bar + kVChunks;                              // [kVChunks]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(conv_bar + kVChunks);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = blockIdx.x >> 1, half = blockIdx.x & 1;
    const int pos = __ldg(b.q_pos + r), seq = __ldg(b.q_seq + r);
    const int n_valid = max(0, min(k_top, pos + 1));
    const int T = (n_valid + kTile - 1) / kTile;  // key tiles
    const int n_chunks = kChunksPerTile * T;

    if (tid == 0) {
        // Landing barriers, one cp.async arrival per loader thread per phase:
        // full_bar[slot] for score chunks (a phase per score chunk in that
        // slot), vfull_bar[v] for value chunk v (a phase per key tile).  Each
        // waiter observes every phase of the barriers it waits on, in order.
        for (int i = 0; i < kRing; i++) {
            mbar_init(full_bar + i, kLoaders);
            mbar_init(empty_bar + i, 1);
        }
        for (int i = 0; i < kVChunks; i++) {
            mbar_init(vfull_bar + i, kLoaders);
            mbar_init(conv_bar + i, kConverters);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(sfull_bar + i, 1);
            mbar_init(sempty_bar + i, 128);
        }
        for (int i = 0; i < kMaskSlots; i++)
            mbar_init(mask_bar + i, kLoaders);
        mbar_init(qready_bar, kLoaders);
        mbar_init(pfull_bar, 128);
        mbar_init(pvdone_bar, 1);
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const uint8_t *kv = static_cast<const uint8_t *>(at.k.data);
    const int64_t row_bytes = at.k.row_stride * 2;

    if (warp < kLoaderWarps) {
        // -------------------------------------------------------------- loaders
        // Thread t owns 16-byte unit u = t & 7 of key rows kr_i = (t >> 3) + 32 i
        // in every chunk.
        const int u = tid & 7, kr0 = tid >> 3;
        // query: 128 heads x 9 chunks x 8 units, SW128 K-major per chunk
        {
            const uint4 *qsrc = reinterpret_cast<const uint4 *>(at.q) + (int64_t)r * kHeads * (kDqk / 8);
            for (int i = tid; i < kHeads * kQChunks * 8; i += kLoaders) {
                const int h = i / (kQChunks * 8), rem = i % (kQChunks * 8);
                const int c = rem >> 3, uu = rem & 7;
                const uint4 v = __ldg(qsrc + (int64_t)h * (kDqk / 8) + rem);
                st_shared_v4(base + kOffQ + c * kChunk + sw128_offset(h, uu), v.x, v.y, v.z, v.w);
            }
            fence_async_smem();
            mbar_arrive(qready_bar);
        }
        // Physical rows of this thread's 4 keys are looked up two tiles ahead
        // (LoaderState) so the dependent loads never stall the stream.
        LoaderState ls;
        ls.have_tile = -1;
        load_idx(idx, r, k_top, 0, T, n_valid, kr0, ls.sv1);
        load_blk(b, seq, pos, ls.sv1, ls.bk1);
        load_idx(idx, r, k_top, 1, T, n_valid, kr0, ls.sv2);
        for (int g = 0; g < n_chunks; g++) {
            const int slot = g % kRing;
            if (g >= kRing && !mbar_wait(empty_bar + slot, (uint32_t)((g / kRing) - 1) & 1, st))
                break;
            issue_chunk(ls, base + kOffRing + slot * kChunk, b, idx, r, k_top, T, n_valid, seq,
                        pos, row_bytes, kr0, u, mask_s, mask_bar, st, kv, half, g);
            const ChunkId id = chunk_of(g, T, half);
            cp_async_arrive(id.v < 0 ? full_bar + slot : vfull_bar + id.v);
        }
        cp_async_wait_all();  // nothing may land after the block has moved on
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------------ MMA
        const uint32_t idesc_s = idesc_f16(kHeads, kTile, 1, 0, 0);   // bf16, K-major A/B
        const uint32_t idesc_pv = idesc_f16(kHeads, 64, 0, 0, 1);     // f16; B (V) MN-major
        bool ok = mbar_wait(qready_bar, 0, st);
        uint32_t s_par = 0;  // phase parity of each slot's score-chunk landings
        for (int g = 0; ok && g < n_chunks; g++) {
            const ChunkId id = chunk_of(g, T, half);
            const int slot = g % kRing;
            if (id.v < 0 && id.c == 0) {
                // S buffer of this tile must be free (softmax read S of tile - 2)
                if (id.tile >= 2 &&
                    !mbar_wait(sempty_bar + (id.tile & 1), (uint32_t)((id.tile >> 1) - 1) & 1, st))
                    break;
            }
            if (id.v == 0) {
                // P of this tile is in shared memory
                if (!mbar_wait(pfull_bar, (uint32_t)id.tile & 1, st))
                    break;
            }
            if (id.v < 0) {
                // score chunk: the loaders' copies have landed; make them
                // visible to the tensor core (async proxy)
                const uint32_t par = (s_par >> slot) & 1u;
                s_par ^= 1u << slot;
                if (!mbar_wait(full_bar + slot, par, st))
                    break;
                fence_async_smem();
            } else if (!mbar_wait(conv_bar + id.v, (uint32_t)id.tile & 1, st)) {
                break;  // value chunk: converted to f16 (the converters fenced)
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t chunk = base + kOffRing + slot * kChunk;
                if (id.v < 0) {
                    const uint32_t d = tmem + kTmemS + (id.tile & 1) * kTile;
#pragma unroll
                    for (int kk = 0; kk < 4; kk++) {
                        const uint64_t ad = smem_desc(base + kOffQ + id.c * kChunk + kk * 32, 16,
                                                      1024, kSwizzle128B);
                        const uint64_t bd = smem_desc(chunk + kk * 32, 16, 1024, kSwizzle128B);
                        umma_f16_ss(d, ad, bd, idesc_s, id.c > 0 || kk > 0);
                    }
                    umma_commit(empty_bar + slot);
                    if (id.c == kQChunks - 1)
                        umma_commit(sfull_bar + (id.tile & 1));
                } else {
                    // O[:, 64 v .. +64] += P[128 x 128 keys] . V_chunk[128 keys x 64]
                    const uint32_t d = tmem + kTmemO + id.v * 64;
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; kk++) {
                        const uint64_t ad = smem_desc(base + kOffP + (kk >> 2) * kChunk +
                                                          (kk & 3) * 32,
                                                      16, 1024, kSwizzle128B);
                        const uint64_t bd = smem_desc(chunk + kk * 2048, 4096, 1024, kSwizzle128B);
                        umma_f16_ss(d, ad, bd, idesc_pv, id.tile > 0 || kk > 0);
                    }
                    umma_commit(empty_bar + slot);
                    if (id.v == kVChunks - 1)
                        umma_commit(pvdone_bar);
                }
            }
            __syncwarp();
        }
    } else if (warp >= kWarpConv0) {
        // ----------------------------------------------------------- converters
        // Value chunks feed the f16 P.V product: rewrite them bf16 -> f16 in
        // place once their copies have landed.
        const int ct = tid - kWarpConv0 * 32;
        for (int g = 0; g < n_chunks; g++) {
            const ChunkId id = chunk_of(g, T, half);
            if (id.v < 0)
                continue;
            const int slot = g % kRing;
            if (!mbar_wait(vfull_bar + id.v, (uint32_t)id.tile & 1, st))
                break;
            const uint32_t src = base + kOffRing + slot * kChunk;
            for (int i = ct; i < (int)(kChunk / 16); i += kConverters) {
                const uint4 x = ld_shared_v4(src + i * 16);
                st_shared_v4(src + i * 16, bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y),
                             bf16x2_to_f16x2(x.z), bf16x2_to_f16x2(x.w));
            }
            fence_async_smem();
            mbar_arrive(conv_bar + id.v);
        }
    } else {
        // -------------------------------------------------------------- softmax
        const int h = tid - kWarpSoft0 * 32;   // head = TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const float sl2 = at.softmax_scale * 1.4426950408889634f;  // scale * log2(e)
        float m_used = -INFINITY;  // exponent reference (log2 units)
        float l = 0.f;
        bool ok = true;
        for (int t = 0; t < T && ok; t++) {
            const int sb = t & 1;
            if (!mbar_wait(mask_bar + (t % kMaskSlots), (uint32_t)(t / kMaskSlots) & 1, st) ||
                !mbar_wait(sfull_bar + sb, (uint32_t)(t >> 1) & 1, st)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // key-valid bits of the tile (bytes 0/1 -> one bit per key)
            uint32_t mw[4];
            {
                const uint32_t *mb = reinterpret_cast<const uint32_t *>(mask_s + (t % kMaskSlots) * kTile);
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    uint32_t bits = 0;
#pragma unroll
                    for (int w = 0; w < 8; w++) {
                        const uint32_t x = mb[q * 8 + w];
                        bits |= ((x & 1u) | ((x >> 7) & 2u) | ((x >> 14) & 4u) | ((x >> 21) & 8u))
                                << (4 * w);
                    }
                    mw[q] = bits;
                }
            }
            // pass 1: tile maximum of the valid logits
            float tmax = -INFINITY;
#pragma unroll 1
            for (int q = 0; q < 4; q++) {
                uint32_t v[32];
                tmem_ld32(tmem + kTmemS + sb * kTile + lane_off + q * 32, v);
                tmem_wait_ld();
                const uint32_t mwq = mw[q];
#pragma unroll
                for (int i = 0; i < 32; i++)
                    if (mwq & (1u << i))
                        tmax = fmaxf(tmax, __uint_as_float(v[i]) * sl2);
            }
            // P.V of the previous tile must be done before P and O are touched
            if (t > 0 && !mbar_wait(pvdone_bar, (uint32_t)(t - 1) & 1, st)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (tmax > m_used + kRescaleThreshold) {
                // raise the exponent reference; rescale O and l accordingly
                const float f = ex2(m_used - tmax);
                if (t > 0) {
#pragma unroll 1
                    for (int q = 0; q < kDvHalf / 32; q++) {
                        uint32_t v[32];
                        tmem_ld32(tmem + kTmemO + lane_off + q * 32, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; i++)
                            v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
                        tmem_st32(tmem + kTmemO + lane_off + q * 32, v);
                    }
                    tmem_wait_st();
                }
                l *= f;
                m_used = tmax;
            }
            // pass 2: p = 2^(x - m_used) as f16 into P (two 64-key chunks)
#pragma unroll 1
            for (int q = 0; q < 4; q++) {
                uint32_t v[32];
                tmem_ld32(tmem + kTmemS + sb * kTile + lane_off + q * 32, v);
                tmem_wait_ld();
                const uint32_t mwq = mw[q];
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float p0 = (mwq & (1u << i)) ? ex2(__uint_as_float(v[i]) * sl2 - m_used) : 0.f;
                    const float p1 =
                        (mwq & (1u << (i + 1))) ? ex2(__uint_as_float(v[i + 1]) * sl2 - m_used) : 0.f;
                    pk[i >> 1] = pack_f16x2(p0, p1);
                    const __half2 pr = *reinterpret_cast<__half2 *>(&pk[i >> 1]);
                    l += __low2float(pr) + __high2float(pr);
                }
                // keys 32q .. 32q+31 -> P chunk q/2, 16-byte units 4(q&1) .. +3
                const uint32_t pc = base + kOffP + (q >> 1) * kChunk;
#pragma unroll
                for (int w = 0; w < 4; w++)
                    st_shared_v4(pc + sw128_offset(h, (q & 1) * 4 + w), pk[4 * w], pk[4 * w + 1],
                                 pk[4 * w + 2], pk[4 * w + 3]);
            }
            tc_fence_before();
            mbar_arrive(sempty_bar + sb);
            fence_async_smem();
            mbar_arrive(pfull_bar);
        }
        // epilogue: wait for the last P.V, normalise, store
        if (ok && T > 0 && !mbar_wait(pvdone_bar, (uint32_t)(T - 1) & 1, st))
            ok = false;
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int64_t obase = ((int64_t)r * kHeads + h) * kDv + half * kDvHalf;
#pragma unroll 1
        for (int q = 0; q < kDvHalf / 32; q++) {
            uint32_t v[32];
            if (ok && T > 0) {
                tmem_ld32(tmem + kTmemO + lane_off + q * 32, v);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < 32; i++)
                    v[i] = 0;
            }
            if (out_dtype == SI_F32) {
                float4 *o4 = reinterpret_cast<float4 *>(static_cast<float *>(out) + obase + q * 32);
#pragma unroll
                for (int i = 0; i < 8; i++)
                    o4[i] = make_float4(__uint_as_float(v[4 * i]) * inv,
                                        __uint_as_float(v[4 * i + 1]) * inv,
                                        __uint_as_float(v[4 * i + 2]) * inv,
                                        __uint_as_float(v[4 * i + 3]) * inv);
            } else {
                uint4 *o4 = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(out) + obase +
                                                      q * 32);
#pragma unroll
                for (int i = 0; i < 4; i++)
                    o4[i] = make_uint4(
                        pack_bf16x2(__uint_as_float(v[8 * i]) * inv, __uint_as_float(v[8 * i + 1]) * inv),
                        pack_bf16x2(__uint_as_float(v[8 * i + 2]) * inv, __uint_as_float(v[8 * i + 3]) * inv),
                        pack_bf16x2(__uint_as_float(v[8 * i + 4]) * inv, __uint_as_float(v[8 * i + 5]) * inv),
                        pack_bf16x2(__uint_as_float(v[8 * i + 6]) * inv, __uint_as_float(v[8 * i + 7]) * inv));
            }
        }
        if (lse && half == 0)
            lse[(int64_t)r * kHeads + h] =
                l > 0.f ? (m_used + log2f(l)) * 0.6931471805599453f : -INFINITY;
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma)
        tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool attn_tc_supported(const si_batch &b, const si_attention &at, int k_top)
{
    (void)b;
    (void)k_top;
    // one shared latent row per position: V is the first 512 entries of the
    // 576-entry key row (the same cache, same stride)
    return at.q_dtype == SI_BF16 && at.n_heads == kHeads && at.d_qk == kDqk && at.d_v == kDv &&
           at.k.dtype == SI_BF16 && at.v.data == at.k.data && at.v.row_stride == at.k.row_stride &&
           at.k.row_stride % 8 == 0 && ((uintptr_t)at.k.data % 16) == 0 &&
           ((uintptr_t)at.q % 16) == 0;
}

cudaError_t launch_attn_tc(const si_batch &b, const si_attention &at, const int32_t *idx,
                           int k_top, void *out, si_dtype out_dtype, float *lse, unsigned int *st,
                           cudaStream_t s)
{
    static std::once_flag once[kMaxDevices];
    static cudaError_t err_of[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::call_once(once[dev], [dev] {
        err_of[dev] = cudaFuncSetAttribute(k_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemBytes);
    });
    if (err_of[dev] != cudaSuccess)
        return err_of[dev];
    count_launch();
    k_attn_tc<<<(unsigned)(2 * b.n_q), kThreads, kSmemBytes, s>>>(b, at, idx, k_top, out,
                                                                  out_dtype, lse, st);
    return cudaGetLastError();
}

}  // namespace si
