// si_indexer_tc.cu -- tensor-core indexer over a paged FP8 key cache.
//
// "Day0 Inference Support and Performance Optimization for New Architecture
// LLMs": section 2.2 (the indexer scores a query against every earlier
// position and aggregates the per-head scores with head weights), section
// 4.1 (the scoring reads the paged K-cache directly and never stores the
// intermediate per-head scores) and section 5.1 (the indexer path is stored in
// FP8).  Score of key s for query row r:
//     k_scale[s] * sum_h w[r,h] * ReLU(q[r,h,:] . k[s,:])
//
// GB300 mapping.  A tile is 128 consecutive key positions of one query row;
// its FP8 key rows are the UMMA A operand (M = 128, K = 128 bytes) exactly as
// the TMA engine lands them in shared memory, so keys are never converted.
// The bf16 query is made FP8 without loss: per head h a power of two s_h
// brings max|q_h| into (224, 448], and the scaled head is written as
// q_hi + q_lo with q_hi = e4m3(q) and q_lo = e4m3(q - q_hi).  A bf16 value
// has 8 significant bits and each term carries 4, so the split is exact
// except where q_lo falls below e4m3's subnormal step (|q| < max|q_h| / 1800,
// error < 2^-10 of the head's scale).  The 64 q_hi heads and the 64 q_lo heads
// form one 128-row B operand; the MMA (kind::f8f6f4, fp32 accumulate) writes
// D[key, 0..63] = q_hi . k and D[key, 64..127] = q_lo . k, one key per TMEM
// lane.  Each epilogue thread then reduces its own key:
//     k_scale * sum_h (w_h * s_h) * ReLU(D[h] + D[64 + h])
// (s_h > 0 is a power of two, so folding it into the weight is exact).
// A query already stored in FP8 with a per-(row, head) scale (section 4.3's
// per-group quantisation, one group per head) needs no split: its codes are
// q_hi, q_lo is zero and the scale multiplies the head weight.
//
// MXFP8 (k_indexer_tc<false, true>; section 5.1: query and keys quantised
// per group of 32 entries with E8M0 scales).  The MMA is the block-scaled
// kind::mxf8f6f4: B is the 64 query heads' codes (N = 64, no split), and the
// tensor core applies each group's pair of scales to its 32-entry partial
// dot product, so D[key, h] is already the MXFP8 dot product.  Scale factors
// live in TMEM.  The producer lands each tile's key scale words (4 bytes per
// key, one byte per group) with cp.async into a 32 x 16-byte block per stage,
// row L holding keys L, L+32, L+64, L+96 -- the order tcgen05.cp spreads over
// TMEM lanes and columns -- and the MMA thread copies that block (and, once
// per query row, the query's block) into TMEM ahead of the tile's four MMAs;
// copies and MMAs of one thread execute in order.  A bf16 query is converted
// by the q-prep threads with the MX rule of section 4.3's per-group query
// quantisation, bit-identical to si_quant_mxfp8.
//
// One persistent CTA per SM runs a warp-specialised pipeline:
//   2 producer warps -- per tile, TMA tensor copies of its key pages (128-byte
//                       swizzle) into a ten-stage ring; tiles alternate
//                       between the warps because a bulk copy holds its
//                       issuing warp for several hundred cycles;
//   2 lanes of work  -- tiles alternate between two (MMA warp, epilogue
//                       warpgroup) pairs: the MMA warp issues four FP8 UMMAs
//                       per tile into its two TMEM accumulators (128 columns
//                       each), the epilogue group fetches the keys' scales,
//                       reduces its accumulator and stores the scores; two
//                       pairs hide UMMA issue and TMEM-load latency;
//   q-prep warpgroup -- splits each query row into the FP8 B operand and the
//                       scaled head weights (double-buffered per row).
// Work is the flattened list of (query row, tile) items split into equal
// contiguous ranges, one per CTA.
//
// Candidate lists (k_indexer_tc<true>; the vLLM article on DeepSeek-V4.1,
// "Kernels": logits over a fixed candidate set per query).  A tile is then
// 128 consecutive slots of the row's candidate list, not of its positions:
// the producer lanes resolve each slot (list entry -> block table -> physical
// row) and gather the key rows with 16-byte cp.async pieces straight into the
// stage's swizzled layout, and each key's scale into the scale ring; a slot
// without a candidate gets a zero row and scale -1 (score -inf).  Everything
// after the stage is the same pipeline.
#include <cuda.h>
#include <cuda_fp16.h>
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

constexpr int kKeys = 128;        // keys per tile = UMMA M
constexpr int kHeads = 64;        // indexer heads
constexpr int kDim = 128;         // head dim = bytes per e4m3 key row = UMMA K
constexpr int kN = 2 * kHeads;    // B rows: q_hi heads, then q_lo heads = UMMA N
constexpr int kStages = 10;       // key-tile ring depth
constexpr int kScStages = kStages / 2;  // per-producer ring of tile scales (128 floats each)
constexpr int kPairs = 2;         // (MMA warp, epilogue group) pairs, alternate tiles
constexpr int kAccPerPair = 2;    // TMEM accumulators per pair (4 x 128 = 512 columns)
// warp roles
constexpr int kWarpProd0 = 0, kWarpProd1 = 2;   // producers
constexpr int kWarpMma0 = 1, kWarpMma1 = 3;     // MMA warps of pair 0 and pair 1
constexpr int kWarpPrep0 = 4;                   // q-prep: 4..7
constexpr int kWarpEpi0 = 8;                    // epilogue groups: 8..11 and 12..15
constexpr int kThreads = 16 * 32;

constexpr uint32_t kTile = kKeys * kDim;    // 16 KB, SW128 K-major
constexpr uint32_t kTileB = kN * kDim;      // 16 KB, SW128 K-major
constexpr uint32_t kOffStage = 0;
constexpr uint32_t kOffQ = kOffStage + kStages * kTile;            // [2]
constexpr uint32_t kOffW = kOffQ + 2 * kTileB;                      // [2][64] fp32 (w * s_h)
constexpr uint32_t kOffWin = kOffW + 2 * kHeads * 4;                // 2 producers x 32 int
constexpr uint32_t kOffSc = kOffWin + 2 * 32 * 4;                   // [2][kScStages][128] fp32
// MXFP8: scale words for tcgen05.cp, 32 rows x 16 bytes per block
constexpr uint32_t kSfBytes = 512;
constexpr uint32_t kOffSfa = kOffSc + 2 * kScStages * kKeys * 4;    // [kStages] key tiles
constexpr uint32_t kOffSfb = kOffSfa + kStages * kSfBytes;          // [2] query rows
constexpr uint32_t kOffBar = kOffSfb + 2 * kSfBytes;
constexpr uint32_t kSmemBytes = kOffBar + 1024 + 1024;             // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
// TMEM columns: accumulators from 0 (kN wide, or kHeads for MXFP8), then for
// MXFP8 four scale columns per accumulator (keys) and per (pair, row buffer)
// (query heads).
constexpr uint32_t kTmemCols = kPairs * kAccPerPair * kN;  // 512
constexpr uint32_t kColSfa = kPairs * kAccPerPair * kHeads;
constexpr uint32_t kColSfb = kColSfa + 4 * kPairs * kAccPerPair;
static_assert(kColSfb + 4 * kPairs * 2 <= kTmemCols, "TMEM columns");

// Advances (row, tile) by `n` items of a row-major list with `tpr` tiles per row.
__device__ __forceinline__ void advance(int &r, int &t, int n, int tpr)
{
    t += n;
    while (t >= tpr) {
        t -= tpr;
        ++r;
    }
}

__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v)
{
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
    return make_float2(__half2float(__ushort_as_half(h.x)), __half2float(__ushort_as_half(h.y)));
}

__device__ __forceinline__ uint16_t float2_to_e4m3x2(float a, float b)
{
    return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Candidate-list operands of k_indexer_tc<true> (row r's list at cand + r * ld,
// its first n entries scored).
struct CandArgs {
    const int32_t *cand;
    int64_t ld;
    int32_t n;
};

__device__ const float kScaleOne = 1.f;    // scale of a key in an unscaled cache
__device__ const float kScaleNone = -1.f;  // scale of a slot without a candidate

// 16-byte global -> shared copy that lands asynchronously; src_bytes = 0
// writes zeros without reading.
__device__ __forceinline__ void cp_async_16z(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// One producer lane's view of the four slots lane + 32 i (i < 4) of one
// candidate tile: list entries, their block-table entries and the row's
// position; `prev` (lane 0) is the list entry before the tile.
struct CandLook {
    int cv[4], bk[4];
    int pos, prev;
};

__device__ __forceinline__ void cand_entries(const CandArgs &ca, const si_batch &b, int r, int t,
                                             int lane, CandLook &L)
{
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int j = t * kKeys + lane + 32 * i;
        L.cv[i] = (r < b.n_q && j < ca.n) ? __ldg(ca.cand + (int64_t)r * ca.ld + j) : -1;
    }
    L.prev = (lane == 0 && r < b.n_q && t > 0 && t * kKeys - 1 < ca.n)
                 ? __ldg(ca.cand + (int64_t)r * ca.ld + t * kKeys - 1)
                 : -1;
}

__device__ __forceinline__ void cand_blocks(const si_batch &b, int r, CandLook &L)
{
    L.pos = r < b.n_q ? __ldg(b.q_pos + r) : -1;
    const int seq = r < b.n_q ? __ldg(b.q_seq + r) : -1;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int s = L.cv[i];
        L.bk[i] = -1;
        if (s >= 0 && s <= L.pos && (unsigned)seq < (unsigned)b.n_seq &&
            s / b.page_size < b.max_blocks)
            L.bk[i] = __ldg(b.block_table + (int64_t)seq * b.max_blocks + s / b.page_size);
    }
}

template <bool CAND, bool MX>
__global__ void __launch_bounds__(kThreads, 1)
k_indexer_tc(const __grid_constant__ CUtensorMap tmap, si_batch b, si_indexer ix, float *scores,
             int64_t ld, int64_t total_items, int tiles_per_row, unsigned int *st, CandArgs ca)
{
    static_assert(!(CAND && MX), "candidate lists take FP8 keys with per-row scales");
    constexpr int nB = MX ? kHeads : kN;  // B rows = accumulator columns
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - smem_u32(smem_raw));
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(gbase + kOffBar);  // [kStages]
    uint64_t *empty_bar = full_bar + kStages;                             // [kStages]
    uint64_t *cfull_bar = empty_bar + kStages;                            // [kPairs][kAccPerPair]
    uint64_t *cempty_bar = cfull_bar + kPairs * kAccPerPair;              // [kPairs][kAccPerPair]
    uint64_t *qfull_bar = cempty_bar + kPairs * kAccPerPair;              // [2]
    uint64_t *qempty_bar = qfull_bar + 2;                                 // [2]
    uint64_t *scfull_bar = qempty_bar + 2;                                // [2][kScStages]
    uint64_t *scempty_bar = scfull_bar + 2 * kScStages;                   // [2][kScStages]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(scempty_bar + 2 * kScStages);
    float *sc_s = reinterpret_cast<float *>(gbase + kOffSc);
    float *w_s = reinterpret_cast<float *>(gbase + kOffW);
    volatile int *win_all = reinterpret_cast<volatile int *>(gbase + kOffWin);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    griddep_launch_dependents();  // the Top-K kernel may be scheduled as CTAs finish
    const int64_t G = gridDim.x;
    const int64_t j0 = total_items * blockIdx.x / G;
    const int64_t j1 = total_items * (blockIdx.x + 1) / G;
    const int64_t n_items = j1 - j0;

    if (tid == 0) {
        for (int i = 0; i < kStages; i++) {
            // producer's expect_tx arrival, or its 32 lanes' cp.async arrivals,
            // or (MXFP8) both
            mbar_init(full_bar + i, CAND ? 32 : (MX ? 33 : 1));
            mbar_init(empty_bar + i, 1);    // MMA commit (or plain arrive)
        }
        for (int i = 0; i < kPairs * kAccPerPair; i++) {
            mbar_init(cfull_bar + i, 1);    // MMA commit
            mbar_init(cempty_bar + i, 128); // epilogue group
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(qfull_bar + i, 128);                   // q-prep threads
            mbar_init(qempty_bar + i, kPairs + kPairs * 128); // MMA commits + epilogues
        }
        for (int i = 0; i < 2 * kScStages; i++) {
            mbar_init(scfull_bar + i, 32);    // producer lanes (copy landed or sentinel)
            mbar_init(scempty_bar + i, 128);  // epilogue group read the scales
        }
        fence_barrier_init();
    }
    if (warp == kWarpMma0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int P = b.page_size;
    const int lp = 31 - __clz(P);  // page_size is a power of two >= 8

    if (CAND && (warp == kWarpProd0 || warp == kWarpProd1)) {
        // ------------------------------------------------- producer, candidates
        // Lane l gathers slots t * 128 + l + 32 i of each item.  The lookups
        // that feed the copies are plain loads, which complete behind the
        // lane's copies in flight, so they run one (block table) and two
        // (list entries) of this producer's items ahead of their use.
        const int pw = warp == kWarpProd0 ? 0 : 1;  // takes items pw, pw + 2, ...
        const uint8_t *kdata = static_cast<const uint8_t *>(ix.k.data);
        int rA = (int)(j0 / tiles_per_row), tA = (int)(j0 % tiles_per_row);
        advance(rA, tA, pw, tiles_per_row);
        int rB = rA, tB = tA;
        advance(rB, tB, 2, tiles_per_row);
        int rC = rB, tC = tB;
        advance(rC, tC, 2, tiles_per_row);
        CandLook A, B, C;
        cand_entries(ca, b, rA, tA, lane, A);
        cand_blocks(b, rA, A);
        cand_entries(ca, b, rB, tB, lane, B);
        cand_blocks(b, rB, B);
        cand_entries(ca, b, rC, tC, lane, C);
        for (int64_t it = pw; it < n_items; it += 2) {
            const int stg = (int)(it % kStages);
            if (it >= kStages &&
                !mbar_wait(empty_bar + stg, (uint32_t)((it / kStages) - 1) & 1, st))
                break;
            int64_t prow[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int s = A.cv[i];
                const bool valid = s >= 0 && s <= A.pos;
                prow[i] = (valid && (unsigned)A.bk[i] < (unsigned)b.n_blocks)
                              ? (int64_t)A.bk[i] * P + s % P
                              : -1;
                if (valid && prow[i] < 0)
                    raise_flag(st, SI_DEVFLAG_BAD_BLOCK);
                // a candidate follows a candidate with a lower position
                // (the slot before lane 0's is lane 31's of the previous group of
                // 32, or the entry before the tile)
                int pv = __shfl_up_sync(0xffffffffu, s, 1);
                const int last = __shfl_sync(0xffffffffu, A.cv[i > 0 ? i - 1 : 0], 31);
                if (lane == 0)
                    pv = i > 0 ? last : A.prev;
                const bool first = tA == 0 && lane == 0 && i == 0;
                if (valid && !first && !(pv >= 0 && pv < s))
                    raise_flag(st, SI_DEVFLAG_BAD_INDEX);
            }
            const uint32_t dst = base + kOffStage + stg * kTile;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int key = lane + 32 * i;
#pragma unroll
                for (int u = 0; u < kDim / 16; u++)
                    cp_async_16z(dst + sw128_offset(key, u),
                                 prow[i] >= 0 ? kdata + prow[i] * kDim + u * 16 : kdata,
                                 prow[i] >= 0 ? 16u : 0u);
            }
            cp_async_arrive_noinc(full_bar + stg);
            // the keys' scales into this producer's scale ring
            const int64_t kit = it >> 1;
            const int ss = (int)(kit % kScStages);
            if (kit >= kScStages &&
                !mbar_wait(scempty_bar + pw * kScStages + ss, (uint32_t)((kit / kScStages) - 1) & 1,
                           st))
                break;
            const uint32_t sd = smem_u32(sc_s + (pw * kScStages + ss) * kKeys);
#pragma unroll
            for (int i = 0; i < 4; i++)
                cp_async_4(sd + (lane + 32 * i) * 4,
                           prow[i] >= 0 ? (ix.k.scale ? fscale(ix.k.scale) + prow[i] : &kScaleOne)
                                        : &kScaleNone);
            cp_async_arrive_noinc(scfull_bar + pw * kScStages + ss);
            // shift the lookahead by one item of this producer
            A = B;
            rA = rB;
            tA = tB;
            B = C;
            rB = rC;
            tB = tC;
            cand_blocks(b, rB, B);
            advance(rC, tC, 2, tiles_per_row);
            cand_entries(ca, b, rC, tC, lane, C);
        }
        // nothing may land after the block has moved on
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp == kWarpProd0 || warp == kWarpProd1) {
        // ------------------------------------------------------------ producer
        const int pw = warp == kWarpProd0 ? 0 : 1;  // takes items pw, pw + 2, ...
        volatile int *win_s = win_all + pw * 32;
        const int span = min(P, kKeys);             // keys of one page inside one tile
        int r = (int)(j0 / tiles_per_row), t = (int)(j0 % tiles_per_row);
        advance(r, t, pw, tiles_per_row);
        int pf_row = -1, pf_pos = -1, pf_seq = 0;
        // window of 32 block-table entries: win_s[l] = page win + l of win_row
        int win_row = -1, win = 0;
        for (int64_t it = pw; it < n_items; it += 2) {
            const int stg = (int)(it % kStages);
            if (it >= kStages &&
                !mbar_wait(empty_bar + stg, (uint32_t)((it / kStages) - 1) & 1, st))
                break;
            if (r != pf_row) {
                pf_row = r;
                pf_pos = __ldg(b.q_pos + r);
                pf_seq = __ldg(b.q_seq + r);
            }
            const int s0 = t * kKeys;
            const bool live = s0 <= pf_pos;
            const int first = s0 >> lp;
            const int last = min(s0 + kKeys - 1, pf_pos) >> lp;
            if (live && (win_row != r || last >= win + 32)) {
                win_row = r;
                win = first;
                const int lb = first + lane;
                int v = -1;
                if ((unsigned)pf_seq < (unsigned)b.n_seq && lb < b.max_blocks)
                    v = __ldg(b.block_table + (int64_t)pf_seq * b.max_blocks + lb);
                win_s[lane] = v;
                __syncwarp();
            }
            // lane l handles page first + l of the tile
            const int lb = first + lane;
            bool copy = false;
            int row = 0, k_lo = 0;
            if (live && lane < 16 && lb <= last) {
                const int blk = win_s[lb - win];
                if (lb < b.max_blocks && (unsigned)blk < (unsigned)b.n_blocks) {
                    copy = true;
                    k_lo = max(lb << lp, s0) - s0;
                    row = (blk << lp) + (s0 + k_lo - (lb << lp));
                } else {
                    raise_flag(st, SI_DEVFLAG_BAD_BLOCK);
                }
            }
            const uint32_t n_copies = __popc(__ballot_sync(0xffffffffu, copy));
            if (lane == 0)
                mbar_arrive_expect_tx(full_bar + stg, n_copies * span * kDim);
            __syncwarp();
            if (copy)
                tma_load_2d(base + kOffStage + stg * kTile + k_lo * kDim, &tmap, 0, row,
                            full_bar + stg);
            if constexpr (MX) {
                // The keys' E8M0 words (byte g = group g) into the stage's block
                // for tcgen05.cp: row `lane` holds keys lane + 32 i.  A key after
                // the row's position or on an invalid page keeps a stale word;
                // its score is -inf whatever the tensor core makes of it.
                const uint32_t sfa = base + kOffSfa + stg * kSfBytes + lane * 16;
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int sk = s0 + lane + 32 * i;
                    if (live && sk <= pf_pos) {
                        const int lbk = sk >> lp;
                        const int blk = win_s[lbk - win];
                        if (lbk < b.max_blocks && (unsigned)blk < (unsigned)b.n_blocks)
                            cp_async_4(sfa + 4 * i,
                                       mxscale(ix.k.scale) +
                                           (((int64_t)blk << lp) + (sk & (P - 1))) * (kDim / 32));
                    }
                }
                cp_async_arrive_noinc(full_bar + stg);
            }
            // The tile's per-key scales into this producer's scale ring (read
            // by the paired epilogue group): lane l copies keys s0 + 4 l .. +3
            // (one page), or writes -1 where the page has no valid block.
            const int64_t kit = it >> 1;
            const int ss = (int)(kit % kScStages);
            uint64_t *sf = scfull_bar + pw * kScStages + ss;
            if (kit >= kScStages &&
                !mbar_wait(scempty_bar + pw * kScStages + ss, (uint32_t)((kit / kScStages) - 1) & 1,
                           st))
                break;
            {
                const int s4 = s0 + 4 * lane, lb4 = s4 >> lp;
                int blk4 = -1;
                if (live && lb4 <= last && lb4 < b.max_blocks) {
                    const int v = win_s[lb4 - win];
                    if ((unsigned)v < (unsigned)b.n_blocks)
                        blk4 = v;
                }
                const uint32_t d = smem_u32(sc_s + (pw * kScStages + ss) * kKeys + 4 * lane);
                if (blk4 >= 0 && ix.k.scale && !MX) {
                    cp_async_16(d, fscale(ix.k.scale) + ((int64_t)blk4 << lp) + (s4 & (P - 1)));
                    cp_async_arrive_noinc(sf);
                } else {  // no per-key scale (MXFP8 scales are the tensor core's)
                    const uint32_t v = __float_as_uint(blk4 >= 0 ? 1.f : -1.f);
                    st_shared_v4(d, v, v, v, v);
                    mbar_arrive(sf);
                }
            }
            advance(r, t, 2, tiles_per_row);
        }
    } else if (warp == kWarpMma0 || warp == kWarpMma1) {
        // ----------------------------------------------------------------- MMA
        const int pr = warp == kWarpMma0 ? 0 : 1;  // pair: items pr, pr + 2, ...
        const uint32_t idesc = idesc_e4m3(kKeys, kN);
        int r = (int)(j0 / tiles_per_row), t = (int)(j0 % tiles_per_row);
        int cur = -1, ri = -1, pos = -1, p = 0;
        int sfb_row = -1;  // MXFP8: query row whose scales this pair's TMEM holds
        int64_t m = 0;  // live tiles of this pair so far
        for (int64_t it = 0; it < n_items; it++) {
            if (r != cur) {
                cur = r;
                ++ri;
                p = ri & 1;
                pos = CAND ? ca.n - 1 : __ldg(b.q_pos + r);
                if (!mbar_wait(qfull_bar + p, (uint32_t)(ri >> 1) & 1, st))
                    break;
            }
            const bool mine = (int)(it & 1) == pr;
            const int stg = (int)(it % kStages);
            const bool live = t * kKeys <= pos;
            advance(r, t, 1, tiles_per_row);
            const bool row_ends = (it + 1 == n_items) || (r != cur);
            if (mine) {
                if (!mbar_wait(full_bar + stg, (uint32_t)(it / kStages) & 1, st))
                    break;
                if constexpr (CAND || MX)
                    fence_async_smem();  // cp.async pieces (generic proxy) -> tensor core
                if (live) {
                    const int c = (int)(m % kAccPerPair);
                    uint64_t *cf = cfull_bar + pr * kAccPerPair + c;
                    if (m >= kAccPerPair &&
                        !mbar_wait(cempty_bar + pr * kAccPerPair + c,
                                   (uint32_t)((m / kAccPerPair) - 1) & 1, st))
                        break;
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t d = tmem + (pr * kAccPerPair + c) * nB;
                        if constexpr (MX) {
                            // scale factors first: the key tile's, and once per
                            // query row this pair scores, the row's
                            const uint32_t sfa = tmem + kColSfa + (pr * kAccPerPair + c) * 4;
                            const uint32_t sfb = tmem + kColSfb + (pr * 2 + p) * 4;
                            tmem_cp_32x128b_x4(sfa, base + kOffSfa + stg * kSfBytes);
                            if (sfb_row != ri) {
                                tmem_cp_32x128b_x4(sfb, base + kOffSfb + p * kSfBytes);
                                sfb_row = ri;
                            }
#pragma unroll
                            for (int kk = 0; kk < kDim / 32; kk++) {
                                const uint64_t ad = smem_desc(
                                    base + kOffStage + stg * kTile + kk * 32, 16, 1024, kSwizzle128B);
                                const uint64_t bd = smem_desc(base + kOffQ + p * kTileB + kk * 32,
                                                              16, 1024, kSwizzle128B);
                                umma_mx_ss(d, ad, bd, idesc_mx_e4m3(kKeys, nB, kk), sfa, sfb,
                                           kk > 0);
                            }
                        } else {
#pragma unroll
                            for (int kk = 0; kk < kDim / 32; kk++) {
                                const uint64_t ad = smem_desc(
                                    base + kOffStage + stg * kTile + kk * 32, 16, 1024, kSwizzle128B);
                                const uint64_t bd = smem_desc(base + kOffQ + p * kTileB + kk * 32,
                                                              16, 1024, kSwizzle128B);
                                umma_f8_ss(d, ad, bd, idesc, kk > 0);
                            }
                        }
                        umma_commit(empty_bar + stg);
                        umma_commit(cf);
                    }
                    m++;
                } else if (lane == 0) {
                    mbar_arrive(empty_bar + stg);  // nothing was copied; release the slot
                }
            }
            if (row_ends && lane == 0)
                umma_commit(qempty_bar + p);  // the row's B operand is free once read
            __syncwarp();
        }
    } else if (warp >= kWarpPrep0 && warp < kWarpEpi0) {
        // -------------------------------------------------------------- q-prep
        // Thread pt splits dims [64 * half, +64) of head h into q_hi / q_lo.
        const int pt = tid - kWarpPrep0 * 32;
        const int h = pt >> 1, half = pt & 1;
        const int r_first = (int)(j0 / tiles_per_row);
        const int r_last = n_items > 0 ? (int)((j1 - 1) / tiles_per_row) : r_first - 1;
        for (int r = r_first; r <= r_last; r++) {
            const int ri = r - r_first, p = ri & 1;
            if (ri >= 2 && !mbar_wait(qempty_bar + p, (uint32_t)((ri - 2) >> 1) & 1, st))
                break;
            const uint32_t qb = base + kOffQ + p * kTileB;
            if constexpr (MX) {
                // dims [64 half, +64) of head h = MX groups 2 half, 2 half + 1
                uint32_t sbytes;  // this thread's two scale bytes, group 2 half in the low one
                if (ix.q_dtype == SI_MXE4M3) {
                    const int64_t rh = (int64_t)r * kHeads + h;
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        static_cast<const uint8_t *>(ix.q) + rh * kDim + half * 64);
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        const uint4 v = __ldg(src + c);
                        st_shared_v4(qb + sw128_offset(h, (uint32_t)(half * 4 + c)), v.x, v.y, v.z,
                                     v.w);
                    }
                    const uint8_t *qs = mxscale(ix.q_scale) + rh * (kDim / 32) + 2 * half;
                    sbytes = (uint32_t)__ldg(qs) | ((uint32_t)__ldg(qs + 1) << 8);
                } else {
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        static_cast<const uint16_t *>(ix.q) + ((int64_t)r * kHeads + h) * kDim +
                        half * 64);
                    sbytes = 0;
#pragma unroll
                    for (int gg = 0; gg < 2; gg++) {  // one MX group = 32 dims = 4 loads
                        uint32_t q2[16];
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            const uint4 v = __ldg(src + 4 * gg + i);
                            q2[4 * i] = v.x;
                            q2[4 * i + 1] = v.y;
                            q2[4 * i + 2] = v.z;
                            q2[4 * i + 3] = v.w;
                        }
                        uint32_t mb = 0;
#pragma unroll
                        for (int i = 0; i < 16; i++)
                            mb = max(mb, max(abs_bits(__uint_as_float(q2[i] << 16)),
                                             abs_bits(__uint_as_float(q2[i] & 0xFFFF0000u))));
                        const uint32_t sb = mx_scale_byte(mb);
                        sbytes |= sb << (8 * gg);
#pragma unroll
                        for (int c = 0; c < 2; c++) {  // 16 dims per 16-byte unit
                            uint32_t w4[4];
#pragma unroll
                            for (int j = 0; j < 4; j++) {
                                const uint32_t a = q2[8 * c + 2 * j], bb = q2[8 * c + 2 * j + 1];
                                w4[j] = mx_codes2(__uint_as_float(a << 16),
                                                  __uint_as_float(a & 0xFFFF0000u), sb) |
                                        (mx_codes2(__uint_as_float(bb << 16),
                                                   __uint_as_float(bb & 0xFFFF0000u), sb)
                                         << 16);
                            }
                            st_shared_v4(qb + sw128_offset(h, (uint32_t)(half * 4 + 2 * gg + c)),
                                         w4[0], w4[1], w4[2], w4[3]);
                        }
                    }
                }
                // head h's scale word (byte g = group g) for tcgen05.cp: row
                // h % 32, word h / 32 of the row buffer's block
                const uint32_t other = __shfl_xor_sync(0xffffffffu, sbytes, 1);
                if (half == 0) {
                    const uint32_t word = sbytes | (other << 16);
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(base + kOffSfb + p * kSfBytes +
                                                                 (h & 31) * 16 + (h >> 5) * 4),
                                 "r"(word)
                                 : "memory");
                    w_s[p * kHeads + h] = __ldg(ix.w + (int64_t)r * kHeads + h);
                }
                fence_async_smem();
                mbar_arrive(qfull_bar + p);
                continue;
            }
            if (ix.q_dtype == SI_E4M3) {
                // Stored FP8 query: its codes are the B operand (q_lo = 0) and
                // the per-(row, head) scale joins the head weight.
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    static_cast<const uint8_t *>(ix.q) + ((int64_t)r * kHeads + h) * kDim +
                    half * 64);
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const uint4 v = __ldg(src + c);
                    const uint32_t u = (uint32_t)(half * 4 + c);
                    st_shared_v4(qb + sw128_offset(h, u), v.x, v.y, v.z, v.w);
                    st_shared_v4(qb + sw128_offset(kHeads + h, u), 0u, 0u, 0u, 0u);
                }
                if (half == 0)
                    w_s[p * kHeads + h] = __ldg(ix.w + (int64_t)r * kHeads + h) *
                                          __ldg(fscale(ix.q_scale) + (int64_t)r * kHeads + h);
                fence_async_smem();
                mbar_arrive(qfull_bar + p);
                continue;
            }
            const uint4 *src = reinterpret_cast<const uint4 *>(
                static_cast<const uint16_t *>(ix.q) + ((int64_t)r * kHeads + h) * kDim + half * 64);
            uint32_t q2[32];  // 64 bf16 dims, two per word
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const uint4 v = __ldg(src + i);
                q2[4 * i] = v.x;
                q2[4 * i + 1] = v.y;
                q2[4 * i + 2] = v.z;
                q2[4 * i + 3] = v.w;
            }
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 32; i++) {
                amax = fmaxf(amax, fabsf(__uint_as_float(q2[i] << 16)));
                amax = fmaxf(amax, fabsf(__uint_as_float(q2[i] & 0xFFFF0000u)));
            }
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            // s_h = 2^e with max|q_h| / s_h in (224, 448]
            int e = 0;
            if (amax > 0.f) {
                e = (int)ceilf(log2f(amax / 448.f));
                while (ldexpf(amax, -e) > 448.f)
                    e++;
                while (ldexpf(amax, -(e - 1)) <= 448.f)
                    e--;
            }
            // x / s_h as one multiply by 2^-e when that is a normal float (the
            // same correctly rounded result as ldexpf)
            const bool pow2 = e >= -126 && e <= 126;
            const float inv_s = pow2 ? __int_as_float((127 - e) << 23) : 0.f;
            auto unscale = [&](float x) { return pow2 ? x * inv_s : ldexpf(x, -e); };
#pragma unroll
            for (int c = 0; c < 4; c++) {  // 16 dims per 16-byte unit
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int j = 0; j < 4; j++) {  // 4 dims per output word
                    uint32_t hw = 0, lw = 0;
#pragma unroll
                    for (int pr2 = 0; pr2 < 2; pr2++) {
                        const uint32_t word = q2[8 * c + 2 * j + pr2];  // dims 16c+4j+2pr2, +1
                        const float x0 = unscale(__uint_as_float(word << 16));
                        const float x1 = unscale(__uint_as_float(word & 0xFFFF0000u));
                        const uint16_t h2 = float2_to_e4m3x2(x0, x1);
                        const float2 hf = e4m3x2_to_float2(h2);
                        const uint16_t l2 = float2_to_e4m3x2(x0 - hf.x, x1 - hf.y);
                        hw |= (uint32_t)h2 << (16 * pr2);
                        lw |= (uint32_t)l2 << (16 * pr2);
                    }
                    hi[j] = hw;
                    lo[j] = lw;
                }
                const uint32_t u = (uint32_t)(half * 4 + c);
                st_shared_v4(qb + sw128_offset(h, u), hi[0], hi[1], hi[2], hi[3]);
                st_shared_v4(qb + sw128_offset(kHeads + h, u), lo[0], lo[1], lo[2], lo[3]);
            }
            if (half == 0)
                w_s[p * kHeads + h] = ldexpf(__ldg(ix.w + (int64_t)r * kHeads + h), e);
            fence_async_smem();
            mbar_arrive(qfull_bar + p);
        }
    } else if (warp >= kWarpEpi0) {
        // ------------------------------------------------------------ epilogue
        // Group g pairs with MMA warp g and owns items g, g + 2, ...; it walks
        // every item to keep the row bookkeeping.
        const int g = (warp - kWarpEpi0) >> 2;
        const int et = (tid - kWarpEpi0 * 32) & 127;  // key row = TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        int r = (int)(j0 / tiles_per_row), t = (int)(j0 % tiles_per_row);
        int cur = -1, ri = -1, pos = -1, p = 0;
        int64_t m = 0;
        for (int64_t it = 0; it < n_items; it++) {
            if (r != cur) {
                cur = r;
                ++ri;
                p = ri & 1;
                pos = CAND ? ca.n - 1 : __ldg(b.q_pos + r);  // candidates: slots 0..n-1
                if (!mbar_wait(qfull_bar + p, (uint32_t)(ri >> 1) & 1, st))
                    break;
            }
            const int rr = r, s0 = t * kKeys, s = s0 + et;
            advance(r, t, 1, tiles_per_row);
            const bool row_ends = (it + 1 == n_items) || (r != cur);
            const bool live = s0 <= pos;
            if ((int)(it & 1) == g) {
                // this key's scale from the producer's ring: -1 marks a key
                // without a valid block (scores -inf), 1 an unscaled cache
                const int64_t kit = it >> 1;
                const int ss = (int)(kit % kScStages);
                if (!mbar_wait(scfull_bar + g * kScStages + ss, (uint32_t)(kit / kScStages) & 1, st))
                    break;
                const float scv = sc_s[(g * kScStages + ss) * kKeys + et];
                mbar_arrive(scempty_bar + g * kScStages + ss);
                if (live) {
                    const float sc = s <= pos ? scv : -1.f;
                    const int c = (int)(m % kAccPerPair);
                    if (!mbar_wait(cfull_bar + g * kAccPerPair + c,
                                   (uint32_t)(m / kAccPerPair) & 1, st))
                        break;
                    tc_fence_after();
                    const float4 *w4 = reinterpret_cast<const float4 *>(w_s + p * kHeads);
                    const uint32_t acc = tmem + (g * kAccPerPair + c) * nB + lane_off;
                    // partial head sums in two packed pairs (0.0f has all bits 0)
                    uint64_t p01 = 0, p23 = 0;
                    if constexpr (MX) {
                        // D[key, h] is the MXFP8 logit: w_h * ReLU(D), two heads per fma
                        uint32_t v0[32], v1[32];
                        tmem_ld32(acc, v0);
                        tmem_ld32(acc + 32, v1);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 64; i += 4) {
                            const float4 wv = w4[i >> 2];
                            const uint32_t *v = i < 32 ? v0 + i : v1 + (i - 32);
                            f32x2_fma(p01, f32x2_pack(wv.x, wv.y),
                                      f32x2_pack(fmaxf(__uint_as_float(v[0]), 0.f),
                                                 fmaxf(__uint_as_float(v[1]), 0.f)));
                            f32x2_fma(p23, f32x2_pack(wv.z, wv.w),
                                      f32x2_pack(fmaxf(__uint_as_float(v[2]), 0.f),
                                                 fmaxf(__uint_as_float(v[3]), 0.f)));
                        }
                    }
#pragma unroll
                    for (int hh = 0; hh < (MX ? 0 : 2); hh++) {  // heads [32 hh, 32 hh + 32)
                        uint32_t vh[32], vl[32];
                        tmem_ld32(acc + hh * 32, vh);
                        tmem_ld32(acc + kHeads + hh * 32, vl);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 wv = w4[(hh * 32 + i) >> 2];
                            // logit = q_hi term + q_lo term, two heads per add
                            float lg[4];
#pragma unroll
                            for (int k = 0; k < 4; k += 2) {
                                const float2 s2 = f32x2_unpack(f32x2_add(
                                    f32x2_pack(__uint_as_float(vh[i + k]),
                                               __uint_as_float(vh[i + k + 1])),
                                    f32x2_pack(__uint_as_float(vl[i + k]),
                                               __uint_as_float(vl[i + k + 1]))));
                                lg[k] = s2.x;
                                lg[k + 1] = s2.y;
                            }
                            // w_h * ReLU(logit), two heads per fma
                            f32x2_fma(p01, f32x2_pack(wv.x, wv.y),
                                      f32x2_pack(fmaxf(lg[0], 0.f), fmaxf(lg[1], 0.f)));
                            f32x2_fma(p23, f32x2_pack(wv.z, wv.w),
                                      f32x2_pack(fmaxf(lg[2], 0.f), fmaxf(lg[3], 0.f)));
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(cempty_bar + g * kAccPerPair + c);
                    const float2 pa = f32x2_unpack(p01), pc = f32x2_unpack(p23);
                    const float sum = (pa.x + pa.y) + (pc.x + pc.y);
                    if (s < ld)
                        scores[(int64_t)rr * ld + s] = sc >= 0.f ? sum * sc + 0.0f : -INFINITY;
                    m++;
                } else if (s < ld) {
                    scores[(int64_t)rr * ld + s] = -INFINITY;  // tile after the query
                }
            }
            if (row_ends)
                mbar_arrive(qempty_bar + p);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma0)
        tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool indexer_tc_supported(const si_batch &b, const si_indexer &ix, int64_t ld)
{
    (void)ld;
    // whole pages are copied as tensor boxes: rows packed (stride 128 bytes),
    // page size a power of two >= 8, physical row indices within int32
    const bool pow2_page = b.page_size >= 8 && (b.page_size & (b.page_size - 1)) == 0;
    const bool mx = ix.k.dtype == SI_MXE4M3;
    const bool q_ok = mx ? (ix.q_dtype == SI_BF16 ||
                            (ix.q_dtype == SI_MXE4M3 && ((uintptr_t)ix.q_scale % 4) == 0))
                         : (ix.q_dtype == SI_BF16 || (ix.q_dtype == SI_E4M3 && ix.q_scale));
    return pow2_page && q_ok && (ix.k.dtype == SI_E4M3 || mx) && ix.n_heads == kHeads &&
           ix.head_dim == kDim && ix.k.row_stride == kDim &&
           (int64_t)b.n_blocks * b.page_size < (int64_t)INT32_MAX &&
           ((uintptr_t)ix.q % 16) == 0 && ((uintptr_t)ix.k.data % 16) == 0 &&
           ((uintptr_t)ix.k.scale % 16) == 0;
}

namespace {

cudaError_t launch_indexer_tc_any(const si_batch &b, const si_indexer &ix, const CandArgs &ca,
                                  float *scores, int64_t ld, unsigned int *st, cudaStream_t s)
{
    // Per-device launch facts (SM count, shared-memory opt-in), set up once.
    static std::once_flag once[kMaxDevices];
    static int sms_of[kMaxDevices];
    static cudaError_t err_of[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::call_once(once[dev], [dev] {
        cudaError_t r = cudaDeviceGetAttribute(&sms_of[dev], cudaDevAttrMultiProcessorCount, dev);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(k_indexer_tc<false, false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(k_indexer_tc<true, false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(k_indexer_tc<false, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        err_of[dev] = r;
    });
    if (err_of[dev] != cudaSuccess)
        return err_of[dev];
    CUtensorMap tmap;
    e = make_tmap_2d_u8_sw128(&tmap, ix.k.data, kDim, (uint64_t)b.n_blocks * b.page_size,
                              (uint64_t)ix.k.row_stride, kDim,
                              (uint32_t)std::min(b.page_size, kKeys));
    if (e != cudaSuccess)
        return e;
    const int tiles_per_row = (int)((ld + kKeys - 1) / kKeys);
    const int64_t total = (int64_t)b.n_q * tiles_per_row;
    const int64_t grid = std::min<int64_t>(total, (int64_t)sms_of[dev]);  // one CTA per SM
    if (ca.cand && ix.k.dtype == SI_MXE4M3)
        return cudaErrorNotSupported;  // candidate lists take per-row FP8 scales
    count_launch();
    if (ca.cand)
        k_indexer_tc<true, false><<<(unsigned)grid, kThreads, kSmemBytes, s>>>(
            tmap, b, ix, scores, ld, total, tiles_per_row, st, ca);
    else if (ix.k.dtype == SI_MXE4M3)
        k_indexer_tc<false, true><<<(unsigned)grid, kThreads, kSmemBytes, s>>>(
            tmap, b, ix, scores, ld, total, tiles_per_row, st, ca);
    else
        k_indexer_tc<false, false><<<(unsigned)grid, kThreads, kSmemBytes, s>>>(
            tmap, b, ix, scores, ld, total, tiles_per_row, st, ca);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer_tc(const si_batch &b, const si_indexer &ix, float *scores, int64_t ld,
                              unsigned int *st, cudaStream_t s)
{
    return launch_indexer_tc_any(b, ix, CandArgs{nullptr, 0, 0}, scores, ld, st, s);
}

cudaError_t launch_indexer_tc_cand(const si_batch &b, const si_indexer &ix, const int32_t *cand,
                                   int64_t ld_cand, int32_t n_cand, float *scores, int64_t ld,
                                   unsigned int *st, cudaStream_t s)
{
    return launch_indexer_tc_any(b, ix, CandArgs{cand, ld_cand, n_cand}, scores, ld, st, s);
}

}  // namespace si
