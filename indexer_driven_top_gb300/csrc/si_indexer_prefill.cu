// si_indexer_prefill.cu -- tensor-core indexer for a causal prefill: many
// query rows of one sequence over a paged FP8 key cache.
//
// "Day0 Inference Support and Performance Optimization for New Architecture
// LLMs": section 2.2 (every query row scores all earlier positions; per-head
// scores are aggregated with head weights), section 4.1 (the scoring reads
// the paged K-cache directly) and section 6.2 (in a causal prefill the
// scoring work of a row grows with its position).  Score of key s for row r:
//     k_scale[s] * sum_h w[r,h] * ReLU(q[r,h,:] . k[s,:])
//
// GB300 mapping.  All rows of a prefill score the same keys, so one key tile
// (128 keys x 128 e4m3 bytes, UMMA A operand, landed by TMA) serves a block
// of query rows at once, and the B operand is always 256 rows wide (UMMA N =
// 256) so that every key byte brought in feeds a full-width UMMA:
//   * bf16 query: four rows per block, each row's 64 heads split exactly into
//     two e4m3 terms as in the decode indexer (q = s_h (q_hi + q_lo), s_h a
//     power of two folded into the head weight).  The two terms are laid
//     side by side along K (a q_hi tile and a q_lo tile), and eight UMMAs
//     accumulate key . q_hi and key . q_lo into the same 64 columns per row,
//     so the epilogue reads one logit per head (the key tile serves as A for
//     both halves of K);
//   * FP8 query with a per-(row, head) scale (section 4.3 quantises the
//     indexer query before scoring): four rows per block, 64 heads each, the
//     scale folded into the head weight: 4 x 64 B rows, twice the scores per
//     UMMA and per TMEM column read.
//   * MXFP8 query and keys (section 5.1; a bf16 query is converted per group
//     of 32 by the q-prep threads, bit-identical to si_quant_mxfp8): the
//     block-scaled kind::mxf8f6f4 UMMA applies each group's scales inside the
//     tensor core.  Its scale factors take TMEM columns, so the accumulators
//     are 192 wide (three rows of 64 heads per block) instead of 256; the
//     keys' scale words land per stage in the 32 x 16-byte block tcgen05.cp
//     copies to TMEM (row L: keys L, L+32, L+64, L+96), the rows' per block.
// The causal triangle is balanced by splitting the list of (row block, key
// tile) items -- block by block, each block's live tiles (those at or before
// its last position) -- into equal contiguous ranges, one per CTA: every CTA
// gets the same number of tiles whatever the number of blocks, and a block
// whose tiles straddle two CTAs has its query prepared by both.  Blocks are
// listed head and tail alternately (0, nb-1, 1, nb-2, ...: the pairing
// section 6.3 uses for context-parallel shards), so that every range mixes
// short and long blocks and the per-block costs spread evenly too.
//
// One persistent CTA per SM, 16 warps:
//   warps 0, 2  -- producers, alternate items (a bulk tensor copy holds its
//                  issuing warp for several hundred cycles): per item (block,
//                  key tile) the TMA copies of the tile's key pages into a
//                  ring of key stages, and the keys' scales into the
//                  producer's scale ring (cp.async);
//   warp 1      -- MMA: four (bf16 query: eight) kind::f8f6f4 UMMAs (M 128,
//                  N 256, K 32) per item into one of two TMEM accumulators
//                  (256 columns each);
//   warp 3      -- writes -inf into each block's score columns past its live
//                  tiles with bulk copies from a -inf buffer in shared memory
//                  (the copy engine does the writing, off the pipeline); the
//                  fused calls, whose Top-K reads only positions up to each
//                  row's own, skip it;
//   warps 4..7  -- q-prep: writes each block's query rows into the B operand
//                  (double-buffered);
//   warps 8..15 -- two epilogue groups that take alternate items: per key
//                  (TMEM lane) and row, ReLU, head weights, scale, store; an
//                  item's accumulator is released as soon as its last piece
//                  has been loaded.
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

constexpr int kKeys = 128;            // keys per tile = UMMA M
constexpr int kHeads = 64;            // indexer heads
constexpr int kDim = 128;             // head dim = bytes per e4m3 key row = UMMA K
constexpr int kN = 256;               // UMMA N (bf16 and FP8 query): B rows of one block
constexpr int kMaxRows = 4;           // query rows per block
// Query modes: a bf16 query split into q_hi / q_lo terms, an FP8 query with a
// per-(row, head) scale, an MXFP8 query (block-scaled MMA).  Every mode puts
// a row's 64 heads in 64 B rows (and accumulator columns).
constexpr int kQBf16 = 0, kQFp8 = 1, kQMx = 2;
template <int QM> constexpr int mma_n() { return QM == kQMx ? 3 * kHeads : kN; }
template <int QM> constexpr int rows_per_block() { return mma_n<QM>() / kHeads; }
// What a block's query preparation costs, in tiles of work, when the balance
// charges it to the CTA whose range holds the block.
template <int QM> constexpr int block_cost() { return QM == kQFp8 ? 4 : 8; }
constexpr int kScStages = 4;          // scale ring depth per epilogue group
constexpr int kThreads = 16 * 32;
constexpr int kWarpProd0 = 0, kWarpProd1 = 2;  // producers: items of parity 0 / 1
constexpr int kWarpMma = 1, kWarpTail = 3, kWarpPrep0 = 4, kWarpEpi0 = 8;

constexpr uint32_t kTile = kKeys * kDim;    // 16 KB, SW128 K-major
constexpr uint32_t kTileB = kN * kDim;      // 32 KB, SW128 K-major
// MXFP8 scale words for tcgen05.cp (32 rows x 16 bytes per block): one block
// per key stage, two per B buffer (B rows 0..127 and 128..255)
constexpr uint32_t kSfBytes = 512;
constexpr uint32_t kNinfBytes = 4096;       // -inf source of the tail writer's copies

// Shared-memory layout of one query mode: the key-tile ring, two B buffers
// (a bf16 query takes a q_hi and a q_lo tile per buffer, so its ring is
// shorter), head weights, block-table windows, the epilogue scale rings, the
// MXFP8 scale blocks, the -inf buffer and the barriers.
template <int QM> struct Lay {
    static constexpr int kStages = QM == kQBf16 ? 5 : 8;
    static constexpr uint32_t kQParts = QM == kQBf16 ? 2 : 1;
    static constexpr uint32_t kQBuf = kQParts * kTileB;
    static constexpr uint32_t kOffStage = 0;
    static constexpr uint32_t kOffQ = kOffStage + kStages * kTile;             // [2] B operands
    static constexpr uint32_t kOffW = kOffQ + 2 * kQBuf;                        // [2][rows][64]
    static constexpr uint32_t kOffWin = kOffW + 2 * kMaxRows * kHeads * 4;      // 2 x 32 entries
    static constexpr uint32_t kOffSc = kOffWin + 2 * 32 * 4;                    // [2][kScStages][128]
    static constexpr uint32_t kOffSfa = kOffSc + 2 * kScStages * kKeys * 4;     // [kStages]
    static constexpr uint32_t kOffSfb = kOffSfa + kStages * kSfBytes;           // [2][2]
    static constexpr uint32_t kOffNinf = kOffSfb + 4 * kSfBytes;
    static constexpr uint32_t kOffBar = kOffNinf + kNinfBytes;
    static constexpr uint32_t kSmemBytes = kOffBar + 512 + 1024;               // + alignment slack
    static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};
// TMEM: two accumulators of mma_n columns; MXFP8 adds 4 scale columns per
// accumulator (keys) and 8 per B buffer (query rows) after them.
constexpr uint32_t kTmemCols = 2 * kN;  // 512
constexpr uint32_t kColSfa = 2 * 3 * kHeads;
constexpr uint32_t kColSfb = kColSfa + 2 * 4;
static_assert(kColSfb + 2 * 8 <= kTmemCols, "TMEM columns");

__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v)
{
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
    return make_float2(__half2float(__ushort_as_half(h.x)), __half2float(__ushort_as_half(h.y)));
}

__device__ __forceinline__ uint16_t float2_to_e4m3x2(float a, float b)
{
    return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Rows of block `blk` and its live key tiles (those holding a key at or
// before the block's last position; at least one, so that every block's
// score rows are written).
template <int kRows>
__device__ __forceinline__ void block_shape(const si_batch &b, int blk, int tiles_ld, int &r0,
                                            int &nrows, int &T)
{
    r0 = blk * kRows;
    nrows = min(kRows, b.n_q - r0);
    int pmax = -1;
    for (int j = 0; j < nrows; j++)
        pmax = max(pmax, __ldg(b.q_pos + r0 + j));
    T = max(1, min(tiles_ld, (pmax + kKeys) / kKeys));
}

// Block at position i of the item list: head and tail blocks alternately.
__device__ __forceinline__ int block_at(int i, int nb) { return (i & 1) ? nb - 1 - (i >> 1) : i >> 1; }

// This CTA's range of the item list: from tile t0 of the block at list
// position b0, n items.
struct Span {
    int b0, t0;
    int64_t n;
};

// The CTAs' ranges are equal shares of a cost in which every block weighs
// its tiles plus kCost: a block's query preparation is not hidden behind a
// block of few tiles, and a range holding more blocks ends later.  Found by
// all threads of the CTA together: thread i sums the tiles of blocks
// [i m, (i + 1) m), a block-wide scan places those sums (the cost before
// block j is the tiles before it plus kCost j), and the threads whose blocks
// hold the range's two ends turn them into items: an end inside a block's
// kCost part is that block's first tile.  `wsum` holds kThreads / 32 + 6
// entries of shared memory.
template <int kRows, int kCost>
__device__ Span find_span(const si_batch &b, int nb, int tiles_ld, long long *wsum)
{
    constexpr int kWarps = kThreads / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m = (nb + kThreads - 1) / kThreads;
    const int lo = min(nb, tid * m), hi = min(nb, lo + m);
    long long local = 0;
    for (int i = lo; i < hi; i++) {
        int r0, nrows, T;
        block_shape<kRows>(b, block_at(i, nb), tiles_ld, r0, nrows, T);
        local += T;
    }
    long long x = local;  // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        long long t = lane < kWarps ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o)
                t += y;
        }
        if (lane < kWarps)
            wsum[lane] = t;  // inclusive warp totals
    }
    __syncthreads();
    const long long before = (warp > 0 ? wsum[warp - 1] : 0) + x - local;  // tiles
    const long long total = wsum[kWarps - 1];
    const long long cbefore = before + (long long)kCost * lo;               // cost
    const long long clocal = local + (long long)kCost * (hi - lo);
    const long long ctotal = total + (long long)kCost * nb;
    const long long c0 = ctotal * blockIdx.x / gridDim.x;
    const long long c1 = ctotal * (blockIdx.x + 1) / gridDim.x;
    __syncthreads();  // every thread has read the totals before they are reused
    // cost position c -> (list position, tile in block, item index)
    auto locate = [&](long long c, int slot) {
        long long acc = before, cacc = cbefore;
        for (int i = lo; i < hi; i++) {
            int r0, nrows, T;
            block_shape<kRows>(b, block_at(i, nb), tiles_ld, r0, nrows, T);
            if (c < cacc + kCost + T) {
                const long long t = c - cacc - kCost > 0 ? c - cacc - kCost : 0;
                wsum[slot] = i;
                wsum[slot + 1] = t;
                wsum[slot + 2] = acc + t;
                return;
            }
            acc += T;
            cacc += kCost + T;
        }
    };
    if (cbefore <= c0 && c0 < cbefore + clocal)
        locate(c0, kWarps);
    if (cbefore <= c1 && c1 < cbefore + clocal)
        locate(c1, kWarps + 3);
    if (tid == 0 && c1 >= ctotal)
        wsum[kWarps + 5] = total;  // the last range ends after the last item
    __syncthreads();
    Span sp{0, 0, 0};
    if (c0 < c1) {
        sp.b0 = (int)wsum[kWarps];
        sp.t0 = (int)wsum[kWarps + 1];
        sp.n = wsum[kWarps + 5] - wsum[kWarps + 2];
    }
    return sp;
}

// Walks a span block by block: the current list position `pos` (block
// block_at(pos, nb)), its first tile in the span `t_first`, and the items
// still to come.
struct SpanWalk {
    int pos, nb, t_first;
    int64_t left;
    __device__ SpanWalk(const Span &sp, int nb_) : pos(sp.b0), nb(nb_), t_first(sp.t0), left(sp.n) {}
    __device__ bool more() const { return left > 0; }
    __device__ int blk() const { return block_at(pos, nb); }
    // one past the last tile of the current block (T tiles) inside the span
    __device__ int end_of(int T) const
    {
        return (int64_t)T < t_first + left ? T : (int)(t_first + left);
    }
    __device__ void next(int t_end)
    {
        left -= t_end - t_first;
        pos++;
        t_first = 0;
    }
};

template <int QM>
__global__ void __launch_bounds__(kThreads, 1)
k_indexer_prefill(const __grid_constant__ CUtensorMap tmap, si_batch b, si_indexer ix,
                  float *scores, int64_t ld, int n_blocks_rows, int fill_tail, unsigned int *st)
{
    constexpr bool MX = QM == kQMx;
    constexpr int kRows = rows_per_block<QM>();
    constexpr int kRowN = kHeads;  // B rows (accumulator columns) per query row
    constexpr int nB = mma_n<QM>();
    using L = Lay<QM>;
    constexpr int kStages = L::kStages;
    constexpr uint32_t kOffStage = L::kOffStage, kOffQ = L::kOffQ, kOffW = L::kOffW,
                       kOffWin = L::kOffWin, kOffSc = L::kOffSc, kOffSfa = L::kOffSfa,
                       kOffSfb = L::kOffSfb, kOffNinf = L::kOffNinf, kOffBar = L::kOffBar;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - smem_u32(smem_raw));
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(gbase + kOffBar);  // [kStages]
    uint64_t *empty_bar = full_bar + kStages;                             // [kStages]
    uint64_t *cfull_bar = empty_bar + kStages;                            // [2]
    uint64_t *cempty_bar = cfull_bar + 2;                                 // [2]
    uint64_t *qfull_bar = cempty_bar + 2;                                 // [2]
    uint64_t *qempty_bar = qfull_bar + 2;                                 // [2]
    uint64_t *scfull_bar = qempty_bar + 2;                                // [2][kScStages]
    uint64_t *scempty_bar = scfull_bar + 2 * kScStages;                   // [2][kScStages]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(scempty_bar + 2 * kScStages);
    float *w_s = reinterpret_cast<float *>(gbase + kOffW);
    volatile int *win_all = reinterpret_cast<volatile int *>(gbase + kOffWin);
    float *sc_s = reinterpret_cast<float *>(gbase + kOffSc);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    griddep_launch_dependents();  // the Top-K kernel may be scheduled as CTAs finish
    const int tiles_ld = (int)((ld + kKeys - 1) / kKeys);

    if (tid == 0) {
        for (int i = 0; i < kStages; i++) {
            // producer's expect_tx arrival (MXFP8: and its 32 lanes' cp.async arrivals)
            mbar_init(full_bar + i, MX ? 33 : 1);
            mbar_init(empty_bar + i, 1);  // MMA commit
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(cfull_bar + i, 1);             // MMA commit
            mbar_init(cempty_bar + i, 128);          // epilogue group
            mbar_init(qfull_bar + i, 128);           // q-prep threads
            mbar_init(qempty_bar + i, 1 + 2 * 128);  // MMA commit + both epilogue groups
        }
        for (int i = 0; i < 2 * kScStages; i++) {
            mbar_init(scfull_bar + i, 32);    // producer lanes (copy landed or sentinel)
            mbar_init(scempty_bar + i, 128);  // epilogue group read the scales
        }
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
    const int P = b.page_size;
    const int lp = 31 - __clz(P);  // page_size is a power of two >= 8
    const int seq = __ldg(b.q_seq);  // every row belongs to this sequence
    __shared__ long long span_scratch[kThreads / 32 + 6];
    const Span work = find_span<kRows, block_cost<QM>()>(b, n_blocks_rows, tiles_ld, span_scratch);

    if (warp == kWarpProd0 || warp == kWarpProd1) {
        // ------------------------------------------------------------ producer
        // Two producer warps take alternate items (a bulk tensor copy holds
        // its issuing warp for several hundred cycles); producer pw also
        // fills the scale ring of epilogue group pw.
        const int pw = warp == kWarpProd0 ? 0 : 1;
        volatile int *win_s = win_all + pw * 32;
        const int span = min(P, kKeys);  // keys of one page inside one tile
        int win = -1;                    // window: win_s[l] = block-table entry win + l
        SpanWalk walk(work, n_blocks_rows);
        int64_t it = 0;
        bool ok = true;
        for (; ok && walk.more(); ) {
            const int blk = walk.blk();
            int r0, nrows, T;
            block_shape<kRows>(b, blk, tiles_ld, r0, nrows, T);
            int pmax = -1;
            for (int j = 0; j < nrows; j++)
                pmax = max(pmax, __ldg(b.q_pos + r0 + j));
            const int t1 = walk.end_of(T);
            for (int t = walk.t_first; t < t1; t++, it++) {
                if ((int)(it & 1) != pw)
                    continue;
                const int stg = (int)(it % kStages);
                if (it >= kStages &&
                    !mbar_wait(empty_bar + stg, (uint32_t)((it / kStages) - 1) & 1, st)) {
                    ok = false;
                    break;
                }
                const int s0 = t * kKeys;
                const int first = s0 >> lp;
                const int last = min(s0 + kKeys - 1, pmax) >> lp;
                if (win < 0 || first < win || last >= win + 32) {
                    win = first;
                    const int lb = first + lane;
                    int v = -1;
                    if ((unsigned)seq < (unsigned)b.n_seq && lb < b.max_blocks)
                        v = __ldg(b.block_table + (int64_t)seq * b.max_blocks + lb);
                    win_s[lane] = v;
                    __syncwarp();
                }
                // lane l handles page first + l of the tile
                const int lb = first + lane;
                bool copy = false;
                int row = 0, k_lo = 0;
                if (lane < 16 && lb <= last) {
                    const int blkid = win_s[lb - win];
                    if (lb < b.max_blocks && (unsigned)blkid < (unsigned)b.n_blocks) {
                        copy = true;
                        k_lo = max(lb << lp, s0) - s0;
                        row = (blkid << lp) + (s0 + k_lo - (lb << lp));
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
                    // the keys' E8M0 words into the stage's tcgen05.cp block, row
                    // `lane` = keys lane + 32 i; a key after the block's last
                    // position or on an invalid page keeps a stale word (its
                    // score is -inf)
                    const uint32_t sfa = base + kOffSfa + stg * kSfBytes + lane * 16;
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const int sk = s0 + lane + 32 * i;
                        if (sk <= pmax) {
                            const int lbk = sk >> lp;
                            const int blkk = win_s[lbk - win];
                            if (lbk < b.max_blocks && (unsigned)blkk < (unsigned)b.n_blocks)
                                cp_async_4(sfa + 4 * i, mxscale(ix.k.scale) +
                                                            (((int64_t)blkk << lp) + (sk & (P - 1))) *
                                                                (kDim / 32));
                        }
                    }
                    cp_async_arrive_noinc(full_bar + stg);
                }
                // scales of the tile's keys into the ring of epilogue group pw
                const int g = pw;
                const int64_t kit = it >> 1;
                const int ss = (int)(kit % kScStages);
                uint64_t *sf = scfull_bar + g * kScStages + ss;
                if (kit >= kScStages &&
                    !mbar_wait(scempty_bar + g * kScStages + ss,
                               (uint32_t)((kit / kScStages) - 1) & 1, st)) {
                    ok = false;
                    break;
                }
                const int s4 = s0 + 4 * lane, lb4 = s4 >> lp;
                int blk4 = -1;
                if (lb4 <= last && lb4 < b.max_blocks) {
                    const int v = win_s[lb4 - win];
                    if ((unsigned)v < (unsigned)b.n_blocks)
                        blk4 = v;
                }
                const uint32_t d = smem_u32(sc_s + (g * kScStages + ss) * kKeys + 4 * lane);
                if (blk4 >= 0 && ix.k.scale && !MX) {
                    cp_async_16(d, fscale(ix.k.scale) + ((int64_t)blk4 << lp) + (s4 & (P - 1)));
                    cp_async_arrive_noinc(sf);
                } else {
                    const uint32_t v = __float_as_uint(blk4 >= 0 ? 1.f : -1.f);
                    st_shared_v4(d, v, v, v, v);
                    mbar_arrive(sf);
                }
            }
            walk.next(t1);
        }
        cp_async_commit();
        cp_async_wait<0>();  // nothing may land after the block has moved on
    } else if (warp == kWarpMma) {
        // ----------------------------------------------------------------- MMA
        const uint32_t idesc = idesc_e4m3(kKeys, nB);
        SpanWalk walk(work, n_blocks_rows);
        int64_t it = 0;
        int bi = 0;
        bool ok = true;
        for (; ok && walk.more(); bi++) {
            int r0, nrows, T;
            block_shape<kRows>(b, walk.blk(), tiles_ld, r0, nrows, T);
            const int t1 = walk.end_of(T);
            const int p = bi & 1;
            if (!mbar_wait(qfull_bar + p, (uint32_t)(bi >> 1) & 1, st))
                break;
            if constexpr (MX) {
                // the block's query scales into TMEM (B rows 0..127, 128..255);
                // the MMAs that read this buffer's columns last (block bi - 2)
                // are done: the q-prep waited for their commit before writing
                fence_async_smem();
                if (lane == 0) {
                    tmem_cp_32x128b_x4(tmem + kColSfb + p * 8, base + kOffSfb + (2 * p) * kSfBytes);
                    tmem_cp_32x128b_x4(tmem + kColSfb + p * 8 + 4,
                                       base + kOffSfb + (2 * p + 1) * kSfBytes);
                }
                __syncwarp();
            }
            for (int t = walk.t_first; t < t1; t++, it++) {
                const int stg = (int)(it % kStages);
                const int g = (int)(it & 1);
                const int64_t mg = it >> 1;  // this accumulator's use count
                if (!mbar_wait(full_bar + stg, (uint32_t)(it / kStages) & 1, st) ||
                    (mg >= 1 && !mbar_wait(cempty_bar + g, (uint32_t)(mg - 1) & 1, st))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if constexpr (MX)
                    fence_async_smem();  // the scale words landed by cp.async (generic proxy)
                if (lane == 0) {
                    const uint32_t dacc = tmem + g * nB;
                    if constexpr (MX) {
                        const uint32_t sfa = tmem + kColSfa + g * 4, sfb = tmem + kColSfb + p * 8;
                        tmem_cp_32x128b_x4(sfa, base + kOffSfa + stg * kSfBytes);
#pragma unroll
                        for (int kk = 0; kk < kDim / 32; kk++) {
                            const uint64_t ad = smem_desc(base + kOffStage + stg * kTile + kk * 32,
                                                          16, 1024, kSwizzle128B);
                            const uint64_t bd = smem_desc(base + kOffQ + p * L::kQBuf + kk * 32, 16,
                                                          1024, kSwizzle128B);
                            umma_mx_ss(dacc, ad, bd, idesc_mx_e4m3(kKeys, nB, kk), sfa, sfb,
                                       kk > 0);
                        }
                    } else {
                        // K blocks of the B buffer: q_hi (and, for a bf16 query,
                        // then q_lo), each against the same K block of the keys
#pragma unroll
                        for (int kk = 0; kk < (int)L::kQParts * (kDim / 32); kk++) {
                            const uint64_t ad =
                                smem_desc(base + kOffStage + stg * kTile + (kk & 3) * 32, 16, 1024,
                                          kSwizzle128B);
                            const uint64_t bd = smem_desc(base + kOffQ + p * L::kQBuf +
                                                              (kk >> 2) * kTileB + (kk & 3) * 32,
                                                          16, 1024, kSwizzle128B);
                            umma_f8_ss(dacc, ad, bd, idesc, kk > 0);
                        }
                    }
                    umma_commit(empty_bar + stg);
                    umma_commit(cfull_bar + g);
                }
                __syncwarp();
            }
            if (ok && lane == 0)
                umma_commit(qempty_bar + p);  // the block's B operand is free once read
            __syncwarp();
            walk.next(t1);
        }
    } else if (warp == kWarpTail && fill_tail) {
        // -------------------------------------------------------- tail writer
        // Score columns past a block's live tiles are -inf; the CTA that
        // scores the block's last tile writes them.  The 16-byte aligned
        // middle of each row's tail goes by bulk copies of a -inf buffer
        // (lane l issues chunks l, l + 32, ...), the ragged ends by plain
        // stores.
        float *ninf_s = reinterpret_cast<float *>(gbase + kOffNinf);
        for (int i = lane; i < (int)(kNinfBytes / 4); i += 32)
            ninf_s[i] = -INFINITY;
        fence_async_smem();  // generic-proxy writes -> the copy engine's reads
        __syncwarp();
        griddep_wait();  // the score rows may still be read by the previous kernel
        constexpr int64_t kChunk = kNinfBytes / 4;  // floats per copy
        SpanWalk walk(work, n_blocks_rows);
        for (; walk.more();) {
            int r0, nrows, T;
            block_shape<kRows>(b, walk.blk(), tiles_ld, r0, nrows, T);
            const int t1 = walk.end_of(T);
            walk.next(t1);
            const int64_t c0 = (int64_t)T * kKeys;
            if (t1 != T || c0 >= ld)
                continue;
            for (int j = 0; j < nrows; j++) {
                float *row = scores + (int64_t)(r0 + j) * ld;
                int64_t a = c0;  // first 16-byte aligned column at or after c0
                while (a < ld && ((uintptr_t)(row + a) & 15) != 0)
                    a++;
                const int64_t nv = (ld - a) & ~(int64_t)3;  // floats of the aligned middle
                if (lane < a - c0)
                    row[c0 + lane] = -INFINITY;
                if (lane < ld - (a + nv))
                    row[a + nv + lane] = -INFINITY;
                for (int64_t c = (int64_t)lane * kChunk; c < nv; c += 32 * kChunk)
                    bulk_s2g(row + a + c, smem_u32(ninf_s),
                             (uint32_t)(4 * (nv - c < kChunk ? nv - c : kChunk)));
            }
        }
        bulk_commit();
        bulk_wait<0>();  // every copy done before the block exits
    } else if (warp >= kWarpPrep0 && warp < kWarpEpi0) {
        // -------------------------------------------------------------- q-prep
        // Thread pt prepares dims [64 half, +64) of head h of every row.
        const int pt = tid - kWarpPrep0 * 32;
        const int h = pt >> 1, half = pt & 1;
        SpanWalk walk(work, n_blocks_rows);
        int bi = 0;
        for (; walk.more(); bi++) {
            int r0, nrows, T;
            block_shape<kRows>(b, walk.blk(), tiles_ld, r0, nrows, T);
            walk.next(walk.end_of(T));
            const int p = bi & 1;
            if (bi >= 2 && !mbar_wait(qempty_bar + p, (uint32_t)((bi - 2) >> 1) & 1, st))
                break;
            const uint32_t qb = base + kOffQ + p * L::kQBuf;
            if constexpr (MX) {
                // dims [64 half, +64) of head h of each row = MX groups 2 half,
                // 2 half + 1; B row n = j * 64 + h
                for (int j = 0; j < kRows; j++) {
                    const bool have = j < nrows;
                    const int64_t rh = (int64_t)(r0 + j) * kHeads + h;
                    const uint32_t n = (uint32_t)(j * kRowN + h);
                    uint32_t sbytes = 0;  // group 2 half in the low byte
                    if (ix.q_dtype == SI_MXE4M3) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(
                            static_cast<const uint8_t *>(ix.q) + rh * kDim + half * 64);
#pragma unroll
                        for (int c = 0; c < 4; c++) {
                            const uint4 v = have ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
                            st_shared_v4(qb + sw128_offset(n, (uint32_t)(half * 4 + c)), v.x, v.y,
                                         v.z, v.w);
                        }
                        if (have) {
                            const uint8_t *qs = mxscale(ix.q_scale) + rh * (kDim / 32) + 2 * half;
                            sbytes = (uint32_t)__ldg(qs) | ((uint32_t)__ldg(qs + 1) << 8);
                        }
                    } else {
                        const uint4 *src = reinterpret_cast<const uint4 *>(
                            static_cast<const uint16_t *>(ix.q) + rh * kDim + half * 64);
#pragma unroll
                        for (int gg = 0; gg < 2; gg++) {  // one MX group = 32 dims = 4 loads
                            uint32_t q2[16];
#pragma unroll
                            for (int i = 0; i < 4; i++) {
                                const uint4 v =
                                    have ? __ldg(src + 4 * gg + i) : make_uint4(0u, 0u, 0u, 0u);
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
                                for (int jj = 0; jj < 4; jj++) {
                                    const uint32_t a = q2[8 * c + 2 * jj],
                                                   bb = q2[8 * c + 2 * jj + 1];
                                    w4[jj] = mx_codes2(__uint_as_float(a << 16),
                                                       __uint_as_float(a & 0xFFFF0000u), sb) |
                                             (mx_codes2(__uint_as_float(bb << 16),
                                                        __uint_as_float(bb & 0xFFFF0000u), sb)
                                              << 16);
                                }
                                st_shared_v4(qb + sw128_offset(n, (uint32_t)(half * 4 + 2 * gg + c)),
                                             w4[0], w4[1], w4[2], w4[3]);
                            }
                        }
                    }
                    // B row n's scale word (byte g = group g) for tcgen05.cp:
                    // block n / 128, row n % 32, word (n / 32) % 4
                    const uint32_t other = __shfl_xor_sync(0xffffffffu, sbytes, 1);
                    if (half == 0) {
                        const uint32_t word = sbytes | (other << 16);
                        asm volatile("st.shared.b32 [%0], %1;" ::"r"(
                                         base + kOffSfb + (2 * p + (n >> 7)) * kSfBytes +
                                         (n & 31) * 16 + ((n >> 5) & 3) * 4),
                                     "r"(word)
                                     : "memory");
                        w_s[(p * kRows + j) * kHeads + h] = have ? __ldg(ix.w + rh) : 0.f;
                    }
                }
            } else if constexpr (QM == kQFp8) {
                // stored FP8 query: codes as they are, the scale joins the weight
                for (int j = 0; j < kRows; j++) {
                    const bool have = j < nrows;
                    const int64_t rh = (int64_t)(r0 + j) * kHeads + h;
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        static_cast<const uint8_t *>(ix.q) + rh * kDim + half * 64);
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        const uint4 v = have ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
                        st_shared_v4(qb + sw128_offset(j * kRowN + h, (uint32_t)(half * 4 + c)),
                                     v.x, v.y, v.z, v.w);
                    }
                    if (half == 0)
                        w_s[(p * kRows + j) * kHeads + h] =
                            have ? __ldg(ix.w + rh) * __ldg(fscale(ix.q_scale) + rh) : 0.f;
                }
            } else {
                for (int j = 0; j < kRows; j++) {
                    const bool have = j < nrows;
                    uint32_t q2[32];  // 64 bf16 dims, two per word
                    if (have) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(
                            static_cast<const uint16_t *>(ix.q) +
                            ((int64_t)(r0 + j) * kHeads + h) * kDim + half * 64);
#pragma unroll
                        for (int i = 0; i < 8; i++) {
                            const uint4 v = __ldg(src + i);
                            q2[4 * i] = v.x;
                            q2[4 * i + 1] = v.y;
                            q2[4 * i + 2] = v.z;
                            q2[4 * i + 3] = v.w;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; i++)
                            q2[i] = 0;
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
                    // x / s_h as one multiply by 2^-e when that is a normal
                    // float (the same correctly rounded result as ldexpf)
                    const bool pow2 = e >= -126 && e <= 126;
                    const float inv_s = pow2 ? __int_as_float((127 - e) << 23) : 0.f;
                    auto unscale = [&](float x) { return pow2 ? x * inv_s : ldexpf(x, -e); };
#pragma unroll
                    for (int c = 0; c < 4; c++) {  // 16 dims per 16-byte unit
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int jj = 0; jj < 4; jj++) {  // 4 dims per output word
                            uint32_t hw = 0, lw = 0;
#pragma unroll
                            for (int pr2 = 0; pr2 < 2; pr2++) {
                                const uint32_t word = q2[8 * c + 2 * jj + pr2];
                                const float x0 = unscale(__uint_as_float(word << 16));
                                const float x1 = unscale(__uint_as_float(word & 0xFFFF0000u));
                                const uint16_t h2 = float2_to_e4m3x2(x0, x1);
                                const float2 hf = e4m3x2_to_float2(h2);
                                const uint16_t l2 = float2_to_e4m3x2(x0 - hf.x, x1 - hf.y);
                                hw |= (uint32_t)h2 << (16 * pr2);
                                lw |= (uint32_t)l2 << (16 * pr2);
                            }
                            hi[jj] = hw;
                            lo[jj] = lw;
                        }
                        const uint32_t u = (uint32_t)(half * 4 + c);
                        // q_hi into the first K half, q_lo into the second
                        st_shared_v4(qb + sw128_offset(j * kRowN + h, u), hi[0], hi[1], hi[2],
                                     hi[3]);
                        st_shared_v4(qb + kTileB + sw128_offset(j * kRowN + h, u), lo[0], lo[1],
                                     lo[2], lo[3]);
                    }
                    if (half == 0)
                        w_s[(p * kRows + j) * kHeads + h] =
                            have ? ldexpf(__ldg(ix.w + (int64_t)(r0 + j) * kHeads + h), e) : 0.f;
                }
            }
            fence_async_smem();
            mbar_arrive(qfull_bar + p);

        }
    } else if (warp >= kWarpEpi0) {
        // ------------------------------------------------------------ epilogue
        // Group g takes items g, g + 2, ...; it walks every item to keep the
        // block bookkeeping.
        const int g = (warp - kWarpEpi0) >> 2;
        const int et = (tid - kWarpEpi0 * 32) & 127;  // key row = TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        // Launched as a programmatic dependent, the kernel prepares queries,
        // loads keys and fills both accumulators while the previous kernel
        // (a Top-K reading the same score rows) finishes; the stores wait.
        griddep_wait();
        SpanWalk walk(work, n_blocks_rows);
        int64_t it = 0;
        int bi = 0;
        bool ok = true;
        for (; ok && walk.more(); bi++) {
            int r0, nrows, T;
            block_shape<kRows>(b, walk.blk(), tiles_ld, r0, nrows, T);
            const int t0 = walk.t_first, t1 = walk.end_of(T);
            walk.next(t1);
            const int p = bi & 1;
            int pos[kRows];
#pragma unroll
            for (int j = 0; j < kRows; j++)
                pos[j] = j < nrows ? __ldg(b.q_pos + r0 + j) : -1;
            if (!mbar_wait(qfull_bar + p, (uint32_t)(bi >> 1) & 1, st))
                break;
            for (int t = t0; t < t1; t++, it++) {
                if ((int)(it & 1) != g)
                    continue;
                const int64_t kit = it >> 1;
                const int ss = (int)(kit % kScStages);
                if (!mbar_wait(scfull_bar + g * kScStages + ss, (uint32_t)(kit / kScStages) & 1,
                               st)) {
                    ok = false;
                    break;
                }
                const float scv = sc_s[(g * kScStages + ss) * kKeys + et];
                mbar_arrive(scempty_bar + g * kScStages + ss);
                if (!mbar_wait(cfull_bar + g, (uint32_t)kit & 1, st)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int s = t * kKeys + et;
                const uint32_t acc = tmem + g * nB + lane_off;
                // The accumulator is read in pieces of 32 heads of one row,
                // each piece's load issued before the previous piece is
                // reduced; the accumulator is released as soon as the last
                // piece has landed in registers.
                constexpr int kPH = 32;                    // heads per piece
                constexpr int kPPR = kHeads / kPH;         // pieces per row
                constexpr int kPieces = kRows * kPPR;
                auto issue = [&](int pc, uint32_t(&v)[32]) {
                    tmem_ld32(acc + (uint32_t)((pc / kPPR) * kRowN + (pc % kPPR) * kPH), v);
                };
                float sum[kRows];
                // partial head sums in two packed pairs (0.0f has all bits 0)
                uint64_t p01 = 0, p23 = 0;
                uint32_t va[32], vb[32];
                issue(0, va);
#pragma unroll
                for (int pc = 0; pc < kPieces; pc++) {
                    uint32_t(&cur)[32] = (pc & 1) ? vb : va;
                    uint32_t(&nxt)[32] = (pc & 1) ? va : vb;
                    tmem_wait_ld();
                    tmem_regs_ready(cur);
                    if (pc + 1 < kPieces) {
                        issue(pc + 1, nxt);
                    } else {
                        tc_fence_before();
                        mbar_arrive(cempty_bar + g);
                    }
                    const int j = pc / kPPR, hq = pc % kPPR;
                    const float4 *w4 =
                        reinterpret_cast<const float4 *>(w_s + (p * kRows + j) * kHeads + hq * kPH);
#pragma unroll
                    for (int i = 0; i < kPH; i += 4) {
                        const float4 wv = w4[i >> 2];
                        // w_h * ReLU(logit), two heads per fma
                        f32x2_fma(p01, f32x2_pack(wv.x, wv.y),
                                  f32x2_pack(fmaxf(__uint_as_float(cur[i]), 0.f),
                                             fmaxf(__uint_as_float(cur[i + 1]), 0.f)));
                        f32x2_fma(p23, f32x2_pack(wv.z, wv.w),
                                  f32x2_pack(fmaxf(__uint_as_float(cur[i + 2]), 0.f),
                                             fmaxf(__uint_as_float(cur[i + 3]), 0.f)));
                    }
                    if (hq == kPPR - 1) {
                        const float2 x01 = f32x2_unpack(p01), x23 = f32x2_unpack(p23);
                        sum[j] = (x01.x + x01.y) + (x23.x + x23.y);
                        p01 = p23 = 0;
                    }
                }
                if (s < ld) {
#pragma unroll
                    for (int j = 0; j < kRows; j++)
                        if (j < nrows)
                            scores[(int64_t)(r0 + j) * ld + s] =
                                (s <= pos[j] && scv >= 0.f) ? sum[j] * scv + 0.0f : -INFINITY;
                }
            }
            if (ok)
                mbar_arrive(qempty_bar + p);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma)
        tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_indexer_prefill(const si_batch &b, const si_indexer &ix, float *scores,
                                   int64_t ld, unsigned int *st, cudaStream_t s, bool fill_tail,
                                   bool after_own_kernel)
{
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
            r = cudaFuncSetAttribute(k_indexer_prefill<kQBf16>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)Lay<kQBf16>::kSmemBytes);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(k_indexer_prefill<kQFp8>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)Lay<kQFp8>::kSmemBytes);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(k_indexer_prefill<kQMx>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)Lay<kQMx>::kSmemBytes);
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
    const int qm = ix.k.dtype == SI_MXE4M3 ? kQMx : (ix.q_dtype == SI_E4M3 ? kQFp8 : kQBf16);
    const int rows = qm == kQMx ? rows_per_block<kQMx>()
                                : (qm == kQFp8 ? rows_per_block<kQFp8>() : rows_per_block<kQBf16>());
    const int nb = (b.n_q + rows - 1) / rows;
    // every SM takes an equal share of the (block, tile) items
    const int64_t tiles_ld = (ld + kKeys - 1) / kKeys;
    const int64_t grid = std::min<int64_t>((int64_t)nb * tiles_ld, (int64_t)sms_of[dev]);
    count_launch();
    // After a kernel of the same call the launch may overlap its end
    // (programmatic dependent launch): everything the kernel reads before its
    // stores was written before the call.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_own_kernel ? 1 : 0;
    const int fill = fill_tail ? 1 : 0;
    if (qm == kQMx) {
        cfg.dynamicSmemBytes = Lay<kQMx>::kSmemBytes;
        return cudaLaunchKernelEx(&cfg, k_indexer_prefill<kQMx>, tmap, b, ix, scores, ld, nb, fill,
                                  st);
    }
    if (qm == kQFp8) {
        cfg.dynamicSmemBytes = Lay<kQFp8>::kSmemBytes;
        return cudaLaunchKernelEx(&cfg, k_indexer_prefill<kQFp8>, tmap, b, ix, scores, ld, nb,
                                  fill, st);
    }
    cfg.dynamicSmemBytes = Lay<kQBf16>::kSmemBytes;
    return cudaLaunchKernelEx(&cfg, k_indexer_prefill<kQBf16>, tmap, b, ix, scores, ld, nb, fill,
                              st);
}

}  // namespace si
