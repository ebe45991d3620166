// si_api.cu -- the extern "C" boundary of libsi: argument validation,
// workspace layout, kernel selection and the fused call.
//
// The path is the "select first, compute later" sparse attention of "Day0
// Inference Support and Performance Optimization for New Architecture LLMs"
// (section 2.2), with the fused indexer of section 4.1 and the index-based
// gather of section 4.2.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>

#include "si_common.cuh"
#include "si_internal.h"

namespace si {
static std::atomic<uint64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
}  // namespace si

namespace {

thread_local char g_err[512];

si_status fail(si_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
si_status fail(si_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

}  // namespace

si_status si::set_error(si_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

namespace {

si_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(SI_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Preferred fused workspace: the score strip stays in the GPU's L2 (about
// 126 MB) between the indexer that writes it and the Top-K that reads it.
constexpr size_t kFusedCap = (size_t)64 << 20;
constexpr int kMaxTop = 16384;

si_status check_batch(const si_batch *b)
{
    if (!b)
        return fail(SI_ERR_INVALID_ARG, "batch is NULL");
    if (b->n_q < 0)
        return fail(SI_ERR_INVALID_ARG, "n_q = %d < 0", b->n_q);
    if (b->n_q == 0)
        return SI_OK;
    if (!b->block_table || !b->ctx_len || !b->q_seq || !b->q_pos)
        return fail(SI_ERR_INVALID_ARG, "batch has a NULL device array");
    if (b->n_seq < 1 || b->max_blocks < 1 || b->n_blocks < 1)
        return fail(SI_ERR_INVALID_ARG, "n_seq, max_blocks and n_blocks must be >= 1");
    if (b->page_size < 1 || b->page_size > 1024)
        return fail(SI_ERR_INVALID_ARG, "page_size %d outside 1..1024", b->page_size);
    if (b->max_ctx < 1 || (int64_t)b->max_ctx > (int64_t)b->max_blocks * b->page_size)
        return fail(SI_ERR_INVALID_ARG, "max_ctx %d outside 1..max_blocks*page_size", b->max_ctx);
    if (b->max_ctx > (1 << 26))
        return fail(SI_ERR_UNSUPPORTED, "max_ctx %d above 2^26", b->max_ctx);
    return SI_OK;
}

si_status check_paged(const si_paged &p, const char *name, int need_dim)
{
    if (!p.data)
        return fail(SI_ERR_INVALID_ARG, "%s.data is NULL", name);
    if (!aligned(p.data, 16))
        return fail(SI_ERR_INVALID_ARG, "%s.data is not 16-byte aligned", name);
    if (p.dtype != SI_F32 && p.dtype != SI_BF16 && p.dtype != SI_E4M3 && p.dtype != SI_E2M1 &&
        p.dtype != SI_MXE4M3)
        return fail(SI_ERR_INVALID_ARG, "%s.dtype %d unknown", name, (int)p.dtype);
    if (p.dtype == SI_MXE4M3 && (p.scale_tile != 32 || !p.scale || p.row_stride % 32 != 0))
        return fail(SI_ERR_INVALID_ARG,
                    "%s: MXFP8 rows need E8M0 scales with scale_tile 32 and a row_stride "
                    "that is a multiple of 32", name);
    if (p.dtype == SI_E2M1 && (p.scale_tile < 1 || !p.scale || p.row_stride % 2 != 0))
        return fail(SI_ERR_INVALID_ARG,
                    "%s: e2m1 rows need per-tile scales and an even row_stride", name);
    if (p.row_dim < need_dim)
        return fail(SI_ERR_INVALID_ARG, "%s.row_dim %d < %d", name, p.row_dim, need_dim);
    if (p.row_stride < p.row_dim)
        return fail(SI_ERR_INVALID_ARG, "%s.row_stride %lld < row_dim %d", name,
                    (long long)p.row_stride, p.row_dim);
    if (p.scale_tile < 0 || (p.scale_tile > 0 && !p.scale))
        return fail(SI_ERR_INVALID_ARG, "%s.scale_tile %d needs a scale array", name, p.scale_tile);
    return SI_OK;
}

si_status check_indexer(const si_indexer *ix)
{
    if (!ix)
        return fail(SI_ERR_INVALID_ARG, "indexer operands are NULL");
    if (!ix->q || !ix->w)
        return fail(SI_ERR_INVALID_ARG, "indexer q or w is NULL");
    if (ix->q_dtype != SI_F32 && ix->q_dtype != SI_BF16 && ix->q_dtype != SI_E4M3 &&
        ix->q_dtype != SI_MXE4M3)
        return fail(SI_ERR_INVALID_ARG, "indexer q dtype must be f32, bf16, e4m3 or mxe4m3");
    if ((ix->q_dtype == SI_E4M3 || ix->q_dtype == SI_MXE4M3) && !ix->q_scale)
        return fail(SI_ERR_INVALID_ARG, "an e4m3 or mxe4m3 indexer q needs q_scale");
    if (ix->n_heads < 1 || ix->n_heads > 128)
        return fail(SI_ERR_INVALID_ARG, "indexer n_heads %d outside 1..128", ix->n_heads);
    if (ix->head_dim < 1 || ix->head_dim > 256)
        return fail(SI_ERR_INVALID_ARG, "indexer head_dim %d outside 1..256", ix->head_dim);
    if (ix->k.dtype == SI_E2M1)
        return fail(SI_ERR_UNSUPPORTED, "indexer keys are f32, bf16, e4m3 or mxe4m3");
    if (ix->k.dtype == SI_MXE4M3) {
        // section 5.1: query and keys both in MXFP8 (a bf16 / f32 query is
        // converted on the device)
        if (ix->head_dim % 32 != 0)
            return fail(SI_ERR_INVALID_ARG, "MXFP8 keys need head_dim a multiple of 32");
        if (ix->q_dtype == SI_E4M3)
            return fail(SI_ERR_UNSUPPORTED,
                        "MXFP8 keys take an mxe4m3, bf16 or f32 query, not e4m3");
    } else {
        if (ix->q_dtype == SI_MXE4M3)
            return fail(SI_ERR_UNSUPPORTED, "an mxe4m3 query needs mxe4m3 keys");
        if (ix->k.scale_tile != 0)
            return fail(SI_ERR_UNSUPPORTED, "indexer keys take one scale per row (scale_tile 0)");
    }
    return check_paged(ix->k, "indexer k", ix->head_dim);
}

si_status check_attention(const si_attention *at)
{
    if (!at)
        return fail(SI_ERR_INVALID_ARG, "attention operands are NULL");
    if (!at->q)
        return fail(SI_ERR_INVALID_ARG, "attention q is NULL");
    if (at->q_dtype != SI_F32 && at->q_dtype != SI_BF16)
        return fail(SI_ERR_INVALID_ARG, "attention q dtype must be f32 or bf16");
    if (at->n_heads < 1 || at->n_heads > 256)
        return fail(SI_ERR_INVALID_ARG, "attention n_heads %d outside 1..256", at->n_heads);
    if (at->d_qk < 1 || at->d_qk > 1024 || at->d_v < 1 || at->d_v > 1024)
        return fail(SI_ERR_INVALID_ARG, "attention d_qk/d_v outside 1..1024");
    si_status s = check_paged(at->k, "attention k", at->d_qk);
    if (s != SI_OK)
        return s;
    s = check_paged(at->v, "attention v", at->d_v);
    if (s != SI_OK)
        return s;
    // keys and values: the dtype of q, or FP8 / FP4 codes with scales (section
    // 5.2; the vLLM article's NVFP4 KV)
    const bool fp8_kv = at->k.dtype == SI_E4M3 && at->v.dtype == SI_E4M3;
    const bool fp4_kv = at->k.dtype == SI_E2M1 && at->v.dtype == SI_E2M1;
    if (!fp8_kv && !fp4_kv && (at->k.dtype != at->q_dtype || at->v.dtype != at->q_dtype))
        return fail(SI_ERR_UNSUPPORTED, "attention k and v must share q's dtype, or both be "
                                        "e4m3 or e2m1 with scales");
    if ((fp8_kv || fp4_kv) && (!at->k.scale || !at->v.scale))
        return fail(SI_ERR_INVALID_ARG, "e4m3 / e2m1 attention k and v need scales");
    return SI_OK;
}

si_status check_ws(void *ws, size_t ws_bytes, size_t need)
{
    if (!ws)
        return fail(SI_ERR_WORKSPACE, "workspace is NULL");
    if (!aligned(ws, SI_WORKSPACE_ALIGN))
        return fail(SI_ERR_WORKSPACE, "workspace is not %d-byte aligned", SI_WORKSPACE_ALIGN);
    if (ws_bytes < need)
        return fail(SI_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
    return SI_OK;
}

si_status check_k(int32_t k_top)
{
    if (k_top < 1 || k_top > kMaxTop)
        return fail(SI_ERR_INVALID_ARG, "k_top %d outside 1..%d", k_top, kMaxTop);
    return SI_OK;
}

int64_t scores_ld(const si_batch *b) { return (int64_t)round_up((size_t)b->max_ctx, 64); }

// Sub-batch of rows [r0, r0 + n) (device pointers advanced).
si_batch row_slice(const si_batch &b, int32_t r0, int32_t n)
{
    si_batch s = b;
    s.q_seq = b.q_seq + r0;
    s.q_pos = b.q_pos + r0;
    s.host_q_seq = b.host_q_seq ? b.host_q_seq + r0 : nullptr;
    s.n_q = n;
    return s;
}

size_t dtype_bytes(si_dtype t) { return t == SI_F32 ? 4 : (t == SI_BF16 ? 2 : 1); }

// Indexer operands of rows [r0, ...): query and head-weight pointers advanced.
si_indexer indexer_slice(const si_indexer &ix, int32_t r0)
{
    si_indexer s = ix;
    s.q = static_cast<const char *>(ix.q) +
          (size_t)r0 * ix.n_heads * ix.head_dim * dtype_bytes(ix.q_dtype);
    s.w = ix.w + (size_t)r0 * ix.n_heads;
    if (ix.q_scale && ix.q_dtype == SI_MXE4M3)
        s.q_scale = si::mxscale(ix.q_scale) + (size_t)r0 * ix.n_heads * (ix.head_dim / 32);
    else if (ix.q_scale)
        s.q_scale = si::fscale(ix.q_scale) + (size_t)r0 * ix.n_heads;
    return s;
}

unsigned int *status_word(void *ws) { return reinterpret_cast<unsigned int *>(ws); }

constexpr int32_t kPrefillRun = 64;  // rows of one sequence worth a prefill launch

cudaError_t launch_indexer_rows(const si_batch &b, const si_indexer &ix, float *scores,
                                int64_t ld, bool one_sequence, bool fill_tail, bool after_own,
                                unsigned int *st, cudaStream_t s)
{
    if (one_sequence && b.n_q >= kPrefillRun && si::indexer_tc_supported(b, ix, ld))
        return si::launch_indexer_prefill(b, ix, scores, ld, st, s, fill_tail, after_own);
    return si::indexer_tc_supported(b, ix, ld) ? si::launch_indexer_tc(b, ix, scores, ld, st, s)
                                               : si::launch_indexer_generic(b, ix, scores, ld, st, s);
}

// With a host copy of q_seq the batch is planned: each run of >= 64 rows of
// one sequence goes to the prefill kernel, the rows between runs to the
// decode kernels (one launch per maximal stretch).  fill_tail false: the
// scores past each row's position may be left unwritten (the caller's Top-K
// reads 0..q_pos only).  after_own: the stream's previous kernel is one of
// this call's (a single prefill launch may then overlap its end).
si_status run_indexer(const si_batch &b, const si_indexer &ix, float *scores, int64_t ld,
                      unsigned int *st, cudaStream_t s, bool fill_tail = true,
                      bool after_own = false)
{
    cudaError_t e = cudaSuccess;
    if (!b.host_q_seq || b.n_seq == 1 || b.n_q < kPrefillRun) {
        e = launch_indexer_rows(b, ix, scores, ld, b.n_seq == 1, fill_tail, after_own, st, s);
        return e == cudaSuccess ? SI_OK : cuda_fail(e, "indexer launch");
    }
    const int32_t *hs = b.host_q_seq;
    auto run_end = [&](int32_t r) {
        int32_t e2 = r + 1;
        while (e2 < b.n_q && hs[e2] == hs[r])
            e2++;
        return e2;
    };
    int32_t r = 0;
    while (e == cudaSuccess && r < b.n_q) {
        int32_t end = run_end(r);
        const bool chunk = end - r >= kPrefillRun;
        if (!chunk) {  // extend over short runs up to the next chunk
            while (end < b.n_q && run_end(end) - end < kPrefillRun)
                end = run_end(end);
        }
        e = launch_indexer_rows(row_slice(b, r, end - r), indexer_slice(ix, r),
                                scores + (int64_t)r * ld, ld, chunk, fill_tail, false, st, s);
        r = end;
    }
    return e == cudaSuccess ? SI_OK : cuda_fail(e, "indexer launch");
}

si_status run_topk(const si_batch &b, const float *scores, int64_t ld, int k_top, int32_t *idx,
                   unsigned int *st, cudaStream_t s)
{
    cudaError_t e = si::launch_topk(b, scores, ld, k_top, idx, st, s);
    return e == cudaSuccess ? SI_OK : cuda_fail(e, "top-k launch");
}

si_status run_attn(const si_batch &b, const si_attention &at, const int32_t *idx, int k_top,
                   void *out, si_dtype odt, float *lse, void *scratch, size_t scratch_bytes,
                   unsigned int *st, cudaStream_t s)
{
    // the tensor-core kernel stores its output with the tensor engine, which
    // needs a 16-byte aligned destination
    const bool tc = si::attn_tc_supported(b, at, k_top) && ((uintptr_t)out % 16) == 0;
    cudaError_t e = tc ? si::launch_attn_tc(b, at, idx, k_top, out, odt, lse, scratch,
                                            scratch_bytes, st, s)
                       : si::launch_attn_generic(b, at, idx, k_top, out, odt, lse, st, s);
    return e == cudaSuccess ? SI_OK : cuda_fail(e, "attention launch");
}

}  // namespace

si_status si::check_fused_args(const si_batch *b, const si_indexer *ix, const si_attention *at,
                               int32_t k_top, const int32_t *idx, const void *out,
                               si_dtype out_dtype)
{
    si_status st = check_batch(b);
    if (st != SI_OK || b->n_q == 0)
        return st;
    if ((st = check_indexer(ix)) != SI_OK || (st = check_attention(at)) != SI_OK ||
        (st = check_k(k_top)) != SI_OK)
        return st;
    if (!idx || !out)
        return fail(SI_ERR_INVALID_ARG, "idx or out is NULL");
    if (out_dtype != SI_F32 && out_dtype != SI_BF16)
        return fail(SI_ERR_INVALID_ARG, "out dtype must be f32 or bf16");
    return SI_OK;
}

namespace {

// Scratch the attention's split partials would use (0 when the batch is
// large enough to fill the GPU unsplit, or the shapes take another kernel).
size_t attn_split_need(const si_batch *b, const si_attention *at, int32_t k_top)
{
    if (!at || b->n_q <= 0 || k_top < 1 || !si::attn_tc_supported(*b, *at, k_top))
        return 0;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return round_up(si::attn_tc_split_bytes(*b, si::attn_tc_split(*b, k_top, sms)), 256);
}

size_t ws_need(si_op op, const si_batch *b, const si_indexer *ix, const si_attention *at,
               int32_t k_top, bool minimal)
{
    (void)ix;
    size_t n = si::kStatusBytes;
    size_t extra = 0;
    if ((op == SI_OP_FUSED || op == SI_OP_SELECT) && b->n_q > 0) {
        const size_t row_bytes = (size_t)scores_ld(b) * sizeof(float);
        size_t rows = minimal ? 1 : (size_t)b->n_q;
        if (!minimal && rows * row_bytes > kFusedCap)
            rows = std::max<size_t>(1, kFusedCap / row_bytes);
        extra = round_up(rows * row_bytes, 256);
    }
    // the full size also lets few-row attention split each row's key tiles
    if (!minimal && (op == SI_OP_FUSED || op == SI_OP_ATTN))
        extra = std::max(extra, attn_split_need(b, at, k_top));
    return n + extra;
}

// Workspace of a candidate-restricted selection: status word, the synthetic
// batch's arrays, gathered key rows and scales, scores.
struct CandLayout {
    si::CandView v;
    size_t keys, scales, scores, total;
    int64_t ld;  // scores row stride when they live in the workspace
};

// With the tensor-core indexer the candidates are gathered inside the
// scoring kernel and the workspace holds only the status word and scores.
bool cand_fused(const si_batch &b, const si_indexer &ix, int32_t n_cand)
{
    return si::indexer_tc_supported(b, ix, (int64_t)round_up((size_t)n_cand, 64));
}

CandLayout cand_layout(const si_batch &b, const si_indexer &ix, int32_t n_cand, void *ws)
{
    CandLayout L{};
    if (cand_fused(b, ix, n_cand)) {
        L.ld = (int64_t)round_up((size_t)n_cand, 64);
        L.scores = si::kStatusBytes;
        L.total = L.scores + round_up((size_t)b.n_q * L.ld * 4, 256);
        return L;
    }
    const int64_t n_q = b.n_q;
    L.v.n_pad = (int32_t)round_up((size_t)n_cand, si::kCandPage);
    L.v.blocks_per_row = L.v.n_pad / si::kCandPage;
    L.v.row_bytes = ix.k.row_stride * (int64_t)dtype_bytes(ix.k.dtype);
    char *base = static_cast<char *>(ws);
    size_t off = si::kStatusBytes;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += round_up(bytes, 256);
        return at;
    };
    const size_t bt = take((size_t)n_q * L.v.blocks_per_row * 4);
    const size_t qs = take((size_t)n_q * 4), qp = take((size_t)n_q * 4),
                 cl = take((size_t)n_q * 4);
    L.keys = take((size_t)n_q * L.v.n_pad * L.v.row_bytes);
    L.scales = take((size_t)n_q * L.v.n_pad * 4);
    L.ld = (int64_t)round_up((size_t)n_cand, 64);
    L.scores = take((size_t)n_q * L.ld * 4);
    L.total = off;
    if (base) {
        L.v.block_table = reinterpret_cast<int32_t *>(base + bt);
        L.v.q_seq = reinterpret_cast<int32_t *>(base + qs);
        L.v.q_pos = reinterpret_cast<int32_t *>(base + qp);
        L.v.ctx_len = reinterpret_cast<int32_t *>(base + cl);
    }
    return L;
}

constexpr int32_t kMaxCand = 1 << 24;

}  // namespace

extern "C" {

size_t si_workspace_size_cand(const si_batch *b, const si_indexer *ix, int32_t n_cand)
{
    if (check_batch(b) != SI_OK || check_indexer(ix) != SI_OK || n_cand < 1 || n_cand > kMaxCand ||
        ix->k.dtype == SI_MXE4M3)
        return 0;
    return cand_layout(*b, *ix, n_cand, nullptr).total;
}

si_status si_indexer_topk_cand(const si_batch *b, const si_indexer *ix, const int32_t *cand,
                               int32_t n_cand, int64_t ld_cand, int32_t k_top, int32_t *idx,
                               float *scores, int64_t ld_scores, void *ws, size_t ws_bytes,
                               void *stream)
{
    si_status st = check_batch(b);
    if (st != SI_OK || b->n_q == 0)
        return st;
    if ((st = check_indexer(ix)) != SI_OK || (st = check_k(k_top)) != SI_OK)
        return st;
    if (ix->k.dtype == SI_MXE4M3)
        return fail(SI_ERR_UNSUPPORTED,
                    "candidate-restricted selection takes f32, bf16 or e4m3 keys");
    if (!cand || !idx)
        return fail(SI_ERR_INVALID_ARG, "cand or idx is NULL");
    if (n_cand < 1 || n_cand > kMaxCand)
        return fail(SI_ERR_INVALID_ARG, "n_cand %d outside 1..%d", n_cand, kMaxCand);
    if (ld_cand < n_cand)
        return fail(SI_ERR_INVALID_ARG, "ld_cand %lld < n_cand %d", (long long)ld_cand, n_cand);
    if (scores && ld_scores < n_cand)
        return fail(SI_ERR_INVALID_ARG, "ld_scores %lld < n_cand %d", (long long)ld_scores,
                    n_cand);
    const CandLayout need = cand_layout(*b, *ix, n_cand, nullptr);
    if ((st = check_ws(ws, ws_bytes, need.total)) != SI_OK)
        return st;
    const CandLayout L = cand_layout(*b, *ix, n_cand, ws);
    cudaStream_t s = (cudaStream_t)stream;
    unsigned int *stw = status_word(ws);
    char *base = static_cast<char *>(ws);
    float *sc = scores ? scores : reinterpret_cast<float *>(base + L.scores);
    const int64_t ld = scores ? ld_scores : L.ld;
    cudaError_t e;
    if (cand_fused(*b, *ix, n_cand)) {
        e = si::launch_indexer_tc_cand(*b, *ix, cand, ld_cand, n_cand, sc, ld, stw, s);
        if (e != cudaSuccess)
            return cuda_fail(e, "candidate indexer launch");
    } else {
        uint8_t *keys = reinterpret_cast<uint8_t *>(base + L.keys);
        float *scl = reinterpret_cast<float *>(base + L.scales);
        // other shapes: the candidates gathered into one private sequence per
        // query row, scored by the CUDA-core indexer
        si_batch cb = *b;
        cb.block_table = L.v.block_table;
        cb.ctx_len = L.v.ctx_len;
        cb.q_seq = L.v.q_seq;
        cb.q_pos = L.v.q_pos;
        cb.n_seq = b->n_q;
        cb.max_blocks = L.v.blocks_per_row;
        cb.page_size = si::kCandPage;
        cb.max_ctx = n_cand;
        cb.n_blocks = b->n_q * L.v.blocks_per_row;
        cb.host_q_seq = nullptr;
        si_indexer cix = *ix;
        cix.k.data = keys;
        cix.k.scale = scl;
        e = si::launch_cand_gather(*b, cand, ld_cand, n_cand, L.v, ix->k, keys, scl, stw, s);
        if (e != cudaSuccess)
            return cuda_fail(e, "candidate gather launch");
        if ((st = run_indexer(cb, cix, sc, ld, stw, s)) != SI_OK)
            return st;
        // the CUDA-core indexer multiplies by the -1 scale of an empty slot
        e = si::launch_cand_mask(b->n_q, n_cand, L.v, scl, sc, ld, s);
        if (e != cudaSuccess)
            return cuda_fail(e, "candidate mask launch");
    }
    // Top-K over the slots, each selected slot written as its position
    e = si::launch_topk(*b, sc, ld, k_top, idx, stw, s, n_cand, cand, ld_cand);
    return e == cudaSuccess ? SI_OK : cuda_fail(e, "top-k launch");
}

size_t si_workspace_size(si_op op, const si_batch *b, const si_indexer *ix,
                         const si_attention *at, int32_t k_top)
{
    if (check_batch(b) != SI_OK)
        return 0;
    return ws_need(op, b, ix, at, k_top, false);
}

size_t si_workspace_min(si_op op, const si_batch *b, const si_indexer *ix,
                        const si_attention *at, int32_t k_top)
{
    if (check_batch(b) != SI_OK)
        return 0;
    return ws_need(op, b, ix, at, k_top, true);
}

si_status si_indexer_scores(const si_batch *b, const si_indexer *ix, float *scores,
                            int64_t ld_scores, void *ws, size_t ws_bytes, void *stream)
{
    si_status st = check_batch(b);
    if (st != SI_OK || b->n_q == 0)
        return st;
    if ((st = check_indexer(ix)) != SI_OK)
        return st;
    if (!scores)
        return fail(SI_ERR_INVALID_ARG, "scores is NULL");
    if (ld_scores < b->max_ctx)
        return fail(SI_ERR_INVALID_ARG, "ld_scores %lld < max_ctx %d", (long long)ld_scores,
                    b->max_ctx);
    if ((st = check_ws(ws, ws_bytes, ws_need(SI_OP_INDEXER, b, ix, nullptr, 0, true))) != SI_OK)
        return st;
    return run_indexer(*b, *ix, scores, ld_scores, status_word(ws), (cudaStream_t)stream);
}

si_status si_topk(const si_batch *b, const float *scores, int64_t ld_scores, int32_t k_top,
                  int32_t *idx, void *ws, size_t ws_bytes, void *stream)
{
    si_status st = check_batch(b);
    if (st != SI_OK || b->n_q == 0)
        return st;
    if ((st = check_k(k_top)) != SI_OK)
        return st;
    if (!scores || !idx)
        return fail(SI_ERR_INVALID_ARG, "scores or idx is NULL");
    if (ld_scores < b->max_ctx)
        return fail(SI_ERR_INVALID_ARG, "ld_scores %lld < max_ctx %d", (long long)ld_scores,
                    b->max_ctx);
    if ((st = check_ws(ws, ws_bytes, ws_need(SI_OP_TOPK, b, nullptr, nullptr, k_top, true))) !=
        SI_OK)
        return st;
    return run_topk(*b, scores, ld_scores, k_top, idx, status_word(ws), (cudaStream_t)stream);
}

si_status si_sparse_attn(const si_batch *b, const si_attention *at, const int32_t *idx,
                         int32_t k_top, void *out, si_dtype out_dtype, float *lse, void *ws,
                         size_t ws_bytes, void *stream)
{
    si_status st = check_batch(b);
    if (st != SI_OK || b->n_q == 0)
        return st;
    if ((st = check_attention(at)) != SI_OK || (st = check_k(k_top)) != SI_OK)
        return st;
    if (!idx || !out)
        return fail(SI_ERR_INVALID_ARG, "idx or out is NULL");
    if (out_dtype != SI_F32 && out_dtype != SI_BF16)
        return fail(SI_ERR_INVALID_ARG, "out dtype must be f32 or bf16");
    if ((st = check_ws(ws, ws_bytes, ws_need(SI_OP_ATTN, b, nullptr, at, k_top, true))) != SI_OK)
        return st;
    return run_attn(*b, *at, idx, k_top, out, out_dtype, lse,
                    static_cast<char *>(ws) + si::kStatusBytes, ws_bytes - si::kStatusBytes,
                    status_word(ws), (cudaStream_t)stream);
}

}  // extern "C"

namespace {

// Scores and Top-K strip by strip (section 4.1's fused operator); the strip
// starts at ws + *head on return.
si_status run_indexer_topk(const si_batch *b, const si_indexer *ix, int32_t k_top, int32_t *idx,
                           void *ws, size_t ws_bytes, cudaStream_t s, size_t *head_out)
{
    si_status st = SI_OK;
    unsigned int *stw = status_word(ws);
    const int64_t ld = scores_ld(b);
    const size_t row_bytes = (size_t)ld * sizeof(float);
    const size_t head = si::kStatusBytes;
    float *scores = reinterpret_cast<float *>(static_cast<char *>(ws) + head);
    const int64_t strip = (int64_t)((ws_bytes - head) / row_bytes);
    for (int64_t r0 = 0; r0 < b->n_q; r0 += strip) {
        const int32_t n = (int32_t)std::min<int64_t>(strip, b->n_q - r0);
        const si_batch sb = row_slice(*b, (int32_t)r0, n);
        const si_indexer si_ = indexer_slice(*ix, (int32_t)r0);
        if ((st = run_indexer(sb, si_, scores, ld, stw, s, false, r0 > 0)) != SI_OK)
            return st;
        if ((st = run_topk(sb, scores, ld, k_top, idx + r0 * k_top, stw, s)) != SI_OK)
            return st;
    }
    *head_out = head;
    return SI_OK;
}

}  // namespace

extern "C" {

si_status si_indexer_topk(const si_batch *b, const si_indexer *ix, int32_t k_top, int32_t *idx,
                          void *ws, size_t ws_bytes, void *stream)
{
    si_status st = check_batch(b);
    if (st != SI_OK || b->n_q == 0)
        return st;
    if ((st = check_indexer(ix)) != SI_OK || (st = check_k(k_top)) != SI_OK)
        return st;
    if (!idx)
        return fail(SI_ERR_INVALID_ARG, "idx is NULL");
    if ((st = check_ws(ws, ws_bytes, ws_need(SI_OP_SELECT, b, ix, nullptr, k_top, true))) != SI_OK)
        return st;
    size_t head = 0;
    return run_indexer_topk(b, ix, k_top, idx, ws, ws_bytes, (cudaStream_t)stream, &head);
}

si_status si_fused_decode(const si_batch *b, const si_indexer *ix, const si_attention *at,
                          int32_t k_top, int32_t *idx, void *out, si_dtype out_dtype,
                          float *lse, void *ws, size_t ws_bytes, void *stream)
{
    si_status st = si::check_fused_args(b, ix, at, k_top, idx, out, out_dtype);
    if (st != SI_OK || b->n_q == 0)
        return st;
    if ((st = check_ws(ws, ws_bytes, ws_need(SI_OP_FUSED, b, ix, at, k_top, true))) != SI_OK)
        return st;
    cudaStream_t s = (cudaStream_t)stream;
    size_t head = 0;
    if ((st = run_indexer_topk(b, ix, k_top, idx, ws, ws_bytes, s, &head)) != SI_OK)
        return st;
    // the score strip is free once every Top-K has run: it may hold the
    // attention's split partials
    return run_attn(*b, *at, idx, k_top, out, out_dtype, lse, static_cast<char *>(ws) + head,
                    ws_bytes - head, status_word(ws), s);
}

si_status si_workspace_status(const void *ws, uint32_t *flags, void *stream)
{
    if (!ws || !flags)
        return fail(SI_ERR_INVALID_ARG, "ws or flags is NULL");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "stream synchronize");
    e = cudaMemcpy(flags, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_fail(e, "status read");
    return *flags ? fail(SI_ERR_DEVICE, "device flags 0x%x", *flags) : SI_OK;
}

const char *si_status_string(si_status s)
{
    switch (s) {
    case SI_OK: return "ok";
    case SI_ERR_INVALID_ARG: return "invalid argument";
    case SI_ERR_UNSUPPORTED: return "unsupported";
    case SI_ERR_WORKSPACE: return "workspace error";
    case SI_ERR_CUDA: return "cuda error";
    case SI_ERR_DEVICE: return "device-side flag raised";
    }
    return "unknown status";
}

const char *si_last_error(void) { return g_err; }

uint64_t si_launch_count(void) { return si::g_launches.load(std::memory_order_relaxed); }

int32_t si_version(void) { return SI_VERSION; }

}  // extern "C"
