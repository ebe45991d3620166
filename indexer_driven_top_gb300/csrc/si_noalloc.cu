// si_noalloc.cu -- the fused path for callers that must not allocate.
//
// Some callers cannot hand the library a workspace: code that runs where
// device allocation is forbidden or unsafe (inside an allocator's own
// callbacks, in a process whose device memory is fully reserved by another
// runtime, or in a plain C program with no allocator at hand).  For them
// si_fused_decode_noalloc runs the same kernels as si_fused_decode, with the
// workspace taken from a fixed scratch array that is part of the library's
// device image.  The call itself allocates nothing: no cudaMalloc, no
// cudaFree, no allocating library routine.
//
// The scratch holds what si_fused_decode keeps in its workspace: the sticky
// status word (first 256 bytes, must be zero when the kernels start; the call
// clears it on the caller's stream before launching) and the score strip
// (needs no initial value: the indexer writes every entry the Top-K reads).
#include <mutex>

#include "si_common.cuh"
#include "si_internal.h"

namespace {

// 8 MiB: the status word plus a score strip of (8 MiB - 256) / (4 * max_ctx)
// rows, e.g. 255 rows at 8192 positions, 15 rows at 131072.
constexpr size_t kScratchBytes = SI_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Scratch address per device, looked up on the first successful call; a
// failed lookup is not remembered, so a later call retries it.
std::mutex g_mu[si::kMaxDevices];
void *g_addr[si::kMaxDevices];

using si::set_error;

}  // namespace

extern "C" {

si_status si_fused_decode_noalloc(const si_batch *b, const si_indexer *ix,
                                  const si_attention *at, int32_t k_top, int32_t *idx,
                                  void *out, si_dtype out_dtype, float *lse,
                                  const void **scratch, void *stream)
{
    if (scratch)
        *scratch = nullptr;
    // Validation and the size check are host arithmetic only, so a bad or
    // oversize request is refused before any CUDA call.
    si_status st = si::check_fused_args(b, ix, at, k_top, idx, out, out_dtype);
    if (st != SI_OK || b->n_q == 0)
        return st;
    const size_t need = si_workspace_min(SI_OP_FUSED, b, ix, at, k_top);
    if (need > kScratchBytes)
        return set_error(SI_ERR_WORKSPACE,
                         "si_fused_decode_noalloc: max_ctx = %d needs %zu bytes of scratch, "
                         "the static scratch holds %zu (use si_fused_decode with a workspace)",
                         b->max_ctx, need, kScratchBytes);
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return set_error(SI_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= si::kMaxDevices)
        return set_error(SI_ERR_UNSUPPORTED, "device ordinal %d beyond %d", dev,
                         si::kMaxDevices);
    void *addr;
    {
        std::lock_guard<std::mutex> lock(g_mu[dev]);
        if (!g_addr[dev]) {
            void *a = nullptr;
            e = cudaGetSymbolAddress(&a, g_scratch);
            if (e != cudaSuccess)
                return set_error(SI_ERR_CUDA, "scratch address on device %d: %s", dev,
                                 cudaGetErrorString(e));
            g_addr[dev] = a;
        }
        addr = g_addr[dev];
    }
    e = cudaMemsetAsync(addr, 0, si::kStatusBytes, (cudaStream_t)stream);
    if (e != cudaSuccess)
        return set_error(SI_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
    st = si_fused_decode(b, ix, at, k_top, idx, out, out_dtype, lse, addr, kScratchBytes, stream);
    if (st == SI_OK && scratch)
        *scratch = addr;
    return st;
}

}  // extern "C"
