// pa_noalloc.cu -- split-K decode for callers that cannot allocate device
// memory.
//
// pa_decode_splitk needs a scratch workspace for its per-partition partial
// states, which the caller normally allocates.  Some callers cannot call
// cudaMalloc: code hosted inside a framework that owns all device memory and
// hands its plugins no allocator, or a latency-critical loop where an
// allocation (which may synchronise the device) is not allowed.
// pa_decode_splitk_noalloc serves them from a fixed scratch array that lives
// in this file as a static device variable, so the call itself allocates
// nothing.
//
// The array holds PA_NOALLOC_SCRATCH_BYTES on every GPU where the library's
// module is loaded, until the process exits.  On each device the entry
// point's first call looks up the array's device address
// (cudaGetSymbolAddress, with that device current) and caches it; that first
// call should therefore come before any stream capture.  All calls on a
// device share the one array: calls that overlap on the GPU race, so callers
// must order them (one stream, or events).
#include <cuda_runtime.h>

#include <mutex>

#include "pa.h"

namespace {

// Scratch in device global memory.  In host code this name is only a
// host-side stand-in for the symbol; the kernels get its real device address
// from scratch_address().
__device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device (looked up once
// per device).  Returns nullptr and sets *err if the lookup fails.
void *scratch_address(cudaError_t *err)
{
    static void *addr[64] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess)
        return nullptr;
    if (dev < 0 || dev >= 64) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (*err != cudaSuccess || !p)
            return nullptr;
        addr[dev] = p;
    }
    *err = cudaSuccess;
    return addr[dev];
}

} // namespace

extern "C" pa_status pa_decode_splitk_noalloc(void *out, const void *q, const void *kv_cache,
                                              const int32_t *block_tables,
                                              const int32_t *seq_lens, int num_seqs,
                                              int num_heads, int num_kv_heads, int head_size,
                                              int block_size, int num_blocks,
                                              int max_blocks_per_seq, float scale,
                                              pa_dtype dtype, int max_seq_len,
                                              int partition_size, void *stream)
{
    const size_t need = pa_decode_splitk_workspace_size(num_seqs, num_heads, head_size,
                                                        max_seq_len, partition_size);
    if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES)
        return PA_ERR_WORKSPACE; // these sizes need more scratch than the array holds
    cudaError_t e;
    void *scratch = scratch_address(&e);
    if (!scratch)
        return PA_ERR_CUDA;
    // Nothing in the scratch has to start at zero: the partition kernel
    // writes every partial state the reduce reads within the same call.
    return pa_decode_splitk(out, q, kv_cache, block_tables, seq_lens, num_seqs, num_heads,
                            num_kv_heads, head_size, block_size, num_blocks,
                            max_blocks_per_seq, scale, dtype, max_seq_len, partition_size,
                            scratch, (size_t)PA_NOALLOC_SCRATCH_BYTES, stream);
}
