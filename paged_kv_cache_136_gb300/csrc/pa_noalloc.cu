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
// (cudaGetSymbolAddress, with that device current) and caches it per device
// and context; that first call (and the first call after a device reset or
// in another driver context) should therefore come before any stream
// capture.  All calls on a
// device share the one array: calls that overlap on the GPU race, so callers
// must order them (one stream, or events).
#include <cuda_runtime.h>

#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace pa {

void *current_driver_context()
{
    typedef int (*ctx_get_current_fn)(void **ctx);
    static ctx_get_current_fn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<ctx_get_current_fn>(p);
    });
    void *ctx = nullptr;
    if (!fn || fn(&ctx) != 0)
        return nullptr;
    return ctx;
}

} // namespace pa

namespace {

// Scratch in device global memory.  In host code this name is only a
// host-side stand-in for the symbol; the kernels get its real device address
// from scratch_address().
__device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch in the current device's current
// context.  The lookup is done once per (device, context) and cached: a new
// context on a device (after cudaDeviceReset, or a caller that switched
// driver contexts) loads the module again with a new copy of the array, so
// its address is looked up again.  Returns nullptr and sets *err if the
// lookup fails.
void *scratch_address(cudaError_t *err)
{
    struct entry {
        int dev;
        void *ctx;
        void *addr;
    };
    static entry cache[64];
    static int n_cached = 0;
    static std::mutex mu;
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess)
        return nullptr;
    void *ctx = pa::current_driver_context();
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_cached; ++i)
        if (cache[i].dev == dev && cache[i].ctx == ctx) {
            *err = cudaSuccess;
            return cache[i].addr;
        }
    void *p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess || !p)
        return nullptr;
    // With no context current before the lookup, the runtime has just made
    // the device's primary context current: key the entry on that one.
    if (!ctx)
        ctx = pa::current_driver_context();
    // Replace an entry of the same device (its context is gone or no longer
    // current), else append; a full table recycles its oldest slot.
    int slot = -1;
    for (int i = 0; i < n_cached; ++i)
        if (cache[i].dev == dev)
            slot = i;
    if (slot < 0)
        slot = n_cached < 64 ? n_cached++ : 0;
    cache[slot] = {dev, ctx, p};
    *err = cudaSuccess;
    return p;
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
