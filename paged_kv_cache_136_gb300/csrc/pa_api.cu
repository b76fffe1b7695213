// pa_api.cu -- the C ABI of libpa.so (declared in include/pa.h): host-side
// argument checks, TMA tensor-map encoding, the cache-write kernel, the split-K
// reduce launcher and the device error word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <math.h>
#include <mutex>
#include <stdint.h>
#include <string.h>
#include <unordered_set>
#include <vector>

#include <stdlib.h>

#include "pa.h"
#include "pa_decode.cuh"
#include "pa_decode_tc.cuh"
#include "pa_internal.h"

namespace pa {

// Sticky per-device error word (PA_DEVERR_* bits).  Kernels receive its
// device address as a parameter.
__device__ unsigned int g_device_errors = 0;

static unsigned int *device_error_word(cudaError_t *err)
{
    static unsigned int *addr[64] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess)
        return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev & 63]) {
        void *p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_device_errors);
        if (*err != cudaSuccess)
            return nullptr;
        addr[dev & 63] = static_cast<unsigned int *>(p);
    }
    return addr[dev & 63];
}

// ---------------------------------------------------------------------------
// TMA tensor map over the pool [2, NB, BS, Hkv, D], seen as 4-D
// {D, Hkv, NB*BS, 2} (innermost first).  A box is 64 elements (128 bytes) of
// `box_heads` consecutive kv heads for `box_rows` consecutive token rows
// (default: one head, one block) of one plane, loaded with the 128-byte
// swizzle.  Rows at or past NB*BS are out of bounds and read as zeros.
// ---------------------------------------------------------------------------
// Measurement aid (pa_profile_kernel_events): events recorded around the main
// attention kernel of this host thread's later decode calls.
static thread_local cudaEvent_t t_mark_before = nullptr;
static thread_local cudaEvent_t t_mark_after = nullptr;

static inline void mark_before(cudaStream_t s)
{
    if (t_mark_before)
        cudaEventRecord(t_mark_before, s);
}

static inline void mark_after(cudaStream_t s)
{
    if (t_mark_after)
        cudaEventRecord(t_mark_after, s);
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn(cudaError_t *err)
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    static cudaError_t init_err = cudaSuccess;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        init_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                    cudaEnableDefault, &q);
        if (init_err == cudaSuccess && q != cudaDriverEntryPointSuccess)
            init_err = cudaErrorNotSupported;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    *err = init_err;
    return fn;
}

static bool make_pool_map(CUtensorMap *map, const void *cache, int dtype, int num_blocks,
                          int block_size, int num_kv_heads, int head_size, int box_heads = 1,
                          int box_rows = 0)
{
    cudaError_t err;
    auto fn = encode_fn(&err);
    if (!fn)
        return false;
    const cuuint64_t es = 2;
    cuuint64_t dims[4] = {(cuuint64_t)head_size, (cuuint64_t)num_kv_heads,
                          (cuuint64_t)num_blocks * block_size, 2};
    cuuint64_t strides[3] = {head_size * es, (cuuint64_t)num_kv_heads * head_size * es,
                             (cuuint64_t)num_blocks * block_size * num_kv_heads * head_size * es};
    cuuint32_t box[4] = {64, (cuuint32_t)box_heads,
                         (cuuint32_t)(box_rows > 0 ? box_rows : block_size), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    4, const_cast<void *>(cache), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Query rows as a 2-D tensor {D, B*H}; a box is 64 elements of `box_rows`
// consecutive query heads (the groups of the CTA's kv heads), loaded with the
// 128-byte swizzle.
static bool make_q_map(CUtensorMap *map, const void *q, int dtype, int rows, int head_size,
                       int box_rows)
{
    cudaError_t err;
    auto fn = encode_fn(&err);
    if (!fn)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)head_size, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)head_size * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    2, const_cast<void *>(q), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// FP8 pool as a 4-D byte tensor {D, Hkv, NB*bs, 2}; a box is one kv head's
// 128-byte rows of `box_rows` tokens, with the 128-byte swizzle.
static bool make_pool_map_fp8(CUtensorMap *map, const void *cache, int num_blocks,
                              int block_size, int num_kv_heads, int head_size, int box_rows,
                              int box_heads = 1)
{
    cudaError_t err;
    auto fn = encode_fn(&err);
    if (!fn)
        return false;
    cuuint64_t dims[4] = {(cuuint64_t)head_size, (cuuint64_t)num_kv_heads,
                          (cuuint64_t)num_blocks * block_size, 2};
    cuuint64_t strides[3] = {(cuuint64_t)head_size, (cuuint64_t)num_kv_heads * head_size,
                             (cuuint64_t)num_blocks * block_size * num_kv_heads * head_size};
    cuuint32_t box[4] = {(cuuint32_t)head_size, (cuuint32_t)box_heads, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(cache), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// e4m3 query parts [3][rows][128] as a 2-D byte tensor {128, 3*rows}; a box
// is `box_rows` rows of one part.
static bool make_q_parts_map(CUtensorMap *map, const void *parts, int rows, int box_rows)
{
    cudaError_t err;
    auto fn = encode_fn(&err);
    if (!fn)
        return false;
    cuuint64_t dims[2] = {128, (cuuint64_t)rows * 3};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(parts), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Packed query rows [T, H, D] as a 3-D tensor {D, H, T}; a box is 64
// elements of one head for 128 consecutive tokens, with the 128-byte swizzle.
static bool make_q_rows_map(CUtensorMap *map, const void *q, int dtype, int num_tokens,
                            int num_heads, int head_size)
{
    cudaError_t err;
    auto fn = encode_fn(&err);
    if (!fn)
        return false;
    cuuint64_t dims[3] = {(cuuint64_t)head_size, (cuuint64_t)num_heads, (cuuint64_t)num_tokens};
    cuuint64_t strides[2] = {(cuuint64_t)head_size * 2, (cuuint64_t)num_heads * head_size * 2};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    3, const_cast<void *>(q), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static int sm_count(cudaError_t *err)
{
    static int count[64] = {0};
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess)
        return 0;
    if (!count[dev & 63]) {
        int c = 0;
        *err = cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
        if (*err != cudaSuccess)
            return 0;
        count[dev & 63] = c;
    }
    return count[dev & 63];
}

// Decode kernel family: PA_DECODE_KERNEL=simt or =tcgen05 forces one
// (head_size 128 only for tcgen05); unset or anything else picks per shape.
enum { kKernelAuto = 0, kKernelSimt = 1, kKernelTc = 2 };
static int kernel_choice()
{
    static int choice = -1;
    if (choice < 0) {
        const char *v = getenv("PA_DECODE_KERNEL");
        choice = (v && !strcmp(v, "simt")) ? kKernelSimt
                 : (v && !strcmp(v, "tcgen05")) ? kKernelTc
                                                : kKernelAuto;
    }
    return choice;
}

static bool use_tc(int head_size, int group, bool split)
{
    if (head_size != 128)
        return false;
    const int c = kernel_choice();
    if (c == kKernelSimt)
        return false;
    if (c == kKernelTc)
        return true;
    return split || group >= 2;
}

cudaError_t launch_decode(const DecodeKey &key, const CUtensorMap &tmap, const DecodeParams &p,
                          dim3 grid, cudaStream_t stream)
{
    if (key.dtype == PA_FP16 && key.head_size == 64)
        return launch_decode_f16_d64(key, tmap, p, grid, stream);
    if (key.dtype == PA_FP16 && key.head_size == 128)
        return launch_decode_f16_d128(key, tmap, p, grid, stream);
    if (key.dtype == PA_BF16 && key.head_size == 64)
        return launch_decode_bf16_d64(key, tmap, p, grid, stream);
    if (key.dtype == PA_BF16 && key.head_size == 128)
        return launch_decode_bf16_d128(key, tmap, p, grid, stream);
    return cudaErrorNotSupported;
}

template <typename T, int D>
static cudaError_t launch_reduce_t(const ReduceParams &p, dim3 grid, cudaStream_t stream)
{
    // Rows of at most 32 partitions: one warp per row.
    if (p.max_parts <= 32)
        return launch_after_previous(
            splitk_reduce_warp_kernel<T, D>,
            dim3((grid.x + kReduceWarpHeads - 1) / kReduceWarpHeads, grid.y),
            dim3(32 * kReduceWarpHeads), 0, stream, p);
    // Rows of many partitions: one CTA per row, its warps split the partitions.
    return launch_after_previous(splitk_reduce_kernel<T, D>, grid, dim3(32 * kWideWarps), 0, stream,
                                 p);
}

cudaError_t launch_reduce(int dtype, int head_size, const ReduceParams &p, int num_seqs,
                          cudaStream_t stream)
{
    // Launched as the dependent of the partition kernel: its launch overlaps
    // that kernel's tail, and it waits for the partial states on the device.
    dim3 grid(p.num_heads, num_seqs);
    if (dtype == PA_FP16 && head_size == 64)
        return launch_reduce_t<__half, 64>(p, grid, stream);
    if (dtype == PA_FP16 && head_size == 128)
        return launch_reduce_t<__half, 128>(p, grid, stream);
    if (dtype == PA_BF16 && head_size == 64)
        return launch_reduce_t<__nv_bfloat16, 64>(p, grid, stream);
    if (dtype == PA_BF16 && head_size == 128)
        return launch_reduce_t<__nv_bfloat16, 128>(p, grid, stream);
    return cudaErrorNotSupported;
}

// ---------------------------------------------------------------------------
// Cache write ("PagedAttention 在 vLLM 中的实现分析", sections 3.2 and 7.4).
// In the NHD pool the row of (block, offset) is block*block_size + offset,
// which is the slot itself, so each token's [Hkv, D] row is copied to row
// `slot` of the key plane and of the value plane with 16-byte moves.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    reshape_and_cache_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                             uint4 *__restrict__ cache, const int64_t *__restrict__ slots,
                             int num_tokens, int row_vecs, int64_t key_stride_vecs,
                             int64_t value_stride_vecs, int64_t num_slots, unsigned int *err)
{
    // Launched as the dependent of the kernel before it (which may write the
    // inputs or read the cache): wait for it, then let the kernel after this
    // one (the split-K plan) get resident while the copy runs.
    griddep_wait();
    griddep_launch_dependents();
    const int tok = blockIdx.y;
    const int64_t slot = slots[tok];
    if (slot < 0)
        return; // padding token
    if (slot >= num_slots) {
        if (threadIdx.x == 0 && blockIdx.x == 0)
            atomicOr(err, PA_DEVERR_SLOT);
        return;
    }
    const int64_t plane = num_slots * row_vecs;
    for (int w = blockIdx.x * blockDim.x + threadIdx.x; w < row_vecs; w += gridDim.x * blockDim.x) {
        const uint4 k = key[tok * key_stride_vecs + w];
        const uint4 v = value[tok * value_stride_vecs + w];
        cache[slot * row_vecs + w] = k;
        cache[plane + slot * row_vecs + w] = v;
    }
}

// ---------------------------------------------------------------------------
// Copy-on-write block copy (k4i.top "paged attention" explainer, parallel
// sampling copy-on-write section: a fresh block receives a copy of the shared
// block before the writer's token goes into it).  Grid: x = chunks of a block plane, y = pair;
// each thread moves 16-byte vectors of both planes.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4 *__restrict__ cache, const int64_t *__restrict__ mapping,
                       int num_blocks, int64_t block_vecs, unsigned int *err)
{
    const int64_t src = mapping[2 * (int64_t)blockIdx.y];
    const int64_t dst = mapping[2 * (int64_t)blockIdx.y + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.x == 0)
            atomicOr(err, PA_DEVERR_BLOCK_ID);
        return;
    }
    const int64_t plane = (int64_t)num_blocks * block_vecs;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < block_vecs;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 k = cache[src * block_vecs + i];
        const uint4 v = cache[plane + src * block_vecs + i];
        cache[dst * block_vecs + i] = k;
        cache[plane + dst * block_vecs + i] = v;
    }
}

// Self-test of the bounded waits: one thread waits on an mbarrier phase that
// nothing completes.  The wait gives up after its time limit, the kernel sets
// PA_DEVERR_TIMEOUT and returns.
__global__ void wait_timeout_selftest_kernel(unsigned int *err)
{
    __shared__ uint64_t bar;
    mbar_init(&bar, 1);
    fence_barrier_init();
    if (!mbar_wait(&bar, 0))
        atomicOr(err, PA_DEVERR_TIMEOUT);
    mbar_arrive(&bar); // complete the phase so the barrier is left consistent
}

} // namespace pa

using namespace pa;

// ---------------------------------------------------------------------------
// Host-side checks
// ---------------------------------------------------------------------------
static bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

static bool supported_shape(int head_size, int block_size, int group, int dtype)
{
    return (head_size == 64 || head_size == 128) && (block_size == 16 || block_size == 32) &&
           (group == 1 || group == 2 || group == 4 || group == 8) &&
           (dtype == PA_FP16 || dtype == PA_BF16);
}

static pa_status check_decode_args(const void *out, const void *q, const void *kv_cache,
                                   const int32_t *block_tables, const int32_t *seq_lens,
                                   int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                   int block_size, int num_blocks, int max_blocks_per_seq,
                                   float scale, pa_dtype dtype)
{
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 ||
        block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 || !isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads != 0)
        return PA_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!out || !q || !kv_cache || !block_tables || !seq_lens))
        return PA_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(kv_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (!supported_shape(head_size, block_size, num_heads / num_kv_heads, (int)dtype))
        return PA_ERR_UNSUPPORTED;
    // TMA row coordinates and kernel token counters are 32-bit.
    if ((int64_t)num_blocks * block_size >= (int64_t)INT32_MAX ||
        (int64_t)max_blocks_per_seq * block_size >= (int64_t)INT32_MAX)
        return PA_ERR_UNSUPPORTED;
    if (num_kv_heads > 65535 || num_seqs > 65535 || (int64_t)num_seqs * num_heads > INT32_MAX)
        return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

static const float kLog2e = 1.4426950408889634f;
// Full partitions per run item of the split-K work list (see the plan kernel).
static const int kSplitRun = 4;

extern "C" {

int pa_version(void) { return 10000; }

pa_status pa_profile_kernel_events(void *before, void *after)
{
    if ((before == nullptr) != (after == nullptr))
        return PA_ERR_INVALID_ARG;
    t_mark_before = static_cast<cudaEvent_t>(before);
    t_mark_after = static_cast<cudaEvent_t>(after);
    return PA_OK;
}

const char *pa_status_string(pa_status status)
{
    switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_OUT_OF_RANGE: return "PA_ERR_OUT_OF_RANGE";
    }
    return "PA_ERR_UNKNOWN";
}

pa_status pa_reshape_and_cache(const void *key, const void *value, void *kv_cache,
                               const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                               int head_size, int block_size, int num_blocks,
                               int64_t key_stride, int64_t value_stride, pa_dtype dtype,
                               void *stream)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 ||
        num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_FP16 && dtype != PA_BF16)
        return PA_ERR_UNSUPPORTED;
    const int64_t row = (int64_t)num_kv_heads * head_size;
    if (key_stride < row || value_stride < row || key_stride % 8 || value_stride % 8 || row % 8)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0)
        return PA_OK;
    if (!key || !value || !kv_cache || !slot_mapping)
        return PA_ERR_INVALID_ARG;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(kv_cache, 16) ||
        !aligned(slot_mapping, 8))
        return PA_ERR_INVALID_ARG;
    if (num_tokens > 65535 || row / 8 > INT32_MAX)
        return PA_ERR_UNSUPPORTED;
    cudaError_t e;
    unsigned int *err = device_error_word(&e);
    if (!err)
        return PA_ERR_CUDA;
    const int row_vecs = (int)(row / 8);
    const int threads = 256;
    int bx = (row_vecs + threads - 1) / threads;
    dim3 grid(bx, num_tokens);
    const cudaError_t le = launch_after_previous(
        reshape_and_cache_kernel, grid, dim3(threads), 0, static_cast<cudaStream_t>(stream),
        static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
        static_cast<uint4 *>(kv_cache), slot_mapping, num_tokens, row_vecs,
        (int64_t)(key_stride / 8), (int64_t)(value_stride / 8), (int64_t)num_blocks * block_size,
        err);
    return le == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_decode(void *out, const void *q, const void *kv_cache, const int32_t *block_tables,
                    const int32_t *seq_lens, int num_seqs, int num_heads, int num_kv_heads,
                    int head_size, int block_size, int num_blocks, int max_blocks_per_seq,
                    float scale, pa_dtype dtype, void *stream)
{
    pa_status st = check_decode_args(out, q, kv_cache, block_tables, seq_lens, num_seqs,
                                     num_heads, num_kv_heads, head_size, block_size, num_blocks,
                                     max_blocks_per_seq, scale, dtype);
    if (st != PA_OK || num_seqs == 0)
        return st;
    cudaError_t e;
    unsigned int *err = device_error_word(&e);
    if (!err)
        return PA_ERR_CUDA;
    alignas(64) CUtensorMap tmap;
    if (!make_pool_map(&tmap, kv_cache, dtype, num_blocks, block_size, num_kv_heads, head_size))
        return PA_ERR_CUDA;
    const int group = num_heads / num_kv_heads;
    if (use_tc(head_size, group, false)) {
        const int hg = tc::heads_per_cta(group, num_kv_heads);
        const int rows = block_size < 128 / hg ? block_size : 128 / hg;
        alignas(64) CUtensorMap pmap, qmap;
        if (!make_pool_map(&pmap, kv_cache, dtype, num_blocks, block_size, num_kv_heads,
                           head_size, hg, rows) ||
            !make_q_map(&qmap, q, dtype, num_seqs * num_heads, head_size, hg * group))
            return PA_ERR_CUDA;
        tc::TcParams t = {};
        t.out = out;
        t.block_tables = block_tables;
        t.seq_lens = seq_lens;
        t.err = err;
        t.num_heads = num_heads;
        t.num_kv_heads = num_kv_heads;
        t.num_groups = num_kv_heads / hg;
        t.num_blocks = num_blocks;
        t.max_blocks = max_blocks_per_seq;
        t.part_tokens = max_blocks_per_seq * block_size;
        t.max_parts = 1;
        t.len_cap = max_blocks_per_seq * block_size;
        t.qscale = scale * kLog2e;
        auto launch = dtype == PA_BF16 ? launch_decode_tc_bf16 : launch_decode_tc_f16;
        mark_before(static_cast<cudaStream_t>(stream));
        e = launch(block_size, group, hg, false, pmap, qmap, t,
                   dim3(num_kv_heads / hg, num_seqs), static_cast<cudaStream_t>(stream));
        mark_after(static_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? PA_OK : (e == cudaErrorNotSupported ? PA_ERR_UNSUPPORTED : PA_ERR_CUDA);
    }
    DecodeParams p = {};
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.err = err;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.num_blocks = num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.part_tokens = 0;
    p.max_parts = 1;
    p.len_cap = max_blocks_per_seq * block_size;
    p.qscale = scale * kLog2e;
    DecodeKey key = {(int)dtype, head_size, block_size, num_heads / num_kv_heads, false};
    mark_before(static_cast<cudaStream_t>(stream));
    e = launch_decode(key, tmap, p, dim3(num_kv_heads, num_seqs, 1),
                      static_cast<cudaStream_t>(stream));
    mark_after(static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : (e == cudaErrorNotSupported ? PA_ERR_UNSUPPORTED : PA_ERR_CUDA);
}

static size_t splitk_parts(int max_seq_len, int partition_size)
{
    size_t parts = ((size_t)max_seq_len + partition_size - 1) / partition_size;
    return parts ? parts : 1;
}

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Split-K workspace: [header 256 B: work counter, item count] [unit list,
// one per (sequence, partition)] [partial o, fp32 D per row] [partial (m, l)],
// each region 256-byte aligned; rows = B * H * partitions.
struct WsLayout {
    size_t units, o, ml, total;
};

static WsLayout ws_layout(int num_seqs, int num_heads, int head_size, size_t parts)
{
    WsLayout w;
    const size_t rows = (size_t)num_seqs * num_heads * parts;
    w.units = 256;
    w.o = w.units + round_up((size_t)num_seqs * parts * 4, 256);
    w.ml = w.o + round_up(rows * head_size * sizeof(float), 256);
    w.total = w.ml + round_up(rows * 2 * sizeof(float), 256);
    return w;
}

size_t pa_decode_splitk_workspace_size(int num_seqs, int num_heads, int head_size,
                                       int max_seq_len, int partition_size)
{
    if (num_seqs < 0 || num_heads <= 0 || head_size <= 0 || max_seq_len < 0 ||
        partition_size <= 0)
        return 0;
    return ws_layout(num_seqs, num_heads, head_size, splitk_parts(max_seq_len, partition_size)).total;
}

} // extern "C"

// out_f32: write float32 output rows (the cascade's parts) instead of dtype.
static pa_status decode_splitk_impl(void *out, float *lse, const void *q, const void *kv_cache,
                                    const int32_t *block_tables, const int32_t *seq_lens,
                                    int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                    int block_size, int num_blocks, int max_blocks_per_seq,
                                    float scale, pa_dtype dtype, int max_seq_len,
                                    int partition_size, void *workspace, size_t workspace_bytes,
                                    void *stream, bool out_f32 = false)
{
    pa_status st = check_decode_args(out, q, kv_cache, block_tables, seq_lens, num_seqs,
                                     num_heads, num_kv_heads, head_size, block_size, num_blocks,
                                     max_blocks_per_seq, scale, dtype);
    if (st != PA_OK)
        return st;
    if (max_seq_len < 0 || partition_size <= 0 || partition_size % kTok != 0 || !aligned(lse, 4))
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0)
        return PA_OK;
    const size_t parts = splitk_parts(max_seq_len, partition_size);
    if (parts > 65535)
        return PA_ERR_UNSUPPORTED;
    const size_t need = pa_decode_splitk_workspace_size(num_seqs, num_heads, head_size,
                                                        max_seq_len, partition_size);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
        return PA_ERR_WORKSPACE;
    cudaError_t e;
    unsigned int *err = device_error_word(&e);
    if (!err)
        return PA_ERR_CUDA;
    alignas(64) CUtensorMap tmap;
    if (!make_pool_map(&tmap, kv_cache, dtype, num_blocks, block_size, num_kv_heads, head_size))
        return PA_ERR_CUDA;
    const WsLayout lay = ws_layout(num_seqs, num_heads, head_size, parts);
    char *wsb = static_cast<char *>(workspace);
    float *ws_o = reinterpret_cast<float *>(wsb + lay.o);
    float *ws_ml = reinterpret_cast<float *>(wsb + lay.ml);
    const int64_t cap_tab = (int64_t)max_blocks_per_seq * block_size;
    const int64_t cap_ws = (int64_t)parts * partition_size;
    const int len_cap = (int)(cap_tab < cap_ws ? cap_tab : cap_ws);
    const int group = num_heads / num_kv_heads;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (use_tc(head_size, group, true)) {
        const int hg = tc::heads_per_cta(group, num_kv_heads);
        const int ngroups = num_kv_heads / hg;
        const int rows = block_size < 128 / hg ? block_size : 128 / hg;
        alignas(64) CUtensorMap pmap, qmap;
        if (!make_pool_map(&pmap, kv_cache, dtype, num_blocks, block_size, num_kv_heads,
                           head_size, hg, rows) ||
            !make_q_map(&qmap, q, dtype, num_seqs * num_heads, head_size, hg * group))
            return PA_ERR_CUDA;
        uint32_t *hdr = reinterpret_cast<uint32_t *>(wsb);
        uint32_t *units = reinterpret_cast<uint32_t *>(wsb + lay.units);
        const int sms = sm_count(&e);
        if (!sms)
            return PA_ERR_CUDA;
        const size_t bound = (size_t)num_seqs * ngroups * parts;
        const unsigned grid = (unsigned)(bound < (size_t)sms ? bound : (size_t)sms);
        // Runs of kSplitRun full partitions per item for long sequences; each
        // sequence keeps enough trailing single partitions that about three
        // waves of single items end the work list.
        int max_run = 1, keep_single = 0;
        if (parts > 1 && parts <= 4096) {
            max_run = kSplitRun;
            const long long pairs = (long long)num_seqs * ngroups;
            const long long want = 3LL * grid;
            keep_single = (int)((want + pairs - 1) / pairs) - 1;
            keep_single = keep_single < 0 ? 0 : keep_single;
        }
        e = dtype == PA_BF16
                ? launch_after_previous(tc::splitk_plan_kernel<__nv_bfloat16>, dim3(1), dim3(1024), 0,
                                        s, seq_lens, num_seqs, num_heads, ngroups, partition_size,
                                        len_cap, hdr, units, static_cast<__nv_bfloat16 *>(out), lse,
                                        err, out_f32 ? 1 : 0, max_run, keep_single)
                : launch_after_previous(tc::splitk_plan_kernel<__half>, dim3(1), dim3(1024), 0, s,
                                        seq_lens, num_seqs, num_heads, ngroups, partition_size,
                                        len_cap, hdr, units, static_cast<__half *>(out), lse, err,
                                        out_f32 ? 1 : 0, max_run, keep_single);
        if (e != cudaSuccess)
            return PA_ERR_CUDA;
        tc::TcParams t = {};
        t.out = out;
        t.block_tables = block_tables;
        t.seq_lens = seq_lens;
        t.err = err;
        t.hdr = hdr;
        t.units = units;
        t.ws_o = ws_o;
        t.ws_ml = ws_ml;
        t.num_heads = num_heads;
        t.num_kv_heads = num_kv_heads;
        t.num_groups = ngroups;
        t.num_blocks = num_blocks;
        t.max_blocks = max_blocks_per_seq;
        t.part_tokens = partition_size;
        t.max_parts = (int)parts;
        t.len_cap = len_cap;
        t.qscale = scale * kLog2e;
        t.lse = lse;
        t.out_f32 = out_f32 ? 1 : 0;
        t.runs = max_run > 1 ? 1 : 0;
        auto launch = dtype == PA_BF16 ? launch_decode_tc_bf16 : launch_decode_tc_f16;
        mark_before(s);
        e = launch(block_size, group, hg, true, pmap, qmap, t, dim3(grid), s);
        mark_after(s);
        if (e != cudaSuccess)
            return e == cudaErrorNotSupported ? PA_ERR_UNSUPPORTED : PA_ERR_CUDA;
        if (parts > 1) {
            // Merge the partitions of multi-partition sequences.
            ReduceParams r = {out, ws_o, ws_ml, seq_lens, num_heads, (int)parts, partition_size,
                              len_cap, 1, lse, out_f32 ? 1 : 0};
            e = launch_reduce((int)dtype, head_size, r, num_seqs, s);
        }
        return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }

    DecodeParams p = {};
    p.ws_o = ws_o;
    p.ws_ml = ws_ml;
    p.q = q;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.err = err;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.num_blocks = num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.part_tokens = partition_size;
    p.max_parts = (int)parts;
    p.len_cap = len_cap;
    p.qscale = scale * kLog2e;
    p.lse = lse;
    DecodeKey key = {(int)dtype, head_size, block_size, group, true};
    mark_before(s);
    e = launch_decode(key, tmap, p, dim3(num_kv_heads, num_seqs, (unsigned)parts), s);
    mark_after(s);
    if (e != cudaSuccess)
        return e == cudaErrorNotSupported ? PA_ERR_UNSUPPORTED : PA_ERR_CUDA;
    ReduceParams r = {out, ws_o, ws_ml, seq_lens, num_heads, (int)parts, partition_size, len_cap,
                      0, lse, out_f32 ? 1 : 0};
    e = launch_reduce((int)dtype, head_size, r, num_seqs, s);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Merge of attention states and cascade (shared-prefix) decode
// ("PagedAttention 在 vLLM 中的实现分析", section 6.4: the shared prefix is
// attended once without the causal mask, each request's own suffix
// separately, and the two results are combined with the online-softmax
// correction -- merge_attn_states).
// ---------------------------------------------------------------------------

// out = (w_a o_a + w_b o_b) / (w_a + w_b), w_x = exp(lse_x - max), lse =
// max + log(w_a + w_b); a part with lse = -inf is empty, two empty parts give
// 0 and -inf.  One thread per 8 elements (16 bytes) of a row.
template <typename T>
__global__ void __launch_bounds__(256)
    merge_attn_states_kernel(T *__restrict__ out, float *__restrict__ out_lse,
                             const T *__restrict__ o_a, const float *__restrict__ lse_a,
                             const T *__restrict__ o_b, const float *__restrict__ lse_b,
                             int64_t rows, int head_size)
{
    const int vpr = head_size / 8;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t row = idx / vpr;
    if (row >= rows)
        return;
    const int v = (int)(idx - row * vpr);
    const float la = lse_a[row], lb = lse_b[row];
    const size_t off = (size_t)row * head_size + (size_t)v * 8;
    uint4 res = make_uint4(0, 0, 0, 0);
    float lse = -INFINITY;
    if (!(la == -INFINITY && lb == -INFINITY)) {
        const float M = fmaxf(la, lb);
        const float wa = __expf(la - M), wb = __expf(lb - M);
        const float inv = 1.f / (wa + wb);
        const uint4 ua = *reinterpret_cast<const uint4 *>(o_a + off);
        const uint4 ub = *reinterpret_cast<const uint4 *>(o_b + off);
        const T *ea = reinterpret_cast<const T *>(&ua);
        const T *eb = reinterpret_cast<const T *>(&ub);
        T *er = reinterpret_cast<T *>(&res);
        // An empty part (weight 0) is not read: its rows may hold anything.
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float xa = wa > 0.f ? wa * Elem<T>::one(ea[i]) : 0.f;
            const float xb = wb > 0.f ? wb * Elem<T>::one(eb[i]) : 0.f;
            er[i] = Elem<T>::from((xa + xb) * inv);
        }
        lse = M + __logf(wa + wb);
    }
    *reinterpret_cast<uint4 *>(out + off) = res;
    if (out_lse && v == 0)
        out_lse[row] = lse;
}

// N-way merge of float32 parts [nparts][rows][head_size] with log-sum-exps
// [nparts][rows]: out = sum_i w_i o_i / sum_i w_i, w_i = exp(lse_i - max).
// The parts stay in float32 so that the only 16-bit rounding is the final
// one.  Parts with lse = -inf carry no weight and are not read; a row whose
// parts are all empty is zero.
constexpr int kMaxMergeParts = 17; // prefix key chunks (<= 16) + the suffix

template <typename T>
__global__ void __launch_bounds__(256)
    merge_parts_kernel(T *__restrict__ out, const float *__restrict__ parts,
                       const float *__restrict__ lse_parts, int nparts, int64_t rows,
                       int head_size)
{
    griddep_wait(); // launched as the dependent of the suffix decode
    const int vpr = head_size / 8;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t row = idx / vpr;
    if (row >= rows)
        return;
    const int v = (int)(idx - row * vpr);
    // All the parts' log-sum-exps first (independent loads), then the
    // weighted sum with the parts' rows loaded side by side.
    float lv[kMaxMergeParts];
    float M = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMaxMergeParts; ++i) {
        lv[i] = i < nparts ? lse_parts[(size_t)i * rows + row] : -INFINITY;
        M = fmaxf(M, lv[i]);
    }
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
        for (int i = 0; i < kMaxMergeParts; ++i) {
            if (lv[i] == -INFINITY)
                continue;
            const float w = __expf(lv[i] - M);
            den += w;
            const float4 *src = reinterpret_cast<const float4 *>(
                parts + ((size_t)i * rows + row) * head_size + (size_t)v * 8);
            const float4 u0 = src[0], u1 = src[1];
            const float e[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j)
                acc[j] = fmaf(w, e[j], acc[j]);
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    uint4 res;
    T *er = reinterpret_cast<T *>(&res);
#pragma unroll
    for (int j = 0; j < 8; ++j)
        er[j] = Elem<T>::from(acc[j] * inv);
    *reinterpret_cast<uint4 *>(out + (size_t)row * head_size + (size_t)v * 8) = res;
}

// Cascade setup, one CTA per sequence: each sequence's suffix length and
// suffix block table (its entries after the prefix blocks), and a check that
// every table starts with row 0's prefix blocks.
__global__ void cascade_setup_kernel(const int32_t *__restrict__ block_tables,
                                     const int32_t *__restrict__ seq_lens, int max_blocks,
                                     int prefix_blocks, int block_size, int suffix_cols,
                                     int32_t *__restrict__ suffix_lens,
                                     int32_t *__restrict__ suffix_tables, unsigned int *err)
{
    // The plan kernel that follows waits for this grid before it reads the
    // suffix lengths written here; it may get resident meanwhile.
    griddep_launch_dependents();
    const int s = blockIdx.x;
    const int P = prefix_blocks * block_size;
    const int32_t *row = block_tables + (size_t)s * max_blocks;
    if (threadIdx.x == 0) {
        const int L = seq_lens[s];
        if (L < P)
            atomicOr(err, PA_DEVERR_PREFIX);
        suffix_lens[s] = L < P ? 0 : L - P;
    }
    for (int j = threadIdx.x; j < suffix_cols; j += blockDim.x)
        suffix_tables[(size_t)s * suffix_cols + j] =
            prefix_blocks + j < max_blocks ? row[prefix_blocks + j] : -1;
    for (int j = threadIdx.x; j < prefix_blocks; j += blockDim.x)
        if (row[j] != block_tables[j])
            atomicOr(err, PA_DEVERR_PREFIX);
}

extern "C" {

pa_status pa_decode_splitk(void *out, const void *q, const void *kv_cache,
                           const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                           int num_heads, int num_kv_heads, int head_size, int block_size,
                           int num_blocks, int max_blocks_per_seq, float scale, pa_dtype dtype,
                           int max_seq_len, int partition_size, void *workspace,
                           size_t workspace_bytes, void *stream)
{
    return decode_splitk_impl(out, nullptr, q, kv_cache, block_tables, seq_lens, num_seqs,
                              num_heads, num_kv_heads, head_size, block_size, num_blocks,
                              max_blocks_per_seq, scale, dtype, max_seq_len, partition_size,
                              workspace, workspace_bytes, stream);
}

pa_status pa_decode_splitk_lse(void *out, float *lse, const void *q, const void *kv_cache,
                               const int32_t *block_tables, const int32_t *seq_lens,
                               int num_seqs, int num_heads, int num_kv_heads, int head_size,
                               int block_size, int num_blocks, int max_blocks_per_seq,
                               float scale, pa_dtype dtype, int max_seq_len, int partition_size,
                               void *workspace, size_t workspace_bytes, void *stream)
{
    if (!lse && num_seqs > 0)
        return PA_ERR_INVALID_ARG;
    return decode_splitk_impl(out, lse, q, kv_cache, block_tables, seq_lens, num_seqs,
                              num_heads, num_kv_heads, head_size, block_size, num_blocks,
                              max_blocks_per_seq, scale, dtype, max_seq_len, partition_size,
                              workspace, workspace_bytes, stream);
}

} // extern "C"

// Prefill launch; key_split > 1 (non-causal only) gives every CTA a chunk of
// chunk_tiles key tiles and writes part c of out / lse at c * part_stride /
// c * lse_part_stride elements.
static pa_status prefill_impl(void *out, float *lse, const void *q, const void *kv_cache,
                              const int32_t *block_tables, int64_t block_table_stride,
                              const int32_t *seq_lens, const int32_t *query_start_loc,
                              int num_reqs, int num_tokens, int max_query_len, int num_heads,
                              int num_kv_heads, int head_size, int block_size, int num_blocks,
                              int max_blocks_per_seq, float scale, int causal, pa_dtype dtype,
                              int key_split, int chunk_tiles, int64_t part_stride,
                              int64_t lse_part_stride, void *stream, bool out_f32 = false,
                              int fixed_len = -1)
{
    if (num_reqs < 0 || num_tokens < 0 || max_query_len < 0 || num_heads <= 0 ||
        num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_size <= 0 ||
        block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 ||
        block_table_stride < max_blocks_per_seq || !isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if ((head_size != 64 && head_size != 128) || (block_size != 16 && block_size != 32) ||
        (dtype != PA_FP16 && dtype != PA_BF16))
        return PA_ERR_UNSUPPORTED;
    if (num_reqs == 0 || num_tokens == 0 || max_query_len == 0)
        return PA_OK;
    // fixed_len >= 0 (the cascade's prefix pass): one request whose
    // metadata is given by value.
    if (fixed_len >= 0 && (num_reqs != 1 || max_query_len != num_tokens ||
                           (int64_t)fixed_len > (int64_t)max_blocks_per_seq * block_size))
        return PA_ERR_INVALID_ARG;
    if (!out || !q || !kv_cache || !block_tables ||
        (fixed_len < 0 && (!seq_lens || !query_start_loc)))
        return PA_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(lse, 4) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4) || !aligned(query_start_loc, 4))
        return PA_ERR_INVALID_ARG;
    if ((int64_t)num_blocks * block_size >= (int64_t)INT32_MAX ||
        (int64_t)max_blocks_per_seq * block_size >= (int64_t)INT32_MAX ||
        (int64_t)num_tokens + 512 >= (int64_t)INT32_MAX || num_heads > 65535 ||
        num_reqs > 65535)
        return PA_ERR_UNSUPPORTED;
    cudaError_t e;
    unsigned int *err = device_error_word(&e);
    if (!err)
        return PA_ERR_CUDA;
    alignas(64) CUtensorMap pmap, qmap;
    if (!make_pool_map(&pmap, kv_cache, dtype, num_blocks, block_size, num_kv_heads, head_size,
                       1, block_size) ||
        !make_q_rows_map(&qmap, q, dtype, num_tokens, num_heads, head_size))
        return PA_ERR_CUDA;
    PrefillParams p{};
    p.out = out;
    p.lse = lse;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.query_start_loc = query_start_loc;
    p.err = err;
    p.bt_stride = block_table_stride;
    p.num_tokens = num_tokens;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.num_blocks = num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.max_query_len = max_query_len;
    p.causal = causal ? 1 : 0;
    p.qscale = scale * kLog2e;
    if (key_split < 1 || (key_split > 1 && (causal || chunk_tiles < 1)))
        return PA_ERR_INVALID_ARG;
    p.key_split = key_split;
    p.chunk_tiles = key_split > 1 ? chunk_tiles : 1;
    p.part_stride = part_stride;
    p.lse_part_stride = lse_part_stride;
    p.out_f32 = out_f32 ? 1 : 0;
    p.fixed_len = fixed_len;
    // At most 128 query rows per request and an even group size: a CTA's
    // two tiles take two query heads of one kv head (both busy, one K/V
    // stream); otherwise one CTA per 256 rows of one head.
    const int group = num_heads / num_kv_heads;
    p.head_pairs = (max_query_len <= 128 && group % 2 == 0) ? 1 : 0;
    const int rows_cta = p.head_pairs ? 128 : 256;
    // x = query head (or pair), y = request, z = query block from the end x key chunk
    const int64_t zdim = (int64_t)((max_query_len + rows_cta - 1) / rows_cta) * key_split;
    if (zdim > 65535 || num_reqs > 65535)
        return PA_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)(p.head_pairs ? num_heads / 2 : num_heads), (unsigned)num_reqs,
                    (unsigned)zdim);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    e = dtype == PA_BF16 ? launch_prefill_bf16(head_size, block_size, pmap, qmap, p, grid, st)
                         : launch_prefill_f16(head_size, block_size, pmap, qmap, p, grid, st);
    if (e == cudaErrorNotSupported)
        return PA_ERR_UNSUPPORTED;
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" {

pa_status pa_prefill(void *out, float *lse, const void *q, const void *kv_cache,
                     const int32_t *block_tables, int64_t block_table_stride,
                     const int32_t *seq_lens, const int32_t *query_start_loc, int num_reqs,
                     int num_tokens, int max_query_len, int num_heads, int num_kv_heads,
                     int head_size, int block_size, int num_blocks, int max_blocks_per_seq,
                     float scale, int causal, pa_dtype dtype, void *stream)
{
    return prefill_impl(out, lse, q, kv_cache, block_tables, block_table_stride, seq_lens,
                        query_start_loc, num_reqs, num_tokens, max_query_len, num_heads,
                        num_kv_heads, head_size, block_size, num_blocks, max_blocks_per_seq,
                        scale, causal, dtype, 1, 1, 0, 0, stream);
}

pa_status pa_reshape_and_cache_fp8(const void *key, const void *value, void *kv_cache,
                                   const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                                   int head_size, int block_size, int num_blocks,
                                   int64_t key_stride, int64_t value_stride, pa_dtype src_dtype,
                                   float k_scale, float v_scale, void *stream)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 ||
        num_blocks <= 0 || !(k_scale > 0.f) || !(v_scale > 0.f) || !isfinite(k_scale) ||
        !isfinite(v_scale))
        return PA_ERR_INVALID_ARG;
    if (head_size != 128 || (src_dtype != PA_FP16 && src_dtype != PA_BF16))
        return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0)
        return PA_OK;
    const int row = num_kv_heads * head_size;
    if (!key || !value || !kv_cache || !slot_mapping || key_stride < row || value_stride < row ||
        key_stride % 8 || value_stride % 8 || !aligned(key, 16) || !aligned(value, 16) ||
        !aligned(kv_cache, 16) || !aligned(slot_mapping, 8))
        return PA_ERR_INVALID_ARG;
    if (num_tokens > 65535)
        return PA_ERR_UNSUPPORTED;
    cudaError_t e;
    unsigned int *err = device_error_word(&e);
    if (!err)
        return PA_ERR_CUDA;
    const int64_t plane = (int64_t)num_blocks * block_size * row;
    auto launch = src_dtype == PA_BF16 ? launch_reshape_fp8_bf16 : launch_reshape_fp8_f16;
    e = launch(key, value, kv_cache, slot_mapping, num_tokens, row, key_stride, value_stride,
               plane, block_size, (int64_t)num_blocks * block_size, k_scale, v_scale, err,
               static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// FP8 split-K workspace: the 16-bit layout, then the query's e4m3 parts
// [3][B*H][128] and its row scales [B*H] (tensor-core path).
static size_t fp8_ws_extra(int num_seqs, int num_heads, int head_size)
{
    const size_t rows = (size_t)num_seqs * num_heads;
    return round_up(3 * rows * head_size, 256) + round_up(rows * 4, 256);
}

size_t pa_decode_splitk_fp8_workspace_size(int num_seqs, int num_heads, int head_size,
                                           int max_seq_len, int partition_size)
{
    const size_t base = pa_decode_splitk_workspace_size(num_seqs, num_heads, head_size,
                                                        max_seq_len, partition_size);
    return base ? base + fp8_ws_extra(num_seqs, num_heads, head_size) : 0;
}

static pa_status decode_fp8_impl(void *out, const void *q, const void *kv_cache,
                                 const int32_t *block_tables, const int32_t *seq_lens,
                                 int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                 int block_size, int num_blocks, int max_blocks_per_seq,
                                 float scale, float k_scale, float v_scale, pa_dtype dtype,
                                 bool split, int max_seq_len, int partition_size,
                                 void *workspace, size_t workspace_bytes, void *stream)
{
    pa_status st = check_decode_args(out, q, kv_cache, block_tables, seq_lens, num_seqs,
                                     num_heads, num_kv_heads, head_size, block_size, num_blocks,
                                     max_blocks_per_seq, scale, dtype);
    if (st != PA_OK)
        return st;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !isfinite(k_scale) || !isfinite(v_scale))
        return PA_ERR_INVALID_ARG;
    if (head_size != 128)
        return PA_ERR_UNSUPPORTED;
    if (split && (max_seq_len < 0 || partition_size <= 0 || partition_size % kTok != 0))
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0)
        return PA_OK;
    cudaError_t e;
    unsigned int *err = device_error_word(&e);
    if (!err)
        return PA_ERR_CUDA;
    alignas(64) CUtensorMap tmap;
    if (!make_pool_map_fp8(&tmap, kv_cache, num_blocks, block_size, num_kv_heads, head_size,
                           block_size))
        return PA_ERR_CUDA;
    const int group = num_heads / num_kv_heads;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto launch = dtype == PA_BF16 ? launch_decode_fp8_bf16 : launch_decode_fp8_f16;
    DecodeParams p = {};
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.err = err;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.num_blocks = num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.qscale = scale * k_scale * kLog2e;
    if (!split) {
        p.part_tokens = 0;
        p.max_parts = 1;
        p.len_cap = max_blocks_per_seq * block_size;
        mark_before(s);
        e = launch(block_size, group, false, tmap, p, v_scale, dim3(num_kv_heads, num_seqs, 1), s);
        mark_after(s);
        return e == cudaSuccess ? PA_OK
                                : (e == cudaErrorNotSupported ? PA_ERR_UNSUPPORTED : PA_ERR_CUDA);
    }
    const size_t parts = splitk_parts(max_seq_len, partition_size);
    if (parts > 65535)
        return PA_ERR_UNSUPPORTED;
    const size_t need = pa_decode_splitk_fp8_workspace_size(num_seqs, num_heads, head_size,
                                                            max_seq_len, partition_size);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
        return PA_ERR_WORKSPACE;
    const WsLayout lay = ws_layout(num_seqs, num_heads, head_size, parts);
    char *wsb = static_cast<char *>(workspace);
    float *ws_o = reinterpret_cast<float *>(wsb + lay.o);
    float *ws_ml = reinterpret_cast<float *>(wsb + lay.ml);
    const int64_t cap_tab = (int64_t)max_blocks_per_seq * block_size;
    const int64_t cap_ws = (int64_t)parts * partition_size;
    const int len_cap = (int)(cap_tab < cap_ws ? cap_tab : cap_ws);
    if (kernel_choice() != kKernelSimt) {
        // Tensor cores: query prepass, plan, persistent split-K, reduce.
        const int rows = num_seqs * num_heads;
        uint8_t *qparts = reinterpret_cast<uint8_t *>(wsb + lay.total);
        float *qscales = reinterpret_cast<float *>(wsb + lay.total +
                                                   round_up(3 * (size_t)rows * head_size, 256));
        const int hg = tc::heads_per_cta(group, num_kv_heads);
        const int ngroups = num_kv_heads / hg;
        // A stage of the FP8 kernel holds 256 (token, head) rows: 256/hg tokens.
        const int stage_tokens = 2 * 128 / hg;
        const int box_rows = block_size < stage_tokens ? block_size : stage_tokens;
        alignas(64) CUtensorMap pmap, qmap;
        if (!make_pool_map_fp8(&pmap, kv_cache, num_blocks, block_size, num_kv_heads, head_size,
                               box_rows, hg) ||
            !make_q_parts_map(&qmap, qparts, rows, hg * group))
            return PA_ERR_CUDA;
        // The plan reads only seq_lens, the query prepass only q: the prepass
        // runs as the plan's dependent (it cannot start before the plan has
        // waited for the kernel before it) and waits for the plan at its end,
        // so the decode kernel's wait on the prepass covers both.
        uint32_t *hdr = reinterpret_cast<uint32_t *>(wsb);
        uint32_t *units = reinterpret_cast<uint32_t *>(wsb + lay.units);
        e = dtype == PA_BF16
                ? launch_after_previous(tc::splitk_plan_kernel<__nv_bfloat16>, dim3(1), dim3(1024), 0,
                                        s, seq_lens, num_seqs, num_heads, ngroups, partition_size,
                                        len_cap, hdr, units, static_cast<__nv_bfloat16 *>(out),
                                        static_cast<float *>(nullptr), err, 0, 1, 0)
                : launch_after_previous(tc::splitk_plan_kernel<__half>, dim3(1), dim3(1024), 0, s,
                                        seq_lens, num_seqs, num_heads, ngroups, partition_size,
                                        len_cap, hdr, units, static_cast<__half *>(out),
                                        static_cast<float *>(nullptr), err, 0, 1, 0);
        if (e != cudaSuccess)
            return PA_ERR_CUDA;
        e = dtype == PA_BF16 ? launch_quantize_q_bf16(q, qparts, qscales, rows, s)
                             : launch_quantize_q_f16(q, qparts, qscales, rows, s);
        if (e != cudaSuccess)
            return PA_ERR_CUDA;
        tc::TcParams t = {};
        t.out = out;
        t.block_tables = block_tables;
        t.seq_lens = seq_lens;
        t.err = err;
        t.hdr = hdr;
        t.units = units;
        t.ws_o = ws_o;
        t.ws_ml = ws_ml;
        t.num_heads = num_heads;
        t.num_kv_heads = num_kv_heads;
        t.num_groups = ngroups;
        t.num_blocks = num_blocks;
        t.max_blocks = max_blocks_per_seq;
        t.part_tokens = partition_size;
        t.max_parts = (int)parts;
        t.len_cap = len_cap;
        t.qscale = scale * k_scale * kLog2e;
        const int sms = sm_count(&e);
        if (!sms)
            return PA_ERR_CUDA;
        const size_t bound = (size_t)num_seqs * ngroups * parts;
        const unsigned grid = (unsigned)(bound < (size_t)sms ? bound : (size_t)sms);
        auto tl = dtype == PA_BF16 ? launch_decode_tc_fp8_bf16 : launch_decode_tc_fp8_f16;
        mark_before(s);
        e = tl(block_size, group, hg, pmap, qmap, t, qscales, rows, v_scale, dim3(grid), s);
        mark_after(s);
        if (e != cudaSuccess)
            return e == cudaErrorNotSupported ? PA_ERR_UNSUPPORTED : PA_ERR_CUDA;
        if (parts > 1) {
            ReduceParams r = {out, ws_o, ws_ml, seq_lens, num_heads, (int)parts, partition_size,
                              len_cap, 1, nullptr};
            e = launch_reduce((int)dtype, head_size, r, num_seqs, s);
        }
        return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }
    p.ws_o = ws_o;
    p.ws_ml = ws_ml;
    p.part_tokens = partition_size;
    p.max_parts = (int)parts;
    p.len_cap = len_cap;
    mark_before(s);
    e = launch(block_size, group, true, tmap, p, v_scale,
               dim3(num_kv_heads, num_seqs, (unsigned)parts), s);
    mark_after(s);
    if (e != cudaSuccess)
        return e == cudaErrorNotSupported ? PA_ERR_UNSUPPORTED : PA_ERR_CUDA;
    ReduceParams r = {out, ws_o, ws_ml, seq_lens, num_heads, (int)parts, partition_size,
                      p.len_cap, 0, nullptr};
    e = launch_reduce((int)dtype, head_size, r, num_seqs, s);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_decode_fp8(void *out, const void *q, const void *kv_cache,
                        const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                        int num_heads, int num_kv_heads, int head_size, int block_size,
                        int num_blocks, int max_blocks_per_seq, float scale, float k_scale,
                        float v_scale, pa_dtype dtype, void *stream)
{
    return decode_fp8_impl(out, q, kv_cache, block_tables, seq_lens, num_seqs, num_heads,
                           num_kv_heads, head_size, block_size, num_blocks, max_blocks_per_seq,
                           scale, k_scale, v_scale, dtype, false, 0, 0, nullptr, 0, stream);
}

pa_status pa_decode_splitk_fp8(void *out, const void *q, const void *kv_cache,
                               const int32_t *block_tables, const int32_t *seq_lens,
                               int num_seqs, int num_heads, int num_kv_heads, int head_size,
                               int block_size, int num_blocks, int max_blocks_per_seq,
                               float scale, float k_scale, float v_scale, pa_dtype dtype,
                               int max_seq_len, int partition_size, void *workspace,
                               size_t workspace_bytes, void *stream)
{
    return decode_fp8_impl(out, q, kv_cache, block_tables, seq_lens, num_seqs, num_heads,
                           num_kv_heads, head_size, block_size, num_blocks, max_blocks_per_seq,
                           scale, k_scale, v_scale, dtype, true, max_seq_len, partition_size,
                           workspace, workspace_bytes, stream);
}

pa_status pa_merge_attn_states(void *out, float *out_lse, const void *o_a, const float *lse_a,
                               const void *o_b, const float *lse_b, int num_tokens,
                               int num_heads, int head_size, pa_dtype dtype, void *stream)
{
    if (num_tokens < 0 || num_heads <= 0 || head_size <= 0)
        return PA_ERR_INVALID_ARG;
    if ((head_size != 64 && head_size != 128) || (dtype != PA_FP16 && dtype != PA_BF16))
        return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0)
        return PA_OK;
    if (!out || !o_a || !o_b || !lse_a || !lse_b || !aligned(out, 16) || !aligned(o_a, 16) ||
        !aligned(o_b, 16) || !aligned(lse_a, 4) || !aligned(lse_b, 4) || !aligned(out_lse, 4))
        return PA_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)num_tokens * num_heads;
    const int64_t threads = rows * (head_size / 8);
    const unsigned grid = (unsigned)((threads + 255) / 256);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == PA_BF16)
        merge_attn_states_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
            static_cast<__nv_bfloat16 *>(out), out_lse, static_cast<const __nv_bfloat16 *>(o_a),
            lse_a, static_cast<const __nv_bfloat16 *>(o_b), lse_b, rows, head_size);
    else
        merge_attn_states_kernel<__half><<<grid, 256, 0, st>>>(
            static_cast<__half *>(out), out_lse, static_cast<const __half *>(o_a), lse_a,
            static_cast<const __half *>(o_b), lse_b, rows, head_size);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Cascade workspace: [256 B header: query_start_loc {0, B}, prefix seq_len]
// [suffix lengths] [suffix tables] [parts: prefix key chunks then the suffix,
// float32] [their lse] [split-K workspace], 256-byte aligned.  The prefix pass
// is split over at most kMaxPrefixSplits key chunks.
constexpr int kMaxPrefixSplits = kMaxMergeParts - 1;

// A side stream for work that may run beside the caller's: per host thread
// and device, a non-blocking stream of the device's highest priority, with
// one event that forks work onto it after the caller's stream and one that
// joins it back.  Created on first use in a (device, driver context) pair and
// kept for the life of the thread.  Returns nullptr, and the caller keeps all
// its work on its own stream, if creation fails or if `caller` is being
// captured into a graph and nothing exists yet (no stream or event is created
// during a capture).
struct SideStream {
    int dev = -1;
    void *ctx = nullptr;
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

static SideStream *side_stream(cudaStream_t caller)
{
    constexpr int kMaxDevices = 16;
    static thread_local SideStream slots[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    void *ctx = current_driver_context();
    SideStream &ss = slots[dev];
    if (ss.stream && ss.dev == dev && ss.ctx == ctx)
        return &ss;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(caller, &cap) != cudaSuccess) {
        cudaGetLastError(); // not this call's error to report
        return nullptr;
    }
    if (cap != cudaStreamCaptureStatusNone)
        return nullptr;
    SideStream n;
    n.dev = dev;
    n.ctx = ctx;
    int least = 0, greatest = 0;
    bool ok = cudaDeviceGetStreamPriorityRange(&least, &greatest) == cudaSuccess &&
              cudaStreamCreateWithPriority(&n.stream, cudaStreamNonBlocking, greatest) ==
                  cudaSuccess &&
              cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        if (n.join)
            cudaEventDestroy(n.join);
        if (n.fork)
            cudaEventDestroy(n.fork);
        if (n.stream)
            cudaStreamDestroy(n.stream);
        cudaGetLastError();
        return nullptr;
    }
    // Objects of an earlier context on this device died with it: not
    // destroyed, only replaced.
    ss = n;
    return &ss;
}

struct CascadeLayout {
    size_t sl, bt, parts, lse, ws, ws_bytes, total;
    int suffix_cols, max_parts;
};

static CascadeLayout cascade_layout(int num_seqs, int num_heads, int head_size,
                                    int max_blocks_per_seq, int prefix_blocks, int block_size,
                                    int max_suffix_len, int partition_size)
{
    CascadeLayout c;
    const size_t rows = (size_t)num_seqs * num_heads;
    const int prefix_tiles = (prefix_blocks * block_size + 127) / 128;
    c.max_parts = (prefix_tiles < kMaxPrefixSplits ? prefix_tiles : kMaxPrefixSplits) + 1;
    c.suffix_cols = max_blocks_per_seq - prefix_blocks > 0 ? max_blocks_per_seq - prefix_blocks : 1;
    c.sl = 0;
    c.bt = c.sl + round_up((size_t)num_seqs * 4, 256);
    c.parts = c.bt + round_up((size_t)num_seqs * c.suffix_cols * 4, 256);
    c.lse = c.parts + round_up((size_t)c.max_parts * rows * head_size * 4, 256);
    c.ws = c.lse + round_up((size_t)c.max_parts * rows * 4, 256);
    c.ws_bytes = ws_layout(num_seqs, num_heads, head_size,
                           splitk_parts(max_suffix_len, partition_size)).total;
    c.total = c.ws + c.ws_bytes;
    return c;
}

size_t pa_cascade_decode_workspace_size(int num_seqs, int num_heads, int head_size,
                                        int max_blocks_per_seq, int prefix_blocks,
                                        int max_seq_len, int block_size, int partition_size)
{
    if (num_seqs < 0 || num_heads <= 0 || head_size <= 0 || max_blocks_per_seq <= 0 ||
        prefix_blocks < 0 || prefix_blocks > max_blocks_per_seq || max_seq_len < 0 ||
        block_size <= 0 || partition_size <= 0)
        return 0;
    const int suffix = max_seq_len - prefix_blocks * block_size;
    return cascade_layout(num_seqs, num_heads, head_size, max_blocks_per_seq, prefix_blocks,
                          block_size, suffix > 0 ? suffix : 0, partition_size).total;
}

pa_status pa_cascade_decode(void *out, const void *q, const void *kv_cache,
                            const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                            int num_heads, int num_kv_heads, int head_size, int block_size,
                            int num_blocks, int max_blocks_per_seq, int prefix_blocks,
                            float scale, pa_dtype dtype, int max_seq_len, int partition_size,
                            void *workspace, size_t workspace_bytes, void *stream)
{
    pa_status st = check_decode_args(out, q, kv_cache, block_tables, seq_lens, num_seqs,
                                     num_heads, num_kv_heads, head_size, block_size, num_blocks,
                                     max_blocks_per_seq, scale, dtype);
    if (st != PA_OK)
        return st;
    if (prefix_blocks < 0 || prefix_blocks > max_blocks_per_seq || max_seq_len < 0 ||
        partition_size <= 0 || partition_size % kTok != 0)
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0)
        return PA_OK;
    if (prefix_blocks == 0)
        return decode_splitk_impl(out, nullptr, q, kv_cache, block_tables, seq_lens, num_seqs,
                                  num_heads, num_kv_heads, head_size, block_size, num_blocks,
                                  max_blocks_per_seq, scale, dtype, max_seq_len, partition_size,
                                  workspace, workspace_bytes, stream);
    const int P = prefix_blocks * block_size;
    const int max_suffix = max_seq_len > P ? max_seq_len - P : 0;
    const CascadeLayout c = cascade_layout(num_seqs, num_heads, head_size, max_blocks_per_seq,
                                           prefix_blocks, block_size, max_suffix, partition_size);
    if (!workspace || workspace_bytes < c.total || !aligned(workspace, 256))
        return PA_ERR_WORKSPACE;
    cudaError_t e;
    unsigned int *err = device_error_word(&e);
    if (!err)
        return PA_ERR_CUDA;
    char *w = static_cast<char *>(workspace);
    int32_t *sl_suf = reinterpret_cast<int32_t *>(w + c.sl);
    int32_t *bt_suf = reinterpret_cast<int32_t *>(w + c.bt);
    const size_t rows = (size_t)num_seqs * num_heads;
    char *parts = w + c.parts;
    float *lse_parts = reinterpret_cast<float *>(w + c.lse);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Key chunks of the prefix pass: enough CTAs for one wave of the SMs.
    const int sms = sm_count(&e);
    if (!sms)
        return PA_ERR_CUDA;
    const int prefix_tiles = (P + 127) / 128;
    const int ctas_per_chunk = (num_seqs <= 128 && (num_heads / num_kv_heads) % 2 == 0)
                                   ? num_heads / 2
                                   : ((num_seqs + 255) / 256) * num_heads;
    int nsplit = (sms + ctas_per_chunk - 1) / ctas_per_chunk;
    nsplit = nsplit < 1 ? 1 : (nsplit > c.max_parts - 1 ? c.max_parts - 1 : nsplit);
    const int chunk_tiles = (prefix_tiles + nsplit - 1) / nsplit;
    nsplit = (prefix_tiles + chunk_tiles - 1) / chunk_tiles;
    // The prefix pass needs nothing from the other kernels (its request
    // metadata goes by value) and the suffix decode nothing the prefix pass
    // writes, so the prefix pass goes to the side stream, forked before the
    // setup kernel and joined before the merge.  Launched first and at the
    // higher priority, its CTAs take SMs while the suffix decode's persistent
    // CTAs take the others and then the SMs the prefix pass frees, instead of
    // the two passes running one after the other.
    SideStream *side = side_stream(s);
    cudaStream_t ps = s;
    if (side) {
        if (cudaEventRecord(side->fork, s) != cudaSuccess ||
            cudaStreamWaitEvent(side->stream, side->fork, 0) != cudaSuccess)
            return PA_ERR_CUDA;
        ps = side->stream;
    }
    // 1. Every query against the shared prefix, no causal mask: one request
    //    whose B query rows are the B sequences' queries, split over nsplit
    //    key chunks (parts 0 .. nsplit-1).
    const int64_t part_elems = (int64_t)rows * head_size;
    st = prefill_impl(parts, lse_parts, q, kv_cache, block_tables, max_blocks_per_seq, nullptr,
                      nullptr, 1, num_seqs, num_seqs, num_heads, num_kv_heads, head_size,
                      block_size, num_blocks, prefix_blocks, scale, 0, dtype, nsplit,
                      chunk_tiles, part_elems, (int64_t)rows, ps, true, P);
    if (st != PA_OK)
        return st;
    if (side && cudaEventRecord(side->join, ps) != cudaSuccess)
        return PA_ERR_CUDA;
    // 2. Each sequence's own suffix (part nsplit), after the setup kernel
    //    has written the suffix lengths and tables.
    cascade_setup_kernel<<<num_seqs, 128, 0, s>>>(block_tables, seq_lens, max_blocks_per_seq,
                                                  prefix_blocks, block_size, c.suffix_cols,
                                                  sl_suf, bt_suf, err);
    if (cudaGetLastError() != cudaSuccess)
        return PA_ERR_CUDA;
    st = decode_splitk_impl(parts + (size_t)nsplit * part_elems * 4, lse_parts + (size_t)nsplit * rows,
                            q, kv_cache, bt_suf, sl_suf, num_seqs, num_heads, num_kv_heads,
                            head_size, block_size, num_blocks, c.suffix_cols, scale, dtype,
                            max_suffix, partition_size, w + c.ws, c.ws_bytes, stream, true);
    if (st != PA_OK)
        return st;
    // 3. Merge the nsplit + 1 parts, after both passes.  After the join the
    //    merge is a plain launch: it waits for everything before it.
    if (side && cudaStreamWaitEvent(s, side->join, 0) != cudaSuccess)
        return PA_ERR_CUDA;
    const int64_t threads = (int64_t)rows * (head_size / 8);
    const unsigned grid = (unsigned)((threads + 255) / 256);
    if (side) {
        if (dtype == PA_BF16)
            merge_parts_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
                static_cast<__nv_bfloat16 *>(out), reinterpret_cast<const float *>(parts),
                static_cast<const float *>(lse_parts), nsplit + 1, (int64_t)rows, head_size);
        else
            merge_parts_kernel<__half><<<grid, 256, 0, s>>>(
                static_cast<__half *>(out), reinterpret_cast<const float *>(parts),
                static_cast<const float *>(lse_parts), nsplit + 1, (int64_t)rows, head_size);
        return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }
    const cudaError_t me =
        dtype == PA_BF16
            ? launch_after_previous(merge_parts_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, s,
                                    static_cast<__nv_bfloat16 *>(out),
                                    reinterpret_cast<const float *>(parts),
                                    static_cast<const float *>(lse_parts), nsplit + 1,
                                    (int64_t)rows, head_size)
            : launch_after_previous(merge_parts_kernel<__half>, dim3(grid), dim3(256), 0, s,
                                    static_cast<__half *>(out),
                                    reinterpret_cast<const float *>(parts),
                                    static_cast<const float *>(lse_parts), nsplit + 1,
                                    (int64_t)rows, head_size);
    return me == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_validate_tables(const int32_t *block_tables, const int32_t *seq_lens,
                             int num_seqs, int max_blocks_per_seq, int block_size,
                             int num_blocks)
{
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!block_tables || !seq_lens))
        return PA_ERR_INVALID_ARG;
    const int64_t cap = (int64_t)max_blocks_per_seq * block_size;
    for (int s = 0; s < num_seqs; ++s) {
        const int64_t L = seq_lens[s];
        if (L < 0 || L > cap)
            return PA_ERR_OUT_OF_RANGE;
        const int64_t nb = (L + block_size - 1) / block_size;
        const int32_t *row = block_tables + (size_t)s * max_blocks_per_seq;
        for (int64_t j = 0; j < nb; ++j)
            if (row[j] < 0 || row[j] >= num_blocks)
                return PA_ERR_OUT_OF_RANGE;
    }
    return PA_OK;
}

pa_status pa_validate_slots(const int64_t *slot_mapping, int num_tokens, int block_size,
                            int num_blocks)
{
    if (num_tokens < 0 || block_size <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_tokens > 0 && !slot_mapping)
        return PA_ERR_INVALID_ARG;
    const int64_t cap = (int64_t)num_blocks * block_size;
    std::unordered_set<int64_t> seen;
    seen.reserve((size_t)num_tokens * 2);
    for (int i = 0; i < num_tokens; ++i) {
        const int64_t s = slot_mapping[i];
        if (s < 0)
            continue;
        if (s >= cap || !seen.insert(s).second)
            return PA_ERR_OUT_OF_RANGE;
    }
    return PA_OK;
}

// ---------------------------------------------------------------------------
// Staging copy on the SMs: 16-byte moves over a grid of a few CTAs per SM.
// Either side may be pinned host memory, which the SMs reach through its
// device mapping over the host link; for the few MB of a decode step's inputs
// and outputs that is faster than a copy-engine transfer.  Pointers that have
// no device mapping, or are not 16-byte aligned, go to cudaMemcpyAsync.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    stage_copy_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src, size_t n16)
{
    // Launched as the dependent of the kernel before it (which may write src
    // or read dst): wait for it, then let the next kernel (the cache write of
    // a step whose inputs this copies in) get resident while the copy runs.
    griddep_wait();
    griddep_launch_dependents();
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
         i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

// The address under which the device reaches p, or null when it has none.
static const void *device_view(const void *p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged ||
        a.type == cudaMemoryTypeHost)
        return a.devicePointer;
    return nullptr;
}

pa_status pa_stage_copy(void *dst, const void *src, size_t bytes, void *stream)
{
    if (bytes == 0)
        return PA_OK;
    if (!dst || !src)
        return PA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *dd = const_cast<void *>(device_view(dst));
    const void *ds = device_view(src);
    cudaError_t e;
    const int sms = (dd && ds) ? sm_count(&e) : 0;
    if (!dd || !ds || !sms || !aligned(dd, 16) || !aligned(ds, 16) || bytes % 16)
        return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, s) == cudaSuccess ? PA_OK
                                                                                : PA_ERR_CUDA;
    const size_t n16 = bytes / 16;
    const size_t want = (n16 + 255) / 256;
    const unsigned grid = (unsigned)(want < (size_t)(4 * sms) ? want : (size_t)(4 * sms));
    return launch_after_previous(stage_copy_kernel, dim3(grid), dim3(256), 0, s,
                                 static_cast<uint4 *>(dd), static_cast<const uint4 *>(ds), n16) ==
                   cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status pa_copy_blocks(void *kv_cache, const int64_t *block_mapping, int num_pairs,
                         int num_blocks, int block_size, int num_kv_heads, int head_size,
                         pa_dtype dtype, void *stream)
{
    if (num_pairs < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_size <= 0)
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_FP16 && dtype != PA_BF16)
        return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0)
        return PA_OK;
    if (!kv_cache || !block_mapping || !aligned(kv_cache, 16) || !aligned(block_mapping, 8))
        return PA_ERR_INVALID_ARG;
    const int64_t block_bytes = (int64_t)block_size * num_kv_heads * head_size * 2;
    if (block_bytes % 16)
        return PA_ERR_INVALID_ARG;
    if (num_pairs > 65535)
        return PA_ERR_UNSUPPORTED;
    cudaError_t e;
    unsigned int *err = device_error_word(&e);
    if (!err)
        return PA_ERR_CUDA;
    const int64_t block_vecs = block_bytes / 16;
    const int64_t per_cta = 256 * 4; // four vectors per thread and plane
    const unsigned gx = (unsigned)((block_vecs + per_cta - 1) / per_cta);
    copy_blocks_kernel<<<dim3(gx, num_pairs), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4 *>(kv_cache), block_mapping, num_blocks, block_vecs, err);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_validate_block_mapping(const int64_t *block_mapping, int num_pairs,
                                    int num_blocks)
{
    if (num_pairs < 0 || num_blocks <= 0 || (num_pairs > 0 && !block_mapping))
        return PA_ERR_INVALID_ARG;
    std::unordered_set<int64_t> dsts, srcs;
    for (int i = 0; i < num_pairs; ++i) {
        const int64_t src = block_mapping[2 * i], dst = block_mapping[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks)
            return PA_ERR_OUT_OF_RANGE;
        if (!dsts.insert(dst).second)
            return PA_ERR_OUT_OF_RANGE;
        srcs.insert(src);
    }
    for (int64_t d : dsts)
        if (srcs.count(d))
            return PA_ERR_OUT_OF_RANGE;
    return PA_OK;
}

pa_status pa_selftest_wait_timeout(void *stream)
{
    cudaError_t e;
    unsigned int *err = device_error_word(&e);
    if (!err)
        return PA_ERR_CUDA;
    wait_timeout_selftest_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(err);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_device_errors(unsigned int *flags, int clear)
{
    if (!flags)
        return PA_ERR_INVALID_ARG;
    cudaError_t e;
    unsigned int *word = device_error_word(&e);
    if (!word)
        return PA_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess)
        return PA_ERR_CUDA;
    if (cudaMemcpy(flags, word, sizeof(unsigned int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return PA_ERR_CUDA;
    if (clear && cudaMemset(word, 0, sizeof(unsigned int)) != cudaSuccess)
        return PA_ERR_CUDA;
    if (clear && cudaDeviceSynchronize() != cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}

} // extern "C"
