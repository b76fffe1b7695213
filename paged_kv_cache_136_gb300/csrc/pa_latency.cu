// pa_latency.cu -- latency floor of the library's C ABI on the 4-sequence
// decode workload (lengths {1, 17, 33, 64}, block_size 16, 4 q / 4 kv heads,
// head_size 64, fp16, a pool of 32 blocks, 4 new tokens of which one is
// padding), measured without any Python in the loop.
//
// Prints one JSON line:
//   enqueue_us      host time of one API call (it only enqueues work), per
//                   entry point, mean over many calls
//   device_us       device time per call, CUDA events around back-to-back
//                   calls on one stream
//   step_sync_us    host wall time of one decode step made synchronously:
//                   pa_reshape_and_cache + pa_decode_splitk, then
//                   cudaStreamSynchronize -- the floor a serving loop sees
//
// Usage: pa_latency [iterations]
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "pa.h"

#define CHECK_CUDA(x)                                                                    \
    do {                                                                                 \
        cudaError_t e_ = (x);                                                            \
        if (e_ != cudaSuccess) {                                                         \
            fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_));              \
            return 1;                                                                    \
        }                                                                                \
    } while (0)
#define CHECK_PA(x)                                                                      \
    do {                                                                                 \
        pa_status s_ = (x);                                                              \
        if (s_ != PA_OK) {                                                               \
            fprintf(stderr, "%s failed: %s\n", #x, pa_status_string(s_));                \
            return 1;                                                                    \
        }                                                                                \
    } while (0)

namespace {

// Deterministic values in [-1, 1) (a 64-bit linear congruential generator).
struct Lcg {
    uint64_t x;
    float next()
    {
        x = x * 6364136223846793005ull + 1442695040888963407ull;
        return (float)((x >> 40) & 0xFFFFFF) / 8388608.0f - 1.0f;
    }
};

double now_us()
{
    return std::chrono::duration<double, std::micro>(
               std::chrono::steady_clock::now().time_since_epoch())
        .count();
}

} // namespace

int main(int argc, char **argv)
{
    const int iters = argc > 1 ? atoi(argv[1]) : 2000;
    const int B = 4, H = 4, Hkv = 4, D = 64, bs = 16, NB = 32, MB = 4, T = 4;
    const int lens[B] = {1, 17, 33, 64};
    const float scale = 0.125f;
    // Block tables: the first 10 entries of a fixed permutation of the pool.
    const int perm[10] = {7, 19, 3, 28, 11, 24, 0, 15, 30, 9};
    std::vector<int32_t> bt(B * MB, -1), sl(lens, lens + B);
    int next = 0;
    for (int s = 0; s < B; ++s)
        for (int j = 0; j < (lens[s] + bs - 1) / bs; ++j)
            bt[s * MB + j] = perm[next++];
    // New tokens land at each sequence's last position; token 2 is padding.
    std::vector<int64_t> slots(T);
    for (int s = 0; s < T; ++s) {
        const int pos = lens[s] - 1;
        slots[s] = (int64_t)bt[s * MB + pos / bs] * bs + pos % bs;
    }
    slots[2] = -1;
    Lcg g{12345};
    const size_t pool_elems = (size_t)2 * NB * bs * Hkv * D;
    std::vector<__half> pool(pool_elems), q((size_t)B * H * D), kv_new((size_t)T * Hkv * D);
    for (auto &v : pool) v = __float2half(g.next());
    for (auto &v : q) v = __float2half(g.next());
    for (auto &v : kv_new) v = __float2half(g.next());

    void *d_pool, *d_q, *d_out, *d_key, *d_value, *d_bt, *d_sl, *d_slots, *d_ws;
    const int msl = 64, P = 64;
    const size_t ws_bytes = pa_decode_splitk_workspace_size(B, H, D, msl, P);
    CHECK_CUDA(cudaMalloc(&d_pool, pool_elems * 2));
    CHECK_CUDA(cudaMalloc(&d_q, q.size() * 2));
    CHECK_CUDA(cudaMalloc(&d_out, q.size() * 2));
    CHECK_CUDA(cudaMalloc(&d_key, kv_new.size() * 2));
    CHECK_CUDA(cudaMalloc(&d_value, kv_new.size() * 2));
    CHECK_CUDA(cudaMalloc(&d_bt, bt.size() * 4));
    CHECK_CUDA(cudaMalloc(&d_sl, sl.size() * 4));
    CHECK_CUDA(cudaMalloc(&d_slots, slots.size() * 8));
    CHECK_CUDA(cudaMalloc(&d_ws, ws_bytes));
    CHECK_CUDA(cudaMemcpy(d_pool, pool.data(), pool_elems * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_q, q.data(), q.size() * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_key, kv_new.data(), kv_new.size() * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_value, kv_new.data(), kv_new.size() * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_bt, bt.data(), bt.size() * 4, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_sl, sl.data(), sl.size() * 4, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_slots, slots.data(), slots.size() * 8, cudaMemcpyHostToDevice));
    cudaStream_t st;
    CHECK_CUDA(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));

    auto reshape = [&]() {
        return pa_reshape_and_cache(d_key, d_value, d_pool, (const int64_t *)d_slots, T, Hkv, D,
                                    bs, NB, (int64_t)Hkv * D, (int64_t)Hkv * D, PA_FP16, st);
    };
    auto decode = [&]() {
        return pa_decode(d_out, d_q, d_pool, (const int32_t *)d_bt, (const int32_t *)d_sl, B, H,
                         Hkv, D, bs, NB, MB, scale, PA_FP16, st);
    };
    auto splitk = [&]() {
        return pa_decode_splitk(d_out, d_q, d_pool, (const int32_t *)d_bt, (const int32_t *)d_sl,
                                B, H, Hkv, D, bs, NB, MB, scale, PA_FP16, msl, P, d_ws, ws_bytes,
                                st);
    };
    for (int i = 0; i < 50; ++i) {
        CHECK_PA(reshape());
        CHECK_PA(decode());
        CHECK_PA(splitk());
    }
    CHECK_CUDA(cudaStreamSynchronize(st));

    // Host time per call (enqueue only), and device time per call.
    double enq[3], dev[3];
    cudaEvent_t e0, e1;
    CHECK_CUDA(cudaEventCreate(&e0));
    CHECK_CUDA(cudaEventCreate(&e1));
    for (int which = 0; which < 3; ++which) {
        CHECK_CUDA(cudaEventRecord(e0, st));
        const double t0 = now_us();
        for (int i = 0; i < iters; ++i) {
            const pa_status s = which == 0 ? reshape() : which == 1 ? decode() : splitk();
            if (s != PA_OK) {
                fprintf(stderr, "call failed: %s\n", pa_status_string(s));
                return 1;
            }
        }
        const double t1 = now_us();
        CHECK_CUDA(cudaEventRecord(e1, st));
        CHECK_CUDA(cudaEventSynchronize(e1));
        float ms = 0.f;
        CHECK_CUDA(cudaEventElapsedTime(&ms, e0, e1));
        enq[which] = (t1 - t0) / iters;
        dev[which] = 1e3 * ms / iters;
    }
    // A synchronous step: cache write + split-K decode + wait.
    const int sync_iters = iters / 4 > 10 ? iters / 4 : 10;
    std::vector<double> samples(sync_iters);
    for (int i = 0; i < sync_iters; ++i) {
        const double t0 = now_us();
        CHECK_PA(reshape());
        CHECK_PA(splitk());
        CHECK_CUDA(cudaStreamSynchronize(st));
        samples[i] = now_us() - t0;
    }
    std::vector<double> sorted = samples;
    std::sort(sorted.begin(), sorted.end());
    unsigned int flags = 0;
    CHECK_PA(pa_device_errors(&flags, 1));
    printf("{\"workload\": \"4 seqs {1,17,33,64}, 4/4 heads, head_size 64, block_size 16, fp16\", "
           "\"iterations\": %d, "
           "\"enqueue_us\": {\"pa_reshape_and_cache\": %.3f, \"pa_decode\": %.3f, "
           "\"pa_decode_splitk\": %.3f}, "
           "\"device_us\": {\"pa_reshape_and_cache\": %.3f, \"pa_decode\": %.3f, "
           "\"pa_decode_splitk\": %.3f}, "
           "\"step_sync_us\": {\"median\": %.3f, \"p10\": %.3f, \"p90\": %.3f}, "
           "\"device_error_flags\": %u}\n",
           iters, enq[0], enq[1], enq[2], dev[0], dev[1], dev[2], sorted[sync_iters / 2],
           sorted[sync_iters / 10], sorted[(sync_iters * 9) / 10], flags);
    return 0;
}
