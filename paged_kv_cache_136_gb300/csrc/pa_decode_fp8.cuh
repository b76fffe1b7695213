// pa_decode_fp8.cuh -- paged decode attention over an FP8 (e4m3) KV pool,
// head_size 128, and the FP8 cache write.
//
// "PagedAttention 在 vLLM 中的实现分析", section 6.3: with an FP8 cache the
// cache write converts each new K/V row with k_scale / v_scale; the attention
// reads k_scale * e4m3(K) and v_scale * e4m3(V).  The pool
// [2, num_blocks, block_size, num_kv_heads, 128] holds one byte per element,
// so a kv head's row is exactly one 128-byte swizzle segment and a stage of
// 64 tokens moves half the bytes of the 16-bit kernel.
//
// Structure as the 16-bit CUDA-core kernel: one CTA per (kv head, sequence
// [, partition]) and all G query heads of that kv head; a producer warp
// TMA-loads each block's K and V rows ({128 bytes, 1 head, block_size rows}
// boxes, one per lane, block table in lane registers) into a 6-slot ring; 4
// consumer warps compute scores with two threads per token (64 codes each),
// the stage max by shuffles and one named barrier, the online-softmax
// rescale, and o += p v with each thread owning 16 codes of a row.  e4m3
// pairs are widened with the cvt.f16x2.e4m3x2 instruction (exact: every e4m3
// value is an fp16 value) and accumulated in fp32.  k_scale is folded into
// the query scale, v_scale into the output.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_decode.cuh"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace f8 {

constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kTok = 64;                       // tokens per stage
constexpr int kStages = 6;                     // 6 x 16 KB
constexpr int kD = 128;
constexpr int kPlaneBytes = kTok * 128;        // K (or V) rows of a stage
constexpr int kStageBytes = 2 * kPlaneBytes;
constexpr int kQRow = kD + kD / 8;             // padded fp32 query row
constexpr int kBar = 1;

template <int G>
constexpr int smem_bytes()
{
    return 1024 + kStages * kStageBytes + (G * kQRow + kConsumerWarps * G + G * kTok) * 4 +
           2 * kStages * 8;
}

// Four e4m3 codes (one 32-bit word, lowest byte first) -> four floats.
__device__ __forceinline__ void widen4(uint32_t w, float *f)
{
    uint32_t lo, hi;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"((unsigned short)(w & 0xFFFFu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"((unsigned short)(w >> 16)));
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&lo));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
    f[0] = a.x;
    f[1] = a.y;
    f[2] = b.x;
    f[3] = b.y;
}

__device__ __forceinline__ void widen16(const uint4 &v, float (&f)[16])
{
    widen4(v.x, f);
    widen4(v.y, f + 4);
    widen4(v.z, f + 8);
    widen4(v.w, f + 12);
}

// Codes of a value row per thread in the values loop: 16 (one 16-byte chunk)
// for G <= 4; 8 for G = 8, which keeps the G x VW accumulators in registers.
template <int G>
struct ValueMap {
    static constexpr int VW = G >= 8 ? 8 : 16;
    static constexpr int kParts = kD / VW;                  // threads per row
    static constexpr int kTokenGroups = kConsumers / kParts;
};

template <typename T, int BS, int G, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 2)
    decode_fp8_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeParams p,
                      float v_scale)
{
    constexpr int SB = kTok / BS; // pool blocks per stage
    static_assert(kTok % BS == 0 && 32 % SB == 0 && 2 * SB <= 32, "stage geometry");
    const int kvh = blockIdx.x;
    const int s = blockIdx.y;
    const int part = SPLIT ? (int)blockIdx.z : 0;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    int L = p.seq_lens[s];
    if (L < 0 || L > p.len_cap) {
        if (tid == 0)
            atomicOr(p.err, PA_DEVERR_SEQ_LEN_);
        L = L < 0 ? 0 : p.len_cap;
    }
    int t0 = 0, t1 = L;
    if (SPLIT) {
        t0 = part * p.part_tokens;
        t1 = min(L, t0 + p.part_tokens);
        if (t0 >= t1)
            return; // partition past the end: the reduce skips it
    } else if (L == 0) {
        T *out = reinterpret_cast<T *>(p.out) + ((size_t)s * p.num_heads + kvh * G) * kD;
        for (int i = tid; i < G * kD; i += kThreads)
            out[i] = Elem<T>::from(0.f);
        if (p.lse && tid < G)
            p.lse[(size_t)s * p.num_heads + kvh * G + tid] = -INFINITY;
        return;
    }

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *q_s = reinterpret_cast<float *>(smem + kStages * kStageBytes);
    float *red = q_s + G * kQRow;
    float *p_s = red + kConsumerWarps * G;
    uint64_t *full = reinterpret_cast<uint64_t *>(p_s + G * kTok);
    uint64_t *empty = full + kStages;
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    const int nst = (t1 - t0 + kTok - 1) / kTok;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        const int jb0 = t0 / BS;
        const int jend = (t1 + BS - 1) / BS;
        const int32_t *bt = p.block_tables + (size_t)s * p.max_blocks;
        int cbase = jb0;
        int cur = (cbase + lane < jend) ? __ldg(bt + cbase + lane) : -1;
        int nxt = (cbase + 32 + lane < jend) ? __ldg(bt + cbase + 32 + lane) : -1;
        const uint64_t policy = policy_evict_first();
        if (lane == 0)
            prefetch_tensormap(&tmap);
        for (int st = 0; st < nst; ++st) {
            const int slot = st % kStages;
            if (st >= kStages) {
                bool ok = true;
                if (lane == 0)
                    ok = mbar_wait(&empty[slot], ((st / kStages) - 1) & 1);
                if (!__shfl_sync(0xffffffffu, (int)ok, 0)) {
                    if (lane == 0)
                        atomicOr(p.err, PA_DEVERR_TIMEOUT_);
                    break;
                }
            }
            const int jf = jb0 + st * SB;
            if (jf >= cbase + 32) {
                cbase += 32;
                cur = nxt;
                nxt = (cbase + 32 + lane < jend) ? __ldg(bt + cbase + 32 + lane) : -1;
            }
            const int nblk = min(SB, jend - jf);
            uint8_t *stage = smem + slot * kStageBytes;
            if (lane == 0)
                mbar_arrive_expect_tx(&full[slot], (uint32_t)(nblk * BS * kD * 2));
            __syncwarp();
            // One box per lane: block jj = lane / 2, plane = lane % 2.
            const int jj = lane >> 1;
            const int phys = __shfl_sync(0xffffffffu, cur, (jf - cbase + (jj < SB ? jj : 0)) & 31);
            if (lane < nblk * 2) {
                const int plane = lane & 1;
                int row;
                if (phys < 0 || phys >= p.num_blocks) {
                    atomicOr(p.err, PA_DEVERR_BLOCK_ID_);
                    row = p.num_blocks * BS; // past the extent: zero fill
                } else {
                    row = phys * BS;
                }
                tma_load_4d_hint(stage + plane * kPlaneBytes + jj * BS * 128, &tmap, &full[slot],
                                 0, kvh, row, plane, policy);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    {
        const T *qg = reinterpret_cast<const T *>(p.q) + ((size_t)s * p.num_heads + kvh * G) * kD;
        for (int i = tid; i < G * kD; i += kConsumers) {
            const int g = i / kD, d = i % kD;
            q_s[g * kQRow + d + (d >> 5) * 4] = Elem<T>::one(qg[i]) * p.qscale;
        }
    }
    bar_sync(kBar, kConsumers);

    using VM = ValueMap<G>;
    constexpr int VW = VM::VW;
    constexpr int kTokenGroups = VM::kTokenGroups;
    const int tq = tid >> 1, hq = tid & 1;                // scores: token, half row
    const int pc = tid % VM::kParts, tg = tid / VM::kParts; // values: row part, token group
    float m_run[G], l_run[G], o[G][VW];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m_run[g] = -INFINITY;
        l_run[g] = 0.f;
#pragma unroll
        for (int k = 0; k < VW; ++k)
            o[g][k] = 0.f;
    }

    bool aborted = false;
    for (int st = 0; st < nst; ++st) {
        const int slot = st % kStages;
        const bool ok = mbar_wait(&full[slot], (st / kStages) & 1);
        const uint8_t *kb = smem + slot * kStageBytes;
        const uint8_t *vb = kb + kPlaneBytes;
        const int nv = min(kTok, t1 - (t0 + st * kTok));

        // ---- scores: each thread 4 chunks (64 codes) of its token's key row
        float sc[G];
#pragma unroll
        for (int g = 0; g < G; ++g)
            sc[g] = 0.f;
        if (ok && tq < nv) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int gc = hq * 4 + i;
                const uint4 kv =
                    *reinterpret_cast<const uint4 *>(kb + tq * 128 + ((gc ^ (tq & 7)) << 4));
                float kf[16];
                widen16(kv, kf);
                const float *qp = q_s + gc * 16 + (gc >> 1) * 4;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float acc = sc[g];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 qa = *reinterpret_cast<const float4 *>(qp + g * kQRow + 4 * j);
                        acc = fmaf(qa.x, kf[4 * j], acc);
                        acc = fmaf(qa.y, kf[4 * j + 1], acc);
                        acc = fmaf(qa.z, kf[4 * j + 2], acc);
                        acc = fmaf(qa.w, kf[4 * j + 3], acc);
                    }
                    sc[g] = acc;
                }
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
            sc[g] += __shfl_xor_sync(0xffffffffu, sc[g], 1);

        // ---- stage max over the consumer group
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float v = (tq < nv) ? sc[g] : -INFINITY;
#pragma unroll
            for (int off = 2; off < 32; off <<= 1)
                v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
            if (lane == 0)
                red[warp * G + g] = v;
        }
        if (bar_sync_or(kBar, kConsumers, !ok)) {
            aborted = true;
            break;
        }
        float alpha[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float mst = red[g];
#pragma unroll
            for (int w = 1; w < kConsumerWarps; ++w)
                mst = fmaxf(mst, red[w * G + g]);
            const float m_new = fmaxf(m_run[g], mst);
            alpha[g] = ex2(m_run[g] - m_new);
            m_run[g] = m_new;
        }
        if (hq == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g)
                p_s[g * kTok + tq] = (tq < nv) ? ex2(sc[g] - m_run[g]) : 0.f;
        }
        bar_sync(kBar, kConsumers);

        // ---- values: VW codes of the row per thread
#pragma unroll
        for (int g = 0; g < G; ++g) {
            l_run[g] *= alpha[g];
#pragma unroll
            for (int k = 0; k < VW; ++k)
                o[g][k] *= alpha[g];
        }
        for (int t = tg; t < nv; t += kTokenGroups) {
            float vf[VW];
            if constexpr (VW == 16) {
                const uint4 vv =
                    *reinterpret_cast<const uint4 *>(vb + t * 128 + ((pc ^ (t & 7)) << 4));
                widen16(vv, vf);
            } else {
                // half a 16-byte chunk: chunk pc/2, bytes (pc&1)*8 .. +8
                const uint2 vv = *reinterpret_cast<const uint2 *>(
                    vb + t * 128 + (((pc >> 1) ^ (t & 7)) << 4) + (pc & 1) * 8);
                widen4(vv.x, vf);
                widen4(vv.y, vf + 4);
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float pg = p_s[g * kTok + t];
                l_run[g] += pg;
#pragma unroll
                for (int k = 0; k < VW; ++k)
                    o[g][k] = fmaf(pg, vf[k], o[g][k]);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[slot]);
    }
    if (aborted)
        return;

    // ---- merge the token groups (they share the running max)
    bar_sync(kBar, kConsumers);
    float *buf = reinterpret_cast<float *>(smem);
    float *lbuf = buf + kTokenGroups * G * kD;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float4 *dst = reinterpret_cast<float4 *>(buf + (tg * G + g) * kD + pc * VW);
#pragma unroll
        for (int j = 0; j < VW / 4; ++j)
            dst[j] = make_float4(o[g][4 * j], o[g][4 * j + 1], o[g][4 * j + 2], o[g][4 * j + 3]);
        if (pc == 0)
            lbuf[tg * G + g] = l_run[g];
    }
    bar_sync(kBar, kConsumers);
    for (int i = tid; i < G * kD; i += kConsumers) {
        const int g = i / kD, d = i % kD;
        float acc = 0.f, l = 0.f;
#pragma unroll
        for (int j = 0; j < kTokenGroups; ++j) {
            acc += buf[(j * G + g) * kD + d];
            l += lbuf[j * G + g];
        }
        acc *= v_scale;
        const int h = kvh * G + g;
        float mg = m_run[0];
#pragma unroll
        for (int gg = 1; gg < G; ++gg)
            if (gg == g)
                mg = m_run[gg];
        if (SPLIT) {
            const size_t row = ((size_t)s * p.num_heads + h) * p.max_parts + part;
            p.ws_o[row * kD + d] = acc;
            if (d == 0) {
                p.ws_ml[row * 2] = mg;
                p.ws_ml[row * 2 + 1] = l;
            }
        } else {
            T *out = reinterpret_cast<T *>(p.out);
            out[((size_t)s * p.num_heads + h) * kD + d] = Elem<T>::from(acc / l);
            if (p.lse && d == 0)
                p.lse[(size_t)s * p.num_heads + h] = (mg + __log2f(l)) * 0.69314718055994531f;
        }
    }
}

// FP8 cache write: token blockIdx.y, 8 elements per thread.  code =
// e4m3(fp32(x / scale)), nearest-even with saturation to +-448.
template <typename T>
__global__ void __launch_bounds__(256)
    reshape_and_cache_fp8_kernel(const T *__restrict__ key, const T *__restrict__ value,
                                 uint8_t *__restrict__ cache, const int64_t *__restrict__ slots,
                                 int row_elems, int64_t key_stride, int64_t value_stride,
                                 int64_t plane_elems, int block_size, int64_t num_slots,
                                 float k_scale, float v_scale, unsigned int *err)
{
    const int i = blockIdx.y;
    const int64_t slot = slots[i];
    if (slot < 0)
        return;
    if (slot >= num_slots) {
        if (threadIdx.x == 0 && blockIdx.x == 0)
            atomicOr(err, PA_DEVERR_SLOT_);
        return;
    }
    const int e0 = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
    if (e0 >= row_elems)
        return;
    const int64_t dst = slot * row_elems + e0; // slot rows are contiguous: [NB*bs][Hkv*D]
#pragma unroll
    for (int plane = 0; plane < 2; ++plane) {
        const T *src = plane == 0 ? key + (size_t)i * key_stride : value + (size_t)i * value_stride;
        const float sc = plane == 0 ? k_scale : v_scale;
        const uint4 raw = *reinterpret_cast<const uint4 *>(src + e0);
        float f[8];
        unpack8<T>(raw, f);
        uint32_t w[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            uint16_t lo, hi;
            // cvt ... e4m3x2.f32 d, a, b puts a in the upper byte, b in the lower.
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
                : "=h"(lo)
                : "f"(__fdiv_rn(f[4 * j + 1], sc)), "f"(__fdiv_rn(f[4 * j], sc)));
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
                : "=h"(hi)
                : "f"(__fdiv_rn(f[4 * j + 3], sc)), "f"(__fdiv_rn(f[4 * j + 2], sc)));
            w[j] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        *reinterpret_cast<uint2 *>(cache + plane * plane_elems + dst) = make_uint2(w[0], w[1]);
    }
}

template <typename T, int BS, int G, bool SPLIT>
cudaError_t launch_one(const CUtensorMap &tmap, const DecodeParams &p, float v_scale, dim3 grid,
                       cudaStream_t stream)
{
    constexpr int smem = smem_bytes<G>();
    auto kern = decode_fp8_kernel<T, BS, G, SPLIT>;
    static unsigned long long done_mask = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        __atomic_fetch_or(&done_mask, bit, __ATOMIC_ACQ_REL);
    }
    kern<<<grid, kThreads, smem, stream>>>(tmap, p, v_scale);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch(int block_size, int group, bool split, const CUtensorMap &tmap,
                   const DecodeParams &p, float v_scale, dim3 grid, cudaStream_t stream)
{
#define PA_F8_CASE(Gv)                                                                        \
    case Gv:                                                                                  \
        if (block_size == 16)                                                                 \
            return split ? launch_one<T, 16, Gv, true>(tmap, p, v_scale, grid, stream)        \
                         : launch_one<T, 16, Gv, false>(tmap, p, v_scale, grid, stream);      \
        if (block_size == 32)                                                                 \
            return split ? launch_one<T, 32, Gv, true>(tmap, p, v_scale, grid, stream)        \
                         : launch_one<T, 32, Gv, false>(tmap, p, v_scale, grid, stream);      \
        return cudaErrorNotSupported;
    switch (group) {
        PA_F8_CASE(1)
        PA_F8_CASE(2)
        PA_F8_CASE(4)
        PA_F8_CASE(8)
    default: return cudaErrorNotSupported;
    }
#undef PA_F8_CASE
}

template <typename T>
cudaError_t launch_reshape(const void *key, const void *value, void *cache, const int64_t *slots,
                           int num_tokens, int row_elems, int64_t key_stride,
                           int64_t value_stride, int64_t plane_elems, int block_size,
                           int64_t num_slots, float k_scale, float v_scale, unsigned int *err,
                           cudaStream_t stream)
{
    const int per_row = (row_elems / 8 + 255) / 256;
    reshape_and_cache_fp8_kernel<T><<<dim3(per_row, num_tokens), 256, 0, stream>>>(
        static_cast<const T *>(key), static_cast<const T *>(value), static_cast<uint8_t *>(cache),
        slots, row_elems, key_stride, value_stride, plane_elems, block_size, num_slots, k_scale,
        v_scale, err);
    return cudaGetLastError();
}

} // namespace f8
} // namespace pa
