// pa_decode_tc.cuh -- paged decode attention on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory), head_size 128.
//
// Work item: (sequence s, kv head, token range).  Its tokens are walked in
// stages of 128.  Roles in a CTA of 192 threads:
//
//   warp 4 (producer)   takes work items, reads each item's block-table
//                       entries into lane registers, and TMA-loads per stage
//                       the item's query rows (Q, G x 128) and, per physical
//                       block, the block's K and V rows of the kv head
//                       ("Paged attention", k4i.top, section "block table").
//   warp 5 (MMA)        allocates 64 TMEM columns and issues, per stage,
//                         S^T[128 tok x 16] = K[128 x 128] . Q^T   (scores)
//                         O^T[128 d  x 16] = V^T[128 x 128 tok] . P (values)
//                       with tcgen05.mma (M=128, N=16, K=16 per instruction).
//                       S and O are double-buffered in TMEM.
//   warps 0-3           one TMEM lane each: read the scores of their token,
//   (softmax/epilogue)  scale, mask the tail, stage max over the 128 tokens,
//                       online-softmax rescale ("Paged attention",
//                       "对非连续 blocks 做 attention"), write P as a bf16/fp16
//                       high part (B rows 0-7) plus low part (rows 8-15), so
//                       one N=16 MMA carries P to ~16 bits, zero V rows past
//                       the sequence end, then read O for their head_size row
//                       and accumulate o = alpha*o + O[g] + O[8+g].
//
// The K and V tiles are read by the tensor cores straight from the TMA
// layout: K as a K-major operand, V as an MN-major (transposed) operand; both
// use the 128-byte swizzle (shared-memory matrix descriptors).
//
// Split-K ("PagedAttention 在 vLLM 中的实现分析", section 7.3): items are
// (partition of P tokens, kv head) pairs dealt dynamically to a persistent
// grid through an atomic counter.  A sequence with one partition writes its
// output directly; otherwise each partition writes its unnormalised (o, m, l)
// to the workspace and the last partition to finish (an arrival counter per
// (sequence, kv head)) merges them with the log-sum-exp rescale.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_decode.cuh"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace tc {

constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kStages = 3;
constexpr int kTT = 128;                  // tokens per stage
constexpr int kD = 128;                   // head_size
constexpr int kRegion = kTT * 128;        // one 64-element half of 128 rows
constexpr int kPlane = 2 * kRegion;       // K (or V) of a stage
constexpr int kStageBytes = 2 * kPlane;   // K + V
constexpr int kQBytes = 2 * 1024;         // two 64-element halves x 8 rows
constexpr int kPBytes = 4 * 1024;         // two 64-token halves x 16 rows (8 high, 8 low)
constexpr int kTmemCols = 64;
constexpr int kBarEpi = 1;                // named barrier of the softmax warps

constexpr int kOffQ = kStages * kStageBytes;
constexpr int kOffP = kOffQ + kStages * kQBytes;
constexpr int kOffMisc = kOffP + 2 * kPBytes;

constexpr int kFlagFirst = 1, kFlagLast = 2, kFlagStop = 4;

struct StageDesc {
    int s, kvh, part, nvalid, flags, nparts, tok0, pad;
};

struct Misc {
    StageDesc desc[kStages];
    float red[2][4][8];   // per-stage max, double-buffered by stage parity
    float red2[4][8];     // normaliser sums at item end
    int bcast[4];
    uint32_t tmem_base;
    uint32_t pad;
    uint64_t full[kStages], empty[kStages];
    uint64_t s_full[2], p_full[2], o_full[2], o_free[2];
    uint64_t mma_done;
};

constexpr int kSmemBytes = 1024 + kOffMisc + (int)sizeof(Misc);

struct TcParams {
    void *out;                   // [B, H, 128]
    const int32_t *block_tables; // [B, max_blocks]
    const int32_t *seq_lens;     // [B]
    unsigned int *err;
    // split-K workspace (null in one-pass mode)
    uint32_t *hdr;               // [0] work counter, [1] total items
    uint32_t *arrive;            // [B * Hkv] arrival counters
    const uint32_t *units;       // (s << 16) | partition
    float *ws_o;                 // [B, H, max_parts, 128]
    float *ws_ml;                // [B, H, max_parts, 2]
    int num_heads, num_kv_heads, num_blocks, max_blocks;
    int part_tokens, max_parts, len_cap;
    float qscale;
};

template <typename T>
struct Bits;
template <>
struct Bits<__half> {
    static __device__ __forceinline__ void split(float p, uint16_t &hi, uint16_t &lo)
    {
        const __half h = __float2half_rn(p);
        const __half l = __float2half_rn(p - __half2float(h));
        hi = __half_as_ushort(h);
        lo = __half_as_ushort(l);
    }
};
template <>
struct Bits<__nv_bfloat16> {
    static __device__ __forceinline__ void split(float p, uint16_t &hi, uint16_t &lo)
    {
        const __nv_bfloat16 h = __float2bfloat16_rn(p);
        const __nv_bfloat16 l = __float2bfloat16_rn(p - __bfloat162float(h));
        hi = __bfloat16_as_ushort(h);
        lo = __bfloat16_as_ushort(l);
    }
};

__device__ __forceinline__ int clamp_len(int L, int cap, unsigned int *err)
{
    if (L < 0 || L > cap) {
        atomicOr(err, PA_DEVERR_SEQ_LEN_);
        return L < 0 ? 0 : cap;
    }
    return L;
}

// Warp-uniform bounded wait driven by lane 0.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, int lane)
{
    bool ok = true;
    if (lane == 0)
        ok = mbar_wait(bar, parity);
    return __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
}

template <typename T, int BS, int G, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap pool_map,
                     const __grid_constant__ CUtensorMap q_map, const TcParams p)
{
    static_assert(G >= 1 && G <= 8, "group size");
    static_assert(kTT % BS == 0, "block size");
    static_assert((kTT / BS) * 4 <= 32, "one TMA box per producer lane");
    constexpr int SB = kTT / BS;               // physical blocks per stage
    constexpr uint32_t kFmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    constexpr uint32_t kIdescQK = idesc_f16_f32(kFmt, 0, 0, 128, 16);
    constexpr uint32_t kIdescPV = idesc_f16_f32(kFmt, 1, 0, 128, 16);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc *m = reinterpret_cast<Misc *>(smem + kOffMisc);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&m->full[i], 1);
            mbar_init(&m->empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&m->s_full[i], 1);
            mbar_init(&m->p_full[i], 4);
            mbar_init(&m->o_full[i], 1);
            mbar_init(&m->o_free[i], 4);
        }
        mbar_init(&m->mma_done, 1);
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&m->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = m->tmem_base;

    if (warp == kProducerWarp) {
        // ================================================================ producer
        const uint64_t policy = policy_evict_first();
        if (lane == 0) {
            prefetch_tensormap(&pool_map);
            prefetch_tensormap(&q_map);
        }
        uint32_t gk = 0; // global stage counter
        bool alive = true;
        uint32_t total = 0;
        if (SPLIT)
            total = __ldcg(p.hdr + 1);
        int static_done = 0;
        while (alive) {
            // ---- next work item
            int s = 0, kvh = 0, part = 0, L = 0, nparts = 1;
            bool have = false;
            if (SPLIT) {
                uint32_t j = 0;
                if (lane == 0)
                    j = atomicAdd(p.hdr, 1u);
                j = __shfl_sync(0xffffffffu, j, 0);
                if (j < total) {
                    const uint32_t u = __ldg(p.units + j / p.num_kv_heads);
                    kvh = (int)(j % p.num_kv_heads);
                    s = (int)(u >> 16);
                    part = (int)(u & 0xFFFFu);
                    L = clamp_len(__ldg(p.seq_lens + s), p.len_cap, p.err);
                    nparts = (L + p.part_tokens - 1) / p.part_tokens;
                    have = true;
                }
            } else if (!static_done) {
                kvh = blockIdx.x;
                s = blockIdx.y;
                int Lr = __ldg(p.seq_lens + s);
                if (lane == 0)
                    Lr = clamp_len(Lr, p.len_cap, p.err);
                L = __shfl_sync(0xffffffffu, Lr < 0 ? 0 : (Lr > p.len_cap ? p.len_cap : Lr), 0);
                nparts = 1;
                have = L > 0;
                static_done = 1;
                if (!have) {
                    // Empty sequence: its output rows are zero.
                    T *out = reinterpret_cast<T *>(p.out) + ((size_t)s * p.num_heads + kvh * G) * kD;
                    for (int i = lane; i < G * kD; i += 32)
                        out[i] = Elem<T>::from(0.f);
                }
            }
            if (!have)
                break;
            const int tok0 = SPLIT ? part * p.part_tokens : 0;
            const int tok1 = SPLIT ? min(L, tok0 + p.part_tokens) : L;
            const int jb0 = tok0 / BS;
            const int jend = (tok1 + BS - 1) / BS;
            const int nst = (tok1 - tok0 + kTT - 1) / kTT;
            const int32_t *bt = p.block_tables + (size_t)s * p.max_blocks;
            int cbase = jb0;
            int cur = (cbase + lane < jend) ? __ldg(bt + cbase + lane) : -1;
            int nxt = (cbase + 32 + lane < jend) ? __ldg(bt + cbase + 32 + lane) : -1;
            const int qrow = s * p.num_heads + kvh * G;
            for (int st = 0; st < nst; ++st, ++gk) {
                const int slot = gk % kStages;
                if (gk >= kStages && !warp_wait(&m->empty[slot], ((gk / kStages) - 1) & 1, lane)) {
                    if (lane == 0)
                        atomicOr(p.err, PA_DEVERR_TIMEOUT_);
                    alive = false;
                    break;
                }
                const int jf = jb0 + st * SB;
                if (jf >= cbase + 32) {
                    cbase += 32;
                    cur = nxt;
                    nxt = (cbase + 32 + lane < jend) ? __ldg(bt + cbase + 32 + lane) : -1;
                }
                const int nblk = min(SB, jend - jf);
                const int t_lo = tok0 + st * kTT;
                uint8_t *kv = smem + slot * kStageBytes;
                uint8_t *qb = smem + kOffQ + slot * kQBytes;
                if (lane == 0) {
                    StageDesc &d = m->desc[slot];
                    d.s = s;
                    d.kvh = kvh;
                    d.part = part;
                    d.nvalid = min(kTT, tok1 - t_lo);
                    d.flags = (st == 0 ? kFlagFirst : 0) | (st == nst - 1 ? kFlagLast : 0);
                    d.nparts = nparts;
                    d.tok0 = t_lo;
                    mbar_arrive_expect_tx(&m->full[slot],
                                          (uint32_t)(nblk * BS * 128 * 2 * 2 + 2 * G * 128));
                    tma_load_2d(qb, &q_map, &m->full[slot], 0, qrow);
                    tma_load_2d(qb + 1024, &q_map, &m->full[slot], 64, qrow);
                }
                __syncwarp();
                // One K/V box per lane (box i: block i/4, plane, 64-element half).
                const int jj = lane >> 2;
                const int phys = __shfl_sync(0xffffffffu, cur, (jf - cbase + (jj < SB ? jj : 0)) & 31);
                if (lane < nblk * 4) {
                    const int plane = (lane >> 1) & 1;
                    const int r = lane & 1;
                    int row;
                    if (phys < 0 || phys >= p.num_blocks) {
                        atomicOr(p.err, PA_DEVERR_BLOCK_ID_);
                        row = p.num_blocks * BS; // past the extent: zero fill
                    } else {
                        row = phys * BS;
                    }
                    tma_load_4d_hint(kv + plane * kPlane + r * kRegion + jj * BS * 128, &pool_map,
                                     &m->full[slot], r * 64, kvh, row, plane, policy);
                }
            }
        }
        // ---- tell the other roles that no work is left
        if (alive) {
            const int slot = gk % kStages;
            if (gk < kStages || warp_wait(&m->empty[slot], ((gk / kStages) - 1) & 1, lane)) {
                if (lane == 0) {
                    m->desc[slot].flags = kFlagStop;
                    mbar_arrive(&m->full[slot]);
                }
            } else if (lane == 0) {
                atomicOr(p.err, PA_DEVERR_TIMEOUT_);
            }
        }
    } else if (warp == kMmaWarp) {
        // ===================================================================== MMA
        int kq = 0, kp = 0, stop_at = -1;
        unsigned long long idle_since = 0;
        while (stop_at < 0 || kp < stop_at) {
            bool progress = false;
            // Scores of stage kq once it has landed and its S buffer is free.
            if (stop_at < 0 && kq <= kp + 1) {
                const int slot = kq % kStages;
                int ready = 0;
                if (lane == 0)
                    ready = mbar_test_wait(&m->full[slot], (kq / kStages) & 1);
                if (__shfl_sync(0xffffffffu, ready, 0)) {
                    progress = true;
                    int stop = 0;
                    if (lane == 0) // lane 0 did the acquiring wait
                        stop = m->desc[slot].flags & kFlagStop;
                    if (__shfl_sync(0xffffffffu, stop, 0)) {
                        stop_at = kq;
                    } else {
                        tc_fence_after_sync();
                        if (lane == 0) {
                            const uint32_t kbase = smem_addr(smem + slot * kStageBytes);
                            const uint32_t qbase = smem_addr(smem + kOffQ + slot * kQBytes);
                            const uint32_t d_tmem = tmem + (uint32_t)((kq & 1) * 16);
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint32_t koff = (uint32_t)((kk >> 2) * kRegion + (kk & 3) * 32);
                                const uint32_t qoff = (uint32_t)((kk >> 2) * 1024 + (kk & 3) * 32);
                                umma_f16(d_tmem, smem_desc_sw128(kbase + koff, 16, 1024),
                                         smem_desc_sw128(qbase + qoff, 16, 1024), kIdescQK,
                                         kk > 0 ? 1u : 0u);
                            }
                            umma_commit(&m->s_full[kq & 1]);
                        }
                        __syncwarp();
                        ++kq;
                    }
                }
            }
            // Values of stage kp once its P is written and its O buffer is free.
            if (kp < kq) {
                const int b = kp & 1;
                const int u = kp >> 1;
                int ready = 0;
                if (lane == 0)
                    ready = mbar_test_wait(&m->p_full[b], u & 1) &&
                            (u == 0 || mbar_test_wait(&m->o_free[b], (u - 1) & 1));
                if (__shfl_sync(0xffffffffu, ready, 0)) {
                    progress = true;
                    tc_fence_after_sync();
                    if (lane == 0) {
                        const int slot = kp % kStages;
                        const uint32_t vbase = smem_addr(smem + slot * kStageBytes + kPlane);
                        const uint32_t pbase = smem_addr(smem + kOffP + b * kPBytes);
                        const uint32_t d_tmem = tmem + (uint32_t)(32 + b * 16);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t a = smem_desc_sw128(vbase + kk * 2048, kRegion, 1024);
                            const uint32_t poff = (uint32_t)((kk >> 2) * 2048 + (kk & 3) * 32);
                            umma_f16(d_tmem, a, smem_desc_sw128(pbase + poff, 16, 1024), kIdescPV,
                                     kk > 0 ? 1u : 0u);
                        }
                        umma_commit(&m->o_full[b]);
                        umma_commit(&m->empty[slot]);
                    }
                    __syncwarp();
                    ++kp;
                }
            }
            if (progress) {
                idle_since = 0;
            } else {
                const unsigned long long now = global_ns();
                if (idle_since == 0) {
                    idle_since = now;
                } else if (now - idle_since > kWaitLimitNs) {
                    if (lane == 0)
                        atomicOr(p.err, PA_DEVERR_TIMEOUT_);
                    break;
                }
            }
        }
        // Drain: every issued MMA completes before TMEM is released.
        if (lane == 0)
            umma_commit(&m->mma_done);
        warp_wait(&m->mma_done, 0, lane);
    } else {
        // ======================================================== softmax/epilogue
        const int t = tid; // token slot of the stage and head_size row of O
        const uint32_t lane_base = (uint32_t)((warp * 32) << 16);
        float m_run[G], l_part[G], o_acc[G], alpha_prev[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m_run[g] = -INFINITY;
            l_part[g] = 0.f;
            o_acc[g] = 0.f;
            alpha_prev[g] = 0.f;
        }
        bool pending = false; // the previous stage's O is still to be accumulated
        // o = alpha*o + O(stage k), then hand the O buffer back to the MMA warp.
        auto take_o = [&](int k, const float (&alpha)[G]) -> bool {
            const int b = k & 1;
            const bool okw = mbar_wait(&m->o_full[b], (k >> 1) & 1);
            __syncwarp();
            tc_fence_after_sync();
            float ov[16];
            tmem_ld16(tmem + lane_base + (uint32_t)(32 + b * 16), ov);
#pragma unroll
            for (int g = 0; g < G; ++g)
                o_acc[g] = fmaf(o_acc[g], alpha[g], ov[g] + ov[8 + g]);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&m->o_free[b]);
            return okw;
        };
        for (int k = 0;; ++k) {
            const int slot = k % kStages;
            const int b = k & 1;
            const int u = k >> 1;
            bool ok = mbar_wait(&m->full[slot], (k / kStages) & 1);
            const StageDesc d = m->desc[slot];
            if (bar_sync_or(kBarEpi, kEpiThreads, !ok)) {
                if (t == 0)
                    atomicOr(p.err, PA_DEVERR_TIMEOUT_);
                break;
            }
            if (d.flags & kFlagStop)
                break;
            if (d.flags & kFlagFirst) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    m_run[g] = -INFINITY;
                    l_part[g] = 0.f;
                    o_acc[g] = 0.f;
                }
                pending = false;
            }
            ok = mbar_wait(&m->s_full[b], u & 1);
            __syncwarp();
            tc_fence_after_sync();
            float sv[8];
            tmem_ld8(tmem + lane_base + (uint32_t)(b * 16), sv);
            const bool valid = t < d.nvalid;
            float x[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                x[g] = valid ? sv[g] * p.qscale : -INFINITY;
                float v = x[g];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
                if (lane == 0)
                    m->red[b][warp][g] = v;
            }
            if (bar_sync_or(kBarEpi, kEpiThreads, !ok)) {
                if (t == 0)
                    atomicOr(p.err, PA_DEVERR_TIMEOUT_);
                break;
            }
            float alpha[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float mst = fmaxf(fmaxf(m->red[b][0][g], m->red[b][1][g]),
                                        fmaxf(m->red[b][2][g], m->red[b][3][g]));
                const float m_new = fmaxf(m_run[g], mst);
                alpha[g] = ex2(m_run[g] - m_new);
                m_run[g] = m_new;
            }
            // P as the K-major B operand: high part in row g, low part in
            // row 8+g (the next 8-row swizzle atom), column = token t.
            uint8_t *phi = smem + kOffP + b * kPBytes;
            uint8_t *plo = phi + 1024;
            const int poff = (t >> 6) * 2048 + (t & 7) * 2;
            const int pc = (t & 63) >> 3;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float pr = ex2(x[g] - m_run[g]);
                l_part[g] = fmaf(l_part[g], alpha[g], pr);
                uint16_t hi, lo;
                Bits<T>::split(pr, hi, lo);
                const int off = poff + g * 128 + ((pc ^ g) << 4);
                *reinterpret_cast<uint16_t *>(phi + off) = hi;
                *reinterpret_cast<uint16_t *>(plo + off) = lo;
            }
            if (!valid) {
                // V rows past the end may hold anything (stale tiles, NaN
                // padding); P is 0 there, but 0 * NaN would still poison O.
                uint8_t *vrow = smem + slot * kStageBytes + kPlane + t * 128;
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4 *>(vrow + r * kRegion + c * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&m->p_full[b]);

            // The previous stage's values ran on the tensor cores while this
            // stage's softmax was computed; fold them in now.
            if (pending && !take_o(k - 1, alpha_prev) && t == 0)
                atomicOr(p.err, PA_DEVERR_TIMEOUT_);
#pragma unroll
            for (int g = 0; g < G; ++g)
                alpha_prev[g] = alpha[g];
            pending = true;

            if (!(d.flags & kFlagLast))
                continue;
            if (!take_o(k, alpha_prev) && t == 0)
                atomicOr(p.err, PA_DEVERR_TIMEOUT_);
            pending = false;
            // ---- end of the item: normaliser over the 128 token slots
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float v = l_part[g];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane == 0)
                    m->red2[warp][g] = v;
            }
            bar_sync(kBarEpi, kEpiThreads);
            float l[G];
#pragma unroll
            for (int g = 0; g < G; ++g)
                l[g] = (m->red2[0][g] + m->red2[1][g]) + (m->red2[2][g] + m->red2[3][g]);
            const int h0 = d.kvh * G;
            if (!SPLIT || d.nparts == 1) {
                T *out = reinterpret_cast<T *>(p.out) + ((size_t)d.s * p.num_heads + h0) * kD;
#pragma unroll
                for (int g = 0; g < G; ++g)
                    out[g * kD + t] = Elem<T>::from(o_acc[g] / l[g]);
            } else {
                const size_t row0 = ((size_t)d.s * p.num_heads + h0) * p.max_parts + d.part;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const size_t row = row0 + (size_t)g * p.max_parts;
                    p.ws_o[row * kD + t] = o_acc[g];
                    if (t == g) {
                        p.ws_ml[row * 2] = m_run[g];
                        p.ws_ml[row * 2 + 1] = l[g];
                    }
                }
                __threadfence();
                bar_sync(kBarEpi, kEpiThreads);
                if (t == 0) {
                    const uint32_t old = atomicAdd(p.arrive + d.s * p.num_kv_heads + d.kvh, 1u);
                    m->bcast[0] = (old == (uint32_t)(d.nparts - 1)) ? 1 : 0;
                }
                bar_sync(kBarEpi, kEpiThreads);
                if (m->bcast[0]) {
                    // Last partition of (s, kv head): merge every partition.
                    __threadfence();
                    T *out = reinterpret_cast<T *>(p.out) + ((size_t)d.s * p.num_heads + h0) * kD;
                    for (int g = 0; g < G; ++g) {
                        const size_t rg = ((size_t)d.s * p.num_heads + h0 + g) * p.max_parts;
                        float M = -INFINITY;
                        for (int q = 0; q < d.nparts; ++q)
                            M = fmaxf(M, __ldcg(p.ws_ml + (rg + q) * 2));
                        float num = 0.f, den = 0.f;
                        for (int q = 0; q < d.nparts; ++q) {
                            const float w = ex2(__ldcg(p.ws_ml + (rg + q) * 2) - M);
                            den = fmaf(w, __ldcg(p.ws_ml + (rg + q) * 2 + 1), den);
                            num = fmaf(w, __ldcg(p.ws_o + (rg + q) * kD + t), num);
                        }
                        out[g * kD + t] = Elem<T>::from(num / den);
                    }
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Split-K plan: zero the work and arrival counters, list every
// (sequence, partition) unit in sequence order, count the work items
// (units x kv heads), and write zero rows for empty sequences.  One CTA.
template <typename T>
__global__ void __launch_bounds__(1024) splitk_plan_kernel(const int32_t *seq_lens, int B, int H,
                                                           int Hkv, int part_tokens, int len_cap,
                                                           uint32_t *hdr, uint32_t *arrive,
                                                           uint32_t *units, T *out,
                                                           unsigned int *err)
{
    __shared__ uint32_t warp_tot[32];
    __shared__ uint32_t carry_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < B * Hkv; i += blockDim.x)
        arrive[i] = 0;
    if (tid == 0) {
        hdr[0] = 0;
        carry_s = 0;
    }
    __syncthreads();
    for (int c0 = 0; c0 < B; c0 += blockDim.x) {
        const int s = c0 + tid;
        uint32_t n = 0;
        if (s < B) {
            int L = seq_lens[s];
            if (L < 0 || L > len_cap) {
                atomicOr(err, PA_DEVERR_SEQ_LEN_);
                L = L < 0 ? 0 : len_cap;
            }
            n = (uint32_t)((L + part_tokens - 1) / part_tokens);
            if (L == 0)
                for (int i = 0; i < H * 128; ++i)
                    out[(size_t)s * H * 128 + i] = Elem<T>::from(0.f);
        }
        // block exclusive scan of n
        uint32_t v = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off)
                v += y;
        }
        if (lane == 31)
            warp_tot[warp] = v;
        __syncthreads();
        if (warp == 0) {
            uint32_t w = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off)
                    w += y;
            }
            warp_tot[lane] = w; // inclusive prefix over warps
        }
        __syncthreads();
        const uint32_t base = carry_s + (warp ? warp_tot[warp - 1] : 0) + v - n;
        for (uint32_t q = 0; q < n; ++q)
            units[base + q] = ((uint32_t)s << 16) | q;
        __syncthreads();
        if (tid == 0)
            carry_s += warp_tot[(blockDim.x >> 5) - 1];
        __syncthreads();
    }
    if (tid == 0)
        hdr[1] = carry_s * (uint32_t)Hkv;
}

template <typename T, int BS, int G, bool SPLIT>
cudaError_t launch_tc_one(const CUtensorMap &pool, const CUtensorMap &qmap, const TcParams &p,
                          dim3 grid, cudaStream_t stream)
{
    auto kern = decode_tc_kernel<T, BS, G, SPLIT>;
    static unsigned long long done_mask = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess)
            return e;
        __atomic_fetch_or(&done_mask, bit, __ATOMIC_ACQ_REL);
    }
    kern<<<grid, kThreads, kSmemBytes, stream>>>(pool, qmap, p);
    return cudaGetLastError();
}

template <typename T, int G>
cudaError_t launch_tc_bs(int block_size, bool split, const CUtensorMap &pool,
                         const CUtensorMap &qmap, const TcParams &p, dim3 grid,
                         cudaStream_t stream)
{
    if (block_size == 16)
        return split ? launch_tc_one<T, 16, G, true>(pool, qmap, p, grid, stream)
                     : launch_tc_one<T, 16, G, false>(pool, qmap, p, grid, stream);
    if (block_size == 32)
        return split ? launch_tc_one<T, 32, G, true>(pool, qmap, p, grid, stream)
                     : launch_tc_one<T, 32, G, false>(pool, qmap, p, grid, stream);
    return cudaErrorNotSupported;
}

template <typename T>
cudaError_t launch_tc(int block_size, int group, bool split, const CUtensorMap &pool,
                      const CUtensorMap &qmap, const TcParams &p, dim3 grid, cudaStream_t stream)
{
    switch (group) {
    case 1: return launch_tc_bs<T, 1>(block_size, split, pool, qmap, p, grid, stream);
    case 2: return launch_tc_bs<T, 2>(block_size, split, pool, qmap, p, grid, stream);
    case 4: return launch_tc_bs<T, 4>(block_size, split, pool, qmap, p, grid, stream);
    case 8: return launch_tc_bs<T, 8>(block_size, split, pool, qmap, p, grid, stream);
    default: return cudaErrorNotSupported;
    }
}

} // namespace tc
} // namespace pa
