// pa_decode.cuh -- paged decode attention kernels for sm_103a.
//
// One CTA handles one (kv head, sequence[, partition]) work item and all G
// query heads that share the kv head (grouped-query attention).  Its tokens
// are walked in stages of kTok tokens:
//
//   producer warp   reads the sequence's block-table entries into registers
//                   (32 at a time, one entry per lane, the next 32 prefetched),
//                   and for each physical block issues TMA tile loads of the
//                   block's [block_size x head_size] K rows and V rows of this
//                   kv head into a shared-memory ring of kStages stages
//                   ("Paged attention", k4i.top, section "block table":
//                   physical_block = block_table[t // block_size]).
//   4 consumer warps for each stage: scores s = (scale*log2 e) q.K in fp32,
//                   stage max by warp shuffles + one named barrier, online
//                   softmax rescale of the running (m, l, o) ("Paged
//                   attention", section "对非连续 blocks 做 attention"), then
//                   o += p V.  The stage slot is handed back to the producer
//                   through an mbarrier.
//
// Tiles land with the TMA 128-byte swizzle: inside each 128-byte row segment
// the 16-byte chunk c of row r sits at position c ^ (r & 7).  Both the score
// and the value loops read 16-byte chunks conflict-free with that pattern.
//
// The one-pass kernel writes out = o / l.  The split-K kernel writes the
// unnormalised (o, m, l) of its partition to the workspace; a second kernel
// merges partitions with the log-sum-exp rescale ("PagedAttention 在 vLLM 中
// 的实现分析", section 7.3).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32; // + one producer warp
constexpr int kTok = 64;                  // tokens per pipeline stage
constexpr int kStages = 3;              // 3 x 32 KB ring: two CTAs fit on an SM
constexpr int kBarConsumers = 1;          // named barrier id of the consumer group

template <int D>
struct Geometry {
    static constexpr int kRegions = D / 64;           // 128-byte segments per row
    static constexpr int kRegionBytes = kTok * 128;   // one segment column of a stage
    static constexpr int kPlaneBytes = kRegions * kRegionBytes; // K (or V) of a stage
    static constexpr int kStageBytes = 2 * kPlaneBytes;
    static constexpr int kChunks = D / 8;             // 16-byte chunks per row
    static constexpr int kTokenGroups = kConsumers / kChunks; // value-loop token groups
    static constexpr int kQRow = D + D / 8;           // padded fp32 query row
};

template <typename T>
struct Elem;
template <>
struct Elem<__half> {
    static __device__ __forceinline__ float2 pair(uint32_t w)
    {
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
    }
    static __device__ __forceinline__ float one(__half x) { return __half2float(x); }
    static __device__ __forceinline__ __half from(float x) { return __float2half_rn(x); }
};
template <>
struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float2 pair(uint32_t w)
    {
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
    }
    static __device__ __forceinline__ float one(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from(float x) { return __float2bfloat16_rn(x); }
};

// Element idx of an output row buffer: the input dtype T, or float32 when
// f32 is set (the cascade keeps its partial results in float32 so that
// merging them adds no 16-bit rounding).
template <typename T>
__device__ __forceinline__ void put_out(void *base, size_t idx, float v, int f32)
{
    if (f32)
        reinterpret_cast<float *>(base)[idx] = v;
    else
        reinterpret_cast<T *>(base)[idx] = Elem<T>::from(v);
}

template <typename T>
__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8])
{
    float2 a = Elem<T>::pair(v.x), b = Elem<T>::pair(v.y), c = Elem<T>::pair(v.z),
           d = Elem<T>::pair(v.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

template <int D, int G>
constexpr int decode_smem_bytes()
{
    using Geo = Geometry<D>;
    return 1024 /* alignment slack */ + kStages * Geo::kStageBytes +
           (G * Geo::kQRow + kConsumerWarps * G + G * kTok) * 4 + 2 * kStages * 8;
}

template <typename T, int D, int BS, int G, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 2)
    decode_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeParams p)
{
    using Geo = Geometry<D>;
    constexpr int SB = kTok / BS; // physical blocks per stage
    static_assert(kTok % BS == 0 && 32 % SB == 0, "stage/block geometry");
    static_assert(SB * 2 * Geometry<D>::kRegions <= 32, "one TMA box per producer lane");
    static_assert(D == 64 || D == 128, "head_size");

    const int kvh = blockIdx.x;
    const int s = blockIdx.y;
    const int part = SPLIT ? (int)blockIdx.z : 0;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // Sequence length, guarded: never walk past the table (or workspace).
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
            return; // partition past the sequence end: the reduce skips it
    } else if (L == 0) {
        T *out = reinterpret_cast<T *>(p.out) + ((size_t)s * p.num_heads + kvh * G) * D;
        for (int i = tid; i < G * D; i += kThreads)
            out[i] = Elem<T>::from(0.f);
        if (p.lse && tid < G)
            p.lse[(size_t)s * p.num_heads + kvh * G + tid] = -INFINITY;
        return;
    }

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *q_s = reinterpret_cast<float *>(smem + kStages * Geo::kStageBytes);
    float *red = q_s + G * Geo::kQRow;
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
        const int jb0 = t0 / BS;                // first logical block
        const int jend = (t1 + BS - 1) / BS;    // one past the last
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
                // One lane waits; the verdict is broadcast so the warp stays
                // converged for the shuffles below.
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
            uint8_t *stage = smem + slot * Geo::kStageBytes;
            if (lane == 0)
                mbar_arrive_expect_tx(&full[slot], (uint32_t)(nblk * BS * D * 2 * 2));
            __syncwarp();
            // One TMA box per lane: box i covers block jj = i / (2*kRegions),
            // plane, 64-element region.  Issuing from many lanes at once keeps
            // the copy engine fed (one issuing thread cannot).
            constexpr int kBoxesPerBlock = 2 * Geo::kRegions;
            const int jj = lane / kBoxesPerBlock;
            const int phys = __shfl_sync(0xffffffffu, cur, (jf - cbase + (jj < SB ? jj : 0)) & 31);
            if (lane < nblk * kBoxesPerBlock) {
                const int rem = lane % kBoxesPerBlock;
                const int plane = rem / Geo::kRegions;
                const int r = rem % Geo::kRegions;
                int row;
                if (phys < 0 || phys >= p.num_blocks) {
                    // Never dereference a bad id: a row past the tensor's
                    // extent makes TMA fill the tile with zeros.
                    atomicOr(p.err, PA_DEVERR_BLOCK_ID_);
                    row = p.num_blocks * BS;
                } else {
                    row = phys * BS;
                }
                tma_load_4d_hint(stage + plane * Geo::kPlaneBytes + r * Geo::kRegionBytes + jj * BS * 128,
                                 &tmap, &full[slot], r * 64, kvh, row, plane, policy);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    {
        const T *qg = reinterpret_cast<const T *>(p.q) + ((size_t)s * p.num_heads + kvh * G) * D;
        for (int i = tid; i < G * D; i += kConsumers) {
            const int g = i / D, d = i % D;
            q_s[g * Geo::kQRow + d + (d >> 5) * 4] = Elem<T>::one(qg[i]) * p.qscale;
        }
    }
    bar_sync(kBarConsumers, kConsumers);

    // Score mapping: two threads per token, each half of head_size.
    const int tq = tid >> 1;
    const int hq = tid & 1;
    // Value mapping: thread owns one 16-byte chunk of the row for a token group.
    const int pc = tid % Geo::kChunks;
    const int tg = tid / Geo::kChunks;

    float m_run[G], l_run[G], o[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m_run[g] = -INFINITY;
        l_run[g] = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            o[g][k] = 0.f;
    }

    bool aborted = false;
    for (int st = 0; st < nst; ++st) {
        const int slot = st % kStages;
        const bool ok = mbar_wait(&full[slot], (st / kStages) & 1);
        const uint8_t *kb = smem + slot * Geo::kStageBytes;
        const uint8_t *vb = kb + Geo::kPlaneBytes;
        const int nv = min(kTok, t1 - (t0 + st * kTok)); // valid tokens this stage

        // ---- scores
        float sc[G];
#pragma unroll
        for (int g = 0; g < G; ++g)
            sc[g] = 0.f;
        if (ok && tq < nv) {
            constexpr int kHalf = Geo::kChunks / 2; // chunks per thread
#pragma unroll
            for (int i = 0; i < kHalf; ++i) {
                // D=128: the two halves walk their 8 chunks in orders that differ
                // in bit 2, so a quarter-warp touches 8 distinct bank groups.
                const int gc = hq * kHalf + (D == 128 ? (i ^ (hq << 2)) : i);
                const int region = gc >> 3, cc = gc & 7;
                const uint4 kv = *reinterpret_cast<const uint4 *>(
                    kb + region * Geo::kRegionBytes + tq * 128 + ((cc ^ (tq & 7)) << 4));
                float kf[8];
                unpack8<T>(kv, kf);
                const float *qp = q_s + gc * 8 + (gc >> 2) * 4;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float4 qa = *reinterpret_cast<const float4 *>(qp + g * Geo::kQRow);
                    const float4 qb = *reinterpret_cast<const float4 *>(qp + g * Geo::kQRow + 4);
                    float acc = sc[g];
                    acc = fmaf(qa.x, kf[0], acc);
                    acc = fmaf(qa.y, kf[1], acc);
                    acc = fmaf(qa.z, kf[2], acc);
                    acc = fmaf(qa.w, kf[3], acc);
                    acc = fmaf(qb.x, kf[4], acc);
                    acc = fmaf(qb.y, kf[5], acc);
                    acc = fmaf(qb.z, kf[6], acc);
                    acc = fmaf(qb.w, kf[7], acc);
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
        if (bar_sync_or(kBarConsumers, kConsumers, !ok)) {
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
        bar_sync(kBarConsumers, kConsumers);

        // ---- values
#pragma unroll
        for (int g = 0; g < G; ++g) {
            l_run[g] *= alpha[g];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                o[g][k] *= alpha[g];
        }
        {
            const int region = pc >> 3, cc = pc & 7;
            const uint8_t *vcol = vb + region * Geo::kRegionBytes;
            for (int t = tg; t < nv; t += Geo::kTokenGroups) {
                const uint4 vv =
                    *reinterpret_cast<const uint4 *>(vcol + t * 128 + ((cc ^ (t & 7)) << 4));
                float vf[8];
                unpack8<T>(vv, vf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float pg = p_s[g * kTok + t];
                    l_run[g] += pg;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        o[g][k] = fmaf(pg, vf[k], o[g][k]);
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[slot]);
    }
    if (aborted)
        return; // every consumer took this branch together (bar.red.or)

    // ---- merge the token groups (all share the same running max)
    bar_sync(kBarConsumers, kConsumers); // everyone is done reading stage memory
    float *buf = reinterpret_cast<float *>(smem);
    float *lbuf = buf + Geo::kTokenGroups * G * D;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float4 *dst = reinterpret_cast<float4 *>(buf + (tg * G + g) * D + pc * 8);
        dst[0] = make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
        dst[1] = make_float4(o[g][4], o[g][5], o[g][6], o[g][7]);
        if (pc == 0)
            lbuf[tg * G + g] = l_run[g];
    }
    bar_sync(kBarConsumers, kConsumers);
    for (int i = tid; i < G * D; i += kConsumers) {
        const int g = i / D, d = i % D;
        float acc = 0.f, l = 0.f;
#pragma unroll
        for (int j = 0; j < Geo::kTokenGroups; ++j) {
            acc += buf[(j * G + g) * D + d];
            l += lbuf[j * G + g];
        }
        const int h = kvh * G + g;
        float mg = m_run[0];
#pragma unroll
        for (int gg = 1; gg < G; ++gg)
            if (gg == g)
                mg = m_run[gg];
        if (SPLIT) {
            const size_t row = ((size_t)s * p.num_heads + h) * p.max_parts + part;
            p.ws_o[row * D + d] = acc;
            if (d == 0) {
                p.ws_ml[row * 2] = mg;
                p.ws_ml[row * 2 + 1] = l;
            }
        } else {
            T *out = reinterpret_cast<T *>(p.out);
            out[((size_t)s * p.num_heads + h) * D + d] = Elem<T>::from(acc / l);
            // m is in log2 units of the scaled score.
            if (p.lse && d == 0)
                p.lse[(size_t)s * p.num_heads + h] = (mg + __log2f(l)) * 0.69314718055994531f;
        }
    }
}

// Log-sum-exp merge of the partitions of one (sequence, query head):
// M = max_p m_p, out = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p.
// Rows of many partitions (long sequences): one CTA per row.  The weights
// w_p = 2^(m_p - M) are formed once per partition in shared memory (chunks
// of kReduceChunk partitions) and the normaliser is a block sum of w_p l_p.
// The kWideWarps warps split the partitions (warp w takes p = w, w + 16, ...);
// lane j loads elements j*E .. j*E+E-1 of a partition's head_size-vector as
// one vector load, so a warp reads a partition's vector in one coalesced
// request and all warps' requests are in flight together; the warps' sums are
// added through shared memory at the end.
constexpr int kReduceChunk = 512;
constexpr int kWideWarps = 16;

template <int E>
struct VecF;
template <>
struct VecF<4> {
    static __device__ __forceinline__ void load(const float *p, float (&v)[4])
    {
        const float4 x = *reinterpret_cast<const float4 *>(p);
        v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w;
    }
};
template <>
struct VecF<2> {
    static __device__ __forceinline__ void load(const float *p, float (&v)[2])
    {
        const float2 x = *reinterpret_cast<const float2 *>(p);
        v[0] = x.x, v[1] = x.y;
    }
};

template <typename T, int D>
__global__ void __launch_bounds__(32 * kWideWarps) splitk_reduce_kernel(const ReduceParams p)
{
    constexpr int NT = 32 * kWideWarps;
    constexpr int E = D / 32; // elements per lane
    __shared__ float w_s[kReduceChunk];
    __shared__ float red_s[kWideWarps];
    __shared__ float acc_s[kWideWarps][D];
    __shared__ float bc_s;
    griddep_wait(); // the partition kernel's states are complete
    const int h = blockIdx.x, s = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int L = p.seq_lens[s];
    L = L < 0 ? 0 : (L > p.len_cap ? p.len_cap : L);
    const int np = (L + p.part_tokens - 1) / p.part_tokens;
    const size_t row0 = ((size_t)s * p.num_heads + h) * p.max_parts;
    const size_t out0 = ((size_t)s * p.num_heads + h) * D;
    if (np == 0) {
        if (tid < D)
            put_out<T>(p.out, out0 + tid, 0.f, p.out_f32);
        if (p.lse && tid == 0)
            p.lse[(size_t)s * p.num_heads + h] = -INFINITY;
        return;
    }
    if (np == 1 && p.skip_single)
        return;
    // Block-wide max / sum of one value per thread, returned to every thread.
    auto block_reduce = [&](float v, bool is_max) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, v, off);
            v = is_max ? fmaxf(v, o) : v + o;
        }
        __syncthreads(); // red_s / bc_s free from the previous use
        if (lane == 0)
            red_s[warp] = v;
        __syncthreads();
        if (tid == 0) {
            float r = red_s[0];
            for (int i = 1; i < kWideWarps; ++i)
                r = is_max ? fmaxf(r, red_s[i]) : r + red_s[i];
            bc_s = r;
        }
        __syncthreads();
        return bc_s;
    };
    float M = -INFINITY;
    for (int q = tid; q < np; q += NT)
        M = fmaxf(M, p.ws_ml[(row0 + q) * 2]);
    M = block_reduce(M, true);
    float den = 0.f; // this thread's share of sum_p w_p l_p
    float a[E];
#pragma unroll
    for (int e = 0; e < E; ++e)
        a[e] = 0.f;
    for (int q0 = 0; q0 < np; q0 += kReduceChunk) {
        const int nq = min(kReduceChunk, np - q0);
        __syncthreads();
        for (int q = tid; q < nq; q += NT) {
            const float w = ex2(p.ws_ml[(row0 + q0 + q) * 2] - M);
            w_s[q] = w;
            den = fmaf(w, p.ws_ml[(row0 + q0 + q) * 2 + 1], den);
        }
        __syncthreads();
        const float *o = p.ws_o + (row0 + q0) * D + lane * E;
#pragma unroll 4
        for (int q = warp; q < nq; q += kWideWarps) {
            // A partition covered by a run of the one before it has weight 0
            // and no vector: skip it.
            const float w = w_s[q];
            if (w == 0.f)
                continue;
            float v[E];
            VecF<E>::load(o + (size_t)q * D, v);
#pragma unroll
            for (int e = 0; e < E; ++e)
                a[e] = fmaf(w, v[e], a[e]);
        }
    }
    den = block_reduce(den, false);
#pragma unroll
    for (int e = 0; e < E; ++e)
        acc_s[warp][lane * E + e] = a[e];
    __syncthreads();
    if (tid < D) {
        float num = 0.f;
#pragma unroll
        for (int w = 0; w < kWideWarps; ++w)
            num += acc_s[w][tid];
        put_out<T>(p.out, out0 + tid, num / den, p.out_f32);
        if (p.lse && tid == 0)
            p.lse[(size_t)s * p.num_heads + h] = (M + __log2f(den)) * 0.69314718055994531f;
    }
}

// The same merge for rows of at most 32 partitions: one warp per
// (sequence, query head), kReduceWarpHeads heads per CTA.  Lane q holds
// partition q's (m_q, l_q), so M and sum_q w_q l_q are warp shuffles with no
// block barrier, and lane j sums output columns j, j+32, ... over the
// partitions (each load instruction of a warp reads 128 contiguous bytes).
// All rows of a decode batch then fit on the GPU at once.
constexpr int kReduceWarpHeads = 8;

template <typename T, int D>
__global__ void __launch_bounds__(32 * kReduceWarpHeads)
    splitk_reduce_warp_kernel(const ReduceParams p)
{
    constexpr int E = D / 32; // output columns per lane
    griddep_wait();           // the partition kernel's states are complete
    const int lane = threadIdx.x & 31;
    const int h = blockIdx.x * kReduceWarpHeads + (threadIdx.x >> 5);
    const int s = blockIdx.y;
    if (h >= p.num_heads)
        return;
    int L = p.seq_lens[s];
    L = L < 0 ? 0 : (L > p.len_cap ? p.len_cap : L);
    const int np = (L + p.part_tokens - 1) / p.part_tokens;
    const size_t row0 = ((size_t)s * p.num_heads + h) * p.max_parts;
    const size_t out0 = ((size_t)s * p.num_heads + h) * D;
    if (np == 0) {
#pragma unroll
        for (int e = 0; e < E; ++e)
            put_out<T>(p.out, out0 + lane + 32 * e, 0.f, p.out_f32);
        if (p.lse && lane == 0)
            p.lse[(size_t)s * p.num_heads + h] = -INFINITY;
        return;
    }
    if (np == 1 && p.skip_single)
        return;
    float m = -INFINITY, l = 0.f;
    if (lane < np) {
        m = p.ws_ml[(row0 + lane) * 2];
        l = p.ws_ml[(row0 + lane) * 2 + 1];
    }
    float M = m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float w = lane < np ? ex2(m - M) : 0.f;
    float den = w * l;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        den += __shfl_xor_sync(0xffffffffu, den, off);
    const float *o = p.ws_o + row0 * D + lane;
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e)
        acc[e] = 0.f;
#pragma unroll 4
    for (int q = 0; q < np; ++q) {
        // A partition covered by a run of the one before it has weight 0 and
        // no vector: skip it.
        const float wq = __shfl_sync(0xffffffffu, w, q);
        if (wq == 0.f)
            continue;
#pragma unroll
        for (int e = 0; e < E; ++e)
            acc[e] = fmaf(wq, o[(size_t)q * D + 32 * e], acc[e]);
    }
#pragma unroll
    for (int e = 0; e < E; ++e)
        put_out<T>(p.out, out0 + lane + 32 * e, acc[e] / den, p.out_f32);
    if (p.lse && lane == 0)
        p.lse[(size_t)s * p.num_heads + h] = (M + __log2f(den)) * 0.69314718055994531f;
}

// Launch helper shared by the instantiation units.
template <typename T, int D, int BS, int G, bool SPLIT>
cudaError_t launch_one(const CUtensorMap &tmap, const DecodeParams &p, dim3 grid,
                       cudaStream_t stream)
{
    constexpr int smem = decode_smem_bytes<D, G>();
    auto kern = decode_kernel<T, D, BS, G, SPLIT>;
    // Opt in to the large dynamic shared-memory carve-out once per device.
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
    kern<<<grid, kThreads, smem, stream>>>(tmap, p);
    return cudaGetLastError();
}

template <typename T, int D, int G>
cudaError_t launch_by_bs(const DecodeKey &key, const CUtensorMap &tmap, const DecodeParams &p,
                         dim3 grid, cudaStream_t stream)
{
    if (key.block_size == 16)
        return key.split ? launch_one<T, D, 16, G, true>(tmap, p, grid, stream)
                         : launch_one<T, D, 16, G, false>(tmap, p, grid, stream);
    if (key.block_size == 32)
        return key.split ? launch_one<T, D, 32, G, true>(tmap, p, grid, stream)
                         : launch_one<T, D, 32, G, false>(tmap, p, grid, stream);
    return cudaErrorNotSupported;
}

template <typename T, int D>
cudaError_t launch_by_group(const DecodeKey &key, const CUtensorMap &tmap, const DecodeParams &p,
                            dim3 grid, cudaStream_t stream)
{
    switch (key.group) {
    case 1: return launch_by_bs<T, D, 1>(key, tmap, p, grid, stream);
    case 2: return launch_by_bs<T, D, 2>(key, tmap, p, grid, stream);
    case 4: return launch_by_bs<T, D, 4>(key, tmap, p, grid, stream);
    case 8: return launch_by_bs<T, D, 8>(key, tmap, p, grid, stream);
    default: return cudaErrorNotSupported;
    }
}

} // namespace pa
