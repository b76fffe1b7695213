// pa_decode_tc_fp8.cuh -- paged decode attention over an FP8 (e4m3) KV pool
// on the 5th-generation tensor cores, head_size 128.
//
// The FP8 cache ("PagedAttention 在 vLLM 中的实现分析", section 6.3: the
// cache write converts K/V to FP8 with k_scale / v_scale) is read by the
// tensor cores as it lies in the pool: tcgen05.mma kind::f8f6f4 takes the
// e4m3 key tile (K-major) and value tile (MN-major) straight from the TMA
// ring.  The other operand of each product must be e4m3 too, so:
//
//   scores  S^T = K8 . Q'^T, Q' the query row divided by its own scale
//           (max |q| / 256) and written as three e4m3 parts whose sum
//           carries about 12 significant bits (a prepass kernel makes them
//           once per call); the three parts are 16 columns each of one N=48
//           operand, and the softmax adds the three score columns and
//           multiplies by the row scale;
//   values  O^T = V8^T . P', P' = 256 p written as three e4m3 parts (N=48);
//           the epilogue adds the three column groups and divides by 256.
//
// Everything else -- roles, the (token, kv head) row order of a stage, head
// groups per CTA, lagged O accumulation, the persistent split-K schedule --
// is the 16-bit tensor-core kernel's (pa_decode_tc.cuh), with one change: a
// stage holds 256 (token, kv head) rows -- two 128-row blocks, each with its
// own score columns, and each softmax thread takes one row of each -- so a
// stage moves the same 64 KB as the 16-bit kernel's and the per-stage
// hand-offs are paid once per 64 KB.  The values MMA contracts over all 256
// rows (K = 256); its P operand is written over the stage's own K, which is
// dead once the scores MMA has run, so no stage waits for another's values
// MMA to release a P buffer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_decode_tc.cuh"

namespace pa {
namespace tc8 {

using namespace tc;
// The roles and the stage row count are the 16-bit kernel's.
constexpr int kThreads = tc::kThreads;
constexpr int kEpiThreads = tc::kEpiThreads;
constexpr int kProducerWarp = tc::kProducerWarp;
constexpr int kQkWarp = tc::kQkWarp;
constexpr int kPvWarp = tc::kPvWarp;
constexpr int kBarEpi = tc::kBarEpi;
constexpr int kRows = tc::kRows;
constexpr int kD = tc::kD;

constexpr int kStages = 3;
constexpr int kStageRows = 2 * kRows;      // (token, kv head) rows per stage
constexpr int kRegion = kRows * 128;       // a block of 128 rows x 128 codes
constexpr int kPlane = 2 * kRegion;        // K (or V) of a stage: two row blocks
constexpr int kStageBytes = 2 * kPlane;
constexpr int kParts = 3;                  // e4m3 parts of q' and of 256 p
constexpr int kPartRows = 16;              // (head, query) columns per part
constexpr int kNQ = kParts * kPartRows;    // score columns
constexpr int kNP = kParts * kPartRows;    // value columns
constexpr int kQBytes = kNQ * 128;
constexpr int kPBytes = 2 * kNP * 128;     // K = 256 stage rows: two 128-byte regions
constexpr int kSCols = 2 * kNQ;            // S of one stage: two row blocks
constexpr int kOCol = 2 * kSCols;          // O after the two S buffers
constexpr uint32_t kTmemCols = 512;        // S: 2 x 2 x 48, O: 2 x 48
constexpr float kPScale = 256.f;
constexpr float kInvPScale = 1.f / 256.f;
constexpr float kQRange = 256.f;           // |q'| <= 256

constexpr int kOffQ = kStages * kStageBytes;
// P of a stage lives in the first kPBytes of the stage's K region (see the
// softmax), so it needs no buffer of its own.
constexpr int kOffMisc = kOffQ + kStages * kQBytes;
static_assert(kPBytes <= kPlane && kPBytes % (16 * kEpiThreads) == 0 && (kNP * 128) % 1024 == 0,
              "P fits the K region, clears in whole 16-byte stores, keeps 1024-byte atoms");

struct Misc {
    StageDesc desc[kStages];
    float red[2][4][16];
    float red2[4][16];
    int bcast[4];
    uint32_t tmem_base;
    uint32_t pad;
    uint64_t full[kStages], empty[kStages];
    uint64_t s_full[2], p_full[2], o_full[2], o_free[2];
    uint64_t mma_done[2];
};

constexpr int kSmemBytes = 1024 + kOffMisc + (int)sizeof(Misc);

// D[tmem] (+)= A[smem] * B[smem] with 8-bit operands, issued by one thread.
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n"
        "  .reg .pred p;\n"
        "  setp.ne.u32 p, %4, 0;\n"
        "  tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Byte offset of element (row n, column k) of a K-major 8-bit operand with
// the 128-byte swizzle (rows of 128 codes, 8-row atoms of 1024 bytes).
__device__ __forceinline__ int sw128_offset_b8(int n, int k)
{
    return (n >> 3) * 1024 + (n & 7) * 128 + ((((k >> 4)) ^ (n & 7)) << 4) + (k & 15);
}

// e4m3 code of x (nearest, ties to even, saturating) and its value.
__device__ __forceinline__ uint32_t e4m3_code(float x, float &value)
{
    unsigned short pair;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.f), "f"(x));
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
    value = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
    return pair & 0xFFu;
}

// x as three e4m3 parts: c0 = e4m3(x), c1 = e4m3(x - c0), c2 = e4m3(x - c0 - c1).
__device__ __forceinline__ void split3_e4m3(float x, uint8_t (&c)[3])
{
    float r = x;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        float v;
        c[i] = (uint8_t)e4m3_code(r, v);
        r -= v;
    }
}

// Two values as three e4m3 parts each, exactly as split3_e4m3 would give, with
// one paired conversion per step for both.
__device__ __forceinline__ void split3_e4m3x2(float a, float b, uint8_t (&ca)[3],
                                              uint8_t (&cb)[3])
{
    float ra = a, rb = b;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        unsigned short pair;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(ra), "f"(rb));
        uint32_t h2;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
        ca[i] = (uint8_t)(pair >> 8);
        cb[i] = (uint8_t)(pair & 0xFFu);
        ra -= __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
        rb -= __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
    }
}

// Query prepass: one warp per (sequence, head) row of 128 elements.  scale =
// max|q| / 256 (1 for an all-zero row); the three e4m3 parts of q / scale go
// to parts[p][row][0..127], the scale to scales[row].
template <typename T>
__global__ void __launch_bounds__(128)
    quantize_q_parts_kernel(const T *__restrict__ q, uint8_t *__restrict__ parts,
                            float *__restrict__ scales, int rows)
{
    // Launched as the dependent of the split-K plan, which has already waited
    // for the kernel before it (so q is final); the decode kernel may start
    // its prologue at once.  Every thread waits for the plan before it exits,
    // so this grid completes only after the plan: the decode kernel's wait on
    // it covers both.
    griddep_launch_dependents();
    const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) {
        griddep_wait();
        return;
    }
    const uint2 raw = *reinterpret_cast<const uint2 *>(q + (size_t)row * kD + lane * 4);
    const T *e = reinterpret_cast<const T *>(&raw);
    float x[4], amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[i] = Elem<T>::one(e[i]);
        amax = fmaxf(amax, fabsf(x[i]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float sc = amax > 0.f ? amax / kQRange : 1.f;
    uint32_t w[3] = {0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint8_t c[3];
        split3_e4m3(__fdiv_rn(x[i], sc), c);
#pragma unroll
        for (int pp = 0; pp < 3; ++pp)
            w[pp] |= (uint32_t)c[pp] << (8 * i);
    }
#pragma unroll
    for (int pp = 0; pp < 3; ++pp)
        *reinterpret_cast<uint32_t *>(parts + ((size_t)pp * rows + row) * kD + lane * 4) = w[pp];
    if (lane == 0)
        scales[row] = sc;
    griddep_wait();
}

template <typename T, int BS, int G, int HG, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_fp8_kernel(const __grid_constant__ CUtensorMap pool_map,
                         const __grid_constant__ CUtensorMap q_map, const TcParams p,
                         const float *__restrict__ q_scales, int q_rows, float v_scale)
{
    constexpr int NV = HG * G;                 // valid (head, query) columns
    constexpr int TPS = kStageRows / HG;       // tokens per stage
    constexpr int R = BS < TPS ? BS : TPS;     // token rows per TMA box
    constexpr int CH = TPS / R;                // row chunks per stage
    constexpr int BOX_BYTES = R * HG * 128;
    static_assert(G >= 1 && NV <= kPartRows && (HG & (HG - 1)) == 0, "heads per CTA");
    static_assert(TPS % R == 0 && BS % R == 0 && CH * 2 <= 32, "stage geometry");
    // kind::f8f6f4 with e4m3 operands (format code 0), fp32 accumulation.
    constexpr uint32_t kIdescQK = idesc_f16_f32(0, 0, 0, 128, kNQ);
    constexpr uint32_t kIdescPV = idesc_f16_f32(0, 1, 0, 128, kNP);

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
            mbar_init(&m->mma_done[i], 1);
        }
        fence_barrier_init();
    }
    if (warp == kQkWarp) {
        tmem_alloc(&m->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = m->tmem_base;
    // Everything above overlaps the previous kernel (the plan) when launched
    // as its dependent; from here on its results are read.
    griddep_wait();
    griddep_launch_dependents();

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
        // Split mode resolves the NEXT work item a step at a time while the last
        // stages of the current item are issued, so its chain of dependent
        // loads (work counter -> unit -> seq_len and block table) overlaps the
        // waits for free stage slots instead of stalling the ring at item
        // changes.
        int nstep = 0;                    // steps of the next item done so far
        uint32_t nj_raw = 0, nj = 0, nu = 0;
        int nL_raw = 0, ncur = -1, nnxt = -1, n_s = 0, n_group = 0, n_part = 0;
        bool n_have = false;
        auto next_step = [&]() {
            if (nstep == 0) {
                if (lane == 0)
                    nj_raw = atomicAdd(p.hdr, 1u);
            } else if (nstep == 1) {
                nj = __shfl_sync(0xffffffffu, nj_raw, 0);
                n_have = nj < total;
                if (n_have)
                    nu = __ldg(p.units + nj / p.num_groups);
            } else if (nstep == 2 && n_have) {
                n_group = (int)(nj % p.num_groups);
                n_s = (int)(nu >> 16);
                n_part = (int)(nu & 0xFFFFu);
                nL_raw = __ldg(p.seq_lens + n_s);
                // Table entries past the item's end are loaded but never used.
                const int jb = n_part * p.part_tokens / BS;
                const int32_t *btn = p.block_tables + (size_t)n_s * p.max_blocks;
                ncur = (jb + lane < p.max_blocks) ? __ldg(btn + jb + lane) : -1;
                nnxt = (jb + 32 + lane < p.max_blocks) ? __ldg(btn + jb + 32 + lane) : -1;
            }
            ++nstep;
        };
        bool have_tab = false; // cur/nxt already hold the item's first table entries
        int cur = -1, nxt = -1;
        while (alive) {
            // ---- next work item: (sequence, group of HG kv heads, partition)
            int s = 0, group = 0, part = 0, L = 0, nparts = 1;
            bool have = false;
            if (SPLIT) {
                while (nstep < 3)
                    next_step();
                if (n_have) {
                    s = n_s;
                    group = n_group;
                    part = n_part;
                    int Lr = nL_raw;
                    if (lane == 0)
                        Lr = clamp_len(Lr, p.len_cap, p.err);
                    L = __shfl_sync(0xffffffffu, Lr, 0);
                    nparts = (L + p.part_tokens - 1) / p.part_tokens;
                    cur = ncur;
                    nxt = nnxt;
                    have_tab = true;
                    have = true;
                    nstep = 0;
                }
            } else if (!static_done) {
                group = blockIdx.x;
                s = blockIdx.y;
                int Lr = __ldg(p.seq_lens + s);
                if (lane == 0)
                    Lr = clamp_len(Lr, p.len_cap, p.err);
                L = __shfl_sync(0xffffffffu, Lr, 0);
                nparts = 1;
                have = L > 0;
                static_done = 1;
                if (!have) {
                    // Empty sequence: its output rows are zero.
                    T *out = reinterpret_cast<T *>(p.out) +
                             ((size_t)s * p.num_heads + group * NV) * kD;
                    for (int i = lane; i < NV * kD; i += 32)
                        out[i] = Elem<T>::from(0.f);
                    if (p.lse && lane < NV)
                        p.lse[(size_t)s * p.num_heads + group * NV + lane] = -INFINITY;
                }
            }
            if (!have)
                break;
            const int kvh0 = group * HG;
            const int tok0 = SPLIT ? part * p.part_tokens : 0;
            const int tok1 = SPLIT ? min(L, tok0 + p.part_tokens) : L;
            const int jb0 = tok0 / BS;
            const int jend = (tok1 + BS - 1) / BS;
            const int nst = (tok1 - tok0 + TPS - 1) / TPS;
            const int32_t *bt = p.block_tables + (size_t)s * p.max_blocks;
            int cbase = jb0;
            if (!have_tab) {
                cur = (cbase + lane < jend) ? __ldg(bt + cbase + lane) : -1;
                nxt = (cbase + 32 + lane < jend) ? __ldg(bt + cbase + 32 + lane) : -1;
            }
            have_tab = false;
            const int qrow = s * p.num_heads + kvh0 * G;
            for (int st = 0; st < nst; ++st, ++gk) {
                const int slot = gk % kStages;
                if (gk >= kStages && !warp_wait(&m->empty[slot], ((gk / kStages) - 1) & 1, lane)) {
                    if (lane == 0)
                        atomicOr(p.err, PA_DEVERR_TIMEOUT_);
                    alive = false;
                    break;
                }
                const int t_lo = tok0 + st * TPS;
                const int nvalid = min(TPS, tok1 - t_lo);
                const int nch = (nvalid + R - 1) / R;
                if (t_lo / BS >= cbase + 32) {
                    cbase += 32;
                    cur = nxt;
                    nxt = (cbase + 32 + lane < jend) ? __ldg(bt + cbase + 32 + lane) : -1;
                }
                uint8_t *kv = smem + slot * kStageBytes;
                uint8_t *qb = smem + kOffQ + slot * kQBytes;
                if (lane == 0) {
                    StageDesc &d = m->desc[slot];
                    d.s = s;
                    d.group = group;
                    d.part = part;
                    d.nvalid = nvalid;
                    d.flags = (st == 0 ? kFlagFirst : 0) | (st == nst - 1 ? kFlagLast : 0);
                    d.nparts = nparts;
                    mbar_arrive_expect_tx(&m->full[slot],
                                          (uint32_t)(nch * 2 * BOX_BYTES + kParts * NV * 128));
#pragma unroll
                    for (int pp = 0; pp < kParts; ++pp)
                        tma_load_2d(qb + pp * kPartRows * 128, &q_map, &m->full[slot], 0,
                                    pp * q_rows + qrow);
                }
                __syncwarp();
                // One K/V box per lane: box i covers row chunk i/2 of plane
                // i&1, all 128 codes of the row, for all HG heads.
                const int c = lane >> 1;
                const int t = t_lo + (c < CH ? c : 0) * R;
                const int phys = __shfl_sync(0xffffffffu, cur, (t / BS - cbase) & 31);
                if (lane < nch * 2) {
                    const int plane = lane & 1;
                    int row;
                    if (phys < 0 || phys >= p.num_blocks) {
                        atomicOr(p.err, PA_DEVERR_BLOCK_ID_);
                        row = p.num_blocks * BS; // past the extent: zero fill
                    } else {
                        row = phys * BS + t % BS;
                    }
                    tma_load_4d_hint(kv + plane * kPlane + c * BOX_BYTES, &pool_map,
                                     &m->full[slot], 0, kvh0, row, plane, policy);
                }
                // Next item: claim it when three stages of this one are left
                // to issue (claiming earlier would unbalance the tail), then
                // its unit, then its length and table.
                if (SPLIT && nst - 1 - st <= 2 && nstep < 3 - (nst - 1 - st))
                    next_step();
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
    } else if (warp == kQkWarp || warp == kPvWarp) {
        // ==================================================== MMA issuers
        const bool qk = warp == kQkWarp;
        for (int k = 0;; ++k) {
            const int slot = k % kStages;
            const int b = k & 1;
            const int u = k >> 1;
            if (!warp_wait(&m->full[slot], (k / kStages) & 1, lane)) {
                if (lane == 0)
                    atomicOr(p.err, PA_DEVERR_TIMEOUT_);
                break;
            }
            int stop = 0;
            if (lane == 0)
                stop = m->desc[slot].flags & kFlagStop;
            if (__shfl_sync(0xffffffffu, stop, 0))
                break;
            bool ok = true;
            if (qk) {
                // S[b] is free once the softmax of stage k-2 is done.
                if (u > 0)
                    ok = warp_wait(&m->p_full[b], (u - 1) & 1, lane);
            } else {
                ok = warp_wait(&m->p_full[b], u & 1, lane);
                if (ok && u > 0)
                    ok = warp_wait(&m->o_free[b], (u - 1) & 1, lane);
            }
            if (!ok) {
                if (lane == 0)
                    atomicOr(p.err, PA_DEVERR_TIMEOUT_);
                break;
            }
            tc_fence_after_sync();
            if (lane == 0) {
                const uint32_t kvbase = smem_addr(smem + slot * kStageBytes);
                if (qk) {
                    const uint32_t qbase = smem_addr(smem + kOffQ + slot * kQBytes);
                    // Each 128-row block of the stage gets its own 48
                    // columns; K = 32 codes per instruction, four steps.
#pragma unroll
                    for (int ub = 0; ub < 2; ++ub) {
                        const uint32_t d_tmem = tmem + (uint32_t)(b * kSCols + ub * kNQ);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_f8(d_tmem, smem_desc_sw128(kvbase + ub * kRegion + kk * 32, 16, 1024),
                                    smem_desc_sw128(qbase + kk * 32, 16, 1024), kIdescQK,
                                    kk > 0 ? 1u : 0u);
                    }
                    umma_commit(&m->s_full[b]);
                } else {
                    const uint32_t vbase = kvbase + kPlane;
                    const uint32_t pbase = kvbase; // P over the stage's K (see the softmax)
                    const uint32_t d_tmem = tmem + (uint32_t)(kOCol + b * kNP);
                    // V^T as the MN-major A operand, 32 stage rows (4 KB) per
                    // step over all 256 rows; P's K runs over two regions.
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_f8(d_tmem, smem_desc_sw128(vbase + kk * 4096, kRegion, 1024),
                                smem_desc_sw128(pbase + (kk >> 2) * (kNP * 128) + (kk & 3) * 32,
                                                16, 1024),
                                kIdescPV, kk > 0 ? 1u : 0u);
                    umma_commit(&m->o_full[b]);
                    umma_commit(&m->empty[slot]);
                }
            }
            __syncwarp();
        }
        // Drain: every MMA this warp issued completes before TMEM is freed.
        const int wi = qk ? 0 : 1;
        if (lane == 0)
            umma_commit(&m->mma_done[wi]);
        warp_wait(&m->mma_done[wi], 0, lane);
    } else if (warp < 4) {
        // ======================================================== softmax/epilogue
        const int t = tid;                 // stage row (token t/HG, head t%HG); O row d = t
        const int h = t % HG;
        const uint32_t lane_base = (uint32_t)((warp * 32) << 16);
        float m_run[NV], o_acc[NV], alpha_prev[NV], l_part[G], qsn[NV];
#pragma unroll
        for (int n = 0; n < NV; ++n) {
            m_run[n] = -INFINITY;
            o_acc[n] = 0.f;
            alpha_prev[n] = 0.f;
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
            l_part[g] = 0.f;
        bool pending = false; // the previous stage's O is still to be accumulated
        // o = alpha*o + O_high + O_low for stage k, then free the O buffer.
        auto take_o = [&](int k, const float (&alpha)[NV]) -> bool {
            const int b = k & 1;
            const bool okw = mbar_wait(&m->o_full[b], (k >> 1) & 1);
            __syncwarp();
            tc_fence_after_sync();
            float o1[16], o2[16], o3[16];
            tmem_ld16(tmem + lane_base + (uint32_t)(kOCol + b * kNP), o1);
            tmem_ld16(tmem + lane_base + (uint32_t)(kOCol + b * kNP + kPartRows), o2);
            tmem_ld16(tmem + lane_base + (uint32_t)(kOCol + b * kNP + 2 * kPartRows), o3);
#pragma unroll
            for (int n = 0; n < NV; ++n)
                o_acc[n] = fmaf(o_acc[n], alpha[n], (o1[n] + o2[n] + o3[n]) * kInvPScale);
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
                // Scales of the item's query rows (the e4m3 parts of row n
                // carry q / q_scales[n]).
                const size_t head0 = (size_t)d.s * p.num_heads + (size_t)d.group * NV;
#pragma unroll
                for (int n = 0; n < NV; ++n) {
                    m_run[n] = -INFINITY;
                    o_acc[n] = 0.f;
                    qsn[n] = __ldg(q_scales + head0 + n) * p.qscale;
                }
#pragma unroll
                for (int g = 0; g < G; ++g)
                    l_part[g] = 0.f;
                pending = false;
            }
            ok = mbar_wait(&m->s_full[b], u & 1);
            __syncwarp();
            tc_fence_after_sync();
            // P of this stage goes over the stage's K: the scores MMA that
            // read K is complete (s_full), and the producer refills the slot
            // only after the values MMA has read P.  Each row writes only the
            // columns of its own head, so the region is cleared first; the
            // barrier after the row maxima orders the clearing before every
            // thread's writes.  Stages therefore never wait for the previous
            // stage's values MMA to release a shared P buffer.
            uint8_t *pb = smem + slot * kStageBytes;
#pragma unroll
            for (int i = 0; i < kPBytes / 16 / kEpiThreads; ++i)
                reinterpret_cast<uint4 *>(pb)[t + i * kEpiThreads] = make_uint4(0, 0, 0, 0);
            // This thread's two stage rows: t (block 0) and 128 + t (block 1),
            // both of head h.
            float x[2][G];
            bool valid[2];
#pragma unroll
            for (int ub = 0; ub < 2; ++ub) {
                float sv[16], sv2[16], sv3[16];
                const uint32_t sc = tmem + lane_base + (uint32_t)(b * kSCols + ub * kNQ);
                tmem_ld16(sc, sv);
                tmem_ld16(sc + kPartRows, sv2);
                tmem_ld16(sc + 2 * kPartRows, sv3);
                valid[ub] = ((ub * kRows + t) / HG) < d.nvalid;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float v = (sv[g] + sv2[g] + sv3[g]) * qsn[g];
#pragma unroll
                    for (int hh = 1; hh < HG; ++hh)
                        if (h == hh)
                            v = (sv[hh * G + g] + sv2[hh * G + g] + sv3[hh * G + g]) *
                                qsn[hh * G + g];
                    x[ub][g] = valid[ub] ? v : -INFINITY;
                }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                // max over this warp's tokens of the same head
                float mx = fmaxf(x[0][g], x[1][g]);
#pragma unroll
                for (int off = HG; off < 32; off <<= 1)
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                if (lane < HG)
                    m->red[b][warp][lane * G + g] = mx;
            }
            if (bar_sync_or(kBarEpi, kEpiThreads, !ok)) {
                if (t == 0)
                    atomicOr(p.err, PA_DEVERR_TIMEOUT_);
                break;
            }
            float alpha[NV];
#pragma unroll
            for (int n = 0; n < NV; ++n) {
                const float mst = fmaxf(fmaxf(m->red[b][0][n], m->red[b][1][n]),
                                        fmaxf(m->red[b][2][n], m->red[b][3][n]));
                const float m_new = fmaxf(m_run[n], mst);
                alpha[n] = ex2(m_run[n] - m_new);
                m_run[n] = m_new;
            }
            // P as the K-major B operand of the values MMA: column (k index)
            // = the stage row; row pp*16 + h*G + g holds part pp.
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float mg = m_run[g], ag = alpha[g];
#pragma unroll
                for (int hh = 1; hh < HG; ++hh)
                    if (h == hh) {
                        mg = m_run[hh * G + g];
                        ag = alpha[hh * G + g];
                    }
                const float pr0 = ex2(x[0][g] - mg);
                const float pr1 = ex2(x[1][g] - mg);
                l_part[g] = fmaf(l_part[g], ag, pr0 + pr1);
                // 256 p as three e4m3 parts (about 12 significant bits).
                const int n = h * G + g;
                uint8_t c3[2][3];
                split3_e4m3x2(pr0 * kPScale, pr1 * kPScale, c3[0], c3[1]);
#pragma unroll
                for (int ub = 0; ub < 2; ++ub)
#pragma unroll
                    for (int pp = 0; pp < kParts; ++pp)
                        pb[ub * (kNP * 128) + sw128_offset_b8(pp * kPartRows + n, t)] = c3[ub][pp];
            }
#pragma unroll
            for (int ub = 0; ub < 2; ++ub)
                if (!valid[ub]) {
                    // V rows past the end may hold anything (stale tiles, NaN
                    // padding); P is 0 there, but 0 * NaN would still poison O.
                    uint8_t *vrow = smem + slot * kStageBytes + kPlane + (ub * kRows + t) * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4 *>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
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
            for (int n = 0; n < NV; ++n)
                alpha_prev[n] = alpha[n];
            pending = true;

            if (!(d.flags & kFlagLast))
                continue;
            if (!take_o(k, alpha_prev) && t == 0)
                atomicOr(p.err, PA_DEVERR_TIMEOUT_);
            pending = false;
            // ---- end of the item: normaliser of each (head, query) column
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float v = l_part[g];
#pragma unroll
                for (int off = HG; off < 32; off <<= 1)
                    v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane < HG)
                    m->red2[warp][lane * G + g] = v;
            }
            bar_sync(kBarEpi, kEpiThreads);
            float l[NV];
#pragma unroll
            for (int n = 0; n < NV; ++n)
                l[n] = (m->red2[0][n] + m->red2[1][n]) + (m->red2[2][n] + m->red2[3][n]);
            const size_t head0 = (size_t)d.s * p.num_heads + (size_t)d.group * NV;
            if (!SPLIT || d.nparts == 1) {
                T *out = reinterpret_cast<T *>(p.out) + head0 * kD;
#pragma unroll
                for (int n = 0; n < NV; ++n)
                    out[n * kD + t] = Elem<T>::from(o_acc[n] * v_scale / l[n]);
                if (p.lse) {
#pragma unroll
                    for (int n = 0; n < NV; ++n)
                        if (t == n)
                            p.lse[head0 + n] = (m_run[n] + __log2f(l[n])) * 0.69314718055994531f;
                }
            } else {
                // Partial state of this partition; the reduce kernel that
                // follows merges the partitions of the sequence.
#pragma unroll
                for (int n = 0; n < NV; ++n) {
                    const size_t row = (head0 + n) * p.max_parts + d.part;
                    p.ws_o[row * kD + t] = o_acc[n] * v_scale;
                    if (t == n) {
                        p.ws_ml[row * 2] = m_run[n];
                        p.ws_ml[row * 2 + 1] = l[n];
                    }
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kQkWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <typename T, int BS, int G, int HG>
cudaError_t launch_one(const CUtensorMap &pool, const CUtensorMap &qmap, const TcParams &p,
                       const float *q_scales, int q_rows, float v_scale, dim3 grid,
                       cudaStream_t stream)
{
    auto kern = decode_tc_fp8_kernel<T, BS, G, HG, true>;
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
    // Follows the plan kernel as its dependent.
    return launch_after_previous(kern, grid, dim3(kThreads), kSmemBytes, stream, pool, qmap, p,
                                 q_scales, q_rows, v_scale);
}

// Split-K only (the query prepass needs the caller's workspace).
template <typename T>
cudaError_t launch(int block_size, int group, int hg, const CUtensorMap &pool,
                   const CUtensorMap &qmap, const TcParams &p, const float *q_scales,
                   int q_rows, float v_scale, dim3 grid, cudaStream_t stream)
{
#define PA_TC8_BS(Gv, HGv)                                                                    \
    (block_size == 16 ? launch_one<T, 16, Gv, HGv>(pool, qmap, p, q_scales, q_rows, v_scale, \
                                                   grid, stream)                              \
                      : (block_size == 32 ? launch_one<T, 32, Gv, HGv>(pool, qmap, p, q_scales, \
                                                                       q_rows, v_scale, grid, \
                                                                       stream)                \
                                          : cudaErrorNotSupported))
#define PA_TC8_CASE(Gv)                                                                       \
    case Gv:                                                                                  \
        return hg == 16 / Gv ? PA_TC8_BS(Gv, 16 / Gv)                                         \
                             : (hg == 1 ? PA_TC8_BS(Gv, 1) : cudaErrorNotSupported);
    switch (group) {
        PA_TC8_CASE(1)
        PA_TC8_CASE(2)
        PA_TC8_CASE(4)
        PA_TC8_CASE(8)
    default: return cudaErrorNotSupported;
    }
#undef PA_TC8_CASE
#undef PA_TC8_BS
}

template <typename T>
cudaError_t launch_quantize_q(const void *q, uint8_t *parts, float *scales, int rows,
                              cudaStream_t stream)
{
    return launch_after_previous(quantize_q_parts_kernel<T>, dim3((rows + 3) / 4), dim3(128), 0,
                                 stream, static_cast<const T *>(q), parts, scales, rows);
}

} // namespace tc8
} // namespace pa
