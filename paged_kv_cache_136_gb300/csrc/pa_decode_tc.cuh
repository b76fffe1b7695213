// pa_decode_tc.cuh -- paged decode attention on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory), head_size 128.
//
// A CTA works on HG kv heads at once (HG = 16/G when num_kv_heads allows).  A
// pipeline stage holds 128 rows ordered (token, kv head) -- TPS = 128/HG
// tokens of all HG heads -- which is the order the NHD pool
// [2, num_blocks, block_size, num_kv_heads, head_size] stores them in, so one
// TMA box {64 elements, HG heads, R token rows} fetches all HG heads of R rows
// ("Paged attention", k4i.top, section "block table": physical_block =
// block_table[t // block_size]).  Roles in a CTA of 224 threads:
//
//   warp 4 (producer)   takes work items, keeps the item's block-table entries
//                       in lane registers, and TMA-loads per stage the query
//                       rows of the HG heads (Q, HG*G x 128) and the K and V
//                       row chunks, one box per lane.
//   warp 5 (scores)     owns 128 TMEM columns and issues
//                         S^T[128 rows x 16] = K[128 x 128] . Q^T
//                       (tcgen05.mma, M=128, N=16, K=16 per instruction); row
//                       (t, h) uses columns h*G .. h*G+G-1.
//   warp 6 (values)     issues O^T[128 d x 32] = V^T[128 x 128 rows] . P,
//                       contracting over all 128 rows of the stage; P holds
//                       row (t, h)'s probabilities only in the columns of head
//                       h (high parts in columns 0-15, low parts in 16-31), so
//                       the other heads' rows add exact zeros.
//   warps 0-3           one TMEM lane (stage row) each: scale and mask the
//   (softmax/epilogue)  scores, stage max per (head, query) over the tokens,
//                       online-softmax rescale ("Paged attention", section
//                       "对非连续 blocks 做 attention"), write P as a bf16/fp16
//                       high part plus low part (~16-bit accuracy), zero V rows
//                       past the sequence end, and as head_size row d
//                       accumulate o = alpha*o + O_high + O_low for every
//                       (head, query) column.  S and O are double-buffered, so
//                       the values of stage k run while stage k+1's softmax is
//                       computed.
//
// The K and V tiles are read by the tensor cores straight from the TMA
// layout: K as a K-major operand, V as an MN-major (transposed) operand, both
// with the 128-byte swizzle (shared-memory matrix descriptors).
//
// Split-K ("PagedAttention 在 vLLM 中的实现分析", section 7.3): items are
// (partition of P tokens, head group) pairs dealt dynamically, longest first,
// to a persistent grid through an atomic counter.  A sequence with one
// partition writes its output directly; otherwise each partition writes its
// unnormalised (o, m, l) to the workspace and the reduce kernel that follows
// merges them with the log-sum-exp rescale.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_decode.cuh"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace tc {

// Warp roles.
constexpr int kThreads = 224;
constexpr int kEpiThreads = 128;          // warps 0-3: softmax / epilogue
constexpr int kProducerWarp = 4;          // TMA
constexpr int kQkWarp = 5;                // scores MMA issuer, owns TMEM
constexpr int kPvWarp = 6;                // values MMA issuer

constexpr int kStages = 3;
constexpr int kRows = 128;                // (token, kv head) rows per stage
constexpr int kD = 128;                   // head_size
constexpr int kRegion = kRows * 128;      // one 64-element half of 128 rows
constexpr int kPlane = 2 * kRegion;       // K (or V) of a stage
constexpr int kStageBytes = 2 * kPlane;   // K + V
constexpr int kNQ = 16;                   // score columns: (head, query) pairs
constexpr int kNP = 32;                   // value columns: high parts, then low parts
constexpr int kQBytes = 2 * kNQ * 128;    // two 64-element halves x 16 rows
constexpr int kPBytes = 2 * kNP * 128;    // two 64-row halves of K x 32 rows
constexpr int kTmemCols = 128;            // S: 2 x 16 columns, O: 2 x 32 columns
constexpr int kBarEpi = 1;                // named barrier of the softmax warps

constexpr int kOffQ = kStages * kStageBytes;
constexpr int kOffP = kOffQ + kStages * kQBytes;
constexpr int kOffMisc = kOffP + 2 * kPBytes;

constexpr int kFlagFirst = 1, kFlagLast = 2, kFlagStop = 4;

struct StageDesc {
    int s, group, part, nvalid, flags, nparts, run, pad1;
};

// Stage descriptors rotate over twice the ring, each with its own barrier:
// the one of stage k is rewritten for stage k + 2 * kStages, once the scores
// MMA of stage k + kStages has freed that slot, by which time the softmax of
// stage k (its last reader) is long done.  The softmax waits on the
// descriptor's barrier, not on the slot's K barrier: K of stage k + kStages
// may land before the softmax of stage k starts, and a parity wait cannot
// tell the two phases apart.
constexpr int kDescs = 2 * kStages;

struct Misc {
    StageDesc desc[kDescs];
    int stop_v[kStages];   // the values warp's stop flag of a slot
    float red[2][4][kNQ];  // per-stage max, double-buffered by stage parity
    float red2[2][4][kNQ]; // normaliser sums at item end, double-buffered by item
    int bcast[4];
    uint32_t tmem_base;
    uint32_t pad;
    uint64_t desc_full[kDescs]; // the stage descriptor written
    uint64_t full_k[kStages];  // K and Q of the slot landed
    uint64_t full_v[kStages];  // V of the slot landed
    uint64_t empty[kStages];   // V of the slot free (its values MMA is done)
    uint64_t empty_k[kStages]; // K and Q of the slot free (its scores MMA is done)
    uint64_t s_full[2], p_full[2], o_full[2], o_free[2];
    uint64_t mma_done[2];
};

constexpr int kSmemBytes = 1024 + kOffMisc + (int)sizeof(Misc);

struct TcParams {
    void *out;                   // [B, H, 128]
    const int32_t *block_tables; // [B, max_blocks]
    const int32_t *seq_lens;     // [B]
    unsigned int *err;
    // split-K workspace (null in one-pass mode)
    uint32_t *hdr;               // [0] work counter, [1] total items
    const uint32_t *units;       // (s << 16) | partition, or with runs
                                 // (s << 16) | ((run - 1) << 12) | partition
    float *ws_o;                 // [B, H, max_parts, 128]
    float *ws_ml;                // [B, H, max_parts, 2]
    int num_heads, num_kv_heads, num_groups, num_blocks, max_blocks;
    int part_tokens, max_parts, len_cap;
    float qscale;
    float *lse;                  // [B, H] natural-log softmax denominators, or null
    int out_f32;                 // out holds float32 rows instead of T
    int runs;                    // units carry a run length (see the plan kernel)
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

// Byte offset of element (row n, column k) of a K-major operand with 128-byte
// swizzle, stored as 64-column regions of `rows` rows each.
__device__ __forceinline__ int sw128_offset(int n, int k, int rows)
{
    return (k >> 6) * rows * 128 + (n >> 3) * 1024 + (n & 7) * 128 +
           ((((k & 63) >> 3) ^ (n & 7)) << 4) + (k & 7) * 2;
}

// HG kv heads per CTA; a stage holds TPS = 128/HG tokens of all HG heads,
// rows ordered (token, head) exactly as the NHD pool stores them, so one TMA
// box covers all HG heads of R consecutive token rows.
template <typename T, int BS, int G, int HG, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap pool_map,
                     const __grid_constant__ CUtensorMap q_map, const TcParams p)
{
    constexpr int NV = HG * G;                 // valid (head, query) columns
    constexpr int TPS = kRows / HG;            // tokens per stage
    constexpr int R = BS < TPS ? BS : TPS;     // token rows per TMA box
    constexpr int CH = TPS / R;                // row chunks per stage
    constexpr int BOX_BYTES = R * HG * 128;
    static_assert(G >= 1 && NV <= kNQ && (HG & (HG - 1)) == 0, "heads per CTA");
    static_assert(TPS % R == 0 && BS % R == 0 && CH * 4 <= 32, "stage geometry");
    constexpr uint32_t kFmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    constexpr uint32_t kIdescQK = idesc_f16_f32(kFmt, 0, 0, 128, kNQ);
    constexpr uint32_t kIdescPV = idesc_f16_f32(kFmt, 1, 0, 128, kNP);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc *m = reinterpret_cast<Misc *>(smem + kOffMisc);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // P entries of other heads' columns stay zero for the whole kernel: a
    // row (token, head h) only ever writes the columns of head h.
    for (int i = tid; i < 2 * kPBytes / 16; i += kThreads)
        reinterpret_cast<uint4 *>(smem + kOffP)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&m->full_k[i], 1);
            mbar_init(&m->full_v[i], 1);
        }
        for (int i = 0; i < kDescs; ++i) {
            mbar_init(&m->desc_full[i], 1);
            mbar_init(&m->empty[i], 1);
            mbar_init(&m->empty_k[i], 1);
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
        int nL_raw = 0, ncur = -1, nnxt = -1, n_s = 0, n_group = 0, n_part = 0, n_run = 1;
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
                n_part = p.runs ? (int)(nu & 0xFFFu) : (int)(nu & 0xFFFFu);
                n_run = p.runs ? (int)((nu >> 12) & 0xFu) + 1 : 1;
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
            int s = 0, group = 0, part = 0, L = 0, nparts = 1, run = 1;
            bool have = false;
            if (SPLIT) {
                while (nstep < 3)
                    next_step();
                if (n_have) {
                    s = n_s;
                    group = n_group;
                    part = n_part;
                    run = n_run;
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
                    const size_t out0 = ((size_t)s * p.num_heads + group * NV) * kD;
                    for (int i = lane; i < NV * kD; i += 32)
                        put_out<T>(p.out, out0 + i, 0.f, p.out_f32);
                    if (p.lse && lane < NV)
                        p.lse[(size_t)s * p.num_heads + group * NV + lane] = -INFINITY;
                }
            }
            if (!have)
                break;
            const int kvh0 = group * HG;
            const int tok0 = SPLIT ? part * p.part_tokens : 0;
            const int tok1 = SPLIT ? min(L, tok0 + run * p.part_tokens) : L;
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
                const uint32_t ph = ((gk / kStages) - 1) & 1;
                // K and Q of the slot are released by the scores MMA, V only by
                // the values MMA after the softmax: K and Q of this stage are
                // loaded as soon as the first is done, so more of the ring is
                // in flight while the softmax runs.
                if (gk >= kStages && !warp_wait(&m->empty_k[slot], ph, lane)) {
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
                // K and Q (with the stage's descriptor) and V land on
                // separate barriers: the scores MMA and the softmax of a stage
                // need not wait for its V, whose slot frees only when the
                // values MMA of the stage kStages back is done.
                if (lane == 0) {
                    StageDesc &d = m->desc[gk % kDescs];
                    d.s = s;
                    d.group = group;
                    d.part = part;
                    d.nvalid = nvalid;
                    d.flags = (st == 0 ? kFlagFirst : 0) | (st == nst - 1 ? kFlagLast : 0);
                    d.nparts = nparts;
                    d.run = run;
                    mbar_arrive(&m->desc_full[gk % kDescs]);
                    mbar_arrive_expect_tx(&m->full_k[slot], (uint32_t)(nch * 2 * BOX_BYTES + 2 * NV * 128));
                    tma_load_2d(qb, &q_map, &m->full_k[slot], 0, qrow);
                    tma_load_2d(qb + kNQ * 128, &q_map, &m->full_k[slot], 64, qrow);
                }
                __syncwarp();
                // One K/V box per lane: box i covers row chunk i/4 of plane
                // (i/2)&1, 64-element half i&1, for all HG heads.
                const int c = lane >> 2;
                const int t = t_lo + (c < CH ? c : 0) * R;
                const int phys = __shfl_sync(0xffffffffu, cur, (t / BS - cbase) & 31);
                const int plane = (lane >> 1) & 1;
                int row = 0;
                if (lane < nch * 4) {
                    if (phys < 0 || phys >= p.num_blocks) {
                        if (plane == 0)
                            atomicOr(p.err, PA_DEVERR_BLOCK_ID_);
                        row = p.num_blocks * BS; // past the extent: zero fill
                    } else {
                        row = phys * BS + t % BS;
                    }
                }
                if (lane < nch * 4 && plane == 0)
                    tma_load_4d_hint(kv + (lane & 1) * kRegion + c * BOX_BYTES, &pool_map,
                                     &m->full_k[slot], (lane & 1) * 64, kvh0, row, 0, policy);
                if (gk >= kStages && !warp_wait(&m->empty[slot], ph, lane)) {
                    // Let the K and Q copies already issued land before leaving;
                    // the values warp sees a stop at this slot (the others time
                    // out at the next stage).
                    if (lane == 0) {
                        atomicOr(p.err, PA_DEVERR_TIMEOUT_);
                        m->stop_v[slot] = 1;
                        mbar_arrive(&m->full_v[slot]);
                    }
                    warp_wait(&m->full_k[slot], (gk / kStages) & 1, lane);
                    alive = false;
                    break;
                }
                if (lane == 0) {
                    m->stop_v[slot] = 0;
                    mbar_arrive_expect_tx(&m->full_v[slot], (uint32_t)(nch * 2 * BOX_BYTES));
                }
                __syncwarp();
                if (lane < nch * 4 && plane == 1)
                    tma_load_4d_hint(kv + kPlane + (lane & 1) * kRegion + c * BOX_BYTES, &pool_map,
                                     &m->full_v[slot], (lane & 1) * 64, kvh0, row, 1, policy);
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
                // The values MMA of stage gk - kStages is done, so its scores
                // MMA is too: both halves of the slot are free.
                if (lane == 0) {
                    m->desc[gk % kDescs].flags = kFlagStop;
                    m->stop_v[slot] = 1;
                    mbar_arrive(&m->desc_full[gk % kDescs]);
                    mbar_arrive(&m->full_k[slot]);
                    mbar_arrive(&m->full_v[slot]);
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
            if (!warp_wait(qk ? &m->full_k[slot] : &m->full_v[slot], (k / kStages) & 1, lane)) {
                if (lane == 0)
                    atomicOr(p.err, PA_DEVERR_TIMEOUT_);
                break;
            }
            int stop = 0;
            if (lane == 0)
                stop = qk ? (m->desc[k % kDescs].flags & kFlagStop) : m->stop_v[slot];
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
                    const uint32_t d_tmem = tmem + (uint32_t)(b * kNQ);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t koff = (uint32_t)((kk >> 2) * kRegion + (kk & 3) * 32);
                        const uint32_t qoff = (uint32_t)((kk >> 2) * kNQ * 128 + (kk & 3) * 32);
                        umma_f16(d_tmem, smem_desc_sw128(kvbase + koff, 16, 1024),
                                 smem_desc_sw128(qbase + qoff, 16, 1024), kIdescQK,
                                 kk > 0 ? 1u : 0u);
                    }
                    umma_commit(&m->s_full[b]);
                    umma_commit(&m->empty_k[slot]);
                } else {
                    const uint32_t vbase = kvbase + kPlane;
                    const uint32_t pbase = smem_addr(smem + kOffP + b * kPBytes);
                    const uint32_t d_tmem = tmem + (uint32_t)(2 * kNQ + b * kNP);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t poff = (uint32_t)((kk >> 2) * kNP * 128 + (kk & 3) * 32);
                        umma_f16(d_tmem, smem_desc_sw128(vbase + kk * 2048, kRegion, 1024),
                                 smem_desc_sw128(pbase + poff, 16, 1024), kIdescPV,
                                 kk > 0 ? 1u : 0u);
                    }
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
        float m_run[NV], o_acc[NV], alpha_prev[NV], l_part[G];
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
        // An item whose last stage's values were still on the tensor cores
        // when its softmax ended: it is normalised and written once that O is
        // folded in, after the next stage's softmax, so the wait for the
        // values MMA overlaps work instead of stalling the ring at every item
        // change.  Its column sums of l wait in red2[fin_par].
        bool fin = false;
        int fin_s = 0, fin_group = 0, fin_part = 0, fin_nparts = 1, fin_par = 0, fin_run = 1;
        float fin_m = 0.f; // running max of column t (t < NV) of that item
        int par = 0;
        // o = alpha*o + O_high + O_low for stage k, then free the O buffer.
        auto take_o = [&](int k, const float (&alpha)[NV]) -> bool {
            const int b = k & 1;
            const bool okw = mbar_wait(&m->o_full[b], (k >> 1) & 1);
            __syncwarp();
            tc_fence_after_sync();
            float lo16[16], hi16[16];
            tmem_ld16(tmem + lane_base + (uint32_t)(2 * kNQ + b * kNP), hi16);
            tmem_ld16(tmem + lane_base + (uint32_t)(2 * kNQ + b * kNP + 16), lo16);
#pragma unroll
            for (int n = 0; n < NV; ++n)
                o_acc[n] = fmaf(o_acc[n], alpha[n], hi16[n] + lo16[n]);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&m->o_free[b]);
            return okw;
        };
        // Normalise and store the finished item (o_acc holds its sums), then
        // clear the accumulator for the item under way.
        auto finish = [&]() {
            float l[NV];
#pragma unroll
            for (int n = 0; n < NV; ++n)
                l[n] = (m->red2[fin_par][0][n] + m->red2[fin_par][1][n]) +
                       (m->red2[fin_par][2][n] + m->red2[fin_par][3][n]);
            const size_t head0 = (size_t)fin_s * p.num_heads + (size_t)fin_group * NV;
            if (!SPLIT || fin_nparts == 1) {
#pragma unroll
                for (int n = 0; n < NV; ++n)
                    put_out<T>(p.out, (head0 + n) * kD + t, o_acc[n] / l[n], p.out_f32);
                if (p.lse) {
#pragma unroll
                    for (int n = 0; n < NV; ++n)
                        if (t == n)
                            p.lse[head0 + n] = (fin_m + __log2f(l[n])) * 0.69314718055994531f;
                }
            } else {
                // Partial state of this partition; the reduce kernel that
                // follows merges the partitions of the sequence.
#pragma unroll
                for (int n = 0; n < NV; ++n) {
                    const size_t row = (head0 + n) * p.max_parts + fin_part;
                    p.ws_o[row * kD + t] = o_acc[n];
                    if (t == n) {
                        p.ws_ml[row * 2] = fin_m;
                        p.ws_ml[row * 2 + 1] = l[n];
                    }
                }
                // A run covered the next fin_run - 1 partitions too: they
                // carry no weight (the reduce skips them).
                if (fin_run > 1 && t < NV) {
                    const size_t row = (head0 + t) * p.max_parts + fin_part;
                    for (int q = 1; q < fin_run; ++q) {
                        p.ws_ml[(row + q) * 2] = -INFINITY;
                        p.ws_ml[(row + q) * 2 + 1] = 0.f;
                    }
                }
            }
#pragma unroll
            for (int n = 0; n < NV; ++n)
                o_acc[n] = 0.f;
            fin = false;
        };
        for (int k = 0;; ++k) {
            const int slot = k % kStages;
            const int b = k & 1;
            const int u = k >> 1;
            bool ok = mbar_wait(&m->desc_full[k % kDescs], (k / kDescs) & 1);
            const StageDesc d = m->desc[k % kDescs];
            if (bar_sync_or(kBarEpi, kEpiThreads, !ok)) {
                if (t == 0)
                    atomicOr(p.err, PA_DEVERR_TIMEOUT_);
                break;
            }
            if (d.flags & kFlagStop) {
                // No more work: the last item's final values are still out.
                if (fin) {
                    if (!take_o(k - 1, alpha_prev) && t == 0)
                        atomicOr(p.err, PA_DEVERR_TIMEOUT_);
                    finish();
                }
                break;
            }
            if (d.flags & kFlagFirst) {
                // o_acc is cleared by finish() of the item before.
#pragma unroll
                for (int n = 0; n < NV; ++n)
                    m_run[n] = -INFINITY;
#pragma unroll
                for (int g = 0; g < G; ++g)
                    l_part[g] = 0.f;
            }
            ok = mbar_wait(&m->s_full[b], u & 1);
            __syncwarp();
            tc_fence_after_sync();
            float sv[16];
            tmem_ld16(tmem + lane_base + (uint32_t)(b * kNQ), sv);
            const bool valid = (t / HG) < d.nvalid;
            float x[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float v = sv[g];
#pragma unroll
                for (int hh = 1; hh < HG; ++hh)
                    if (h == hh)
                        v = sv[hh * G + g];
                x[g] = valid ? v * p.qscale : -INFINITY;
                // max over this warp's tokens of the same head
                float mx = x[g];
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
            // = this row t; row h*G+g holds the high part, 16+h*G+g the low.
            uint8_t *pb = smem + kOffP + b * kPBytes;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float mg = m_run[g], ag = alpha[g];
#pragma unroll
                for (int hh = 1; hh < HG; ++hh)
                    if (h == hh) {
                        mg = m_run[hh * G + g];
                        ag = alpha[hh * G + g];
                    }
                const float pr = ex2(x[g] - mg);
                l_part[g] = fmaf(l_part[g], ag, pr);
                uint16_t hi, lo;
                Bits<T>::split(pr, hi, lo);
                const int n = h * G + g;
                *reinterpret_cast<uint16_t *>(pb + sw128_offset(n, t, kNP)) = hi;
                *reinterpret_cast<uint16_t *>(pb + sw128_offset(kNQ + n, t, kNP)) = lo;
            }
            if (!valid) {
                // V rows past the end may hold anything (stale tiles, NaN
                // padding); P is 0 there, but 0 * NaN would still poison O.
                // They are zeroed once V has landed.
                if (!mbar_wait(&m->full_v[slot], (k / kStages) & 1))
                    atomicOr(p.err, PA_DEVERR_TIMEOUT_);
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
            // stage's softmax was computed; fold them in now.  If that stage
            // ended an item, the item is complete: store it.
            if (pending && !take_o(k - 1, alpha_prev) && t == 0)
                atomicOr(p.err, PA_DEVERR_TIMEOUT_);
            if (fin)
                finish();
#pragma unroll
            for (int n = 0; n < NV; ++n)
                alpha_prev[n] = alpha[n];
            pending = true;

            if (!(d.flags & kFlagLast))
                continue;
            // ---- last stage of the item: its normaliser sums go to red2[par]
            // and column t's running max to fin_m; the values of this stage
            // are folded in (and the item stored) after the next stage's
            // softmax.
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float v = l_part[g];
#pragma unroll
                for (int off = HG; off < 32; off <<= 1)
                    v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane < HG)
                    m->red2[par][warp][lane * G + g] = v;
            }
#pragma unroll
            for (int n = 0; n < NV; ++n)
                if (t == n)
                    fin_m = m_run[n];
            fin = true;
            fin_s = d.s;
            fin_group = d.group;
            fin_part = d.part;
            fin_run = d.run;
            fin_nparts = d.nparts;
            fin_par = par;
            par ^= 1;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kQkWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Split-K plan (one CTA): zero the work counter, write zero rows for empty
// sequences, and list the work units of every sequence longest first, so the
// dynamically claimed work ends with the shortest items:
//   1. runs: max_run consecutive full partitions of one sequence, taken by
//      one CTA as one item (fewer item changes, one partial state per run);
//   2. single full partitions: a sequence's last keep_single full
//      partitions (and those left over from its runs), in sequence order;
//   3. each sequence's last, possibly partial, partition, in descending size
//      (a counting sort over kPlanBuckets size buckets).
// max_run == 1 lists every full partition singly.  A unit is (s << 16) |
// partition, or with runs (s << 16) | ((run - 1) << 12) | partition (the
// host enables runs only with fewer than 4096 partitions per sequence).  The
// item count (units x head groups) goes to hdr[1].
constexpr int kPlanBuckets = 256;
constexpr int kRunShift = 12; // run length field of a unit, when runs are on

template <typename T>
__global__ void __launch_bounds__(1024) splitk_plan_kernel(const int32_t *seq_lens, int B, int H,
                                                           int num_groups, int part_tokens,
                                                           int len_cap, uint32_t *hdr,
                                                           uint32_t *units,
                                                           T *out, float *lse,
                                                           unsigned int *err, int out_f32,
                                                           int max_run, int keep_single)
{
    __shared__ unsigned long long warp_tot[32];
    __shared__ uint32_t bucket[kPlanBuckets];
    __shared__ unsigned long long carry_s;
    __shared__ uint32_t total_runs_s;
    // Launched as the dependent of the kernel before it (the cache write):
    // wait for its results, let the decode grid start its prologue.
    griddep_wait();
    griddep_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int R = max_run > 1 ? max_run : 1;
    for (int i = tid; i < kPlanBuckets; i += blockDim.x)
        bucket[i] = 0;
    if (tid == 0) {
        hdr[0] = 0;
        carry_s = 0;
        total_runs_s = 0;
    }
    __syncthreads();
    auto seq_len = [&](int s, bool flag) {
        int L = seq_lens[s];
        if (L < 0 || L > len_cap) {
            if (flag)
                atomicOr(err, PA_DEVERR_SEQ_LEN_);
            L = L < 0 ? 0 : len_cap;
        }
        return L;
    };
    // Runs and single full partitions of a sequence of L tokens.
    auto split_full = [&](int L, uint32_t &nruns, uint32_t &nsingle) {
        const int n = (L + part_tokens - 1) / part_tokens;
        const int nfull = n > 0 ? n - 1 : 0;
        const int in_runs = (R > 1 && nfull > keep_single) ? nfull - keep_single : 0;
        nruns = (uint32_t)(in_runs / R);
        nsingle = (uint32_t)(nfull - (int)nruns * R);
    };
    // Size bucket of a last partition of `last` tokens: larger first.
    auto size_bucket = [&](int last) {
        const int b = (int)(((long long)(last - 1) * kPlanBuckets) / part_tokens);
        return kPlanBuckets - 1 - (b < kPlanBuckets - 1 ? b : kPlanBuckets - 1);
    };
    // Pass 0: how many run units come before the single partitions.
    if (R > 1) {
        uint32_t mine = 0;
        for (int s = tid; s < B; s += blockDim.x) {
            uint32_t nr, ns;
            split_full(seq_len(s, false), nr, ns);
            mine += nr;
        }
        if (mine)
            atomicAdd(&total_runs_s, mine);
        __syncthreads();
    }
    const uint32_t total_runs = total_runs_s;
    // Pass 1: runs and single full partitions in sequence order (two
    // prefix sums packed in one 64-bit scan: runs high, singles low);
    // histogram of the last partitions.
    for (int c0 = 0; c0 < B; c0 += blockDim.x) {
        const int s = c0 + tid;
        uint32_t nr = 0, ns = 0;
        int L = 0;
        if (s < B) {
            L = seq_len(s, true);
            const int n = (L + part_tokens - 1) / part_tokens;
            if (n > 0) {
                split_full(L, nr, ns);
                atomicAdd(&bucket[size_bucket(L - (n - 1) * part_tokens)], 1u);
            } else {
                for (int i = 0; i < H * 128; ++i)
                    put_out<T>(out, (size_t)s * H * 128 + i, 0.f, out_f32);
                if (lse)
                    for (int h = 0; h < H; ++h)
                        lse[(size_t)s * H + h] = -INFINITY;
            }
        }
        const unsigned long long mine = ((unsigned long long)nr << 32) | ns;
        unsigned long long v = mine;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off)
                v += y;
        }
        if (lane == 31)
            warp_tot[warp] = v;
        __syncthreads();
        if (warp == 0) {
            unsigned long long w = lane < nwarps ? warp_tot[lane] : 0ull;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off)
                    w += y;
            }
            warp_tot[lane] = w; // inclusive prefix over warps
        }
        __syncthreads();
        const unsigned long long base = carry_s + (warp ? warp_tot[warp - 1] : 0ull) + v - mine;
        const uint32_t rbase = (uint32_t)(base >> 32);
        const uint32_t sbase = total_runs + (uint32_t)(base & 0xFFFFFFFFull);
        for (uint32_t q = 0; q < nr; ++q)
            units[rbase + q] = ((uint32_t)s << 16) | ((uint32_t)(R - 1) << kRunShift) |
                               (q * (uint32_t)R);
        for (uint32_t q = 0; q < ns; ++q)
            units[sbase + q] = ((uint32_t)s << 16) | (nr * (uint32_t)R + q);
        __syncthreads();
        if (tid == 0)
            carry_s += warp_tot[nwarps - 1];
        __syncthreads();
    }
    // Bucket start offsets after the runs and single partitions (buckets in
    // size order): an exclusive scan of the counts over the first
    // kPlanBuckets threads, one bucket each (the kernel is launched with
    // 1024 threads).
    static_assert(kPlanBuckets % 32 == 0 && kPlanBuckets <= 1024, "one bucket per thread");
    const uint32_t first_last = total_runs + (uint32_t)(carry_s & 0xFFFFFFFFull);
    __shared__ uint32_t warp_tot32[32];
    uint32_t bc = 0, bi = 0; // this thread's bucket count, inclusive scan in its warp
    if (tid < kPlanBuckets) {
        bc = bucket[tid];
        bi = bc;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, bi, off);
            if (lane >= off)
                bi += y;
        }
        if (lane == 31)
            warp_tot32[warp] = bi;
    }
    __syncthreads();
    if (tid < kPlanBuckets) {
        uint32_t before = first_last;
        for (int w = 0; w < warp; ++w)
            before += warp_tot32[w];
        bucket[tid] = before + bi - bc;
        if (tid == kPlanBuckets - 1)
            hdr[1] = (before + bi) * (uint32_t)num_groups;
    }
    __syncthreads();
    // Pass 2: place each last partition in its bucket.
    for (int s = tid; s < B; s += blockDim.x) {
        const int L = seq_len(s, false);
        const int n = (L + part_tokens - 1) / part_tokens;
        if (n > 0) {
            const uint32_t pos = atomicAdd(&bucket[size_bucket(L - (n - 1) * part_tokens)], 1u);
            units[pos] = ((uint32_t)s << 16) | (uint32_t)(n - 1);
        }
    }
}

template <typename T, int BS, int G, int HG, bool SPLIT>
cudaError_t launch_tc_one(const CUtensorMap &pool, const CUtensorMap &qmap, const TcParams &p,
                          dim3 grid, cudaStream_t stream)
{
    auto kern = decode_tc_kernel<T, BS, G, HG, SPLIT>;
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
    // The split kernel follows the plan kernel as its dependent.
    if (SPLIT)
        return launch_after_previous(kern, grid, dim3(kThreads), kSmemBytes, stream, pool, qmap, p);
    kern<<<grid, kThreads, kSmemBytes, stream>>>(pool, qmap, p);
    return cudaGetLastError();
}

template <typename T, int G, int HG>
cudaError_t launch_tc_bs(int block_size, bool split, const CUtensorMap &pool,
                         const CUtensorMap &qmap, const TcParams &p, dim3 grid,
                         cudaStream_t stream)
{
    if (block_size == 16)
        return split ? launch_tc_one<T, 16, G, HG, true>(pool, qmap, p, grid, stream)
                     : launch_tc_one<T, 16, G, HG, false>(pool, qmap, p, grid, stream);
    if (block_size == 32)
        return split ? launch_tc_one<T, 32, G, HG, true>(pool, qmap, p, grid, stream)
                     : launch_tc_one<T, 32, G, HG, false>(pool, qmap, p, grid, stream);
    return cudaErrorNotSupported;
}

// Kv heads per CTA for group size G: 16/G when num_kv_heads allows it, else 1.
__host__ __device__ constexpr int heads_per_cta(int group, int num_kv_heads)
{
    return (num_kv_heads % (16 / group) == 0) ? 16 / group : 1;
}

template <typename T>
cudaError_t launch_tc(int block_size, int group, int hg, bool split, const CUtensorMap &pool,
                      const CUtensorMap &qmap, const TcParams &p, dim3 grid, cudaStream_t stream)
{
#define PA_TC_CASE(Gv)                                                                        \
    case Gv:                                                                                  \
        return hg == 16 / Gv ? launch_tc_bs<T, Gv, 16 / Gv>(block_size, split, pool, qmap, p, \
                                                             grid, stream)                    \
                             : (hg == 1 ? launch_tc_bs<T, Gv, 1>(block_size, split, pool,      \
                                                                 qmap, p, grid, stream)       \
                                        : cudaErrorNotSupported);
    switch (group) {
        PA_TC_CASE(1)
        PA_TC_CASE(2)
        PA_TC_CASE(4)
        PA_TC_CASE(8)
    default: return cudaErrorNotSupported;
    }
#undef PA_TC_CASE
}

} // namespace tc
} // namespace pa
