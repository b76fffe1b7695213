// pa_prefill_tc.cuh -- prefill and chunked prefill over the paged KV cache on
// the 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// What it computes ("PagedAttention 在 vLLM 中的实现分析", section 6.2: the
// batch's new query tokens, packed by query_start_loc, attend the paged keys
// of their request with seqlen_k = seq_lens, through the block table, with
// causal masking; section 6.4: the shared-prefix pass is the same attention
// without the causal mask).  Query row i of request r sits at position
// seq_len - q_len + i and attends keys 0..position (causal) or every key.
//
// A CTA owns 256 query rows of one (request, query head): two tiles of 128
// rows that share every K/V tile, each with its own softmax warpgroup.  Roles
// in a CTA of 320 threads:
//
//   warp 8 (producer)  TMA-loads the two query tiles once, then K and V tiles
//                      of 128 keys into a ring of shared-memory slots, one
//                      box {64 elements, 1 kv head, block_size rows} per lane
//                      and block ("Paged attention", k4i.top, section "block
//                      table": physical_block = block_table[t // block_size]).
//   warp 9 (MMA)       owns the 512 TMEM columns and issues, for both tiles,
//                        S_t = Q_t K_k^T          (M=128, N=128, K=head_size)
//                        O_t (+)= P_t V_k         (M=128, N=head_size, K=128)
//                      with P_t read from tensor memory (A operand) and V_k as
//                      an MN-major shared-memory operand, in the order
//                        PV_0(k), QK_0(k+1), PV_1(k), QK_1(k+1), ...
//                      so tile 0's softmax of key tile k+1 runs while the
//                      tensor cores work on tile 1, and the other way round.
//   warps 0-3 / 4-7    one query row per thread (TMEM lane): scale and mask
//   (softmax, tile 0/1) the row's 128 scores, row max, base-2 exponentials,
//                      write P over S as a 16-bit high part (the buffer's
//                      first 64 columns) plus the rounded remainder (the
//                      next 64), so P keeps 16 or more significant bits, and
//                      at the end out = O / l (and the log-sum-exp when
//                      asked).
//
// Tensor memory: tile t's scores (then P) in columns t*128 .. t*128+127, O_t
// at 256 + t*128.  The scores of key tile k+1 go over P of key tile k, so a
// tile's chain is QK -> softmax -> PV -> QK; the two tiles' chains interleave
// on the tensor cores.  MMAs issued by one thread run in issue order and a
// commit tracks all of them, so when the scores of key tile k are committed
// the values MMA of tile k-1 is complete too, and the softmax may rescale O.
//
// The running maximum is updated lazily: O and l are rescaled only when a key
// tile raises a row's maximum by more than 2^8, so most tiles skip the rescale
// and P stays below 2^8 (exact in fp16/bf16 range).  Every key row past
// seq_len that a tile could hold is zeroed in shared memory before the values
// MMA reads it, so stale or NaN bytes never reach O.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace pf {

constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;         // the MMA issuer of both query tiles
constexpr int kTileM = 128;         // query rows per tile
constexpr int kRowsPerCta = 2 * kTileM;
constexpr int kTileN = 128;         // keys per K/V tile
constexpr float kRescaleLog2 = 8.f; // lazy-rescale threshold, log2 units
constexpr uint32_t kTmemCols = 512;
constexpr int kQRegion = kTileM * 128;  // 128 query rows x 64 elements x 2 bytes

template <int D>
struct Geo {
    static constexpr int kHalves = D / 64;
    static constexpr int kKVRegion = kTileN * 128;        // 128 key rows x 64 elements x 2 bytes
    static constexpr int kTileBytes = kHalves * kQRegion; // a Q tile
    static constexpr int kKVBytes = kHalves * kKVRegion;  // a K or V tile
    static constexpr int kSlots = kKVBytes >= 32768 ? 4 : 8; // K/V ring of 128 KB
    static constexpr int kOffKV = 2 * kTileBytes;         // after the two Q tiles
    static constexpr int kOffMisc = kOffKV + kSlots * kKVBytes;
};

struct Misc {
    uint64_t q_full;
    uint64_t kv_full[8], kv_empty[8];
    uint64_t s_full[2], p_full[2]; // per query tile
    uint64_t o_done[2];            // the tile's last values MMA done
    uint64_t drain;
    uint32_t tmem_base;
};

template <int D>
constexpr int smem_bytes()
{
    return 1024 + Geo<D>::kOffMisc + (int)sizeof(Misc);
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b)
{
    const __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// The two values of a packed pair, back to float.
template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t w);
template <>
__device__ __forceinline__ float2 unpack2<__half>(uint32_t w)
{
    return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}
template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Warp-uniform bounded wait driven by lane 0.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, int lane)
{
    bool ok = true;
    if (lane == 0)
        ok = mbar_wait(bar, parity);
    return __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
}

template <typename T, int D, int BS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap pool_map,
                      const __grid_constant__ CUtensorMap q_map, const PrefillParams p)
{
    using Gm = Geo<D>;
    constexpr int kKVRegion = Gm::kKVRegion;
    constexpr int NH = Gm::kHalves;
    constexpr int TB = Gm::kTileBytes;
    constexpr int KB = Gm::kKVBytes;
    constexpr int S = Gm::kSlots;
    constexpr int BPT = kTileN / BS; // pool blocks per key tile
    static_assert(32 % BPT == 0 && BPT * NH <= 32, "key tile geometry");
    constexpr uint32_t kFmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    // P travels as a high part plus the rounded remainder (two MMAs on the
    // same V): a 16-bit P alone (8 or 11 significant bits) puts the
    // relative error of a row whose keys' values cancel above 1e-2.
    constexpr uint32_t kIdescS = idesc_f16_f32(kFmt, 0, 0, kTileM, kTileN);
    constexpr uint32_t kIdescO = idesc_f16_f32(kFmt, 0, 1, kTileM, D);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc *m = reinterpret_cast<Misc *>(smem + Gm::kOffMisc);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // Launched as the dependent of the kernel before it (which may write the
    // request metadata, q or the pool): wait for it before reading anything.
    griddep_wait();
    // ---- this CTA's rows: request r, query head h, query rows i0 .. i0+255
    // Grid: x = query head (or head pair), y = request, z = query block
    // counted from the request's last one (times the key chunks).  CTAs start
    // in linear order, x fastest, so the last blocks of all requests -- under
    // the causal mask the ones that attend to the most keys -- start first and
    // the short first blocks fill the tail.
    const int r = blockIdx.y;
    // Head pairs (grouped-query heads 2j, 2j+1 share a kv head): tile t
    // takes the same 128 rows for head 2j+t.  Otherwise tile t takes rows
    // 128t.. of one head.
    const bool hp = p.head_pairs != 0;
    const int h = hp ? 2 * (int)blockIdx.x : (int)blockIdx.x;
    const int nsplit = p.key_split;
    const int csplit = (int)blockIdx.z % nsplit;
    const int rank = (int)blockIdx.z / nsplit;
    const int rows_cta = hp ? kTileM : kRowsPerCta;
    auto toff = [&](int t) { return hp ? 0 : t * kTileM; };  // tile t's first row
    auto thead = [&](int t) { return hp ? h + t : h; };       // tile t's query head
    const bool fixed = p.fixed_len >= 0;
    const int q0 = fixed ? 0 : __ldg(p.query_start_loc + r);
    const int q1 = fixed ? p.num_tokens : __ldg(p.query_start_loc + r + 1);
    const int L = fixed ? p.fixed_len : __ldg(p.seq_lens + r);
    const int q_len = q1 - q0;
    if (q0 < 0 || q1 > p.num_tokens || q_len < 0 || q_len > p.max_query_len || L < q_len ||
        L > p.max_blocks * BS) {
        if (tid == 0 && rank == 0 && csplit == 0 && h == 0)
            atomicOr(p.err, PA_DEVERR_SEQ_LEN_);
        return;
    }
    const int qb = (q_len + rows_cta - 1) / rows_cta - 1 - rank;
    if (qb < 0)
        return;
    const int i0 = qb * rows_cta;
    const int ctx = L - q_len;
    // Keys of this CTA: [kt0 * 128, key_hi) (the whole request unless split).
    const int kt0 = csplit * p.chunk_tiles;
    const int key_hi = nsplit > 1 ? min(L, (kt0 + p.chunk_tiles) * kTileN) : L;
    // Output rows in T, or float32 (out_f32: the cascade's parts).
    const size_t out_elem0 = (size_t)csplit * (size_t)p.part_stride;
    float *const lse_base = p.lse ? p.lse + (size_t)csplit * (size_t)p.lse_part_stride : nullptr;
    int nv[2], nt[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        nv[t] = min(max(q_len - (i0 + toff(t)), 0), kTileM);
        const int ext = p.causal ? min(L, ctx + i0 + toff(t) + nv[t]) : key_hi;
        nt[t] = nv[t] > 0 ? max(0, (ext - kt0 * kTileN + kTileN - 1) / kTileN) : 0;
    }
    const int n = max(nt[0], nt[1]); // key tiles loaded
    if (n == 0) {
        // An empty key chunk: zero rows and -inf log-sum-exps (an empty part).
        for (int t = 0; t < 2; ++t) {
            for (int i = tid; i < nv[t] * D; i += kThreads) {
                const size_t tok = (size_t)(q0 + i0 + toff(t) + i / D);
                const size_t e = out_elem0 + (tok * p.num_heads + thead(t)) * D + i % D;
                if (p.out_f32)
                    static_cast<float *>(p.out)[e] = 0.f;
                else
                    static_cast<T *>(p.out)[e] = T(0.f);
            }
            if (lse_base)
                for (int i = tid; i < nv[t]; i += kThreads)
                    lse_base[(size_t)(q0 + i0 + toff(t) + i) * p.num_heads + thead(t)] = -INFINITY;
        }
        return;
    }
    const bool tail = (kt0 + n) * kTileN > L; // the last key tile reaches past seq_len
    // The softmax warpgroup that zeroes the last key tile's V rows past
    // seq_len: tile 0 whenever it reads that tile (its values MMA comes
    // first), else tile 1.
    const int fixer = nt[0] == n ? 0 : 1;

    if (tid == 0) {
        mbar_init(&m->q_full, 1);
        for (int i = 0; i < S; ++i) {
            mbar_init(&m->kv_full[i], 1);
            mbar_init(&m->kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&m->s_full[i], 1);
            mbar_init(&m->p_full[i], 4);
            mbar_init(&m->o_done[i], 1);
        }
        mbar_init(&m->drain, 1);
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
    griddep_launch_dependents();

    if (warp == kProducerWarp) {
        // ================================================================ producer
        const int kvh = h / (p.num_heads / p.num_kv_heads);
        if (lane == 0) {
            prefetch_tensormap(&pool_map);
            prefetch_tensormap(&q_map);
            mbar_arrive_expect_tx(&m->q_full, (uint32_t)((nv[1] > 0 ? 2 : 1) * TB));
#pragma unroll
            for (int t = 0; t < 2; ++t)
                if (nv[t] > 0)
#pragma unroll
                    for (int hf = 0; hf < NH; ++hf)
                        tma_load_3d(smem + t * TB + hf * kQRegion, &q_map, &m->q_full, hf * 64,
                                    thead(t), q0 + i0 + toff(t));
        }
        // Block-table entries of 64 blocks live in lane registers (this
        // window and the next), refreshed every 32 blocks.
        const int nblk_req = (key_hi + BS - 1) / BS;
        const int32_t *bt = p.block_tables + (size_t)r * (size_t)p.bt_stride;
        int cb = (kt0 * BPT) & ~31;
        int cur = cb + lane < nblk_req ? __ldg(bt + cb + lane) : -1;
        int nxt = cb + 32 + lane < nblk_req ? __ldg(bt + cb + 32 + lane) : -1;
        for (int g = 0; g < 2 * n; ++g) {
            const int k = g >> 1, plane = g & 1, slot = g % S;
            if (g >= S && !warp_wait(&m->kv_empty[slot], ((g / S) - 1) & 1, lane)) {
                if (lane == 0)
                    atomicOr(p.err, PA_DEVERR_TIMEOUT_);
                break;
            }
            const int jt = (kt0 + k) * BPT;
            if (jt >= cb + 32) {
                cb += 32;
                cur = nxt;
                nxt = cb + 32 + lane < nblk_req ? __ldg(bt + cb + 32 + lane) : -1;
            }
            const int nblk = min(BPT, nblk_req - jt);
            if (lane == 0)
                mbar_arrive_expect_tx(&m->kv_full[slot], (uint32_t)(nblk * BS * D * 2));
            __syncwarp();
            const int c = lane / NH, hf = lane % NH;
            const int phys = __shfl_sync(0xffffffffu, cur, (jt + min(c, BPT - 1) - cb) & 31);
            if (lane < nblk * NH) {
                int row;
                if (phys < 0 || phys >= p.num_blocks) {
                    atomicOr(p.err, PA_DEVERR_BLOCK_ID_);
                    row = p.num_blocks * BS; // past the extent: zero fill
                } else {
                    row = phys * BS;
                }
                tma_load_4d(smem + Gm::kOffKV + slot * KB + hf * kKVRegion + c * BS * 128,
                            &pool_map, &m->kv_full[slot], hf * 64, kvh, row, plane);
            }
        }
    } else if (warp == kMmaWarp) {
        // ============================================ MMA issuer of both tiles
        // Shared-memory descriptors are formed once: a K/V slot's descriptor is
        // the ring's base descriptor plus the slot offset, and each 16-wide
        // step adds a constant, so issuing an MMA costs one 64-bit add
        // instead of a chain of address arithmetic.
        const uint64_t q_desc[2] = {smem_desc_sw128(smem_addr(smem), 16, 1024),
                                    smem_desc_sw128(smem_addr(smem + TB), 16, 1024)};
        const uint64_t k_desc0 = smem_desc_sw128(smem_addr(smem + Gm::kOffKV), 16, 1024);
        const uint64_t v_desc0 = smem_desc_sw128(smem_addr(smem + Gm::kOffKV), kKVRegion, 1024);
        auto slot_off = [](int slot) { return (uint64_t)((uint32_t)(slot * KB) >> 4); };
        // S_t = Q_t K^T into tile t's score buffer.
        auto issue_qk = [&](int t, int slot) {
            const uint64_t kd = k_desc0 + slot_off(slot);
            const uint64_t qd = q_desc[t];
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t qo = (uint64_t)(((kk >> 2) * kQRegion + (kk & 3) * 32) >> 4);
                const uint64_t ko = (uint64_t)(((kk >> 2) * kKVRegion + (kk & 3) * 32) >> 4);
                umma_f16(tmem + (uint32_t)(t * 128), qd + qo, kd + ko, kIdescS, kk > 0 ? 1u : 0u);
            }
            umma_commit(&m->s_full[t]);
        };
        // O_t (+)= P_t V with P (high parts, then low parts 64 columns on)
        // read from the score buffer it was written over.
        auto issue_pv = [&](int t, int slot, bool acc) {
            const uint64_t vd0 = v_desc0 + slot_off(slot);
            const uint32_t pa = tmem + (uint32_t)(t * 128);
            const uint32_t od = tmem + (uint32_t)(256 + t * 128);
#pragma unroll
            for (int kk = 0; kk < kTileN / 16; ++kk) {
                const uint64_t vd = vd0 + (uint64_t)((kk * 2048) >> 4);
                umma_f16_tmem_a(od, pa + (uint32_t)(kk * 8), vd, kIdescO, (acc || kk > 0) ? 1u : 0u);
                umma_f16_tmem_a(od, pa + (uint32_t)(kTileN / 2 + kk * 8), vd, kIdescO, 1u);
            }
        };
        bool ok = warp_wait(&m->q_full, 0, lane) && warp_wait(&m->kv_full[0], 0, lane);
        if (ok) {
            tc_fence_after_sync();
            if (lane == 0) {
#pragma unroll
                for (int t = 0; t < 2; ++t)
                    if (nt[t] > 0)
                        issue_qk(t, 0);
                umma_commit(&m->kv_empty[0]); // K of key tile 0 read by both
            }
            __syncwarp();
        }
        // Per key tile k: for each tile t that needs it, the values of k once
        // P_t(k) is written, then the scores of k+1 over that P (the MMAs run
        // in issue order).  V of k is released after both tiles' values
        // MMAs, K of k+1 after both tiles' scores MMAs.  Tile 0 goes first,
        // so tile 0's softmax of k+1 overlaps tile 1's MMAs and tile 1's
        // softmax overlaps tile 0's next values and scores.
        for (int k = 0; ok && k < n; ++k) {
            const int gv = 2 * k + 1, sv = gv % S;
            const int gk = 2 * k + 2, sk = gk % S;
            const bool next = k + 1 < n;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (!ok || k >= nt[t])
                    continue;
                // Before tile 0's MMAs: V of k, K of k+1 and P_0(k), each
                // awaited by its own lane at the same time; before tile 1's
                // (issued after tile 0's when both need k): P_1(k).
                bool w = true;
                if (t == 0 || k >= nt[0]) {
                    if (lane == 0)
                        w = mbar_wait(&m->kv_full[sv], (gv / S) & 1);
                    else if (lane == 1 && next)
                        w = mbar_wait(&m->kv_full[sk], (gk / S) & 1);
                    else if (lane == 2)
                        w = mbar_wait(&m->p_full[t], k & 1);
                } else if (lane == 2) {
                    w = mbar_wait(&m->p_full[t], k & 1);
                }
                ok = __all_sync(0xffffffffu, w);
                if (!ok)
                    break;
                tc_fence_after_sync();
                if (lane == 0) {
                    issue_pv(t, sv, k > 0);
                    if (k + 1 < nt[t])
                        issue_qk(t, sk);
                    else
                        umma_commit(&m->o_done[t]); // the tile's last values MMA
                }
                __syncwarp();
            }
            if (!ok)
                break;
            if (lane == 0) {
                umma_commit(&m->kv_empty[sv]);
                if (next)
                    umma_commit(&m->kv_empty[sk]);
            }
            __syncwarp();
        }
        if (!ok && lane == 0)
            atomicOr(p.err, PA_DEVERR_TIMEOUT_);
        // Drain: every MMA issued completes before TMEM is freed.
        if (lane == 0)
            umma_commit(&m->drain);
        warp_wait(&m->drain, 0, lane);
    } else {
        // =========================================== softmax / epilogue (tiles 0, 1)
        const int wg = warp >> 2;
        const int row = tid & 127;
        const uint32_t lane_base = (uint32_t)(((warp & 3) * 32) << 16);
        const uint32_t s_addr = tmem + lane_base + (uint32_t)(wg * 128);
        const uint32_t o_addr = tmem + lane_base + (uint32_t)(256 + wg * 128);
        const int ntt = nt[wg];
        if (ntt > 0) {
            const int pos = ctx + i0 + toff(wg) + row;
            const int lim = p.causal ? min(L, pos + 1) : key_hi;         // keys < lim
            const int lim_lo = p.causal ? min(L, ctx + i0 + toff(wg) + 1) : key_hi;
            const float qs = p.qscale;
            float m_used = -INFINITY, l = 0.f;
            bool ok = true;
            for (int k = 0; k < ntt; ++k) {
                const uint32_t sb = s_addr; // this tile's score buffer
                ok = warp_wait(&m->s_full[wg], k & 1, lane);
                if (!ok)
                    break;
                tc_fence_after_sync();
                // The row's kTileN raw scores (bits).
                uint32_t sv[kTileN];
#pragma unroll
                for (int c = 0; c < kTileN / 32; ++c)
                    tmem_ld32_nowait(sb + (uint32_t)(c * 32),
                                     *reinterpret_cast<uint32_t(*)[32]>(sv + c * 32));
                tmem_wait_ld();
                // Row max over the raw scores (scale > 0 commutes with max),
                // three-input maxima in 4 independent chains; masked keys
                // become -inf.
                if ((kt0 + k + 1) * kTileN > lim_lo) {
                    const int kl = lim - (kt0 + k) * kTileN; // keys of this tile below the limit
#pragma unroll
                    for (int i = 0; i < kTileN; ++i)
                        if (i >= kl)
                            sv[i] = __float_as_uint(-INFINITY);
                }
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int i = 0; i < kTileN / 2; ++i)
                    m4[i & 3] = fmax3(m4[i & 3], __uint_as_float(sv[2 * i]),
                                      __uint_as_float(sv[2 * i + 1]));
                const float mx = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * qs;
                float alpha = 1.f;
                bool need = false;
                if (k == 0) {
                    m_used = mx;
                } else if (mx > m_used + kRescaleLog2) {
                    alpha = ex2(m_used - mx);
                    m_used = mx;
                    l *= alpha;
                    need = true;
                }
                // p = 2^(S * scale*log2e - m): one packed FFMA per two keys and
                // one ex2 per key; the row sum in two packed chains.  P goes
                // over the scores it came from: high parts in the first
                // kTileN / 2 columns of the buffer, rounded remainders after.
                const float nmu = m_used == -INFINITY ? 0.f : -m_used;
                const float2 qs2 = make_float2(qs, qs), nmu2 = make_float2(nmu, nmu);
                float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < kTileN / 32; ++c) {
                    uint32_t pk[16], lo[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float2 z = __ffma2_rn(make_float2(__uint_as_float(sv[c * 32 + 2 * j]),
                                                                __uint_as_float(sv[c * 32 + 2 * j + 1])),
                                                    qs2, nmu2);
                        const float2 pp = make_float2(ex2(z.x), ex2(z.y));
                        l2[j & 1] = __fadd2_rn(l2[j & 1], pp);
                        pk[j] = pack2<T>(pp.x, pp.y);
                        const float2 hf = unpack2<T>(pk[j]);
                        lo[j] = pack2<T>(pp.x - hf.x, pp.y - hf.y);
                    }
                    tmem_st16(sb + (uint32_t)(c * 16), pk);
                    tmem_st16(sb + (uint32_t)(kTileN / 2 + c * 16), lo);
                }
                l += (l2[0].x + l2[1].x) + (l2[0].y + l2[1].y);
                if (__any_sync(0xffffffffu, need)) {
                    // O holds the values of key tiles 0..k-1: the scores of k
                    // were committed after that values MMA was issued.  Done
                    // after P is written so the scores' registers are free.
                    tc_fence_after_sync();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32_nowait(o_addr + (uint32_t)(c * 32), v);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
                        tmem_st32(o_addr + (uint32_t)(c * 32), v);
                    }
                }
                tmem_wait_st();
                if (tail && wg == fixer && k == n - 1) {
                    // Zero the V rows of keys >= seq_len in the last tile (one
                    // thread per key row).
                    const int gv = 2 * k + 1;
                    if (!warp_wait(&m->kv_full[gv % S], (gv / S) & 1, lane))
                        ok = false;
                    if (ok && row < kTileN && (kt0 + k) * kTileN + row >= L) {
                        uint8_t *vrow = smem + Gm::kOffKV + (gv % S) * KB + row * 128;
#pragma unroll
                        for (int hf = 0; hf < NH; ++hf)
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                *reinterpret_cast<uint4 *>(vrow + hf * kKVRegion + c * 16) =
                                    make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&m->p_full[wg]);
                if (!ok)
                    break;
            }
            if (ok)
                ok = warp_wait(&m->o_done[wg], 0, lane);
            if (!ok) {
                if (lane == 0)
                    atomicOr(p.err, PA_DEVERR_TIMEOUT_);
            } else {
                tc_fence_after_sync();
                const bool valid = row < nv[wg];
                const size_t tok = (size_t)(q0 + i0 + toff(wg) + row);
                const int hw = thead(wg);
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const size_t o_elem = out_elem0 + (tok * p.num_heads + hw) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32_nowait(o_addr + (uint32_t)(c * 32), v);
                    tmem_wait_ld();
                    if (p.out_f32) {
                        if (valid) {
                            float4 *dst =
                                reinterpret_cast<float4 *>(static_cast<float *>(p.out) + o_elem + c * 32);
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                dst[j] = make_float4(__uint_as_float(v[4 * j]) * inv,
                                                     __uint_as_float(v[4 * j + 1]) * inv,
                                                     __uint_as_float(v[4 * j + 2]) * inv,
                                                     __uint_as_float(v[4 * j + 3]) * inv);
                        }
                        continue;
                    }
                    uint32_t w[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        w[j] = pack2<T>(__uint_as_float(v[2 * j]) * inv,
                                        __uint_as_float(v[2 * j + 1]) * inv);
                    if (valid) {
                        uint4 *dst =
                            reinterpret_cast<uint4 *>(static_cast<T *>(p.out) + o_elem + c * 32);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                    }
                }
                if (lse_base && valid)
                    lse_base[tok * p.num_heads + hw] =
                        l > 0.f ? (m_used + __log2f(l)) * 0.69314718055994531f : -INFINITY;
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

template <typename T, int D, int BS>
cudaError_t launch_one(const CUtensorMap &pool, const CUtensorMap &qmap, const PrefillParams &p,
                       dim3 grid, cudaStream_t stream)
{
    auto kern = prefill_tc_kernel<T, D, BS>;
    constexpr int kSmem = smem_bytes<D>();
    static unsigned long long done_mask = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess)
            return e;
        __atomic_fetch_or(&done_mask, bit, __ATOMIC_ACQ_REL);
    }
    return launch_after_previous(kern, grid, dim3(kThreads), (size_t)kSmem, stream, pool, qmap, p);
}

template <typename T>
cudaError_t launch(int head_size, int block_size, const CUtensorMap &pool, const CUtensorMap &qmap,
                   const PrefillParams &p, dim3 grid, cudaStream_t stream)
{
    if (head_size == 128 && block_size == 16)
        return launch_one<T, 128, 16>(pool, qmap, p, grid, stream);
    if (head_size == 128 && block_size == 32)
        return launch_one<T, 128, 32>(pool, qmap, p, grid, stream);
    if (head_size == 64 && block_size == 16)
        return launch_one<T, 64, 16>(pool, qmap, p, grid, stream);
    if (head_size == 64 && block_size == 32)
        return launch_one<T, 64, 32>(pool, qmap, p, grid, stream);
    return cudaErrorNotSupported;
}

} // namespace pf
} // namespace pa
