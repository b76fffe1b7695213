// pa_internal.h -- declarations shared by the library's translation units
// (kernel parameter blocks and the per-instantiation launchers).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

// Bits of the sticky device error word (the same values as PA_DEVERR_* in
// pa.h, which the kernels' translation units do not include).
#define PA_DEVERR_BLOCK_ID_ 0x1u
#define PA_DEVERR_SEQ_LEN_ 0x2u
#define PA_DEVERR_SLOT_ 0x4u
#define PA_DEVERR_TIMEOUT_ 0x8u

namespace pa {

// Launch `kern` so that it may start while the previous kernel on the stream
// is finishing (programmatic dependent launch); the kernel calls
// griddep_wait() before it reads anything that kernel wrote.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_after_previous(void (*kern)(KArgs...), dim3 grid, dim3 block,
                                         size_t smem, cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Kernel parameters of the decode kernels (one-pass and split-K partition).
struct DecodeParams {
    void *out;                   // [B, H, D] (one-pass)
    float *ws_o;                 // [B, H, max_parts, D] unnormalised partial outputs
    float *ws_ml;                // [B, H, max_parts, 2] running max (log2 units), normaliser
    const void *q;               // [B, H, D]
    const int32_t *block_tables; // [B, max_blocks]
    const int32_t *seq_lens;     // [B]
    unsigned int *err;           // sticky device error word
    int num_heads;
    int num_kv_heads;
    int num_blocks;
    int max_blocks;
    int part_tokens;             // split-K: tokens per partition
    int max_parts;               // split-K: partitions reserved per (seq, head)
    int len_cap;                 // largest seq_len the tables (and workspace) allow
    float qscale;                // scale * log2(e)
    float *lse;                  // [B, H] natural-log softmax denominators, or null
};

// Parameters of the split-K log-sum-exp reduce.
struct ReduceParams {
    void *out;
    const float *ws_o;
    const float *ws_ml;
    const int32_t *seq_lens;
    int num_heads;
    int max_parts;
    int part_tokens;
    int len_cap;
    int skip_single; // rows of one-partition sequences are already final
    float *lse;      // [B, H] natural-log softmax denominators, or null
    int out_f32;     // out holds float32 rows instead of the input dtype
};

// Key of a decode kernel instantiation.
struct DecodeKey {
    int dtype;      // 0 fp16, 1 bf16
    int head_size;  // 64, 128
    int block_size; // 16, 32
    int group;      // 1, 2, 4, 8
    bool split;
};

// Launch the decode kernel matching `key` on grid (Hkv, B, parts).  Returns
// cudaErrorNotSupported if no instantiation matches.
cudaError_t launch_decode(const DecodeKey &key, const CUtensorMap &tmap, const DecodeParams &p,
                          dim3 grid, cudaStream_t stream);

cudaError_t launch_decode_f16_d64(const DecodeKey &, const CUtensorMap &, const DecodeParams &,
                                  dim3, cudaStream_t);
cudaError_t launch_decode_f16_d128(const DecodeKey &, const CUtensorMap &, const DecodeParams &,
                                   dim3, cudaStream_t);
cudaError_t launch_decode_bf16_d64(const DecodeKey &, const CUtensorMap &, const DecodeParams &,
                                   dim3, cudaStream_t);
cudaError_t launch_decode_bf16_d128(const DecodeKey &, const CUtensorMap &, const DecodeParams &,
                                    dim3, cudaStream_t);

// Launch the split-K reduce on grid (H, B).
cudaError_t launch_reduce(int dtype, int head_size, const ReduceParams &p, int num_seqs,
                          cudaStream_t stream);

namespace tc {
struct TcParams;
}
// Tensor-core (tcgen05) decode kernels, head_size 128, `hg` kv heads per
// CTA.  One-pass: grid (Hkv/hg, B), one (head group, sequence) per CTA.
// Split: persistent 1-D grid fed by the work counter of the plan.
cudaError_t launch_decode_tc_f16(int block_size, int group, int hg, bool split,
                                 const CUtensorMap &pool, const CUtensorMap &qmap,
                                 const tc::TcParams &p, dim3 grid, cudaStream_t stream);
cudaError_t launch_decode_tc_bf16(int block_size, int group, int hg, bool split,
                                  const CUtensorMap &pool, const CUtensorMap &qmap,
                                  const tc::TcParams &p, dim3 grid, cudaStream_t stream);

// FP8 (e4m3) pool, head_size 128: decode on grid (Hkv, B[, parts]) and the
// cache write on grid (ceil(Hkv*128/8/256), T).
cudaError_t launch_decode_fp8_f16(int block_size, int group, bool split, const CUtensorMap &tmap,
                                  const DecodeParams &p, float v_scale, dim3 grid,
                                  cudaStream_t stream);
cudaError_t launch_decode_fp8_bf16(int block_size, int group, bool split, const CUtensorMap &tmap,
                                   const DecodeParams &p, float v_scale, dim3 grid,
                                   cudaStream_t stream);
cudaError_t launch_reshape_fp8_f16(const void *key, const void *value, void *cache,
                                   const int64_t *slots, int num_tokens, int row_elems,
                                   int64_t key_stride, int64_t value_stride, int64_t plane_elems,
                                   int block_size, int64_t num_slots, float k_scale,
                                   float v_scale, unsigned int *err, cudaStream_t stream);
cudaError_t launch_reshape_fp8_bf16(const void *key, const void *value, void *cache,
                                    const int64_t *slots, int num_tokens, int row_elems,
                                    int64_t key_stride, int64_t value_stride,
                                    int64_t plane_elems, int block_size, int64_t num_slots,
                                    float k_scale, float v_scale, unsigned int *err,
                                    cudaStream_t stream);

// FP8 pool on the tensor cores (split-K, persistent grid fed by the plan):
// the query prepass writes three e4m3 parts [3][rows][128] and row scales.
cudaError_t launch_decode_tc_fp8_f16(int block_size, int group, int hg, const CUtensorMap &pool,
                                     const CUtensorMap &qmap, const tc::TcParams &p,
                                     const float *q_scales, int q_rows, float v_scale, dim3 grid,
                                     cudaStream_t stream);
cudaError_t launch_decode_tc_fp8_bf16(int block_size, int group, int hg,
                                      const CUtensorMap &pool, const CUtensorMap &qmap,
                                      const tc::TcParams &p, const float *q_scales, int q_rows,
                                      float v_scale, dim3 grid, cudaStream_t stream);
cudaError_t launch_quantize_q_f16(const void *q, uint8_t *parts, float *scales, int rows,
                                  cudaStream_t stream);
cudaError_t launch_quantize_q_bf16(const void *q, uint8_t *parts, float *scales, int rows,
                                   cudaStream_t stream);

// Parameters of the tensor-core prefill kernel.
struct PrefillParams {
    void *out;                      // [num_tokens, H, D]
    float *lse;                     // [num_tokens, H] natural log, or null
    const int32_t *block_tables;    // row r at block_tables + r * bt_stride
    const int32_t *seq_lens;        // [R]
    const int32_t *query_start_loc; // [R + 1]
    unsigned int *err;
    long long bt_stride;
    int num_tokens, num_heads, num_kv_heads, num_blocks, max_blocks, max_query_len;
    int causal;
    float qscale;                   // scale * log2(e)
    // Key split (non-causal only): CTA chunk c attends keys
    // [c*chunk_tiles*128, (c+1)*chunk_tiles*128) and writes part c of out
    // and lse, part_stride / lse_part_stride elements apart.  key_split 1:
    // every key, out and lse as given.
    int key_split, chunk_tiles;
    long long part_stride, lse_part_stride;
    // Head pairs: grid.y = H/2 and a CTA's two tiles are query heads 2j and
    // 2j+1 (same kv head) over the same 128 rows.
    int head_pairs;
    int out_f32;                    // out holds float32 rows instead of the input dtype
    // >= 0: one request of num_tokens query rows over fixed_len keys, and
    // query_start_loc / seq_lens are not read.
    int fixed_len;
};

// The calling thread's current driver context (cuCtxGetCurrent, reached
// through the runtime's driver entry point), or nullptr if there is none or
// the driver does not export the call.  Caches of device objects key on it so
// that a new context on a device (after cudaDeviceReset, or a caller that
// switched driver contexts) gets new objects.
void *current_driver_context();

// Prefill over the paged cache on grid (ceil(max_query_len/128) x key_split, H, R).
cudaError_t launch_prefill_f16(int head_size, int block_size, const CUtensorMap &pool,
                               const CUtensorMap &qmap, const PrefillParams &p, dim3 grid,
                               cudaStream_t stream);
cudaError_t launch_prefill_bf16(int head_size, int block_size, const CUtensorMap &pool,
                                const CUtensorMap &qmap, const PrefillParams &p, dim3 grid,
                                cudaStream_t stream);

} // namespace pa
