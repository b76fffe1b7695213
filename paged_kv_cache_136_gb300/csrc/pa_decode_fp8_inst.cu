// pa_decode_fp8_inst.cu -- instantiates the FP8-pool kernels for one query
// dtype, chosen by -DPA_INST_DTYPE (0 fp16, 1 bf16).
#include "pa_decode_fp8.cuh"
#include "pa_decode_tc_fp8.cuh"

#if !defined(PA_INST_DTYPE)
#error "compile with -DPA_INST_DTYPE=<0|1>"
#endif

namespace pa {
#if PA_INST_DTYPE == 0
using InstT = __half;
#define PA_F8_DECODE launch_decode_fp8_f16
#define PA_F8_RESHAPE launch_reshape_fp8_f16
#define PA_F8_TC launch_decode_tc_fp8_f16
#define PA_F8_QUANT launch_quantize_q_f16
#else
using InstT = __nv_bfloat16;
#define PA_F8_DECODE launch_decode_fp8_bf16
#define PA_F8_RESHAPE launch_reshape_fp8_bf16
#define PA_F8_TC launch_decode_tc_fp8_bf16
#define PA_F8_QUANT launch_quantize_q_bf16
#endif

cudaError_t PA_F8_DECODE(int block_size, int group, bool split, const CUtensorMap &tmap,
                         const DecodeParams &p, float v_scale, dim3 grid, cudaStream_t stream)
{
    return f8::launch<InstT>(block_size, group, split, tmap, p, v_scale, grid, stream);
}

cudaError_t PA_F8_RESHAPE(const void *key, const void *value, void *cache, const int64_t *slots,
                          int num_tokens, int row_elems, int64_t key_stride, int64_t value_stride,
                          int64_t plane_elems, int block_size, int64_t num_slots, float k_scale,
                          float v_scale, unsigned int *err, cudaStream_t stream)
{
    return f8::launch_reshape<InstT>(key, value, cache, slots, num_tokens, row_elems, key_stride,
                                     value_stride, plane_elems, block_size, num_slots, k_scale,
                                     v_scale, err, stream);
}
cudaError_t PA_F8_TC(int block_size, int group, int hg, const CUtensorMap &pool,
                     const CUtensorMap &qmap, const tc::TcParams &p, const float *q_scales,
                     int q_rows, float v_scale, dim3 grid, cudaStream_t stream)
{
    return tc8::launch<InstT>(block_size, group, hg, pool, qmap, p, q_scales, q_rows, v_scale,
                              grid, stream);
}

cudaError_t PA_F8_QUANT(const void *q, uint8_t *parts, float *scales, int rows,
                        cudaStream_t stream)
{
    return tc8::launch_quantize_q<InstT>(q, parts, scales, rows, stream);
}
} // namespace pa
