// pa_prefill_inst.cu -- instantiates the tensor-core prefill kernels for one
// dtype, chosen by -DPA_INST_DTYPE (0 fp16, 1 bf16), so the two units compile
// in parallel.
#include "pa_prefill_tc.cuh"

#if !defined(PA_INST_DTYPE)
#error "compile with -DPA_INST_DTYPE=<0|1>"
#endif

namespace pa {
#if PA_INST_DTYPE == 0
cudaError_t launch_prefill_f16(int head_size, int block_size, const CUtensorMap &pool,
                               const CUtensorMap &qmap, const PrefillParams &p, dim3 grid,
                               cudaStream_t stream)
{
    return pf::launch<__half>(head_size, block_size, pool, qmap, p, grid, stream);
}
#else
cudaError_t launch_prefill_bf16(int head_size, int block_size, const CUtensorMap &pool,
                                const CUtensorMap &qmap, const PrefillParams &p, dim3 grid,
                                cudaStream_t stream)
{
    return pf::launch<__nv_bfloat16>(head_size, block_size, pool, qmap, p, grid, stream);
}
#endif
} // namespace pa
