// pa_decode_inst.cu -- instantiates the decode kernels for one (dtype,
// head_size) pair, chosen by -DPA_INST_DTYPE (0 fp16, 1 bf16) and
// -DPA_INST_D (64, 128).  The build compiles this file once per pair so the
// four units compile in parallel.
#include "pa_decode.cuh"
#if PA_INST_D == 128
#include "pa_decode_tc.cuh"
#endif

#if !defined(PA_INST_DTYPE) || !defined(PA_INST_D)
#error "compile with -DPA_INST_DTYPE=<0|1> -DPA_INST_D=<64|128>"
#endif

#if PA_INST_DTYPE == 0
using InstT = __half;
#define PA_DT_NAME f16
#else
using InstT = __nv_bfloat16;
#define PA_DT_NAME bf16
#endif

#define PA_CAT3(a, b, c) a##b##c
#define PA_CAT(a, b, c) PA_CAT3(a, b, c)
#define PA_LAUNCHER PA_CAT(launch_decode_, PA_DT_NAME, PA_CAT(_d, PA_INST_D, ))

namespace pa {
cudaError_t PA_LAUNCHER(const DecodeKey &key, const CUtensorMap &tmap, const DecodeParams &p,
                        dim3 grid, cudaStream_t stream)
{
    return launch_by_group<InstT, PA_INST_D>(key, tmap, p, grid, stream);
}

#if PA_INST_D == 128
#define PA_TC_LAUNCHER PA_CAT(launch_decode_tc_, PA_DT_NAME, )
cudaError_t PA_TC_LAUNCHER(int block_size, int group, int hg, bool split,
                           const CUtensorMap &pool, const CUtensorMap &qmap,
                           const tc::TcParams &p, dim3 grid, cudaStream_t stream)
{
    return tc::launch_tc<InstT>(block_size, group, hg, split, pool, qmap, p, grid, stream);
}
#endif
} // namespace pa
