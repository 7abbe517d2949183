// decode_f16.cu -- split-KV decode kernels for f16 K/V pools.
#include "decode_dispatch.cuh"

namespace fd {

cudaError_t launch_decode_f16(const fd_problem &p, const KernelShape &ks, const DecodeParams &dp,
                             const CUtensorMap &tmk, const CUtensorMap &tmv, int grid, size_t smem,
                             cudaStream_t stream) {
    return launch_decode_kind<KV_F16, false>(p, ks, dp, tmk, tmv, grid, smem, stream);
}

cudaError_t decode_occupancy_f16(const fd_problem &p, const KernelShape &ks, size_t smem, int *blocks) {
    return occupancy_kind<KV_F16, false>(p, ks, smem, blocks);
}

size_t decode_smem_f16(const fd_problem &p, const KernelShape &ks, int stages, bool in_stage) {
    return decode_smem_kind<KV_F16, false>(p, ks, stages, in_stage);
}

}  // namespace fd
