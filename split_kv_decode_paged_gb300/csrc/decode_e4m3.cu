// decode_e4m3.cu -- split-KV decode kernels for e4m3 K/V pools.
#include "decode_dispatch.cuh"

namespace fd {

cudaError_t launch_decode_e4m3(const fd_problem &p, const KernelShape &ks, const DecodeParams &dp,
                             const CUtensorMap &tmk, const CUtensorMap &tmv, int grid, size_t smem,
                             cudaStream_t stream) {
    if (p.q_dtype == FD_BF16) return launch_decode_kind<KV_E4M3, true>(p, ks, dp, tmk, tmv, grid, smem, stream);
    return launch_decode_kind<KV_E4M3, false>(p, ks, dp, tmk, tmv, grid, smem, stream);
}

cudaError_t decode_occupancy_e4m3(const fd_problem &p, const KernelShape &ks, size_t smem, int *blocks) {
    if (p.q_dtype == FD_BF16) return occupancy_kind<KV_E4M3, true>(p, ks, smem, blocks);
    return occupancy_kind<KV_E4M3, false>(p, ks, smem, blocks);
}

size_t decode_smem_e4m3(const fd_problem &p, const KernelShape &ks, int stages, bool in_stage) {
    return decode_smem_kind<KV_E4M3, false>(p, ks, stages, in_stage);
}

}  // namespace fd
