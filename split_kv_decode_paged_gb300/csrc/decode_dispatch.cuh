// decode_dispatch.cuh -- explicit instantiation helper for one K/V storage kind.
#pragma once
#include "decode_kernel.cuh"

namespace fd {

template <int KV, bool QBF16>
cudaError_t launch_decode_kind(const fd_problem &p, const KernelShape &ks, const DecodeParams &dp,
                               const CUtensorMap &tmk, const CUtensorMap &tmv, int grid, size_t smem,
                               cudaStream_t stream) {
    if (ks.consumer_warps != 4) return cudaErrorInvalidValue;
    if (p.D == 128) {
        if (ks.nt == 1) return launch_decode_t<KV, 128, 1, 4, QBF16>(dp, tmk, tmv, grid, smem, stream);
        return launch_decode_t<KV, 128, 2, 4, QBF16>(dp, tmk, tmv, grid, smem, stream);
    }
    if (p.D == 64) {
        if (ks.nt == 1) return launch_decode_t<KV, 64, 1, 4, QBF16>(dp, tmk, tmv, grid, smem, stream);
        return launch_decode_t<KV, 64, 2, 4, QBF16>(dp, tmk, tmv, grid, smem, stream);
    }
    return cudaErrorInvalidValue;
}

template <int KV, bool QBF16>
size_t decode_smem_kind(const fd_problem &p, const KernelShape &ks, int stages) {
    if (p.D == 128)
        return ks.nt == 1 ? decode_smem_for<KV, 128, 1, 4, QBF16>(stages, p.B)
                          : decode_smem_for<KV, 128, 2, 4, QBF16>(stages, p.B);
    return ks.nt == 1 ? decode_smem_for<KV, 64, 1, 4, QBF16>(stages, p.B)
                      : decode_smem_for<KV, 64, 2, 4, QBF16>(stages, p.B);
}

}  // namespace fd
