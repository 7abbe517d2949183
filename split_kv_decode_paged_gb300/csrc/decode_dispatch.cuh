// decode_dispatch.cuh -- explicit instantiation helper for one K/V storage kind.
#pragma once
#include "decode_kernel.cuh"

namespace fd {

// (consumer warps, sub-tiles per warp) pairs built for each storage kind:
// 16-bit K/V: (4,1) = 64-token stages, (8,1) = 128-token stages;
// E4M3 K/V:   (4,1) = 64-token stages, (8,1) = 128-token stages, (8,2) = 256-token stages,
//             (4,2) = 128-token stages for two CTAs per SM.
template <int KV, int D, int NT, bool QBF16>
cudaError_t launch_decode_d(const KernelShape &ks, const DecodeParams &dp, const CUtensorMap &tmk,
                            const CUtensorMap &tmv, int grid, size_t smem, cudaStream_t stream) {
    if (dp.qn > 1) {
        // several causal query tokens per KV row: the 128-token, 8-warp shape only
        if (ks.consumer_warps == 8 && ks.subtiles == 1)
            return launch_decode_t<KV, D, NT, 8, 1, QBF16, true>(dp, tmk, tmv, grid, smem, stream);
        return cudaErrorInvalidValue;
    }
    if (ks.consumer_warps == 4 && ks.subtiles == 1)
        return launch_decode_t<KV, D, NT, 4, 1, QBF16>(dp, tmk, tmv, grid, smem, stream);
    if constexpr (KV == KV_E4M3) {
        if (ks.consumer_warps == 8 && ks.subtiles == 1)
            return launch_decode_t<KV, D, NT, 8, 1, QBF16>(dp, tmk, tmv, grid, smem, stream);
        if (ks.consumer_warps == 8 && ks.subtiles == 2)
            return launch_decode_t<KV, D, NT, 8, 2, QBF16>(dp, tmk, tmv, grid, smem, stream);
        if (ks.consumer_warps == 4 && ks.subtiles == 2) {
            if constexpr (NT == 1) {
                if (dp.scr_in_stage)
                    return launch_decode_t<KV, D, NT, 4, 2, QBF16, false, true>(dp, tmk, tmv, grid, smem, stream);
            }
            return launch_decode_t<KV, D, NT, 4, 2, QBF16>(dp, tmk, tmv, grid, smem, stream);
        }
    } else {
        if (ks.consumer_warps == 8 && ks.subtiles == 1)
            return launch_decode_t<KV, D, NT, 8, 1, QBF16>(dp, tmk, tmv, grid, smem, stream);
    }
    return cudaErrorInvalidValue;
}

template <int KV, int D, int NT, bool QBF16>
cudaError_t occupancy_d(const KernelShape &ks, size_t smem, int *blocks) {
    if (ks.consumer_warps == 4 && ks.subtiles == 1) return occupancy_t<KV, D, NT, 4, 1, QBF16>(smem, blocks);
    if constexpr (KV == KV_E4M3) {
        if (ks.consumer_warps == 8 && ks.subtiles == 2) return occupancy_t<KV, D, NT, 8, 2, QBF16>(smem, blocks);
        if (ks.consumer_warps == 4 && ks.subtiles == 2) return occupancy_t<KV, D, NT, 4, 2, QBF16>(smem, blocks);
    }
    if (ks.consumer_warps == 8 && ks.subtiles == 1) return occupancy_t<KV, D, NT, 8, 1, QBF16>(smem, blocks);
    return cudaErrorInvalidValue;
}

template <int KV, bool QBF16>
cudaError_t occupancy_kind(const fd_problem &p, const KernelShape &ks, size_t smem, int *blocks) {
    if (p.D == 128)
        return ks.nt == 1 ? occupancy_d<KV, 128, 1, QBF16>(ks, smem, blocks) : occupancy_d<KV, 128, 2, QBF16>(ks, smem, blocks);
    if (p.D == 64)
        return ks.nt == 1 ? occupancy_d<KV, 64, 1, QBF16>(ks, smem, blocks) : occupancy_d<KV, 64, 2, QBF16>(ks, smem, blocks);
    return cudaErrorInvalidValue;
}

template <int KV, int D, int NT, bool QBF16>
size_t decode_smem_d(const KernelShape &ks, int stages, int B, bool in_stage) {
    if (ks.consumer_warps == 4 && ks.subtiles == 1) return decode_smem_for<KV, D, NT, 4, 1, QBF16>(stages, B, in_stage);
    if (ks.consumer_warps == 8 && ks.subtiles == 2) return decode_smem_for<KV, D, NT, 8, 2, QBF16>(stages, B, in_stage);
    if (ks.consumer_warps == 4 && ks.subtiles == 2) return decode_smem_for<KV, D, NT, 4, 2, QBF16>(stages, B, in_stage);
    return decode_smem_for<KV, D, NT, 8, 1, QBF16>(stages, B, in_stage);
}

template <int KV, bool QBF16>
cudaError_t launch_decode_kind(const fd_problem &p, const KernelShape &ks, const DecodeParams &dp,
                               const CUtensorMap &tmk, const CUtensorMap &tmv, int grid, size_t smem,
                               cudaStream_t stream) {
    if (p.D == 128) {
        if (ks.nt == 1) return launch_decode_d<KV, 128, 1, QBF16>(ks, dp, tmk, tmv, grid, smem, stream);
        return launch_decode_d<KV, 128, 2, QBF16>(ks, dp, tmk, tmv, grid, smem, stream);
    }
    if (p.D == 64) {
        if (ks.nt == 1) return launch_decode_d<KV, 64, 1, QBF16>(ks, dp, tmk, tmv, grid, smem, stream);
        return launch_decode_d<KV, 64, 2, QBF16>(ks, dp, tmk, tmv, grid, smem, stream);
    }
    return cudaErrorInvalidValue;
}

template <int KV, bool QBF16>
size_t decode_smem_kind(const fd_problem &p, const KernelShape &ks, int stages, bool in_stage) {
    if (p.D == 128)
        return ks.nt == 1 ? decode_smem_d<KV, 128, 1, QBF16>(ks, stages, p.B, in_stage)
                          : decode_smem_d<KV, 128, 2, QBF16>(ks, stages, p.B, in_stage);
    return ks.nt == 1 ? decode_smem_d<KV, 64, 1, QBF16>(ks, stages, p.B, in_stage)
                      : decode_smem_d<KV, 64, 2, QBF16>(ks, stages, p.B, in_stage);
}

}  // namespace fd
