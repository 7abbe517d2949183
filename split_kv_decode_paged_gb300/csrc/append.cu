// append.cu -- write one new token's K and V per sequence into the paged pools
// ("Inference Cookbook" §3.2-3.3: the new k, v are written into the cache and
// the cached lengths are not advanced by the call; §4.2 page addressing).
// Token position L = seq_lens[b] goes to page block_table[b][L / page_size],
// slot L % page_size.  FP8 (E4M3) pools: code = rne_satfinite(x / scale) with
// the page's fp32 scale and an IEEE fp32 division.
// One warp per (b, kvh, K-or-V) row; lanes stride over D.
#include "fd_internal.h"
#include "ptx.cuh"

namespace fd {

constexpr int kAppendWarps = 4;

__device__ __forceinline__ float load_16bit_as_float(const void *base, size_t idx, bool bf16) {
    const uint16_t bits = reinterpret_cast<const uint16_t *>(base)[idx];
    if (bf16) return __uint_as_float(static_cast<uint32_t>(bits) << 16);
    return __half2float(__ushort_as_half(bits));
}

__global__ void __launch_bounds__(kAppendWarps * 32) fd_append_kv_kernel(const AppendParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long job = (long long)blockIdx.x * kAppendWarps + warp;  // (b, kvh, which)
    if (job >= 2LL * p.B * p.Hkv) return;
    const int which = (int)(job & 1);
    const int bk = (int)(job >> 1);
    const int b = bk / p.Hkv, kvh = bk - (bk / p.Hkv) * p.Hkv;
    const int L = p.seq_lens[b];
    const int col = L >= 0 ? L / p.page_size : -1;
    int page = -1;
    if (col >= 0 && col < p.max_blocks) page = p.block_table[(size_t)b * p.max_blocks + col];
    if (page < 0 || page >= p.num_pages) {
        if (lane == 0 && which == 0 && kvh == 0 && p.status) atomicOr(p.status, FD_DEV_BAD_PAGE);
        return;
    }
    const int slot = L - col * p.page_size;
    const size_t src = ((size_t)b * p.Hkv + kvh) * p.D;
    const size_t dst = (((size_t)page * p.page_size + slot) * p.Hkv + kvh) * p.D;
    const void *in = which ? p.v_new : p.k_new;
    void *pool = which ? p.v_pages : p.k_pages;
    if (p.kv_kind != KV_E4M3) {
        const uint16_t *s16 = reinterpret_cast<const uint16_t *>(in) + src;
        uint16_t *d16 = reinterpret_cast<uint16_t *>(pool) + dst;
        for (int d = lane; d < p.D; d += 32) d16[d] = s16[d];
        return;
    }
    const float sc = (which ? p.v_scale : p.k_scale)[(size_t)page * p.Hkv + kvh];
    uint8_t *d8 = reinterpret_cast<uint8_t *>(pool) + dst;
    for (int d = 2 * lane; d < p.D; d += 64) {
        const float x0 = load_16bit_as_float(in, src + d, p.new_is_bf16);
        const float x1 = load_16bit_as_float(in, src + d + 1, p.new_is_bf16);
        const uint16_t codes = f32x2_to_e4m3x2(__fdiv_rn(x1, sc), __fdiv_rn(x0, sc));
        *reinterpret_cast<uint16_t *>(d8 + d) = codes;
    }
}

cudaError_t launch_append(const AppendParams &ap, cudaStream_t stream) {
    const long long jobs = 2LL * ap.B * ap.Hkv;
    if (jobs == 0) return cudaSuccess;
    const long long blocks = (jobs + kAppendWarps - 1) / kAppendWarps;
    fd_append_kv_kernel<<<(unsigned)blocks, kAppendWarps * 32, 0, stream>>>(ap);
    return cudaGetLastError();
}

}  // namespace fd
