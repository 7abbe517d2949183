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

// Rotary embedding of element d of a row x (fp32 values) at position pos:
// pairs (i, i + rotary_dim/2) or (2i, 2i+1) of the first rotary_dim elements,
// y1 = (x1*cos) - (x2*sin), y2 = (x2*cos) + (x1*sin), every product and sum
// rounded to fp32 (no fused multiply-add); other elements pass through.
template <typename LoadFn>
__device__ __forceinline__ float rotate_elem(const AppendParams &p, LoadFn x, int d, int pos) {
    const float xd = x(d);
    if (d >= p.rotary_dim) return xd;
    const int half = p.rotary_dim >> 1;
    int i, partner;
    bool first;
    if (p.interleaved) {
        i = d >> 1;
        first = (d & 1) == 0;
        partner = d ^ 1;
    } else {
        first = d < half;
        i = first ? d : d - half;
        partner = first ? d + half : d - half;
    }
    const float c = p.cos[(size_t)pos * half + i];
    const float s = p.sin[(size_t)pos * half + i];
    const float xp = x(partner);
    return first ? __fsub_rn(__fmul_rn(xd, c), __fmul_rn(xp, s)) : __fadd_rn(__fmul_rn(xd, c), __fmul_rn(xp, s));
}

__device__ __forceinline__ uint16_t round_16bit(float v, bool bf16) {
    return bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
}

__global__ void __launch_bounds__(kAppendWarps * 32) fd_append_kv_kernel(const AppendParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long job = (long long)blockIdx.x * kAppendWarps + warp;  // (b, kvh, which), then q rows
    const long long kv_jobs = 2LL * p.B * p.Hkv;
    const bool rotary = p.cos != nullptr;
    if (job >= kv_jobs) {
        // q row (b, hq), rotated in place at position seq_lens[b].
        if (!rotary || !p.q_inout || job >= kv_jobs + (long long)p.B * p.Hq) return;
        const int r = (int)(job - kv_jobs);
        const int b = r / p.Hq;
        const int pos = p.seq_lens[b];
        if (pos < 0 || pos >= p.max_pos) return;  // flagged by the K/V job of this sequence
        uint16_t *row = reinterpret_cast<uint16_t *>(p.q_inout) + (size_t)r * p.D;
        const bool qbf = p.q_is_bf16 != 0;
        auto x = [&](int d) { return load_16bit_as_float(row, d, qbf); };
        uint16_t outv[8];  // D <= 256: at most 8 elements per lane
        int k = 0;
        for (int d = lane; d < p.D; d += 32) outv[k++] = round_16bit(rotate_elem(p, x, d, pos), qbf);
        __syncwarp();      // every read of the row happens before any write
        k = 0;
        for (int d = lane; d < p.D; d += 32) row[d] = outv[k++];
        return;
    }
    const int which = (int)(job & 1);
    const int bk = (int)(job >> 1);
    const int b = bk / p.Hkv, kvh = bk - (bk / p.Hkv) * p.Hkv;
    const size_t src = ((size_t)b * p.Hkv + kvh) * p.D;
    const void *in = which ? p.v_new : p.k_new;
    // The new row does not depend on where it goes: request it before the
    // seq_lens -> block table -> page chain (16-bit bits, D <= 256).
    uint16_t raw[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int d = lane + 32 * k;
        raw[k] = d < p.D ? reinterpret_cast<const uint16_t *>(in)[src + d] : (uint16_t)0;
    }
    const int L = p.seq_lens[b];
    const int col = L >= 0 ? L / p.page_size : -1;
    int page = -1;
    if (col >= 0 && col < p.max_blocks) page = p.block_table[(size_t)b * p.max_blocks + col];
    if (page < 0 || page >= p.num_pages) {
        if (lane == 0 && which == 0 && kvh == 0 && p.status) atomicOr(p.status, FD_DEV_BAD_PAGE);
        return;
    }
    if (rotary && (L >= p.max_pos)) {
        if (lane == 0 && which == 0 && kvh == 0 && p.status) atomicOr(p.status, FD_DEV_CAPACITY);
        return;
    }
    const int slot = L - col * p.page_size;
    const size_t dst = (((size_t)page * p.page_size + slot) * p.Hkv + kvh) * p.D;
    void *pool = which ? p.v_pages : p.k_pages;
    const bool rot_k = rotary && which == 0;  // V is never rotated
    if (p.kv_kind != KV_E4M3) {
        const uint16_t *s16 = reinterpret_cast<const uint16_t *>(in) + src;
        uint16_t *d16 = reinterpret_cast<uint16_t *>(pool) + dst;
        if (!rot_k) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int d = lane + 32 * k;
                if (d < p.D) d16[d] = raw[k];
            }
            return;
        }
        const bool bf = p.kv_kind == KV_BF16;
        auto x = [&](int d) { return load_16bit_as_float(s16, d, bf); };
        for (int d = lane; d < p.D; d += 32) d16[d] = round_16bit(rotate_elem(p, x, d, L), bf);
        return;
    }
    const float sc = (which ? p.v_scale : p.k_scale)[(size_t)page * p.Hkv + kvh];
    uint8_t *d8 = reinterpret_cast<uint8_t *>(pool) + dst;
    const void *srow = reinterpret_cast<const uint16_t *>(in) + src;
    auto x = [&](int d) { return load_16bit_as_float(srow, d, p.new_is_bf16); };
    if (!rot_k) {
        // element lane + 32k sits in raw[k]; one byte per element
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int d = lane + 32 * k;
            if (d < p.D) {
                const float xv = p.new_is_bf16 ? __uint_as_float(static_cast<uint32_t>(raw[k]) << 16)
                                               : __half2float(__ushort_as_half(raw[k]));
                d8[d] = (uint8_t)(f32x2_to_e4m3x2(0.f, __fdiv_rn(xv, sc)) & 0xffu);
            }
        }
        return;
    }
    for (int d = 2 * lane; d < p.D; d += 64) {
        const float x0 = rotate_elem(p, x, d, L);
        const float x1 = rotate_elem(p, x, d + 1, L);
        const uint16_t codes = f32x2_to_e4m3x2(__fdiv_rn(x1, sc), __fdiv_rn(x0, sc));
        *reinterpret_cast<uint16_t *>(d8 + d) = codes;
    }
}

cudaError_t launch_append(const AppendParams &ap, cudaStream_t stream) {
    long long jobs = 2LL * ap.B * ap.Hkv;
    if (ap.cos && ap.q_inout) jobs += (long long)ap.B * ap.Hq;
    if (jobs == 0) return cudaSuccess;
    const long long blocks = (jobs + kAppendWarps - 1) / kAppendWarps;
    fd_append_kv_kernel<<<(unsigned)blocks, kAppendWarps * 32, 0, stream>>>(ap);
    return cudaGetLastError();
}

}  // namespace fd
