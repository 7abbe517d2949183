// merge.cu -- merge of partial attention states (lpnh.cn "FlashDecoding 核心原理",
// stage two; "FlashDecoding 与 FlashInfer 深度解析" §2.1 step 3):
//   m = max_i m_i, alpha_i = exp(m_i - m), d = sum_i alpha_i d_i,
//   out = sum_i alpha_i O_i / d, lse = m + ln d.
// One warp per (b, hq) row: lane i holds split i's (m_i, d_i) (splits past
// 32 are re-read from global memory), and each lane owns VEC-wide groups of
// the D outputs.  The first eight splits' partial outputs are requested
// before the weights are formed, so a row costs about one round of loads.
#include <math.h>

#include "fd_internal.h"
#include "ptx.cuh"

namespace fd {

constexpr int kMergeWarps = 4;

__device__ __forceinline__ void merge_store(void *out, size_t idx, float v, int out_dtype) {
    if (out_dtype == FD_BF16)
        reinterpret_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
    else if (out_dtype == FD_F16)
        reinterpret_cast<__half *>(out)[idx] = __float2half_rn(v);
    else
        reinterpret_cast<float *>(out)[idx] = v;
}

template <int VEC>
__device__ __forceinline__ void load_vec(const float *src, float *v) {
    if constexpr (VEC == 4) {
        const float4 t = *reinterpret_cast<const float4 *>(src);
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else if constexpr (VEC == 2) {
        const float2 t = *reinterpret_cast<const float2 *>(src);
        v[0] = t.x; v[1] = t.y;
    } else {
        v[0] = *src;
    }
}

// VEC consecutive outputs at idx (idx and out aligned for a VEC-wide store).
template <int VEC>
__device__ __forceinline__ void store_vec(void *out, size_t idx, const float *v, int out_dtype) {
    if constexpr (VEC == 1) {
        merge_store(out, idx, v[0], out_dtype);
    } else if (out_dtype == FD_F32) {
        if constexpr (VEC == 4)
            *reinterpret_cast<float4 *>(reinterpret_cast<float *>(out) + idx) = make_float4(v[0], v[1], v[2], v[3]);
        else
            *reinterpret_cast<float2 *>(reinterpret_cast<float *>(out) + idx) = make_float2(v[0], v[1]);
    } else {
        uint32_t w[VEC / 2];
#pragma unroll
        for (int k = 0; k < VEC / 2; ++k)
            w[k] = out_dtype == FD_BF16 ? pack_bf16x2(v[2 * k], v[2 * k + 1]) : pack_f16x2(v[2 * k], v[2 * k + 1]);
        if constexpr (VEC == 4)
            *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(out) + idx) = make_uint2(w[0], w[1]);
        else
            *reinterpret_cast<uint32_t *>(reinterpret_cast<uint16_t *>(out) + idx) = w[0];
    }
}

template <int VEC>
__global__ void __launch_bounds__(kMergeWarps * 32) fd_merge_states_kernel(const MergeParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kMergeWarps + warp;  // b * Hq + hq
    if (row >= (long long)p.B * p.Hq) return;
    const int b = (int)(row / p.Hq);
    int n = p.S;
    if (p.seq_lens) {
        // Rows of sequences that were not split were written by the decode
        // kernel itself; only the split ones are merged here.
        int cb = b / p.fold;  // KV row of this q sequence
        if (p.batch_idx) {
            cb = p.batch_idx[b];
            if (cb < 0 || cb >= p.cache_rows) return;
        }
        int L = p.seq_lens[cb];
        if (p.leftpad) {
            const int lp = p.leftpad[cb];
            L = (lp < 0 || lp > L) ? 0 : L - lp;
        }
        L = L < 0 ? 0 : (L > p.cap ? p.cap : L);
        n = (L == 0) ? 1 : (L + p.chunk - 1) / p.chunk;
        if (n <= 1) return;
    }
    const int D = p.D;
    const float *pm = p.part_m + row * p.S;
    const float *pd = p.part_d + row * p.S;
    const float *po = p.part_o + row * (size_t)p.S * D;
    const int ng = (D / VEC + 31) / 32;  // VEC-wide output groups per lane

    // The first batch of partial outputs of this lane's first group.
    float v0[8][VEC];
    {
        const bool live = lane * VEC < D;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (live && k < n)
                load_vec<VEC>(po + (size_t)k * D + lane * VEC, v0[k]);
            else
#pragma unroll
                for (int e = 0; e < VEC; ++e) v0[k][e] = 0.f;
        }
    }
    // Weights: max, then w_i = exp(m_i - m) and d = sum w_i d_i.
    const float ml = lane < n ? pm[lane] : -INFINITY;
    const float dl = lane < n ? pd[lane] : 0.f;
    float mx = ml;
    for (int s = lane + 32; s < n; s += 32) mx = fmaxf(mx, pm[s]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float al = (ml == -INFINITY || mx == -INFINITY) ? 0.f : __expf(ml - mx);
    float sum = al * dl;
    for (int s = lane + 32; s < n; s += 32) {
        const float ms = pm[s];
        sum += ((ms == -INFINITY) ? 0.f : __expf(ms - mx)) * pd[s];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const bool empty = (mx == -INFINITY) || !(sum > 0.f);
    const float inv = empty ? 0.f : 1.f / sum;
    auto weight = [&](int s) -> float {  // uniform s; every lane calls it
        const float a = __shfl_sync(0xffffffffu, al, s & 31);
        if (s < 32) return a;
        const float ms = pm[s];
        return (ms == -INFINITY) ? 0.f : __expf(ms - mx);
    };

    for (int grp = 0; grp < ng; ++grp) {
        const int e0 = (lane + 32 * grp) * VEC;
        const bool live = e0 < D;
        float acc[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
        for (int s0 = 0; s0 < n; s0 += 8) {
            float v[8][VEC];
            if (grp == 0 && s0 == 0) {
#pragma unroll
                for (int k = 0; k < 8; ++k)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) v[k][e] = v0[k][e];
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if (live && s0 + k < n)
                        load_vec<VEC>(po + (size_t)(s0 + k) * D + e0, v[k]);
                    else
#pragma unroll
                        for (int e = 0; e < VEC; ++e) v[k][e] = 0.f;
                }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float w = (s0 + k < n) ? weight(s0 + k) : 0.f;
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[e] = fmaf(w, v[k][e], acc[e]);
            }
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] *= inv;
        if (live) store_vec<VEC>(p.out, (size_t)row * D + e0, acc, p.out_dtype);
    }
    if (lane == 0 && p.lse) p.lse[row] = empty ? -INFINITY : mx + logf(sum);
}

// Two normalised states (out_a, lse_a) and (out_b, lse_b) of the same query
// over disjoint token sets: m = max(lse_a, lse_b), w = exp(lse - m),
// out = (w_a out_a + w_b out_b) / (w_a + w_b), lse = m + ln(w_a + w_b).
// One thread per (row, 4 elements of D).
__global__ void fd_merge_two_kernel(const float *oa, const float *la, const float *ob, const float *lb, int rows,
                                    int D, int out_dtype, void *out, float *lse) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const int per_row = D / 4;
    if (i >= (long long)rows * per_row) return;
    const long long row = i / per_row;
    const int d = (int)(i - row * per_row) * 4;
    const float a = la[row], b = lb[row];
    const float m = fmaxf(a, b);
    float wa = 0.f, wb = 0.f;
    if (m != -INFINITY) {
        wa = (a == -INFINITY) ? 0.f : __expf(a - m);
        wb = (b == -INFINITY) ? 0.f : __expf(b - m);
    }
    const float den = wa + wb;
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const float4 va = *reinterpret_cast<const float4 *>(oa + row * D + d);
    const float4 vb = *reinterpret_cast<const float4 *>(ob + row * D + d);
    const float r[4] = {(wa * va.x + wb * vb.x) * inv, (wa * va.y + wb * vb.y) * inv, (wa * va.z + wb * vb.z) * inv,
                        (wa * va.w + wb * vb.w) * inv};
    for (int k = 0; k < 4; ++k) merge_store(out, row * D + d + k, r[k], out_dtype);
    if (d == 0 && lse) lse[row] = den > 0.f ? m + logf(den) : -INFINITY;
}

cudaError_t launch_merge_two(const float *oa, const float *la, const float *ob, const float *lb, int rows, int D,
                             int out_dtype, void *out, float *lse, cudaStream_t stream) {
    const long long n = (long long)rows * (D / 4);
    if (n == 0) return cudaSuccess;
    fd_merge_two_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(oa, la, ob, lb, rows, D, out_dtype, out,
                                                                         lse);
    return cudaGetLastError();
}

cudaError_t launch_merge(const MergeParams &mp, cudaStream_t stream) {
    if (mp.S < 1) return cudaErrorInvalidValue;
    const long long rows = (long long)mp.B * mp.Hq;
    if (rows == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((rows + kMergeWarps - 1) / kMergeWarps);
    const size_t eb = mp.out_dtype == FD_F32 ? 4 : 2;
    auto al = [](const void *ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; };
    // Widest access the layout allows: every row start stays aligned when D
    // is a multiple of the width and the bases are aligned to it.
    if (mp.D % 4 == 0 && al(mp.part_o, 16) && al(mp.out, 4 * eb))
        fd_merge_states_kernel<4><<<grid, kMergeWarps * 32, 0, stream>>>(mp);
    else if (mp.D % 2 == 0 && al(mp.part_o, 8) && al(mp.out, 2 * eb))
        fd_merge_states_kernel<2><<<grid, kMergeWarps * 32, 0, stream>>>(mp);
    else
        fd_merge_states_kernel<1><<<grid, kMergeWarps * 32, 0, stream>>>(mp);
    return cudaGetLastError();
}

}  // namespace fd
