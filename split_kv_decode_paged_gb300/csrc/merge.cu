// merge.cu -- merge of partial attention states (lpnh.cn "FlashDecoding 核心原理",
// stage two; "FlashDecoding 与 FlashInfer 深度解析" §2.1 step 3):
//   m = max_i m_i, alpha_i = exp(m_i - m), d = sum_i alpha_i d_i,
//   out = sum_i alpha_i O_i / d, lse = m + ln d.
// One CTA per (b, hq); warp 0 computes the normalised weights alpha_i / d
// into shared memory, then all threads form the D outputs (coalesced).
#include <math.h>

#include "fd_internal.h"
#include "ptx.cuh"

namespace fd {

constexpr int kMergeThreads = 128;
constexpr int kMergeMaxS = 4096;

__device__ __forceinline__ void merge_store(void *out, size_t idx, float v, int out_dtype) {
    if (out_dtype == FD_BF16)
        reinterpret_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
    else if (out_dtype == FD_F16)
        reinterpret_cast<__half *>(out)[idx] = __float2half_rn(v);
    else
        reinterpret_cast<float *>(out)[idx] = v;
}

__global__ void __launch_bounds__(kMergeThreads) fd_merge_states_kernel(const MergeParams p) {
    __shared__ float w[kMergeMaxS];
    const size_t row = blockIdx.x;  // b * Hq + hq
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
    const float *pm = p.part_m + row * p.S;
    const float *pd = p.part_d + row * p.S;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ float s_lse_m, s_inv;
    if (warp == 0) {
        float mx = -INFINITY;
        for (int s = lane; s < n; s += 32) mx = fmaxf(mx, pm[s]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float sum = 0.f;
        for (int s = lane; s < n; s += 32) {
            const float ms = pm[s];
            const float a = (ms == -INFINITY || mx == -INFINITY) ? 0.f : __expf(ms - mx);
            w[s] = a;
            sum += a * pd[s];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) {
            const bool empty = (mx == -INFINITY) || !(sum > 0.f);
            s_inv = empty ? 0.f : 1.f / sum;
            s_lse_m = empty ? -INFINITY : mx + logf(sum);
        }
    }
    __syncthreads();
    const float inv = s_inv;
    if (threadIdx.x == 0 && p.lse) p.lse[row] = s_lse_m;
    const float *po = p.part_o + row * (size_t)p.S * p.D;
    // 8 independent loads in flight per batch of splits.
    for (int d = threadIdx.x; d < p.D; d += kMergeThreads) {
        float acc = 0.f;
        for (int s0 = 0; s0 < n; s0 += 8) {
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = (s0 + k < n) ? po[(size_t)(s0 + k) * p.D + d] : 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) acc += (s0 + k < n) ? w[s0 + k] * v[k] : 0.f;
        }
        merge_store(p.out, row * p.D + d, acc * inv, p.out_dtype);
    }
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
    if (mp.S > kMergeMaxS || mp.S < 1) return cudaErrorInvalidValue;
    const long long rows = (long long)mp.B * mp.Hq;
    if (rows == 0) return cudaSuccess;
    fd_merge_states_kernel<<<(unsigned)rows, kMergeThreads, 0, stream>>>(mp);
    return cudaGetLastError();
}

}  // namespace fd
