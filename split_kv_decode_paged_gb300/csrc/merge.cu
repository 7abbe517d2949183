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
        int cb = b;
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
    for (int d = threadIdx.x; d < p.D; d += kMergeThreads) {
        float acc = 0.f;
        for (int s = 0; s < n; ++s) acc += w[s] * po[(size_t)s * p.D + d];
        merge_store(p.out, row * p.D + d, acc * inv, p.out_dtype);
    }
}

cudaError_t launch_merge(const MergeParams &mp, cudaStream_t stream) {
    if (mp.S > kMergeMaxS || mp.S < 1) return cudaErrorInvalidValue;
    const long long rows = (long long)mp.B * mp.Hq;
    if (rows == 0) return cudaSuccess;
    fd_merge_states_kernel<<<(unsigned)rows, kMergeThreads, 0, stream>>>(mp);
    return cudaGetLastError();
}

}  // namespace fd
