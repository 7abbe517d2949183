// decode_kernel.cuh -- persistent split-KV paged decode attention for sm_103a.
//
// What one launch computes (lpnh.cn "FlashDecoding 核心原理", stages one and
// two; "FlashDecoding 与 FlashInfer 深度解析" §2.1): for every sequence b and
// query head hq, softmax(q k^T / sqrt(D)) V over the tokens [0, seq_lens[b])
// of its KV head kvh = hq / G, plus the log-sum-exp.
//
// Work decomposition.  A work item is (sequence b, split s, KV head kvh,
// head sub-group): the contiguous token range [s*C, min(L_b, (s+1)*C)) of one
// KV head, with the query heads of the group (up to 16 rows) packed into the
// same CTA so each K/V byte is read once (lpnh.cn "进阶突破", KV-reused layout
// for GQA).  Sequences shorter than one chunk are not split.  Items are
// dispatched longest first -- every full chunk, then each sequence's partial
// chunk sorted by length -- through an atomic counter to a persistent grid.
// Every CTA builds the same order in shared memory from seq_lens at start:
// the producer alone for small batches, all warps for large ones.
//
// CTA layout: NC consumer warps + 1 producer warp.
//   producer: claims items one ahead, reads the block table a batch of 32
//     boxes ahead, and issues TMA tensor loads of K and V boxes (page-size x D
//     slices of one KV head) into a ring of shared-memory stages, plus one
//     bulk copy of the item's query rows; stage hand-off through full/empty
//     mbarriers with bounded waits.
//   consumers: each warp takes SUBT sub-tiles of 16 tokens of every stage:
//     S^T[16 tok x 8 heads] = K[16 x D] . Q^T  (mma.sync m16n8k16, K from
//     swizzled shared memory via ldmatrix, Q in registers),
//     one online-softmax step over the warp's sub-tiles in the exp2 domain
//     (the reference maximum moves only when a score passes it by more than
//     kMaxSlack), P^T moved into the B operand
//     with movmatrix, O^T[D x 8] += V^T[D x 16] . P^T (ldmatrix.trans on V).
//     At the end of an item the warps merge their states (warp w+NC/2 into
//     warp w, then through shared memory); a single-split item writes
//     out/lse, a multi-split item writes its partial state (unnormalised O,
//     m, d) and the CTA that completes the last split of a group merges all
//     of them (atomic counter, no spin-wait), per the merge formula of stage
//     two.
// FP8 (E4M3) K/V are converted to f16 in registers (exact); the per-(page,
// KV head) scales multiply the scores and the P.V product.  A bf16 q enters
// that f16 product scaled per head by a power of two (exact in f16 over the
// head's whole range), undone on the scores.
#pragma once

#include <float.h>
#include <math.h>

#include "fd_internal.h"
#include "ptx.cuh"

namespace fd {

constexpr int kOrderBuckets = 64;  // length buckets of the partial-chunk dispatch order (2 per lane)
constexpr int kCoopBlocks = 4;     // 32-row blocks from which every warp builds the dispatch tables
constexpr int kFlagFirst = 1;
constexpr int kFlagLast = 2;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kMaxSlack = 8.f;  // log2 headroom of the softmax reference maximum

struct StageMeta {
    int b, kvh, s, t0, nvalid, flags, nsplit, vlo;  // b: KV row; valid tile rows [vlo, nvalid)
    int hg, nrows;                                  // head sub-group and its number of q rows
    float kscale[kMaxBoxesPerTile];
    float vscale[kMaxBoxesPerTile];
};
// The stage barriers (8-byte mbarriers) follow the array of StageMeta in
// shared memory.
static_assert(sizeof(StageMeta) % 8 == 0, "StageMeta keeps the barriers after it 8-byte aligned");

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int KV, int D, int NT, int NC, int SUBT>
struct DecodeShape {
    static constexpr int E = (KV == KV_E4M3) ? 1 : 2;  // K/V bytes per element
    static constexpr int RB = D * E;                   // bytes per K/V row
    static constexpr int SUBROW = RB > 128 ? 128 : RB; // swizzle span (bytes)
    static constexpr int NHALF = RB / SUBROW;          // sub-row regions per row
    static constexpr int TILE = NC * SUBT * kTokensPerWarp;  // tokens per stage
    static constexpr int QROWS = 8 * NT;               // padded query rows
    static constexpr int KV_REGION = TILE * RB;
    static constexpr int Q_REGION = align_up(QROWS * D * 2, 1024);
    static constexpr int STAGE = 2 * KV_REGION + Q_REGION;
    static constexpr int SS = D + 4;                   // scratch row stride (floats)
    // Epilogue slots of per-warp O rows: with 8 or more consumer warps, warp
    // w + NC/2 first hands its state to warp w, so half as many slots.
    // Reused for the merge weights (QROWS x kMaxSplits).
    static constexpr int NSLOT = NC >= 8 ? NC / 2 : NC;
    static constexpr int SCR_O = (NSLOT * QROWS * SS > QROWS * kMaxSplits) ? NSLOT * QROWS * SS : QROWS * kMaxSplits;
    // The slots and merge weights take a region of their own, or (16-bit
    // K/V, where a stage holds them and the plan asks for it) the item's
    // last stage, which the consumers then release only when the item's
    // epilogue and merge are over: the shared memory this frees goes to
    // another stage.  Not for 4 warps with two head tiles, whose two CTAs
    // per SM would no longer fit the register file.  E4M3: only the two-CTA
    // shape of 4 warps x 2 sub-tiles with one head tile, in an instance of
    // its own (the other E4M3 instances keep their registers).
    static constexpr bool SCR_STAGE_OK =
        (KV != KV_E4M3 || (NC == 4 && SUBT == 2 && NT == 1)) && SCR_O * 4 <= STAGE && !(NC == 4 && NT == 2);
    static constexpr int SCRATCH_SMALL = 2 * NC * QROWS * 4 + 2 * QROWS * 4 + 16;  // per-row m, l, 1/sum, max; flag
    static constexpr int SCRATCH = SCR_O * 4 + SCRATCH_SMALL;
    static constexpr int THREADS = (NC + 1) * 32;
    static_assert(D == 64 || D == 128, "D");
    static_assert(SUBROW == 128 || SUBROW == 64, "swizzle span");
};

// Offset of 16-byte chunk `chunk` of row `row` in a TMA-swizzled region.
template <int SUBROW>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    if constexpr (SUBROW == 128)
        return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
    else
        return static_cast<uint32_t>(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}

// Lanes of the warp whose 7-bit key equals this lane's (what match.any
// returns), from one ballot per key bit: a fixed cost whatever the number of
// distinct keys in the warp.
__device__ __forceinline__ unsigned same_key_lanes(unsigned key) {
    unsigned m = 0xffffffffu;
#pragma unroll
    for (int bit = 0; bit < 7; ++bit) {
        const bool set = (key >> bit) & 1u;
        const unsigned v = __ballot_sync(0xffffffffu, set);
        m &= set ? v : ~v;
    }
    return m;
}

// Idle for ns nanoseconds (the stall test hook of the timeout path).
__device__ __forceinline__ void idle_ns(uint64_t ns) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < ns) __nanosleep(1000);
}

__device__ __forceinline__ void flag_status(int *status, int bit) {
    if (status) atomicOr(status, bit);
}

template <typename T>
__device__ __forceinline__ T ldcg(const T *p) {
    return __ldcg(p);
}

// Four consecutive outputs (idx a multiple of 4).
__device__ __forceinline__ void store_out4(void *out, size_t idx, float a, float b, float c, float d,
                                           int out_dtype) {
    if (out_dtype == FD_BF16) {
        uint2 v;
        v.x = pack_bf16x2(a, b);
        v.y = pack_bf16x2(c, d);
        *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(out) + idx) = v;
    } else if (out_dtype == FD_F16) {
        uint2 v;
        v.x = pack_f16x2(a, b);
        v.y = pack_f16x2(c, d);
        *reinterpret_cast<uint2 *>(reinterpret_cast<__half *>(out) + idx) = v;
    } else {
        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(out) + idx) = make_float4(a, b, c, d);
    }
}

// Global q row (b * Hq + hq) of row j of head sub-group hg of (KV row bkv, kvh).
__device__ __forceinline__ size_t q_row(const DecodeParams &p, int bkv, int kvh, int hg, int j, int qrows) {
    const int i = hg * qrows + j;
    const int bq = bkv * p.fold + i / p.G;
    return (size_t)bq * p.Hq + (size_t)kvh * p.G + (i % p.G);
}

// Fused merge of the nsplit partial states of the nrows q rows of one
// (KV row, kvh, head sub-group), run by the consumer warps of the CTA that
// completed the last split: m_g = max m_i, w_i = exp(m_i - m_g),
// O = sum w_i O_i / sum w_i d_i, lse = m_g + log(sum w_i d_i).
// alpha: >= nrows*nsplit floats of shared memory.
template <int NC, int kInFlight>
__device__ void merge_group(const DecodeParams &p, int b, int kvh, int hg, int nrows, int qrows, int nsplit,
                            float *alpha, int warp, int lane, int D) {
    const int S = p.S;
    const int tid = warp * 32 + lane;
    constexpr int kFew = 8;
    if (nsplit <= kFew) {
        // Few splits: every thread reads the m, d and O of its four outputs
        // for all splits in one round of loads and merges them itself.
        for (int idx = tid; idx < nrows * (D / 4); idx += NC * 32) {
            const int h = idx / (D / 4), d = (idx - h * (D / 4)) * 4;
            const size_t row = q_row(p, b, kvh, hg, h, qrows);
            float m[kFew], dd[kFew];
            float4 v[kFew];
#pragma unroll
            for (int k = 0; k < kFew; ++k) {
                const bool in = k < nsplit;
                m[k] = in ? ldcg(p.part_m + row * S + k) : -INFINITY;
                dd[k] = in ? ldcg(p.part_d + row * S + k) : 0.f;
                v[k] = in ? __ldcg(reinterpret_cast<const float4 *>(p.part_o + (row * S + k) * D + d))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float mx = -INFINITY;
#pragma unroll
            for (int k = 0; k < kFew; ++k) mx = fmaxf(mx, m[k]);
            float sum = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kFew; ++k) {
                const float a = (m[k] == -INFINITY) ? 0.f : __expf(m[k] - mx);
                sum = fmaf(a, dd[k], sum);
                acc.x = fmaf(a, v[k].x, acc.x);
                acc.y = fmaf(a, v[k].y, acc.y);
                acc.z = fmaf(a, v[k].z, acc.z);
                acc.w = fmaf(a, v[k].w, acc.w);
            }
            const bool empty = (mx == -INFINITY) || !(sum > 0.f);
            const float inv = empty ? 0.f : 1.f / sum;
            store_out4(p.out, row * D + d, acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv, p.out_dtype);
            if (d == 0 && p.lse) p.lse[row] = empty ? -INFINITY : mx + logf(sum);
        }
        return;
    }
    // Many splits: a warp per q row finds the weights (m and d read in one
    // round), then the outputs in float4 groups with kInFlight split loads
    // in flight (16 where the caller's state is dead here, else 8: the
    // registers of the two-CTA shapes).
    for (int h = warp; h < nrows; h += NC) {
        const size_t row = q_row(p, b, kvh, hg, h, qrows);
        const float *pm = p.part_m + row * S;
        const float *pd = p.part_d + row * S;
        float mx = -INFINITY;
        float d_lane = 0.f;  // d of split `lane`, requested with its m
        for (int s = lane; s < nsplit; s += 32) {
            const float ms = ldcg(pm + s);
            if (s < 32) d_lane = ldcg(pd + s);
            alpha[h * nsplit + s] = ms;
            mx = fmaxf(mx, ms);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float sum = 0.f;
        for (int s = lane; s < nsplit; s += 32) {
            const float ms = alpha[h * nsplit + s];
            const float a = (ms == -INFINITY) ? 0.f : __expf(ms - mx);
            alpha[h * nsplit + s] = a;
            sum += a * (s < 32 ? d_lane : ldcg(pd + s));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const bool empty = (mx == -INFINITY) || !(sum > 0.f);
        const float inv = empty ? 0.f : 1.f / sum;
        for (int s = lane; s < nsplit; s += 32) alpha[h * nsplit + s] *= inv;
        if (lane == 0 && p.lse) p.lse[row] = empty ? -INFINITY : mx + logf(sum);
    }
    named_bar_sync(1, NC * 32);
    for (int idx = tid; idx < nrows * (D / 4); idx += NC * 32) {
        const int h = idx / (D / 4), d = (idx - h * (D / 4)) * 4;
        const size_t row = q_row(p, b, kvh, hg, h, qrows);
        const float *po = p.part_o + row * S * D + d;
        const float *al = alpha + h * nsplit;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = 0; s0 < nsplit; s0 += kInFlight) {
            float4 v[kInFlight];
#pragma unroll
            for (int k = 0; k < kInFlight; ++k)
                v[k] = (s0 + k < nsplit) ? __ldcg(reinterpret_cast<const float4 *>(po + (size_t)(s0 + k) * D))
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kInFlight; ++k) {
                const float a = (s0 + k < nsplit) ? al[s0 + k] : 0.f;
                acc.x = fmaf(a, v[k].x, acc.x);
                acc.y = fmaf(a, v[k].y, acc.y);
                acc.z = fmaf(a, v[k].z, acc.z);
                acc.w = fmaf(a, v[k].w, acc.w);
            }
        }
        store_out4(p.out, row * D + d, acc.x, acc.y, acc.z, acc.w, p.out_dtype);
    }
}

// Dispatch tables of a large batch (at least kCoopBlocks 32-row blocks),
// built by all NC + 1 warps of the CTA: the consumers have nothing to do
// before the first stage lands.  The result is the one the producer builds
// alone for small batches (same lengths, block prefixes, bucket function and
// stable order).  Every warp takes a contiguous run of blocks with its own
// bucket counts: (1) lengths, per-block item counts and per-warp bucket
// counts; (2) the last warp scans both into block prefixes (bpre[nb] = all
// full-chunk items) and per-warp bucket offsets (hist[(NC + 1) * 64] = all
// partial-chunk rows); (3) every warp places its rows.  hist is scratch of
// (NC + 1) * 64 + 1 ints.  Called by every thread of the CTA (it holds CTA
// barriers); kept out of line so the small-batch kernel body stays as it is.
template <int NC>
__device__ __noinline__ void build_dispatch_tables_coop(const DecodeParams &p, int *bpre, int *lens, int *hist,
                                                        uint16_t *order, int warp, int lane) {
    constexpr int NW = NC + 1;
    const int Bkv = p.Bkv, C = p.chunk, HG = p.Hkv * p.nhg;  // HG: items per chunk of a KV row
    const int nb = (Bkv + 31) >> 5;
    const int blk0 = (warp * nb) / NW, blk1 = ((warp + 1) * nb) / NW;
    int *hw = hist + warp * kOrderBuckets;  // this warp's bucket counts, then offsets
    auto tail_of = [&](int L) { return (L == 0 || L % C) ? L % C : -1; };  // -1: no partial chunk
    const int bsh = max(0, 26 - __clz(C));  // as in the kernel's producer
    auto bucket_of = [&](int r) { return (kOrderBuckets - 1) - (r >> bsh); };
    // Warm L2 with the block table (a slice per thread of every CTA).
    {
        const long long bt_bytes = (long long)p.cache_rows * p.max_blocks * (long long)sizeof(int32_t);
        if (bt_bytes <= (4 << 20)) {
            const char *bt = reinterpret_cast<const char *>(p.block_table);
            for (int off = ((int)blockIdx.x * 32 * NW + warp * 32 + lane) * 128; off < (int)bt_bytes;
                 off += (int)gridDim.x * 32 * NW * 128)
                prefetch_l2(bt + off);
        }
    }
    for (int i = lane; i < kOrderBuckets; i += 32) hw[i] = 0;
    __syncwarp();
    // (1) Four blocks per round, every load issued before any is used.
    for (int k0 = blk0; k0 < blk1; k0 += 4) {
        bool row[4];
        int cbv[4], slv[4], lpv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int b = (k0 + u) * 32 + lane;
            row[u] = k0 + u < blk1 && b < Bkv;
            cbv[u] = !row[u] ? -1 : (p.batch_idx ? __ldg(p.batch_idx + b) : b);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const bool in = row[u] && cbv[u] >= 0 && cbv[u] < p.cache_rows;
            slv[u] = in ? __ldg(p.seq_lens + cbv[u]) : 0;
            lpv[u] = (in && p.leftpad) ? __ldg(p.leftpad + cbv[u]) : 0;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (k0 + u >= blk1) break;  // warp-uniform
            const int b = (k0 + u) * 32 + lane;
            int bucket = kOrderBuckets;  // sentinel: past B or no partial chunk
            int vA = 0;
            if (row[u]) {
                int L = 0;
                if (cbv[u] < 0 || cbv[u] >= p.cache_rows) {
                    flag_status(p.status, FD_DEV_BAD_PAGE);
                } else {
                    L = slv[u];
                    if (p.leftpad) L = (lpv[u] < 0 || lpv[u] > L) ? -1 : L - lpv[u];
                }
                if (L < 0 || L > p.cap) {
                    flag_status(p.status, FD_DEV_CAPACITY);
                    L = L < 0 ? 0 : p.cap;
                }
                lens[b] = L;
                vA = (L / C) * HG;
                const int r = tail_of(L);
                if (r >= 0) bucket = bucket_of(r);
            }
            const unsigned peers = same_key_lanes((unsigned)bucket);
            if (bucket < kOrderBuckets && lane == __ffs(peers) - 1) hw[bucket] += __popc(peers);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) vA += __shfl_xor_sync(0xffffffffu, vA, o);
            if (lane == 0) bpre[k0 + u] = vA;  // the block's item count, scanned below
            __syncwarp();
        }
    }
    __syncthreads();
    if (warp == NC) {
        // (2a) Block item counts -> exclusive prefix.
        const int per = (nb + 31) >> 5;
        int sum = 0;
        for (int i = 0; i < per; ++i) {
            const int k = lane * per + i;
            if (k < nb) sum += bpre[k];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        int run = incl - sum;
        for (int i = 0; i < per; ++i) {
            const int k = lane * per + i;
            if (k < nb) {
                const int v = bpre[k];
                bpre[k] = run;
                run += v;
            }
        }
        if (lane == 31) bpre[nb] = incl;
        // (2b) Bucket counts (2 buckets per lane) -> where each warp's rows
        // of each bucket start.
        int t0 = 0, t1 = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            t0 += hist[w * kOrderBuckets + 2 * lane];
            t1 += hist[w * kOrderBuckets + 2 * lane + 1];
        }
        int v = t0 + t1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        int r0 = v - t0 - t1, r1 = v - t1;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            int *h = hist + w * kOrderBuckets + 2 * lane;
            const int c0 = h[0], c1 = h[1];
            h[0] = r0;
            h[1] = r1;
            r0 += c0;
            r1 += c1;
        }
        if (lane == 31) hist[NW * kOrderBuckets] = v;
    }
    __syncthreads();
    // (3) Place this warp's rows in the partial-chunk order.
    for (int k = blk0; k < blk1; ++k) {
        const int b = k * 32 + lane;
        const int r = b < Bkv ? tail_of(lens[b]) : -1;
        const int bucket = r >= 0 ? bucket_of(r) : kOrderBuckets;
        const unsigned peers = same_key_lanes((unsigned)bucket);
        if (bucket < kOrderBuckets) {
            const unsigned below = peers & ((1u << lane) - 1u);
            order[hw[bucket] + __popc(below)] = (uint16_t)b;
        }
        __syncwarp();
        if (bucket < kOrderBuckets && lane == __ffs(peers) - 1) hw[bucket] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
}

// CAUSAL: several query tokens per KV row (DecodeParams::qn > 1), each with
// its own causal limit; a separate instance so the one-token decode carries
// none of it.
// SCR: the E4M3 instance that may keep its epilogue scratch in the held stage.
template <int KV, int D, int NT, int NC, int SUBT, bool QBF16, bool CAUSAL, bool SCR = false>
__global__ void __launch_bounds__((NC + 1) * 32, 1)
    fd_split_kv_decode_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                              const __grid_constant__ CUtensorMap tmv) {
    using Sh = DecodeShape<KV, D, NT, NC, SUBT>;
    constexpr int TILE = Sh::TILE, SUBROW = Sh::SUBROW, NHALF = Sh::NHALF;
    constexpr int QROWS = Sh::QROWS, SS = Sh::SS;
    constexpr bool FP8 = (KV == KV_E4M3);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int NST = p.stages;
    uint8_t *stages = smem;
    const bool scr_in_stage = Sh::SCR_STAGE_OK && (KV != KV_E4M3 || SCR) && p.scr_in_stage;
    float *scr_own = reinterpret_cast<float *>(stages + (size_t)NST * Sh::STAGE);
    float *scr_m = scr_own + (scr_in_stage ? 0 : Sh::SCR_O);
    float *scr_l = scr_m + NC * QROWS;
    float *scr_inv = scr_l + NC * QROWS;   // per head: 1 / combined denominator
    float *scr_lse = scr_inv + QROWS;      // per head: combined max (log2 units)
    int *scr_flag = reinterpret_cast<int *>(scr_lse + QROWS);
    StageMeta *meta = reinterpret_cast<StageMeta *>(reinterpret_cast<uint8_t *>(scr_own) +
                                                    align_up(scr_in_stage ? Sh::SCRATCH_SMALL : Sh::SCRATCH, 128));
    uint64_t *full_bar = reinterpret_cast<uint64_t *>((reinterpret_cast<uintptr_t>(meta + NST) + 7) & ~uintptr_t(7));
    uint64_t *empty_bar = full_bar + NST;
    // Dispatch tables of the KV rows: item prefix at 32-row block
    // boundaries, attended length per row, partial-chunk row order.
    const int nblk = (p.Bkv + 31) / 32;
    int *bpre = reinterpret_cast<int *>(empty_bar + NST);  // nblk + 1
    int *lens = bpre + nblk + 1;                           // Bkv
    int *hist = lens + p.Bkv;                              // kOrderBuckets
    uint16_t *order = reinterpret_cast<uint16_t *>(hist + kOrderBuckets);  // Bkv

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), NC);
        }
        fence_barrier_init();
    }
    if (warp == NC && lane == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }
    __syncthreads();
    // Everything above touches only this CTA's shared memory and the kernel
    // parameters; global inputs and the workspace are read after the
    // preceding grid (e.g. the previous decode call) has completed.
    grid_dependency_wait();
    // Large batches: every warp builds the dispatch tables (see
    // build_dispatch_tables_coop); small ones: the producer alone, below.
    // Shapes at the register limit (two head tiles of D = 128) keep the
    // producer-only build: the out-of-line call would make them spill.
    constexpr bool kCoopTables = !(NT == 2 && D == 128);
    const bool coop = kCoopTables && ((p.Bkv + 31) >> 5) >= kCoopBlocks;  // the same in every thread
    // Its per-warp bucket tables live in the first stage, unused until the
    // producer issues the first load, after the tables are complete.
    static_assert(Sh::STAGE >= ((NC + 1) * kOrderBuckets + 1) * (int)sizeof(int), "bucket tables fit in a stage");
    int *coop_hist = reinterpret_cast<int *>(stages);  // (NC + 1) * kOrderBuckets + 1
    if constexpr (kCoopTables)
        if (coop) build_dispatch_tables_coop<NC>(p, bpre, lens, coop_hist, order, warp, lane);

    if (warp == NC) {
        // ================================================================ producer
        const int B = p.Bkv, Hkv = p.Hkv, C = p.chunk, ps = p.page_size, boxr = p.boxr;
        const int NHG = p.nhg, HG = Hkv * p.nhg;  // items per chunk of a KV row
        // K/V are streamed once per call: keep them from displacing other lines in L2.
        const uint64_t kv_policy = l2_policy_evict_first();
        const int BPT = TILE / boxr;  // boxes per tile: 1, 2, 4 (or 8)
        // boxr divides the power-of-two tile, so it is a power of two itself.
        const int bxs = __ffs(boxr) - 1;
        const int bpp = ps >> bxs;    // boxes per page
        int totalA = 0, nB = 0;
        if (coop) {
            totalA = bpre[(B + 31) >> 5];
            nB = coop_hist[(NC + 1) * kOrderBuckets];
        } else {
            // Warm L2 with the block table (each CTA one slice of it) while the
            // dispatch tables are built, so the first items' page ids hit L2.
            {
                const long long bt_bytes = (long long)p.cache_rows * p.max_blocks * (long long)sizeof(int32_t);
                if (bt_bytes <= (4 << 20)) {
                    const char *bt = reinterpret_cast<const char *>(p.block_table);
                    for (int off = ((int)blockIdx.x * 32 + lane) * 128; off < (int)bt_bytes; off += (int)gridDim.x * 32 * 128)
                        prefetch_l2(bt + off);
                }
            }
            // Dispatch order, identical in every CTA (it depends only on seq_lens):
            //  A: every full chunk (C tokens) of every KV row, in row order;
            //  B: the last, partial chunk of each row (or the single empty item of
            //     an empty row), rows sorted by that chunk's length, longest first
            //     (stable counting sort into kOrderBuckets buckets).
            // Largest items go first and the smallest fill the tail.
            // Attended length of every row: tokens [leftpad, seq_len) of its cache
            // row (block table, seq_lens and leftpad are indexed by the cache row;
            // an index outside the cache is flagged and the row attends nothing).
            // Four rows per lane per round, every load issued before any is used,
            // so a round costs one memory latency.
            for (int b0 = 0; b0 < B; b0 += 4 * 32) {
                int cbv[4], slv[4], lpv[4];
    #pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int b = b0 + u * 32 + lane;
                    cbv[u] = b >= B ? -1 : (p.batch_idx ? __ldg(p.batch_idx + b) : b);
                }
    #pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const bool in = cbv[u] >= 0 && cbv[u] < p.cache_rows;
                    slv[u] = in ? __ldg(p.seq_lens + cbv[u]) : 0;
                    lpv[u] = (in && p.leftpad) ? __ldg(p.leftpad + cbv[u]) : 0;
                }
    #pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int b = b0 + u * 32 + lane;
                    if (b >= B) continue;
                    int L = 0;
                    if (cbv[u] < 0 || cbv[u] >= p.cache_rows) {
                        flag_status(p.status, FD_DEV_BAD_PAGE);
                    } else {
                        L = slv[u];
                        if (p.leftpad) L = (lpv[u] < 0 || lpv[u] > L) ? -1 : L - lpv[u];
                    }
                    if (L < 0 || L > p.cap) {
                        flag_status(p.status, FD_DEV_CAPACITY);
                        L = L < 0 ? 0 : p.cap;
                    }
                    lens[b] = L;
                }
            }
            auto tail_of = [&](int L) { return (L == 0 || L % C) ? L % C : -1; };  // -1: no partial chunk
            if (B == 1) {
                // One KV row (a single long request): its full chunks, then
                // its partial chunk; no ordering to build.
                __syncwarp();
                const int L = lens[0];
                totalA = (L / C) * HG;
                nB = tail_of(L) >= 0 ? 1 : 0;
                if (lane == 0) {
                    bpre[0] = 0;
                    bpre[1] = totalA;
                    order[0] = 0;
                }
                __syncwarp();
            } else {
            for (int i = lane; i < kOrderBuckets; i += 32) hist[i] = 0;
            __syncwarp();
            // Bucket of a partial chunk of r < C tokens: r >> bsh < 64 for all of
            // them (buckets 2^bsh tokens wide, C / 64 < 2^bsh <= C / 32), longer
            // chunks in lower buckets.  A shift, not a division: this runs once
            // per row, twice, on the path to the first load.
            static_assert(kOrderBuckets == 64, "bucket_of assumes 64 buckets");
            const int bsh = max(0, 26 - __clz(C));
            auto bucket_of = [&](int r) { return (kOrderBuckets - 1) - (r >> bsh); };
            int runningA = 0;
            for (int base = 0; base < B; base += 32) {
                const int b = base + lane;
                int bucket = kOrderBuckets;  // sentinel: past B or no partial chunk
                int vA = 0;
                if (b < B) {
                    const int L = lens[b];
                    vA = (L / C) * HG;
                    const int r = tail_of(L);
                    if (r >= 0) bucket = bucket_of(r);
                }
                const unsigned peers = same_key_lanes((unsigned)bucket);
                if (bucket < kOrderBuckets && lane == __ffs(peers) - 1) hist[bucket] += __popc(peers);
    #pragma unroll
                for (int o = 16; o > 0; o >>= 1) vA += __shfl_xor_sync(0xffffffffu, vA, o);
                if (lane == 0) bpre[base >> 5] = runningA;
                runningA += vA;
                __syncwarp();
            }
            if (lane == 0) bpre[(B + 31) >> 5] = runningA;
            {   // exclusive scan of the bucket counts (2 buckets per lane)
                const int h0 = hist[2 * lane], h1 = hist[2 * lane + 1];
                int v = h0 + h1;
    #pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int t = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v += t;
                }
                nB = __shfl_sync(0xffffffffu, v, 31);
                const int excl = v - h0 - h1;
                __syncwarp();
                hist[2 * lane] = excl;
                hist[2 * lane + 1] = excl + h0;
                __syncwarp();
            }
            for (int base = 0; base < B; base += 32) {
                const int b = base + lane;
                const int r = b < B ? tail_of(lens[b]) : -1;
                const int bucket = r >= 0 ? bucket_of(r) : kOrderBuckets;
                const unsigned peers = same_key_lanes((unsigned)bucket);
                if (bucket < kOrderBuckets) {
                    const unsigned below = peers & ((1u << lane) - 1u);
                    order[hist[bucket] + __popc(below)] = (uint16_t)b;
                }
                __syncwarp();
                if (bucket < kOrderBuckets && lane == __ffs(peers) - 1) hist[bucket] += __popc(peers);
                __syncwarp();
            }
            totalA = runningA;
            }
        }
        const int total = totalA + nB * HG;

        // Item -> (b, split, kvh) and its token range.
        // Tokens [t_begin, t_end) of cache row cb; tiles start at the box
        // boundary a <= t_begin, and the first tile masks its vlo leading rows.
        struct Item {
            int b, cb, s, kvh, hg, nrows, L, nsplit, t_begin, t_end, ntok, ntiles, nbox, box0, vlo;
        };
        auto decode_item = [&](int item) -> Item {
            Item it;
            int r2;
            if (B == 1) {
                // One KV row: its full chunks, then its partial chunk, so
                // the chunk of item i is i / HG either way.
                it.b = 0;
                it.s = item / HG;
                r2 = item - it.s * HG;
            } else if (item < totalA) {
                // The 32-row block by binary search over the block prefix,
                // then the row by a warp scan of the block's item counts.
                int lo = 0, hi = ((B + 31) >> 5) - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (bpre[mid] <= item) lo = mid; else hi = mid - 1;
                }
                const int bl = lo * 32 + lane;
                const int v = bl < B ? (lens[bl] / C) * HG : 0;
                int incl = v;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                const int off = item - bpre[lo];
                const int ln = __ffs(__ballot_sync(0xffffffffu, incl > off)) - 1;
                it.b = lo * 32 + ln;
                // within a KV row: split-major, then kvh, then head sub-group
                // (the sub-groups of one (split, kvh) read the same K/V back to back)
                const int rem = off - __shfl_sync(0xffffffffu, incl - v, ln);
                it.s = rem / HG;
                r2 = rem - it.s * HG;
            } else {
                const int k = (item - totalA) / HG;
                it.b = order[k];
                it.s = lens[it.b] / C;
                r2 = (item - totalA) - k * HG;
            }
            it.kvh = r2 / NHG;
            it.hg = r2 - it.kvh * NHG;
            it.nrows = min(QROWS, p.G * p.fold - it.hg * QROWS);
            it.L = lens[it.b];
            // several query tokens per row need at least that many cached tokens
            if constexpr (CAUSAL)
                if (it.L < p.qn && lane == 0) flag_status(p.status, FD_DEV_CAPACITY);
            it.nsplit = it.L == 0 ? 1 : (it.L + C - 1) / C;
            it.cb = it.b;
            int lp = 0;
            if (p.batch_idx) {
                it.cb = __ldg(p.batch_idx + it.b);
                if (it.cb < 0 || it.cb >= p.cache_rows) { it.cb = 0; it.L = 0; }
            }
            if (p.leftpad && it.L > 0) lp = __ldg(p.leftpad + it.cb);
            it.t_begin = lp + it.s * C;
            it.t_end = lp + min(it.L, it.s * C + C);
            it.ntok = max(0, it.t_end - it.t_begin);
            const int a = it.ntok > 0 ? (it.t_begin >> bxs) << bxs : it.t_begin;
            it.vlo = it.t_begin - a;
            const int span = it.ntok > 0 ? it.t_end - a : 0;
            it.ntiles = max(1, (span + TILE - 1) / TILE);
            it.nbox = (span + boxr - 1) >> bxs;
            it.box0 = a >> bxs;
            it.t_begin = a;  // tiles are laid out from the aligned start
            return it;
        };
        // Page id of box k of an item (-1 past its end; -2 for a block-table
        // column out of range).
        auto page_of = [&](const Item &it, int k) -> int {
            if (k >= it.nbox) return -1;
            const int col = (it.box0 + k) / bpp;
            if (col >= p.max_blocks) return -2;
            return __ldg(p.block_table + (size_t)it.cb * p.max_blocks + col);
        };
        // Item ids: CTA i starts with item i; later items come from the
        // atomic counter, offset by the grid size.
        int st = 0;
        uint32_t ph = 0;
        bool ok = true;
        long long n_issued = 0;
        // One item of lookahead: the next item is claimed, and its first two
        // batches of page ids requested, while the current one streams.  The
        // claim is made late, in the item's last tiles, so that an item is
        // bound to the CTA that will be free first (a claim made as a long
        // item starts would hold the next item back for that item's whole
        // duration), while the stages still in flight cover the claim's
        // round trip and the page-id requests.
        int next_item = (int)blockIdx.x;
        Item nx{};
        int npg0 = -1, npg1 = -1;
        if (next_item < total) {
            nx = decode_item(next_item);
            npg0 = page_of(nx, lane);
            npg1 = page_of(nx, 32 + lane);
        }
        if (p.stall_role == 1) idle_ns(p.stall_ns);  // test hook: late producer
        while (ok && next_item < total) {
            const Item cur = nx;
            int pg_cur = npg0, pg_nxt = npg1;
            int claim_raw = 0;
            const int b = cur.b, s = cur.s, kvh = cur.kvh, nsplit = cur.nsplit;
            const int t_begin = cur.t_begin, t_end = cur.t_end, ntok = cur.ntok, ntiles = cur.ntiles;
            // Claim with the second-to-last tile and read it after the last
            // one; with only two stages, one tile earlier each (the claim's
            // round trip and the next item's page ids then have a tile's
            // time more to arrive).
            const int j_claim = NST >= 3 ? max(0, ntiles - 2) : max(0, ntiles - 3);
            const int j_read = NST >= 3 ? ntiles - 1 : (ntiles >= 3 ? ntiles - 2 : 0);
            const int nbox = cur.nbox, box0 = cur.box0;
            int batch = 0;
            for (int j = 0; j < ntiles; ++j) {
                if (j == j_claim && lane == 0) claim_raw = atomicAdd(p.work_ctr, 1);
                const int kb = j * BPT;
                if (kb >= (batch + 1) * 32) {
                    ++batch;
                    pg_cur = pg_nxt;
                    pg_nxt = page_of(cur, (batch + 1) * 32 + lane);
                }
                const int src_lane = (kb + (lane < BPT ? lane : 0)) & 31;
                const int pg = __shfl_sync(0xffffffffu, pg_cur, src_lane);
                const bool live = lane < BPT && (kb + lane) < nbox;
                const bool good = live && pg >= 0 && pg < p.num_pages;
                if (live && !good) flag_status(p.status, FD_DEV_BAD_PAGE);
                const unsigned good_mask = __ballot_sync(0xffffffffu, good);

                if (!mbar_wait_bounded(smem_u32(&empty_bar[st]), ph ^ 1u, p.timeout_ns)) {
                    flag_status(p.status, FD_DEV_TIMEOUT);
                    ok = false;
                    break;
                }
                const int t0 = t_begin + j * TILE;
                const bool load_q = (j == 0) && (ntok > 0);
                const uint32_t bytes = (uint32_t)__popc(good_mask) * 2u * (uint32_t)(boxr * Sh::RB) +
                                       (load_q ? (uint32_t)(cur.nrows * D * 2) : 0u);
                StageMeta *m = &meta[st];
                if (lane == 0) {
                    m->b = b; m->kvh = kvh; m->s = s; m->t0 = t0;
                    m->nvalid = max(0, min(TILE, t_end - t0));
                    m->vlo = j == 0 ? cur.vlo : 0;
                    m->hg = cur.hg;
                    m->nrows = cur.nrows;
                    m->flags = (j == 0 ? kFlagFirst : 0) | (j == ntiles - 1 ? kFlagLast : 0);
                    m->nsplit = nsplit;
                }
                const uint32_t fb = smem_u32(&full_bar[st]);
                if constexpr (FP8) {
                    // Per-(page, KV head) scales of the tile's boxes, copied
                    // asynchronously; the stage's full barrier also waits for
                    // them (registered before lane 0's arrival below).
                    if (good) {
                        cp_async_4(smem_u32(&m->kscale[lane]), p.k_scale + (size_t)pg * Hkv + kvh);
                        cp_async_4(smem_u32(&m->vscale[lane]), p.v_scale + (size_t)pg * Hkv + kvh);
                        cp_async_mbar_arrive(fb);
                    } else if (lane < BPT) {
                        m->kscale[lane] = 1.f;
                        m->vscale[lane] = 1.f;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(fb, bytes);
                __syncwarp();
                uint8_t *sb = stages + (size_t)st * Sh::STAGE;
                auto issue_kv = [&]() {
                    if (good) {
                        // One box = boxr token rows x the whole D of one KV head,
                        // stored as NHALF swizzled regions of boxr x SUBROW bytes.
                        const int tok = (box0 + kb + lane) * boxr;
                        const int slot = tok % ps;
                        const uint32_t off = (uint32_t)(lane * NHALF * boxr * SUBROW);
                        tma_load_5d(smem_u32(sb + off), &tmk, fb, 0, slot, 0, kvh, pg, kv_policy);
                        tma_load_5d(smem_u32(sb + Sh::KV_REGION + off), &tmv, fb, 0, slot, 0, kvh, pg, kv_policy);
                    }
                };
                auto issue_q = [&]() {
                    if (load_q) {
                        // The item's q rows: one contiguous run of heads per q
                        // sequence it spans; lane t copies run t.
                        const int i0 = cur.hg * QROWS, i1 = i0 + cur.nrows, Gh = p.G;
                        const int bq0 = i0 / Gh;
                        const int ia = max(i0, (bq0 + lane) * Gh), ib = min(i1, (bq0 + lane + 1) * Gh);
                        if (ia < ib) {
                            const int bq = b * p.fold + ia / Gh;
                            const uint8_t *qsrc = reinterpret_cast<const uint8_t *>(p.q) +
                                                  ((size_t)bq * p.Hq + (size_t)kvh * Gh + (ia % Gh)) * D * 2;
                            bulk_load(smem_u32(sb + 2 * Sh::KV_REGION + (ia - i0) * D * 2), qsrc,
                                      (uint32_t)((ib - ia) * D * 2), fb);
                        }
                    }
                };
                // 16-bit K/V: the K/V boxes first, so the large copies start
                // earlier; E4M3 K/V: q first (measured the faster order each).
                if constexpr (!FP8) { issue_kv(); issue_q(); } else { issue_q(); issue_kv(); }
                ++n_issued;
                if (++st == NST) { st = 0; ph ^= 1u; }
                if (j == j_read) {
                    next_item = (int)gridDim.x + __shfl_sync(0xffffffffu, claim_raw, 0);
                    if (next_item < total) {
                        nx = decode_item(next_item);
                        npg0 = page_of(nx, lane);
                        npg1 = page_of(nx, 32 + lane);
                    }
                }
            }
        }
        // No more items to claim: the next grid in the stream may start
        // launching onto SMs as they free up.
        grid_launch_dependents();
        // Wait (bounded) until the copies into the stages issued most recently
        // have landed: the consumers leave early when one of their own waits
        // runs out, and no copy may still be in flight when the CTA exits.
        // Only this warp arrives on the full barriers, so the phase of each
        // stage's last issue is still the one its parity names.
        for (int k = 1; k <= NST && k <= n_issued; ++k) {
            const int s2 = (st - k + NST) % NST;
            const uint32_t par = (s2 < st) ? ph : (ph ^ 1u);
            if (!mbar_wait_bounded(smem_u32(&full_bar[s2]), par, p.timeout_ns)) ok = false;
        }
        // Stop marker for the consumers.
        if (ok && mbar_wait_bounded(smem_u32(&empty_bar[st]), ph ^ 1u, p.timeout_ns)) {
            if (lane == 0) {
                meta[st].b = -1;
                mbar_arrive(smem_u32(&full_bar[st]));
            }
        } else {
            flag_status(p.status, FD_DEV_TIMEOUT);
        }
        // Last producer out resets the work counters for the next launch
        // (the release orders this CTA's claims before its count; the
        // acquire orders every CTA's claims before the reset).
        if (lane == 0) {
            const int done = atom_add_acq_rel_gpu(p.done_ctr, 1);
            if (done == (int)gridDim.x - 1) {
                atomicExch(p.work_ctr, 0);
                atomicExch(p.done_ctr, 0);
            }
        }
        return;
    }

    // ==================================================================== consumers
    const int g = lane >> 2, c = lane & 3;
    constexpr int KT = D / 16;  // k-steps of QK (f16/bf16 path)
    constexpr int MT = D / 16;  // m-tiles of PV
    uint32_t qf[KT][NT][2];
    // E4M3 K/V with bf16 q: q enters the f16 MMA scaled per head by a power
    // of two; qd[n][r] undoes it for score column 2c + r of head tile n.
    float qd[NT][2];
#pragma unroll
    for (int n = 0; n < NT; ++n) qd[n][0] = qd[n][1] = 1.f;
    float o[MT][NT][4];
    float mrow[NT][2], lrow[NT][2];
    const float scale_log2 = p.scale_log2;

    if (p.stall_role == 2) {
        // Test hook: slow consumers.  Hold the first stage (the producer
        // cannot refill it before it is released) for stall_ns.
        if (mbar_wait_bounded(smem_u32(&full_bar[0]), 0, p.timeout_ns)) idle_ns(p.stall_ns);
    }
    int st = 0;
    uint32_t ph = 0;
    while (true) {
        if (!mbar_wait_bounded(smem_u32(&full_bar[st]), ph, p.timeout_ns)) {
            flag_status(p.status, FD_DEV_TIMEOUT);
            break;
        }
        const StageMeta &mt = meta[st];
        const int mb = mt.b;
        if (mb < 0) break;
        const int flags = mt.flags, nvalid = mt.nvalid, vlo = mt.vlo;
        const uint8_t *sb = stages + (size_t)st * Sh::STAGE;
        const uint32_t kbase = smem_u32(sb), vbase = kbase + Sh::KV_REGION, qbase = kbase + 2 * Sh::KV_REGION;

        if (flags & kFlagFirst) {
            // Query fragments (B operand of QK), zero for padded heads.
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const bool live_head = (n * 8 + g) < mt.nrows;
                if constexpr (!FP8) {
#pragma unroll
                    for (int kk = 0; kk < KT; kk += 2) {
                        const int row = n * 8 + (lane & 7);
                        const int chunk = 2 * kk + (lane >> 3);
                        uint32_t r0, r1, r2, r3;
                        ldsm_x4(qbase + (uint32_t)(row * D * 2 + chunk * 16), r0, r1, r2, r3);
                        qf[kk][n][0] = live_head ? r0 : 0u;
                        qf[kk][n][1] = live_head ? r1 : 0u;
                        qf[kk + 1][n][0] = live_head ? r2 : 0u;
                        qf[kk + 1][n][1] = live_head ? r3 : 0u;
                    }
                } else {
                    // f16 fragments in the E4M3 k-order: k-step ks covers
                    // d = 32*(ks/2) + 16*(ks%2) + {4c..4c+3}.
                    const int row = n * 8 + g;
                    const uint8_t *qrow = sb + 2 * Sh::KV_REGION + row * D * 2;
                    if constexpr (QBF16) {
                        // bf16 q into the f16 product.  Direct conversion is
                        // exact for elements in [2^-17, 65504] and loses at
                        // most 2^-25 below; it is kept when every element of
                        // the head is below 2^15 and its largest is at least
                        // 2^-3 (small elements then lose < 2^-22 of the
                        // largest).  A head tile with any other head is
                        // redone with a per-head power of two 2^e that brings
                        // each head's largest |q| into [2^14, 2^15): every
                        // element within 2^31 of it is then exact (8
                        // significant bits into 11), smaller ones lose less
                        // than 2^-39 of it, and the scores get 2^-e back.
                        float amax = 0.f;  // this lane's elements of head row g
#pragma unroll
                        for (int ks = 0; ks < KT; ++ks) {
                            const int d0 = 32 * (ks >> 1) + 16 * (ks & 1) + 4 * c;
                            const uint2 raw = *reinterpret_cast<const uint2 *>(qrow + d0 * 2);
                            const float x0 = __uint_as_float(raw.x << 16), x1 = __uint_as_float(raw.x & 0xffff0000u);
                            const float x2 = __uint_as_float(raw.y << 16), x3 = __uint_as_float(raw.y & 0xffff0000u);
                            amax = fmaxf(fmaxf(amax, fmaxf(fabsf(x0), fabsf(x1))), fmaxf(fabsf(x2), fabsf(x3)));
                            qf[ks][n][0] = live_head ? pack_f16x2(x0, x1) : 0u;
                            qf[ks][n][1] = live_head ? pack_f16x2(x2, x3) : 0u;
                        }
                        // head row g is small when all four of its lanes are
                        const unsigned small = __ballot_sync(0xffffffffu, !(amax >= 0.125f));
                        const bool row_small = ((small >> (4 * g)) & 0xfu) == 0xfu;
                        if (__any_sync(0xffffffffu, live_head && (amax >= 32768.f || row_small))) {
                            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                            // e = 141 - biased exponent of amax, kept in
                            // [-126, 126] so that 2^e and 2^-e are normal
                            const int be = (int)((__float_as_uint(amax) >> 23) & 0xffu);
                            const int e = (live_head && amax > 0.f) ? max(-126, min(126, 141 - be)) : 0;
                            const float up = __uint_as_float((uint32_t)(127 + e) << 23);
                            const float down = __uint_as_float((uint32_t)(127 - e) << 23);
                            qd[n][0] = __shfl_sync(0xffffffffu, down, 8 * c);      // head 2c
                            qd[n][1] = __shfl_sync(0xffffffffu, down, 8 * c + 4);  // head 2c + 1
#pragma unroll
                            for (int ks = 0; ks < KT; ++ks) {
                                const int d0 = 32 * (ks >> 1) + 16 * (ks & 1) + 4 * c;
                                const uint2 raw = *reinterpret_cast<const uint2 *>(qrow + d0 * 2);
                                const uint32_t w0 = pack_f16x2(__uint_as_float(raw.x << 16) * up,
                                                               __uint_as_float(raw.x & 0xffff0000u) * up);
                                const uint32_t w1 = pack_f16x2(__uint_as_float(raw.y << 16) * up,
                                                               __uint_as_float(raw.y & 0xffff0000u) * up);
                                qf[ks][n][0] = live_head ? w0 : 0u;
                                qf[ks][n][1] = live_head ? w1 : 0u;
                            }
                        } else {
                            qd[n][0] = qd[n][1] = 1.f;
                        }
                    } else {
#pragma unroll
                        for (int ks = 0; ks < KT; ++ks) {
                            const int d0 = 32 * (ks >> 1) + 16 * (ks & 1) + 4 * c;
                            const uint2 raw = *reinterpret_cast<const uint2 *>(qrow + d0 * 2);
                            qf[ks][n][0] = live_head ? raw.x : 0u;
                            qf[ks][n][1] = live_head ? raw.y : 0u;
                        }
                    }
                }
            }
#pragma unroll
            for (int mi = 0; mi < MT; ++mi)
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int r = 0; r < 4; ++r) o[mi][n][r] = 0.f;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                mrow[n][0] = mrow[n][1] = -INFINITY;
                lrow[n][0] = lrow[n][1] = 0.f;
            }
        }

        // The warp's SUBT sub-tiles of 16 tokens (tile rows r0 .. r0+15 with
        // r0 = (sub*NC + warp)*16, each inside box r0 / boxr: sub-tiles are
        // dealt to the warps in turn, so a ragged last tile leaves every warp
        // about the same number of valid rows) share one
        // online-softmax step: scores of every sub-tile, one check of the
        // reference maxima (and, when needed, one reduction and O rescale),
        // then P.V of every sub-tile.  Valid rows of a sub-tile: [ll, nl).
        int nl[SUBT], ll[SUBT];
        bool any_act = false;
#pragma unroll
        for (int sub = 0; sub < SUBT; ++sub) {
            const int r0 = (sub * NC + warp) * kTokensPerWarp;
            nl[sub] = max(0, min(kTokensPerWarp, nvalid - r0));
            ll[sub] = max(0, vlo - r0);
            any_act |= nl[sub] > ll[sub];
        }
        if (any_act) {
            const uint32_t hstride = (uint32_t)(p.boxr * SUBROW);
            // ---------------------------------------------------------- S = K Q^T
            // Two independent accumulator chains per sub-tile (even / odd
            // k-steps) halve the dependent MMA latency of the dot products.
            float sv[SUBT][NT][4];
#pragma unroll
            for (int sub = 0; sub < SUBT; ++sub) {
                const int r0 = (sub * NC + warp) * kTokensPerWarp;
                const uint32_t kbox = kbase + (uint32_t)((r0 / p.boxr) * NHALF) * hstride;
                const int row_a = r0 % p.boxr + (lane & 7) + ((lane >> 3) & 1) * 8;
                float s2[NT][4];
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int r = 0; r < 4; ++r) sv[sub][n][r] = s2[n][r] = 0.f;
                if (nl[sub] > ll[sub]) {
                    if constexpr (!FP8) {
#pragma unroll
                        for (int kk = 0; kk < KT; ++kk) {
                            const int byte = kk * 32;
                            const int h = byte / SUBROW;
                            const int chunk = (byte % SUBROW) / 16 + (lane >> 4);
                            uint32_t a0, a1, a2, a3;
                            ldsm_x4(kbox + (uint32_t)h * hstride + swz<SUBROW>(row_a, chunk), a0, a1, a2, a3);
#pragma unroll
                            for (int n = 0; n < NT; ++n) {
                                float *acc = (kk & 1) ? s2[n] : sv[sub][n];
                                if constexpr (KV == KV_BF16)
                                    mma_bf16(acc, a0, a1, a2, a3, qf[kk][n][0], qf[kk][n][1]);
                                else
                                    mma_f16(acc, a0, a1, a2, a3, qf[kk][n][0], qf[kk][n][1]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int jg = 0; jg < D / 32; ++jg) {
                            const int byte = jg * 32;
                            const int h = byte / SUBROW;
                            const int chunk = (byte % SUBROW) / 16 + (lane >> 4);
                            uint32_t q0, q1, q2, q3;
                            ldsm_x4(kbox + (uint32_t)h * hstride + swz<SUBROW>(row_a, chunk), q0, q1, q2, q3);
                            const uint32_t a00 = e4m3x2_to_f16x2((uint16_t)(q0 & 0xffff));
                            const uint32_t a01 = e4m3x2_to_f16x2((uint16_t)(q1 & 0xffff));
                            const uint32_t a02 = e4m3x2_to_f16x2((uint16_t)(q0 >> 16));
                            const uint32_t a03 = e4m3x2_to_f16x2((uint16_t)(q1 >> 16));
                            const uint32_t a10 = e4m3x2_to_f16x2((uint16_t)(q2 & 0xffff));
                            const uint32_t a11 = e4m3x2_to_f16x2((uint16_t)(q3 & 0xffff));
                            const uint32_t a12 = e4m3x2_to_f16x2((uint16_t)(q2 >> 16));
                            const uint32_t a13 = e4m3x2_to_f16x2((uint16_t)(q3 >> 16));
#pragma unroll
                            for (int n = 0; n < NT; ++n) {
                                mma_f16(sv[sub][n], a00, a01, a02, a03, qf[2 * jg][n][0], qf[2 * jg][n][1]);
                                mma_f16(s2[n], a10, a11, a12, a13, qf[2 * jg + 1][n][0], qf[2 * jg + 1][n][1]);
                            }
                        }
                    }
                }
                // scaled, masked scores
                float sc = scale_log2;
                if constexpr (FP8) sc *= mt.kscale[r0 / p.boxr];
                const bool v0 = g >= ll[sub] && g < nl[sub], v1 = (g + 8) >= ll[sub] && (g + 8) < nl[sub];
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    float sc0 = sc, sc1 = sc;
                    if constexpr (FP8 && QBF16) {
                        sc0 *= qd[n][0];
                        sc1 *= qd[n][1];
                    }
                    bool v00 = v0, v01 = v0, v10 = v1, v11 = v1;
                    if constexpr (CAUSAL) {
                        // causal: q row i of the item is query token i / G of
                        // the KV row and sees the cached tokens
                        // [0, L - qn + i / G + 1); token t of the tile row is
                        // hidden from the score columns (q rows 2c, 2c + 1 of
                        // head tile n) whose limit it reaches
                        const int ta = mt.t0 + r0 + g;
                        const int i0 = mt.hg * QROWS + n * 8 + 2 * c;
                        const int L = lens[mt.b];  // the row's attended length (dispatch table)
                        const int l0 = L - p.qn + i0 / p.G + 1, l1 = L - p.qn + (i0 + 1) / p.G + 1;
                        v00 = v00 && ta < l0;
                        v01 = v01 && ta < l1;
                        v10 = v10 && ta + 8 < l0;
                        v11 = v11 && ta + 8 < l1;
                    }
                    sv[sub][n][0] = v00 ? (sv[sub][n][0] + s2[n][0]) * sc0 : -INFINITY;
                    sv[sub][n][1] = v01 ? (sv[sub][n][1] + s2[n][1]) * sc1 : -INFINITY;
                    sv[sub][n][2] = v10 ? (sv[sub][n][2] + s2[n][2]) * sc0 : -INFINITY;
                    sv[sub][n][3] = v11 ? (sv[sub][n][3] + s2[n][3]) * sc1 : -INFINITY;
                }
            }

            // ------------------------------------------------- online softmax (exp2)
            // The reference maximum mrow only moves when some score exceeds it
            // by more than kMaxSlack (log2 units): softmax does not depend on
            // the reference, and the weights stay <= 2^kMaxSlack.  Then the
            // warp reduces the step's row maxima (three shuffle rounds) and
            // rescales; otherwise it skips both.
            float mx[NT][2];
            bool need = false;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                mx[n][0] = mx[n][1] = -INFINITY;
#pragma unroll
                for (int sub = 0; sub < SUBT; ++sub) {
                    mx[n][0] = fmaxf(mx[n][0], fmaxf(sv[sub][n][0], sv[sub][n][2]));
                    mx[n][1] = fmaxf(mx[n][1], fmaxf(sv[sub][n][1], sv[sub][n][3]));
                }
                need |= mx[n][0] > mrow[n][0] + kMaxSlack;
                need |= mx[n][1] > mrow[n][1] + kMaxSlack;
            }
            float alpha[NT][2];
            const bool moved = __any_sync(0xffffffffu, need);
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                alpha[n][0] = alpha[n][1] = 1.f;
                if (moved) {
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        mx[n][0] = fmaxf(mx[n][0], shfl_xor(mx[n][0], off));
                        mx[n][1] = fmaxf(mx[n][1], shfl_xor(mx[n][1], off));
                    }
                    const float mn0 = fmaxf(mrow[n][0], mx[n][0]), mn1 = fmaxf(mrow[n][1], mx[n][1]);
                    alpha[n][0] = (mn0 == -INFINITY) ? 1.f : ex2(mrow[n][0] - mn0);
                    alpha[n][1] = (mn1 == -INFINITY) ? 1.f : ex2(mrow[n][1] - mn1);
                    mrow[n][0] = mn0;
                    mrow[n][1] = mn1;
                }
            }
            uint32_t pb[SUBT][NT][2];
            uint32_t pl[SUBT][NT][2];  // bf16 V: low parts of the weights (P = hi + lo)
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const float mn0 = mrow[n][0], mn1 = mrow[n][1];
                float add0 = 0.f, add1 = 0.f;
#pragma unroll
                for (int sub = 0; sub < SUBT; ++sub) {
                    const float p0 = (mn0 == -INFINITY) ? 0.f : ex2(sv[sub][n][0] - mn0);
                    const float p1 = (mn1 == -INFINITY) ? 0.f : ex2(sv[sub][n][1] - mn1);
                    const float p2 = (mn0 == -INFINITY) ? 0.f : ex2(sv[sub][n][2] - mn0);
                    const float p3 = (mn1 == -INFINITY) ? 0.f : ex2(sv[sub][n][3] - mn1);
                    uint32_t x0, x1;
                    float wr0, wr1, wr2, wr3;  // the rounded weights actually used
                    if constexpr (KV == KV_BF16) {
                        // bf16 keeps 8 significant bits; the weights enter P.V
                        // as hi + lo bf16 pairs (two MMAs on one V fragment),
                        // so the product sees them to ~2^-17 relative.
                        x0 = pack_bf16x2(p0, p1);
                        x1 = pack_bf16x2(p2, p3);
                        const float h0 = __uint_as_float(x0 << 16), h1 = __uint_as_float(x0 & 0xffff0000u);
                        const float h2 = __uint_as_float(x1 << 16), h3 = __uint_as_float(x1 & 0xffff0000u);
                        const uint32_t y0 = pack_bf16x2(p0 - h0, p1 - h1);
                        const uint32_t y1 = pack_bf16x2(p2 - h2, p3 - h3);
                        wr0 = h0 + __uint_as_float(y0 << 16); wr1 = h1 + __uint_as_float(y0 & 0xffff0000u);
                        wr2 = h2 + __uint_as_float(y1 << 16); wr3 = h3 + __uint_as_float(y1 & 0xffff0000u);
                        pl[sub][n][0] = movmatrix_t(y0);
                        pl[sub][n][1] = movmatrix_t(y1);
                    } else {
                        x0 = pack_f16x2(p0, p1);
                        x1 = pack_f16x2(p2, p3);
                        const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&x0));
                        const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&x1));
                        wr0 = f0.x; wr1 = f0.y; wr2 = f1.x; wr3 = f1.y;
                    }
                    add0 += wr0 + wr2;
                    add1 += wr1 + wr3;
                    pb[sub][n][0] = movmatrix_t(x0);
                    pb[sub][n][1] = movmatrix_t(x1);
                }
                lrow[n][0] = lrow[n][0] * alpha[n][0] + add0;
                lrow[n][1] = lrow[n][1] * alpha[n][1] + add1;
            }
            if (moved) {
#pragma unroll
                for (int mi = 0; mi < MT; ++mi)
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        o[mi][n][0] *= alpha[n][0];
                        o[mi][n][1] *= alpha[n][1];
                        o[mi][n][2] *= alpha[n][0];
                        o[mi][n][3] *= alpha[n][1];
                    }
            }

            // ---------------------------------------------------- O^T += V^T P^T
#pragma unroll
            for (int sub = 0; sub < SUBT; ++sub) {
                if (!(nl[sub] > ll[sub])) continue;
                const int r0 = (sub * NC + warp) * kTokensPerWarp;
                const int rib = r0 % p.boxr;
                const uint32_t vbox = vbase + (uint32_t)((r0 / p.boxr) * NHALF) * hstride;
                // Rows outside [ll, nl) may hold any bits (stale or NaN):
                // partial sub-tiles zero their V fragments.
                const bool part = nl[sub] < kTokensPerWarp || ll[sub] > 0;
                uint32_t msk01 = 0xffffffffu, msk23 = 0xffffffffu;
                if (part) {
                    const int lo_t = ll[sub], hi_t = nl[sub];
                    auto ok_t = [&](int t) { return t >= lo_t && t < hi_t; };
                    msk01 = (ok_t(2 * c) ? 0x0000ffffu : 0u) | (ok_t(2 * c + 1) ? 0xffff0000u : 0u);
                    msk23 = (ok_t(2 * c + 8) ? 0x0000ffffu : 0u) | (ok_t(2 * c + 9) ? 0xffff0000u : 0u);
                }
                if constexpr (!FP8) {
                    const int row_t = rib + (lane & 7) + (lane >> 4) * 8;
#pragma unroll
                    for (int mi = 0; mi < MT; ++mi) {
                        const int byte = mi * 32;
                        const int h = byte / SUBROW;
                        const int chunk = (byte % SUBROW) / 16 + ((lane >> 3) & 1);
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4_t(vbox + (uint32_t)h * hstride + swz<SUBROW>(row_t, chunk), a0, a1, a2, a3);
                        if (part) { a0 &= msk01; a1 &= msk01; a2 &= msk23; a3 &= msk23; }
#pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            if constexpr (KV == KV_BF16) {
                                mma_bf16(o[mi][n], a0, a1, a2, a3, pb[sub][n][0], pb[sub][n][1]);
                                mma_bf16(o[mi][n], a0, a1, a2, a3, pl[sub][n][0], pl[sub][n][1]);
                            } else {
                                mma_f16(o[mi][n], a0, a1, a2, a3, pb[sub][n][0], pb[sub][n][1]);
                            }
                        }
                    }
                } else {
                    const int row_a = rib + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const float vsc = mt.vscale[r0 / p.boxr];
#pragma unroll
                    for (int jg = 0; jg < D / 32; ++jg) {
                        const int byte = jg * 32;
                        const int h = byte / SUBROW;
                        const int chunk = (byte % SUBROW) / 16 + (lane >> 4);
                        uint32_t q0, q1, q2, q3;
                        ldsm_x4_t(vbox + (uint32_t)h * hstride + swz<SUBROW>(row_a, chunk), q0, q1, q2, q3);
                        // the 16-bit halves of q0, q2 hold tokens 2c, 2c+1; of
                        // q1, q3 tokens 2c+8, 2c+9 (E4M3 zero bytes convert to +0)
                        if (part) { q0 &= msk01; q1 &= msk23; q2 &= msk01; q3 &= msk23; }
                        const uint32_t t0 = __byte_perm(q0, 0, 0x3120), t1 = __byte_perm(q1, 0, 0x3120);
                        const uint32_t t2 = __byte_perm(q2, 0, 0x3120), t3 = __byte_perm(q3, 0, 0x3120);
                        uint32_t A[2][4];
                        A[0][0] = e4m3x2_to_f16x2((uint16_t)(t0 & 0xffff));
                        A[0][1] = e4m3x2_to_f16x2((uint16_t)(t0 >> 16));
                        A[0][2] = e4m3x2_to_f16x2((uint16_t)(t1 & 0xffff));
                        A[0][3] = e4m3x2_to_f16x2((uint16_t)(t1 >> 16));
                        A[1][0] = e4m3x2_to_f16x2((uint16_t)(t2 & 0xffff));
                        A[1][1] = e4m3x2_to_f16x2((uint16_t)(t2 >> 16));
                        A[1][2] = e4m3x2_to_f16x2((uint16_t)(t3 & 0xffff));
                        A[1][3] = e4m3x2_to_f16x2((uint16_t)(t3 >> 16));
#pragma unroll
                        for (int hs = 0; hs < 2; ++hs)
#pragma unroll
                            for (int n = 0; n < NT; ++n) {
                                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                                mma_f16(acc, A[hs][0], A[hs][1], A[hs][2], A[hs][3], pb[sub][n][0], pb[sub][n][1]);
                                float *od = o[2 * jg + hs][n];
                                od[0] = fmaf(acc[0], vsc, od[0]);
                                od[1] = fmaf(acc[1], vsc, od[1]);
                                od[2] = fmaf(acc[2], vsc, od[2]);
                                od[3] = fmaf(acc[3], vsc, od[3]);
                            }
                    }
                }
            }
        }
        // Release the stage (all reads of it are done); an item's last stage
        // holding the epilogue scratch is released after the epilogue.
        const int m_kvh = mt.kvh, m_s = mt.s, m_nsplit = mt.nsplit, m_hg = mt.hg, m_nrows = mt.nrows;
        __syncwarp();
        if (lane == 0 && !(scr_in_stage && (flags & kFlagLast))) mbar_arrive(smem_u32(&empty_bar[st]));
        if (++st == NST) { st = 0; ph ^= 1u; }
        if (!(flags & kFlagLast)) continue;
        // the stage just consumed: st - 1 (mod NST)
        float *scratch = scr_in_stage ? reinterpret_cast<float *>(stages + (size_t)((st == 0 ? NST : st) - 1) * Sh::STAGE)
                                      : scr_own;
        // every warp's reads of that stage are done before it is written
        if (scr_in_stage) named_bar_sync(1, NC * 32);

        // ========================================================== item epilogue
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                float v = lrow[n][r];
                v += shfl_xor(v, 4);
                v += shfl_xor(v, 8);
                v += shfl_xor(v, 16);
                lrow[n][r] = v;
            }
        constexpr int NSLOT = Sh::NSLOT;
        // Warp state (o, m, l) into epilogue slot `slot`.
        auto put_state = [&](int slot) {
            float *so = scratch + slot * QROWS * SS;
#pragma unroll
            for (int mi = 0; mi < MT; ++mi) {
                const int d0 = FP8 ? 16 * mi + 2 * g : 16 * mi + g;
                const int d1 = FP8 ? d0 + 1 : d0 + 8;
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const int h0 = n * 8 + 2 * c, h1 = h0 + 1;
                    so[h0 * SS + d0] = o[mi][n][0];
                    so[h1 * SS + d0] = o[mi][n][1];
                    so[h0 * SS + d1] = o[mi][n][2];
                    so[h1 * SS + d1] = o[mi][n][3];
                }
            }
            if (g == 0) {
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const int h0 = n * 8 + 2 * c;
                    scr_m[slot * QROWS + h0] = mrow[n][0];
                    scr_m[slot * QROWS + h0 + 1] = mrow[n][1];
                    scr_l[slot * QROWS + h0] = lrow[n][0];
                    scr_l[slot * QROWS + h0 + 1] = lrow[n][1];
                }
            }
        };
        if constexpr (NSLOT < NC) {
            // Warp w + NSLOT hands its state to warp w, which merges it into
            // its own registers (same rescale as the final combine).
            if (warp >= NSLOT) put_state(warp - NSLOT);
            named_bar_sync(1, NC * 32);
            if (warp < NSLOT) {
                const float *so = scratch + warp * QROWS * SS;
                float wo[NT][2], wp[NT][2];
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int h = n * 8 + 2 * c + r;
                        const float pm = scr_m[warp * QROWS + h], pl = scr_l[warp * QROWS + h];
                        const float mn = fmaxf(mrow[n][r], pm);
                        wo[n][r] = (mn == -INFINITY) ? 0.f : ex2(mrow[n][r] - mn);
                        wp[n][r] = (mn == -INFINITY) ? 0.f : ex2(pm - mn);
                        lrow[n][r] = wo[n][r] * lrow[n][r] + wp[n][r] * pl;
                        mrow[n][r] = mn;
                    }
#pragma unroll
                for (int mi = 0; mi < MT; ++mi) {
                    const int d0 = FP8 ? 16 * mi + 2 * g : 16 * mi + g;
                    const int d1 = FP8 ? d0 + 1 : d0 + 8;
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        const int h0 = n * 8 + 2 * c, h1 = h0 + 1;
                        o[mi][n][0] = wo[n][0] * o[mi][n][0] + wp[n][0] * so[h0 * SS + d0];
                        o[mi][n][1] = wo[n][1] * o[mi][n][1] + wp[n][1] * so[h1 * SS + d0];
                        o[mi][n][2] = wo[n][0] * o[mi][n][2] + wp[n][0] * so[h0 * SS + d1];
                        o[mi][n][3] = wo[n][1] * o[mi][n][3] + wp[n][1] * so[h1 * SS + d1];
                    }
                }
                __syncwarp();  // every lane has read the slot before it is rewritten
                put_state(warp);
            }
        } else {
            put_state(warp);
        }
        named_bar_sync(1, NC * 32);
        const int tid = warp * 32 + lane;
        const int G = m_nrows;  // q rows of this item
        // Per head: combined max, the warps' weights (in place of their max)
        // and the combined denominator; then the D outputs in float4 groups.
        if (tid < G) {
            const int h = tid;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NSLOT; ++w) M = fmaxf(M, scr_m[w * QROWS + h]);
            float Ls = 0.f;
#pragma unroll
            for (int w = 0; w < NSLOT; ++w) {
                const float a = (M == -INFINITY) ? 0.f : ex2(scr_m[w * QROWS + h] - M);
                scr_m[w * QROWS + h] = a;
                Ls += a * scr_l[w * QROWS + h];
            }
            const bool empty = !(Ls > 0.f);
            const size_t row = q_row(p, mb, m_kvh, m_hg, h, QROWS);
            if (m_nsplit == 1) {
                scr_inv[h] = empty ? 0.f : 1.f / Ls;
                if (p.lse) p.lse[row] = empty ? -INFINITY : (M + __log2f(Ls)) * kLn2;
            } else {
                scr_inv[h] = 1.f;
                p.part_m[row * p.S + m_s] = (M == -INFINITY) ? -INFINITY : M * kLn2;
                p.part_d[row * p.S + m_s] = Ls;
            }
        }
        named_bar_sync(1, NC * 32);
        for (int idx = tid; idx < G * (D / 4); idx += NC * 32) {
            const int h = idx / (D / 4), d = (idx - h * (D / 4)) * 4;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < NSLOT; ++w) {
                const float a = scr_m[w * QROWS + h];
                const float4 v = *reinterpret_cast<const float4 *>(scratch + (w * QROWS + h) * SS + d);
                acc.x = fmaf(a, v.x, acc.x);
                acc.y = fmaf(a, v.y, acc.y);
                acc.z = fmaf(a, v.z, acc.z);
                acc.w = fmaf(a, v.w, acc.w);
            }
            const size_t row = q_row(p, mb, m_kvh, m_hg, h, QROWS);
            if (m_nsplit == 1) {
                const float inv = scr_inv[h];
                store_out4(p.out, row * D + d, acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv, p.out_dtype);
            } else {
                *reinterpret_cast<float4 *>(p.part_o + (row * p.S + m_s) * D + d) = acc;
            }
        }
        if (m_nsplit > 1 && p.fuse_merge) {
            // Publish the partial state: the barrier orders every consumer
            // thread's stores before thread 0's GPU-scope counter update,
            // whose release makes them visible to the other CTAs; its
            // acquire makes theirs visible to the CTA that sees the last
            // count (the barrier below passes that on to its threads).
            named_bar_sync(1, NC * 32);
            if (tid == 0) {
                const int prev = atom_add_acq_rel_gpu(p.merge_ctr + ((size_t)mb * p.Hkv + m_kvh) * p.nhg + m_hg, 1);
                *scr_flag = (prev == m_nsplit - 1);
            }
            named_bar_sync(1, NC * 32);
            if (*scr_flag) {
                merge_group<NC, FP8 ? 8 : 16>(p, mb, m_kvh, m_hg, m_nrows, QROWS, m_nsplit, scratch, warp, lane, D);
                if (tid == 0) atomicExch(p.merge_ctr + ((size_t)mb * p.Hkv + m_kvh) * p.nhg + m_hg, 0);
            }
        }
        // 16-bit K/V: the item's state and q fragments are spent; set them
        // here (the next item's first stage sets them again) so that they
        // are not live across the epilogue and the merge (fewer registers;
        // measured faster for 16-bit K/V, not for E4M3).
        if constexpr (!FP8)
#pragma unroll
        for (int n = 0; n < NT; ++n) {
#pragma unroll
            for (int mi = 0; mi < MT; ++mi)
#pragma unroll
                for (int r = 0; r < 4; ++r) o[mi][n][r] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) qf[kk][n][0] = qf[kk][n][1] = 0u;
            mrow[n][0] = mrow[n][1] = -INFINITY;
            lrow[n][0] = lrow[n][1] = 0.f;
            qd[n][0] = qd[n][1] = 1.f;
        }
        // The scratch stage goes back to the producer: this thread's writes
        // to it are ordered before the copies that refill it.
        if (scr_in_stage) fence_proxy_async_shared();
        named_bar_sync(1, NC * 32);
        if (scr_in_stage && lane == 0) mbar_arrive(smem_u32(&empty_bar[(st == 0 ? NST : st) - 1]));
    }
}

// Dynamic shared memory of this instance with `stages` stages and B KV rows;
// 0 if the epilogue scratch is asked to live in a stage and cannot.
template <int KV, int D, int NT, int NC, int SUBT, bool QBF16>
size_t decode_smem_for(int stages, int B, bool scr_in_stage) {
    using Sh = DecodeShape<KV, D, NT, NC, SUBT>;
    if (scr_in_stage && !Sh::SCR_STAGE_OK) return 0;
    size_t n = 1024;  // alignment slack
    n += (size_t)stages * Sh::STAGE;
    n += align_up(scr_in_stage ? Sh::SCRATCH_SMALL : Sh::SCRATCH, 128);
    n += (size_t)stages * sizeof(StageMeta);
    n += (size_t)stages * 16;
    n += (size_t)((B + 31) / 32 + 1 + B + kOrderBuckets) * 4 + (size_t)align_up(2 * B, 4);  // dispatch tables
    return n;
}

// Resident CTAs per SM of this instance with `smem` bytes of dynamic shared
// memory (registers, threads and shared memory all counted).
template <int KV, int D, int NT, int NC, int SUBT, bool QBF16>
cudaError_t occupancy_t(size_t smem, int *blocks) {
    auto kern = fd_split_kv_decode_kernel<KV, D, NT, NC, SUBT, QBF16, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, kern, DecodeShape<KV, D, NT, NC, SUBT>::THREADS, smem);
}

template <int KV, int D, int NT, int NC, int SUBT, bool QBF16, bool CAUSAL = false, bool SCR = false>
cudaError_t launch_decode_t(const DecodeParams &dp, const CUtensorMap &tmk, const CUtensorMap &tmv, int grid,
                            size_t smem, cudaStream_t stream) {
    auto kern = fd_split_kv_decode_kernel<KV, D, NT, NC, SUBT, QBF16, CAUSAL, SCR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // Programmatic dependent launch: the kernel may begin its prologue while
    // the previous grid in the stream drains; it waits (griddepcontrol.wait)
    // before reading any global input.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(DecodeShape<KV, D, NT, NC, SUBT>::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, dp, tmk, tmv);
}

}  // namespace fd
