// fd_internal.h -- parameters shared between the C ABI layer (fd_api.cu) and
// the kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fd_api.h"

namespace fd {

// Consumer warps per CTA, tokens per consumer warp per stage, and the
// pipeline tile (tokens per stage) that follows from them.
constexpr int kTokensPerWarp = 16;
constexpr int kMaxConsumerWarps = 8;
constexpr int kMaxBoxesPerTile = 8;  // tile / gcd(page_size, tile) <= 128 / 16
constexpr int kMaxSplits = 512;      // partial slots per (b, hq)
constexpr int kMaxBatch = 8192;
constexpr int kMinChunkTokens = 256; // below this a sequence is not split

enum KvKind { KV_F16 = 0, KV_BF16 = 1, KV_E4M3 = 2 };

struct DecodeParams {
    const void *q;             // [B, Hq, D]
    const int32_t *block_table;
    const int32_t *seq_lens;
    const int32_t *batch_idx;  // [B] cache row of q row b, or null (row b)
    const int32_t *leftpad;    // [cache rows] first attended token, or null (0)
    int cache_rows;            // rows of block_table / seq_lens / leftpad
    const float *k_scale;      // [num_pages, Hkv] or null
    const float *v_scale;
    void *out;                 // [B, Hq, D]
    float *lse;                // [B, Hq] or null
    float *part_o;             // [B, Hq, S, D]
    float *part_m;             // [B, Hq, S]
    float *part_d;             // [B, Hq, S]
    int *merge_ctr;            // [B, Hkv]
    int *work_ctr;             // 1
    int *done_ctr;             // 1
    int *status;               // null allowed
    int B, Hq, Hkv, G;
    // Query rows of one work item: the G*fold rows that read KV head kvh of
    // KV row bkv (fold > 1: several q sequences share one KV row), sliced
    // into nhg sub-groups of at most 8*NT rows.  Row i of the group is q
    // sequence bkv*fold + i/G, head kvh*G + i%G.
    int fold, nhg, Bkv;
    int page_size, max_blocks, num_pages;
    int S;                     // partial slots per (b, hq)
    int chunk;                 // tokens per split
    int cap;                   // S * chunk
    int boxr;                  // token rows per TMA box: gcd(page_size, tile)
    int out_dtype;             // fd_dtype
    int fuse_merge;
    int stages;
    int scr_in_stage;          // epilogue scratch in the item's last stage (16-bit K/V)
    float scale_log2;          // log2(e) / sqrt(D)
    uint64_t timeout_ns;       // limit of every device-side wait
    uint64_t stall_ns;         // test hook (0 = off): idle time of stall_role
    int stall_role;            // 1: producer before its first load; 2: consumers before the first release
    int qn;                    // query tokens per KV row, causal among them (1: one-token decode)
};

struct MergeParams {
    const float *part_o, *part_m, *part_d;
    void *out;
    float *lse;
    const int32_t *seq_lens;   // non-null: per-sequence split counts from lengths
    const int32_t *batch_idx;  // as in DecodeParams (with seq_lens only)
    const int32_t *leftpad;
    int cache_rows;
    int B, Hq, S, D, chunk, cap;
    int fold;                  // q sequences per KV row
    int out_dtype;
};

struct AppendParams {
    const void *k_new, *v_new;
    void *k_pages, *v_pages;
    const float *k_scale, *v_scale;
    const int32_t *block_table, *seq_lens;
    int *status;
    int B, Hkv, D, page_size, max_blocks, num_pages;
    int kv_kind;               // KvKind
    int new_is_bf16;           // for E4M3 caches: input dtype bf16 (1) or f16 (0)
    // Rotary embedding (cos == null: none): tables [max_pos, rotary_dim/2].
    const float *cos, *sin;
    int rotary_dim, max_pos, interleaved;
    void *q_inout;             // [B, Hq, D] rotated in place, or null
    int Hq;
    int q_is_bf16;
};

// Kernel configuration chosen at plan time.
struct KernelShape {
    int consumer_warps;  // 4 or 8
    int subtiles;        // 16-token sub-tiles per consumer warp per stage: 1 or 2
    int tile;            // tokens per stage = consumer_warps * subtiles * 16
    int nt;              // 8-wide head tiles: 1 (G <= 8) or 2 (G <= 16)
};

// tile_tokens: 64, 128 or 256 (0 = default for the K/V type); fold: q
// sequences per KV row (1 = ordinary decode); ctas_per_sm: persistent CTAs
// per SM (E4M3 128-token stages with two or more CTAs per SM take 4 consumer
// warps x 2 sub-tiles, which fit two to an SM).
KernelShape kernel_shape(const fd_problem &p, int tile_tokens, int fold, int ctas_per_sm);
// Dynamic shared memory of the decode kernel of this shape with `stages`
// stages (p.B = KV rows: the dispatch tables); scr_in_stage: the epilogue
// scratch in the item's last stage (16-bit K/V; 0 where a stage cannot hold it).
size_t decode_smem_bytes(const fd_problem &p, const KernelShape &ks, int stages, bool scr_in_stage);
// Resident CTAs per SM of the decode kernel of this shape with smem bytes of
// dynamic shared memory (needs a device).
cudaError_t decode_occupancy(const fd_problem &p, const KernelShape &ks, size_t smem, int *blocks);

cudaError_t launch_decode(const fd_problem &p, const KernelShape &ks, const DecodeParams &dp,
                          const CUtensorMap &tmk, const CUtensorMap &tmv, int grid, size_t smem,
                          cudaStream_t stream);
cudaError_t launch_merge(const MergeParams &mp, cudaStream_t stream);
cudaError_t launch_append(const AppendParams &ap, cudaStream_t stream);
cudaError_t launch_merge_two(const float *oa, const float *la, const float *ob, const float *lb, int rows, int D,
                             int out_dtype, void *out, float *lse, cudaStream_t stream);

}  // namespace fd
