/*
 * fd_api.h -- C ABI of libfd: paged, GQA-shared, split-KV decode attention
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation (one query token per sequence against its cached keys and
 * values) is the decode step described on these pages:
 *   [P1] "FlashDecoding 与 FlashInfer 深度解析" (tbr8.org), §2.1: split the KV
 *        sequence into contiguous chunks, compute per chunk the scores
 *        q k^T / sqrt(d), a local softmax, the weighted sum of V and the local
 *        max and sum, then merge the chunks exactly.
 *   [P2] lpnh.cn/news/1601758, "FlashDecoding 核心原理": stage one writes the
 *        partial state (unnormalised O_i, max m_i, denominator d_i); stage two
 *        merges with m = max m_i, alpha_i = exp(m_i - m), d = sum alpha_i d_i,
 *        O = sum alpha_i O_i / d; "进阶突破": a cost model picks the split count
 *        from batch, heads, length and SM count, and short sequences are not
 *        split; map and reduce may be fused into one kernel through atomics.
 *   [P3] "Inference Cookbook" (FlashAttention): §4.2 paged pools
 *        [num_pages, page_size, Hkv, D] and an int32 block table with -1 in
 *        unused entries; §3.2-3.3 new K/V are written into the cache and the
 *        cached lengths are not advanced by the call; §3.5 the softmax LSE per
 *        (batch, head); §6 split-KV with num_splits (0 = automatic) and its
 *        heuristic; §7 FP8 (E4M3) KV with fp32 descale factors.
 *   [P4] "FlashAttention 與 FlashInfer:兩大 GPU 注意力後端": page (block) sizes
 *        must be multiples of 16.
 *
 * Conventions for every entry point:
 *  - All pointers except seq_lens_host (fd_plan) are DEVICE pointers on the
 *    current CUDA device.  The library never allocates, frees or copies
 *    device memory; every buffer belongs to the caller.
 *  - Calls are asynchronous on the given stream (cudaStream_t passed as a
 *    void*; NULL = the legacy default stream) and never synchronise.
 *  - Errors found on the host are returned before anything is launched.
 *    Errors only the device can see (a block-table entry out of range inside
 *    a live range, a length beyond the plan's capacity, a wait that ran past
 *    its time limit) are OR-ed into *status_dev as FD_DEV_* bits when
 *    status_dev is not NULL; the kernel skips the offending access and never
 *    traps.  fd_status_from_device() maps a status word to an fd_status.
 *  - Nothing is thrown across the ABI.
 */
#ifndef FD_API_H
#define FD_API_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FD_API_VERSION 5

typedef enum {
    FD_OK = 0,
    FD_ERR_INVALID_ARG = 1,         /* null pointer, bad size, bad alignment          */
    FD_ERR_UNSUPPORTED = 2,         /* a valid problem this library does not serve    */
    FD_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < plan->workspace_bytes        */
    FD_ERR_BAD_PAGE = 4,            /* device saw a block-table entry out of range    */
    FD_ERR_CUDA = 5,                /* a CUDA runtime/driver call failed              */
    FD_ERR_CAPACITY = 6,            /* device saw seq_lens[b] above the plan capacity */
    FD_ERR_TIMEOUT = 7              /* a device-side wait hit its time limit          */
} fd_status;

/* Bits of the device status word. */
#define FD_DEV_BAD_PAGE 0x1
#define FD_DEV_CAPACITY 0x2
#define FD_DEV_TIMEOUT  0x4

typedef enum { FD_F16 = 0, FD_BF16 = 1, FD_E4M3 = 2, FD_F32 = 3 } fd_dtype;

/* Shapes and types of one decode problem.
 *   q            [B, Hq, D]                      q_dtype (FD_F16 or FD_BF16)
 *   k/v pages    [num_pages, page_size, Hkv, D]  kv_dtype; row-major, D fastest
 *   block_table  int32 [B, max_blocks_per_seq], entry j of row b is the page
 *                holding tokens [j*page_size, (j+1)*page_size) of sequence b
 *   seq_lens     int32 [B]
 *   out          [B, Hq, D]                      out_dtype (q_dtype or FD_F32)
 *   lse          fp32 [B, Hq], natural log
 * Constraints: Hq % Hkv == 0 (the query heads of KV head kvh are the
 * contiguous group hq / (Hq / Hkv) == kvh; groups larger than 16 heads are
 * split into 16-head work items); D in {64, 128};
 * page_size % 16 == 0 [P4]; kv_dtype FD_E4M3 requires q_dtype FD_BF16 or
 * FD_F16, otherwise kv_dtype == q_dtype; 1 <= B <= 8192. */
typedef struct {
    int B, Hq, Hkv, D;
    int page_size;
    int max_blocks_per_seq;
    int num_pages;
    fd_dtype q_dtype, kv_dtype, out_dtype;
} fd_problem;

typedef struct {
    int num_splits;     /* 0 = cost model [P2 进阶突破, P3 §6.3]; >0 forces the
                           number of contiguous chunks of the longest sequence   */
    int num_sms;        /* 0 = query the device; >0 overrides (planning only)   */
    int fuse_merge;     /* 1 = the CTA that finishes the last chunk of a (b, kvh)
                           merges in place (default); 0 = a separate merge kernel */
    int max_seq_len;    /* 0 = max of seq_lens_host; otherwise the capacity the
                           plan must cover when it is reused as lengths grow    */
    int ctas_per_sm;    /* 0 = automatic; persistent CTAs per SM                */
    int split_margin_pct; /* 0 = default (2): pick the fewest splits whose
                           estimated time is within this many percent of the
                           best; 18 reproduces the cookbook's "smallest split
                           count reaching 85% of the best efficiency" [P3 §6.3] */
    int tile_tokens;    /* tokens per pipeline stage: 64, 128, or 256 (E4M3 pools
                           with page_size % 32 == 0); 0 = default: 256 for E4M3
                           when pages allow and 3 stages fit, else 128 */
    int shared_kv;      /* 1: every q sequence attends the same KV row (one
                           block-table row, seq_lens[0]; e.g. a shared prefix):
                           the B*G q rows of each KV head are packed 16 to a
                           work item so each K/V tile feeds 16 rows; plan with
                           seq_lens_host[0] = the shared length */
    int timeout_us;     /* limit of every device-side wait, in microseconds;
                           0 = 2 s.  A wait that runs past it sets
                           FD_DEV_TIMEOUT, and the kernel drains its copies in
                           flight and returns (no trap, no hang)  */
    int debug_stall_us; /* TEST HOOK, 0 = off: with debug_stall_role 1 the
                           producer warp of every CTA idles this long before
                           its first load; with 2 the consumer warps idle this
                           long before releasing their first stage.  Longer
                           than timeout_us, it makes the other side's waits
                           run out, exercising the timeout path.  <= 1 s.   */
    int debug_stall_role; /* 0, 1 (producer) or 2 (consumers)                */
    int q_len;          /* query tokens per sequence, 0 or 1 = one (decode).
                           q_len > 1 (at most 64): the last q_len cached tokens
                           of every sequence are its queries and token i of
                           them attends the cached tokens
                           [0, seq_lens[b] - q_len + i + 1) -- causal attention
                           aligned to the end of the cache, after the new
                           tokens' K/V were appended ("Inference Cookbook"
                           §3.2-3.3, causal=True; [P1] §3.1, the append mode).
                           q and out are [B, q_len, Hq, D], lse [B, q_len, Hq];
                           problem->B counts sequences; not with shared_kv or
                           the fd_decode_extras indirections               */
} fd_plan_options;

/* A plan: plain data in host memory, owned by the caller, reusable for any
 * number of calls while 0 <= seq_lens[b] <= capacity_tokens on the device. */
typedef struct {
    fd_problem problem;
    int num_splits;       /* partial-state slots per (b, hq)                     */
    int chunk_tokens;     /* tokens per split (a multiple of tile_tokens)        */
    int tile_tokens;      /* tokens per pipeline stage                           */
    int capacity_tokens;  /* num_splits * chunk_tokens                           */
    int grid_ctas;        /* persistent CTAs launched                            */
    int num_sms;
    int fuse_merge;
    int stages;           /* shared-memory pipeline depth                        */
    int smem_bytes;       /* dynamic shared memory per CTA                       */
    size_t workspace_bytes;
    size_t ws_partial_o;  /* byte offsets inside the workspace                   */
    size_t ws_partial_md;
    size_t ws_counters;
    long long work_items_hint; /* items for the host lengths (information)      */
    int kv_rows;          /* block-table / seq_lens rows the call reads          */
    int row_fold;         /* q sequences per KV row (1, or B with shared_kv)     */
    int head_subgroups;   /* work items per (KV row, split, KV head)             */
    int ctas_per_sm;      /* persistent CTAs per SM the shape was chosen for     */
    int timeout_us;       /* device wait limit (0 = 2 s), from the options       */
    int debug_stall_us;   /* test hook copied from the options (0 = off)         */
    int debug_stall_role;
    int q_len;            /* query tokens per sequence (1 = decode); problem.B
                             then counts query rows, B * q_len               */
    int scratch_in_stage; /* 1: the item epilogue's scratch lives in the item's
                             last pipeline stage (16-bit K/V, where that makes
                             room for another stage); 0: a region of its own */
    int reserved[2];
} fd_plan_t;

/* Plan a decode call [P1 §2.1 step 1; P2 进阶突破; P3 §6.3, §8.2].
 *   problem        shapes/types (copied into the plan)
 *   seq_lens_host  HOST int32 [B]: the lengths the split count is chosen for
 *   options        may be NULL (all defaults)
 *   plan           out: filled on FD_OK
 * The split count follows the pages' rules: no split when the sequences are
 * short or when B*Hkv already fills the SMs with equal work; otherwise the
 * smallest split count whose estimated SM efficiency is within a margin of
 * the best.  The workspace the call needs is plan->workspace_bytes; it must be
 * zero-filled once after allocation (the kernels leave their counters at zero
 * when they finish), and again after any call reported an FD_DEV_* error.
 * Returns FD_ERR_INVALID_ARG / FD_ERR_UNSUPPORTED on bad problems, FD_ERR_CUDA
 * if the device cannot be queried. */
fd_status fd_plan(const fd_problem *problem, const int32_t *seq_lens_host,
                  const fd_plan_options *options, fd_plan_t *plan);

/* One decode step [P1 §2.1; P2 stages one and two; P3 §3.5, §4, §6, §7].
 *   q, k_pages, v_pages  device, 16-byte aligned, layouts as in fd_problem
 *                        (with plan->q_len > 1: q and out [B, q_len, Hq, D],
 *                        lse [B, q_len, Hq], the q_len causal query tokens of
 *                        each sequence; see fd_plan_options.q_len)
 *   k_scale, v_scale     device fp32 [num_pages, Hkv] for FD_E4M3 (value =
 *                        e4m3 code * scale); must be NULL otherwise
 *   block_table, seq_lens device int32; the call attends over tokens
 *                        [0, seq_lens[b]) of every sequence
 *   out                  device [B, Hq, D] in problem.out_dtype
 *   lse                  device fp32 [B, Hq] or NULL
 *   workspace            device, 256-byte aligned, >= plan->workspace_bytes,
 *                        zero-filled before its first use; one workspace per
 *                        call in flight (calls sharing one must not overlap)
 *   status_dev           device int32 or NULL; FD_DEV_* bits are OR-ed in
 *   stream               cudaStream_t
 * A sequence of length 0 gives out = 0 and lse = -inf.  Output rounding is
 * round-to-nearest-even from fp32. */
fd_status fd_decode_paged(const fd_plan_t *plan, const void *q, const void *k_pages,
                          const void *v_pages, const float *k_scale, const float *v_scale,
                          const int32_t *block_table, const int32_t *seq_lens, void *out,
                          float *lse, void *workspace, size_t workspace_bytes,
                          int32_t *status_dev, void *stream);

/* Optional indirections of a decode call ("Inference Cookbook" §5.2
 * cache_batch_idx, §5.3 cache_leftpad).  All device pointers, NULL = off.
 *   cache_batch_idx  int32 [B]: q row b reads cache row cache_batch_idx[b]
 *                    (its block-table row, seq_lens entry and leftpad entry);
 *                    out/lse stay indexed by q row.  Lets the active subset
 *                    of a larger batch decode without copying its metadata.
 *   cache_leftpad    int32 [cache rows]: the first cached token of the row;
 *                    q row b attends tokens [leftpad[cb], seq_lens[cb]).
 *   cache_rows       rows of block_table / seq_lens / cache_leftpad when
 *                    cache_batch_idx is set (an index outside [0, cache_rows)
 *                    sets FD_DEV_BAD_PAGE and that row gets out = 0, lse = -inf).
 * Plan such a call with the attended lengths seq_lens[cb] - leftpad[cb] of
 * the q rows as seq_lens_host; a leftpad outside [0, seq_len] sets
 * FD_DEV_CAPACITY. */
typedef struct {
    const int32_t *cache_batch_idx;
    const int32_t *cache_leftpad;
    int cache_rows;
} fd_decode_extras;

/* fd_decode_paged with the indirections of fd_decode_extras (NULL extras is
 * the plain call).  Same arguments, errors and guarantees otherwise. */
fd_status fd_decode_paged_ex(const fd_plan_t *plan, const void *q, const void *k_pages,
                             const void *v_pages, const float *k_scale, const float *v_scale,
                             const int32_t *block_table, const int32_t *seq_lens,
                             const fd_decode_extras *extras, void *out, float *lse,
                             void *workspace, size_t workspace_bytes, int32_t *status_dev,
                             void *stream);

/* Merge S partial states per (b, hq) into the output [P1 §2.1 step 3 merge;
 * P2 stage two].
 *   o_part   device fp32 [B, Hq, S, D]: unnormalised sum_t exp(s_t - m) v_t
 *   m        device fp32 [B, Hq, S]: max score of the chunk (natural units,
 *            score = q.k/sqrt(D)); -inf marks an empty chunk
 *   d        device fp32 [B, Hq, S]: sum_t exp(s_t - m); 0 for an empty chunk
 *   out      device [B, Hq, D] in out_dtype (FD_F16, FD_BF16 or FD_F32)
 *   lse      device fp32 [B, Hq] or NULL
 * All-empty rows give out = 0 and lse = -inf.  1 <= S <= 4096, D <= 256. */
fd_status fd_merge_states(const float *o_part, const float *m, const float *d, int B, int Hq,
                          int S, int D, fd_dtype out_dtype, void *out, float *lse,
                          void *stream);

/* Merge two normalised attention states of the same queries over disjoint
 * token sets (cascade / shared-prefix decode: a state over the shared prefix
 * and one over each sequence's own suffix) [P2 stage two with d = 1:
 * m = max(lse_a, lse_b), w = exp(lse - m), out = (w_a out_a + w_b out_b) /
 * (w_a + w_b), lse = m + ln(w_a + w_b)].
 *   out_a, out_b  device fp32 [rows, D], 16-byte aligned; lse_a, lse_b fp32 [rows]
 *   out           device [rows, D] in out_dtype; lse fp32 [rows] or NULL
 * An empty state has lse = -inf; both empty give out = 0, lse = -inf.
 * D % 4 == 0. */
fd_status fd_merge_two(const float *out_a, const float *lse_a, const float *out_b,
                       const float *lse_b, int rows, int D, fd_dtype out_dtype, void *out,
                       float *lse, void *stream);

/* Append one token per sequence [P3 §3.2-3.3, §4.2].
 *   k_new, v_new  device [B, Hkv, D] in problem.q_dtype for an FD_E4M3 cache
 *                 (quantised as code = e4m3_rne_satfinite(x / scale[page, kvh]),
 *                 the division in fp32), otherwise in kv_dtype (bits copied)
 *   k/v_pages     device pools, modified in place at position seq_lens[b]:
 *                 page block_table[b][seq_lens[b] / page_size], slot
 *                 seq_lens[b] % page_size
 *   k/v_scale     device fp32 [num_pages, Hkv] for FD_E4M3, else NULL
 *   status_dev    device int32 or NULL: FD_DEV_BAD_PAGE when the target page
 *                 is out of range (that sequence is skipped)
 * seq_lens is NOT advanced; the caller adds 1 after the call. */
fd_status fd_append_kv(const fd_problem *problem, const void *k_new, const void *v_new,
                       void *k_pages, void *v_pages, const float *k_scale,
                       const float *v_scale, const int32_t *block_table,
                       const int32_t *seq_lens, int32_t *status_dev, void *stream);

/* Size of the library-owned workspace used by fd_decode_paged_noalloc: 16 MiB
 * per GPU that loads the library, held until the process exits. */
#define FD_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* fd_decode_paged without a caller-provided workspace.  (The pages have no
 * counterpart: this is a convenience of this library.)
 *
 * Who needs it: callers that cannot allocate device memory at the point of
 * the call -- code hosted by an engine or plugin interface that owns every
 * device allocation and hands out only input and output pointers, real-time
 * loops that must not take cudaMalloc's device-wide synchronisation, and
 * plain C callers that have no device allocator at hand.
 *
 * The workspace is a fixed buffer of FD_NOALLOC_SCRATCH_BYTES inside libfd,
 * one per device.  Arguments are those of fd_decode_paged minus the
 * workspace.  The caller still owns q, the pools, the block table, seq_lens,
 * out, lse and status_dev.
 *  - Returns FD_ERR_WORKSPACE_TOO_SMALL, with nothing launched, when
 *    plan->workspace_bytes exceeds FD_NOALLOC_SCRATCH_BYTES (plan with fewer
 *    splits, or call fd_decode_paged with a workspace of your own).
 *  - The first call on each device looks up the device address of that
 *    device's buffer; make that first call before any stream capture.
 *  - Every call on a device uses the same buffer, which keeps what the last
 *    call left in it; each call clears the buffer's counters with an
 *    asynchronous memset on `stream` before the decode launch.  Calls whose
 *    GPU work overlaps (other streams, other threads) race on the buffer and
 *    give wrong results: order them, e.g. on one stream.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
fd_status fd_decode_paged_noalloc(const fd_plan_t *plan, const void *q, const void *k_pages,
                                  const void *v_pages, const float *k_scale,
                                  const float *v_scale, const int32_t *block_table,
                                  const int32_t *seq_lens, void *out, float *lse,
                                  int32_t *status_dev, void *stream);

/* fd_append_kv with rotary position embedding fused in ("Inference Cookbook"
 * §3.4: the new key is rotated before it is written, so the cache holds
 * rotated keys; the query is rotated at the same position).
 *   rotary_cos, rotary_sin  device fp32 [max_pos, rotary_dim / 2]
 *   rotary_dim              even, <= D: the first rotary_dim elements rotate
 *   interleaved             0: pairs (i, i + rotary_dim/2) (GPT-NeoX style);
 *                           1: pairs (2i, 2i+1)
 *   q_inout                 device [B, Hq, D] in q_dtype rotated in place, or NULL
 * Position = seq_lens[b].  Pair (x1, x2) at angle index i becomes
 * ((x1*cos) - (x2*sin), (x2*cos) + (x1*sin)), each product and sum rounded to
 * fp32, then rounded to the storage type (RNE; E4M3 caches quantise the
 * rotated value as fd_append_kv does).  V is copied unrotated.  A sequence
 * whose position is >= max_pos is skipped and sets FD_DEV_CAPACITY.
 * seq_lens is not advanced. */
fd_status fd_append_kv_rotary(const fd_problem *problem, const void *k_new, const void *v_new,
                              void *k_pages, void *v_pages, const float *k_scale,
                              const float *v_scale, const int32_t *block_table,
                              const int32_t *seq_lens, const float *rotary_cos,
                              const float *rotary_sin, int rotary_dim, int max_pos,
                              int interleaved, void *q_inout, int32_t *status_dev, void *stream);

/* One decode step from and to host memory.  (The pages have no counterpart:
 * a convenience of this library for serving loops whose per-step inputs are
 * prepared on the host.)
 *
 * The step's inputs live in one host block and its results in another, so a
 * step is one host-to-device copy and the decode (fd_decode_paged), plus one
 * device-to-host copy unless the output block is mapped (below), all queued
 * on `stream`:
 *   input block   q [B, Hq, D] (q_dtype) at q_offset,
 *                 block_table int32 [kv_rows, max_blocks_per_seq] at
 *                 block_table_offset, seq_lens int32 [kv_rows] at
 *                 seq_lens_offset; in_bytes in all
 *   output block  out [B, Hq, D] (out_dtype) at out_offset, lse fp32 [B, Hq]
 *                 at lse_offset; out_bytes in all
 * Offsets are multiples of 256 bytes; kv_rows is the plan's (B unless the
 * plan folds sequences onto shared KV rows). */
typedef struct {
    size_t q_offset, block_table_offset, seq_lens_offset, in_bytes;
    size_t out_offset, lse_offset, out_bytes;
} fd_host_io_layout;

/* Fill *layout for plan.  Returns FD_ERR_INVALID_ARG on NULL arguments. */
fd_status fd_host_io_layout_for(const fd_plan_t *plan, fd_host_io_layout *layout);

/*   host_in    host input block (in_bytes), read by the copy; page-locked
 *              (cudaHostAlloc / pinned) memory keeps the call asynchronous
 *   dev_in     device buffer of in_bytes, 256-byte aligned, overwritten
 *   dev_out    device buffer of out_bytes, 256-byte aligned, overwritten
 *   host_out   host output block (out_bytes), valid once `stream` has been
 *              synchronised.  Page-locked memory mapped for the device (any
 *              cudaHostAlloc / pinned block under unified addressing) is
 *              written by the decode kernel itself and no copy is queued;
 *              other host memory is filled by a copy from dev_out
 *   other arguments as fd_decode_paged (pools, scales, workspace, status_dev).
 * Errors as fd_decode_paged; FD_ERR_CUDA when a copy cannot be queued.  The
 * caller owns all four blocks and must not change host_in or read host_out
 * until the stream has passed the call. */
fd_status fd_decode_paged_host(const fd_plan_t *plan, const void *host_in, void *dev_in,
                               const void *k_pages, const void *v_pages, const float *k_scale,
                               const float *v_scale, void *dev_out, void *host_out,
                               void *workspace, size_t workspace_bytes, int32_t *status_dev,
                               void *stream);

/* The parts of fd_decode_paged_host, for callers that queue them on
 * different streams: the input copy of one step on a copy stream while the
 * decode of the previous step runs, and (optionally) the output copy of a
 * step on a copy stream while the next one decodes (several block sets in
 * turn; the caller orders each decode after its input copy, each input copy
 * into dev_in after the decode that last read it, each output copy after its
 * decode, and each decode into dev_out after the output copy that last read
 * it, e.g. with CUDA events).
 *
 * fd_host_copy_in: queue the copy of host_in (in_bytes) to dev_in on
 *   `stream`.  Arguments as fd_decode_paged_host.  FD_ERR_INVALID_ARG on NULL
 *   blocks or an unaligned dev_in; FD_ERR_CUDA when the copy cannot be queued.
 * fd_decode_paged_staged: the decode of fd_decode_paged_host from an input
 *   block already in dev_in (its copy queued before, in stream order or behind
 *   an event).  host_out as fd_decode_paged_host (stores straight into a
 *   mapped block, else a copy from dev_out), or NULL: the results stay in
 *   dev_out.  Other arguments and errors as fd_decode_paged_host.
 * fd_host_copy_out: queue the copy of dev_out (out_bytes) to host_out on
 *   `stream`.  FD_ERR_INVALID_ARG on NULL blocks or an unaligned dev_out;
 *   FD_ERR_CUDA when the copy cannot be queued. */
fd_status fd_host_copy_in(const fd_plan_t *plan, const void *host_in, void *dev_in, void *stream);
fd_status fd_decode_paged_staged(const fd_plan_t *plan, const void *dev_in, const void *k_pages,
                                 const void *v_pages, const float *k_scale, const float *v_scale,
                                 void *dev_out, void *host_out, void *workspace, size_t workspace_bytes,
                                 int32_t *status_dev, void *stream);
fd_status fd_host_copy_out(const fd_plan_t *plan, const void *dev_out, void *host_out, void *stream);

/* Map a device status word to a status code (FD_OK when zero). */
fd_status fd_status_from_device(int32_t status_word);

/* Static description of a status code. */
const char *fd_status_string(fd_status status);

/* FD_API_VERSION of the loaded library. */
int fd_api_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FD_API_H */
