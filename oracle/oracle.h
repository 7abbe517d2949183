/*
 * oracle.h -- fp64 CPU oracle for paged, GQA-shared decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This library is what the CUDA path is checked
 * against.  Only the test suite, the package smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header, table or helper
 * with the CUDA library (split_kv_decode_paged_gb300/csrc), and the CUDA
 * library never calls it.
 *
 * What it computes is the plain definition of one-token decode attention:
 * for every (sequence b, query head hq) the full softmax over all cached
 * tokens, in double precision, with no splitting and no online softmax.
 * The split/merge method of the pages reaches this result exactly up to
 * rounding ("FlashDecoding 与 FlashInfer 深度解析", §2.1 step 3: merging the
 * partial softmaxes equals the softmax over the whole sequence).
 *
 * Storage formats are decoded by the oracle's own decoders, written from the
 * format definitions (IEEE 754 binary16, bfloat16 = the top half of binary32,
 * OCP FP8 E4M3 with bias 7, no infinities and S.1111.111 = NaN).
 *
 * Parity pins: every function here is pinned by tests/test_oracle_*.py
 * against closed forms, brute force in arbitrary precision, library
 * conversions and the pages' worked examples.
 */
#ifndef FD_ORACLE_H
#define FD_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Storage type codes (the oracle's own numbering). */
enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_F32 = 3 };

/* Return codes. */
enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_BAD_PAGE = 2, ORC_ERR_NOMEM = 3 };

typedef struct {
    int B;                  /* sequences                                   */
    int Hq;                 /* query heads                                 */
    int Hkv;                /* key/value heads, Hq % Hkv == 0              */
    int D;                  /* head dimension                              */
    int page_size;          /* tokens per page                             */
    int max_blocks_per_seq; /* columns of the block table                  */
    int num_pages;          /* pages in the K (and V) pool                 */
    int q_dtype;            /* ORC_F16 / ORC_BF16 / ORC_F32                */
    int kv_dtype;           /* ORC_F16 / ORC_BF16 / ORC_E4M3 / ORC_F32     */
} orc_problem;

/* Format decoders (exact). */
double orc_f16_to_double(uint16_t bits);
double orc_bf16_to_double(uint16_t bits);
double orc_e4m3_to_double(uint8_t bits);

/* E4M3 encoder: round to nearest, ties to even mantissa; magnitudes at or
 * above the largest finite value (448) saturate to +-448; NaN maps to the
 * NaN code with the input's sign. */
uint8_t orc_e4m3_from_float(float x);

/* Full-softmax decode attention over the paged cache.
 *   q            [B, Hq, D]                     (q_dtype)
 *   k/v_pages    [num_pages, page_size, Hkv, D] (kv_dtype)
 *   k/v_scale    [num_pages, Hkv] fp32, used only for ORC_E4M3
 *   block_table  [B, max_blocks_per_seq] int32, -1 = unused
 *   seq_lens     [B] int32
 *   out          [B, Hq, D] fp64;  lse [B, Hq] fp64 (natural log)
 * A sequence with seq_len 0 yields out = 0 and lse = -inf.
 * nthreads <= 0 uses every online core.  Returns ORC_ERR_BAD_PAGE if a page
 * index inside a live range is out of [0, num_pages). */
int orc_decode_paged(const orc_problem *p, const void *q, const void *k_pages,
                     const void *v_pages, const float *k_scale, const float *v_scale,
                     const int32_t *block_table, const int32_t *seq_lens,
                     double *out, double *lse, int nthreads);

/* Same, for a subset of (b, hq) pairs: pairs[2*i] = b, pairs[2*i+1] = hq.
 * out is [npairs, D], lse [npairs]. */
int orc_decode_paged_pairs(const orc_problem *p, const void *q, const void *k_pages,
                           const void *v_pages, const float *k_scale, const float *v_scale,
                           const int32_t *block_table, const int32_t *seq_lens,
                           const int32_t *pairs, int npairs,
                           double *out, double *lse, int nthreads);

/* Decode with the "Inference Cookbook" §5.2-5.3 indirections: q row b reads
 * cache row cb = cache_batch_idx[b] (identity when NULL) -- its block-table
 * row, seq_lens entry and leftpad entry -- and attends tokens
 * [leftpad[cb], seq_lens[cb]) (leftpad 0 when NULL).  cache_rows = rows of
 * block_table / seq_lens / leftpad.  Returns ORC_ERR_ARG for an index outside
 * the cache or a leftpad outside [0, seq_len]. */
/* Several query tokens per sequence, causal among them ("Inference Cookbook"
 * §3.2-3.3: flash_attn_with_kvcache with seqlen_q >= 1 and causal=True after
 * the new tokens' K/V were written into the cache; "FlashDecoding 与
 * FlashInfer 深度解析" §3.1, the append mode).  q [B, q_len, Hq, D]: query
 * token i of sequence b is the i-th of its last q_len cached tokens and
 * attends the tokens [0, L_b - q_len + i + 1) (the causal mask aligned to the
 * end of the cache).  out [B, q_len, Hq, D], lse [B, q_len, Hq].  Requires
 * L_b >= q_len. */
int orc_decode_paged_multi(const orc_problem *p, int q_len, const void *q, const void *k_pages,
                           const void *v_pages, const float *k_scale, const float *v_scale,
                           const int32_t *block_table, const int32_t *seq_lens,
                           double *out, double *lse);

int orc_decode_paged_ex(const orc_problem *p, int cache_rows, const int32_t *cache_batch_idx,
                        const int32_t *cache_leftpad, const void *q, const void *k_pages,
                        const void *v_pages, const float *k_scale, const float *v_scale,
                        const int32_t *block_table, const int32_t *seq_lens,
                        double *out, double *lse);

/* Contiguous-cache decode: k/v_cache [B, max_seqlen, Hkv, D] (kv_dtype, no
 * scales).  The comparator for the paged gather. */
int orc_decode_contiguous(const orc_problem *p, int max_seqlen, const void *q,
                          const void *k_cache, const void *v_cache,
                          const int32_t *seq_lens, double *out, double *lse);

/* Partial state of one (b, hq) over the token range [t_begin, t_end):
 * o = sum_t exp(s_t - m) v_t (unnormalised), m = max_t s_t, d = sum_t exp(s_t - m).
 * An empty range gives o = 0, m = -inf, d = 0. */
int orc_partial_state(const orc_problem *p, const void *q, const void *k_pages,
                      const void *v_pages, const float *k_scale, const float *v_scale,
                      const int32_t *block_table, int b, int hq, int t_begin, int t_end,
                      double *o, double *m, double *d);

/* Merge of n partial states (o [n, D], m [n], d [n]) into the normalised
 * output and its log-sum-exp, by the rescale formula of the pages. */
void orc_merge_states(int n, int D, const double *o, const double *m, const double *d,
                      double *out, double *lse);

/* KV append: write k_new/v_new [B, Hkv, D] (new_dtype) at position
 * seq_lens[b] of each sequence, in place into k/v_pages.  For an E4M3 cache
 * the value is divided by the page's scale in fp32 and encoded with
 * orc_e4m3_from_float; otherwise new_dtype must equal kv_dtype and the bits
 * are copied.  seq_lens is not modified. */
int orc_append_kv(const orc_problem *p, int new_dtype, const void *k_new, const void *v_new,
                  void *k_pages, void *v_pages, const float *k_scale, const float *v_scale,
                  const int32_t *block_table, const int32_t *seq_lens);

/* Rotary position embedding applied at append time ("Inference Cookbook"
 * §3.4: the new key is rotated before it is written into the cache, and the
 * query is rotated at the same position).  cos_tab/sin_tab: fp32
 * [max_pos, rotary_dim / 2].  Pair (i, i + rotary_dim/2) (interleaved == 0,
 * GPT-NeoX style) or (2i, 2i+1) (interleaved != 0) of the first rotary_dim
 * elements is rotated by angle index i at position pos:
 *   y1 = (x1 * cos) - (x2 * sin),  y2 = (x2 * cos) + (x1 * sin)
 * with every product and sum rounded to fp32 (no fused multiply-add); the
 * other elements pass through.  x: n fp32 values, y: n fp32 values. */
void orc_rotary_f32(const float *x, int n, int rotary_dim, int interleaved, const float *cos_tab,
                    const float *sin_tab, int pos, float *y);

/* orc_append_kv with the key rotated (V is not) before it is stored, and q
 * [B, Hq, D] (q_dtype, may be NULL) rotated in place, both at position
 * seq_lens[b].  Rotated 16-bit values are rounded to nearest even. */
int orc_append_kv_rotary(const orc_problem *p, int new_dtype, const void *k_new, const void *v_new,
                         void *k_pages, void *v_pages, const float *k_scale, const float *v_scale,
                         const int32_t *block_table, const int32_t *seq_lens,
                         const float *cos_tab, const float *sin_tab, int rotary_dim, int max_pos,
                         int interleaved, void *q_inout);

#ifdef __cplusplus
}
#endif
#endif
