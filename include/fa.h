/*
 * fa.h -- C ABI of libfa.so: masked attention over a block-sparse BlockMask on GB300 (sm_103a).
 *
 * Three operations, as described on the pages this library implements:
 *   fa_create_block_mask  -- evaluate a mask rule tile by tile and emit the BlockMask tables
 *                            ("5.1.2 FlexAttention: from rules to fused kernels", sections 2.1-2.2;
 *                             "FlexAttention: compiler optimisation of custom attention", section 4).
 *   fa_flex_forward       -- FlashAttention-style forward that visits only the non-empty KV blocks of each
 *                            query block, applies the score rule, masks partial blocks only, and writes O
 *                            and LSE ("5.1.2 FlexAttention ...", section 3.1; "FlexAttention: compiler
 *                            optimisation ...", section 3).
 *   fa_flex_decode        -- one new query token per request over a paged KV cache, split along KV and
 *                            merged by the online-softmax law ("5.1.2 FlexAttention ...", sections 3.2 and
 *                            5; "FlexAttention: compiler optimisation ...", section 6; "5 Kernels: turning
 *                            logical sparsity into real speed-ups", section 3).
 *
 * Conventions shared by every entry point
 *  - Memory: the caller owns all memory. Pointers marked "device" must be device pointers of the current
 *    CUDA device; "host" pointers are read during the call only. The library keeps no state between
 *    calls and allocates no device memory.
 *  - Streams: all device work is enqueued on `stream` (NULL = legacy default stream). No entry point
 *    synchronises except fa_check_status.
 *  - Argument errors are detected on the host before anything is launched and return FA_ERR_* without
 *    side effects. Errors only the device can see (an out-of-range page id, a pipeline wait that timed
 *    out) are written to *dev_status (first error wins) and read back with fa_check_status.
 *  - Layouts are row-major and contiguous unless stated. bf16 = IEEE bfloat16 bit patterns (uint16).
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

typedef struct CUstream_st* fa_stream_t; /* the same type as cudaStream_t */

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,     /* NULL where a pointer is required, malformed rule, bad enum */
  FA_ERR_SHAPE = 2,           /* sizes inconsistent with each other or with the BlockMask */
  FA_ERR_UNSUPPORTED = 3,     /* valid but not implemented (head dim, block size, GQA group > 16) */
  FA_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed (launch, copy, tensor-map encode) */
  FA_ERR_TIMEOUT = 5,         /* device: a bounded pipeline wait gave up (the kernel returned early) */
  FA_ERR_DEVICE_CHECK = 6,    /* device: an index read from memory was out of range (e.g. a page id) */
  FA_ERR_BUFFER_TOO_SMALL = 7 /* caller-provided buffer/workspace smaller than required */
} fa_status;

FA_API const char* fa_status_string(fa_status s);

/* ------------------------------------------------------------------------------------------------
 * Mask rule (mask_mod): a postfix program over (b, h, q_idx, kv_idx) -> allowed.
 * "5.1.2 FlexAttention ...", section 1.1 (causal i >= j, left window i - j < W, document equality,
 * and_masks / or_masks); prefix-LM j < P OR causal as in the causal-pruning article, section 5.
 * i is the GLOBAL query position i = q_idx + q_offset[b] ("FlexAttention: compiler optimisation ...",
 * section 6: a decode query at position t must be compared as t, not 0).
 * Atoms push one value, FA_M_AND / FA_M_OR pop two and push one; exactly one value must remain.
 * The library rewrites the program into at most FA_MAX_RULE_TERMS OR-ed conjunctions; larger
 * expansions return FA_ERR_UNSUPPORTED.
 * ---------------------------------------------------------------------------------------------- */
#define FA_MAX_RULE_OPS 16
#define FA_MAX_RULE_TERMS 8

typedef enum {
  FA_M_TRUE = 0,   /* every pair */
  FA_M_CAUSAL = 1, /* kv_idx <= i */
  FA_M_WINDOW = 2, /* i - kv_idx < arg  (arg = W >= 1; the window includes the current token) */
  FA_M_PREFIX = 3, /* kv_idx < arg      (arg = P >= 0) */
  FA_M_DOC = 4,    /* doc_ids[b][i] == doc_ids[b][kv_idx] */
  FA_M_AND = 5,
  FA_M_OR = 6
} fa_mask_op;

typedef struct {
  int32_t n_ops;                   /* 1..FA_MAX_RULE_OPS */
  int32_t op[FA_MAX_RULE_OPS];     /* fa_mask_op */
  int64_t arg[FA_MAX_RULE_OPS];    /* W for FA_M_WINDOW, P for FA_M_PREFIX, ignored otherwise */
  const int32_t* doc_ids;          /* device int32 [doc_batch, doc_len]; required iff a FA_M_DOC op */
  int32_t doc_batch;               /* 1 (one sequence layout for all b) or B */
  int32_t doc_len;                 /* >= KV_LEN (every key position; else FA_ERR_SHAPE). A global query
                                      position outside [0, doc_len) (reachable through q_offset or
                                      Q_LEN > doc_len) reads as id -1: it shares a document with exactly
                                      the keys whose id is -1 (none when all ids are >= 0) */
  const int32_t* q_offset;         /* device int32 [B] or NULL (= all zero) */
  int32_t batch_dependent;         /* 0: table broadcast over b (Bm = 1); 1: Bm = B */
  int32_t head_dependent;          /* 0: table broadcast over h (Hm = 1); 1: Hm = H */
} fa_mask_rule;

/* ------------------------------------------------------------------------------------------------
 * Score rule (score_mod), applied to the already-scaled score s = scale * <q_i, k_j> in the fixed
 * order  s -> s + alibi -> + rel_bias -> softcap  (the c(a*s + r) order; "5.1.2 FlexAttention ...",
 * section 1.2). Every absent part is the identity. Head index = the QUERY head (GQA: section 1.2).
 * ---------------------------------------------------------------------------------------------- */
typedef struct {
  const float* alibi_slopes; /* device fp32 [Hq] or NULL:  s += -slope[h] * (i - j) */
  const float* rel_bias;     /* device fp32 [Hq, 2*KV_LEN-1] or NULL:  s += rel_bias[h][(i - j) + KV_LEN - 1] */
  float softcap;             /* > 0: s = softcap * tanh(s / softcap);  <= 0: off. The 128x128 forward
                                specialises the soft-cap alone for softcap <= 62.3 (a fixed softmax
                                reference; see fa_flex_forward); a larger cap, or a cap with a bias,
                                takes its generic score path (same results, slower). */
} fa_score_rule;

/* ------------------------------------------------------------------------------------------------
 * BlockMask ("5.1.2 FlexAttention ...", sections 2.1-2.2; "5 Kernels ...", section 4): per query block
 * row r (Bq rows) the partial KV blocks (kv_num / kv_idx) and the full ones (full_kv_num / full_kv_idx),
 * column ids ascending, unused slots 0; the query-side transpose per KV block c (q_num / q_idx,
 * full_q_num / full_q_idx), row ids ascending, unused slots 0. A block is full when every pair of its
 * Bq x Bk footprint is allowed, empty when none is, partial otherwise; pairs outside [0,Q_LEN) x
 * [0,KV_LEN) count as not allowed, so a ragged tail block is at most partial.
 * All arrays point into the caller's buffer given to fa_create_block_mask. The rule is kept by value
 * (its device pointers must stay valid while the mask is used).
 * ---------------------------------------------------------------------------------------------- */
typedef struct {
  int32_t Bm, Hm, q_len, kv_len, bq, bk, nq, nk;
  int32_t* kv_num;          /* [Bm,Hm,nq]    */
  int32_t* kv_idx;          /* [Bm,Hm,nq,nk] */
  int32_t* full_kv_num;     /* [Bm,Hm,nq]    */
  int32_t* full_kv_idx;     /* [Bm,Hm,nq,nk] */
  int32_t* q_num;           /* [Bm,Hm,nk]    */
  int32_t* q_idx;           /* [Bm,Hm,nk,nq] */
  int32_t* full_q_num;      /* [Bm,Hm,nk]    */
  int32_t* full_q_idx;      /* [Bm,Hm,nk,nq] */
  uint8_t* block_class;     /* [Bm,Hm,nq,nk]: 0 empty, 1 partial, 2 full */
  int32_t* doc_run;         /* rules that read document ids: [doc_batch,2,doc_len], per position the first
                               and one-past-last position of the run of equal ids around it; else NULL */
  int32_t* doc_sorted;      /* [doc_batch]: 1 where the ids never decrease (each id is then one run, and
                               the kernels test document equality as a column interval); else NULL */
  int32_t* row_order;       /* [Bm,Hm,nq]: the query block rows by visited length (full + partial) from the
                               longest, ties by the higher row first ("5.1.2 FlexAttention ...", section 5:
                               row lengths as the load signal; longest work first). The forward and the
                               dQ kernel take their query blocks in this order. NULL (one row per table):
                               rows nq-1 .. 0. Tables of more than 2048 key blocks keep nq-1 .. 0 too. */
  fa_mask_rule rule;
} fa_block_mask;

/* Bytes of device buffer fa_create_block_mask needs for these sizes (0 on invalid arguments). */
FA_API size_t fa_block_mask_bytes(const fa_mask_rule* rule, int32_t B, int32_t H, int32_t Q_LEN, int32_t KV_LEN,
                           int32_t Bq, int32_t Bk);

/* create_block_mask(mask_mod, B, H, Q_LEN, KV_LEN, BLOCK_SIZE) ("FlexAttention: compiler optimisation
 * ...", section 5; "5.1.2 FlexAttention ...", section 2.2 "building the table from mask_mod"):
 * classify every (b_m, h_m, r, c) block by evaluating the rule over its footprint, compact the partial
 * and full lists, and build the query-side transpose.
 *   rule      host pointer, copied into *out
 *   B, H      batch and query-head counts the mask is used with (Bm = B or 1, Hm = H or 1 per the rule)
 *   Bq, Bk    block sizes, 1..128 each
 *   dev_buf   device buffer of >= fa_block_mask_bytes(...) bytes, 256-byte aligned
 *   out       host struct, filled with pointers into dev_buf
 * Returns FA_ERR_BUFFER_TOO_SMALL, FA_ERR_SHAPE (non-positive sizes, Bq/Bk out of range, doc ids too
 * short), FA_ERR_INVALID_ARG (malformed rule, a rule that reads per-batch state with
 * batch_dependent = 0), FA_ERR_UNSUPPORTED (rule expands to more than FA_MAX_RULE_TERMS terms). */
FA_API fa_status fa_create_block_mask(const fa_mask_rule* rule, int32_t B, int32_t H, int32_t Q_LEN, int32_t KV_LEN,
                               int32_t Bq, int32_t Bk, void* dev_buf, size_t buf_bytes, fa_block_mask* out,
                               fa_stream_t stream);

/* Prebuilt table, sliced per decode step ("5.1.2 FlexAttention ...", section 5.2; "FlexAttention:
 * compiler optimisation ...", section 6): from a mask built once for the longest context in global
 * positions (src->rule.q_offset == NULL), take for each request b the query block row that holds its
 * token's position q_pos[b] and emit a one-row-per-request mask for fa_flex_decode: Bm = Bz, Hm =
 * src->Hm, q_len = nq = Bq = 1, the same kv_len / Bk / nk, and the rule of src with q_offset = q_pos
 * (batch_dependent = 1). A block that is full or empty for the whole block row is so for each of its
 * rows; only the row's partial blocks are evaluated again, at the one position, as the slice must match
 * the actual query length. The tables are then exactly those fa_create_block_mask builds for one query
 * at q_pos[b] (lists, classes and the one-row transpose), at the cost of the partial blocks only.
 *   src          host pointer to a mask from fa_create_block_mask; src->Bm is 1 or Bz
 *   dev_q_pos    device int32 [Bz], global query positions; must stay valid while *out is used
 *   dev_buf      device buffer of >= fa_block_mask_select_bytes(src, Bz) bytes, 256-byte aligned
 *   out          host struct, filled with pointers into dev_buf (and src's document run arrays)
 *   dev_status   device int32 or NULL: a position outside [0, src->q_len) sets FA_ERR_DEVICE_CHECK
 *                and that request's row is empty
 * Returns FA_ERR_INVALID_ARG (NULL pointers, src with a query offset), FA_ERR_SHAPE (src->Bm or the
 * document batch not 1 or Bz), FA_ERR_BUFFER_TOO_SMALL. */
FA_API size_t fa_block_mask_select_bytes(const fa_block_mask* src, int32_t Bz);
FA_API fa_status fa_block_mask_select_rows(const fa_block_mask* src, const int32_t* dev_q_pos, int32_t Bz,
                                           void* dev_buf, size_t buf_bytes, fa_block_mask* out,
                                           int32_t* dev_status, fa_stream_t stream);

/* Element type of O. The softmax statistics and the accumulator are fp32 in every case; FA_OUT_F32
 * stores the fp32 result as is, FA_OUT_BF16 rounds it to bf16 (round to nearest even) on the store. */
typedef enum { FA_OUT_BF16 = 0, FA_OUT_F32 = 1 } fa_out_dtype;

/* flex_attention(q, k, v, score_mod, block_mask, scale) forward ("5.1.2 FlexAttention ...", section
 * 3.1: for each query block visit the full list without the mask and the partial list with it, keep the
 * online-softmax state (m, l, acc), write O = acc / l and LSE = m + ln l; an empty row writes O = 0,
 * LSE = -inf).
 *   q            device bf16 [B, Hq, Q_LEN, d]
 *   k, v         device bf16 [B, Hkv, KV_LEN, d]; query head h reads KV head floor(h / (Hq/Hkv))
 *   block_mask   host pointer to a mask made by fa_create_block_mask with q_len == Q_LEN, kv_len ==
 *                KV_LEN, Bm in {1, B}, Hm in {1, Hq} (a length mismatch is an error, never trimmed)
 *   score_rule   host pointer or NULL (no score rule)
 *   scale        > 0, or <= 0 for 1/sqrt(d)
 *   out          device [B, Hq, Q_LEN, d] of type out_dtype;  lse  device fp32 [B, Hq, Q_LEN] (natural log)
 *   dev_status   device int32 or NULL (device-side errors are then not reported)
 *   dev_counters device int64[4] or NULL: += {query tiles, full blocks visited, partial blocks visited,
 *                K/V tile loads issued}. Empty blocks issue no load; a K/V tile load serves every query
 *                tile of the CTA that reads it (sibling query heads of one KV head with one mask row).
 * Supported: d in {64, 128}; Bq, Bk in {16, 32, 64, 128}; Q_LEN, KV_LEN >= 1; Hq % Hkv == 0;
 * q/k/v/out 16-byte aligned. Bq == Bk == 128 runs the tcgen05/TMEM kernel, other block sizes the
 * mma.sync kernel. The softmax reference m of a row is the running maximum, moved only when a block
 * exceeds it by 2^8 in log2 units, except under a soft-cap alone with softcap <= 62.3 on the tcgen05
 * kernel: the scores then lie in (-c, c) and m is fixed at c log2(e) - 64 (log2 units), every P staying
 * a normal fp32/bf16 number in [2^(64 - 2c log2 e), 2^64]. The choice of m changes O and LSE only by
 * rounding. */
FA_API fa_status fa_flex_forward(const void* q, const void* k, const void* v, const fa_block_mask* block_mask,
                                 const fa_score_rule* score_rule, float scale, void* out, int32_t out_dtype,
                                 float* lse, int32_t B, int32_t Hq, int32_t Hkv, int32_t Q_LEN, int32_t KV_LEN,
                                 int32_t d, int32_t* dev_status, int64_t* dev_counters, fa_stream_t stream);

/* The same forward with Q, K, V, O and LSE in host memory (pinned memory for full copy speed), for callers
 * whose tensors live on the host: the batch's KV heads are cut into chunks (about eight per call) that
 * stream through three device slots of `dev_workspace`; each chunk's copies in, its kernel and its copies
 * out run on separate streams, so copies overlap the neighbouring chunks' work. The mask stays on the
 * device (build it with fa_create_block_mask on `stream` first).
 *   host_q, host_k, host_v, host_out, host_lse  host pointers, layouts as fa_flex_forward; they must stay
 *                valid until `stream` has completed
 *   dev_workspace  device buffer of >= fa_forward_host_workspace_bytes(...) bytes, 256-byte aligned
 *   stream       everything queued on it before the call runs first; the call's last copy out completes
 *                on it (synchronise `stream` before reading host_out / host_lse)
 * Returns the errors of fa_flex_forward, FA_ERR_BUFFER_TOO_SMALL, FA_ERR_CUDA (stream or event creation). */
FA_API size_t fa_forward_host_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t Q_LEN, int32_t KV_LEN,
                                              int32_t d, int32_t out_dtype);
FA_API fa_status fa_flex_forward_host(const void* host_q, const void* host_k, const void* host_v,
                                      const fa_block_mask* block_mask, const fa_score_rule* score_rule, float scale,
                                      void* host_out, int32_t out_dtype, float* host_lse, int32_t B, int32_t Hq,
                                      int32_t Hkv, int32_t Q_LEN, int32_t KV_LEN, int32_t d, void* dev_workspace,
                                      size_t workspace_bytes, int32_t* dev_status, fa_stream_t stream);

/* The same forward with K and V in a paged cache ("5.1.2 FlexAttention ...", section 5, the paragraph on
 * turning the logical BlockMask into physical pages; "FlexAttention: compiler optimisation ...", section
 * 6): the rules stay in logical positions (the mask, causal / window bounds, the score rule and the query
 * offset all see token positions), and only the K / V fetch of logical key block c of batch row b goes to
 * physical page page_table[b * max_pages + c]. Several rows may name the same page (a shared prefix).
 *   k_pages, v_pages  device bf16 [n_pages_total, Hkv, page, d], page == the mask's Bk (one page per key
 *                     block), 16-byte aligned
 *   page_table        device int32 [B, max_pages], max_pages >= the mask's nk; entries of blocks the mask
 *                     never lists are not read. Slots of a page past KV_LEN must hold finite values (they
 *                     are masked, so any finite value gives the same result).
 *   other arguments   as fa_flex_forward (no counters)
 * Returns FA_ERR_SHAPE (page != Bk, max_pages < nk, n_pages_total < 1), FA_ERR_INVALID_ARG (NULL table,
 * misaligned pointers), and the errors of fa_flex_forward. A listed page id outside [0, n_pages_total)
 * sets *dev_status = FA_ERR_DEVICE_CHECK (page 0 is read in its place; the output is then not valid). */
FA_API fa_status fa_flex_forward_paged(const void* q, const void* k_pages, const void* v_pages,
                                       const int32_t* page_table, int32_t n_pages_total, int32_t page,
                                       int32_t max_pages, const fa_block_mask* block_mask,
                                       const fa_score_rule* score_rule, float scale, void* out, int32_t out_dtype,
                                       float* lse, int32_t B, int32_t Hq, int32_t Hkv, int32_t Q_LEN,
                                       int32_t KV_LEN, int32_t d, int32_t* dev_status, fa_stream_t stream);

/* The same forward with long rows split ("5 Kernels: turning logical sparsity into real speed-ups",
 * section 5: a long row becomes several tasks, each with its own softmax state, merged once; the merge law
 * of its section 3; "5.1.2 FlexAttention ...", section 5.2 on the long tail of row lengths). Each query
 * block row's visited blocks, in column order, are cut into chunks of at most chunk_blocks blocks; every
 * chunk runs as its own query tile (the tcgen05 kernel) and writes its normalised O and LSE to the
 * workspace, and a second kernel merges the chunks of each row: with m = max_c LSE_c,
 * O = sum_c e^(LSE_c - m) O_c / sum_c e^(LSE_c - m), LSE = m + ln sum_c e^(LSE_c - m) (an empty chunk has no
 * weight; a row with no visited block gets O = 0, LSE = -inf). A row of up to chunk_blocks blocks is one
 * chunk. The result equals fa_flex_forward's up to the summation order.
 *   arguments as fa_flex_forward (no counters), plus
 *   chunk_blocks   >= 1, key blocks per chunk
 *   workspace      device buffer of >= fa_forward_split_workspace_bytes(block_mask, B, Hq, d, chunk_blocks)
 *                  bytes, 256-byte aligned: the split tables and the per-chunk O (fp32) and LSE, about
 *                  B * Hq * nq * ceil(nk / chunk_blocks) * 128 * (d + 1) * 4 bytes
 * Supported: Bq == Bk == 128, d in {64, 128}. Returns the errors of fa_flex_forward, FA_ERR_UNSUPPORTED
 * (other block sizes), FA_ERR_INVALID_ARG (chunk_blocks < 1, workspace NULL or misaligned),
 * FA_ERR_BUFFER_TOO_SMALL. */
FA_API size_t fa_forward_split_workspace_bytes(const fa_block_mask* block_mask, int32_t B, int32_t Hq, int32_t d,
                                               int32_t chunk_blocks);
FA_API fa_status fa_flex_forward_split(const void* q, const void* k, const void* v, const fa_block_mask* block_mask,
                                       const fa_score_rule* score_rule, float scale, void* out, int32_t out_dtype,
                                       float* lse, int32_t B, int32_t Hq, int32_t Hkv, int32_t Q_LEN, int32_t KV_LEN,
                                       int32_t d, int32_t chunk_blocks, void* workspace, size_t workspace_bytes,
                                       int32_t* dev_status, fa_stream_t stream);

/* Same as fa_flex_forward but always uses the mma.sync kernel (a second, independent kernel over the
 * same tables; used to cross-check the tcgen05 path). */
FA_API fa_status fa_flex_forward_mma(const void* q, const void* k, const void* v, const fa_block_mask* block_mask,
                                     const fa_score_rule* score_rule, float scale, void* out, int32_t out_dtype,
                                     float* lse, int32_t B, int32_t Hq, int32_t Hkv, int32_t Q_LEN, int32_t KV_LEN,
                                     int32_t d, int32_t* dev_status, int64_t* dev_counters, fa_stream_t stream);

/* Gradients of fa_flex_forward's output ("5.1.2 FlexAttention ...", section 4.2: the backward reuses the
 * BlockMask and its query-side transpose; FlashAttention self-test questions on the backward pass).
 * With P recomputed from the forward's LSE and the score rule: D = rowsum(dout * out), dV = P^T dout,
 * dS = P (dout V^T - D) times the soft-cap's chain factor, dQ = scale dS K, dK = scale dS^T Q; dK and dV
 * summed over the query heads sharing a KV head (no atomics: one pass over the BlockMask rows for dQ, one
 * over its columns for dK / dV).
 *   q, k, v, block_mask, score_rule, scale, B .. d   as given to fa_flex_forward
 *   out, out_dtype, lse   the forward's outputs (device; out bf16 or fp32 per out_dtype)
 *   dout                  device bf16 [B,Hq,Q_LEN,d], the gradient of the loss with respect to out
 *   dq, dk, dv            device fp32 [B,Hq,Q_LEN,d], [B,Hkv,KV_LEN,d], [B,Hkv,KV_LEN,d]; overwritten
 *   delta                 device fp32 [B,Hq,Q_LEN] scratch (overwritten)
 * Block sizes 64 or 128 (both dimensions), d in {64, 128}. Pointers 16-byte aligned. Errors as for
 * fa_flex_forward; nothing is launched on an argument error. */
FA_API fa_status fa_flex_backward(const void* q, const void* k, const void* v, const void* out, int32_t out_dtype,
                                  const void* dout, const float* lse, const fa_block_mask* block_mask,
                                  const fa_score_rule* score_rule, float scale, float* dq, float* dk, float* dv,
                                  float* delta, int32_t B, int32_t Hq, int32_t Hkv, int32_t Q_LEN, int32_t KV_LEN,
                                  int32_t d, int32_t* dev_status, fa_stream_t stream);

/* Paged split-KV decode ("5.1.2 FlexAttention ...", sections 3.2 "split-KV exact merge" and 5.1-5.2;
 * "FlexAttention: compiler optimisation ...", section 6; the merge law of "5 Kernels ...", section 3).
 * One query token per request. Logical KV block c of request b lives in physical page
 * page_table[b][c]; rules use logical positions. Each (request, KV head, split) program reads every K/V
 * byte of its pages once for all Hq/Hkv query heads, keeps (m, l, u) for its pages, and a second kernel
 * merges the splits: m = max m_s, l = sum e^(m_s - m) l_s, O = sum e^(m_s - m) u_s / l.
 *   q            device bf16 [Bz, Hq, d]
 *   k_pages,
 *   v_pages      device bf16 [n_pages_total, Hkv, page, d]
 *   page_table   device int32 [Bz, max_pages]
 *   block_mask   made with Bq = 1, Bk = page, Q_LEN = 1, KV_LEN = max_pages * page, Bm in {1, Bz},
 *                Hm == 1; its rule's q_offset[b] is the query's global position (cur_pos = L_b - 1)
 *   workspace    device buffer of >= fa_decode_workspace_bytes(...) bytes, 16-byte aligned; holds the
 *                per-split (m, l, u) between the two kernels
 *   out          device [Bz, Hq, d] of type out_dtype;  lse  device fp32 [Bz, Hq]
 * Supported: d in {64, 128}; page in {32, 64, 128}; 1 <= Hq/Hkv <= 16.
 * A page id outside [0, n_pages_total) sets FA_ERR_DEVICE_CHECK in *dev_status (that page is skipped). */
FA_API size_t fa_decode_workspace_bytes(int32_t Bz, int32_t Hq, int32_t d, int32_t max_pages, int32_t page);
FA_API fa_status fa_flex_decode(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                                int32_t n_pages_total, const fa_block_mask* block_mask,
                                const fa_score_rule* score_rule, float scale, void* out, int32_t out_dtype,
                                float* lse, int32_t Bz, int32_t Hq, int32_t Hkv, int32_t d, int32_t page,
                                int32_t max_pages, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                int64_t* dev_counters, fa_stream_t stream);

/* Allocation-free decode. The pages this library follows have no counterpart to this entry point; it
 * exists for callers that cannot provide device memory: a host program whose device memory belongs to
 * another runtime's pool, or a serving loop that must never call cudaMalloc / cudaFree (cudaFree
 * synchronises the whole device). It computes exactly what fa_flex_decode computes (same arguments
 * minus the workspace) and keeps the per-split state in one file-scope device array of
 * FA_DECODE_NOALLOC_SCRATCH_BYTES bytes that every GPU loading libfa.so holds until the process exits.
 *  - Set-up: the first call on a device, with that device current, looks up the array's device address
 *    (cudaGetSymbolAddress) and caches it; make that first call before any stream capture. A
 *    cudaDeviceReset (or any other teardown of the device's context) invalidates the cached address
 *    without the library noticing: do not use this entry point on a device after resetting it.
 *  - Size limit: a problem whose fa_decode_workspace_bytes(...) exceeds the array returns
 *    FA_ERR_BUFFER_TOO_SMALL and launches nothing (fa_decode_noalloc_scratch_bytes() reports the size).
 *    Every other argument is checked first, with the codes fa_flex_decode returns for it. The need is
 *    about Bz * Hq * n_splits * (d + 3) * 4 bytes, n_splits = ceil(max_pages / min(max_pages,
 *    4096 / page)): with d = 128, 128-token pages, a 32768-token table (8 splits) and Hq = 32, up to 250
 *    requests fit.
 *  - Sharing: all calls use the same array. Calls that overlap on the GPU (different streams with no
 *    ordering between them) race on it; calls on one stream are fine. Nothing in it needs clearing
 *    between calls.
 *  - It allocates no memory and calls no allocating routine. */
#define FA_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
FA_API fa_status fa_flex_decode_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                        const int32_t* page_table, int32_t n_pages_total,
                                        const fa_block_mask* block_mask, const fa_score_rule* score_rule,
                                        float scale, void* out, int32_t out_dtype, float* lse, int32_t Bz,
                                        int32_t Hq, int32_t Hkv, int32_t d, int32_t page, int32_t max_pages,
                                        int32_t* dev_status, int64_t* dev_counters, fa_stream_t stream);
FA_API size_t fa_decode_noalloc_scratch_bytes(void);

/* Block statistics of a BlockMask ("5.1.2 FlexAttention ...", sections 2.2 and 6.3: full/partial/empty
 * counts and row lengths). dev_out: device int64[6] = {full, partial, empty, max row length (full +
 * partial), sum of row lengths, rows}. Enqueued on stream, no synchronisation. */
FA_API fa_status fa_block_mask_stats(const fa_block_mask* block_mask, int64_t* dev_out, fa_stream_t stream);

/* Synchronise `stream`, read *dev_status and return it as an fa_status (FA_ERR_CUDA if the stream
 * reported a CUDA error). Does not clear *dev_status. */
FA_API fa_status fa_check_status(const int32_t* dev_status, fa_stream_t stream);

/* Bounded waits. Every pipeline wait inside the kernels gives up after this many nanoseconds, sets
 * FA_ERR_TIMEOUT and returns. Default 2e9 (2 s). Process-wide setting read at launch time. */
FA_API void fa_set_wait_timeout_ns(uint64_t ns);
FA_API uint64_t fa_get_wait_timeout_ns(void);

/* Self-test of the bounded wait: launches one CTA that waits on an mbarrier nothing ever arrives on,
 * with a limit of timeout_ns; the kernel must return and set FA_ERR_TIMEOUT in *dev_status. */
FA_API fa_status fa_debug_wait_timeout(int32_t* dev_status, uint64_t timeout_ns, fa_stream_t stream);

/* Self-test of one tcgen05 MMA chain (128 x 128 x K, bf16 in, fp32 accumulate in tensor memory):
 * C = A * B^T with A device bf16 [128, K] and B device bf16 [128, K] (b_mn_major = 0, B K-major), or
 * C = A * B with B device bf16 [K, 128] (b_mn_major = 1, B MN-major); C device fp32 [128, 128].
 * K in {64, 128}. use_tma = 1 stages the tiles with TMA (128-byte swizzle), 0 with plain stores in the
 * same swizzled layout, 2 puts A in tensor memory (row per lane, two bf16 per 32-bit column) and B in
 * shared memory. Used by the tests to pin the shared-memory, tensor-memory and instruction descriptors. */
FA_API fa_status fa_debug_tc5_gemm(const void* A, const void* B, float* C, int32_t K, int32_t b_mn_major,
                            int32_t use_tma, int32_t* dev_status, fa_stream_t stream);

/* Self-test of the soft-cap every kernel applies: y[i] = c * tanh(x[i] / c) ("5.1.2 FlexAttention: from
 * rules to fused kernels", section 1.2). x, y: device fp32 [n]; c > 0. */
FA_API fa_status fa_debug_softcap(const float* x, float* y, int32_t n, float c, fa_stream_t stream);

/* Library version string. */
FA_API const char* fa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FA_H_ */
