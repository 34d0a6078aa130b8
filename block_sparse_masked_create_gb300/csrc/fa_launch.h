// Internal launch interfaces between the C-ABI layer (fa_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fa_internal.cuh"

namespace fa {

// Table pointers and geometry of a BlockMask, as the kernels read it.
struct DevMask {
  int32_t Bm, Hm, q_len, kv_len, bq, bk, nq, nk;
  const int32_t* kv_num;
  const int32_t* kv_idx;
  const int32_t* full_kv_num;
  const int32_t* full_kv_idx;
  const int32_t* q_num;        // query-side transpose (the backward's key-block columns)
  const int32_t* q_idx;
  const int32_t* full_q_num;
  const int32_t* full_q_idx;
  const int32_t* row_order;    // [Bm,Hm,nq] rows by visited length, longest first (NULL: nq-1 .. 0)
};

struct MaskOut {
  int32_t Bm, Hm, q_len, kv_len, bq, bk, nq, nk;
  int32_t* kv_num;
  int32_t* kv_idx;
  int32_t* full_kv_num;
  int32_t* full_kv_idx;
  int32_t* q_num;
  int32_t* q_idx;
  int32_t* full_q_num;
  int32_t* full_q_idx;
  uint8_t* block_class;
  int32_t* doc_run;     // [doc_batch][2][doc_len] or NULL
  int32_t* doc_sorted;  // [doc_batch] or NULL
  int32_t* row_order;   // [Bm][Hm][nq] or NULL
};

cudaError_t launch_mask_build(const DevRule& R, const MaskOut& T, cudaStream_t st);
cudaError_t launch_mask_stats(const MaskOut& T, int64_t* dev_out, cudaStream_t st);
// row block q_pos[b] / S.bq of S per request b, re-classified at position q_pos[b] = R.q_offset[b] -> D with
// Bm = Bz, nq = 1 (D's buffers laid out by the caller)
cudaError_t launch_mask_select(const DevRule& R, const MaskOut& S, int Bz, const MaskOut& D, int32_t* status,
                               cudaStream_t st);

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  int32_t out_f32;  // 1: O stored as fp32, 0: bf16
  float* lse;
  int32_t B, Hq, Hkv, q_len, kv_len, d;
  float scale;
  DevRule rule;
  DevScore score;
  DevMask mask;
  int32_t* status;
  int64_t* counters;
  uint64_t timeout_ns;
  // paged K/V (NULL: contiguous [B, Hkv, kv_len, d]): k and v point at pages [n_pages_total, Hkv, Bk, d]
  // and key block c of batch row b lives in page page_table[b * max_pages + c] (one page per key block)
  const int32_t* page_table;
  int32_t max_pages, n_pages_total;
  // split rows (tcgen05 kernel only): the mask's rows are entries e = r * split_ncm + c, chunk c of query
  // block r; Q and every position come from block e / split_ncm, while O (fp32) and LSE of entry e are
  // written at rows e * 128 .. of [B, Hq, out_q_len]. split_ncm = 1 and out_q_len = q_len otherwise.
  int32_t split_ncm, out_q_len;
};

cudaError_t launch_fwd_mma(const FwdArgs& a, cudaStream_t st);
// Returns FA_OK / FA_ERR_UNSUPPORTED / FA_ERR_CUDA.
int launch_fwd_tc5(const FwdArgs& a, cudaStream_t st);

struct DecArgs {
  const void* q;
  const void* k_pages;
  const void* v_pages;
  const int32_t* page_table;
  int32_t n_pages_total;
  void* out;
  int32_t out_f32;
  float* lse;
  int32_t Bz, Hq, Hkv, d, page, max_pages;
  float scale;
  DevRule rule;
  DevScore score;
  DevMask mask;
  float* ws_m;      // [Bz, Hq, n_splits]
  float* ws_l;      // [Bz, Hq, n_splits]  sum of the bf16-rounded P (normalises O)
  float* ws_le;     // [Bz, Hq, n_splits]  sum of the unrounded P (LSE)
  float* ws_u;      // [Bz, Hq, n_splits, d]
  int32_t pages_per_split, n_splits;
  int32_t* status;
  int64_t* counters;
  uint64_t timeout_ns;
};

int launch_decode(const DecArgs& a, cudaStream_t st);

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* out;     // the forward's O
  int32_t out_f32;     // 1: O is fp32, 0: bf16
  const void* dout;    // bf16, layout of q
  const float* lse;    // the forward's LSE (natural log)
  float* dq;           // fp32, layout of q
  float* dk;           // fp32, layout of k
  float* dv;           // fp32, layout of v
  float* delta;        // [B, Hq, q_len] scratch: rowsum(dO * O)
  int32_t B, Hq, Hkv, q_len, kv_len, d;
  float scale;
  DevRule rule;
  DevScore score;
  DevMask mask;
  int32_t* status;
  uint64_t timeout_ns;  // bound of every in-kernel wait (tcgen05 kernels)
};

cudaError_t launch_backward(const BwdArgs& a, cudaStream_t st);
// dQ and dK/dV on tcgen05 for 128 x 128 blocks; FA_OK / FA_ERR_UNSUPPORTED / FA_ERR_CUDA
int launch_bwd_tc5(const BwdArgs& a, cudaStream_t st);

cudaError_t launch_debug_wait(int32_t* status, uint64_t timeout_ns, cudaStream_t st);

// Split rows. From a BlockMask S (q_len rows of Bq = 128), the derived tables D: per (b_m, h_m) and
// entry e = r * ncm + c, chunk c of block row r's visited blocks (full and partial merged in column
// order, chunk = positions [c C, c C + C) of that order), as full / partial lists of row stride C; and a
// row order that takes chunk c of every row (rows from the last) before chunk c + 1.
cudaError_t launch_mask_split(const MaskOut& S, int C, int ncm, const MaskOut& D, cudaStream_t st);
// Merge the entries of each query row (normalised O_e fp32 [B, Hq, nq * ncm * 128, d], LSE_e [B, Hq,
// nq * ncm * 128]) into O (bf16 or fp32) [B, Hq, q_len, d] and LSE [B, Hq, q_len].
cudaError_t launch_split_combine(const float* o_part, const float* lse_part, int B, int Hq, int q_len, int nq,
                                 int ncm, int d, void* out, int out_f32, float* lse, cudaStream_t st);

// Host helpers: encode a bf16 / fp32 tensor map (dims innermost first) with 128-byte swizzle.
int encode_tmap_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides_bytes /* rank-1 entries */, const uint32_t* box);
int encode_tmap_f32(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box);

}  // namespace fa
