// Split rows of the prefill forward ("5 Kernels: turning logical sparsity into real speed-ups", section 5:
// a long row is cut into several tasks, each keeping its own softmax state, merged once at the end; the
// merge law of section 3 of the same page; "5.1.2 FlexAttention: from rules to fused kernels", section 5.2
// on taming the long tail of row lengths).
//
// mask_split_kernel   cuts each query block row's visited blocks (its full and partial lists merged in
//                     column order) into chunks of at most C blocks and writes them as the rows of a
//                     derived BlockMask (entry e = r * ncm + c), with a row order that takes chunk c of
//                     every row before chunk c + 1. The forward kernel then runs each entry as a query
//                     tile of block r and writes that entry's normalised O and its LSE.
// split_combine_kernel merges the entries of each query row: with m = max_e LSE_e,
//                     O = sum_e e^(LSE_e - m) O_e / sum_e e^(LSE_e - m), LSE = m + ln sum_e e^(LSE_e - m);
//                     an entry with LSE = -inf (an empty chunk) has no weight and its O is not read.
#include "fa_launch.h"

namespace fa {
namespace {

// One warp per (query block row, chunk). The row's visited blocks in column order are the merge of its
// full and partial lists (each ascending, no column in both); the number of full blocks among the first
// k of them is found by a binary search over the two lists (a merge path), so every lane places its own
// positions of the chunk without walking the row.
__device__ __forceinline__ int full_before(const int32_t* fi, int nf, const int32_t* pi, int np, int k) {
  int lo = max(0, k - np), hi = min(k, nf);
  while (lo < hi) {  // more full blocks while the next full one precedes the partial one it would displace
    const int mid = (lo + hi) >> 1;
    if (__ldg(fi + mid) < __ldg(pi + (k - mid - 1))) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(256) mask_split_kernel(MaskOut S, int C, int ncm, MaskOut D) {
  const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int bh = blockIdx.y;  // b_m * Hm + h_m
  if (w >= S.nq * ncm) return;
  const int r = w / ncm, c = w - r * ncm;
  const size_t srow = (size_t)bh * S.nq + r;
  const int nf = S.full_kv_num[srow], np = S.kv_num[srow];
  const int32_t* fi = S.full_kv_idx + srow * S.nk;
  const int32_t* pi = S.kv_idx + srow * S.nk;
  const int n = nf + np;
  const int k0 = min(c * C, n), k1 = min(k0 + C, n);  // the chunk's positions in column order
  const int f0 = full_before(fi, nf, pi, np, k0), p0 = k0 - f0;
  const int cf = full_before(fi, nf, pi, np, k1) - f0, cp = (k1 - k0) - cf;
  const size_t nqd = (size_t)S.nq * ncm;
  const size_t drow = (size_t)bh * nqd + (size_t)r * ncm + c;
  int32_t* dfi = D.full_kv_idx + drow * C;
  int32_t* dpi = D.kv_idx + drow * C;
  for (int k = k0 + lane; k < k1; k += 32) {
    const int f = full_before(fi, nf, pi, np, k);
    const int vf = f < nf ? __ldg(fi + f) : 0x7FFFFFFF, vp = k - f < np ? __ldg(pi + (k - f)) : 0x7FFFFFFF;
    if (vf < vp) dfi[f - f0] = vf;
    else dpi[(k - f) - p0] = vp;
  }
  for (int k = cf + lane; k < C; k += 32) dfi[k] = 0;  // unused slots 0, as in every table
  for (int k = cp + lane; k < C; k += 32) dpi[k] = 0;
  if (lane == 0) {
    D.full_kv_num[drow] = cf;
    D.kv_num[drow] = cp;
    D.row_order[(size_t)bh * nqd + (size_t)c * S.nq + (S.nq - 1 - r)] = r * ncm + c;
  }
}

// one warp per query row; lane l holds columns 4 l .. 4 l + 3
__global__ void __launch_bounds__(256) split_combine_kernel(const float* __restrict__ o_part,
                                                            const float* __restrict__ lse_part, int rows, int q_len,
                                                            int nq, int ncm, int d, void* out, int out_f32,
                                                            float* lse) {
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (gw >= rows) return;
  const int bh = gw / q_len, i = gw - bh * q_len;
  const int r = i >> 7, rr = i & 127;
  const size_t part_rows = (size_t)nq * ncm * 128;
  const float* L = lse_part + (size_t)bh * part_rows;
  float m = -INFINITY;
  for (int c = 0; c < ncm; ++c) m = fmaxf(m, L[((size_t)r * ncm + c) * 128 + rr]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float sum = 0.f;
  const bool has = lane * 4 < d;
  if (m != -INFINITY) {
    for (int c = 0; c < ncm; ++c) {
      const size_t pr = ((size_t)r * ncm + c) * 128 + rr;
      const float lc = L[pr];
      if (lc == -INFINITY) continue;
      const float w = expf(lc - m);
      sum += w;
      if (has) {
        const float4 o = *reinterpret_cast<const float4*>(o_part + ((size_t)bh * part_rows + pr) * d + lane * 4);
        acc.x += w * o.x;
        acc.y += w * o.y;
        acc.z += w * o.z;
        acc.w += w * o.w;
      }
    }
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  if (has) {
    const size_t off = ((size_t)bh * q_len + i) * d + lane * 4;
    if (out_f32) {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + off) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
      uint2 v;
      v.x = *reinterpret_cast<uint32_t*>(&lo);
      v.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + off) = v;
    }
  }
  if (lane == 0) lse[(size_t)bh * q_len + i] = m == -INFINITY ? -INFINITY : m + logf(sum);
}

}  // namespace

cudaError_t launch_mask_split(const MaskOut& S, int C, int ncm, const MaskOut& D, cudaStream_t st) {
  dim3 grid((unsigned)(((int64_t)S.nq * ncm + 7) / 8), S.Bm * S.Hm);
  mask_split_kernel<<<grid, 256, 0, st>>>(S, C, ncm, D);
  return cudaGetLastError();
}

cudaError_t launch_split_combine(const float* o_part, const float* lse_part, int B, int Hq, int q_len, int nq,
                                 int ncm, int d, void* out, int out_f32, float* lse, cudaStream_t st) {
  const int rows = B * Hq * q_len;
  split_combine_kernel<<<(rows + 7) / 8, 256, 0, st>>>(o_part, lse_part, rows, q_len, nq, ncm, d, out, out_f32, lse);
  return cudaGetLastError();
}

}  // namespace fa
