// create_block_mask on the device ("5.1.2 FlexAttention: from rules to fused kernels", section 2.2,
// "building the table from mask_mod": evaluate the rule inside every block, reduce any/all, compact to
// indices; the query-side transpose of section 2.1).
//
// Kernel 1 (one CTA per (b_m, h_m, query block r)): every thread owns one query row of the block and
// evaluates the rule as a 128-bit vector per KV block (interval arithmetic per OR-term, document ids
// compared per column only when the rule reads them). Rows vote "some pair allowed" / "some pair not
// allowed" per KV block; a CTA-wide prefix sum then compacts the partial and full column ids in
// ascending order and zero-fills the unused slots.
// Kernel 2 (one CTA per (b_m, h_m, KV block c)): the same compaction down a column of the class matrix.
#include "fa_launch.h"

namespace fa {

namespace {

constexpr int kThreads = 128;
constexpr int kChunk = 4096;  // KV (or query) blocks classified per pass of a CTA

struct ScanOut {
  int excl_a, excl_b, tot_a, tot_b;
};

// CTA-wide exclusive scan of two counters (128 threads).
__device__ __forceinline__ ScanOut block_scan2(int a, int b, int* s_tmp /* [8] */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int ta = __shfl_up_sync(0xFFFFFFFFu, ia, o);
    int tb = __shfl_up_sync(0xFFFFFFFFu, ib, o);
    if (lane >= o) {
      ia += ta;
      ib += tb;
    }
  }
  if (lane == 31) {
    s_tmp[warp] = ia;
    s_tmp[4 + warp] = ib;
  }
  __syncthreads();
  int wa = 0, wb = 0, ta = 0, tb = 0;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    if (w < warp) {
      wa += s_tmp[w];
      wb += s_tmp[4 + w];
    }
    ta += s_tmp[w];
    tb += s_tmp[4 + w];
  }
  __syncthreads();
  ScanOut r;
  r.excl_a = wa + ia - a;
  r.excl_b = wb + ib - b;
  r.tot_a = ta;
  r.tot_b = tb;
  return r;
}

__global__ void __launch_bounds__(kThreads) mask_classify_kernel(DevRule R, MaskOut T) {
  const int r = blockIdx.x, hm = blockIdx.y, bm = blockIdx.z;
  const int tid = threadIdx.x;
  const int Bq = T.bq, Bk = T.bk, nk = T.nk;
  const int lanes = kThreads / Bq;  // KV blocks evaluated side by side
  const int rho = tid % Bq, lam = tid / Bq;
  const bool active = lam < lanes;
  const int64_t i = (int64_t)r * Bq + rho;
  const bool row_in = active && i < T.q_len;
  const int64_t ig = i + (R.q_offset ? (int64_t)__ldg(R.q_offset + bm) : 0);
  const int doc_i = (R.any_doc && row_in) ? doc_at(R, bm, ig) : -1;

  __shared__ uint8_t s_any[kChunk];
  __shared__ uint8_t s_notall[kChunk];
  __shared__ int s_tmp[8];

  const size_t row = ((size_t)bm * T.Hm + hm) * T.nq + r;
  int32_t* kv_idx = T.kv_idx + row * nk;
  int32_t* full_idx = T.full_kv_idx + row * nk;
  uint8_t* cls_row = T.block_class + row * nk;
  const Bits128 full_bk = range_bits(0, Bk);

  int run_p = 0, run_f = 0;
  for (int c0 = 0; c0 < nk; c0 += kChunk) {
    const int cn = min(kChunk, nk - c0);
    for (int x = tid; x < cn; x += kThreads) {
      s_any[x] = 0;
      s_notall[x] = 0;
    }
    __syncthreads();
    if (active) {
      for (int cc = lam; cc < cn; cc += lanes) {
        const int64_t j0 = (int64_t)(c0 + cc) * Bk;
        const int w = (int)min((int64_t)Bk, (int64_t)T.kv_len - j0);
        bool any = false, all = false;
        if (row_in) {
          Bits128 b = rule_row_bits(R, ig, j0, w, doc_i, [&](int d) {
            Bits128 db = {{0u, 0u, 0u, 0u}};
            for (int c = 0; c < w; ++c)
              if (doc_at(R, bm, j0 + c) == d) db.w[c >> 5] |= 1u << (c & 31);
            return db;
          });
          any = (b.w[0] | b.w[1] | b.w[2] | b.w[3]) != 0u;
          all = (w == Bk) && b.w[0] == full_bk.w[0] && b.w[1] == full_bk.w[1] && b.w[2] == full_bk.w[2] &&
                b.w[3] == full_bk.w[3];
        }
        if (any) s_any[cc] = 1;
        if (!all) s_notall[cc] = 1;
      }
    }
    __syncthreads();
    // classify the chunk and compact (each thread owns a contiguous segment -> ascending order)
    const int seg = (cn + kThreads - 1) / kThreads;
    const int s0 = min(tid * seg, cn), s1 = min(s0 + seg, cn);
    int np = 0, nf = 0;
    for (int x = s0; x < s1; ++x) {
      const uint8_t cl = s_any[x] ? (s_notall[x] ? FA_BLOCK_PARTIAL : FA_BLOCK_FULL) : FA_BLOCK_EMPTY;
      cls_row[c0 + x] = cl;
      np += cl == FA_BLOCK_PARTIAL;
      nf += cl == FA_BLOCK_FULL;
    }
    ScanOut so = block_scan2(np, nf, s_tmp);
    int p = run_p + so.excl_a, f = run_f + so.excl_b;
    for (int x = s0; x < s1; ++x) {
      const bool a = s_any[x] != 0, na = s_notall[x] != 0;
      if (a && na) kv_idx[p++] = c0 + x;
      if (a && !na) full_idx[f++] = c0 + x;
    }
    run_p += so.tot_a;
    run_f += so.tot_b;
    __syncthreads();
  }
  for (int x = run_p + tid; x < nk; x += kThreads) kv_idx[x] = 0;
  for (int x = run_f + tid; x < nk; x += kThreads) full_idx[x] = 0;
  if (tid == 0) {
    T.kv_num[row] = run_p;
    T.full_kv_num[row] = run_f;
  }
}

__global__ void __launch_bounds__(kThreads) mask_transpose_kernel(MaskOut T) {
  const int c = blockIdx.x, hm = blockIdx.y, bm = blockIdx.z;
  const int tid = threadIdx.x;
  const int nq = T.nq, nk = T.nk;
  __shared__ int s_tmp[8];
  const size_t head = (size_t)bm * T.Hm + hm;
  const uint8_t* cls = T.block_class + head * nq * nk + c;  // column c, stride nk
  const size_t col = head * nk + c;
  int32_t* q_idx = T.q_idx + col * nq;
  int32_t* fq_idx = T.full_q_idx + col * nq;
  int run_p = 0, run_f = 0;
  for (int r0 = 0; r0 < nq; r0 += kChunk) {
    const int rn = min(kChunk, nq - r0);
    const int seg = (rn + kThreads - 1) / kThreads;
    const int s0 = min(tid * seg, rn), s1 = min(s0 + seg, rn);
    int np = 0, nf = 0;
    for (int x = s0; x < s1; ++x) {
      const uint8_t cl = cls[(size_t)(r0 + x) * nk];
      np += cl == FA_BLOCK_PARTIAL;
      nf += cl == FA_BLOCK_FULL;
    }
    ScanOut so = block_scan2(np, nf, s_tmp);
    int p = run_p + so.excl_a, f = run_f + so.excl_b;
    for (int x = s0; x < s1; ++x) {
      const uint8_t cl = cls[(size_t)(r0 + x) * nk];
      if (cl == FA_BLOCK_PARTIAL) q_idx[p++] = r0 + x;
      if (cl == FA_BLOCK_FULL) fq_idx[f++] = r0 + x;
    }
    run_p += so.tot_a;
    run_f += so.tot_b;
  }
  for (int x = run_p + tid; x < nq; x += kThreads) q_idx[x] = 0;
  for (int x = run_f + tid; x < nq; x += kThreads) fq_idx[x] = 0;
  if (tid == 0) {
    T.q_num[col] = run_p;
    T.full_q_num[col] = run_f;
  }
}

// dev_out = {full, partial, empty, max row length, sum of row lengths, rows} (zeroed by the launcher)
__global__ void __launch_bounds__(256) mask_stats_kernel(MaskOut T, unsigned long long* out) {
  const long long rows = (long long)T.Bm * T.Hm * T.nq;
  long long f = 0, p = 0, mx = 0;
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < rows; x += (long long)gridDim.x * blockDim.x) {
    const long long a = T.full_kv_num[x], b = T.kv_num[x];
    f += a;
    p += b;
    mx = max(mx, a + b);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    f += __shfl_xor_sync(0xFFFFFFFFu, f, o);
    p += __shfl_xor_sync(0xFFFFFFFFu, p, o);
    mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  }
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(out + 0, (unsigned long long)f);
    atomicAdd(out + 1, (unsigned long long)p);
    atomicMax(out + 3, (unsigned long long)mx);
    atomicAdd(out + 4, (unsigned long long)(f + p));
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    atomicAdd(out + 5, (unsigned long long)rows);
  }
}

__global__ void mask_stats_finish(MaskOut T, unsigned long long* out) {
  const unsigned long long total = (unsigned long long)T.Bm * T.Hm * T.nq * T.nk;
  out[2] = total - out[0] - out[1];
}

}  // namespace

cudaError_t launch_mask_build(const DevRule& R, const MaskOut& T, cudaStream_t st) {
  dim3 g1(T.nq, T.Hm, T.Bm);
  mask_classify_kernel<<<g1, kThreads, 0, st>>>(R, T);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 g2(T.nk, T.Hm, T.Bm);
  mask_transpose_kernel<<<g2, kThreads, 0, st>>>(T);
  return cudaGetLastError();
}

cudaError_t launch_mask_stats(const MaskOut& T, int64_t* dev_out, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(dev_out, 0, 6 * sizeof(int64_t), st);
  if (e != cudaSuccess) return e;
  const long long rows = (long long)T.Bm * T.Hm * T.nq;
  long long nb = (rows + 255) / 256;
  int blocks = (int)(nb > 1024 ? 1024 : nb);
  if (blocks < 1) blocks = 1;
  mask_stats_kernel<<<blocks, 256, 0, st>>>(T, reinterpret_cast<unsigned long long*>(dev_out));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mask_stats_finish<<<1, 1, 0, st>>>(T, reinterpret_cast<unsigned long long*>(dev_out));
  return cudaGetLastError();
}

}  // namespace fa
