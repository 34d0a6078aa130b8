// create_block_mask on the device ("5.1.2 FlexAttention: from rules to fused kernels", section 2.2,
// "building the table from mask_mod": evaluate the rule inside every block, reduce any/all, compact to
// indices; the query-side transpose of section 2.1).
//
// Kernel 1 (one CTA per (b_m, h_m, query block r)): each KV block is first classified from the rule's
// terms at block level (interval tests, document-id ranges); only the blocks that test cannot decide
// are visited pair by pair: every thread owns one query row and evaluates the rule as a 128-bit vector
// over the block's columns (interval arithmetic per OR-term, document ids compared per column), rows
// vote "some pair allowed" / "some pair not allowed". A CTA-wide prefix sum then compacts the partial
// and full column ids in ascending order and zero-fills the unused slots.
// Kernel 2 (one CTA per (b_m, h_m, KV block c)): the same compaction down a column of the class matrix.
#include <climits>

#include "fa_launch.h"

namespace fa {

namespace {

constexpr int kThreads = 128;
constexpr int kChunk = 2048;  // KV (or query) blocks classified per pass of a CTA

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

// Document-id runs, one thread per position (grid.y = batch row). Where the ids never decrease, the
// run of equal ids around position t is [first position with id >= d[t], first with id > d[t]) of the
// row: two binary searches. Any decrease clears the row's `sorted` flag (set beforehand); the bounds
// of an unsorted row are then never read.
__global__ void __launch_bounds__(256) doc_runs_kernel(DevRule R, int32_t* run, int32_t* sorted) {
  const int b = blockIdx.y;
  const int n = R.doc_len;
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n) return;
  const int32_t* d = R.doc_ids + (size_t)b * n;
  const int v = __ldg(d + t);
  if (t > 0 && __ldg(d + t - 1) > v) sorted[b] = 0;
  int a = 0, z = t;  // lower bound of v in [0, t]
  while (a < z) {
    const int m = (a + z) >> 1;
    if (__ldg(d + m) < v) a = m + 1; else z = m;
  }
  int c = t + 1, e = n;  // upper bound of v in [t + 1, n)
  while (c < e) {
    const int m = (c + e) >> 1;
    if (__ldg(d + m) <= v) c = m + 1; else e = m;
  }
  int32_t* lo = run + (size_t)b * 2 * n;
  lo[t] = a;
  lo[n + t] = c;
}

constexpr uint8_t kUnknown = 0xFF;  // class not decided by the block-level test
constexpr int kDocStage = 4096;     // column document ids staged in shared memory per visiting round

// Min / max over the CTA (128 threads) of two values.
__device__ __forceinline__ void block_minmax(int& mn, int& mx, int* s_tmp /* [8] */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  }
  if (lane == 0) {
    s_tmp[warp] = mn;
    s_tmp[4 + warp] = mx;
  }
  __syncthreads();
  mn = min(min(s_tmp[0], s_tmp[1]), min(s_tmp[2], s_tmp[3]));
  mx = max(max(s_tmp[4], s_tmp[5]), max(s_tmp[6], s_tmp[7]));
  __syncthreads();
}

// Class of block (rows [g0, g1) in global positions, all of the query block's valid rows; columns
// [j0, j1)) decided from the rule's terms without visiting pairs. Per term the columns allowed by
// "j < pre" form an interval and causal / window bound d = i - j to an interval; over a rectangle of
// rows x columns d takes every integer between its extremes, so "some pair" and "every pair" are
// exact interval tests. Document equality is decided only when the row and column document ranges
// are disjoint (no equal pair) or both a single equal id (always equal); otherwise, and for an OR of
// terms none of which covers the block alone, the answer is kUnknown and the caller visits the pairs.
__device__ __forceinline__ uint8_t classify_block(const DevRule& R, int64_t g0, int64_t g1, int64_t j0, int64_t j1,
                                                  bool full_shape, int rdmin, int rdmax, int cdmin, int cdmax) {
  if (g1 <= g0 || j1 <= j0) return FA_BLOCK_EMPTY;
  bool any = false, all = false, unknown = false;
  for (int t = 0; t < R.n_terms; ++t) {
    const DevTerm T = R.t[t];
    const int64_t jhi = T.pre != INT64_MAX ? min(j1, T.pre) : j1;
    if (jhi <= j0) continue;  // no column of the block is allowed by this term
    const bool all_j = T.pre == INT64_MAX || j1 <= T.pre;
    const int64_t dlo = T.causal ? 0 : INT64_MIN;
    const int64_t dhi = T.win != INT64_MAX ? T.win - 1 : INT64_MAX;
    bool any_t = !((g1 - 1) - j0 < dlo || g0 - (jhi - 1) > dhi);
    bool all_t = all_j && g0 - (j1 - 1) >= dlo && (g1 - 1) - j0 <= dhi;
    if (T.doc) {
      if (cdmax < rdmin || cdmin > rdmax) {
        any_t = all_t = false;
      } else if (!(rdmin == rdmax && cdmin == cdmax)) {
        all_t = false;
        if (any_t) {
          unknown = true;
          any_t = false;
        }
      }
    }
    any = any || any_t;
    all = all || all_t;
  }
  if (!full_shape) return any ? FA_BLOCK_PARTIAL : (unknown ? kUnknown : FA_BLOCK_EMPTY);
  if (all) return FA_BLOCK_FULL;
  if (unknown) return kUnknown;
  if (!any) return FA_BLOCK_EMPTY;
  return R.n_terms > 1 ? kUnknown : FA_BLOCK_PARTIAL;
}

// Hull of a table row (or column): ascending, disjoint intervals of block indices that hold every block
// with at least one allowed pair, so that blocks outside them are empty without being looked at (the
// structured interval builder of "5.1.2 FlexAttention: from rules to fused kernels", section 2.2: for
// interval rules the work is proportional to the visited blocks, not to nq x nk). Per OR-term the
// allowed keys of a row range [g0, g1) (global positions) lie in one interval: "j < pre" bounds it
// above, causal (j <= i) by g1, a window (i - j < W) below by g0 - W + 1, and document equality, where
// the ids never decrease and the rows lie inside the id array with a non-negative first id, by the
// runs of the first and last row. The same reasoning bounds the rows of a column range. Conservative
// by construction: the blocks inside still go through the exact classification.
struct Hull {
  int n;
  int lo[FA_MAX_RULE_TERMS], hi[FA_MAX_RULE_TERMS], pre[FA_MAX_RULE_TERMS + 1];
};

constexpr int64_t kHullWinMax = (int64_t)1 << 40;  // wider windows bound nothing at int32 lengths

// add positions [lo, hi) (lo >= 0) as blocks of size bs, clipped to [0, nblk), keeping the list sorted
__device__ void hull_add(Hull& h, int64_t lo, int64_t hi, int bs, int nblk) {
  if (hi <= lo) return;
  const int a = (int)(lo / bs);
  const int b = (int)min((hi + bs - 1) / bs, (int64_t)nblk);
  if (b <= a) return;
  int k = h.n++;
  while (k > 0 && h.lo[k - 1] > a) {
    h.lo[k] = h.lo[k - 1];
    h.hi[k] = h.hi[k - 1];
    --k;
  }
  h.lo[k] = a;
  h.hi[k] = b;
}

__device__ void hull_merge(Hull& h) {
  int m = 0;
  for (int k = 0; k < h.n; ++k) {
    if (m > 0 && h.lo[k] <= h.hi[m - 1]) {
      h.hi[m - 1] = max(h.hi[m - 1], h.hi[k]);
    } else {
      h.lo[m] = h.lo[k];
      h.hi[m] = h.hi[k];
      ++m;
    }
  }
  h.n = m;
  h.pre[0] = 0;
  for (int k = 0; k < m; ++k) h.pre[k + 1] = h.pre[k] + h.hi[k] - h.lo[k];
}

// block index of the v-th block of the hull (v < pre[n])
__device__ __forceinline__ int hull_at(const Hull& h, int v) {
  int k = 0;
  while (k + 1 < h.n && v >= h.pre[k + 1]) ++k;
  return h.lo[k] + v - h.pre[k];
}

// KV blocks that rows [g0, g1) (global positions) can reach
__device__ void row_hull(const DevRule& R, int bm, int64_t g0, int64_t g1, int64_t kv_len, int Bk, int nk,
                         Hull& h) {
  h.n = 0;
  if (g1 > g0) {
    bool refine = false;
    int64_t rlo = 0, rhi = 0, unused = 0;
    if (R.any_doc && doc_runs_usable(R, bm) && g0 >= 0 && g1 <= R.doc_len && doc_at(R, bm, g0) >= 0) {
      doc_run_of(R, bm, g0, rlo, unused);
      doc_run_of(R, bm, g1 - 1, unused, rhi);
      refine = true;
    }
    for (int t = 0; t < R.n_terms; ++t) {
      const DevTerm T = R.t[t];
      int64_t lo = 0, hi = kv_len;
      if (T.pre != INT64_MAX) hi = min(hi, T.pre);
      if (T.causal) hi = min(hi, g1);
      if (T.win != INT64_MAX && T.win < kHullWinMax) lo = max(lo, g0 - T.win + 1);
      if (T.doc && refine) {
        lo = max(lo, rlo);
        hi = min(hi, rhi);
      }
      hull_add(h, lo, hi, Bk, nk);
    }
  }
  hull_merge(h);
}

// query blocks (local rows, offset off to global) that can reach keys [j0, j1)
__device__ void col_hull(const DevRule& R, int bm, int64_t off, int64_t j0, int64_t j1, int64_t q_len, int Bq,
                         int nq, Hull& h) {
  h.n = 0;
  if (j1 > j0) {
    bool refine = false;
    int64_t clo = 0, chi = 0, unused = 0;
    if (R.any_doc && doc_runs_usable(R, bm) && j1 <= R.doc_len && doc_at(R, bm, j0) >= 0) {
      doc_run_of(R, bm, j0, clo, unused);
      doc_run_of(R, bm, j1 - 1, unused, chi);
      refine = true;
    }
    for (int t = 0; t < R.n_terms; ++t) {
      const DevTerm T = R.t[t];
      if (T.pre != INT64_MAX && j0 >= T.pre) continue;
      int64_t lo = 0, hi = q_len;
      if (T.causal) lo = max(lo, j0 - off);
      if (T.win != INT64_MAX && T.win < kHullWinMax) hi = min(hi, j1 - 1 + T.win - off);
      if (T.doc && refine) {
        lo = max(lo, clo - off);
        hi = min(hi, chi - off);
      }
      hull_add(h, max(lo, (int64_t)0), hi, Bq, nq);
    }
  }
  hull_merge(h);
}

__global__ void __launch_bounds__(kThreads) mask_classify_kernel(DevRule R, MaskOut T) {
  const int r = blockIdx.x, hm = blockIdx.y, bm = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Bq = T.bq, Bk = T.bk, nk = T.nk;
  const int64_t off = R.q_offset ? (int64_t)__ldg(R.q_offset + bm) : 0;
  const int64_t i0 = (int64_t)r * Bq, i1 = min(i0 + Bq, (int64_t)T.q_len);  // valid rows [i0, i1)
  const bool rows_full = i1 - i0 == Bq;

  __shared__ uint8_t s_cls[kChunk];
  __shared__ int s_a[kChunk];  // column-block document minimum, then "some pair allowed"
  __shared__ int s_b[kChunk];  // column-block document maximum, then "some pair not allowed"
  __shared__ int s_tmp[8];
  __shared__ int s_doc[kDocStage];  // column document ids of the blocks visited side by side
  __shared__ Hull s_h;               // the KV blocks this query block can reach

  if (tid == 0) row_hull(R, bm, i0 + off, i1 + off, T.kv_len, Bk, nk, s_h);

  // document range of the query block's valid rows (ids that never decrease: first and last row)
  int rdmin = INT_MAX, rdmax = INT_MIN;
  const bool sorted_ids = R.any_doc && doc_runs_usable(R, bm);
  if (sorted_ids) {
    if (i1 > i0) {
      const int da = doc_at(R, bm, i0 + off), db = doc_at(R, bm, i1 - 1 + off);
      rdmin = min(da, db);  // -1 (outside the id array) may sit at either end
      rdmax = max(da, db);
      if (da == -1 || db == -1) {  // mixed inside / outside: fall back to the full reduction
        rdmin = INT_MAX;
        rdmax = INT_MIN;
        for (int64_t i = i0 + tid; i < i1; i += kThreads) {
          const int d = doc_at(R, bm, i + off);
          rdmin = min(rdmin, d);
          rdmax = max(rdmax, d);
        }
        block_minmax(rdmin, rdmax, s_tmp);
      }
    }
  } else if (R.any_doc) {
    for (int64_t i = i0 + tid; i < i1; i += kThreads) {
      const int d = doc_at(R, bm, i + off);
      rdmin = min(rdmin, d);
      rdmax = max(rdmax, d);
    }
    block_minmax(rdmin, rdmax, s_tmp);
  }

  // per-row state of the exact evaluation (row rho of lam-th block evaluated side by side)
  const int lanes = kThreads / Bq;
  const int rho = tid % Bq, lam = tid / Bq;
  const bool active = lam < lanes;
  const int64_t i = i0 + rho;
  const bool row_in = active && i < T.q_len;
  const int64_t ig = i + off;
  const int doc_i = (R.any_doc && row_in) ? doc_at(R, bm, ig) : -1;
  const bool runs = R.any_doc && row_in && ig >= 0 && ig < R.doc_len && doc_runs_usable(R, bm);
  int64_t run_lo = 0, run_hi = 0;
  if (runs) doc_run_of(R, bm, ig, run_lo, run_hi);
  const Bits128 full_bk = range_bits(0, Bk);

  const size_t row = ((size_t)bm * T.Hm + hm) * T.nq + r;
  int32_t* kv_idx = T.kv_idx + row * nk;
  int32_t* full_idx = T.full_kv_idx + row * nk;
  uint8_t* cls_row = T.block_class + row * nk;

  __syncthreads();
  const int nh = s_h.pre[s_h.n];  // blocks in the hull; the rest are empty
  for (int x = tid; x < nk; x += kThreads) {
    bool in = false;
    for (int k = 0; k < s_h.n; ++k) in = in || (x >= s_h.lo[k] && x < s_h.hi[k]);
    if (!in) cls_row[x] = FA_BLOCK_EMPTY;
  }
  auto col = [&](int v) { return hull_at(s_h, v); };

  int run_p = 0, run_f = 0;
  for (int c0 = 0; c0 < nh; c0 += kChunk) {
    const int cn = min(kChunk, nh - c0);
    // 1. document range of every column block of the chunk: first and last id when the ids never
    // decrease, else a warp per block (coalesced)
    if (sorted_ids) {
      for (int x = tid; x < cn; x += kThreads) {
        const int64_t j0 = (int64_t)col(c0 + x) * Bk;
        const int64_t j1 = min(j0 + Bk, (int64_t)T.kv_len);
        s_a[x] = doc_at(R, bm, j0);
        s_b[x] = doc_at(R, bm, j1 - 1);
      }
      __syncthreads();
    } else if (R.any_doc) {
      for (int x = warp; x < cn; x += kThreads / 32) {
        const int64_t j0 = (int64_t)col(c0 + x) * Bk;
        const int w = (int)min((int64_t)Bk, (int64_t)T.kv_len - j0);
        int mn = INT_MAX, mx = INT_MIN;
        for (int cc = lane; cc < w; cc += 32) {
          const int d = doc_at(R, bm, j0 + cc);
          mn = min(mn, d);
          mx = max(mx, d);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
          mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        }
        if (lane == 0) {
          s_a[x] = mn;
          s_b[x] = mx;
        }
      }
      __syncthreads();
    }
    // 2. block-level classification
    bool has_unknown = false;
    for (int x = tid; x < cn; x += kThreads) {
      const int64_t j0 = (int64_t)col(c0 + x) * Bk, j1 = min(j0 + Bk, (int64_t)T.kv_len);
      const uint8_t cl = classify_block(R, i0 + off, i1 + off, j0, j1, rows_full && j1 - j0 == Bk, rdmin, rdmax,
                                        R.any_doc ? s_a[x] : 0, R.any_doc ? s_b[x] : 0);
      s_cls[x] = cl;
      has_unknown = has_unknown || cl == kUnknown;
    }
    // 3. undecided blocks: every valid row evaluates the rule over the block's columns
    if (__syncthreads_or(has_unknown)) {
      for (int x = tid; x < cn; x += kThreads) {
        s_a[x] = 0;
        s_b[x] = 0;
      }
      __syncthreads();
      // rounds of `lanes` blocks side by side; the blocks' column document ids are staged in shared
      // memory when they fit (every thread of the CTA takes part in the rounds and their barriers)
      const bool stage = R.any_doc && !doc_runs_usable(R, bm) && lanes * Bk <= kDocStage;  // uniform in the CTA
      for (int base = 0; base < cn; base += lanes) {
        bool round_has = false;  // same answer in every thread (s_cls is stable here)
        for (int l = 0; l < lanes && base + l < cn; ++l) round_has = round_has || s_cls[base + l] == kUnknown;
        if (!round_has) continue;
        if (stage) {
          for (int x = tid; x < lanes * Bk; x += kThreads) {
            const int cc = base + x / Bk;
            const int64_t j = (int64_t)col(c0 + cc) * Bk + x % Bk;
            s_doc[x] = (cc < cn && s_cls[cc] == kUnknown && j < T.kv_len) ? doc_at(R, bm, j) : 0;
          }
          __syncthreads();
        }
        const int cc = base + lam;
        if (active && cc < cn && s_cls[cc] == kUnknown) {
          const int64_t j0 = (int64_t)col(c0 + cc) * Bk;
          const int w = (int)min((int64_t)Bk, (int64_t)T.kv_len - j0);
          bool any = false, all = false;
          if (row_in) {
            const int* cdoc = s_doc + lam * Bk;
            Bits128 b = rule_row_bits(R, ig, j0, w, doc_i, [&](int d) {
              if (runs) return range_bits(clamp_rel(run_lo - j0, w), clamp_rel(run_hi - j0, w));
              return stage ? doc_bits<4>(w, d, [&](int c) { return cdoc[c]; })
                           : doc_bits<4>(w, d, [&](int c) { return doc_at(R, bm, j0 + c); });
            });
            any = (b.w[0] | b.w[1] | b.w[2] | b.w[3]) != 0u;
            all = (w == Bk) && b.w[0] == full_bk.w[0] && b.w[1] == full_bk.w[1] && b.w[2] == full_bk.w[2] &&
                  b.w[3] == full_bk.w[3];
          }
          if (any) s_a[cc] = 1;
          if (!all) s_b[cc] = 1;
        }
        if (stage) __syncthreads();
      }
      __syncthreads();
      for (int x = tid; x < cn; x += kThreads)
        if (s_cls[x] == kUnknown) s_cls[x] = s_a[x] ? (s_b[x] ? FA_BLOCK_PARTIAL : FA_BLOCK_FULL) : FA_BLOCK_EMPTY;
    }
    __syncthreads();
    // 4. compaction (each thread owns a contiguous segment -> ascending order)
    const int seg = (cn + kThreads - 1) / kThreads;
    const int s0 = min(tid * seg, cn), s1 = min(s0 + seg, cn);
    int np = 0, nf = 0;
    for (int x = s0; x < s1; ++x) {
      const uint8_t cl = s_cls[x];
      cls_row[col(c0 + x)] = cl;
      np += cl == FA_BLOCK_PARTIAL;
      nf += cl == FA_BLOCK_FULL;
    }
    ScanOut so = block_scan2(np, nf, s_tmp);
    int p = run_p + so.excl_a, f = run_f + so.excl_b;
    for (int x = s0; x < s1; ++x) {
      const uint8_t cl = s_cls[x];
      if (cl == FA_BLOCK_PARTIAL) kv_idx[p++] = col(c0 + x);
      if (cl == FA_BLOCK_FULL) full_idx[f++] = col(c0 + x);
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

// Rows of the table by visited length (full + partial), longest first, ties by the higher row first:
// a stable counting sort over the key nk - length, one CTA per (b_m, h_m). The forward and the dQ kernel
// take their query blocks in this order, so the longest rows start first and the short ones fill the
// tail ("5.1.2 FlexAttention ...", section 5: row lengths as the load signal). For causal tables this is
// the order nq-1 .. 0. Tables wider than kOrderBins - 1 blocks (keys past 2048 x Bk) keep that order.
// Runs in one extra CTA per (b_m, h_m) of the transpose launch (the row tables are complete by then);
// the histogram is static shared memory of every CTA of that launch, hence kept small.
constexpr int kOrderBins = 2049;

__device__ void mask_row_order(const MaskOut& T, int hm, int bm, int* s_cnt /* [kOrderBins] */,
                               int* s_tmp /* [8] */) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int nq = T.nq, nk = T.nk;
  const size_t base = ((size_t)bm * T.Hm + hm) * nq;
  int32_t* order = T.row_order + base;
  if (nk + 1 > kOrderBins) {
    for (int x = tid; x < nq; x += kThreads) order[x] = nq - 1 - x;
    return;
  }
  auto len = [&](int r) { return __ldg(T.kv_num + base + r) + __ldg(T.full_kv_num + base + r); };
  for (int x = tid; x <= nk; x += kThreads) s_cnt[x] = 0;
  __syncthreads();
  for (int r = tid; r < nq; r += kThreads) atomicAdd(&s_cnt[nk - len(r)], 1);
  __syncthreads();
  // exclusive scan of the counts: the first position of each key
  const int nb = nk + 1, seg = (nb + kThreads - 1) / kThreads;
  const int s0 = min(tid * seg, nb), s1 = min(s0 + seg, nb);
  int sum = 0;
  for (int x = s0; x < s1; ++x) sum += s_cnt[x];
  const ScanOut so = block_scan2(sum, 0, s_tmp);
  int run = so.excl_a;
  for (int x = s0; x < s1; ++x) {
    const int c = s_cnt[x];
    s_cnt[x] = run;
    run += c;
  }
  __syncthreads();
  // placement by one warp, 32 rows per step from the highest row down: lanes with the same key take
  // consecutive positions in lane order (higher rows first), then the key's cursor moves past them
  if (tid < 32) {
    for (int r0 = nq - 1; r0 >= 0; r0 -= 32) {
      const int r = r0 - lane;
      const bool valid = r >= 0;
      const int key = valid ? nk - len(r) : -1 - lane;  // lanes past row 0 get keys of their own
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, key);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int pos = valid ? s_cnt[key] + rank : 0;
      __syncwarp();
      if (valid && rank == 0) s_cnt[key] += __popc(peers);
      __syncwarp();
      if (valid) order[pos] = r;
    }
  }
}

__global__ void __launch_bounds__(kThreads) mask_transpose_kernel(DevRule R, MaskOut T) {
  const int c = blockIdx.x, hm = blockIdx.y, bm = blockIdx.z;
  const int tid = threadIdx.x;
  const int nq = T.nq, nk = T.nk;
  __shared__ int s_tmp[8];
  if (c == nk) {  // the extra CTA: the row order
    __shared__ int s_cnt[kOrderBins];
    mask_row_order(T, hm, bm, s_cnt, s_tmp);
    return;
  }
  __shared__ Hull s_h;  // the query blocks that can reach this KV block; the class matrix is empty elsewhere
  if (tid == 0) {
    const int64_t off = R.q_offset ? (int64_t)__ldg(R.q_offset + bm) : 0;
    const int64_t j0 = (int64_t)c * T.bk, j1 = min(j0 + T.bk, (int64_t)T.kv_len);
    col_hull(R, bm, off, j0, j1, T.q_len, T.bq, nq, s_h);
  }
  __syncthreads();
  const int nh = s_h.pre[s_h.n];
  const size_t head = (size_t)bm * T.Hm + hm;
  const uint8_t* cls = T.block_class + head * nq * nk + c;  // column c, stride nk
  const size_t col = head * nk + c;
  int32_t* q_idx = T.q_idx + col * nq;
  int32_t* fq_idx = T.full_q_idx + col * nq;
  int run_p = 0, run_f = 0;
  for (int r0 = 0; r0 < nh; r0 += kChunk) {
    const int rn = min(kChunk, nh - r0);
    const int seg = (rn + kThreads - 1) / kThreads;
    const int s0 = min(tid * seg, rn), s1 = min(s0 + seg, rn);
    int np = 0, nf = 0;
    for (int x = s0; x < s1; ++x) {
      const uint8_t cl = cls[(size_t)hull_at(s_h, r0 + x) * nk];
      np += cl == FA_BLOCK_PARTIAL;
      nf += cl == FA_BLOCK_FULL;
    }
    ScanOut so = block_scan2(np, nf, s_tmp);
    int p = run_p + so.excl_a, f = run_f + so.excl_b;
    for (int x = s0; x < s1; ++x) {
      const int r = hull_at(s_h, r0 + x);
      const uint8_t cl = cls[(size_t)r * nk];
      if (cl == FA_BLOCK_PARTIAL) q_idx[p++] = r;
      if (cl == FA_BLOCK_FULL) fq_idx[f++] = r;
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

// One row of a prebuilt table per request ("5.1.2 FlexAttention ...", section 5.2: build the table once
// for the longest context, then at each decode step take the query block that holds each request's
// position and keep the exact rule for its partial blocks). One CTA per (request, h_m). The block row's
// full and empty blocks are full / empty for each of its valid rows, so only its partial blocks are
// looked at again, for the one query row at the request's position: they become empty, full or stay
// partial. The result is the table a one-row build at that position gives, without the classification
// of the row's other blocks (for a paged cache this also drops blocks past the request's own length,
// whose pages may not exist). A position outside [0, src q_len) reports a device-check error and yields
// an empty row.
__global__ void __launch_bounds__(kThreads) mask_select_kernel(DevRule R, MaskOut S, MaskOut D, int32_t* status) {
  const int bz = blockIdx.x, hm = blockIdx.y, tid = threadIdx.x;
  const int nk = S.nk, Bk = S.bk;
  __shared__ uint8_t s_cls[kChunk];
  __shared__ int s_tmp[8];
  const int64_t pos = __ldg(R.q_offset + bz);
  const bool ok = pos >= 0 && pos < S.q_len;
  if (!ok && tid == 0) report(status, FA_ERR_DEVICE_CHECK);
  const int sb = S.Bm > 1 ? bz : 0;
  const size_t srow = ((size_t)sb * S.Hm + hm) * S.nq + (ok ? pos / S.bq : 0);
  const size_t drow = (size_t)bz * D.Hm + hm;  // nq = 1
  const int doc_i = (R.any_doc && ok) ? doc_at(R, bz, pos) : -1;
  const Bits128 full_bk = range_bits(0, Bk);
  int run_p = 0, run_f = 0;
  for (int c0 = 0; c0 < nk; c0 += kChunk) {
    const int cn = min(kChunk, nk - c0);
    for (int x = tid; x < cn; x += kThreads) {
      uint8_t cl = ok ? S.block_class[srow * nk + c0 + x] : (uint8_t)FA_BLOCK_EMPTY;
      if (cl == FA_BLOCK_PARTIAL) {
        const int64_t j0 = (int64_t)(c0 + x) * Bk;
        const int w = (int)min((int64_t)Bk, (int64_t)S.kv_len - j0);
        const Bits128 bits = rule_row_bits(R, pos, j0, w, doc_i, [&](int d) {
          return doc_bits<4>(w, d, [&](int c) { return doc_at(R, bz, j0 + c); });
        });
        const bool any = (bits.w[0] | bits.w[1] | bits.w[2] | bits.w[3]) != 0u;
        const bool all = w == Bk && bits.w[0] == full_bk.w[0] && bits.w[1] == full_bk.w[1] &&
                         bits.w[2] == full_bk.w[2] && bits.w[3] == full_bk.w[3];
        cl = any ? (all ? FA_BLOCK_FULL : FA_BLOCK_PARTIAL) : FA_BLOCK_EMPTY;
      }
      s_cls[x] = cl;
    }
    __syncthreads();
    const int seg = (cn + kThreads - 1) / kThreads;
    const int s0 = min(tid * seg, cn), s1 = min(s0 + seg, cn);
    int np = 0, nf = 0;
    for (int x = s0; x < s1; ++x) {
      const uint8_t cl = s_cls[x];
      const size_t e = drow * nk + c0 + x;
      D.block_class[e] = cl;
      D.q_num[e] = cl == FA_BLOCK_PARTIAL;  // the transpose of a one-row table
      D.full_q_num[e] = cl == FA_BLOCK_FULL;
      D.q_idx[e] = 0;
      D.full_q_idx[e] = 0;
      np += cl == FA_BLOCK_PARTIAL;
      nf += cl == FA_BLOCK_FULL;
    }
    ScanOut so = block_scan2(np, nf, s_tmp);
    int p = run_p + so.excl_a, f = run_f + so.excl_b;
    for (int x = s0; x < s1; ++x) {
      const uint8_t cl = s_cls[x];
      if (cl == FA_BLOCK_PARTIAL) D.kv_idx[drow * nk + p++] = c0 + x;
      if (cl == FA_BLOCK_FULL) D.full_kv_idx[drow * nk + f++] = c0 + x;
    }
    run_p += so.tot_a;
    run_f += so.tot_b;
    __syncthreads();
  }
  for (int x = run_p + tid; x < nk; x += kThreads) D.kv_idx[drow * nk + x] = 0;
  for (int x = run_f + tid; x < nk; x += kThreads) D.full_kv_idx[drow * nk + x] = 0;
  if (tid == 0) {
    D.kv_num[drow] = run_p;
    D.full_kv_num[drow] = run_f;
  }
}

}  // namespace

cudaError_t launch_mask_build(const DevRule& R0, const MaskOut& T, cudaStream_t st) {
  DevRule R = R0;
  if (R.any_doc && T.doc_run && T.doc_sorted) {
    cudaError_t e = cudaMemsetAsync(T.doc_sorted, 0xFF, sizeof(int32_t) * R.doc_batch, st);  // nonzero: sorted
    if (e != cudaSuccess) return e;
    doc_runs_kernel<<<dim3((R.doc_len + 255) / 256, R.doc_batch), 256, 0, st>>>(R, T.doc_run, T.doc_sorted);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    R.doc_run = T.doc_run;
    R.doc_sorted = T.doc_sorted;
  }
  dim3 g1(T.nq, T.Hm, T.Bm);
  mask_classify_kernel<<<g1, kThreads, 0, st>>>(R, T);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  dim3 g2(T.nk + (T.row_order ? 1 : 0), T.Hm, T.Bm);  // + one CTA per (b_m, h_m) for the row order
  mask_transpose_kernel<<<g2, kThreads, 0, st>>>(R, T);
  return cudaGetLastError();
}

cudaError_t launch_mask_select(const DevRule& R, const MaskOut& S, int Bz, const MaskOut& D, int32_t* status,
                               cudaStream_t st) {
  mask_select_kernel<<<dim3(Bz, D.Hm), kThreads, 0, st>>>(R, S, D, status);
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
