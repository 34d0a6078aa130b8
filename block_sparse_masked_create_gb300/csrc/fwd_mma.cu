// Block-sparse masked attention forward with warp-level mma.sync (m16n8k16, bf16 -> fp32).
//
// One CTA per (query block r, query head h, batch b); each warp owns 16 query rows. The CTA walks the
// BlockMask row of its query block: the full blocks (no mask), then the partial blocks (rule evaluated per
// element after the score rule) -- "5.1.2 FlexAttention: from rules to fused kernels", sections 2.2 and
// 3.1. K/V tiles of visited blocks only are copied into shared memory with cp.async (double buffered);
// empty blocks issue no loads. Online softmax per row in the exp2 domain; O = acc / l, LSE = m + ln l.
// This kernel serves block sizes other than 128 x 128 and is the independent cross-check of the
// tcgen05 kernel.
#include "fa_launch.h"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Byte offset of 16-byte chunk `ch` of row `row` in a [rows][D] bf16 tile with chunk ^= (row & 7).
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int ch) {
  return (uint32_t)(row * (D * 2) + ((ch ^ (row & 7)) << 4));
}

template <int D, int BQ, int BK>
struct MmaCfg {
  static constexpr int kWarps = BQ / 16;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kQBytes = BQ * D * 2;
  static constexpr int kKVBytes = BK * D * 2;
  static constexpr int kSmem = kQBytes + 4 * kKVBytes + BK * 4 /* doc ids */ + 64;
};

template <int D, int BQ, int BK>
__global__ void __launch_bounds__(MmaCfg<D, BQ, BK>::kThreads)
    fwd_mma_kernel(const __grid_constant__ FwdArgs a) {
  using C = MmaCfg<D, BQ, BK>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sQ = smem;
  uint8_t* sK = smem + C::kQBytes;                    // [2][BK][D]
  uint8_t* sV = sK + 2 * C::kKVBytes;                 // [2][BK][D]
  int32_t* sDoc = reinterpret_cast<int32_t*>(sV + 2 * C::kKVBytes);

  const int r = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = a.Hq / a.Hkv, hk = h / g;
  const DevMask& M = a.mask;
  const int bm = M.Bm > 1 ? b : 0, hm = M.Hm > 1 ? h : 0;
  const size_t mrow = ((size_t)bm * M.Hm + hm) * M.nq + r;
  const int n_full = __ldg(M.full_kv_num + mrow), n_part = __ldg(M.kv_num + mrow);
  const int n_vis = n_full + n_part;
  const int32_t* full_idx = M.full_kv_idx + mrow * M.nk;
  const int32_t* part_idx = M.kv_idx + mrow * M.nk;

  const __nv_bfloat16* Qg = reinterpret_cast<const __nv_bfloat16*>(a.q) + ((size_t)b * a.Hq + h) * a.q_len * D;
  const __nv_bfloat16* Kg = reinterpret_cast<const __nv_bfloat16*>(a.k) + ((size_t)b * a.Hkv + hk) * a.kv_len * D;
  const __nv_bfloat16* Vg = reinterpret_cast<const __nv_bfloat16*>(a.v) + ((size_t)b * a.Hkv + hk) * a.kv_len * D;
  __nv_bfloat16* Og = reinterpret_cast<__nv_bfloat16*>(a.out) + ((size_t)b * a.Hq + h) * a.q_len * D;
  float* Lg = a.lse + ((size_t)b * a.Hq + h) * a.q_len;

  if (tid == 0 && a.counters) {
    atomicAdd(reinterpret_cast<unsigned long long*>(a.counters) + 0, 1ull);
    atomicAdd(reinterpret_cast<unsigned long long*>(a.counters) + 1, (unsigned long long)n_full);
    atomicAdd(reinterpret_cast<unsigned long long*>(a.counters) + 2, (unsigned long long)n_part);
    atomicAdd(reinterpret_cast<unsigned long long*>(a.counters) + 3, (unsigned long long)(2 * n_vis));
  }

  const int q0 = r * BQ;
  // rows of this thread: ra (c0, c1) and ra + 8 (c2, c3)
  const int row_a = q0 + warp * 16 + (lane >> 2);
  const int row_b = row_a + 8;

  if (n_vis == 0) {  // empty row block: O = 0, LSE = -inf, no K/V loads
    const int kChunks = a.out_f32 ? D / 4 : D / 8;  // 16-byte chunks per row
    uint8_t* Ob = reinterpret_cast<uint8_t*>(a.out) + ((size_t)b * a.Hq + h) * a.q_len * D * (a.out_f32 ? 4 : 2);
    for (int x = tid; x < BQ * kChunks; x += C::kThreads) {
      int rr = x / kChunks, ch = x % kChunks;
      if (q0 + rr < a.q_len)
        *reinterpret_cast<uint4*>(Ob + ((size_t)(q0 + rr) * kChunks + ch) * 16) = make_uint4(0, 0, 0, 0);
    }
    for (int x = tid; x < BQ; x += C::kThreads)
      if (q0 + x < a.q_len) Lg[q0 + x] = -INFINITY;
    return;
  }

  // ---- Q tile -> shared memory (rows past q_len are zero)
  constexpr int kChunks = D / 8;
  for (int x = tid; x < BQ * kChunks; x += C::kThreads) {
    int rr = x / kChunks, ch = x % kChunks;
    bool ok = q0 + rr < a.q_len;
    const __nv_bfloat16* src = Qg + (size_t)(ok ? q0 + rr : 0) * D + ch * 8;
    cp_async_16(smem_u32(sQ) + swz<D>(rr, ch), src, ok);
  }
  cp_async_commit();

  auto load_kv = [&](int n, int stage) {
    const int c = n < n_full ? __ldg(full_idx + n) : __ldg(part_idx + n - n_full);
    const int j0 = c * BK;
    uint32_t kb = smem_u32(sK + stage * C::kKVBytes), vb = smem_u32(sV + stage * C::kKVBytes);
    const __nv_bfloat16* Kb = Kg;  // rows of the block start at Kb + row * D
    const __nv_bfloat16* Vb = Vg;
    int rbase = j0;
    if (a.page_table) {  // key block c is one whole page of BK rows; a bad id is reported and page 0 read
      int pg = __ldg(a.page_table + (size_t)b * a.max_pages + c);
      if (pg < 0 || pg >= a.n_pages_total) {
        if (tid == 0) report(a.status, FA_ERR_DEVICE_CHECK);
        pg = 0;
      }
      const size_t page_off = ((size_t)pg * a.Hkv + hk) * BK * D;
      Kb = reinterpret_cast<const __nv_bfloat16*>(a.k) + page_off;
      Vb = reinterpret_cast<const __nv_bfloat16*>(a.v) + page_off;
      rbase = 0;
    }
    for (int x = tid; x < BK * kChunks; x += C::kThreads) {
      int rr = x / kChunks, ch = x % kChunks;
      bool ok = j0 + rr < a.kv_len;
      size_t off = (size_t)(ok ? rbase + rr : 0) * D + ch * 8;
      cp_async_16(kb + swz<D>(rr, ch), Kb + off, ok);
      cp_async_16(vb + swz<D>(rr, ch), Vb + off, ok);
    }
  };

  load_kv(0, 0);
  cp_async_commit();

  // softmax state per row (log2 domain)
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f, le_a = 0.f, le_b = 0.f;
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  uint32_t qf[D / 16][4];

  const int64_t off_b = a.rule.q_offset ? (int64_t)__ldg(a.rule.q_offset + (M.Bm > 1 ? b : 0)) : 0;
  const int64_t ig_a = row_a + off_b, ig_b = row_b + off_b;
  const int doc_a = a.rule.any_doc ? doc_at(a.rule, bm, ig_a) : -1;
  const int doc_b = a.rule.any_doc ? doc_at(a.rule, bm, ig_b) : -1;
  const float scale_log2 = a.scale * kLog2e;
  const bool has_score = a.score.alibi || a.score.rel || a.score.softcap > 0.f;
  const float slope = a.score.alibi ? __ldg(a.score.alibi + h) : 0.f;

  for (int n = 0; n < n_vis; ++n) {
    const int stage = n & 1;
    if (n + 1 < n_vis) {
      load_kv(n + 1, stage ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    const bool partial = n >= n_full;
    const int c = partial ? __ldg(part_idx + n - n_full) : __ldg(full_idx + n);
    const int j0 = c * BK;
    if (partial && a.rule.any_doc) {
      for (int x = tid; x < BK; x += C::kThreads) sDoc[x] = doc_at(a.rule, bm, (int64_t)j0 + x);
    }
    __syncthreads();
    if (n == 0) {
      // Q fragments (A operand, row-major): matrices (rows 0-7|8-15) x (k 0-7|8-15)
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        int mi = lane >> 3, rr = warp * 16 + (mi & 1) * 8 + (lane & 7), ch = ks * 2 + (mi >> 1);
        ldsm_x4(smem_u32(sQ) + swz<D>(rr, ch), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
      }
    }
    const uint32_t kb = smem_u32(sK + stage * C::kKVBytes), vb = smem_u32(sV + stage * C::kKVBytes);

    // ---- S = Q K^T (fp32)
    float s[BK / 8][4];
#pragma unroll
    for (int i = 0; i < BK / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int nt = 0; nt < BK / 8; nt += 2) {
        int mi = lane >> 3, rr = nt * 8 + (mi >> 1) * 8 + (lane & 7), ch = ks * 2 + (mi & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + swz<D>(rr, ch), b0, b1, b2, b3);
        mma_bf16_16816(s[nt], qf[ks], b0, b1);
        mma_bf16_16816(s[nt + 1], qf[ks], b2, b3);
      }
    }

    // ---- scale, score rule, mask (partial blocks only); to the log2 domain
    Bits128 bits_a = {{~0u, ~0u, ~0u, ~0u}}, bits_b = bits_a;
    if (partial) {
      const int w = min(BK, a.kv_len - j0);
      auto docbits = [&](int d) { return doc_bits<(BK + 31) / 32>(w, d, [&](int c) { return sDoc[c]; }); };
      bits_a = row_a < a.q_len ? rule_row_bits(a.rule, ig_a, j0, w, doc_a, docbits) : Bits128{{0u, 0u, 0u, 0u}};
      bits_b = row_b < a.q_len ? rule_row_bits(a.rule, ig_b, j0, w, doc_b, docbits) : Bits128{{0u, 0u, 0u, 0u}};
    }
    float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < BK / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = nt * 8 + (lane & 3) * 2 + (e & 1);
        const bool upper = e >= 2;
        float x;
        if (has_score) {
          x = s[nt][e] * a.scale;
          const int64_t dist = (upper ? ig_b : ig_a) - (int64_t)(j0 + col);
          if (a.score.alibi) x -= slope * (float)dist;
          if (a.score.rel) {
            int64_t ix = dist + a.score.kv_len - 1;
            ix = ix < 0 ? 0 : (ix > 2 * (int64_t)a.score.kv_len - 2 ? 2 * (int64_t)a.score.kv_len - 2 : ix);
            x += __ldg(a.score.rel + (size_t)h * (2 * (size_t)a.score.kv_len - 1) + ix);
          }
          if (a.score.softcap > 0.f) x = softcap_apply(x, a.score.softcap, a.score.inv_softcap);
          x *= kLog2e;
        } else {
          x = s[nt][e] * scale_log2;
        }
        if (partial) {
          const Bits128& bb = upper ? bits_b : bits_a;
          if (!((bb.w[col >> 5] >> (col & 31)) & 1u)) x = -INFINITY;
        }
        s[nt][e] = x;
        if (upper) mx_b = fmaxf(mx_b, x); else mx_a = fmaxf(mx_a, x);
      }
    }
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xFFFFFFFFu, mx_a, 1));
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xFFFFFFFFu, mx_a, 2));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xFFFFFFFFu, mx_b, 1));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xFFFFFFFFu, mx_b, 2));
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float ref_a = mn_a == -INFINITY ? 0.f : mn_a, ref_b = mn_b == -INFINITY ? 0.f : mn_b;
    const float al_a = ex2_approx(m_a - ref_a), al_b = ex2_approx(m_b - ref_b);  // 0 when m was -inf
    m_a = mn_a;
    m_b = mn_b;
    float ps_a = 0.f, ps_b = 0.f, pe_a = 0.f, pe_b = 0.f;
    uint32_t pf[BK / 16][4];
#pragma unroll
    for (int nt = 0; nt < BK / 8; ++nt) {
      const float p0 = ex2_approx(s[nt][0] - ref_a), p1 = ex2_approx(s[nt][1] - ref_a);
      const float p2 = ex2_approx(s[nt][2] - ref_b), p3 = ex2_approx(s[nt][3] - ref_b);
      // C-fragment of n-tiles (2k, 2k+1) -> A-fragment of k-step k. Two row sums: of the rounded P the
      // P V product sees (normalises O: an exact convex combination of V rows) and of the unrounded P (LSE)
      const uint32_t pa = pack_bf16x2(p0, p1), pb = pack_bf16x2(p2, p3);
      pf[nt >> 1][(nt & 1) * 2 + 0] = pa;
      pf[nt >> 1][(nt & 1) * 2 + 1] = pb;
      ps_a += bf16x2_sum(pa);
      ps_b += bf16x2_sum(pb);
      pe_a += p0 + p1;
      pe_b += p2 + p3;
    }
    l_a = l_a * al_a + ps_a;
    l_b = l_b * al_b + ps_b;
    le_a = le_a * al_a + pe_a;
    le_b = le_b * al_b + pe_b;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) {
      o[dt][0] *= al_a;
      o[dt][1] *= al_a;
      o[dt][2] *= al_b;
      o[dt][3] *= al_b;
    }
    // ---- O += P V
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
#pragma unroll
      for (int dt = 0; dt < D / 8; dt += 2) {
        int mi = lane >> 3, rr = kk * 16 + (mi & 1) * 8 + (lane & 7), ch = dt + (mi >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swz<D>(rr, ch), b0, b1, b2, b3);
        mma_bf16_16816(o[dt], pf[kk], b0, b1);
        mma_bf16_16816(o[dt + 1], pf[kk], b2, b3);
      }
    }
    __syncthreads();  // this stage is refilled by the next iteration's prefetch
  }

  // ---- epilogue: row sums across the 4 lanes of a row, O / l, LSE
  l_a += __shfl_xor_sync(0xFFFFFFFFu, l_a, 1);
  l_a += __shfl_xor_sync(0xFFFFFFFFu, l_a, 2);
  l_b += __shfl_xor_sync(0xFFFFFFFFu, l_b, 1);
  l_b += __shfl_xor_sync(0xFFFFFFFFu, l_b, 2);
  le_a += __shfl_xor_sync(0xFFFFFFFFu, le_a, 1);
  le_a += __shfl_xor_sync(0xFFFFFFFFu, le_a, 2);
  le_b += __shfl_xor_sync(0xFFFFFFFFu, le_b, 1);
  le_b += __shfl_xor_sync(0xFFFFFFFFu, le_b, 2);
  const bool emp_a = m_a == -INFINITY, emp_b = m_b == -INFINITY;
  const float inv_a = emp_a ? 0.f : 1.f / l_a, inv_b = emp_b ? 0.f : 1.f / l_b;
  if ((lane & 3) == 0) {
    if (row_a < a.q_len) Lg[row_a] = emp_a ? -INFINITY : (m_a + __log2f(le_a)) * kLn2;
    if (row_b < a.q_len) Lg[row_b] = emp_b ? -INFINITY : (m_b + __log2f(le_b)) * kLn2;
  }
  if (a.out_f32) {
    float* Of = reinterpret_cast<float*>(a.out) + ((size_t)b * a.Hq + h) * a.q_len * D;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) {
      const int col = dt * 8 + (lane & 3) * 2;
      if (row_a < a.q_len) *reinterpret_cast<float2*>(Of + (size_t)row_a * D + col) = make_float2(o[dt][0] * inv_a, o[dt][1] * inv_a);
      if (row_b < a.q_len) *reinterpret_cast<float2*>(Of + (size_t)row_b * D + col) = make_float2(o[dt][2] * inv_b, o[dt][3] * inv_b);
    }
    return;
  }
  // stage O through this warp's own Q rows in shared memory, then 16-byte coalesced stores
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) {
    const int col = dt * 8 + (lane & 3) * 2;
    const int ra = warp * 16 + (lane >> 2), rb = ra + 8;
    *reinterpret_cast<uint32_t*>(sQ + swz<D>(ra, col >> 3) + (col & 7) * 2) = pack_bf16x2(o[dt][0] * inv_a, o[dt][1] * inv_a);
    *reinterpret_cast<uint32_t*>(sQ + swz<D>(rb, col >> 3) + (col & 7) * 2) = pack_bf16x2(o[dt][2] * inv_b, o[dt][3] * inv_b);
  }
  __syncwarp();
  for (int x = lane; x < 16 * kChunks; x += 32) {
    const int rr = warp * 16 + x / kChunks, ch = x % kChunks;
    if (q0 + rr < a.q_len)
      *reinterpret_cast<uint4*>(Og + (size_t)(q0 + rr) * D + ch * 8) = *reinterpret_cast<const uint4*>(sQ + swz<D>(rr, ch));
  }
}

template <int D, int BQ, int BK>
cudaError_t launch_one(const FwdArgs& a, cudaStream_t st) {
  using C = MmaCfg<D, BQ, BK>;
  auto kern = fwd_mma_kernel<D, BQ, BK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.mask.nq, a.Hq, a.B);
  kern<<<grid, C::kThreads, C::kSmem, st>>>(a);
  return cudaGetLastError();
}

template <int D, int BQ>
cudaError_t launch_bk(const FwdArgs& a, cudaStream_t st) {
  switch (a.mask.bk) {
    case 16: return launch_one<D, BQ, 16>(a, st);
    case 32: return launch_one<D, BQ, 32>(a, st);
    case 64: return launch_one<D, BQ, 64>(a, st);
    case 128: return launch_one<D, BQ, 128>(a, st);
  }
  return cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_bq(const FwdArgs& a, cudaStream_t st) {
  switch (a.mask.bq) {
    case 16: return launch_bk<D, 16>(a, st);
    case 32: return launch_bk<D, 32>(a, st);
    case 64: return launch_bk<D, 64>(a, st);
    case 128: return launch_bk<D, 128>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_fwd_mma(const FwdArgs& a, cudaStream_t st) {
  if (a.d == 64) return launch_bq<64>(a, st);
  if (a.d == 128) return launch_bq<128>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace fa
