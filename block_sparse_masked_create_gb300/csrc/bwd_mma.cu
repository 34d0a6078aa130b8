// Backward of the block-sparse masked attention forward, with warp-level mma.sync (m16n8k16, bf16 ->
// fp32). What it computes (FlashAttention self-test questions on the backward pass; "5.1.2 FlexAttention:
// from rules to fused kernels", section 4.2, the backward reusing the BlockMask and its transpose):
//   P = exp(s' - LSE) recomputed from the forward's LSE, s' = score rule (scale q.k), masked pairs 0;
//   D_i = sum_d dO_id O_id;  dV = P^T dO;  dP = dO V^T;  dS = P (dP - D) times ds'/ds (1 - (s'/c)^2 under
//   the soft-cap c);  dQ = scale dS K;  dK = scale dS^T Q; dK, dV summed over the query heads of a KV head.
// Three launches, no atomics:
//   delta: one warp per query row, D_i.
//   dQ:    one CTA per 64 query rows (4 warps x 16 rows); walks the BlockMask row of its query block (full
//          blocks, then partial ones with the rule evaluated per pair), 64 key columns at a time, K / V
//          chunks double-buffered with cp.async; dQ accumulates in registers.
//   dK/dV: one CTA per 64 key rows of one KV head; for every query head of the group, walks the column of
//          its key block in the query-side transpose, 64 query rows at a time (Q, dO, LSE, D chunks
//          double-buffered); dK and dV accumulate in registers.
#include "fa_launch.h"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBwdThreads = 128;  // 4 warps x 16 rows = 64 rows per CTA

// Byte offset of 16-byte chunk `ch` of row `row` in a [64][D] bf16 tile, chunk ^= (row & 7).
template <int D>
__device__ __forceinline__ uint32_t swzb(int row, int ch) {
  return (uint32_t)(row * (D * 2) + ((ch ^ (row & 7)) << 4));
}

// rows [r0, r0 + 64) of a [n][D] bf16 tensor into a swizzled tile; rows past n read as zero
template <int D>
__device__ __forceinline__ void load_tile64(uint8_t* dst, const __nv_bfloat16* src, int r0, int n) {
  constexpr int kChunks = D / 8;
  for (int x = threadIdx.x; x < 64 * kChunks; x += kBwdThreads) {
    const int rr = x / kChunks, ch = x % kChunks;
    const bool ok = r0 + rr < n;
    cp_async_16(smem_u32(dst) + swzb<D>(rr, ch), src + (size_t)(ok ? r0 + rr : 0) * D + ch * 8, ok);
  }
}

// C[16 x 64] += A[16 rows of a] . B[64 rows of b]^T over D (both tiles [rows][D] swizzled, K-major):
// S = Q K^T and dP = dO V^T shapes. Fragments of the four 8-row column groups pairs as in mma m16n8k16.
template <int D>
__device__ __forceinline__ void mma_abt(float (&c)[8][4], uint32_t a_tile, int a_row0, uint32_t b_tile) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    uint32_t af[4];
    {
      const int mi = lane >> 3, rr = a_row0 + (mi & 1) * 8 + (lane & 7), ch = ks * 2 + (mi >> 1);
      ldsm_x4(a_tile + swzb<D>(rr, ch), af[0], af[1], af[2], af[3]);
    }
#pragma unroll
    for (int nt = 0; nt < 8; nt += 2) {
      const int mi = lane >> 3, rr = nt * 8 + (mi >> 1) * 8 + (lane & 7), ch = ks * 2 + (mi & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(b_tile + swzb<D>(rr, ch), b0, b1, b2, b3);
      mma_bf16_16816(c[nt], af, b0, b1);
      mma_bf16_16816(c[nt + 1], af, b2, b3);
    }
  }
}

// acc[16 x D] += A[16 x 64] (bf16 A-fragments, 4 k-steps) . B[64 rows][D] (tile rows are the k index)
template <int D>
__device__ __forceinline__ void mma_ab(float (&acc)[D / 8][4], const uint32_t (&af)[4][4], uint32_t b_tile) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
    for (int dt = 0; dt < D / 8; dt += 2) {
      const int mi = lane >> 3, rr = kk * 16 + (mi & 1) * 8 + (lane & 7), ch = dt + (mi >> 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(b_tile + swzb<D>(rr, ch), b0, b1, b2, b3);
      mma_bf16_16816(acc[dt], af[kk], b0, b1);
      mma_bf16_16816(acc[dt + 1], af[kk], b2, b3);
    }
  }
}

// The score rule on a scaled score (ALiBi, relative bias, then soft-cap); *g = ds'/ds.
__device__ __forceinline__ float score_and_slope(const DevScore& sc, int h, float x, int64_t dist, float slope,
                                                 float* g) {
  if (sc.alibi) x -= slope * (float)dist;
  if (sc.rel) {
    int64_t ix = dist + sc.kv_len - 1;
    ix = ix < 0 ? 0 : (ix > 2 * (int64_t)sc.kv_len - 2 ? 2 * (int64_t)sc.kv_len - 2 : ix);
    x += __ldg(sc.rel + (size_t)h * (2 * (size_t)sc.kv_len - 1) + ix);
  }
  *g = 1.f;
  if (sc.softcap > 0.f) {
    x = softcap_apply(x, sc.softcap, sc.inv_softcap);
    const float t = x * sc.inv_softcap;
    *g = 1.f - t * t;
  }
  return x;
}

// ---------------------------------------------------------------------------------------------- delta
__global__ void __launch_bounds__(256) bwd_delta_kernel(const __grid_constant__ BwdArgs a) {
  const long long rows = (long long)a.B * a.Hq * a.q_len;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const __nv_bfloat16* dO = reinterpret_cast<const __nv_bfloat16*>(a.dout) + row * a.d;
  float acc = 0.f;
  if (a.out_f32) {
    const float* O = reinterpret_cast<const float*>(a.out) + row * a.d;
    for (int c = lane; c < a.d; c += 32) acc += __bfloat162float(dO[c]) * O[c];
  } else {
    const __nv_bfloat16* O = reinterpret_cast<const __nv_bfloat16*>(a.out) + row * a.d;
    for (int c = lane; c < a.d; c += 32) acc += __bfloat162float(dO[c]) * __bfloat162float(O[c]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  if (lane == 0) a.delta[row] = acc;
}

// ---------------------------------------------------------------------------------------------- dQ
template <int D>
struct BwdCfg {
  static constexpr int kTile = 64 * D * 2;                 // one [64][D] bf16 tile
  // 2 fixed tiles + 2 x 2 streamed tiles, then per stage 64 LSE, 64 delta and 64 document ids
  static constexpr int kSmem = 6 * kTile + 3 * 2 * 64 * 4;
};

template <int D, int BQ, int BK>
__global__ void __launch_bounds__(kBwdThreads) bwd_dq_kernel(const __grid_constant__ BwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sQ = smem;
  uint8_t* sdO = smem + C::kTile;
  uint8_t* sK = smem + 2 * C::kTile;  // [2][64][D]
  uint8_t* sV = smem + 4 * C::kTile;  // [2][64][D]
  int32_t* sDoc = reinterpret_cast<int32_t*>(smem + 6 * C::kTile);  // [2][64]

  const int q0 = blockIdx.x * 64, h = blockIdx.y, b = blockIdx.z;
  const int r = q0 / BQ;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hk = h / (a.Hq / a.Hkv);
  const DevMask& M = a.mask;
  const int bm = M.Bm > 1 ? b : 0, hm = M.Hm > 1 ? h : 0;
  const size_t mrow = ((size_t)bm * M.Hm + hm) * M.nq + r;
  const int n_full = __ldg(M.full_kv_num + mrow), n_vis = n_full + __ldg(M.kv_num + mrow);
  const int32_t* full_idx = M.full_kv_idx + mrow * M.nk;
  const int32_t* part_idx = M.kv_idx + mrow * M.nk;
  constexpr int kCh = BK / 64;  // 64-column chunks per key block
  const int n_chunks = n_vis * kCh;

  const __nv_bfloat16* Qg = reinterpret_cast<const __nv_bfloat16*>(a.q) + ((size_t)b * a.Hq + h) * a.q_len * D;
  const __nv_bfloat16* dOg = reinterpret_cast<const __nv_bfloat16*>(a.dout) + ((size_t)b * a.Hq + h) * a.q_len * D;
  const __nv_bfloat16* Kg = reinterpret_cast<const __nv_bfloat16*>(a.k) + ((size_t)b * a.Hkv + hk) * a.kv_len * D;
  const __nv_bfloat16* Vg = reinterpret_cast<const __nv_bfloat16*>(a.v) + ((size_t)b * a.Hkv + hk) * a.kv_len * D;
  const float* Lg = a.lse + ((size_t)b * a.Hq + h) * a.q_len;
  const float* Dg = a.delta + ((size_t)b * a.Hq + h) * a.q_len;

  const int row_a = q0 + warp * 16 + (lane >> 2), row_b = row_a + 8;
  float dq[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;

  if (n_chunks > 0) {
    load_tile64<D>(sQ, Qg, q0, a.q_len);
    load_tile64<D>(sdO, dOg, q0, a.q_len);
    cp_async_commit();
    auto chunk_col = [&](int n, bool& partial) {
      const int nb = n / kCh;
      partial = nb >= n_full;
      const int c = partial ? __ldg(part_idx + nb - n_full) : __ldg(full_idx + nb);
      return c * BK + (n % kCh) * 64;
    };
    auto load_chunk = [&](int n, int stage) {
      bool partial;
      const int j0 = chunk_col(n, partial);
      load_tile64<D>(sK + stage * C::kTile, Kg, j0, a.kv_len);
      load_tile64<D>(sV + stage * C::kTile, Vg, j0, a.kv_len);
      if (partial && a.rule.any_doc)
        for (int x = threadIdx.x; x < 64; x += kBwdThreads) sDoc[stage * 64 + x] = doc_at(a.rule, bm, (int64_t)j0 + x);
    };
    load_chunk(0, 0);
    cp_async_commit();

    const int64_t off_b = a.rule.q_offset ? (int64_t)__ldg(a.rule.q_offset + (M.Bm > 1 ? b : 0)) : 0;
    const int64_t ig_a = row_a + off_b, ig_b = row_b + off_b;
    const int doc_a = a.rule.any_doc ? doc_at(a.rule, bm, ig_a) : -1;
    const int doc_b = a.rule.any_doc ? doc_at(a.rule, bm, ig_b) : -1;
    const bool in_a = row_a < a.q_len, in_b = row_b < a.q_len;
    const float la = in_a ? __ldg(Lg + row_a) * kLog2e : -INFINITY, lb = in_b ? __ldg(Lg + row_b) * kLog2e : -INFINITY;
    const float da = in_a ? __ldg(Dg + row_a) : 0.f, db = in_b ? __ldg(Dg + row_b) : 0.f;
    const float slope = a.score.alibi ? __ldg(a.score.alibi + h) : 0.f;

    for (int n = 0; n < n_chunks; ++n) {
      const int stage = n & 1;
      if (n + 1 < n_chunks) {
        load_chunk(n + 1, stage ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();
      bool partial;
      const int j0 = chunk_col(n, partial);
      const uint32_t kb = smem_u32(sK + stage * C::kTile), vb = smem_u32(sV + stage * C::kTile);
      float s[8][4], dp[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = dp[i][0] = dp[i][1] = dp[i][2] = dp[i][3] = 0.f;
      mma_abt<D>(s, smem_u32(sQ), warp * 16, kb);
      mma_abt<D>(dp, smem_u32(sdO), warp * 16, vb);
      Bits128 bits_a = {{~0u, ~0u, ~0u, ~0u}}, bits_b = bits_a;
      const int w = min(64, a.kv_len - j0);
      if (partial) {
        const int* cdoc = sDoc + stage * 64;
        auto docbits = [&](int d) { return doc_bits<2>(w, d, [&](int c) { return cdoc[c]; }); };
        bits_a = in_a ? rule_row_bits(a.rule, ig_a, j0, w, doc_a, docbits) : Bits128{{0u, 0u, 0u, 0u}};
        bits_b = in_b ? rule_row_bits(a.rule, ig_b, j0, w, doc_b, docbits) : Bits128{{0u, 0u, 0u, 0u}};
      }
      uint32_t dsf[4][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = nt * 8 + (lane & 3) * 2 + (e & 1);
          const bool upper = e >= 2;
          const float lrow = upper ? lb : la;
          bool ok = col < w && lrow != -INFINITY;
          if (partial) {
            const Bits128& bb = upper ? bits_b : bits_a;
            ok = ok && ((bb.w[col >> 5] >> (col & 31)) & 1u);
          }
          float gsc;
          const float x = score_and_slope(a.score, h, s[nt][e] * a.scale, (upper ? ig_b : ig_a) - (int64_t)(j0 + col),
                                          slope, &gsc);
          const float p = ok ? ex2_approx(x * kLog2e - lrow) : 0.f;
          v[e] = p * (dp[nt][e] - (upper ? db : da)) * gsc;
        }
        dsf[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(v[0], v[1]);
        dsf[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(v[2], v[3]);
      }
      mma_ab<D>(dq, dsf, kb);
      __syncthreads();  // this stage is refilled by the next iteration's prefetch
    }
  }
  // dQ = scale * dS K, fp32 (rows past q_len and empty rows: written as computed, i.e. zero)
  float* dQg = a.dq + ((size_t)b * a.Hq + h) * a.q_len * D;
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) {
    const int col = dt * 8 + (lane & 3) * 2;
    if (row_a < a.q_len) *reinterpret_cast<float2*>(dQg + (size_t)row_a * D + col) = make_float2(dq[dt][0] * a.scale, dq[dt][1] * a.scale);
    if (row_b < a.q_len) *reinterpret_cast<float2*>(dQg + (size_t)row_b * D + col) = make_float2(dq[dt][2] * a.scale, dq[dt][3] * a.scale);
  }
}

// ---------------------------------------------------------------------------------------------- dK, dV
template <int D, int BQ, int BK>
__global__ void __launch_bounds__(kBwdThreads) bwd_dkdv_kernel(const __grid_constant__ BwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::kTile;
  uint8_t* sQ = smem + 2 * C::kTile;   // [2][64][D]
  uint8_t* sdO = smem + 4 * C::kTile;  // [2][64][D]
  float* sL = reinterpret_cast<float*>(smem + 6 * C::kTile);  // [2][64] LSE (log2 domain)
  float* sD = sL + 128;                                         // [2][64] delta
  int32_t* sDocQ = reinterpret_cast<int32_t*>(sD + 128);        // [2][64]

  const int j0 = blockIdx.x * 64, hk = blockIdx.y, b = blockIdx.z;
  const int c = j0 / BK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = a.Hq / a.Hkv;
  const DevMask& M = a.mask;
  const int bm = M.Bm > 1 ? b : 0;
  constexpr int kCh = BQ / 64;  // 64-row chunks per query block

  const __nv_bfloat16* Kg = reinterpret_cast<const __nv_bfloat16*>(a.k) + ((size_t)b * a.Hkv + hk) * a.kv_len * D;
  const __nv_bfloat16* Vg = reinterpret_cast<const __nv_bfloat16*>(a.v) + ((size_t)b * a.Hkv + hk) * a.kv_len * D;
  load_tile64<D>(sK, Kg, j0, a.kv_len);
  load_tile64<D>(sV, Vg, j0, a.kv_len);
  cp_async_commit();

  const int row_a = j0 + warp * 16 + (lane >> 2), row_b = row_a + 8;  // key rows of this thread
  const bool in_a = row_a < a.kv_len, in_b = row_b < a.kv_len;
  const int docj_a = (a.rule.any_doc && in_a) ? doc_at(a.rule, bm, row_a) : -1;
  const int docj_b = (a.rule.any_doc && in_b) ? doc_at(a.rule, bm, row_b) : -1;
  const int64_t off_b = a.rule.q_offset ? (int64_t)__ldg(a.rule.q_offset + (M.Bm > 1 ? b : 0)) : 0;

  float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) dk[i][0] = dk[i][1] = dk[i][2] = dk[i][3] = dv[i][0] = dv[i][1] = dv[i][2] = dv[i][3] = 0.f;

  for (int gi = 0; gi < g; ++gi) {
    const int h = hk * g + gi;
    const int hm = M.Hm > 1 ? h : 0;
    const size_t mcol = ((size_t)bm * M.Hm + hm) * M.nk + c;
    const int n_full = __ldg(M.full_q_num + mcol), n_vis = n_full + __ldg(M.q_num + mcol);
    const int32_t* full_idx = M.full_q_idx + mcol * M.nq;
    const int32_t* part_idx = M.q_idx + mcol * M.nq;
    const int n_chunks = n_vis * kCh;
    if (n_chunks == 0) continue;
    const __nv_bfloat16* Qg = reinterpret_cast<const __nv_bfloat16*>(a.q) + ((size_t)b * a.Hq + h) * a.q_len * D;
    const __nv_bfloat16* dOg = reinterpret_cast<const __nv_bfloat16*>(a.dout) + ((size_t)b * a.Hq + h) * a.q_len * D;
    const float* Lg = a.lse + ((size_t)b * a.Hq + h) * a.q_len;
    const float* Dg = a.delta + ((size_t)b * a.Hq + h) * a.q_len;
    const float slope = a.score.alibi ? __ldg(a.score.alibi + h) : 0.f;
    auto chunk_row = [&](int n, bool& partial) {
      const int nb = n / kCh;
      partial = nb >= n_full;
      const int r = partial ? __ldg(part_idx + nb - n_full) : __ldg(full_idx + nb);
      return r * BQ + (n % kCh) * 64;
    };
    auto load_chunk = [&](int n, int stage) {
      bool partial;
      const int i0 = chunk_row(n, partial);
      load_tile64<D>(sQ + stage * C::kTile, Qg, i0, a.q_len);
      load_tile64<D>(sdO + stage * C::kTile, dOg, i0, a.q_len);
      for (int x = threadIdx.x; x < 64; x += kBwdThreads) {
        const bool ok = i0 + x < a.q_len;
        sL[stage * 64 + x] = ok ? __ldg(Lg + i0 + x) * kLog2e : -INFINITY;
        sD[stage * 64 + x] = ok ? __ldg(Dg + i0 + x) : 0.f;
        if (partial && a.rule.any_doc) sDocQ[stage * 64 + x] = doc_at(a.rule, bm, (int64_t)i0 + x + off_b);
      }
    };
    __syncthreads();  // the previous head's last chunk is no longer read
    load_chunk(0, 0);
    cp_async_commit();
    for (int n = 0; n < n_chunks; ++n) {
      const int stage = n & 1;
      if (n + 1 < n_chunks) {
        load_chunk(n + 1, stage ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();
      bool partial;
      const int i0 = chunk_row(n, partial);
      const uint32_t qb = smem_u32(sQ + stage * C::kTile), ob = smem_u32(sdO + stage * C::kTile);
      // S^T = K Q^T and dP^T = V dO^T: rows are this warp's 16 keys, columns the chunk's 64 queries
      float st[8][4], dpt[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) st[i][0] = st[i][1] = st[i][2] = st[i][3] = dpt[i][0] = dpt[i][1] = dpt[i][2] = dpt[i][3] = 0.f;
      mma_abt<D>(st, smem_u32(sK), warp * 16, qb);
      mma_abt<D>(dpt, smem_u32(sV), warp * 16, ob);
      uint32_t pf[4][4], dsf[4][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        float pv[4], dsv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = nt * 8 + (lane & 3) * 2 + (e & 1);  // query row i0 + col
          const bool upper = e >= 2;
          const int j = upper ? row_b : row_a;
          const int64_t ig = (int64_t)i0 + col + off_b;
          const float lrow = sL[stage * 64 + col];
          bool ok = (upper ? in_b : in_a) && lrow != -INFINITY;
          if (partial) ok = ok && rule_allows(a.rule, ig, j, a.rule.any_doc ? sDocQ[stage * 64 + col] : -1, upper ? docj_b : docj_a);
          float gsc;
          const float x = score_and_slope(a.score, h, st[nt][e] * a.scale, ig - j, slope, &gsc);
          const float p = ok ? ex2_approx(x * kLog2e - lrow) : 0.f;
          pv[e] = p;
          dsv[e] = p * (dpt[nt][e] - sD[stage * 64 + col]) * gsc;
        }
        pf[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(pv[0], pv[1]);
        pf[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(pv[2], pv[3]);
        dsf[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(dsv[0], dsv[1]);
        dsf[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(dsv[2], dsv[3]);
      }
      mma_ab<D>(dv, pf, ob);   // dV += P^T dO
      mma_ab<D>(dk, dsf, qb);  // dK += dS^T Q
      __syncthreads();  // this stage is refilled by the next iteration's prefetch
    }
  }
  cp_async_wait<0>();  // K / V of a CTA that visited nothing
  float* dKg = a.dk + ((size_t)b * a.Hkv + hk) * a.kv_len * D;
  float* dVg = a.dv + ((size_t)b * a.Hkv + hk) * a.kv_len * D;
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) {
    const int col = dt * 8 + (lane & 3) * 2;
    if (in_a) {
      *reinterpret_cast<float2*>(dKg + (size_t)row_a * D + col) = make_float2(dk[dt][0] * a.scale, dk[dt][1] * a.scale);
      *reinterpret_cast<float2*>(dVg + (size_t)row_a * D + col) = make_float2(dv[dt][0], dv[dt][1]);
    }
    if (in_b) {
      *reinterpret_cast<float2*>(dKg + (size_t)row_b * D + col) = make_float2(dk[dt][2] * a.scale, dk[dt][3] * a.scale);
      *reinterpret_cast<float2*>(dVg + (size_t)row_b * D + col) = make_float2(dv[dt][2], dv[dt][3]);
    }
  }
}

template <int D, int BQ, int BK>
cudaError_t launch_shapes(const BwdArgs& a, cudaStream_t st) {
  using C = BwdCfg<D>;
  auto kq = bwd_dq_kernel<D, BQ, BK>;
  auto kk = bwd_dkdv_kernel<D, BQ, BK>;
  cudaError_t e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  kq<<<dim3((a.q_len + 63) / 64, a.Hq, a.B), kBwdThreads, C::kSmem, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kk<<<dim3((a.kv_len + 63) / 64, a.Hkv, a.B), kBwdThreads, C::kSmem, st>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const BwdArgs& a, cudaStream_t st) {
  const int bq = a.mask.bq, bk = a.mask.bk;
  if (bq == 64 && bk == 64) return launch_shapes<D, 64, 64>(a, st);
  if (bq == 64 && bk == 128) return launch_shapes<D, 64, 128>(a, st);
  if (bq == 128 && bk == 64) return launch_shapes<D, 128, 64>(a, st);
  if (bq == 128 && bk == 128) return launch_shapes<D, 128, 128>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_backward(const BwdArgs& a, cudaStream_t st) {
  const long long rows = (long long)a.B * a.Hq * a.q_len;
  bwd_delta_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int t = launch_bwd_tc5(a, st);
  if (t == FA_OK) return cudaSuccess;
  if (t != FA_ERR_UNSUPPORTED) return cudaErrorLaunchFailure;
  if (a.d == 64) return launch_d<64>(a, st);
  if (a.d == 128) return launch_d<128>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace fa
