// Paged split-KV decode ("5.1.2 FlexAttention: from rules to fused kernels", sections 3.2 and 5.1-5.2;
// "FlexAttention: compiler optimisation of custom attention", section 6; merge law of "5 Kernels:
// turning logical sparsity into real speed-ups", section 3).
//
// Kernel 1: one CTA per (split s, KV head hk, request b). The CTA takes pages [s*PS, (s+1)*PS) of the
// request's visit list (its BlockMask row: full blocks, then partial blocks) and serves all g = Hq/Hkv
// query heads of hk at once, so every K/V byte is read once. Logical block c is physical page
// page_table[b][c] (the gather is fused: no KV copy). Each of the 4 warps streams 32-token sub-tiles of
// those pages through its own 3-stage TMA ring (128-byte swizzle), computes S = Q K^T and O += P V with
// mma.sync (the g query heads are rows of a 16-row tile), and keeps an online-softmax state; the warps'
// states are merged in shared memory and written as (m_s, l_s, u_s) (u unnormalised, log2 domain).
// Kernel 2: one CTA per (query head, request) merges its splits: m = max m_s, l = sum 2^(m_s-m) l_s,
// O = sum 2^(m_s-m) u_s / l, LSE = (m + log2 l) ln 2. A request with no visible block writes O = 0,
// LSE = -inf; a split with no block is never read.
#include "fa_launch.h"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kDecWarps = 4;
constexpr int kSub = 32;   // tokens per sub-tile
constexpr int kStages = 3;

template <int D>
struct DecCfg {
  static constexpr int kBoxBytes = kSub * 128;                 // one [32][64] bf16 box
  static constexpr int kTileBytes = kSub * D * 2;              // K or V sub-tile
  static constexpr int kStageBytes = 2 * kTileBytes;           // K + V
  static constexpr int kWarpBytes = kStages * kStageBytes;
  static constexpr int kSmem = kDecWarps * kWarpBytes + 1024 /* alignment slack */ + 256;
};

// byte offset of 16-byte chunk c16 (0 .. D/8-1) of row `row` in a TMA-written [32][D] sub-tile made of
// D/64 boxes of [32][64] with the 128-byte swizzle (chunk ^= row & 7 inside each box)
__device__ __forceinline__ uint32_t dswz(int row, int c16) {
  return (uint32_t)((c16 >> 3) * (kSub * 128) + row * 128 + (((c16 & 7) ^ (row & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kDecWarps * 32)
    decode_split_kernel(const __grid_constant__ DecArgs a, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, int PAGE) {
  using C = DecCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bars[kDecWarps][kStages];
  __shared__ int32_t s_abort;

  const int s = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = a.Hq / a.Hkv;
  const DevMask& M = a.mask;
  const int bm = M.Bm > 1 ? b : 0;
  const size_t mrow = (size_t)bm * M.Hm * M.nq;  // Hm == 1, nq == 1
  const int n_full = __ldg(M.full_kv_num + mrow), n_part = __ldg(M.kv_num + mrow);
  const int n_vis = n_full + n_part;
  const int e0 = s * a.pages_per_split;
  if (e0 >= n_vis) return;  // this split has no block: the combine never reads it
  const int e1 = min(n_vis, e0 + a.pages_per_split);
  const int32_t* full_idx = M.full_kv_idx + mrow * M.nk;
  const int32_t* part_idx = M.kv_idx + mrow * M.nk;
  const int subs_per_page = PAGE / kSub;
  const int n_sub = (e1 - e0) * subs_per_page;

  if (tid == 0) {
    s_abort = 0;
    for (int w = 0; w < kDecWarps; ++w)
      for (int st = 0; st < kStages; ++st) mbar_init(&bars[w][st], 1);
    fence_mbar_init();
    if (a.counters) {
      atomicAdd(reinterpret_cast<unsigned long long*>(a.counters) + 0, 1ull);
      int nf = max(0, min(e1, n_full) - e0), np = (e1 - e0) - nf;
      atomicAdd(reinterpret_cast<unsigned long long*>(a.counters) + 1, (unsigned long long)nf);
      atomicAdd(reinterpret_cast<unsigned long long*>(a.counters) + 2, (unsigned long long)np);
      atomicAdd(reinterpret_cast<unsigned long long*>(a.counters) + 3, (unsigned long long)(2 * (e1 - e0)));
    }
  }
  if (tid == 32) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  __syncthreads();
  WaitCtl wc{a.timeout_ns, a.status, &s_abort};

  uint8_t* my = smem + warp * C::kWarpBytes;
  // sub-tiles of this warp: u = warp, warp + 4, ...
  const int my_count = warp < n_sub ? (n_sub - warp + kDecWarps - 1) / kDecWarps : 0;

  // resolve sub-tile -> (logical block c, token offset, physical page or -1)
  auto sub_info = [&](int k, int& c, int& t0, int& pid) {
    const int u = warp + k * kDecWarps;
    const int e = e0 + u / subs_per_page;
    t0 = (u % subs_per_page) * kSub;
    c = e < n_full ? __ldg(full_idx + e) : __ldg(part_idx + e - n_full);
    pid = __ldg(a.page_table + (size_t)b * a.max_pages + c);
    if (pid < 0 || pid >= a.n_pages_total) pid = -1;
  };
  auto issue = [&](int k) {  // lane 0 only
    int c, t0, pid;
    sub_info(k, c, t0, pid);
    uint64_t* bar = &bars[warp][k % kStages];
    uint8_t* st = my + (k % kStages) * C::kStageBytes;
    if (pid < 0) {
      report(a.status, FA_ERR_DEVICE_CHECK);
      mbar_arrive(bar);
      return;
    }
    mbar_arrive_expect_tx(bar, C::kStageBytes);
    const int yrow = (pid * a.Hkv + hk) * PAGE + t0;
#pragma unroll
    for (int x = 0; x < D / 64; ++x) {
      tma_load_2d(st + x * C::kBoxBytes, &tmK, x * 64, yrow, bar);
      tma_load_2d(st + C::kTileBytes + x * C::kBoxBytes, &tmV, x * 64, yrow, bar);
    }
  };
  if (lane == 0)
    for (int k = 0; k < min(kStages, my_count); ++k) issue(k);

  // Q fragments: row = query head hk*g + row (rows >= g are zero)
  const int ra = lane >> 2, rb = ra + 8;
  const __nv_bfloat16* Qb = reinterpret_cast<const __nv_bfloat16*>(a.q) + ((size_t)b * a.Hq + (size_t)hk * g) * D;
  uint32_t qf[D / 16][4];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int k0 = ks * 16 + (lane & 3) * 2;
    auto ld = [&](int row, int col) -> uint32_t {
      return row < g ? *reinterpret_cast<const uint32_t*>(Qb + (size_t)row * D + col) : 0u;
    };
    qf[ks][0] = ld(ra, k0);
    qf[ks][1] = ld(rb, k0);
    qf[ks][2] = ld(ra, k0 + 8);
    qf[ks][3] = ld(rb, k0 + 8);
  }
  const int64_t ig = a.rule.q_offset ? (int64_t)__ldg(a.rule.q_offset + (M.Bm > 1 ? b : 0)) : 0;
  const int doc_i = a.rule.any_doc ? doc_at(a.rule, bm, ig) : -1;
  const bool has_score = a.score.alibi || a.score.rel || a.score.softcap > 0.f;
  const float slope_a = (a.score.alibi && ra < g) ? __ldg(a.score.alibi + hk * g + ra) : 0.f;
  const float slope_b = (a.score.alibi && rb < g) ? __ldg(a.score.alibi + hk * g + rb) : 0.f;
  const float scale_log2 = a.scale * kLog2e;

  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f, le_a = 0.f, le_b = 0.f;
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  bool ok = true;
  int k_fail = my_count;
  for (int k = 0; k < my_count; ++k) {
    const int stg = k % kStages;
    ok = mbar_wait(&bars[warp][stg], (uint32_t)((k / kStages) & 1), wc);
    if (!ok) {
      k_fail = k;
      break;
    }
    int c, t0, pid;
    sub_info(k, c, t0, pid);
    const uint32_t kb = smem_u32(my + stg * C::kStageBytes), vb = kb + C::kTileBytes;
    if (pid >= 0) {
      const int e = e0 + (warp + k * kDecWarps) / subs_per_page;
      const bool partial = e >= n_full;
      const int64_t j0 = (int64_t)c * PAGE + t0;
      float sc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int nt = 0; nt < 4; nt += 2) {
          const int mi = lane >> 3, rr = nt * 8 + (mi >> 1) * 8 + (lane & 7), c16 = ks * 2 + (mi & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + dswz(rr, c16), b0, b1, b2, b3);
          mma_bf16_16816(sc[nt], qf[ks], b0, b1);
          mma_bf16_16816(sc[nt + 1], qf[ks], b2, b3);
        }
      }
      uint32_t bits = 0xFFFFFFFFu;
      if (partial) {
        const int w = (int)min((int64_t)kSub, (int64_t)a.mask.kv_len - j0);
        Bits128 bb = rule_row_bits(a.rule, ig, j0, w, doc_i, [&](int d) {
          return doc_bits<1>(w, d, [&](int c) { return doc_at(a.rule, bm, j0 + c); });
        });
        bits = bb.w[0];
      }
      float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const int col = nt * 8 + (lane & 3) * 2 + (e2 & 1);
          const bool up = e2 >= 2;
          float x;
          if (has_score) {
            x = sc[nt][e2] * a.scale;
            const int64_t dist = ig - (j0 + col);
            if (a.score.alibi) x -= (up ? slope_b : slope_a) * (float)dist;
            if (a.score.rel) {
              const int hq = hk * g + (up ? rb : ra);
              if ((up ? rb : ra) < g) {
                int64_t ix = dist + a.score.kv_len - 1;
                ix = ix < 0 ? 0 : (ix > 2 * (int64_t)a.score.kv_len - 2 ? 2 * (int64_t)a.score.kv_len - 2 : ix);
                x += __ldg(a.score.rel + (size_t)hq * (2 * (size_t)a.score.kv_len - 1) + ix);
              }
            }
            if (a.score.softcap > 0.f) x = softcap_apply(x, a.score.softcap, a.score.inv_softcap);
            x *= kLog2e;
          } else {
            x = sc[nt][e2] * scale_log2;
          }
          if (!((bits >> col) & 1u)) x = -INFINITY;
          sc[nt][e2] = x;
          if (up) mx_b = fmaxf(mx_b, x); else mx_a = fmaxf(mx_a, x);
        }
      }
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xFFFFFFFFu, mx_a, 1));
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xFFFFFFFFu, mx_a, 2));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xFFFFFFFFu, mx_b, 1));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xFFFFFFFFu, mx_b, 2));
      const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
      const float ref_a = mn_a == -INFINITY ? 0.f : mn_a, ref_b = mn_b == -INFINITY ? 0.f : mn_b;
      const float al_a = ex2_approx(m_a - ref_a), al_b = ex2_approx(m_b - ref_b);
      m_a = mn_a;
      m_b = mn_b;
      uint32_t pf[2][4];
      float ps_a = 0.f, ps_b = 0.f, pe_a = 0.f, pe_b = 0.f;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const float p0 = ex2_approx(sc[nt][0] - ref_a), p1 = ex2_approx(sc[nt][1] - ref_a);
        const float p2 = ex2_approx(sc[nt][2] - ref_b), p3 = ex2_approx(sc[nt][3] - ref_b);
        const uint32_t pa = pack_bf16x2(p0, p1), pb = pack_bf16x2(p2, p3);
        pf[nt >> 1][(nt & 1) * 2 + 0] = pa;
        pf[nt >> 1][(nt & 1) * 2 + 1] = pb;
        ps_a += bf16x2_sum(pa);  // sums of the rounded P the product uses (normalise O)
        ps_b += bf16x2_sum(pb);
        pe_a += p0 + p1;         // sums of the unrounded P (LSE)
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
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
        for (int dt = 0; dt < D / 8; dt += 2) {
          const int mi = lane >> 3, rr = kk * 16 + (mi & 1) * 8 + (lane & 7), c16 = dt + (mi >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + dswz(rr, c16), b0, b1, b2, b3);
          mma_bf16_16816(o[dt], pf[kk], b0, b1);
          mma_bf16_16816(o[dt + 1], pf[kk], b2, b3);
        }
      }
    }
    __syncwarp();
    if (lane == 0 && k + kStages < my_count) {
      fence_proxy_async_smem();
      issue(k + kStages);
    }
  }
  if (!ok) {
    // drain this warp's copies still in flight (sub-tiles k_fail .. k_fail + kStages - 1 were issued and
    // not consumed) before the CTA and its shared memory go away
    if (lane == 0) {
      for (int k = k_fail; k < min(my_count, k_fail + kStages); ++k)
        mbar_wait_drain(&bars[warp][k % kStages], (uint32_t)((k / kStages) & 1), a.timeout_ns);
    }
    __syncwarp();
  }
  __syncthreads();
  if (s_abort) return;

  // ---- merge the 4 warps' states (shared memory reuse: all copies have landed)
  l_a += __shfl_xor_sync(0xFFFFFFFFu, l_a, 1);
  l_a += __shfl_xor_sync(0xFFFFFFFFu, l_a, 2);
  l_b += __shfl_xor_sync(0xFFFFFFFFu, l_b, 1);
  l_b += __shfl_xor_sync(0xFFFFFFFFu, l_b, 2);
  le_a += __shfl_xor_sync(0xFFFFFFFFu, le_a, 1);
  le_a += __shfl_xor_sync(0xFFFFFFFFu, le_a, 2);
  le_b += __shfl_xor_sync(0xFFFFFFFFu, le_b, 1);
  le_b += __shfl_xor_sync(0xFFFFFFFFu, le_b, 2);
  float* sO = reinterpret_cast<float*>(smem);             // [4][16][D]
  float* sM = sO + kDecWarps * 16 * D;                    // [4][16]
  float* sL = sM + kDecWarps * 16;                        // [4][16]
  float* sLe = sL + kDecWarps * 16;                       // [4][16]
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) {
    const int col = dt * 8 + (lane & 3) * 2;
    sO[(warp * 16 + ra) * D + col] = o[dt][0];
    sO[(warp * 16 + ra) * D + col + 1] = o[dt][1];
    sO[(warp * 16 + rb) * D + col] = o[dt][2];
    sO[(warp * 16 + rb) * D + col + 1] = o[dt][3];
  }
  if ((lane & 3) == 0) {
    sM[warp * 16 + ra] = m_a;
    sM[warp * 16 + rb] = m_b;
    sL[warp * 16 + ra] = l_a;
    sL[warp * 16 + rb] = l_b;
    sLe[warp * 16 + ra] = le_a;
    sLe[warp * 16 + rb] = le_b;
  }
  __syncthreads();
  const size_t ns = (size_t)a.n_splits;
  for (int x = tid; x < g * D; x += kDecWarps * 32) {
    const int row = x / D, col = x % D;
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) mm = fmaxf(mm, sM[w * 16 + row]);
    const float ref = mm == -INFINITY ? 0.f : mm;
    float u = 0.f, l = 0.f, le = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      const float wt = ex2_approx(sM[w * 16 + row] - ref);
      u += wt * sO[(w * 16 + row) * D + col];
      l += wt * sL[w * 16 + row];
      le += wt * sLe[w * 16 + row];
    }
    const size_t hq = (size_t)hk * g + row;
    const size_t slot = ((size_t)b * a.Hq + hq) * ns + s;
    a.ws_u[slot * D + col] = u;
    if (col == 0) {
      a.ws_m[slot] = mm;
      a.ws_l[slot] = l;
      a.ws_le[slot] = le;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const __grid_constant__ DecArgs a) {
  const int hq = blockIdx.x, b = blockIdx.y;
  const DevMask& M = a.mask;
  const size_t mrow = (size_t)(M.Bm > 1 ? b : 0) * M.Hm * M.nq;
  const int n_vis = __ldg(M.full_kv_num + mrow) + __ldg(M.kv_num + mrow);
  const int ns = (n_vis + a.pages_per_split - 1) / a.pages_per_split;
  const size_t base = ((size_t)b * a.Hq + hq) * (size_t)a.n_splits;
  const size_t obase = ((size_t)b * a.Hq + hq) * D;
  float mm = -INFINITY;
  for (int s = 0; s < ns; ++s) mm = fmaxf(mm, a.ws_m[base + s]);
  const float ref = mm == -INFINITY ? 0.f : mm;
  float l = 0.f, le = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float wt = ex2_approx(a.ws_m[base + s] - ref);
    l += wt * a.ws_l[base + s];
    le += wt * a.ws_le[base + s];
  }
  const bool empty = mm == -INFINITY;
  const float inv = empty ? 0.f : 1.f / l;
  for (int col = threadIdx.x; col < D; col += blockDim.x) {
    float u = 0.f;
    for (int s = 0; s < ns; ++s) u += ex2_approx(a.ws_m[base + s] - ref) * a.ws_u[(base + s) * D + col];
    if (a.out_f32)
      reinterpret_cast<float*>(a.out)[obase + col] = u * inv;
    else
      reinterpret_cast<__nv_bfloat16*>(a.out)[obase + col] = __float2bfloat16_rn(u * inv);
  }
  if (threadIdx.x == 0) a.lse[(size_t)b * a.Hq + hq] = empty ? -INFINITY : (mm + __log2f(le)) * kLn2;
}

template <int D>
int launch_d(const DecArgs& a, cudaStream_t st) {
  using C = DecCfg<D>;
  CUtensorMap tk, tv;
  const uint64_t rows = (uint64_t)a.n_pages_total * a.Hkv * a.page;
  const uint64_t dims[2] = {(uint64_t)D, rows};
  const uint64_t strides[1] = {(uint64_t)D * 2};
  const uint32_t box[2] = {64, kSub};
  if (encode_tmap_bf16(&tk, a.k_pages, 2, dims, strides, box) != 0) return FA_ERR_CUDA;
  if (encode_tmap_bf16(&tv, a.v_pages, 2, dims, strides, box) != 0) return FA_ERR_CUDA;
  auto kern = decode_split_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess)
    return FA_ERR_CUDA;
  dim3 g1(a.n_splits, a.Hkv, a.Bz);
  kern<<<g1, kDecWarps * 32, C::kSmem, st>>>(a, tk, tv, a.page);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  dim3 g2(a.Hq, a.Bz);
  decode_combine_kernel<D><<<g2, 128, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace

int launch_decode(const DecArgs& a, cudaStream_t st) {
  if (a.d == 64) return launch_d<64>(a, st);
  if (a.d == 128) return launch_d<128>(a, st);
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
