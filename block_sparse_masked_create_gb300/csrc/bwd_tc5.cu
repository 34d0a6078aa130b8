// Backward of the block-sparse masked attention forward on the 5th-generation tensor cores (tcgen05,
// accumulators in tensor memory, operands staged by TMA), for 128 x 128 blocks. Same arithmetic as the
// mma.sync backward (FlashAttention self-test questions on the backward pass; "5.1.2 FlexAttention: from
// rules to fused kernels", section 4, the two aggregation directions of the backward):
//   P = exp(s' - LSE) from the forward's LSE, s' = score rule (scale q.k), masked pairs 0; D_i from the
//   delta kernel; dV = P^T dO; dP = dO V^T; dS = P (dP - D) g with g = ds'/ds; dQ = scale dS K;
//   dK = scale dS^T Q; dK and dV summed over the query heads of a KV head, without atomics.
//
// dK/dV kernel: one CTA per (key block c, KV head, batch row). K_c and V_c stay in shared memory; the CTA
// walks, for every query head of the group, the column of block c in the query-side transpose (full
// blocks, then partial ones). Per query block, with the key rows in the TMEM lanes:
//   S^T = K Q^T and dP^T = V dO^T (both operands in shared memory) -> TMEM;
//   eight gradient warps turn S^T into P^T (bf16, written over S^T) and dP^T into dS^T (over dP^T);
//   dV += P^T dO and dK += dS^T Q with the A operand read from TMEM; the accumulators stay in TMEM.
// dQ kernel: one CTA per (query block, head); walks the block's kv lists: S = Q K^T and dP = dO V^T,
//   dS (bf16, over dP) and dQ += dS K; S is double-buffered so the next block's S overlaps the math.
// Warp roles (both): warps 0-7 gradient math (warpgroup w owns 64 of the 128 columns, warp w % 4 its
// 32 TMEM lanes), warp 8 TMA producer, warp 9 MMA issuer (one elected lane issues). Every wait is bounded;
// a wait that runs out sets FA_ERR_TIMEOUT and the CTA drains its copies and MMAs before it exits.
#include <cstring>

#include "fa_launch.h"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kLoadWarp = 8, kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr int kGradThreads = 256;

template <int D>
struct BwdTc5 {
  static constexpr int kTile = 128 * D * 2;  // one [128 x D] bf16 tile: D / 64 swizzled halves of 16 KB
  // tensor memory columns (512 allocated). dK/dV kernel: S^T, dP^T, then the dV and dK accumulators;
  // dQ kernel: two S buffers, dP, then the dQ accumulator
  static constexpr uint32_t kKvColS = 0, kKvColDP = 128, kKvColDV = 256, kKvColDK = 256 + D;
  static constexpr uint32_t kQColS0 = 0, kQColDP = 256, kQColDQ = 384;
  static constexpr uint32_t kTmemCols = 512;
  // dK/dV kernel shared memory: K, V, two stages of (Q, dO), the stage statistics, barriers
  static constexpr int kKvOffK = 0, kKvOffV = kTile, kKvOffStage = 2 * kTile;
  static constexpr int kKvOffStat = 6 * kTile;  // float [2][3][128]: LSE*log2e, D, query document ids
  static constexpr int kKvOffBar = kKvOffStat + 2 * 3 * 128 * 4;
  static constexpr int kKvSmem = kKvOffBar + 256;
  // dQ kernel shared memory: Q, dO, a 3-slot K ring (K(k) is read by S(k) and, last, by dQ(k); the
  // third slot lets K(k+1) arrive while dQ(k-1) still reads its slot), a 2-slot V ring (V(k) is read by
  // dP(k) only), key document ids [2][128], barriers
  static constexpr int kQOffQ = 0, kQOffDO = kTile, kQOffK = 2 * kTile, kQOffV = 5 * kTile;
  static constexpr int kQOffDoc = 7 * kTile;
  static constexpr int kQOffBar = kQOffDoc + 2 * 128 * 4;
  static constexpr int kQSmem = kQOffBar + 256;
  static_assert(kKvSmem <= 232448 && kQSmem <= 232448, "shared memory per CTA");
};

// K-major operand tile (TMA box {64, 128} with the 128-byte swizzle): k-step ks (16 elements) starts at
// this descriptor offset (16-byte units)
__device__ __forceinline__ uint64_t kmaj_step(int ks) { return (uint64_t)(((ks >> 2) * 16384 + (ks & 3) * 32) >> 4); }
// MN-major operand (the rows of the tile are the k index): k-step ks = 16 rows
__device__ __forceinline__ uint64_t mnmaj_step(int ks) { return (uint64_t)((ks * 2048) >> 4); }
// A operand packed as bf16 pairs in TMEM by the gradient warps: k-step ks of warpgroup ks / 4
__device__ __forceinline__ uint32_t packed_step(int ks) { return (uint32_t)(ks * 8 + (ks >= 4 ? 32 : 0)); }

// Barrier of the 256 gradient threads (named barrier 1) that also ORs a flag over them, so that a
// failed wait makes every gradient thread leave its loop at the same iteration (a thread that left
// alone would leave the others waiting at this barrier).
__device__ __forceinline__ bool grad_bar_any(bool flag) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbarrier.cta.red.or.pred p, 1, 256, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)flag)
      : "memory");
  return r != 0;
}

// Score-rule variants compiled separately: none, ALiBi alone, soft-cap alone, anything else (generic).
// The first three take the forward's log2-domain arithmetic (scale * log2e folded into one FMA, ALiBi as
// a bias linear in the column, c log2e tanh(scale x / c)), so P is recomputed as the forward formed it.
enum ScoreKind { SK_NONE = 0, SK_ALIBI = 1, SK_SOFTCAP = 2, SK_GENERIC = 3 };

// Generic score rule on a scaled score (ALiBi, relative bias, then soft-cap) and g = ds'/ds; dist = i_g - j.
__device__ __forceinline__ float score_g(const DevScore& sc, int h, float x, int64_t dist, float slope, float& g) {
  g = 1.f;
  if (sc.alibi) x -= slope * (float)dist;
  if (sc.rel) {
    int64_t ix = dist + sc.kv_len - 1;
    ix = ix < 0 ? 0 : (ix > 2 * (int64_t)sc.kv_len - 2 ? 2 * (int64_t)sc.kv_len - 2 : ix);
    x += __ldg(sc.rel + (size_t)h * (2 * (size_t)sc.kv_len - 1) + ix);
  }
  if (sc.softcap > 0.f) {
    x = softcap_apply(x, sc.softcap, sc.inv_softcap);
    const float t = x * sc.inv_softcap;
    g = 1.f - t * t;
  }
  return x;
}

// Allowed query rows (global positions [ig0, ig0 + w), w <= 128) of one key position j: the rule's terms
// read with the roles of row and column swapped (causal: i >= j; window: i < j + W; prefix: j < P;
// document: doc(i) == doc(j), as the run [run_lo, run_hi) of j's id when `use_run` (ids that never
// decrease, and an id other than -1, which rows outside the id array also read), else from the rows' ids
// in `qdoc`).
__device__ __forceinline__ Bits128 rule_key_bits(const DevRule& R, int64_t j, int64_t ig0, int w, int doc_j,
                                                 const int* qdoc, bool use_run, int64_t run_lo, int64_t run_hi) {
  Bits128 db = {{0u, 0u, 0u, 0u}};
  if (R.any_doc && use_run) {
    db = range_bits(clamp_rel(run_lo - ig0, w), clamp_rel(run_hi - ig0, w));
  } else if (R.any_doc) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t wd = 0u;
#pragma unroll 8
      for (int b = 0; b < 32; ++b)
        if (32 * k + b < w && qdoc[32 * k + b] == doc_j) wd |= 1u << b;
      db.w[k] = wd;
    }
  }
  Bits128 acc = {{0u, 0u, 0u, 0u}};
  for (int t = 0; t < R.n_terms; ++t) {
    const DevTerm T = R.t[t];
    if (T.pre != INT64_MAX && j >= T.pre) continue;
    int64_t lo = ig0, hi = ig0 + w;
    if (T.causal) lo = max(lo, j);
    if (T.win != INT64_MAX) hi = min(hi, j + T.win);
    Bits128 b = range_bits(clamp_rel(lo - ig0, w), clamp_rel(hi - ig0, w));
    if (T.doc) {
#pragma unroll
      for (int k = 0; k < 4; ++k) b.w[k] &= db.w[k];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) acc.w[k] |= b.w[k];
  }
  return acc;
}

struct Tc5BwdParams {
  BwdArgs a;
};

// The (query head, query block, partial?) of item k of the dK/dV walk over key block c: the query heads
// of the group in order, each with its full list, then its partial list.
__device__ __forceinline__ void kv_item(const BwdArgs& a, int b, int hk, int c, int k, int& h, int& r, bool& partial) {
  const DevMask& M = a.mask;
  const int g = a.Hq / a.Hkv;
  const int bm = M.Bm > 1 ? b : 0;
  for (int gi = 0; gi < g; ++gi) {
    const int hh = hk * g + gi;
    const int hm = M.Hm > 1 ? hh : 0;
    const size_t col = ((size_t)bm * M.Hm + hm) * M.nk + c;
    const int nf = __ldg(M.full_q_num + col), np = __ldg(M.q_num + col);
    if (k < nf + np) {
      h = hh;
      partial = k >= nf;
      r = partial ? __ldg(M.q_idx + col * M.nq + (k - nf)) : __ldg(M.full_q_idx + col * M.nq + k);
      return;
    }
    k -= nf + np;
  }
  h = hk * g;
  r = 0;
  partial = true;
}

__device__ __forceinline__ int kv_items(const BwdArgs& a, int b, int hk, int c) {
  const DevMask& M = a.mask;
  const int g = a.Hq / a.Hkv;
  const int bm = M.Bm > 1 ? b : 0;
  int n = 0;
  for (int gi = 0; gi < g; ++gi) {
    const int hm = M.Hm > 1 ? hk * g + gi : 0;
    const size_t col = ((size_t)bm * M.Hm + hm) * M.nk + c;
    n += __ldg(M.full_q_num + col) + __ldg(M.q_num + col);
  }
  return n;
}

// ============================================================================================ dK / dV
template <int D, int SK>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kv_tc5_kernel(const __grid_constant__ Tc5BwdParams P, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmDO) {
  using C = BwdTc5<D>;
  const BwdArgs& a = P.a;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (smem_u32(smem) & 1023u) {  // uniform across the CTA, before any barrier or allocation
    if (tid == 0) report(a.status, FA_ERR_DEVICE_CHECK);
    return;
  }
  const int c = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int n = kv_items(a, b, hk, c);
  uint8_t* sK = smem + C::kKvOffK;
  uint8_t* sV = smem + C::kKvOffV;
  float* sStat = reinterpret_cast<float*>(smem + C::kKvOffStat);  // [2][3][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kKvOffBar);
  uint64_t* bar_kv = bars + 0;
  uint64_t* bar_ld = bars + 1;    // [2]
  uint64_t* bar_free = bars + 3;  // [2]
  uint64_t* bar_s = bars + 5;
  uint64_t* bar_dp = bars + 6;
  uint64_t* bar_p = bars + 7;
  uint64_t* bar_ds = bars + 8;
  uint64_t* bar_done = bars + 9;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 10);
  volatile int32_t* s_abort = reinterpret_cast<volatile int32_t*>(bars + 11);
  auto stageQ = [&](int st) { return smem + C::kKvOffStage + st * 2 * C::kTile; };
  auto stageDO = [&](int st) { return smem + C::kKvOffStage + st * 2 * C::kTile + C::kTile; };

  if (warp == kLoadWarp) {
    if (lane == 0) {
      *s_abort = 0;
      mbar_init(bar_kv, 1);
      for (int i = 0; i < 2; ++i) {
        mbar_init(bar_ld + i, 1);
        mbar_init(bar_free + i, 1);
      }
      mbar_init(bar_s, 1);
      mbar_init(bar_dp, 1);
      mbar_init(bar_p, kGradThreads);
      mbar_init(bar_ds, kGradThreads);
      mbar_init(bar_done, 1);
      fence_mbar_init();
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
    }
    __syncwarp();
    if (n > 0) {
      mbar_arrive_expect_tx_elect(bar_kv, 2 * C::kTile);
#pragma unroll
      for (int x = 0; x < D / 64; ++x) {
        tma_load_3d_elect(sK + x * 16384, &tmK, x * 64, c * 128, b * a.Hkv + hk, bar_kv);
        tma_load_3d_elect(sV + x * 16384, &tmV, x * 64, c * 128, b * a.Hkv + hk, bar_kv);
      }
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(s_tmem, C::kTmemCols);
    tmem_relinquish();
  }
  tc5_fence_before();
  __syncthreads();
  tc5_fence_after();
  const uint32_t tmem = *s_tmem;
  WaitCtl wc{a.timeout_ns, a.status, s_abort};

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------------ TMA producer: Q, dO per item
    int issued[2] = {0, 0};
    for (int k = 0; k < n; ++k) {
      const int st = k & 1;
      if (k >= 2 && !__all_sync(0xFFFFFFFFu, mbar_wait(bar_free + st, (uint32_t)(((k >> 1) - 1) & 1), wc))) break;
      int h, r;
      bool partial;
      kv_item(a, b, hk, c, k, h, r, partial);
      mbar_arrive_expect_tx_elect(bar_ld + st, 2 * C::kTile);
#pragma unroll
      for (int x = 0; x < D / 64; ++x) {
        tma_load_3d_elect(stageQ(st) + x * 16384, &tmQ, x * 64, r * 128, b * a.Hq + h, bar_ld + st);
        tma_load_3d_elect(stageDO(st) + x * 16384, &tmDO, x * 64, r * 128, b * a.Hq + h, bar_ld + st);
      }
      issued[st] = (k >> 1) + 1;
    }
    // every copy this CTA issued lands before the CTA may exit (its shared memory stays valid)
    if (n > 0) mbar_wait_drain(bar_kv, 0, a.timeout_ns);
    for (int st = 0; st < 2; ++st)
      if (issued[st] > 0) mbar_wait_drain(bar_ld + st, (uint32_t)((issued[st] - 1) & 1), a.timeout_ns);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_t = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T: N = 128 query rows
    constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, false, true);   // dV, dK: B MN-major, N = D
    const uint64_t kdesc = sdesc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t vdesc = sdesc_sw128(smem_u32(sV), 16, 1024);
    bool ok = n > 0 && __all_sync(0xFFFFFFFFu, mbar_wait(bar_kv, 0, wc));
    auto issue_st = [&](int k) -> bool {  // S^T(k) once Q(k) is in
      const int st = k & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_ld + st, (uint32_t)((k >> 1) & 1), wc))) return false;
      tc5_fence_after();
      const uint64_t qd = sdesc_sw128(smem_u32(stageQ(st)), 16, 1024);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        tc5_mma_ss_elect(tmem + C::kKvColS, kdesc + kmaj_step(ks), qd + kmaj_step(ks), idesc_t, ks > 0 ? 1u : 0u);
      tc5_commit_elect(bar_s);
      return true;
    };
    if (ok) ok = issue_st(0);
    for (int k = 0; k < n && ok; ++k) {
      const int st = k & 1;
      const uint64_t dod = sdesc_sw128(smem_u32(stageDO(st)), 16, 1024);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        tc5_mma_ss_elect(tmem + C::kKvColDP, vdesc + kmaj_step(ks), dod + kmaj_step(ks), idesc_t, ks > 0 ? 1u : 0u);
      tc5_commit_elect(bar_dp);
      if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_p, (uint32_t)(k & 1), wc)))) break;
      tc5_fence_after();
      const uint64_t do_mn = sdesc_sw128(smem_u32(stageDO(st)), 16384, 1024);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        tc5_mma_ts_elect(tmem + C::kKvColDV, tmem + C::kKvColS + packed_step(ks), do_mn + mnmaj_step(ks), idesc_acc,
                         (k > 0 || ks > 0) ? 1u : 0u);
      if (k + 1 < n && !(ok = issue_st(k + 1))) break;  // S^T(k+1) overwrites P^T(k) after dV(k) read it
      if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_ds, (uint32_t)(k & 1), wc)))) break;
      tc5_fence_after();
      const uint64_t q_mn = sdesc_sw128(smem_u32(stageQ(st)), 16384, 1024);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        tc5_mma_ts_elect(tmem + C::kKvColDK, tmem + C::kKvColDP + packed_step(ks), q_mn + mnmaj_step(ks), idesc_acc,
                         (k > 0 || ks > 0) ? 1u : 0u);
      tc5_commit_elect(bar_free + st);
    }
    tc5_commit_elect(bar_done);  // completes when every MMA issued above has
  } else {
    // ------------------------------------------------------------------ gradient warps
    const int wg = warp >> 2, quarter = warp & 3;
    const int row = quarter * 32 + lane;  // key row of the block = TMEM lane
    const int64_t j = (int64_t)c * 128 + row;
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    const int64_t off = a.rule.q_offset ? (int64_t)__ldg(a.rule.q_offset + (a.mask.Bm > 1 ? b : 0)) : 0;
    const int doc_j = a.rule.any_doc ? doc_at(a.rule, b, j) : -1;
    // document equality of this key as the run of its id (ids that never decrease)
    const bool runs = a.rule.any_doc && doc_j != -1 && doc_runs_usable(a.rule, b);
    int64_t run_lo = 0, run_hi = 0;
    if (runs) doc_run_of(a.rule, b, j, run_lo, run_hi);
    const float sl2 = a.scale * kLog2e;
    const float ain = a.scale * a.score.inv_softcap, aout = a.score.softcap * kLog2e;
    // Per-query statistics of an item, one value per thread: LSE * log2(e) (+inf past the sequence or
    // for an empty row, so P = 0 there) in threads 0-127, D and the query row's document id in threads
    // 128-255. Item k + 1's are loaded into registers at the start of item k and stored to the shared
    // buffer (k + 1) & 1 at its end, so their latency hides behind item k; the barrier at the top of each
    // item publishes them, and the buffer they overwrite was last read before the previous barrier.
    int h_n = 0, r_n = 0;
    bool p_n = false;
    float v_n = 0.f;
    int doc_n = -1;
    auto fetch = [&](int kk) {
      kv_item(a, b, hk, c, kk, h_n, r_n, p_n);
      const int64_t i = (int64_t)r_n * 128 + (tid & 127);
      const size_t qrow = ((size_t)b * a.Hq + h_n) * a.q_len + i;
      const bool in = i < a.q_len;
      v_n = tid < 128 ? (in ? __ldg(a.lse + qrow) : -INFINITY) : (in ? __ldg(a.delta + qrow) : 0.f);
      if (a.rule.any_doc && tid >= 128) doc_n = doc_at(a.rule, b, i + off);
    };
    auto publish = [&](int kk) {
      float* st = sStat + (kk & 1) * 384;
      const int x = tid & 127;
      if (tid < 128) {
        st[x] = v_n == -INFINITY ? INFINITY : v_n * kLog2e;
      } else {
        st[128 + x] = v_n;
        if (a.rule.any_doc) reinterpret_cast<int*>(st)[256 + x] = doc_n;
      }
    };
    if (n > 0) {
      fetch(0);
      publish(0);
    }
    bool ok = true;  // warp-uniform; made CTA-uniform among the gradient warps at each item's barrier
    for (int k = 0; k < n; ++k) {
      if (grad_bar_any(!ok)) {
        ok = false;
        break;
      }
      const int h = h_n, r = r_n;
      const bool partial = p_n;
      float* st_l = sStat + (k & 1) * 384;
      if (k + 1 < n) fetch(k + 1);
      const float slope = (SK == SK_ALIBI || SK == SK_GENERIC) && a.score.alibi ? __ldg(a.score.alibi + h) : 0.f;
      // ALiBi (log2 domain): -slope log2e (i_g - j), i_g - j = d0 + column; base at this warpgroup's first
      const int64_t d0 = (int64_t)r * 128 + off - j;
      const float nsl2 = -slope * kLog2e, base_w = nsl2 * (float)(d0 + 64 * wg);
      uint32_t allowed[2] = {0xFFFFFFFFu, 0xFFFFFFFFu};  // this warpgroup's 64 query columns
      if (partial) {
        const Bits128 bits = rule_key_bits(a.rule, j, (int64_t)r * 128 + off, (int)min((int64_t)128, (int64_t)a.q_len - (int64_t)r * 128),
                                           doc_j, reinterpret_cast<const int*>(st_l) + 256, runs, run_lo, run_hi);
        allowed[0] = bits.w[2 * wg];
        allowed[1] = bits.w[2 * wg + 1];
      }
      // ---- P^T = exp2(s' log2e - LSE log2e), written over S^T as bf16 pairs; pg = P g kept for dS^T
      if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_s, (uint32_t)(k & 1), wc)))) continue;
      tc5_fence_after();
      float pg[64];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t sv[32];
        tc5_ld32(lane_addr + C::kKvColS + 64 * wg + 32 * half, sv);
        tc5_wait_ld();
        uint32_t pk[16];
        const float4* l4 = reinterpret_cast<const float4*>(st_l + 64 * wg + 32 * half);
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 L4 = l4[e >> 2];
          const float L[4] = {L4.x, L4.y, L4.z, L4.w};
          float pv[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int cl = 32 * half + e + u;  // column within this warpgroup's 64
            const float xr = __uint_as_float(sv[e + u]);
            float lg, g = 1.f;
            if constexpr (SK == SK_NONE) {
              lg = fmaf(xr, sl2, -L[u]);
            } else if constexpr (SK == SK_ALIBI) {
              lg = fmaf(xr, sl2, fmaf(nsl2, (float)cl, base_w) - L[u]);
            } else if constexpr (SK == SK_SOFTCAP) {
              const float t = tanh_approx(xr * ain);
              lg = fmaf(t, aout, -L[u]);
              g = 1.f - t * t;
            } else {
              lg = score_g(a.score, h, xr * a.scale, d0 + 64 * wg + cl, slope, g) * kLog2e - L[u];
            }
            float p = ex2_approx(lg);
            if (partial && !((allowed[half] >> (e + u)) & 1u)) p = 0.f;
            pv[u] = p;
            pg[cl] = SK == SK_SOFTCAP || SK == SK_GENERIC ? p * g : p;
          }
          pk[e >> 1] = pack_bf16x2(pv[0], pv[1]);
          pk[(e >> 1) + 1] = pack_bf16x2(pv[2], pv[3]);
        }
        tc5_st16(lane_addr + C::kKvColS + 64 * wg + 16 * half, pk);
      }
      tc5_wait_st();
      tc5_fence_before();
      mbar_arrive(bar_p);
      // ---- dS^T = P g (dP^T - D), written over dP^T as bf16 pairs
      if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_dp, (uint32_t)(k & 1), wc)))) continue;
      tc5_fence_after();
      uint32_t dv2[2][32];
      tc5_ld32(lane_addr + C::kKvColDP + 64 * wg, dv2[0]);
      tc5_ld32(lane_addr + C::kKvColDP + 64 * wg + 32, dv2[1]);
      tc5_wait_ld();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t (&dv)[32] = dv2[half];
        uint32_t pk[16];
        const float4* dl4 = reinterpret_cast<const float4*>(st_l + 128 + 64 * wg + 32 * half);
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 Dl = dl4[e >> 2];
          const int cl = 32 * half + e;
          pk[e >> 1] = pack_bf16x2(pg[cl] * (__uint_as_float(dv[e]) - Dl.x), pg[cl + 1] * (__uint_as_float(dv[e + 1]) - Dl.y));
          pk[(e >> 1) + 1] =
              pack_bf16x2(pg[cl + 2] * (__uint_as_float(dv[e + 2]) - Dl.z), pg[cl + 3] * (__uint_as_float(dv[e + 3]) - Dl.w));
        }
        tc5_st16(lane_addr + C::kKvColDP + 64 * wg + 16 * half, pk);
      }
      tc5_wait_st();
      tc5_fence_before();
      mbar_arrive(bar_ds);
      if (k + 1 < n) publish(k + 1);
    }
    // ---- epilogue: dV and scale * dK of this key row, fp32 (rows past kv_len are not written)
    // (tcgen05.ld is warp-collective: every lane loads, only rows inside the sequence store)
    const bool done = __all_sync(0xFFFFFFFFu, n == 0 || mbar_wait_drain(bar_done, 0, a.timeout_ns));
    tc5_fence_after();
    const bool in = j < a.kv_len;
    if (ok && done) {
      float* dVg = a.dv + (((size_t)b * a.Hkv + hk) * a.kv_len + (in ? j : 0)) * D + wg * (D / 2);
      float* dKg = a.dk + (((size_t)b * a.Hkv + hk) * a.kv_len + (in ? j : 0)) * D + wg * (D / 2);
#pragma unroll
      for (int part = 0; part < D / 64; ++part) {
        uint32_t v[32];
        if (n > 0) {
          tc5_ld32(lane_addr + C::kKvColDV + wg * (D / 2) + 32 * part, v);
          tc5_wait_ld();
        }
#pragma unroll
        for (int e = 0; e < 32 && in; e += 4)
          *reinterpret_cast<float4*>(dVg + 32 * part + e) =
              n > 0 ? make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]),
                                  __uint_as_float(v[e + 3]))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
        if (n > 0) {
          tc5_ld32(lane_addr + C::kKvColDK + wg * (D / 2) + 32 * part, v);
          tc5_wait_ld();
        }
#pragma unroll
        for (int e = 0; e < 32 && in; e += 4)
          *reinterpret_cast<float4*>(dKg + 32 * part + e) =
              n > 0 ? make_float4(__uint_as_float(v[e]) * a.scale, __uint_as_float(v[e + 1]) * a.scale,
                                  __uint_as_float(v[e + 2]) * a.scale, __uint_as_float(v[e + 3]) * a.scale)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  tc5_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc5_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ================================================================================================= dQ
template <int D, int SK>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_q_tc5_kernel(const __grid_constant__ Tc5BwdParams P, const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmDO) {
  using C = BwdTc5<D>;
  const BwdArgs& a = P.a;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (smem_u32(smem) & 1023u) {
    if (tid == 0) report(a.status, FA_ERR_DEVICE_CHECK);
    return;
  }
  const DevMask& M = a.mask;
  const int h = blockIdx.y, b = blockIdx.z;
  // long rows first: the mask's row order (causal: nq-1 .. 0)
  const int r = M.row_order
                    ? __ldg(M.row_order + ((size_t)(M.Bm > 1 ? b : 0) * M.Hm + (M.Hm > 1 ? h : 0)) * M.nq + blockIdx.x)
                    : M.nq - 1 - (int)blockIdx.x;
  const int hk = h / (a.Hq / a.Hkv);
  const size_t mrow = ((size_t)(M.Bm > 1 ? b : 0) * M.Hm + (M.Hm > 1 ? h : 0)) * M.nq + r;
  const int nf = __ldg(M.full_kv_num + mrow), n = nf + __ldg(M.kv_num + mrow);
  const int32_t* full_idx = M.full_kv_idx + mrow * M.nk;
  const int32_t* part_idx = M.kv_idx + mrow * M.nk;
  auto item_col = [&](int k) { return k < nf ? __ldg(full_idx + k) : __ldg(part_idx + k - nf); };

  uint8_t* sQ = smem + C::kQOffQ;
  uint8_t* sDO = smem + C::kQOffDO;
  int* sDoc = reinterpret_cast<int*>(smem + C::kQOffDoc);  // [2][128] key document ids
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kQOffBar);
  uint64_t* bar_qdo = bars + 0;
  uint64_t* bar_kfull = bars + 1;   // [3]
  uint64_t* bar_kempty = bars + 4;  // [3]
  uint64_t* bar_vfull = bars + 7;   // [2]
  uint64_t* bar_vempty = bars + 9;  // [2]
  uint64_t* bar_s = bars + 11;      // [2] S buffers
  uint64_t* bar_dp = bars + 13;
  uint64_t* bar_ds = bars + 14;
  uint64_t* bar_done = bars + 15;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int32_t* s_abort = reinterpret_cast<volatile int32_t*>(bars + 17);
  auto slotK = [&](int k) { return smem + C::kQOffK + (k % 3) * C::kTile; };
  auto slotV = [&](int k) { return smem + C::kQOffV + (k & 1) * C::kTile; };

  if (warp == kLoadWarp) {
    if (lane == 0) {
      *s_abort = 0;
      mbar_init(bar_qdo, 1);
      for (int i = 0; i < 3; ++i) {
        mbar_init(bar_kfull + i, 1);
        mbar_init(bar_kempty + i, 1);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(bar_vfull + i, 1);
        mbar_init(bar_vempty + i, 1);
        mbar_init(bar_s + i, 1);
      }
      mbar_init(bar_dp, 1);
      mbar_init(bar_ds, kGradThreads);
      mbar_init(bar_done, 1);
      fence_mbar_init();
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
    }
    __syncwarp();
    if (n > 0) {
      mbar_arrive_expect_tx_elect(bar_qdo, 2 * C::kTile);
#pragma unroll
      for (int x = 0; x < D / 64; ++x) {
        tma_load_3d_elect(sQ + x * 16384, &tmQ, x * 64, r * 128, b * a.Hq + h, bar_qdo);
        tma_load_3d_elect(sDO + x * 16384, &tmDO, x * 64, r * 128, b * a.Hq + h, bar_qdo);
      }
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(s_tmem, C::kTmemCols);
    tmem_relinquish();
  }
  tc5_fence_before();
  __syncthreads();
  tc5_fence_after();
  const uint32_t tmem = *s_tmem;
  WaitCtl wc{a.timeout_ns, a.status, s_abort};

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------------ TMA producer: K, V per block
    int issuedK[3] = {0, 0, 0}, issuedV[2] = {0, 0};
    for (int k = 0; k < n; ++k) {
      const int c = item_col(k);
      const int sk = k % 3, sv = k & 1;
      if (k >= 3 && !__all_sync(0xFFFFFFFFu, mbar_wait(bar_kempty + sk, (uint32_t)((k / 3 - 1) & 1), wc))) break;
      mbar_arrive_expect_tx_elect(bar_kfull + sk, C::kTile);
#pragma unroll
      for (int x = 0; x < D / 64; ++x)
        tma_load_3d_elect(slotK(k) + x * 16384, &tmK, x * 64, c * 128, b * a.Hkv + hk, bar_kfull + sk);
      issuedK[sk] = k / 3 + 1;
      if (k >= 2 && !__all_sync(0xFFFFFFFFu, mbar_wait(bar_vempty + sv, (uint32_t)(((k >> 1) - 1) & 1), wc))) break;
      mbar_arrive_expect_tx_elect(bar_vfull + sv, C::kTile);
#pragma unroll
      for (int x = 0; x < D / 64; ++x)
        tma_load_3d_elect(slotV(k) + x * 16384, &tmV, x * 64, c * 128, b * a.Hkv + hk, bar_vfull + sv);
      issuedV[sv] = (k >> 1) + 1;
    }
    if (n > 0) mbar_wait_drain(bar_qdo, 0, a.timeout_ns);
    for (int i = 0; i < 3; ++i)
      if (issuedK[i] > 0) mbar_wait_drain(bar_kfull + i, (uint32_t)((issuedK[i] - 1) & 1), a.timeout_ns);
    for (int i = 0; i < 2; ++i)
      if (issuedV[i] > 0) mbar_wait_drain(bar_vfull + i, (uint32_t)((issuedV[i] - 1) & 1), a.timeout_ns);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);  // S, dP: N = 128 keys
    constexpr uint32_t idesc_q = idesc_bf16_f32(128, D, false, true);     // dQ: B = K MN-major, N = D
    const uint64_t qdesc = sdesc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t dodesc = sdesc_sw128(smem_u32(sDO), 16, 1024);
    bool ok = n > 0 && __all_sync(0xFFFFFFFFu, mbar_wait(bar_qdo, 0, wc));
    auto issue_s = [&](int k) -> bool {  // S(k) = Q K(k)^T into S buffer k & 1
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_kfull + k % 3, (uint32_t)((k / 3) & 1), wc))) return false;
      tc5_fence_after();
      const uint64_t kd = sdesc_sw128(smem_u32(slotK(k)), 16, 1024);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        tc5_mma_ss_elect(tmem + C::kQColS0 + 128 * (k & 1), qdesc + kmaj_step(ks), kd + kmaj_step(ks), idesc_s,
                         ks > 0 ? 1u : 0u);
      tc5_commit_elect(bar_s + (k & 1));
      return true;
    };
    if (ok) ok = issue_s(0);
    for (int k = 0; k < n && ok; ++k) {
      if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_vfull + (k & 1), (uint32_t)((k >> 1) & 1), wc)))) break;
      tc5_fence_after();
      const uint64_t vd = sdesc_sw128(smem_u32(slotV(k)), 16, 1024);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        tc5_mma_ss_elect(tmem + C::kQColDP, dodesc + kmaj_step(ks), vd + kmaj_step(ks), idesc_s, ks > 0 ? 1u : 0u);
      tc5_commit_elect(bar_dp);
      tc5_commit_elect(bar_vempty + (k & 1));
      if (k + 1 < n && !(ok = issue_s(k + 1))) break;  // its buffer held S(k-1), read before dS(k-1)
      if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_ds, (uint32_t)(k & 1), wc)))) break;
      tc5_fence_after();
      const uint64_t k_mn = sdesc_sw128(smem_u32(slotK(k)), 16384, 1024);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        tc5_mma_ts_elect(tmem + C::kQColDQ, tmem + C::kQColDP + packed_step(ks), k_mn + mnmaj_step(ks), idesc_q,
                         (k > 0 || ks > 0) ? 1u : 0u);
      tc5_commit_elect(bar_kempty + k % 3);
    }
    tc5_commit_elect(bar_done);
  } else {
    // ------------------------------------------------------------------ gradient warps
    const int wg = warp >> 2, quarter = warp & 3;
    const int row = quarter * 32 + lane;  // query row of the block = TMEM lane
    const int64_t i = (int64_t)r * 128 + row;
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    const int64_t off = a.rule.q_offset ? (int64_t)__ldg(a.rule.q_offset + (M.Bm > 1 ? b : 0)) : 0;
    const int64_t ig = i + off;
    const size_t qrow = ((size_t)b * a.Hq + h) * a.q_len + i;
    float lse2 = INFINITY, dlt = 0.f;  // rows past the sequence and empty rows: P = 0
    if (i < a.q_len) {
      const float l = __ldg(a.lse + qrow);
      lse2 = l == -INFINITY ? INFINITY : l * kLog2e;
      dlt = __ldg(a.delta + qrow);
    }
    const int doc_i = a.rule.any_doc ? doc_at(a.rule, b, ig) : -1;
    // document equality of this row as the run of its id (ids that never decrease; every key position
    // lies inside the id array)
    const bool runs = a.rule.any_doc && ig >= 0 && ig < a.rule.doc_len && doc_runs_usable(a.rule, b);
    int64_t run_lo = 0, run_hi = 0;
    if (runs) doc_run_of(a.rule, b, ig, run_lo, run_hi);
    const float slope = (SK == SK_ALIBI || SK == SK_GENERIC) && a.score.alibi ? __ldg(a.score.alibi + h) : 0.f;
    const float sl2 = a.scale * kLog2e, psl2 = slope * kLog2e;
    const float ain = a.scale * a.score.inv_softcap, aout = a.score.softcap * kLog2e;
    bool ok = true;
    for (int k = 0; k < n; ++k) {
      const int c = item_col(k);
      const bool partial = k >= nf;
      const int64_t j0 = (int64_t)c * 128;
      int* kdoc = sDoc + (k & 1) * 128;
      if (partial && a.rule.any_doc && tid < 128) kdoc[tid] = doc_at(a.rule, b, j0 + tid);
      if (grad_bar_any(!ok)) {
        ok = false;
        break;
      }
      uint32_t allowed[2] = {0xFFFFFFFFu, 0xFFFFFFFFu};  // this warpgroup's 64 key columns
      if (partial) {
        const int w = (int)min((int64_t)128, (int64_t)a.kv_len - j0);
        const Bits128 bits = rule_row_bits(a.rule, ig, j0, w, doc_i, [&](int d) {
          if (runs) return range_bits(clamp_rel(run_lo - j0, w), clamp_rel(run_hi - j0, w));
          return doc_bits<4>(w, d, [&](int cc) { return kdoc[cc]; });
        });
        allowed[0] = bits.w[2 * wg];
        allowed[1] = bits.w[2 * wg + 1];
      }
      if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_s + (k & 1), (uint32_t)((k >> 1) & 1), wc)))) continue;
      tc5_fence_after();
      float pg[64];
      uint32_t sv2[2][32];
      tc5_ld32(lane_addr + C::kQColS0 + 128 * (k & 1) + 64 * wg, sv2[0]);
      tc5_ld32(lane_addr + C::kQColS0 + 128 * (k & 1) + 64 * wg + 32, sv2[1]);
      tc5_wait_ld();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t (&sv)[32] = sv2[half];
        // ALiBi (log2 domain): -slope log2e (i_g - j) = base_w + slope log2e (column - 64 wg)
        const float base_w = -psl2 * (float)(ig - (j0 + 64 * wg));
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int cl = 32 * half + e;  // key column within this warpgroup's 64
          const float xr = __uint_as_float(sv[e]);
          float lg, g = 1.f;
          if constexpr (SK == SK_NONE) {
            lg = fmaf(xr, sl2, -lse2);
          } else if constexpr (SK == SK_ALIBI) {
            lg = fmaf(xr, sl2, fmaf(psl2, (float)cl, base_w) - lse2);
          } else if constexpr (SK == SK_SOFTCAP) {
            const float t = tanh_approx(xr * ain);
            lg = fmaf(t, aout, -lse2);
            g = 1.f - t * t;
          } else {
            lg = score_g(a.score, h, xr * a.scale, ig - (j0 + 64 * wg + cl), slope, g) * kLog2e - lse2;
          }
          float p = ex2_approx(lg);
          if (partial && !((allowed[half] >> e) & 1u)) p = 0.f;
          pg[cl] = SK == SK_SOFTCAP || SK == SK_GENERIC ? p * g : p;
        }
      }
      if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_dp, (uint32_t)(k & 1), wc)))) continue;
      tc5_fence_after();
      uint32_t dv2[2][32];
      tc5_ld32(lane_addr + C::kQColDP + 64 * wg, dv2[0]);
      tc5_ld32(lane_addr + C::kQColDP + 64 * wg + 32, dv2[1]);
      tc5_wait_ld();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t (&dv)[32] = dv2[half];
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          pk[e >> 1] = pack_bf16x2(pg[32 * half + e] * (__uint_as_float(dv[e]) - dlt),
                                 pg[32 * half + e + 1] * (__uint_as_float(dv[e + 1]) - dlt));
        tc5_st16(lane_addr + C::kQColDP + 64 * wg + 16 * half, pk);
      }
      tc5_wait_st();
      tc5_fence_before();
      mbar_arrive(bar_ds);
    }
    // ---- epilogue: dQ = scale * (dS K) of this query row, fp32 (rows past q_len are not written)
    // (tcgen05.ld is warp-collective: every lane loads, only rows inside the sequence store)
    const bool done = __all_sync(0xFFFFFFFFu, n == 0 || mbar_wait_drain(bar_done, 0, a.timeout_ns));
    tc5_fence_after();
    const bool in = i < a.q_len;
    if (ok && done) {
      float* dQg = a.dq + (in ? qrow : 0) * D + wg * (D / 2);
#pragma unroll
      for (int part = 0; part < D / 64; ++part) {
        uint32_t v[32];
        if (n > 0) {
          tc5_ld32(lane_addr + C::kQColDQ + wg * (D / 2) + 32 * part, v);
          tc5_wait_ld();
        }
#pragma unroll
        for (int e = 0; e < 32 && in; e += 4)
          *reinterpret_cast<float4*>(dQg + 32 * part + e) =
              n > 0 ? make_float4(__uint_as_float(v[e]) * a.scale, __uint_as_float(v[e + 1]) * a.scale,
                                  __uint_as_float(v[e + 2]) * a.scale, __uint_as_float(v[e + 3]) * a.scale)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  tc5_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc5_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int SK>
int launch_tc5(const BwdArgs& a, cudaStream_t st) {
  using C = BwdTc5<D>;
  CUtensorMap tq, tk, tv, tdo;
  const uint64_t dq[3] = {(uint64_t)D, (uint64_t)a.q_len, (uint64_t)a.B * a.Hq};
  const uint64_t dk[3] = {(uint64_t)D, (uint64_t)a.kv_len, (uint64_t)a.B * a.Hkv};
  const uint64_t sq[2] = {(uint64_t)D * 2, (uint64_t)a.q_len * D * 2};
  const uint64_t sk[2] = {(uint64_t)D * 2, (uint64_t)a.kv_len * D * 2};
  const uint32_t box[3] = {64, 128, 1};
  if (encode_tmap_bf16(&tq, a.q, 3, dq, sq, box) || encode_tmap_bf16(&tk, a.k, 3, dk, sk, box) ||
      encode_tmap_bf16(&tv, a.v, 3, dk, sk, box) || encode_tmap_bf16(&tdo, a.dout, 3, dq, sq, box))
    return FA_ERR_CUDA;
  Tc5BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.a = a;
  auto kq = bwd_q_tc5_kernel<D, SK>;
  auto kk = bwd_kv_tc5_kernel<D, SK>;
  if (cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kQSmem) != cudaSuccess ||
      cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kKvSmem) != cudaSuccess)
    return FA_ERR_CUDA;
  kq<<<dim3(a.mask.nq, a.Hq, a.B), kThreads, C::kQSmem, st>>>(p, tq, tk, tv, tdo);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  kk<<<dim3(a.mask.nk, a.Hkv, a.B), kThreads, C::kKvSmem, st>>>(p, tq, tk, tv, tdo);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

// dQ and dK/dV on tcgen05 for 128 x 128 blocks (the delta kernel has run). FA_ERR_UNSUPPORTED: other
// shapes, which the mma.sync kernels take.
int launch_bwd_tc5(const BwdArgs& a, cudaStream_t st) {
  if (a.mask.bq != 128 || a.mask.bk != 128) return FA_ERR_UNSUPPORTED;
  if (a.mask.nq > 65535 * 1024 || a.Hq > 65535 || a.B > 65535) return FA_ERR_UNSUPPORTED;
  const bool al = a.score.alibi != nullptr, rel = a.score.rel != nullptr, cap = a.score.softcap > 0.f;
  const int sk = (!al && !rel && !cap) ? SK_NONE : (al && !rel && !cap) ? SK_ALIBI : (!al && !rel && cap) ? SK_SOFTCAP : SK_GENERIC;
  if (a.d == 128) {
    if (sk == SK_NONE) return launch_tc5<128, SK_NONE>(a, st);
    if (sk == SK_ALIBI) return launch_tc5<128, SK_ALIBI>(a, st);
    if (sk == SK_SOFTCAP) return launch_tc5<128, SK_SOFTCAP>(a, st);
    return launch_tc5<128, SK_GENERIC>(a, st);
  }
  if (a.d == 64) {
    if (sk == SK_NONE) return launch_tc5<64, SK_NONE>(a, st);
    if (sk == SK_ALIBI) return launch_tc5<64, SK_ALIBI>(a, st);
    if (sk == SK_SOFTCAP) return launch_tc5<64, SK_SOFTCAP>(a, st);
    return launch_tc5<64, SK_GENERIC>(a, st);
  }
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
