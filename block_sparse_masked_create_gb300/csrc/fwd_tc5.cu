// Block-sparse masked attention forward on 5th-generation tensor cores (tcgen05, accumulators in tensor
// memory), 128 x 128 blocks, head dim 64 or 128.
//
// What it computes is "5.1.2 FlexAttention: from rules to fused kernels", section 3.1 (and
// "FlexAttention: compiler optimisation of custom attention", section 3): per query block, visit the
// BlockMask's full blocks without the mask and its partial blocks with it; per block S = scale * Q K^T,
// score rule, -inf for masked pairs (partial blocks only), online softmax (m, l), acc += P V; finally
// O = acc / l and LSE = m + ln l, an empty row giving O = 0, LSE = -inf.
//
// How (one CTA = NT query tiles of 128 rows: two tiles of sibling heads of the same query block in 18
// warps, or, for short sliding windows of MHA, one tile in 10 warps with two CTAs per SM):
//   warps 8t .. 8t+7  the softmax of tile t, two warpgroups each owning 64 of a block's 128 key columns
//                    (TMEM lane = query row = 32 * (warp % 4) + lane). Per block: S from TMEM to
//                    registers, score rule, mask (partial blocks only), half-row max exchanged through
//                    shared memory, P = 2^(x - m) with packed fp32x2 FMAs, two row sums, P as bf16 back into
//                    tensor memory over the S columns it came from, "P ready". The O accumulator is
//                    rescaled in TMEM only when the running max grows by more than 2^8 (exact for any
//                    reference max; the bound keeps P <= 256). Epilogue O / l -> shared memory -> TMA store.
//   warp 8 NT        TMA producer: Q tiles, then K / V tiles of the visited blocks only (an empty block
//                    issues no load) into a shared-memory ring, in exactly the order the MMA warp consumes
//                    them. Sibling query heads of one KV head with the same mask row share each K / V load.
//   warp 8 NT + 1    allocates TMEM (S/P and O of every tile: 256 columns per tile) and issues every
//                    tcgen05.mma from one thread: when P_t(j) is ready, O_t += P_t(j) V(j) (A read from
//                    TMEM) and then S_t(j+1) = Q_t K(j+1)^T (A, B from shared memory). The tensor pipe runs a
//                    thread's MMAs in issue order, so S_t(j+1) overwrites P_t(j) only after the product has
//                    read it, and the completion of S_t(j) implies that of O_t's previous update.
// Two tiles in flight keep the tensor core busy while each tile's softmax runs. Every wait is bounded (an
// abort flag stops all roles; copies and MMAs in flight are drained before tensor memory is freed and the
// CTA exits).
#include <cstring>

#include "fa_launch.h"

namespace fa {
namespace {

// NT query tiles per CTA (2: one CTA per SM; 1: two CTAs per SM, whose start-up and epilogue then
// overlap each other's work). Per tile 8 softmax warps (2 warpgroups), then the TMA producer and the MMA
// issuer. At most five warps share an SM sub-partition either way, which caps a thread at 96 registers;
// the softmax fits (it holds 64 scores).
template <int NT>
struct Roles {
  static constexpr int kLoadWarp = 8 * NT;
  static constexpr int kMmaWarp = 8 * NT + 1;
  static constexpr int kThreads = (8 * NT + 2) * 32;
  static constexpr int kCtasPerSm = NT == 2 ? 1 : 2;
};
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P values stay <= 2^8
constexpr int kGroupPairs = 8;             // (batch, head pair) units sharing the L2 at a time

enum ScoreKind { SK_NONE = 0, SK_ALIBI = 1, SK_SOFTCAP = 2, SK_GENERIC = 3 };

template <int D, int NT>
struct Tc5Cfg {
  static constexpr int kQBytes = 128 * D * 2;      // one Q tile (also the O staging tile)
  static constexpr int kSlotBytes = 128 * D * 2;   // one K or V tile
  // K / V ring: what is left of the shared memory of an SM (two CTAs: half of it each)
  static constexpr int kStages = NT == 2 ? (D == 128 ? 5 : 12) : (D == 128 ? 2 : 5);
  static constexpr int kOffRing = NT * kQBytes;
  static constexpr int kOffRed = kOffRing + kStages * kSlotBytes;  // float [tile][half][row] exchange
  static constexpr int kOffBar = kOffRed + 2 * 2 * 128 * 4;        // mbarriers, TMEM address, abort flag
  static constexpr int kSmem = kOffBar + 512;
  static_assert(kSmem * (NT == 2 ? 1 : 2) + (NT == 2 ? 0 : 1024) <= 227 * 1024, "shared memory budget");
  static constexpr uint32_t kTmemCols = 256 * NT;
  // tensor-memory columns: S_t at [256 t, 256 t + 128), with P_t (bf16 pairs) over columns [0, 32) and
  // [64, 96) of it (keys 0..63 and 64..127); O_t at [256 t + 128, 256 t + 128 + D)
  __device__ static constexpr uint32_t col_s(int t) { return (uint32_t)t * 256u; }
  __device__ static constexpr uint32_t col_o(int t) { return (uint32_t)t * 256u + 128u; }
};

struct Tc5Params {
  FwdArgs a;
  int ahead;  // CTAs per wave: the CTA this many ids later runs next on the SM this one frees
};

// byte offset of 16-byte chunk c16 of row `row` in a [128][D] tile stored as D/64 sub-tiles [128][64]
// with the 128-byte swizzle (TMA SWIZZLE_128B layout; also the UMMA K-major SW128 layout)
__device__ __forceinline__ uint32_t tile_off(int row, int c16) {
  return (uint32_t)((c16 >> 3) * 16384 + row * 128 + (((c16 & 7) ^ (row & 7)) << 4));
}

struct Tile {
  int valid;     // a tile exists (Hq may be odd)
  int h, hk;     // query head, KV head
  int n_full, n;
  const int32_t* full_idx;
  const int32_t* part_idx;
  __device__ __forceinline__ int col(int j) const {
    return j < n_full ? __ldg(full_idx + j) : __ldg(part_idx + j - n_full);
  }
};

__device__ __forceinline__ Tile make_tile(const FwdArgs& a, int b, int h, int r) {
  const DevMask& M = a.mask;
  Tile T;
  T.valid = h < a.Hq;
  T.h = T.valid ? h : 0;
  T.hk = T.h / (a.Hq / a.Hkv);
  const int bm = M.Bm > 1 ? b : 0, hm = M.Hm > 1 ? T.h : 0;
  const size_t mrow = ((size_t)bm * M.Hm + hm) * M.nq + r;
  T.n_full = T.valid ? __ldg(M.full_kv_num + mrow) : 0;
  T.n = T.valid ? T.n_full + __ldg(M.kv_num + mrow) : 0;
  T.full_idx = M.full_kv_idx + mrow * M.nk;
  T.part_idx = M.kv_idx + mrow * M.nk;
  return T;
}

// Work item p -> (batch b, head group hp of NT heads, query block r). The (b, hp) units are taken in groups of
// kGroupPairs; within a group the query blocks follow the mask's row order (longest rows first, so the
// short ones fill the tail; for causal masks the last block first) with the group's pairs side by side,
// so the CTAs resident at any time share the K / V of a few heads in L2 instead of streaming every
// head's K / V from DRAM once per query block.
template <int NT>
__device__ __forceinline__ void work_item(const FwdArgs& a, int p, int& b, int& hp, int& r) {
  const int HP = (a.Hq + NT - 1) / NT;
  const int nq = a.mask.nq;
  const int NP = a.B * HP;
  const int GS = NP < kGroupPairs ? NP : kGroupPairs;
  const int g = p / (GS * nq), g0 = g * GS, gs = min(GS, NP - g0);
  const int rem = p - g * GS * nq;
  const int pair = g0 + rem % gs;
  hp = pair % HP;
  b = pair / HP;
  // query blocks by visited length, longest first (the mask's row order; causal: nq-1 .. 0)
  const DevMask& M = a.mask;
  r = M.row_order ? __ldg(M.row_order + ((size_t)(M.Bm > 1 ? b : 0) * M.Hm + (M.Hm > 1 ? NT * hp : 0)) * nq + rem / gs)
                  : nq - 1 - rem / gs;
}

template <int D, int SK, int NT>
__global__ void __launch_bounds__(Roles<NT>::kThreads, Roles<NT>::kCtasPerSm)
    fwd_tc5_kernel(const __grid_constant__ Tc5Params P, const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmO) {
  using C = Tc5Cfg<D, NT>;
  constexpr int kLoadWarp = Roles<NT>::kLoadWarp;
  constexpr int kMmaWarp = Roles<NT>::kMmaWarp;
  constexpr int NST = C::kStages;
  const FwdArgs& a = P.a;
  // All shared state is dynamic (no static __shared__), so the buffer starts at the CTA's shared
  // window and keeps the 1024-byte alignment the 128-byte swizzle needs; checked below, never assumed.
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* const bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* const bar_q = bars;          // [2] Q tile landed
  uint64_t* const bar_s = bars + 2;      // [2] S = Q K^T complete
  uint64_t* const bar_p = bars + 4;      // [2] P stored in tensor memory (both halves, 256 arrivals)
  uint64_t* const bar_o = bars + 6;      // [2] O += P V complete
  uint64_t* const bar_full = bars + 8;   // [NST] ring slot landed
  uint64_t* const bar_empty = bars + 8 + NST;  // [NST] ring slot consumed
  uint64_t& bar_drain = bars[8 + 2 * NST];
  uint32_t& s_tmem = *reinterpret_cast<uint32_t*>(bars + 9 + 2 * NST);
  int32_t& s_abort = *(reinterpret_cast<int32_t*>(bars + 9 + 2 * NST) + 1);
  // Half-row maxima of the current block, [tile][half][row]; one buffer suffices: a half writes block
  // j+1's value only after S(j+1) completed, which the MMA issues only after both halves signalled P(j),
  // i.e. after both had read block j's values. The epilogue reuses it for the row sums.
  float (*const s_red)[2][128] = reinterpret_cast<float (*)[2][128]>(smem + C::kOffRed);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (smem_u32(smem) & 1023u) {  // uniform across the CTA, before any barrier or allocation
    if (tid == 0) report(a.status, FA_ERR_DEVICE_CHECK);
    return;
  }

  // ---- work item: (query block r, batch b, head pair hp)
  const DevMask& M = a.mask;
  int b, hp, r;
  work_item<NT>(a, blockIdx.x, b, hp, r);
  const Tile T0 = make_tile(a, b, NT * hp, r);
  const Tile T1 = make_tile(a, b, NT == 2 ? 2 * hp + 1 : a.Hq, r);  // NT = 1: no second tile
  // sibling heads of one KV head with the same mask row share K / V loads
  const bool shared_kv = T1.valid && T0.hk == T1.hk && T0.n > 0 && M.Hm == 1;
  const int nmax = max(T0.n, T1.n);

  uint8_t* sQ0 = smem;
  uint8_t* sQ1 = smem + C::kQBytes;
  uint8_t* sRing = smem + C::kOffRing;

  // ring loads issued so far (producer warp); the ring fill starts before the CTA-wide barrier below
  int issued = 0;
  auto load_slot = [&](const Tile& T, bool is_v, int j) {  // into the next slot, which must be free
    const int s = issued % NST;
    const int c = T.col(j);
    int yk = c * 128, zk = b * a.Hkv + T.hk;
    if (a.page_table) {  // key block c is one whole page; a bad page id is reported and page 0 read instead
      int pg = __ldg(a.page_table + (size_t)b * a.max_pages + c);
      if (pg < 0 || pg >= a.n_pages_total) {
        if (lane == 0) report(a.status, FA_ERR_DEVICE_CHECK);
        pg = 0;
      }
      yk = 0;
      zk = pg * a.Hkv + T.hk;
    }
    uint8_t* dst = sRing + s * C::kSlotBytes;
    mbar_arrive_expect_tx_elect(&bar_full[s], C::kSlotBytes);
#pragma unroll
    for (int x = 0; x < D / 64; ++x)
      tma_load_3d_elect(dst + x * 16384, is_v ? &tmV : &tmK, x * 64, yk, zk, &bar_full[s]);
    ++issued;
  };
  if (warp == kLoadWarp) {
    // The producer sets up the barriers and sends the Q tiles and the first K tiles at once (they need
    // nothing else), while the MMA warp allocates tensor memory.
    if (lane == 0) {
      s_abort = 0;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        mbar_init(&bar_q[t], 1);
        mbar_init(&bar_s[t], 1);
        mbar_init(&bar_p[t], 256);
        mbar_init(&bar_o[t], 1);
      }
      for (int s = 0; s < NST; ++s) {
        mbar_init(&bar_full[s], 1);
        mbar_init(&bar_empty[s], 1);
      }
      mbar_init(&bar_drain, 1);
      fence_mbar_init();
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmO);
    }
    __syncwarp();
    if (T0.n > 0) {
      mbar_arrive_expect_tx_elect(&bar_q[0], C::kQBytes);
#pragma unroll
      for (int x = 0; x < D / 64; ++x) tma_load_3d_elect(sQ0 + x * 16384, &tmQ, x * 64, r * 128, b * a.Hq + T0.h, &bar_q[0]);
    }
    if (T1.n > 0) {
      mbar_arrive_expect_tx_elect(&bar_q[1], C::kQBytes);
#pragma unroll
      for (int x = 0; x < D / 64; ++x) tma_load_3d_elect(sQ1 + x * 16384, &tmQ, x * 64, r * 128, b * a.Hq + T1.h, &bar_q[1]);
    }
    // first K tiles in load order (K(0) shared, or K0(0) K1(0)); at most two, the ring has more slots
    if (shared_kv) {
      load_slot(T0, false, 0);
    } else {
      if (T0.n > 0) load_slot(T0, false, 0);
      if (T1.n > 0) load_slot(T1, false, 0);
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&s_tmem, C::kTmemCols);
    tmem_relinquish();
  }
  tc5_fence_before();
  __syncthreads();
  tc5_fence_after();
  const uint32_t tmem = s_tmem;
  WaitCtl wc{a.timeout_ns, a.status, &s_abort};

  if (warp == kLoadWarp) {
    // =============================== TMA producer ===============================
    // The whole warp runs this code (operands stay warp-uniform); elect.sync picks the lane that issues.
    // Load order == consumption order of the MMA warp:
    //   separate K/V: K0(0) K1(0), then per j: V0(j) K0(j+1) V1(j) K1(j+1)   (each only if it exists)
    //   shared K/V:   K(0), then per j: V(j) K(j+1)
    if (a.counters && lane == 0) {
      unsigned long long* cnt = reinterpret_cast<unsigned long long*>(a.counters);
      const int vis = T0.n + T1.n;
      atomicAdd(cnt + 0, (unsigned long long)(T0.valid + T1.valid));
      atomicAdd(cnt + 1, (unsigned long long)(T0.n_full + T1.n_full));
      atomicAdd(cnt + 2, (unsigned long long)(T0.n - T0.n_full + T1.n - T1.n_full));
      atomicAdd(cnt + 3, (unsigned long long)(shared_kv ? vis : 2 * vis));
    }
    __syncwarp();
    // the Q tiles of the CTA that will take this SM after the next wave go to L2 now, so its start does
    // not wait on DRAM
    if (P.ahead > 0 && blockIdx.x + P.ahead < gridDim.x && lane == 0) {
      int bn, hpn, rn;
      work_item<NT>(a, blockIdx.x + P.ahead, bn, hpn, rn);
#pragma unroll
      for (int tt = 0; tt < NT; ++tt) {
        const Tile Tn = make_tile(a, bn, NT * hpn + tt, rn);
        if (Tn.n == 0) continue;
#pragma unroll
        for (int x = 0; x < D / 64; ++x) tma_prefetch_l2_3d(&tmQ, x * 64, rn * 128, bn * a.Hq + Tn.h);
      }
    }
    __syncwarp();
    bool ok = true;
    auto load = [&](const Tile& T, bool is_v, int j) -> bool {
      const int s = issued % NST;
      if (issued >= NST &&
          !__all_sync(0xFFFFFFFFu, mbar_wait(&bar_empty[s], (uint32_t)(((issued / NST) - 1) & 1), wc)))
        return false;
      load_slot(T, is_v, j);
      return true;
    };
    // K(0) / K0(0) K1(0) went out before the CTA-wide barrier
    if (shared_kv) {
      for (int j = 0; j < T0.n && ok; ++j) {
        ok = load(T0, true, j);
        if (ok && j + 1 < T0.n) ok = load(T0, false, j + 1);
      }
    } else {
      for (int j = 0; j < nmax && ok; ++j) {
        if (j < T0.n) {
          ok = load(T0, true, j);
          if (ok && j + 1 < T0.n) ok = load(T0, false, j + 1);
        }
        if (ok && j < T1.n) {
          ok = load(T1, true, j);
          if (ok && j + 1 < T1.n) ok = load(T1, false, j + 1);
        }
      }
    }
    if (!ok || *wc.abort) {
      // drain: the last NST issued copies may still be landing in shared memory
      for (int i = max(0, issued - NST); i < issued; ++i)
        mbar_wait_drain(&bar_full[i % NST], (uint32_t)((i / NST) & 1), a.timeout_ns);
      if (T0.n > 0) mbar_wait_drain(&bar_q[0], 0, a.timeout_ns);
      if (T1.n > 0) mbar_wait_drain(&bar_q[1], 0, a.timeout_ns);
    }
  } else if (warp == kMmaWarp) {
    // =============================== MMA issuer ===============================
    // Warp-uniform like the producer; each tcgen05.mma / commit is issued by one elected lane.
    // Descriptors: base values computed once, per-MMA offsets added to the 14-bit address field.
    constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
    const uint64_t qdesc0 = sdesc_sw128(smem_u32(sQ0), 16, 1024), qdesc1 = sdesc_sw128(smem_u32(sQ1), 16, 1024);
    const uint64_t kdesc = sdesc_sw128(smem_u32(sRing), 16, 1024);
    const uint64_t vdesc = sdesc_sw128(smem_u32(sRing), 128 * 128, 1024);
    int consumed = 0;
    bool ok = true;
    if (T0.n > 0) ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar_q[0], 0, wc));
    if (ok && T1.n > 0) ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar_q[1], 0, wc));
    tc5_fence_after();
    auto take = [&]() -> int {  // wait for the next ring slot in load order
      const int s = consumed % NST;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_full[s], (uint32_t)((consumed / NST) & 1), wc))) return -1;
      tc5_fence_after();
      ++consumed;
      return s;
    };
    auto mma_qk = [&](int t, int s) {
      const uint64_t qd = t ? qdesc1 : qdesc0;
      const uint64_t kd = kdesc + (uint64_t)(s * (C::kSlotBytes >> 4));
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t off = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
        tc5_mma_ss_elect(tmem + C::col_s(t), qd + off, kd + off, idesc_qk, ks > 0 ? 1u : 0u);
      }
      tc5_commit_elect(&bar_s[t]);
    };
    auto mma_pv = [&](int t, int s, bool acc) {
      const uint64_t vd = vdesc + (uint64_t)(s * (C::kSlotBytes >> 4));
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        tc5_mma_ts_elect(tmem + C::col_o(t), tmem + C::col_s(t) + (uint32_t)(ks * 8 + (ks >= 4 ? 32 : 0)),
                         vd + (uint64_t)((ks * 2048) >> 4),
                         idesc_pv, (acc || ks > 0) ? 1u : 0u);
      tc5_commit_elect(&bar_o[t]);
    };
    auto wait_p = [&](int t, int j) -> bool {
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_p[t], (uint32_t)(j & 1), wc))) return false;
      tc5_fence_after();
      return true;
    };
    if (ok) {
      if (shared_kv) {
        const int n = T0.n;
        int sk = take();
        ok = sk >= 0;
        if (ok) {
          mma_qk(0, sk);
          mma_qk(1, sk);
          tc5_commit_elect(&bar_empty[sk]);
        }
        for (int j = 0; j < n && ok; ++j) {
          // V(j) and K(j+1) landed long ago: take their slots before waiting for P, so that the wait on
          // their barriers is off the path from P(j) to the next products
          const int sv = take();
          if (sv < 0) { ok = false; break; }
          sk = -1;
          if (j + 1 < n && (sk = take()) < 0) { ok = false; break; }
          if (!(ok = wait_p(0, j))) break;
          mma_pv(0, sv, j > 0);
          if (sk >= 0) mma_qk(0, sk);
          if (!(ok = wait_p(1, j))) break;
          mma_pv(1, sv, j > 0);
          tc5_commit_elect(&bar_empty[sv]);
          if (sk >= 0) {
            mma_qk(1, sk);
            tc5_commit_elect(&bar_empty[sk]);
          }
        }
      } else {
        if (T0.n > 0) {
          const int s = take();
          if (s < 0) ok = false;
          else { mma_qk(0, s); tc5_commit_elect(&bar_empty[s]); }
        }
        if (ok && T1.n > 0) {
          const int s = take();
          if (s < 0) ok = false;
          else { mma_qk(1, s); tc5_commit_elect(&bar_empty[s]); }
        }
        for (int j = 0; j < nmax && ok; ++j) {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int nt = t ? T1.n : T0.n;
            if (!ok || j >= nt) continue;
            // V_t(j) and K_t(j+1): slots taken before the wait for P (see above)
            const int sv = take();
            if (sv < 0) { ok = false; break; }
            int sk = -1;
            if (j + 1 < nt && (sk = take()) < 0) { ok = false; break; }
            if (!(ok = wait_p(t, j))) break;
            mma_pv(t, sv, j > 0);
            tc5_commit_elect(&bar_empty[sv]);
            if (sk >= 0) {
              mma_qk(t, sk);
              tc5_commit_elect(&bar_empty[sk]);
            }
          }
        }
      }
    }
    // every MMA issued so far has completed before tensor memory is read back or freed
    tc5_commit_elect(&bar_drain);
    mbar_wait_drain(&bar_drain, 0, a.timeout_ns);
  } else {
    // =============================== softmax warpgroups ===============================
    // Two warpgroups per tile: warpgroup (t, h) owns columns [64 h, 64 h + 64) of the 128 rows of tile t
    // (TMEM lane == query row == 32 * (warp % 4) + lane). The row maximum is exchanged through shared
    // memory once per block; the row sums stay per half and are added in the epilogue.
    const int t = warp >> 3;                 // tile
    const int h = (warp >> 2) & 1;           // column half
    const int row = (warp & 3) * 32 + lane;  // query row in the tile
    const Tile TT = t ? T1 : T0;
    uint8_t* const sQt = t ? sQ1 : sQ0;
    const int q_row = r * 128 + row;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::col_s(t);
    const uint32_t tO = tmem + lane_base + C::col_o(t);
    float* Lg = a.lse + ((size_t)b * a.Hq + TT.h) * a.q_len;
    if (TT.valid && TT.n == 0) {
      // empty query block: O = 0, LSE = -inf, nothing loaded (each half writes its half of the row)
      const int row_bytes = D * (a.out_f32 ? 4 : 2);
      uint8_t* Ob = reinterpret_cast<uint8_t*>(a.out) + (((size_t)b * a.Hq + TT.h) * a.q_len) * row_bytes;
      if (q_row < a.q_len) {
        const uint4 z = make_uint4(0, 0, 0, 0);
        for (int c16 = h * (row_bytes / 32); c16 < (h + 1) * (row_bytes / 32); ++c16)
          *reinterpret_cast<uint4*>(Ob + (size_t)q_row * row_bytes + c16 * 16) = z;
        if (h == 0) Lg[q_row] = -INFINITY;
      }
    } else if (TT.valid) {
      const int64_t off_b = a.rule.q_offset ? (int64_t)__ldg(a.rule.q_offset + (M.Bm > 1 ? b : 0)) : 0;
      const int64_t ig = (int64_t)q_row + off_b;
      const int bm = M.Bm > 1 ? b : 0;
      const int doc_i = a.rule.any_doc ? doc_at(a.rule, bm, ig) : -1;
      // document equality as the column interval of this row's run when the ids never decrease
      const bool runs = a.rule.any_doc && ig >= 0 && ig < a.rule.doc_len && doc_runs_usable(a.rule, bm);
      int64_t run_lo = 0, run_hi = 0;
      if (runs) doc_run_of(a.rule, bm, ig, run_lo, run_hi);
      const float sl2 = a.scale * kLog2e;
      float slope2 = 0.f;
      if (SK == SK_ALIBI || SK == SK_GENERIC) slope2 = a.score.alibi ? __ldg(a.score.alibi + TT.h) * kLog2e : 0.f;
      const int c_lo = 64 * h;                 // first column of this half within the block
      float m_ref = -INFINITY;  // reference max (log2 domain) used for P and for O
      // this half's row sum of P (for the LSE), and the correction that turns it into the sum O is divided
      // by: per block, the bf16 rounding error of the half's largest P (see the P loop)
      float le = 0.f, lc = 0.f;
      bool ok = true;
      // tcgen05.ld / st are warp-collective (.sync.aligned): every decision that guards one is made
      // uniform across the warp (wait results with __all_sync, the O rescale with __any_sync). The
      // loop always runs TT.n times so that both halves reach the tile's barrier equally often; after
      // a failed wait a warp only keeps the barrier count (its waits then return at once).
      // Each half touches only its own S columns [64 h, 64 h + 64); its P (64 keys as bf16 pairs) goes
      // over the first 32 of them.
      for (int j = 0; j < TT.n; ++j) {
        if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar_s[t], (uint32_t)(j & 1), wc));
        if (!ok) {
          named_bar_sync(1 + t, 256);
          continue;
        }
        tc5_fence_after();
        float x[64];
        tc5_ld32(tS + c_lo, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
        tc5_ld32(tS + c_lo + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
        tc5_wait_ld();
        const bool partial = j >= TT.n_full;
        const bool need_col = partial || SK != SK_NONE;
        const int c = need_col ? TT.col(j) : 0;
        const int64_t j0 = (int64_t)c * 128;
        // ---- score rule (log2 domain); SK_NONE defers the scale into the exponent's FMA
        const float mult = SK == SK_NONE ? sl2 : 1.f;
        if (SK == SK_ALIBI) {
          const float base = -slope2 * (float)(ig - j0 - c_lo);  // bias at this half's first column
          const uint64_t s2 = f2_pack(sl2, sl2), sp2 = f2_pack(slope2, slope2), b2 = f2_pack(base, base);
#pragma unroll
          for (int i = 0; i < 64; i += 2) {
            const uint64_t bias = f2_fma(sp2, f2_pack((float)i, (float)(i + 1)), b2);
            f2_unpack(f2_fma(f2_pack(x[i], x[i + 1]), s2, bias), x[i], x[i + 1]);
          }
        } else if (SK == SK_SOFTCAP) {
          // log2(e) c tanh(scale x / c), packed multiplies around the tanh
          const float ain = a.scale * a.score.inv_softcap, aout = a.score.softcap * kLog2e;
          const uint64_t in2 = f2_pack(ain, ain), out2 = f2_pack(aout, aout);
#pragma unroll
          for (int i = 0; i < 64; i += 2) {
            float u0, u1;
            f2_unpack(f2_mul(f2_pack(x[i], x[i + 1]), in2), u0, u1);
            f2_unpack(f2_mul(f2_pack(tanh_approx(u0), tanh_approx(u1)), out2), x[i], x[i + 1]);
          }
        } else if (SK == SK_GENERIC) {
          for (int i = 0; i < 64; ++i) {
            float v = x[i] * a.scale;
            const int64_t dist = ig - (j0 + c_lo + i);
            if (a.score.alibi) v -= (slope2 * kLn2) * (float)dist;
            if (a.score.rel) {
              int64_t ix = dist + a.score.kv_len - 1;
              ix = ix < 0 ? 0 : (ix > 2 * (int64_t)a.score.kv_len - 2 ? 2 * (int64_t)a.score.kv_len - 2 : ix);
              v += __ldg(a.score.rel + (size_t)TT.h * (2 * (size_t)a.score.kv_len - 1) + ix);
            }
            if (a.score.softcap > 0.f) v = softcap_apply(v, a.score.softcap, a.score.inv_softcap);
            x[i] = v * kLog2e;
          }
        }
        // ---- mask after the score rule, partial blocks only
        if (partial) {
          // this half's 64 columns only
          const int64_t jh = j0 + c_lo;
          const int w = (int)max((int64_t)0, min((int64_t)64, (int64_t)a.kv_len - jh));
          Bits128 bits = {{0u, 0u, 0u, 0u}};
          if (q_row < a.q_len && w > 0) {
            bits = rule_row_bits(a.rule, ig, jh, w, doc_i, [&](int dq) {
              if (runs) return range_bits(clamp_rel(run_lo - jh, w), clamp_rel(run_hi - jh, w));
              return doc_bits<2>(w, dq, [&](int cc) { return doc_at(a.rule, bm, jh + cc); });
            });
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const uint32_t wd = bits.w[k];
#pragma unroll
            for (int i = 0; i < 32; ++i) x[k * 32 + i] = ((wd >> i) & 1u) ? x[k * 32 + i] : -INFINITY;
          }
        }
        // ---- this half's max: 4 independent 3-input max chains; then the row max across both halves
        float mxk[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) mxk[k] = fmaxf(x[k], x[k + 4]);
#pragma unroll
        for (int i = 8; i < 64; i += 8)
#pragma unroll
          for (int k = 0; k < 4; ++k) mxk[k] = fmax3(mxk[k], x[i + k], x[i + 4 + k]);
        const float hmax = fmaxf(fmaxf(mxk[0], mxk[1]), fmaxf(mxk[2], mxk[3]));
        s_red[t][h][row] = hmax * mult;
        named_bar_sync(1 + t, 256);
        const float mb = fmaxf(s_red[t][0][row], s_red[t][1][row]);
        // ---- reference max: move it only when the block max exceeds it by more than 2^8
        float alpha = 1.f;
        bool rescale = false;
        if (mb > m_ref + kRescaleThreshold || (m_ref == -INFINITY && mb > -INFINITY)) {
          alpha = m_ref == -INFINITY ? 0.f : ex2_approx(m_ref - mb);
          rescale = j > 0 && m_ref != -INFINITY;
          m_ref = mb;
        }
        const float mr = m_ref == -INFINITY ? 0.f : m_ref;
        // ---- P = 2^(mult * x - m), stored as bf16 16 columns (32 keys) at a time, and the row sum of the
        // unrounded P. The product multiplies the bf16-rounded P; O is divided by the unrounded sum plus, per
        // block, the rounding error of this half's largest P (the same FMA and ex2 on the same input give
        // that element's P bit for bit). A row dominated by one key then gets that key's V row with an exact
        // weight, as if O were divided by the sum of the rounded values; what is left is the rounding of
        // the smaller weights, at most 2^-9 of their share.
        const uint64_t mul2 = f2_pack(mult, mult), neg2 = f2_pack(-mr, -mr);
        uint64_t se[2] = {0, 0};
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float y0, y1;
            f2_unpack(f2_fma(f2_pack(x[32 * ch + 2 * i], x[32 * ch + 2 * i + 1]), mul2, neg2), y0, y1);
            const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
            pk[i] = pack_bf16x2(p0, p1);
            se[i & 1] = f2_add(se[i & 1], f2_pack(p0, p1));
          }
          tc5_st16(tS + c_lo + 16 * ch, pk);
        }
        const float ph = ex2_approx(fmaf(hmax, mult, -mr));
        const float ch_err = __uint_as_float(pack_bf16x2(ph, 0.f) << 16) - ph;
        float e0, e1;
        f2_unpack(f2_add(se[0], se[1]), e0, e1);
        le = le * alpha + (e0 + e1);
        lc = lc * alpha + ch_err;
        // ---- O is stable here: S_t(j) completed, and O_t's previous update was issued before it.
        // Each half rescales its half of O's columns.
        if (__any_sync(0xFFFFFFFFu, rescale)) {
          const float f = rescale ? alpha : 1.f;
#pragma unroll
          for (int c0 = 0; c0 < D / 2; c0 += 32) {
            uint32_t o[32];
            tc5_ld32(tO + h * (D / 2) + c0, o);
            tc5_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
            tc5_st32(tO + h * (D / 2) + c0, o);
          }
        }
        tc5_wait_st();
        tc5_fence_before();
        mbar_arrive(&bar_p[t]);
      }
      // ---- epilogue: add the two halves' sums, wait for the last O update, normalise and store
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar_o[t], (uint32_t)((TT.n - 1) & 1), wc));
      tc5_fence_after();
      // the last O update completed after both halves read the last block's maxima: the exchange
      // buffer is free for the two sums, one at a time
      s_red[t][h][row] = le + lc;
      named_bar_sync(1 + t, 256);
      const float lt = s_red[t][0][row] + s_red[t][1][row];
      named_bar_sync(1 + t, 256);
      s_red[t][h][row] = le;
      named_bar_sync(1 + t, 256);
      const float let = s_red[t][0][row] + s_red[t][1][row];
      const bool empty = m_ref == -INFINITY;
      const float inv = empty ? 0.f : 1.f / lt;
      if (ok && h == 0 && q_row < a.q_len) Lg[q_row] = empty ? -INFINITY : (m_ref + __log2f(let)) * kLn2;
      const bool issuer = h == 0 && (warp & 3) == 0 && lane == 0;
      // fp32 O (two slots' worth) is staged in the K / V ring when both tiles visit the same number of
      // blocks (or one visits none): then, once this tile's last product completed, every ring slot but
      // the one of the CTA's last load has been consumed, in both load orders. Tile t takes the slots of
      // the loads 2 + 2t and 3 + 2t from the end (distinct, the ring has at least five slots); boxes
      // [128][32] (128-byte rows, 128-byte swizzle), half h filling its D/64 boxes.
      const int n_loads = shared_kv ? 2 * T0.n : 2 * (T0.n + T1.n);
      const bool ring_stage = a.out_f32 && (T0.n == T1.n || T0.n == 0 || T1.n == 0);
      auto box_smem = [&](int kb) -> uint8_t* {
        // one tile per CTA: its last product is the CTA's last MMA, so every slot is free
        int sl = (n_loads - ((NT == 2 ? 2 + 2 * t : 1) + (kb * 16384) / C::kSlotBytes)) % NST;
        sl = sl < 0 ? sl + NST : sl;
        return sRing + sl * C::kSlotBytes + (kb * 16384) % C::kSlotBytes;
      };
      if (ring_stage) {
        if (ok) {
#pragma unroll
          for (int kb = h * (D / 64); kb < (h + 1) * (D / 64); ++kb) {
            uint8_t* const stg = box_smem(kb);
            uint32_t o[32];
            tc5_ld32(tO + kb * 32, o);
            tc5_wait_ld();
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              float4 v = make_float4(__uint_as_float(o[4 * q4 + 0]) * inv, __uint_as_float(o[4 * q4 + 1]) * inv,
                                     __uint_as_float(o[4 * q4 + 2]) * inv, __uint_as_float(o[4 * q4 + 3]) * inv);
              *reinterpret_cast<float4*>(stg + row * 128 + ((q4 ^ (row & 7)) << 4)) = v;
            }
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1 + t, 256);
        if (!*wc.abort && issuer) {
#pragma unroll
          for (int kb = 0; kb < D / 32; ++kb) tma_store_3d(&tmO, box_smem(kb), kb * 32, r * 128, b * a.Hq + TT.h);
          bulk_commit_group();
        }
      }
      // otherwise staging in this tile's Q buffer (D/64 sub-buffers of 16 KB; free: every Q K^T of the
      // tile has completed). bf16: one round of D/64 boxes [128][64], each half filling its columns. fp32:
      // two rounds of boxes [128][32]; with D = 128 half h fills sub-buffer h with its columns 32 rd..
      // each round, with D = 64 half rd fills the only sub-buffer in round rd.
      const int rounds = ring_stage ? 0 : (a.out_f32 ? 2 : 1);
      for (int rd = 0; rd < rounds; ++rd) {
        if (rd > 0) {
          if (issuer) bulk_wait_group_read0();  // the previous round's boxes have left shared memory
          named_bar_sync(1 + t, 256);
        }
        if (ok) {
          if (!a.out_f32) {
#pragma unroll
            for (int c0 = 0; c0 < D / 2; c0 += 32) {
              uint32_t o[32];
              tc5_ld32(tO + h * (D / 2) + c0, o);
              tc5_wait_ld();
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(o[8 * q4 + 0]) * inv, __uint_as_float(o[8 * q4 + 1]) * inv);
                v.y = pack_bf16x2(__uint_as_float(o[8 * q4 + 2]) * inv, __uint_as_float(o[8 * q4 + 3]) * inv);
                v.z = pack_bf16x2(__uint_as_float(o[8 * q4 + 4]) * inv, __uint_as_float(o[8 * q4 + 5]) * inv);
                v.w = pack_bf16x2(__uint_as_float(o[8 * q4 + 6]) * inv, __uint_as_float(o[8 * q4 + 7]) * inv);
                *reinterpret_cast<uint4*>(sQt + tile_off(row, (h * (D / 2) + c0) / 8 + q4)) = v;
              }
            }
          } else if (D == 128 || h == rd) {
            uint8_t* const stg = sQt + (D == 128 ? h * 16384 : 0);
            uint32_t o[32];
            tc5_ld32(tO + (D == 128 ? h * 64 + rd * 32 : rd * 32), o);
            tc5_wait_ld();
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              float4 v = make_float4(__uint_as_float(o[4 * q4 + 0]) * inv, __uint_as_float(o[4 * q4 + 1]) * inv,
                                     __uint_as_float(o[4 * q4 + 2]) * inv, __uint_as_float(o[4 * q4 + 3]) * inv);
              *reinterpret_cast<float4*>(stg + row * 128 + ((q4 ^ (row & 7)) << 4)) = v;
            }
          }
        }
        // every thread of the tile reaches these barriers (ok or not); the store runs only if no role
        // gave up (a failed wait always sets the CTA's abort flag)
        fence_proxy_async_smem();
        named_bar_sync(1 + t, 256);
        if (!*wc.abort && issuer) {
          if (!a.out_f32) {
#pragma unroll
            for (int x = 0; x < D / 64; ++x) tma_store_3d(&tmO, sQt + x * 16384, x * 64, r * 128, b * a.Hq + TT.h);
          } else {
#pragma unroll
            for (int x = 0; x < D / 64; ++x)
              tma_store_3d(&tmO, sQt + x * 16384, D == 128 ? x * 64 + rd * 32 : rd * 32, r * 128, b * a.Hq + TT.h);
          }
          bulk_commit_group();
        }
      }
      // the staging buffer must stay untouched until the last boxes have been read out of it
      if (issuer) bulk_wait_group_read0();
    }
  }
  tc5_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc5_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int SK, int NT>
int launch_k(const FwdArgs& a, cudaStream_t st) {
  using C = Tc5Cfg<D, NT>;
  CUtensorMap tq, tk, tv, to;
  const uint64_t dq[3] = {(uint64_t)D, (uint64_t)a.q_len, (uint64_t)a.B * a.Hq};
  // K / V: [B * Hkv, kv_len, D], or pages [n_pages_total * Hkv, 128, D] read one whole page per block
  const bool paged = a.page_table != nullptr;
  const uint64_t dk[3] = {(uint64_t)D, paged ? 128u : (uint64_t)a.kv_len,
                          paged ? (uint64_t)a.n_pages_total * a.Hkv : (uint64_t)a.B * a.Hkv};
  const uint64_t sq[2] = {(uint64_t)D * 2, (uint64_t)a.q_len * D * 2};
  const uint64_t sk[2] = {(uint64_t)D * 2, (paged ? 128u : (uint64_t)a.kv_len) * D * 2};
  const uint32_t box[3] = {64, 128, 1};
  if (encode_tmap_bf16(&tq, a.q, 3, dq, sq, box) || encode_tmap_bf16(&tk, a.k, 3, dk, sk, box) ||
      encode_tmap_bf16(&tv, a.v, 3, dk, sk, box))
    return FA_ERR_CUDA;
  if (a.out_f32) {
    const uint64_t so[2] = {(uint64_t)D * 4, (uint64_t)a.q_len * D * 4};
    const uint32_t boxo[3] = {32, 128, 1};
    if (encode_tmap_f32(&to, a.out, 3, dq, so, boxo)) return FA_ERR_CUDA;
  } else if (encode_tmap_bf16(&to, a.out, 3, dq, sq, box)) {
    return FA_ERR_CUDA;
  }
  Tc5Params p;
  std::memset(&p, 0, sizeof(p));
  p.a = a;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  p.ahead = sms * Roles<NT>::kCtasPerSm;
  const int n_items = a.B * a.mask.nq * ((a.Hq + NT - 1) / NT);
  auto kern = fwd_tc5_kernel<D, SK, NT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess)
    return FA_ERR_CUDA;
  kern<<<n_items, Roles<NT>::kThreads, C::kSmem, st>>>(p, tq, tk, tv, to);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D, int NT>
int launch_sk(const FwdArgs& a, cudaStream_t st) {
  const bool al = a.score.alibi != nullptr, rel = a.score.rel != nullptr, cap = a.score.softcap > 0.f;
  if (!al && !rel && !cap) return launch_k<D, SK_NONE, NT>(a, st);
  if (al && !rel && !cap) return launch_k<D, SK_ALIBI, NT>(a, st);
  if (!al && !rel && cap) return launch_k<D, SK_SOFTCAP, NT>(a, st);
  return launch_k<D, SK_GENERIC, NT>(a, st);
}

// Tiles per CTA. Two tiles of sibling heads share one CTA (and, for grouped query heads, every K / V
// load); one tile per CTA lets two CTAs share an SM, which pays where rows are short and a CTA's
// start-up and epilogue are a large part of its life.
// Measured: sliding windows of up to 2048 keys (at most 17 blocks a row) with one KV head per query head
// gain about 5 % with one tile per CTA; long rows lose about 8 % (the ring is then two slots deep), and
// grouped query heads would lose their shared K / V loads.
int tiles_per_cta(const FwdArgs& a) {
#ifdef FA_TC5_TILES
  (void)a;
  return FA_TC5_TILES;
#else
  bool windowed = a.rule.n_terms > 0;
  for (int i = 0; i < a.rule.n_terms; ++i)
    if (a.rule.t[i].win == INT64_MAX || a.rule.t[i].win > 2048) windowed = false;
  return (windowed && a.Hq == a.Hkv) ? 1 : 2;
#endif
}

template <int D>
int launch_d(const FwdArgs& a, cudaStream_t st) {
  return tiles_per_cta(a) == 1 ? launch_sk<D, 1>(a, st) : launch_sk<D, 2>(a, st);
}

}  // namespace

int launch_fwd_tc5(const FwdArgs& a, cudaStream_t st) {
  if (a.mask.bq != 128 || a.mask.bk != 128) return FA_ERR_UNSUPPORTED;
  if (a.B * (int64_t)a.mask.nq * ((a.Hq + 1) / 2) > 0x7FFFFFFF) return FA_ERR_UNSUPPORTED;
  if (a.d == 128) return launch_d<128>(a, st);
  if (a.d == 64) return launch_d<64>(a, st);
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
