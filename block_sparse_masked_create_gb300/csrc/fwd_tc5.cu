// Block-sparse masked attention forward on 5th-generation tensor cores (tcgen05, accumulators in tensor
// memory), 128 x 128 blocks, head dim 64 or 128.
//
// What it computes is "5.1.2 FlexAttention: from rules to fused kernels", section 3.1 (and
// "FlexAttention: compiler optimisation of custom attention", section 3): per query block, visit the
// BlockMask's full blocks without the mask and its partial blocks with it; per block S = scale * Q K^T,
// score rule, -inf for masked pairs (partial blocks only), online softmax (m, l), acc += P V; finally
// O = acc / l and LSE = m + ln l, an empty row giving O = 0, LSE = -inf.
//
// How (one CTA = two 128-row query tiles that read the same K / V: two query blocks of one head, or one
// query block of two sibling heads of a KV head; 10 warps):
//   warps 4t .. 4t+3  the softmax of tile t, one thread per query row (TMEM lane = query row = 32 * (warp
//                    % 4) + lane) over all 128 key columns of a block, so no value is exchanged between
//                    threads. Per block: S from TMEM to registers, score rule, mask (partial blocks only),
//                    row max, P = 2^(x - m) with packed fp32x2 FMAs, the row sum, P as bf16 back into
//                    tensor memory over the S columns it came from, "P ready" (one arrival per warp). The
//                    O accumulator is rescaled in TMEM only when the running max grows by more than 2^8
//                    (exact for any reference max; the bound keeps P <= 256); soft-capped scores take a
//                    fixed reference and no max pass. Epilogue O / l -> shared memory -> TMA store.
//   warp 8           TMA producer: Q tiles, then K / V tiles of the union of the two tiles' block lists
//                    (each block once; an empty block issues no load) into a shared-memory ring, in the
//                    order the MMA warp consumes them; with each K tile, the element's flags (which tiles
//                    visit it, whether it is the last), so the MMA warp does not walk the lists.
//   warp 9           allocates TMEM (S/P and O of both tiles: 512 columns) and issues every tcgen05.mma from
//                    one thread: per element of the union, for each tile that visits it, O_t += P_t V(prev)
//                    (A read from TMEM) once P_t is ready and then S_t = Q_t K^T (A, B from shared memory),
//                    each product one asm statement under one elect.
//                    The tensor pipe runs a thread's MMAs in issue order, so S_t overwrites P_t only after
//                    the product has read it, and the completion of S_t implies that of O_t's previous update.
// Each tile's softmax runs while the tensor core works on the other tile. Every wait is bounded (an abort
// flag stops all roles; copies and MMAs in flight are drained before tensor memory is freed and the CTA
// exits).
#include <cstring>

#include "fa_launch.h"

namespace fa {
namespace {

// Roles: two softmax warpgroups (one per tile), the TMA producer and the MMA issuer. At most three warps
// share an SM sub-partition, so a thread may hold 168 registers; the softmax holds a row's 128 scores.
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 10 * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P values stay <= 2^8
// A soft-capped score lies in (-c, c), so its exponent x log2(e) c spans less than 2 c log2(e): with the
// fixed reference c log2(e) - 64, P = 2^(x log2(e) c - m) stays within [2^(64 - 2 c log2(e)), 2^64], normal in
// fp32 and bf16 (and O, a sum of at most 2^31 such P times bf16 V, far from overflow) for c log2(e) <= 90.
// The softmax then needs no running maximum: no max pass before P, no O rescale.
constexpr float kCapFixedMax = 90.0f;   // largest c log2(e) that takes the fixed reference
constexpr float kCapFixedSpan = 64.0f;  // P <= 2^64

enum ScoreKind { SK_NONE = 0, SK_ALIBI = 1, SK_SOFTCAP = 2, SK_GENERIC = 3 };

template <int D>
struct Tc5Cfg {
  static constexpr int kQBytes = 128 * D * 2;      // one Q tile (also the O staging tile)
  static constexpr int kSlotBytes = 128 * D * 2;   // one K or V tile
  // K / V ring: what is left of the shared memory of an SM
  static constexpr int kStages = D == 128 ? 5 : 12;
  static constexpr int kOffRing = 2 * kQBytes;
  static constexpr int kOffBar = kOffRing + kStages * kSlotBytes;  // mbarriers, TMEM address, abort flag
  static constexpr int kSmem = kOffBar + 512;
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  static_assert((13 + 2 * kStages) * 8 + 4 * kStages <= 512, "barrier region");
  static constexpr uint32_t kTmemCols = 512;
  // tensor-memory columns: S_t at [256 t, 256 t + 128), with P_t (bf16 pairs: keys 2i, 2i+1 in column i)
  // over its first 64 columns; O_t at [256 t + 128, 256 t + 128 + D)
  __device__ static constexpr uint32_t col_s(int t) { return (uint32_t)t * 256u; }
  __device__ static constexpr uint32_t col_o(int t) { return (uint32_t)t * 256u + 128u; }
};

struct Tc5Params {
  FwdArgs a;
  int ahead;      // CTAs per wave: the CTA this many ids later runs next on the SM this one frees
  int pair_rows;  // two tiles: 1 = two query blocks of one head, 0 = sibling heads (one KV head), one block
  int desc;       // 1: visit each row's blocks from the highest column down, 0: from the lowest up
  int group;      // units whose items are interleaved (sharing the L2 at a time)
};

// byte offset of 16-byte chunk c16 of row `row` in a [128][D] tile stored as D/64 sub-tiles [128][64]
// with the 128-byte swizzle (TMA SWIZZLE_128B layout; also the UMMA K-major SW128 layout)
__device__ __forceinline__ uint32_t tile_off(int row, int c16) {
  return (uint32_t)((c16 >> 3) * 16384 + row * 128 + (((c16 & 7) ^ (row & 7)) << 4));
}

// One 128-row query tile: query head h (KV head hk), BlockMask row r, and the query block rq it reads
// (rq = r, or with split rows the block of entry r). O and LSE go to rows r * 128 .. of the output.
struct Tile {
  int valid;     // a tile exists (Hq or the number of query blocks may be odd)
  int h, hk, r, rq;
  int n_full, n_part, n;
  const int32_t* full_idx;
  const int32_t* part_idx;
};

__device__ __forceinline__ Tile make_tile(const FwdArgs& a, int b, int h, int r) {
  const DevMask& M = a.mask;
  Tile T;
  T.valid = h < a.Hq && r >= 0;
  T.h = T.valid ? h : 0;
  T.r = T.valid ? r : 0;
  T.rq = a.split_ncm > 1 ? T.r / a.split_ncm : T.r;
  T.hk = T.h / (a.Hq / a.Hkv);
  const int bm = M.Bm > 1 ? b : 0, hm = M.Hm > 1 ? T.h : 0;
  const size_t mrow = ((size_t)bm * M.Hm + hm) * M.nq + T.r;
  T.n_full = T.valid ? __ldg(M.full_kv_num + mrow) : 0;
  T.n_part = T.valid ? __ldg(M.kv_num + mrow) : 0;
  T.n = T.n_full + T.n_part;
  T.full_idx = M.full_kv_idx + mrow * M.nk;
  T.part_idx = M.kv_idx + mrow * M.nk;
  return T;
}

// A tile's visited blocks in column order, its full and partial lists (each ascending) merged. Ordering
// keys are the column (ascending walk) or minus the column (descending walk); an exhausted list has key
// INT_MAX. Every role of the CTA walks the same lists the same way.
struct Walk {
  int f, p, kf, kp;
  // The load is issued where the walk advances and read one element later; as a volatile asm statement
  // it keeps its place in the program (a read-only __ldg may be sunk to its first use, which would put a
  // cache round trip on the issuing warp's critical path at every element).
  static __device__ __forceinline__ int key(const int32_t* idx, int n, int i, bool desc) {
    const int k = i < n ? (desc ? n - 1 - i : i) : 0;
    int v;
    asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(idx + k));
    return i >= n ? INT_MAX : (desc ? -v : v);
  }
  __device__ __forceinline__ void init(const Tile& T, bool desc) {
    f = p = 0;
    kf = key(T.full_idx, T.n_full, 0, desc);
    kp = key(T.part_idx, T.n_part, 0, desc);
  }
  __device__ __forceinline__ int next_key() const { return min(kf, kp); }
  __device__ __forceinline__ bool next_partial() const { return kp < kf; }
  __device__ __forceinline__ void advance(const Tile& T, bool desc) {
    if (kp < kf) {
      ++p;
      kp = key(T.part_idx, T.n_part, p, desc);
    } else {
      ++f;
      kf = key(T.full_idx, T.n_full, f, desc);
    }
  }
};
__device__ __forceinline__ int key_col(int key, bool desc) { return desc ? -key : key; }

// The same walk with the loaded column ids kept as loaded: the ordering keys are derived where they are
// compared, so the load that advance() issues is first waited for at the next element rather than at once
// (the producer walks the union between its loads; a cache round trip per element would delay them).
struct LazyWalk {
  int f, p, nf, np, vf, vp, dsc;
  static __device__ __forceinline__ int load(const int32_t* idx, int n, int i, bool desc) {
    const int k = i < n ? (desc ? n - 1 - i : i) : 0;
    int v;
    asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(idx + k));
    return v;
  }
  __device__ __forceinline__ void init(const Tile& T, bool desc) {
    f = p = 0;
    nf = T.n_full;
    np = T.n_part;
    dsc = desc;
    vf = load(T.full_idx, nf, 0, desc);
    vp = load(T.part_idx, np, 0, desc);
  }
  __device__ __forceinline__ int kf() const { return f < nf ? (dsc ? -vf : vf) : INT_MAX; }
  __device__ __forceinline__ int kp() const { return p < np ? (dsc ? -vp : vp) : INT_MAX; }
  __device__ __forceinline__ int next_key() const { return min(kf(), kp()); }
  __device__ __forceinline__ bool next_partial() const { return kp() < kf(); }
  __device__ __forceinline__ void advance(const Tile& T, bool desc) {
    if (kp() < kf()) {
      ++p;
      vp = load(T.part_idx, np, p, desc);
    } else {
      ++f;
      vf = load(T.full_idx, nf, f, desc);
    }
  }
};

// The union of the two tiles' block sequences (both tiles read the same K / V: one batch row, one KV
// head), in the same order; each element says which tiles visit it. The producer walks it, loads K and V of
// each element once and passes the element's flags to the MMA warp with its K slot; the MMA warp issues each
// tile's products on its own elements.
struct Union {
  LazyWalk w0, w1;
  __device__ __forceinline__ void init(const Tile& T0, const Tile& T1, bool desc) {
    w0.init(T0, desc);
    w1.init(T1, desc);
  }
  __device__ __forceinline__ bool done() const { return min(w0.next_key(), w1.next_key()) == INT_MAX; }
  // column of the next element, which tiles visit it (and whether it is partial for them); then step past it
  __device__ __forceinline__ int take(const Tile& T0, const Tile& T1, bool desc, bool& in0, bool& in1,
                                      bool* part0 = nullptr, bool* part1 = nullptr) {
    const int k = min(w0.next_key(), w1.next_key());
    in0 = w0.next_key() == k;
    in1 = w1.next_key() == k;
    if (part0) *part0 = w0.next_partial();
    if (part1) *part1 = w1.next_partial();
    if (in0) w0.advance(T0, desc);
    if (in1) w1.advance(T1, desc);
    return key_col(k, desc);
  }
};

// Work item p -> batch b and the two tiles' (head, query block). Units of work, (batch, head pair) for
// sibling heads or (batch, head) for row pairs, are taken in groups of `group`; within a group the
// query blocks follow the mask's row order (longest rows first, so the short ones fill the tail; for
// causal masks the last block first) with the group's units side by side, so the CTAs resident at any
// time share the K / V of a few heads in L2. Row pairs are consecutive entries of the row order (for
// causal and sliding-window masks two adjacent query blocks), whose block lists mostly coincide.
__device__ __forceinline__ void work_item(const FwdArgs& a, int pair_rows, int group, int p, int& b, int& h0,
                                          int& h1, int& r0, int& r1) {
  const int HP = pair_rows ? a.Hq : (a.Hq + 1) / 2;         // units per batch row
  const int nq = a.mask.nq;
  const int RPU = pair_rows ? (nq + 1) / 2 : nq;             // items per unit
  const int NP = a.B * HP;
  const int GS = NP < group ? NP : group;
  const int g = p / (GS * RPU), g0 = g * GS, gs = min(GS, NP - g0);
  const int rem = p - g * GS * RPU;
  const int unit = g0 + rem % gs;
  const int k = rem / gs;                                    // rank of the item within its unit
  const int hu = unit % HP;
  b = unit / HP;
  const DevMask& M = a.mask;
  const int hm_head = pair_rows ? hu : 2 * hu;
  const int32_t* ro = M.row_order ? M.row_order + ((size_t)(M.Bm > 1 ? b : 0) * M.Hm + (M.Hm > 1 ? hm_head : 0)) * nq
                                  : nullptr;
  auto row = [&](int i) { return ro ? __ldg(ro + i) : nq - 1 - i; };
  if (pair_rows) {
    h0 = h1 = hu;
    r0 = row(2 * k);
    r1 = 2 * k + 1 < nq ? row(2 * k + 1) : -1;
  } else {
    h0 = 2 * hu;
    h1 = 2 * hu + 1;
    r0 = r1 = row(k);
  }
}

// A whole product is issued from one asm statement: one elect.sync picks the issuing lane for all its
// K-steps (an elect and a separate statement per K-step cost the single MMA warp more issue time than the
// tensor core spends on the step). Operand offsets per K-step ks, in 16-byte descriptor units:
//  S = Q K^T (K-major, 128-byte swizzle, [128][64] sub-tiles of 16 KiB): (ks / 4) * 1024 + (ks % 4) * 2 on
//  both operands; the first step overwrites S, the others accumulate.
//  O += P V: P (bf16 pairs) at tensor-memory column 8 ks, V rows 16 ks .. 16 ks + 15 at 128 ks; the first
//  step accumulates only if `acc`.
#define FA_MMA_HEAD                                                                                       \
  "{\n\t.reg .pred P, Q, T;\n\t.reg .b64 da, db;\n\t.reg .b32 ta;\n\telect.sync _|P, 0xffffffff;\n\t" \
  "setp.ne.b32 Q, %4, 0;\n\tsetp.eq.b32 T, %4, %4;\n\t"
#define FA_QK_FIRST "@P tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, Q;\n\t"
#define FA_QK_STEP(OFF) \
  "add.s64 da, %1, " #OFF ";\n\tadd.s64 db, %2, " #OFF ";\n\t@P tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, T;\n\t"
#define FA_PV_FIRST "@P tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, Q;\n\t"
#define FA_PV_STEP(COL, OFF)                                                                               \
  "add.s32 ta, %1, " #COL ";\n\tadd.s64 db, %2, " #OFF ";\n\t@P tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, " \
  "%3, T;\n\t"

template <int NK>  // D / 16 K-steps
__device__ __forceinline__ void mma_qk_product(uint32_t d_tmem, uint64_t qdesc, uint64_t kdesc, uint32_t idesc) {
  static_assert(NK == 4 || NK == 8, "d = 64 or 128");
  if constexpr (NK == 8) {
    asm volatile(FA_MMA_HEAD FA_QK_FIRST FA_QK_STEP(2) FA_QK_STEP(4) FA_QK_STEP(6) FA_QK_STEP(1024) FA_QK_STEP(1026)
                     FA_QK_STEP(1028) FA_QK_STEP(1030) "}" ::"r"(d_tmem),
                 "l"(qdesc), "l"(kdesc), "r"(idesc), "r"(0u)
                 : "memory");
  } else {
    asm volatile(FA_MMA_HEAD FA_QK_FIRST FA_QK_STEP(2) FA_QK_STEP(4) FA_QK_STEP(6) "}" ::"r"(d_tmem), "l"(qdesc),
                 "l"(kdesc), "r"(idesc), "r"(0u)
                 : "memory");
  }
}
__device__ __forceinline__ void mma_pv_product(uint32_t d_tmem, uint32_t p_tmem, uint64_t vdesc, uint32_t idesc,
                                               uint32_t acc) {
  asm volatile(FA_MMA_HEAD FA_PV_FIRST FA_PV_STEP(8, 128) FA_PV_STEP(16, 256) FA_PV_STEP(24, 384) FA_PV_STEP(32, 512)
                   FA_PV_STEP(40, 640) FA_PV_STEP(48, 768) FA_PV_STEP(56, 896) "}" ::"r"(d_tmem),
               "r"(p_tmem), "l"(vdesc), "r"(idesc), "r"(acc)
               : "memory");
}
#undef FA_MMA_HEAD
#undef FA_QK_FIRST
#undef FA_QK_STEP
#undef FA_PV_FIRST
#undef FA_PV_STEP

template <int D, int SK>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc5_kernel(const __grid_constant__ Tc5Params P, const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmO) {
  using C = Tc5Cfg<D>;
  constexpr int NST = C::kStages;
  const FwdArgs& a = P.a;
  // All shared state is dynamic (no static __shared__), so the buffer starts at the CTA's shared
  // window and keeps the 1024-byte alignment the 128-byte swizzle needs; checked below, never assumed.
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* const bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* const bar_q = bars;          // [2] Q tile landed
  uint64_t* const bar_s = bars + 2;      // [2] S = Q K^T complete
  uint64_t* const bar_p = bars + 4;      // [2] P stored in tensor memory (each softmax warp arrives once)
  uint64_t* const bar_o = bars + 6;      // [2] O += P V complete
  uint64_t* const bar_full = bars + 8;   // [NST] ring slot landed
  uint64_t* const bar_empty = bars + 8 + NST;  // [NST] ring slot consumed
  uint64_t& bar_drain = bars[8 + 2 * NST];
  uint64_t& bar_info = bars[9 + 2 * NST];  // the union summary below is written
  uint32_t& s_tmem = *reinterpret_cast<uint32_t*>(bars + 10 + 2 * NST);
  int32_t& s_abort = *(reinterpret_cast<int32_t*>(bars + 10 + 2 * NST) + 1);
  // union summary from the MMA warp: elements, each tile's last element (-1: none), tile 1 visits tile 0's last
  volatile int32_t* const s_info = reinterpret_cast<volatile int32_t*>(bars + 11 + 2 * NST);
  // per ring slot holding a K tile: which tiles visit its element (bits 0, 1) and whether it is the union's last
  // (bit 2); written by the producer before the slot's load is armed, read by the MMA warp after it landed
  volatile int32_t* const s_uflag = reinterpret_cast<volatile int32_t*>(bars + 13 + 2 * NST);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (smem_u32(smem) & 1023u) {  // uniform across the CTA, before any barrier or allocation
    if (tid == 0) report(a.status, FA_ERR_DEVICE_CHECK);
    return;
  }

  // ---- work item: batch b and the two tiles
  const DevMask& M = a.mask;
  const bool desc = P.desc != 0;
  int b, h0, h1, r0, r1;
  work_item(a, P.pair_rows, P.group, blockIdx.x, b, h0, h1, r0, r1);
  const Tile T0 = make_tile(a, b, h0, r0);
  const Tile T1 = make_tile(a, b, h1, r1);
  // both tiles read the same K / V (one batch row, one KV head): each block of the union of their lists is
  // loaded once; the two lists are the same when they come from the same mask row

  uint8_t* sQ0 = smem;
  uint8_t* sQ1 = smem + C::kQBytes;
  uint8_t* sRing = smem + C::kOffRing;

  // ring loads issued so far (producer warp); the ring fill starts before the CTA-wide barrier below
  int issued = 0;
  Union uw;            // producer: the union walk
  int c_cur = -1;      // producer: column of the last K load
  auto load_slot = [&](bool is_v, int c, int fl) {  // into the next slot, which must be free
    const int s = issued % NST;
    if (!is_v) {
      if (lane == 0) s_uflag[s] = fl;
      __syncwarp();
    }
    int yk = c * 128, zk = b * a.Hkv + T0.hk;
    if (a.page_table) {  // key block c is one whole page; a bad page id is reported and page 0 read instead
      int pg = __ldg(a.page_table + (size_t)b * a.max_pages + c);
      if (pg < 0 || pg >= a.n_pages_total) {
        if (lane == 0) report(a.status, FA_ERR_DEVICE_CHECK);
        pg = 0;
      }
      yk = 0;
      zk = pg * a.Hkv + T0.hk;
    }
    uint8_t* dst = sRing + s * C::kSlotBytes;
    mbar_arrive_expect_tx_elect(&bar_full[s], C::kSlotBytes);
#pragma unroll
    for (int x = 0; x < D / 64; ++x)
      tma_load_3d_elect(dst + x * 16384, is_v ? &tmV : &tmK, x * 64, yk, zk, &bar_full[s]);
    ++issued;
  };
  if (warp == kLoadWarp) {
    // The producer sets up the barriers and sends the Q tiles and the first K tile at once (they need
    // nothing else), while the MMA warp allocates tensor memory.
    if (lane == 0) {
      s_abort = 0;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        mbar_init(&bar_q[t], 1);
        mbar_init(&bar_s[t], 1);
        mbar_init(&bar_p[t], 4);  // one lane of each warp of the tile's softmax warpgroup
        mbar_init(&bar_o[t], 1);
      }
      for (int s = 0; s < NST; ++s) {
        mbar_init(&bar_full[s], 1);
        mbar_init(&bar_empty[s], 1);
      }
      mbar_init(&bar_drain, 1);
      mbar_init(&bar_info, 1);
      fence_mbar_init();
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmO);
    }
    __syncwarp();
    // a Q tile is read by this CTA only: its lines may go first
    const uint64_t qpol = l2_evict_first_policy();
    if (T0.n > 0) {
      mbar_arrive_expect_tx_elect(&bar_q[0], C::kQBytes);
#pragma unroll
      for (int x = 0; x < D / 64; ++x)
        tma_load_3d_elect_hint(sQ0 + x * 16384, &tmQ, x * 64, T0.rq * 128, b * a.Hq + T0.h, &bar_q[0], qpol);
    }
    if (T1.n > 0) {
      mbar_arrive_expect_tx_elect(&bar_q[1], C::kQBytes);
#pragma unroll
      for (int x = 0; x < D / 64; ++x)
        tma_load_3d_elect_hint(sQ1 + x * 16384, &tmQ, x * 64, T1.rq * 128, b * a.Hq + T1.h, &bar_q[1], qpol);
    }
    uw.init(T0, T1, desc);
    if (!uw.done()) {  // K of the first element (the ring has more slots than this)
      bool i0, i1;
      c_cur = uw.take(T0, T1, desc, i0, i1);
      load_slot(false, c_cur, (int)i0 | ((int)i1 << 1) | (uw.done() ? 4 : 0));
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
    // Load order == the MMA warp's order of taking slots: K(u0), then V(u_k) K(u_k+1) for each element
    // u_k of the union.
    __syncwarp();
    // the Q tiles of the CTA that will take this SM after the next wave go to L2 now, so its start does
    // not wait on DRAM
    if (P.ahead > 0 && blockIdx.x + P.ahead < gridDim.x && lane == 0) {
      int bn, hn0, hn1, rn0, rn1;
      work_item(a, P.pair_rows, P.group, blockIdx.x + P.ahead, bn, hn0, hn1, rn0, rn1);
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        const Tile Tn = make_tile(a, bn, tt ? hn1 : hn0, tt ? rn1 : rn0);
        if (Tn.n == 0) continue;
#pragma unroll
        for (int x = 0; x < D / 64; ++x) tma_prefetch_l2_3d(&tmQ, x * 64, Tn.rq * 128, bn * a.Hq + Tn.h);
      }
    }
    __syncwarp();
    bool ok = true;
    auto load = [&](bool is_v, int c, int fl) -> bool {
      const int s = issued % NST;
      if (issued >= NST &&
          !__all_sync(0xFFFFFFFFu, mbar_wait(&bar_empty[s], (uint32_t)(((issued / NST) - 1) & 1), wc)))
        return false;
      load_slot(is_v, c, fl);
      return true;
    };
    while (c_cur >= 0 && ok) {
      ok = load(true, c_cur, 0);
      if (!ok || uw.done()) break;
      bool i0, i1;
      c_cur = uw.take(T0, T1, desc, i0, i1);
      ok = load(false, c_cur, (int)i0 | ((int)i1 << 1) | (uw.done() ? 4 : 0));
    }
    if (a.counters && lane == 0) {
      unsigned long long* cnt = reinterpret_cast<unsigned long long*>(a.counters);
      atomicAdd(cnt + 0, (unsigned long long)(T0.valid + T1.valid));
      atomicAdd(cnt + 1, (unsigned long long)(T0.n_full + T1.n_full));
      atomicAdd(cnt + 2, (unsigned long long)(T0.n_part + T1.n_part));
      atomicAdd(cnt + 3, (unsigned long long)issued);
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
    // Warp-uniform like the producer; each product (all its K-steps) and each commit is issued by one
    // elected lane. Descriptors: base values computed once, per-K-step offsets added to the address field.
    // Order: at union step k, for tile 0 then tile 1 (each only on its own elements), O_t += P_t(u_k-1)
    // V(u_k-1) once P_t is ready, then S_t = Q_t K(u_k)^T. The tensor pipe runs one thread's MMAs in issue
    // order, so S_t overwrites P_t only after the product has read it, and the completion of S_t implies
    // that of O_t's previous update. Waiting for P_0 before P_1 keeps the two tiles' softmaxes apart: each
    // runs while the tensor core works on the other tile. A ring slot is released (commit to its "empty"
    // barrier) after the last product that reads it. Which tiles visit an element, and whether it is the last,
    // come with its K slot (flags written by the producer): this warp does not walk the block lists, and
    // between two products it only waits on barriers (walking them here cost the tensor core 2-4 %).
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
      mma_qk_product<D / 16>(tmem + C::col_s(t), qd, kd, idesc_qk);
      tc5_commit_elect(&bar_s[t]);
    };
    auto mma_pv = [&](int t, int s, bool acc) {
      const uint64_t vd = vdesc + (uint64_t)(s * (C::kSlotBytes >> 4));
      mma_pv_product(tmem + C::col_o(t), tmem + C::col_s(t), vd, idesc_pv, acc ? 1u : 0u);
      tc5_commit_elect(&bar_o[t]);
    };
    auto wait_p = [&](int t, int j) -> bool {
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_p[t], (uint32_t)(j & 1), wc))) return false;
      tc5_fence_after();
      return true;
    };
    struct Step {
      bool live, in0, in1;
      int sk, sv;  // ring slots of the element's K and V
    };
    Step cur{false, false, false, -1, -1}, prev = cur;
    bool more = T0.n + T1.n > 0;  // an element of the union is still to come
    int np[2] = {0, 0};  // P blocks consumed so far per tile
    int uk = 0, last0 = -1, last1 = -1, both0 = 0;  // union elements taken; each tile's last; tile 1 on last0
    bool info = false;
    while (ok) {
      cur.live = more;
      if (!cur.live && !info) {  // the union is known: its summary for the epilogues' staging plans
        if (lane == 0) {
          s_info[0] = uk;
          s_info[1] = last0;
          s_info[2] = last1;
          s_info[3] = both0;
          mbar_arrive(&bar_info);
        }
        __syncwarp();
        info = true;
      }
      if (!cur.live && !prev.live) break;
      // slots of V(prev) and K(cur), taken before the waits for P, so that their barrier waits are off the
      // path from P to the next products
      if (prev.live && (prev.sv = take()) < 0) { ok = false; break; }
      if (cur.live) {
        if ((cur.sk = take()) < 0) { ok = false; break; }
        const int fl = s_uflag[cur.sk];
        cur.in0 = fl & 1;
        cur.in1 = (fl >> 1) & 1;
        more = !(fl & 4);
        if (cur.in0) {
          last0 = uk;
          both0 = cur.in1;
        }
        if (cur.in1) last1 = uk;
        ++uk;
      }
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const bool use_v = prev.live && (t ? prev.in1 : prev.in0);
        const bool use_k = cur.live && (t ? cur.in1 : cur.in0);
        if (use_v) {  // O_t += P_t(prev) V(prev)
          if (!(ok = wait_p(t, np[t]))) break;
          mma_pv(t, prev.sv, np[t] > 0);
          ++np[t];
          if (t == 1 || !prev.in1) tc5_commit_elect(&bar_empty[prev.sv]);  // its last reader
        }
        if (use_k) {  // S_t = Q_t K(cur)^T, over P_t(prev), which the product above has read
          mma_qk(t, cur.sk);
          if (t == 1 || !cur.in1) tc5_commit_elect(&bar_empty[cur.sk]);
        }
      }
      prev = cur;
    }
    // every MMA issued so far has completed before tensor memory is read back or freed
    tc5_commit_elect(&bar_drain);
    mbar_wait_drain(&bar_drain, 0, a.timeout_ns);
  } else {
    // =============================== softmax warpgroups ===============================
    // Warpgroup t (warps 4t .. 4t + 3) runs the softmax of tile t, one thread per query row (TMEM lane ==
    // query row == 32 * (warp % 4) + lane), over all 128 key columns of each block: no exchange between
    // threads, neither of the row maximum nor of the row sums. The two tiles' softmaxes run on different
    // warps and meet only in the MMA warp's order.
    const int t = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const Tile TT = t ? T1 : T0;
    uint8_t* const sQt = t ? sQ1 : sQ0;
    const int q_row = TT.rq * 128 + row;  // query position within the sequence (rule, score, validity)
    const int o_row = TT.r * 128 + row;   // output row (the same unless rows are split)
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::col_s(t);
    const uint32_t tO = tmem + lane_base + C::col_o(t);
    float* Lg = a.lse + ((size_t)b * a.Hq + TT.h) * a.out_q_len;
    const bool issuer = (warp & 3) == 0 && lane == 0;
    if (TT.valid && TT.n == 0) {
      // empty query block: O = 0, LSE = -inf, nothing loaded (an empty chunk of a split row only needs its
      // LSE: the merge gives it no weight)
      const int row_bytes = D * (a.out_f32 ? 4 : 2);
      uint8_t* Ob = reinterpret_cast<uint8_t*>(a.out) + (((size_t)b * a.Hq + TT.h) * a.out_q_len) * row_bytes;
      if (q_row < a.q_len) {
        const uint4 z = make_uint4(0, 0, 0, 0);
        if (a.split_ncm <= 1)
          for (int c16 = 0; c16 < row_bytes / 16; ++c16)
            *reinterpret_cast<uint4*>(Ob + (size_t)o_row * row_bytes + c16 * 16) = z;
        Lg[o_row] = -INFINITY;
      }
    } else if (TT.valid) {
      const int64_t off_b = a.rule.q_offset ? (int64_t)__ldg(a.rule.q_offset + (M.Bm > 1 ? b : 0)) : 0;
      const int64_t ig = (int64_t)q_row + off_b;
      const int bm = M.Bm > 1 ? b : 0;
      const float sl2 = a.scale * kLog2e;
      float slope2 = 0.f;
      if (SK == SK_ALIBI || SK == SK_GENERIC) slope2 = a.score.alibi ? __ldg(a.score.alibi + TT.h) * kLog2e : 0.f;
      // the factor the exponent's FMA applies: the scale (no score rule) or log2(e) c (soft-cap), else 1
      const float mult = SK == SK_NONE ? sl2 : SK == SK_SOFTCAP ? a.score.softcap * kLog2e : 1.f;
      // reference max (log2 domain) used for P and for O; fixed for soft-capped scores
      float m_ref = SK == SK_SOFTCAP ? mult - kCapFixedSpan : -INFINITY;
      // the row sum of P (for the LSE), and the correction that turns it into the sum O is divided by: per
      // block, the bf16 rounding error of the row's largest P (see the P loop)
      float le = 0.f, lc = 0.f;
      bool ok = true;
      Walk wk;  // this tile's blocks, in the order the MMA warp issues them
      wk.init(TT, desc);
      // tcgen05.ld / st are warp-collective (.sync.aligned): every decision that guards one is made uniform
      // across the warp (wait results with __all_sync, the O rescale with __any_sync).
      for (int j = 0; j < TT.n; ++j) {
        const bool partial = wk.next_partial();
        const int c = key_col(wk.next_key(), desc);
        wk.advance(TT, desc);
        const int64_t j0 = (int64_t)c * 128;
        // the allowed pairs of a partial block depend on positions only: evaluated while S is computed, and
        // before the row's 128 scores occupy the registers
        Bits128 bits = {{0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu}};
        if (partial) {
          const int w = (int)max((int64_t)0, min((int64_t)128, (int64_t)a.kv_len - j0));
          bits = {{0u, 0u, 0u, 0u}};
          if (q_row < a.q_len && w > 0) {
            // the row's document and (ids that never decrease) its run as a column interval, looked up per
            // partial block so that they hold no registers through the block loop
            const int doc_i = a.rule.any_doc ? doc_at(a.rule, bm, ig) : -1;
            const bool runs = a.rule.any_doc && ig >= 0 && ig < a.rule.doc_len && doc_runs_usable(a.rule, bm);
            int64_t run_lo = 0, run_hi = 0;
            if (runs) doc_run_of(a.rule, bm, ig, run_lo, run_hi);
            bits = rule_row_bits(a.rule, ig, j0, w, doc_i, [&](int dq) {
              if (runs) return range_bits(clamp_rel(run_lo - j0, w), clamp_rel(run_hi - j0, w));
              return doc_bits<4>(w, dq, [&](int cc) { return doc_at(a.rule, bm, j0 + cc); });
            });
          }
        }
        if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar_s[t], (uint32_t)(j & 1), wc));
        if (!ok) continue;
        tc5_fence_after();
        float x[128];
#pragma unroll
        for (int k = 0; k < 4; ++k) tc5_ld32(tS + 32 * k, *reinterpret_cast<uint32_t(*)[32]>(&x[32 * k]));
        tc5_wait_ld();
        // ---- score rule (log2 domain)
        if (SK == SK_ALIBI) {
          const float base = -slope2 * (float)(ig - j0);  // bias at the block's first column
          // The bias is linear in the column: four chains hold it for columns 8q + 2r and 8q + 2r + 1 (r =
          // 0..3) and step by 8 columns with one packed add (no per-column constants to materialise; each
          // step rounds once, so after q steps the bias is off by at most q half-ulps of its size, and only
          // keys near the diagonal, where the bias is small, carry weight).
          const uint64_t s2 = f2_pack(sl2, sl2), step = f2_pack(8.f * slope2, 8.f * slope2);
          uint64_t bch[4];
#pragma unroll
          for (int r = 0; r < 4; ++r)
            bch[r] = f2_pack(fmaf(slope2, (float)(2 * r), base), fmaf(slope2, (float)(2 * r + 1), base));
#pragma unroll
          for (int i = 0; i < 128; i += 2) {
            const int r = (i >> 1) & 3;
            f2_unpack(f2_fma(f2_pack(x[i], x[i + 1]), s2, bch[r]), x[i], x[i + 1]);
            bch[r] = f2_add(bch[r], step);
          }
        } else if (SK == SK_SOFTCAP) {
          // tanh(scale x / c); the factor log2(e) c is applied in the exponent's FMA (mult)
          const float ain = a.scale * a.score.inv_softcap;
          const uint64_t in2 = f2_pack(ain, ain);
#pragma unroll
          for (int i = 0; i < 128; i += 2) {
            float u0, u1;
            f2_unpack(f2_mul(f2_pack(x[i], x[i + 1]), in2), u0, u1);
            x[i] = tanh_approx(u0);
            x[i + 1] = tanh_approx(u1);
          }
        } else if (SK == SK_GENERIC) {
          for (int i = 0; i < 128; ++i) {
            float v = x[i] * a.scale;
            const int64_t dist = ig - (j0 + i);
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
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t wd = bits.w[k];
#pragma unroll
            for (int i = 0; i < 32; ++i) x[k * 32 + i] = ((wd >> i) & 1u) ? x[k * 32 + i] : -INFINITY;
          }
        }
        // ---- the row's block max: 4 independent chains of 3-input maxima (with the fixed reference of a
        // soft-cap, taken inside the P loop instead: only the correction term below needs it)
        float mxk[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (SK != SK_SOFTCAP) {
#pragma unroll
          for (int k = 0; k < 4; ++k) mxk[k] = fmaxf(x[k], x[k + 4]);
#pragma unroll
          for (int i = 8; i < 128; i += 8)
#pragma unroll
            for (int k = 0; k < 4; ++k) mxk[k] = fmax3(mxk[k], x[i + k], x[i + 4 + k]);
        }
        float xmax = fmaxf(fmaxf(mxk[0], mxk[1]), fmaxf(mxk[2], mxk[3]));
        const float mb = xmax * mult;
        // ---- reference max: move it only when the block max exceeds it by more than 2^8
        float alpha = 1.f;
        bool rescale = false;
        if (SK != SK_SOFTCAP && (mb > m_ref + kRescaleThreshold || (m_ref == -INFINITY && mb > -INFINITY))) {
          alpha = m_ref == -INFINITY ? 0.f : ex2_approx(m_ref - mb);
          rescale = j > 0 && m_ref != -INFINITY;
          m_ref = mb;
        }
        const float mr = m_ref == -INFINITY ? 0.f : m_ref;
        // ---- P = 2^(mult * x - m), stored as bf16 8 columns (16 keys) at a time over the first 64 of the
        // S columns (small store groups keep the loop under the register limit: fewer spills, about 2 %
        // faster than 16 columns at a time), and the row sum of the unrounded P. The product multiplies
        // the bf16-rounded P; O is divided by the unrounded sum plus, per block, the rounding error of the
        // row's largest P (the same FMA and ex2 on the same input give that element's P bit for bit). A row
        // dominated by one key then gets that key's V row with an exact weight, as if O were divided by the
        // sum of the rounded values; what is left is the rounding of the smaller weights, at most 2^-9 of
        // their share.
        const uint64_t mul2 = f2_pack(mult, mult), neg2 = f2_pack(-mr, -mr);
        uint64_t se[2] = {0, 0};
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float y0, y1;
            f2_unpack(f2_fma(f2_pack(x[16 * ch + 2 * i], x[16 * ch + 2 * i + 1]), mul2, neg2), y0, y1);
            const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
            if (SK == SK_SOFTCAP) mxk[i & 3] = fmax3(mxk[i & 3], x[16 * ch + 2 * i], x[16 * ch + 2 * i + 1]);
            pk[i] = pack_bf16x2(p0, p1);
            se[i & 1] = f2_add(se[i & 1], f2_pack(p0, p1));
          }
          tc5_st8(tS + 8 * ch, pk);
        }
        if (SK == SK_SOFTCAP) xmax = fmaxf(fmaxf(mxk[0], mxk[1]), fmaxf(mxk[2], mxk[3]));
        const float ph = ex2_approx(fmaf(xmax, mult, -mr));
        const float ch_err = __uint_as_float(pack_bf16x2(ph, 0.f) << 16) - ph;
        float e0, e1;
        f2_unpack(f2_add(se[0], se[1]), e0, e1);
        le = le * alpha + (e0 + e1);
        lc = lc * alpha + ch_err;
        // ---- O is stable here: S_t completed, and O_t's previous update was issued before it
        if (__any_sync(0xFFFFFFFFu, rescale)) {
          const float f = rescale ? alpha : 1.f;
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tc5_ld32(tO + c0, o);
            tc5_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
            tc5_st32(tO + c0, o);
          }
        }
        tc5_wait_st();
        tc5_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_p[t]);
      }
      // ---- epilogue: wait for the tile's last O update, normalise and store
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar_o[t], (uint32_t)((TT.n - 1) & 1), wc));
      tc5_fence_after();
      // no key of the row visible: no reference max, or (fixed reference) a zero sum, every P of a visible
      // key being at least 2^(64 - 2 c log2(e)) > 0
      const bool empty = SK == SK_SOFTCAP ? le == 0.f : m_ref == -INFINITY;
      const float inv = empty ? 0.f : 1.f / (le + lc);
      if (ok && q_row < a.q_len) Lg[o_row] = empty ? -INFINITY : (m_ref + __log2f(le)) * kLn2;
      // fp32 O ([128][D], D / 32 boxes of [128][32]: 128-byte rows, 128-byte swizzle; two ring slots) is
      // staged in K / V ring slots that no product reads any more and no load refills, in one round. Loads
      // are numbered K(u0) = 0, V(u0) = 1, K(u1) = 2, ... over the union's U elements (n = 2 U loads); load i
      // sits in slot i % NST and has not been refilled if i >= n - NST. The tile whose last product comes
      // first (earlier last element, or the same one and tile 0) finds free every such load up to the V of
      // its last element (which tile 1 may still read when tile 0 is first) and takes the two lowest; the
      // other tile's last product is the CTA's last, so it takes the two highest the first did not take.
      // Without two free slots, O goes through the tile's Q buffer (free: every product reading it has
      // completed): bf16 in one round ([128][64] boxes), fp32 in rounds of QB = D / 64 boxes.
      int stg0 = -1, stg1 = -1;  // ring slots of the fp32 O, or -1: the Q buffer
      if (a.out_f32 && ok) {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar_info, 0u, wc));
        if (ok) {
          const int n = 2 * s_info[0], lo = max(0, n - NST);
          const int l[2] = {s_info[1], s_info[2]};
          const int o = 1 - t;
          const bool first = l[o] >= 0 && (l[t] < l[o] || (l[t] == l[o] && t == 0));
          // the first tile's free range ends at its last V, or one before it when tile 1 reads that V too
          const int f = first ? t : o;
          const int hi_f = l[o] < 0 ? -1 : 2 * l[f] + 1 - (f == 0 && s_info[3] ? 1 : 0);
          const bool f_ring = l[o] >= 0 && hi_f - lo + 1 >= 2;
          if (first) {
            if (f_ring) {
              stg0 = lo;
              stg1 = lo + 1;
            }
          } else {  // the CTA's last product is this tile's: every load n - NST .. n - 1 is free
            int k = n - 1;
            if (f_ring && k <= lo + 1) k = -1;
            if (k >= lo) {
              stg0 = k;
              stg1 = k - 1;
              if (f_ring && stg1 <= lo + 1) stg0 = stg1 = -1;
            }
          }
          if (stg1 < lo) stg0 = stg1 = -1;
        }
      }
      const bool ring_stage = stg0 >= 0;
      auto box_ring = [&](int kb) -> uint8_t* {
        const int sl = ((kb * 16384) / C::kSlotBytes ? stg1 : stg0) % NST;
        return sRing + sl * C::kSlotBytes + (kb * 16384) % C::kSlotBytes;
      };
      constexpr int QB = D / 64;
      const int rounds = a.out_f32 ? (ring_stage ? 1 : (D / 32) / QB) : 1;
      for (int rd = 0; rd < rounds; ++rd) {
        if (rd > 0) {
          if (issuer) bulk_wait_group_read0();  // the previous round's boxes have left shared memory
          named_bar_sync(1 + t, 128);
        }
        if (ok) {
#pragma unroll
          for (int col = 0; col < D; col += 32) {
            const int kb = col / 32;  // fp32 box
            if (a.out_f32 && !ring_stage && kb / QB != rd) continue;
            uint32_t o[32];
            tc5_ld32(tO + col, o);
            tc5_wait_ld();
            if (!a.out_f32) {
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(o[8 * q4 + 0]) * inv, __uint_as_float(o[8 * q4 + 1]) * inv);
                v.y = pack_bf16x2(__uint_as_float(o[8 * q4 + 2]) * inv, __uint_as_float(o[8 * q4 + 3]) * inv);
                v.z = pack_bf16x2(__uint_as_float(o[8 * q4 + 4]) * inv, __uint_as_float(o[8 * q4 + 5]) * inv);
                v.w = pack_bf16x2(__uint_as_float(o[8 * q4 + 6]) * inv, __uint_as_float(o[8 * q4 + 7]) * inv);
                *reinterpret_cast<uint4*>(sQt + tile_off(row, col / 8 + q4)) = v;
              }
            } else {
              uint8_t* const stg = ring_stage ? box_ring(kb) : sQt + (kb % QB) * 16384;
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4) {
                float4 v = make_float4(__uint_as_float(o[4 * q4 + 0]) * inv, __uint_as_float(o[4 * q4 + 1]) * inv,
                                       __uint_as_float(o[4 * q4 + 2]) * inv, __uint_as_float(o[4 * q4 + 3]) * inv);
                *reinterpret_cast<float4*>(stg + row * 128 + ((q4 ^ (row & 7)) << 4)) = v;
              }
            }
          }
        }
        // every thread of the tile reaches these barriers (ok or not); the store runs only if no role gave
        // up (a failed wait always sets the CTA's abort flag)
        fence_proxy_async_smem();
        named_bar_sync(1 + t, 128);
        if (!*wc.abort && issuer) {
          // O is written once and read by no later CTA: its lines go first when L2 needs room, ahead of the
          // K / V lines neighbouring CTAs still read
          const uint64_t pol = l2_evict_first_policy();
          if (!a.out_f32) {
#pragma unroll
            for (int x = 0; x < D / 64; ++x) tma_store_3d_hint(&tmO, sQt + x * 16384, x * 64, TT.r * 128, b * a.Hq + TT.h, pol);
          } else if (ring_stage) {
#pragma unroll
            for (int kb = 0; kb < D / 32; ++kb)
              tma_store_3d_hint(&tmO, box_ring(kb), kb * 32, TT.r * 128, b * a.Hq + TT.h, pol);
          } else {
#pragma unroll
            for (int x = 0; x < QB; ++x)
              tma_store_3d_hint(&tmO, sQt + x * 16384, (rd * QB + x) * 32, TT.r * 128, b * a.Hq + TT.h, pol);
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

template <int D, int SK>
int launch_k(const FwdArgs& a, cudaStream_t st) {
  using C = Tc5Cfg<D>;
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
  // O: [B * Hq, out_q_len, D] (out_q_len = q_len unless rows are split)
  const uint64_t dout[3] = {(uint64_t)D, (uint64_t)a.out_q_len, (uint64_t)a.B * a.Hq};
  if (a.out_f32) {
    const uint64_t so[2] = {(uint64_t)D * 4, (uint64_t)a.out_q_len * D * 4};
    const uint32_t boxo[3] = {32, 128, 1};
    if (encode_tmap_f32(&to, a.out, 3, dout, so, boxo)) return FA_ERR_CUDA;
  } else {
    const uint64_t so[2] = {(uint64_t)D * 2, (uint64_t)a.out_q_len * D * 2};
    if (encode_tmap_bf16(&to, a.out, 3, dout, so, box)) return FA_ERR_CUDA;
  }
  Tc5Params p;
  std::memset(&p, 0, sizeof(p));
  p.a = a;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  p.ahead = sms;
  // sibling heads share a KV head when the group size is even; otherwise a CTA takes two query blocks of
  // one head
  const int g = a.Hq / a.Hkv;
  p.pair_rows = g % 2 != 0;
  // ALiBi is largest next to the diagonal: visiting the highest columns first fixes the running maximum
  // early, so the O accumulator is rarely rescaled
  p.desc = a.score.alibi != nullptr;
  const int n_items = p.pair_rows ? a.B * a.Hq * ((a.mask.nq + 1) / 2) : a.B * ((a.Hq + 1) / 2) * a.mask.nq;
  // Eight units side by side keep the longest-rows-first order over stretches of several waves where a
  // unit has few items; with 128 or more row pairs per head, four units already span several waves, and
  // the K / V window of fewer heads stays in L2 (sliding window over 65536 tokens: DRAM reads 844 MB
  // against 865 MB, the same time)
  p.group = p.pair_rows && (a.mask.nq + 1) / 2 >= 128 ? 4 : 8;
  auto kern = fwd_tc5_kernel<D, SK>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess)
    return FA_ERR_CUDA;
  kern<<<n_items, kThreads, C::kSmem, st>>>(p, tq, tk, tv, to);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D>
int launch_sk(const FwdArgs& a, cudaStream_t st) {
  const bool al = a.score.alibi != nullptr, rel = a.score.rel != nullptr, cap = a.score.softcap > 0.f;
  if (!al && !rel && !cap) return launch_k<D, SK_NONE>(a, st);
  if (al && !rel && !cap) return launch_k<D, SK_ALIBI>(a, st);
  if (!al && !rel && cap && a.score.softcap * kLog2e <= kCapFixedMax) return launch_k<D, SK_SOFTCAP>(a, st);
  return launch_k<D, SK_GENERIC>(a, st);
}

}  // namespace

int launch_fwd_tc5(const FwdArgs& a, cudaStream_t st) {
  if (a.mask.bq != 128 || a.mask.bk != 128) return FA_ERR_UNSUPPORTED;
  if (a.B * (int64_t)a.mask.nq * a.Hq > 0x7FFFFFFF) return FA_ERR_UNSUPPORTED;  // grid size
  if (a.d == 128) return launch_sk<128>(a, st);
  if (a.d == 64) return launch_sk<64>(a, st);
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
