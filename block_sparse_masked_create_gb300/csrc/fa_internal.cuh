// Internal device-side helpers of libfa.so (sm_103a): rule evaluation on 128-column bit vectors,
// bounded mbarrier waits, TMA, tcgen05 and mma.sync wrappers written as inline PTX.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fa.h"

namespace fa {

constexpr uint8_t FA_BLOCK_EMPTY = 0, FA_BLOCK_PARTIAL = 1, FA_BLOCK_FULL = 2;

// ------------------------------------------------------------------------------------------------
// Rule in the form the kernels evaluate: an OR of up to FA_MAX_RULE_TERMS conjunctions. A conjunction
// of the atoms {true, causal, window W, prefix P, doc} is one interval of KV positions
//     lo(i) = (win ? i - W + 1 : -inf)  <=  j  <  hi(i) = min(causal ? i + 1 : +inf, prefix P)
// intersected with {j : doc(j) == doc(i)} when `doc` is set. The host rewrites the postfix program into
// this form (fa_api.cu); the mask builder and both attention kernels evaluate it the same way.
// ------------------------------------------------------------------------------------------------
struct DevTerm {
  int32_t causal;   // j <= i
  int32_t doc;      // doc(j) == doc(i)
  int64_t win;      // i - j < win   (INT64_MAX: none)
  int64_t pre;      // j < pre       (INT64_MAX: none)
};

struct DevRule {
  int32_t n_terms;
  int32_t any_doc;
  DevTerm t[FA_MAX_RULE_TERMS];
  const int32_t* doc_ids;
  int32_t doc_batch;
  int32_t doc_len;
  const int32_t* q_offset;
  // run bounds of the document ids, filled by the block-mask builder: doc_run [doc_batch][2][doc_len]
  // holds, per position, the first and one-past-last position of the run of equal ids around it;
  // doc_sorted [doc_batch] is 1 where the ids never decrease (then every id is one run, and document
  // equality with position p is exactly the column interval of p's run). NULL: not available.
  const int32_t* doc_run;
  const int32_t* doc_sorted;
};

struct Bits128 {
  uint32_t w[4];
};

__device__ __forceinline__ uint32_t bits_below(int n) {  // n in [0, 32]
  return n >= 32 ? 0xFFFFFFFFu : ((1u << n) - 1u);
}

// bits c in [lo, hi) of a 128-bit vector (lo, hi already clamped to [0, 128])
__device__ __forceinline__ Bits128 range_bits(int lo, int hi) {
  Bits128 r;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    int a = min(max(lo - 32 * k, 0), 32);
    int b = min(max(hi - 32 * k, 0), 32);
    r.w[k] = b > a ? (bits_below(b) & ~bits_below(a)) : 0u;
  }
  return r;
}

__device__ __forceinline__ int clamp_rel(int64_t x, int w) {
  return (int)(x < 0 ? 0 : (x > w ? (int64_t)w : x));
}

__device__ __forceinline__ int doc_at(const DevRule& R, int b, int64_t pos) {
  const int32_t* row = R.doc_ids + (int64_t)(R.doc_batch > 1 ? b : 0) * R.doc_len;
  return (pos >= 0 && pos < R.doc_len) ? __ldg(row + pos) : -1;
}

// Whether the rule allows the pair (query position ig, key position j), one pair at a time; doc_i /
// doc_j are the two positions' document ids (read only by document terms). Same terms as rule_row_bits.
__device__ __forceinline__ bool rule_allows(const DevRule& R, int64_t ig, int64_t j, int doc_i, int doc_j) {
  for (int t = 0; t < R.n_terms; ++t) {
    const DevTerm T = R.t[t];
    if (T.causal && j > ig) continue;
    if (T.win != INT64_MAX && ig - j >= T.win) continue;
    if (T.pre != INT64_MAX && j >= T.pre) continue;
    if (T.doc && doc_i != doc_j) continue;
    return true;
  }
  return false;
}

// Whether document equality of batch row b can be read from run bounds (ids non-decreasing).
__device__ __forceinline__ bool doc_runs_usable(const DevRule& R, int b) {
  return R.doc_run != nullptr && __ldg(R.doc_sorted + (R.doc_batch > 1 ? b : 0)) != 0;
}

// Positions [lo, hi) holding the same document id as position pos, for pos inside the id array (a
// position outside has id -1, which the caller compares id by id instead) and doc_runs_usable.
__device__ __forceinline__ void doc_run_of(const DevRule& R, int b, int64_t pos, int64_t& lo, int64_t& hi) {
  const int32_t* run = R.doc_run + (int64_t)(R.doc_batch > 1 ? b : 0) * 2 * R.doc_len;
  lo = __ldg(run + pos);
  hi = __ldg(run + R.doc_len + pos);
}

// Bits c < w (of NW 32-bit words) whose column document id coldoc(c) equals d. Fully unrolled with
// constant word indices, so the words stay in registers.
template <int NW, class ColDocFn>
__device__ __forceinline__ Bits128 doc_bits(int w, int d, ColDocFn coldoc) {
  Bits128 db = {{0u, 0u, 0u, 0u}};
#pragma unroll
  for (int k = 0; k < NW; ++k) {
    uint32_t wd = 0u;
#pragma unroll
    for (int b = 0; b < 32; ++b) {
      const int c = 32 * k + b;
      if (c < w && coldoc(c) == d) wd |= 1u << b;
    }
    db.w[k] = wd;
  }
  return db;
}

// Allowed bits of one query row (global position ig) over KV columns [j0, j0 + w), w <= 128.
// `docbits(d)` returns the bits of columns whose document id equals d (only called if R.any_doc).
template <class DocBitsFn>
__device__ __forceinline__ Bits128 rule_row_bits(const DevRule& R, int64_t ig, int64_t j0, int w,
                                                 int doc_i, DocBitsFn docbits) {
  Bits128 acc = {{0u, 0u, 0u, 0u}};
  Bits128 db = {{0u, 0u, 0u, 0u}};
  if (R.any_doc) db = docbits(doc_i);
  for (int t = 0; t < R.n_terms; ++t) {
    const DevTerm T = R.t[t];
    int64_t lo = j0, hi = j0 + w;
    if (T.win != INT64_MAX) lo = max(lo, ig - T.win + 1);
    if (T.causal) hi = min(hi, ig + 1);
    if (T.pre != INT64_MAX) hi = min(hi, T.pre);
    Bits128 b = range_bits(clamp_rel(lo - j0, w), clamp_rel(hi - j0, w));
    if (T.doc) {
#pragma unroll
      for (int k = 0; k < 4; ++k) b.w[k] &= db.w[k];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) acc.w[k] |= b.w[k];
  }
  return acc;
}

// ------------------------------------------------------------------------------------------------
// Status reporting and bounded waits
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared by all roles of a CTA: a wait that runs out sets *abort so every other wait returns quickly.
struct WaitCtl {
  uint64_t limit_ns;
  int32_t* status;
  volatile int32_t* abort;  // shared memory flag
};

// Wait for phase `parity` of `bar` to complete. Returns false (after setting FA_ERR_TIMEOUT and the
// CTA's abort flag) if it did not complete within limit_ns, or if another role already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtl& w) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if ((it & 15u) == 0) {
      if (*w.abort) return false;
      if (globaltimer() - t0 > w.limit_ns) {
        report(w.status, FA_ERR_TIMEOUT);
        *w.abort = 1;
        return false;
      }
    }
  }
}

// A wait used only while shutting down after an abort: same bound, no abort check.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  uint64_t t0 = globaltimer();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if ((it & 15u) == 15u && globaltimer() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------------------------------------
// TMA (tensor maps encoded on the host with cuTensorMapEncodeTiled)
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* m, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// Bring a tile of a 3-D tensor into L2 ahead of its load (no shared memory, nothing to wait for).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* m, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(reinterpret_cast<uint64_t>(m)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* m, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* smem_src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}

// L2 eviction priority for a bulk copy's lines (all of them: fraction 1.0)
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_store_3d_hint(const CUtensorMap* m, const void* smem_src, int x, int y, int z,
                                                  uint64_t policy) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%2, %3, %4}], [%1], %5;" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z), "l"(policy)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// ------------------------------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
// ------------------------------------------------------------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2), descriptor version 1.
//   K-major operand:  rows of 64 bf16 (128 B), 8-row groups SBO bytes apart; LBO unused.
//   MN-major operand: 64-element MN chunks LBO bytes apart, 8-row K groups SBO bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulation.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc5_mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::
          "r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// A operand in tensor memory (M rows in lanes, K packed two bf16 per 32-bit column), B from shared memory.
__device__ __forceinline__ void tc5_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::
          "r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// ---- elected issue: the whole warp executes the surrounding code (so operands stay warp-uniform) and
// exactly one lane, chosen by elect.sync, issues the instruction. Issuing from a lane-0 branch instead
// measured about half the MMA rate on this part.
__device__ __forceinline__ void tc5_mma_ss_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred P, Q;\n\telect.sync _|P, 0xffffffff;\n\tsetp.ne.b32 Q, %4, 0;\n\t"
      "@P tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, Q;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc5_mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred P, Q;\n\telect.sync _|P, 0xffffffff;\n\tsetp.ne.b32 Q, %4, 0;\n\t"
      "@P tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, Q;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc5_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\t"
      "@P tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_elect_hint(void* smem_dst, const CUtensorMap* m, int x, int y, int z,
                                                       uint64_t* bar, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\t"
      "@P cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
      "{%2, %3, %4}], [%5], %6;\n\t}" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred P;\n\t.reg .b64 st;\n\telect.sync _|P, 0xffffffff;\n\t"
      "@P mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred P;\n\t.reg .b64 st;\n\telect.sync _|P, 0xffffffff;\n\t"
      "@P mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_elect(void* smem_dst, const CUtensorMap* m, int x, int y, int z,
                                                  uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\t"
      "@P cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4}], [%5];\n\t}" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// Arrive (once) on an mbarrier when all previously issued tcgen05 async ops of this thread complete.
__device__ __forceinline__ void tc5_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc5_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc5_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc5_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc5_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 columns of 32-bit: thread t of the warp gets lane (taddr.lane + t), columns [c, c+32).
__device__ __forceinline__ void tc5_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tc5_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 32 lanes x 16 columns of 32-bit: thread t gets lane (taddr.lane + t), columns [c, c+16).
__device__ __forceinline__ void tc5_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tc5_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tc5_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// ------------------------------------------------------------------------------------------------
// Legacy warp-level tensor-core path (mma.sync m16n8k16, bf16 -> fp32), used by the mma.sync forward
// and by the HBM-bound decode kernel where FLOPs are negligible.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ---- packed fp32x2 arithmetic (one instruction for two lanes of fp32 work) and a 3-input max
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// sum of the two bf16 halves of a packed pair, in fp32 (exact widening)
__device__ __forceinline__ float bf16x2_sum(uint32_t v) {
  return __uint_as_float(v << 16) + __uint_as_float(v & 0xFFFF0000u);
}

__device__ __forceinline__ void cp_async_16(uint32_t saddr, const void* gptr, bool pred) {
  int sz = pred ? 16 : 0;  // zero-fill when pred is false
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr), "l"(gptr), "r"(sz) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------------------------------------
// Score rule on the device (fixed order: + ALiBi, + relative bias, soft-cap)
// ------------------------------------------------------------------------------------------------
struct DevScore {
  const float* alibi;   // [Hq] or null
  const float* rel;     // [Hq, 2*kv_len-1] or null
  float softcap;        // > 0: on
  float inv_softcap;
  int32_t kv_len;
};

// 2^x on the special-function unit (flushes subnormal results to zero)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// tanh on the special-function unit (one instruction; measured on this part: absolute error below 8e-6
// over [-8, 8], relative error below 1e-5; checked by fa_debug_softcap's test)
__device__ __forceinline__ float tanh_approx(float x) {
  float r;
  asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// soft-cap c * tanh(x / c)
__device__ __forceinline__ float softcap_apply(float x, float c, float inv_c) { return c * tanh_approx(x * inv_c); }

}  // namespace fa
