// Self-tests of the building blocks the kernels rely on, callable through the C ABI:
//  - fa_debug_wait_timeout: the bounded mbarrier wait returns and reports FA_ERR_TIMEOUT when nothing
//    ever arrives (no fault, no hang);
//  - fa_debug_tc5_gemm: one 128x128xK tcgen05 MMA chain from 128-byte-swizzled shared memory into tensor
//    memory, with B either K-major (the S = Q K^T operand) or MN-major (the O += P V operand), the tiles
//    written either by TMA or by plain stores with the same swizzle. Compared against a library GEMM by
//    the tests, it pins the descriptor encodings the attention kernel uses.
#include <cstring>

#include "fa_launch.h"

namespace fa {
namespace {

__global__ void debug_wait_kernel(int32_t* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int32_t s_abort;
  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  WaitCtl w{timeout_ns, status, &s_abort};
  if (threadIdx.x == 0) mbar_wait(&bar, 0, w);  // nothing arrives: must give up after timeout_ns
  __syncthreads();
}

// K in {64, 128}; 128 threads
__global__ void __launch_bounds__(128) debug_tc5_gemm_kernel(const __nv_bfloat16* A, const __nv_bfloat16* B,
                                                             float* C, int K, int b_mn, int use_tma,
                                                             const __grid_constant__ CUtensorMap tmA,
                                                             const __grid_constant__ CUtensorMap tmB,
                                                             int32_t* status, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                  // K/64 sub-tiles [128][64]
  uint8_t* sB = smem + 128 * K * 2;    // K-major: K/64 sub-tiles [128][64]; MN-major: 2 sub-tiles [K][64]
  __shared__ uint64_t bar_load, bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ int32_t s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    s_abort = 0;
    mbar_init(&bar_load, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 256);  // D at columns [0, 128), A (mode 2) at [128, 128 + K/2)
    tmem_relinquish();
  }
  tc5_fence_before();
  __syncthreads();
  tc5_fence_after();
  WaitCtl wc{timeout_ns, status, &s_abort};
  const uint32_t tmem = tmem_base;
  bool ok = true;
  if (use_tma == 2) {
    // A into tensor memory: thread = row, K packed two bf16 per 32-bit column
    const int row = warp * 32 + lane;
    for (int c0 = 0; c0 < K / 2; c0 += 32) {
      uint32_t r[32];
      for (int j = 0; j < 32; ++j)
        r[j] = *reinterpret_cast<const uint32_t*>(A + (size_t)row * K + 2 * (c0 + j));
      tc5_st32(tmem + ((uint32_t)(warp * 32) << 16) + 128u + (uint32_t)c0, r);
    }
    tc5_wait_st();
  }
  if (use_tma == 1) {
    if (tid == 0) {
      const uint32_t bytes = 2u * 128u * (uint32_t)K * 2u;
      mbar_arrive_expect_tx(&bar_load, bytes);
      for (int kt = 0; kt < K / 64; ++kt) tma_load_2d(sA + kt * 16384, &tmA, kt * 64, 0, &bar_load);
      if (!b_mn) {
        for (int kt = 0; kt < K / 64; ++kt) tma_load_2d(sB + kt * 16384, &tmB, kt * 64, 0, &bar_load);
      } else {
        for (int nt = 0; nt < 2; ++nt) tma_load_2d(sB + nt * (K * 128), &tmB, nt * 64, 0, &bar_load);
      }
    }
    ok = mbar_wait(&bar_load, 0, wc);
  } else {
    for (int x = tid; use_tma == 0 && x < 128 * K / 8; x += 128) {  // A: 16-byte chunks
      const int row = x / (K / 8), ch = x % (K / 8);
      const uint4 val = *reinterpret_cast<const uint4*>(A + (size_t)row * K + ch * 8);
      *reinterpret_cast<uint4*>(sA + (ch >> 3) * 16384 + row * 128 + (((ch & 7) ^ (row & 7)) << 4)) = val;
    }
    if (!b_mn) {
      for (int x = tid; x < 128 * K / 8; x += 128) {
        const int row = x / (K / 8), ch = x % (K / 8);
        const uint4 val = *reinterpret_cast<const uint4*>(B + (size_t)row * K + ch * 8);
        *reinterpret_cast<uint4*>(sB + (ch >> 3) * 16384 + row * 128 + (((ch & 7) ^ (row & 7)) << 4)) = val;
      }
    } else {
      for (int x = tid; x < K * 16; x += 128) {  // B[K][128]: row k, chunk of n
        const int k = x / 16, ch = x % 16;
        const uint4 val = *reinterpret_cast<const uint4*>(B + (size_t)k * 128 + ch * 8);
        *reinterpret_cast<uint4*>(sB + (ch >> 3) * (K * 128) + k * 128 + (((ch & 7) ^ (k & 7)) << 4)) = val;
      }
    }
    fence_proxy_async_smem();
  }
  tc5_fence_before();  // orders the tensor-memory stores of mode 2 before the MMA issue
  __syncthreads();
  tc5_fence_after();
  if (ok && tid == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, 128, false, b_mn != 0);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
    for (int ks = 0; ks < K / 16; ++ks) {
      const uint64_t ad = sdesc_sw128(a0 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
      const uint64_t bd = b_mn ? sdesc_sw128(b0 + ks * 16 * 128, K * 128, 1024)
                               : sdesc_sw128(b0 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
      if (use_tma == 2)
        tc5_mma_ts(tmem, tmem + 128u + (uint32_t)(ks * 8), bd, idesc, ks > 0 ? 1u : 0u);
      else
        tc5_mma_ss(tmem, ad, bd, idesc, ks > 0 ? 1u : 0u);
    }
    tc5_commit(&bar_mma);
  }
  __syncwarp();
  if (ok) ok = mbar_wait(&bar_mma, 0, wc);
  tc5_fence_after();
  ok = __all_sync(0xFFFFFFFFu, ok);  // tcgen05.ld below is warp-collective
  if (ok) {
    for (int c0 = 0; c0 < 128; c0 += 32) {
      uint32_t r[32];
      tc5_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, r);
      tc5_wait_ld();
      const int row = warp * 32 + lane;
      for (int j = 0; j < 32; ++j) C[(size_t)row * 128 + c0 + j] = __uint_as_float(r[j]);
    }
  }
  if (!ok && tid == 0) {  // nothing may still be writing shared or tensor memory when the CTA leaves
    if (use_tma == 1) mbar_wait_drain(&bar_load, 0, timeout_ns);
    mbar_wait_drain(&bar_mma, 0, timeout_ns);
  }
  tc5_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

__global__ void debug_softcap_kernel(const float* x, float* y, int n, float c) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) y[i] = softcap_apply(x[i], c, 1.0f / c);
}

}  // namespace

cudaError_t launch_debug_wait(int32_t* status, uint64_t timeout_ns, cudaStream_t st) {
  debug_wait_kernel<<<1, 32, 0, st>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace fa

extern "C" fa_status fa_debug_softcap(const float* x, float* y, int32_t n, float c, fa_stream_t stream) {
  if (!x || !y || n < 1 || !(c > 0.f)) return FA_ERR_INVALID_ARG;
  fa::debug_softcap_kernel<<<(n + 255) / 256, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(x, y, n, c);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

extern "C" fa_status fa_debug_tc5_gemm(const void* A, const void* B, float* C, int32_t K, int32_t b_mn_major,
                                       int32_t use_tma, int32_t* dev_status, fa_stream_t stream) {
  using namespace fa;
  if (!A || !B || !C || (K != 64 && K != 128)) return FA_ERR_INVALID_ARG;
  CUtensorMap ta, tb;
  std::memset(&ta, 0, sizeof(ta));
  std::memset(&tb, 0, sizeof(tb));
  if (use_tma) {
    const uint64_t da[2] = {(uint64_t)K, 128}, sa[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {64, 128};
    if (encode_tmap_bf16(&ta, A, 2, da, sa, box) != 0) return FA_ERR_CUDA;
    if (!b_mn_major) {
      if (encode_tmap_bf16(&tb, B, 2, da, sa, box) != 0) return FA_ERR_CUDA;
    } else {
      const uint64_t db[2] = {128, (uint64_t)K}, sb[1] = {256};
      const uint32_t boxb[2] = {64, (uint32_t)K};
      if (encode_tmap_bf16(&tb, B, 2, db, sb, boxb) != 0) return FA_ERR_CUDA;
    }
  }
  const int smem = 2 * 128 * K * 2 + 1024;
  auto kern = debug_tc5_gemm_kernel;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return FA_ERR_CUDA;
  kern<<<1, 128, smem, reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const __nv_bfloat16*>(A), reinterpret_cast<const __nv_bfloat16*>(B), C, K, b_mn_major, use_tma,
      ta, tb, dev_status, fa_get_wait_timeout_ns());
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
