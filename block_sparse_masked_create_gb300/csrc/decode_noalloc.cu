// Allocation-free variant of the paged split-KV decode.
//
// Some callers cannot hand this library a device workspace: a host program whose device memory is
// owned by another runtime's pool (where a stray cudaMalloc would bypass or fragment it), or a serving
// loop that must not call cudaMalloc / cudaFree at all because cudaFree synchronises the whole device.
// For them, fa_flex_decode_noalloc keeps the split workspace in one file-scope device array of fixed size
// instead. Each GPU that loads libfa.so holds this array until the process exits.
//
// Set-up: the first call on a device (with that device current) looks up the array's device address with
// cudaGetSymbolAddress and caches it for that device. Make that first call before any stream capture.
// The cached address belongs to the device's context of that moment: after cudaDeviceReset (or anything
// else that tears down and recreates the context) the module is loaded again and the array may move, which
// the library cannot see, so this entry point must not be used on that device after such a reset.
// The array is shared by every call: two calls that overlap on the GPU (different streams, no ordering
// between them) race on it. Its previous contents never matter: the split kernel writes every slot the
// combine kernel reads within the same call, so nothing has to be cleared.
#include <mutex>

#include "fa_launch.h"

namespace fa {
namespace {

constexpr size_t kNoAllocScratchBytes = FA_DECODE_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return FA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_flex_decode_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                            const int32_t* page_table, int32_t n_pages_total,
                                            const fa_block_mask* block_mask, const fa_score_rule* score_rule,
                                            float scale, void* out, int32_t out_dtype, float* lse, int32_t Bz,
                                            int32_t Hq, int32_t Hkv, int32_t d, int32_t page, int32_t max_pages,
                                            int32_t* dev_status, int64_t* dev_counters, fa_stream_t stream) {
  // fa_flex_decode checks every argument first and the workspace size last, so an oversized problem with
  // otherwise valid arguments returns FA_ERR_BUFFER_TOO_SMALL, and other argument errors keep the codes
  // they have there; in both cases nothing is launched.
  void* ws = nullptr;
  const int s = fa::scratch_address(&ws);
  if (s != FA_OK) return (fa_status)s;
  return fa_flex_decode(q, k_pages, v_pages, page_table, n_pages_total, block_mask, score_rule, scale, out,
                        out_dtype, lse, Bz, Hq, Hkv, d, page, max_pages, ws, fa::kNoAllocScratchBytes, dev_status,
                        dev_counters, stream);
}

extern "C" size_t fa_decode_noalloc_scratch_bytes(void) { return fa::kNoAllocScratchBytes; }
