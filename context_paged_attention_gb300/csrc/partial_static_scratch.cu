// cp_paged_attn_partial_noalloc: the partner-partial attention call for callers
// that cannot allocate device memory.
//
// Who needs this: code that runs where cudaMalloc is off limits or unavailable
// -- a host that hands a plugin raw pointers for its inputs and outputs but no
// allocator, a runtime whose memory pool owns every byte of the GPU, or a step
// that must not allocate once it has started.  cp_paged_attn_partial asks such
// a caller for a workspace it cannot provide.  This entry point instead uses a
// scratch buffer that lives inside this library as a file-scope __device__
// array, sized once at build time; the caller still passes every input and
// output.
//
// Costs and limits:
// * Every GPU that loads the library holds kScratchBytes (16 MiB) for this
//   array until the process exits, whether or not this entry point is called.
// * Problems whose split-KV scratch (cp_paged_attn_workspace_bytes) exceeds
//   kScratchBytes are refused with CPATTN_ERR_WORKSPACE_TOO_SMALL, nothing
//   launched.
// * All calls share the one array.  The array keeps whatever the previous call
//   left; the only part that must start at zero, the split tickets, is
//   cleared on the caller's stream whenever the call splits a stripe (the only
//   time the tickets are read).  Two calls whose kernels can overlap on the
//   GPU (different streams, or different host threads) race on the array:
//   order them on one stream.
// * The first call on each device looks up the array's device address
//   (cudaGetSymbolAddress, with that device current) and remembers it; make
//   that first call before any stream capture begins.  The address belongs to
//   the device's primary context: after cudaDeviceReset it is stale, so this
//   entry point is not to be called again in that process.
#include <cuda_runtime.h>

#include <mutex>

#include "cpattn.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// symbol, never a device address: the address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_partial_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CPATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_partial_scratch) != cudaSuccess || p == nullptr) return CPATTN_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return CPATTN_OK;
}

}  // namespace

extern "C" {

size_t cp_paged_attn_noalloc_scratch_bytes(void) { return kScratchBytes; }

int cp_paged_attn_partial_noalloc(const cpattn_pool_desc* desc, const void* pool_k, const void* pool_v,
                                  const void* q, int32_t num_q_heads, int32_t num_rows, int32_t num_tokens,
                                  const int32_t* qo_indptr, const int32_t* kv_len, int32_t max_kv_len,
                                  const int32_t* kv_page_indptr, const int32_t* kv_page_indices, float scale,
                                  float* o_part, float* lse_part, int32_t* dev_status, cudaStream_t stream) {
  // the same sizing rule as the workspace of cp_paged_attn_partial; 0 means bad arguments
  const size_t need = cp_paged_attn_workspace_bytes(desc, num_q_heads, num_tokens, max_kv_len);
  if (need > kScratchBytes) return CPATTN_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != CPATTN_OK) return st;
  // the regular entry point validates the rest, clears the tickets on `stream`
  // and launches; the library's own scratch stands in for the caller's workspace
  return cp_paged_attn_partial(desc, pool_k, pool_v, q, num_q_heads, num_rows, num_tokens, qo_indptr, kv_len,
                               max_kv_len, kv_page_indptr, kv_page_indices, scale, o_part, lse_part, scratch,
                               kScratchBytes, dev_status, stream);
}

}  // extern "C"
