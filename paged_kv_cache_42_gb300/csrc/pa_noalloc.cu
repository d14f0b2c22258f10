// pa_attention_noalloc: pa_attention for callers that cannot allocate device
// memory.
//
// pa_attention needs a device workspace for its planner output and split-KV
// partial results, and expects the caller to provide it. Some callers have no
// way to get one: code running where cudaMalloc is forbidden or unavailable
// (inside a custom allocator's own callbacks, a plugin host that owns all
// device memory and exposes no allocation hook, or a latency-critical path
// that must never enter the driver's allocator). This entry point serves
// them with a fixed scratch area that lives in the library image itself: a
// file-scope device array, created when the library's module is loaded onto
// a GPU and held by every GPU that loads the library until the process exits.
//
// Nothing here allocates: no cudaMalloc / cudaFree, no library allocator.
// The array's device address is looked up once per device (with that device
// current) and then handed to the unchanged pa_attention as its workspace.
// With lazy module loading, that first lookup is also when the driver places
// the array in device memory, so the first call on a device belongs outside
// any context that must not allocate. The cached address is valid for the
// life of the CUDA context (cudaDeviceReset is not supported).
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pa_api.h"
#include "pa_internal.h"

namespace {

constexpr size_t kScratchBytes = PA_NOALLOC_SCRATCH_BYTES;  // 64 MiB

// The scratch area. Host code must not use this name as an address: on the
// host it denotes a stand-in object, not device memory; the device address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Per-device set-up: the scratch array's device address on the current device.
pa_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) return PA_ERR_CUDA;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" {

size_t pa_noalloc_scratch_bytes(void) { return kScratchBytes; }

pa_status pa_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* seq_lens,
                               const int32_t* query_start_loc, float scale, void* out,
                               int num_reqs, int num_tokens, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks,
                               int max_blocks_per_req, int max_query_len, int max_seq_len,
                               void* stream) {
  // argument errors first, as pa_attention reports them, whatever the batch size
  bool nothing = false;
  if (pa_status st = pa::check_attention_args(
          q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale, out, num_reqs,
          num_tokens, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
          max_blocks_per_req, max_query_len, max_seq_len, 0, 0, 1.f, 1.f, &nothing))
    return st;
  if (nothing) return PA_OK;
  const size_t need =
      pa_attention_workspace_size(num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim);
  if (need == 0) return PA_ERR_INVALID_ARG;
  if (need > kScratchBytes) return PA_ERR_WORKSPACE;  // batch too large for the fixed scratch
  void* scratch = nullptr;
  if (pa_status st = scratch_for_current_device(&scratch)) return st;
  return pa_attention(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale, out,
                      num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim, block_size,
                      num_blocks, max_blocks_per_req, max_query_len, max_seq_len, scratch,
                      kScratchBytes, stream);
}

}  // extern "C"
