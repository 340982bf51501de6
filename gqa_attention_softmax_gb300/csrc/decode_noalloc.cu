// Split-KV decode for callers that cannot allocate device memory.
//
// sinkattn_decode needs a caller-provided workspace for the per-chunk
// partials. Some callers cannot provide one: code that runs inside another
// runtime whose memory manager owns all device memory and exposes no
// allocator to plugins, or serving loops where a cudaMalloc (which may
// synchronise the whole device) is not acceptable. For them,
// sinkattn_decode_noalloc keeps the partials in a fixed array that lives in
// this library's own device memory.
//
// The array is a file-scope __device__ buffer of kNoAllocScratchBytes
// (32 MiB). Every GPU that loads the library holds it until the process
// exits. Host code cannot use the array's name as a device address (on the
// host it is only a stand-in symbol), so the first call on each device looks
// up the real address with cudaGetSymbolAddress while that device is current,
// and caches it.
#include <mutex>

#include "internal.h"
#include "sinkattn.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t{32} << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {};

// Device address of the scratch array on the current device (set up once
// per device, under a lock). Returns a SINKATTN_* status.
int scratch_address(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    sinkattn::set_error("cudaGetDevice: %s", cudaGetErrorString(e));
    return SINKATTN_CUDA_ERROR;
  }
  if (dev < 0 || dev >= 64) {
    sinkattn::set_error("device ordinal %d out of range", dev);
    return SINKATTN_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      sinkattn::set_error("cudaGetSymbolAddress of the scratch array: %s", cudaGetErrorString(e));
      return SINKATTN_CUDA_ERROR;
    }
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return SINKATTN_OK;
}

}  // namespace

extern "C" SINKATTN_API int sinkattn_decode_noalloc(
    const void* q, const void* k, const void* v, const int32_t* kv_indptr, int32_t batch,
    int32_t q_len, int32_t max_kv_len, int32_t num_qo_heads, int32_t num_kv_heads,
    int32_t head_dim, float sm_scale, int32_t causal, int32_t window, int32_t num_splits,
    const float* sinks, void* out, float* lse, void* stream) {
  int rc;
  if (num_splits <= 0) {
    rc = sinkattn_decode_default_splits(batch, q_len, num_qo_heads, num_kv_heads, head_dim,
                                        max_kv_len, &num_splits);
    if (rc) return rc;
  }
  size_t need = 0;
  rc = sinkattn_decode_workspace_bytes(batch, q_len, num_qo_heads, head_dim, num_splits, &need);
  if (rc) return rc;
  if (need > kNoAllocScratchBytes) {
    sinkattn::set_error(
        "this decode needs %zu bytes of partials; the built-in scratch holds %zu bytes "
        "(use sinkattn_decode with a caller workspace, or fewer splits)",
        need, kNoAllocScratchBytes);
    return SINKATTN_UNSUPPORTED;
  }
  void* scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc) return rc;
  // Nothing in the scratch needs clearing: the split kernel writes every
  // (row, head, chunk) slot that the merge reads, empty chunks included.
  return sinkattn_decode(q, k, v, kv_indptr, batch, q_len, max_kv_len, num_qo_heads,
                         num_kv_heads, head_dim, sm_scale, causal, window, num_splits, sinks,
                         scratch, kNoAllocScratchBytes, out, lse, stream);
}
