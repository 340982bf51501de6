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
// host it is only a stand-in symbol), so the first call in each CUDA context
// looks up the real address with cudaGetSymbolAddress while that context is
// current, and caches it under the context's unique id (cuCtxGetId). A
// context made after cudaDeviceReset, or a non-primary context made current
// by another runtime, has a new id and gets its own lookup, so no cached
// address outlives the module it points into.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "sinkattn.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t{32} << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxFns& ctx_fns() {
  static CtxFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  return f;
}

// Unique id of the current CUDA context, or 0 if there is none yet.
unsigned long long current_ctx_id() {
  const CtxFns& f = ctx_fns();
  if (!f.get_current || !f.get_id) return 0;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (f.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

constexpr int kCacheSlots = 64;
std::mutex g_scratch_mu;
unsigned long long g_cache_ctx[kCacheSlots] = {};
void* g_cache_addr[kCacheSlots] = {};
int g_cache_next = 0;

// Device address of the scratch array in the current context, after checking
// that `stream` belongs to the current device (the partial and merge kernels
// run on `stream`, and the address is only valid in the context it was
// looked up in). Returns a SINKATTN_* status; nothing is launched.
int scratch_address(cudaStream_t stream, void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    sinkattn::set_error("cudaGetDevice: %s", cudaGetErrorString(e));
    return SINKATTN_CUDA_ERROR;
  }
  int sdev = dev;
  e = cudaStreamGetDevice(stream, &sdev);
  if (e != cudaSuccess) {
    sinkattn::set_error("cudaStreamGetDevice: %s", cudaGetErrorString(e));
    return SINKATTN_CUDA_ERROR;
  }
  if (sdev != dev) {
    sinkattn::set_error(
        "the stream belongs to device %d but device %d is current; make the stream's device "
        "current before calling sinkattn_decode_noalloc", sdev, dev);
    return SINKATTN_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long id = current_ctx_id();
  if (id != 0) {
    for (int i = 0; i < kCacheSlots; ++i)
      if (g_cache_ctx[i] == id) {
        *addr = g_cache_addr[i];
        return SINKATTN_OK;
      }
  }
  // Set-up for this context: look the address up with the context current.
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr) {
    sinkattn::set_error("cudaGetSymbolAddress of the scratch array: %s", cudaGetErrorString(e));
    return SINKATTN_CUDA_ERROR;
  }
  if (id == 0) id = current_ctx_id();   // the lookup may have made the primary context current
  if (id != 0) {
    g_cache_ctx[g_cache_next] = id;
    g_cache_addr[g_cache_next] = p;
    g_cache_next = (g_cache_next + 1) % kCacheSlots;
  }
  *addr = p;
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
  rc = scratch_address(static_cast<cudaStream_t>(stream), &scratch);
  if (rc) return rc;
  // Nothing in the scratch needs clearing: the split kernel writes every
  // (row, head, chunk) slot that the merge reads, empty chunks included.
  return sinkattn_decode(q, k, v, kv_indptr, batch, q_len, max_kv_len, num_qo_heads,
                         num_kv_heads, head_dim, sm_scale, causal, window, num_splits, sinks,
                         scratch, kNoAllocScratchBytes, out, lse, stream);
}
