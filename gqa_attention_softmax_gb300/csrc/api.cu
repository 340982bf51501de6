// C ABI of libsinkattn: argument validation, tensor-map encoding, launch
// selection. Every entry point checks its arguments on the host before any
// CUDA call and returns a status; nothing here allocates, frees or
// synchronises (except the diagnostic sinkattn_debug_status).
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "internal.h"
#include "sinkattn.h"

namespace sinkattn {

static thread_local char g_last_error[512] = "";
static std::atomic<int> g_decode_kernel{SINKATTN_DECODE_AUTO};
static std::atomic<int> g_prefill_kernel{SINKATTN_PREFILL_AUTO};

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
}

int sm_count() {
  // host threads may call the library concurrently: entries are atomics (a
  // racing first fill stores the same value twice)
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 0 || dev >= 64) return 148;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int make_rows_tmap(CUtensorMap* map, const void* base, uint64_t rows, int d, int box_rows,
                   int swizzle_bytes) {
  auto fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return SINKATTN_CUDA_ERROR;
  }
  if (rows == 0) rows = 1;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUtensorMapSwizzle sw =
      swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return SINKATTN_CUDA_ERROR;
  }
  return SINKATTN_OK;
}

int make_rows_tmap_u8(CUtensorMap* map, const void* base, uint64_t rows, int d, int box_rows,
                      int swizzle_bytes) {
  auto fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return SINKATTN_CUDA_ERROR;
  }
  if (rows == 0) rows = 1;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(d), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUtensorMapSwizzle sw = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                               : swizzle_bytes == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                                                      : CU_TENSOR_MAP_SWIZZLE_NONE;
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled (u8) failed (CUresult %d)", static_cast<int>(r));
    return SINKATTN_CUDA_ERROR;
  }
  return SINKATTN_OK;
}

int make_q_tmap(CUtensorMap* map, const void* q, uint64_t total_q, int Hq, int d, int G, int QB) {
  auto fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return SINKATTN_CUDA_ERROR;
  }
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hq),
                              total_q > 0 ? total_q : 1};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(Hq) * d * 2};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(QB)};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled (q) failed (CUresult %d)", static_cast<int>(r));
    return SINKATTN_CUDA_ERROR;
  }
  return SINKATTN_OK;
}

}  // namespace sinkattn

using namespace sinkattn;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  set_error("%s", buf);
  return status;
}

// Checks shared by every attention entry point.
int check_common(const void* q, const void* k, const void* v, int32_t Hq, int32_t Hkv,
                 int32_t d, float sm_scale, int32_t causal, int32_t window) {
  if (!q || !k || !v) return fail(SINKATTN_INVALID_ARG, "q, k and v must be non-null");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v))
    return fail(SINKATTN_INVALID_ARG, "q, k and v must be 16-byte aligned");
  if (Hq <= 0 || Hkv <= 0) return fail(SINKATTN_INVALID_ARG, "head counts must be positive");
  if (Hq % Hkv != 0)
    return fail(SINKATTN_UNSUPPORTED, "num_qo_heads (%d) is not a multiple of num_kv_heads (%d)",
                Hq, Hkv);
  if (d != 64 && d != 128) return fail(SINKATTN_UNSUPPORTED, "head_dim %d is not 64 or 128", d);
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale))
    return fail(SINKATTN_INVALID_ARG, "sm_scale must be positive and finite");
  if (causal != 0 && causal != 1) return fail(SINKATTN_INVALID_ARG, "causal must be 0 or 1");
  if (window > 0 && !causal)
    return fail(SINKATTN_UNSUPPORTED, "a sliding window requires causal masking");
  return SINKATTN_OK;
}

// Paged KV: page pools [num_pages, Hkv, page_size, d] and per-sequence page lists.
struct PagedKv {
  const int32_t* page_indptr;
  const int32_t* page_indices;
  int32_t num_pages;
  int32_t page_size;
};

int check_paged(const PagedKv& pg, int32_t Hkv) {
  if (!pg.page_indptr || !pg.page_indices)
    return fail(SINKATTN_INVALID_ARG, "page_indptr and page_indices must be non-null");
  if (pg.page_size < 16 || pg.page_size > 256 || (pg.page_size & (pg.page_size - 1)))
    return fail(SINKATTN_UNSUPPORTED, "page_size %d is not a power of two in [16, 256]",
                pg.page_size);
  if (pg.num_pages < 1) return fail(SINKATTN_INVALID_ARG, "num_pages must be positive");
  if (static_cast<int64_t>(pg.num_pages) * Hkv * pg.page_size >= (int64_t{1} << 31))
    return fail(SINKATTN_UNSUPPORTED, "page pools exceed 2^31 rows");
  return SINKATTN_OK;
}

void set_paged(AttnArgs* a, const PagedKv* pg) {
  a->page_size = pg ? pg->page_size : 0;
  a->num_pages = pg ? pg->num_pages : 0;
  a->page_indptr = pg ? pg->page_indptr : nullptr;
  a->page_indices = pg ? pg->page_indices : nullptr;
}

}  // namespace

extern "C" {

const char* sinkattn_status_string(int status) {
  switch (status) {
    case SINKATTN_OK: return "SINKATTN_OK";
    case SINKATTN_INVALID_ARG: return "SINKATTN_INVALID_ARG";
    case SINKATTN_UNSUPPORTED: return "SINKATTN_UNSUPPORTED";
    case SINKATTN_CUDA_ERROR: return "SINKATTN_CUDA_ERROR";
    case SINKATTN_TIMEOUT: return "SINKATTN_TIMEOUT";
    case SINKATTN_BAD_LENGTHS: return "SINKATTN_BAD_LENGTHS";
    default: return "SINKATTN_UNKNOWN_STATUS";
  }
}

const char* sinkattn_last_error(void) { return g_last_error; }

}  // extern "C"

namespace {

int prefill_impl(const void* q, const void* k, const void* v, const float* sinks,
                 const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const PagedKv* pg,
                 int32_t batch, int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k,
                 int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim, float sm_scale,
                 int32_t causal, int32_t window, void* out, float* lse, void* stream) {
  g_last_error[0] = '\0';
  int rc = check_common(q, k, v, num_qo_heads, num_kv_heads, head_dim, sm_scale, causal, window);
  if (rc) return rc;
  if (pg && (rc = check_paged(*pg, num_kv_heads))) return rc;
  if (!out || !aligned16(out)) return fail(SINKATTN_INVALID_ARG, "out must be non-null and 16-byte aligned");
  if (!cu_seqlens_q || !cu_seqlens_k) return fail(SINKATTN_INVALID_ARG, "cu_seqlens must be non-null");
  if (batch < 0 || total_q < 0 || max_seqlen_q < 0 || max_seqlen_k < 0)
    return fail(SINKATTN_INVALID_ARG, "sizes must be non-negative");
  if (batch > 65535) return fail(SINKATTN_UNSUPPORTED, "batch %d exceeds 65535", batch);
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(SINKATTN_INVALID_ARG, "lse must be 4-byte aligned");
  if (max_seqlen_q > max_seqlen_k)
    return fail(SINKATTN_INVALID_ARG, "max_seqlen_q (%d) exceeds max_seqlen_k (%d)", max_seqlen_q,
                max_seqlen_k);
  if (static_cast<int64_t>(num_kv_heads) * batch * max_seqlen_k >= (int64_t{1} << 31) ||
      static_cast<int64_t>(total_q) * num_qo_heads >= (int64_t{1} << 31))
    return fail(SINKATTN_UNSUPPORTED, "problem exceeds 2^31 rows");
  if (batch == 0 || total_q == 0 || max_seqlen_q == 0) return SINKATTN_OK;

  AttnArgs a{};
  a.q = q; a.k = k; a.v = v;
  a.cu_q = cu_seqlens_q; a.cu_k = cu_seqlens_k;
  a.batch = batch; a.q_len = 0; a.max_q = max_seqlen_q; a.max_kv = max_seqlen_k;
  a.total_q = total_q;
  a.Hq = num_qo_heads; a.Hkv = num_kv_heads; a.d = head_dim;
  a.sm_scale = sm_scale; a.causal = causal; a.window = window; a.num_splits = 1;
  a.sinks = sinks; a.out = out; a.lse = lse;
  set_paged(&a, pg);
  if (num_qo_heads / num_kv_heads > 128)
    return fail(SINKATTN_UNSUPPORTED, "GQA group of %d heads exceeds 128", num_qo_heads / num_kv_heads);
  return launch_prefill_tc(a, g_prefill_kernel.load(std::memory_order_relaxed),
                           static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int sinkattn_prefill(const void* q, const void* k, const void* v, const float* sinks,
                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
                     int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k,
                     int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                     float sm_scale, int32_t causal, int32_t window, void* out, float* lse,
                     void* stream) {
  return prefill_impl(q, k, v, sinks, cu_seqlens_q, cu_seqlens_k, nullptr, batch, total_q,
                      max_seqlen_q, max_seqlen_k, num_qo_heads, num_kv_heads, head_dim, sm_scale,
                      causal, window, out, lse, stream);
}

int sinkattn_prefill_paged(const void* q, const void* k_pages, const void* v_pages,
                           const float* sinks, const int32_t* cu_seqlens_q,
                           const int32_t* cu_seqlens_k, const int32_t* page_indptr,
                           const int32_t* page_indices, int32_t num_pages, int32_t page_size,
                           int32_t batch, int32_t total_q, int32_t max_seqlen_q,
                           int32_t max_seqlen_k, int32_t num_qo_heads, int32_t num_kv_heads,
                           int32_t head_dim, float sm_scale, int32_t causal, int32_t window,
                           void* out, float* lse, void* stream) {
  const PagedKv pg{page_indptr, page_indices, num_pages, page_size};
  return prefill_impl(q, k_pages, v_pages, sinks, cu_seqlens_q, cu_seqlens_k, &pg, batch,
                      total_q, max_seqlen_q, max_seqlen_k, num_qo_heads, num_kv_heads, head_dim,
                      sm_scale, causal, window, out, lse, stream);
}

}  // extern "C"

namespace {

// Validation shared by the split-KV decode entry points; fills `a` (without
// the output pointers). Returns SINKATTN_OK or the failing status.
int decode_args(const void* q, const void* k, const void* v, const int32_t* kv_indptr,
                int32_t batch, int32_t q_len, int32_t max_kv_len, int32_t num_qo_heads,
                int32_t num_kv_heads, int32_t head_dim, float sm_scale, int32_t causal,
                int32_t window, int32_t num_splits, AttnArgs* a) {
  int rc = check_common(q, k, v, num_qo_heads, num_kv_heads, head_dim, sm_scale, causal, window);
  if (rc) return rc;
  if (!kv_indptr) return fail(SINKATTN_INVALID_ARG, "kv_indptr must be non-null");
  if (batch < 0 || max_kv_len < 0) return fail(SINKATTN_INVALID_ARG, "sizes must be non-negative");
  if (batch > 65535) return fail(SINKATTN_UNSUPPORTED, "batch %d exceeds 65535", batch);
  if (q_len < 1) return fail(SINKATTN_INVALID_ARG, "q_len must be at least 1");
  if (num_splits < 1) return fail(SINKATTN_INVALID_ARG, "num_splits must be at least 1");
  if (num_splits > 4096) return fail(SINKATTN_UNSUPPORTED, "num_splits %d exceeds 4096", num_splits);
  if (q_len > max_kv_len)
    return fail(SINKATTN_INVALID_ARG, "q_len (%d) exceeds max_kv_len (%d)", q_len, max_kv_len);
  if (num_qo_heads / num_kv_heads > 64)
    return fail(SINKATTN_UNSUPPORTED, "GQA group of %d heads exceeds 64", num_qo_heads / num_kv_heads);
  if (static_cast<int64_t>(num_kv_heads) * batch * max_kv_len >= (int64_t{1} << 31) ||
      static_cast<int64_t>(batch) * q_len * num_qo_heads * num_splits * head_dim >=
          (int64_t{1} << 40))
    return fail(SINKATTN_UNSUPPORTED, "problem too large");
  *a = AttnArgs{};
  a->q = q; a->k = k; a->v = v;
  a->cu_q = nullptr; a->cu_k = kv_indptr;
  a->batch = batch; a->q_len = q_len; a->max_q = q_len; a->max_kv = max_kv_len;
  a->Hq = num_qo_heads; a->Hkv = num_kv_heads; a->d = head_dim;
  a->sm_scale = sm_scale; a->causal = causal; a->window = window; a->num_splits = num_splits;
  return SINKATTN_OK;
}

// Partials with the selected kernel (a.part_acc / a.part_md set).
// FP8 KV: e4m3 K/V codes and their per-KV-head scales.
struct Fp8Kv {
  const float* k_scale;
  const float* v_scale;
};

int launch_partials(const AttnArgs& a, cudaStream_t stream) {
  const int kind = g_decode_kernel.load(std::memory_order_relaxed);
  if (a.kv_fp8) {   // tcgen05 up to 64 rows per tile at head_dim 128, else the warp-level kernel
    const bool tc8 = decode_tc_supported(a);
    if (kind == SINKATTN_DECODE_TCGEN05 && !tc8)
      return fail(SINKATTN_UNSUPPORTED,
                  "the tcgen05 FP8 decode needs head_dim 128 and at most 64 heads per group");
    if (kind == SINKATTN_DECODE_TCGEN05 || (kind == SINKATTN_DECODE_AUTO && tc8))
      return launch_decode_tc(a, stream);
    return launch_attn_mma(a, stream);
  }
  const bool tc_ok = decode_tc_supported(a);
  if (kind == SINKATTN_DECODE_TCGEN05 && !tc_ok)
    return fail(SINKATTN_UNSUPPORTED,
                "the tcgen05 decode kernel needs head_dim 128");
  if (kind == SINKATTN_DECODE_TCGEN05 || (kind == SINKATTN_DECODE_AUTO && tc_ok))
    return launch_decode_tc(a, stream);
  return launch_attn_mma(a, stream);
}

int decode_split_impl(const void* q, const void* k, const void* v, const int32_t* kv_indptr,
                      const PagedKv* pg, int32_t batch, int32_t q_len, int32_t max_kv_len,
                      int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                      float sm_scale, int32_t causal, int32_t window, int32_t num_splits,
                      float* part_acc, float* part_md, void* stream,
                      const Fp8Kv* f8 = nullptr) {
  g_last_error[0] = '\0';
  AttnArgs a;
  int rc = decode_args(q, k, v, kv_indptr, batch, q_len, max_kv_len, num_qo_heads, num_kv_heads,
                       head_dim, sm_scale, causal, window, num_splits, &a);
  if (rc) return rc;
  if (pg && (rc = check_paged(*pg, num_kv_heads))) return rc;
  if (!part_acc || !part_md || !aligned16(part_acc) || !aligned16(part_md))
    return fail(SINKATTN_INVALID_ARG, "partial buffers must be non-null and 16-byte aligned");
  if (f8) {
    if (!f8->k_scale || !f8->v_scale ||
        (reinterpret_cast<uintptr_t>(f8->k_scale) | reinterpret_cast<uintptr_t>(f8->v_scale)) & 3u)
      return fail(SINKATTN_INVALID_ARG, "k_scale and v_scale must be non-null and 4-byte aligned");
    a.kv_fp8 = 1;
    a.k_scale = f8->k_scale;
    a.v_scale = f8->v_scale;
  }
  if (batch == 0) return SINKATTN_OK;
  a.part_acc = part_acc; a.part_md = part_md;
  set_paged(&a, pg);
  return launch_partials(a, static_cast<cudaStream_t>(stream));
}

int decode_impl(const void* q, const void* k, const void* v, const int32_t* kv_indptr,
                const PagedKv* pg, int32_t batch, int32_t q_len, int32_t max_kv_len,
                int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim, float sm_scale,
                int32_t causal, int32_t window, int32_t num_splits, const float* sinks,
                void* workspace, size_t workspace_bytes, void* out, float* lse, void* stream,
                const Fp8Kv* f8 = nullptr) {
  g_last_error[0] = '\0';
  int rc;
  if (num_splits <= 0) {
    rc = sinkattn_decode_default_splits(batch, q_len, num_qo_heads, num_kv_heads, head_dim,
                                        max_kv_len, &num_splits);
    if (rc) return rc;
  }
  size_t need = 0;
  rc = sinkattn_decode_workspace_bytes(batch, q_len, num_qo_heads, head_dim, num_splits, &need);
  if (rc) return rc;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(SINKATTN_INVALID_ARG, "workspace must be non-null and 256-byte aligned");
  if (workspace_bytes < need)
    return fail(SINKATTN_INVALID_ARG, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  if (!out || !aligned16(out)) return fail(SINKATTN_INVALID_ARG, "out must be non-null and 16-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(SINKATTN_INVALID_ARG, "lse must be 4-byte aligned");
  // More query rows per KV head than one 128-row tile holds (G x q_len > 128,
  // e.g. 16 MTP drafts of 16 heads): the split kernels would read every KV
  // tile once per 128-row block; the single-pass prefill kernel (decode
  // drafts are its queries, bottom-right causal) reads each once and needs
  // no partials. Only under the default kernel choice, bf16 KV.
  if (!f8 && batch > 0 && static_cast<int64_t>(num_qo_heads / num_kv_heads) * q_len > 128 &&
      g_decode_kernel.load(std::memory_order_relaxed) == SINKATTN_DECODE_AUTO &&
      (head_dim == 64 || head_dim == 128)) {
    AttnArgs a;
    rc = decode_args(q, k, v, kv_indptr, batch, q_len, max_kv_len, num_qo_heads, num_kv_heads,
                     head_dim, sm_scale, causal, window, num_splits, &a);
    if (rc) return rc;
    if (pg && (rc = check_paged(*pg, num_kv_heads))) return rc;
    if (static_cast<int64_t>(batch) * q_len >= (int64_t{1} << 31))
      return fail(SINKATTN_UNSUPPORTED, "too many query rows");
    set_paged(&a, pg);
    a.total_q = batch * q_len;
    a.sinks = sinks;
    a.out = out;
    a.lse = lse;
    return launch_prefill_tc(a, g_prefill_kernel.load(std::memory_order_relaxed),
                             static_cast<cudaStream_t>(stream));
  }
  const size_t slots = static_cast<size_t>(batch) * q_len * num_qo_heads * num_splits;
  float* part_acc = static_cast<float*>(workspace);
  float* part_md = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                            ((slots * head_dim * 4 + 255) & ~static_cast<size_t>(255)));
  rc = decode_split_impl(q, k, v, kv_indptr, pg, batch, q_len, max_kv_len, num_qo_heads,
                         num_kv_heads, head_dim, sm_scale, causal, window, num_splits, part_acc,
                         part_md, stream, f8);
  if (rc) return rc;
  if (batch == 0) return SINKATTN_OK;
  // the partials are this call's scratch: the merge may drop them from L2
  return launch_merge(part_acc, part_md, sinks, batch * q_len, num_qo_heads, head_dim,
                      num_splits, out, lse, static_cast<cudaStream_t>(stream), true);
}

}  // namespace

extern "C" {

int sinkattn_decode_split(const void* q, const void* k, const void* v,
                          const int32_t* kv_indptr, int32_t batch, int32_t q_len,
                          int32_t max_kv_len, int32_t num_qo_heads, int32_t num_kv_heads,
                          int32_t head_dim, float sm_scale, int32_t causal, int32_t window,
                          int32_t num_splits, float* part_acc, float* part_md, void* stream) {
  return decode_split_impl(q, k, v, kv_indptr, nullptr, batch, q_len, max_kv_len, num_qo_heads,
                           num_kv_heads, head_dim, sm_scale, causal, window, num_splits, part_acc,
                           part_md, stream);
}

int sinkattn_decode_split_paged(const void* q, const void* k_pages, const void* v_pages,
                                const int32_t* kv_indptr, const int32_t* page_indptr,
                                const int32_t* page_indices, int32_t num_pages, int32_t page_size,
                                int32_t batch, int32_t q_len, int32_t max_kv_len,
                                int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                                float sm_scale, int32_t causal, int32_t window, int32_t num_splits,
                                float* part_acc, float* part_md, void* stream) {
  const PagedKv pg{page_indptr, page_indices, num_pages, page_size};
  return decode_split_impl(q, k_pages, v_pages, kv_indptr, &pg, batch, q_len, max_kv_len,
                           num_qo_heads, num_kv_heads, head_dim, sm_scale, causal, window,
                           num_splits, part_acc, part_md, stream);
}

int sinkattn_decode_split_fp8(const void* q, const void* k, const void* v,
                              const float* k_scale, const float* v_scale,
                              const int32_t* kv_indptr, int32_t batch, int32_t q_len,
                              int32_t max_kv_len, int32_t num_qo_heads, int32_t num_kv_heads,
                              int32_t head_dim, float sm_scale, int32_t causal, int32_t window,
                              int32_t num_splits, float* part_acc, float* part_md, void* stream) {
  const Fp8Kv f8{k_scale, v_scale};
  return decode_split_impl(q, k, v, kv_indptr, nullptr, batch, q_len, max_kv_len, num_qo_heads,
                           num_kv_heads, head_dim, sm_scale, causal, window, num_splits, part_acc,
                           part_md, stream, &f8);
}

int sinkattn_decode_fp8(const void* q, const void* k, const void* v, const float* k_scale,
                        const float* v_scale, const int32_t* kv_indptr, int32_t batch,
                        int32_t q_len, int32_t max_kv_len, int32_t num_qo_heads,
                        int32_t num_kv_heads, int32_t head_dim, float sm_scale, int32_t causal,
                        int32_t window, int32_t num_splits, const float* sinks, void* workspace,
                        size_t workspace_bytes, void* out, float* lse, void* stream) {
  const Fp8Kv f8{k_scale, v_scale};
  return decode_impl(q, k, v, kv_indptr, nullptr, batch, q_len, max_kv_len, num_qo_heads,
                     num_kv_heads, head_dim, sm_scale, causal, window, num_splits, sinks,
                     workspace, workspace_bytes, out, lse, stream, &f8);
}

int sinkattn_set_prefill_kernel(int kind) {
  g_last_error[0] = '\0';
  if (kind != SINKATTN_PREFILL_AUTO && kind != SINKATTN_PREFILL_ONE_BLOCK &&
      kind != SINKATTN_PREFILL_PERSISTENT)
    return fail(SINKATTN_INVALID_ARG, "unknown prefill kernel %d", kind);
  g_prefill_kernel.store(kind, std::memory_order_relaxed);
  return SINKATTN_OK;
}

int sinkattn_set_decode_kernel(int kind) {
  g_last_error[0] = '\0';
  if (kind != SINKATTN_DECODE_AUTO && kind != SINKATTN_DECODE_WARP &&
      kind != SINKATTN_DECODE_TCGEN05)
    return fail(SINKATTN_INVALID_ARG, "unknown decode kernel %d", kind);
  g_decode_kernel.store(kind, std::memory_order_relaxed);
  return SINKATTN_OK;
}

int sinkattn_merge(const float* part_acc, const float* part_md, const float* sinks, int32_t rows,
                   int32_t num_qo_heads, int32_t head_dim, int32_t num_splits, void* out,
                   float* lse, void* stream) {
  g_last_error[0] = '\0';
  if (!part_acc || !part_md || !out)
    return fail(SINKATTN_INVALID_ARG, "part_acc, part_md and out must be non-null");
  if (!aligned16(part_acc) || !aligned16(part_md) || !aligned16(out))
    return fail(SINKATTN_INVALID_ARG, "part_acc, part_md and out must be 16-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(SINKATTN_INVALID_ARG, "lse must be 4-byte aligned");
  if (rows < 0 || num_qo_heads <= 0) return fail(SINKATTN_INVALID_ARG, "bad sizes");
  if (head_dim != 64 && head_dim != 128)
    return fail(SINKATTN_UNSUPPORTED, "head_dim %d is not 64 or 128", head_dim);
  if (num_splits < 1) return fail(SINKATTN_INVALID_ARG, "num_splits must be at least 1");
  return launch_merge(part_acc, part_md, sinks, rows, num_qo_heads, head_dim, num_splits, out,
                      lse, static_cast<cudaStream_t>(stream), false);
}

int sinkattn_decode_workspace_bytes(int32_t batch, int32_t q_len, int32_t num_qo_heads,
                                    int32_t head_dim, int32_t num_splits, size_t* bytes) {
  g_last_error[0] = '\0';
  if (!bytes) return fail(SINKATTN_INVALID_ARG, "bytes must be non-null");
  if (batch < 0 || q_len < 1 || num_qo_heads <= 0 || num_splits < 1)
    return fail(SINKATTN_INVALID_ARG, "bad sizes");
  if (head_dim != 64 && head_dim != 128)
    return fail(SINKATTN_UNSUPPORTED, "head_dim %d is not 64 or 128", head_dim);
  const size_t slots = static_cast<size_t>(batch) * q_len * num_qo_heads * num_splits;
  const size_t acc = (slots * head_dim * 4 + 255) & ~static_cast<size_t>(255);
  *bytes = acc + slots * 2 * 4;
  return SINKATTN_OK;
}

int sinkattn_decode_default_splits(int32_t batch, int32_t q_len, int32_t num_qo_heads,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t max_kv_len,
                                   int32_t* num_splits) {
  g_last_error[0] = '\0';
  if (!num_splits) return fail(SINKATTN_INVALID_ARG, "num_splits must be non-null");
  if (batch < 0 || q_len < 1 || num_qo_heads <= 0 || num_kv_heads <= 0 || max_kv_len < 0)
    return fail(SINKATTN_INVALID_ARG, "bad sizes");
  if (head_dim != 64 && head_dim != 128)
    return fail(SINKATTN_UNSUPPORTED, "head_dim %d is not 64 or 128", head_dim);
  // Aim for ~4 work items per SM slot so variable lengths even out, but keep
  // each chunk at least 4 KV tiles long (shorter chunks mostly cost partials).
  const int64_t items = static_cast<int64_t>(batch) * num_kv_heads;
  const int64_t target = 8 * static_cast<int64_t>(sm_count());
  int64_t s = items > 0 ? (target + items - 1) / items : 1;
  const int kt = head_dim == 64 ? 64 : 32;
  const int64_t cap = max_kv_len / (4 * kt);
  if (s > cap) s = cap;
  if (s < 1) s = 1;
  if (s > 16) s = 16;
  *num_splits = static_cast<int32_t>(s);
  return SINKATTN_OK;
}

int sinkattn_decode(const void* q, const void* k, const void* v, const int32_t* kv_indptr,
                    int32_t batch, int32_t q_len, int32_t max_kv_len, int32_t num_qo_heads,
                    int32_t num_kv_heads, int32_t head_dim, float sm_scale, int32_t causal,
                    int32_t window, int32_t num_splits, const float* sinks, void* workspace,
                    size_t workspace_bytes, void* out, float* lse, void* stream) {
  return decode_impl(q, k, v, kv_indptr, nullptr, batch, q_len, max_kv_len, num_qo_heads,
                     num_kv_heads, head_dim, sm_scale, causal, window, num_splits, sinks,
                     workspace, workspace_bytes, out, lse, stream);
}

int sinkattn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                          const int32_t* kv_indptr, const int32_t* page_indptr,
                          const int32_t* page_indices, int32_t num_pages, int32_t page_size,
                          int32_t batch, int32_t q_len, int32_t max_kv_len, int32_t num_qo_heads,
                          int32_t num_kv_heads, int32_t head_dim, float sm_scale, int32_t causal,
                          int32_t window, int32_t num_splits, const float* sinks, void* workspace,
                          size_t workspace_bytes, void* out, float* lse, void* stream) {
  const PagedKv pg{page_indptr, page_indices, num_pages, page_size};
  return decode_impl(q, k_pages, v_pages, kv_indptr, &pg, batch, q_len, max_kv_len, num_qo_heads,
                     num_kv_heads, head_dim, sm_scale, causal, window, num_splits, sinks,
                     workspace, workspace_bytes, out, lse, stream);
}

int sinkattn_decode_fused(const void* q, const void* k, const void* v, const int32_t* kv_indptr,
                          int32_t batch, int32_t q_len, int32_t max_kv_len, int32_t num_qo_heads,
                          int32_t num_kv_heads, int32_t head_dim, float sm_scale, int32_t causal,
                          int32_t window, int32_t num_splits, const float* sinks, void* out,
                          float* lse, void* stream) {
  g_last_error[0] = '\0';
  int rc = check_common(q, k, v, num_qo_heads, num_kv_heads, head_dim, sm_scale, causal, window);
  if (rc) return rc;
  if (!kv_indptr) return fail(SINKATTN_INVALID_ARG, "kv_indptr must be non-null");
  if (!out || !aligned16(out)) return fail(SINKATTN_INVALID_ARG, "out must be non-null and 16-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(SINKATTN_INVALID_ARG, "lse must be 4-byte aligned");
  if (batch < 0 || max_kv_len < 0) return fail(SINKATTN_INVALID_ARG, "sizes must be non-negative");
  if (batch > 65535) return fail(SINKATTN_UNSUPPORTED, "batch %d exceeds 65535", batch);
  if (q_len < 1) return fail(SINKATTN_INVALID_ARG, "q_len must be at least 1");
  if (q_len > max_kv_len)
    return fail(SINKATTN_INVALID_ARG, "q_len (%d) exceeds max_kv_len (%d)", q_len, max_kv_len);
  if (num_qo_heads / num_kv_heads > 64)
    return fail(SINKATTN_UNSUPPORTED, "GQA group of %d heads exceeds 64", num_qo_heads / num_kv_heads);
  if (static_cast<int64_t>(num_kv_heads) * batch * max_kv_len >= (int64_t{1} << 31))
    return fail(SINKATTN_UNSUPPORTED, "problem too large");
  if (num_splits <= 0) {
    rc = sinkattn_decode_default_splits(batch, q_len, num_qo_heads, num_kv_heads, head_dim,
                                        max_kv_len, &num_splits);
    if (rc) return rc;
  }
  if (num_splits > 16)
    return fail(SINKATTN_UNSUPPORTED, "num_splits %d exceeds the 16 CTAs of a cluster", num_splits);
  if (batch == 0) return SINKATTN_OK;
  AttnArgs a{};
  a.q = q; a.k = k; a.v = v;
  a.cu_q = nullptr; a.cu_k = kv_indptr;
  a.batch = batch; a.q_len = q_len; a.max_q = q_len; a.max_kv = max_kv_len;
  a.Hq = num_qo_heads; a.Hkv = num_kv_heads; a.d = head_dim;
  a.sm_scale = sm_scale; a.causal = causal; a.window = window; a.num_splits = num_splits;
  a.sinks = sinks; a.out = out; a.lse = lse;
  return launch_attn_mma_fused(a, static_cast<cudaStream_t>(stream));
}

int sinkattn_debug_status(void* stream, int* status) {
  g_last_error[0] = '\0';
  if (!status) return fail(SINKATTN_INVALID_ARG, "status must be non-null");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  int a = 0, m = 0, t = 0, dt = 0;
  if (read_status_attn_mma(s, &a) || read_status_merge(s, &m) || read_status_prefill_tc(s, &t) ||
      read_status_decode_tc(s, &dt))
    return fail(SINKATTN_CUDA_ERROR, "reading the device status failed: %s",
                cudaGetErrorString(cudaGetLastError()));
  *status = a ? a : (dt ? dt : (t ? t : m));
  return SINKATTN_OK;
}

int sinkattn_debug_set_hooks(long long wait_limit_cycles, int skip_tile) {
  g_last_error[0] = '\0';
  if (skip_tile < -1) return fail(SINKATTN_INVALID_ARG, "skip_tile must be -1 or a tile index");
  if (set_hooks_attn_mma(wait_limit_cycles, skip_tile) ||
      set_hooks_prefill_tc(wait_limit_cycles, skip_tile) ||
      set_hooks_decode_tc(wait_limit_cycles, skip_tile))
    return fail(SINKATTN_CUDA_ERROR, "setting the test hooks failed: %s",
                cudaGetErrorString(cudaGetLastError()));
  return SINKATTN_OK;
}

}  // extern "C"
