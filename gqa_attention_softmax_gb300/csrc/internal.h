// Host-side interface between the C ABI (api.cu) and the kernel translation
// units. Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sinkattn {

// Everything the attention kernels need besides the K/V tensor maps.
struct AttnArgs {
  const void* q;            // bf16 [total_q, Hq, d]
  const void* k;            // bf16 ragged HND
  const void* v;            // bf16 ragged HND
  const int32_t* cu_q;      // [B+1] (prefill) or nullptr (decode: uniform q_len)
  const int32_t* cu_k;      // [B+1]
  int32_t batch, q_len, max_q, max_kv;
  int32_t total_q;          // rows of q (prefill)
  int32_t Hq, Hkv, d;
  float sm_scale;
  int32_t causal, window;
  int32_t num_splits;       // 1 for the single-pass (final) mode
  // final mode
  const float* sinks;
  void* out;
  float* lse;
  // split mode
  float* part_acc;
  float* part_md;
  // paged KV (page_size > 0): k and v are page pools [num_pages, Hkv, page_size, d];
  // sequence b's keys [e * page_size, (e + 1) * page_size) live in page
  // page_indices[page_indptr[b] + e]; cu_k still gives the key counts
  int32_t page_size;
  int32_t num_pages;
  const int32_t* page_indptr;   // [B+1]
  const int32_t* page_indices;  // [page_indptr[B]]
  // FP8 KV (kv_fp8 != 0): k and v hold e4m3 codes (one byte per element, same
  // layout); KV head g's keys are code * k_scale[g], values code * v_scale[g]
  int32_t kv_fp8;
  const float* k_scale;         // [Hkv], device
  const float* v_scale;         // [Hkv], device
};

// Rows of the 2-D tensor map over K or V, and the box height: contiguous HND
// rows, or page-pool rows (page, head, slot) with boxes of min(page, tile) rows.
inline uint64_t kv_map_rows(const AttnArgs& a) {
  return a.page_size > 0 ? static_cast<uint64_t>(a.num_pages) * a.Hkv * a.page_size
                         : static_cast<uint64_t>(a.Hkv) * a.batch * a.max_kv;
}
// Paged KV: boxes of min(page_size, the largest power of two dividing the
// tile) rows, so a box starting on a multiple of its height never crosses a
// page; contiguous KV: one box per tile.
inline int kv_box_rows(const AttnArgs& a, int tile_keys) {
  if (a.page_size <= 0) return tile_keys;
  const int pow2 = tile_keys & -tile_keys;
  return a.page_size < pow2 ? a.page_size : pow2;
}

// Encodes a 2-D tensor map over a [rows, d] bf16 buffer with [box_rows, 64]
// boxes and 128-byte swizzling. Returns 0 or a SINKATTN_* status.
int make_rows_tmap(CUtensorMap* map, const void* base, uint64_t rows, int d, int box_rows,
                   int swizzle_bytes);
// The same over a [rows, d] array of bytes (e4m3 codes), [box_rows, d] boxes,
// swizzled in 16-byte chunks over swizzle_bytes (64 or 128; 0: none; the
// row must be that wide).
int make_rows_tmap_u8(CUtensorMap* map, const void* base, uint64_t rows, int d, int box_rows,
                      int swizzle_bytes = 0);

// Encodes a 3-D tensor map over q [total_q, Hq, d] bf16 whose box is
// [QB tokens][G heads][64 columns] (128 rows of one GQA group), 128-byte swizzled.
int make_q_tmap(CUtensorMap* map, const void* q, uint64_t total_q, int Hq, int d, int G, int QB);

// Split-KV decode (per-chunk partial outputs) on the warp-level tensor-core
// path. Returns a SINKATTN_* status.
int launch_attn_mma(const AttnArgs& a, cudaStream_t stream);

// Split-KV decode with the merge done on chip: the num_splits (<= 16) chunks
// of one (sequence, KV head) form a thread-block cluster that folds its
// partials through distributed shared memory. Writes out / lse directly.
int launch_attn_mma_fused(const AttnArgs& a, cudaStream_t stream);


// Split-KV decode on the tcgen05/TMEM path (head_dim 128; 16, 32, 48 or 64
// query rows per KV head and query block). Same partial layout as
// launch_attn_mma.
bool decode_tc_supported(const AttnArgs& a);
int launch_decode_tc(const AttnArgs& a, cudaStream_t stream);

// Single-pass prefill on the tcgen05/TMEM path. Returns a SINKATTN_* status.
int launch_prefill_tc(const AttnArgs& a, int kind, cudaStream_t stream);

// drop_partials: the partials are the library's scratch (sinkattn_decode's
// workspace): after folding a row, drop its accumulator lines from L2 without
// write-back. Never for caller-visible partials.
int launch_merge(const float* part_acc, const float* part_md, const float* sinks, int32_t rows,
                 int32_t Hq, int32_t d, int32_t num_splits, void* out, float* lse,
                 cudaStream_t stream, bool drop_partials);

// Reads and clears the device status word of one translation unit.
int read_status_attn_mma(cudaStream_t s, int* status);
int read_status_merge(cudaStream_t s, int* status);
int read_status_prefill_tc(cudaStream_t s, int* status);
int read_status_decode_tc(cudaStream_t s, int* status);

// Failure-detection test hooks of one translation unit (wait limit in clock
// cycles, <= 0: the default; KV tile the first thread block's producer leaves
// out, -1: none). Host, synchronous.
int set_hooks_attn_mma(long long limit, int skip);
int set_hooks_prefill_tc(long long limit, int skip);
int set_hooks_decode_tc(long long limit, int skip);

// Thread-local error text used by the C ABI.
void set_error(const char* fmt, ...);

// Number of SMs on the current device (queried once).
int sm_count();

}  // namespace sinkattn
