// Device helpers shared by the sinkattn kernels (sm_103a): shared-memory
// barriers, TMA tile loads, ldmatrix / mma.sync fragments, status reporting.
#pragma once

#include <cuda.h>
#include <math.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sinkattn.h"

namespace sinkattn {

// Every spin-wait in the library gives up after this many SM clock cycles
// (about 1 s at the GB300's 2.07 GHz maximum), records SINKATTN_TIMEOUT in
// the kernel's status word and unwinds.
constexpr long long kWaitLimitCycles = 2000000000LL;

// Failure-detection test hooks (sinkattn_debug_set_hooks), one copy per
// translation unit: the limit every bounded wait uses, and the KV tile whose
// copies the producer of the grid's first thread block leaves out (-1: none),
// so that the waits for that tile run out and take the timeout path.
static __device__ long long g_wait_limit_cycles = kWaitLimitCycles;
static __device__ int g_skip_tile = -1;

// Sets this translation unit's hooks (host; synchronous). limit <= 0 restores
// the default.
#define SINKATTN_DEFINE_SET_HOOKS(fn)                                                        \
  int fn(long long limit, int skip) {                                                        \
    if (limit <= 0) limit = kWaitLimitCycles;                                                \
    if (cudaMemcpyToSymbol(g_wait_limit_cycles, &limit, sizeof limit) != cudaSuccess ||      \
        cudaMemcpyToSymbol(g_skip_tile, &skip, sizeof skip) != cudaSuccess)                  \
      return SINKATTN_CUDA_ERROR;                                                            \
    return SINKATTN_OK;                                                                      \
  }

// The tile the calling thread block's producer leaves out (test hook).
__device__ __forceinline__ int hook_skip_tile() {
  return (blockIdx.x | blockIdx.y | blockIdx.z) == 0 ? g_skip_tile : -1;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -INFINITY;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete. Returns false
// if the CTA-wide abort flag is (or becomes) set, or after the wait limit
// (kWaitLimitCycles unless a test hook changed it); in the latter case it sets
// the abort flag and records a timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  const long long limit = g_wait_limit_cycles;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      atomicExch(status, SINKATTN_TIMEOUT);
      return false;
    }
  }
}

// Bounded wait that ignores the abort flag: used only to drain copies that
// are still in flight before a CTA exits.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  const long long limit = g_wait_limit_cycles;
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return;
  }
}

// ---------------------------------------------------------------------------
// TMA (tiled tensor copies, global -> shared, completion on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y,
                                                 uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Byte offset of element (row, col) inside a [rows][64] bf16 tile written by
// TMA with 128-byte swizzling: the 16-byte chunk index (col / 8) is XORed
// with (row % 8). The tile base must be 1024-byte aligned.
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// ---------------------------------------------------------------------------
// Warp-level tensor-core fragments (mma.sync m16n8k16, bf16 in, fp32 accumulate)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// A 16 x 16 matrix of bytes, transposed: lanes 0-15 address rows 0-15 (16
// bytes each); lane (g, c) = (lane / 4, lane % 4) receives rows 4c .. 4c + 3
// of column g in r0 and of column g + 8 in r1, row 4c in the lowest byte.
__device__ __forceinline__ void ldsm_b8_trans(uint32_t& r0, uint32_t& r1, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m16n16.x1.trans.shared.b8 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same with f16 operands (the FP8 KV path widens e4m3 to f16, which holds
// every e4m3 value exactly).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Two e4m3 codes (low byte first) -> two f16 (low half first), exact: one
// conversion instruction straight into the packed register.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(codes));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Sum of the two f16 halves of a packed pair, in fp32 (exact widening).
__device__ __forceinline__ float f16x2_sum(uint32_t v) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
  return f.x + f.y;
}

// Sum of the two bf16 halves of a packed pair, in fp32 (exact widening).
__device__ __forceinline__ float bf16x2_sum(uint32_t v) {
  return __uint_as_float(v << 16) + __uint_as_float(v & 0xffff0000u);
}

// Split-KV chunk length for Lk keys in S chunks: ceil(Lk / S) rounded up to
// whole 64-key tiles, so every chunk but the last starts and ends on a tile
// boundary and no tile is loaded by two chunks.
__host__ __device__ __forceinline__ int split_chunk(int Lk, int S) {
  return ((Lk + S - 1) / S + 63) / 64 * 64;
}

// ---------------------------------------------------------------------------
// Paged KV: a producer warp's view of one sequence's page list.
// Entry e of the list (global memory) is the page holding keys
// [e * page_size, (e + 1) * page_size). Lane l caches entry base + l and the
// entry 32 further, so a warp reads the list 32 entries per load, one batch
// ahead of use; entries past the end repeat the last page (its keys are
// masked wherever they fall outside the sequence); an empty list reads page 0
// (the caller records the length error). get() is warp-collective: it moves
// the cursor to entry `e_first` (non-decreasing across calls) and returns to
// each lane the page of its own entry `e`, which must lie in
// [e_first, e_first + 32) -- the entries of one KV tile (at most 8).
// ---------------------------------------------------------------------------
struct PageCursor {
  const int32_t* list;
  int count, base, cur, nxt;
  __device__ __forceinline__ int load(int e) const {
    return count > 0 ? list[e < count ? e : count - 1] : 0;
  }
  __device__ __forceinline__ void start(const int32_t* list_, int count_, int e0, int lane) {
    list = list_;
    count = count_;
    base = e0 & ~31;
    cur = load(base + lane);
    nxt = load(base + 32 + lane);
  }
  __device__ __forceinline__ int get(int e_first, int e, int lane) {
    while (e_first >= base + 32) {
      base += 32;
      cur = nxt;
      nxt = load(base + 32 + lane);
    }
    const int from_cur = __shfl_sync(0xffffffffu, cur, (e - base) & 31);
    const int from_nxt = __shfl_sync(0xffffffffu, nxt, (e - base) & 31);
    return e - base < 32 ? from_cur : from_nxt;
  }
};

// max(a, b, c) in one instruction (sm_100 family); like fmaxf, a NaN operand
// is ignored.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 2^x on the SFU (MUFU.EX2); exact 0 for -inf.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Every thread of every CTA of the cluster arrives, then waits (release /
// acquire at cluster scope). All threads of the kernel reach each call.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Load from the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_dsmem(const float* p, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(p)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

template <int N>
__device__ __forceinline__ void ld_dsmem_vec(const float* p, uint32_t rank, float (&v)[N]) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(p)), "r"(rank));
  if constexpr (N == 4) {
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
                 : "r"(ra)
                 : "memory");
  } else {
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
                 : "=f"(v[0]), "=f"(v[1])
                 : "r"(ra)
                 : "memory");
  }
}

// Within each group of 8 lanes, lane i holds chunk e (e = 0..7, 16 bytes
// each) of row i of the group in ch[e]; afterwards it holds chunk i of row e
// in ch[e]. Three shfl_xor stages: at lane bit m, for each chunk pair
// (e, e | m), the lane with bit m clear gives chunk e | m and takes its
// partner's chunk e into that slot, and the partner does the mirror image.
// Rows stored as ch[e] of lane i at chunk i then make a store instruction
// write 4 whole 128-byte row segments per warp. Warp-collective.
template <typename V4>
__device__ __forceinline__ void transpose8_chunks(V4 (&ch)[8], int lane) {
  const int i = lane & 7;
#pragma unroll
  for (int m = 4; m >= 1; m >>= 1) {
    const bool up = (i & m) != 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (e & m) continue;
      V4 snd = up ? ch[e] : ch[e | m];
      V4 rcv;
      rcv.x = __shfl_xor_sync(0xffffffffu, snd.x, m);
      rcv.y = __shfl_xor_sync(0xffffffffu, snd.y, m);
      rcv.z = __shfl_xor_sync(0xffffffffu, snd.z, m);
      rcv.w = __shfl_xor_sync(0xffffffffu, snd.w, m);
      if (up) ch[e] = rcv;
      else ch[e | m] = rcv;
    }
  }
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace sinkattn
