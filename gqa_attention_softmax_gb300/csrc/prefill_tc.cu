// Varlen prefill with a per-head softmax sink on the 5th-generation tensor
// cores (tcgen05.mma, accumulators and P in TMEM, operands staged by TMA).
//
// Prefill is the one dense contraction of the path ("Hosting Qwen on
// Blackwell", section "Prefillers": prefill is compute-intensive, thousands
// of tokens processed at once). Per CTA:
//
//  * rows: NT query tiles of 128 (query token, head-in-group) pairs of one KV
//    head -- each tile is QB = 128/G consecutive tokens times the G query
//    heads sharing that KV head -- so one K/V tile in shared memory serves
//    every tile and the whole GQA group, and the causal diagonal cuts only a
//    few keys of the last KV tile. NT is 3 at head_dim 64 and 2 at 128, in
//    both launches;
//  * warp 0: TMA producer (the Q tiles once as 3-D boxes, then K/V tiles of
//    KT keys -- 96 at head_dim 64, 128 at 128 -- into an NST-stage ring,
//    right-aligned to the end of the key range so no copy reads past the
//    last key needed);
//  * warp 1: allocates TMEM and issues every MMA from one elected lane (the
//    warp runs the schedule uniformly), with S_t = Q_t K^T (M 128, N KT,
//    K d; both operands in shared memory) and O_t += P_t V (M 128, N d, K KT;
//    P_t read from TMEM, V from shared memory). With one S buffer per tile
//    the order is S_t(0) for every tile, then per KV tile j and tile t:
//    PV_t(j), then S_t(j+1) once PV_t(j) has completed (S overwrites P), so
//    the tiles' chains interleave on the tensor core;
//  * warps 2 + 4t .. 5 + 4t: softmax of tile t, one thread per row (= TMEM
//    lane). The running max starts at the head's sink and the running sum at
//    1 ("GPT-OSS on Day 0", section "Kernels for GPT-OSS / Sink attention").
//    Each thread loads its row's KT scores from TMEM in one batch, so the
//    row maximum and sums need no exchange between threads; P goes back as
//    bf16 into the first KT/2 columns of the same S buffer. The running
//    maximum is exact, so a row's largest weight is exactly 1 in bf16; O_t is
//    rescaled in TMEM when a row maximum grows, and out is divided by the
//    exact fp32 row sum.
//
// Every wait is bounded; on a timeout the CTA records SINKATTN_TIMEOUT,
// drains its copies and MMAs, frees TMEM and exits.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace sinkattn {

__device__ int g_status_prefill_tc;

struct TcParams {
  const int32_t* cu_q;      // nullptr: every sequence has q_len queries (decode drafts)
  const int32_t* cu_k;
  int q_len;
  int batch, n_items;
  int Hq, Hkv, G, QB, nqb, max_kv;
  float sm_scale, scale_log2;
  int causal, window;
  const float* sinks;
  __nv_bfloat16* out;
  float* lse;
  // paged KV (page_size > 0): page-pool rows, boxes of box_rows keys
  int page_size, box_rows;
  const int32_t* page_indptr;
  const int32_t* page_indices;
};

template <int D, int NST, int NT = 2>
struct TcCfg {
  // NT query tiles per CTA (one softmax warpgroup each), one S buffer per
  // tile: three tiles at d 64, two at d 128 (TMEM holds no more).
  static constexpr int NO = D;                    // O_t columns
  static constexpr int NSUB = D / 64;
  static constexpr int KT = D == 64 ? 96 : 128;   // keys per KV tile
  static constexpr int NSB = NT;                  // S buffers
  static constexpr int QSUB = 128 * 128;          // [128 rows][64 bf16], 128B-swizzled: 16 KB
  static constexpr int KVSUB = KT * 128;          // [KT rows][64 bf16], 128B-swizzled
  static constexpr int Q_TILE = NSUB * QSUB;
  static constexpr int KV_TILE = NSUB * KVSUB;
  static constexpr int STAGE = 2 * KV_TILE;       // K and V of one KV tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + NT * Q_TILE;
  static constexpr int LIST_CAP = 512;            // items per CTA in the snake list
  static constexpr int CUQ_CAP = 1025;            // sequences staged for the item scan
  static constexpr int OFF_LIST = OFF_KV + NST * STAGE;   // [LIST_CAP + 32 + CUQ_CAP] ints
  static constexpr int OFF_BAR = OFF_LIST + ((LIST_CAP + 32 + CUQ_CAP) * 4 + 15) / 16 * 16;
  static constexpr int N_BARS = 2 + 2 * NST + NSB + NT + NT + 1;
  static constexpr int SMEM = 1024 + OFF_BAR + N_BARS * 8 + 64;
  static constexpr int THREADS = (2 + 4 * NT) * 32;   // TMA, MMA, NT tiles x 4 softmax warps
  // registers per thread: 14 warps put 4 on two SM sub-partitions, whose
  // 16384 registers then allow 128 a thread (bounded by a 512-thread launch)
  static constexpr int LB_THREADS = NT == 2 ? 320 : 512;
  static constexpr uint32_t TMEM_COLS = 512;
  // TMEM columns: S buffers (P in the first KT / 2 columns of its S) at KT b,
  // O_t after them.
  __host__ __device__ static constexpr uint32_t col_s(int buf) { return static_cast<uint32_t>(KT) * buf; }
  __host__ __device__ static constexpr uint32_t col_o(int t) {
    return static_cast<uint32_t>(NSB * KT + NO * t);
  }
  static_assert(NSB * KT + NT * NO <= 512, "TMEM budget");
  static_assert(NT == 2 || (NT == 3 && D == 64), "tiles per CTA");
  static_assert(KVSUB % 1024 == 0 && KT % 32 == 0, "tile shape");
};

// Epilogue: out row = O_t row / l, as bf16. Each lane owns one row of the
// tile; D / 64 blocks of 64 columns (128 bytes) are read from TMEM, scaled
// and packed into eight 16-byte chunks. An 8 x 8 transpose of the chunks
// within each group of 8 lanes leaves lane i with chunk i of each of the
// group's rows, so a store instruction writes 4 whole 128-byte rows per warp
// rather than 16 bytes of each of 32 rows: 4 L1 wavefronts instead of 32,
// which keeps the load/store unit free for the next item's copies into
// shared memory.
// Warp-collective; `zero` (warp-uniform) stores zeros without reading TMEM.
template <int D>
__device__ __forceinline__ void store_o_rows(uint32_t o_addr, bool zero, float inv,
                                             __nv_bfloat16* orow, bool valid, int lane) {
  const int i = lane & 7;
#pragma unroll
  for (int blk = 0; blk < D / 64; ++blk) {
    uint4 ch[8];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float o[32];
      if (!zero) {
        tc::tmem_ld32(o_addr + blk * 64 + half * 32, o);
        tc::tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0.f;
      }
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint4& pk = ch[half * 4 + q4];
        pk.x = pack_bf16x2(o[q4 * 8 + 0] * inv, o[q4 * 8 + 1] * inv);
        pk.y = pack_bf16x2(o[q4 * 8 + 2] * inv, o[q4 * 8 + 3] * inv);
        pk.z = pack_bf16x2(o[q4 * 8 + 4] * inv, o[q4 * 8 + 5] * inv);
        pk.w = pack_bf16x2(o[q4 * 8 + 6] * inv, o[q4 * 8 + 7] * inv);
      }
    }
    transpose8_chunks(ch, lane);   // now ch[e] of lane i: chunk i of the group's row e
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int src = (lane & ~7) + e;
      const unsigned long long row =
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(orow), src);
      const int v = __shfl_sync(0xffffffffu, valid ? 1 : 0, src);
      if (v)
        *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(row) + blk * 64 + i * 8) =
            ch[e];
    }
  }
}

// One block per item: block (x, y, z) runs query block nqb - 1 - x of KV head
// y of sequence z (longest query blocks launch first), the hardware deals the
// blocks out to the SMs as they free up.
template <int D, int NST, int NT>
__global__ void __launch_bounds__(TcCfg<D, NST, NT>::LB_THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const TcParams p) {
  using C = TcCfg<D, NST, NT>;
  constexpr int KT = C::KT;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* kv_full = q_full + 1;
  uint64_t* kv_empty = kv_full + NST;
  uint64_t* s_full = kv_empty + NST;   // [NSB]: S written into buffer b
  uint64_t* p_full = s_full + C::NSB;  // [NT]: P_t(j) written and O_t rescaled (128 arrivals)
  uint64_t* pv_done = p_full + NT;     // [NT]: PV_t(j) completed
  uint64_t* drain = pv_done + NT;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* status = &g_status_prefill_tc;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.z;
  const int kvh = blockIdx.y;
  const int qb = p.nqb - 1 - static_cast<int>(blockIdx.x);   // longest query blocks first

  const int q_start = p.cu_q ? p.cu_q[b] : b * p.q_len;
  const int Lq = p.cu_q ? p.cu_q[b + 1] - q_start : p.q_len;
  const int k_start = p.cu_k[b];
  const int Lk = p.cu_k[b + 1] - k_start;
  const int q0 = qb * NT * p.QB;  // first token of tile 0
  if (q0 >= Lq) return;           // uniform over the CTA, before any barrier or TMEM use
  const int nq = min(NT * p.QB, Lq - q0);
  if (threadIdx.x == 0 && (Lk < Lq || Lk > p.max_kv)) atomicExch(status, SINKATTN_BAD_LENGTHS);

  const int pos0 = Lk - Lq + q0;
  const int posN = pos0 + nq - 1;
  int k_lo = 0, k_hi = Lk;
  if (p.causal) k_hi = min(k_hi, posN + 1);
  if (p.window > 0) k_lo = max(k_lo, pos0 - p.window + 1);
  // Tiles end at k_hi (contiguous: no copy reads past the last key needed),
  // or start on a multiple of KT (paged: no box straddles a page).
  const bool paged = p.page_size > 0;
  const int t0 = k_lo / KT * KT;
  const int n = (k_hi > k_lo) ? (k_hi - (paged ? t0 : k_lo) + KT - 1) / KT : 0;
  const int first = paged ? t0 : k_hi - n * KT;   // key of tile 0's first column

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NST; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < C::NSB; ++i) mbar_init(&s_full[i], 1);
    for (int t = 0; t < NT; ++t) {
      mbar_init(&p_full[t], 128);
      mbar_init(&pv_done[t], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  int issued = 0;   // producer: KV tiles whose copies were issued (or left out by the test hook)

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    // The warp runs the loop (page lists are read 32 entries per warp load);
    // lane 0 issues every copy.
    const bool leader = (lane == 0);
    if (leader) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint32_t q_bytes = static_cast<uint32_t>(NT * C::NSUB * 128 * p.G * p.QB);
      mbar_arrive_expect_tx(q_full, q_bytes);
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int sub = 0; sub < C::NSUB; ++sub)
          tc::tma_load_3d(smem + C::OFF_Q + t * C::Q_TILE + sub * C::QSUB, &tmQ, sub * 64,
                          kvh * p.G, q_start + q0 + t * p.QB, q_full);
    }
    const uint64_t policy = policy_evict_last();   // K/V are re-read by every query block
    const int slab = k_start * p.Hkv + kvh * Lk;     // contiguous: tensor-map row of key 0
    PageCursor pc;
    if (paged && n > 0) {
      const int e0 = p.page_indptr[b];
      const int np = p.page_indptr[b + 1] - e0;
      if (leader && Lk > np * p.page_size) atomicExch(status, SINKATTN_BAD_LENGTHS);
      pc.start(p.page_indices + e0, np, first / p.page_size, lane);
    }
    const int skip_tile = hook_skip_tile();
    for (int i = 0; i < n; ++i) {
      const int st = i % NST;
      if (!__all_sync(0xffffffffu, mbar_wait(&kv_empty[st], ((i / NST) & 1) ^ 1, abort_flag, status)))
        break;
      if (i == skip_tile) {   // test hook: the waits for this tile run out
        issued = i + 1;
        continue;
      }
      uint8_t* kt = smem + C::OFF_KV + st * C::STAGE;
      if (leader) mbar_arrive_expect_tx(&kv_full[st], C::STAGE);
      const int j0 = first + i * KT;
      if (!paged) {
        if (leader) {
#pragma unroll
          for (int sub = 0; sub < C::NSUB; ++sub) {
            tma_load_2d_hint(kt + sub * C::KVSUB, &tmK, sub * 64, slab + j0, &kv_full[st], policy);
            tma_load_2d_hint(kt + C::KV_TILE + sub * C::KVSUB, &tmV, sub * 64, slab + j0,
                             &kv_full[st], policy);
          }
        }
      } else {
        // one box per page segment, lane i issuing box i: rows (page, head,
        // slot) of the pool
        const int nbox = KT / p.box_rows;
        const int a = j0 + min(lane, nbox - 1) * p.box_rows;
        const int page = pc.get(j0 / p.page_size, a / p.page_size, lane);
        if (lane < nbox) {
          const int row = (page * p.Hkv + kvh) * p.page_size + a % p.page_size;
          const int off = (a - j0) * 128;
#pragma unroll
          for (int sub = 0; sub < C::NSUB; ++sub) {
            tma_load_2d_hint(kt + sub * C::KVSUB + off, &tmK, sub * 64, row, &kv_full[st], policy);
            tma_load_2d_hint(kt + C::KV_TILE + sub * C::KVSUB + off, &tmV, sub * 64, row,
                             &kv_full[st], policy);
          }
        }
      }
      issued = i + 1;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp runs the schedule (waits and descriptor arithmetic stay
    // warp-uniform); one elected lane issues each MMA and commit.
    const bool leader = tc::elect_one();
    auto wwait1 = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, status));
    };
    {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(128, KT, false);
      constexpr uint32_t idesc_o = tc::idesc_bf16_f32(128, C::NO, true);
      constexpr uint64_t STAGE16 = C::STAGE >> 4;   // one K/V stage, in descriptor address units
      constexpr uint64_t QSUB16 = C::QSUB >> 4;
      constexpr uint64_t KVSUB16 = C::KVSUB >> 4;
      // Descriptors prepared once: a K step (16 elements = 32 bytes) within a
      // 128-byte swizzle row adds 2 to the address field, the next 64-column
      // block adds its size / 16, a stage adds STAGE / 16, 16 keys of V add 128.
      const uint64_t qd0 = tc::smem_desc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
      const uint64_t kd0 = tc::smem_desc_sw128(smem_u32(smem + C::OFF_KV), 16, 1024);
      // V is MN-major: its 64-column blocks are KVSUB bytes apart.
      const uint32_t v_base0 = smem_u32(smem + C::OFF_KV + C::KV_TILE);
      const uint64_t vd0 = tc::smem_desc_sw128(v_base0, static_cast<uint32_t>(C::KVSUB), 1024);
      auto issue_s = [&](int t, int j) {
        const int buf = t;
        const uint64_t kd = kd0 + static_cast<uint64_t>(j % NST) * STAGE16;
        const uint64_t qd = qd0 + static_cast<uint64_t>(t) * (C::Q_TILE >> 4);
        const uint32_t d_tm = tmem + C::col_s(buf);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t step = static_cast<uint64_t>(kk & 3) * 2;
            tc::mma_ss(d_tm, qd + static_cast<uint64_t>(kk >> 2) * QSUB16 + step,
                       kd + static_cast<uint64_t>(kk >> 2) * KVSUB16 + step, idesc_s,
                       kk > 0 ? 1u : 0u);
          }
          tc::commit(&s_full[buf]);
        }
        __syncwarp();
      };
      auto issue_pv = [&](int t, int j) {
        const uint64_t vd = vd0 + static_cast<uint64_t>(j % NST) * STAGE16;
        const uint32_t d_tm = tmem + C::col_o(t);
        const uint32_t a_tm = tmem + C::col_s(t);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < KT / 16; ++kk)
            tc::mma_ts(d_tm, a_tm + kk * 8, vd + static_cast<uint64_t>(kk) * 128u, idesc_o,
                       (j > 0 || kk > 0) ? 1u : 0u);
          tc::commit(&pv_done[t]);
        }
        __syncwarp();
      };
      // Order, one buffer per tile: S_t(0) for every tile, then per KV tile j
      // and tile t: PV_t(j), then S_t(j+1) into the same buffer once PV_t(j) is
      // done (the tensor core may not overwrite P before the MMA has read it).
      bool ok = wwait1(q_full, 0);
      if (ok && n > 0) {
        ok = wwait1(&kv_full[0], 0);
        if (ok) {
          tc::fence_after_sync();
          for (int t = 0; t < NT; ++t) issue_s(t, 0);
        }
      }
      for (int j = 0; ok && j < n; ++j) {
        for (int t = 0; t < NT; ++t) {
          if (!wwait1(&p_full[t], j & 1)) { ok = false; break; }
          tc::fence_after_sync();
          issue_pv(t, j);
          if (t == NT - 1) {
            if (leader) tc::commit(&kv_empty[j % NST]);
            __syncwarp();
          }
          if (j + 1 < n) {
            // the first tile's S of KV tile j + 1 waits for its K; S_t(j + 1)
            // overwrites the buffer PV_t(j) reads P from
            if (t == 0 && !wwait1(&kv_full[(j + 1) % NST], ((j + 1) / NST) & 1)) { ok = false; break; }
            if (!wwait1(&pv_done[t], j & 1)) { ok = false; break; }
            tc::fence_after_sync();
            issue_s(t, j + 1);
          }
        }
      }
      // every MMA this warp issued has completed before the CTA frees TMEM
      if (leader) tc::commit(drain);
      __syncwarp();
      mbar_drain(drain, 0);
    }
  } else {
    // ---------------------------------------------------------------- softmax
    // 4 NT warps: tile t = (warp - 2) / 4; warp w may access TMEM lanes 32 (w % 4) ...
    const int t = (warp - 2) >> 2;
    const int quad = warp & 3;       // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    const int G = p.G;
    const int rg = row / G;          // token within the tile
    const int tl = t * p.QB + rg;    // token within the CTA
    const bool valid = rg < p.QB && tl < nq;
    const int pos = pos0 + tl;
    const int h = kvh * G + (row - rg * G);
    const int tok = q_start + q0 + tl;
    int lo_r = k_lo, hi_r = k_hi - 1;
    if (p.window > 0) lo_r = max(lo_r, pos - p.window + 1);
    if (p.causal) hi_r = min(hi_r, pos);
    const float c2 = p.scale_log2;

    // l: the row's running sum, the sink's term included (for out and lse).
    // The running maximum is exact, so the row's largest weight is exactly 1
    // and the P.V MMA's bf16 rounding of the others stays below 2^-8 of each.
    float m_used = kNegInf, l = 0.f;
    if (p.sinks != nullptr && valid) {
      const float s = p.sinks[h];
      if (s != kNegInf) {
        m_used = s / p.sm_scale;   // the sink, in raw logit units
        l = 1.f;
      }
    }
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t o_addr = lane_base + C::col_o(t);
    constexpr int NCH = KT / 32;     // 32-column chunks of a score row
    bool ok = true;
    // A wait that gives up in any lane makes the whole warp leave, so the
    // warp-collective TMEM loads/stores below never run with missing lanes.
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, status));
    };

    for (int j = 0; j < n; ++j) {
      const int buf = t;
      if (!wwait(&s_full[buf], j & 1)) { ok = false; break; }
      tc::fence_after_sync();
      const uint32_t s_addr = lane_base + C::col_s(buf);
      const int j0 = first + j * KT;
      const bool masked = (j0 < lo_r || j0 + KT - 1 > hi_r);
      const int clo = lo_r - j0, chi = hi_r - j0;

      // the row's KT scores, one batch of loads
      float v[NCH][32];
#pragma unroll
      for (int c = 0; c < NCH; ++c) tc::tmem_ld32(s_addr + 32 * c, v[c]);
      tc::tmem_wait_ld();
      if (masked) {
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const int lo_c = clo - c * 32, hi_c = chi - c * 32;
          if (lo_c <= 0 && hi_c >= 31) continue;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e < lo_c || e > hi_c) v[c][e] = kNegInf;
        }
      }
      // row maximum: 2 NCH independent chains of three-input maxima
      float mxc[2 * NCH];
#pragma unroll
      for (int i = 0; i < 2 * NCH; ++i)
        mxc[i] = fmaxf(v[i >> 1][(i & 1) * 16], v[i >> 1][(i & 1) * 16 + 1]);
#pragma unroll
      for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int e = 2; e < 16; e += 2) {
          mxc[2 * c] = fmax3(mxc[2 * c], v[c][e], v[c][e + 1]);
          mxc[2 * c + 1] = fmax3(mxc[2 * c + 1], v[c][16 + e], v[c][16 + e + 1]);
        }
      float mx = fmax3(mxc[0], mxc[1], mxc[2]);
#pragma unroll
      for (int i = 3; i < 2 * NCH; i += 2)
        mx = (i + 1 < 2 * NCH) ? fmax3(mx, mxc[i], mxc[i + 1]) : fmaxf(mx, mxc[i]);

      float alpha = 1.f;
      bool rescale = false;
      if (mx > m_used) {
        alpha = (m_used == kNegInf) ? 0.f : ex2((m_used - mx) * c2);
        m_used = mx;
        rescale = true;
      }
      const float mb = (m_used == kNegInf) ? 0.f : m_used * c2;

      // P = 2^(s*c2 - mb) as bf16 into the first KT / 2 columns of this S
      // buffer (all KT scores are already in registers). Scale-subtract and
      // the exact sum run two lanes per instruction (paired fp32 FMA / add).
      const float2 c2x2 = make_float2(c2, c2), nmb2 = make_float2(-mb, -mb);
      float2 rs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                       make_float2(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const int k = hh * 16 + e;
            const float2 x = __ffma2_rn(make_float2(v[c][k], v[c][k + 1]), c2x2, nmb2);
            const float2 a = make_float2(ex2(x.x), ex2(x.y));
            rs2[(e >> 1) & 3] = __fadd2_rn(rs2[(e >> 1) & 3], a);
            pk[e >> 1] = pack_bf16x2(a.x, a.y);
          }
          tc::tmem_st8(s_addr + 16 * c + 8 * hh, pk);
        }
      const float2 rsa = __fadd2_rn(__fadd2_rn(rs2[0], rs2[1]), __fadd2_rn(rs2[2], rs2[3]));
      const float rs = rsa.x + rsa.y;

      // S_t(j) was issued after PV_t(j-1) had completed, so O_t is free to
      // touch and p_full[t] cannot run two phases ahead of the MMA warp.
      // Rescale the row's O_t when some row of this warp moved its maximum
      // (warp-uniform branch).
      if (j >= 1 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tc::tmem_ld32(o_addr + c * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tc::tmem_st32(o_addr + c * 32, o);
        }
      }
      tc::tmem_wait_st();
      l = l * alpha + rs;
      tc::fence_before_sync();
      mbar_arrive(&p_full[t]);
    }

    // ------------------------------------------------------------ epilogue
    if (ok && n >= 1) {
      ok = wwait(&pv_done[t], (n - 1) & 1);
      tc::fence_after_sync();
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat16* orow = p.out + (static_cast<size_t>(tok) * p.Hq + h) * D;
    store_o_rows<D>(o_addr, !(n >= 1 && ok), inv, orow, valid, lane);
    if (valid && p.lse != nullptr)
      p.lse[static_cast<size_t>(tok) * p.Hq + h] =
          l > 0.f ? (m_used * c2 + lg2(l)) * kLn2 : kNegInf;
  }

  // a warp that left its loop early may still have TMEM loads or stores in flight
  tc::tmem_wait_ld();
  tc::tmem_wait_st();
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag) {
    // a wait gave up: let every issued copy land before the CTA's shared
    // memory goes away (a left-out tile's phase never completes: bounded)
    mbar_drain(q_full, 0);
    for (int i = max(0, issued - NST); i < issued; ++i) mbar_drain(&kv_full[i % NST], (i / NST) & 1);
  }
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// One work item: both query tiles of (sequence b, KV head kvh, query block qb)
// and the KV tiles they visit. n < 0: the block has no query rows; n == 0:
// rows but no visible key (the epilogue alone runs).
struct PfItem {
  int b, kvh, q_start, Lq, q0, nq, k_start, Lk, pos0, k_lo, k_hi, n, first;
};

template <int KT, int NT>
__device__ __forceinline__ PfItem pf_item(const TcParams& p, int it) {
  PfItem t;
  const int per = p.Hkv * p.batch;
  const int qb = p.nqb - 1 - it / per;   // longest query blocks first
  const int r = it % per;
  t.kvh = r % p.Hkv;
  t.b = r / p.Hkv;
  t.q_start = p.cu_q ? p.cu_q[t.b] : t.b * p.q_len;
  t.Lq = p.cu_q ? p.cu_q[t.b + 1] - t.q_start : p.q_len;
  t.k_start = p.cu_k[t.b];
  t.Lk = p.cu_k[t.b + 1] - t.k_start;
  t.q0 = qb * NT * p.QB;   // first token of the item's first tile
  t.nq = 0;
  t.pos0 = t.k_lo = t.k_hi = t.first = 0;
  t.n = -1;
  if (t.q0 >= t.Lq) return t;
  t.nq = min(NT * p.QB, t.Lq - t.q0);
  t.pos0 = t.Lk - t.Lq + t.q0;
  const int posN = t.pos0 + t.nq - 1;
  t.k_hi = t.Lk;
  if (p.causal) t.k_hi = min(t.k_hi, posN + 1);
  if (p.window > 0) t.k_lo = max(0, t.pos0 - p.window + 1);
  // Tiles end at k_hi (contiguous: no copy reads past the last key needed),
  // or start on a multiple of KT (paged: no box straddles a page).
  const bool paged = p.page_size > 0;
  const int t0 = t.k_lo / KT * KT;
  t.n = (t.k_hi > t.k_lo) ? (t.k_hi - (paged ? t0 : t.k_lo) + KT - 1) / KT : 0;
  t.first = paged ? t0 : t.k_hi - t.n * KT;
  return t;
}

// Persistent: CTA c runs items c, c + gridDim.x, ... (one CTA per SM, TMEM
// allocated once). KV tiles, S buffers and every barrier phase are counted
// across items, so the K/V ring streams on from one item into the next; the
// next item's Q is loaded as soon as the tensor core has finished the
// current item's last S.
template <int D, int NST, int NT>
__global__ void __launch_bounds__(TcCfg<D, NST, NT>::LB_THREADS, 1)
    prefill_tc_persistent_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const TcParams p) {
  using C = TcCfg<D, NST, NT>;
  constexpr int KT = C::KT;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;             // Q of the item landed (by active item ordinal)
  uint64_t* q_empty = q_full + 1;      // the item's last S completed: Q may be replaced
  uint64_t* kv_full = q_empty + 1;
  uint64_t* kv_empty = kv_full + NST;
  uint64_t* s_full = kv_empty + NST;   // [NSB]: S written into buffer b
  uint64_t* p_full = s_full + C::NSB;  // [NT]: P_t written and O_t rescaled (128 arrivals)
  uint64_t* pv_done = p_full + NT;     // [NT]: PV_t completed (one buffer per tile)
  uint64_t* drain = pv_done + NT;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* status = &g_status_prefill_tc;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int* list = reinterpret_cast<int*>(smem + C::OFF_LIST);      // [LIST_CAP] this CTA's items
  int* scan = list + C::LIST_CAP;                               // [16] per-warp counts, [16] misc
  int* cuq_s = scan + 32;                                       // [CUQ_CAP] staged cu_seqlens_q

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < NST; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < C::NSB; ++i) mbar_init(&s_full[i], 1);
    for (int t = 0; t < NT; ++t) {
      mbar_init(&p_full[t], 128);
      mbar_init(&pv_done[t], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc::tmem_relinquish();
  }

  // This CTA's items. Items (the rectangle of query blocks x KV heads x
  // sequences, longest query blocks first) that have query rows are ranked in
  // that order and dealt out in snake order -- rank r of round r / G goes to
  // CTA r % G on even rounds and G - 1 - r % G on odd ones -- so every CTA
  // gets one item of each round and the loads differ by about one small
  // item. Without room for the list, items go round-robin.
  const int G = static_cast<int>(gridDim.x);
  const bool staged = p.batch + 1 <= C::CUQ_CAP;
  if (staged)
    for (int i = threadIdx.x; i <= p.batch; i += blockDim.x) cuq_s[i] = p.cu_q ? p.cu_q[i] : i * p.q_len;
  __syncthreads();
  const int per = p.Hkv * p.batch;
  auto has_rows = [&](int it) -> bool {
    const int qb = p.nqb - 1 - it / per;
    const int b = (it % per) / p.Hkv;
    const int Lq = staged ? cuq_s[b + 1] - cuq_s[b] : (p.cu_q ? p.cu_q[b + 1] - p.cu_q[b] : p.q_len);
    return qb * NT * p.QB < Lq;
  };
  int n_list = 0, total = 0;
  bool use_list = staged;
  if (use_list) {
    const int nw = blockDim.x >> 5;
    for (int base = 0; base < p.n_items; base += blockDim.x) {
      const int it = base + static_cast<int>(threadIdx.x);
      const bool f = it < p.n_items && has_rows(it);
      const uint32_t bal = __ballot_sync(0xffffffffu, f);
      if (lane == 0) scan[warp] = __popc(bal);
      __syncthreads();
      int before = total;
      for (int w = 0; w < warp; ++w) before += scan[w];
      int chunk = 0;
      for (int w = 0; w < nw; ++w) chunk += scan[w];
      if (f) {
        const int r = before + __popc(bal & ((1u << lane) - 1u));
        const int round = r / G, pos = r - round * G;
        const int cta = (round & 1) ? G - 1 - pos : pos;
        if (cta == static_cast<int>(blockIdx.x) && round < C::LIST_CAP) list[round] = it;
      }
      total += chunk;
      __syncthreads();
    }
    const int rounds = (total + G - 1) / G;
    if (rounds > C::LIST_CAP) {
      use_list = false;
    } else {
      // rounds in which this CTA got an item: all but possibly the last
      const int last = rounds - 1;
      const int last_n = total - last * G;   // items of the last round
      const int pos_last = (last & 1) ? G - 1 - static_cast<int>(blockIdx.x)
                                      : static_cast<int>(blockIdx.x);
      n_list = (rounds > 0 && pos_last >= last_n) ? last : rounds;
    }
  }
  const int n_mine = use_list ? n_list
                              : (p.n_items - static_cast<int>(blockIdx.x) + G - 1) / G;
  auto item_of = [&](int k) -> int {
    return use_list ? list[k] : static_cast<int>(blockIdx.x) + k * G;
  };

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  int g_prod = 0, qi_prod = 0;   // producer: KV tiles and Q loads issued

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    // The warp runs the loop (page lists are read 32 entries per warp load);
    // lane 0 issues every other copy.
    const bool leader = (lane == 0);
    auto pwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, status));
    };
    if (leader) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    const uint64_t policy = policy_evict_last();   // K/V are re-read by every query block
    const uint32_t q_bytes = static_cast<uint32_t>(NT * C::NSUB * 128 * p.G * p.QB);
    int g = 0, qi = 0;   // KV tiles and active items so far
    bool ok = true;
    const int skip_tile = hook_skip_tile();
    for (int k = 0; ok && k < n_mine; ++k) {
      const PfItem t = pf_item<KT, NT>(p, item_of(k));
      if (t.n < 0) continue;
      if (leader && (t.Lk < t.Lq || t.Lk > p.max_kv)) atomicExch(status, SINKATTN_BAD_LENGTHS);
      if (t.n == 0) continue;
      if (qi > 0 && !pwait(q_empty, (qi - 1) & 1)) { ok = false; break; }
      if (leader) {
        mbar_arrive_expect_tx(q_full, q_bytes);
#pragma unroll
        for (int tt = 0; tt < NT; ++tt)
#pragma unroll
          for (int sub = 0; sub < C::NSUB; ++sub)
            tc::tma_load_3d(smem + C::OFF_Q + tt * C::Q_TILE + sub * C::QSUB, &tmQ, sub * 64,
                            t.kvh * p.G, t.q_start + t.q0 + tt * p.QB, q_full);
      }
      ++qi;
      const int slab = t.k_start * p.Hkv + t.kvh * t.Lk;   // contiguous: tensor-map row of key 0
      PageCursor pc;
      if (p.page_size > 0) {
        const int e0 = p.page_indptr[t.b];
        const int np = p.page_indptr[t.b + 1] - e0;
        if (leader && t.Lk > np * p.page_size) atomicExch(status, SINKATTN_BAD_LENGTHS);
        pc.start(p.page_indices + e0, np, t.first / p.page_size, lane);
      }
      for (int i = 0; i < t.n; ++i, ++g) {
        const int st = g % NST;
        if (!pwait(&kv_empty[st], ((g / NST) & 1) ^ 1)) { ok = false; break; }
        if (g == skip_tile) continue;   // test hook: the waits for this tile run out
        uint8_t* kt = smem + C::OFF_KV + st * C::STAGE;
        if (leader) mbar_arrive_expect_tx(&kv_full[st], C::STAGE);
        const int j0 = t.first + i * KT;
        if (p.page_size == 0) {
          if (leader) {
#pragma unroll
            for (int sub = 0; sub < C::NSUB; ++sub) {
              tma_load_2d_hint(kt + sub * C::KVSUB, &tmK, sub * 64, slab + j0, &kv_full[st],
                               policy);
              tma_load_2d_hint(kt + C::KV_TILE + sub * C::KVSUB, &tmV, sub * 64, slab + j0,
                               &kv_full[st], policy);
            }
          }
        } else {
          // one box per page segment, lane i issuing box i: rows (page,
          // head, slot) of the pool
          const int nbox = KT / p.box_rows;
          const int a = j0 + min(lane, nbox - 1) * p.box_rows;
          const int page = pc.get(j0 / p.page_size, a / p.page_size, lane);
          if (lane < nbox) {
            const int row = (page * p.Hkv + t.kvh) * p.page_size + a % p.page_size;
            const int off = (a - j0) * 128;
#pragma unroll
            for (int sub = 0; sub < C::NSUB; ++sub) {
              tma_load_2d_hint(kt + sub * C::KVSUB + off, &tmK, sub * 64, row, &kv_full[st],
                               policy);
              tma_load_2d_hint(kt + C::KV_TILE + sub * C::KVSUB + off, &tmV, sub * 64, row,
                               &kv_full[st], policy);
            }
          }
        }
      }
    }
    g_prod = g;
    qi_prod = qi;
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp runs the schedule (waits and descriptor arithmetic stay
    // warp-uniform); one elected lane issues each MMA and commit.
    const bool leader = tc::elect_one();
    auto wwait1 = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, status));
    };
    constexpr uint32_t idesc_s = tc::idesc_bf16_f32(128, KT, false);
    constexpr uint32_t idesc_o = tc::idesc_bf16_f32(128, C::NO, true);
    constexpr uint64_t STAGE16 = C::STAGE >> 4;   // one K/V stage, in descriptor address units
    constexpr uint64_t QSUB16 = C::QSUB >> 4;
    constexpr uint64_t KVSUB16 = C::KVSUB >> 4;
    // Descriptors prepared once: a K step (16 elements = 32 bytes) within a
    // 128-byte swizzle row adds 2 to the address field, the next 64-column
    // block adds its size / 16, a stage adds STAGE / 16, 16 keys of V add 128.
    const uint64_t qd0 = tc::smem_desc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
    const uint64_t kd0 = tc::smem_desc_sw128(smem_u32(smem + C::OFF_KV), 16, 1024);
    // V is MN-major: its 64-column blocks are KVSUB bytes apart.
    const uint32_t v_base0 = smem_u32(smem + C::OFF_KV + C::KV_TILE);
    const uint64_t vd0 = tc::smem_desc_sw128(v_base0, static_cast<uint32_t>(C::KVSUB), 1024);
    // S_t of global KV tile g
    auto issue_s = [&](int t, int g) {
      const int buf = t;
      const uint64_t kd = kd0 + static_cast<uint64_t>(g % NST) * STAGE16;
      const uint64_t qd = qd0 + static_cast<uint64_t>(t) * (C::Q_TILE >> 4);
      const uint32_t d_tm = tmem + C::col_s(buf);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t step = static_cast<uint64_t>(kk & 3) * 2;
          tc::mma_ss(d_tm, qd + static_cast<uint64_t>(kk >> 2) * QSUB16 + step,
                     kd + static_cast<uint64_t>(kk >> 2) * KVSUB16 + step, idesc_s,
                     kk > 0 ? 1u : 0u);
        }
        tc::commit(&s_full[buf]);
      }
      __syncwarp();
    };
    // PV_t of global KV tile g; the item's first PV overwrites O_t
    auto issue_pv = [&](int t, int g, bool first_of_item) {
      const uint64_t vd = vd0 + static_cast<uint64_t>(g % NST) * STAGE16;
      const uint32_t d_tm = tmem + C::col_o(t);
      const uint32_t a_tm = tmem + C::col_s(t);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk)
          tc::mma_ts(d_tm, a_tm + kk * 8, vd + static_cast<uint64_t>(kk) * 128u, idesc_o,
                     (!first_of_item || kk > 0) ? 1u : 0u);
        tc::commit(&pv_done[t]);   // S_t of the next KV tile may overwrite P_t
      }
      __syncwarp();
    };
    auto commit1 = [&](uint64_t* bar) {
      if (leader) tc::commit(bar);
      __syncwarp();
    };
    int g = 0, qi = 0;   // KV tiles and active items so far
    bool ok = true;
    // this CTA's next item with KV tiles after item k0 (n_mine when none)
    auto next_item = [&](int k0, PfItem& t) -> int {
      for (int k = k0 + 1; k < n_mine; ++k) {
        t = pf_item<KT, NT>(p, item_of(k));
        if (t.n > 0) return k;
      }
      return n_mine;
    };
    PfItem t_nx;
    int k_nx = next_item(-1, t_nx);
    while (ok && k_nx < n_mine) {
      const int k = k_nx;
      const PfItem t = t_nx;
      if (!wwait1(q_full, qi & 1)) { ok = false; break; }
      const int g0 = g, n = t.n;
      // One buffer per tile: S_t(g0) of every tile, then per KV tile g and
      // tile t: PV_t(g), then S_t(g+1) into the same buffer once PV_t(g) is done.
      for (int tt = 0; ok && tt < NT; ++tt) {
        if (tt == 0 && !wwait1(&kv_full[g0 % NST], (g0 / NST) & 1)) { ok = false; break; }
        if (g0 > 0 && !wwait1(&pv_done[tt], (g0 - 1) & 1)) { ok = false; break; }
        tc::fence_after_sync();
        issue_s(tt, g0);
        if (n == 1 && tt == NT - 1) commit1(q_empty);
      }
      // the next item's geometry, looked up while this item's first softmax
      // runs (its sequence offsets are global loads of about a microsecond)
      k_nx = next_item(k, t_nx);
      for (int jj = 0; ok && jj < n; ++jj) {
        const int gg = g0 + jj;
        for (int tt = 0; tt < NT; ++tt) {
          if (!wwait1(&p_full[tt], gg & 1)) { ok = false; break; }
          tc::fence_after_sync();
          issue_pv(tt, gg, jj == 0);
          if (tt == NT - 1) commit1(&kv_empty[gg % NST]);
          if (jj + 1 < n) {
            if (tt == 0 && !wwait1(&kv_full[(gg + 1) % NST], ((gg + 1) / NST) & 1)) { ok = false; break; }
            if (!wwait1(&pv_done[tt], gg & 1)) { ok = false; break; }
            tc::fence_after_sync();
            issue_s(tt, gg + 1);
            if (jj + 2 == n && tt == NT - 1) commit1(q_empty);
          }
        }
      }
      g += n;
      ++qi;
    }
    // every MMA this warp issued has completed before the CTA frees TMEM
    commit1(drain);
    mbar_drain(drain, 0);
  } else {
    // ---------------------------------------------------------------- softmax
    // 4 NT warps: tile t; warp w may access TMEM lanes 32 (w % 4) ...
    const int t = (warp - 2) >> 2;
    const int quad = warp & 3;       // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    const int G = p.G;
    const int rg = row / G;          // token within the tile
    const int hig = row - rg * G;    // head within the group
    const float c2 = p.scale_log2;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t o_addr = lane_base + C::col_o(t);
    constexpr int NCH = KT / 32;     // 32-column chunks of a score row
    // A wait that gives up in any lane makes the whole warp leave, so the
    // warp-collective TMEM loads/stores below never run with missing lanes.
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, status));
    };
    // wait for PV_t of global KV tile gg
    auto pv_wait = [&](int gg) -> bool { return wwait(&pv_done[t], gg & 1); };
    int g = 0;   // KV tiles so far
    bool ok = true;
    for (int k = 0; ok && k < n_mine; ++k) {
      const PfItem it_ = pf_item<KT, NT>(p, item_of(k));
      if (it_.n < 0) continue;
      const int n = it_.n;
      const int tl = t * p.QB + rg;    // token within the item
      const bool valid = rg < p.QB && tl < it_.nq;
      const int pos = it_.pos0 + tl;
      const int h = it_.kvh * G + hig;
      const int tok = it_.q_start + it_.q0 + tl;
      int lo_r = it_.k_lo, hi_r = it_.k_hi - 1;
      if (p.window > 0) lo_r = max(lo_r, pos - p.window + 1);
      if (p.causal) hi_r = min(hi_r, pos);

      // l: the row's running sum, the sink's term included (for out and
      // lse). The running maximum is exact, so the row's largest weight is
      // exactly 1 and the P.V MMA's bf16 rounding of the others stays below
      // 2^-8 of each.
      float m_used = kNegInf, l = 0.f;
      if (p.sinks != nullptr && valid) {
        const float s = p.sinks[h];
        if (s != kNegInf) {
          m_used = s / p.sm_scale;   // the sink, in raw logit units
          l = 1.f;
        }
      }

      for (int j = 0; j < n; ++j) {
        const int gg = g + j;
        const int buf = t;
        if (!wwait(&s_full[buf], gg & 1)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t s_addr = lane_base + C::col_s(buf);
        const int j0 = it_.first + j * KT;
        const bool masked = (j0 < lo_r || j0 + KT - 1 > hi_r);
        const int clo = lo_r - j0, chi = hi_r - j0;

        // the row's KT scores, one batch of loads
        float v[NCH][32];
#pragma unroll
        for (int c = 0; c < NCH; ++c) tc::tmem_ld32(s_addr + 32 * c, v[c]);
        tc::tmem_wait_ld();
        if (masked) {
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            const int lo_c = clo - c * 32, hi_c = chi - c * 32;
            if (lo_c <= 0 && hi_c >= 31) continue;
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (e < lo_c || e > hi_c) v[c][e] = kNegInf;
          }
        }
        // row maximum: 2 NCH independent chains of three-input maxima
        float mxc[2 * NCH];
#pragma unroll
        for (int i = 0; i < 2 * NCH; ++i)
          mxc[i] = fmaxf(v[i >> 1][(i & 1) * 16], v[i >> 1][(i & 1) * 16 + 1]);
#pragma unroll
        for (int c = 0; c < NCH; ++c)
#pragma unroll
          for (int e = 2; e < 16; e += 2) {
            mxc[2 * c] = fmax3(mxc[2 * c], v[c][e], v[c][e + 1]);
            mxc[2 * c + 1] = fmax3(mxc[2 * c + 1], v[c][16 + e], v[c][16 + e + 1]);
          }
        float mx = fmax3(mxc[0], mxc[1], mxc[2]);
#pragma unroll
        for (int i = 3; i < 2 * NCH; i += 2)
          mx = (i + 1 < 2 * NCH) ? fmax3(mx, mxc[i], mxc[i + 1]) : fmaxf(mx, mxc[i]);

        float alpha = 1.f;
        bool rescale = false;
        if (mx > m_used) {
          alpha = (m_used == kNegInf) ? 0.f : ex2((m_used - mx) * c2);
          m_used = mx;
          rescale = true;
        }
        const float mb = (m_used == kNegInf) ? 0.f : m_used * c2;

        // P = 2^(s*c2 - mb) as bf16 into the first KT / 2 columns of this S
        // buffer (all KT scores are already in registers). Scale-subtract and
        // the exact sum run two lanes per instruction (paired fp32 FMA / add).
        const float2 c2x2 = make_float2(c2, c2), nmb2 = make_float2(-mb, -mb);
        float2 rs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < NCH; ++c)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const int k = hh * 16 + e;
              const float2 x = __ffma2_rn(make_float2(v[c][k], v[c][k + 1]), c2x2, nmb2);
              const float2 a = make_float2(ex2(x.x), ex2(x.y));
              rs2[(e >> 1) & 3] = __fadd2_rn(rs2[(e >> 1) & 3], a);
              pk[e >> 1] = pack_bf16x2(a.x, a.y);
            }
            tc::tmem_st8(s_addr + 16 * c + 8 * hh, pk);
          }
        const float2 rsa = __fadd2_rn(__fadd2_rn(rs2[0], rs2[1]), __fadd2_rn(rs2[2], rs2[3]));
        const float rs = rsa.x + rsa.y;

        // S_t(j) was issued after PV_t(j-1) had completed (at j = 0 the
        // previous item's epilogue waited for its last PV_t), so O_t is free
        // to touch and p_full[t] cannot run two phases ahead of the MMA warp.
        // Rescale the row's O_t when some row of this warp moved its maximum
        // (warp-uniform branch).
        if (j >= 1 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tc::tmem_ld32(o_addr + c * 32, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tc::tmem_st32(o_addr + c * 32, o);
          }
        }
        tc::tmem_wait_st();
        l = l * alpha + rs;
        tc::fence_before_sync();
        mbar_arrive(&p_full[t]);
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      // O_t is read out before this thread hands P of the next item over,
      // so the next item's first PV (which overwrites O_t) comes after it.
      if (n >= 1) {
        if (!pv_wait(g + n - 1)) { ok = false; break; }
        tc::fence_after_sync();
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.out + (static_cast<size_t>(tok) * p.Hq + h) * D;
      store_o_rows<D>(o_addr, n < 1, inv, orow, valid, lane);
      if (valid && p.lse != nullptr)
        p.lse[static_cast<size_t>(tok) * p.Hq + h] =
            l > 0.f ? (m_used * c2 + lg2(l)) * kLn2 : kNegInf;
      g += n;
    }
  }

  // a warp that left its loop early may still have TMEM loads or stores in flight
  tc::tmem_wait_ld();
  tc::tmem_wait_st();
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag) {
    // a wait gave up: let every issued copy land before the CTA's shared
    // memory goes away (a left-out tile's phase never completes: bounded)
    if (qi_prod > 0) mbar_drain(q_full, (qi_prod - 1) & 1);
    for (int i = max(0, g_prod - NST); i < g_prod; ++i) mbar_drain(&kv_full[i % NST], (i / NST) & 1);
  }
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// NT query tiles per CTA, in both launches.
template <int D, int NST, int NT>
static int launch_tc(const AttnArgs& a, bool persistent, cudaStream_t stream) {
  static_assert(NT >= 2, "tiles per CTA");
  using C = TcCfg<D, NST, NT>;
  const int G = a.Hq / a.Hkv;
  CUtensorMap tmQ, tmK, tmV;
  const int QB = 128 / G;
  int rc = make_q_tmap(&tmQ, a.q, static_cast<uint64_t>(a.total_q), a.Hq, D, G, QB);
  if (rc) return rc;
  const uint64_t rows = kv_map_rows(a);
  const int box = kv_box_rows(a, C::KT);
  rc = make_rows_tmap(&tmK, a.k, rows, D, box, 128);
  if (rc) return rc;
  rc = make_rows_tmap(&tmV, a.v, rows, D, box, 128);
  if (rc) return rc;

  TcParams p{};
  p.page_size = a.page_size;
  p.box_rows = box;
  p.page_indptr = a.page_indptr;
  p.page_indices = a.page_indices;
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.q_len = a.q_len;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = G;
  p.QB = QB;
  const int tiles = NT;   // query tiles per item
  p.nqb = (a.max_q + tiles * QB - 1) / (tiles * QB);
  p.batch = a.batch;
  const int64_t items = static_cast<int64_t>(p.nqb) * a.Hkv * a.batch;
  if (items >= (int64_t{1} << 31)) {
    set_error("too many prefill work items");
    return SINKATTN_UNSUPPORTED;
  }
  p.n_items = static_cast<int>(items);
  p.max_kv = a.max_kv;
  p.sm_scale = a.sm_scale;
  p.scale_log2 = a.sm_scale * kLog2e;
  p.causal = a.causal;
  p.window = a.window;
  p.sinks = a.sinks;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;

  auto kern = persistent ? prefill_tc_persistent_kernel<D, NST, NT> : prefill_tc_kernel<D, NST, NT>;
  const int smem = C::SMEM;
  const int threads = C::THREADS;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) {
    set_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    return SINKATTN_CUDA_ERROR;
  }
  if (p.n_items == 0) return SINKATTN_OK;
  const dim3 grid = persistent ? dim3(static_cast<unsigned>(std::min<int64_t>(items, sm_count())))
                               : dim3(static_cast<unsigned>(p.nqb), static_cast<unsigned>(a.Hkv),
                                      static_cast<unsigned>(a.batch));
  kern<<<grid, threads, smem, stream>>>(tmQ, tmK, tmV, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("prefill kernel launch: %s", cudaGetErrorString(e));
    return SINKATTN_CUDA_ERROR;
  }
  return SINKATTN_OK;
}

// Persistent CTAs pay off when items are short (a few KV tiles: a sliding
// window, short prompts), where the one-block-per-item launch spends much of
// its time starting and finishing blocks.
static bool prefer_persistent(const AttnArgs& a, int kt, int tiles) {
  const int G = a.Hq / a.Hkv;
  const int tokens = tiles * (128 / G);   // query tokens per item
  const long long keys = a.window > 0 ? static_cast<long long>(a.window) + tokens
                                      : (a.causal ? a.max_kv / 2 : a.max_kv);
  return keys <= 6LL * kt;
}

// Both launches run the same tiles per CTA (three at d 64, two at d 128), and
// the persistent one also wins when every SM gets many items, so that the
// snake order evens out their lengths: full-causal gpt-oss-shaped prefill
// 846 against 796 TFLOP/s, Qwen-shaped prefill (3000 items of 2 x 6000
// tokens) 1390 against 1340. With few long items per SM (1024 items of a
// 16-draft decode) the hardware's dynamic block dealing balances better
// (0.69 against 0.73 ms).
static bool many_items_per_sm(const AttnArgs& a, int tiles) {
  const int G = a.Hq / a.Hkv;
  const long long tokens = tiles * (128 / G);
  const long long items = (a.max_q + tokens - 1) / tokens * a.Hkv * a.batch;
  return items >= 16LL * sm_count();
}

int launch_prefill_tc(const AttnArgs& a, int kind, cudaStream_t stream) {
  const int G = a.Hq / a.Hkv;
  if (G > 128) {
    set_error("GQA group of %d query heads exceeds the 128 rows of a tile", G);
    return SINKATTN_UNSUPPORTED;
  }
  if (a.d == 64) {
    const bool pers = kind == SINKATTN_PREFILL_PERSISTENT ||
                      (kind == SINKATTN_PREFILL_AUTO &&
                       (prefer_persistent(a, TcCfg<64, 4, 3>::KT, 3) || many_items_per_sm(a, 3)));
    return launch_tc<64, 4, 3>(a, pers, stream);
  }
  const bool pers = kind == SINKATTN_PREFILL_PERSISTENT ||
                    (kind == SINKATTN_PREFILL_AUTO &&
                     (prefer_persistent(a, TcCfg<128, 2>::KT, 2) || many_items_per_sm(a, 2)));
  return launch_tc<128, 2, 2>(a, pers, stream);
}

SINKATTN_DEFINE_SET_HOOKS(set_hooks_prefill_tc)

int read_status_prefill_tc(cudaStream_t s, int* status) {
  int zero = 0;
  if (cudaMemcpyFromSymbolAsync(status, g_status_prefill_tc, sizeof(int), 0,
                                cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SINKATTN_CUDA_ERROR;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SINKATTN_CUDA_ERROR;
  if (cudaMemcpyToSymbolAsync(g_status_prefill_tc, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                              s) != cudaSuccess)
    return SINKATTN_CUDA_ERROR;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SINKATTN_CUDA_ERROR;
  return SINKATTN_OK;
}

}  // namespace sinkattn
