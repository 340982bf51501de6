// Split-KV decode / MTP on the 5th-generation tensor cores, head_dim 128.
//
// Decoding is bound by HBM bandwidth ("Hosting Qwen on Blackwell", section
// "Decoders"), and with MTP drafts sharing a KV head (3 tokens x 16 query
// heads = 48 rows per Qwen3 KV head) every streamed KV byte costs 48
// multiply-adds -- more than the warp-level mma.sync path sustains at HBM
// speed on GB300. Here both products run on tcgen05 with a 128-row tile, an
// item's R = G x QB real rows in its first R lanes and the rest padding:
//
//   S = Q K^T   M 128 rows, N 64 keys, K 128 d   (both operands in shared memory)
//   O += P V    M 128 rows, N 128 d,  K 64 keys (P from TMEM, V from shared memory)
//
// A work item is (sequence b, KV head, query block, KV chunk), as in the
// warp-level split kernel, and it writes the same partials: the chunk's
// (m, d, acc) WITHOUT the sink, which the merge folds in once ("GPT-OSS on
// Day 0", section "Kernels for GPT-OSS / Sink attention"). One persistent
// CTA per SM runs items back to back (warp roles, buffers and the schedule
// are described at the kernel below). The Q tile holds only RR rows in
// shared memory; the MMA's other 128 - RR rows read whatever follows, which
// only reaches padding lanes. Every wait is bounded.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace sinkattn {

__device__ int g_status_decode_tc;

struct DtcParams {
  const int32_t* cu_k;
  int batch;
  int q_len, Hq, Hkv, G, QB, nqb, num_splits, max_kv;
  int n_items;   // batch * Hkv * nqb * num_splits
  float sm_scale, scale_log2;
  int causal, window;
  float* part_acc;
  float* part_md;
  // paged KV (page_size > 0): page-pool rows, boxes of box_rows keys
  int page_size, box_rows;
  const int32_t* page_indptr;
  const int32_t* page_indices;
  // FP8 KV: per-KV-head scales of the e4m3 codes
  const float* k_scale;
  const float* v_scale;
};

// One work item: (sequence b, KV head, query block, KV chunk) and its keys.
struct DtcItem {
  int b, kvh, split, q_start, q0, nq, k_start, Lk, pos0, k_lo, k_hi, n;
  int first;   // key of tile 0's first column: tiles end at k_hi (contiguous) or
               // start on a multiple of the tile (paged, so boxes never straddle pages)
};

// cu_k is read from `cu` (a shared-memory copy when the batch fits, else
// global memory): every role derives every item's keys from it.
template <int KT, bool PAGED, bool ROTATE>
__device__ __forceinline__ DtcItem dtc_item(const DtcParams& p, const int32_t* cu, int it) {
  DtcItem t;
  const int S = p.num_splits;
  int r = it / S;
  // ROTATE: the chunk index rotates with the group, so the CTAs that take
  // every gridDim.x-th item see every chunk position (late chunks are often
  // short or empty: a fixed position per CTA leaves some CTAs idle). Measured
  // +4% on the bf16 MTP decode, -4% with FP8 KV (bound by per-tile work).
  t.split = ROTATE ? (it % S + r) % S : it % S;
  const int qb = p.nqb - 1 - r % p.nqb;   // longer query blocks first
  r /= p.nqb;
  t.kvh = r % p.Hkv;
  t.b = r / p.Hkv;
  t.q_start = t.b * p.q_len;
  t.q0 = qb * p.QB;
  t.nq = min(p.QB, p.q_len - t.q0);
  t.k_start = cu[t.b];
  t.Lk = cu[t.b + 1] - t.k_start;
  t.pos0 = t.Lk - p.q_len + t.q0;
  const int posN = t.pos0 + t.nq - 1;
  const int chunk = split_chunk(t.Lk, S);
  t.k_lo = min(t.split * chunk, t.Lk);
  t.k_hi = min(t.k_lo + chunk, t.Lk);
  if (p.causal) t.k_hi = min(t.k_hi, posN + 1);
  if (p.window > 0) t.k_lo = max(t.k_lo, t.pos0 - p.window + 1);
  if (PAGED) {
    const int t0 = t.k_lo / KT * KT;
    t.n = (t.k_hi > t.k_lo) ? (t.k_hi - t0 + KT - 1) / KT : 0;
    t.first = t0;
  } else {
    t.n = (t.k_hi > t.k_lo) ? (t.k_hi - t.k_lo + KT - 1) / KT : 0;
    t.first = t.k_hi - t.n * KT;
  }
  return t;
}

template <int RR, bool FP8 = false>
struct DtcCfg {
  static constexpr int D = 128;
  static constexpr int KT = 64;                 // keys per KV tile
  static constexpr int SUB_KV = KT * 128;       // [64 keys][64 bf16], 128B-swizzled: 8 KB
  static constexpr int KV_TILE = 2 * SUB_KV;    // K or V of one tile, d 128
  static constexpr int STAGE = 2 * KV_TILE;     // K and V: 32 KB
  static constexpr int Q_SUB = RR * 128;        // [RR rows][64 bf16]
  static constexpr int Q_BUF = 2 * Q_SUB;       // one item's Q (two 64-column blocks)
  static constexpr int XS = D + 4;              // staging row stride (floats)
  static constexpr int OFF_Q = 0;               // two Q buffers
  static constexpr int OFF_RING = (2 * Q_BUF + 1023) / 1024 * 1024;
  static constexpr int CU_CAP = 2048;           // sequences whose kv_indptr is staged in smem
  // FP8: a ring of e4m3 K/V code stages feeds the f16 tile ring
  static constexpr int CODE_STAGE = 2 * KT * D; // 16 KB
  static constexpr int NSTF = FP8 ? 2 : 0;   // (two code stages leave room for a deeper f16 ring)
  static constexpr int NSTF_MOD = FP8 ? NSTF : 1;   // (a non-zero modulus for the bf16 build)
  static constexpr int FIXED = OFF_RING + RR * XS * 4 + 2 * 128 * 16 + (CU_CAP + 1) * 4 + 16 +
                               (40 + 2 * NSTF + 2) * 8 + 64 + 1024 + NSTF * CODE_STAGE;
  static constexpr int NST = (232448 - FIXED) / STAGE < 6 ? (232448 - FIXED) / STAGE : 6;
  static constexpr int OFF_CODE = OFF_RING + NST * STAGE;  // FP8: [NSTF][K | V] codes
  static constexpr int OFF_STG = OFF_CODE + NSTF * CODE_STAGE;   // [RR][XS] fp32 partial rows
  static constexpr int OFF_ML = OFF_STG + RR * XS * 4;     // [2][128] (m, l, lr) per row
  static constexpr int OFF_CU = OFF_ML + 2 * 128 * 16;     // [CU_CAP + 1] kv_indptr copy
  static constexpr int OFF_BAR = OFF_CU + ((CU_CAP + 1) * 4 + 15) / 16 * 16;
  static constexpr int NSB = 4;                 // S buffers in TMEM
  static constexpr int N_BARS =
      2 + 2 + 2 * NST + 3 * NSB + 2 + 2 + 2 + 1 + (FP8 ? 2 * NSTF + 2 : 0);
  static constexpr int SMEM = 1024 + OFF_BAR + N_BARS * 8 + 64;
  // 12 warps. bf16: 0-3 softmax, 4-7 epilogue, 10 producer, 11 MMA. FP8 (at
  // most 64 rows, so TMEM lane quarters 0 and 1): 0-1 softmax, 2-3 and 10-11
  // convert (sub-partitions 2 and 3), 4-7 epilogue, 8 producer, 9 MMA.
  static constexpr int THREADS = 12 * 32;
  static constexpr int W_PROD = FP8 ? 8 : 10;
  static constexpr int W_MMA = FP8 ? 9 : 11;
  static constexpr int N_CVT = 4;               // FP8 converter warps
  static constexpr int N_SMX = FP8 ? 2 : 4;     // softmax warps
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_O = NSB * KT;   // O buffers at 256 and 384
  static_assert(COL_O + 2 * D <= TMEM_COLS, "TMEM budget");
  static_assert(RR % 8 == 0 && RR >= 8 && RR <= 128, "rows");
  static_assert(NST >= 2, "ring depth");
  static_assert(!FP8 || NST >= 3, "FP8: the f16 ring keeps three tiles for the S look-ahead");
  // S runs LA tiles ahead of PV: tile g + LA reuses tile g's ring stage at the
  // latest. FP8 keeps a stage of slack (LA = NST - 1), so the conversion of
  // tile g + LA starts when PV(g - 1) completes rather than PV(g).
  static constexpr int LA = FP8 ? NST - 1 : (NST < 3 ? NST : 3);
  // the A operand reads 128 rows from each Q sub-tile: keep them inside the allocation
  static_assert(OFF_Q + Q_BUF + Q_SUB + 128 * 128 <= OFF_BAR, "Q over-read stays in shared memory");
  // one CTA per SM, so the 512-column TMEM allocation always succeeds
  static_assert(SMEM <= 232448 && 2 * (SMEM + 1024) > 233472, "one CTA per SM");
};

// Persistent: CTA c runs items c, c + gridDim.x, ... back to back, so the
// ring keeps streaming across item boundaries. Warps 0-3 softmax (thread =
// row = TMEM lane), 4-7 epilogue (read O, write the partial), 10 TMA
// producer, 11 TMEM allocation + MMA issue (8, 9 idle for bf16 KV: the
// producer and the issuer sit on the SM sub-partitions of the softmax warps
// with the fewest real rows). Q and O are double-buffered by item; S has four
// buffers: the issuer keeps S three tiles ahead, issuing S(g+3) right after
// PV(g) (it reuses P(g-1)'s buffer, whose PV has completed by then), so the
// chain softmax -> PV -> S spans three tiles of softmax work. Tile g+3 takes
// tile g's ring stage at the latest, so a two-stage ring (128-row tiles)
// runs two tiles ahead instead.
//
// Lazy rescaling: a row's weights are taken relative to a reference maximum
// that moves only when a score exceeds it by more than 2^8 in exp2 units,
// so O is rarely rescaled (each rescale must wait for the previous PV) and
// weights stay below 256. Two sums are kept: l over the exact weights and
// lr over the bf16-rounded weights the MMA applies. The partial is written
// as (m', lr) with m' = m + ln(l / lr): m' + ln lr is the chunk's exact
// log-sum-exp and acc / lr its output normalised by the weights actually
// applied -- the same state, rescaled, as (chunk max, exact sum).
//
// FP8 KV (e4m3 codes with per-KV-head scales): the producer copies the codes
// into a ring of code stages; warps 2-3 and 10-11 (the sub-partitions
// without real softmax rows, as tiles have at most 64 rows) convert each
// item's Q in place to f16 and widen each tile's codes to f16 into the tile
// ring (the layout the MMAs read), and every MMA runs on f16 operands (P is
// packed as f16). The producer moves to warp 8 and the MMA issuer to 9. The
// key scale joins the item's logit scale, the value scale multiplies the
// staged accumulator. Rows are normalised by the exact weight sum: f16
// weights are within 2^-11 of it.
template <int RR, bool PAGED, bool FP8>
__global__ void __launch_bounds__(DtcCfg<RR, FP8>::THREADS, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const DtcParams p) {
  using C = DtcCfg<RR, FP8>;
  constexpr int D = C::D, KT = C::KT, NST = C::NST;
  constexpr float NEG_INF = kNegInf;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;              // [2] by non-empty item ordinal
  uint64_t* q_empty = q_full + 2;       // [2] the item's last S has completed
  uint64_t* kv_full = q_empty + 2;      // [NST] by tile ordinal
  uint64_t* kv_empty = kv_full + NST;
  uint64_t* s_full = kv_empty + NST;    // [4] S(g) in buffer g % 4
  uint64_t* p_full = s_full + 4;        // [4] P(g) written and O rescaled (128 arrivals)
  uint64_t* pv_done = p_full + 4;       // [4] PV(g) completed
  uint64_t* o_full = pv_done + 4;       // [2] by item: its last PV has completed
  uint64_t* o_free = o_full + 2;        // [2] by item: epilogue has read O and (m, l)
  uint64_t* ml_full = o_free + 2;       // [2] by item: softmax wrote (m, l) (128 arrivals)
  uint64_t* drain = ml_full + 2;
  uint64_t* c_full = drain + 1;         // FP8: [NSTF] codes of the stage landed
  uint64_t* c_empty = c_full + C::NSTF; // FP8: [NSTF] codes of the stage converted
  uint64_t* q_cvt = c_empty + C::NSTF;  // FP8: [2] the item's Q is f16
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_cvt + (FP8 ? 2 : 0));
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  float4* ml = reinterpret_cast<float4*>(smem + C::OFF_ML);
  int* status = &g_status_decode_tc;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_mine = (p.n_items - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                     static_cast<int>(gridDim.x);
  // kv_indptr in shared memory (global-memory loads under a saturated HBM
  // stream take microseconds, and every role needs every item's keys)
  int32_t* cu_s = reinterpret_cast<int32_t*>(smem + C::OFF_CU);
  const int n_cu = p.batch + 1;
  const bool cu_in_smem = n_cu <= C::CU_CAP + 1;
  if (cu_in_smem)
    for (int i = threadIdx.x; i < n_cu; i += blockDim.x) cu_s[i] = p.cu_k[i];
  const int32_t* cu = cu_in_smem ? cu_s : p.cu_k;
  auto item_of = [&](int k) {
    return dtc_item<KT, PAGED, !FP8>(p, cu, static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x));
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 32 * C::N_SMX);
      mbar_init(&pv_done[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_free[i], 128);
      mbar_init(&ml_full[i], 32 * C::N_SMX);
    }
    for (int i = 0; i < NST; ++i) {
      mbar_init(&kv_full[i], FP8 ? C::N_CVT : 1);   // FP8: the converter warps
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < C::NSTF; ++i) {
      mbar_init(&c_full[i], 1);
      mbar_init(&c_empty[i], C::N_CVT);
    }
    if (FP8)
      for (int i = 0; i < 2; ++i) mbar_init(&q_cvt[i], C::N_CVT);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == C::W_MMA) {
    tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, status));
  };
  int g_prod = 0, qi_prod = 0;   // producer: tiles and Q loads issued

  if (warp == C::W_PROD) {
    // ---------------------------------------------------------------- producer
    // Contiguous KV: lane 0 runs the loop alone. Paged KV: the whole warp runs
    // it (page lists are read 32 entries per warp load, lane i issues box i of
    // a tile) and lane 0 issues the other copies.
    const bool leader = (lane == 0);
    if (PAGED || leader) {
      auto pwait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if constexpr (PAGED) return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, status));
        else return mbar_wait(bar, parity, abort_flag, status);
      };
      if (leader) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
      }
      const uint64_t policy = policy_evict_first();   // K/V are streamed once
      [[maybe_unused]] PageCursor pc;
      int g = 0, qi = 0;                               // tile and non-empty item ordinals
      bool ok = true;
      const int skip_tile = hook_skip_tile();
      for (int k = 0; ok && k < n_mine; ++k) {
        const DtcItem t = item_of(k);
        if (leader && (t.Lk < p.q_len || t.Lk > p.max_kv)) atomicExch(status, SINKATTN_BAD_LENGTHS);
        if (t.n == 0) continue;
        if (!pwait(&q_empty[qi & 1], ((qi >> 1) & 1) ^ 1)) { ok = false; break; }
        if (leader) {
          mbar_arrive_expect_tx(&q_full[qi & 1], static_cast<uint32_t>(2 * 128 * p.G * p.QB));
          for (int sub = 0; sub < 2; ++sub)
            tc::tma_load_3d(smem + C::OFF_Q + (qi & 1) * C::Q_BUF + sub * C::Q_SUB, &tmQ,
                            sub * 64, t.kvh * p.G, t.q_start + t.q0, &q_full[qi & 1]);
        }
        ++qi;
        if constexpr (PAGED) {
          const int e0 = p.page_indptr[t.b];
          const int np = p.page_indptr[t.b + 1] - e0;
          if (leader && t.Lk > np * p.page_size) atomicExch(status, SINKATTN_BAD_LENGTHS);
          pc.start(p.page_indices + e0, np, t.first / p.page_size, lane);
        }
        const int slab = t.k_start * p.Hkv + t.kvh * t.Lk;   // contiguous: tensor-map row of key 0
        for (int j = 0; j < t.n; ++j, ++g) {
          const int j0 = t.first + j * KT;
          if constexpr (FP8) {
            // the tile's e4m3 codes into the code ring (the converters fill the tile ring)
            const int sc = g % C::NSTF_MOD;
            if (!pwait(&c_empty[sc], ((g / C::NSTF_MOD) & 1) ^ 1)) { ok = false; break; }
            if (g == skip_tile) continue;   // test hook: the waits for this tile run out
            uint8_t* codes = smem + C::OFF_CODE + sc * C::CODE_STAGE;
            if (leader) {
              mbar_arrive_expect_tx(&c_full[sc], C::CODE_STAGE);
              tma_load_2d_hint(codes, &tmK, 0, slab + j0, &c_full[sc], policy);
              tma_load_2d_hint(codes + KT * D, &tmV, 0, slab + j0, &c_full[sc], policy);
            }
            continue;
          }
          const int st = g % NST;
          if (!pwait(&kv_empty[st], ((g / NST) & 1) ^ 1)) { ok = false; break; }
          if (g == skip_tile) continue;   // test hook: the waits for this tile run out
          uint8_t* kt = smem + C::OFF_RING + st * C::STAGE;
          if (leader) mbar_arrive_expect_tx(&kv_full[st], C::STAGE);
          if constexpr (!PAGED) {
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
              tma_load_2d_hint(kt + sub * C::SUB_KV, &tmK, sub * 64, slab + j0, &kv_full[st],
                               policy);
              tma_load_2d_hint(kt + C::KV_TILE + sub * C::SUB_KV, &tmV, sub * 64, slab + j0,
                               &kv_full[st], policy);
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
              for (int sub = 0; sub < 2; ++sub) {
                tma_load_2d_hint(kt + sub * C::SUB_KV + off, &tmK, sub * 64, row, &kv_full[st],
                                 policy);
                tma_load_2d_hint(kt + C::KV_TILE + sub * C::SUB_KV + off, &tmV, sub * 64, row,
                                 &kv_full[st], policy);
              }
            }
          }
        }
      }
      g_prod = g;
      qi_prod = qi;
    }
  } else if (warp == C::W_MMA) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp runs the schedule (waits, cursors, descriptor arithmetic
    // stay warp-uniform) and one elected lane issues each MMA and commit.
    const bool leader = tc::elect_one();
    constexpr uint32_t idesc_s = FP8 ? tc::idesc_f16_f32(128, KT, false)
                                     : tc::idesc_bf16_f32(128, KT, false);
    constexpr uint32_t idesc_o = FP8 ? tc::idesc_f16_f32(128, D, true)
                                     : tc::idesc_bf16_f32(128, D, true);
    constexpr uint64_t STAGE16 = C::STAGE >> 4;   // descriptor address units
    // A K step (16 elements = 32 bytes) inside a 128-byte swizzle row adds 2
    // to the address field; the next 64-column block adds its sub-tile size.
    const uint64_t qd0 = tc::smem_desc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
    const uint64_t kd0 = tc::smem_desc_sw128(smem_u32(smem + C::OFF_RING), 16, 1024);
    // V as the MN-major B operand: d blocks of 64 one sub-tile apart, 8-key
    // groups 1024 bytes apart; 16 keys advance 2048 bytes.
    const uint64_t vd0 =
        tc::smem_desc_sw128(smem_u32(smem + C::OFF_RING + C::KV_TILE), C::SUB_KV, 1024);

    // S cursor: runs LA (three, or two with a two-stage ring) tiles ahead of the PV cursor.
    int sk = 0, sj = 0, sg = 0, sqi = 0;
    DtcItem st_ = n_mine > 0 ? item_of(0) : DtcItem{};
    auto s_skip_empty = [&]() {
      while (sk < n_mine && st_.n == 0) {
        ++sk;
        if (sk < n_mine) st_ = item_of(sk);
      }
    };
    auto issue_next_s = [&]() -> bool {
      // the item's Q has landed (FP8: and has been converted to f16)
      if (sj == 0 && !wwait(FP8 ? &q_cvt[sqi & 1] : &q_full[sqi & 1], (sqi >> 1) & 1)) return false;
      if (!wwait(&kv_full[sg % NST], (sg / NST) & 1)) return false;
      // S(sg) overwrites P(sg - 4): PV(sg - 4) must have read it
      if (sg >= 4 && !wwait(&pv_done[sg & 3], ((sg - 4) >> 2) & 1)) return false;
      tc::fence_after_sync();
      const uint64_t qd = qd0 + static_cast<uint64_t>(sqi & 1) * (C::Q_BUF >> 4);
      const uint64_t kd = kd0 + static_cast<uint64_t>(sg % NST) * STAGE16;
      const uint32_t d_tm = tmem + static_cast<uint32_t>((sg & 3) * KT);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t oq = static_cast<uint64_t>(kk >> 2) * (C::Q_SUB >> 4) + (kk & 3) * 2;
          const uint64_t ok = static_cast<uint64_t>(kk >> 2) * (C::SUB_KV >> 4) + (kk & 3) * 2;
          tc::mma_ss(d_tm, qd + oq, kd + ok, idesc_s, kk > 0 ? 1u : 0u);
        }
        tc::commit(&s_full[sg & 3]);
      }
      __syncwarp();
      ++sg;
      if (++sj == st_.n) {   // the item's last S: its Q buffer frees when this completes
        if (leader) tc::commit(&q_empty[sqi & 1]);
        __syncwarp();
        ++sqi;
        sj = 0;
        ++sk;
        if (sk < n_mine) st_ = item_of(sk);
        s_skip_empty();
      }
      return true;
    };

    bool ok = true;
    s_skip_empty();
    for (int w = 0; w < C::LA && ok && sk < n_mine; ++w) ok = issue_next_s();
    int g = 0;   // PV cursor: tile ordinal
    for (int k = 0; ok && k < n_mine; ++k) {
      const int n = item_of(k).n;
      // O buffer k & 1 is reused: the epilogue of item k - 2 has read it
      if (k >= 2 && !wwait(&o_free[k & 1], ((k - 2) >> 1) & 1)) {
        ok = false;
        break;
      }
      const uint32_t o_tm = tmem + C::COL_O + static_cast<uint32_t>((k & 1) * D);
      for (int j = 0; j < n; ++j, ++g) {
        if (!wwait(&p_full[g & 3], (g >> 2) & 1)) { ok = false; break; }
        tc::fence_after_sync();
        const uint64_t vd = vd0 + static_cast<uint64_t>(g % NST) * STAGE16;
        const uint32_t a_tm = tmem + static_cast<uint32_t>((g & 3) * KT);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < KT / 16; ++kk)
            tc::mma_ts(o_tm, a_tm + kk * 8, vd + static_cast<uint64_t>(kk) * 128u, idesc_o,
                       (j > 0 || kk > 0) ? 1u : 0u);
          tc::commit(&pv_done[g & 3]);
          tc::commit(&kv_empty[g % NST]);
        }
        __syncwarp();
        // S(g+LA) into P(g+LA-4)'s buffer: PV(g+LA-4) was issued at least a tile ago
        if (sk < n_mine && !issue_next_s()) { ok = false; break; }
      }
      if (!ok) break;
      if (leader) tc::commit(&o_full[k & 1]);   // also for an empty item: nothing to wait for
      __syncwarp();
    }
    // every MMA this warp issued has completed before the CTA frees TMEM
    if (leader) tc::commit(drain);
    __syncwarp();
    mbar_drain(drain, 0);
  } else if (FP8 && (warp == 2 || warp == 3 || warp == 10 || warp == 11)) {
    // ------------------------------------------------------------ converters
    // Per item: its Q in place, bf16 -> f16 (same swizzled positions); per
    // tile: 16-byte chunks of e4m3 codes -> f16 into the tile ring stage.
    // Generic-proxy writes the tensor core reads: fenced before each hand-over.
    constexpr int NT = C::N_CVT * 32;
    const int ct = ((warp < 4 ? warp - 2 : warp - 8) << 5) + lane;   // 0 .. NT - 1
    constexpr int CH_ROW = D / 16;          // 16-byte chunks per row of codes
    constexpr int CH_TILE = KT * CH_ROW;
    int g = 0, qi = 0;
    bool ok = true;
    for (int k = 0; ok && k < n_mine; ++k) {
      const DtcItem t = item_of(k);
      if (t.n == 0) continue;
      if (!wwait(&q_full[qi & 1], (qi >> 1) & 1)) break;
      uint8_t* qb = smem + C::OFF_Q + (qi & 1) * C::Q_BUF;
      for (int c = ct; c < C::Q_BUF / 16; c += NT) {
        uint4 w = *reinterpret_cast<const uint4*>(qb + c * 16);
        w.x = pack_f16x2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
        w.y = pack_f16x2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
        w.z = pack_f16x2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u));
        w.w = pack_f16x2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
        *reinterpret_cast<uint4*>(qb + c * 16) = w;
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_cvt[qi & 1]);
      ++qi;
      for (int j = 0; j < t.n; ++j, ++g) {
        const int sc = g % C::NSTF_MOD, st = g % NST;
        if (!wwait(&c_full[sc], (g / C::NSTF_MOD) & 1)) { ok = false; break; }
        const uint8_t* codes = smem + C::OFF_CODE + sc * C::CODE_STAGE;
        uint8_t* dst = smem + C::OFF_RING + st * C::STAGE;
        // all of this thread's codes into registers first (the loads do not
        // wait behind the stores), then the code stage is handed back
        constexpr int PER = 2 * CH_TILE / NT;
        uint4 w[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const int c = ct + i * NT;
          w[i] = *reinterpret_cast<const uint4*>(codes + c * 16);   // row-major [2][KT][D] codes
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&c_empty[sc]);
        if (!wwait(&kv_empty[st], ((g / NST) & 1) ^ 1)) { ok = false; break; }
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const int c = ct + i * NT;
          const int tensor = c / CH_TILE;   // 0: K, 1: V
          const int rem = c - tensor * CH_TILE;
          const int row = rem / CH_ROW, cb = rem - row * CH_ROW;
          uint4 h0, h1;
          h0.x = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i].x));
          h0.y = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i].x >> 16));
          h0.z = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i].y));
          h0.w = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i].y >> 16));
          h1.x = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i].z));
          h1.y = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i].z >> 16));
          h1.z = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i].w));
          h1.w = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i].w >> 16));
          // columns 16 cb .. 16 cb + 15: sub-tile cb / 4, 16-byte chunks 2 (cb % 4) and + 1
          // (lanes cb and cb + 4 of a row share bank groups; an order that
          // avoids it measured slower)
          uint8_t* sub = dst + tensor * C::KV_TILE + (cb >> 2) * C::SUB_KV;
          const int ch = (cb & 3) * 2;
          *reinterpret_cast<uint4*>(sub + sw128_offset(row, ch)) = h0;
          *reinterpret_cast<uint4*>(sub + sw128_offset(row, ch + 1)) = h1;
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&kv_full[st]);
      }
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------------- softmax
    const int row = warp * 32 + lane;   // TMEM lane; warp w owns lanes 32w..32w+31
    const int G = p.G;
    const int tl = row / G;
    const bool warp_rows = warp * 32 < p.G * p.QB;   // the warp holds a real row of some item
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    bool ok = true;
    int g = 0;
    for (int k = 0; ok && k < n_mine; ++k) {
      const DtcItem t = item_of(k);
      // raw logits -> base-2 exponents (FP8: the key scale of the item's head)
      const float c2 = p.scale_log2 * (FP8 ? p.k_scale[t.kvh] : 1.f);
      const bool valid = tl < t.nq;
      const int pos = t.pos0 + tl;
      int lo_r = t.k_lo, hi_r = t.k_hi - 1;
      if (p.window > 0) lo_r = max(lo_r, pos - p.window + 1);
      if (p.causal) hi_r = min(hi_r, pos);
      const uint32_t o_addr = lane_base + C::COL_O + static_cast<uint32_t>((k & 1) * D);
      // reference maximum (raw logits), exact and rounded weight sums
      float m = NEG_INF, l = 0.f, lr = 0.f;
      for (int j = 0; j < t.n; ++j, ++g) {
        if (!wwait(&s_full[g & 3], (g >> 2) & 1)) { ok = false; break; }
        if (!warp_rows) {   // padding rows only: nothing to compute, keep the barriers' count
          mbar_arrive(&p_full[g & 3]);
          continue;
        }
        tc::fence_after_sync();
        const uint32_t s_addr = lane_base + static_cast<uint32_t>((g & 3) * KT);
        const int j0 = t.first + j * KT;   // key of tile column 0
        float v[2][32];
        tc::tmem_ld32(s_addr, v[0]);
        tc::tmem_ld32(s_addr + 32, v[1]);
        tc::tmem_wait_ld();
        // (padding lanes skip the mask: their weights are zeroed below)
        if (valid && (j0 < lo_r || j0 + KT - 1 > hi_r)) {
          const int clo = lo_r - j0, chi = hi_r - j0;
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c * 32 + e < clo || c * 32 + e > chi) v[c][e] = NEG_INF;
        }
        float mx4[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            mx4[(e >> 1) & 3] = fmax3(mx4[(e >> 1) & 3], v[c][e], v[c][e + 1]);
        const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        float alpha = 1.f;
        bool rescale = false;
        if (valid && (m == NEG_INF ? mx > m : (mx - m) * c2 > 8.f)) {
          alpha = (m == NEG_INF) ? 0.f : ex2((m - mx) * c2);
          m = mx;
          rescale = true;
        }
        // padding lanes: an infinite offset makes every weight 0 (their S rows
        // are garbage; only their own P and O rows see it)
        const float mb = !valid ? INFINITY : (m == NEG_INF) ? 0.f : m * c2;
        float rs4[4] = {0.f, 0.f, 0.f, 0.f};
        float rr4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float a0 = ex2(fmaf(v[c][e], c2, -mb));
            const float a1 = ex2(fmaf(v[c][e + 1], c2, -mb));
            rs4[(e >> 1) & 3] += a0 + a1;
            if constexpr (FP8) {
              pk[e >> 1] = pack_f16x2(a0, a1);   // (normalised by the exact sum)
            } else {
              pk[e >> 1] = pack_bf16x2(a0, a1);
              rr4[(e >> 1) & 3] += bf16x2_sum(pk[e >> 1]);
            }
          }
          // P columns [16c, 16c + 16) hold scores this thread already loaded
          tc::tmem_st16(s_addr + 16 * c, pk);
        }
        // O rescale (rare): PV(g - 1) of this item must have completed; warp-uniform
        if (j >= 1 && __any_sync(0xffffffffu, rescale)) {
          if (!wwait(&pv_done[(g - 1) & 3], ((g - 1) >> 2) & 1)) { ok = false; break; }
          tc::fence_after_sync();
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
        l = l * alpha + ((rs4[0] + rs4[1]) + (rs4[2] + rs4[3]));
        if constexpr (FP8) lr = l;
        else lr = lr * alpha + ((rr4[0] + rr4[1]) + (rr4[2] + rr4[3]));
        tc::fence_before_sync();
        mbar_arrive(&p_full[g & 3]);
      }
      if (!ok) break;
      // hand (m, l) to the epilogue once it is done with item k - 2's
      if (k >= 2 && !wwait(&o_free[k & 1], ((k - 2) >> 1) & 1)) { ok = false; break; }
      ml[(k & 1) * 128 + row] = make_float4(m, l, lr, 0.f);
      mbar_arrive(&ml_full[k & 1]);
    }
  } else if (warp < 8) {
    // ---------------------------------------------------------------- epilogue
    const int quad = warp - 4;
    const int row = quad * 32 + lane;
    const int G = p.G;
    const int tl = row / G;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    float* stage = reinterpret_cast<float*>(smem + C::OFF_STG);
    const int S = p.num_splits;
    const uint64_t keep_policy = policy_evict_last();
    for (int k = 0; k < n_mine; ++k) {
      const DtcItem t = item_of(k);
      if (!wwait(&o_full[k & 1], (k >> 1) & 1) || !wwait(&ml_full[k & 1], (k >> 1) & 1)) break;
      tc::fence_after_sync();
      const float4 mlr = ml[(k & 1) * 128 + row];
      const uint32_t o_addr = lane_base + C::COL_O + static_cast<uint32_t>((k & 1) * D);
      const float vscale = FP8 ? p.v_scale[t.kvh] : 1.f;   // accumulator -> value units
      const float lscale = FP8 ? p.sm_scale * p.k_scale[t.kvh] : p.sm_scale;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        if (t.n >= 1) {
          tc::tmem_ld32(o_addr + c * 32, o);
          tc::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0.f;
        }
        if (row < RR) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(stage + row * C::XS + c * 32 + e) =
                make_float4(o[e] * vscale, o[e + 1] * vscale, o[e + 2] * vscale, o[e + 3] * vscale);
        }
      }
      tc::fence_before_sync();
      mbar_arrive(&o_free[k & 1]);
      if (tl < t.nq) {
        const size_t rowid =
            static_cast<size_t>(t.q_start + t.q0 + tl) * p.Hq + t.kvh * G + (row - tl * G);
        // (m', lr): m' + ln lr = m + ln l, the chunk's exact log-sum-exp
        float2 md;
        if (mlr.x == NEG_INF || !(mlr.z > 0.f)) {
          md = make_float2(NEG_INF, 0.f);
        } else {
          md.x = mlr.x * lscale + (lg2(mlr.y) - lg2(mlr.z)) * kLn2;
          md.y = mlr.z;
        }
        *reinterpret_cast<float2*>(p.part_md + (rowid * S + t.split) * 2) = md;
      }
      named_barrier_sync(1, 128);   // staging written
      const int nrows = t.nq * G;
      for (int r = quad; r < nrows; r += 4) {
        const int t2 = r / G;
        const size_t rowid =
            static_cast<size_t>(t.q_start + t.q0 + t2) * p.Hq + t.kvh * G + (r - t2 * G);
        const float4 val = *reinterpret_cast<const float4*>(stage + r * C::XS + lane * 4);
        // kept in L2 as long as possible: the merge reads the newest partials first
        asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(
                         p.part_acc + (rowid * S + t.split) * D + lane * 4),
                     "f"(val.x), "f"(val.y), "f"(val.z), "f"(val.w), "l"(keep_policy)
                     : "memory");
      }
      named_barrier_sync(1, 128);   // staging read before the next item overwrites it
    }
  }

  // a warp that left its loop early may still have TMEM loads or stores in flight
  tc::tmem_wait_ld();
  tc::tmem_wait_st();
  tc::fence_before_sync();
  __syncthreads();
  if (warp == C::W_PROD && lane == 0 && *abort_flag) {
    // a wait gave up: let every issued copy land before the CTA's shared
    // memory goes away (a left-out tile's phase never completes: bounded)
    for (int i = max(0, qi_prod - 2); i < qi_prod; ++i) mbar_drain(&q_full[i & 1], (i >> 1) & 1);
    if constexpr (FP8) {
      for (int i = max(0, g_prod - C::NSTF_MOD); i < g_prod; ++i)
        mbar_drain(&c_full[i % C::NSTF_MOD], (i / C::NSTF_MOD) & 1);
    } else {
      for (int i = max(0, g_prod - NST); i < g_prod; ++i)
        mbar_drain(&kv_full[i % NST], (i / NST) & 1);
    }
  }
  // this CTA's partials are written: a dependent merge may start launching
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == C::W_MMA) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
template <int RR, bool PAGED, bool FP8 = false>
static int launch_dtc(const AttnArgs& a, int QB, cudaStream_t stream) {
  using C = DtcCfg<RR, FP8>;
  const int G = a.Hq / a.Hkv;
  CUtensorMap tmQ, tmK, tmV;
  int rc = make_q_tmap(&tmQ, a.q, static_cast<uint64_t>(a.batch) * a.q_len, a.Hq, C::D, G, QB);
  if (rc) return rc;
  const uint64_t rows = kv_map_rows(a);
  const int box = kv_box_rows(a, C::KT);
  rc = FP8 ? make_rows_tmap_u8(&tmK, a.k, rows, C::D, box)
           : make_rows_tmap(&tmK, a.k, rows, C::D, box, 128);
  if (rc) return rc;
  rc = FP8 ? make_rows_tmap_u8(&tmV, a.v, rows, C::D, box)
           : make_rows_tmap(&tmV, a.v, rows, C::D, box, 128);
  if (rc) return rc;
  DtcParams p{};
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.page_size = a.page_size;
  p.box_rows = box;
  p.page_indptr = a.page_indptr;
  p.page_indices = a.page_indices;
  p.cu_k = a.cu_k;
  p.batch = a.batch;
  p.q_len = a.q_len;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = G;
  p.QB = QB;
  p.nqb = (a.q_len + QB - 1) / QB;
  p.num_splits = a.num_splits;
  const int64_t items = static_cast<int64_t>(a.batch) * a.Hkv * p.nqb * a.num_splits;
  if (items >= (int64_t{1} << 31)) {
    set_error("too many work items");
    return SINKATTN_UNSUPPORTED;
  }
  p.n_items = static_cast<int>(items);
  p.max_kv = a.max_kv;
  p.sm_scale = a.sm_scale;
  p.scale_log2 = a.sm_scale * kLog2e;
  p.causal = a.causal;
  p.window = a.window;
  p.part_acc = a.part_acc;
  p.part_md = a.part_md;
  auto kern = decode_tc_kernel<RR, PAGED, FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) {
    set_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    return SINKATTN_CUDA_ERROR;
  }
  if (p.n_items == 0) return SINKATTN_OK;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(items, sm_count()));
  kern<<<grid, C::THREADS, C::SMEM, stream>>>(tmQ, tmK, tmV, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("decode kernel launch: %s", cudaGetErrorString(e));
    return SINKATTN_CUDA_ERROR;
  }
  return SINKATTN_OK;
}

bool decode_tc_supported(const AttnArgs& a) {
  const int G = a.Hq / a.Hkv;
  // FP8 (contiguous KV only): tiles of at most 64 rows, so the code ring fits
  if (a.kv_fp8) return a.d == 128 && G >= 1 && G <= 64 && a.page_size == 0;
  return a.d == 128 && G >= 1 && G <= 128;
}

int launch_decode_tc(const AttnArgs& a, cudaStream_t stream) {
  const int G = a.Hq / a.Hkv;
  if (!decode_tc_supported(a)) {
    set_error("the tcgen05 decode kernel needs head_dim 128 and at most 128 heads per group");
    return SINKATTN_UNSUPPORTED;
  }
  if (a.kv_fp8) {
    const int QB = min(a.q_len, 64 / G);  // at most 64 rows per tile
    const int R = G * QB;
    if (R <= 16) return launch_dtc<16, false, true>(a, QB, stream);
    if (R <= 32) return launch_dtc<32, false, true>(a, QB, stream);
    if (R <= 48) return launch_dtc<48, false, true>(a, QB, stream);
    return launch_dtc<64, false, true>(a, QB, stream);
  }
  const int QB = min(a.q_len, 128 / G);   // query tokens per CTA
  const int R = G * QB;                   // real rows of the 128-row tile
  if (a.page_size > 0) {
    if (R <= 16) return launch_dtc<16, true>(a, QB, stream);
    if (R <= 32) return launch_dtc<32, true>(a, QB, stream);
    if (R <= 48) return launch_dtc<48, true>(a, QB, stream);
    if (R <= 64) return launch_dtc<64, true>(a, QB, stream);
    return launch_dtc<128, true>(a, QB, stream);
  }
  if (R <= 16) return launch_dtc<16, false>(a, QB, stream);
  if (R <= 32) return launch_dtc<32, false>(a, QB, stream);
  if (R <= 48) return launch_dtc<48, false>(a, QB, stream);
  if (R <= 64) return launch_dtc<64, false>(a, QB, stream);
  return launch_dtc<128, false>(a, QB, stream);
}

SINKATTN_DEFINE_SET_HOOKS(set_hooks_decode_tc)

int read_status_decode_tc(cudaStream_t s, int* status) {
  int zero = 0;
  if (cudaMemcpyFromSymbolAsync(status, g_status_decode_tc, sizeof(int), 0,
                                cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SINKATTN_CUDA_ERROR;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SINKATTN_CUDA_ERROR;
  if (cudaMemcpyToSymbolAsync(g_status_decode_tc, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                              s) != cudaSuccess)
    return SINKATTN_CUDA_ERROR;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SINKATTN_CUDA_ERROR;
  return SINKATTN_OK;
}

}  // namespace sinkattn
