// Split-KV decode / MTP on the 5th-generation tensor cores, head_dim 128.
//
// Decoding is bound by HBM bandwidth ("Hosting Qwen on Blackwell", section
// "Decoders"), and with MTP drafts sharing a KV head (3 tokens x 16 query
// heads = 48 rows per Qwen3 KV head) every streamed KV byte costs 48
// multiply-adds -- more than the warp-level mma.sync path sustains at HBM
// speed on GB300. Here both products run on tcgen05 with a 128-row tile, the
// CTA's R = G x QB real rows in its first R lanes and the rest padding:
//
//   S = Q K^T   M 128 rows, N 64 keys, K 128 d   (both operands in shared memory)
//   O += P V    M 128 rows, N 128 d,  K 64 keys (P from TMEM, V from shared memory)
//
// One CTA = (sequence b, KV head, query block, KV chunk), as the warp-level
// split kernel, and it writes the same partials: the chunk's (m, d, acc)
// WITHOUT the sink, which the merge folds in once ("GPT-OSS on Day 0",
// section "Kernels for GPT-OSS / Sink attention").
//
//  * warps 0-3: softmax, one thread per row (= TMEM lane, so each warp may
//    only touch its own 32-lane quadrant): all 64 scores of a KV tile in
//    registers, so the row maximum and sum need no exchange between threads.
//    P goes back as bf16 into the first 32 columns of the same TMEM buffer.
//    O is rescaled in TMEM only when some row of the warp raised its maximum.
//  * warp 4: TMA producer -- Q once (a 3-D box of QB tokens x G heads), then
//    K/V tiles of 64 keys into an NST-stage ring, right-aligned to the end of
//    the chunk so no copy reads past the last key the CTA needs.
//  * warp 5: TMEM allocation and every MMA, from one thread. Two S buffers
//    alternate, so S(j+1) is computed while the softmax works on S(j):
//      S(0), S(1), then per tile j:  PV(j), [PV(j) done] S(j+2).
//
// The Q tile holds only R rows in shared memory; the MMA's other 128 - R
// rows read whatever follows (the ring), which only reaches padding lanes.
// TMEM: S0 | S1 | O = 64 + 64 + 128 of 256 columns, so two CTAs share an SM
// (shared memory admits at most two, and exactly two up to 48 rows), one
// streaming while the other is in its prologue or epilogue. The partial rows
// are staged in the (then idle) ring and written with coalesced stores.
// Every wait is bounded.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace sinkattn {

__device__ int g_status_decode_tc;

struct DtcParams {
  const int32_t* cu_k;
  int q_len, Hq, Hkv, G, QB, nqb, num_splits, max_kv;
  float sm_scale, scale_log2;
  int causal, window;
  float* part_acc;
  float* part_md;
};

template <int RR>
struct DtcCfg {
  static constexpr int D = 128;
  static constexpr int KT = 64;                 // keys per KV tile
  static constexpr int NST = 3;                 // ring stages
  static constexpr int SUB_KV = KT * 128;       // [64 keys][64 bf16], 128B-swizzled: 8 KB
  static constexpr int KV_TILE = 2 * SUB_KV;    // K or V of one tile, d 128
  static constexpr int STAGE = 2 * KV_TILE;     // K and V: 32 KB
  static constexpr int Q_SUB = RR * 128;        // [RR rows][64 bf16]
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = (2 * Q_SUB + 1023) / 1024 * 1024;
  static constexpr int OFF_BAR = OFF_RING + NST * STAGE;
  static constexpr int N_BARS = 1 + 2 * NST + 2 + 2 + 2 + 1;
  static constexpr int SMEM = 1024 + OFF_BAR + N_BARS * 8 + 64;
  static constexpr int THREADS = 6 * 32;
  static constexpr uint32_t TMEM_COLS = 256;
  static constexpr uint32_t COL_O = 2 * KT;
  static constexpr int XS = D + 4;              // staging row stride (floats)
  static_assert(RR % 8 == 0 && RR >= 8 && RR <= 128, "rows");
  // the A operand reads 128 rows from each Q sub-tile: keep them inside the allocation
  static_assert(OFF_Q + Q_SUB + 128 * 128 <= OFF_BAR, "Q over-read stays in shared memory");
  static_assert(RR * XS * 4 <= NST * STAGE, "partial staging fits in the ring");
  // at most two CTAs per SM, so two 256-column TMEM allocations always fit;
  // up to 48 rows exactly two fit
  static_assert(SMEM > 233472 / 3 - 1024 && SMEM <= 232448, "CTAs per SM");
  static_assert(RR > 48 || 2 * (SMEM + 1024) <= 233472, "two CTAs per SM");
};

template <int RR>
__global__ void __launch_bounds__(DtcCfg<RR>::THREADS, 2)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const DtcParams p) {
  using C = DtcCfg<RR>;
  constexpr int D = C::D, KT = C::KT, NST = C::NST;
  constexpr float NEG_INF = kNegInf;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* kv_full = q_full + 1;
  uint64_t* kv_empty = kv_full + NST;
  uint64_t* s_full = kv_empty + NST;   // [2]: S(j) written to buffer j & 1
  uint64_t* p_full = s_full + 2;       // [2]: P(j) written, O rescaled (128 arrivals)
  uint64_t* pv_done = p_full + 2;      // [2]: PV(j) completed
  uint64_t* drain = pv_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* status = &g_status_decode_tc;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.z;
  const int kvh = blockIdx.y;
  const int S = p.num_splits;
  const int split = blockIdx.x % S;
  const int qb = p.nqb - 1 - static_cast<int>(blockIdx.x / S);

  const int q_start = b * p.q_len;
  const int Lq = p.q_len;
  const int k_start = p.cu_k[b];
  const int Lk = p.cu_k[b + 1] - k_start;
  const int q0 = qb * p.QB;
  if (q0 >= Lq) return;   // uniform over the CTA, before any barrier or TMEM use
  const int nq = min(p.QB, Lq - q0);
  if (threadIdx.x == 0 && (Lk < Lq || Lk > p.max_kv)) atomicExch(status, SINKATTN_BAD_LENGTHS);
  const int pos0 = Lk - Lq + q0;
  const int posN = pos0 + nq - 1;
  const int chunk = (Lk + S - 1) / S;
  int k_lo = min(split * chunk, Lk);
  int k_hi = min(k_lo + chunk, Lk);
  if (p.causal) k_hi = min(k_hi, posN + 1);
  if (p.window > 0) k_lo = max(k_lo, pos0 - p.window + 1);
  const int n = (k_hi > k_lo) ? (k_hi - k_lo + KT - 1) / KT : 0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NST; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(2 * 128 * p.G * p.QB));
      for (int sub = 0; sub < 2; ++sub)
        tc::tma_load_3d(smem + C::OFF_Q + sub * C::Q_SUB, &tmQ, sub * 64, kvh * p.G,
                        q_start + q0, q_full);
      const uint64_t policy = policy_evict_first();   // K/V are streamed once
      const int slab = k_start * p.Hkv + kvh * Lk;     // tensor-map row of key 0
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int st = i % NST;
        if (!mbar_wait(&kv_empty[st], ((i / NST) & 1) ^ 1, abort_flag, status)) break;
        uint8_t* kt = smem + C::OFF_RING + st * C::STAGE;
        mbar_arrive_expect_tx(&kv_full[st], C::STAGE);
        const int row = slab + k_hi - (n - i) * KT;
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          tma_load_2d_hint(kt + sub * C::SUB_KV, &tmK, sub * 64, row, &kv_full[st], policy);
          tma_load_2d_hint(kt + C::KV_TILE + sub * C::SUB_KV, &tmV, sub * 64, row, &kv_full[st],
                           policy);
        }
        issued = i + 1;
      }
      if (*abort_flag) {   // let every copy land before the CTA's shared memory goes away
        mbar_drain(q_full, 0);
        for (int i = max(0, issued - NST); i < issued; ++i)
          mbar_drain(&kv_full[i % NST], (i / NST) & 1);
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(128, KT, false);
      constexpr uint32_t idesc_o = tc::idesc_bf16_f32(128, D, true);
      constexpr uint64_t STAGE16 = C::STAGE >> 4;   // descriptor address units
      // A K step (16 elements = 32 bytes) inside a 128-byte swizzle row adds 2
      // to the address field; the next 64-column block adds its sub-tile size.
      const uint64_t qd0 = tc::smem_desc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
      const uint64_t kd0 = tc::smem_desc_sw128(smem_u32(smem + C::OFF_RING), 16, 1024);
      // V as the MN-major B operand: d blocks of 64 one sub-tile apart, 8-key
      // groups 1024 bytes apart; 16 keys advance 2048 bytes.
      const uint64_t vd0 =
          tc::smem_desc_sw128(smem_u32(smem + C::OFF_RING + C::KV_TILE), C::SUB_KV, 1024);
      auto issue_s = [&](int j) {
        const uint64_t kd = kd0 + static_cast<uint64_t>(j % NST) * STAGE16;
        const uint32_t d_tm = tmem + static_cast<uint32_t>((j & 1) * KT);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t oq = static_cast<uint64_t>(kk >> 2) * (C::Q_SUB >> 4) + (kk & 3) * 2;
          const uint64_t ok = static_cast<uint64_t>(kk >> 2) * (C::SUB_KV >> 4) + (kk & 3) * 2;
          tc::mma_ss(d_tm, qd0 + oq, kd + ok, idesc_s, kk > 0 ? 1u : 0u);
        }
        tc::commit(&s_full[j & 1]);
      };
      auto issue_pv = [&](int j) {
        const uint64_t vd = vd0 + static_cast<uint64_t>(j % NST) * STAGE16;
        const uint32_t a_tm = tmem + static_cast<uint32_t>((j & 1) * KT);
#pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk)
          tc::mma_ts(tmem + C::COL_O, a_tm + kk * 8, vd + static_cast<uint64_t>(kk) * 128u,
                     idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        tc::commit(&pv_done[j & 1]);
        tc::commit(&kv_empty[j % NST]);
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, status);
      for (int j = 0; ok && j < min(n, 2); ++j) {
        ok = mbar_wait(&kv_full[j], 0, abort_flag, status);
        if (ok) {
          tc::fence_after_sync();
          issue_s(j);
        }
      }
      for (int j = 0; ok && j < n; ++j) {
        if (!mbar_wait(&p_full[j & 1], (j >> 1) & 1, abort_flag, status)) break;
        tc::fence_after_sync();
        issue_pv(j);
        if (j + 2 < n) {
          // S(j+2) overwrites P(j): wait until PV(j) has read it.
          if (!mbar_wait(&kv_full[(j + 2) % NST], ((j + 2) / NST) & 1, abort_flag, status) ||
              !mbar_wait(&pv_done[j & 1], (j >> 1) & 1, abort_flag, status))
            break;
          tc::fence_after_sync();
          issue_s(j + 2);
        }
      }
      // every MMA this thread issued has completed before the CTA frees TMEM
      tc::commit(drain);
      mbar_drain(drain, 0);
    }
  } else {
    // ---------------------------------------------------------------- softmax
    const int row = warp * 32 + lane;   // TMEM lane; warp w owns lanes 32w..32w+31
    const int G = p.G;
    const int tl = row / G;
    const bool valid = tl < nq;
    const int pos = pos0 + tl;
    int lo_r = k_lo, hi_r = k_hi - 1;
    if (p.window > 0) lo_r = max(lo_r, pos - p.window + 1);
    if (p.causal) hi_r = min(hi_r, pos);
    if (!valid) {   // padding lanes see no key: P = 0
      lo_r = 1;
      hi_r = 0;
    }
    const float c2 = p.scale_log2;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t o_addr = lane_base + C::COL_O;
    float m = NEG_INF, l = 0.f;   // running max (raw logits) and exact sum
    bool ok = true;
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, status));
    };

    for (int j = 0; j < n; ++j) {
      if (!wwait(&s_full[j & 1], (j >> 1) & 1)) { ok = false; break; }
      tc::fence_after_sync();
      const uint32_t s_addr = lane_base + static_cast<uint32_t>((j & 1) * KT);
      const int j0 = k_hi - (n - j) * KT;   // key of tile column 0
      float v[2][32];
      tc::tmem_ld32(s_addr, v[0]);
      tc::tmem_ld32(s_addr + 32, v[1]);
      tc::tmem_wait_ld();
      if (j0 < lo_r || j0 + KT - 1 > hi_r) {
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
        for (int e = 0; e < 32; ++e) mx4[e & 3] = fmaxf(mx4[e & 3], v[c][e]);
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      float alpha = 1.f;
      bool rescale = false;
      if (mx > m) {
        alpha = (m == NEG_INF) ? 0.f : ex2((m - mx) * c2);
        m = mx;
        rescale = true;
      }
      const float mb = (m == NEG_INF) ? 0.f : m * c2;
      float rs4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float a0 = ex2(fmaf(v[c][e], c2, -mb));
          const float a1 = ex2(fmaf(v[c][e + 1], c2, -mb));
          rs4[(e >> 1) & 3] += a0 + a1;
          pk[e >> 1] = pack_bf16x2(a0, a1);
        }
        // P columns [16c, 16c + 16) hold scores this thread already loaded
        tc::tmem_st16(s_addr + 16 * c, pk);
      }
      // O rescale (PV(j-1) must have completed; warp-uniform branch)
      if (j >= 1 && __any_sync(0xffffffffu, rescale)) {
        if (!wwait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1)) { ok = false; break; }
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
      tc::fence_before_sync();
      mbar_arrive(&p_full[j & 1]);
    }

    // ------------------------------------------------------------ epilogue
    if (ok && n >= 1) {
      ok = wwait(&pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1);
      tc::fence_after_sync();
    }
    // Every tile has been consumed and every PV has completed: the ring is
    // free and stages this CTA's partial rows for coalesced stores.
    float* stage = reinterpret_cast<float*>(smem + C::OFF_RING);
    const bool have_o = ok && n >= 1;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float o[32];
      if (have_o) {
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
              make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
      }
    }
    if (valid) {
      const size_t rowid =
          static_cast<size_t>(q_start + q0 + tl) * p.Hq + kvh * G + (row - tl * G);
      float2 md;
      md.x = (m == NEG_INF) ? NEG_INF : m * p.sm_scale;
      md.y = l;
      *reinterpret_cast<float2*>(p.part_md + (rowid * S + split) * 2) = md;
    }
    named_barrier_sync(1, 128);
    const int nrows = nq * G;
    for (int r = warp; r < nrows; r += 4) {
      const int t2 = r / G;
      const size_t rowid = static_cast<size_t>(q_start + q0 + t2) * p.Hq + kvh * G + (r - t2 * G);
      const float4 val = *reinterpret_cast<const float4*>(stage + r * C::XS + lane * 4);
      *reinterpret_cast<float4*>(p.part_acc + (rowid * S + split) * D + lane * 4) = val;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
template <int RR>
static int launch_dtc(const AttnArgs& a, int QB, cudaStream_t stream) {
  using C = DtcCfg<RR>;
  const int G = a.Hq / a.Hkv;
  CUtensorMap tmQ, tmK, tmV;
  int rc = make_q_tmap(&tmQ, a.q, static_cast<uint64_t>(a.batch) * a.q_len, a.Hq, C::D, G, QB);
  if (rc) return rc;
  const uint64_t rows = static_cast<uint64_t>(a.Hkv) * a.batch * a.max_kv;
  rc = make_rows_tmap(&tmK, a.k, rows, C::D, C::KT, 128);
  if (rc) return rc;
  rc = make_rows_tmap(&tmV, a.v, rows, C::D, C::KT, 128);
  if (rc) return rc;
  DtcParams p{};
  p.cu_k = a.cu_k;
  p.q_len = a.q_len;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = G;
  p.QB = QB;
  p.nqb = (a.q_len + QB - 1) / QB;
  p.num_splits = a.num_splits;
  p.max_kv = a.max_kv;
  p.sm_scale = a.sm_scale;
  p.scale_log2 = a.sm_scale * kLog2e;
  p.causal = a.causal;
  p.window = a.window;
  p.part_acc = a.part_acc;
  p.part_md = a.part_md;
  auto kern = decode_tc_kernel<RR>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) {
    set_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    return SINKATTN_CUDA_ERROR;
  }
  const dim3 grid(static_cast<unsigned>(p.nqb * p.num_splits), static_cast<unsigned>(a.Hkv),
                  static_cast<unsigned>(a.batch));
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
  return a.d == 128 && G >= 1 && G <= 128;
}

int launch_decode_tc(const AttnArgs& a, cudaStream_t stream) {
  const int G = a.Hq / a.Hkv;
  if (!decode_tc_supported(a)) {
    set_error("the tcgen05 decode kernel needs head_dim 128 and at most 128 heads per group");
    return SINKATTN_UNSUPPORTED;
  }
  const int QB = min(a.q_len, 128 / G);   // query tokens per CTA
  const int R = G * QB;                   // real rows of the 128-row tile
  if (R <= 16) return launch_dtc<16>(a, QB, stream);
  if (R <= 32) return launch_dtc<32>(a, QB, stream);
  if (R <= 48) return launch_dtc<48>(a, QB, stream);
  if (R <= 64) return launch_dtc<64>(a, QB, stream);
  return launch_dtc<128>(a, QB, stream);
}

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
