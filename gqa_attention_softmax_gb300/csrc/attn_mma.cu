// Split-KV decode / MTP attention with a per-head softmax sink, on the
// warp-level tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate).
//
// Decode is bound by HBM bandwidth ("Hosting Qwen on Blackwell", section
// "Decoders": decoding is memory-bound), so this kernel is built to stream
// each (sequence, KV head) slab of the HND cache exactly once:
//
//  * One CTA = (sequence b, KV head, query block, KV chunk). Its rows are
//    (query token, head-in-group) pairs packed 16 per warp tile, so one K/V
//    tile in shared memory serves the whole GQA group and every MTP draft.
//  * A producer warp streams K and V tiles with TMA (128-byte swizzled boxes)
//    into an NST-stage mbarrier ring; consumer warps own one 16-row tile each
//    and split the KV tiles of the chunk round-robin into TG token groups.
//  * Per tile: S = Q K^T on mma.sync, mask, online softmax (running max and
//    sum per row, max reduced over the 4-lane quads with warp shuffles),
//    O += P V with P re-packed to bf16 straight from the S accumulators.
//  * FP8 KV (e4m3 codes, per-KV-head scales): the producer's TMA copies the
//    raw codes into the stage ring (K and V codes swizzled in 16-byte
//    chunks), and both products read their fragments straight from the
//    codes, widened to f16 in registers (exact: f16 holds every e4m3 value).
//    S: one 32-bit load of four adjacent K codes per fragment, with the head
//    dimensions of Q's fragments relabelled to match (q . k is unchanged).
//    P.V: ldmatrix's transposed 8-bit load hands each lane four consecutive
//    keys of a V column, which become the B fragment's k-slots (2c, 2c + 1,
//    2c + 8, 2c + 9); S is computed with its key columns permuted to the
//    same order, so P's fragments need no change (a sum over keys does not
//    depend on their order). Q is converted to f16 once. The key scale joins
//    the logit scale, the value scale multiplies the chunk's accumulator.
//  * Tiles are right-aligned to the end of the CTA's key range, so no copy
//    ever reads past the last key the CTA needs; keys before the range that a
//    tile covers are masked (and are real data or TMA zero-fill, never NaN).
//
// Output, split mode: the chunk's (m, d, acc) WITHOUT the sink, to HBM; the
// merge kernel seeds with the sink so it counts exactly once ("GPT-OSS on
// Day 0", section "Kernels for GPT-OSS / Sink attention": online softmax with
// a running max, the sink in one block only when the sequence is split).
//
// Output, fused mode: the S chunks of one (sequence, KV head, query block)
// form a thread-block cluster. Each CTA leaves its partial in its own shared
// memory; after a cluster barrier, CTA r folds rows r, r + S, ... of all S
// partials read through distributed shared memory, seeded with the sink, and
// writes out and lse; a second cluster barrier keeps every CTA's shared
// memory alive until its peers have read it. No partials go to HBM.
#include <cstdio>

#include "common.cuh"
#include "internal.h"

namespace sinkattn {

__device__ int g_status_attn_mma;

struct MmaParams {
  const __nv_bfloat16* q;
  const int32_t* cu_q;
  const int32_t* cu_k;
  int q_len;
  int Hq, Hkv, G;
  int QB;          // query tokens per CTA
  int nqb;         // query blocks per sequence in the grid
  int num_splits;
  int max_kv;
  float sm_scale, scale_log2;
  int causal, window;
  float* part_acc;
  float* part_md;
  const float* sinks;     // fused mode
  __nv_bfloat16* out;     // fused mode
  float* lse;             // fused mode
  // paged KV (page_size > 0): page-pool rows, boxes of box_rows keys
  int page_size, box_rows;
  const int32_t* page_indptr;
  const int32_t* page_indices;
  // FP8 KV: per-KV-head scales of the e4m3 codes
  const float* k_scale;
  const float* v_scale;
};

template <int D, int RT, int TG, int KT, int NST, bool FP8 = false>
struct MmaCfg {
  static constexpr int NW = RT * TG;               // consumer warps
  static constexpr int THREADS = (NW + 1) * 32;    // + producer warp
  static constexpr int NSUB = D / 64;              // 64-column sub-tiles
  static constexpr int SUB_BYTES = KT * 128;
  static constexpr int TILE_BYTES = NSUB * SUB_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int F8_TILE = KT * D;           // one K or V tile of e4m3 codes
  static constexpr int F8_STAGE = 2 * F8_TILE;
  // bf16: the stage ring of tiles; FP8: the ring of e4m3 stages
  static constexpr int OFF_F8 = FP8 ? 0 : NST * STAGE_BYTES;
  static constexpr int OFF_BAR = OFF_F8 + (FP8 ? NST * F8_STAGE : 0);
  static constexpr int XCHG_FLOATS_PER_LANE = D / 2 + 4;
  static constexpr int XCHG_BYTES = (TG - 1) * RT * 32 * XCHG_FLOATS_PER_LANE * 4;
  static constexpr int BAR_BYTES = 2 * NST * 8 + 16;
  static constexpr int SMEM_BYTES = 1024 + OFF_BAR + BAR_BYTES + XCHG_BYTES;
  // fused mode: one CTA's partial, [16 RT rows][m, d, pad, pad, acc[D]], over the tile ring
  static constexpr int XOUT_STRIDE = D + 4;
  static_assert(FP8 || 16 * RT * XOUT_STRIDE * 4 <= NST * STAGE_BYTES,
                "partial fits in the tile ring");
  // Token group tg takes tiles tg, tg + TG, ...; tile i lives in stage i % NST
  // with barrier phase (i / NST) % 2. Each stage must serve one group only,
  // which consumes its tiles in order: a stage shared by two groups lets one
  // of them wait for a tile two phases ahead while the stage's previous tile
  // is still in flight, and the parity wait would pass on the wrong phase.
  static_assert(NST % TG == 0, "every ring stage serves one token group");
  // Two resident CTAs per SM: one CTA's prologue (barrier set-up, first TMA
  // round trip, Q fragments) and epilogue overlap the other's streaming.
  static constexpr int MIN_CTAS = 2;
};

template <int D, int RT, int TG, int KT, int NST, bool FUSED, bool FP8>
__global__ void __launch_bounds__(MmaCfg<D, RT, TG, KT, NST, FP8>::THREADS,
                                  MmaCfg<D, RT, TG, KT, NST, FP8>::MIN_CTAS)
    attn_mma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const MmaParams p) {
  using C = MmaCfg<D, RT, TG, KT, NST, FP8>;
  constexpr int NW = C::NW;
  constexpr float NEG_INF = kNegInf;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* tiles = smem;                 // bf16: stage ring
  uint8_t* f8 = smem + C::OFF_F8;        // FP8: e4m3 stage ring [NST][K | V]
  // bf16: full / empty of the stage ring; FP8: codes landed / codes read
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + NST;
  int* abort_flag = reinterpret_cast<int*>(empty + NST);
  float* xchg = reinterpret_cast<float*>(smem + C::OFF_BAR + C::BAR_BYTES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.z;
  const int kvh = blockIdx.y;
  const int S = p.num_splits;
  const int split = blockIdx.x % S;
  const int qb = p.nqb - 1 - static_cast<int>(blockIdx.x / S);   // longest query blocks first

  const int q_start = p.cu_q ? p.cu_q[b] : b * p.q_len;
  const int Lq = p.cu_q ? p.cu_q[b + 1] - q_start : p.q_len;
  const int k_start = p.cu_k[b];
  const int Lk = p.cu_k[b + 1] - k_start;
  const int q0 = qb * p.QB;
  if (q0 >= Lq) return;   // uniform over the CTA (and the cluster), before any barrier
  const int nq = min(p.QB, Lq - q0);
  if (threadIdx.x == 0 && (Lk < Lq || Lk > p.max_kv || Lq < 0))
    atomicExch(&g_status_attn_mma, SINKATTN_BAD_LENGTHS);

  // Positions of the CTA's first and last query (queries are the last Lq keys).
  const int pos0 = Lk - Lq + q0;
  const int posN = pos0 + nq - 1;

  // Key range [k_lo, k_hi) this CTA must visit.
  const int chunk = split_chunk(Lk, S);
  int k_lo = min(split * chunk, Lk);
  int k_hi = min(k_lo + chunk, Lk);
  if (p.causal) k_hi = min(k_hi, posN + 1);
  if (p.window > 0) k_lo = max(k_lo, pos0 - p.window + 1);
  // Tiles end at k_hi (contiguous: no copy reads past the last key needed),
  // or start on a multiple of KT (paged: no box straddles a page).
  const bool paged = p.page_size > 0;
  const int t0 = k_lo / KT * KT;
  const int ntiles = (k_hi > k_lo) ? (k_hi - (paged ? t0 : k_lo) + KT - 1) / KT : 0;
  const int first = paged ? t0 : k_hi - ntiles * KT;   // key of tile 0's first row

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], RT);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // ------------------------------------------------------------------ producer
  bool writer = false;   // consumer warps holding the CTA's combined state
  if (warp == NW) {
    // Contiguous KV: lane 0 runs the loop alone. Paged KV: the whole warp runs
    // it (page lists are read 32 entries per warp load, lane i issues box i of
    // a tile).
    const bool leader = (lane == 0);
    if (ntiles > 0 && (paged || leader)) {
      const unsigned members = paged ? 0xffffffffu : 1u;
      if (leader) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
      }
      const uint64_t policy = policy_evict_first();
      const int slab = k_start * p.Hkv + kvh * Lk;   // contiguous: tensor-map row of key 0
      PageCursor pc;
      if (paged) {
        const int e0 = p.page_indptr[b];
        const int np = p.page_indptr[b + 1] - e0;
        if (leader && Lk > np * p.page_size) atomicExch(&g_status_attn_mma, SINKATTN_BAD_LENGTHS);
        pc.start(p.page_indices + e0, np, first / p.page_size, lane);
      }
      int issued = 0;
      const int skip_tile = hook_skip_tile();
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % NST;
        const uint32_t ph = static_cast<uint32_t>(i / NST) & 1u;
        const int j0 = first + i * KT;
        if constexpr (FP8) {
          // e4m3 codes into the code ring
          if (!__all_sync(members, mbar_wait(&empty[st], ph ^ 1u, abort_flag, &g_status_attn_mma)))
            break;
          if (i == skip_tile) {   // test hook: the waits for this tile run out
            issued = i + 1;
            continue;
          }
          uint8_t* kc = f8 + st * C::F8_STAGE;
          uint8_t* vc = kc + C::F8_TILE;
          if (leader) mbar_arrive_expect_tx(&full[st], C::F8_STAGE);
          if (!paged) {
            tma_load_2d_hint(kc, &tmK, 0, slab + j0, &full[st], policy);
            tma_load_2d_hint(vc, &tmV, 0, slab + j0, &full[st], policy);
          } else {
            const int nbox = KT / p.box_rows;
            const int a = j0 + min(lane, nbox - 1) * p.box_rows;
            const int page = pc.get(j0 / p.page_size, a / p.page_size, lane);
            if (lane < nbox) {
              const int row = (page * p.Hkv + kvh) * p.page_size + a % p.page_size;
              const int off = (a - j0) * D;
              tma_load_2d_hint(kc + off, &tmK, 0, row, &full[st], policy);
              tma_load_2d_hint(vc + off, &tmV, 0, row, &full[st], policy);
            }
          }
          issued = i + 1;
          continue;
        }
        if (!__all_sync(members, mbar_wait(&empty[st], ph ^ 1u, abort_flag, &g_status_attn_mma)))
          break;
        if (i == skip_tile) {   // test hook: the waits for this tile run out
          issued = i + 1;
          continue;
        }
        uint8_t* kt = tiles + st * C::STAGE_BYTES;
        uint8_t* vt = kt + C::TILE_BYTES;
        if (leader) mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
        if (!paged) {
#pragma unroll
          for (int sub = 0; sub < C::NSUB; ++sub) {
            tma_load_2d_hint(kt + sub * C::SUB_BYTES, &tmK, sub * 64, slab + j0, &full[st], policy);
            tma_load_2d_hint(vt + sub * C::SUB_BYTES, &tmV, sub * 64, slab + j0, &full[st], policy);
          }
        } else {
          // one box per page segment, lane i issuing box i: rows (page,
          // head, slot) of the pool
          const int nbox = KT / p.box_rows;
          const int a = j0 + min(lane, nbox - 1) * p.box_rows;
          const int page = pc.get(j0 / p.page_size, a / p.page_size, lane);
          if (lane < nbox) {
            const int row = (page * p.Hkv + kvh) * p.page_size + a % p.page_size;
            const int off = (a - j0) * 128;
#pragma unroll
            for (int sub = 0; sub < C::NSUB; ++sub) {
              tma_load_2d_hint(kt + sub * C::SUB_BYTES + off, &tmK, sub * 64, row, &full[st], policy);
              tma_load_2d_hint(vt + sub * C::SUB_BYTES + off, &tmV, sub * 64, row, &full[st], policy);
            }
          }
        }
        issued = i + 1;
      }
      // Let every issued copy land before this warp exits: the kernel has no
      // final block-wide barrier, and when a wait gives up (the abort flag
      // may be set after this loop ends) the consumers leave without reading
      // every tile. A copy the consumers read has long landed, so this costs
      // nothing otherwise; a left-out tile's phase never completes (bounded).
      if (leader)
        for (int i = max(0, issued - NST); i < issued; ++i)
          mbar_drain(&full[i % NST], static_cast<uint32_t>(i / NST) & 1u);
    }
  } else {
  // ------------------------------------------------------------------ consumers
  const int rt = warp % RT;
  const int tg = warp / RT;
  const int G = p.G;

  int pos[2], tok[2], head[2];
  bool valid[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = rt * 16 + (lane >> 2) + 8 * i;
    const int tl = r / G;
    valid[i] = tl < nq;
    pos[i] = pos0 + tl;
    tok[i] = q_start + q0 + tl;
    head[i] = kvh * G + (r - tl * G);
  }

  // Q fragments (A operand, row-major 16 x 16 per k-step), loaded once.
  // FP8: the k-slots (2c, 2c + 1, 2c + 8, 2c + 9) of lane c = lane % 4 hold
  // head dims 4c .. 4c + 3 of each 16-dim step, the relabelling under which
  // the K fragment is one 32-bit load of four adjacent codes; q . k is a sum
  // over the head dims, so the same relabelling on both operands leaves it
  // unchanged.
  uint32_t qa[D / 16][4];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
    for (int reg = 0; reg < 4; ++reg) {
      const int i = reg & 1;
      const int col = FP8 ? kk * 16 + (lane & 3) * 4 + ((reg >> 1) << 1)
                          : kk * 16 + (lane & 3) * 2 + ((reg >> 1) << 3);
      uint32_t qv = valid[i]
                        ? *reinterpret_cast<const uint32_t*>(
                              p.q + (static_cast<size_t>(tok[i]) * p.Hq + head[i]) * D + col)
                        : 0u;
      if constexpr (FP8)   // f16 operands: bf16 -> f32 (exact) -> f16
        qv = pack_f16x2(__uint_as_float(qv << 16), __uint_as_float(qv & 0xffff0000u));
      qa[kk][reg] = qv;
    }
  }

  // Running state per row, in raw logit units (before sm_scale).
  float m[2], l[2];
  float o[D / 8][4];
#pragma unroll
  for (int jd = 0; jd < D / 8; ++jd) o[jd][0] = o[jd][1] = o[jd][2] = o[jd][3] = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    m[i] = NEG_INF;
    l[i] = 0.f;
  }

  // logits in raw units q . k (k the e4m3 value with FP8 KV); c2 turns them
  // into base-2 exponents
  const float kscale = FP8 ? p.k_scale[kvh] : 1.f;
  const float c2 = p.scale_log2 * kscale;
  for (int i = tg; i < ntiles; i += TG) {
    const int st = i % NST;
    const uint32_t ph = static_cast<uint32_t>(i / NST) & 1u;
    uint32_t kbase = 0;
    if constexpr (FP8) {
      if (!__all_sync(0xffffffffu, mbar_wait(&full[st], ph, abort_flag, &g_status_attn_mma))) break;
    } else {
      if (!mbar_wait(&full[st], ph, abort_flag, &g_status_attn_mma)) break;
      kbase = smem_u32(tiles + st * C::STAGE_BYTES);
    }
    const uint32_t vbase = kbase + C::TILE_BYTES;
    const int j0 = first + i * KT;   // key index of tile row 0

    float s[KT / 8][4];
#pragma unroll
    for (int j = 0; j < KT / 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;

    // S = Q K^T
    if constexpr (FP8) {
      // K fragments straight from the e4m3 codes: one 32-bit load of four
      // codes (head dims 4c .. 4c + 3 of the step, lane c = lane % 4) per key
      // column and 16-dim step, widened to the two f16 pairs of the B
      // fragment in the relabelled order the Q fragments use. Block j of S
      // holds, in column n, key 16 (j / 2) + kr(n) + 2 (j % 2) with
      // kr(n) = 2n - (n % 2): the order in which the P.V product below takes
      // its V fragments.
      // The code rows are swizzled: 16-byte chunk k of key row r sits at chunk
      // k ^ ((r / 2) % 4) (64-byte rows) or k ^ (r % 8) (128-byte rows); for
      // r = 16 i + kr(lane / 4) + 2 (j % 2) that is a constant of the lane.
      const int kr = 2 * (lane >> 2) - ((lane >> 2) & 1);
      int xr[2];
      const uint8_t* kc[2];
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const int r = kr + 2 * blk;
        xr[blk] = D == 64 ? ((r >> 1) & 3) : (r & 7);
        kc[blk] = f8 + st * C::F8_STAGE + r * D + (lane & 3) * 4;
      }
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int j = 0; j < KT / 8; ++j) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(kc[j & 1] + 16 * (j >> 1) * D +
                                                                ((kk ^ xr[j & 1]) << 4));
          mma_f16_16816(s[j], qa[kk], e4m3x2_to_f16x2(static_cast<uint16_t>(w)),
                        e4m3x2_to_f16x2(static_cast<uint16_t>(w >> 16)));
        }
      }
    } else
#pragma unroll
    for (int kk = 0; kk < D / 16; kk += 2) {
#pragma unroll
      for (int j = 0; j < KT / 8; ++j) {
        const int trow = 8 * j + (lane & 7);
        const int chunk = 2 * kk + (lane >> 3);
        uint32_t bf[4];
        ldsm_x4(bf, kbase + (chunk >> 3) * C::SUB_BYTES + sw128_offset(trow, chunk & 7));
        if constexpr (FP8) {
          mma_f16_16816(s[j], qa[kk], bf[0], bf[1]);
          mma_f16_16816(s[j], qa[kk + 1], bf[2], bf[3]);
        } else {
          mma_bf16_16816(s[j], qa[kk], bf[0], bf[1]);
          mma_bf16_16816(s[j], qa[kk + 1], bf[2], bf[3]);
        }
      }
    }

    // Mask (skipped for tiles that every row sees whole).
    const bool whole = (j0 >= k_lo) && (j0 + KT <= k_hi) && (!p.causal || j0 + KT - 1 <= pos0) &&
                       (p.window <= 0 || j0 > posN - p.window);
    if (!whole) {
#pragma unroll
      for (int j = 0; j < KT / 8; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = FP8 ? j0 + 16 * (j >> 1) + 4 * (lane & 3) + 2 * (j & 1) + (e & 1)
                              : j0 + 8 * j + (lane & 3) * 2 + (e & 1);
          const int ps = pos[e >> 1];
          const bool vis = key >= k_lo && key < k_hi && (!p.causal || key <= ps) &&
                           (p.window <= 0 || key > ps - p.window);
          if (!vis) s[j][e] = NEG_INF;
        }
      }
    }

    // Online softmax.
    float mx[2] = {m[0], m[1]};
#pragma unroll
    for (int j = 0; j < KT / 8; ++j) {
      mx[0] = fmaxf(mx[0], fmaxf(s[j][0], s[j][1]));
      mx[1] = fmaxf(mx[1], fmaxf(s[j][2], s[j][3]));
    }
    float sc[2], alpha[2];
#pragma unroll
    for (int i2 = 0; i2 < 2; ++i2) {
      mx[i2] = fmaxf(mx[i2], __shfl_xor_sync(0xffffffffu, mx[i2], 1));
      mx[i2] = fmaxf(mx[i2], __shfl_xor_sync(0xffffffffu, mx[i2], 2));
      alpha[i2] = (mx[i2] == NEG_INF) ? 1.f : ex2((m[i2] - mx[i2]) * c2);
      sc[i2] = (mx[i2] == NEG_INF) ? 0.f : mx[i2] * c2;
      m[i2] = mx[i2];
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < KT / 8; ++j) {
      s[j][0] = ex2(fmaf(s[j][0], c2, -sc[0]));
      s[j][1] = ex2(fmaf(s[j][1], c2, -sc[0]));
      s[j][2] = ex2(fmaf(s[j][2], c2, -sc[1]));
      s[j][3] = ex2(fmaf(s[j][3], c2, -sc[1]));
      rs[0] += s[j][0] + s[j][1];
      rs[1] += s[j][2] + s[j][3];
    }
    l[0] = l[0] * alpha[0] + rs[0];
    l[1] = l[1] * alpha[1] + rs[1];
#pragma unroll
    for (int jd = 0; jd < D / 8; ++jd) {
      o[jd][0] *= alpha[0];
      o[jd][1] *= alpha[0];
      o[jd][2] *= alpha[1];
      o[jd][3] *= alpha[1];
    }

    // O += P V
#pragma unroll
    for (int kt2 = 0; kt2 < KT / 16; ++kt2) {
      uint32_t a[4];
      if constexpr (FP8) {
        a[0] = pack_f16x2(s[2 * kt2][0], s[2 * kt2][1]);
        a[1] = pack_f16x2(s[2 * kt2][2], s[2 * kt2][3]);
        a[2] = pack_f16x2(s[2 * kt2 + 1][0], s[2 * kt2 + 1][1]);
        a[3] = pack_f16x2(s[2 * kt2 + 1][2], s[2 * kt2 + 1][3]);
      } else {
        a[0] = pack_bf16x2(s[2 * kt2][0], s[2 * kt2][1]);
        a[1] = pack_bf16x2(s[2 * kt2][2], s[2 * kt2][3]);
        a[2] = pack_bf16x2(s[2 * kt2 + 1][0], s[2 * kt2 + 1][1]);
        a[3] = pack_bf16x2(s[2 * kt2 + 1][2], s[2 * kt2 + 1][3]);
      }
      if constexpr (FP8) {
        // V fragments straight from the codes: the transposed 8-bit load of
        // keys 16 kt2 .. + 15 x columns 16 jd2 .. + 15 gives lane (g, c) keys
        // 4c .. 4c + 3 of columns g and g + 8, the k-slots (2c, 2c + 1,
        // 2c + 8, 2c + 9) of the B fragments in the key order of S above.
        // Lanes 0-15 address the 16 key rows (swizzled like K's).
        const int vr = lane & 15;
        const int vxr = D == 64 ? ((vr >> 1) & 3) : (vr & 7);
        const uint8_t* vrow = f8 + st * C::F8_STAGE + C::F8_TILE + (16 * kt2 + vr) * D;
#pragma unroll
        for (int jd2 = 0; jd2 < D / 16; ++jd2) {
          uint32_t r0, r1;
          ldsm_b8_trans(r0, r1, smem_u32(vrow + ((jd2 ^ vxr) << 4)));
          mma_f16_16816(o[2 * jd2], a, e4m3x2_to_f16x2(static_cast<uint16_t>(r0)),
                        e4m3x2_to_f16x2(static_cast<uint16_t>(r0 >> 16)));
          mma_f16_16816(o[2 * jd2 + 1], a, e4m3x2_to_f16x2(static_cast<uint16_t>(r1)),
                        e4m3x2_to_f16x2(static_cast<uint16_t>(r1 >> 16)));
        }
      } else {
#pragma unroll
        for (int jd = 0; jd < D / 8; jd += 2) {
          const int mi = lane >> 3;
          const int trow = 16 * kt2 + (mi & 1) * 8 + (lane & 7);
          const int chunk = jd + (mi >> 1);
          uint32_t bf[4];
          ldsm_x4_trans(bf, vbase + (chunk >> 3) * C::SUB_BYTES + sw128_offset(trow, chunk & 7));
          mma_bf16_16816(o[jd], a, bf[0], bf[1]);
          mma_bf16_16816(o[jd + 1], a, bf[2], bf[3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);   // this warp has read the tile
  }

  // Row sums are split over the 4 lanes of each quad.
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l[i] += __shfl_xor_sync(0xffffffffu, l[i], 1);
    l[i] += __shfl_xor_sync(0xffffffffu, l[i], 2);
  }

  // Combine the token groups of each row tile.
  if (TG > 1) {
    if (tg > 0) {
      float* slot = xchg + ((tg - 1) * RT + rt) * 32 * C::XCHG_FLOATS_PER_LANE +
                    lane * C::XCHG_FLOATS_PER_LANE;
#pragma unroll
      for (int jd = 0; jd < D / 8; ++jd)
#pragma unroll
        for (int e = 0; e < 4; ++e) slot[jd * 4 + e] = o[jd][e];
      slot[D / 2 + 0] = m[0];
      slot[D / 2 + 1] = m[1];
      slot[D / 2 + 2] = l[0];
      slot[D / 2 + 3] = l[1];
    }
    named_barrier_sync(1, NW * 32);
  }
  writer = (tg == 0);
  if (TG > 1 && writer) {
#pragma unroll 1
    for (int t = 1; t < TG; ++t) {
      const float* slot = xchg + ((t - 1) * RT + rt) * 32 * C::XCHG_FLOATS_PER_LANE +
                          lane * C::XCHG_FLOATS_PER_LANE;
      float a0[2], a1[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float m2 = slot[D / 2 + i];
        const float l2 = slot[D / 2 + 2 + i];
        const float mn = fmaxf(m[i], m2);
        a0[i] = (m[i] == NEG_INF) ? 0.f : ex2((m[i] - mn) * c2);
        a1[i] = (m2 == NEG_INF) ? 0.f : ex2((m2 - mn) * c2);
        l[i] = l[i] * a0[i] + l2 * a1[i];
        m[i] = mn;
      }
#pragma unroll
      for (int jd = 0; jd < D / 8; ++jd) {
        o[jd][0] = o[jd][0] * a0[0] + slot[jd * 4 + 0] * a1[0];
        o[jd][1] = o[jd][1] * a0[0] + slot[jd * 4 + 1] * a1[0];
        o[jd][2] = o[jd][2] * a0[1] + slot[jd * 4 + 2] * a1[1];
        o[jd][3] = o[jd][3] * a0[1] + slot[jd * 4 + 3] * a1[1];
      }
    }
  }

  // ------------------------------------------------------------------ epilogue
  if (!FUSED && writer) {
    // FP8: the value scale turns the accumulator into value units
    const float vscale = FP8 ? p.v_scale[kvh] : 1.f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (!valid[i]) continue;
      const size_t rowid = static_cast<size_t>(tok[i]) * p.Hq + head[i];
      float* arow = p.part_acc + (rowid * S + split) * D;
#pragma unroll
      for (int jd = 0; jd < D / 8; ++jd) {
        const int col = jd * 8 + (lane & 3) * 2;
        *reinterpret_cast<float2*>(arow + col) =
            make_float2(o[jd][2 * i] * vscale, o[jd][2 * i + 1] * vscale);
      }
      if ((lane & 3) == 0) {
        float2 md;
        md.x = (m[i] == NEG_INF) ? NEG_INF : m[i] * (p.sm_scale * kscale);
        md.y = l[i];
        *reinterpret_cast<float2*>(p.part_md + (rowid * S + split) * 2) = md;
      }
    }
  }
  if (FUSED && writer) {
    // this CTA's partial (raw-logit m, d, acc) into its own shared memory; the
    // tile ring is free: every tile has been consumed
    float* xout = reinterpret_cast<float*>(tiles);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = rt * 16 + (lane >> 2) + 8 * i;
      float* xr = xout + r * C::XOUT_STRIDE;
#pragma unroll
      for (int jd = 0; jd < D / 8; ++jd) {
        const int col = jd * 8 + (lane & 3) * 2;
        *reinterpret_cast<float2*>(xr + 4 + col) = make_float2(o[jd][2 * i], o[jd][2 * i + 1]);
      }
      if ((lane & 3) == 0) {
        xr[0] = m[i];
        xr[1] = l[i];
      }
    }
  }
  }   // consumers

  if (FUSED) {
    cluster_sync_all();
    // Fold rows rank, rank + S, ... over the S partials of the cluster, seeded
    // with the sink (the sink counts once). One consumer warp per row; lane s
    // reads peer s's (m, d); each lane owns D/32 output columns.
    constexpr int VEC = D / 32;
    const float* xout = reinterpret_cast<const float*>(tiles);
    const uint32_t rank = static_cast<uint32_t>(split);
    if (warp < NW) {
      const float c2 = p.scale_log2;
      for (int r = static_cast<int>(rank) + S * warp; r < 16 * RT; r += S * NW) {
        const int tl = r / p.G;
        if (tl >= nq) continue;
        const int tk = q_start + q0 + tl;
        const int hh = kvh * p.G + (r - tl * p.G);
        const float* xr = xout + r * C::XOUT_STRIDE;
        float ms = NEG_INF, ls = 0.f;
        if (lane < S) {
          ms = ld_dsmem(xr + 0, static_cast<uint32_t>(lane));
          ls = ld_dsmem(xr + 1, static_cast<uint32_t>(lane));
        }
        float M = ms;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float sk = p.sinks ? p.sinks[hh] : NEG_INF;
        const float sink_raw = (sk == NEG_INF) ? NEG_INF : sk / p.sm_scale;
        M = fmaxf(M, sink_raw);
        const float ws = (ms == NEG_INF) ? 0.f : ex2((ms - M) * c2);
        float L = ws * ls;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
        if (sink_raw != NEG_INF) L += ex2((sink_raw - M) * c2);
        float acc[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
        for (int s2 = 0; s2 < S; ++s2) {
          const float w = __shfl_sync(0xffffffffu, ws, s2);
          if (w == 0.f) continue;
          float v[VEC];
          ld_dsmem_vec<VEC>(xr + 4 + lane * VEC, static_cast<uint32_t>(s2), v);
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[e] = fmaf(w, v[e], acc[e]);
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        __nv_bfloat16* orow = p.out + (static_cast<size_t>(tk) * p.Hq + hh) * D + lane * VEC;
        if constexpr (VEC == 4) {
          uint2 pk;
          pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
          pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
          *reinterpret_cast<uint2*>(orow) = pk;
        } else {
          *reinterpret_cast<uint32_t*>(orow) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        }
        if (p.lse != nullptr && lane == 0)
          p.lse[static_cast<size_t>(tk) * p.Hq + hh] = L > 0.f ? (M * c2 + lg2(L)) * kLn2 : NEG_INF;
      }
    }
    cluster_sync_all();   // peers may still be reading this CTA's partial
  }
  // split mode: this thread's partial writes are issued; a dependent merge
  // may start launching (it waits for the whole grid before reading)
  if (!FUSED) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int D, int RT, int TG, int KT, int NST, bool FUSED, bool FP8>
static int launch_cfg(const AttnArgs& a, cudaStream_t stream) {
  using C = MmaCfg<D, RT, TG, KT, NST, FP8>;
  CUtensorMap tmK, tmV;
  const uint64_t rows = kv_map_rows(a);
  const int box = kv_box_rows(a, KT);
  // FP8: K and V codes land swizzled (16-byte chunks over the D-byte row), so
  // the S product's 32-bit fragment loads and the P.V product's transposed
  // 16-row loads are free of bank conflicts.
  int rc = FP8 ? make_rows_tmap_u8(&tmK, a.k, rows, D, box, D) : make_rows_tmap(&tmK, a.k, rows, D, box, 128);
  if (rc) return rc;
  rc = FP8 ? make_rows_tmap_u8(&tmV, a.v, rows, D, box, D) : make_rows_tmap(&tmV, a.v, rows, D, box, 128);
  if (rc) return rc;

  MmaParams p{};
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.q_len = a.q_len;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.Hq / a.Hkv;
  p.QB = (a.q_len * p.G <= 16 * RT) ? a.q_len : (16 * RT) / p.G;
  const int maxq = a.cu_q ? a.max_q : a.q_len;
  p.nqb = (maxq + p.QB - 1) / p.QB;
  p.num_splits = a.num_splits;
  p.max_kv = a.max_kv;
  p.sm_scale = a.sm_scale;
  p.scale_log2 = a.sm_scale * kLog2e;
  p.causal = a.causal;
  p.window = a.window;
  p.part_acc = a.part_acc;
  p.part_md = a.part_md;
  p.page_size = a.page_size;
  p.box_rows = box;
  p.page_indptr = a.page_indptr;
  p.page_indices = a.page_indices;
  p.sinks = a.sinks;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;

  auto kern = attn_mma_kernel<D, RT, TG, KT, NST, FUSED, FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) {
    set_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    return SINKATTN_CUDA_ERROR;
  }
  const dim3 grid(static_cast<unsigned>(p.nqb * p.num_splits), static_cast<unsigned>(a.Hkv),
                  static_cast<unsigned>(a.batch));
  if (FUSED) {
    // the S chunks of one (sequence, KV head, query block) form a cluster
    if (p.num_splits > 8) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) {
        set_error("cluster size %d not allowed: %s", p.num_splits, cudaGetErrorString(e));
        return SINKATTN_UNSUPPORTED;
      }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.num_splits);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, tmK, tmV, p);
  } else {
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tmK, tmV, p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_error("attention kernel launch: %s", cudaGetErrorString(e));
    return SINKATTN_CUDA_ERROR;
  }
  return SINKATTN_OK;
}

template <bool FUSED, bool FP8>
static int launch_attn_mma_t(const AttnArgs& a, cudaStream_t stream) {
  const int G = a.Hq / a.Hkv;
  const int rows = G * a.q_len;
  const int rt_needed = (rows + 15) / 16;
  if (G > 64) {
    set_error("GQA group of %d query heads exceeds 64 rows per CTA", G);
    return SINKATTN_UNSUPPORTED;
  }
  // stages of the ring: an FP8 stage holds half the bytes of a bf16 one, so
  // twice as many keep the same bytes in flight per SM
  constexpr int NS = FP8 ? 8 : 4;
  if (a.d == 64) {
    if (rt_needed <= 1) return launch_cfg<64, 1, 4, 64, NS, FUSED, FP8>(a, stream);
    if (rt_needed <= 2) return launch_cfg<64, 2, 2, 64, NS, FUSED, FP8>(a, stream);
    if (rt_needed <= 3) return launch_cfg<64, 3, 2, 64, NS, FUSED, FP8>(a, stream);
    return launch_cfg<64, 4, 2, 64, NS, FUSED, FP8>(a, stream);
  }
  if (rt_needed <= 1) return launch_cfg<128, 1, 4, 32, NS, FUSED, FP8>(a, stream);
  if (rt_needed <= 2) return launch_cfg<128, 2, 2, 32, NS, FUSED, FP8>(a, stream);
  if (rt_needed <= 3) return launch_cfg<128, 3, 2, 32, NS, FUSED, FP8>(a, stream);
  return launch_cfg<128, 4, 2, 32, NS, FUSED, FP8>(a, stream);
}

int launch_attn_mma(const AttnArgs& a, cudaStream_t stream) {
  return a.kv_fp8 ? launch_attn_mma_t<false, true>(a, stream)
                  : launch_attn_mma_t<false, false>(a, stream);
}

int launch_attn_mma_fused(const AttnArgs& a, cudaStream_t stream) {
  return launch_attn_mma_t<true, false>(a, stream);
}

SINKATTN_DEFINE_SET_HOOKS(set_hooks_attn_mma)

int read_status_attn_mma(cudaStream_t s, int* status) {
  int zero = 0;
  if (cudaMemcpyFromSymbolAsync(status, g_status_attn_mma, sizeof(int), 0,
                                cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SINKATTN_CUDA_ERROR;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SINKATTN_CUDA_ERROR;
  if (cudaMemcpyToSymbolAsync(g_status_attn_mma, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                              s) != cudaSuccess)
    return SINKATTN_CUDA_ERROR;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SINKATTN_CUDA_ERROR;
  return SINKATTN_OK;
}

}  // namespace sinkattn
