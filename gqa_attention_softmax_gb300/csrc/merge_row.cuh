// Fold of one (row, query head)'s split-KV partials with the sink counted
// exactly once, by one warp ("GPT-OSS on Day 0", section "Kernels for
// GPT-OSS / Sink attention": the sink belongs to one block only when the
// sequence is split). With M the maximum of the sink and every chunk's m_s:
//   w_s = e^{m_s - M},  D = e^{s_h - M} + sum_s w_s d_s,
//   out = sum_s w_s acc_s / D,  lse = M + ln D
// (the sink term is absent without a sink; an empty chunk has m_s = -inf).
// Lane s computes w_s; every lane owns D/32 output columns and reads each
// chunk's accumulator slice with one vector load. Up to 16 chunks, all loads
// (the (m, d) pairs and every slice) are in flight at once, one memory round
// trip per row; beyond that, eight slices at a time after a pass over the
// maxima. Partials are read once, through L2 only (ld.global.cg).
#pragma once

#include "common.cuh"

namespace sinkattn {

template <int D>
__device__ __forceinline__ void merge_row(const float* md, const float* acc, float sink, int S,
                                          int lane, __nv_bfloat16* orow, float* lse_out) {
  constexpr int VEC = D / 32;   // 2 or 4 floats per lane
  constexpr float NEG_INF = kNegInf;
  float o[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) o[e] = 0.f;
  float M = sink, dpart = 0.f;
  if (S <= 16) {
    // one round trip: lane s's (m_s, d_s) and every chunk's accumulator
    // slice are loaded together; the weights follow from the maximum
    const float2 mdl = lane < S ? __ldcg(reinterpret_cast<const float2*>(md + 2 * lane))
                                : make_float2(NEG_INF, 0.f);
    float a[16][VEC];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      if (u < S) {
        const float* src = acc + u * D + lane * VEC;
        if constexpr (VEC == 4) {
          const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
          a[u][0] = t.x; a[u][1] = t.y; a[u][2] = t.z; a[u][3] = t.w;
        } else {
          const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
          a[u][0] = t.x; a[u][1] = t.y;
        }
      }
    }
    M = fmaxf(M, mdl.x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float w = 0.f;
    if (mdl.x != NEG_INF) {
      w = ex2((mdl.x - M) * kLog2e);
      dpart = mdl.y * w;
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const float wu = __shfl_sync(0xffffffffu, w, u);
      if (u < S) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = fmaf(a[u][e], wu, o[e]);
      }
    }
  } else {
    for (int s = lane; s < S; s += 32) M = fmaxf(M, __ldcg(md + 2 * s));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    for (int s0 = 0; s0 < S; s0 += 32) {
      float w = 0.f;
      if (s0 + lane < S) {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(md + 2 * (s0 + lane)));
        if (v.x != NEG_INF) {
          w = ex2((v.x - M) * kLog2e);
          dpart = fmaf(v.y, w, dpart);
        }
      }
      const int cnt = min(32, S - s0);
      for (int i = 0; i < cnt; i += 8) {
        float a[8][VEC];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (i + u < cnt) {
            const float* src = acc + (s0 + i + u) * D + lane * VEC;
            if constexpr (VEC == 4) {
              const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
              a[u][0] = t.x; a[u][1] = t.y; a[u][2] = t.z; a[u][3] = t.w;
            } else {
              const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
              a[u][0] = t.x; a[u][1] = t.y;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float wu = __shfl_sync(0xffffffffu, w, (i + u) & 31);
          if (i + u < cnt) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) o[e] = fmaf(a[u][e], wu, o[e]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dpart += __shfl_xor_sync(0xffffffffu, dpart, off);
  const float dsum = dpart + ((sink == NEG_INF) ? 0.f : ex2((sink - M) * kLog2e));
  const float inv = dsum > 0.f ? 1.f / dsum : 0.f;
  __nv_bfloat16* op = orow + lane * VEC;
  if constexpr (VEC == 4) {
    uint2 pk;
    pk.x = pack_bf16x2(o[0] * inv, o[1] * inv);
    pk.y = pack_bf16x2(o[2] * inv, o[3] * inv);
    *reinterpret_cast<uint2*>(op) = pk;
  } else {
    *reinterpret_cast<uint32_t*>(op) = pack_bf16x2(o[0] * inv, o[1] * inv);
  }
  if (lse_out != nullptr && lane == 0) *lse_out = dsum > 0.f ? M + lg2(dsum) * kLn2 : NEG_INF;
}

}  // namespace sinkattn
