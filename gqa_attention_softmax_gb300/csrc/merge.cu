// Merge of split-KV partials with the sink counted exactly once.
//
// For every (row, query head): the state starts from the sink alone
// (m = s_h, d = 1; m = -inf, d = 0 without a sink) and absorbs every chunk's
// (m_s, d_s, acc_s) with the rescale to the common maximum; out = acc / d,
// lse = m + ln d ("GPT-OSS on Day 0", section "Kernels for GPT-OSS / Sink
// attention": the sink belongs to one block only when the sequence is split).
// The common maximum over the sink and all chunk maxima is taken first, so
// every chunk is rescaled once.
//
// One warp per (row, head); each lane owns d/32 contiguous output columns, so
// each chunk's accumulator row is read with one coalesced vector load.
#include "common.cuh"
#include "internal.h"

namespace sinkattn {

template <int D>
__global__ void __launch_bounds__(256)
    merge_kernel(const float* __restrict__ part_acc, const float* __restrict__ part_md,
                 const float* __restrict__ sinks, int n_rows, int Hq, int S,
                 __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  constexpr int VEC = D / 32;   // 2 or 4 floats per lane
  constexpr float NEG_INF = kNegInf;
  const int lane = threadIdx.x & 31;
  const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (w >= static_cast<long long>(n_rows) * Hq) return;
  const int h = static_cast<int>(w % Hq);
  const float* md = part_md + w * S * 2;
  const float* acc = part_acc + w * S * D;

  const float sink = sinks ? sinks[h] : NEG_INF;
  float M = sink;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, md[2 * s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  float dsum = (sink == NEG_INF) ? 0.f : ex2((sink - M) * kLog2e);
  float o[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) o[e] = 0.f;
  for (int s = 0; s < S; ++s) {
    const float2 mds = *reinterpret_cast<const float2*>(md + 2 * s);
    if (mds.x == NEG_INF) continue;   // empty chunk
    const float wgt = ex2((mds.x - M) * kLog2e);
    dsum = fmaf(mds.y, wgt, dsum);
    const float* a = acc + s * D + lane * VEC;
    if (VEC == 4) {
      const float4 v = *reinterpret_cast<const float4*>(a);
      o[0] = fmaf(v.x, wgt, o[0]);
      o[1] = fmaf(v.y, wgt, o[1]);
      o[2] = fmaf(v.z, wgt, o[2]);
      o[3] = fmaf(v.w, wgt, o[3]);
    } else {
      const float2 v = *reinterpret_cast<const float2*>(a);
      o[0] = fmaf(v.x, wgt, o[0]);
      o[1] = fmaf(v.y, wgt, o[1]);
    }
  }
  const float inv = dsum > 0.f ? 1.f / dsum : 0.f;
  __nv_bfloat16* orow = out + w * D + lane * VEC;
  if (VEC == 4) {
    uint2 pk;
    pk.x = pack_bf16x2(o[0] * inv, o[1] * inv);
    pk.y = pack_bf16x2(o[2] * inv, o[3] * inv);
    *reinterpret_cast<uint2*>(orow) = pk;
  } else {
    *reinterpret_cast<uint32_t*>(orow) = pack_bf16x2(o[0] * inv, o[1] * inv);
  }
  if (lse != nullptr && lane == 0) lse[w] = dsum > 0.f ? M + lg2(dsum) * kLn2 : NEG_INF;
}

int launch_merge(const float* part_acc, const float* part_md, const float* sinks, int32_t rows,
                 int32_t Hq, int32_t d, int32_t num_splits, void* out, float* lse,
                 cudaStream_t stream) {
  const long long warps = static_cast<long long>(rows) * Hq;
  if (warps == 0) return SINKATTN_OK;
  const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
  auto* o = static_cast<__nv_bfloat16*>(out);
  if (d == 64)
    merge_kernel<64><<<blocks, 256, 0, stream>>>(part_acc, part_md, sinks, rows, Hq, num_splits, o, lse);
  else
    merge_kernel<128><<<blocks, 256, 0, stream>>>(part_acc, part_md, sinks, rows, Hq, num_splits, o, lse);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("merge kernel launch: %s", cudaGetErrorString(e));
    return SINKATTN_CUDA_ERROR;
  }
  return SINKATTN_OK;
}

int read_status_merge(cudaStream_t s, int* status) {
  *status = SINKATTN_OK;   // the merge kernel has no waits and no length checks
  (void)s;
  return SINKATTN_OK;
}

}  // namespace sinkattn
