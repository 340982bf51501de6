// Merge of split-KV partials with the sink counted exactly once: one warp
// per (row, query head) runs merge_row (merge_row.cuh).
#include "common.cuh"
#include "internal.h"
#include "merge_row.cuh"

namespace sinkattn {

template <int D>
__global__ void __launch_bounds__(256)
    merge_kernel(const float* __restrict__ part_acc, const float* __restrict__ part_md,
                 const float* __restrict__ sinks, int n_rows, int Hq, int S,
                 __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int drop) {
  // Launched as a programmatic dependent of the partial kernel: wait until
  // that grid has completed and its writes are visible (immediate otherwise).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long n = static_cast<long long>(n_rows) * Hq;
  const long long w0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (w0 >= n) return;
  // newest rows first: the partial kernels finish the last sequences last,
  // so those partials are the ones still in L2
  const long long w = n - 1 - w0;
  const int h = static_cast<int>(w % Hq);
  const float* acc = part_acc + w * S * D;
  merge_row<D>(part_md + w * S * 2, acc, sinks ? sinks[h] : kNegInf, S, lane, out + w * D,
               lse != nullptr ? lse + w : nullptr);
  if (drop) {   // library-owned scratch: the row's accumulator lines are dead
    __syncwarp();
    const char* base = reinterpret_cast<const char*>(acc);
    for (int off = lane * 128; off < S * D * 4; off += 32 * 128)
      asm volatile("discard.global.L2 [%0], 128;" ::"l"(base + off) : "memory");
  }
}

int launch_merge(const float* part_acc, const float* part_md, const float* sinks, int32_t rows,
                 int32_t Hq, int32_t d, int32_t num_splits, void* out, float* lse,
                 cudaStream_t stream, bool drop_partials) {
  const long long warps = static_cast<long long>(rows) * Hq;
  if (warps == 0) return SINKATTN_OK;
  const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
  auto* o = static_cast<__nv_bfloat16*>(out);
  // Programmatic stream serialisation: the launch may be processed while the
  // previous kernel on the stream (the partial kernel) drains its last CTAs;
  // the kernel's griddepcontrol.wait keeps the data dependency.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e =
      d == 64 ? cudaLaunchKernelEx(&cfg, merge_kernel<64>, part_acc, part_md, sinks, rows, Hq,
                                   num_splits, o, lse, drop_partials ? 1 : 0)
              : cudaLaunchKernelEx(&cfg, merge_kernel<128>, part_acc, part_md, sinks, rows, Hq,
                                   num_splits, o, lse, drop_partials ? 1 : 0);
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
