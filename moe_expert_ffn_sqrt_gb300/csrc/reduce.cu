// Weighted unpermute-reduce: out[t] = bf16( sum_k topk_w[t,k] * y[inv_perm[t,k]] ), fp32 sum in k order.
// Note "INT8 高吞吐/低延迟 EP 代码梳理" §9.6 (gather: look up inv_perm, read the row, multiply by
// topk_weights, accumulate); MegaMoE page 二、阶段 5 (float32 accumulation, bf16 result).
// Each thread owns 8 consecutive columns (one 16-byte load per slot, one 16-byte store).
#include <cuda_bf16.h>

#include "kernels.h"

namespace moe {

__global__ void __launch_bounds__(128) unpermute_reduce_kernel(const uint16_t* __restrict__ y,
                                                               const int32_t* __restrict__ inv_perm,
                                                               const float* __restrict__ topk_w, int K, int H,
                                                               uint16_t* __restrict__ out) {
  const int t = blockIdx.x;
  const int c = (blockIdx.y * 128 + threadIdx.x) * 8;
  if (c >= H) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int k = 0; k < K; ++k) {
    const int row = __ldg(inv_perm + static_cast<size_t>(t) * K + k);
    const float w = topk_w ? __ldg(topk_w + static_cast<size_t>(t) * K + k) : 1.f;   // nullptr: plain sum
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(y + static_cast<size_t>(row) * H + c));
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[2 * j] = fmaf(w, __uint_as_float(u[j] << 16), acc[2 * j]);
      acc[2 * j + 1] = fmaf(w, __uint_as_float(u[j] & 0xFFFF0000u), acc[2 * j + 1]);
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * j]));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * j + 1]));
    o[j] = lo | (hi << 16);
  }
  *reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
}

cudaError_t launch_unpermute_reduce(const uint16_t* y, const int32_t* inv_perm, const float* topk_w, int T, int K,
                                    int H, uint16_t* out, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  dim3 grid(T, (H / 8 + 127) / 128);
  unpermute_reduce_kernel<<<grid, 128, 0, stream>>>(y, inv_perm, topk_w, K, H, out);
  return cudaGetLastError();
}

// Failure-path self-test: one bounded wait that nothing can satisfy, through the same primitives
// the hot-path kernels use.  Mode 0: a counter that is never incremented (the L2-after-L1 waits);
// mode 1: an mbarrier phase that never completes (the pipeline waits).  The wait gives up after
// its cycle budget, records a timeout in the status word and the kernel returns.
__global__ void wait_selftest_kernel(const uint32_t* never_set, uint32_t* status, int mode) {
  __shared__ uint64_t bar;
  if (mode == 0) {
    if (threadIdx.x == 0) wait_counter(never_set, 1u, status);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, status);
}

cudaError_t launch_wait_selftest(const uint32_t* never_set, uint32_t* status, int mode, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(never_set, status, mode);
  return cudaGetLastError();
}

}  // namespace moe
