// Gate GEMM on the tensor cores for batches of more than 16 tokens:
//   partial[s][t][e] = sum over the s-th slice of H of hidden[t, h] * w_gate[e, h]
// Page "DeepSeek V4 MegaMoE Kernel 深度解析", 经典 MoE 的计算过程 / 第一步：路由 (gate logits from the
// hidden states and the fp32 gate weight); the scoring and top-K that follow are route.cu's.
//
// Design (this file's own):
//  * Each call splits the fp32 gate weight into three bf16 parts, w = hi + mid + lo, each part the
//    round-to-nearest bf16 of what the parts before it leave over.  Three 8-bit significands cover
//    fp32's 24, so the split is exact; a bf16 hidden value times a part is exact in fp32, and the
//    tensor core adds these exact products in fp32, like the fma chain of a SIMT dot product.
//  * MMA: M = 128 experts (A = one weight part), N = 128 tokens (B = hidden rows), K = 16.  A stage
//    holds the three 128 x 64 part tiles and the 128 x 64 hidden tile (64 KB; three stages), loaded
//    by TMA with 128-byte swizzle.
//  * The tensor core's fp32 accumulation drops low bits at every step (measured: over the 1344
//    steps of H = 7168 the logit error grows linearly to ~2e-6 of sum |x w|, twenty times an fma
//    chain's).  So one TMEM accumulator holds only one 64-column k-block (12 MMAs); the epilogue
//    adds it into fp32 registers in k order while the MMAs fill the other accumulator.
//  * Grid = expert tiles x token tiles x H slices.  A CTA owns one (tile, slice): warp 0 loads,
//    warp 1 issues the MMAs, warps 2..5 sum and write the fp32 partial sums (thread = expert, so
//    each token's 32 consecutive experts per warp form one 128-byte store).  route_finish_kernel
//    adds the slices in a fixed order.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kGateThreads = 192;
constexpr int kGateM = 128;                       // experts per tile
constexpr int kGateN = 128;                       // tokens per tile
constexpr int kGateKB = 64;                       // bf16 columns per k-block (one swizzled 128-byte row)
constexpr int kGateA = kGateM * kGateKB * 2;      // 16 KB: one weight-part tile
constexpr int kGateB = kGateN * kGateKB * 2;      // 16 KB: hidden tile
constexpr int kGateStage = 3 * kGateA + kGateB;   // 64 KB
constexpr int kGateStages = 3;
constexpr int kGateSmem = 1024 + kGateStages * kGateStage + 256;
constexpr int kGateMaxSplit = 16;
constexpr uint32_t kGateTmemCols = 2 * kGateN;   // two accumulators

// w [n] fp32 -> parts[0 .. n) hi, [n .. 2n) mid, [2n .. 3n) lo (bf16 bits).  n % 4 == 0.
__global__ void __launch_bounds__(256) gate_split_kernel(const float* __restrict__ w, size_t n,
                                                         uint16_t* __restrict__ parts) {
  const size_t n4 = n / 4;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float4 v = reinterpret_cast<const float4*>(w)[i];
    const float x[4] = {v.x, v.y, v.z, v.w};
    uint16_t p[3][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(x[j]);
      const float r1 = x[j] - __bfloat162float(hi);
      const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
      const float r2 = r1 - __bfloat162float(mid);
      const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
      p[0][j] = __bfloat16_as_ushort(hi);
      p[1][j] = __bfloat16_as_ushort(mid);
      p[2][j] = __bfloat16_as_ushort(lo);
    }
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const uint2 o = make_uint2(static_cast<uint32_t>(p[q][0]) | (static_cast<uint32_t>(p[q][1]) << 16),
                                 static_cast<uint32_t>(p[q][2]) | (static_cast<uint32_t>(p[q][3]) << 16));
      reinterpret_cast<uint2*>(parts + static_cast<size_t>(q) * n)[i] = o;
    }
  }
}

struct GateArgs {
  float* partial;        // [nsplit][T][E]
  uint32_t* status;
  int T, E;
  int nkb;               // H / 64
  int kb_per_split;
};

__global__ void __launch_bounds__(kGateThreads, 1)
    gate_mma_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                    const GateArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGateStages * kGateStage);
  uint64_t* empty = full + kGateStages;
  uint64_t* acc_full = empty + kGateStages;    // [2]
  uint64_t* acc_empty = acc_full + 2;          // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int e0 = blockIdx.x * kGateM, t0 = blockIdx.y * kGateN, split = blockIdx.z;
  const int kb0 = split * a.kb_per_split, kb1 = min(a.nkb, kb0 + a.kb_per_split);   // never empty (host)
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGateStages; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(acc_full + b), 1);
      mbar_init(smem_u32(acc_empty + b), 128);
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_x);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kGateTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer (whole warp iterates, lane 0 issues) ----------------
    const uint64_t pol = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(empty + stage), phase ^ 1, a.status))) {
        *abort_flag = 1;
        break;
      }
      if (lane == 0) {
        uint8_t* st = smem + stage * kGateStage;
        const uint32_t fb = smem_u32(full + stage);
        mbar_arrive_expect_tx(fb, kGateStage);
#pragma unroll
        for (int p = 0; p < 3; ++p) tma_load_2d(smem_u32(st + p * kGateA), &tmap_w, kb * kGateKB, p * a.E + e0, fb, pol);
        tma_load_2d(smem_u32(st + 3 * kGateA), &tmap_x, kb * kGateKB, t0, fb, pol);
      }
      __syncwarp();
      if (++stage == kGateStages) {
        stage = 0;
        phase ^= 1;
      }
    }
    if (__any_sync(0xffffffffu, *abort_flag != 0)) {
      // let every copy issued into shared memory land before the CTA exits
      for (int s = 0; s < kGateStages; ++s) mbar_wait(smem_u32(full + s), (s < stage) ? phase : (phase ^ 1), nullptr);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: k-block i goes to accumulator i & 1 ----------------
    const uint32_t id = idesc_bf16(kGateM, kGateN);
    int stage = 0;
    uint32_t phase = 0;
    for (int kb = kb0, i = 0; kb < kb1; ++kb, ++i) {
      const int b = i & 1;
      const uint32_t use = static_cast<uint32_t>(i >> 1) & 1u;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(acc_empty + b), use ^ 1u, a.status) &&
                                                  mbar_wait(smem_u32(full + stage), phase, a.status) && *abort_flag == 0);
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t st = smem_u32(smem + stage * kGateStage);
        const uint32_t d = tmem + static_cast<uint32_t>(b * kGateN);
#pragma unroll
        for (int p = 0; p < 3; ++p)
#pragma unroll
          for (int k = 0; k < kGateKB / 16; ++k)
            mma_bf16(d, desc_sw128(st + p * kGateA + k * 32), desc_sw128(st + 3 * kGateA + k * 32), id,
                     (p > 0 || k > 0) ? 1u : 0u);
        tc_commit(smem_u32(empty + stage));
        tc_commit(smem_u32(acc_full + b));
      }
      __syncwarp();
      if (++stage == kGateStages) {
        stage = 0;
        phase ^= 1;
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5): thread = expert row of the tile ----------------
    const int q = warp & 3;
    const int e = e0 + q * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    float sum[kGateN];
#pragma unroll
    for (int c = 0; c < kGateN; ++c) sum[c] = 0.f;
    bool ok = true;
    for (int kb = kb0, i = 0; kb < kb1; ++kb, ++i) {
      const int b = i & 1;
      const uint32_t use = static_cast<uint32_t>(i >> 1) & 1u;
      ok = mbar_wait(smem_u32(acc_full + b), use, a.status) && *abort_flag == 0;
      ok = named_barrier_and(1, 128, ok);
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t acc = lane_base + static_cast<uint32_t>(b * kGateN);
#pragma unroll
      for (int h = 0; h < kGateN; h += 64) {
        uint32_t v[4][16];
#pragma unroll
        for (int j = 0; j < 4; ++j) tc_ld_x16(acc + h + 16 * j, v[j]);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int c = 0; c < 16; ++c) sum[h + 16 * j + c] += __uint_as_float(v[j][c]);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(acc_empty + b));
    }
    if (ok && e < a.E) {
#pragma unroll
      for (int c = 0; c < kGateN; ++c) {
        const int t = t0 + c;
        if (t < a.T) a.partial[(static_cast<size_t>(split) * a.T + t) * a.E + e] = sum[c];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kGateTmemCols);
  }
}

int gate_nsplit(int T, int H, int E) {
  const int tiles = ((E + kGateM - 1) / kGateM) * ((T + kGateN - 1) / kGateN);
  const int nkb = H / kGateKB;
  int ns = num_sms() / tiles;                // about one CTA per SM
  if (ns > kGateMaxSplit) ns = kGateMaxSplit;
  if (ns > nkb) ns = nkb;
  if (ns < 1) ns = 1;
  const int kps = (nkb + ns - 1) / ns;
  return (nkb + kps - 1) / kps;             // every slice non-empty
}

size_t gate_parts_bytes(int T, int H, int E) {
  (void)T;
  return (static_cast<size_t>(3) * E * H * sizeof(uint16_t) + 255) / 256 * 256;
}

cudaError_t launch_gate_mma(const uint16_t* hidden, const float* w_gate, int T, int H, int E, int nsplit,
                            uint16_t* parts, float* partial, uint32_t* status, cudaStream_t stream) {
  const size_t n = static_cast<size_t>(E) * H;
  int sblocks = static_cast<int>((n / 4 + 255) / 256);
  if (sblocks > 4 * num_sms()) sblocks = 4 * num_sms();
  gate_split_kernel<<<sblocks, 256, 0, stream>>>(w_gate, n, parts);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  CUtensorMap mw, mx;
  // parts viewed as [3E, H] bf16 (hi rows, then mid rows, then lo rows); hidden as [T, H]
  if (!make_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, parts, H, static_cast<uint64_t>(3) * E,
                   static_cast<uint64_t>(H) * 2, kGateKB, kGateM))
    return cudaErrorInvalidValue;
  if (!make_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, hidden, H, T, static_cast<uint64_t>(H) * 2, kGateKB, kGateN))
    return cudaErrorInvalidValue;
  GateArgs a;
  a.partial = partial;
  a.status = status;
  a.T = T;
  a.E = E;
  a.nkb = H / kGateKB;
  a.kb_per_split = (a.nkb + nsplit - 1) / nsplit;
  err = cudaFuncSetAttribute(gate_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGateSmem);
  if (err != cudaSuccess) return err;
  dim3 grid((E + kGateM - 1) / kGateM, (T + kGateN - 1) / kGateN, nsplit);
  gate_mma_kernel<<<grid, kGateThreads, kGateSmem, stream>>>(mw, mx, a);
  return cudaGetLastError();
}

}  // namespace moe
