// Grouped GEMMs with NVFP4 weights (E2M1 codes, one E4M3 scale per 16 along K, one fp32 scale per
// expert matrix) on tcgen05 (sm_103a).  Same contract as gemm.cu: L1 = SwiGLU + FP8 requant, L2 =
// bf16.  Weight format: CUDA tag page teaser (MXFP4 vs NVFP4, chosen by moe_quant_algo).
//
// No tcgen05 MMA kind multiplies E4M3 activations by E2M1 weights with E4M3 per-16 scales, and
// rounding code x scale to an 8-bit format would lose bits.  Both operands are exact in bfloat16,
// though: an E2M1 value times an E4M3 scale has at most 6 significant bits, and an E4M3 activation
// times its power-of-two scale at most 4.  So this path runs kind::f16 (bf16 x bf16 -> fp32):
//  * activations are dequantised once per call into bf16 rows (act_to_bf16_kernel);
//  * each pipeline stage brings 256 weight rows x 64 codes + their scales with one bulk copy, and
//    the four epilogue warps turn them into a 128-byte-swizzled bf16 tile (byte-permute table for
//    E2M1 -> bf16, exact bf16 multiply by the scale) before the MMA warp consumes it;
//  * the per-expert fp32 tensor scale multiplies the accumulator in the epilogue.
// Layout and scheduling otherwise follow gemm.cu: M = 128 token rows x N = 256 weight rows, one
// persistent CTA per SM, TMA producer warp, single-thread MMA issue, 128x256 fp32 accumulator.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kNvThreads = 192;          // warp 0 TMA, warp 1 MMA, warps 2..5 convert + epilogue
constexpr int kNvBudget = 227 * 1024;
constexpr uint32_t kNvTmemCols = 512;
constexpr int kNvTile = 256;             // weight rows per tile (MMA N)
constexpr int kNvSlab = 64;              // K per pipeline stage (64 bf16 = one 128-byte row)
constexpr int kNvChunk = kNvTile * 32 + kNvTile * 4;   // packed bytes per (tile, slab): codes + scales

template <int BN>
struct NvCfg {
  static constexpr int A_OFF = 0;                               // bf16 tokens, MMA reads 128 rows
  static constexpr int A_BYTES = BN * 128;
  static constexpr int B_OFF = 16384;                           // bf16 weights 256 x 128 B
  static constexpr int P_OFF = B_OFF + kNvTile * 128;           // packed codes + scales
  static constexpr int STAGE = (P_OFF + kNvChunk + 1023) / 1024 * 1024;
  static constexpr int EXTRA = 1024;
  static constexpr int S_FIT = (kNvBudget - EXTRA - 1024) / STAGE;
  static constexpr int STAGES = S_FIT > 4 ? 4 : S_FIT;
  static constexpr int SMEM = 1024 + STAGES * STAGE + EXTRA;
  static_assert(STAGES >= 2, "shared memory too small");
};

struct NvArgs {
  const uint8_t* w;             // packed NVFP4 weight stream
  const float* tscale;          // [E]
  const int32_t* expert_ids;
  const int32_t* m_sum;
  uint8_t* h_q;
  uint8_t* h_sf;
  uint16_t* y;
  uint32_t* status;
  size_t w_bytes;
  int n_slabs;                  // K / 64
  int n_wt;
  int out_cols;
  int sf_nb;
  int n_tiles;
  int one_expert_blocks;        // permute alignment is a multiple of BN: one expert per row block
  FusedReduce red;              // L2: unpermute-reduce in the epilogue when red.out != nullptr
};

template <int BN>
__device__ __forceinline__ bool nv_next_item(const NvArgs& a, int msum, int& t, int& e) {
  // as next_item in gemm.cu: called by whole warps; one load per block when blocks hold one expert
  const int lane = threadIdx.x & 31;
  while (t < a.n_tiles) {
    const int r0 = (t / a.n_wt) * BN;
    if (r0 >= msum) return false;
    if (a.one_expert_blocks) {
      if (e < 0) {
        const int x = __ldg(a.expert_ids + r0);
        if (x >= 0) {
          e = x;
          return true;
        }
      }
    } else {
      const int rend = min(r0 + BN, msum);
      int best = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < (BN + 31) / 32; ++j) {
        const int r = r0 + j * 32 + lane;
        if (r < rend) {
          const int x = __ldg(a.expert_ids + r);
          if (x > e && x < best) best = x;
        }
      }
      best = __reduce_min_sync(0xffffffffu, best);
      if (best != 0x7fffffff) {
        e = best;
        return true;
      }
    }
    t += gridDim.x;
    e = -1;
  }
  return false;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Four E2M1 codes (the low 16 bits of `w`, element i in nibble i) -> four bf16 values as two
// bf16x2 words.  Magnitude codes 0..7 are 0, .5, 1, 1.5, 2, 3, 4, 6, whose bf16 patterns split
// into the low-byte table {00,00,80,C0,00,40,80,C0} and the high-byte table {00,3F,3F,3F,40,40,
// 40,40}; prmt looks up four bytes at once.  The code's sign bit becomes the bf16 sign bit.
__device__ __forceinline__ void e2m1x4_to_bf16(uint32_t w, uint32_t& p0, uint32_t& p1) {
  const uint32_t sel = w & 0x7777u;
  const uint32_t lo = prmt(0xC0800000u, 0xC0804000u, sel);
  const uint32_t hi = prmt(0x3F3F3F00u, 0x40404040u, sel);
  p0 = prmt(lo, hi, 0x5140u) | ((w << 12) & 0x8000u) | ((w << 24) & 0x80000000u);
  p1 = prmt(lo, hi, 0x7362u) | ((w << 4) & 0x8000u) | ((w << 16) & 0x80000000u);
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a), y = *reinterpret_cast<__nv_bfloat162*>(&b);
  __nv_bfloat162 r = __hmul2(x, y);
  return *reinterpret_cast<uint32_t*>(&r);
}

// E4M3 code -> bf16 bits (exact).
__device__ __forceinline__ uint32_t e4m3_to_bf16_bits(uint32_t c) {
  const __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3);
  const float f = __half2float(*reinterpret_cast<const __half*>(&hr));
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Converts the packed (codes, scales) of one stage into the 128-byte-swizzled bf16 weight tile.
// 128 threads, two weight rows each.
__device__ __forceinline__ void convert_stage(const uint8_t* packed, uint8_t* btile, int tid) {
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int n = tid * 2 + rr;
    const uint4 c0 = *reinterpret_cast<const uint4*>(packed + n * 32);
    const uint4 c1 = *reinterpret_cast<const uint4*>(packed + n * 32 + 16);
    const uint32_t scw = *reinterpret_cast<const uint32_t*>(packed + kNvTile * 32 + n * 4);
    const uint32_t codes[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    uint8_t* rowp = btile + n * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {           // 16-byte chunk c = elements 8c .. 8c+7 (group c/2)
      const uint32_t s = e4m3_to_bf16_bits((scw >> (8 * (c >> 1))) & 0xFF);
      const uint32_t s2 = s | (s << 16);
      uint32_t p[4];
      e2m1x4_to_bf16(codes[c], p[0], p[1]);
      e2m1x4_to_bf16(codes[c] >> 16, p[2], p[3]);
#pragma unroll
      for (int j = 0; j < 4; ++j) p[j] = bf16x2_mul(p[j], s2);
      *reinterpret_cast<uint4*>(rowp + ((c ^ (n & 7)) << 4)) = make_uint4(p[0], p[1], p[2], p[3]);
    }
  }
}

__device__ __forceinline__ float silu_mul_nv(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

template <int BN, bool L1>
__global__ void __launch_bounds__(kNvThreads, 1)
    moe_gemm_nv_kernel(const __grid_constant__ CUtensorMap tmap_x, const NvArgs a) {
  using C = NvCfg<BN>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* extra = smem + C::STAGES * C::STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(extra);
  uint64_t* conv = full + C::STAGES;
  uint64_t* empty = conv + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(conv + s), 128);
      mbar_init(smem_u32(empty + s), 1);
    }
    mbar_init(smem_u32(acc_full), 1);
    mbar_init(smem_u32(acc_empty), 128);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmap_x);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kNvTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int msum = *a.m_sum;

  if (warp == 0) {
    // ---------------- producer: bf16 token rows by TMA, packed weights by one bulk copy ----------------
    const uint64_t pol_x = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    int t = blockIdx.x, e = -1;
    while (!__any_sync(0xffffffffu, *abort_flag != 0) && nv_next_item<BN>(a, msum, t, e)) {
      const int r0 = (t / a.n_wt) * BN, wt = t % a.n_wt;
      const size_t chunk0 = (static_cast<size_t>(e) * a.n_wt + wt) * a.n_slabs;
      bool ok = true;
      for (int s = 0; s < a.n_slabs; ++s) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(empty + stage), phase ^ 1, a.status));
        if (!ok) break;
        if (lane == 0) {
          uint8_t* st = stages + stage * C::STAGE;
          const uint32_t fb = smem_u32(full + stage);
          const size_t wbase = (chunk0 + s) * kNvChunk;
          if (wbase + kNvChunk > a.w_bytes || (reinterpret_cast<uintptr_t>(a.w) & 15)) {
            record_error(a.status, kDevErrCheck);
            *abort_flag = 1;
          } else {
            mbar_arrive_expect_tx(fb, C::A_BYTES + kNvChunk);
            tma_load_2d(smem_u32(st + C::A_OFF), &tmap_x, s * kNvSlab, r0, fb, pol_x);
            bulk_load(smem_u32(st + C::P_OFF), a.w + wbase, kNvChunk, fb);
          }
        }
        __syncwarp();
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        break;
      }
    }
    if (__any_sync(0xffffffffu, *abort_flag != 0)) {
      for (int s = 0; s < C::STAGES; ++s) mbar_wait(smem_u32(full + s), (s < stage) ? phase : (phase ^ 1), nullptr);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: kind::f16, M=128, N=256, K=16 x 4 per stage ----------------
    int stage = 0;
    uint32_t phase = 0;
    uint32_t acc_phase = 0;
    int t = blockIdx.x, e = -1;
    const uint32_t id = idesc_bf16(128, kNvTile);
    while (!__any_sync(0xffffffffu, *abort_flag != 0) && nv_next_item<BN>(a, msum, t, e)) {
      bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(acc_empty), acc_phase ^ 1, a.status));
      if (ok) {
        tc_fence_after();
        for (int s = 0; s < a.n_slabs; ++s) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(conv + stage), phase, a.status));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t st = smem_u32(stages + stage * C::STAGE);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16(tmem, desc_sw128(st + C::A_OFF + k * 32), desc_sw128(st + C::B_OFF + k * 32), id,
                       (s > 0 || k > 0) ? 1u : 0u);
            tc_commit(smem_u32(empty + stage));
          }
          __syncwarp();
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      if (lane == 0) tc_commit(smem_u32(acc_full));
      __syncwarp();
      acc_phase ^= 1;
    }
  } else {
    // ---------------- warps 2..5: convert each stage's weights, then the epilogue per item ----------------
    const int tid = threadIdx.x - 64;
    const int q = warp & 3;
    const int m = q * 32 + lane;
    const bool warp_has_rows = q * 32 < BN;
    const uint32_t acc = tmem + (static_cast<uint32_t>(q * 32) << 16);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t acc_phase = 0;
    int t = blockIdx.x, e = -1;
    while (nv_next_item<BN>(a, msum, t, e)) {
      const int r0 = (t / a.n_wt) * BN, wt = t % a.n_wt;
      bool ok = true;
      for (int s = 0; s < a.n_slabs; ++s) {
        ok = mbar_wait(smem_u32(full + stage), phase, a.status) && *abort_flag == 0;
        ok = named_barrier_and(1, 128, ok);
        if (!ok) break;
        uint8_t* st = stages + stage * C::STAGE;
        convert_stage(st + C::P_OFF, st + C::B_OFF, tid);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(smem_u32(conv + stage));
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (ok) {
        ok = mbar_wait(smem_u32(acc_full), acc_phase, a.status) && *abort_flag == 0;
        ok = named_barrier_and(1, 128, ok);
      }
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int row = r0 + m;
      const bool mine = m < BN && row < msum && __ldg(a.expert_ids + row) == e;
      const float ts = __ldg(a.tscale + e);
      if (L1) {
        float h[128];
        float amax = 0.f;
        if (warp_has_rows) {
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 16) {
            uint32_t g[16], u[16];
            tc_ld_x16(acc + c0, g);
            tc_ld_x16(acc + 128 + c0, u);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              h[c0 + j] = silu_mul_nv(__uint_as_float(g[j]) * ts, __uint_as_float(u[j]) * ts);
              amax = fmaxf(amax, fabsf(h[c0 + j]));
            }
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(acc_empty));
        if (mine) {
          const int ex = ue8m0_exponent(amax);
          const float sc = pow2_neg(ex);
          a.h_sf[act_sf_offset(BN, a.sf_nb, row, wt)] = static_cast<uint8_t>(ex + 127);
          uint4* dst = reinterpret_cast<uint4*>(a.h_q + static_cast<size_t>(row) * a.out_cols + wt * 128);
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 16) {
            uint32_t packed[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int c = c0 + 4 * j;
              const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(h[c] * sc, h[c + 1] * sc), __NV_SATFINITE, __NV_E4M3);
              const uint32_t hi =
                  __nv_cvt_float2_to_fp8x2(make_float2(h[c + 2] * sc, h[c + 3] * sc), __NV_SATFINITE, __NV_E4M3);
              packed[j] = lo | (hi << 16);
            }
            dst[c0 / 16] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
          }
        }
      } else {
        uint32_t packed[128];
        const int ncols = min(kNvTile, a.out_cols - wt * kNvTile);
        if (warp_has_rows) {
#pragma unroll
          for (int c0 = 0; c0 < kNvTile; c0 += 16) {
            uint32_t v[16];
            tc_ld_x16(acc + c0, v);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[2 * j]) * ts));
              const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[2 * j + 1]) * ts));
              packed[c0 / 2 + j] = lo | (hi << 16);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(acc_empty));
        if (mine) {
          uint4* dst = reinterpret_cast<uint4*>(a.y + static_cast<size_t>(row) * a.out_cols + wt * kNvTile);
#pragma unroll
          for (int c = 0; c < kNvTile / 8; ++c)
            if (c * 8 < ncols) dst[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
        }
        if (a.red.out) fused_reduce_tail(a.red, a.y, a.out_cols, mine, row, wt, a.n_wt, wt * kNvTile, ncols);
      }
      acc_phase ^= 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kNvTmemCols);
  }
}

// Activation rows (E4M3 codes + tiled UE8M0 scales) -> bf16 rows, exactly, for rows that hold a
// (token, expert) pair.  One warp per row, 8 codes per lane step.
__global__ void __launch_bounds__(256) act_to_bf16_kernel(const uint8_t* __restrict__ x, const uint8_t* __restrict__ sf,
                                                          const int32_t* __restrict__ expert_ids,
                                                          const int32_t* __restrict__ m_sum, int U, int Kd, int bt,
                                                          int nb, uint16_t* __restrict__ xb) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int msum = *m_sum;
  for (int r = blockIdx.x * 8 + warp; r < msum && r < U; r += gridDim.x * 8) {
    if (__ldg(expert_ids + r) < 0) continue;
    for (int k0 = lane * 8; k0 < Kd; k0 += 256) {
      const uint32_t b = sf[act_sf_offset(bt, nb, r, k0 / 128)];
      const float sc = b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);   // 2^(b-127)
      const uint2 c = *reinterpret_cast<const uint2*>(x + static_cast<size_t>(r) * Kd + k0);
      const uint32_t cw[2] = {c.x, c.y};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t two = (cw[j >> 1] >> (16 * (j & 1))) & 0xFFFF;
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
        const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(f.x * sc));
        const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(f.y * sc));
        o[j] = lo | (hi << 16);
      }
      *reinterpret_cast<uint4*>(xb + static_cast<size_t>(r) * Kd + k0) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// NVFP4 packing: per (expert, 256-row tile, 64-deep slab) 256 rows x 32 bytes of codes followed by
// 256 rows x 4 E4M3 scales (one per 16 codes); tiles formed as in pack_mx_weights_kernel.
__global__ void pack_nv_weights_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf, int E, int N,
                                       int Kd, int pair, uint8_t* __restrict__ out) {
  const int n_slabs = Kd / kNvSlab, n_wt = pair == 2 ? N / kNvTile : (N + kNvTile - 1) / kNvTile;
  const size_t total = static_cast<size_t>(E) * n_wt * n_slabs * kNvChunk;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const size_t c = i / kNvChunk;
    const int o = static_cast<int>(i % kNvChunk);
    const int s = static_cast<int>(c % n_slabs);
    const size_t ew = c / n_slabs;
    const int wt = static_cast<int>(ew % n_wt), e = static_cast<int>(ew / n_wt);
    const bool code = o < kNvTile * 32;
    const int n = code ? o / 32 : (o - kNvTile * 32) / 4;
    const int h = n / 128, mm = n % 128;
    const int r = pair == 2 ? h * (N / 2) + wt * 128 + mm : wt * 256 + n;
    if (code)
      out[i] = r < N ? q[(static_cast<size_t>(e) * N + r) * (Kd / 2) + s * 32 + (o % 32)] : 0;
    else
      out[i] = r < N ? sf[(static_cast<size_t>(e) * N + r) * (Kd / 16) + s * 4 + (o - kNvTile * 32) % 4] : 0;
  }
}

typedef CUresult (*EncodeTiledFnNv)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFnNv get_encode_nv() {
  static EncodeTiledFnNv fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFnNv>(p);
  }
  return fn;
}

template <int BN, bool L1>
cudaError_t launch_nv_t(const NvLaunch& L, cudaStream_t stream) {
  using C = NvCfg<BN>;
  EncodeTiledFnNv enc = get_encode_nv();
  if (!enc) return cudaErrorInvalidValue;
  CUtensorMap mx;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(L.Kd), static_cast<cuuint64_t>(L.U)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(L.Kd) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kNvSlab), static_cast<cuuint32_t>(BN)};
  cuuint32_t es[2] = {1, 1};
  if (enc(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(L.xb), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  NvArgs a;
  a.w = L.w;
  a.tscale = L.tscale;
  a.expert_ids = L.expert_ids;
  a.m_sum = L.m_sum;
  a.h_q = L.h_q;
  a.h_sf = L.h_sf;
  a.y = L.y;
  a.red = L.red;
  a.status = L.status;
  const int pair = L1 ? 2 : 1;
  a.n_wt = pair == 2 ? L.w_rows / kNvTile : (L.w_rows + kNvTile - 1) / kNvTile;
  a.n_slabs = L.Kd / kNvSlab;
  a.w_bytes = static_cast<size_t>(L.E) * a.n_wt * a.n_slabs * kNvChunk;
  a.out_cols = L1 ? L.I : L.w_rows;
  a.sf_nb = act_sf_blocks(L.U, BN);
  a.n_tiles = ((L.U + BN - 1) / BN) * a.n_wt;
  a.one_expert_blocks = L.align % BN == 0;
  int grid = num_sms();
  if (grid > a.n_tiles) grid = a.n_tiles;
  if (grid < 1) grid = 1;
  cudaError_t err = cudaFuncSetAttribute(moe_gemm_nv_kernel<BN, L1>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (err != cudaSuccess) return err;
  moe_gemm_nv_kernel<BN, L1><<<grid, kNvThreads, C::SMEM, stream>>>(mx, a);
  return cudaGetLastError();
}

}  // namespace

size_t packed_nv_weight_bytes(int E, int N, int Kd, int pair) {
  const int n_wt = pair == 2 ? N / kNvTile : (N + kNvTile - 1) / kNvTile;
  return static_cast<size_t>(E) * n_wt * (Kd / kNvSlab) * kNvChunk;
}

cudaError_t launch_pack_nv(const uint8_t* q, const uint8_t* sf, int E, int N, int Kd, int pair, uint8_t* out,
                           cudaStream_t stream) {
  pack_nv_weights_kernel<<<4 * num_sms(), 256, 0, stream>>>(q, sf, E, N, Kd, pair, out);
  return cudaGetLastError();
}

cudaError_t launch_act_to_bf16(const uint8_t* x, const uint8_t* sf, const int32_t* expert_ids, const int32_t* m_sum,
                               int U, int Kd, int align, uint16_t* xb, cudaStream_t stream) {
  const int bt = act_sf_block_rows(align);
  const int blocks = (U + 7) / 8 < 4 * num_sms() ? (U + 7) / 8 : 4 * num_sms();
  act_to_bf16_kernel<<<blocks > 0 ? blocks : 1, 256, 0, stream>>>(x, sf, expert_ids, m_sum, U, Kd, bt,
                                                                  act_sf_blocks(U, bt), xb);
  return cudaGetLastError();
}

cudaError_t launch_gemm_nv(const NvLaunch& L, bool l1, cudaStream_t stream) {
  const int bn = act_sf_block_rows(L.align);
  if (l1) {
    switch (bn) {
      case 16: return launch_nv_t<16, true>(L, stream);
      case 32: return launch_nv_t<32, true>(L, stream);
      case 64: return launch_nv_t<64, true>(L, stream);
      default: return launch_nv_t<128, true>(L, stream);
    }
  }
  switch (bn) {
    case 16: return launch_nv_t<16, false>(L, stream);
    case 32: return launch_nv_t<32, false>(L, stream);
    case 64: return launch_nv_t<64, false>(L, stream);
    default: return launch_nv_t<128, false>(L, stream);
  }
}

}  // namespace moe
