// Grouped GEMMs with NVFP4 weights (E2M1 codes, one E4M3 scale per 16 along K, one fp32 scale per
// expert matrix) on tcgen05 (sm_103a).  Same contract as gemm.cu: L1 = SwiGLU + FP8 requant, L2 =
// bf16.  Weight format: CUDA tag page teaser (MXFP4 vs NVFP4, chosen by moe_quant_algo).
//
// No tcgen05 MMA kind multiplies E4M3 activations by E2M1 weights with E4M3 per-16 scales, and
// rounding code x scale to an 8-bit format would lose bits.  Both operands are exact in bfloat16,
// though: an E2M1 value times an E4M3 scale has at most 6 significant bits, and an E4M3 activation
// times its power-of-two scale at most 4.  So this path runs kind::f16 (bf16 x bf16 -> fp32):
//  * activations are dequantised once per call into bf16 rows (act_to_bf16_kernel);
//  * a load ring (3 slots) receives each slab's bf16 token rows (one or two row blocks) by TMA and
//    its packed weights (256 rows x 64 codes + scales) by one bulk copy; ten converter warps turn
//    the packed weights into a 128-byte-swizzled bf16 tile in a second ring (3 slots; byte-permute
//    table for E2M1 -> bf16, exact bf16 multiply by the scale) before the MMA warp consumes it;
//  * two 256-column TMEM accumulators (kind::f16 keeps no scale factors in TMEM) hold two row
//    blocks of one expert that share each converted tile; four epilogue warps drain them 32
//    columns at a time;
//  * the per-expert fp32 tensor scale multiplies the accumulator in the epilogue.
// Layout and scheduling otherwise follow gemm.cu: M = 128 token rows x N = 256 weight rows, one
// persistent CTA per SM, TMA producer warp, single-thread MMA issue.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"
#include "passes.cuh"

namespace moe {

namespace {

constexpr int kNvThreads = 448;          // warp 0 TMA, 1 MMA, 2..9 convert, 10..13 epilogue
constexpr int kNvConvThreads = 256;      // one weight row of the tile per converter thread
constexpr int kNvBudget = 227 * 1024;
constexpr uint32_t kNvTmemCols = 512;    // two 256-column accumulators
constexpr int kNvTile = 256;             // weight rows per tile (MMA N)
constexpr int kNvSlab = 64;              // K per pipeline stage (64 bf16 = one 128-byte row)
// Packed bytes per (tile, slab): the codes as two 4 KB halves (bytes 0..15, then 16..31, of each
// row's 32 code bytes, rows consecutive: a converter thread's 16-byte loads are conflict-free),
// then 256 rows x 4 E4M3 scales.
constexpr int kNvChunk = kNvTile * 32 + kNvTile * 4;
// Load ring slot: bf16 token rows of up to two row blocks (the MMA reads 128 rows = 16 KB each) +
// one packed weight chunk.
constexpr int kNvABytes = 16384;
constexpr int kNvPOff = 2 * kNvABytes;
constexpr int kNvLoadStage = (kNvPOff + kNvChunk + 1023) / 1024 * 1024;   // 41 KB
constexpr int kNvLoadStages = 3;
// bf16 weight ring slot: 256 rows x 128 B, 128-byte swizzle.
constexpr int kNvBStage = kNvTile * 128;                                     // 32 KB
constexpr int kNvBStages = 3;
constexpr int kNvExtra = 1024;
constexpr int kNvSmem = 1024 + kNvLoadStages * kNvLoadStage + kNvBStages * kNvBStage + kNvExtra;
static_assert(kNvSmem <= kNvBudget, "shared memory budget");
static_assert(kNvConvThreads % 32 == 0 && 2 + kNvConvThreads / 32 + 4 == kNvThreads / 32, "warp roles");

// One GEMM of the layer as the kernel sees it (L1: W13 with SwiGLU + requant; L2: W2, bf16 out).
struct NvPhase {
  const uint8_t* w;             // packed NVFP4 weight stream
  const float* tscale;          // [E]
  size_t w_bytes;
  int n_slabs;                  // K / 64
  int n_wt;                     // weight tiles per expert
  int out_cols;                 // L1: I, L2: H
  int n_tiles;                  // items of this phase (0: not run by this launch)
};

struct NvArgs {
  NvPhase ph[2];                // [0] L1, [1] L2
  const int32_t* expert_ids;
  const int32_t* m_sum;
  uint8_t* h_q;
  uint8_t* h_sf;
  uint16_t* y;
  uint32_t* status;
  int sf_nb;
  int one_expert_blocks;        // permute alignment is a multiple of BN: one expert per row block
  int split_pairs;              // items are halves of row-block pairs (small blocks) or whole pairs
  FusedReduce red;              // L2: unpermute-reduce in the epilogue when red.out != nullptr
  const int32_t* row_ids;       // L1: h of row r scaled by row_w[row_ids[r]] when row_w != nullptr
  const float* row_w;
};

// The per-phase view next_row_pass walks.
struct NvPassView {
  int n_tiles, n_wt, one_expert_blocks, split_pairs, pair_blocks;
  const int32_t* expert_ids;
};

__device__ __forceinline__ NvPassView pass_view(const NvArgs& a, int ph) {
  return NvPassView{a.ph[ph].n_tiles, a.ph[ph].n_wt, a.one_expert_blocks, a.split_pairs, 1, a.expert_ids};
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// E2M1 magnitude codes 0..7 are 0, .5, 1, 1.5, 2, 3, 4, 6: their bf16 patterns split into the
// low-byte table {00,00,80,C0,00,40,80,C0} and the high-byte table {00,3F,3F,3F,40,40,40,40}, which
// prmt looks up four at a time.
constexpr uint32_t kLoA = 0xC0800000u, kLoB = 0xC0804000u, kHiA = 0x3F3F3F00u, kHiB = 0x40404040u;

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a), y = *reinterpret_cast<__nv_bfloat162*>(&b);
  __nv_bfloat162 r = __hmul2(x, y);
  return *reinterpret_cast<uint32_t*>(&r);
}

// Eight E2M1 codes (element i in nibble i of w) times one bf16 scale s2 (in both halves; positive)
// -> eight bf16 values, exactly (a 2-bit E2M1 significand times a 4-bit E4M3 one fits bf16's 8):
// magnitudes by table lookup, scaled, then each code's sign bit xor-ed into the bf16 sign bit.  The
// signs come from a prmt in sign-replicate mode: byte k of w << 4 carries element 2k's sign in its
// top bit and byte k of w element 2k+1's.
__device__ __forceinline__ void e2m1x8_to_bf16(uint32_t w, uint32_t s2, uint32_t (&q)[4]) {
  const uint32_t sel0 = w & 0x7777u, sel1 = (w >> 16) & 0x7777u;
  const uint32_t lo0 = prmt(kLoA, kLoB, sel0), hi0 = prmt(kHiA, kHiB, sel0);
  const uint32_t lo1 = prmt(kLoA, kLoB, sel1), hi1 = prmt(kHiA, kHiB, sel1);
  const uint32_t w4 = w << 4;
  q[0] = bf16x2_mul(prmt(lo0, hi0, 0x5140), s2) ^ (prmt(w4, w, 0xC080) & 0x80008000u);
  q[1] = bf16x2_mul(prmt(lo0, hi0, 0x7362), s2) ^ (prmt(w4, w, 0xD090) & 0x80008000u);
  q[2] = bf16x2_mul(prmt(lo1, hi1, 0x5140), s2) ^ (prmt(w4, w, 0xE0A0) & 0x80008000u);
  q[3] = bf16x2_mul(prmt(lo1, hi1, 0x7362), s2) ^ (prmt(w4, w, 0xF0B0) & 0x80008000u);
}

// Two E4M3 codes (low 16 bits of v) -> their bf16 values, each in both halves of a word (exact).
__device__ __forceinline__ void e4m3x2_to_bf16x2(uint32_t v, uint32_t& s0, uint32_t& s1) {
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v & 0xFFFFu), __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  const uint32_t u = *reinterpret_cast<const uint32_t*>(&b);
  s0 = prmt(u, u, 0x1010);
  s1 = prmt(u, u, 0x3232);
}

__device__ __forceinline__ float silu_mul_nv(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

// Converts weight row n (one converter thread) of one slab: 64 codes (two conflict-free 16-byte
// loads), four E4M3 scales, eight 16-byte stores into the row's 128-byte-swizzled chunks (chunk c
// holds K positions 8c .. 8c+7 at byte ((c ^ (n & 7)) << 4) of the row).
__device__ __forceinline__ void convert_row(const uint8_t* __restrict__ packed, uint8_t* __restrict__ btile, int n) {
  const uint4 c0 = *reinterpret_cast<const uint4*>(packed + n * 16);
  const uint4 c1 = *reinterpret_cast<const uint4*>(packed + kNvTile * 16 + n * 16);
  const uint32_t sc = *reinterpret_cast<const uint32_t*>(packed + kNvTile * 32 + n * 4);
  uint32_t s2[4];
  e4m3x2_to_bf16x2(sc, s2[0], s2[1]);
  e4m3x2_to_bf16x2(sc >> 16, s2[2], s2[3]);
  const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const uint32_t row = smem_u32(btile) + static_cast<uint32_t>(n) * 128;
  const uint32_t x = static_cast<uint32_t>(n & 7) << 4;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t q[4];
    e2m1x8_to_bf16(words[c], s2[c >> 1], q);
    const uint32_t addr = row | ((static_cast<uint32_t>(c) << 4) ^ x);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(q[0]), "r"(q[1]), "r"(q[2]), "r"(q[3])
                 : "memory");
  }
}

// Warp roles: 0 loads (TMA token rows + bulk copy of packed weights into the load ring), 1 issues
// the MMAs, 2..9 convert packed weights into the bf16 ring, 10..13 drain the accumulators.
// A pass with two row blocks accumulates block j into TMEM columns [256j, 256j+256); the
// epilogue releases the accumulators after the pass.
// MODE 1: the L1 items (W13, SwiGLU + requant); 2: the L2 items (W2, bf16 out).  Items are assigned
// statically, CTA c taking items c, c + gridDim, ...
template <int BN, int MODE>
__global__ void __launch_bounds__(kNvThreads, 1)
    moe_gemm_nv_kernel(const __grid_constant__ CUtensorMap tmap_x, const NvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* lring = smem;                                   // [kNvLoadStages] token tiles + packed weights
  uint8_t* bring = smem + kNvLoadStages * kNvLoadStage;    // [kNvBStages] bf16 weight tiles
  uint8_t* extra = bring + kNvBStages * kNvBStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(extra);     // load slot filled (TMA)
  uint64_t* lempty = full + kNvLoadStages;                 // load slot consumed (MMA commit)
  uint64_t* bready = lempty + kNvLoadStages;               // bf16 tile written (converters)
  uint64_t* bempty = bready + kNvBStages;                  // bf16 tile consumed (MMA commit)
  uint64_t* acc_full = bempty + kNvBStages;
  uint64_t* acc_empty = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  constexpr int kPh0 = (MODE & 1) ? 0 : 1, kPh1 = (MODE & 2) ? 1 : 0;   // phases run, in order

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kNvLoadStages; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(lempty + s), 1);
    }
    for (int s = 0; s < kNvBStages; ++s) {
      mbar_init(smem_u32(bready + s), kNvConvThreads);
      mbar_init(smem_u32(bempty + s), 1);
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
    int ls = 0;
    uint32_t lph = 0;
    bool ok = true;
    for (int ph = kPh0; ok && ph <= kPh1; ++ph) {
      const NvPhase& F = a.ph[ph];
      const NvPassView V = pass_view(a, ph);
      const CUtensorMap* mx = &tmap_x;
      int t = blockIdx.x, p = 0, ep = -1;
      RowPass P;
      while (!__any_sync(0xffffffffu, *abort_flag != 0) && next_row_pass<BN>(V, msum, t, p, ep, P)) {
        const int wt = t % F.n_wt;
        const size_t chunk0 = (static_cast<size_t>(P.e) * F.n_wt + wt) * F.n_slabs;
        for (int s = 0; s < F.n_slabs; ++s) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(lempty + ls), lph ^ 1, a.status));
          if (!ok) break;
          if (lane == 0) {
            uint8_t* st = lring + ls * kNvLoadStage;
            const uint32_t fb = smem_u32(full + ls);
            const size_t wbase = (chunk0 + s) * kNvChunk;
            if (wbase + kNvChunk > F.w_bytes || (reinterpret_cast<uintptr_t>(F.w) & 15)) {
              record_error(a.status, kDevErrCheck);
              *abort_flag = 1;
            } else {
              mbar_arrive_expect_tx(fb, P.nb * BN * 128 + kNvChunk);
              for (int j = 0; j < P.nb; ++j)
                tma_load_2d(smem_u32(st + j * kNvABytes), mx, s * kNvSlab, (P.rb + j) * BN, fb, pol_x);
              bulk_load(smem_u32(st + kNvPOff), F.w + wbase, kNvChunk, fb);
            }
          }
          __syncwarp();
          if (++ls == kNvLoadStages) {
            ls = 0;
            lph ^= 1;
          }
        }
        if (!ok) break;
      }
    }
    if (!ok) *abort_flag = 1;
    if (__any_sync(0xffffffffu, *abort_flag != 0)) {
      // let every copy issued into shared memory land before the CTA exits
      for (int s = 0; s < kNvLoadStages; ++s) mbar_wait(smem_u32(full + s), (s < ls) ? lph : (lph ^ 1), nullptr);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: kind::f16, M=128, N=256, K=16 x 4 per slab and block ----------------
    int ls = 0, bs = 0;
    uint32_t lph = 0, bph = 0, acc_phase = 0;
    const uint32_t id = idesc_bf16(128, kNvTile);
    bool ok = true;
    for (int ph = kPh0; ok && ph <= kPh1; ++ph) {
      const NvPhase& F = a.ph[ph];
      const NvPassView V = pass_view(a, ph);
      int t = blockIdx.x, p = 0, ep = -1;
      RowPass P;
      while (!__any_sync(0xffffffffu, *abort_flag != 0) && next_row_pass<BN>(V, msum, t, p, ep, P)) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(acc_empty), acc_phase ^ 1, a.status));
        if (ok) {
          tc_fence_after();
          for (int s = 0; s < F.n_slabs; ++s) {
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(full + ls), lph, a.status) &&
                                             mbar_wait(smem_u32(bready + bs), bph, a.status));
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) {
              const uint32_t sa = smem_u32(lring + ls * kNvLoadStage);
              const uint32_t sb = smem_u32(bring + bs * kNvBStage);
              for (int j = 0; j < P.nb; ++j)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  mma_bf16(tmem + static_cast<uint32_t>(j * kNvTile), desc_sw128(sa + j * kNvABytes + k * 32),
                           desc_sw128(sb + k * 32), id, (s > 0 || k > 0) ? 1u : 0u);
              tc_commit(smem_u32(lempty + ls));
              tc_commit(smem_u32(bempty + bs));
            }
            __syncwarp();
            if (++ls == kNvLoadStages) {
              ls = 0;
              lph ^= 1;
            }
            if (++bs == kNvBStages) {
              bs = 0;
              bph ^= 1;
            }
          }
        }
        if (!ok) break;
        if (lane == 0) tc_commit(smem_u32(acc_full));
        __syncwarp();
        acc_phase ^= 1;
      }
    }
    if (!ok) *abort_flag = 1;
  } else if (warp < 2 + kNvConvThreads / 32) {
    // ---------------- converters: packed NVFP4 slab -> 128-byte-swizzled bf16 tile, a row each ----------------
    const int ctid = threadIdx.x - 64;
    int ls = 0, bs = 0;
    uint32_t lph = 0, bph = 0;
    bool ok = true;
    for (int ph = kPh0; ok && ph <= kPh1; ++ph) {
      const NvPhase& F = a.ph[ph];
      const NvPassView V = pass_view(a, ph);
      int t = blockIdx.x, p = 0, ep = -1;
      RowPass P;
      while (!__any_sync(0xffffffffu, *abort_flag != 0) && next_row_pass<BN>(V, msum, t, p, ep, P)) {
        for (int s = 0; s < F.n_slabs; ++s) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(full + ls), lph, a.status) &&
                                           mbar_wait(smem_u32(bempty + bs), bph ^ 1, a.status));
          if (!ok) break;
          convert_row(lring + ls * kNvLoadStage + kNvPOff, bring + bs * kNvBStage, ctid);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(smem_u32(bready + bs));
          if (++ls == kNvLoadStages) {
            ls = 0;
            lph ^= 1;
          }
          if (++bs == kNvBStages) {
            bs = 0;
            bph ^= 1;
          }
        }
        if (!ok) break;
      }
    }
    if (!ok) *abort_flag = 1;
  } else {
    // ---------------- epilogue (warps 10..13): thread = token row m of each block ----------------
    const int q = warp & 3;
    const int m = q * 32 + lane;
    const bool warp_has_rows = q * 32 < BN;   // warp-uniform
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int ph = kPh0; ok && ph <= kPh1; ++ph) {
      const NvPhase& F = a.ph[ph];
      const NvPassView V = pass_view(a, ph);
      int t = blockIdx.x, p = 0, ep = -1;
      RowPass P;
      while (next_row_pass<BN>(V, msum, t, p, ep, P)) {
        const int wt = t % F.n_wt;
        ok = mbar_wait(smem_u32(acc_full), acc_phase, a.status) && *abort_flag == 0;
        ok = named_barrier_and(1, 128, ok);
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const float ts = __ldg(F.tscale + P.e);
        for (int j = 0; j < P.nb; ++j) {
          const uint32_t acc = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(j * kNvTile);
          const int row = (P.rb + j) * BN + m;
          const int row_e = (m < BN && row < msum) ? __ldg(a.expert_ids + row) : -1;
          const bool mine = row_e == P.e;
          if (ph == 0) {
            const float wr = (a.row_w != nullptr && mine) ? __ldg(a.row_w + __ldg(a.row_ids + row)) : 1.f;
            // pass 1: h over the 128 columns, written back over the gate columns of the accumulator,
            // and its amax; pass 2: read h back, quantise, store
            if (warp_has_rows) {
              float amax = 0.f;
#pragma unroll 1
              for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t g[2][16], u[2][16];
                tc_ld_x16(acc + c0, g[0]);
                tc_ld_x16(acc + c0 + 16, g[1]);
                tc_ld_x16(acc + 128 + c0, u[0]);
                tc_ld_x16(acc + 128 + c0 + 16, u[1]);
                tc_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  const float h = silu_mul_nv(__uint_as_float(g[i >> 4][i & 15]) * ts,
                                              __uint_as_float(u[i >> 4][i & 15]) * ts) * wr;
                  amax = fmaxf(amax, fabsf(h));
                  g[i >> 4][i & 15] = __float_as_uint(h);
                }
                tc_st_x16(acc + c0, g[0]);
                tc_st_x16(acc + c0 + 16, g[1]);
              }
              tc_wait_st();
              const int ex = ue8m0_exponent(amax);
              const float sc = pow2_neg(ex);
              uint4* dst = reinterpret_cast<uint4*>(a.h_q + static_cast<size_t>(row) * F.out_cols + wt * 128);
#pragma unroll 1
              for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t g[2][16];
                tc_ld_x16(acc + c0, g[0]);
                tc_ld_x16(acc + c0 + 16, g[1]);
                tc_wait_ld();
                uint32_t packed[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  float h[4];
#pragma unroll
                  for (int v = 0; v < 4; ++v) {
                    const int c = 4 * i + v;
                    h[v] = __uint_as_float(g[c >> 4][c & 15]);
                  }
                  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(h[0] * sc, h[1] * sc), __NV_SATFINITE, __NV_E4M3);
                  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(h[2] * sc, h[3] * sc), __NV_SATFINITE, __NV_E4M3);
                  packed[i] = lo | (hi << 16);
                }
                if (mine) {
                  dst[c0 / 16] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                  dst[c0 / 16 + 1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                }
              }
              if (mine) a.h_sf[act_sf_offset(BN, a.sf_nb, row, wt)] = static_cast<uint8_t>(ex + 127);
            }
          } else {
            const int ncols = min(kNvTile, F.out_cols - wt * kNvTile);
            if (warp_has_rows) {
              uint4* dst = reinterpret_cast<uint4*>(a.y + static_cast<size_t>(row) * F.out_cols + wt * kNvTile);
#pragma unroll 1
              for (int c0 = 0; c0 < kNvTile; c0 += 32) {
                uint32_t v[2][16];
                tc_ld_x16(acc + c0, v[0]);
                tc_ld_x16(acc + c0 + 16, v[1]);
                tc_wait_ld();
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[i >> 3][(2 * i) & 15]) * ts));
                  const uint32_t hi =
                      __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[i >> 3][(2 * i + 1) & 15]) * ts));
                  packed[i] = lo | (hi << 16);
                }
                if (mine && c0 < ncols) {
#pragma unroll
                  for (int c = 0; c < 4; ++c)
                    dst[c0 / 8 + c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
                }
              }
            }
            if (a.red.out) fused_reduce_tail(a.red, a.y, F.out_cols, mine, row, wt, F.n_wt, wt * kNvTile, ncols);
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(acc_empty));
        acc_phase ^= 1;
      }
    }
    if (!ok) *abort_flag = 1;
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
// gather_ids non-null: x and sf are token-order ([T, Kd] codes, [T, Kd/128] plain scales) and row r
// reads token gather_ids[r] / K.
__global__ void __launch_bounds__(256) act_to_bf16_kernel(const uint8_t* __restrict__ x, const uint8_t* __restrict__ sf,
                                                          const int32_t* __restrict__ expert_ids,
                                                          const int32_t* __restrict__ m_sum, int U, int Kd, int bt,
                                                          int nb, uint16_t* __restrict__ xb,
                                                          const int32_t* __restrict__ gather_ids, int K, int T) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int msum = *m_sum;
  for (int r = blockIdx.x * 8 + warp; r < msum && r < U; r += gridDim.x * 8) {
    if (__ldg(expert_ids + r) < 0) continue;
    int src = r;
    if (gather_ids != nullptr) {
      src = __ldg(gather_ids + r) / K;
      if (src < 0 || src >= T) continue;
    }
    for (int k0 = lane * 8; k0 < Kd; k0 += 256) {
      const uint32_t b = gather_ids != nullptr ? sf[static_cast<size_t>(src) * (Kd / 128) + k0 / 128]
                                               : sf[act_sf_offset(bt, nb, r, k0 / 128)];
      const float sc = b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);   // 2^(b-127)
      const uint2 c = *reinterpret_cast<const uint2*>(x + static_cast<size_t>(src) * Kd + k0);
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
    // codes: byte o = (half, row n, j) -> code byte 16 * half + j of row n's 32 (see kNvChunk)
    const int n = code ? (o % (kNvTile * 16)) / 16 : (o - kNvTile * 32) / 4;
    const int cb = code ? (o / (kNvTile * 16)) * 16 + o % 16 : 0;
    const int h = n / 128, mm = n % 128;
    const int r = pair == 2 ? h * (N / 2) + wt * 128 + mm : wt * 256 + n;
    if (code)
      out[i] = r < N ? q[(static_cast<size_t>(e) * N + r) * (Kd / 2) + s * 32 + cb] : 0;
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

// Tensor map over bf16 activation rows [U, Kd] (box: 64 columns x BN rows, 128-byte swizzle).
static bool make_rows_map(CUtensorMap* m, const uint16_t* rows, int Kd, int U, int BN) {
  EncodeTiledFnNv enc = get_encode_nv();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(Kd), static_cast<cuuint64_t>(U)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(Kd) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kNvSlab), static_cast<cuuint32_t>(BN)};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(rows), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static void fill_phase(const NvLaunch& L, bool l1, int nitems_per_wt, NvPhase& F) {
  const int pair = l1 ? 2 : 1;
  F.w = L.w;
  F.tscale = L.tscale;
  F.n_wt = pair == 2 ? L.w_rows / kNvTile : (L.w_rows + kNvTile - 1) / kNvTile;
  F.n_slabs = L.Kd / kNvSlab;
  F.w_bytes = static_cast<size_t>(L.E) * F.n_wt * F.n_slabs * kNvChunk;
  F.out_cols = l1 ? L.I : L.w_rows;
  F.n_tiles = nitems_per_wt * F.n_wt;
}

// L1 (l1 non-null) or L2 (l2 non-null).
template <int BN>
static cudaError_t launch_nv_t(const NvLaunch* l1, const NvLaunch* l2, cudaStream_t stream) {
  const NvLaunch& L = l1 ? *l1 : *l2;
  CUtensorMap mx = {};
  if (!make_rows_map(&mx, L.xb, L.Kd, L.U, BN)) return cudaErrorInvalidValue;
  NvArgs a{};
  a.one_expert_blocks = L.align % BN == 0;
  // items: halves of row-block pairs (blocks of up to 32 rows), whole pairs, or blocks
  a.split_pairs = BN <= 32;
  const int nrb = (L.U + BN - 1) / BN;
  const int per_wt = a.one_expert_blocks ? (a.split_pairs ? (nrb + 1) / 2 * 2 : (nrb + 1) / 2) : nrb;
  fill_phase(L, l1 != nullptr, per_wt, a.ph[l1 ? 0 : 1]);
  a.expert_ids = L.expert_ids;
  a.m_sum = L.m_sum;
  a.h_q = L.h_q;
  a.h_sf = L.h_sf;
  a.y = L.y;
  a.status = L.status;
  a.sf_nb = act_sf_blocks(L.U, BN);
  a.red = L.red;
  a.row_ids = L.row_ids;
  a.row_w = L.row_w;
  const int total = a.ph[l1 ? 0 : 1].n_tiles;
  int grid = num_sms();
  if (grid > total) grid = total;
  if (grid < 1) grid = 1;
  if (l1) {
    cudaError_t err = cudaFuncSetAttribute(moe_gemm_nv_kernel<BN, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kNvSmem);
    if (err != cudaSuccess) return err;
    moe_gemm_nv_kernel<BN, 1><<<grid, kNvThreads, kNvSmem, stream>>>(mx, a);
  } else {
    cudaError_t err = cudaFuncSetAttribute(moe_gemm_nv_kernel<BN, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kNvSmem);
    if (err != cudaSuccess) return err;
    moe_gemm_nv_kernel<BN, 2><<<grid, kNvThreads, kNvSmem, stream>>>(mx, a);
  }
  return cudaGetLastError();
}

static cudaError_t launch_nv(const NvLaunch* l1, const NvLaunch* l2, cudaStream_t stream) {
  switch (act_sf_block_rows((l1 ? l1 : l2)->align)) {
    case 16: return launch_nv_t<16>(l1, l2, stream);
    case 32: return launch_nv_t<32>(l1, l2, stream);
    case 64: return launch_nv_t<64>(l1, l2, stream);
    default: return launch_nv_t<128>(l1, l2, stream);
  }
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
                               int U, int Kd, int align, uint16_t* xb, cudaStream_t stream, const int32_t* gather_ids,
                               int K, int T) {
  const int bt = act_sf_block_rows(align);
  const int blocks = (U + 7) / 8 < 4 * num_sms() ? (U + 7) / 8 : 4 * num_sms();
  act_to_bf16_kernel<<<blocks > 0 ? blocks : 1, 256, 0, stream>>>(x, sf, expert_ids, m_sum, U, Kd, bt,
                                                                  act_sf_blocks(U, bt), xb, gather_ids, K, T);
  return cudaGetLastError();
}

cudaError_t launch_gemm_nv(const NvLaunch& L, bool l1, cudaStream_t stream) {
  return l1 ? launch_nv(&L, nullptr, stream) : launch_nv(nullptr, &L, stream);
}

}  // namespace moe
