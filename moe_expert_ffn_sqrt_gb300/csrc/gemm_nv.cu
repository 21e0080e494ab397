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
// Packed bytes per (tile, slab): two 4608-byte halves, one per 128 rows of the tile (the CTA of a
// pair that converts those rows loads its half with one copy).  A half holds code bytes 0..15 of
// its 128 rows (2 KB, rows consecutive: a converter thread's 16-byte loads are conflict-free), then
// code bytes 16..31 (2 KB), then the rows' 4 E4M3 scales (512 B).
constexpr int kNvHalfChunk = 128 * 36;
constexpr int kNvChunk = 2 * kNvHalfChunk;
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
  const uint8_t* hp = packed + (n >> 7) * kNvHalfChunk;
  const int m = n & 127;
  const uint4 c0 = *reinterpret_cast<const uint4*>(hp + m * 16);
  const uint4 c1 = *reinterpret_cast<const uint4*>(hp + 2048 + m * 16);
  const uint32_t sc = *reinterpret_cast<const uint32_t*>(hp + 4096 + m * 4);
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

// Drains one accumulator (this warp's lane quarter at TMEM address acc) for token row `row` (stored
// when mine) of weight tile wt: L1 (ph 0) SwiGLU + FP8 requant into h_q / h_sf, L2 bf16 y (+ the
// fused reduce).  Called by all four epilogue warps together.
template <int BN>
__device__ __forceinline__ void nv_drain(const NvArgs& a, const NvPhase& F, int ph, uint32_t acc, int row,
                                         bool mine, int wt, float ts, bool warp_has_rows) {
  // 32-byte stores when the output base allows (row strides are multiples of 32 bytes)
  const bool v8 = ((reinterpret_cast<uintptr_t>(ph == 0 ? static_cast<const void*>(a.h_q) : static_cast<const void*>(a.y)) &
                    31) == 0);
  if (ph == 0) {
    const float wr = (a.row_w != nullptr && mine) ? __ldg(a.row_w + __ldg(a.row_ids + row)) : 1.f;
    // pass 1: h over the 128 channels, written back over the gate columns of the accumulator,
    // and its amax; pass 2: read h back, quantise, store.  Channel c's gate product is in column
    // gcol(c) = (c & 63) + 128 * (c >> 6), its up product in gcol(c) + 64 (the W13 tile order).
    if (warp_has_rows) {
      float amax = 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 32) {
        const uint32_t gc = static_cast<uint32_t>((c0 & 63) + 128 * (c0 >> 6));
        uint32_t g[2][16], u[2][16];
        tc_ld_x16(acc + gc, g[0]);
        tc_ld_x16(acc + gc + 16, g[1]);
        tc_ld_x16(acc + gc + 64, u[0]);
        tc_ld_x16(acc + gc + 80, u[1]);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float h = silu_mul_nv(__uint_as_float(g[i >> 4][i & 15]) * ts,
                                      __uint_as_float(u[i >> 4][i & 15]) * ts) * wr;
          amax = fmaxf(amax, fabsf(h));
          g[i >> 4][i & 15] = __float_as_uint(h);
        }
        tc_st_x16(acc + gc, g[0]);
        tc_st_x16(acc + gc + 16, g[1]);
      }
      tc_wait_st();
      const int ex = ue8m0_exponent(amax);
      const float sc = pow2_neg(ex);
      uint4* dst = reinterpret_cast<uint4*>(a.h_q + static_cast<size_t>(row) * F.out_cols + wt * 128);
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 32) {
        const uint32_t gc = static_cast<uint32_t>((c0 & 63) + 128 * (c0 >> 6));
        uint32_t g[2][16];
        tc_ld_x16(acc + gc, g[0]);
        tc_ld_x16(acc + gc + 16, g[1]);
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
          if (v8)   // 32 codes as one whole-sector store
            st_global_v8(dst + c0 / 16, packed[0], packed[1], packed[2], packed[3], packed[4], packed[5], packed[6],
                         packed[7]);
          else {
            dst[c0 / 16] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            dst[c0 / 16 + 1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
          }
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
          if (v8) {   // whole-sector stores
            st_global_v8(dst + c0 / 8, packed[0], packed[1], packed[2], packed[3], packed[4], packed[5], packed[6],
                         packed[7]);
            st_global_v8(dst + c0 / 8 + 2, packed[8], packed[9], packed[10], packed[11], packed[12], packed[13],
                         packed[14], packed[15]);
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              dst[c0 / 8 + c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
          }
        }
      }
    }
    if (a.red.out) fused_reduce_tail(a.red, a.y, F.out_cols, mine, row, wt, F.n_wt, wt * kNvTile, ncols);
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
          nv_drain<BN>(a, F, ph, acc, row, mine, wt, ts, warp_has_rows);
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

// ------------------------------------------------------------------------------------------
// CTA pairs for 128-row blocks (cta_group::2).  The two CTAs of a cluster run one MMA of M = 256
// token rows (two row blocks, one per CTA) x N = 256 weight rows, each CTA holding half of the
// weight tile: so each converts 128 weight rows per slab instead of 256, for the same tensor work
// per SM.  With both TMEM accumulators a pass covers up to four row blocks of one expert (a
// "quad": blocks 4q, 4q+1 in the even CTA, 4q+2, 4q+3 in the odd one).  The even CTA issues the
// MMAs; each CTA loads its own token rows and its half of the packed chunk, converts its half, and
// drains its own accumulator rows.  Cross-CTA signals: converter warps and epilogue warps of both
// CTAs arrive on the even CTA's bf16-ready and accumulator-empty barriers; the MMA commits arrive
// on both CTAs' slot-empty and accumulator-full barriers (multicast).

constexpr int kNvHalfRows = kNvTile / 2;
static_assert(kNvHalfChunk == kNvHalfRows * 36, "a half chunk is 128 rows x (32 code bytes + 4 scales)");
constexpr int kNvPairLoadStage = (2 * kNvABytes + kNvHalfChunk + 1023) / 1024 * 1024;   // 37 KB
constexpr int kNvPairLoadStages = 4;
constexpr int kNvPairBStage = kNvHalfRows * 128;                                        // 16 KB
constexpr int kNvPairBStages = 4;
// The load slot and the bf16 slot of a slab advance together, so one barrier (the load slot's
// "empty") releases both: one MMA commit per slab.
static_assert(kNvPairBStages == kNvPairLoadStages, "load and bf16 slots advance together");
constexpr int kNvMaxRuns = 1024;                                        // experts with rows
constexpr int kNvRunBytes = kNvMaxRuns * 2 * 2 + (kNvMaxRuns + 2) * 4;   // run table
constexpr int kNvPairSmem =
    1024 + kNvPairLoadStages * kNvPairLoadStage + kNvPairBStages * kNvPairBStage + kNvExtra + kNvRunBytes;
static_assert(kNvPairSmem <= kNvBudget, "shared memory budget (pair)");
// Row blocks whose first-row experts the prologue stages in the (then unused) load ring.
constexpr int kNvPairMaxBlocks = kNvPairLoadStages * kNvPairLoadStage / 4;
constexpr uint32_t kNvConvWarps = kNvConvThreads / 32;

// Passes of a CTA pair.  An expert's row blocks are consecutive (a run); its passes take them four
// at a time (c <= 4 blocks from b0).  Slot j of a pass is an accumulator: with 2j + 1 < c it holds two
// blocks, b0 + 2j in the even CTA and b0 + 2j + 1 in the odd one (an M = 256 MMA); with 2j + 1 == c it
// holds block b0 + 2j alone, split by rows: rows 0..63 in the even CTA, 64..127 in the odd one (an
// M = 128 MMA, so a lone block costs no more tensor time than on one SM).  A run of n blocks makes
// ceil(n / 4) passes and a pass never mixes experts.
struct PairPass {
  int e, b0, c;
};

// Run table in shared memory, built by every CTA at kernel start from expert_ids (one entry per
// block: its first row's expert; blocks hold one expert each).
struct RunTable {
  uint16_t* start;   // [kNvMaxRuns] first block of run i
  uint16_t* len;     // [kNvMaxRuns] blocks of run i
  int* pfx;          // [kNvMaxRuns + 2] passes before run i; pfx[n] = all passes; last: n
  int n;             // runs
};

// Pass `pi` of the table (pfx[i] <= pi < pfx[i + 1] for run i).
__device__ __forceinline__ PairPass pair_pass(const RunTable& R, const int32_t* expert_ids, int pi) {
  int lo = 0, hi = R.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (R.pfx[mid] <= pi) lo = mid;
    else hi = mid - 1;
  }
  const int o = 4 * (pi - R.pfx[lo]);
  PairPass P;
  P.b0 = R.start[lo] + o;
  P.c = min(4, static_cast<int>(R.len[lo]) - o);
  P.e = __ldg(expert_ids + static_cast<size_t>(P.b0) * 128);
  return P;
}

// Slot j of the pass: 2 = a block per CTA (M = 256), 1 = one block split by rows (M = 128), 0 = unused.
__device__ __forceinline__ int pair_slot(const PairPass& P, int j) {
  return 2 * j + 1 < P.c ? 2 : (2 * j + 1 == P.c ? 1 : 0);
}

// Converts part h (codes 32h .. 32h+31) of weight row n of this CTA's half tile.  The half chunk in
// shared memory: code bytes 0..15 of its 128 rows (2 KB), then bytes 16..31 (2 KB), then 128 x 4
// E4M3 scales.
__device__ __forceinline__ void convert_half_row(const uint8_t* __restrict__ packed, uint8_t* __restrict__ btile,
                                                 int n, int h) {
  const uint4 c = *reinterpret_cast<const uint4*>(packed + h * (kNvHalfRows * 16) + n * 16);
  const uint32_t sc = *reinterpret_cast<const uint32_t*>(packed + kNvHalfRows * 32 + n * 4) >> (16 * h);
  uint32_t s2[2];
  e4m3x2_to_bf16x2(sc, s2[0], s2[1]);
  const uint32_t words[4] = {c.x, c.y, c.z, c.w};
  const uint32_t row = smem_u32(btile) + static_cast<uint32_t>(n) * 128;
  const uint32_t x = static_cast<uint32_t>(n & 7) << 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t q[4];
    e2m1x8_to_bf16(words[i], s2[i >> 1], q);
    const uint32_t addr = row | ((static_cast<uint32_t>(4 * h + i) << 4) ^ x);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(q[0]), "r"(q[1]), "r"(q[2]), "r"(q[3])
                 : "memory");
  }
}

// Drains a split slot (an M = 128 MMA over the pair): this CTA's 64 rows of the block, each row in
// two lanes.  Lanes 0..63 (epilogue warps 0, 1) hold output columns 0..127 of row lane, lanes
// 64..127 (warps 2, 3) columns 128..255 of row lane - 64; `half` is 0 or 1 accordingly and acc
// already names this warp's lane quarter.  L1: a half holds 64 channels (gate products in columns
// 0..63, up in 64..127), and the row's amax is combined through xa[64] in shared memory.  Called by
// all four epilogue warps together.
template <int BN>
__device__ __forceinline__ void nv_drain_split(const NvArgs& a, const NvPhase& F, int ph, uint32_t acc, int row,
                                               bool mine, int half, int rl, int wt, float ts, float* xa) {
  const bool v8 = ((reinterpret_cast<uintptr_t>(ph == 0 ? static_cast<const void*>(a.h_q) : static_cast<const void*>(a.y)) &
                    31) == 0);
  if (ph == 0) {
    const float wr = (a.row_w != nullptr && mine) ? __ldg(a.row_w + __ldg(a.row_ids + row)) : 1.f;
    float amax = 0.f;
#pragma unroll 1
    for (int c0 = 0; c0 < 64; c0 += 32) {
      uint32_t g[2][16], u[2][16];
      tc_ld_x16(acc + c0, g[0]);
      tc_ld_x16(acc + c0 + 16, g[1]);
      tc_ld_x16(acc + 64 + c0, u[0]);
      tc_ld_x16(acc + 64 + c0 + 16, u[1]);
      tc_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float h = silu_mul_nv(__uint_as_float(g[i >> 4][i & 15]) * ts, __uint_as_float(u[i >> 4][i & 15]) * ts) * wr;
        amax = fmaxf(amax, fabsf(h));
        g[i >> 4][i & 15] = __float_as_uint(h);
      }
      tc_st_x16(acc + c0, g[0]);
      tc_st_x16(acc + c0 + 16, g[1]);
    }
    tc_wait_st();
    if (half) xa[rl] = amax;
    named_barrier(1, 128);
    if (!half) {
      amax = fmaxf(amax, xa[rl]);
      xa[rl] = amax;
    }
    named_barrier(1, 128);
    if (half) amax = xa[rl];
    const int ex = ue8m0_exponent(amax);
    const float sc = pow2_neg(ex);
    uint4* dst = reinterpret_cast<uint4*>(a.h_q + static_cast<size_t>(row) * F.out_cols + wt * 128 + 64 * half);
#pragma unroll 1
    for (int c0 = 0; c0 < 64; c0 += 32) {
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
        if (v8)
          st_global_v8(dst + c0 / 16, packed[0], packed[1], packed[2], packed[3], packed[4], packed[5], packed[6],
                       packed[7]);
        else {
          dst[c0 / 16] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
          dst[c0 / 16 + 1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        }
      }
    }
    if (mine && !half) a.h_sf[act_sf_offset(BN, a.sf_nb, row, wt)] = static_cast<uint8_t>(ex + 127);
  } else {
    const int tcols = min(kNvTile, F.out_cols - wt * kNvTile);
    const int ncols = tcols - 128 * half;   // this half's columns (a last half tile may have none)
    if (ncols > 0) {
      uint4* dst = reinterpret_cast<uint4*>(a.y + static_cast<size_t>(row) * F.out_cols + wt * kNvTile + 128 * half);
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 32) {
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
          if (v8) {   // whole-sector stores
            st_global_v8(dst + c0 / 8, packed[0], packed[1], packed[2], packed[3], packed[4], packed[5], packed[6],
                         packed[7]);
            st_global_v8(dst + c0 / 8 + 2, packed[8], packed[9], packed[10], packed[11], packed[12], packed[13],
                         packed[14], packed[15]);
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              dst[c0 / 8 + c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
          }
        }
      }
    }
    if (a.red.out) {
      named_barrier(1, 128);   // both halves of each row stored before its row owner takes a ticket
      fused_reduce_tail(a.red, a.y, F.out_cols, mine && !half, row, wt, F.n_wt, wt * kNvTile, tcols);
    }
  }
}

// Warp roles as in moe_gemm_nv_kernel; warp 1 of the odd CTA only takes part in the tensor-memory
// allocation.  MODE 1: L1 items, 2: L2 items.  Launched in clusters of two CTAs; item t = pass
// (t / n_wt) of the run table against weight tile t % n_wt, cluster c taking items c, c + clusters, ...
template <int MODE>
__global__ void __launch_bounds__(kNvThreads, 1)
    moe_gemm_nv_pair_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_x64,
                            const NvArgs a) {
  constexpr int BN = 128;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* lring = smem;                                       // token rows of two blocks + half chunk
  uint8_t* bring = smem + kNvPairLoadStages * kNvPairLoadStage;   // bf16 half tiles
  uint8_t* extra = bring + kNvPairBStages * kNvPairBStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(extra);         // load slot filled (TMA + bulk copies)
  uint64_t* lempty = full + kNvPairLoadStages;                 // load + bf16 slot consumed (pair MMA commit)
  uint64_t* bready = lempty + kNvPairLoadStages;               // even CTA: both halves written
  uint64_t* bempty = bready + kNvPairBStages;                  // unused (lempty releases both slots)
  uint64_t* acc_full = bempty + kNvPairBStages;                // [2] accumulator b written
  uint64_t* acc_empty = acc_full + 2;                          // [2] even CTA: both CTAs drained b
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xa = reinterpret_cast<float*>(extra + 256);          // [64] row amax of split slots (L1)
  RunTable R;
  R.start = reinterpret_cast<uint16_t*>(extra + kNvExtra);
  R.len = R.start + kNvMaxRuns;
  R.pfx = reinterpret_cast<int*>(R.len + kNvMaxRuns);
  constexpr int kPh = (MODE & 1) ? 0 : 1;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const int cluster = static_cast<int>(blockIdx.x >> 1), nclusters = static_cast<int>(gridDim.x >> 1);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kNvPairLoadStages; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(lempty + s), 1);
    }
    for (int s = 0; s < kNvPairBStages; ++s) {
      mbar_init(smem_u32(bready + s), 2 * kNvConvWarps);
      mbar_init(smem_u32(bempty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(acc_full + b), 1);
      mbar_init(smem_u32(acc_empty + b), 2 * 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmap_x);
    prefetch_tmap(&tmap_x64);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kNvTmemCols);
    tmem_relinquish_pair();
  }
  // run table: each block's expert staged in the load ring, then runs and their pass counts
  const int msum = *a.m_sum;
  const int nrb = min((msum + BN - 1) / BN, kNvPairMaxBlocks);
  int* eb = reinterpret_cast<int*>(lring);
  for (int b = threadIdx.x; b < nrb; b += blockDim.x) eb[b] = __ldg(a.expert_ids + static_cast<size_t>(b) * BN);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the ring's next writers are copies
  __syncthreads();
  if (warp == 0) {
    int ns = 0, ne = 0;
    for (int b0 = 0; b0 < nrb; b0 += 32) {
      const int b = b0 + lane;
      const int e = b < nrb ? eb[b] : -1;
      const int ep = (b > 0 && b < nrb) ? eb[b - 1] : -1;
      const int en = b + 1 < nrb ? eb[b + 1] : -1;
      const uint32_t fs = __ballot_sync(0xffffffffu, e >= 0 && e != ep);
      const uint32_t fe = __ballot_sync(0xffffffffu, e >= 0 && e != en);
      const uint32_t lt = (1u << lane) - 1u;
      if (e >= 0 && e != ep) {
        const int i = ns + __popc(fs & lt);
        if (i < kNvMaxRuns) R.start[i] = static_cast<uint16_t>(b);
      }
      if (e >= 0 && e != en) {
        const int i = ne + __popc(fe & lt);
        if (i < kNvMaxRuns) R.len[i] = static_cast<uint16_t>(b + 1);   // end, turned into a length below
      }
      ns += __popc(fs);
      ne += __popc(fe);
    }
    if (ns > kNvMaxRuns) {
      if (lane == 0) record_error(a.status, kDevErrCheck);
      ns = 0;   // no passes: every role ends at once
    }
    int base = 0;
    for (int i0 = 0; i0 < ns; i0 += 32) {
      const int i = i0 + lane;
      int np = 0;
      if (i < ns) {
        const int l = static_cast<int>(R.len[i]) - static_cast<int>(R.start[i]);
        R.len[i] = static_cast<uint16_t>(l);
        np = (l + 3) / 4;
      }
      int incl = np;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
      }
      if (i < ns) R.pfx[i] = base + incl - np;
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      R.pfx[ns] = base;
      R.pfx[kNvMaxRuns + 1] = ns;   // run count for the other roles
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers exist before any cross-CTA arrival
  tc_fence_after();
  R.n = R.pfx[kNvMaxRuns + 1];
  const uint32_t tmem = *tmem_slot;
  const NvPhase& F = a.ph[kPh];
  const int n_items = R.pfx[R.n] * F.n_wt;

  if (warp == 0) {
    // ---------------- producer: own token rows by TMA, own half of the packed chunk ----------------
    const uint64_t pol_x = policy_evict_last();
    int ls = 0;
    uint32_t lph = 0;
    bool ok = true;
    for (int t = cluster; ok && t < n_items && !__any_sync(0xffffffffu, *abort_flag != 0); t += nclusters) {
      const PairPass P = pair_pass(R, a.expert_ids, t / F.n_wt);
      const int k0 = pair_slot(P, 0), k1 = pair_slot(P, 1);
      const uint32_t tx = (k0 == 2 ? 128 : 64) * 128 + (k1 == 2 ? 128 * 128 : k1 == 1 ? 64 * 128 : 0);
      const int wt = t % F.n_wt;
      const size_t chunk0 = (static_cast<size_t>(P.e) * F.n_wt + wt) * F.n_slabs;
      for (int s = 0; s < F.n_slabs; ++s) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(lempty + ls), lph ^ 1, a.status));
        if (!ok) break;
        if (lane == 0) {
          uint8_t* st = lring + ls * kNvPairLoadStage;
          const uint32_t fb = smem_u32(full + ls);
          const size_t wbase = (chunk0 + s) * kNvChunk;
          if (wbase + kNvChunk > F.w_bytes || (reinterpret_cast<uintptr_t>(F.w) & 15)) {
            record_error(a.status, kDevErrCheck);
            *abort_flag = 1;
          } else {
            mbar_arrive_expect_tx(fb, tx + kNvHalfChunk);
            for (int j = 0; j < 2; ++j) {
              const int k = j ? k1 : k0;
              if (k == 2)
                tma_load_2d(smem_u32(st + j * kNvABytes), &tmap_x, s * kNvSlab, (P.b0 + 2 * j + rank) * BN, fb,
                            pol_x);
              else if (k == 1)
                tma_load_2d(smem_u32(st + j * kNvABytes), &tmap_x64, s * kNvSlab, (P.b0 + 2 * j) * BN + rank * 64,
                            fb, pol_x);
            }
            uint8_t* hp = st + 2 * kNvABytes;
            bulk_load(smem_u32(hp), F.w + wbase + rank * kNvHalfChunk, kNvHalfChunk, fb);
          }
        }
        __syncwarp();
        if (++ls == kNvPairLoadStages) {
          ls = 0;
          lph ^= 1;
        }
      }
    }
    if (!ok) *abort_flag = 1;
    if (__any_sync(0xffffffffu, *abort_flag != 0)) {
      // let every copy issued into shared memory land before the CTA exits
      for (int s = 0; s < kNvPairLoadStages; ++s)
        mbar_wait(smem_u32(full + s), (s < ls) ? lph : (lph ^ 1), nullptr);
    } else {
      // every slot released: the pair MMA's commits into this CTA's barriers have all landed
      for (int s = 0; s < kNvPairLoadStages; ++s) {
        mbar_wait(smem_u32(lempty + ls), lph ^ 1, a.status);
        if (++ls == kNvPairLoadStages) {
          ls = 0;
          lph ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    if (rank == 0) {
      // ---------------- MMA issuer: kind::f16 over the pair, M=256, N=256, K=16 x 4 per slab ----------------
      // One thread: the issue of a pair MMA takes ~100 cycles of its 128 cycles of tensor work, so
      // the loop between slabs is kept short (no warp votes, descriptors advanced by adding).
      if (lane == 0) {
        int ls = 0;
        uint32_t lph = 0;
        // accumulators: a two-slot pass takes both; one-slot passes alternate between them, so that
        // one pass's drain overlaps the next one's MMAs (bit b of aph: accumulator b's phase)
        uint32_t aph = 0;
        int nb = 0;
        const uint32_t id2 = idesc_bf16(2 * BN, kNvTile), id1 = idesc_bf16(BN, kNvTile);
        const uint64_t da0 = desc_sw128(smem_u32(lring)), db0 = desc_sw128(smem_u32(bring));
        bool ok = true;
        for (int t = cluster; ok && t < n_items && *abort_flag == 0; t += nclusters) {
          const PairPass P = pair_pass(R, a.expert_ids, t / F.n_wt);
          const int nacc = P.c > 2 ? 2 : 1;
          const uint32_t ids[2] = {pair_slot(P, 0) == 2 ? id2 : id1, pair_slot(P, 1) == 2 ? id2 : id1};
          const int b0 = nacc == 2 ? 0 : nb;   // accumulator of slot j: b0 + j
          for (int j = 0; ok && j < nacc; ++j)
            ok = mbar_wait(smem_u32(acc_empty + b0 + j), ((aph >> (b0 + j)) & 1u) ^ 1u, a.status);
          if (!ok) break;
          tc_fence_after();
          for (int s = 0; s < F.n_slabs; ++s) {
            // the converters of both CTAs arrive only after their CTA's load slot is full
            ok = mbar_wait(smem_u32(bready + ls), lph, a.status);
            if (!ok) break;
            tc_fence_after();
            // descriptor start addresses count 16-byte units: + 2 per 32-byte K step
            const uint64_t da = da0 + static_cast<uint64_t>(ls * (kNvPairLoadStage >> 4));
            const uint64_t db = db0 + static_cast<uint64_t>(ls * (kNvPairBStage >> 4));
            for (int j = 0; j < nacc; ++j)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_bf16_pair(tmem + static_cast<uint32_t>((b0 + j) * kNvTile),
                              da + static_cast<uint64_t>(j * (kNvABytes >> 4) + 2 * k), db + static_cast<uint64_t>(2 * k),
                              ids[j], (s > 0 || k > 0) ? 1u : 0u);
            tc_commit_pair(smem_u32(lempty + ls), 0x3);
            if (++ls == kNvPairLoadStages) {
              ls = 0;
              lph ^= 1;
            }
          }
          if (!ok) break;
          for (int j = 0; j < nacc; ++j) {
            tc_commit_pair(smem_u32(acc_full + b0 + j), 0x3);
            aph ^= 1u << (b0 + j);
          }
          if (nacc == 1) nb ^= 1;
        }
        if (!ok) *abort_flag = 1;
      }
      __syncwarp();
    }
  } else if (warp < 2 + static_cast<int>(kNvConvWarps)) {
    // ---------------- converters: half a weight row each (128 rows x 2 parts) ----------------
    const int ctid = threadIdx.x - 64;
    const int n = ctid & (kNvHalfRows - 1), h = ctid / kNvHalfRows;
    const uint32_t peer_bready = mapa_shared(smem_u32(bready), 0);
    int ls = 0, bs = 0;
    uint32_t lph = 0, bph = 0;
    bool ok = true;
    for (int t = cluster; ok && t < n_items && !__any_sync(0xffffffffu, *abort_flag != 0); t += nclusters) {
      for (int s = 0; s < F.n_slabs; ++s) {
        // the bf16 slot bs == ls is free once the slab that last used it was consumed (lempty)
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(full + ls), lph, a.status) &&
                                         mbar_wait(smem_u32(lempty + bs), bph ^ 1, a.status));
        if (!ok) break;
        convert_half_row(lring + ls * kNvPairLoadStage + 2 * kNvABytes, bring + bs * kNvPairBStage, n, h);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(peer_bready + static_cast<uint32_t>(bs * 8));
        if (++ls == kNvPairLoadStages) {
          ls = 0;
          lph ^= 1;
        }
        if (++bs == kNvPairBStages) {
          bs = 0;
          bph ^= 1;
        }
      }
    }
    if (!ok) *abort_flag = 1;
    if (ok && *abort_flag == 0) {
      // every slot released (the pair MMA's commits into this CTA have landed)
      for (int s = 0; s < kNvPairBStages; ++s) {
        mbar_wait(smem_u32(lempty + bs), bph ^ 1, a.status);
        if (++bs == kNvPairBStages) {
          bs = 0;
          bph ^= 1;
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 10..13): thread = token row m of this CTA's blocks ----------------
    const int q = warp & 3;
    const int m = q * 32 + lane;
    const uint32_t peer_acc_empty = mapa_shared(smem_u32(acc_empty), 0);
    uint32_t aph = 0;   // the MMA thread's accumulator choice, repeated
    int nb = 0;
    bool ok = true;
    for (int t = cluster; t < n_items; t += nclusters) {
      const PairPass P = pair_pass(R, a.expert_ids, t / F.n_wt);
      const int wt = t % F.n_wt;
      const int nacc = P.c > 2 ? 2 : 1;
      const int b0 = nacc == 2 ? 0 : nb;
      ok = *abort_flag == 0;
      for (int j = 0; ok && j < nacc; ++j) ok = mbar_wait(smem_u32(acc_full + b0 + j), (aph >> (b0 + j)) & 1u, a.status);
      ok = named_barrier_and(1, 128, ok);
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const float ts = __ldg(F.tscale + P.e);
      for (int j = 0; j < 2; ++j) {
        const int k = pair_slot(P, j);
        if (k == 0) continue;
        const uint32_t acc = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>((b0 + j) * kNvTile);
        if (k == 2) {
          // M = 256: this CTA's block, row m in lane m
          const int row = (P.b0 + 2 * j + static_cast<int>(rank)) * BN + m;
          const int row_e = row < msum ? __ldg(a.expert_ids + row) : -1;
          nv_drain<BN>(a, F, kPh, acc, row, row_e == P.e, wt, ts, true);
        } else {
          // M = 128: rows rank * 64 + (m & 63) of the block, output columns 128 * (m >> 6) + ...
          const int rl = m & 63;
          const int row = (P.b0 + 2 * j) * BN + static_cast<int>(rank) * 64 + rl;
          const int row_e = row < msum ? __ldg(a.expert_ids + row) : -1;
          nv_drain_split<BN>(a, F, kPh, acc, row, row_e == P.e, m >> 6, rl, wt, ts, xa);
        }
      }
      tc_fence_before();
      __syncwarp();
      for (int j = 0; j < nacc; ++j) {
        if (lane == 0) mbar_arrive_cluster(peer_acc_empty + static_cast<uint32_t>((b0 + j) * 8));
        aph ^= 1u << (b0 + j);
      }
      if (nacc == 1) nb ^= 1;
    }
    if (!ok) *abort_flag = 1;
  }
  tc_fence_before();
  cluster_sync();   // no CTA leaves while the pair MMA or the other CTA's arrivals may touch it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kNvTmemCols);
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

// Token-order activation rows -> bf16, one warp per token: the token's row (E4M3 codes x its plain
// UE8M0 scales) is read and converted once and stored to each of its K permuted rows inv_perm[t*K+k]
// (the by-row kernel above reads it once per row).  The same conversion, so the same bits.
__global__ void __launch_bounds__(256) act_to_bf16_tokens_kernel(const uint8_t* __restrict__ x,
                                                                 const uint8_t* __restrict__ sf,
                                                                 const int32_t* __restrict__ inv_perm, int T, int K,
                                                                 int U, int Kd, uint16_t* __restrict__ xb) {
  __shared__ int s_rows[8][32];   // the warp's token's K row positions (read by lanes that diverge at the row's end)
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int t = blockIdx.x * 8 + warp; t < T; t += gridDim.x * 8) {
    int rv = -1;
    if (lane < K) {
      rv = __ldg(inv_perm + static_cast<size_t>(t) * K + lane);
      if (rv < 0 || rv >= U) rv = -1;
    }
    s_rows[warp][lane] = rv;
    __syncwarp();
    const uint8_t* xr = x + static_cast<size_t>(t) * Kd;
    const uint8_t* sr = sf + static_cast<size_t>(t) * (Kd / 128);
    // four lane steps (1024 codes of the row) loaded before any is converted and stored
    for (int kb = 0; kb < Kd; kb += 1024) {
      uint2 c[4];
      uint32_t b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k0 = kb + u * 256 + lane * 8;
        c[u] = k0 < Kd ? __ldg(reinterpret_cast<const uint2*>(xr + k0)) : make_uint2(0, 0);
        b[u] = k0 < Kd ? __ldg(sr + k0 / 128) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k0 = kb + u * 256 + lane * 8;
        if (k0 >= Kd) break;
        const float sc = b[u] ? __uint_as_float(b[u] << 23) : __uint_as_float(0x00400000u);   // 2^(b-127)
        const uint32_t cw[2] = {c[u].x, c[u].y};
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
        const uint4 v = make_uint4(o[0], o[1], o[2], o[3]);
        for (int k = 0; k < K; ++k) {
          const int r = s_rows[warp][k];
          if (r >= 0) *reinterpret_cast<uint4*>(xb + static_cast<size_t>(r) * Kd + k0) = v;
        }
      }
    }
    __syncwarp();   // every lane has read s_rows before the next token's rows replace them
  }
}

// NVFP4 packing: per (expert, 256-row tile, 64-deep slab) 256 rows x 32 bytes of codes and 4 E4M3
// scales (one per 16 codes), in two halves of 128 rows (layout at kNvChunk).  A W2 tile is 256 consecutive rows; a W13 tile is
// 128 gate channels and their up rows, in the order gate 0..63, up 0..63, gate 64..127, up 64..127.
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
    // byte o: half hh of the tile (rows 128hh ..), then within the half p: codes (part, row m, j) ->
    // code byte 16 * part + j of row m's 32, then row m's 4 scales (see kNvChunk)
    const int hh = o / kNvHalfChunk, p = o % kNvHalfChunk;
    const bool code = p < 4096;
    const int n = 128 * hh + (code ? (p % 2048) / 16 : (p - 4096) / 4);
    const int cb = code ? (p / 2048) * 16 + p % 16 : 0;
    // W13 tile rows in quarters of 64: gate channels 128wt + 0..63, their up rows, gate 128wt + 64..127,
    // their up rows (a channel's gate and up products sit 64 accumulator columns apart)
    const int qd = n / 64;
    const int r = pair == 2 ? (qd & 1) * (N / 2) + wt * 128 + 64 * (qd >> 1) + (n & 63) : wt * 256 + n;
    if (code)
      out[i] = r < N ? q[(static_cast<size_t>(e) * N + r) * (Kd / 2) + s * 32 + cb] : 0;
    else
      out[i] = r < N ? sf[(static_cast<size_t>(e) * N + r) * (Kd / 16) + s * 4 + (p - 4096) % 4] : 0;
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

// The CTA-pair kernel in clusters of two: as many clusters as can be resident at once (0 when
// the device cannot host one, then the caller runs the single-CTA kernel).
template <int MODE>
static int nv_pair_clusters() {
  static int n = -1;
  if (n < 0) {
    int c = 0;
    if (cudaFuncSetAttribute(moe_gemm_nv_pair_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kNvPairSmem) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 2;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(2 * (num_sms() / 2));
      cfg.blockDim = dim3(kNvThreads);
      cfg.dynamicSmemBytes = kNvPairSmem;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&c, moe_gemm_nv_pair_kernel<MODE>, &cfg) != cudaSuccess) c = 0;
    }
    (void)cudaGetLastError();
    n = c;
  }
  return n;
}

template <int MODE>
static cudaError_t launch_nv_pair(const CUtensorMap& mx, const CUtensorMap& mx64, const NvArgs& a, int items,
                                  int clusters, cudaStream_t stream) {
  if (clusters > items) clusters = items;
  if (clusters < 1) clusters = 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(kNvThreads);
  cfg.dynamicSmemBytes = kNvPairSmem;
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_gemm_nv_pair_kernel<MODE>, mx, mx64, a);
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
  if (BN == 128 && a.one_expert_blocks && L.E <= kNvMaxRuns && nrb <= kNvPairMaxBlocks) {
    // 128-row blocks: CTA pairs over each expert's blocks, four at a time (the kernel counts the
    // passes; nrb bounds them for the grid)
    const int clusters = l1 ? nv_pair_clusters<1>() : nv_pair_clusters<2>();
    if (clusters > 0) {
      CUtensorMap mx64 = {};
      if (!make_rows_map(&mx64, L.xb, L.Kd, L.U, 64)) return cudaErrorInvalidValue;
      NvArgs b = a;
      fill_phase(L, l1 != nullptr, nrb, b.ph[l1 ? 0 : 1]);
      const int items = b.ph[l1 ? 0 : 1].n_tiles;
      return l1 ? launch_nv_pair<1>(mx, mx64, b, items, clusters, stream)
                : launch_nv_pair<2>(mx, mx64, b, items, clusters, stream);
    }
  }
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

cudaError_t launch_act_to_bf16_tokens(const uint8_t* x, const uint8_t* sf, const int32_t* inv_perm, int T, int K, int U,
                                      int Kd, uint16_t* xb, cudaStream_t stream) {
  if (K < 1 || K > 32) return cudaErrorInvalidValue;
  const int blocks = (T + 7) / 8 < 8 * num_sms() ? (T + 7) / 8 : 8 * num_sms();
  act_to_bf16_tokens_kernel<<<blocks > 0 ? blocks : 1, 256, 0, stream>>>(x, sf, inv_perm, T, K, U, Kd, xb);
  return cudaGetLastError();
}

cudaError_t launch_gemm_nv(const NvLaunch& L, bool l1, cudaStream_t stream) {
  return l1 ? launch_nv(&L, nullptr, stream) : launch_nv(nullptr, &L, stream);
}

}  // namespace moe
