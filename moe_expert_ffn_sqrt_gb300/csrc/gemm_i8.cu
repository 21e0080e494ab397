// Grouped GEMMs of the INT8 (W8A8) variant on tcgen05 (sm_103a).  Page "INT8 高吞吐/低延迟 EP 代码梳理"
// §2 (INT8 dispatch, quant_dtype int8), §3.1 (INT8 with channel-wise weights), §11.6.2 (activations
// quantised per token): weights are int8 codes with one fp32 scale per output channel, activations
// int8 codes with one fp32 scale per row.  L1 = SwiGLU of x W13^T, stored as bf16 h (quantised per
// row afterwards by quant_rows_i8_kernel, which needs the whole row's amax); L2 = h W2^T, bf16 y
// (+ the fused unpermute-reduce, as in gemm.cu).
//
// GB300's int8 tensor rate is far below its 16-bit rate, so the products run on kind::f16 with fp16
// operands: every int8 code is exact in fp16 and so is every product of two codes (|p| <= 16129);
// the tensor core sums them in fp32, which is exact while the partial sums keep within fp32's 24-bit
// significand.  The row and channel scales multiply the fp32 accumulator in the epilogue.
//  * activation rows become fp16 rows of codes once per call (i8_rows_to_f16_kernel; for L1 it also
//    gathers the token rows through sorted_token_ids) and reach shared memory by TMA;
//  * each (expert, 256-row weight tile, 64-deep slab) chunk of int8 codes (16 KB) arrives by one bulk
//    copy, and ten converter warps turn it into a 128-byte-swizzled fp16 tile;
//  * two 256-column TMEM accumulators hold two row blocks of one expert that share each converted
//    tile; four epilogue warps drain them 32 columns at a time.
// The load ring keeps only the rows a row block holds (BN x 128 bytes per block and slab), so small
// blocks leave room for a deeper ring; the MMA's 128-row operand window of a block stays inside its
// ring slot (rows past BN are never stored).
//
// [256, 256] block-quantised weights (BLOCK): the scale of a product changes every 256 columns of
// the reduction (one per activation row and group, one per weight block), so one fp32 accumulator
// cannot take the whole reduction.  Each 256-deep K-block (four slabs) is accumulated alone in TMEM
// columns [0, 256) -- exact, since 256 products of two int8 codes sum to less than 2^24 -- and the
// epilogue folds it, times the row's group scale and the weight block's scale, into a running fp32
// sum kept in TMEM columns [256, 512); the last K-block's fold feeds the SwiGLU (L1) or the bf16
// output (L2) directly.  A pass then holds one row block (the second accumulator's columns hold the
// sum), and the MMA waits for each fold.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "passes.cuh"

namespace moe {

namespace {

constexpr int kI8Threads = 512;          // warp 0 TMA, 1 MMA, 2..11 convert, 12..15 epilogue
constexpr int kI8ConvThreads = 320;
constexpr int kI8ConvBatch = 4;          // conversion tasks per thread with loads issued together
constexpr int kI8Budget = 227 * 1024;
constexpr uint32_t kI8TmemCols = 512;    // two 256-column accumulators
constexpr int kI8Tile = 256;             // weight rows per tile (MMA N)
constexpr int kI8Slab = 64;              // K per pipeline stage (64 fp16 = one 128-byte row)
constexpr int kI8Chunk = kI8Tile * kI8Slab;   // int8 codes per (tile, slab)
constexpr int kI8BStage = kI8Tile * 128;      // fp16 weight tile, 128-byte swizzle
constexpr int kI8Extra = 1024;
static_assert(kI8ConvThreads % 32 == 0 && 2 + kI8ConvThreads / 32 + 4 == kI8Threads / 32, "warp roles");

// Shared-memory plan for row blocks of BN rows: load slots of [block 0 rows][block 1 rows][codes].
// Block-quantised weights with blocks of up to 32 rows keep the running K-block sum in shared
// memory ([BN rows][257 floats], conflict-free column walks), so that the two TMEM accumulators take
// alternate K-blocks and each fold overlaps the next K-block's MMAs.
template <int BN, bool BLOCK = false>
struct I8Cfg {
  static constexpr int kABytes = BN * 128;
  static constexpr int kPOff = 2 * kABytes;
  static constexpr int kStage = (kPOff + kI8Chunk + 1023) / 1024 * 1024;
  static constexpr int kBStages = 2;
  static constexpr bool kSumSmem = BLOCK && BN <= 32;
  static constexpr int kSumStride = 257;
  static constexpr int kSumBytes = kSumSmem ? (BN * kSumStride * 4 + 1023) / 1024 * 1024 : 0;
  static constexpr int kFit = (kI8Budget - 1024 - kBStages * kI8BStage - kSumBytes - kI8Extra) / kStage;
  static constexpr int kStages = kFit > 8 ? 8 : kFit;
  static constexpr int kSmem = 1024 + kStages * kStage + kBStages * kI8BStage + kSumBytes + kI8Extra;
  static_assert(kStages >= 2 && kSmem <= kI8Budget, "shared memory budget");
  static_assert(kABytes + 128 * 128 <= kStage, "the MMA's 128-row window of block 1 stays in its slot");
};

struct I8Args {
  const uint8_t* w;             // packed int8 weight stream
  const float* col_scale;       // [E, w_rows] per-output-channel scales, logical row order
  const float* row_scale;       // [U] per-row activation scales
  const int32_t* expert_ids;
  const int32_t* m_sum;
  uint16_t* out;                // L1: h [U, I] bf16; L2: y [U, H] bf16
  uint32_t* status;
  size_t w_bytes;
  int n_slabs;                  // K / 64
  int n_wt;
  int w_rows;                   // 2I (L1) or H (L2)
  int out_cols;                 // I (L1) or H (L2)
  int n_tiles;
  int one_expert_blocks;        // permute alignment is a multiple of BN: one expert per row block
  int split_pairs;              // items are halves of row-block pairs (small blocks) or whole pairs
  int pair_blocks;              // two blocks of one expert may share a pass (not with block scales)
  int nkb;                      // BLOCK: 256-deep K-blocks (row_scale [U, nkb], col_scale [E, w_rows/256, nkb])
  FusedReduce red;              // L2: unpermute-reduce in the epilogue when red.out != nullptr
};

__device__ __forceinline__ uint32_t prmt_i8(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Four int8 codes (bytes of w, code i in byte i) -> four fp16 values as two half2 words, exactly:
// the offset byte u = code + 128 becomes the fp16 value 1024 + u (bits 0x64uu: exponent 10, u in the
// low mantissa bits), and one packed subtract of 1152 leaves the code.
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = hsub2_bits(prmt_i8(u, 0x64646464u, 0x4140u), 0x64806480u);
  hi = hsub2_bits(prmt_i8(u, 0x64646464u, 0x4342u), 0x64806480u);
}

__device__ __forceinline__ void i8x16_to_f16(uint4 v, uint32_t (&q)[8]) {
  i8x4_to_f16(v.x, q[0], q[1]);
  i8x4_to_f16(v.y, q[2], q[3]);
  i8x4_to_f16(v.z, q[4], q[5]);
  i8x4_to_f16(v.w, q[6], q[7]);
}

__device__ __forceinline__ float silu_mul_i8(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

// Converts one slab: 256 rows x 4 pieces of 16 codes = 1024 tasks over the converter threads, each
// task one 16-byte load and two 16-byte stores at the row's 128-byte-swizzled chunk positions.
__device__ __forceinline__ void convert_slab_i8(const uint8_t* __restrict__ codes, uint8_t* __restrict__ btile,
                                                int ctid) {
  constexpr int kTasks = kI8Tile * 4;
  for (int t0 = ctid; t0 < kTasks; t0 += kI8ConvThreads * kI8ConvBatch) {
    uint4 v[kI8ConvBatch];
#pragma unroll
    for (int j = 0; j < kI8ConvBatch; ++j) {
      const int task = t0 + j * kI8ConvThreads;
      if (task < kTasks) v[j] = *reinterpret_cast<const uint4*>(codes + task * 16);   // row task/4, piece task%4
    }
#pragma unroll
    for (int j = 0; j < kI8ConvBatch; ++j) {
      const int task = t0 + j * kI8ConvThreads;
      if (task < kTasks) {
        const int n = task >> 2, p = task & 3;
        uint32_t q[8];
        i8x16_to_f16(v[j], q);
        uint8_t* row = btile + n * 128;
        *reinterpret_cast<uint4*>(row + (((2 * p) ^ (n & 7)) << 4)) = make_uint4(q[0], q[1], q[2], q[3]);
        *reinterpret_cast<uint4*>(row + (((2 * p + 1) ^ (n & 7)) << 4)) = make_uint4(q[4], q[5], q[6], q[7]);
      }
    }
  }
}

// Warp roles: 0 loads (TMA token rows + bulk copy of the int8 codes into the load ring), 1 issues the
// MMAs, 2..11 convert codes into the fp16 ring, 12..15 drain the accumulators.  A pass with two row
// blocks accumulates block j into TMEM columns [256j, 256j+256); the epilogue releases the
// accumulators after the pass.
template <int BN, bool L1, bool BLOCK>
__global__ void __launch_bounds__(kI8Threads, 1)
    moe_gemm_i8_kernel(const __grid_constant__ CUtensorMap tmap_x, const I8Args a) {
  using C = I8Cfg<BN, BLOCK>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* lring = smem;                                   // [kStages] token rows + int8 codes
  uint8_t* bring = smem + C::kStages * C::kStage;          // [kBStages] fp16 weight tiles
  float* ssum = reinterpret_cast<float*>(bring + C::kBStages * kI8BStage);   // running K-block sums
  uint8_t* extra = bring + C::kBStages * kI8BStage + C::kSumBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(extra);     // load slot filled (TMA)
  uint64_t* lempty = full + C::kStages;                    // load slot consumed (MMA commit)
  uint64_t* bready = lempty + C::kStages;                  // fp16 tile written (converters)
  uint64_t* bempty = bready + C::kBStages;                 // fp16 tile consumed (MMA commit)
  uint64_t* acc_full = bempty + C::kBStages;               // [2]: accumulator 0 / 1 written
  uint64_t* acc_empty = acc_full + 2;                      // [2]: accumulator 0 / 1 drained
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(lempty + s), 1);
    }
    for (int s = 0; s < C::kBStages; ++s) {
      mbar_init(smem_u32(bready + s), kI8ConvThreads);
      mbar_init(smem_u32(bempty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(acc_full + b), 1);
      mbar_init(smem_u32(acc_empty + b), 128);
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmap_x);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kI8TmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int msum = *a.m_sum;

  if (warp == 0) {
    // ---------------- producer: fp16 token rows by TMA, int8 codes by one bulk copy ----------------
    const uint64_t pol_x = policy_evict_last();
    int ls = 0;
    uint32_t lph = 0;
    int t = blockIdx.x, p = 0, ep = -1;
    RowPass P;
    while (!__any_sync(0xffffffffu, *abort_flag != 0) && next_row_pass<BN>(a, msum, t, p, ep, P)) {
      const int wt = t % a.n_wt;
      const size_t chunk0 = (static_cast<size_t>(P.e) * a.n_wt + wt) * a.n_slabs;
      bool ok = true;
      for (int s = 0; s < a.n_slabs; ++s) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(lempty + ls), lph ^ 1, a.status));
        if (!ok) break;
        if (lane == 0) {
          uint8_t* st = lring + ls * C::kStage;
          const uint32_t fb = smem_u32(full + ls);
          const size_t wbase = (chunk0 + s) * kI8Chunk;
          if (wbase + kI8Chunk > a.w_bytes || (reinterpret_cast<uintptr_t>(a.w) & 15)) {
            record_error(a.status, kDevErrCheck);
            *abort_flag = 1;
          } else {
            mbar_arrive_expect_tx(fb, P.nb * C::kABytes + kI8Chunk);
            for (int j = 0; j < P.nb; ++j)
              tma_load_2d(smem_u32(st + j * C::kABytes), &tmap_x, s * kI8Slab, (P.rb + j) * BN, fb, pol_x);
            bulk_load(smem_u32(st + C::kPOff), a.w + wbase, kI8Chunk, fb);
          }
        }
        __syncwarp();
        if (++ls == C::kStages) {
          ls = 0;
          lph ^= 1;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        break;
      }
    }
    if (__any_sync(0xffffffffu, *abort_flag != 0)) {
      // let every copy issued into shared memory land before the CTA exits
      for (int s = 0; s < C::kStages; ++s) mbar_wait(smem_u32(full + s), (s < ls) ? lph : (lph ^ 1), nullptr);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: kind::f16 (fp16 operands), M=128, N=256, K=16 x 4 per slab ----------------
    int ls = 0, bs = 0;
    uint32_t lph = 0, bph = 0;
    uint32_t aph = 0;   // bit b: phase of accumulator b
    int rnd = 0;   // accumulator rounds so far (alternating accumulators with kSumSmem)
    int t = blockIdx.x, p = 0, ep = -1;
    RowPass P;
    const uint32_t id = idesc_f16(128, kI8Tile);
    // BLOCK: one accumulator round per 256-deep K-block (4 slabs); otherwise one per pass
    const int slabs_per_round = BLOCK ? 4 : a.n_slabs;
    while (!__any_sync(0xffffffffu, *abort_flag != 0) && next_row_pass<BN>(a, msum, t, p, ep, P)) {
      bool ok = true;
      for (int s0 = 0; ok && s0 < a.n_slabs; s0 += slabs_per_round) {
        const int buf = C::kSumSmem ? (rnd & 1) : 0;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(acc_empty + buf), ((aph >> buf) & 1u) ^ 1u, a.status));
        if (!ok) break;
        tc_fence_after();
        for (int s = s0; s < s0 + slabs_per_round; ++s) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(full + ls), lph, a.status) &&
                                           mbar_wait(smem_u32(bready + bs), bph, a.status));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t sa = smem_u32(lring + ls * C::kStage);
            const uint32_t sb = smem_u32(bring + bs * kI8BStage);
            for (int j = 0; j < P.nb; ++j)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_bf16(tmem + static_cast<uint32_t>((buf + j) * kI8Tile), desc_sw128(sa + j * C::kABytes + k * 32),
                         desc_sw128(sb + k * 32), id, (s > s0 || k > 0) ? 1u : 0u);
            tc_commit(smem_u32(lempty + ls));
            tc_commit(smem_u32(bempty + bs));
          }
          __syncwarp();
          if (++ls == C::kStages) {
            ls = 0;
            lph ^= 1;
          }
          if (++bs == C::kBStages) {
            bs = 0;
            bph ^= 1;
          }
        }
        if (!ok) break;
        if (lane == 0) tc_commit(smem_u32(acc_full + buf));
        __syncwarp();
        aph ^= 1u << buf;
        ++rnd;
      }
      if (!ok) {
        *abort_flag = 1;
        break;
      }
    }
  } else if (warp < 2 + kI8ConvThreads / 32) {
    // ---------------- converters: int8 codes -> 128-byte-swizzled fp16 tile ----------------
    const int ctid = threadIdx.x - 64;
    int ls = 0, bs = 0;
    uint32_t lph = 0, bph = 0;
    int t = blockIdx.x, p = 0, ep = -1;
    RowPass P;
    while (!__any_sync(0xffffffffu, *abort_flag != 0) && next_row_pass<BN>(a, msum, t, p, ep, P)) {
      bool ok = true;
      for (int s = 0; s < a.n_slabs; ++s) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(full + ls), lph, a.status) &&
                                         mbar_wait(smem_u32(bempty + bs), bph ^ 1, a.status));
        if (!ok) break;
        convert_slab_i8(lring + ls * C::kStage + C::kPOff, bring + bs * kI8BStage, ctid);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(smem_u32(bready + bs));
        if (++ls == C::kStages) {
          ls = 0;
          lph ^= 1;
        }
        if (++bs == C::kBStages) {
          bs = 0;
          bph ^= 1;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        break;
      }
    }
  } else {
    // ---------------- epilogue (warps 12..15): thread = token row m of each block ----------------
    const int q = warp & 3;
    const int m = q * 32 + lane;
    const bool warp_has_rows = q * 32 < BN;   // warp-uniform
    uint32_t acc_phase = 0;
    uint32_t aph = 0;   // bit b: phase of accumulator b
    int rnd = 0;
    int t = blockIdx.x, p = 0, ep = -1;
    RowPass P;
    while (next_row_pass<BN>(a, msum, t, p, ep, P)) {
      const int wt = t % a.n_wt;
      if (C::kSumSmem) {
        // K-blocks alternate between the two accumulators; thread m folds its row into its row of the
        // shared-memory sum (same fma order as the tensor-memory sum), the last K-block's fold feeding
        // the SwiGLU or the bf16 output.  Each accumulator is released once read.
        const uint32_t lq = static_cast<uint32_t>(q * 32) << 16;
        const int row = P.rb * BN + m;
        const bool act = m < BN;
        const bool mine = act && row < msum && __ldg(a.expert_ids + row) == P.e;
        const int nbw = (a.w_rows + 255) / 256;
        const float* wsa = a.col_scale + (static_cast<size_t>(P.e) * nbw + (L1 ? (wt * 128) / 256 : wt)) * a.nkb;
        const float* wsb = a.col_scale + (static_cast<size_t>(P.e) * nbw + (L1 ? (a.out_cols + wt * 128) / 256 : wt)) * a.nkb;
        const float* rsp = a.row_scale + static_cast<size_t>(mine ? row : 0) * a.nkb;
        float* srow = ssum + (act ? m : 0) * C::kSumStride;
        const int ncols = L1 ? 128 : min(kI8Tile, a.out_cols - wt * kI8Tile);
        bool okb = true;
        for (int kb = 0; kb < a.nkb; ++kb) {
          const int buf = rnd & 1;
          okb = mbar_wait(smem_u32(acc_full + buf), (aph >> buf) & 1u, a.status) && *abort_flag == 0;
          okb = named_barrier_and(1, 128, okb);
          if (!okb) break;
          tc_fence_after();
          const uint32_t acc = tmem + lq + static_cast<uint32_t>(buf * kI8Tile);
          const bool last = kb == a.nkb - 1;
          const float rs = mine ? __ldg(rsp + kb) : 0.f;
          const float fa = rs * __ldg(wsa + kb), fb = rs * __ldg(wsb + kb);
          if (warp_has_rows) {
            // four tensor-memory loads in flight per wait (one warp holds all the rows of a small block)
            if (L1) {
              uint4* dst = reinterpret_cast<uint4*>(a.out + static_cast<size_t>(row) * a.out_cols + wt * 128);
#pragma unroll 1
              for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t g[2][16], u[2][16];
                tc_ld_x16(acc + c0, g[0]);
                tc_ld_x16(acc + c0 + 16, g[1]);
                tc_ld_x16(acc + 128 + c0, u[0]);
                tc_ld_x16(acc + 128 + c0 + 16, u[1]);
                tc_wait_ld();
                if (act) {
#pragma unroll
                  for (int i = 0; i < 32; ++i) {
                    const float sg = fmaf(__uint_as_float(g[i >> 4][i & 15]), fa, kb > 0 ? srow[c0 + i] : 0.f);
                    const float su = fmaf(__uint_as_float(u[i >> 4][i & 15]), fb, kb > 0 ? srow[128 + c0 + i] : 0.f);
                    if (!last) {
                      srow[c0 + i] = sg;
                      srow[128 + c0 + i] = su;
                    } else {
                      g[i >> 4][i & 15] = __float_as_uint(silu_mul_i8(sg, su));
                    }
                  }
                  if (last && mine) {
                    uint32_t packed[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                      packed[i] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(g[i >> 3][(2 * i) & 15]))) |
                                  (static_cast<uint32_t>(__bfloat16_as_ushort(
                                       __float2bfloat16_rn(__uint_as_float(g[i >> 3][(2 * i + 1) & 15])))) << 16);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                      dst[c0 / 8 + c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
                  }
                }
              }
            } else {
              uint4* dst = reinterpret_cast<uint4*>(a.out + static_cast<size_t>(row) * a.out_cols + wt * kI8Tile);
#pragma unroll 1
              for (int c0 = 0; c0 < kI8Tile; c0 += 64) {
                uint32_t v[4][16];
#pragma unroll
                for (int k = 0; k < 4; ++k) tc_ld_x16(acc + c0 + 16 * k, v[k]);
                tc_wait_ld();
                if (act) {
#pragma unroll
                  for (int i = 0; i < 64; ++i) {
                    const float sv = fmaf(__uint_as_float(v[i >> 4][i & 15]), fa, kb > 0 ? srow[c0 + i] : 0.f);
                    if (!last) srow[c0 + i] = sv;
                    else v[i >> 4][i & 15] = __float_as_uint(sv);
                  }
                  if (last && mine && c0 < ncols) {
                    uint32_t packed[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                      packed[i] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[i >> 3][(2 * i) & 15]))) |
                                  (static_cast<uint32_t>(__bfloat16_as_ushort(
                                       __float2bfloat16_rn(__uint_as_float(v[i >> 3][(2 * i + 1) & 15])))) << 16);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                      dst[c0 / 8 + c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
                  }
                }
              }
            }
          }
          tc_fence_before();
          mbar_arrive(smem_u32(acc_empty + buf));
          aph ^= 1u << buf;
          ++rnd;
          if (!L1 && last && a.red.out)
            fused_reduce_tail(a.red, a.out, a.out_cols, mine, row, wt, a.n_wt, wt * kI8Tile, ncols);
        }
        if (!okb) {
          *abort_flag = 1;
          break;
        }
        continue;
      }
      if (BLOCK) {
        // one pass = one row block; fold each K-block into the running sum, finish on the last
        const uint32_t acc = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const uint32_t sum = acc + static_cast<uint32_t>(kI8Tile);
        const int row = P.rb * BN + m;
        const bool mine = m < BN && row < msum && __ldg(a.expert_ids + row) == P.e;
        const int nbw = (a.w_rows + 255) / 256;     // weight row blocks
        // weight blocks of the tile's columns: L1 gate rows 128 wt.. and up rows I + 128 wt..; L2 rows 256 wt..
        const float* wsa = a.col_scale + (static_cast<size_t>(P.e) * nbw + (L1 ? (wt * 128) / 256 : wt)) * a.nkb;
        const float* wsb = a.col_scale + (static_cast<size_t>(P.e) * nbw + (L1 ? (a.out_cols + wt * 128) / 256 : wt)) * a.nkb;
        const float* rsp = a.row_scale + static_cast<size_t>(mine ? row : 0) * a.nkb;
        bool okb = true;
        for (int kb = 0; kb < a.nkb; ++kb) {
          okb = mbar_wait(smem_u32(acc_full), acc_phase, a.status) && *abort_flag == 0;
          okb = named_barrier_and(1, 128, okb);
          if (!okb) break;
          tc_fence_after();
          const bool last = kb == a.nkb - 1;
          const float rs = mine ? __ldg(rsp + kb) : 0.f;
          const float fa = rs * __ldg(wsa + kb), fb = rs * __ldg(wsb + kb);
          if (L1) {
            // column c: gate channel wt*128 + c (scale fa) with its up channel in column 128 + c (fb)
            uint4* dst = reinterpret_cast<uint4*>(a.out + static_cast<size_t>(row) * a.out_cols + wt * 128);
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 16) {
              uint32_t g[16], u[16], sg[16], su[16];
              tc_ld_x16(acc + c0, g);
              tc_ld_x16(acc + 128 + c0, u);
              if (kb > 0) {
                tc_ld_x16(sum + c0, sg);
                tc_ld_x16(sum + 128 + c0, su);
              }
              tc_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float pg = kb > 0 ? __uint_as_float(sg[i]) : 0.f;
                const float pu = kb > 0 ? __uint_as_float(su[i]) : 0.f;
                sg[i] = __float_as_uint(fmaf(__uint_as_float(g[i]), fa, pg));
                su[i] = __float_as_uint(fmaf(__uint_as_float(u[i]), fb, pu));
              }
              if (!last) {
                tc_st_x16(sum + c0, sg);
                tc_st_x16(sum + 128 + c0, su);
              } else if (mine) {
                uint32_t packed[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float h0 = silu_mul_i8(__uint_as_float(sg[2 * i]), __uint_as_float(su[2 * i]));
                  const float h1 = silu_mul_i8(__uint_as_float(sg[2 * i + 1]), __uint_as_float(su[2 * i + 1]));
                  packed[i] = __bfloat16_as_ushort(__float2bfloat16_rn(h0)) |
                              (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(h1))) << 16);
                }
                dst[c0 / 8] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                dst[c0 / 8 + 1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
              }
            }
          } else {
            const int ncols = min(kI8Tile, a.out_cols - wt * kI8Tile);
            uint4* dst = reinterpret_cast<uint4*>(a.out + static_cast<size_t>(row) * a.out_cols + wt * kI8Tile);
#pragma unroll 1
            for (int c0 = 0; c0 < kI8Tile; c0 += 16) {
              uint32_t v[16], sv[16];
              tc_ld_x16(acc + c0, v);
              if (kb > 0) tc_ld_x16(sum + c0, sv);
              tc_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i)
                sv[i] = __float_as_uint(fmaf(__uint_as_float(v[i]), fa, kb > 0 ? __uint_as_float(sv[i]) : 0.f));
              if (!last) {
                tc_st_x16(sum + c0, sv);
              } else if (mine && c0 < ncols) {
                uint32_t packed[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  packed[i] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(sv[2 * i]))) |
                              (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(sv[2 * i + 1])))) << 16);
                dst[c0 / 8] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                dst[c0 / 8 + 1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
              }
            }
            if (last && a.red.out)
              fused_reduce_tail(a.red, a.out, a.out_cols, mine, row, wt, a.n_wt, wt * kI8Tile, ncols);
          }
          if (!last) tc_wait_st();
          tc_fence_before();
          mbar_arrive(smem_u32(acc_empty));
          acc_phase ^= 1;
        }
        if (!okb) {
          *abort_flag = 1;
          break;
        }
        continue;
      }
      bool ok = mbar_wait(smem_u32(acc_full), acc_phase, a.status) && *abort_flag == 0;
      ok = named_barrier_and(1, 128, ok);
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const float* cs = a.col_scale + static_cast<size_t>(P.e) * a.w_rows;
      for (int j = 0; j < P.nb; ++j) {
        const uint32_t acc = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(j * kI8Tile);
        const int row = (P.rb + j) * BN + m;
        const bool mine = m < BN && row < msum && __ldg(a.expert_ids + row) == P.e;
        const float rs = mine ? __ldg(a.row_scale + row) : 0.f;
        if (L1) {
          // columns c of the tile: gate channel wt*128 + c, up channel I + wt*128 + c
          const float* cg = cs + wt * 128;
          const float* cu = cs + a.out_cols + wt * 128;
          if (warp_has_rows) {
            uint4* dst = reinterpret_cast<uint4*>(a.out + static_cast<size_t>(row) * a.out_cols + wt * 128);
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 32) {
              uint32_t g[2][16], u[2][16];
              tc_ld_x16(acc + c0, g[0]);
              tc_ld_x16(acc + c0 + 16, g[1]);
              tc_ld_x16(acc + 128 + c0, u[0]);
              tc_ld_x16(acc + 128 + c0 + 16, u[1]);
              tc_wait_ld();
              uint32_t packed[16];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 sg = __ldg(reinterpret_cast<const float4*>(cg + c0) + i);
                const float4 su = __ldg(reinterpret_cast<const float4*>(cu + c0) + i);
                const float sgv[4] = {sg.x, sg.y, sg.z, sg.w}, suv[4] = {su.x, su.y, su.z, su.w};
                float h[4];
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                  const int c = 4 * i + v;
                  h[v] = silu_mul_i8(__uint_as_float(g[c >> 4][c & 15]) * rs * sgv[v],
                                     __uint_as_float(u[c >> 4][c & 15]) * rs * suv[v]);
                }
                packed[2 * i] = __bfloat16_as_ushort(__float2bfloat16_rn(h[0])) |
                                (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(h[1]))) << 16);
                packed[2 * i + 1] = __bfloat16_as_ushort(__float2bfloat16_rn(h[2])) |
                                    (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(h[3]))) << 16);
              }
              if (mine) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                  dst[c0 / 8 + c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
              }
            }
          }
        } else {
          const int ncols = min(kI8Tile, a.out_cols - wt * kI8Tile);
          const float* cy = cs + wt * kI8Tile;
          if (warp_has_rows) {
            uint4* dst = reinterpret_cast<uint4*>(a.out + static_cast<size_t>(row) * a.out_cols + wt * kI8Tile);
#pragma unroll 1
            for (int c0 = 0; c0 < kI8Tile; c0 += 32) {
              uint32_t v[2][16];
              tc_ld_x16(acc + c0, v[0]);
              tc_ld_x16(acc + c0 + 16, v[1]);
              tc_wait_ld();
              if (c0 < ncols) {   // ncols is a multiple of 128: whole 32-column groups
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float4 sc = __ldg(reinterpret_cast<const float4*>(cy + c0) + i);
                  const int c = 4 * i;
                  const float y0 = __uint_as_float(v[c >> 4][c & 15]) * rs * sc.x;
                  const float y1 = __uint_as_float(v[(c + 1) >> 4][(c + 1) & 15]) * rs * sc.y;
                  const float y2 = __uint_as_float(v[(c + 2) >> 4][(c + 2) & 15]) * rs * sc.z;
                  const float y3 = __uint_as_float(v[(c + 3) >> 4][(c + 3) & 15]) * rs * sc.w;
                  packed[2 * i] = __bfloat16_as_ushort(__float2bfloat16_rn(y0)) |
                                  (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(y1))) << 16);
                  packed[2 * i + 1] = __bfloat16_as_ushort(__float2bfloat16_rn(y2)) |
                                      (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(y3))) << 16);
                }
                if (mine) {
#pragma unroll
                  for (int c = 0; c < 4; ++c)
                    dst[c0 / 8 + c] =
                        make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
                }
              }
            }
          }
          if (a.red.out) fused_reduce_tail(a.red, a.out, a.out_cols, mine, row, wt, a.n_wt, wt * kI8Tile, ncols);
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(acc_empty));
      acc_phase ^= 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kI8TmemCols);
  }
}

// Int8 activation rows -> fp16 rows of the codes (exact) plus each row's scale, for the rows r < m_sum
// that hold a (token, expert) pair.  With src_map (L1) row r reads source row src_map[r] / K (the
// token of the row's pair: sorted_token_ids holds t*K + k); otherwise source row r.  One warp per
// row, 16 codes per lane step.
__global__ void __launch_bounds__(256) i8_rows_to_f16_kernel(const int8_t* __restrict__ src,
                                                             const float* __restrict__ src_scale, int src_rows,
                                                             const int32_t* __restrict__ src_map, int K,
                                                             const int32_t* __restrict__ expert_ids,
                                                             const int32_t* __restrict__ m_sum, int U, int C,
                                                             uint16_t* __restrict__ dst, float* __restrict__ dst_scale,
                                                             uint32_t* status, int nsc) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int msum = *m_sum;
  for (int r = blockIdx.x * 8 + warp; r < msum && r < U; r += gridDim.x * 8) {
    if (__ldg(expert_ids + r) < 0) continue;
    const int s = src_map ? __ldg(src_map + r) / K : r;
    if (s < 0 || s >= src_rows) {
      if (lane == 0) record_error(status, kDevErrCheck);
      continue;
    }
    for (int j = lane; j < nsc; j += 32) dst_scale[static_cast<size_t>(r) * nsc + j] = __ldg(src_scale + static_cast<size_t>(s) * nsc + j);
    const int8_t* in = src + static_cast<size_t>(s) * C;
    uint16_t* out = dst + static_cast<size_t>(r) * C;
    for (int k0 = lane * 16; k0 < C; k0 += 512) {
      uint32_t q[8];
      i8x16_to_f16(*reinterpret_cast<const uint4*>(in + k0), q);
      *reinterpret_cast<uint4*>(out + k0) = make_uint4(q[0], q[1], q[2], q[3]);
      *reinterpret_cast<uint4*>(out + k0 + 8) = make_uint4(q[4], q[5], q[6], q[7]);
    }
  }
}

// Symmetric int8 quantisation of bf16 rows, per group of G columns (G = C: per row): amax = max |x|
// over the group; inv = 127 / amax and s = amax / 127, each one correctly rounded fp32 division;
// q = clamp(rint(x * inv), -127, 127) with one fp32 multiply per value (rint: to nearest, ties to
// even).  A group with amax = 0 gives q = 0, s = 0; s is [rows, C/G].  Rows: all of [0, R), or with
// expert_ids the rows r < min(R, m_sum) that hold a pair.  With f16 non-null the codes are also
// written as fp16 values (the next GEMM's operand).  One warp per row, 8 values per lane step.
__global__ void __launch_bounds__(256) quant_rows_i8_kernel(const uint16_t* __restrict__ x, int R, int C,
                                                            const int32_t* __restrict__ expert_ids,
                                                            const int32_t* __restrict__ m_sum,
                                                            int8_t* __restrict__ q, float* __restrict__ s,
                                                            uint16_t* __restrict__ f16, int G) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int rows = m_sum ? min(R, *m_sum) : R;
  const int ng = C / G;
  for (int rg = blockIdx.x * 8 + warp; rg < rows * ng; rg += gridDim.x * 8) {
    const int r = rg / ng, g = rg - r * ng;
    if (expert_ids && __ldg(expert_ids + r) < 0) continue;
    const uint16_t* in = x + static_cast<size_t>(r) * C + static_cast<size_t>(g) * G;
    float amax = 0.f;
    for (int k0 = lane * 8; k0 < G; k0 += 256) {
      const uint4 v = *reinterpret_cast<const uint4*>(in + k0);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
    }
    amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));   // amax >= 0: bits order
    const float inv = amax > 0.f ? __fdiv_rn(127.f, amax) : 0.f;
    if (lane == 0) s[static_cast<size_t>(r) * ng + g] = __fdiv_rn(amax, 127.f);
    int8_t* qo = q + static_cast<size_t>(r) * C + static_cast<size_t>(g) * G;
    for (int k0 = lane * 8; k0 < G; k0 += 256) {
      const uint4 v = *reinterpret_cast<const uint4*>(in + k0);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      int c[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        c[2 * j] = max(-127, min(127, __float2int_rn(__fmul_rn(__uint_as_float(w[j] << 16), inv))));
        c[2 * j + 1] = max(-127, min(127, __float2int_rn(__fmul_rn(__uint_as_float(w[j] & 0xFFFF0000u), inv))));
      }
      uint32_t b[2];
#pragma unroll
      for (int h = 0; h < 2; ++h)
        b[h] = (static_cast<uint32_t>(c[4 * h]) & 0xFF) | ((static_cast<uint32_t>(c[4 * h + 1]) & 0xFF) << 8) |
               ((static_cast<uint32_t>(c[4 * h + 2]) & 0xFF) << 16) | (static_cast<uint32_t>(c[4 * h + 3]) << 24);
      *reinterpret_cast<uint2*>(qo + k0) = make_uint2(b[0], b[1]);
      if (f16) {
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          o[j] = __half_as_ushort(__int2half_rn(c[2 * j])) |
                 (static_cast<uint32_t>(__half_as_ushort(__int2half_rn(c[2 * j + 1]))) << 16);
        *reinterpret_cast<uint4*>(f16 + static_cast<size_t>(r) * C + static_cast<size_t>(g) * G + k0) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
}

// INT8 packing: per (expert, 256-row tile, 64-deep slab) the tile's 256 rows x 64 codes, row n at
// byte 64n; tiles formed as in pack_mx_weights_kernel (pair = 2: rows 128t.. of the gate half then of
// the up half; pair = 1: rows 256t..; rows past N read as zero).  16 bytes per thread step.
__global__ void pack_i8_weights_kernel(const int8_t* __restrict__ q, int E, int N, int Kd, int pair,
                                       uint8_t* __restrict__ out) {
  const int n_slabs = Kd / kI8Slab, n_wt = pair == 2 ? N / kI8Tile : (N + kI8Tile - 1) / kI8Tile;
  const size_t total = static_cast<size_t>(E) * n_wt * n_slabs * (kI8Chunk / 16);
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const size_t c = i / (kI8Chunk / 16);
    const int o = static_cast<int>(i % (kI8Chunk / 16)) * 16;
    const int s = static_cast<int>(c % n_slabs);
    const size_t ew = c / n_slabs;
    const int wt = static_cast<int>(ew % n_wt), e = static_cast<int>(ew / n_wt);
    const int n = o / kI8Slab;
    const int h = n / 128, mm = n % 128;
    const int r = pair == 2 ? h * (N / 2) + wt * 128 + mm : wt * kI8Tile + n;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < N) v = *reinterpret_cast<const uint4*>(q + (static_cast<size_t>(e) * N + r) * Kd + s * kI8Slab + o % kI8Slab);
    *reinterpret_cast<uint4*>(out + i * 16) = v;
  }
}

template <int BN, bool L1, bool BLOCK>
cudaError_t launch_i8_t(const I8Launch& L, cudaStream_t stream) {
  CUtensorMap mx;
  if (!make_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, L.xf, static_cast<uint64_t>(L.Kd),
                   static_cast<uint64_t>(L.U), static_cast<uint64_t>(L.Kd) * 2, kI8Slab, BN))
    return cudaErrorInvalidValue;
  I8Args a;
  a.w = L.w;
  a.col_scale = L.col_scale;
  a.row_scale = L.row_scale;
  a.expert_ids = L.expert_ids;
  a.m_sum = L.m_sum;
  a.out = L.out;
  a.status = L.status;
  a.red = L.red;
  const int pair = L1 ? 2 : 1;
  a.n_wt = pair == 2 ? L.w_rows / kI8Tile : (L.w_rows + kI8Tile - 1) / kI8Tile;
  a.n_slabs = L.Kd / kI8Slab;
  a.w_bytes = static_cast<size_t>(L.E) * a.n_wt * a.n_slabs * kI8Chunk;
  a.w_rows = L.w_rows;
  a.out_cols = L1 ? L.I : L.w_rows;
  a.one_expert_blocks = L.align % BN == 0;
  const int nrb = (L.U + BN - 1) / BN;
  // items: halves of row-block pairs (blocks of up to 32 rows), whole pairs, or blocks
  a.split_pairs = BN <= 32;
  a.pair_blocks = BLOCK ? 0 : 1;
  a.nkb = L.Kd / 256;
  if (BLOCK && (L.Kd % 256 != 0 || L.w_rows % 256 != 0)) return cudaErrorInvalidValue;
  a.n_tiles = (a.one_expert_blocks ? (a.split_pairs ? (nrb + 1) / 2 * 2 : (nrb + 1) / 2) : nrb) * a.n_wt;
  int grid = num_sms();
  if (grid > a.n_tiles) grid = a.n_tiles;
  if (grid < 1) grid = 1;
  constexpr int kSmem = I8Cfg<BN, BLOCK>::kSmem;
  cudaError_t err = cudaFuncSetAttribute(moe_gemm_i8_kernel<BN, L1, BLOCK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmem);
  if (err != cudaSuccess) return err;
  moe_gemm_i8_kernel<BN, L1, BLOCK><<<grid, kI8Threads, kSmem, stream>>>(mx, a);
  return cudaGetLastError();
}

int rows_grid(int rows) {
  const int b = (rows + 7) / 8;
  return b < 1 ? 1 : (b < 4 * num_sms() ? b : 4 * num_sms());
}

}  // namespace

size_t packed_i8_weight_bytes(int E, int N, int Kd, int pair) {
  const int n_wt = pair == 2 ? N / kI8Tile : (N + kI8Tile - 1) / kI8Tile;
  return static_cast<size_t>(E) * n_wt * (Kd / kI8Slab) * kI8Chunk;
}

cudaError_t launch_pack_i8(const int8_t* q, int E, int N, int Kd, int pair, uint8_t* out, cudaStream_t stream) {
  pack_i8_weights_kernel<<<4 * num_sms(), 256, 0, stream>>>(q, E, N, Kd, pair, out);
  return cudaGetLastError();
}

cudaError_t launch_i8_rows_to_f16(const int8_t* src, const float* src_scale, int src_rows, const int32_t* src_map,
                                  int K, const int32_t* expert_ids, const int32_t* m_sum, int U, int C, uint16_t* dst,
                                  float* dst_scale, uint32_t* status, cudaStream_t stream, int nsc) {
  i8_rows_to_f16_kernel<<<rows_grid(U), 256, 0, stream>>>(src, src_scale, src_rows, src_map, K, expert_ids, m_sum, U,
                                                           C, dst, dst_scale, status, nsc);
  return cudaGetLastError();
}

cudaError_t launch_quant_rows_i8(const uint16_t* x, int R, int C, const int32_t* expert_ids, const int32_t* m_sum,
                                 int8_t* q, float* s, uint16_t* f16, cudaStream_t stream, int group) {
  const int G = group > 0 ? group : C;
  const long long units = static_cast<long long>(R) * (C / G);
  const int grid = static_cast<int>(units / 8 + 1 < 4LL * num_sms() ? units / 8 + 1 : 4LL * num_sms());
  quant_rows_i8_kernel<<<grid, 256, 0, stream>>>(x, R, C, expert_ids, m_sum, q, s, f16, G);
  return cudaGetLastError();
}

template <bool BLOCK>
static cudaError_t launch_gemm_i8_b(const I8Launch& L, bool l1, cudaStream_t stream) {
  const int bn = act_sf_block_rows(L.align);
  if (l1) {
    switch (bn) {
      case 16: return launch_i8_t<16, true, BLOCK>(L, stream);
      case 32: return launch_i8_t<32, true, BLOCK>(L, stream);
      case 64: return launch_i8_t<64, true, BLOCK>(L, stream);
      default: return launch_i8_t<128, true, BLOCK>(L, stream);
    }
  }
  switch (bn) {
    case 16: return launch_i8_t<16, false, BLOCK>(L, stream);
    case 32: return launch_i8_t<32, false, BLOCK>(L, stream);
    case 64: return launch_i8_t<64, false, BLOCK>(L, stream);
    default: return launch_i8_t<128, false, BLOCK>(L, stream);
  }
}

cudaError_t launch_gemm_i8(const I8Launch& L, bool l1, cudaStream_t stream) {
  return L.block ? launch_gemm_i8_b<true>(L, l1, stream) : launch_gemm_i8_b<false>(L, l1, stream);
}

}  // namespace moe
