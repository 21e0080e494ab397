// Block-scaled grouped GEMMs of the MoE layer on tcgen05 (sm_103a):
//   L1: gu = X @ W13[e]^T, h = silu(gu[:I]) * gu[I:], FP8 requant per 128 along I
//   L2: y  = h @ W2[e]^T, bf16
// Page "DeepSeek V4 MegaMoE Kernel 深度解析", 二、阶段 2-4 (FP8 E4M3 activations x FP4 E2M1
// weights with UE8M0 scales, TMA -> shared memory -> scales copied into TMEM -> UMMA ->
// TMEM accumulators, full/empty barrier pipeline, SwiGLU + amax -> UE8M0 -> E4M3 epilogue).
//
// Design (this file's own, for one GPU):
//  * Weights are the MMA's M side (128 rows per tile) and tokens the N side (BN rows), so a
//    3-row expert at decode costs an N=16 MMA, not a 128-row one.  L1 tiles hold the gate rows
//    i0..i0+127 and the up rows I+i0..I+i0+127 in two accumulators, so one CTA sees both halves
//    of SwiGLU and the full 128-wide requant group.
//  * A work item is (row block of BN permuted rows, weight tile, expert).  BN divides the
//    permute alignment in the common case, so a block holds one expert; otherwise each expert
//    present in the block is a separate pass whose stores are masked by expert_ids.
//  * Persistent CTAs (one per SM) walk the items in a fixed order; producer warp (TMA),
//    MMA warp (one thread issues tcgen05.cp + tcgen05.mma) and four epilogue warps run
//    decoupled through mbarriers; accumulators are double-buffered in TMEM when they fit.
//  * FP4 weights are loaded with the padded 4-bit TMA type (each 16 codes -> 16 bytes of shared
//    memory), 128-byte swizzle, which is the operand layout kind::mxf8f6f4 reads.
//  * Scale factors: weight scales arrive pre-arranged (moe_pack_weight_scales) as one 512-byte
//    32x(4x4 bytes) image per (128-row tile, 128-deep slab); token scales as the tiled layout.
//    Both are copied into TMEM with tcgen05.cp .32x128b.warpx4.  Row m of the weight tile reads
//    its scale from column (m/32), byte (k-step); token n from column (n/32), byte (slab % 4).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kGemmThreads = 192;        // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kSmemBudget = 227 * 1024;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: accumulators in [0, 384); scale factors in [384, 512), every region starting
// on a 16-column boundary (weight scales of the gate / up tiles and token scales, 2 slots each).
constexpr uint32_t kAccCols = 384;
constexpr uint32_t kSfaGate = 384;
constexpr uint32_t kSfaUp = 416;
constexpr uint32_t kSfbCol = 448;

template <int BN, bool L1>
struct GemmCfg {
  static constexpr int NW = L1 ? 2 : 1;                          // weight tiles per stage
  static constexpr int W_BYTES = 16384;                          // 128 x 128 codes, padded
  static constexpr int X_BYTES = BN * 128;
  static constexpr int SFA_OFF = NW * W_BYTES + X_BYTES;
  static constexpr int SFB_OFF = SFA_OFF + NW * 512;
  static constexpr int STAGE_RAW = SFB_OFF + 512;
  static constexpr int STAGE = (STAGE_RAW + 1023) / 1024 * 1024;
  static constexpr int EXTRA = 4096;                             // barriers, reductions, flags
  static constexpr int S_FIT = (kSmemBudget - EXTRA - 1024) / STAGE;
  static constexpr int STAGES = S_FIT > 8 ? 8 : S_FIT;
  static constexpr int UP_OFF = (BN + 31) / 32 * 32;            // column offset of the up accumulator
  static constexpr int ACC_COLS = NW * UP_OFF;                   // columns per accumulator buffer
  static constexpr int NBUF = (2 * ACC_COLS <= (int)kAccCols) ? 2 : 1;
  static constexpr int SFB_BYTES = 512;                          // one token-scale chunk
  static constexpr int SMEM = 1024 + STAGES * STAGE + EXTRA;
  static constexpr uint32_t TX_W = 8192;                         // global bytes of one FP4 tile
  static_assert(STAGES >= 2, "shared memory too small for two stages");
  static_assert(ACC_COLS * NBUF <= (int)kAccCols, "accumulators overlap the scale columns");
};

struct GemmArgs {
  const uint8_t* w_sf;          // packed weight scale images
  const uint8_t* x_sf;          // tiled token scales (rows U)
  const int32_t* expert_ids;    // [U]
  const int32_t* m_sum;         // [1]
  uint8_t* h_q;                 // L1 out [U, I]
  uint8_t* h_sf;                // L1 out, tiled (rows U, slabs I/128)
  uint16_t* y;                  // L2 out [U, H] bf16
  uint32_t* status;
  size_t w_sf_bytes;            // sizes, for the kernel's own bounds checks
  size_t x_sf_bytes;
  int n_slabs;                  // reduction depth / 128
  int w_rows;                   // rows per expert in the weight tensor (2I or H)
  int n_wt;                     // weight tiles per item row (I/128 or H/128)
  int up_off;                   // L1: I (row offset of the up half)
  int out_cols;                 // L1: I, L2: H
  int sf_nb;                    // blocks of the tiled token-scale layouts (rows U, block rows BN)
  int n_tiles;                  // ceil(U/BN) * n_wt
};

// Next work item after (t, e): smallest expert id > e present in the row block of tile t,
// else the first expert of the next tile of this CTA.  Rows are sorted by expert (ignoring -1).
template <int BN>
__device__ __forceinline__ bool next_item(const GemmArgs& a, int msum, int& t, int& e) {
  while (t < a.n_tiles) {
    const int r0 = (t / a.n_wt) * BN;
    if (r0 >= msum) return false;
    const int rend = min(r0 + BN, msum);
    for (int r = r0; r < rend; ++r) {
      const int x = __ldg(a.expert_ids + r);
      if (x > e) {
        e = x;
        return true;
      }
    }
    t += gridDim.x;
    e = -1;
  }
  return false;
}

template <int BN, bool L1>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                    const GemmArgs a) {
  using C = GemmCfg<BN, L1>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* extra = smem + C::STAGES * C::STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(extra);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(extra + 256);              // [4][BN] warp partial maxima
  uint8_t* row_ok = extra + 256 + 4 * BN * 4;                      // [BN]

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
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
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int msum = *a.m_sum;

  if (warp == 0) {
    // ---------------- TMA producer (whole warp iterates, lane 0 issues) ----------------
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    int t = blockIdx.x, e = -1;
    while (!__any_sync(0xffffffffu, *abort_flag != 0) && next_item<BN>(a, msum, t, e)) {
      const int r0 = (t / a.n_wt) * BN, wt = t % a.n_wt;
      const int wrow = e * a.w_rows + wt * 128;
      const size_t sfa_chunk = static_cast<size_t>(wrow / 128) * a.n_slabs;
      bool ok = true;
      for (int s = 0; s < a.n_slabs; ++s) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(empty + stage), phase ^ 1, a.status));
        if (!ok) break;
        if (lane == 0) {
          uint8_t* st = stages + stage * C::STAGE;
          const uint32_t fb = smem_u32(full + stage);
          const int urow = wrow + a.up_off;
          const size_t sfa_g = (sfa_chunk + s) * 512;
          const size_t sfa_u = (static_cast<size_t>(urow / 128) * a.n_slabs + s) * 512;
          const size_t sfb = (static_cast<size_t>(s >> 2) * a.sf_nb + r0 / BN) * act_sf_chunk_bytes(BN);
          // self-check: every bulk copy inside its buffer and 16-byte aligned
          const bool good = sfa_g + 512 <= a.w_sf_bytes && (!L1 || sfa_u + 512 <= a.w_sf_bytes) &&
                            ((s & 3) != 0 || sfb + C::SFB_BYTES <= a.x_sf_bytes) &&
                            ((reinterpret_cast<uintptr_t>(a.w_sf) | reinterpret_cast<uintptr_t>(a.x_sf)) & 15) == 0;
          if (!good) {
            record_error(a.status, kDevErrCheck);
            *abort_flag = 1;
          } else {
            uint32_t bytes = C::NW * (C::TX_W + 512) + C::X_BYTES;
            if ((s & 3) == 0) bytes += C::SFB_BYTES;
            mbar_arrive_expect_tx(fb, bytes);
            tma_load_2d(smem_u32(st), &tmap_w, s * 128, wrow, fb, pol_w);
            bulk_load(smem_u32(st + C::SFA_OFF), a.w_sf + sfa_g, 512, fb);
            if (L1) {
              tma_load_2d(smem_u32(st + C::W_BYTES), &tmap_w, s * 128, urow, fb, pol_w);
              bulk_load(smem_u32(st + C::SFA_OFF + 512), a.w_sf + sfa_u, 512, fb);
            }
            tma_load_2d(smem_u32(st + C::NW * C::W_BYTES), &tmap_x, s * 128, r0, fb, pol_x);
            if ((s & 3) == 0) bulk_load(smem_u32(st + C::SFB_OFF), a.x_sf + sfb, C::SFB_BYTES, fb);
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
      // let every copy issued into shared memory land before the CTA exits
      for (int s = 0; s < C::STAGES; ++s) mbar_wait(smem_u32(full + s), (s < stage) ? phase : (phase ^ 1), nullptr);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (whole warp iterates, lane 0 issues) ----------------
    int stage = 0;
    uint32_t phase = 0;
    int buf = 0;
    uint32_t acc_phase = 0;
    int t = blockIdx.x, e = -1;
    while (!__any_sync(0xffffffffu, *abort_flag != 0) && next_item<BN>(a, msum, t, e)) {
      bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(acc_empty + buf), acc_phase ^ 1, a.status));
      if (ok) {
        tc_fence_after();
        const uint32_t acc = tmem + buf * C::ACC_COLS;
        for (int s = 0; s < a.n_slabs; ++s) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(full + stage), phase, a.status));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t st = smem_u32(stages + stage * C::STAGE);
            const uint32_t sfa = tmem + kSfaGate + (s & 1) * 16;
            const uint32_t sfu = tmem + kSfaUp + (s & 1) * 16;
            const uint32_t sfb = tmem + kSfbCol + ((s >> 2) & 1) * 16;
            tc_cp_32x128b_x4(sfa, smem_desc(st + C::SFA_OFF, 0, 128, 0));
            if (L1) tc_cp_32x128b_x4(sfu, smem_desc(st + C::SFA_OFF + 512, 0, 128, 0));
            if ((s & 3) == 0) tc_cp_32x128b_x4(sfb, smem_desc(st + C::SFB_OFF, 0, 128, 0));
            const uint32_t xs = st + C::NW * C::W_BYTES;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t id = idesc_mxf8f6f4(5, 0, 128, BN, k, s & 3);
              const uint32_t accum = (s > 0 || k > 0) ? 1u : 0u;
              mma_mxf8f6f4(acc, desc_sw128(st + k * 32), desc_sw128(xs + k * 32), id, sfa, sfb, accum);
              if (L1)
                mma_mxf8f6f4(acc + C::UP_OFF, desc_sw128(st + C::W_BYTES + k * 32), desc_sw128(xs + k * 32), id, sfu,
                             sfb, accum);
            }
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
      if (lane == 0) tc_commit(smem_u32(acc_full + buf));
      __syncwarp();
      if (++buf == C::NBUF) {
        buf = 0;
        acc_phase ^= 1;
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5, 128 threads) ----------------
    const int q = warp & 3;                  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;           // weight row within the tile (L1: i, L2: output col)
    const int et = threadIdx.x - 64;         // 0..127
    int buf = 0;
    uint32_t acc_phase = 0;
    int t = blockIdx.x, e = -1;
    while (next_item<BN>(a, msum, t, e)) {
      const int r0 = (t / a.n_wt) * BN, wt = t % a.n_wt;
      if (et < BN) row_ok[et] = (r0 + et < msum && __ldg(a.expert_ids + r0 + et) == e) ? 1 : 0;
      bool ok = mbar_wait(smem_u32(acc_full + buf), acc_phase, a.status) && *abort_flag == 0;
      // one vote over the four epilogue warps (also orders the row_ok writes before their reads)
      ok = named_barrier_and(1, 128, ok);
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t acc = tmem + buf * C::ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
      if (L1) {
        // pass 1: per-token amax of h over the 128 rows of this tile
        for (int n0 = 0; n0 < BN; n0 += 16) {
          uint32_t g[16], u[16];
          tc_ld_x16(acc + n0, g);
          tc_ld_x16(acc + C::UP_OFF + n0, u);
          tc_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float gv = __uint_as_float(g[j]);
            float m = fabsf(gv / (1.0f + expf(-gv)) * __uint_as_float(u[j]));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            if (lane == 0) red[q * BN + n0 + j] = m;
          }
        }
        named_barrier(1, 128);
        if (et < BN && row_ok[et]) {
          const float am = fmaxf(fmaxf(red[et], red[BN + et]), fmaxf(red[2 * BN + et], red[3 * BN + et]));
          a.h_sf[act_sf_offset(BN, a.sf_nb, r0 + et, wt)] = static_cast<uint8_t>(ue8m0_exponent(am) + 127);
        }
        // pass 2: quantise and store
        for (int n0 = 0; n0 < BN; n0 += 16) {
          uint32_t g[16], u[16];
          tc_ld_x16(acc + n0, g);
          tc_ld_x16(acc + C::UP_OFF + n0, u);
          tc_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int n = n0 + j;
            if (!row_ok[n]) continue;
            const float am = fmaxf(fmaxf(red[n], red[BN + n]), fmaxf(red[2 * BN + n], red[3 * BN + n]));
            const float sc = pow2_neg(ue8m0_exponent(am));
            const float gv = __uint_as_float(g[j]);
            const float h = gv / (1.0f + expf(-gv)) * __uint_as_float(u[j]);
            const __nv_fp8x2_storage_t p = __nv_cvt_float2_to_fp8x2(make_float2(h * sc, 0.f), __NV_SATFINITE, __NV_E4M3);
            a.h_q[static_cast<size_t>(r0 + n) * a.out_cols + wt * 128 + row] = static_cast<uint8_t>(p & 0xFF);
          }
        }
      } else {
        for (int n0 = 0; n0 < BN; n0 += 16) {
          uint32_t v[16];
          tc_ld_x16(acc + n0, v);
          tc_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int n = n0 + j;
            if (!row_ok[n]) continue;
            const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(v[j]));
            a.y[static_cast<size_t>(r0 + n) * a.out_cols + wt * 128 + row] = __bfloat16_as_ushort(b);
          }
        }
      }
      tc_fence_before();
      named_barrier(1, 128);               // row_ok / red reuse on the next item
      mbar_arrive(smem_u32(acc_empty + buf));
      if (++buf == C::NBUF) {
        buf = 0;
        acc_phase ^= 1;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------------------------------
// Host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

static bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

template <int BN, bool L1>
static cudaError_t launch_gemm_t(const GemmLaunch& L, cudaStream_t stream) {
  using C = GemmCfg<BN, L1>;
  CUtensorMap mw, mx;
  const int E_rows = L.E * L.w_rows;
  if (!make_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, L.w_q, L.Kd, E_rows, L.Kd / 2, 128, 128))
    return cudaErrorInvalidValue;
  if (!make_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.x, L.Kd, L.U, L.Kd, 128, BN)) return cudaErrorInvalidValue;
  GemmArgs a;
  a.w_sf = L.w_sf;
  a.x_sf = L.x_sf;
  a.expert_ids = L.expert_ids;
  a.m_sum = L.m_sum;
  a.h_q = L.h_q;
  a.h_sf = L.h_sf;
  a.y = L.y;
  a.status = L.status;
  a.w_sf_bytes = static_cast<size_t>(L.E) * L.w_rows * (L.Kd / 32);
  a.x_sf_bytes = act_sf_bytes(L.U, L.Kd / 128, BN);
  a.n_slabs = L.Kd / 128;
  a.w_rows = L.w_rows;
  a.n_wt = L1 ? L.I / 128 : L.w_rows / 128;
  a.up_off = L1 ? L.I : 0;
  a.out_cols = L1 ? L.I : L.w_rows;
  a.sf_nb = act_sf_blocks(L.U, BN);
  const int nrb = (L.U + BN - 1) / BN;
  a.n_tiles = nrb * a.n_wt;
  int grid = num_sms();
  if (grid > a.n_tiles) grid = a.n_tiles;
  if (grid < 1) grid = 1;
  cudaError_t err = cudaFuncSetAttribute(moe_gemm_kernel<BN, L1>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (err != cudaSuccess) return err;
  moe_gemm_kernel<BN, L1><<<grid, kGemmThreads, C::SMEM, stream>>>(mw, mx, a);
  return cudaGetLastError();
}

int gemm_block_n(int align) { return act_sf_block_rows(align); }

cudaError_t launch_gemm(const GemmLaunch& L, bool l1, cudaStream_t stream) {
  const int bn = gemm_block_n(L.align);
  if (l1) {
    switch (bn) {
      case 16: return launch_gemm_t<16, true>(L, stream);
      case 32: return launch_gemm_t<32, true>(L, stream);
      case 64: return launch_gemm_t<64, true>(L, stream);
      default: return launch_gemm_t<128, true>(L, stream);
    }
  }
  switch (bn) {
    case 16: return launch_gemm_t<16, false>(L, stream);
    case 32: return launch_gemm_t<32, false>(L, stream);
    case 64: return launch_gemm_t<64, false>(L, stream);
    default: return launch_gemm_t<128, false>(L, stream);
  }
}

// ------------------------------------------------------------------------------------------
// Weight scale packing: logical [E*N, Kd/32] UE8M0 -> per (128-row tile, 128-deep slab) a
// 512-byte image whose byte l*16 + w*4 + b holds row (32w + l), k-block (4*slab + b).
__global__ void pack_mx_scales_kernel(const uint8_t* __restrict__ sf, int rows, int kblocks,
                                      uint8_t* __restrict__ out) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(rows) * kblocks;
  if (i >= total) return;
  const int nslab = kblocks / 4;
  const long long chunk = i / 512;
  const int within = static_cast<int>(i % 512);
  const int rt = static_cast<int>(chunk / nslab), s = static_cast<int>(chunk % nslab);
  const int l = within / 16, w = (within / 4) & 3, b = within & 3;
  const int r = rt * 128 + w * 32 + l;
  out[i] = sf[static_cast<size_t>(r) * kblocks + s * 4 + b];
}

cudaError_t launch_pack_mx(const uint8_t* sf, int rows, int Kd, uint8_t* out, cudaStream_t stream) {
  const int kblocks = Kd / 32;
  const long long total = static_cast<long long>(rows) * kblocks;
  if (total == 0) return cudaSuccess;
  pack_mx_scales_kernel<<<static_cast<int>((total + 255) / 256), 256, 0, stream>>>(sf, rows, kblocks, out);
  return cudaGetLastError();
}

}  // namespace moe
