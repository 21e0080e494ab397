// Block-scaled grouped GEMMs of the MoE layer on tcgen05 (sm_103a):
//   L1: gu = X @ W13[e]^T, h = silu(gu[:I]) * gu[I:], FP8 requant per 128 along I
//   L2: y  = h @ W2[e]^T, bf16
// Page "DeepSeek V4 MegaMoE Kernel 深度解析", 二、阶段 2-4 (FP8 E4M3 activations x FP4 E2M1
// weights with UE8M0 scales, TMA -> shared memory -> scales copied into TMEM -> UMMA ->
// TMEM accumulators, full/empty barrier pipeline, SwiGLU + amax -> UE8M0 -> E4M3 epilogue).
//
// Design (this file's own, for one GPU):
//  * One MMA is M = 128 token rows x N = 256 weight rows x K = 32.  On this part a block-scaled
//    M=128 MMA occupies the tensor pipe for about the same time at N = 16 as at N = 128, and an
//    N = 256 one for ~1.3x that, so the weights go on the N side, 256 rows at a time: at decode
//    (a handful of tokens per expert) the tensor pipe then moves weights at ~2x HBM speed.
//    L1 tiles are 128 gate rows + the matching 128 up rows, so one thread (= one token, one TMEM
//    lane) holds both SwiGLU halves and the whole 128-wide requant group of its row.
//  * A work item is (row block of BN permuted rows, weight tile, expert).  Only the block's BN
//    token rows are loaded; the MMA's other rows read unrelated shared memory and their results
//    are never stored.  BN divides the permute alignment in the common case, so a block holds
//    one expert; otherwise each expert in the block is a separate pass with masked stores.
//  * moe_forward runs L1 and L2 as one launch: L2 items wait (bounded) on per-row-block counters of
//    finished L1 tiles, so the L1 tail wave and the launch gap are filled with L2 work.
//  * Persistent CTAs (one per SM) draw the items in index order from a counter in the workspace
//    (BatchedExperts: only the row blocks that hold tokens, from expert_num_tokens); a producer
//    warp (TMA), an MMA warp (one thread issues tcgen05.cp + tcgen05.mma) and eight epilogue
//    warps run decoupled through mbarriers.  The 128x256 fp32 accumulator takes half of TMEM and is single-buffered;
//    the shared-memory ring keeps the weights streaming while the epilogue drains it.
//  * Weights come pre-packed (moe_pack_weights): per (expert, tile, 128-deep slab) one chunk of
//    256 rows of FP4 codes followed by two 512-byte scale images.  The codes are loaded with the
//    padded 4-bit TMA type (16 codes -> 16 bytes of shared memory, 128-byte swizzle), the operand
//    layout kind::mxf8f6f4 reads; the scale images go to TMEM with tcgen05.cp .32x128b.warpx4,
//    where weight row n is read from column n/32 (byte = k-step) and token row m from column m/32
//    (byte = slab % 4).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "permute_small.cuh"
#include "route_small.cuh"

namespace moe {

constexpr int kGemmThreads = 352;        // warps 0 and 10 TMA, warp 1 MMA, warps 2..9 epilogue
constexpr int kProducer2Warp = 10;       // second copy-issuing warp (odd slabs)
constexpr int kEpiThreads = 256;         // two warps per TMEM lane quarter, one per column half
constexpr int kEpiThread0 = 64;          // first epilogue thread
constexpr int kSmemBudget = 227 * 1024;
constexpr int kGemmStaticSmem = 6 * 1024;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: accumulator [0, 256); token scales 2 slots x 16 at 256; weight scales 2 x 16 at 288.
constexpr uint32_t kSfaCol = 256;
constexpr uint32_t kSfbCol = 288;
constexpr int kTileRows = 256;           // weight rows per tile (MMA N)

template <int BN>
struct GemmCfg {
  static constexpr int X_BYTES = BN * 128;                       // token rows loaded per slab
  static constexpr int X_SLOT = (X_BYTES + 1023) / 1024 * 1024;  // MMA reads 16 KB from here
  static constexpr int W_OFF = X_SLOT;
  static constexpr int W_BYTES = kTileRows * 128;                // 256 rows of padded FP4 codes
  static constexpr int SFB_OFF = W_OFF + W_BYTES;                // weight scale images (2 x 512 B)
  static constexpr int SFA_OFF = SFB_OFF + 1024;                 // token scale chunk (every 4th slab)
  static constexpr int SFA_BYTES = 512;
  static constexpr int STAGE = (SFA_OFF + SFA_BYTES + 1023) / 1024 * 1024;
  static constexpr int EXTRA = 1024;                             // barriers and flags
  // dynamic + static shared memory (6 KB: the row-block prefix and the amax exchange) within the budget
  static constexpr int S_FIT = (kSmemBudget - kGemmStaticSmem - EXTRA - 1024) / STAGE;
  static constexpr int STAGES = S_FIT > 8 ? 8 : S_FIT;
  static constexpr int SMEM = 1024 + STAGES * STAGE + EXTRA;
  static constexpr uint32_t TX_W = kTileRows * 64;               // global bytes of the FP4 box
  static constexpr size_t W_CHUNK = 2 * (8192 + 512);            // packed bytes per (tile, slab)
  static_assert(STAGES >= 3, "shared memory too small");
  static_assert(X_SLOT + 16384 <= STAGE, "MMA A reads must stay inside the stage");
};

// Single-launch forward: the small-batch routing and permute run inside the GEMM launch first.
struct PreludeArgs {
  RouteFinishArgs r;            // routing (its topk_ids, topk_w, logits, x_q, x_sf are stored by CTA 0 / all)
  const float* w_gate;          // [E, H]
  float* partial;               // [kGemvSplit, T, E] gate partial sums
  PermuteArgs p;                // the small permute over the routing's ids
  const uint8_t* x_q;           // [T, H] E4M3 (written by the routing phase)
  const uint8_t* x_sf;          // [T, H/128]
  uint8_t* x_perm;              // [U, H]
  uint8_t* x_perm_sf;           // tiled
  int H, bt, nb;
};

// One GEMM of the layer as the kernel sees it.
struct GemmPhase {
  const uint8_t* w;             // packed weight stream
  const uint8_t* x_sf;          // tiled token scales (rows U, block rows BN)
  size_t w_bytes;               // sizes, for the kernel's own bounds checks
  size_t x_sf_bytes;
  int n_slabs;                  // reduction depth / 128
  int n_wt;                     // weight tiles per expert
  int out_cols;                 // L1: I, L2: H
  int n_tiles;                  // ceil(U/BN) * n_wt; 0 = phase not run by this launch
  // Gather mode (L1): the activation tensor map covers the token-order rows [T, Kd], and permuted
  // row r reads token gather_ids[r] / gather_k (gather_ids = sorted_token_ids [U]; padding rows
  // name token T, past the tensor, and read zeros).  nullptr: the map covers the permuted rows.
  const int32_t* gather_ids;
  int gather_k;
  int gather_rows;              // T
  int gather_u;                 // entries of gather_ids
};

struct GemmArgs {
  GemmPhase ph[2];              // [0] L1: W13, SwiGLU, FP8 requant; [1] L2: W2, bf16
  const int32_t* expert_ids;    // [U]
  const int32_t* m_sum;         // [1]
  uint8_t* h_q;                 // L1 out [U, I]
  uint8_t* h_sf;                // L1 out, tiled (rows U, slabs I/128)
  uint16_t* y;                  // L2 out [U, H] bf16
  uint32_t* status;
  int sf_nb;                    // blocks of the tiled token-scale layouts
  uint32_t* sched;              // [n_ready + 4] words, zero at launch and left at zero by the last CTA
                                // to exit: [0, n_ready) finished L1 tiles per row block (fused
                                // launches), [n_ready] next work item, [n_ready + 1] exited CTAs,
                                // [n_ready + 2, + 3] the single-launch forward's grid barriers
  int n_ready;                  // ceil(U/BN)
  int fused;                    // both phases in one launch: L2 items wait for their block's L1 tiles
  int one_expert_blocks;        // permute alignment is a multiple of BN: one expert per row block
  FusedReduce red;              // L2: unpermute-reduce in the epilogue when red.out != nullptr
  const int32_t* row_ids;       // L1: h of row r scaled by row_w[row_ids[r]] when row_w != nullptr
  const float* row_w;
  // BatchedExperts (masked) mode: expert e owns slot_blocks row blocks from row block
  // e * slot_blocks, of which ceil(counts[e] / BN) hold tokens; only those are work items
  const int32_t* counts;        // nullptr: every row block below m_sum is an item
  int slot_blocks;
  int E;
};

// The kernel's last parameter: the prelude's arguments in the single-launch instance, nothing
// (an empty struct) in the others, so that their parameter block stays as small as before.
struct NoPrelude {};
template <bool PRELUDE>
using PreludeParam = typename std::conditional<PRELUDE, PreludeArgs, NoPrelude>::type;

constexpr int kMaxMaskedExperts = 1024;   // masked mode: experts in the shared prefix table

// Work items: the L1 tiles of the row blocks below m_sum, then their L2 tiles, each phase
// row-block major (t = row_block * n_wt + weight_tile).  The producer warp of each CTA takes the
// next index from a global counter, so items start in index order and a CTA that drew short
// items draws more of them.  It hands (t, expert) to the MMA and epilogue warps through a small
// ring in shared memory.
struct Item {
  int phase, rb, wt;
};

// bpre (masked mode, shared memory): bpre[e] = active row blocks of experts < e, bpre[E] = all.
__device__ __forceinline__ Item decode_item(const GemmArgs& a, int n0, int t, const int* bpre) {
  Item it;
  it.phase = t >= n0 ? 1 : 0;
  const int l = it.phase ? t - n0 : t;
  const int ab = l / a.ph[it.phase].n_wt;
  it.wt = l - ab * a.ph[it.phase].n_wt;
  if (bpre == nullptr) {
    it.rb = ab;
  } else {                                 // expert e with bpre[e] <= ab < bpre[e + 1]
    int lo = 0, hi = a.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (bpre[mid] <= ab) lo = mid;
      else hi = mid;
    }
    it.rb = lo * a.slot_blocks + (ab - bpre[lo]);
  }
  return it;
}

// Smallest expert id > e among the rows of the block starting at row r0 (rows are sorted by
// expert, ignoring -1).  Called by whole warps.  When the permute alignment is a multiple of BN every block lies
// inside one expert's segment (real rows first, then padding), so the block's first entry names
// its only expert (-1: the block is padding); otherwise the warp scans the block in one round.
template <int BN>
__device__ __forceinline__ bool find_expert(const GemmArgs& a, int msum, int r0, int& e) {
  if (a.one_expert_blocks) {
    if (e >= 0) return false;
    const int x = __ldg(a.expert_ids + r0);
    if (x < 0) return false;
    e = x;
    return true;
  }
  const int lane = threadIdx.x & 31;
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
  if (best == 0x7fffffff) return false;
  e = best;
  return true;
}

// Two floats -> bf16 (round to nearest even) packed low | high << 16, one conversion instruction.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// silu(g) * u with the fast exponential and division intrinsics: the result is requantised to
// E4M3 (3 mantissa bits), far coarser than their few-ulp error, and unlike the IEEE division they
// have no slow path for the infinities that unused accumulator rows may hold.
__device__ __forceinline__ float silu_mul(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

constexpr int kItemSlots = 4;

// One thread issues the copies of an item's slabs whose running slab index gslab has parity
// `mine`: the two producer warps take alternate slabs, since a thread issues a bulk copy only
// every ~300 cycles and one thread could not keep the ring full.  stage / phase / gslab advance
// over every slab of the item (both producers see every item); a failed wait or range check stops
// the loop and returns false.  The copy ranges are checked once per item.
template <int BN>
__device__ __forceinline__ bool issue_mx_slabs(const GemmArgs& a, const GemmPhase& P, const CUtensorMap* mw,
                                               const CUtensorMap* mx, int r0, size_t chunk0, uint32_t mine,
                                               uint8_t* stages, uint64_t* full, uint64_t* empty, int& stage,
                                               uint32_t& phase, uint32_t& gslab, uint64_t pol_w, uint64_t pol_x) {
  using C = GemmCfg<BN>;
  const size_t wend = (chunk0 + P.n_slabs) * C::W_CHUNK;
  const size_t sfa_last = (static_cast<size_t>((P.n_slabs - 1) >> 2) * a.sf_nb + r0 / BN) * act_sf_chunk_bytes(BN);
  if (!(wend <= P.w_bytes && sfa_last + C::SFA_BYTES <= P.x_sf_bytes &&
        ((reinterpret_cast<uintptr_t>(P.w) | reinterpret_cast<uintptr_t>(P.x_sf)) & 15) == 0)) {
    record_error(a.status, kDevErrCheck);
    return false;
  }
  const uint32_t stages0 = smem_u32(stages);
  const uint8_t* wsrc = P.w + chunk0 * C::W_CHUNK;
  int wrow = static_cast<int>(chunk0 * C::W_CHUNK / 64);
  for (int s = 0; s < P.n_slabs; ++s) {
    if ((gslab & 1u) == mine) {
      if (!mbar_wait(smem_u32(empty + stage), phase ^ 1, a.status)) return false;
      const uint32_t st = stages0 + static_cast<uint32_t>(stage * C::STAGE);
      const uint32_t fb = smem_u32(full + stage);
      const bool sf4 = (s & 3) == 0;
      mbar_arrive_expect_tx(fb, C::TX_W + 1024 + C::X_BYTES + (sf4 ? C::SFA_BYTES : 0));
      tma_load_2d(st + C::W_OFF, mw, 0, wrow, fb, pol_w);
      bulk_load(st + C::SFB_OFF, wsrc + C::TX_W, 1024, fb);
      tma_load_2d(st, mx, s * 128, r0, fb, pol_x);
      if (sf4)
        bulk_load(st + C::SFA_OFF, P.x_sf + (static_cast<size_t>(s >> 2) * a.sf_nb + r0 / BN) * act_sf_chunk_bytes(BN),
                  C::SFA_BYTES, fb);
    }
    wsrc += C::W_CHUNK;
    wrow += static_cast<int>(C::W_CHUNK / 64);
    ++gslab;
    if (++stage == C::STAGES) {
      stage = 0;
      phase ^= 1;
    }
  }
  return true;
}

// Every CTA of a cooperative launch arrives on the counter and waits until all have (bounded:
// false, with the status recorded, if the wait runs out).  Thread 0 arrives and waits, with fences
// on both sides as a grid-wide barrier needs; the CTA's barriers spread the result.
__device__ __forceinline__ bool grid_barrier(uint32_t* ctr, uint32_t* status, volatile int* flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ctr, 1u);
    const bool ok = wait_counter(ctr, gridDim.x, status);
    __threadfence();
    *flag = ok ? 1 : 0;
  }
  __syncthreads();
  return *flag != 0;
}

// Runs the L1 items, the L2 items, or both.  With both, an L2 item of row block rb reads h rows
// written by other CTAs: its producer first waits until sched[rb] counts all n_wt L1 tiles of the
// block (each L1 item's epilogue adds one after its stores).  Items are drawn in index order, all
// L1 items before any L2 item; a producer waits only while holding an L2 item, after issuing every
// load of the items it drew before.  So every awaited L1 item was drawn by a CTA that is running
// (or has finished it), and that CTA's MMA and epilogue warps complete it whatever its producer
// waits for: progress needs no co-residency of the CTAs, and the wait is bounded all the same.
// The last CTA to exit sets all counters back to zero: no CTA can still be waiting or drawing then.
// GATHER: the L1 phase reads its token rows with four-row gathers (GemmPhase::gather_ids); a
// separate instance, so that the permuted-copy path carries none of that bookkeeping.
// PRELUDE (the single-launch forward, small batches; the launch is cooperative, so every CTA is
// resident): before the FFN work the CTAs run the small-batch routing (the blocks of its grid
// spread over the CTAs, threads 0..255 of each), meet at a grid barrier, then each CTA computes
// the top-K of every token into shared memory (CTA 0 stores the routing outputs) and runs the
// small permute on it (CTA 0 stores the indices; padding, tail and row copies are split over the
// CTAs), and they meet again.  The same device functions as the routing and permute launches,
// so the results are the same bits.
template <int BN, bool GATHER, bool PRELUDE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w1, const __grid_constant__ CUtensorMap tmap_x1,
                    const __grid_constant__ CUtensorMap tmap_w2, const __grid_constant__ CUtensorMap tmap_x2,
                    const GemmArgs a, const PreludeParam<PRELUDE> pre) {
  using C = GemmCfg<BN>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* extra = smem + C::STAGES * C::STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(extra);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* item_full = acc_empty + 1;             // [kItemSlots], producer arrives
  uint64_t* item_empty = item_full + kItemSlots;   // [kItemSlots], MMA warp, epilogue, producer 2 arrive
  // (t, e, row block, weight tile | phase << 16), decoded once by the producer; t < 0 ends the work
  int4* items = reinterpret_cast<int4*>(item_empty + kItemSlots);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(items + kItemSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 1);
    }
    mbar_init(smem_u32(acc_full), 1);
    mbar_init(smem_u32(acc_empty), kEpiThreads);
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(smem_u32(item_full + s), 1);
      mbar_init(smem_u32(item_empty + s), 3);   // MMA thread, epilogue, second producer
    }
    *abort_flag = 0;
    fence_barrier_init();
    if (a.ph[0].n_tiles) {
      prefetch_tmap(&tmap_w1);
      prefetch_tmap(&tmap_x1);
    }
    if (a.ph[1].n_tiles) {
      prefetch_tmap(&tmap_w2);
      prefetch_tmap(&tmap_x2);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if constexpr (PRELUDE) {
    // scratch in the ring (not yet in use): partial-sum exchange [8][4 * 16] floats, the top-K ids
    // (<= 128), the permute's counts, segment starts, ids and ranks (256 each), total and a flag
    float(*red)[kGemvE * kGemvT] = reinterpret_cast<float(*)[kGemvE * kGemvT]>(stages);
    int32_t* s_topk = reinterpret_cast<int32_t*>(stages + 8 * kGemvE * kGemvT * sizeof(float));
    int32_t* p_cnt = s_topk + 128;
    int32_t* p_seg = p_cnt + 256;
    int32_t* p_ids = p_seg + 256;
    int32_t* p_rank = p_ids + 256;
    int32_t* p_total = p_rank + 256;
    volatile int* p_flag = reinterpret_cast<volatile int*>(p_total + 1);
    const PreludeArgs& q = pre;
    const int gx = (q.r.E + kGemvE - 1) / kGemvE;
    const auto sync256 = [] { named_barrier(2, 256); };
    for (int vb = blockIdx.x; vb < gx * kGemvSplit; vb += gridDim.x) {
      if (threadIdx.x < 256) {
        route_small_gemv<kGemvT>(q.r, q.w_gate, q.partial, vb % gx, vb / gx, gx, threadIdx.x, red, sync256);
        named_barrier(2, 256);   // red is reused by the next block
      }
    }
    bool pre_ok = grid_barrier(a.sched + a.n_ready + 2, a.status, p_flag);
    if (pre_ok) {
      if (threadIdx.x < 256) {
        if (blockIdx.x == 0)   // CTA 0 also stores the routing outputs
          route_small_topk<kGemvT, 8, true, true>(q.r, q.partial, threadIdx.x / 32, threadIdx.x % 32, s_topk);
        else
          route_small_topk<kGemvT, 8, true, false>(q.r, q.partial, threadIdx.x / 32, threadIdx.x % 32, s_topk);
        named_barrier(2, 256);   // every token's ids in s_topk
        permute_small_body<256, true>(q.p, s_topk, q.x_q, q.x_sf, q.H, q.x_perm, q.x_perm_sf, q.bt, q.nb, p_cnt, p_seg, p_ids,
                                p_rank, p_total, threadIdx.x, blockIdx.x, gridDim.x, sync256);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the ring's next writers are copies
      fence_proxy_async_global();   // x_perm and its scales are read next by TMA and bulk copies
      pre_ok = grid_barrier(a.sched + a.n_ready + 3, a.status, p_flag);
      fence_proxy_async_global();
    }
    if (!pre_ok && threadIdx.x == 0) *abort_flag = 1;   // every role then stops before its first item
  }
  // masked mode: each expert's row blocks that hold tokens, loaded by all threads at once; the
  // prefix over experts is formed after the barrier below
  __shared__ int s_bpre[kMaxMaskedExperts + 1];
  grid_dependency_wait();          // everything below reads the previous launch's results
  if (a.counts)
    for (int e = threadIdx.x; e < a.E; e += kGemmThreads)
      s_bpre[e] = min((max(__ldg(a.counts + e), 0) + BN - 1) / BN, a.slot_blocks);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int msum = *a.m_sum;
  // masked mode: exclusive prefix of the experts' active row blocks, in place (an epilogue warp,
  // idle at this point)
  const int* bpre = nullptr;
  if (a.counts) {
    if (warp == 2) {
      int run = 0;
      for (int e0 = 0; e0 < a.E; e0 += 32) {
        const int e = e0 + lane;
        const int nb = e < a.E ? s_bpre[e] : 0;
        int incl = nb;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += v;
        }
        if (e < a.E) s_bpre[e] = run + incl - nb;
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) s_bpre[a.E] = run;
    }
    __syncthreads();
    bpre = s_bpre;
  }
  const int nrb = bpre ? bpre[a.E] : (msum + BN - 1) / BN;
  const int n0 = a.ph[0].n_tiles ? nrb * a.ph[0].n_wt : 0;
  const int n_items = n0 + (a.ph[1].n_tiles ? nrb * a.ph[1].n_wt : 0);

  if (warp == 0) {
    // ---------------- TMA producer (whole warp iterates, lane 0 issues) ----------------
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0, gslab = 0;
    uint32_t islot = 0, iphase = 0;
    int t = -1, e = -1;
    Item it{0, 0, 0};
    bool ok = true;
    while (ok && !__any_sync(0xffffffffu, *abort_flag != 0)) {
      bool have = t >= 0 && find_expert<BN>(a, msum, it.rb * BN, e);    // another expert of the same block
      while (!have) {
        int nt = 0;
        if (lane == 0) nt = static_cast<int>(atomicAdd(a.sched + a.n_ready, 1u));
        nt = __shfl_sync(0xffffffffu, nt, 0);
        if (nt >= n_items) {
          t = -1;
          break;
        }
        t = nt;
        e = -1;
        it = decode_item(a, n0, t, bpre);
        have = find_expert<BN>(a, msum, it.rb * BN, e);
      }
      if (!have) break;
      // hand the item to the MMA and epilogue warps
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(item_empty + islot), iphase ^ 1, a.status));
      if (!ok) break;
      if (lane == 0) {
        items[islot] = make_int4(t, e, it.rb, it.wt | (it.phase << 16));
        mbar_arrive(smem_u32(item_full + islot));
      }
      __syncwarp();
      if (++islot == kItemSlots) {
        islot = 0;
        iphase ^= 1;
      }
      const GemmPhase& P = a.ph[it.phase];
      const CUtensorMap* mw = it.phase ? &tmap_w2 : &tmap_w1;
      const CUtensorMap* mx = it.phase ? &tmap_x2 : &tmap_x1;
      const int r0 = it.rb * BN;
      const size_t chunk0 = (static_cast<size_t>(e) * P.n_wt + it.wt) * P.n_slabs;
      // gather mode: lane j (< BN / 4) copies rows 4j .. 4j + 3 of the block, tokens looked up once
      const bool gather = GATHER && P.gather_ids != nullptr;
      int g_tok[4] = {0, 0, 0, 0};
      if (gather && lane < BN / 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = r0 + 4 * lane + i;
          const int tk = r < P.gather_u ? __ldg(P.gather_ids + r) / P.gather_k : P.gather_rows;
          g_tok[i] = (tk < 0 || tk > P.gather_rows) ? P.gather_rows : tk;
        }
      }
      if (it.phase == 1 && a.fused) {
        // h rows of this block come from other CTAs' L1 epilogues
        if (lane == 0) {
          const uint32_t need = static_cast<uint32_t>(a.ph[0].n_wt);
          if (ld_acquire_gpu(a.sched + it.rb) < need) {
            // start the item's weights towards L2 while waiting
            const size_t wb = chunk0 * C::W_CHUNK, nb = static_cast<size_t>(P.n_slabs) * C::W_CHUNK;
            if (wb + nb <= P.w_bytes && nb < (size_t(1) << 31)) bulk_prefetch_l2(P.w + wb, static_cast<uint32_t>(nb));
            ok = wait_counter(a.sched + it.rb, need, a.status);
          }
          fence_proxy_async_global();
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (!gather) {
        // lane 0 issues the item's even slabs (warp 10 the odd ones)
        if (lane == 0 && ok) {
          ok = issue_mx_slabs<BN>(a, P, mw, mx, r0, chunk0, 0u, stages, full, empty, stage, phase, gslab, pol_w, pol_x);
          if (!ok) *abort_flag = 1;
        }
        // lane 0's ring position and status for the whole warp
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        stage = __shfl_sync(0xffffffffu, stage, 0);
        phase = __shfl_sync(0xffffffffu, phase, 0);
        gslab = __shfl_sync(0xffffffffu, gslab, 0);
        continue;
      }
      for (int s = 0; ok && s < P.n_slabs; ++s) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(empty + stage), phase ^ 1, a.status));
        if (!ok) break;
        bool good = true;
        if (lane == 0) {
          uint8_t* st = stages + stage * C::STAGE;
          const uint32_t fb = smem_u32(full + stage);
          const size_t wbase = (chunk0 + s) * C::W_CHUNK;
          const size_t sfa = (static_cast<size_t>(s >> 2) * a.sf_nb + r0 / BN) * act_sf_chunk_bytes(BN);
          // self-check: every copy inside its buffer and 16-byte aligned
          good = wbase + C::W_CHUNK <= P.w_bytes &&
                 ((s & 3) != 0 || sfa + C::SFA_BYTES <= P.x_sf_bytes) &&
                 ((reinterpret_cast<uintptr_t>(P.w) | reinterpret_cast<uintptr_t>(P.x_sf)) & 15) == 0;
          if (!good) {
            record_error(a.status, kDevErrCheck);
            *abort_flag = 1;
          } else {
            uint32_t bytes = C::TX_W + 1024 + C::X_BYTES;
            if ((s & 3) == 0) bytes += C::SFA_BYTES;
            mbar_arrive_expect_tx(fb, bytes);
            tma_load_2d(smem_u32(st + C::W_OFF), mw, 0, static_cast<int>(wbase / 64), fb, pol_w);
            bulk_load(smem_u32(st + C::SFB_OFF), P.w + wbase + C::TX_W, 1024, fb);
            if (!gather) tma_load_2d(smem_u32(st), mx, s * 128, r0, fb, pol_x);
            if ((s & 3) == 0) bulk_load(smem_u32(st + C::SFA_OFF), P.x_sf + sfa, C::SFA_BYTES, fb);
          }
        }
        if (gather) {                          // warp-uniform: the other lanes copy the token rows
          good = __shfl_sync(0xffffffffu, good, 0);
          if (good && lane < BN / 4)
            tma_gather4(smem_u32(stages + stage * C::STAGE + lane * 512), mx, s * 128, g_tok[0], g_tok[1], g_tok[2],
                        g_tok[3], smem_u32(full + stage), pol_x);
        }
        __syncwarp();
        ++gslab;
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok) *abort_flag = 1;
    // end of work for the other warps (if the ring does not free up they stop on their own waits)
    if (__all_sync(0xffffffffu, mbar_wait(smem_u32(item_empty + islot), iphase ^ 1, a.status))) {
      if (lane == 0) {
        items[islot] = make_int4(-1, -1, 0, 0);
        mbar_arrive(smem_u32(item_full + islot));
      }
      __syncwarp();
    }
    if (__any_sync(0xffffffffu, *abort_flag != 0)) {
      // let every copy issued into shared memory land before the CTA exits
      for (int s = 0; s < C::STAGES; ++s) mbar_wait(smem_u32(full + s), (s < stage) ? phase : (phase ^ 1), nullptr);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (one thread) ----------------
    // The loop between slabs is kept short (no warp votes; descriptors advanced by addition): the
    // MMA thread's time per slab must stay below the slab's arrival interval.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      uint32_t islot = 0, iphase = 0;
      const uint64_t dst0 = desc_sw128(smem_u32(stages));
      const uint32_t id0 = idesc_mxf8f6f4(0, 5, 128, kTileRows, 0, 0);
      while (true) {
        bool ok = mbar_wait(smem_u32(item_full + islot), iphase, a.status);
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        const int4 item = items[islot];
        mbar_arrive(smem_u32(item_empty + islot));
        if (++islot == kItemSlots) {
          islot = 0;
          iphase ^= 1;
        }
        if (item.x < 0 || *abort_flag != 0) break;
        const int n_slabs = a.ph[item.w >> 16].n_slabs;
        ok = mbar_wait(smem_u32(acc_empty), acc_phase ^ 1, a.status);
        if (ok) {
          tc_fence_after();
          for (int s = 0; s < n_slabs; ++s) {
            ok = mbar_wait(smem_u32(full + stage), phase, a.status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t st = smem_u32(stages + stage * C::STAGE);
            const uint32_t sfa = tmem + kSfaCol + ((s >> 2) & 1) * 16;
            const uint32_t sfb = tmem + kSfbCol + (s & 1) * 16;
            if ((s & 3) == 0) tc_cp_32x128b_x4(sfa, smem_desc(st + C::SFA_OFF, 0, 128, 0));
            tc_cp_32x128b_x4(sfb, smem_desc(st + C::SFB_OFF, 0, 128, 0));
            tc_cp_32x128b_x4(sfb + 4, smem_desc(st + C::SFB_OFF + 512, 0, 128, 0));
            // descriptor start addresses count 16-byte units: + 2 per 32-byte K step
            const uint64_t da = dst0 + static_cast<uint64_t>(stage * (C::STAGE >> 4));
            const uint64_t dw = da + static_cast<uint64_t>(C::W_OFF >> 4);
            const uint32_t ids = id0 | (static_cast<uint32_t>(s & 3) << 29);   // scale-factor id of A
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_mxf8f6f4(tmem, da + 2 * k, dw + 2 * k, ids | (static_cast<uint32_t>(k) << 4), sfa, sfb,
                           (s > 0 || k > 0) ? 1u : 0u);
            tc_commit(smem_u32(empty + stage));
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
        tc_commit(smem_u32(acc_full));
        acc_phase ^= 1;
      }
    }
    __syncwarp();
  } else if (warp == kProducer2Warp) {
    // ---------------- second producer (one thread): the odd slabs of every copy-path item ----------------
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, gslab = 0;
      uint32_t islot = 0, iphase = 0;
      while (true) {
        bool ok = mbar_wait(smem_u32(item_full + islot), iphase, a.status);
        const int4 item = items[islot];
        if (ok) mbar_arrive(smem_u32(item_empty + islot));
        if (++islot == kItemSlots) {
          islot = 0;
          iphase ^= 1;
        }
        if (!ok) *abort_flag = 1;
        if (!ok || item.x < 0 || *abort_flag != 0) break;
        const int ph = item.w >> 16;
        const GemmPhase& P = a.ph[ph];
        if (GATHER && P.gather_ids != nullptr) {
          // the first producer's whole warp issues gathered items; keep the ring position
          gslab += static_cast<uint32_t>(P.n_slabs);
          stage += P.n_slabs;
          phase ^= static_cast<uint32_t>((stage / C::STAGES) & 1);
          stage %= C::STAGES;
          continue;
        }
        if (ph == 1 && a.fused) {
          // the item's h rows come from other CTAs' L1 epilogues (the first producer waits too)
          const uint32_t need = static_cast<uint32_t>(a.ph[0].n_wt);
          if (ld_acquire_gpu(a.sched + item.z) < need) ok = wait_counter(a.sched + item.z, need, a.status);
          fence_proxy_async_global();
          if (!ok) {
            *abort_flag = 1;
            break;
          }
        }
        const size_t chunk0 = (static_cast<size_t>(item.y) * P.n_wt + (item.w & 0xFFFF)) * P.n_slabs;
        if (!issue_mx_slabs<BN>(a, P, ph ? &tmap_w2 : &tmap_w1, ph ? &tmap_x2 : &tmap_x1, item.z * BN, chunk0, 1u, stages,
                                full, empty, stage, phase, gslab, pol_w, pol_x)) {
          *abort_flag = 1;
          break;
        }
      }
      if (*abort_flag != 0) {
        // let every copy issued into shared memory land before the CTA exits
        for (int s = 0; s < C::STAGES; ++s) mbar_wait(smem_u32(full + s), (s < stage) ? phase : (phase ^ 1), nullptr);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..9): thread = token row m of the block, one column half --------
    // Warps 2..5 take the first half of the accumulator's columns and warps 6..9 the second, so each
    // thread drains half a row: two TMEM load rounds before the accumulator is released.
    __shared__ float s_amax[2][128];
    const int q = warp & 3;                  // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;
    const int m = q * 32 + lane;
    // Every epilogue warp drains its lane quarter, also when the block has no rows there (BN < 128):
    // those values are never stored (`mine` is false), and one code path for all warps keeps the
    // epilogue within the 168 registers a thread has without spilling (a per-warp branch around the
    // loads spilled 56 bytes at BN = 16, 32, 64).
    const bool warp_has_rows = true;
    const uint32_t acc = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t acc_phase = 0;
    uint32_t islot = 0, iphase = 0;
    while (true) {
      bool ok = mbar_wait(smem_u32(item_full + islot), iphase, a.status);
      const int4 item = items[islot];
      ok = named_barrier_and(1, kEpiThreads, ok);    // every epilogue thread has read the slot
      if (ok && threadIdx.x == kEpiThread0) mbar_arrive(smem_u32(item_empty + islot));
      if (++islot == kItemSlots) {
        islot = 0;
        iphase ^= 1;
      }
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      if (item.x < 0) break;
      const int e = item.y;
      const Item it{item.w >> 16, item.z, item.w & 0xFFFF};
      const int r0 = it.rb * BN, wt = it.wt;
      const int row = r0 + m;
      const int row_e = (m < BN && row < msum) ? __ldg(a.expert_ids + row) : -1;
      const bool mine = row_e == e;
      // the routing weight of this row's (token, slot) pair when it is applied in L1 (else 1)
      const float wr = (it.phase == 0 && a.row_w != nullptr && mine) ? __ldg(a.row_w + __ldg(a.row_ids + row)) : 1.f;
      ok = mbar_wait(smem_u32(acc_full), acc_phase, a.status) && *abort_flag == 0;
      ok = named_barrier_and(1, kEpiThreads, ok);    // one vote over the eight epilogue warps
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      if (it.phase == 0) {
        const int I = a.ph[0].out_cols;
        // This thread's 64 gate and 64 up values (of the tile's 128 columns) are read from TMEM in
        // one round and the accumulator is released before h = silu(gate) * up is formed; the
        // 128-wide amax combines both halves through shared memory
        float h[64];
        float amax = 0.f;
        if (warp_has_rows) {
          uint32_t g[4][16], u[4][16];
          const uint32_t col = static_cast<uint32_t>(half * 64);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            tc_ld_x16(acc + col + 16 * j, g[j]);
            tc_ld_x16(acc + 128 + col + 16 * j, u[j]);
          }
          tc_wait_ld();
          tc_fence_before();
          mbar_arrive(smem_u32(acc_empty));
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            h[j] = silu_mul(__uint_as_float(g[j >> 4][j & 15]), __uint_as_float(u[j >> 4][j & 15])) * wr;
            amax = fmaxf(amax, fabsf(h[j]));
          }
        } else {
          tc_fence_before();
          mbar_arrive(smem_u32(acc_empty));
        }
        s_amax[half][m] = amax;
        named_barrier(1, kEpiThreads);
        if (warp_has_rows && mine) {
          amax = fmaxf(amax, s_amax[half ^ 1][m]);
          const int ex = ue8m0_exponent(amax);
          const float sc = pow2_neg(ex);
          if (half == 0) a.h_sf[act_sf_offset(BN, a.sf_nb, row, wt)] = static_cast<uint8_t>(ex + 127);
          uint4* dst = reinterpret_cast<uint4*>(a.h_q + static_cast<size_t>(row) * I + wt * 128 + half * 64);
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 16) {
            uint32_t packed[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int c = c0 + 4 * j;
              const uint32_t lo =
                  __nv_cvt_float2_to_fp8x2(make_float2(h[c] * sc, h[c + 1] * sc), __NV_SATFINITE, __NV_E4M3);
              const uint32_t hi =
                  __nv_cvt_float2_to_fp8x2(make_float2(h[c + 2] * sc, h[c + 3] * sc), __NV_SATFINITE, __NV_E4M3);
              packed[j] = lo | (hi << 16);
            }
            dst[c0 / 16] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
          }
          if (a.fused) fence_proxy_async_global();
        }
        if (a.fused) {
          // publish the tile once the block's last expert pass is stored: bar.red doubles as the
          // barrier that orders all epilogue threads' stores before the release below
          const bool later = row_e > e;
          if (!named_barrier_or(1, kEpiThreads, later) && threadIdx.x == kEpiThread0) {
            __threadfence();
            atomicAdd(a.sched + it.rb, 1u);
          }
        }
      } else {
        const int H = a.ph[1].out_cols;
        const int ncols = min(kTileRows, H - wt * kTileRows) - half * (kTileRows / 2);   // this half's columns
        // 128 outputs in two rounds of 64 columns: round 0 is packed to bf16 pairs while round 1's
        // TMEM loads are issued; the accumulator is released once round 1 has landed, and both
        // rounds are stored after that
        if (warp_has_rows) {
          uint4* dst = reinterpret_cast<uint4*>(a.y + static_cast<size_t>(row) * H + wt * kTileRows +
                                                half * (kTileRows / 2));
          const uint32_t col = static_cast<uint32_t>(half * (kTileRows / 2));
          uint32_t v[4][16];
          uint32_t p0[32];
#pragma unroll
          for (int j = 0; j < 4; ++j) tc_ld_x16(acc + col + 16 * j, v[j]);
          tc_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) p0[j] = pack_bf16x2(__uint_as_float(v[j >> 3][(2 * j) & 15]),
                                                            __uint_as_float(v[j >> 3][(2 * j + 1) & 15]));
#pragma unroll
          for (int j = 0; j < 4; ++j) tc_ld_x16(acc + col + 64 + 16 * j, v[j]);
          tc_wait_ld();
          tc_fence_before();
          mbar_arrive(smem_u32(acc_empty));
          if (mine) {
#pragma unroll
            for (int c = 0; c < 8; ++c)
              if (c * 8 < ncols) dst[c] = make_uint4(p0[4 * c], p0[4 * c + 1], p0[4 * c + 2], p0[4 * c + 3]);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              if (64 + c * 8 < ncols) {
                uint32_t q4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const int j = 4 * c + i;
                  q4[i] = pack_bf16x2(__uint_as_float(v[j >> 3][(2 * j) & 15]),
                                      __uint_as_float(v[j >> 3][(2 * j + 1) & 15]));
                }
                dst[8 + c] = make_uint4(q4[0], q4[1], q4[2], q4[3]);
              }
            }
          }
        } else {
          tc_fence_before();
          mbar_arrive(smem_u32(acc_empty));
        }
        if (a.red.out && ncols > 0)
          fused_reduce_tail(a.red, a.y, H, mine, row, wt * 2 + half, a.ph[1].n_wt * 2,
                            wt * kTileRows + half * (kTileRows / 2), min(ncols, kTileRows / 2));
      }
      acc_phase ^= 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  __shared__ int s_last_cta;
  if (threadIdx.x == 0) {
    __threadfence();
    s_last_cta = atomicAdd(a.sched + a.n_ready + 1, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (s_last_cta) {
    __threadfence();
    for (int i = threadIdx.x; i < a.n_ready + 4; i += blockDim.x) a.sched[i] = 0;
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

bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
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

int weight_tiles(int N, int pair) { return pair == 2 ? N / kTileRows : (N + kTileRows - 1) / kTileRows; }

size_t packed_weight_bytes(int E, int N, int Kd, int pair) {
  return static_cast<size_t>(E) * weight_tiles(N, pair) * (Kd / 128) * (2 * (8192 + 512));
}

// Fills one phase's arguments and tensor maps.  L1 reads x_perm [U, H] against W13 (2I rows,
// gate/up paired tiles), L2 reads h [U, I] against W2 (H rows).
template <int BN>
static bool make_phase(const GemmLaunch& L, bool l1, GemmPhase& P, CUtensorMap& mw, CUtensorMap& mx) {
  const int pair = l1 ? 2 : 1;
  P.w = L.w;
  P.x_sf = L.x_sf;
  P.w_bytes = packed_weight_bytes(L.E, L.w_rows, L.Kd, pair);
  P.x_sf_bytes = act_sf_bytes(L.U, L.Kd / 128, BN);
  P.n_slabs = L.Kd / 128;
  P.n_wt = weight_tiles(L.w_rows, pair);
  P.out_cols = l1 ? L.I : L.w_rows;
  P.n_tiles = (L.U + BN - 1) / BN * P.n_wt;
  P.gather_ids = nullptr;
  P.gather_k = 1;
  P.gather_rows = 0;
  P.gather_u = 0;
  // the packed stream viewed as rows of 128 FP4 codes (64 bytes); a box is 256 rows
  if (!make_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, L.w, 128, P.w_bytes / 64, 64, 128, kTileRows))
    return false;
  if (l1 && L.gather_ids) {
    // token-order rows [T, Kd], one-row box for the four-row gathers
    if (L.gather_rows <= 0 || L.gather_k <= 0) return false;
    P.gather_ids = L.gather_ids;
    P.gather_k = L.gather_k;
    P.gather_rows = L.gather_rows;
    P.gather_u = L.U;
    return make_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.x, L.Kd, L.gather_rows, L.Kd, 128, 1);
  }
  return make_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.x, L.Kd, L.U, L.Kd, 128, BN);
}

// l1 and/or l2 (non-null ones run).  `sched` holds gemm_sched_words(U, align) words that are zero
// before the launch and zero again after it (work counter; with both phases also the per-row-block
// counters that order them).
template <int BN, bool GATHER, bool PRELUDE = false>
static cudaError_t launch_gemm_t(const GemmLaunch* l1, const GemmLaunch* l2, uint32_t* sched, cudaStream_t stream,
                                 const PreludeArgs* pre = nullptr) {
  using C = GemmCfg<BN>;
  GemmArgs a{};
  CUtensorMap m[4] = {};
  if (!sched || (!l1 && !l2)) return cudaErrorInvalidValue;
  const GemmLaunch& any = l1 ? *l1 : *l2;
  if (l1 && !make_phase<BN>(*l1, true, a.ph[0], m[0], m[1])) return cudaErrorInvalidValue;
  if (l2 && !make_phase<BN>(*l2, false, a.ph[1], m[2], m[3])) return cudaErrorInvalidValue;
  if (!l1) {
    a.ph[0] = a.ph[1];
    a.ph[0].n_tiles = 0;
    m[0] = m[2];
    m[1] = m[3];
  }
  if (!l2) {
    a.ph[1] = a.ph[0];
    a.ph[1].n_tiles = 0;
    m[2] = m[0];
    m[3] = m[1];
  }
  a.expert_ids = any.expert_ids;
  a.m_sum = any.m_sum;
  a.h_q = l1 ? l1->h_q : nullptr;
  a.h_sf = l1 ? l1->h_sf : nullptr;
  a.y = l2 ? l2->y : nullptr;
  a.status = any.status;
  a.sf_nb = act_sf_blocks(any.U, BN);
  a.sched = sched;
  a.n_ready = (any.U + BN - 1) / BN;
  a.fused = (l1 && l2) ? 1 : 0;
  a.one_expert_blocks = any.align % BN == 0;
  if (l2) a.red = l2->red;
  if (l1) {
    a.row_ids = l1->row_ids;
    a.row_w = l1->row_w;
  }
  a.E = any.E;
  if (any.counts) {
    // masked mode needs one expert per row block and whole blocks per slot
    if (any.slot % BN != 0 || any.align % BN != 0 || any.E > kMaxMaskedExperts) return cudaErrorInvalidValue;
    a.counts = any.counts;
    a.slot_blocks = any.slot / BN;
  }
  const int total = a.ph[0].n_tiles + a.ph[1].n_tiles;
  int grid = num_sms();
  if (grid > total) grid = total;
  if (grid < 1) grid = 1;
  PreludeParam<PRELUDE> pp{};
  if constexpr (PRELUDE) {
    if (!pre) return cudaErrorInvalidValue;
    pp = *pre;
    grid = num_sms();   // one CTA per SM, all resident (cooperative launch): the routing blocks need them all
  }
  cudaError_t err = cudaFuncSetAttribute(moe_gemm_kernel<BN, GATHER, PRELUDE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  // Programmatic stream serialization lets the CTAs start their prologue (barriers, TMEM, tensor
  // maps) while the permute finishes; they wait for it before reading its results.  Should the
  // runtime refuse it, the launch is repeated without it.
  // The single-launch forward is cooperative instead (its grid barriers need every CTA resident)
  // and starts only after the previous launch, whose outputs its routing phase overwrites.
  static bool pdl_ok = true;
  cudaLaunchAttribute attr[1];
  int n = 0;
  if (PRELUDE) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
    ++n;
  } else if (pdl_ok) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  err = cudaLaunchKernelEx(&cfg, moe_gemm_kernel<BN, GATHER, PRELUDE>, m[0], m[1], m[2], m[3], a, pp);
  if (err != cudaSuccess && !PRELUDE && pdl_ok) {
    (void)cudaGetLastError();
    cfg.numAttrs = n - 1;
    err = cudaLaunchKernelEx(&cfg, moe_gemm_kernel<BN, GATHER, PRELUDE>, m[0], m[1], m[2], m[3], a, pp);
    if (err == cudaSuccess) pdl_ok = false;   // only the attribute was refused
  }
  if (err != cudaSuccess) (void)cudaGetLastError();   // a refused launch leaves no error for later calls
  return err;
}

int gemm_block_n(int align) { return act_sf_block_rows(align); }

template <bool GATHER>
static cudaError_t launch_bn_t(const GemmLaunch* l1, const GemmLaunch* l2, uint32_t* sched, cudaStream_t stream) {
  switch (gemm_block_n((l1 ? l1 : l2)->align)) {
    case 16: return launch_gemm_t<16, GATHER>(l1, l2, sched, stream);
    case 32: return launch_gemm_t<32, GATHER>(l1, l2, sched, stream);
    case 64: return launch_gemm_t<64, GATHER>(l1, l2, sched, stream);
    default: return launch_gemm_t<128, GATHER>(l1, l2, sched, stream);
  }
}

static cudaError_t launch_bn(const GemmLaunch* l1, const GemmLaunch* l2, uint32_t* sched, cudaStream_t stream) {
  if (l1 && l1->gather_ids) return launch_bn_t<true>(l1, l2, sched, stream);
  return launch_bn_t<false>(l1, l2, sched, stream);
}

cudaError_t launch_gemm(const GemmLaunch& L, bool l1, uint32_t* sched, cudaStream_t stream) {
  return l1 ? launch_bn(&L, nullptr, sched, stream) : launch_bn(nullptr, &L, sched, stream);
}

cudaError_t launch_ffn(const GemmLaunch& l1, const GemmLaunch& l2, uint32_t* sched, cudaStream_t stream) {
  return launch_bn(&l1, &l2, sched, stream);
}

cudaError_t launch_ffn_prelude(const GemmLaunch& l1, const GemmLaunch& l2, const PreludeLaunch& p, uint32_t* sched,
                               cudaStream_t stream) {
  if (!prelude_supported(p.T, p.E, p.K, p.align) || gemm_block_n(l1.align) != 16 || l1.gather_ids || l1.counts)
    return cudaErrorInvalidValue;
  PreludeArgs q{};
  q.r.partial = p.partial;
  q.r.nsplit = kGemvSplit;
  q.r.gate_bias = p.gate_bias;
  q.r.e_bias = p.e_bias;
  q.r.T = p.T;
  q.r.H = p.H;
  q.r.E = p.E;
  q.r.K = p.K;
  q.r.score_fn = p.score_fn;
  q.r.renormalize = p.renormalize;
  q.r.logits_out = p.logits_out;
  q.r.topk_ids = p.topk_ids;
  q.r.topk_w = p.topk_w;
  q.r.hidden = p.hidden;
  q.r.x_q = p.x_q;
  q.r.x_sf = p.x_sf;
  q.r.topk_blocks = p.T;
  q.r.nv = NaiveLayout{};
  q.r.gate_failed = nullptr;
  q.w_gate = p.w_gate;
  q.partial = p.partial;
  q.p = PermuteArgs{p.topk_ids, p.T, p.K, p.E, p.align, p.U, p.sorted_ids, p.expert_ids, p.inv_perm, p.m_sum,
                    p.counts, p.status, 0};
  q.x_q = p.x_q;
  q.x_sf = p.x_sf;
  q.x_perm = p.x_perm;
  q.x_perm_sf = p.x_perm_sf;
  q.H = p.H;
  q.bt = act_sf_block_rows(p.align);
  q.nb = act_sf_blocks(p.U, q.bt);
  return launch_gemm_t<16, false, true>(&l1, &l2, sched, stream, &q);
}

bool prelude_supported(int T, int E, int K, int align) {
  // the routing's 16-token and 256-expert register tiles, one thread per (token, slot) pair in a
  // 256-thread permute that also copies the rows (up to 128 pairs), 16-row GEMM blocks
  return T >= 1 && T <= kGemvT && E >= 1 && E <= 256 && T * K <= 128 && gemm_block_n(align) == 16;
}

size_t gemm_sched_words(int U, int align) {
  const int bn = gemm_block_n(align);
  return static_cast<size_t>((U + bn - 1) / bn) + 4;   // row-block counters, work, exit, two grid barriers
}

// ------------------------------------------------------------------------------------------
// Weight packing (once per weight tensor): logical codes [E, N, Kd/2] and UE8M0 scales
// [E, N, Kd/32] -> a stream of chunks, one per (expert, 256-row tile, 128-deep slab), in the order
// the GEMM reads them.  A tile is two halves of 128 rows: pair = 2 (W13) joins the gate rows
// 128t.. with the up rows N/2 + 128t..; pair = 1 (W2) takes rows 256t .. 256t+255 (rows past N
// are zero codes with scale 1).  Chunk = 2 x [128 rows x 64 B codes], then 2 x 512-byte scale
// images whose byte l*16 + w*4 + b holds the scale of half-row (32w + l), k-block (4*slab + b):
// the layout tcgen05.cp .32x128b.warpx4 turns into "row n at TMEM column n/32, byte = k-step".
__global__ void pack_mx_weights_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf, int E, int N,
                                       int Kd, int pair, uint8_t* __restrict__ out) {
  const size_t chunk_bytes = 2 * (8192 + 512);
  const int n_slabs = Kd / 128, n_wt = pair == 2 ? N / kTileRows : (N + kTileRows - 1) / kTileRows;
  const size_t total = static_cast<size_t>(E) * n_wt * n_slabs * chunk_bytes;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const size_t c = i / chunk_bytes;
    const int o = static_cast<int>(i % chunk_bytes);
    const int s = static_cast<int>(c % n_slabs);
    const size_t ew = c / n_slabs;
    const int wt = static_cast<int>(ew % n_wt), e = static_cast<int>(ew / n_wt);
    if (o < 2 * 8192) {
      const int h = o / 8192, m = (o % 8192) / 64, j = o % 64;
      const int r = pair == 2 ? h * (N / 2) + wt * 128 + m : wt * 256 + h * 128 + m;
      out[i] = r < N ? q[(static_cast<size_t>(e) * N + r) * (Kd / 2) + s * 64 + j] : 0;
    } else {
      const int o2 = o - 2 * 8192;
      const int h = o2 / 512, within = o2 % 512;
      const int l = within / 16, w = (within / 4) & 3, b = within & 3;
      const int mm = 32 * w + l;
      const int r = pair == 2 ? h * (N / 2) + wt * 128 + mm : wt * 256 + h * 128 + mm;
      out[i] = r < N ? sf[(static_cast<size_t>(e) * N + r) * (Kd / 32) + s * 4 + b] : 127;
    }
  }
}

cudaError_t launch_pack_mx(const uint8_t* q, const uint8_t* sf, int E, int N, int Kd, int pair, uint8_t* out,
                           cudaStream_t stream) {
  pack_mx_weights_kernel<<<4 * num_sms(), 256, 0, stream>>>(q, sf, E, N, Kd, pair, out);
  return cudaGetLastError();
}

}  // namespace moe
