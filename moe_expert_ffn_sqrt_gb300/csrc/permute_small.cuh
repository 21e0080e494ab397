// The small permute (T * K <= 1024 pairs) as a device function for the single-launch forward
// (gemm.cu): the steps of permute_small_kernel (permute.cu) in the same order with the same
// arithmetic, so the results are the same bits (the single-launch tests assert it).  The launch
// keeps its own copy: passing its shared-memory arrays through this function cost it ~0.5 us.
// Note "INT8 高吞吐/低延迟 EP 代码梳理" §9.3-9.4 (scatter, inv_perm, M_sum), §10 (M_sum_upper) and the
// m_indices paragraph (expert_ids, -1 on padding); MegaMoE page 路径 A (moe_align_block_size).
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace moe {

// The alignment is a power of two (checked by the host), so rounding up is a mask, not a division.
__device__ __forceinline__ int round_up_pow2(int n, int align) { return (n + align - 1) & ~(align - 1); }

struct PermuteArgs {
  const int32_t* topk_ids;
  int T, K, E, align, U;
  int32_t* sorted_ids;
  int32_t* expert_ids;
  int32_t* inv_perm;
  int32_t* m_sum;
  int32_t* counts;       // optional
  uint32_t* status;
  int slot;              // 0: contiguous segments padded to align; > 0: BatchedExperts, expert e's rows
                         // start at e * slot and its segment is slot rows.  A pair that would land past
                         // its expert's slot is dropped (inv_perm -1) and recorded as an index error.
};

// Small problems (T*K <= 1024): one thread per (t,k) pair.  A pair's rank within its expert is
// the number of earlier pairs (smaller flat index) with the same expert, counted in shared
// memory; one warp scans the expert counts.  CTA 0 writes the permutation.  When there are few
// pairs the same launch also copies the activation rows: every CTA recomputes the (cheap)
// permutation and each warp copies a 1 KB piece of one pair's row (two 16-byte loads per lane,
// issued before the stores), so the copy is spread over N * H / 1024 warps.
constexpr int kSmallPairs = 1024;
constexpr int kSmallCopyPairs = 128;
constexpr int kCopyPiece = 64;       // 16-byte chunks of a row one warp copies (1 KB)

// The small permute over NT threads of block `cta` of `ncta` (each block recomputes the indices;
// block 0 writes them, and the padding, tail and row copies are split over the blocks).  ids:
// the [T, K] expert ids (global or shared memory); cnt, seg: [E] each; s_ids, s_rank: [NT];
// T * K <= NT.  sync() is a barrier over exactly the NT threads.  COHERENT: x_q is written by the
// same launch (the single-launch forward), so its rows are read past the non-coherent cache.
template <int NT, bool COHERENT, class Sync>
__device__ __forceinline__ void permute_small_body(const PermuteArgs& a, const int32_t* ids, const uint8_t* x_q,
                                                   const uint8_t* x_sf, int H, uint8_t* x_perm, uint8_t* x_perm_sf,
                                                   int bt, int nb, int32_t* cnt, int32_t* seg, int32_t* s_ids,
                                                   int32_t* s_rank, int32_t* s_total, int tid, int cta, int ncta,
                                                   Sync sync) {
  const int warp = tid / 32, lane = tid % 32;
  const int N = a.T * a.K;
  for (int e = tid; e < a.E; e += NT) cnt[e] = 0;
  int e_mine = -1;
  if (tid < N) {
    e_mine = ids[tid];
    if (e_mine < 0 || e_mine >= a.E) {
      if (cta == 0) record_error(a.status, kDevErrIndex);
      e_mine = -1;
    }
    s_ids[tid] = e_mine;
  }
  sync();
  int rank = 0;
  if (e_mine >= 0) {
    atomicAdd(&cnt[e_mine], 1);
    for (int j = 0; j < tid; ++j) rank += (s_ids[j] == e_mine);
  }
  if (tid < N) s_rank[tid] = rank;
  sync();
  if (a.slot > 0) {                  // BatchedExperts: fixed slots
    for (int e = tid; e < a.E; e += NT) seg[e] = e * a.slot;
    if (tid == 0) *s_total = a.E * a.slot;
  } else if (warp == 0) {            // exclusive scan of the aligned segment sizes
    const int per = (a.E + 31) / 32;
    int local = 0;
    for (int j = 0; j < per; ++j) {
      const int e = lane * per + j;
      if (e < a.E) local += round_up_pow2(cnt[e], a.align);
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int run = incl - local;
    for (int j = 0; j < per; ++j) {
      const int e = lane * per + j;
      if (e < a.E) {
        seg[e] = run;
        run += round_up_pow2(cnt[e], a.align);
      }
    }
    if (lane == 31) *s_total = incl;
  }
  sync();
  const int msum = *s_total;
  if (cta == 0) {
    if (e_mine >= 0) {
      if (a.slot > 0 && rank >= a.slot) {
        record_error(a.status, kDevErrIndex);
        a.inv_perm[tid] = -1;
      } else {
        const int pos = seg[e_mine] + rank;
        a.inv_perm[tid] = pos;
        a.sorted_ids[pos] = tid;
        a.expert_ids[pos] = e_mine;
      }
    }
    if (a.counts)
      for (int e = tid; e < a.E; e += NT) a.counts[e] = cnt[e];
    if (tid == 0) *a.m_sum = msum;
  }
  // padding rows of each segment and the tail [M_sum, U), split over every CTA of the launch (each
  // holds the same counts and segment starts)
  for (int e = cta * (NT / 32) + warp; e < a.E; e += ncta * (NT / 32)) {
    const int c = cnt[e];
    const int padded = a.slot > 0 ? a.slot : round_up_pow2(c, a.align);
    for (int r = c + lane; r < padded; r += 32) {
      a.sorted_ids[seg[e] + r] = N;
      a.expert_ids[seg[e] + r] = -1;
    }
  }
  for (int r = msum + cta * NT + tid; r < a.U; r += ncta * NT) {
    a.sorted_ids[r] = N;
    a.expert_ids[r] = -1;
  }
  if ((x_perm != nullptr || x_perm_sf != nullptr) && N <= kSmallCopyPairs) {
    // one warp per (pair, 1 KB piece of its row); the piece-0 warp also copies the row's scales
    // (x_perm null: the scales alone, one warp per pair)
    const int chunks = x_perm != nullptr ? H / 16 : 0, slabs = H / 128;
    const int pieces = x_perm != nullptr ? (chunks + kCopyPiece - 1) / kCopyPiece : 1;
    for (int u = cta * (NT / 32) + warp; u < N * pieces; u += ncta * (NT / 32)) {
      const int p = u / pieces, piece = u - p * pieces;
      const int e = s_ids[p];
      if (e < 0 || (a.slot > 0 && s_rank[p] >= a.slot)) continue;
      const int dst = seg[e] + s_rank[p];
      const int t = p / a.K;
      const uint4* src = reinterpret_cast<const uint4*>(x_q + static_cast<size_t>(t) * H);
      uint4* out = reinterpret_cast<uint4*>(x_perm + static_cast<size_t>(dst) * H);
      uint4 v[kCopyPiece / 32];
#pragma unroll
      for (int i = 0; i < kCopyPiece / 32; ++i) {
        const int j = piece * kCopyPiece + i * 32 + lane;
        if (j < chunks) v[i] = COHERENT ? __ldcg(src + j) : __ldg(src + j);
      }
#pragma unroll
      for (int i = 0; i < kCopyPiece / 32; ++i) {
        const int j = piece * kCopyPiece + i * 32 + lane;
        if (j < chunks) out[j] = v[i];
      }
      if (piece == 0)
        for (int s2 = lane; s2 < slabs; s2 += 32)
          x_perm_sf[act_sf_offset(bt, nb, dst, s2)] = x_sf[static_cast<size_t>(t) * slabs + s2];
    }
  }
}

}  // namespace moe
