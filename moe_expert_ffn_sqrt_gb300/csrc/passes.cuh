// Row-block passes shared by the bf16-MMA grouped GEMMs (NVFP4 and INT8 weights): which expert a
// CTA's work item runs against which rows.  Used inside the kernels' anonymous namespaces.
#pragma once

#include <cstdint>

namespace moe {

// One pass of the pipeline: expert e against rows [rb*BN, (rb+nb)*BN), nb = 1 or 2 row blocks
// (two blocks share each converted weight tile, halving the conversion work per MMA).
struct RowPass {
  int e, rb, nb;
};

// Walks this CTA's items and their passes.  With one expert per row block (alignment a multiple of
// BN) the blocks go in pairs 2k, 2k+1.  With split_pairs (small blocks), item t = (2k + h) * n_wt + wt
// is half h of pair k against weight tile wt: if both blocks hold the same expert, half 0 is one pass
// over both (sharing each converted weight tile) and half 1 is empty; otherwise half h is a pass over
// block 2k + h when that block holds rows.  Items of one pass each spread the passes evenly over the
// CTAs when consecutive blocks belong to different experts (small batches, where most pairs hold two
// experts).  Without split_pairs (large blocks, where most pairs hold one expert and a split would
// leave every other item empty and the passes unevenly spread over the CTAs), item t = k * n_wt + wt
// is the whole pair: one pass over both blocks, or a pass per block.  Without one expert per block,
// item t is block t / n_wt and each expert present in it is a pass (smallest expert id first).
// With pair_blocks == 0 a pair's two blocks of one expert are two passes (one block each).
// Called by whole warps; every role walks the same sequence.  Args needs n_tiles, n_wt,
// one_expert_blocks, split_pairs, pair_blocks and expert_ids; the item index modulo n_wt is the
// weight tile.
template <int BN, class Args>
__device__ __forceinline__ bool next_row_pass(const Args& a, int msum, int& t, int& p, int& e_prev, RowPass& P) {
  const int lane = threadIdx.x & 31;
  while (t < a.n_tiles) {
    const int k = t / a.n_wt;
    if (a.one_expert_blocks) {
      const int pair = a.split_pairs ? k >> 1 : k;
      const int rb0 = 2 * pair, rb1 = 2 * pair + 1;
      if (rb0 * BN >= msum) return false;
      const int e0 = __ldg(a.expert_ids + rb0 * BN);
      const int e1 = rb1 * BN < msum ? __ldg(a.expert_ids + rb1 * BN) : -1;
      const bool joint = a.pair_blocks && e1 == e0;   // one pass over both blocks
      if (a.split_pairs) {
        const int h = k & 1;
        if (p == 0) {
          p = 1;
          if (h == 0 && e0 >= 0) {
            P = RowPass{e0, rb0, joint ? 2 : 1};
            return true;
          }
          if (h == 1 && e1 >= 0 && !joint) {
            P = RowPass{e1, rb1, 1};
            return true;
          }
        }
      } else {
        if (p == 0) {
          p = 1;
          if (e0 >= 0) {
            P = RowPass{e0, rb0, joint ? 2 : 1};
            return true;
          }
        }
        if (p == 1) {
          p = 2;
          if (e1 >= 0 && !joint) {
            P = RowPass{e1, rb1, 1};
            return true;
          }
        }
      }
    } else {
      const int r0 = k * BN;
      if (r0 >= msum) return false;
      const int rend = min(r0 + BN, msum);
      int best = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < (BN + 31) / 32; ++j) {
        const int r = r0 + j * 32 + lane;
        if (r < rend) {
          const int x = __ldg(a.expert_ids + r);
          if (x > e_prev && x < best) best = x;
        }
      }
      best = __reduce_min_sync(0xffffffffu, best);
      if (best != 0x7fffffff) {
        e_prev = best;
        P = RowPass{best, k, 1};
        return true;
      }
    }
    t += gridDim.x;
    p = 0;
    e_prev = -1;
  }
  return false;
}

}  // namespace moe
