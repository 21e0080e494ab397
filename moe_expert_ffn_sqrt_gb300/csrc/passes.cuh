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
// BN) item t covers blocks 2k and 2k+1 (k = t / n_wt): one pass if both hold the same expert, else
// a pass per block that holds rows.  Otherwise item t is one block and each expert present in it
// is a pass (smallest expert id first).  Called by whole warps; every role walks the same sequence.
// Args needs n_tiles, n_wt, one_expert_blocks and expert_ids.
template <int BN, class Args>
__device__ __forceinline__ bool next_row_pass(const Args& a, int msum, int& t, int& p, int& e_prev, RowPass& P) {
  const int lane = threadIdx.x & 31;
  while (t < a.n_tiles) {
    const int k = t / a.n_wt;
    if (a.one_expert_blocks) {
      const int rb0 = 2 * k, rb1 = 2 * k + 1;
      if (rb0 * BN >= msum) return false;
      const int e0 = __ldg(a.expert_ids + rb0 * BN);
      const int e1 = rb1 * BN < msum ? __ldg(a.expert_ids + rb1 * BN) : -1;
      if (e0 >= 0 && e1 == e0) {
        if (p == 0) {
          P = RowPass{e0, rb0, 2};
          p = 2;
          return true;
        }
      } else {
        if (p == 0) {
          p = 1;
          if (e0 >= 0) {
            P = RowPass{e0, rb0, 1};
            return true;
          }
        }
        if (p == 1) {
          p = 2;
          if (e1 >= 0) {
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
