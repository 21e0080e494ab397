// Small-batch routing (T <= kGemvT) as device functions for the single-launch forward (gemm.cu):
// the steps of route_small_kernel (route.cu) in the same order with the same arithmetic, so the
// results are the same bits (the single-launch tests assert it).  The launch keeps its own copy:
// calling these functions cost it ~0.5 us.
// Page "DeepSeek V4 MegaMoE Kernel 深度解析", 经典 MoE 的计算过程 / 第一步：路由, and the CUDA tag page
// teaser row "Fused TopK Bias Routing" (sqrt(softplus), e_score_correction_bias).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// ------------------------------------------------------------------------------------------
// Small batches (T <= kGemvT): blocks of 4 experts x one quarter of H (route_small_kernel).
constexpr int kGemvT = 16;
constexpr int kGemvE = 4;
constexpr int kGemvSplit = 4;

// ------------------------------------------------------------------------------------------
// Arguments of the routing's scoring, top-K and FP8 activation quantisation (route_finish_kernel
// above kGemvT tokens, the small-batch functions below up to it).
struct RouteFinishArgs {
  const float* partial;
  int nsplit;
  const float* gate_bias;
  const float* e_bias;
  int T, H, E, K;
  int score_fn;      // 0 softmax, 1 sqrt(softplus)
  int renormalize;
  float* logits_out;
  int32_t* topk_ids;
  float* topk_w;
  const uint16_t* hidden;
  uint8_t* x_q;
  uint8_t* x_sf;
  int topk_blocks;   // blocks [0, topk_blocks) do top-K
  NaiveLayout nv;    // small batches: the tiny-batch layout written by the same launch (nv.eids null: off)
  // Optional: a word that is zero unless this call's gate GEMM gave up on a wait (and so left its
  // partial sums unwritten); when set, the top-K writes id -1 and NaN weights and logits instead.
  const uint32_t* gate_failed;
};

// Warp arg-max of (key, id), ties to the lower id, with the warp reduction instructions: the keys
// as order-preserving unsigned integers (-0 folded into +0, so that equal floats stay equal), the
// maximum, then the smallest id among the lanes that hold it.  Keys are finite or -inf.
__device__ __forceinline__ int warp_argmax_id(float key, int id) {
  const uint32_t u = __float_as_uint(key + 0.0f);
  const uint32_t ok = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  const uint32_t best = __reduce_max_sync(0xffffffffu, ok);
  return static_cast<int>(__reduce_min_sync(0xffffffffu, ok == best ? static_cast<uint32_t>(id) : 0xffffffffu));
}

// Parts 1-3 of the small-batch routing for block (bx, by) of a gx x kGemvSplit grid of 256-thread
// blocks: gate partial sums of experts 4bx .. 4bx+3 over H quarter by, this block's share of the
// FP8 activation groups and of the tiny-batch layout.  Run by 256 threads (tid); sync() is a
// barrier over exactly those threads.
template <int TT, class Sync>
__device__ __forceinline__ void route_small_gemv(const RouteFinishArgs& a, const float* __restrict__ wg,
                                                 float* __restrict__ partial, int bx, int by, int gx, int tid,
                                                 float (*red)[kGemvE * TT], Sync sync) {
  const int warp = tid / 32, lane = tid % 32;
  const int nblocks = gx * kGemvSplit;
  const int bid = by * gx + bx;
  const int T = a.T, H = a.H, E = a.E;
  // the biases are read only by the last CTA, after every other CTA's work: start them towards L2
  if (bid == 0 && warp == 0)
    for (int off = lane * 32; off < E; off += 32 * 32) {     // one 128-byte line per lane and round
      if (a.gate_bias) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.gate_bias + off));
      if (a.e_bias) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.e_bias + off));
    }
  // 1. gate GEMV partial: experts e0..e0+3 over one quarter of H
  const int e0 = bx * kGemvE, split = by;
  const int hq = H / kGemvSplit, hbeg = split * hq;   // hq is a multiple of 32 (H multiple of 128)
  float acc[kGemvE][TT];
#pragma unroll
  for (int i = 0; i < kGemvE; ++i)
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[i][t] = 0.f;
  for (int h = hbeg + tid * 8; h < hbeg + hq; h += 256 * 8) {
    float w[kGemvE][8];
#pragma unroll
    for (int i = 0; i < kGemvE; ++i) {
      const int e = e0 + i;
      if (e < E) {
        const float4 p = __ldg(reinterpret_cast<const float4*>(wg + static_cast<size_t>(e) * H + h));
        const float4 q = __ldg(reinterpret_cast<const float4*>(wg + static_cast<size_t>(e) * H + h + 4));
        w[i][0] = p.x; w[i][1] = p.y; w[i][2] = p.z; w[i][3] = p.w;
        w[i][4] = q.x; w[i][5] = q.y; w[i][6] = q.z; w[i][7] = q.w;
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) w[i][j] = 0.f;
      }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      if (t < T) {
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(a.hidden + static_cast<size_t>(t) * H + h));
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
        float xv[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          xv[2 * j] = __uint_as_float(xw[j] << 16);
          xv[2 * j + 1] = __uint_as_float(xw[j] & 0xFFFF0000u);
        }
#pragma unroll
        for (int i = 0; i < kGemvE; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][t] = fmaf(xv[j], w[i][j], acc[i][t]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kGemvE; ++i)
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      float v = acc[i][t];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) red[warp][i * TT + t] = v;
    }
  sync();
  for (int j = tid; j < kGemvE * TT; j += 256) {
    const int i = j / TT, t = j % TT, e = e0 + i;
    if (t < T && e < E) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) v += red[w][j];
      partial[(static_cast<size_t>(split) * T + t) * E + e] = v;
    }
  }
  // 2. FP8 activation quantisation of this CTA's share of the 128-column groups
  if (a.x_q || a.nv.xp) {
    const int gpt = H / 128;
    for (long long gidx = static_cast<long long>(bid) * 8 + warp; gidx < static_cast<long long>(T) * gpt;
         gidx += static_cast<long long>(nblocks) * 8) {
      const int t = static_cast<int>(gidx / gpt), g = static_cast<int>(gidx % gpt);
      const size_t base = static_cast<size_t>(t) * H + g * 128 + lane * 4;
      const uint2 raw = *reinterpret_cast<const uint2*>(a.hidden + base);
      float v[4];
      v[0] = __uint_as_float(raw.x << 16);
      v[1] = __uint_as_float(raw.x & 0xFFFF0000u);
      v[2] = __uint_as_float(raw.y << 16);
      v[3] = __uint_as_float(raw.y & 0xFFFF0000u);
      float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const int ex = ue8m0_exponent(amax);
      const float sc = pow2_neg(ex);
      const __nv_fp8x2_storage_t lo =
          __nv_cvt_float2_to_fp8x2(make_float2(v[0] * sc, v[1] * sc), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t hi =
          __nv_cvt_float2_to_fp8x2(make_float2(v[2] * sc, v[3] * sc), __NV_SATFINITE, __NV_E4M3);
      const uint32_t packed = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      if (a.x_q) {
        *reinterpret_cast<uint32_t*>(a.x_q + base) = packed;
        if (lane == 0) a.x_sf[static_cast<size_t>(t) * gpt + g] = static_cast<uint8_t>(ex + 127);
      }
      if (a.nv.xp) {                               // the token's row of each of its K pairs
        for (int k = 0; k < a.K; ++k) {
          const int r = (t * a.K + k) * kNaiveRows;
          *reinterpret_cast<uint32_t*>(a.nv.xp + static_cast<size_t>(r) * H + g * 128 + lane * 4) = packed;
          if (lane == 0) a.nv.xp_sf[act_sf_offset(kNaiveRows, a.nv.sf_nb, r, g)] = static_cast<uint8_t>(ex + 127);
        }
      }
    }
  }
  // 3. tiny-batch layout: every entry that does not depend on the routing (pair p owns row
  //    kNaiveRows * p; the other rows of its block and the rows up to U are padding)
  if (a.nv.eids) {
    const int npairs = T * a.K;
    for (int r = bid * 256 + tid; r < a.nv.U; r += nblocks * 256) {
      const bool real = r % kNaiveRows == 0 && r / kNaiveRows < npairs;
      a.nv.sorted[r] = real ? r / kNaiveRows : npairs;
      if (!real) a.nv.eids[r] = -1;                // real rows: the top-K below
      if (r < npairs) a.nv.inv[r] = r * kNaiveRows;
    }
    if (bid == 0 && tid == 0) *a.nv.m_sum = npairs * kNaiveRows;
  }
}

// Part 4: the top-K of every token from the kGemvSplit partial sums (summed in split order), one
// warp per token (warps warp, warp + 8, ...).  IDS: the ids also go to ids_out as [T, K] (shared
// memory); OUTPUTS: the ids, weights, logits and tiny-batch ids are stored.  Compile-time flags,
// so that the routing launch's serial tail carries no extra branches.
template <int TT, int PER, bool IDS, bool OUTPUTS>
__device__ __forceinline__ void route_small_topk(const RouteFinishArgs& a, const float* __restrict__ partial, int warp,
                                                 int lane, int32_t* ids_out) {
  const int T = a.T, E = a.E;
  // the biases first, in registers: their loads then overlap the partial-sum loads instead of
  // waiting behind the optional logits stores
  float gbias[PER], ebias[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = lane + 32 * j;
    gbias[j] = (a.gate_bias && e < E) ? __ldg(a.gate_bias + e) : 0.f;
    ebias[j] = (a.e_bias && e < E) ? __ldg(a.e_bias + e) : 0.f;
  }
  for (int t = warp; t < T; t += 8) {
    float s[PER], key[PER];
    float lmax = -INFINITY;
    // partial sums of 8 experts per lane at a time: every load of a group is issued before the
    // optional logits stores (which the compiler may not move loads across)
#pragma unroll
    for (int j0 = 0; j0 < PER; j0 += 8) {
      constexpr int G = PER < 8 ? PER : 8;
      float v[G][kGemvSplit];
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        const int e = lane + 32 * (j0 + jj);
#pragma unroll
        for (int sp = 0; sp < kGemvSplit; ++sp)
          v[jj][sp] = e < E ? __ldcg(partial + (static_cast<size_t>(sp) * T + t) * E + e) : 0.f;
      }
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        const int j = j0 + jj, e = lane + 32 * j;
        float l = -INFINITY;
        if (e < E) {
          l = (v[jj][0] + v[jj][1]) + (v[jj][2] + v[jj][3]);   // the order route_finish_kernel sums 4 splits in
          if (a.gate_bias) l += gbias[j];
          if (OUTPUTS && a.logits_out) a.logits_out[static_cast<size_t>(t) * E + e] = l;
        }
        s[j] = l;
        lmax = fmaxf(lmax, l);
      }
    }
    if (a.score_fn == 0) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, off));
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        s[j] = (lane + 32 * j < E) ? expf(s[j] - lmax) : 0.f;
        sum += s[j];
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
#pragma unroll
      for (int j = 0; j < PER; ++j) s[j] = s[j] / sum;
    } else {
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const float l = s[j];
        s[j] = (lane + 32 * j < E) ? sqrtf(fmaxf(l, 0.f) + log1pf(expf(-fabsf(l)))) : 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int e = lane + 32 * j;
      key[j] = (e < E) ? s[j] + (a.e_bias ? ebias[j] : 0.f) : -INFINITY;
    }
    float wsum = 0.f, wmine = 0.f;
    for (int k = 0; k < a.K; ++k) {
      float bk = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int e = lane + 32 * j;
        if (key[j] > bk || (key[j] == bk && e < bi)) {
          bk = key[j];
          bi = e;
        }
      }
      bi = warp_argmax_id(bk, bi);
      // the winner's lane takes its score and retires its key; selects with compile-time indices
      // keep s[] and key[] in registers
      float sw = 0.f;
      const bool won = (bi & 31) == lane;
      const int jw = bi >> 5;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const bool hit = won && j == jw;
        sw = hit ? s[j] : sw;
        key[j] = hit ? -INFINITY : key[j];
      }
      sw = __shfl_sync(0xffffffffu, sw, bi & 31);
      wsum += sw;
      if (lane == k) wmine = sw;
      if (lane == 0) {
        if (IDS) ids_out[t * a.K + k] = bi;
        if (OUTPUTS) {
          a.topk_ids[static_cast<size_t>(t) * a.K + k] = bi;
          if (a.nv.eids) a.nv.eids[(t * a.K + k) * kNaiveRows] = bi;
        }
      }
    }
    if (OUTPUTS && lane < a.K) a.topk_w[static_cast<size_t>(t) * a.K + lane] = a.renormalize ? wmine / wsum : wmine;
  }
}

}  // namespace moe
