// Routing: gate GEMM (split over H, deterministic; on the tensor cores above 16 tokens, see
// gate.cu), scoring + biased top-K, FP8 activation quantisation.  Page "DeepSeek V4 MegaMoE Kernel 深度解析", 经典 MoE 的计算过程 / 第一步：路由,
// and the CUDA tag page teaser row "Fused TopK Bias Routing" (sqrt(softplus), e_score_correction_bias).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"
#include "route_small.cuh"

namespace moe {

__device__ __forceinline__ float block_reduce(float v, float* sh, bool is_max) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, v, off);
    v = is_max ? fmaxf(v, o) : v + o;
  }
  __syncthreads();
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  float r = sh[0];
  for (int w = 1; w < 8; ++w) r = is_max ? fmaxf(r, sh[w]) : r + sh[w];
  return r;
}

// Top-K above kGemvT tokens: one CTA (256 threads) per token.  Threads sum the split partials of
// one expert each (independent loads, fixed split order), score, and stage scores/keys in shared
// memory; warp 0 then holds PER = E/32 keys per lane in registers and runs K rounds of warp
// arg-max (ties to the lower expert id).  FP8 activation quantisation (one warp per 128-column
// group) runs in the blocks after the top-K blocks of the same launch.
template <int PER>
__global__ void __launch_bounds__(256) route_finish_kernel(const RouteFinishArgs a) {
  __shared__ float s_score[32 * PER];
  __shared__ float s_key[32 * PER];
  __shared__ float s_red[8];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (static_cast<int>(blockIdx.x) < a.topk_blocks) {
    const int t = blockIdx.x;
    if (a.gate_failed != nullptr && *a.gate_failed != 0) {
      // the partial sums of this call were never written: mark the token's routing invalid
      for (int e = threadIdx.x; e < a.E; e += 256)
        if (a.logits_out) a.logits_out[static_cast<size_t>(t) * a.E + e] = __int_as_float(0x7fc00000);
      if (threadIdx.x < a.K) {
        a.topk_ids[static_cast<size_t>(t) * a.K + threadIdx.x] = -1;
        a.topk_w[static_cast<size_t>(t) * a.K + threadIdx.x] = __int_as_float(0x7fc00000);
      }
      return;
    }
    // logits: one expert per thread per pass, splits summed in a fixed order
    float lmax = -INFINITY;
    for (int e = threadIdx.x; e < 32 * PER; e += 256) {
      float l = -INFINITY;
      if (e < a.E) {
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        int sp = 0;
        for (; sp + 4 <= a.nsplit; sp += 4)
#pragma unroll
          for (int u = 0; u < 4; ++u) v[u] += a.partial[(static_cast<size_t>(sp + u) * a.T + t) * a.E + e];
        l = (v[0] + v[1]) + (v[2] + v[3]);
        for (; sp < a.nsplit; ++sp) l += a.partial[(static_cast<size_t>(sp) * a.T + t) * a.E + e];
        if (a.gate_bias) l += a.gate_bias[e];
        if (a.logits_out) a.logits_out[static_cast<size_t>(t) * a.E + e] = l;
      }
      s_score[e] = l;
      lmax = fmaxf(lmax, l);
    }
    if (a.score_fn == 0) {
      lmax = block_reduce(lmax, s_red, true);
      float sum = 0.f;
      for (int e = threadIdx.x; e < 32 * PER; e += 256) {
        const float p = (e < a.E) ? expf(s_score[e] - lmax) : 0.f;
        s_score[e] = p;
        sum += p;
      }
      sum = block_reduce(sum, s_red, false);
      for (int e = threadIdx.x; e < 32 * PER; e += 256) s_score[e] = s_score[e] / sum;
    } else {
      for (int e = threadIdx.x; e < 32 * PER; e += 256) {
        const float l = s_score[e];
        s_score[e] = (e < a.E) ? sqrtf(fmaxf(l, 0.f) + log1pf(expf(-fabsf(l)))) : 0.f;
      }
    }
    for (int e = threadIdx.x; e < 32 * PER; e += 256)
      s_key[e] = (e < a.E) ? s_score[e] + (a.e_bias ? a.e_bias[e] : 0.f) : -INFINITY;
    __syncthreads();
    if (warp != 0) return;
    float key[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) key[j] = s_key[lane + 32 * j];
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
      const bool won = (bi & 31) == lane;   // selects with compile-time indices keep key[] in registers
      const int jw = bi >> 5;
#pragma unroll
      for (int j = 0; j < PER; ++j) key[j] = (won && j == jw) ? -INFINITY : key[j];
      const float sw = s_score[bi];
      wsum += sw;
      if (lane == k) wmine = sw;
      if (lane == 0) a.topk_ids[static_cast<size_t>(t) * a.K + k] = bi;
    }
    if (lane < a.K) a.topk_w[static_cast<size_t>(t) * a.K + lane] = a.renormalize ? wmine / wsum : wmine;
    return;
  }
  // FP8 activation quantisation: group g of token t = 128 columns, 4 per lane.
  const int gpt = a.H / 128;
  const long long gidx = static_cast<long long>(blockIdx.x - a.topk_blocks) * 8 + warp;
  if (gidx >= static_cast<long long>(a.T) * gpt) return;
  const int t = static_cast<int>(gidx / gpt), g = static_cast<int>(gidx % gpt);
  const size_t base = static_cast<size_t>(t) * a.H + g * 128 + lane * 4;
  const uint2 raw = *reinterpret_cast<const uint2*>(a.hidden + base);
  float v[4];
  v[0] = __uint_as_float(raw.x << 16);
  v[1] = __uint_as_float(raw.x & 0xFFFF0000u);
  v[2] = __uint_as_float(raw.y << 16);
  v[3] = __uint_as_float(raw.y & 0xFFFF0000u);
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const int e = ue8m0_exponent(amax);
  const float sc = pow2_neg(e);
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(v[0] * sc, v[1] * sc), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(v[2] * sc, v[3] * sc), __NV_SATFINITE, __NV_E4M3);
  *reinterpret_cast<uint32_t*>(a.x_q + base) = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  if (lane == 0) a.x_sf[static_cast<size_t>(t) * gpt + g] = static_cast<uint8_t>(e + 127);
}

// ------------------------------------------------------------------------------------------
// Small batches (T <= kGemvT), one launch.  Each CTA (4 experts x one quarter of H) writes its
// gate partial sums for all T tokens, then quantises its share of the FP8 activation groups.  The
// last CTA to finish (ticket counter in the scratch buffer) sums the 4 partials per (t, e) in
// split order and runs the top-K of every token, one warp per token, as route_finish_kernel does.
// It resets the counter to zero for the next call.
template <int TT, int PER>
__global__ void __launch_bounds__(256) route_small_kernel(const RouteFinishArgs a, const float* __restrict__ wg,
                                                          float* __restrict__ partial, uint32_t* __restrict__ ticket) {
  __shared__ float red[8][kGemvE * TT];
  __shared__ int s_last;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nblocks = gridDim.x * gridDim.y;
  const int bid = blockIdx.y * gridDim.x + blockIdx.x;
  const int T = a.T, H = a.H, E = a.E;
  grid_launch_dependents();        // the permute may start (it waits for this launch's results)
  // the biases are read only by the last CTA, after every other CTA's work: start them towards L2
  if (bid == 0 && warp == 0)
    for (int off = lane * 32; off < E; off += 32 * 32) {     // one 128-byte line per lane and round
      if (a.gate_bias) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.gate_bias + off));
      if (a.e_bias) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.e_bias + off));
    }
  // 1. gate GEMV partial: experts e0..e0+3 over one quarter of H
  const int e0 = blockIdx.x * kGemvE, split = blockIdx.y;
  const int hq = H / kGemvSplit, hbeg = split * hq;   // hq is a multiple of 32 (H multiple of 128)
  float acc[kGemvE][TT];
#pragma unroll
  for (int i = 0; i < kGemvE; ++i)
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[i][t] = 0.f;
  for (int h = hbeg + threadIdx.x * 8; h < hbeg + hq; h += 256 * 8) {
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
  __syncthreads();
  for (int j = threadIdx.x; j < kGemvE * TT; j += 256) {
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
    for (int r = bid * 256 + threadIdx.x; r < a.nv.U; r += nblocks * 256) {
      const bool real = r % kNaiveRows == 0 && r / kNaiveRows < npairs;
      a.nv.sorted[r] = real ? r / kNaiveRows : npairs;
      if (!real) a.nv.eids[r] = -1;                // real rows: the top-K below
      if (r < npairs) a.nv.inv[r] = r * kNaiveRows;
    }
    if (bid == 0 && threadIdx.x == 0) *a.nv.m_sum = npairs * kNaiveRows;
  }
  // 4. the last CTA to finish does the top-K
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(ticket, 1u) == static_cast<uint32_t>(nblocks - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();
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
          if (a.logits_out) a.logits_out[static_cast<size_t>(t) * E + e] = l;
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
        a.topk_ids[static_cast<size_t>(t) * a.K + k] = bi;
        if (a.nv.eids) a.nv.eids[(t * a.K + k) * kNaiveRows] = bi;
      }
    }
    if (lane < a.K) a.topk_w[static_cast<size_t>(t) * a.K + lane] = a.renormalize ? wmine / wsum : wmine;
  }
  if (threadIdx.x == 0) *ticket = 0;     // ready for the next call (the kernel boundary orders it)
}

int route_nsplit(int T, int H, int E) { return T <= kGemvT ? kGemvSplit : gate_nsplit(T, H, E); }

static size_t partial_bytes(int T, int H, int E) {
  return (static_cast<size_t>(route_nsplit(T > 0 ? T : 1, H, E)) * T * E * sizeof(float) + 255) / 256 * 256;
}

// Routing scratch: [0, 256) the small-batch kernel's ticket counter, at the same place for every T,
// H and E, so that a buffer reused for another problem size still finds it at zero (each launch
// that takes tickets sets it back to zero at its end); then the split partial sums; then, above 16
// tokens, the three bf16 parts of the gate weight.  Partial sums and parts are written by a call
// before the same call reads them.
constexpr size_t kTicketSlot = 256;

float* route_partials(void* scratch) { return reinterpret_cast<float*>(static_cast<char*>(scratch) + kTicketSlot); }

size_t route_scratch_bytes(int T, int H, int E) {
  return kTicketSlot + partial_bytes(T, H, E) + (T > kGemvT ? gate_parts_bytes(T, H, E) : 0);
}

template <int TT>
static void launch_route_small(const RouteFinishArgs& a, const float* w_gate, float* partial, uint32_t* ticket,
                               cudaStream_t stream) {
  dim3 g((a.E + kGemvE - 1) / kGemvE, kGemvSplit);
  const int per = (a.E + 31) / 32;
  if (per <= 1) route_small_kernel<TT, 1><<<g, 256, 0, stream>>>(a, w_gate, partial, ticket);
  else if (per <= 2) route_small_kernel<TT, 2><<<g, 256, 0, stream>>>(a, w_gate, partial, ticket);
  else if (per <= 4) route_small_kernel<TT, 4><<<g, 256, 0, stream>>>(a, w_gate, partial, ticket);
  else if (per <= 8) route_small_kernel<TT, 8><<<g, 256, 0, stream>>>(a, w_gate, partial, ticket);
  else if (per <= 16) route_small_kernel<TT, 16><<<g, 256, 0, stream>>>(a, w_gate, partial, ticket);
  else route_small_kernel<TT, 32><<<g, 256, 0, stream>>>(a, w_gate, partial, ticket);
}

cudaError_t launch_route(const uint16_t* hidden, const float* w_gate, const float* gate_bias, const float* e_bias,
                         int T, int H, int E, int K, int score_fn, int renormalize, float* logits_out,
                         int32_t* topk_ids, float* topk_w, uint8_t* x_q, uint8_t* x_sf, void* scratch,
                         uint32_t* status, cudaStream_t stream, const NaiveLayout* nv, const uint32_t* gate_failed) {
  const int ns = route_nsplit(T, H, E);
  uint32_t* ticket = static_cast<uint32_t*>(scratch);
  float* partial = reinterpret_cast<float*>(static_cast<char*>(scratch) + kTicketSlot);
  RouteFinishArgs a;
  a.partial = partial;
  a.nsplit = ns;
  a.gate_bias = gate_bias;
  a.e_bias = e_bias;
  a.T = T;
  a.H = H;
  a.E = E;
  a.K = K;
  a.score_fn = score_fn;
  a.renormalize = renormalize;
  a.logits_out = logits_out;
  a.topk_ids = topk_ids;
  a.topk_w = topk_w;
  a.hidden = hidden;
  a.x_q = x_q;
  a.x_sf = x_sf;
  a.topk_blocks = T;
  a.nv = NaiveLayout{};
  a.gate_failed = gate_failed;
  if (nv) {
    if (T > kGemvT) return cudaErrorInvalidValue;
    a.nv = *nv;
  }
  if (T <= kGemvT) {
    if (T <= 8) launch_route_small<8>(a, w_gate, partial, ticket, stream);
    else launch_route_small<16>(a, w_gate, partial, ticket, stream);
    return cudaGetLastError();
  }
  {
    uint16_t* parts = reinterpret_cast<uint16_t*>(reinterpret_cast<char*>(partial) + partial_bytes(T, H, E));
    const cudaError_t err = launch_gate_mma(hidden, w_gate, T, H, E, ns, parts, partial, status, stream);
    if (err != cudaSuccess) return err;
  }
  const long long qgroups = (x_q != nullptr) ? static_cast<long long>(T) * (H / 128) : 0;
  const int blocks = T + static_cast<int>((qgroups + 7) / 8);
  const int per = (E + 31) / 32;
  if (per <= 1) route_finish_kernel<1><<<blocks, 256, 0, stream>>>(a);
  else if (per <= 2) route_finish_kernel<2><<<blocks, 256, 0, stream>>>(a);
  else if (per <= 4) route_finish_kernel<4><<<blocks, 256, 0, stream>>>(a);
  else if (per <= 8) route_finish_kernel<8><<<blocks, 256, 0, stream>>>(a);
  else if (per <= 16) route_finish_kernel<16><<<blocks, 256, 0, stream>>>(a);
  else route_finish_kernel<32><<<blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
