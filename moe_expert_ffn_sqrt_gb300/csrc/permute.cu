// Expert-contiguous permute with per-expert alignment.
// Note "INT8 高吞吐/低延迟 EP 代码梳理" §9.3-9.4 (scatter, inv_perm, M_sum), §10 (M_sum_upper) and the
// m_indices paragraph (expert_ids, -1 on padding); MegaMoE page 路径 A (moe_align_block_size).
//
// Up to 1024 (t,k) pairs one small kernel does the index computation (and, up to 128 pairs, the
// row copy); above that two launches over up to 128 CTAs of 1024 threads do it, deterministically:
//   1. each CTA counts its contiguous chunk of the flat (t,k) list per expert;
//   2. each CTA sums the chunk counts per expert (total, and the CTAs before it), scans the aligned
//      segment sizes -> segment starts, M_sum; per (warp, expert) base row = segment start +
//      pairs of that expert in earlier CTAs and earlier warps of this CTA;
//   3. each warp walks its sub-range in order, 32 pairs at a time; __match_any_sync groups equal
//      experts so that each pair's rank among earlier pairs of its expert is exact.
// Padding rows get expert_ids = -1 and sorted_token_ids = T*K.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "permute_small.cuh"

namespace moe {

constexpr int kPermThreads = 1024;
constexpr int kPermWarps = kPermThreads / 32;

// Larger problems: G CTAs, CTA c owning the contiguous pairs [c*CH, (c+1)*CH) and each of its 32
// warps a contiguous sub-range, so that "earlier pair" order is (CTA, warp, lane).
// permute_count_kernel: per-CTA expert counts, stored expert-major as ccount[e*G + c].
// permute_place_kernel: each CTA sums its expert rows of ccount (total, and the part of earlier
// CTAs), scans the aligned segment sizes over experts, adds its per-warp histograms and places
// its pairs with __match_any_sync ranks; padding rows and the tail [M_sum, U) are split over CTAs.
constexpr int kPermMaxCtas = 128;

int permute_ctas(long long N) {
  long long g = (N + kPermThreads - 1) / kPermThreads;
  if (g > kPermMaxCtas) g = kPermMaxCtas;
  return g < 1 ? 1 : static_cast<int>(g);
}

static int permute_warp_chunk(long long N, int G) {
  const long long ch = (N + G - 1) / G;
  return static_cast<int>((ch + kPermWarps - 1) / kPermWarps);
}

size_t permute_scratch_bytes(int T, int K, int E) {
  const long long N = static_cast<long long>(T) * K;
  if (N <= 1024) return 0;
  return (static_cast<size_t>(permute_ctas(N)) * E * sizeof(int32_t) + 255) / 256 * 256;
}

__global__ void __launch_bounds__(kPermThreads, 1) permute_count_kernel(const PermuteArgs a, int W, int32_t* ccount) {
  extern __shared__ int32_t cnt[];                 // [E]
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int N = a.T * a.K, G = gridDim.x, c = blockIdx.x;
  for (int e = tid; e < a.E; e += kPermThreads) cnt[e] = 0;
  grid_dependency_wait();                          // topk_ids come from the previous launch
  __syncthreads();
  const int beg = min(N, (c * kPermWarps + warp) * W), end = min(N, beg + W);
  for (int i = beg + lane; i < end; i += 32) {
    const int e = a.topk_ids[i];
    if (e < 0 || e >= a.E) {
      record_error(a.status, kDevErrIndex);
      continue;
    }
    atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  for (int e = tid; e < a.E; e += kPermThreads) ccount[static_cast<size_t>(e) * G + c] = cnt[e];
}

__global__ void __launch_bounds__(kPermThreads, 1) permute_place_kernel(const PermuteArgs a, int W,
                                                                        const int32_t* __restrict__ ccount) {
  extern __shared__ int32_t sh[];
  int32_t* hist = sh;                              // [kPermWarps][E] -> per-warp base rows
  int32_t* seg = sh + kPermWarps * a.E;            // [E] segment start
  int32_t* tot = seg + a.E;                        // [E] pairs per expert
  __shared__ int32_t s_total;
  __shared__ int32_t s_scan[kPermThreads];
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int N = a.T * a.K, G = gridDim.x, c = blockIdx.x;
  const int beg = min(N, (c * kPermWarps + warp) * W), end = min(N, beg + W);
  for (int i = tid; i < kPermWarps * a.E; i += kPermThreads) hist[i] = 0;
  __syncthreads();
  // 1. per-warp histograms of this CTA's pairs
  for (int i = beg + lane; i < end; i += 32) {
    const int e = a.topk_ids[i];
    if (e >= 0 && e < a.E) atomicAdd(&hist[warp * a.E + e], 1);
  }
  // 2. totals and the earlier CTAs' share per expert; exclusive scan of aligned sizes
  const int per = (a.E + kPermThreads - 1) / kPermThreads;
  int local = 0;
  int pre_mine[4] = {0, 0, 0, 0};                  // per <= 4 (E <= 4096; E <= 1024 here)
  for (int j = 0; j < per; ++j) {
    const int e = tid * per + j;
    if (e < a.E) {
      const int32_t* row = ccount + static_cast<size_t>(e) * G;
      int t_all = 0, t_pre = 0;
#pragma unroll 8
      for (int cc = 0; cc < G; ++cc) {
        const int v = __ldg(row + cc);
        t_all += v;
        if (cc < c) t_pre += v;
      }
      tot[e] = t_all;
      pre_mine[j] = t_pre;
      local += a.slot > 0 ? a.slot : round_up_pow2(t_all, a.align);
    }
  }
  s_scan[tid] = local;
  __syncthreads();
  for (int off = 1; off < kPermThreads; off <<= 1) {   // inclusive Hillis-Steele scan
    const int v = (tid >= off) ? s_scan[tid - off] : 0;
    __syncthreads();
    s_scan[tid] += v;
    __syncthreads();
  }
  int run = s_scan[tid] - local;
  for (int j = 0; j < per; ++j) {
    const int e = tid * per + j;
    if (e < a.E) {
      seg[e] = run;
      int base = run + pre_mine[j];
      for (int w = 0; w < kPermWarps; ++w) {
        const int h = hist[w * a.E + e];
        hist[w * a.E + e] = base;
        base += h;
      }
      run += a.slot > 0 ? a.slot : round_up_pow2(tot[e], a.align);
    }
  }
  if (tid == kPermThreads - 1) s_total = s_scan[tid];
  __syncthreads();
  const int msum = s_total;
  // 3. ranks in (t,k) order within each warp's sub-range
  for (int i0 = beg; i0 < end; i0 += 32) {
    const int i = i0 + lane;
    const bool live = i < end;
    int e = live ? a.topk_ids[i] : -1;
    const bool ok = live && e >= 0 && e < a.E;
    if (!ok) e = -1 - lane;                            // unique dummy key for dead lanes
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    int pos = 0;
    if (ok) pos = hist[warp * a.E + e] + rank;
    __syncwarp();
    if (ok && rank == 0) hist[warp * a.E + e] += __popc(peers);
    __syncwarp();
    if (ok) {
      if (a.slot > 0 && pos - seg[e] >= a.slot) {
        record_error(a.status, kDevErrIndex);
        a.inv_perm[i] = -1;
      } else {
        a.inv_perm[i] = pos;
        a.sorted_ids[pos] = i;
        a.expert_ids[pos] = e;
      }
    }
  }
  // 4. padding rows inside each segment (experts split over CTAs), then the tail [M_sum, U)
  for (int e = c * kPermWarps + warp; e < a.E; e += G * kPermWarps) {
    const int n = tot[e];
    const int padded = a.slot > 0 ? a.slot : round_up_pow2(n, a.align);
    for (int r = n + lane; r < padded; r += 32) {
      a.sorted_ids[seg[e] + r] = N;
      a.expert_ids[seg[e] + r] = -1;
    }
  }
  for (int r = msum + c * kPermThreads + tid; r < a.U; r += G * kPermThreads) {
    a.sorted_ids[r] = N;
    a.expert_ids[r] = -1;
  }
  if (c == 0) {
    if (a.counts)
      for (int e = tid; e < a.E; e += kPermThreads) a.counts[e] = tot[e];
    if (tid == 0) *a.m_sum = msum;
  }
}

// The small permute (method in permute_small.cuh), one launch; permute_small_body there is the
// single-launch forward's copy of the same steps.
__global__ void __launch_bounds__(kPermThreads, 1) permute_small_kernel(const PermuteArgs a, const uint8_t* x_q,
                                                                        const uint8_t* x_sf, int H, uint8_t* x_perm,
                                                                        uint8_t* x_perm_sf, int bt, int nb) {
  extern __shared__ int32_t sh[];
  int32_t* cnt = sh;                 // [E]
  int32_t* seg = sh + a.E;           // [E]
  __shared__ int32_t s_ids[kSmallPairs];
  __shared__ int32_t s_rank[kSmallPairs];
  __shared__ int32_t s_total;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int N = a.T * a.K;
  for (int e = tid; e < a.E; e += kPermThreads) cnt[e] = 0;
  grid_dependency_wait();                          // topk_ids come from the previous launch
  grid_launch_dependents();                        // the expert FFN may start its prologue
  int e_mine = -1;
  if (tid < N) {
    e_mine = a.topk_ids[tid];
    if (e_mine < 0 || e_mine >= a.E) {
      if (blockIdx.x == 0) record_error(a.status, kDevErrIndex);
      e_mine = -1;
    }
    s_ids[tid] = e_mine;
  }
  __syncthreads();
  int rank = 0;
  if (e_mine >= 0) {
    atomicAdd(&cnt[e_mine], 1);
    for (int j = 0; j < tid; ++j) rank += (s_ids[j] == e_mine);
  }
  if (tid < N) s_rank[tid] = rank;
  __syncthreads();
  if (a.slot > 0) {                  // BatchedExperts: fixed slots
    for (int e = tid; e < a.E; e += kPermThreads) seg[e] = e * a.slot;
    if (tid == 0) s_total = a.E * a.slot;
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
    if (lane == 31) s_total = incl;
  }
  __syncthreads();
  const int msum = s_total;
  if (blockIdx.x == 0) {
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
      for (int e = tid; e < a.E; e += kPermThreads) a.counts[e] = cnt[e];
    if (tid == 0) *a.m_sum = msum;
  }
  // padding rows of each segment and the tail [M_sum, U), split over every CTA of the launch (each
  // holds the same counts and segment starts)
  for (int e = blockIdx.x * kPermWarps + warp; e < a.E; e += gridDim.x * kPermWarps) {
    const int c = cnt[e];
    const int padded = a.slot > 0 ? a.slot : round_up_pow2(c, a.align);
    for (int r = c + lane; r < padded; r += 32) {
      a.sorted_ids[seg[e] + r] = N;
      a.expert_ids[seg[e] + r] = -1;
    }
  }
  for (int r = msum + blockIdx.x * kPermThreads + tid; r < a.U; r += gridDim.x * kPermThreads) {
    a.sorted_ids[r] = N;
    a.expert_ids[r] = -1;
  }
  if ((x_perm != nullptr || x_perm_sf != nullptr) && N <= kSmallCopyPairs) {
    // one warp per (pair, 1 KB piece of its row); the piece-0 warp also copies the row's scales
    // (x_perm null: the scales alone, one warp per pair)
    const int chunks = x_perm != nullptr ? H / 16 : 0, slabs = H / 128;
    const int pieces = x_perm != nullptr ? (chunks + kCopyPiece - 1) / kCopyPiece : 1;
    for (int u = blockIdx.x * kPermWarps + warp; u < N * pieces; u += gridDim.x * kPermWarps) {
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
        if (j < chunks) v[i] = __ldg(src + j);
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

// Row copy: x_perm[inv_perm[t,k]] = x_q[t] (skipped when x_perm is null), scales into the tiled
// layout.  One warp per pair.
__global__ void __launch_bounds__(256) permute_rows_kernel(const int32_t* __restrict__ inv_perm,
                                                           const int32_t* __restrict__ topk_ids, int T, int K, int E,
                                                           int H, const uint8_t* __restrict__ x_q,
                                                           const uint8_t* __restrict__ x_sf, uint8_t* __restrict__ x_perm,
                                                           uint8_t* __restrict__ x_perm_sf, int bt, int nb) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  grid_launch_dependents();                        // the expert FFN may start its prologue
  const long long pair = static_cast<long long>(blockIdx.x) * 8 + warp;
  if (pair >= static_cast<long long>(T) * K) return;
  const int e = topk_ids[pair];
  if (e < 0 || e >= E) return;
  const int t = static_cast<int>(pair / K);
  const int dst = inv_perm[pair];
  if (dst < 0) return;                         // dropped by a full BatchedExperts slot
  const uint4* src = reinterpret_cast<const uint4*>(x_q + static_cast<size_t>(t) * H);
  uint4* out = reinterpret_cast<uint4*>(x_perm + static_cast<size_t>(dst) * H);
  const int chunks = x_perm != nullptr ? H / 16 : 0;
  for (int j0 = 0; j0 < chunks; j0 += 8 * 32) {      // eight 16-byte loads per lane in flight, then stores
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u * 32 + lane;
      if (j < chunks) v[u] = __ldg(src + j);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u * 32 + lane;
      if (j < chunks) out[j] = v[u];
    }
  }
  const int slabs = H / 128;
  for (int s = lane; s < slabs; s += 32) x_perm_sf[act_sf_offset(bt, nb, dst, s)] = x_sf[static_cast<size_t>(t) * slabs + s];
}

size_t permute_smem_bytes(int E) { return static_cast<size_t>(kPermWarps + 2) * E * sizeof(int32_t); }


// BatchedExperts row map from per-expert live-row counts: row r of slot e = r / slot is live
// (expert_ids[r] = e) when r % slot < count[e], else padding (-1).  A count above the slot size
// is an index error (the slot's rows are then all taken as live).  m_sum = E * slot.
__global__ void __launch_bounds__(256) batched_rows_kernel(const int32_t* __restrict__ counts, int E, int slot,
                                                           int32_t* __restrict__ expert_ids, int32_t* m_sum,
                                                           uint32_t* status) {
  const long long U = static_cast<long long>(E) * slot;
  for (long long r = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; r < U;
       r += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int e = static_cast<int>(r / slot), i = static_cast<int>(r - static_cast<long long>(e) * slot);
    const int n = __ldg(counts + e);
    if (i == 0 && (n < 0 || n > slot)) record_error(status, kDevErrIndex);
    expert_ids[r] = i < n ? e : -1;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *m_sum = static_cast<int>(U);
}

cudaError_t launch_batched_rows(const int32_t* counts, int E, int slot, int32_t* expert_ids, int32_t* m_sum,
                                uint32_t* status, cudaStream_t stream) {
  const long long U = static_cast<long long>(E) * slot;
  const int grid = static_cast<int>(std::min<long long>((U + 255) / 256, 4 * 152));
  batched_rows_kernel<<<grid < 1 ? 1 : grid, 256, 0, stream>>>(counts, E, slot, expert_ids, m_sum, status);
  return cudaGetLastError();
}

cudaError_t launch_permute(const int32_t* topk_ids, int T, int K, int E, int align, int U, int32_t* sorted_ids,
                           int32_t* expert_ids, int32_t* inv_perm, int32_t* m_sum, int32_t* counts,
                           const uint8_t* x_q, const uint8_t* x_sf, int H, uint8_t* x_perm, uint8_t* x_perm_sf,
                           uint32_t* status, int32_t* scratch, cudaStream_t stream, int slot) {
  PermuteArgs a{topk_ids, T, K, E, align, U, sorted_ids, expert_ids, inv_perm, m_sum, counts, status, slot};
  const int bt = act_sf_block_rows(align), nb = act_sf_blocks(U, bt);
  const long long npairs = static_cast<long long>(T) * K;
  cudaError_t err;
  if (npairs <= kSmallPairs) {
    const size_t smem = 2 * static_cast<size_t>(E) * sizeof(int32_t);
    err = cudaFuncSetAttribute(permute_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    const bool any = x_perm != nullptr || x_perm_sf != nullptr;     // rows and scales, or scales alone
    const bool copy = any && npairs <= kSmallCopyPairs;
    const long long units = npairs * (x_perm != nullptr ? (H / 16 + kCopyPiece - 1) / kCopyPiece : 1);
    const int grid = copy && npairs > 0 ? static_cast<int>((units + kPermWarps - 1) / kPermWarps) : 1;
    err = launch_pdl(permute_small_kernel, dim3(grid), dim3(kPermThreads), smem, stream, a, x_q, x_sf, H, x_perm,
                     x_perm_sf, bt, nb);
    if (err != cudaSuccess || !any || copy) return err;
  } else {
    if (scratch == nullptr) return cudaErrorInvalidValue;
    const int G = permute_ctas(npairs), W = permute_warp_chunk(npairs, G);
    err = cudaFuncSetAttribute(permute_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(E * sizeof(int32_t)));
    if (err != cudaSuccess) return err;
    err = launch_pdl(permute_count_kernel, dim3(G), dim3(kPermThreads), E * sizeof(int32_t), stream, a, W, scratch);
    if (err != cudaSuccess) return err;
    const size_t smem = permute_smem_bytes(E);
    err = cudaFuncSetAttribute(permute_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    permute_place_kernel<<<G, kPermThreads, smem, stream>>>(a, W, scratch);
    err = cudaGetLastError();
    if (err != cudaSuccess || (x_perm == nullptr && x_perm_sf == nullptr)) return err;
  }
  if (npairs == 0) return cudaSuccess;
  permute_rows_kernel<<<static_cast<int>((npairs + 7) / 8), 256, 0, stream>>>(inv_perm, topk_ids, T, K, E, H, x_q, x_sf,
                                                                               x_perm, x_perm_sf, bt, nb);
  return cudaGetLastError();
}

// Scales of the permuted rows from token-order scales: row r < M_sum with expert_ids[r] >= 0 takes
// the scales of token sorted_ids[r] / K into the tiled layout.  One thread per (row, slab).
__global__ void __launch_bounds__(256) permute_act_sf_kernel(const int32_t* __restrict__ sorted_ids, int K,
                                                             const int32_t* __restrict__ expert_ids,
                                                             const int32_t* __restrict__ m_sum, int U, int T,
                                                             const uint8_t* __restrict__ x_sf, int slabs, int bt,
                                                             int nb, uint8_t* __restrict__ out) {
  const int msum = min(*m_sum, U);
  const long long n = static_cast<long long>(msum) * slabs;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / slabs), s = static_cast<int>(i - static_cast<long long>(r) * slabs);
    if (__ldg(expert_ids + r) < 0) continue;
    const int t = __ldg(sorted_ids + r) / K;
    if (t < 0 || t >= T) continue;
    out[act_sf_offset(bt, nb, r, s)] = __ldg(x_sf + static_cast<size_t>(t) * slabs + s);
  }
}

cudaError_t launch_permute_act_sf(const int32_t* sorted_ids, int K, const int32_t* expert_ids, const int32_t* m_sum,
                                  int U, int T, const uint8_t* x_sf, int slabs, int align, uint8_t* out,
                                  cudaStream_t stream) {
  const int bt = act_sf_block_rows(align);
  const long long n = static_cast<long long>(U) * slabs;
  const int grid = static_cast<int>(std::min<long long>((n + 255) / 256, 4 * 152));
  permute_act_sf_kernel<<<grid < 1 ? 1 : grid, 256, 0, stream>>>(sorted_ids, K, expert_ids, m_sum, U, T, x_sf, slabs,
                                                                  bt, act_sf_blocks(U, bt), out);
  return cudaGetLastError();
}

}  // namespace moe
