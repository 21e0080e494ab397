// Device helpers shared by the kernels: status word, mbarrier, TMA, tcgen05 (UMMA/TMEM).
// sm_103a only.  Every wait is bounded: on expiry the status word records MOE_ERR_TIMEOUT
// and the caller unwinds instead of spinning forever.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace moe {

constexpr uint32_t kDevErrIndex = 5;     // matches MOE_ERR_DEVICE_INDEX
constexpr uint32_t kDevErrTimeout = 6;   // matches MOE_ERR_TIMEOUT
constexpr long long kWaitBudgetCycles = 4000000000LL;   // ~2 s at 2 GHz

__device__ __forceinline__ void record_error(uint32_t* status, uint32_t code) {
  if (status) atomicCAS(status, 0u, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------------------------------
// mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false (and records a
// timeout in *status) if it has not completed within the cycle budget.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* status) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_test(bar, parity)) {
    if (clock64() - t0 > kWaitBudgetCycles) {
      record_error(status, kDevErrTimeout);
      return false;
    }
  }
  return true;
}

// ------------------------------------------------------------------------------------------
// Counters shared between CTAs of one launch

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Orders this thread's generic-proxy global accesses with its async-proxy (TMA / bulk copy)
// accesses: used on both sides when one CTA's plain stores are read by another CTA's TMA.
// Programmatic dependent launch: a kernel launched with programmatic stream serialization may start
// while the previous kernel of the stream still runs; this waits until that kernel has completed
// and its memory operations are visible (returns at once for an ordinary launch).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the stream's next kernel, if launched with programmatic stream serialization, start its
// CTAs now (they still wait for this kernel's completion before reading its results).
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Waits until *p >= target (acquire).  Bounded like mbar_wait.
__device__ __forceinline__ bool wait_counter(const uint32_t* p, uint32_t target, uint32_t* status) {
  if (ld_acquire_gpu(p) >= target) return true;
  const long long t0 = clock64();
  while (ld_acquire_gpu(p) < target) {
    if (clock64() - t0 > kWaitBudgetCycles) {
      record_error(status, kDevErrTimeout);
      return false;
    }
    __nanosleep(128);
  }
  return true;
}

// ------------------------------------------------------------------------------------------
// TMA and bulk copies (global -> shared, completion counted on an mbarrier)

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}

// Four rows of a 2D tensor map with a one-row box, rows y0..y3 at column c0, landing as rows 0..3 of
// a tile at dst (the tensor map's swizzle applies as for a four-row box at that address).  Rows
// outside the tensor read as zeros.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int c0, int y0, int y1, int y2,
                                            int y3, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
      "l"(map), "r"(c0), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Starts pulling [src, src + bytes) into L2 (no completion tracking).  16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ------------------------------------------------------------------------------------------
// tcgen05: tensor memory, UMMA, copies and loads

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor.  swz: 0 none, 2 = 128-byte swizzle (K-major tiles whose
// rows are 128 bytes and whose 8-row groups are 1024 bytes apart).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
  d |= 1ull << 46;   // descriptor version for tcgen05
  d |= static_cast<uint64_t>(swz & 7) << 61;
  return d;
}
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) { return smem_desc(saddr, 16, 1024, 2); }

// Instruction descriptor of kind::mxf8f6f4 with UE8M0 block scales (scale_vec::1X, K = 32).
// a_fmt / b_fmt: 0 = E4M3, 5 = E2M1.  Both operands K-major.
__device__ __forceinline__ uint32_t idesc_mxf8f6f4(uint32_t a_fmt, uint32_t b_fmt, uint32_t M, uint32_t N,
                                                   uint32_t sfa_id, uint32_t sfb_id) {
  return (sfb_id << 4) | (a_fmt << 7) | (b_fmt << 10) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24) |
         (sfa_id << 29);
}

__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::f16 with bf16 A/B and fp32 accumulation.
__device__ __forceinline__ uint32_t idesc_bf16(uint32_t M, uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Instruction descriptor of kind::f16 with fp16 A/B and fp32 accumulation.
__device__ __forceinline__ uint32_t idesc_f16(uint32_t M, uint32_t N) {
  return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// kind::f16 MMA (bf16 or fp16 operands, as the instruction descriptor says).
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 rows x 16 bytes from shared memory, broadcast into the four 32-lane quarters, 4 columns.
__device__ __forceinline__ void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Each thread of the warp reads its lane (quarter base + lane id), 16 consecutive columns.
__device__ __forceinline__ void tc_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Each thread of the warp writes its lane (quarter base + lane id), 16 consecutive columns.
__device__ __forceinline__ void tc_st_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------------------------------
// CTA pairs: a cluster of two CTAs on neighbouring SMs sharing one tcgen05 MMA (cta_group::2).
// A kernel that uses these uses cta_group::2 for every tcgen05 instruction that names a group.

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
  return d;
}

// Arrive on an mbarrier of either CTA of the cluster, given by its shared::cluster address (the
// default release semantics of mbarrier.arrive, as for a local arrive: a release at cluster scope
// makes every arriving warp wait for a cluster-wide memory barrier).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Every thread of both CTAs (the two CTAs of a cluster are co-scheduled, so it always completes).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// One warp of each CTA of the pair, together: the same columns in both CTAs' tensor memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// kind::f16 MMA over the pair, issued by one thread of the even CTA: A rows [0, M/2) from the even
// CTA's shared memory and [M/2, M) from the odd CTA's (same address), B rows [0, N/2) from the even
// CTA and [N/2, N) from the odd one; each CTA's tensor memory receives its M/2 rows x N.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives on the mbarrier at shared-memory offset `bar` in every CTA of `cta_mask` once the pair's
// earlier MMAs have completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

// One 32-byte global store (a whole sector); p must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* p, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3, uint32_t w4,
                                             uint32_t w5, uint32_t w6, uint32_t w7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w0), "r"(w1), "r"(w2),
               "r"(w3), "r"(w4), "r"(w5), "r"(w6), "r"(w7)
               : "memory");
}

__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Barrier over `nthreads` threads that also returns the AND of `pred` over all of them.
__device__ __forceinline__ bool named_barrier_and(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.and.pred q, %2, %3, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ bool named_barrier_or(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, %2, %3, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// ------------------------------------------------------------------------------------------
// FP8 (E4M3) quantisation with a power-of-two scale: the smallest e with amax <= 448 * 2^e,
// clamped to [-127, 127], 0 when amax == 0.  Exact integer arithmetic on the fp32 bits.
__device__ __forceinline__ int ue8m0_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax) & 0x7FFFFFFFu;
  if (b == 0) return 0;
  if (b >= 0x7F800000u) return 127;                     // inf / nan: saturate the scale
  const int ex = static_cast<int>(b >> 23);             // biased exponent, 0 for subnormals
  if (ex == 0) return -127;                             // amax < 2^-126: e would be < -134
  const uint32_t mant = b & 0x7FFFFFu;
  // amax = (1 + mant/2^23) * 2^(ex-127);  448 = 1.75 * 2^8
  int e = ex - 127 - 8 + (mant > 0x600000u ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as an exact float for e in [-127, 127].
__device__ __forceinline__ float pow2_neg(int e) {
  const int be = 127 - e;                               // biased exponent of 2^-e
  return be >= 1 ? __uint_as_float(static_cast<uint32_t>(be) << 23) : __uint_as_float(0x00400000u);
}

// Tiled activation-scale layout (see include/moe.h).  Bt = rows per GEMM block (16..128);
// nb = ceil(rows / Bt) + 1 blocks (one spare); chunk bytes CB = 256 for Bt = 16, else 512.
__host__ __device__ __forceinline__ int act_sf_block_rows(int align) {
  int bt = 16;
  while (bt < 128 && bt * 2 <= align) bt *= 2;
  return bt;
}
__host__ __device__ __forceinline__ int act_sf_chunk_bytes(int bt) { return bt == 16 ? 256 : 512; }
__host__ __device__ __forceinline__ int act_sf_blocks(int rows, int bt) { return (rows + bt - 1) / bt + 1; }
__host__ __device__ __forceinline__ size_t act_sf_offset(int bt, int nb, int r, int s) {
  const int rb = r % bt;
  return (static_cast<size_t>(s >> 2) * nb + r / bt) * act_sf_chunk_bytes(bt) + (rb & 31) * 16 + (rb >> 5) * 4 +
         (s & 3);
}
__host__ __device__ __forceinline__ size_t act_sf_bytes(int rows, int slabs, int bt) {
  return static_cast<size_t>((slabs + 3) / 4) * act_sf_blocks(rows, bt) * act_sf_chunk_bytes(bt);
}

constexpr uint32_t kDevErrCheck = 7;    // a kernel self-check (bounds / alignment) failed

// ------------------------------------------------------------------------------------------
// Weighted unpermute-reduce folded into the L2 epilogue: out[t] = bf16(sum_k w[t,k] y[inv[t,k]]).
// After an epilogue has stored the y values of column tile `tile` for its rows, each real row
// takes a ticket for (token, tile); the row that brings the count to K completes the token.
struct FusedReduce {
  uint16_t* out;                 // [T, H] bf16; nullptr = not fused
  const int32_t* inv_perm;       // [T, K]
  const float* topk_w;           // [T, K]; nullptr: plain sum (the weights were applied in L1)
  const int32_t* sorted_ids;     // [U]
  uint32_t* tickets;             // [T, n_col_tiles], zero between calls
  int K;
};

// Called by a whole epilogue warp after its rows' y values for column tile `tile` are stored.
// Each lane that holds a real row counts that row's (token, tile) ticket; a lane that completes
// a token's K-th arrival marks the token, and the warp then reduces the marked tokens one at a
// time, 8 columns per lane, in slot order k = 0..K-1 with fp32 fma (the order of the separate
// unpermute-reduce kernel, so both give identical bits).  The completing warp resets the ticket.
__device__ __forceinline__ void fused_reduce_tail(const FusedReduce& f, const uint16_t* y, int H, bool mine, int row,
                                                  int tile, int n_tiles, int c0, int ncols) {
  const int lane = threadIdx.x & 31;
  int t = 0;
  bool last = false;
  if (mine) {
    t = __ldg(f.sorted_ids + row) / f.K;
    __threadfence();
    last = atomicAdd(f.tickets + static_cast<size_t>(t) * n_tiles + tile, 1u) == static_cast<uint32_t>(f.K - 1);
  }
  unsigned todo = __ballot_sync(0xffffffffu, last);
  if (todo == 0) return;
  __threadfence();
  while (todo) {
    const int src = __ffs(todo) - 1;
    todo &= todo - 1;
    const int tt = __shfl_sync(0xffffffffu, t, src);
    int rk = 0;
    float wk = 0.f;
    if (lane < f.K) {
      rk = __ldg(f.inv_perm + static_cast<size_t>(tt) * f.K + lane);
      wk = f.topk_w ? __ldg(f.topk_w + static_cast<size_t>(tt) * f.K + lane) : 1.f;
    }
    for (int cb = 0; cb < ncols; cb += 256) {
      const int c = c0 + cb + lane * 8;
      const bool active = cb + lane * 8 < ncols;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int k = 0; k < f.K; ++k) {
        const int r = __shfl_sync(0xffffffffu, rk, k);
        const float w = __shfl_sync(0xffffffffu, wk, k);
        if (active) {
          const uint4 v = __ldcg(reinterpret_cast<const uint4*>(y + static_cast<size_t>(r) * H + c));
          const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc[2 * j] = fmaf(w, __uint_as_float(u[j] << 16), acc[2 * j]);
            acc[2 * j + 1] = fmaf(w, __uint_as_float(u[j] & 0xFFFF0000u), acc[2 * j + 1]);
          }
        }
      }
      if (active) {
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * j]));
          const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * j + 1]));
          o[j] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(f.out + static_cast<size_t>(tt) * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    if (lane == 0) f.tickets[static_cast<size_t>(tt) * n_tiles + tile] = 0;
  }
}

}  // namespace moe
