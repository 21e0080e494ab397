// Internal launchers shared between the kernel files and the C ABI layer.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace moe {

// route.cu
int route_nsplit(int T, int H, int E);
size_t route_scratch_bytes(int T, int H, int E);   // ticket slot (first 256 bytes) + partial sums + gate parts
// Tiny-batch layout (no sort): pair p = t*K + k owns row kNaiveRows * p of the permuted buffers,
// the other rows of its block and the rows [kNaiveRows * T * K, U) are padding.  Written by the
// small-batch routing launch (T <= 16).
constexpr int kNaiveRows = 16;
struct NaiveLayout {
  int32_t* sorted = nullptr;   // [U]
  int32_t* eids = nullptr;     // [U]
  int32_t* inv = nullptr;      // [T*K]
  int32_t* m_sum = nullptr;    // [1]
  uint8_t* xp = nullptr;       // [U, H] E4M3
  uint8_t* xp_sf = nullptr;    // tiled (block rows kNaiveRows, rows U, slabs H/128)
  int U = 0, sf_nb = 0;
};
// The gate partial sums inside a routing scratch buffer (route_scratch_bytes of it).
float* route_partials(void* scratch);
cudaError_t launch_route(const uint16_t* hidden, const float* w_gate, const float* gate_bias, const float* e_bias,
                         int T, int H, int E, int K, int score_fn, int renormalize, float* logits_out,
                         int32_t* topk_ids, float* topk_w, uint8_t* x_q, uint8_t* x_sf, void* scratch,
                         uint32_t* status, cudaStream_t stream, const NaiveLayout* nv = nullptr,
                         const uint32_t* gate_failed = nullptr);

// permute.cu
size_t permute_smem_bytes(int E);
size_t permute_scratch_bytes(int T, int K, int E);   // per-CTA expert counts of the multi-CTA path
cudaError_t launch_batched_rows(const int32_t* counts, int E, int slot, int32_t* expert_ids, int32_t* m_sum,
                                uint32_t* status, cudaStream_t stream);   // BatchedExperts row map from counts
cudaError_t launch_permute(const int32_t* topk_ids, int T, int K, int E, int align, int U, int32_t* sorted_ids,
                           int32_t* expert_ids, int32_t* inv_perm, int32_t* m_sum, int32_t* counts,
                           const uint8_t* x_q, const uint8_t* x_sf, int H, uint8_t* x_perm, uint8_t* x_perm_sf,
                           uint32_t* status, int32_t* scratch, cudaStream_t stream, int slot = 0);

// Tiled scales of the permuted rows gathered from token-order scales x_sf [T, slabs] through
// sorted_ids (row r < M_sum with expert_ids[r] >= 0 takes token sorted_ids[r] / K).
cudaError_t launch_permute_act_sf(const int32_t* sorted_ids, int K, const int32_t* expert_ids, const int32_t* m_sum,
                                  int U, int T, const uint8_t* x_sf, int slabs, int align, uint8_t* out,
                                  cudaStream_t stream);

// gate.cu (T > 16: gate GEMM on the tensor cores, three exact bf16 parts of the fp32 gate weight)
int gate_nsplit(int T, int H, int E);
size_t gate_parts_bytes(int T, int H, int E);
cudaError_t launch_gate_mma(const uint16_t* hidden, const float* w_gate, int T, int H, int E, int nsplit,
                            uint16_t* parts, float* partial, uint32_t* status, cudaStream_t stream);

// gemm.cu
// 2D tiled tensor map with 128-byte swizzle (inner extent `inner` elements, `outer` rows).
bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);
struct GemmLaunch {
  const uint8_t* w;            // packed weight stream
  const uint8_t* x;            // [U, Kd] E4M3
  const uint8_t* x_sf;         // tiled (rows U, slabs Kd/128)
  const int32_t* expert_ids;
  const int32_t* m_sum;
  uint8_t* h_q;
  uint8_t* h_sf;
  uint16_t* y;
  uint32_t* status;
  int E, w_rows, Kd, I, U, align;
  FusedReduce red{};           // L2: fold the unpermute-reduce into the epilogue when red.out is set
  const int32_t* row_ids = nullptr;   // L1 with row weights: h of row r is scaled by
  const float* row_w = nullptr;       // row_w[row_ids[r]] (the routing weight of the row's pair)
  const int32_t* counts = nullptr;    // BatchedExperts: tokens per expert slot (masked work list)
  int slot = 0;                       // BatchedExperts slot rows (a multiple of the block height)
  // L1 gather mode: x is the token-order [gather_rows, Kd] activation and permuted row r reads row
  // gather_ids[r] / gather_k of it (x_sf stays the tiled permuted scales)
  const int32_t* gather_ids = nullptr;
  int gather_k = 1;
  int gather_rows = 0;
};
int num_sms();
int weight_tiles(int N, int pair);
size_t packed_weight_bytes(int E, int N, int Kd, int pair);
int gemm_block_n(int align);
// `sched`: gemm_sched_words(U, align) words of the workspace, zero before a launch and left at zero.
cudaError_t launch_gemm(const GemmLaunch& L, bool l1, uint32_t* sched, cudaStream_t stream);
// L1 and L2 in one launch (L2 tiles wait for their row block's L1 tiles).
cudaError_t launch_ffn(const GemmLaunch& l1, const GemmLaunch& l2, uint32_t* sched, cudaStream_t stream);
size_t gemm_sched_words(int U, int align);
// Single-launch forward (small batches, MXFP4, 16-row GEMM blocks): the small-batch routing and
// permute run inside the FFN launch before its GEMM work (cooperative launch, two grid barriers).
// The fields are those of launch_route and launch_permute; partial = the routing scratch's partial
// sums (route_partials).
struct PreludeLaunch {
  const uint16_t* hidden;
  const float* w_gate;
  const float* gate_bias;
  const float* e_bias;
  int T, H, E, K, score_fn, renormalize;
  float* logits_out;
  int32_t* topk_ids;
  float* topk_w;
  uint8_t* x_q;
  uint8_t* x_sf;
  float* partial;
  int align, U;
  int32_t* sorted_ids;
  int32_t* expert_ids;
  int32_t* inv_perm;
  int32_t* m_sum;
  int32_t* counts;
  uint8_t* x_perm;
  uint8_t* x_perm_sf;
  uint32_t* status;
};
bool prelude_supported(int T, int E, int K, int align);
cudaError_t launch_ffn_prelude(const GemmLaunch& l1, const GemmLaunch& l2, const PreludeLaunch& p, uint32_t* sched,
                               cudaStream_t stream);
cudaError_t launch_pack_mx(const uint8_t* q, const uint8_t* sf, int E, int N, int Kd, int pair, uint8_t* out,
                           cudaStream_t stream);

// gemm_nv.cu (NVFP4 weights, bf16 MMA)
struct NvLaunch {
  const uint8_t* w;            // packed NVFP4 weight stream
  const float* tscale;         // [E]
  const uint16_t* xb;          // [U, Kd] bf16 activation rows
  const int32_t* expert_ids;
  const int32_t* m_sum;
  uint8_t* h_q;
  uint8_t* h_sf;
  uint16_t* y;
  uint32_t* status;
  int E, w_rows, Kd, I, U, align;
  FusedReduce red{};
  const int32_t* row_ids = nullptr;   // L1 row weights, as in GemmLaunch
  const float* row_w = nullptr;
};
size_t packed_nv_weight_bytes(int E, int N, int Kd, int pair);
cudaError_t launch_pack_nv(const uint8_t* q, const uint8_t* sf, int E, int N, int Kd, int pair, uint8_t* out,
                           cudaStream_t stream);
// bf16 rows of the activation for rows r < m_sum with expert_ids[r] >= 0.  gather_ids null: x is
// [U, Kd] with tiled scales (block rows from align); else x is token-order [T, Kd] with plain scales
// [T, Kd/128] and row r reads token gather_ids[r] / K.
cudaError_t launch_act_to_bf16(const uint8_t* x, const uint8_t* sf, const int32_t* expert_ids, const int32_t* m_sum,
                               int U, int Kd, int align, uint16_t* xb, cudaStream_t stream,
                               const int32_t* gather_ids = nullptr, int K = 1, int T = 0);
// The same rows from token-order x [T, Kd] with plain scales [T, Kd/128], one pass per token: row
// inv_perm[t*K + k] (entries outside [0, U) skipped) gets token t's converted row.  K <= 32.
cudaError_t launch_act_to_bf16_tokens(const uint8_t* x, const uint8_t* sf, const int32_t* inv_perm, int T, int K, int U,
                                      int Kd, uint16_t* xb, cudaStream_t stream);
cudaError_t launch_gemm_nv(const NvLaunch& L, bool l1, cudaStream_t stream);

// gemm_i8.cu (INT8 W8A8 variant: int8 codes as fp16 on the 16-bit MMA, row and channel scales in the
// epilogue)
struct I8Launch {
  const uint8_t* w;            // packed int8 weight stream
  const float* col_scale;      // [E, w_rows] per-output-channel scales (block: [E, w_rows/256, Kd/256])
  const uint16_t* xf;          // [U, Kd] fp16 activation codes
  const float* row_scale;      // [U] per-row activation scales (block: [U, Kd/256])
  const int32_t* expert_ids;
  const int32_t* m_sum;
  uint16_t* out;               // L1: h [U, I] bf16; L2: y [U, H] bf16
  uint32_t* status;
  int E, w_rows, Kd, I, U, align;
  FusedReduce red{};
  int block = 0;               // [256, 256] block-quantised weights, per-256-group activation scales
};
size_t packed_i8_weight_bytes(int E, int N, int Kd, int pair);
cudaError_t launch_pack_i8(const int8_t* q, int E, int N, int Kd, int pair, uint8_t* out, cudaStream_t stream);
// fp16 rows of int8 codes (+ the row's nsc scales) for rows r < m_sum with expert_ids[r] >= 0;
// source row src_map[r] / K when src_map is given, else r.
cudaError_t launch_i8_rows_to_f16(const int8_t* src, const float* src_scale, int src_rows, const int32_t* src_map,
                                  int K, const int32_t* expert_ids, const int32_t* m_sum, int U, int C, uint16_t* dst,
                                  float* dst_scale, uint32_t* status, cudaStream_t stream, int nsc = 1);
// Int8 quantisation of bf16 rows per group of `group` columns (0: the whole row; s is [rows, C/group])
// (all R rows, or with expert_ids the pair rows below m_sum); f16 (nullable) receives the codes as fp16.
cudaError_t launch_quant_rows_i8(const uint16_t* x, int R, int C, const int32_t* expert_ids, const int32_t* m_sum,
                                 int8_t* q, float* s, uint16_t* f16, cudaStream_t stream, int group = 0);
cudaError_t launch_gemm_i8(const I8Launch& L, bool l1, cudaStream_t stream);

// reduce.cu
cudaError_t launch_wait_selftest(const uint32_t* never_set, uint32_t* status, int mode, cudaStream_t stream);
cudaError_t launch_unpermute_reduce(const uint16_t* y, const int32_t* inv_perm, const float* topk_w, int T, int K,
                                    int H, uint16_t* out, cudaStream_t stream);

// Launches `kernel` with programmatic stream serialization: it may begin (up to its
// grid_dependency_wait) while the stream's previous kernel finishes.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace moe
