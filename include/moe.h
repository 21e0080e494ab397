/*
 * moe.h - C ABI of the GB300 (sm_103a) single-GPU Mixture-of-Experts layer forward.
 *
 * The layer (page "DeepSeek V4 MegaMoE Kernel 深度解析", section 经典 MoE 的计算过程):
 *   gate GEMM -> score (softmax | sqrt(softplus)) -> top-K with e_score_correction_bias
 *   -> expert-contiguous permute padded per expert to `align` rows
 *   -> L1 grouped GEMM against W13 [2I,H] + SwiGLU + FP8 requant
 *   -> L2 grouped GEMM against W2 [H,I] (bf16 out)
 *   -> topk-weighted unpermute-reduce back to [T,H] (bf16).
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers owned by the caller, contiguous, row-major,
 *     unless a comment says "host".  Nothing here allocates, frees or synchronises the
 *     device, except moe_get_error (which synchronises the given stream).
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL = legacy default
 *     stream) and runs asynchronously.  No call reads a device value back to the host:
 *     M_sum stays in device memory and buffers are sized by moe_msum_upper().
 *   - bf16 values are passed as their uint16 bit patterns.  E4M3 / E2M1 / UE8M0 values are
 *     passed as their codes (uint8; E2M1 two per byte, element 2j in the low nibble).
 *   - Host-side argument errors are returned at once and nothing is launched.  Errors the
 *     device detects (an expert id outside [0,E) in topk_ids, a bounded wait that expired)
 *     are recorded in a status word inside the workspace; moe_get_error reads and clears it.
 *   - Calls are stateless and reentrant; calls that share a workspace must not overlap.
 *   - H and I must be multiples of 128 (the pages state this limit for the fused kernel);
 *     K <= E; align is a power of two in [1, 256]; all pointers 16-byte aligned
 *     (W q pointers 32-byte aligned).
 *
 * Scale layouts used between the calls (documented so callers can interpret them):
 *   - Activation scales "tiled" (x_perm_sf, h_sf): one UE8M0 byte per (row r, 128-column
 *     slab s) of a permuted activation matrix with `rows` rows and `slabs` slabs.  With
 *     Bt = moe_act_sf_block_rows(align) (the grouped GEMMs' row-block size: the largest power
 *     of two <= align, clamped to [16, 128]), nb = ceil(rows/Bt) + 1 and CB = 256 for Bt = 16,
 *     else 512, the byte of (r, s) is at
 *       ((s/4)*nb + r/Bt)*CB + ((r%Bt)%32)*16 + ((r%Bt)/32)*4 + (s%4)
 *     so each (row block, 4 slabs) is one contiguous chunk that the GEMM copies into tensor
 *     memory as is.  Total moe_act_sf_tiled_bytes(rows, slabs, align); the _host helpers
 *     convert to and from the plain [rows, slabs] layout.
 *   - Weights: read from the packed stream produced once per tensor by moe_pack_weights().
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or enum */
  MOE_ERR_UNSUPPORTED = 2,   /* valid but not supported (e.g. E too large for the permute kernel) */
  MOE_ERR_WORKSPACE = 3,     /* ws NULL or smaller than moe_workspace_size() */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
  MOE_ERR_DEVICE_INDEX = 5,  /* device saw an expert id outside [0, E) */
  MOE_ERR_TIMEOUT = 6,       /* a device-side bounded wait expired */
  MOE_ERR_DEVICE_CHECK = 7   /* a kernel's own bounds / alignment check failed; the access was skipped */
} moe_status;

typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SQRT_SOFTPLUS = 1 } moe_score_fn;

/* Weight formats (CUDA tag page teaser: MXFP4 vs NVFP4, chosen by moe_quant_algo; note
 * "INT8 高吞吐/低延迟 EP 代码梳理" §2, §3.1: INT8 with channel-wise weights).
 *   MXFP4: E2M1 codes + one UE8M0 scale per 32 along the reduction dim.
 *   NVFP4: E2M1 codes + one E4M3 scale per 16 along the reduction dim + one fp32 scale per
 *          expert matrix.
 *   INT8:  int8 codes + one fp32 scale per output channel (row); only the *_i8 calls take it.
 *   INT8_B256: int8 codes + one fp32 scale per block of 256 output rows x 256 reduction columns
 *          (§3.1 "INT8 with block_shape [256, 256]"); only the *_i8 calls take it. */
typedef enum { MOE_W_MXFP4 = 0, MOE_W_NVFP4 = 1, MOE_W_INT8 = 2, MOE_W_INT8_B256 = 3 } moe_wfmt;

/* One stacked expert weight tensor with logical shape [E, N, Kd] (N output rows, Kd the
 * reduction dim), in the packed stream written by moe_pack_weights.  W13: N = 2I, Kd = H,
 * rows 0..I-1 are the gate projection W1 and rows I..2I-1 the up projection W3 (MegaMoE page,
 * 第三步), packed with pair = 2.  W2: N = H, Kd = I, packed with pair = 1. */
typedef struct {
  const uint8_t* packed;  /* moe_pack_weights output (32-byte aligned)                        */
  const float* tscale;    /* NVFP4: [E] fp32 per-matrix scale; INT8: [E, N] fp32 per-output-  *
                           * channel scales (logical row order, 16-byte aligned); INT8_B256:    *
                           * [E, N/256, Kd/256] fp32 block scales; MXFP4: NULL                 */
  moe_wfmt fmt;
  int E, N, Kd;           /* logical shape                                                    */
  int pair;               /* 2 for W13 (gate/up row tiles interleaved), 1 for W2              */
} moe_weight;

/* --------------------------------------------------------------------------------------
 * Sizes and host-side helpers (no device work).
 * ------------------------------------------------------------------------------------ */

/* M_sum_upper = T*K + E*(align-1): the most rows the aligned expert-contiguous layout can
 * need (note "INT8 高吞吐/低延迟 EP 代码梳理", §10).  Every [U, ...] buffer below has U rows. */
size_t moe_msum_upper(int T, int K, int E, int align);

/* Rows per block of the tiled activation-scale layout for a permute alignment `align`. */
int moe_act_sf_block_rows(int align);

/* Bytes of a "tiled" activation-scale buffer for an activation with `rows` rows and
 * `slabs` = columns/128 slabs, for permute alignment `align` (layout in the file header). */
size_t moe_act_sf_tiled_bytes(int rows, int slabs, int align);

/* Host memory: tiled [moe_act_sf_tiled_bytes(rows,slabs,align)] -> plain [rows, slabs]. */
moe_status moe_act_sf_untile_host(const uint8_t* tiled, int rows, int slabs, int align, uint8_t* out);

/* Host memory: plain [rows, slabs] -> tiled [moe_act_sf_tiled_bytes(rows,slabs,align)]; bytes of
 * the tiled buffer that no (row, slab) maps to are set to 127 (scale 1.0). */
moe_status moe_act_sf_tile_host(const uint8_t* plain, int rows, int slabs, int align, uint8_t* tiled);

/* Bytes of the packed stream of a weight tensor [E, N, Kd] in format fmt with the given pairing
 * (0 if the shape is not supported). */
size_t moe_weight_packed_bytes(moe_wfmt fmt, int E, int N, int Kd, int pair);

/* Rearranges a weight tensor (codes [E, N, Kd/2] packed E2M1; scales [E, N, Kd/32] UE8M0 for
 * MXFP4) into the stream the grouped GEMMs read: one contiguous chunk per (expert, weight tile,
 * 128-deep slab) in reading order, so that weights stream from HBM in long sequential runs.
 * A weight tile is 256 rows: pair = 2 joins rows 128t.. with rows N/2 + 128t.. (W13: gate with
 * up); pair = 1 takes rows 256t.. (W2; rows past N read as zero).  Each chunk holds the tile's
 * codes, then its scales arranged for tensor memory.  Done once per weight tensor (weights are
 * static).  Kd must be a multiple of 128; N of 256 (pair = 2) or 128 (pair = 1).
 * INT8: q is the int8 codes [E, N, Kd] (16-byte aligned), sf is ignored (may be NULL); each
 * chunk is a tile's 256 rows x 64 codes (the channel scales stay in the caller's [E, N] array). */
moe_status moe_pack_weights(moe_wfmt fmt, const uint8_t* q, const uint8_t* sf, int E, int N, int Kd, int pair,
                            uint8_t* packed, void* stream);

/* Bytes of workspace needed by moe_route, moe_permute, the grouped GEMMs and moe_forward
 * for this problem.  The first 256 bytes hold the device status word.  A workspace must
 * be zero-filled once before first use (it is then kept consistent by the calls). */
moe_status moe_workspace_size(int T, int H, int I, int E, int K, int align, size_t* bytes);

/* --------------------------------------------------------------------------------------
 * Hot-path calls.
 * ------------------------------------------------------------------------------------ */

/* Routing and activation quantisation (MegaMoE page 第一步：路由; CUDA tag page teaser
 * "Fused TopK Bias Routing": sqrt(softplus), e_score_correction_bias).
 *   hidden       [T, H] bf16
 *   w_gate       [E, H] fp32;  logits = hidden @ w_gate^T (+ gate_bias[E] if non-NULL)
 *   e_score_bias [E] fp32 or NULL: added to the scores for top-K selection only
 *   fn           softmax over E, or sqrt(ln(1 + e^logit)) per expert
 *   topk_ids     [T, K] int32 out: the K largest (score + e_score_bias), ties to the lower
 *                expert id, ordered by descending key
 *   topk_w       [T, K] fp32 out: the selected unbiased scores, divided by their sum when
 *                renormalize != 0
 *   logits_out   [T, E] fp32 out or NULL
 *   x_q, x_sf    [T, H] E4M3 and [T, H/128] UE8M0 out, or both NULL: per 128 columns the
 *                scale is the smallest power of two 2^e with amax <= 448 * 2^e (e in
 *                [-127,127], e = 0 when amax = 0) and x_q = RNE_e4m3(x / 2^e).
 *   ws           workspace (status word; routing scratch: a counter slot at a fixed offset that
 *                every call leaves at zero, then split-K partial sums that each call writes
 *                before it reads them). */
moe_status moe_route(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                     const float* e_score_bias, int T, int H, int E, int K, moe_score_fn fn,
                     int renormalize, float* logits_out, int32_t* topk_ids, float* topk_w,
                     uint8_t* x_q, uint8_t* x_sf, void* ws, size_t ws_bytes, void* stream);

/* moe_route without a workspace and without allocating anything.  This call has no counterpart in
 * the method's description; it exists for callers that can neither pass a workspace nor allocate
 * device memory (an engine that plans all device buffers up front and forbids cudaMalloc later,
 * a plugin interface that supplies only inputs and outputs).  Same arguments and results as
 * moe_route minus ws/ws_bytes.  Its scratch is a fixed 4 MiB array in device memory inside the
 * library (held on every GPU that loads the library until exit): 256 bytes for a failure word,
 * a 256-byte counter slot at a fixed place (every call leaves it at zero), nsplit*T*E*4 bytes of
 * partial sums (nsplit = 4 for T <= 16) rounded up to 256, and for T > 16 another 3*E*H*2 bytes
 * (bf16 parts of the gate weight); the call returns MOE_ERR_UNSUPPORTED when that exceeds 4 MiB.
 * The partial sums and parts a call reads are the ones it wrote; the array keeps the last call's.
 * Without a workspace there is no status word: if the tensor-core gate GEMM (T > 16) gives up on
 * a bounded wait, the call still returns MOE_OK but writes -1 to every topk_ids entry and NaN to
 * every weight (and logit).  All calls on a device share the array, so calls that may overlap on
 * the GPU race.  The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress): make it before any stream capture starts. */
moe_status moe_route_noalloc(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                             const float* e_score_bias, int T, int H, int E, int K, moe_score_fn fn,
                             int renormalize, float* logits_out, int32_t* topk_ids, float* topk_w,
                             uint8_t* x_q, uint8_t* x_sf, void* stream);

/* Expert-contiguous permute (note "INT8 高吞吐/低延迟 EP 代码梳理" §9.3-9.4, §10 and the
 * m_indices paragraph; MegaMoE page 路径 A moe_align_block_size).
 * With cnt_e = #(t,k) routed to e and seg_e = sum_{e'<e} round_up(cnt_e', align):
 *   inv_perm[t,k]          [T, K] out: seg_e + (rank of (t,k) among expert e's pairs in
 *                          ascending t*K+k order)
 *   sorted_token_ids[row]  [U] out: t*K + k of the pair on that row, T*K on padding rows
 *   expert_ids[row]        [U] out: expert of the row, -1 on padding rows and rows >= M_sum
 *   m_sum                  [1] out (device): sum_e round_up(cnt_e, align)
 *   expert_counts          [E] out or NULL: cnt_e
 *   x_q, x_sf, x_perm, x_perm_sf: optional (all NULL, all set, or only x_sf and x_perm_sf): x_perm
 *   [U, H] gets row x_q[t] on row inv_perm[t,k]; x_perm_sf (tiled for `align`, rows = U, slabs =
 *   H/128) its scales.  With x_sf and x_perm_sf alone only the scales move (the input of the
 *   token-order L1, which reads the rows through sorted_token_ids).  Rows of x_perm at padding
 *   positions are left unwritten.
 * An id outside [0, E) records MOE_ERR_DEVICE_INDEX and the outputs are unspecified. */
moe_status moe_permute(const int32_t* topk_ids, int T, int K, int E, int align,
                       int32_t* sorted_token_ids, int32_t* expert_ids, int32_t* inv_perm,
                       int32_t* m_sum, int32_t* expert_counts, const uint8_t* x_q,
                       const uint8_t* x_sf, int H, uint8_t* x_perm, uint8_t* x_perm_sf,
                       void* ws, size_t ws_bytes, void* stream);

/* L1 grouped GEMM + SwiGLU + FP8 requant (MegaMoE page 二、阶段 2 and 阶段 3).
 * For every row r < M_sum with e = expert_ids[r] >= 0 and x_r the activation of that row:
 *   gu = dequant(x_r) @ dequant(W13[e])^T   ([2I], fp32 accumulate)
 *   h  = silu(gu[0:I]) * gu[I:2I]
 *   h_q[r] / h_sf: h requantised per 128 along I by the rule of moe_route.
 * The activation comes in one of two forms:
 *   a_is_permuted != 0: a_q = x_perm [U, H] E4M3 (x_r = a_q[r]), a_sf = x_perm_sf tiled (rows U,
 *     slabs H/128), both from moe_permute; sorted_token_ids may be NULL.
 *   a_is_permuted == 0: a_q = x_q [T, H] E4M3 and a_sf = x_sf [T, H/128] UE8M0 in token order, as
 *     moe_route writes them; x_r = a_q[sorted_token_ids[r] / K] (MegaMoE page, 什么时候需要
 *     permute/unpermute, 路径 A: the rows are read through the index, never copied).
 *     sorted_token_ids [U] from moe_permute is required.  The rows' scales are first gathered
 *     into the workspace (tiled), the rows themselves are read by the GEMM with row-gather copies.
 * h_q [U, I] E4M3 out, h_sf tiled (rows U, slabs I/128) out.  Rows with expert_ids = -1 are
 * unspecified. */
moe_status moe_grouped_gemm_l1_swiglu(const uint8_t* a_q, const uint8_t* a_sf, int a_is_permuted,
                                      const int32_t* sorted_token_ids, const int32_t* expert_ids,
                                      const int32_t* m_sum, int T, int K, int H, int I, int E,
                                      int align, moe_weight w13, uint8_t* h_q, uint8_t* h_sf,
                                      void* ws, size_t ws_bytes, void* stream);

/* moe_grouped_gemm_l1_swiglu with the routing weight applied in the L1 epilogue (MegaMoE page
 * 二、阶段 3: the SwiGLU output is silu(gate) * up * topk_weight, then amax -> UE8M0 -> E4M3):
 *   h = (silu(gu[0:I]) * gu[I:2I]) * topk_w[sorted_token_ids[r]]   before the requant.
 * sorted_token_ids [U] and topk_w [T*K] fp32 as produced by moe_permute / moe_route.  The reduce
 * that follows then sums without weights (moe_unpermute_reduce with topk_w = NULL). */
moe_status moe_grouped_gemm_l1_swiglu_weighted(const uint8_t* x_perm, const uint8_t* x_perm_sf,
                                               const int32_t* expert_ids, const int32_t* m_sum,
                                               const int32_t* sorted_token_ids, const float* topk_w,
                                               int T, int K, int H, int I, int E, int align,
                                               moe_weight w13, uint8_t* h_q, uint8_t* h_sf, void* ws,
                                               size_t ws_bytes, void* stream);

/* L2 grouped GEMM (MegaMoE page 二、阶段 4; L2 results are bf16, 阶段 5).
 * For every row r < M_sum with e = expert_ids[r] >= 0:
 *   y_perm[r] = bf16_rne( dequant(h_q[r]) @ dequant(W2[e])^T )   ([H], fp32 accumulate)
 *   h_q [U, I] E4M3, h_sf tiled (rows U, slabs I/128); y_perm [U, H] bf16 out. */
moe_status moe_grouped_gemm_l2(const uint8_t* h_q, const uint8_t* h_sf, const int32_t* expert_ids,
                               const int32_t* m_sum, int T, int K, int H, int I, int E,
                               int align, moe_weight w2, uint16_t* y_perm, void* ws,
                               size_t ws_bytes, void* stream);

/* Both expert GEMMs in one call (MegaMoE page 二、阶段 2-5 as one persistent kernel): the results
 * of moe_grouped_gemm_l1_swiglu (h_q, h_sf) and of moe_grouped_gemm_l2 (y_perm), bit for bit.
 * With MXFP4 weights it is one launch in which an L2 tile starts once every L1 tile
 * of its row block is stored; it needs the full moe_workspace_size() workspace (per-row-block
 * counters that the launch leaves at zero).  With NVFP4 weights the two calls run in turn.
 * Arguments as for the two calls (the L1 input permuted or token-order, as in
 * moe_grouped_gemm_l1_swiglu); h_q/h_sf/y_perm 16-byte aligned. */
moe_status moe_grouped_ffn(const uint8_t* a_q, const uint8_t* a_sf, int a_is_permuted,
                           const int32_t* sorted_token_ids, const int32_t* expert_ids,
                           const int32_t* m_sum, int T, int K, int H, int I, int E, int align,
                           moe_weight w13, moe_weight w2, uint8_t* h_q, uint8_t* h_sf,
                           uint16_t* y_perm, void* ws, size_t ws_bytes, void* stream);

/* Weighted unpermute-reduce (note §9.6 "gather 再讲一遍"; MegaMoE page 阶段 5):
 *   out[t] = bf16_rne( sum_{k=0}^{K-1} topk_w[t,k] * y_perm[inv_perm[t,k]] ), summed in fp32
 *   in k order.  y_perm [>= max(inv_perm)+1, H] bf16, inv_perm [T,K], topk_w [T,K] fp32 or NULL
 *   (plain sum, for weights already applied in L1: MegaMoE page 阶段 5 accumulates the
 *   contributions in float32 without weights), out [T, H] bf16. */
moe_status moe_unpermute_reduce(const uint16_t* y_perm, const int32_t* inv_perm,
                                const float* topk_w, int T, int K, int H, uint16_t* out,
                                void* stream);

/* The whole layer in one call: route -> permute -> L1 -> L2 -> reduce on `stream`, with all
 * intermediates in the workspace (L1 and L2 as in moe_grouped_ffn; up to 32 tokens the reduce
 * runs inside the L2 epilogue, with the same arithmetic as moe_unpermute_reduce).  The optional index outputs (any may be NULL) receive the
 * same values as the individual calls would produce; out [T, H] bf16. */
moe_status moe_forward(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                       const float* e_score_bias, int T, int H, int I, int E, int K, int align,
                       moe_score_fn fn, int renormalize, moe_weight w13, moe_weight w2,
                       uint16_t* out, int32_t* topk_ids, float* topk_w,
                       int32_t* sorted_token_ids, int32_t* expert_ids, int32_t* inv_perm,
                       int32_t* m_sum, void* ws, size_t ws_bytes, void* stream);

/* moe_forward as one launch: the single persistent kernel of page "DeepSeek V4 MegaMoE Kernel
 * 深度解析", 一、架构概览 整体思路 (one launch for the whole layer) and 二、Fused 了什么 (stages 1-5),
 * for small batches: the routing (gate, scores, top-K, FP8 activations), the permute, L1 with
 * SwiGLU and requant, L2 and the weighted reduce run as phases of one cooperative kernel, with two
 * grid-wide barriers between routing, permute and the expert GEMMs.  Same arguments, workspace
 * (moe_workspace_size) and results as moe_forward, bit for bit.  Supported: MXFP4 weights,
 * 1 <= T <= 16, E <= 256, T*K <= 128, align <= 16; other problems return MOE_ERR_UNSUPPORTED
 * (moe_forward covers them).  A barrier wait that runs out is reported as MOE_ERR_TIMEOUT by
 * moe_get_error, with out unspecified.  The calls of one stream must not overlap: the launch
 * starts after the previous one and reuses the workspace's routing scratch.  Like moe_forward it
 * can be captured into a CUDA graph (a cooperative kernel node). */
moe_status moe_forward_single_launch(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                                     const float* e_score_bias, int T, int H, int I, int E, int K,
                                     int align, moe_score_fn fn, int renormalize, moe_weight w13,
                                     moe_weight w2, uint16_t* out, int32_t* topk_ids, float* topk_w,
                                     int32_t* sorted_token_ids, int32_t* expert_ids,
                                     int32_t* inv_perm, int32_t* m_sum, void* ws, size_t ws_bytes,
                                     void* stream);

/* --------------------------------------------------------------------------------------
 * BatchedExperts layout (MegaMoE page, vLLM 的两种 Activation Format and 路径 B: each expert
 * owns a fixed slot of max_tokens rows filled through a boolean mask over the tokens; note
 * "INT8 高吞吐/低延迟 EP 代码梳理" §11.2: the low-latency (E, max_tokens, H) buffer with
 * expert_num_tokens).  Rows of the permuted buffers: U = E * max_tokens, expert e's slot is rows
 * [e * max_tokens, (e + 1) * max_tokens), its first expert_num_tokens[e] rows live, the rest
 * padding.  max_tokens is a power of two in [1, 4096].  Scale tensors are tiled as for the
 * contiguous calls with align = moe_batched_align(T, K, E, max_tokens) (the GEMM row-block height:
 * max_tokens below 16, else min(max_tokens, 64), or min(max_tokens, 128) when T*K > 64*E).
 * max_tokens >= 16 keeps every GEMM row block inside one expert's slot. */
int moe_batched_align(int T, int K, int E, int max_tokens);

/* Workspace bytes of the BatchedExperts calls (zero-filled once before first use). */
moe_status moe_workspace_size_batched(int T, int H, int I, int E, int K, int max_tokens, size_t* bytes);

/* BatchedExperts permute.  With n_e = #(t,k) routed to e:
 *   inv_perm[t,k]          [T, K] out: e * max_tokens + (rank of (t,k) among expert e's pairs
 *                          in ascending t*K+k order)
 *   sorted_token_ids[row]  [U] out: t*K + k of the pair on that row, T*K on padding rows
 *   expert_ids[row]        [U] out: expert of the row, -1 on padding rows
 *   m_sum                  [1] out (device): U
 *   expert_num_tokens      [E] out or NULL: n_e
 *   x_q, x_sf, x_perm, x_perm_sf: as for moe_permute (x_perm [U, H]).
 * A pair that would land past its expert's slot (n_e > max_tokens, possible only when a token
 * names one expert twice or T > max_tokens) is dropped: inv_perm = -1, nothing else written
 * for it, and MOE_ERR_DEVICE_INDEX is recorded.  An id outside [0, E) as for moe_permute. */
moe_status moe_permute_batched(const int32_t* topk_ids, int T, int K, int E, int max_tokens,
                               int32_t* sorted_token_ids, int32_t* expert_ids, int32_t* inv_perm,
                               int32_t* m_sum, int32_t* expert_num_tokens, const uint8_t* x_q,
                               const uint8_t* x_sf, int H, uint8_t* x_perm, uint8_t* x_perm_sf,
                               void* ws, size_t ws_bytes, void* stream);

/* Both expert GEMMs over a BatchedExperts buffer: moe_grouped_ffn's arithmetic on every live row
 * (row i of slot e with i < expert_num_tokens[e], expert e); padding rows of h_q and y_perm are
 * unspecified.  x_perm [U, H] E4M3, x_perm_sf tiled (rows U, slabs H/128); h_q [U, I], h_sf,
 * y_perm [U, H] bf16 out.  expert_num_tokens [E] int32 on the device (a count above max_tokens
 * records MOE_ERR_DEVICE_INDEX).  The row map (expert of each row) is written into the
 * workspace by a small kernel before the GEMMs.  ws: moe_workspace_size_batched(T, H, I, E, K,
 * max_tokens) bytes; T and K only size that workspace (T = max_tokens, K = 1 when the buffer
 * comes from elsewhere). */
moe_status moe_grouped_ffn_batched(const uint8_t* x_perm, const uint8_t* x_perm_sf,
                                   const int32_t* expert_num_tokens, int T, int K, int H, int I, int E,
                                   int max_tokens, moe_weight w13, moe_weight w2, uint8_t* h_q,
                                   uint8_t* h_sf, uint16_t* y_perm, void* ws, size_t ws_bytes,
                                   void* stream);

/* moe_forward over the BatchedExperts layout: route -> moe_permute_batched -> L1 -> L2 ->
 * reduce.  `out` equals moe_forward's bit for bit (each row's arithmetic does not depend on the
 * row it sits on).  Requires T <= max_tokens (an expert receives at most T tokens).  The index
 * outputs (any may be NULL) are those of moe_permute_batched. */
moe_status moe_forward_batched(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                               const float* e_score_bias, int T, int H, int I, int E, int K,
                               int max_tokens, moe_score_fn fn, int renormalize, moe_weight w13,
                               moe_weight w2, uint16_t* out, int32_t* topk_ids, float* topk_w,
                               int32_t* sorted_token_ids, int32_t* expert_ids, int32_t* inv_perm,
                               int32_t* m_sum, int32_t* expert_num_tokens, void* ws, size_t ws_bytes,
                               void* stream);

/* moe_forward with the routing weights applied in the L1 epilogue instead of the reduce (MegaMoE
 * page 二、阶段 3 and 阶段 5): L1 as moe_grouped_gemm_l1_swiglu_weighted, L2 as usual, and the
 * reduce an unweighted fp32 sum.  Same arguments, workspace and index outputs as moe_forward; the
 * output differs from moe_forward's only through the FP8 requant and bf16 roundings of the
 * weighted intermediate values (identical when every routing weight is a power of two). */
moe_status moe_forward_l1_weighted(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                                   const float* e_score_bias, int T, int H, int I, int E, int K,
                                   int align, moe_score_fn fn, int renormalize, moe_weight w13,
                                   moe_weight w2, uint16_t* out, int32_t* topk_ids, float* topk_w,
                                   int32_t* sorted_token_ids, int32_t* expert_ids, int32_t* inv_perm,
                                   int32_t* m_sum, void* ws, size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------------------
 * Tiny-batch path (MegaMoE page, the permute-path table 何时选择什么: with very few tokens,
 * T * topk * 4 <= E, even sorted_token_ids is skipped and each (token, expert) pair is given its
 * own block).  Pair p = t*K + k owns row 16 * p of the permuted buffers; the other 15 rows of its
 * block, and the rows [16 * T * K, U) with U = moe_msum_upper(T, K, E, 16), are padding.  No
 * counting or sorting: the routing launch itself writes the activation rows (each token's FP8
 * row K times) and the index arrays, and the expert GEMMs then run with align = 16, one pair
 * per row block.  Requires T <= 16 and T * K <= E (else MOE_ERR_UNSUPPORTED); meant for
 * T * K * 4 <= E, where two pairs rarely share an expert (a shared expert's weights are read once
 * per pair).
 * ------------------------------------------------------------------------------------ */

/* Routing (as moe_route) plus the tiny-batch layout:
 *   sorted_token_ids [U] out: p on row 16p, T*K elsewhere
 *   expert_ids [U] out: topk_ids[p] on row 16p, -1 elsewhere
 *   inv_perm [T, K] out: 16 * (t*K + k);  m_sum [1] out: 16 * T * K
 *   x_perm [U, H] E4M3 out (row 16p = x_q[t], other rows unwritten), x_perm_sf out, tiled for
 *   align 16 (rows U, slabs H/128).
 * ws as for moe_route.  The index arrays and buffers feed moe_grouped_ffn / the grouped GEMMs
 * with align = 16 and the same T, K, E. */
moe_status moe_route_naive(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                           const float* e_score_bias, int T, int H, int E, int K, moe_score_fn fn,
                           int renormalize, int32_t* topk_ids, float* topk_w, int32_t* sorted_token_ids,
                           int32_t* expert_ids, int32_t* inv_perm, int32_t* m_sum, uint8_t* x_perm,
                           uint8_t* x_perm_sf, void* ws, size_t ws_bytes, void* stream);

/* moe_forward over the tiny-batch layout: two launches (routing with the layout, then L1 + L2
 * with the weighted reduce in the L2 epilogue).  ws: moe_workspace_size(T, H, I, E, K, 16)
 * bytes.  `out` equals moe_forward's (align 16) bit for bit; the optional index outputs are
 * those of moe_route_naive. */
moe_status moe_forward_naive(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                             const float* e_score_bias, int T, int H, int I, int E, int K,
                             moe_score_fn fn, int renormalize, moe_weight w13, moe_weight w2,
                             uint16_t* out, int32_t* topk_ids, float* topk_w,
                             int32_t* sorted_token_ids, int32_t* expert_ids, int32_t* inv_perm,
                             int32_t* m_sum, void* ws, size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------------------
 * INT8 (W8A8) variant (note "INT8 高吞吐/低延迟 EP 代码梳理": §2 INT8 dispatch with quant_dtype
 * int8, §3.1 INT8 with channel-wise weights, §11.6.2 the high-throughput INT8 path quantises the
 * activations per token).  Weights: MOE_W_INT8 (int8 codes, fp32 scale per output channel).
 * Activations, both the layer input and the SwiGLU output: int8 codes with one fp32 scale per row,
 *   amax = max |x| over the row, inv = fp32(127 / amax), s = fp32(amax / 127),
 *   q = clamp(rint(fp32(x * inv)), -127, 127)   (rint: to nearest, ties to even),
 * every division correctly rounded; a zero row gives q = 0, s = 0 (rows with 0 < amax <
 * 127 / FLT_MAX are not supported).  The expert GEMMs are integer dot products of the codes (run on
 * the 16-bit tensor cores with fp16 operands, summed in fp32) times the row scale times the channel
 * scale; L1 rounds silu(gate) * up to bf16 and then quantises each row of h.  Routing, the permute
 * and the reduce are those of the FP4 path; the index arrays have the same meaning.
 * With MOE_W_INT8_B256 weights (both w13 and w2; H and I multiples of 256) every activation scale
 * is per row and 256-column group instead ([rows, cols/256], each group quantised by the rule
 * above), and the GEMMs sum, over the 256-deep blocks kb of the reduction, the integer dot product
 * of the block times the row's group scale of kb times the weight block's scale (fp32 sums); the
 * x_s / h_s arguments below are then [T, H/256] / [U, I/256].
 * ------------------------------------------------------------------------------------ */

/* Workspace bytes of the INT8 calls (moe_workspace_size's layout plus the INT8 row scales and a
 * bf16 [U, I] h); zero-filled once before first use, as moe_workspace_size's. */
moe_status moe_workspace_size_i8(int T, int H, int I, int E, int K, int align, size_t* bytes);

/* Per-row int8 quantisation by the rule above: x [rows, cols] bf16 -> x_q [rows, cols] int8,
 * x_s [rows] fp32.  cols a multiple of 128; x and x_q 16-byte aligned.  No workspace. */
moe_status moe_act_quant_i8(const uint16_t* x, int rows, int cols, int8_t* x_q, float* x_s, void* stream);

/* The same rule per 256-column group (the activations of the MOE_W_INT8_B256 layer): x [rows, cols]
 * bf16 -> x_q [rows, cols] int8, x_s [rows, cols/256] fp32.  cols a multiple of 256. */
moe_status moe_act_quant_i8_b256(const uint16_t* x, int rows, int cols, int8_t* x_q, float* x_s, void* stream);

/* L1 + SwiGLU + per-row int8 requant.  The activation rows are read in token order and gathered
 * through sorted_token_ids (row r of the permuted layout is token sorted_token_ids[r] / K):
 *   x_q [T, H] int8, x_s [T] fp32 (moe_act_quant_i8 of the layer input)
 *   sorted_token_ids, expert_ids [U], m_sum [1]: moe_permute's outputs for (T, K, E, align)
 *   w13: MOE_W_INT8, N = 2I, Kd = H, pair = 2 (tscale = [E, 2I] channel scales)
 *   h_q [U, I] int8 out, h_s [U] fp32 out: for rows r < M_sum with expert_ids[r] >= 0,
 *     h = bf16(silu(g) * u), g / u = (integer dot of x_q row and W13 row) * x_s * channel scale,
 *     then the per-row rule; other rows unspecified.
 * ws: moe_workspace_size_i8 bytes (fp16 operand rows, row scales, bf16 h). */
moe_status moe_grouped_gemm_l1_swiglu_i8(const int8_t* x_q, const float* x_s, const int32_t* sorted_token_ids,
                                         const int32_t* expert_ids, const int32_t* m_sum, int T, int K, int H,
                                         int I, int E, int align, moe_weight w13, int8_t* h_q, float* h_s,
                                         void* ws, size_t ws_bytes, void* stream);

/* L2: y_perm[r] = bf16((integer dot of h_q row r and W2 row j) * h_s[r] * channel scale j) for rows
 * r < M_sum with expert_ids[r] >= 0 (others unspecified).  h_q [U, I] int8, h_s [U] fp32; w2:
 * MOE_W_INT8, N = H, Kd = I, pair = 1; y_perm [U, H] bf16; ws: moe_workspace_size_i8 bytes. */
moe_status moe_grouped_gemm_l2_i8(const int8_t* h_q, const float* h_s, const int32_t* expert_ids,
                                  const int32_t* m_sum, int T, int K, int H, int I, int E, int align,
                                  moe_weight w2, uint16_t* y_perm, void* ws, size_t ws_bytes, void* stream);

/* The INT8 layer: moe_route (without the FP8 activation output) -> moe_act_quant_i8 -> moe_permute
 * (indices only) -> INT8 L1 (h requantised per row) -> INT8 L2 -> the topk-weighted reduce, inside
 * the L2 epilogue up to 32 tokens.  Arguments and optional index outputs as moe_forward's; w13, w2
 * MOE_W_INT8; ws: moe_workspace_size_i8 bytes. */
moe_status moe_forward_i8(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                          const float* e_score_bias, int T, int H, int I, int E, int K, int align,
                          moe_score_fn fn, int renormalize, moe_weight w13, moe_weight w2, uint16_t* out,
                          int32_t* topk_ids, float* topk_w, int32_t* sorted_token_ids, int32_t* expert_ids,
                          int32_t* inv_perm, int32_t* m_sum, void* ws, size_t ws_bytes, void* stream);

/* The INT8 layer over the BatchedExperts layout (note "INT8 高吞吐/低延迟 EP 代码梳理" §2: the INT8
 * dispatch flag is passed to the low-latency path, whose experts receive fixed [max_tokens] slots,
 * §11.2): moe_forward_i8 with moe_permute_batched's layout (expert e's rows at e * max_tokens, in
 * token order, unused rows padding).  `out` equals moe_forward_i8's bit for bit (each row's
 * arithmetic does not depend on the row it sits on).  Requires T <= max_tokens; max_tokens a power
 * of two in [1, 4096]; ws: moe_workspace_size_batched_i8 bytes; the optional index outputs are
 * those of moe_permute_batched (expert_num_tokens [E]). */
moe_status moe_workspace_size_batched_i8(int T, int H, int I, int E, int K, int max_tokens, size_t* bytes);
moe_status moe_forward_batched_i8(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                                  const float* e_score_bias, int T, int H, int I, int E, int K,
                                  int max_tokens, moe_score_fn fn, int renormalize, moe_weight w13,
                                  moe_weight w2, uint16_t* out, int32_t* topk_ids, float* topk_w,
                                  int32_t* sorted_token_ids, int32_t* expert_ids, int32_t* inv_perm,
                                  int32_t* m_sum, int32_t* expert_num_tokens, void* ws, size_t ws_bytes,
                                  void* stream);

/* Self-test of the device failure path (no counterpart in the method's description): launches one
 * bounded wait that nothing can satisfy, through the primitives the hot path uses.  mode 0: a
 * counter that is never incremented (word 32 of the workspace's reserved first 256 bytes, which
 * stays zero), as the L2-after-L1 waits of the expert FFN; mode 1: an mbarrier phase that never
 * completes, as the pipeline waits.  After its cycle budget (~2 s) the wait gives up, records
 * MOE_ERR_TIMEOUT in the status word and the kernel returns: moe_get_error then reports it, and
 * the context stays usable.  No fault and no unbounded wait is involved. */
moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, int mode, void* stream);

/* Synchronises `stream`, returns the device status word recorded in `ws` through
 * *device_status (MOE_OK if none) and clears it.  The return value reports host errors. */
moe_status moe_get_error(void* ws, void* stream, moe_status* device_status);

/* Static string for a status code. */
const char* moe_status_str(moe_status s);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
