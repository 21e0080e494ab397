// C ABI of the MoE layer (declarations and contracts in include/moe.h).
// Host-side validation, workspace layout, and launches on the caller's stream.
#include <cstring>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

using namespace moe;

namespace {

constexpr size_t kAlign = 256;
inline size_t up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline cudaStream_t S(void* s) { return static_cast<cudaStream_t>(s); }


bool dims_ok(int T, int H, int I, int E, int K, int align) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || K <= 0 || K > E || K > 32) return false;
  if (H % 128 || I % 128) return false;
  if (align < 1 || align > 256 || (align & (align - 1))) return false;
  return true;
}

// Workspace layout for one problem size.  Offsets are relative to the workspace base.
struct WsLayout {
  size_t status = 0;
  size_t perm = 0, partial = 0, partial_bytes = 0;
  size_t topk_ids = 0, topk_w = 0, x_q = 0, x_sf = 0, sorted = 0, expert_ids = 0, inv_perm = 0, m_sum = 0;
  size_t x_perm = 0, x_perm_sf = 0, h_q = 0, h_sf = 0, y = 0, xb = 0, tickets = 0, sched = 0, counts = 0;
  size_t total = 0;
};

// U: rows of the permuted buffers (moe_msum_upper for the contiguous layout, E * max_tokens for
// the BatchedExperts layout).
WsLayout layout_rows(int T, int H, int I, int E, int K, int align, size_t U) {
  WsLayout L;
  size_t off = kAlign;                             // [0, 256): status word
  L.perm = off;       off = up(off + permute_scratch_bytes(T, K, E));   // permute chunk counts
  L.partial = off;
  L.partial_bytes = route_scratch_bytes(T, H, E);
  off = up(off + L.partial_bytes);
  L.topk_ids = off;   off = up(off + static_cast<size_t>(T) * K * 4);
  L.topk_w = off;     off = up(off + static_cast<size_t>(T) * K * 4);
  L.x_q = off;        off = up(off + static_cast<size_t>(T) * H);
  L.x_sf = off;       off = up(off + static_cast<size_t>(T) * (H / 128));
  L.sorted = off;     off = up(off + U * 4);
  L.expert_ids = off; off = up(off + U * 4);
  L.inv_perm = off;   off = up(off + static_cast<size_t>(T) * K * 4);
  L.m_sum = off;      off = up(off + 4);
  L.x_perm = off;     off = up(off + U * H);
  L.x_perm_sf = off;  off = up(off + moe_act_sf_tiled_bytes(static_cast<int>(U), H / 128, align));
  L.h_q = off;        off = up(off + U * I);
  L.h_sf = off;       off = up(off + moe_act_sf_tiled_bytes(static_cast<int>(U), I / 128, align));
  L.y = off;          off = up(off + U * H * 2);
  L.xb = off;         off = up(off + U * (H > I ? H : I) * 2);   // bf16 activation rows (NVFP4 GEMMs)
  L.tickets = off;    off = up(off + static_cast<size_t>(T) * ((H + 255) / 256) * 2 * 4);   // fused reduce
  L.sched = off;      off = up(off + gemm_sched_words(static_cast<int>(U), align) * 4);   // GEMM work counters
  L.counts = off;     off = up(off + static_cast<size_t>(E) * 4);                     // tokens per expert
  L.total = off;
  return L;
}

WsLayout layout(int T, int H, int I, int E, int K, int align) {
  return layout_rows(T, H, I, E, K, align, moe_msum_upper(T, K, E, align));
}

// BatchedExperts slot size: a power of two, at most kMaxSlot rows.
constexpr int kMaxSlot = 4096;
bool slot_ok(int max_tokens) {
  return max_tokens >= 1 && max_tokens <= kMaxSlot && (max_tokens & (max_tokens - 1)) == 0;
}
// Alignment the GEMMs and the scale tiling see for a slot size, i.e. their row-block height.
// Below 16 rows a 16-row block spans several slots (the GEMM walks each block's experts).  From 16
// rows on the block stays inside one slot: 64 rows when an expert receives at most 64 tokens on
// average (deeper TMA ring per SM for the weight stream; a slot's blocks past its tokens are
// skipped), else 128 (one block per expert's rows, weights read once).
int slot_align(int T, int K, int E, int max_tokens) {
  if (max_tokens < 16) return max_tokens;
  const int cap = static_cast<long long>(T) * K > 64LL * E ? 128 : 64;
  return max_tokens < cap ? max_tokens : cap;
}
size_t slot_rows(int E, int max_tokens) { return static_cast<size_t>(E) * max_tokens; }

// moe_forward folds the unpermute-reduce into the L2 epilogue up to this many tokens.  With many
// tokens per row block one epilogue warp would reduce tokens one after another; the separate
// reduce kernel is faster there.
constexpr int kFusedReduceMaxTokens = 32;

inline uint32_t* status_of(void* ws) { return static_cast<uint32_t*>(ws); }
inline moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// A packed weight of logical shape [E, N, Kd] with the given pairing.
bool weight_ok(const moe_weight& w, int E, int N, int Kd, int pair) {
  if (!w.packed || !aligned(w.packed, 32)) return false;
  if (w.E != E || w.N != N || w.Kd != Kd || w.pair != pair) return false;
  if (w.fmt == MOE_W_NVFP4) return w.tscale != nullptr;
  return w.fmt == MOE_W_MXFP4;
}

// An INT8 weight (the INT8 calls take no other format, and the FP4 calls no INT8 weight).
bool weight_ok_i8(const moe_weight& w, int E, int N, int Kd, int pair) {
  if (!w.packed || !aligned(w.packed, 32) || !w.tscale || !aligned(w.tscale, 16)) return false;
  if (w.fmt == MOE_W_INT8_B256 && (N % 256 || Kd % 256)) return false;
  return (w.fmt == MOE_W_INT8 || w.fmt == MOE_W_INT8_B256) && w.E == E && w.N == N && w.Kd == Kd && w.pair == pair;
}

// Scales per activation row of an INT8 operand with `cols` columns: one, or one per 256 columns.
inline int i8_row_scales(bool block, int cols) { return block ? cols / 256 : 1; }

// INT8 variant: the common layout (its x_q, h_q and xb regions hold the int8 token rows, the int8 h
// and the fp16 operand rows) plus the per-row scales and the bf16 h between L1 and its quantisation.
struct I8Layout {
  WsLayout L;
  size_t x_s = 0, a_s = 0, h_s = 0, hb = 0, total = 0;
};

// U: rows of the permuted buffers (0: moe_msum_upper for the contiguous layout).
I8Layout layout_i8(int T, int H, int I, int E, int K, int align, size_t U = 0) {
  if (U == 0) U = moe_msum_upper(T, K, E, align);
  I8Layout r;
  r.L = layout_rows(T, H, I, E, K, align, U);
  size_t off = r.L.total;
  // scale regions sized for the block format too (a scale per row and 256-column group)
  const size_t nh = H >= 256 ? static_cast<size_t>(H) / 256 : 1, ni = I >= 256 ? static_cast<size_t>(I) / 256 : 1;
  r.x_s = off;  off = up(off + static_cast<size_t>(T) * nh * 4);            // token scales
  r.a_s = off;  off = up(off + U * (nh > ni ? nh : ni) * 4);                 // scales of the GEMM operand rows
  r.h_s = off;  off = up(off + U * ni * 4);                                  // h scales (forward)
  r.hb = off;   off = up(off + U * I * 2);                     // bf16 h
  r.total = off;
  return r;
}

}  // namespace

extern "C" {

size_t moe_msum_upper(int T, int K, int E, int align) {
  if (T < 0 || K < 0 || E < 0 || align < 1) return 0;
  return static_cast<size_t>(T) * K + static_cast<size_t>(E) * (align - 1);
}

int moe_act_sf_block_rows(int align) { return align >= 1 ? act_sf_block_rows(align) : 0; }

size_t moe_act_sf_tiled_bytes(int rows, int slabs, int align) {
  if (rows < 0 || slabs <= 0 || align < 1) return 0;
  return act_sf_bytes(rows, slabs, act_sf_block_rows(align));
}

moe_status moe_act_sf_untile_host(const uint8_t* tiled, int rows, int slabs, int align, uint8_t* out) {
  if (!tiled || !out || rows < 0 || slabs <= 0 || align < 1) return MOE_ERR_INVALID_ARG;
  const int bt = act_sf_block_rows(align), nb = act_sf_blocks(rows, bt);
  for (int r = 0; r < rows; ++r)
    for (int s = 0; s < slabs; ++s) out[static_cast<size_t>(r) * slabs + s] = tiled[act_sf_offset(bt, nb, r, s)];
  return MOE_OK;
}

moe_status moe_act_sf_tile_host(const uint8_t* plain, int rows, int slabs, int align, uint8_t* tiled) {
  if (!tiled || !plain || rows < 0 || slabs <= 0 || align < 1) return MOE_ERR_INVALID_ARG;
  const int bt = act_sf_block_rows(align), nb = act_sf_blocks(rows, bt);
  memset(tiled, 127, act_sf_bytes(rows, slabs, bt));
  for (int r = 0; r < rows; ++r)
    for (int s = 0; s < slabs; ++s) tiled[act_sf_offset(bt, nb, r, s)] = plain[static_cast<size_t>(r) * slabs + s];
  return MOE_OK;
}

size_t moe_weight_packed_bytes(moe_wfmt fmt, int E, int N, int Kd, int pair) {
  if (E <= 0 || N <= 0 || Kd <= 0 || Kd % 128 || (pair != 1 && pair != 2)) return 0;
  if (pair == 2 ? N % 256 : N % 128) return 0;
  if (fmt == MOE_W_MXFP4) return packed_weight_bytes(E, N, Kd, pair);
  if (fmt == MOE_W_NVFP4) return packed_nv_weight_bytes(E, N, Kd, pair);
  if (fmt == MOE_W_INT8 || fmt == MOE_W_INT8_B256) return packed_i8_weight_bytes(E, N, Kd, pair);
  return 0;
}

moe_status moe_pack_weights(moe_wfmt fmt, const uint8_t* q, const uint8_t* sf, int E, int N, int Kd, int pair,
                            uint8_t* packed, void* stream) {
  if (!q || !packed || E <= 0 || N <= 0 || Kd <= 0 || Kd % 128) return MOE_ERR_INVALID_ARG;
  if ((pair != 1 && pair != 2) || (pair == 2 ? N % 256 : N % 128)) return MOE_ERR_INVALID_ARG;
  if (fmt == MOE_W_INT8 || fmt == MOE_W_INT8_B256) {
    if (!aligned(q, 16) || !aligned(packed, 16)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_pack_i8(reinterpret_cast<const int8_t*>(q), E, N, Kd, pair, packed, S(stream)));
  }
  if (!sf) return MOE_ERR_INVALID_ARG;
  if (fmt == MOE_W_MXFP4) return cuda_status(launch_pack_mx(q, sf, E, N, Kd, pair, packed, S(stream)));
  if (fmt == MOE_W_NVFP4) return cuda_status(launch_pack_nv(q, sf, E, N, Kd, pair, packed, S(stream)));
  return MOE_ERR_INVALID_ARG;
}

moe_status moe_workspace_size(int T, int H, int I, int E, int K, int align, size_t* bytes) {
  if (!bytes || !dims_ok(T, H, I, E, K, align)) return MOE_ERR_INVALID_ARG;
  *bytes = layout(T, H, I, E, K, align).total;
  return MOE_OK;
}

moe_status moe_route(const uint16_t* hidden, const float* w_gate, const float* gate_bias, const float* e_score_bias,
                     int T, int H, int E, int K, moe_score_fn fn, int renormalize, float* logits_out,
                     int32_t* topk_ids, float* topk_w, uint8_t* x_q, uint8_t* x_sf, void* ws, size_t ws_bytes,
                     void* stream) {
  if (!dims_ok(T, H, 128, E, K, 1) || E > 1024) return MOE_ERR_INVALID_ARG;
  if (!hidden || !w_gate || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (fn != MOE_SCORE_SOFTMAX && fn != MOE_SCORE_SQRT_SOFTPLUS) return MOE_ERR_INVALID_ARG;
  if ((x_q == nullptr) != (x_sf == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(w_gate, 16)) return MOE_ERR_INVALID_ARG;
  if (x_q && !aligned(x_q, 4)) return MOE_ERR_INVALID_ARG;
  if (!ws) return MOE_ERR_WORKSPACE;
  const size_t poff = up(kAlign + permute_scratch_bytes(T, K, E));   // as in layout()
  const size_t need = poff + route_scratch_bytes(T, H, E);
  if (ws_bytes < need) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  void* scratch = static_cast<char*>(ws) + poff;
  return cuda_status(launch_route(hidden, w_gate, gate_bias, e_score_bias, T, H, E, K, static_cast<int>(fn),
                                  renormalize, logits_out, topk_ids, topk_w, x_q, x_sf, scratch, status_of(ws),
                                  S(stream)));
}

}  // extern "C"

// Routing plus the tiny-batch layout in one launch: pair p = t*K + k owns row kNaiveRows * p of
// [U, H] buffers with U = moe_msum_upper(T, K, E, kNaiveRows) (T*K <= E makes T*K*kNaiveRows fit).
static moe_status route_naive_common(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                                     const float* e_score_bias, int T, int H, int E, int K, moe_score_fn fn,
                                     int renormalize, int32_t* topk_ids, float* topk_w, int32_t* sorted_token_ids,
                                     int32_t* expert_ids, int32_t* inv_perm, int32_t* m_sum, uint8_t* x_perm,
                                     uint8_t* x_perm_sf, void* ws, size_t ws_bytes, void* stream) {
  if (!dims_ok(T, H, 128, E, K, kNaiveRows) || E > 1024) return MOE_ERR_INVALID_ARG;
  if (T > 16 || T * K > E) return MOE_ERR_UNSUPPORTED;
  if (!hidden || !w_gate || !topk_ids || !topk_w || !sorted_token_ids || !expert_ids || !inv_perm || !m_sum ||
      !x_perm || !x_perm_sf)
    return MOE_ERR_INVALID_ARG;
  if (fn != MOE_SCORE_SOFTMAX && fn != MOE_SCORE_SQRT_SOFTPLUS) return MOE_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(w_gate, 16) || !aligned(x_perm, 16)) return MOE_ERR_INVALID_ARG;
  if (!ws) return MOE_ERR_WORKSPACE;
  const size_t poff = up(kAlign + permute_scratch_bytes(T, K, E));   // as in layout()
  if (ws_bytes < poff + route_scratch_bytes(T, H, E)) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  NaiveLayout nv;
  nv.sorted = sorted_token_ids;
  nv.eids = expert_ids;
  nv.inv = inv_perm;
  nv.m_sum = m_sum;
  nv.xp = x_perm;
  nv.xp_sf = x_perm_sf;
  nv.U = static_cast<int>(moe_msum_upper(T, K, E, kNaiveRows));
  nv.sf_nb = act_sf_blocks(nv.U, kNaiveRows);
  void* scratch = static_cast<char*>(ws) + poff;
  return cuda_status(launch_route(hidden, w_gate, gate_bias, e_score_bias, T, H, E, K, static_cast<int>(fn),
                                  renormalize, nullptr, topk_ids, topk_w, nullptr, nullptr, scratch, status_of(ws),
                                  S(stream), &nv));
}

extern "C" {

moe_status moe_route_naive(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                           const float* e_score_bias, int T, int H, int E, int K, moe_score_fn fn, int renormalize,
                           int32_t* topk_ids, float* topk_w, int32_t* sorted_token_ids, int32_t* expert_ids,
                           int32_t* inv_perm, int32_t* m_sum, uint8_t* x_perm, uint8_t* x_perm_sf, void* ws,
                           size_t ws_bytes, void* stream) {
  return route_naive_common(hidden, w_gate, gate_bias, e_score_bias, T, H, E, K, fn, renormalize, topk_ids, topk_w,
                            sorted_token_ids, expert_ids, inv_perm, m_sum, x_perm, x_perm_sf, ws, ws_bytes, stream);
}

}  // extern "C"

// slot 0: contiguous layout padded to align; slot > 0: BatchedExperts (align = slot_align(slot)).
static moe_status permute_common(const int32_t* topk_ids, int T, int K, int E, int align, int slot,
                                 int32_t* sorted_token_ids, int32_t* expert_ids, int32_t* inv_perm, int32_t* m_sum,
                                 int32_t* expert_counts, const uint8_t* x_q, const uint8_t* x_sf, int H,
                                 uint8_t* x_perm, uint8_t* x_perm_sf, void* ws, size_t ws_bytes, void* stream) {
  if (T < 0 || K <= 0 || E <= 0 || K > E || align < 1 || align > 256 || (align & (align - 1)))
    return MOE_ERR_INVALID_ARG;
  if (E > 1024) return MOE_ERR_UNSUPPORTED;
  if (!topk_ids || !sorted_token_ids || !expert_ids || !inv_perm || !m_sum) return MOE_ERR_INVALID_ARG;
  // rows and scales (x_q, x_sf, x_perm, x_perm_sf), the scales alone (x_sf, x_perm_sf), or neither
  const bool copy = x_perm != nullptr, scales = x_perm_sf != nullptr;
  if (copy != (x_q != nullptr) || scales != (x_sf != nullptr) || (copy && !scales)) return MOE_ERR_INVALID_ARG;
  if (scales && (H <= 0 || H % 128)) return MOE_ERR_INVALID_ARG;
  if (copy && (!aligned(x_q, 16) || !aligned(x_perm, 16))) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < kAlign + permute_scratch_bytes(T, K, E)) return MOE_ERR_WORKSPACE;
  const size_t U = slot ? slot_rows(E, slot) : moe_msum_upper(T, K, E, align);
  int32_t* scratch = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kAlign);   // layout().perm
  return cuda_status(launch_permute(topk_ids, T, K, E, align, static_cast<int>(U), sorted_token_ids, expert_ids,
                                    inv_perm, m_sum, expert_counts, x_q, x_sf, H, x_perm, x_perm_sf,
                                    status_of(ws), scratch, S(stream), slot));
}

extern "C" {

moe_status moe_permute(const int32_t* topk_ids, int T, int K, int E, int align, int32_t* sorted_token_ids,
                       int32_t* expert_ids, int32_t* inv_perm, int32_t* m_sum, int32_t* expert_counts,
                       const uint8_t* x_q, const uint8_t* x_sf, int H, uint8_t* x_perm, uint8_t* x_perm_sf,
                       void* ws, size_t ws_bytes, void* stream) {
  return permute_common(topk_ids, T, K, E, align, 0, sorted_token_ids, expert_ids, inv_perm, m_sum, expert_counts,
                        x_q, x_sf, H, x_perm, x_perm_sf, ws, ws_bytes, stream);
}

int moe_batched_align(int T, int K, int E, int max_tokens) {
  if (T < 0 || K <= 0 || E <= 0 || !slot_ok(max_tokens)) return 0;
  return slot_align(T, K, E, max_tokens);
}

moe_status moe_workspace_size_batched(int T, int H, int I, int E, int K, int max_tokens, size_t* bytes) {
  if (!bytes || !slot_ok(max_tokens) || !dims_ok(T, H, I, E, K, slot_align(T, K, E, max_tokens))) return MOE_ERR_INVALID_ARG;
  *bytes = layout_rows(T, H, I, E, K, slot_align(T, K, E, max_tokens), slot_rows(E, max_tokens)).total;
  return MOE_OK;
}

moe_status moe_permute_batched(const int32_t* topk_ids, int T, int K, int E, int max_tokens,
                               int32_t* sorted_token_ids, int32_t* expert_ids, int32_t* inv_perm, int32_t* m_sum,
                               int32_t* expert_num_tokens, const uint8_t* x_q, const uint8_t* x_sf, int H,
                               uint8_t* x_perm, uint8_t* x_perm_sf, void* ws, size_t ws_bytes, void* stream) {
  if (!slot_ok(max_tokens)) return MOE_ERR_INVALID_ARG;
  return permute_common(topk_ids, T, K, E, slot_align(T, K, E, max_tokens), max_tokens, sorted_token_ids, expert_ids,
                        inv_perm, m_sum, expert_num_tokens, x_q, x_sf, H, x_perm, x_perm_sf, ws, ws_bytes, stream);
}

// Launch description of one MXFP4 GEMM (L1: x = x_perm [U, H] against W13; L2: x = h [U, I] against W2).
static GemmLaunch mx_launch(bool l1, const uint8_t* x, const uint8_t* x_sf, const int32_t* expert_ids,
                            const int32_t* m_sum, int H, int I, int E, int align, size_t U, const moe_weight& w,
                            uint8_t* h_q, uint8_t* h_sf, uint16_t* y, void* ws) {
  GemmLaunch L;
  L.w = w.packed;
  L.x = x;
  L.x_sf = x_sf;
  L.expert_ids = expert_ids;
  L.m_sum = m_sum;
  L.h_q = h_q;
  L.h_sf = h_sf;
  L.y = y;
  L.status = status_of(ws);
  L.E = E;
  L.w_rows = l1 ? 2 * I : H;
  L.Kd = l1 ? H : I;
  L.I = I;
  L.U = static_cast<int>(U);
  L.align = align;
  return L;
}

// gather_ids non-null (L1 only): x = token-order activation [T, H] and x_sf its plain scales
// [T, H/128]; permuted row r reads token gather_ids[r] / K (the MXFP4 path first writes the
// permuted rows' tiled scales into the workspace; the rows themselves are gathered by the GEMM).
// Launch description of one NVFP4 GEMM (bf16 operand rows xb [U, Kd]).
static NvLaunch nv_launch(bool l1, const uint16_t* xb, const int32_t* expert_ids, const int32_t* m_sum, int H, int I,
                          int E, int align, size_t U, const moe_weight& w, uint8_t* h_q, uint8_t* h_sf, uint16_t* y,
                          void* ws) {
  NvLaunch N;
  N.w = w.packed;
  N.tscale = w.tscale;
  N.xb = xb;
  N.expert_ids = expert_ids;
  N.m_sum = m_sum;
  N.h_q = h_q;
  N.h_sf = h_sf;
  N.y = y;
  N.status = status_of(ws);
  N.E = E;
  N.w_rows = l1 ? 2 * I : H;
  N.Kd = l1 ? H : I;
  N.I = I;
  N.U = static_cast<int>(U);
  N.align = align;
  return N;
}

static moe_status gemm_common(bool l1, const uint8_t* x, const uint8_t* x_sf, const int32_t* expert_ids,
                              const int32_t* m_sum, int T, int K, int H, int I, int E, int align,
                              const moe_weight& w, uint8_t* h_q, uint8_t* h_sf, uint16_t* y, void* ws,
                              size_t ws_bytes, void* stream, const FusedReduce* red = nullptr, size_t rows = 0,
                              const int32_t* row_ids = nullptr, const float* row_w = nullptr,
                              const int32_t* gather_ids = nullptr, const int32_t* gather_inv = nullptr) {
  if (!dims_ok(T, H, I, E, K, align)) return MOE_ERR_INVALID_ARG;
  if (!x || !x_sf || !expert_ids || !m_sum) return MOE_ERR_INVALID_ARG;
  if (gather_ids && !l1) return MOE_ERR_INVALID_ARG;
  if (!(l1 ? weight_ok(w, E, 2 * I, H, 2) : weight_ok(w, E, H, I, 1))) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || (!gather_ids && !aligned(x_sf, 16))) return MOE_ERR_INVALID_ARG;
  if (l1 && (!h_q || !h_sf)) return MOE_ERR_INVALID_ARG;
  if (!l1 && (!y || !aligned(y, 16))) return MOE_ERR_INVALID_ARG;
  if ((row_ids == nullptr) != (row_w == nullptr) || (!l1 && row_w)) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < kAlign) return MOE_ERR_WORKSPACE;
  const size_t U = rows ? rows : moe_msum_upper(T, K, E, align);
  if (U == 0) return MOE_OK;
  if (w.fmt == MOE_W_NVFP4) {
    // bf16 copy of the activation rows in the workspace, then the bf16 MMA path
    const WsLayout Lw = layout_rows(T, H, I, E, K, align, U);
    if (ws_bytes < Lw.total) return MOE_ERR_WORKSPACE;
    uint16_t* xb = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + Lw.xb);
    const int Kd = l1 ? H : I;
    // token-order rows with the pairs' row positions at hand: one pass per token
    cudaError_t err =
        (gather_ids && gather_inv)
            ? launch_act_to_bf16_tokens(x, x_sf, gather_inv, T, K, static_cast<int>(U), Kd, xb, S(stream))
            : launch_act_to_bf16(x, x_sf, expert_ids, m_sum, static_cast<int>(U), Kd, align, xb, S(stream), gather_ids,
                                 K, T);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    NvLaunch N = nv_launch(l1, xb, expert_ids, m_sum, H, I, E, align, U, w, h_q, h_sf, y, ws);
    if (red) N.red = *red;
    N.row_ids = row_ids;
    N.row_w = row_w;
    return cuda_status(launch_gemm_nv(N, l1, S(stream)));
  }
  const WsLayout Lw = layout_rows(T, H, I, E, K, align, U);
  if (ws_bytes < Lw.total) return MOE_ERR_WORKSPACE;
  const uint8_t* sf = x_sf;
  if (gather_ids) {
    // the permuted rows' scales, tiled for the GEMM, into the workspace
    uint8_t* psf = reinterpret_cast<uint8_t*>(static_cast<char*>(ws) + Lw.x_perm_sf);
    if (launch_permute_act_sf(gather_ids, K, expert_ids, m_sum, static_cast<int>(U), T, x_sf, H / 128, align, psf,
                              S(stream)) != cudaSuccess)
      return MOE_ERR_CUDA;
    sf = psf;
  }
  GemmLaunch L = mx_launch(l1, x, sf, expert_ids, m_sum, H, I, E, align, U, w, h_q, h_sf, y, ws);
  if (red) L.red = *red;
  L.row_ids = row_ids;
  L.row_w = row_w;
  if (gather_ids) {
    L.gather_ids = gather_ids;
    L.gather_k = K;
    L.gather_rows = T;
  }
  uint32_t* sched = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + Lw.sched);
  return cuda_status(launch_gemm(L, l1, sched, S(stream)));
}

moe_status moe_grouped_gemm_l1_swiglu(const uint8_t* a_q, const uint8_t* a_sf, int a_is_permuted,
                                      const int32_t* sorted_token_ids, const int32_t* expert_ids,
                                      const int32_t* m_sum, int T, int K, int H, int I, int E, int align,
                                      moe_weight w13, uint8_t* h_q, uint8_t* h_sf, void* ws, size_t ws_bytes,
                                      void* stream) {
  if (!a_is_permuted && !sorted_token_ids) return MOE_ERR_INVALID_ARG;
  return gemm_common(true, a_q, a_sf, expert_ids, m_sum, T, K, H, I, E, align, w13, h_q, h_sf, nullptr, ws,
                     ws_bytes, stream, nullptr, 0, nullptr, nullptr, a_is_permuted ? nullptr : sorted_token_ids);
}

moe_status moe_grouped_gemm_l1_swiglu_weighted(const uint8_t* x_perm, const uint8_t* x_perm_sf,
                                               const int32_t* expert_ids, const int32_t* m_sum,
                                               const int32_t* sorted_token_ids, const float* topk_w, int T, int K,
                                               int H, int I, int E, int align, moe_weight w13, uint8_t* h_q,
                                               uint8_t* h_sf, void* ws, size_t ws_bytes, void* stream) {
  if (!sorted_token_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  return gemm_common(true, x_perm, x_perm_sf, expert_ids, m_sum, T, K, H, I, E, align, w13, h_q, h_sf, nullptr, ws,
                     ws_bytes, stream, nullptr, 0, sorted_token_ids, topk_w);
}

moe_status moe_grouped_gemm_l2(const uint8_t* h_q, const uint8_t* h_sf, const int32_t* expert_ids,
                               const int32_t* m_sum, int T, int K, int H, int I, int E, int align, moe_weight w2,
                               uint16_t* y_perm, void* ws, size_t ws_bytes, void* stream) {
  return gemm_common(false, h_q, h_sf, expert_ids, m_sum, T, K, H, I, E, align, w2, nullptr, nullptr, y_perm, ws,
                     ws_bytes, stream);
}

// L1 + SwiGLU + requant and L2.  MXFP4: one launch (L2 tiles start as soon as the
// h rows of their block are stored).  NVFP4: the two GEMM calls one after the other.
static moe_status ffn_common(const uint8_t* x_perm, const uint8_t* x_perm_sf, const int32_t* expert_ids,
                             const int32_t* m_sum, int T, int K, int H, int I, int E, int align, const moe_weight& w13,
                             const moe_weight& w2, uint8_t* h_q, uint8_t* h_sf, uint16_t* y, void* ws,
                             size_t ws_bytes, void* stream, const FusedReduce* red, size_t rows = 0,
                             const int32_t* row_ids = nullptr, const float* row_w = nullptr,
                             const int32_t* slot_counts = nullptr, int slot = 0,
                             const int32_t* gather_ids = nullptr, const int32_t* gather_inv = nullptr) {
  if (w13.fmt != MOE_W_MXFP4 || w2.fmt != MOE_W_MXFP4) {
    // NVFP4: the two calls in turn.  (Both GEMMs in one cooperative launch, the L1 epilogue also
    // writing the bf16 h rows L2 reads, measured 8.50 ms against 8.02 ms for the skewed workload:
    // the heavier L1 epilogue holds both accumulators longer while the MMA waits.)
    moe_status st = gemm_common(true, x_perm, x_perm_sf, expert_ids, m_sum, T, K, H, I, E, align, w13, h_q, h_sf,
                                nullptr, ws, ws_bytes, stream, nullptr, rows, row_ids, row_w, gather_ids, gather_inv);
    if (st != MOE_OK) return st;
    return gemm_common(false, h_q, h_sf, expert_ids, m_sum, T, K, H, I, E, align, w2, nullptr, nullptr, y, ws,
                       ws_bytes, stream, red, rows);
  }
  if (!dims_ok(T, H, I, E, K, align)) return MOE_ERR_INVALID_ARG;
  if (!x_perm || !x_perm_sf || !expert_ids || !m_sum || !h_q || !h_sf || !y) return MOE_ERR_INVALID_ARG;
  if (!weight_ok(w13, E, 2 * I, H, 2) || !weight_ok(w2, E, H, I, 1)) return MOE_ERR_INVALID_ARG;
  if (!aligned(x_perm, 16) || !aligned(h_q, 16) || !aligned(h_sf, 16) || !aligned(y, 16))
    return MOE_ERR_INVALID_ARG;
  if (!gather_ids && !aligned(x_perm_sf, 16)) return MOE_ERR_INVALID_ARG;
  if (!ws) return MOE_ERR_WORKSPACE;
  const size_t U = rows ? rows : moe_msum_upper(T, K, E, align);
  const WsLayout L = layout_rows(T, H, I, E, K, align, U);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (U == 0) return MOE_OK;
  if ((row_ids == nullptr) != (row_w == nullptr)) return MOE_ERR_INVALID_ARG;
  if (gather_ids && slot_counts) return MOE_ERR_INVALID_ARG;
  const uint8_t* sf = x_perm_sf;
  uint8_t* psf = reinterpret_cast<uint8_t*>(static_cast<char*>(ws) + L.x_perm_sf);
  if (gather_ids && x_perm_sf != psf) {
    // token-order scales: the permuted rows' tiled scales into the workspace (moe_forward's permute
    // writes them there itself)
    if (launch_permute_act_sf(gather_ids, K, expert_ids, m_sum, static_cast<int>(U), T, x_perm_sf, H / 128, align,
                              psf, S(stream)) != cudaSuccess)
      return MOE_ERR_CUDA;
    sf = psf;
  }
  GemmLaunch l1 = mx_launch(true, x_perm, sf, expert_ids, m_sum, H, I, E, align, U, w13, h_q, h_sf, nullptr, ws);
  l1.row_ids = row_ids;
  l1.row_w = row_w;
  if (gather_ids) {
    l1.gather_ids = gather_ids;
    l1.gather_k = K;
    l1.gather_rows = T;
  }
  if (slot_counts && slot % gemm_block_n(align) == 0 && align % gemm_block_n(align) == 0) {
    // BatchedExperts with one expert per row block: only the blocks holding tokens are work
    l1.counts = slot_counts;
    l1.slot = slot;
  }
  GemmLaunch l2 = mx_launch(false, h_q, h_sf, expert_ids, m_sum, H, I, E, align, U, w2, nullptr, nullptr, y, ws);
  if (red) l2.red = *red;
  uint32_t* sched = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + L.sched);
  return cuda_status(launch_ffn(l1, l2, sched, S(stream)));
}

moe_status moe_grouped_ffn(const uint8_t* a_q, const uint8_t* a_sf, int a_is_permuted,
                           const int32_t* sorted_token_ids, const int32_t* expert_ids, const int32_t* m_sum, int T,
                           int K, int H, int I, int E, int align, moe_weight w13, moe_weight w2, uint8_t* h_q,
                           uint8_t* h_sf, uint16_t* y_perm, void* ws, size_t ws_bytes, void* stream) {
  if (!a_is_permuted && !sorted_token_ids) return MOE_ERR_INVALID_ARG;
  return ffn_common(a_q, a_sf, expert_ids, m_sum, T, K, H, I, E, align, w13, w2, h_q, h_sf, y_perm, ws, ws_bytes,
                    stream, nullptr, 0, nullptr, nullptr, nullptr, 0, a_is_permuted ? nullptr : sorted_token_ids);
}

moe_status moe_grouped_ffn_batched(const uint8_t* x_perm, const uint8_t* x_perm_sf, const int32_t* expert_num_tokens,
                                   int T, int K, int H, int I, int E, int max_tokens, moe_weight w13, moe_weight w2,
                                   uint8_t* h_q, uint8_t* h_sf, uint16_t* y_perm, void* ws, size_t ws_bytes,
                                   void* stream) {
  if (!slot_ok(max_tokens) || !expert_num_tokens) return MOE_ERR_INVALID_ARG;
  const int align = slot_align(T, K, E, max_tokens);
  if (!dims_ok(T, H, I, E, K, align)) return MOE_ERR_INVALID_ARG;
  const size_t U = slot_rows(E, max_tokens);
  if (U > static_cast<size_t>(INT32_MAX)) return MOE_ERR_UNSUPPORTED;
  const WsLayout L = layout_rows(T, H, I, E, K, align, U);
  if (!ws) return MOE_ERR_WORKSPACE;
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  char* b = static_cast<char*>(ws);
  int32_t* eids = reinterpret_cast<int32_t*>(b + L.expert_ids);
  int32_t* ms = reinterpret_cast<int32_t*>(b + L.m_sum);
  if (launch_batched_rows(expert_num_tokens, E, max_tokens, eids, ms, status_of(ws), S(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return ffn_common(x_perm, x_perm_sf, eids, ms, T, K, H, I, E, align, w13, w2, h_q, h_sf, y_perm, ws, ws_bytes,
                    stream, nullptr, U, nullptr, nullptr, E <= 1024 ? expert_num_tokens : nullptr, max_tokens);
}

moe_status moe_unpermute_reduce(const uint16_t* y_perm, const int32_t* inv_perm, const float* topk_w, int T, int K,
                                int H, uint16_t* out, void* stream) {
  if (T < 0 || K <= 0 || H <= 0 || H % 8) return MOE_ERR_INVALID_ARG;
  if (!y_perm || !inv_perm || !out) return MOE_ERR_INVALID_ARG;   // topk_w NULL: plain sum
  if (!aligned(y_perm, 16) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_unpermute_reduce(y_perm, inv_perm, topk_w, T, K, H, out, S(stream)));
}

}  // extern "C"

// moe_forward's L1 input: the token-order activation read through sorted_token_ids (MegaMoE page,
// 路径 A), or the permuted copy x_perm.  NVFP4 converts the rows to bf16 before its GEMM anyway, and
// that pass reads them through the index at no cost, so the permute copies nothing.  The MXFP4 GEMM
// would fetch the rows with four-row TMA gathers, 32 copies per 128-row slab where the copy path
// issues one; measured on GB300 that made the layer slower (prefill 1.77 -> 3.9 ms, decode
// 0.195 -> 0.243 ms), so MXFP4 keeps the copy.  The BatchedExperts and tiny-batch layouts keep
// their copies too.
static bool forward_reads_token_order(moe_wfmt fmt) { return fmt == MOE_W_NVFP4; }

// slot 0: contiguous layout padded to align; slot > 0: BatchedExperts (align = slot_align(slot)).
static moe_status forward_common(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                                 const float* e_score_bias, int T, int H, int I, int E, int K, int align, int slot,
                                 bool l1w, bool naive, moe_score_fn fn, int renormalize, const moe_weight& w13, const moe_weight& w2,
                                 uint16_t* out, int32_t* topk_ids, float* topk_w, int32_t* sorted_token_ids,
                                 int32_t* expert_ids, int32_t* inv_perm, int32_t* m_sum, int32_t* expert_counts,
                                 void* ws, size_t ws_bytes, void* stream) {
  if (!dims_ok(T, H, I, E, K, align) || E > 1024) return MOE_ERR_INVALID_ARG;
  if (!hidden || !w_gate || !out || !weight_ok(w13, E, 2 * I, H, 2) || !weight_ok(w2, E, H, I, 1))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
  if (!ws) return MOE_ERR_WORKSPACE;
  const size_t U = slot ? slot_rows(E, slot) : moe_msum_upper(T, K, E, align);
  if (U > static_cast<size_t>(INT32_MAX)) return MOE_ERR_UNSUPPORTED;
  const WsLayout L = layout_rows(T, H, I, E, K, align, U);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  char* b = static_cast<char*>(ws);
  int32_t* ids = topk_ids ? topk_ids : reinterpret_cast<int32_t*>(b + L.topk_ids);
  float* tw = topk_w ? topk_w : reinterpret_cast<float*>(b + L.topk_w);
  int32_t* sorted = sorted_token_ids ? sorted_token_ids : reinterpret_cast<int32_t*>(b + L.sorted);
  int32_t* eids = expert_ids ? expert_ids : reinterpret_cast<int32_t*>(b + L.expert_ids);
  int32_t* inv = inv_perm ? inv_perm : reinterpret_cast<int32_t*>(b + L.inv_perm);
  int32_t* ms = m_sum ? m_sum : reinterpret_cast<int32_t*>(b + L.m_sum);
  int32_t* cnt = expert_counts ? expert_counts : reinterpret_cast<int32_t*>(b + L.counts);
  uint8_t* xq = reinterpret_cast<uint8_t*>(b + L.x_q);
  uint8_t* xsf = reinterpret_cast<uint8_t*>(b + L.x_sf);
  uint8_t* xp = reinterpret_cast<uint8_t*>(b + L.x_perm);
  uint8_t* xpsf = reinterpret_cast<uint8_t*>(b + L.x_perm_sf);
  uint8_t* hq = reinterpret_cast<uint8_t*>(b + L.h_q);
  uint8_t* hsf = reinterpret_cast<uint8_t*>(b + L.h_sf);
  uint16_t* y = reinterpret_cast<uint16_t*>(b + L.y);
  // token-order L1 input: the permute moves no rows (MXFP4: only the scales, tiled for the GEMM;
  // NVFP4: nothing, its bf16 conversion reads the token-order scales)
  const bool gather = !naive && slot == 0 && forward_reads_token_order(w13.fmt);
  const bool mx = w13.fmt == MOE_W_MXFP4;
  moe_status st;
  if (naive) {
    st = route_naive_common(hidden, w_gate, gate_bias, e_score_bias, T, H, E, K, fn, renormalize, ids, tw, sorted,
                            eids, inv, ms, xp, xpsf, ws, ws_bytes, stream);
    if (st != MOE_OK) return st;
  } else {
    st = moe_route(hidden, w_gate, gate_bias, e_score_bias, T, H, E, K, fn, renormalize, nullptr, ids, tw, xq, xsf, ws,
                   ws_bytes, stream);
    if (st != MOE_OK) return st;
    if (gather)
      st = permute_common(ids, T, K, E, align, slot, sorted, eids, inv, ms, expert_counts, nullptr,
                          mx ? xsf : nullptr, H, nullptr, mx ? xpsf : nullptr, ws, ws_bytes, stream);
    else
      st = permute_common(ids, T, K, E, align, slot, sorted, eids, inv, ms, slot ? cnt : expert_counts, xq, xsf, H,
                          xp, xpsf, ws, ws_bytes, stream);
    if (st != MOE_OK) return st;
  }
  const bool fuse_reduce = T <= kFusedReduceMaxTokens;
  FusedReduce red{};
  if (fuse_reduce) {
    red.out = out;
    red.inv_perm = inv;
    red.topk_w = l1w ? nullptr : tw;
    red.sorted_ids = sorted;
    red.tickets = reinterpret_cast<uint32_t*>(b + L.tickets);
    red.K = K;
  }
  st = ffn_common(gather ? xq : xp, gather && !mx ? xsf : xpsf, eids, ms, T, K, H, I, E, align, w13, w2, hq, hsf, y,
                  ws, ws_bytes, stream, fuse_reduce ? &red : nullptr, U, l1w ? sorted : nullptr, l1w ? tw : nullptr,
                  slot ? cnt : nullptr, slot, gather ? sorted : nullptr, gather ? inv : nullptr);
  if (st != MOE_OK || fuse_reduce) return st;
  return cuda_status(launch_unpermute_reduce(y, inv, l1w ? nullptr : tw, T, K, H, out, S(stream)));
}

// moe_forward in one launch (small batches, MXFP4): the same workspace layout, the same routing,
// permute and GEMM code, run as phases of one cooperative kernel.
static moe_status forward_single_launch(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                                        const float* e_score_bias, int T, int H, int I, int E, int K, int align,
                                        moe_score_fn fn, int renormalize, const moe_weight& w13, const moe_weight& w2,
                                        uint16_t* out, int32_t* topk_ids, float* topk_w, int32_t* sorted_token_ids,
                                        int32_t* expert_ids, int32_t* inv_perm, int32_t* m_sum, void* ws,
                                        size_t ws_bytes, void* stream) {
  if (!dims_ok(T, H, I, E, K, align) || E > 1024) return MOE_ERR_INVALID_ARG;
  if (!hidden || !w_gate || !out || !weight_ok(w13, E, 2 * I, H, 2) || !weight_ok(w2, E, H, I, 1))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
  if (!ws) return MOE_ERR_WORKSPACE;
  const size_t U = moe_msum_upper(T, K, E, align);
  const WsLayout L = layout_rows(T, H, I, E, K, align, U);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  if (w13.fmt != MOE_W_MXFP4 || w2.fmt != MOE_W_MXFP4 || !prelude_supported(T, E, K, align) ||
      T > kFusedReduceMaxTokens)
    return MOE_ERR_UNSUPPORTED;
  char* b = static_cast<char*>(ws);
  int32_t* ids = topk_ids ? topk_ids : reinterpret_cast<int32_t*>(b + L.topk_ids);
  float* tw = topk_w ? topk_w : reinterpret_cast<float*>(b + L.topk_w);
  int32_t* sorted = sorted_token_ids ? sorted_token_ids : reinterpret_cast<int32_t*>(b + L.sorted);
  int32_t* eids = expert_ids ? expert_ids : reinterpret_cast<int32_t*>(b + L.expert_ids);
  int32_t* inv = inv_perm ? inv_perm : reinterpret_cast<int32_t*>(b + L.inv_perm);
  int32_t* ms = m_sum ? m_sum : reinterpret_cast<int32_t*>(b + L.m_sum);
  uint8_t* xq = reinterpret_cast<uint8_t*>(b + L.x_q);
  uint8_t* xsf = reinterpret_cast<uint8_t*>(b + L.x_sf);
  uint8_t* xp = reinterpret_cast<uint8_t*>(b + L.x_perm);
  uint8_t* xpsf = reinterpret_cast<uint8_t*>(b + L.x_perm_sf);
  uint8_t* hq = reinterpret_cast<uint8_t*>(b + L.h_q);
  uint8_t* hsf = reinterpret_cast<uint8_t*>(b + L.h_sf);
  uint16_t* y = reinterpret_cast<uint16_t*>(b + L.y);
  // the routing scratch where moe_route keeps it
  const size_t poff = up(kAlign + permute_scratch_bytes(T, K, E));
  if (poff + route_scratch_bytes(T, H, E) > ws_bytes) return MOE_ERR_WORKSPACE;
  FusedReduce red{};
  red.out = out;
  red.inv_perm = inv;
  red.topk_w = tw;
  red.sorted_ids = sorted;
  red.tickets = reinterpret_cast<uint32_t*>(b + L.tickets);
  red.K = K;
  GemmLaunch l1 = mx_launch(true, xp, xpsf, eids, ms, H, I, E, align, U, w13, hq, hsf, nullptr, ws);
  GemmLaunch l2 = mx_launch(false, hq, hsf, eids, ms, H, I, E, align, U, w2, nullptr, nullptr, y, ws);
  l2.red = red;
  PreludeLaunch p{};
  p.hidden = hidden;
  p.w_gate = w_gate;
  p.gate_bias = gate_bias;
  p.e_bias = e_score_bias;
  p.T = T;
  p.H = H;
  p.E = E;
  p.K = K;
  p.score_fn = static_cast<int>(fn);
  p.renormalize = renormalize;
  p.logits_out = nullptr;
  p.topk_ids = ids;
  p.topk_w = tw;
  p.x_q = xq;
  p.x_sf = xsf;
  p.partial = route_partials(b + poff);
  p.align = align;
  p.U = static_cast<int>(U);
  p.sorted_ids = sorted;
  p.expert_ids = eids;
  p.inv_perm = inv;
  p.m_sum = ms;
  p.counts = nullptr;
  p.x_perm = xp;
  p.x_perm_sf = xpsf;
  p.status = status_of(ws);
  uint32_t* sched = reinterpret_cast<uint32_t*>(b + L.sched);
  return cuda_status(launch_ffn_prelude(l1, l2, p, sched, S(stream)));
}

extern "C" {

moe_status moe_forward_single_launch(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                                     const float* e_score_bias, int T, int H, int I, int E, int K, int align,
                                     moe_score_fn fn, int renormalize, moe_weight w13, moe_weight w2, uint16_t* out,
                                     int32_t* topk_ids, float* topk_w, int32_t* sorted_token_ids, int32_t* expert_ids,
                                     int32_t* inv_perm, int32_t* m_sum, void* ws, size_t ws_bytes, void* stream) {
  return forward_single_launch(hidden, w_gate, gate_bias, e_score_bias, T, H, I, E, K, align, fn, renormalize, w13, w2,
                               out, topk_ids, topk_w, sorted_token_ids, expert_ids, inv_perm, m_sum, ws, ws_bytes,
                               stream);
}

moe_status moe_forward(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                       const float* e_score_bias, int T, int H, int I, int E, int K, int align, moe_score_fn fn,
                       int renormalize, moe_weight w13, moe_weight w2, uint16_t* out, int32_t* topk_ids,
                       float* topk_w, int32_t* sorted_token_ids, int32_t* expert_ids, int32_t* inv_perm,
                       int32_t* m_sum, void* ws, size_t ws_bytes, void* stream) {
  return forward_common(hidden, w_gate, gate_bias, e_score_bias, T, H, I, E, K, align, 0, false, false, fn,
                        renormalize, w13, w2, out, topk_ids, topk_w, sorted_token_ids, expert_ids, inv_perm, m_sum,
                        nullptr, ws, ws_bytes, stream);
}

moe_status moe_forward_naive(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                             const float* e_score_bias, int T, int H, int I, int E, int K, moe_score_fn fn,
                             int renormalize, moe_weight w13, moe_weight w2, uint16_t* out, int32_t* topk_ids,
                             float* topk_w, int32_t* sorted_token_ids, int32_t* expert_ids, int32_t* inv_perm,
                             int32_t* m_sum, void* ws, size_t ws_bytes, void* stream) {
  if (T > 16 || T * K > E) return MOE_ERR_UNSUPPORTED;
  return forward_common(hidden, w_gate, gate_bias, e_score_bias, T, H, I, E, K, kNaiveRows, 0, false, true, fn,
                        renormalize, w13, w2, out, topk_ids, topk_w, sorted_token_ids, expert_ids, inv_perm, m_sum,
                        nullptr, ws, ws_bytes, stream);
}

moe_status moe_forward_l1_weighted(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                                   const float* e_score_bias, int T, int H, int I, int E, int K, int align,
                                   moe_score_fn fn, int renormalize, moe_weight w13, moe_weight w2, uint16_t* out,
                                   int32_t* topk_ids, float* topk_w, int32_t* sorted_token_ids, int32_t* expert_ids,
                                   int32_t* inv_perm, int32_t* m_sum, void* ws, size_t ws_bytes, void* stream) {
  return forward_common(hidden, w_gate, gate_bias, e_score_bias, T, H, I, E, K, align, 0, true, false, fn,
                        renormalize, w13, w2, out, topk_ids, topk_w, sorted_token_ids, expert_ids, inv_perm, m_sum,
                        nullptr, ws, ws_bytes, stream);
}

moe_status moe_forward_batched(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                               const float* e_score_bias, int T, int H, int I, int E, int K, int max_tokens,
                               moe_score_fn fn, int renormalize, moe_weight w13, moe_weight w2, uint16_t* out,
                               int32_t* topk_ids, float* topk_w, int32_t* sorted_token_ids, int32_t* expert_ids,
                               int32_t* inv_perm, int32_t* m_sum, int32_t* expert_num_tokens, void* ws,
                               size_t ws_bytes, void* stream) {
  // a token's K experts are distinct, so no expert receives more than T tokens
  if (!slot_ok(max_tokens) || max_tokens < T) return MOE_ERR_INVALID_ARG;
  return forward_common(hidden, w_gate, gate_bias, e_score_bias, T, H, I, E, K, slot_align(T, K, E, max_tokens), max_tokens,
                        false, false, fn, renormalize, w13, w2, out, topk_ids, topk_w, sorted_token_ids, expert_ids, inv_perm, m_sum,
                        expert_num_tokens, ws, ws_bytes, stream);
}

moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, int mode, void* stream) {
  if (!ws || ws_bytes < kAlign || (mode != 0 && mode != 1)) return MOE_ERR_INVALID_ARG;
  // word 32 of the reserved first 256 bytes: zero in a zero-filled workspace, never written
  const uint32_t* never_set = static_cast<const uint32_t*>(ws) + 32;
  return cuda_status(launch_wait_selftest(never_set, status_of(ws), mode, S(stream)));
}

moe_status moe_get_error(void* ws, void* stream, moe_status* device_status) {
  if (!ws || !device_status) return MOE_ERR_INVALID_ARG;
  uint32_t v = 0;
  if (cudaStreamSynchronize(S(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (v != 0 && cudaMemset(ws, 0, sizeof(v)) != cudaSuccess) return MOE_ERR_CUDA;
  *device_status = static_cast<moe_status>(v);
  return MOE_OK;
}

const char* moe_status_str(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_INDEX: return "expert id out of range (device)";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "kernel self-check failed (bounds or alignment)";
  }
  return "unknown status";
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------
// INT8 (W8A8) variant

// L1 of the INT8 variant into bf16 h (workspace), then h quantised per row into h_q / h_s; with
// h_f16 the codes are also written as fp16 rows for the L2 GEMM.
static moe_status l1_i8_common(const int8_t* x_q, const float* x_s, int x_rows, const int32_t* sorted_token_ids,
                               const int32_t* expert_ids, const int32_t* m_sum, int T, int K, int H, int I, int E,
                               int align, const moe_weight& w13, int8_t* h_q, float* h_s, uint16_t* h_f16, void* ws,
                               size_t ws_bytes, void* stream, size_t rows = 0) {
  if (!dims_ok(T, H, I, E, K, align)) return MOE_ERR_INVALID_ARG;
  if (!x_q || !x_s || !sorted_token_ids || !expert_ids || !m_sum || !h_q || !h_s) return MOE_ERR_INVALID_ARG;
  if (!weight_ok_i8(w13, E, 2 * I, H, 2)) return MOE_ERR_INVALID_ARG;
  if (!aligned(x_q, 16) || !aligned(h_q, 16)) return MOE_ERR_INVALID_ARG;
  if (!ws) return MOE_ERR_WORKSPACE;
  const size_t U = rows ? rows : moe_msum_upper(T, K, E, align);
  const I8Layout L = layout_i8(T, H, I, E, K, align, U);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (U == 0 || T == 0) return MOE_OK;
  char* b = static_cast<char*>(ws);
  uint16_t* xf = reinterpret_cast<uint16_t*>(b + L.L.xb);
  float* as = reinterpret_cast<float*>(b + L.a_s);
  uint16_t* hb = reinterpret_cast<uint16_t*>(b + L.hb);
  const bool block = w13.fmt == MOE_W_INT8_B256;
  if (launch_i8_rows_to_f16(x_q, x_s, x_rows, sorted_token_ids, K, expert_ids, m_sum, static_cast<int>(U), H, xf, as,
                            status_of(ws), S(stream), i8_row_scales(block, H)) != cudaSuccess)
    return MOE_ERR_CUDA;
  I8Launch G;
  G.block = block ? 1 : 0;
  G.w = w13.packed;
  G.col_scale = w13.tscale;
  G.xf = xf;
  G.row_scale = as;
  G.expert_ids = expert_ids;
  G.m_sum = m_sum;
  G.out = hb;
  G.status = status_of(ws);
  G.E = E;
  G.w_rows = 2 * I;
  G.Kd = H;
  G.I = I;
  G.U = static_cast<int>(U);
  G.align = align;
  if (launch_gemm_i8(G, true, S(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(launch_quant_rows_i8(hb, static_cast<int>(U), I, expert_ids, m_sum, h_q, h_s, h_f16, S(stream),
                                          block ? 256 : 0));
}

// L2 of the INT8 variant from fp16 h codes already in the workspace's operand rows.
static moe_status l2_i8_launch(const float* h_s, const int32_t* expert_ids, const int32_t* m_sum, int H, int I, int E,
                               int align, size_t U, const moe_weight& w2, uint16_t* y, const FusedReduce* red,
                               void* ws, const I8Layout& L, void* stream) {
  I8Launch G;
  G.w = w2.packed;
  G.col_scale = w2.tscale;
  G.xf = reinterpret_cast<const uint16_t*>(static_cast<char*>(ws) + L.L.xb);
  G.row_scale = h_s;
  G.expert_ids = expert_ids;
  G.m_sum = m_sum;
  G.out = y;
  G.status = status_of(ws);
  G.E = E;
  G.w_rows = H;
  G.Kd = I;
  G.I = I;
  G.U = static_cast<int>(U);
  G.align = align;
  G.block = w2.fmt == MOE_W_INT8_B256 ? 1 : 0;
  if (red) G.red = *red;
  return cuda_status(launch_gemm_i8(G, false, S(stream)));
}

// The INT8 layer.  slot 0: contiguous layout padded to align; slot > 0: BatchedExperts (align =
// slot_align(slot)), the slot mode of the permute, U = E * slot rows.
static moe_status forward_i8_common(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                                    const float* e_score_bias, int T, int H, int I, int E, int K, int align, int slot,
                                    moe_score_fn fn, int renormalize, const moe_weight& w13, const moe_weight& w2,
                                    uint16_t* out, int32_t* topk_ids, float* topk_w, int32_t* sorted_token_ids,
                                    int32_t* expert_ids, int32_t* inv_perm, int32_t* m_sum, int32_t* expert_counts,
                                    void* ws, size_t ws_bytes, void* stream) {
  if (!dims_ok(T, H, I, E, K, align) || E > 1024) return MOE_ERR_INVALID_ARG;
  if (!hidden || !w_gate || !out || !weight_ok_i8(w13, E, 2 * I, H, 2) || !weight_ok_i8(w2, E, H, I, 1))
    return MOE_ERR_INVALID_ARG;
  if (w13.fmt != w2.fmt) return MOE_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
  if (!ws) return MOE_ERR_WORKSPACE;
  const size_t U = slot ? slot_rows(E, slot) : moe_msum_upper(T, K, E, align);
  if (U > static_cast<size_t>(INT32_MAX)) return MOE_ERR_UNSUPPORTED;
  const I8Layout L = layout_i8(T, H, I, E, K, align, U);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  char* b = static_cast<char*>(ws);
  int32_t* ids = topk_ids ? topk_ids : reinterpret_cast<int32_t*>(b + L.L.topk_ids);
  float* tw = topk_w ? topk_w : reinterpret_cast<float*>(b + L.L.topk_w);
  int32_t* sorted = sorted_token_ids ? sorted_token_ids : reinterpret_cast<int32_t*>(b + L.L.sorted);
  int32_t* eids = expert_ids ? expert_ids : reinterpret_cast<int32_t*>(b + L.L.expert_ids);
  int32_t* inv = inv_perm ? inv_perm : reinterpret_cast<int32_t*>(b + L.L.inv_perm);
  int32_t* ms = m_sum ? m_sum : reinterpret_cast<int32_t*>(b + L.L.m_sum);
  int32_t* cnt = expert_counts ? expert_counts : reinterpret_cast<int32_t*>(b + L.L.counts);
  int8_t* xq = reinterpret_cast<int8_t*>(b + L.L.x_q);
  float* xs = reinterpret_cast<float*>(b + L.x_s);
  int8_t* hq = reinterpret_cast<int8_t*>(b + L.L.h_q);
  float* hs = reinterpret_cast<float*>(b + L.h_s);
  uint16_t* xf = reinterpret_cast<uint16_t*>(b + L.L.xb);
  uint16_t* y = reinterpret_cast<uint16_t*>(b + L.L.y);
  moe_status st = moe_route(hidden, w_gate, gate_bias, e_score_bias, T, H, E, K, fn, renormalize, nullptr, ids, tw,
                            nullptr, nullptr, ws, ws_bytes, stream);
  if (st != MOE_OK) return st;
  if (launch_quant_rows_i8(hidden, T, H, nullptr, nullptr, xq, xs, nullptr, S(stream),
                           w13.fmt == MOE_W_INT8_B256 ? 256 : 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  st = permute_common(ids, T, K, E, align, slot, sorted, eids, inv, ms, slot ? cnt : nullptr, nullptr, nullptr, H,
                      nullptr, nullptr, ws, ws_bytes, stream);
  if (st != MOE_OK) return st;
  // L1, then h quantised per row with its codes also written as the L2 operand rows
  st = l1_i8_common(xq, xs, T, sorted, eids, ms, T, K, H, I, E, align, w13, hq, hs, xf, ws, ws_bytes, stream, U);
  if (st != MOE_OK) return st;
  const bool fuse_reduce = T <= kFusedReduceMaxTokens;
  FusedReduce red{};
  if (fuse_reduce) {
    red.out = out;
    red.inv_perm = inv;
    red.topk_w = tw;
    red.sorted_ids = sorted;
    red.tickets = reinterpret_cast<uint32_t*>(b + L.L.tickets);
    red.K = K;
  }
  st = l2_i8_launch(hs, eids, ms, H, I, E, align, U, w2, y, fuse_reduce ? &red : nullptr, ws, L, stream);
  if (st != MOE_OK || fuse_reduce) return st;
  return cuda_status(launch_unpermute_reduce(y, inv, tw, T, K, H, out, S(stream)));
}

extern "C" {

moe_status moe_workspace_size_i8(int T, int H, int I, int E, int K, int align, size_t* bytes) {
  if (!bytes || !dims_ok(T, H, I, E, K, align)) return MOE_ERR_INVALID_ARG;
  *bytes = layout_i8(T, H, I, E, K, align).total;
  return MOE_OK;
}

moe_status moe_act_quant_i8(const uint16_t* x, int rows, int cols, int8_t* x_q, float* x_s, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 128 || !x || !x_q || !x_s) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(x_q, 16)) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  return cuda_status(launch_quant_rows_i8(x, rows, cols, nullptr, nullptr, x_q, x_s, nullptr, S(stream)));
}

moe_status moe_act_quant_i8_b256(const uint16_t* x, int rows, int cols, int8_t* x_q, float* x_s, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 256 || !x || !x_q || !x_s) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(x_q, 16)) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  return cuda_status(launch_quant_rows_i8(x, rows, cols, nullptr, nullptr, x_q, x_s, nullptr, S(stream), 256));
}

moe_status moe_grouped_gemm_l1_swiglu_i8(const int8_t* x_q, const float* x_s, const int32_t* sorted_token_ids,
                                         const int32_t* expert_ids, const int32_t* m_sum, int T, int K, int H, int I,
                                         int E, int align, moe_weight w13, int8_t* h_q, float* h_s, void* ws,
                                         size_t ws_bytes, void* stream) {
  return l1_i8_common(x_q, x_s, T, sorted_token_ids, expert_ids, m_sum, T, K, H, I, E, align, w13, h_q, h_s, nullptr,
                      ws, ws_bytes, stream);
}

moe_status moe_grouped_gemm_l2_i8(const int8_t* h_q, const float* h_s, const int32_t* expert_ids,
                                  const int32_t* m_sum, int T, int K, int H, int I, int E, int align, moe_weight w2,
                                  uint16_t* y_perm, void* ws, size_t ws_bytes, void* stream) {
  if (!dims_ok(T, H, I, E, K, align)) return MOE_ERR_INVALID_ARG;
  if (!h_q || !h_s || !expert_ids || !m_sum || !y_perm) return MOE_ERR_INVALID_ARG;
  if (!weight_ok_i8(w2, E, H, I, 1)) return MOE_ERR_INVALID_ARG;
  if (!aligned(h_q, 16) || !aligned(y_perm, 16)) return MOE_ERR_INVALID_ARG;
  if (!ws) return MOE_ERR_WORKSPACE;
  const I8Layout L = layout_i8(T, H, I, E, K, align);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  const size_t U = moe_msum_upper(T, K, E, align);
  if (U == 0 || T == 0) return MOE_OK;
  char* b = static_cast<char*>(ws);
  uint16_t* xf = reinterpret_cast<uint16_t*>(b + L.L.xb);
  float* as = reinterpret_cast<float*>(b + L.a_s);
  if (launch_i8_rows_to_f16(h_q, h_s, static_cast<int>(U), nullptr, 1, expert_ids, m_sum, static_cast<int>(U), I, xf,
                            as, status_of(ws), S(stream), i8_row_scales(w2.fmt == MOE_W_INT8_B256, I)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return l2_i8_launch(as, expert_ids, m_sum, H, I, E, align, U, w2, y_perm, nullptr, ws, L, stream);
}

moe_status moe_forward_i8(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                          const float* e_score_bias, int T, int H, int I, int E, int K, int align, moe_score_fn fn,
                          int renormalize, moe_weight w13, moe_weight w2, uint16_t* out, int32_t* topk_ids,
                          float* topk_w, int32_t* sorted_token_ids, int32_t* expert_ids, int32_t* inv_perm,
                          int32_t* m_sum, void* ws, size_t ws_bytes, void* stream) {
  return forward_i8_common(hidden, w_gate, gate_bias, e_score_bias, T, H, I, E, K, align, 0, fn, renormalize, w13, w2,
                           out, topk_ids, topk_w, sorted_token_ids, expert_ids, inv_perm, m_sum, nullptr, ws, ws_bytes,
                           stream);
}

moe_status moe_workspace_size_batched_i8(int T, int H, int I, int E, int K, int max_tokens, size_t* bytes) {
  if (!bytes || !slot_ok(max_tokens) || !dims_ok(T, H, I, E, K, slot_align(T, K, E, max_tokens)))
    return MOE_ERR_INVALID_ARG;
  *bytes = layout_i8(T, H, I, E, K, slot_align(T, K, E, max_tokens), slot_rows(E, max_tokens)).total;
  return MOE_OK;
}

moe_status moe_forward_batched_i8(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                                  const float* e_score_bias, int T, int H, int I, int E, int K, int max_tokens,
                                  moe_score_fn fn, int renormalize, moe_weight w13, moe_weight w2, uint16_t* out,
                                  int32_t* topk_ids, float* topk_w, int32_t* sorted_token_ids, int32_t* expert_ids,
                                  int32_t* inv_perm, int32_t* m_sum, int32_t* expert_num_tokens, void* ws,
                                  size_t ws_bytes, void* stream) {
  if (!slot_ok(max_tokens) || max_tokens < T) return MOE_ERR_INVALID_ARG;
  return forward_i8_common(hidden, w_gate, gate_bias, e_score_bias, T, H, I, E, K, slot_align(T, K, E, max_tokens),
                           max_tokens, fn, renormalize, w13, w2, out, topk_ids, topk_w, sorted_token_ids, expert_ids,
                           inv_perm, m_sum, expert_num_tokens, ws, ws_bytes, stream);
}

}  // extern "C"
