"""Plain CPU statement of the INT8 (W8A8) variant of the MoE layer forward.

TEST INFRASTRUCTURE ONLY, like ``oracle.moe``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` use it, and it
shares no code with the CUDA path.

Source.  Page "INT8 高吞吐/低延迟 EP 代码梳理、疑问、流程差异、DeepEP 通信差异"
(hncyxsy.com): §2 (an INT8 dispatch, ``quant_dtype == torch.int8``, beside the
FP8 one), §3.1 (the batched expert GEMM relaxed to accept INT8 and
channel-wise weights), §11.6.2 (the high-throughput INT8 path quantises the
activations per token before the dispatch).  The routing, the permute, M_sum
and the weighted gather are those of ``oracle.moe`` (same page, §9-§10).

Readings where the page is silent:
* weights: int8 codes, one float32 scale per output channel (row of W13 and
  of W2): w[n, k] = q[n, k] * s[n].  The page's ``[256, 256]`` is the
  alignment shape (§11.6.1: the 256 passed in was meant for the per-expert
  padding, not as a quantisation block), so no block scales.
* activations (the layer input, and the SwiGLU output feeding L2) are int8
  with one float32 scale per row (token), symmetric: amax = max|x| over the
  row, s = fp32(amax / 127), q = clamp(RNE(fp32(x * fp32(127 / amax))),
  -127, 127); an all-zero row gives q = 0, s = 0.  Each step that decides a
  code is one IEEE float32 operation, so both sides take it in float32.
* the SwiGLU output is rounded to bfloat16 (the activation dtype) before its
  per-row quantisation.
* the expert GEMMs are exact integer dot products of the codes, then scaled
  by the row scale and the channel scale (here in float64); L2 rounds to
  bfloat16 per row as in the FP8 path; topk_weight is applied in the gather.

Block-quantised weights, the page's ``[256, 256]`` read the other way (§3.1
relaxes the batched expert GEMM's checks "to support INT8 with
block_shape [256, 256]"): ``fmt = "int8b"``.
* weights: int8 codes, one float32 scale per block of 256 output rows x 256
  reduction columns: w[n, k] = q[n, k] * s[n // 256, k // 256].
* activations (the layer input and the SwiGLU output) are int8 with one
  float32 scale per row and 256-column group, each group quantised by the
  per-row rule above (a group's amax, its own scale).
* the expert GEMMs: per 256-deep block kb of the reduction, the exact
  integer dot product of the codes, times the row's group scale of kb and
  the weight block's scale of kb; the blocks' terms summed (float64 here).
"""
from typing import Callable, Dict

import numpy as np

from .formats import bf16_to_f64, round_bf16_rne
from .moe import permute, route, silu

I8_QMAX = 127


def quantize_i8_rows(x: np.ndarray):
    """x [R, C] (every value exact in float32) -> (q [R, C] int8, s [R] float32).

    Per row: amax = max|x|; inv = fp32(127 / amax); q = clamp(RNE(fp32(x * inv)), -127, 127);
    s = fp32(amax / 127).  A row with amax = 0 gives q = 0 and s = 0.
    """
    x = np.asarray(x)
    x32 = x.astype(np.float32)
    assert np.array_equal(x32.astype(np.float64), x.astype(np.float64)), "values must be exact in float32"
    R, C = x32.shape
    amax = np.abs(x32).max(axis=1) if C else np.zeros(R, np.float32)
    nz = amax > 0
    inv = np.zeros(R, dtype=np.float32)
    inv[nz] = np.float32(I8_QMAX) / amax[nz]                 # float32 / float32: one IEEE rounding
    s = (amax / np.float32(I8_QMAX)).astype(np.float32)
    prod = (x32 * inv[:, None]).astype(np.float32)           # one IEEE float32 multiply per value
    q = np.clip(np.rint(prod), -I8_QMAX, I8_QMAX).astype(np.int8)   # rint: round half to even
    return q, s


def act_quant_i8(hidden_bits: np.ndarray):
    """hidden bf16 bits [T, H] -> x_q int8 [T, H], x_s float32 [T] (per-token quantisation, §11.6.2)."""
    return quantize_i8_rows(bf16_to_f64(hidden_bits))


def dequant_i8(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """codes [R, C] int8 with one scale per row [R] -> float64 [R, C] (weights: a row is an output channel)."""
    return np.asarray(q, dtype=np.float64) * np.asarray(s, dtype=np.float32).astype(np.float64)[:, None]


def i8_dot(a_q: np.ndarray, w_q: np.ndarray) -> np.ndarray:
    """Exact integer dot products: a [R, Kd] int8 x w [N, Kd] int8 -> [R, N] int64 (sum over Kd)."""
    return np.asarray(a_q, dtype=np.int64) @ np.asarray(w_q, dtype=np.int64).T


def expert_l1_swiglu_i8(x_q: np.ndarray, x_s: np.ndarray, w13_q: np.ndarray, w13_s: np.ndarray, I: int):
    """gate_up[r, n] = (sum_k x_q[r, k] * w13_q[n, k]) * x_s[r] * w13_s[n]; gate = columns 0..I-1,
    up = I..2I-1; h = bf16(silu(gate) * up); h quantised per row.

    Returns (h float64 [R, I] (the bf16-rounded values), h_q int8 [R, I], h_s float32 [R]).
    """
    acc = i8_dot(x_q, w13_q).astype(np.float64)               # |acc| < 2**53: exact
    gu = acc * np.asarray(x_s, np.float64)[:, None] * np.asarray(w13_s, np.float64)[None, :]
    g, u = gu[:, :I], gu[:, I:]
    h = bf16_to_f64(round_bf16_rne(silu(g) * u))
    h_q, h_s = quantize_i8_rows(h)
    return h, h_q, h_s


def expert_l2_i8(h_q: np.ndarray, h_s: np.ndarray, w2_q: np.ndarray, w2_s: np.ndarray) -> np.ndarray:
    """y[r, j] = bf16((sum_i h_q[r, i] * w2_q[j, i]) * h_s[r] * w2_s[j]) as bf16 bits [R, H]."""
    acc = i8_dot(h_q, w2_q).astype(np.float64)
    return round_bf16_rne(acc * np.asarray(h_s, np.float64)[:, None] * np.asarray(w2_s, np.float64)[None, :])


# ----------------------------------------------------------------------------
# [256, 256] block-quantised weights ("int8b")

I8_BLOCK = 256


def quantize_i8_groups(x: np.ndarray, group: int = I8_BLOCK):
    """x [R, C] (C a multiple of group) -> (q [R, C] int8, s [R, C/group] float32): every group of
    ``group`` columns of a row quantised as its own row (quantize_i8_rows)."""
    x = np.asarray(x)
    R, C = x.shape
    assert C % group == 0
    q, s = quantize_i8_rows(x.reshape(R * (C // group), group))
    return q.reshape(R, C), s.reshape(R, C // group)


def act_quant_i8_groups(hidden_bits: np.ndarray, group: int = I8_BLOCK):
    """hidden bf16 bits [T, H] -> x_q int8 [T, H], x_s float32 [T, H/group]."""
    return quantize_i8_groups(bf16_to_f64(hidden_bits), group)


def dequant_i8_groups(q: np.ndarray, s: np.ndarray, group: int = I8_BLOCK) -> np.ndarray:
    """codes [R, C] with one scale per (row, group) [R, C/group] -> float64 [R, C]."""
    q = np.asarray(q, dtype=np.float64)
    R, C = q.shape
    sc = np.asarray(s, dtype=np.float32).astype(np.float64)
    return (q.reshape(R, C // group, group) * sc[:, :, None]).reshape(R, C)


def dequant_i8_blocks(q: np.ndarray, s: np.ndarray, block: int = I8_BLOCK) -> np.ndarray:
    """weight codes [N, Kd] with one scale per (block x block) [N/block, Kd/block] -> float64 [N, Kd]."""
    q = np.asarray(q, dtype=np.float64)
    sc = np.asarray(s, dtype=np.float32).astype(np.float64)
    return q * np.repeat(np.repeat(sc, block, axis=0), block, axis=1)


def i8_block_gemm(a_q: np.ndarray, a_s: np.ndarray, w_q: np.ndarray, w_s: np.ndarray,
                  block: int = I8_BLOCK) -> np.ndarray:
    """out[r, n] = sum_kb a_s[r, kb] * w_s[n // block, kb] * (sum_{k in kb} a_q[r, k] * w_q[n, k]), float64.

    a_q [R, Kd] int8, a_s [R, Kd/block]; w_q [N, Kd] int8, w_s [N/block, Kd/block]."""
    R, Kd = a_q.shape
    N = w_q.shape[0]
    out = np.zeros((R, N), dtype=np.float64)
    ws_rows = np.repeat(np.asarray(w_s, dtype=np.float32).astype(np.float64), block, axis=0)   # [N, Kd/block]
    for kb in range(Kd // block):
        cols = slice(kb * block, (kb + 1) * block)
        d = i8_dot(a_q[:, cols], w_q[:, cols]).astype(np.float64)        # exact integers
        out += d * np.asarray(a_s, np.float32).astype(np.float64)[:, kb:kb + 1] * ws_rows[None, :, kb][0]
    return out


def expert_l1_swiglu_i8_block(x_q, x_s, w13_q, w13_s, I: int):
    """L1 with [256, 256] weight blocks and per-256-group activation scales; h = bf16(silu(gate) * up)
    quantised per (row, 256-group).  Returns (h float64 [R, I], h_q int8 [R, I], h_s float32 [R, I/256])."""
    gu = i8_block_gemm(x_q, x_s, w13_q, w13_s)
    g, u = gu[:, :I], gu[:, I:]
    h = bf16_to_f64(round_bf16_rne(silu(g) * u))
    h_q, h_s = quantize_i8_groups(h)
    return h, h_q, h_s


def expert_l2_i8_block(h_q, h_s, w2_q, w2_s) -> np.ndarray:
    """y = bf16(block GEMM of h against W2) as bf16 bits [R, H]."""
    return round_bf16_rne(i8_block_gemm(h_q, h_s, w2_q, w2_s))


WeightProvider = Callable[[int], dict]
"""expert e -> dict(w13_q int8 [2I, H], w13_sf float32 [2I], w2_q int8 [H, I], w2_sf float32 [H])."""


def forward_i8(inp: dict, weights: WeightProvider, K: int, align: int, score_fn: str,
               renormalize: bool = True, tokens=None, topk_w_dtype=np.float64, routing=None,
               block: bool = False) -> Dict[str, object]:
    """Route -> per-token int8 quantisation -> permute -> per expert: integer L1, SwiGLU, bf16,
    per-row int8 requant, integer L2 -> bf16 rows -> weighted reduce (bf16).

    ``tokens``: optional subset of token indices (routing and the permute still use every token);
    ``out`` and ``x_q``/``x_s`` then hold only those tokens' rows, in the order given.
    ``topk_w_dtype``: precision of the routing weights in the final sum.
    ``routing``: optional dict with topk_ids [T,K] and topk_w [T,K] used in place of the computed routing.
    ``block``: [256, 256] block-quantised weights (w*_sf [N/256, Kd/256]) and per-256-group activation
    scales (``x_s`` then [len(tokens), H/256]).
    """
    hidden = inp["hidden"]
    T, H = hidden.shape
    E = inp["w_gate"].shape[0]
    if routing is None:
        r = route(hidden, inp["w_gate"], inp.get("gate_bias"), inp.get("e_score_bias"), K, score_fn, renormalize)
    else:
        r = dict(topk_ids=np.asarray(routing["topk_ids"], dtype=np.int32),
                 topk_w=np.asarray(routing["topk_w"], dtype=np.float64))
    p = permute(r["topk_ids"], E, align)
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    q_rows, s_rows = act_quant_i8_groups(hidden[tok]) if block else act_quant_i8(hidden[tok])
    x_q = {int(t): q_rows[i] for i, t in enumerate(tok)}
    x_s = {int(t): s_rows[i] for i, t in enumerate(tok)}
    need = {}
    for t in tok:
        for k in range(K):
            need.setdefault(int(r["topk_ids"][t, k]), []).append(int(t))
    y_rows, h_rows = {}, {}
    for e, ts in sorted(need.items()):
        w = weights(e)
        I = w["w13_q"].shape[0] // 2
        ts = sorted(set(ts))
        xq_e, xs_e = np.stack([x_q[t] for t in ts]), np.array([x_s[t] for t in ts])
        if block:
            _, hq, hs = expert_l1_swiglu_i8_block(xq_e, xs_e, w["w13_q"], w["w13_sf"], I)
            y = expert_l2_i8_block(hq, hs, w["w2_q"], w["w2_sf"])
        else:
            _, hq, hs = expert_l1_swiglu_i8(xq_e, xs_e, w["w13_q"], w["w13_sf"], I)
            y = expert_l2_i8(hq, hs, w["w2_q"], w["w2_sf"])
        for j, t in enumerate(ts):
            y_rows[(t, e)] = y[j]
            h_rows[(t, e)] = (hq[j], hs[j])
    out = np.zeros((len(tok), H), dtype=np.uint16)
    wts = r["topk_w"].astype(topk_w_dtype).astype(np.float64)
    for i, t in enumerate(tok):
        acc = np.zeros(H, dtype=np.float64)
        for k in range(K):
            acc += wts[t, k] * bf16_to_f64(y_rows[(int(t), int(r["topk_ids"][t, k]))])
        out[i] = round_bf16_rne(acc)
    return dict(route=r, x_q=q_rows, x_s=s_rows, perm=p, out=out, tokens=tok, y_rows=y_rows, h_rows=h_rows)
