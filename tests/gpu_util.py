"""Helpers for the GPU parity tests: device upload, library build, and the comparison rules."""
import os

import numpy as np
import torch

from oracle import formats as F
from oracle import moe as O

# Output tolerance of the whole layer: max |gpu - oracle| <= OUT_TOL * RMS(oracle out).
OUT_TOL = 2e-2
# Relative key gap below which fp32 (kernel) and float64 (oracle) routing may legitimately
# order two experts differently: the kernel's logits are fp32 sums in another order.  Such
# "near-tie" tokens are checked against the oracle's routing run on the kernel's own fp32 logits.
TIE_DELTA = 1e-5
# Relative key gap below which even the oracle's routing on the kernel's own logits may order two
# experts differently from the kernel (fp32 scoring vs float64 scoring of the same logits: a few
# fp32 ulps of the largest key).  Tokens this close are counted and checked for a valid top-K.
GPU_TIE_DELTA = 1e-6


def ensure_lib():
    import moe_expert_ffn_sqrt_gb300 as M
    if not os.path.exists(M.LIB_PATH):
        from moe_expert_ffn_sqrt_gb300 import build
        build.build()
    M.lib()
    return M


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def device_weights(M, stack, fmt):
    if fmt in ("int8", "int8b"):   # int8 codes; the channel or block scales travel as the weight's tscale
        return (M.Weight(dev(stack["w13_q"]), None, dev(stack["w13_sf"]), fmt, pair=2),
                M.Weight(dev(stack["w2_q"]), None, dev(stack["w2_sf"]), fmt, pair=1))
    w13 = M.Weight(dev(stack["w13_q"]), dev(stack["w13_sf"]),
                   None if stack["w13_ts"] is None else dev(stack["w13_ts"]), fmt, pair=2)
    w2 = M.Weight(dev(stack["w2_q"]), dev(stack["w2_sf"]),
                  None if stack["w2_ts"] is None else dev(stack["w2_ts"]), fmt, pair=1)
    return w13, w2


def near_tie_tokens(keys, K, delta=TIE_DELTA):
    """Tokens whose top-(K+1) keys (oracle, float64) contain a gap below delta * max|key|."""
    srt = -np.sort(-keys, axis=1)[:, : K + 1]
    gaps = srt[:, :-1] - srt[:, 1:]
    scale = np.abs(keys).max(axis=1)
    return np.where((gaps < delta * np.maximum(scale, 1e-30)[:, None]).any(axis=1))[0]


def _valid_topk(ids, keys, K, delta):
    kth = -np.sort(-keys)[K - 1]
    tol = delta * np.abs(keys).max()
    return len(set(ids.tolist())) == K and all(keys[e] >= kth - tol for e in ids)


def check_topk(gpu_ids, gpu_w, r, K, r_gpu=None):
    """Routing of every token against the oracle.

    * Tokens whose oracle keys (float64 logits) have every gap among the top K+1 above TIE_DELTA
      x max|key|: ids bit-exact, weights within rtol 2e-5 of the oracle's.
    * Near-tie tokens: with ``r_gpu`` (the oracle's routing run on the kernel's own fp32 logits),
      ids bit-exact and weights within rtol 2e-5 of r_gpu's ("resolved"), unless even r_gpu's keys
      are closer than GPU_TIE_DELTA and the ids differ (then a valid top-K is required and the
      token is counted as unresolved); without ``r_gpu`` a valid top-K is required.
    Returns the counts {"near": ..., "resolved": ..., "unresolved": ...}.
    """
    keys = r["keys"]
    ties = set(near_tie_tokens(keys, K, TIE_DELTA).tolist())
    gties = set(near_tie_tokens(r_gpu["keys"], K, GPU_TIE_DELTA).tolist()) if r_gpu is not None else set()
    counts = {"near": len(ties), "resolved": 0, "unresolved": 0}
    for t in range(keys.shape[0]):
        if t not in ties:
            assert np.array_equal(gpu_ids[t], r["topk_ids"][t]), f"token {t}: {gpu_ids[t]} vs {r['topk_ids'][t]}"
            assert np.allclose(gpu_w[t], r["topk_w"][t], rtol=2e-5, atol=1e-7), f"token {t} weights"
        elif r_gpu is not None and (t not in gties or np.array_equal(gpu_ids[t], r_gpu["topk_ids"][t])):
            assert np.array_equal(gpu_ids[t], r_gpu["topk_ids"][t]), \
                f"near-tie token {t}: {gpu_ids[t]} vs oracle on the kernel's logits {r_gpu['topk_ids'][t]}"
            assert np.allclose(gpu_w[t], r_gpu["topk_w"][t], rtol=2e-5, atol=1e-7), f"near-tie token {t} weights"
            counts["resolved"] += 1
        else:
            assert _valid_topk(gpu_ids[t], keys[t], K, TIE_DELTA), f"token {t}: invalid top-K"
            counts["unresolved"] += 1
    return counts


def gpu_route(M, w, inp):
    """moe_route on the layer inputs: (topk_ids, topk_w, fp32 logits) as numpy arrays.  moe_forward's
    routing stage runs the same kernels on the same inputs, so these are also its logits."""
    T = inp["hidden"].shape[0]
    ws = M.new_workspace(T, w.H, w.I, w.E, w.K, w.align)
    ids = torch.full((T, w.K), -1, dtype=torch.int32, device="cuda")
    tw = torch.full((T, w.K), float("nan"), dtype=torch.float32, device="cuda")
    logits = torch.full((T, w.E), float("nan"), dtype=torch.float32, device="cuda")
    M.route(dev_bf16(inp["hidden"]), dev(inp["w_gate"]), None if inp["gate_bias"] is None else dev(inp["gate_bias"]),
            None if inp["e_score_bias"] is None else dev(inp["e_score_bias"]), w.K, w.score_fn, w.renormalize,
            ids, tw, ws, logits_out=logits)
    assert M.get_error(ws) == M.OK
    return ids.cpu().numpy(), tw.cpu().numpy(), logits.cpu().numpy()


def oracle_route_on(logits, w, inp):
    """The oracle's scoring, selection and weights run on the given (kernel) logits."""
    return O.route_from_logits(logits.astype(np.float64), inp["e_score_bias"], w.K, w.score_fn, w.renormalize)


def check_out(gpu_bits, ref_bits, tol=OUT_TOL):
    g = F.bf16_to_f64(gpu_bits)
    r = F.bf16_to_f64(ref_bits)
    rms = float(np.sqrt(np.mean(r * r)))
    err = float(np.abs(g - r).max())
    assert np.isfinite(g).all()
    assert err <= tol * rms, f"max err {err:.3e} > {tol} x RMS {rms:.3e}"
    return err / rms


def bf16_ulp_diff(a_bits, b_bits):
    """|difference| in units of the bf16 grid (ordered-integer distance)."""
    def key(b):
        b = b.astype(np.int64)
        return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + b)
    return np.abs(key(a_bits) - key(b_bits))


def dequant_act(codes, sf, group=128):
    return O.dequant_fp8_groups(codes, sf, group)


PERM_KEYS = ("sorted_token_ids", "expert_ids", "inv_perm")


def out_errors(gpu_bits, ref_bits):
    """Per-row max |gpu - oracle| and the oracle output's RMS."""
    g = F.bf16_to_f64(gpu_bits)
    r = F.bf16_to_f64(ref_bits)
    assert np.isfinite(g).all()
    return np.abs(g - r).max(axis=1), float(np.sqrt(np.mean(r * r)))


def check_layer(M, w, inp, g, ref, oracle_rerun, perm_fn=None, explain=None):
    """Parity of one whole-layer call with the oracle.

    g: the call's outputs as numpy (topk_ids, topk_w, out bf16 bits of every token, and the index
    outputs sorted_token_ids / expert_ids / inv_perm / m_sum when the call returns them).
    ref: the oracle's forward on the same inputs with its own routing (ref["tokens"] checked).
    oracle_rerun(tokens, routing): the oracle's forward on those tokens with the given routing.
    perm_fn(topk_ids): the oracle's permute of the layout the call uses.

    1. Routing: check_topk, near-tie tokens against the oracle's routing on the kernel's own fp32
       logits (moe_route runs the same kernels; its ids must equal the call's).
    2. Permute: the index outputs bit-exact against the oracle's permute run on the call's own
       topk_ids (whether or not every token agreed with the oracle's routing), and against the
       oracle's own permute when they all agree.
    3. Output of every checked token: against the oracle with its own routing where the ids agree,
       else (resolved near ties) with the oracle's routing on the kernel's logits: max |err| <=
       OUT_TOL x RMS.  With ``explain(tokens, rms)``, tokens beyond that bound are handed to it, and it
       must account for every one of them (see test_gpu_parity's SwiGLU-requant straddle check);
       without it the bound holds for every token.
    Returns (max err / RMS over the tokens within the bound, routing counts).
    """
    gids, gw = g["topk_ids"], g["topk_w"]
    T = gids.shape[0]
    rids, _, logits = gpu_route(M, w, inp)
    assert np.array_equal(rids, gids), "moe_route and the layer call disagree on topk_ids"
    r = ref["route"]
    r_gpu = oracle_route_on(logits, w, inp)
    counts = check_topk(gids, gw, r, w.K, r_gpu)
    assert counts["unresolved"] <= max(2, T // 100), counts
    agree = (gids == r["topk_ids"]).all(axis=1)
    if perm_fn is not None and "inv_perm" in g:
        p = perm_fn(gids)
        for k in PERM_KEYS:
            assert np.array_equal(g[k], p[k]), k
        assert int(np.asarray(g["m_sum"]).reshape(-1)[0]) == p["m_sum"]
        if agree.all():
            for k in PERM_KEYS:
                assert np.array_equal(g[k], ref["perm"][k]), k
    toks = np.asarray(ref["tokens"])
    keep = agree[toks]
    if explain is None:
        rel = check_out(g["out"][toks[keep]], ref["out"][keep])
    else:
        err, rms = out_errors(g["out"][toks[keep]], ref["out"][keep])
        over = err > OUT_TOL * rms
        counts["beyond_bound"] = int(over.sum())
        if over.any():
            explain(toks[keep][over], rms)
        rel = float(err[~over].max() / rms) if (~over).any() else 0.0
    flipped = toks[~keep]
    flipped = flipped[[np.array_equal(gids[t], r_gpu["topk_ids"][t]) for t in flipped]] if flipped.size else flipped
    if flipped.size:
        ids = r["topk_ids"].copy()
        tw = np.asarray(r["topk_w"], dtype=np.float64).copy()
        ids[flipped] = r_gpu["topk_ids"][flipped]
        tw[flipped] = r_gpu["topk_w"][flipped]
        ref2 = oracle_rerun(flipped, dict(topk_ids=ids, topk_w=tw))
        rel = max(rel, check_out(g["out"][flipped], ref2["out"]))
    counts["outputs_checked"] = int(keep.sum() + flipped.size)
    print(f"routing parity {w.name} T={T}: {counts}")
    return rel, counts
