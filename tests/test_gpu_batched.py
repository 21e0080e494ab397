"""GPU parity of the BatchedExperts layout (fixed slot of max_tokens rows per expert) through the C ABI.

Index outputs are compared with the oracle's BatchedExperts permute bit for bit.  The layer output
must equal the expert-contiguous moe_forward's bit for bit: a row's arithmetic does not depend on the
row it sits on, and that output is itself checked against the float64 oracle in test_gpu_parity.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import check_out, dev, dev_bf16, device_weights, ensure_lib, host_bits
from oracle import moe as O

pytestmark = pytest.mark.gpu

I32 = dict(dtype=torch.int32, device="cuda")
U8 = dict(dtype=torch.uint8, device="cuda")


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_lib()


def _pow2_at_least(n):
    s = 1
    while s < n:
        s *= 2
    return s


def _permute_batched(M, ids, E, S, xq=None, xsf=None):
    T, K = ids.shape
    H = 0 if xq is None else xq.shape[1]
    U = E * S
    align = M.batched_align(T, K, E, S)
    o = dict(sorted_token_ids=torch.empty(U, **I32), expert_ids=torch.empty(U, **I32),
             inv_perm=torch.empty(T, K, **I32), m_sum=torch.empty(1, **I32), expert_num_tokens=torch.empty(E, **I32))
    ws = M.new_workspace_batched(T, max(H, 128), 128, E, K, S)
    kw = {}
    if xq is not None:
        o["x_perm"] = torch.full((U, H), 0xAA, **U8)
        o["x_perm_sf"] = torch.zeros(M.act_sf_tiled_bytes(U, H // 128, align), **U8)
        kw = dict(x_q=dev(xq), x_sf=dev(xsf), x_perm=o["x_perm"], x_perm_sf=o["x_perm_sf"])
    M.permute_batched(dev(ids), E, S, o["sorted_token_ids"], o["expert_ids"], o["inv_perm"], o["m_sum"], ws,
                      expert_num_tokens=o["expert_num_tokens"], **kw)
    return o, M.get_error(ws)


@pytest.mark.parametrize("T,K,E,S,skew", [(3, 2, 3, 4, 0.0), (8, 6, 256, 8, 0.0), (1, 1, 1, 1, 0.0),
                                          (37, 4, 16, 64, 0.5), (171, 6, 32, 256, 0.7), (500, 8, 64, 512, 1.5),
                                          (2000, 8, 1024, 2048, 1.0), (100, 1, 2, 128, 0.0), (300, 6, 16, 512, 0.3)])
def test_permute_batched_parity(M, T, K, E, S, skew):
    # covers the single-CTA (T*K <= 1024) and multi-CTA kernels, slots below 16 rows (several per
    # GEMM block) and above (64- and 128-row blocks)
    rng = np.random.default_rng(T * 17 + E)
    ids = synth.topk_ids_random(rng, T, E, K, skew)
    H = 256
    xq = synth.e4m3_codes(rng, (T, H))
    xsf = synth.act_scale_codes(rng, (T, H // 128))
    p = O.permute_batched(ids, E, S)
    g, err = _permute_batched(M, ids, E, S, xq, xsf)
    assert err == M.OK
    assert int(g["m_sum"].item()) == p["m_sum"] == E * S
    for k in ("sorted_token_ids", "expert_ids", "inv_perm", "expert_num_tokens"):
        assert np.array_equal(g[k].cpu().numpy(), p[k]), k
    inv = p["inv_perm"].reshape(-1)
    assert np.array_equal(g["x_perm"].cpu().numpy()[inv], np.repeat(xq, K, axis=0))
    psf = M.act_sf_untile(g["x_perm_sf"].cpu().numpy(), E * S, H // 128, M.batched_align(T, K, E, S))
    assert np.array_equal(psf[inv], np.repeat(xsf, K, axis=0))


@pytest.mark.parametrize("T,S", [(6, 4), (2000, 1024)])
def test_permute_batched_drops_pairs_past_a_full_slot(M, T, S):
    # every pair names expert 0 (a token repeats it), so the slot overflows: the first S pairs in
    # (t, k) order keep their rows, the rest are dropped (inv_perm -1) and an index error is recorded
    K, E = 2 if T < 100 else 1, 2
    ids = np.zeros((T, K), dtype=np.int32)
    g, err = _permute_batched(M, ids, E, S)
    assert err == M.ERR_DEVICE_INDEX
    inv = g["inv_perm"].cpu().numpy().reshape(-1)
    n = T * K
    assert np.array_equal(inv[:S], np.arange(S)) and (inv[S:] == -1).all()
    assert np.array_equal(g["sorted_token_ids"].cpu().numpy()[:S], np.arange(S))
    assert (g["expert_ids"].cpu().numpy()[:S] == 0).all() and (g["expert_ids"].cpu().numpy()[S:] == -1).all()
    assert int(g["expert_num_tokens"][0].item()) == n


def _run_forward(M, w, inp, stack, S=None):
    """moe_forward (S None) or moe_forward_batched with slot size S; returns host copies."""
    T = inp["hidden"].shape[0]
    w13, w2 = device_weights(M, stack, w.fmt)
    if S is None:
        ws = M.new_workspace(T, w.H, w.I, w.E, w.K, w.align)
        U = M.msum_upper(T, w.K, w.E, w.align)
    else:
        ws = M.new_workspace_batched(T, w.H, w.I, w.E, w.K, S)
        U = w.E * S
    o = dict(out=torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda"), topk_ids=torch.empty(T, w.K, **I32),
             topk_w=torch.empty(T, w.K, dtype=torch.float32, device="cuda"),
             sorted_token_ids=torch.empty(U, **I32), expert_ids=torch.empty(U, **I32),
             inv_perm=torch.empty(T, w.K, **I32), m_sum=torch.empty(1, **I32))
    args = (dev_bf16(inp["hidden"]), dev(inp["w_gate"]), None if inp["gate_bias"] is None else dev(inp["gate_bias"]),
            None if inp["e_score_bias"] is None else dev(inp["e_score_bias"]), w.I, w.K)
    idx = {k: o[k] for k in ("topk_ids", "topk_w", "sorted_token_ids", "expert_ids", "inv_perm", "m_sum")}
    if S is None:
        M.forward(*args, w.align, w.score_fn, w.renormalize, w13, w2, o["out"], ws, **idx)
    else:
        o["expert_num_tokens"] = torch.empty(w.E, **I32)
        M.forward_batched(*args, S, w.score_fn, w.renormalize, w13, w2, o["out"], ws,
                          expert_num_tokens=o["expert_num_tokens"], **idx)
    assert M.get_error(ws) == M.OK
    return {k: v.cpu() for k, v in o.items()}


def _case(name):
    T = None
    if name == "align1":
        w = synth.custom(T=23, H=512, I=256, E=16, K=4, align=1, score_fn="sqrt_softplus", e_bias=True, seed=5)
    elif name == "nvfp4":
        w = synth.custom(T=40, H=512, I=256, E=16, K=4, align=16, score_fn="sqrt_softplus", e_bias=True,
                         fmt="nvfp4", seed=9)
    elif name == "pad_only":
        w = synth.custom(T=12, H=256, I=256, E=8, K=2, align=256, score_fn="sqrt_softplus", e_bias=True, seed=11)
    elif name == "tiny300":
        w, T = synth.WORKLOADS["tiny"], 300
    elif name == "tiny1":
        w, T = synth.WORKLOADS["tiny"], 1
    else:
        w = synth.WORKLOADS[name]
    return w, T


@pytest.mark.parametrize("case,extra", [("tiny", 1), ("tiny1", 1), ("tiny1", 8), ("align1", 1), ("nvfp4", 1),
                                        ("pad_only", 1), ("tiny300", 1), ("decode", 1), ("decode", 16)])
def test_forward_batched_equals_forward(M, case, extra):
    # extra: slot size = extra x the smallest power of two >= T (larger slots, more padding rows)
    w, T = _case(case)
    inp = synth.layer_inputs(w, T)
    T = inp["hidden"].shape[0]
    stack = synth.all_expert_weights(w)
    S = _pow2_at_least(T) * extra
    a = _run_forward(M, w, inp, stack)
    b = _run_forward(M, w, inp, stack, S)
    assert torch.equal(a["out"].view(torch.int16), b["out"].view(torch.int16))
    assert torch.equal(a["topk_ids"], b["topk_ids"]) and torch.equal(a["topk_w"], b["topk_w"])
    p = O.permute_batched(b["topk_ids"].numpy(), w.E, S)
    for k in ("sorted_token_ids", "expert_ids", "inv_perm", "expert_num_tokens"):
        assert np.array_equal(b[k].numpy(), p[k]), k
    assert int(b["m_sum"].item()) == w.E * S


def test_forward_batched_tiny_against_oracle(M):
    w = synth.WORKLOADS["tiny"]
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    g = _run_forward(M, w, inp, stack, _pow2_at_least(w.T))
    ref = O.forward(inp, lambda e: {k: (v[e] if v is not None else None) for k, v in stack.items()}, w.fmt, w.K,
                    w.align, w.score_fn, w.renormalize)
    agree = (g["topk_ids"].numpy() == ref["route"]["topk_ids"]).all(axis=1)   # near-ties may differ
    assert agree.sum() >= w.T - 1
    check_out(host_bits(g["out"])[agree], ref["out"][agree])


@pytest.mark.parametrize("case", ["tiny", "align1", "nvfp4", "tiny300"])
def test_grouped_ffn_batched_equals_grouped_ffn(M, case):
    # the BatchedExperts FFN on a buffer laid out by moe_permute_batched gives every pair's L2 row the
    # bits the contiguous FFN gives it; called twice in a row (its counters must return to zero)
    w, T = _case(case)
    inp = synth.layer_inputs(w, T)
    T = inp["hidden"].shape[0]
    stack = synth.all_expert_weights(w)
    w13, w2 = device_weights(M, stack, w.fmt)
    ids, tw = torch.empty(T, w.K, **I32), torch.empty(T, w.K, dtype=torch.float32, device="cuda")
    xq, xsf = torch.empty(T, w.H, **U8), torch.empty(T, w.H // 128, **U8)
    ws = M.new_workspace(T, w.H, w.I, w.E, w.K, w.align)
    M.route(dev_bf16(inp["hidden"]), dev(inp["w_gate"]), None if inp["gate_bias"] is None else dev(inp["gate_bias"]),
            None if inp["e_score_bias"] is None else dev(inp["e_score_bias"]), w.K, w.score_fn, w.renormalize,
            ids, tw, ws, x_q=xq, x_sf=xsf)
    # contiguous reference
    U = M.msum_upper(T, w.K, w.E, w.align)
    srt, eid, inv, ms = torch.empty(U, **I32), torch.empty(U, **I32), torch.empty(T, w.K, **I32), torch.empty(1, **I32)
    xp = torch.zeros(U, w.H, **U8)
    xpsf = torch.zeros(M.act_sf_tiled_bytes(U, w.H // 128, w.align), **U8)
    M.permute(ids, w.E, w.align, srt, eid, inv, ms, ws, x_q=xq, x_sf=xsf, x_perm=xp, x_perm_sf=xpsf)
    hq = torch.zeros(U, w.I, **U8)
    hsf = torch.zeros(M.act_sf_tiled_bytes(U, w.I // 128, w.align), **U8)
    y = torch.zeros(U, w.H, dtype=torch.bfloat16, device="cuda")
    M.grouped_ffn(xp, xpsf, eid, ms, T, w.K, w.H, w.I, w.E, w.align, w13, w2, hq, hsf, y, ws)
    assert M.get_error(ws) == M.OK
    # BatchedExperts
    S = _pow2_at_least(T)
    Ub, align_b = w.E * S, M.batched_align(T, w.K, w.E, S)
    wsb = M.new_workspace_batched(T, w.H, w.I, w.E, w.K, S)
    bs, be, bi, bm, bn = (torch.empty(Ub, **I32), torch.empty(Ub, **I32), torch.empty(T, w.K, **I32),
                          torch.empty(1, **I32), torch.empty(w.E, **I32))
    bxp = torch.zeros(Ub, w.H, **U8)
    bxpsf = torch.zeros(M.act_sf_tiled_bytes(Ub, w.H // 128, align_b), **U8)
    M.permute_batched(ids, w.E, S, bs, be, bi, bm, wsb, expert_num_tokens=bn, x_q=xq, x_sf=xsf, x_perm=bxp,
                      x_perm_sf=bxpsf)
    inv_c, inv_b = inv.flatten().long(), bi.flatten().long()
    for _ in range(2):
        bhq = torch.full((Ub, w.I), 0x7F, **U8)
        bhsf = torch.zeros(M.act_sf_tiled_bytes(Ub, w.I // 128, align_b), **U8)
        by = torch.zeros(Ub, w.H, dtype=torch.bfloat16, device="cuda")
        M.grouped_ffn_batched(bxp, bxpsf, bn, T, w.K, w.H, w.I, w.E, S, w13, w2, bhq, bhsf, by, wsb)
        assert M.get_error(wsb) == M.OK
        assert torch.equal(bhq[inv_b], hq[inv_c])
        assert torch.equal(by[inv_b].view(torch.int16), y[inv_c].view(torch.int16))
        sf_b = M.act_sf_untile(bhsf.cpu().numpy(), Ub, w.I // 128, align_b)
        sf_c = M.act_sf_untile(hsf.cpu().numpy(), U, w.I // 128, w.align)
        assert np.array_equal(sf_b[inv_b.cpu().numpy()], sf_c[inv_c.cpu().numpy()])


def test_grouped_ffn_batched_reports_overfull_count(M):
    # a count above the slot size is an index error; the call still runs on the slot's rows
    w = synth.WORKLOADS["tiny"]
    S = 8
    Ub = w.E * S
    stack = synth.all_expert_weights(w)
    w13, w2 = device_weights(M, stack, w.fmt)
    ws = M.new_workspace_batched(S, w.H, w.I, w.E, 1, S)
    counts = torch.zeros(w.E, **I32)
    counts[3] = S + 1
    xp = torch.zeros(Ub, w.H, **U8)
    align = M.batched_align(S, 1, w.E, S)
    xpsf = torch.full((M.act_sf_tiled_bytes(Ub, w.H // 128, align),), 127, **U8)
    hq = torch.zeros(Ub, w.I, **U8)
    hsf = torch.zeros(M.act_sf_tiled_bytes(Ub, w.I // 128, align), **U8)
    y = torch.full((Ub, w.H), 1.0, dtype=torch.bfloat16, device="cuda")
    M.grouped_ffn_batched(xp, xpsf, counts, S, 1, w.H, w.I, w.E, S, w13, w2, hq, hsf, y, ws)
    assert M.get_error(ws) == M.ERR_DEVICE_INDEX
    assert (y[3 * S:4 * S].float() == 0).all()          # zero activations give zero rows
