"""GPU parity of the INT8 (W8A8) variant through the C ABI against the float64 oracle (oracle.int8).

Bars, from the arithmetic:
  * moe_act_quant_i8: codes and scales bit-exact (both sides take every decision in IEEE float32);
  * L1 + SwiGLU + per-row requant: the kernel forms h in fp32 and rounds it to bf16, the oracle in
    float64, so h can differ by one bf16 step where the two straddle a rounding boundary.  Hence h_s
    within 2^-7 relative, every code within one of the oracle's, >= 98% of the codes identical, and
    the dequantised h within half a quantisation step + 2^-7 |h| of the oracle's h;
  * L2 on the GPU's own h: each y within one bf16 step of the oracle, or within 2^-16 of its row's
    sum of |terms| (the fp32 accumulation order of the tensor core);
  * the layer: index outputs bit-exact, every token within 2e-2 x RMS of the oracle, and
    moe_forward_i8 equal bit for bit to its stage calls.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from gpu_util import bf16_ulp_diff, check_layer, check_out, dev, dev_bf16, device_weights, ensure_lib, host_bits
from oracle import formats as F
from oracle import int8 as QI
from oracle import moe as O

pytestmark = pytest.mark.gpu

I32 = dict(dtype=torch.int32, device="cuda")
I8 = dict(dtype=torch.int8, device="cuda")
F32 = dict(dtype=torch.float32, device="cuda")


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_lib()


def _args(inp):
    return (dev_bf16(inp["hidden"]), dev(inp["w_gate"]), None if inp["gate_bias"] is None else dev(inp["gate_bias"]),
            None if inp["e_score_bias"] is None else dev(inp["e_score_bias"]))


@pytest.mark.parametrize("R,C", [(1, 128), (5, 512), (77, 7168), (300, 256)])
def test_act_quant_i8_bit_exact(M, R, C):
    rng = np.random.default_rng(R + C)
    bits = synth.bf16_rows(rng, R, C)
    bits[0, :8] = F.round_bf16_rne(np.array([127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, -126.5]))  # ties at inv = 1
    bits[0, 8:] = 0
    if R > 2:
        bits[2] = 0                                   # a zero row
        bits[1] *= 0
        bits[1, :3] = F.round_bf16_rne(np.array([3.0, 1.5, -1.0]))   # the float32 tie 63.5 -> 64
    q = torch.empty(R, C, **I8)
    s = torch.empty(R, **F32)
    M.act_quant_i8(dev_bf16(bits), q, s)
    rq, rs = QI.act_quant_i8(bits)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy(), rs)


def _permute(M, ids, E, align):
    T, K = ids.shape
    U = M.msum_upper(T, K, E, align)
    srt, eid, inv, ms = torch.empty(U, **I32), torch.empty(U, **I32), torch.empty(T, K, **I32), torch.empty(1, **I32)
    return U, srt, eid, inv, ms


L1_CASES = [(8, 4, 16, 512, 256, 16), (37, 4, 16, 512, 256, 16), (200, 6, 32, 1024, 512, 64), (64, 4, 8, 512, 384, 1),
            (300, 2, 4, 256, 256, 128), (5, 1, 64, 384, 128, 4), (16, 6, 32, 7168, 2048, 16)]


@pytest.mark.parametrize("T,K,E,H,I,align", L1_CASES)
def test_l1_i8_parity(M, T, K, E, H, I, align):
    rng = np.random.default_rng(T + 7 * H + I)
    wl = synth.custom(T=T, H=H, I=I, E=E, K=K, align=align, seed=T + H, fmt="int8")
    stack = synth.all_expert_weights(wl)
    ids = synth.topk_ids_random(rng, T, E, K, 0.5)
    xq, xs = QI.act_quant_i8(synth.bf16_rows(rng, T, H))
    w13, _ = device_weights(M, stack, "int8")
    U, srt, eid, inv, ms = _permute(M, ids, E, align)
    ws = M.new_workspace_i8(T, H, I, E, K, align)
    M.permute(dev(ids), E, align, srt, eid, inv, ms, ws)
    p = O.permute(ids, E, align)
    assert np.array_equal(srt.cpu().numpy(), p["sorted_token_ids"]) and int(ms.item()) == p["m_sum"]
    hq_d = torch.zeros(U, I, **I8)
    hs_d = torch.zeros(U, **F32)
    M.grouped_gemm_l1_swiglu_i8(dev(xq), dev(xs), srt, eid, ms, T, K, H, I, E, align, w13, hq_d, hs_d, ws)
    assert M.get_error(ws) == M.OK
    hq, hs = hq_d.cpu().numpy(), hs_d.cpu().numpy()
    n_codes = n_same = 0
    for e in range(E):
        rows = np.where(p["expert_ids"] == e)[0]
        if rows.size == 0:
            continue
        toks = p["sorted_token_ids"][rows] // K
        h, hq_ref, hs_ref = QI.expert_l1_swiglu_i8(xq[toks], xs[toks], stack["w13_q"][e], stack["w13_sf"][e], I)
        got_q, got_s = hq[rows].astype(np.int64), hs[rows].astype(np.float64)
        assert (np.abs(got_s - hs_ref) <= hs_ref.astype(np.float64) * 2.0 ** -7).all(), f"expert {e}: h_s"
        assert (np.abs(got_q - hq_ref) <= 1).all(), f"expert {e}: codes off by more than one"
        deq = got_q * got_s[:, None]
        bad = np.abs(deq - h) > got_s[:, None] * (0.5 + 1e-5) + np.abs(h) * 2.0 ** -7 + 1e-30
        assert not bad.any(), f"expert {e}: {bad.sum()} values off"
        n_codes += hq_ref.size
        n_same += int((got_q == hq_ref).sum())
    assert n_same >= 0.98 * n_codes


@pytest.mark.parametrize("T,K,E,H,I,align", L1_CASES[:5] + [(8, 6, 64, 7168, 2048, 16)])
def test_l2_i8_parity(M, T, K, E, H, I, align):
    rng = np.random.default_rng(3 * T + H + I)
    wl = synth.custom(T=T, H=H, I=I, E=E, K=K, align=align, seed=2 * T + H, fmt="int8")
    stack = synth.all_expert_weights(wl)
    ids = synth.topk_ids_random(rng, T, E, K, 0.5)
    _, w2 = device_weights(M, stack, "int8")
    U, srt, eid, inv, ms = _permute(M, ids, E, align)
    ws = M.new_workspace_i8(T, H, I, E, K, align)
    M.permute(dev(ids), E, align, srt, eid, inv, ms, ws)
    p = O.permute(ids, E, align)
    hq = synth.i8_codes(rng, U, I)
    hs = rng.uniform(1e-3, 1e-1, size=U).astype(np.float32)
    y = torch.zeros(U, H, dtype=torch.bfloat16, device="cuda")
    M.grouped_gemm_l2_i8(dev(hq), dev(hs), eid, ms, T, K, H, I, E, align, w2, y, ws)
    assert M.get_error(ws) == M.OK
    yb = host_bits(y)
    for e in range(E):
        rows = np.where(p["expert_ids"] == e)[0]
        if rows.size == 0:
            continue
        ref = QI.expert_l2_i8(hq[rows], hs[rows], stack["w2_q"][e], stack["w2_sf"][e])
        terms = (np.abs(hq[rows].astype(np.float64)) @ np.abs(stack["w2_q"][e].astype(np.float64)).T) \
            * hs[rows, None].astype(np.float64) * stack["w2_sf"][e][None, :].astype(np.float64)
        ulp = bf16_ulp_diff(yb[rows], ref)
        diff = np.abs(F.bf16_to_f64(yb[rows]) - F.bf16_to_f64(ref))
        ok = (ulp <= 1) | (diff <= terms * 2.0 ** -16)
        assert ok.all(), f"expert {e}: {(~ok).sum()} values off"


CASES = {
    "tiny": dict(T=8, H=512, I=256, E=16, K=4, align=16, score_fn="softmax", seed=41),
    "T77_tensor_gate": dict(T=77, H=512, I=256, E=16, K=4, align=16, score_fn="softmax", seed=42),
    "align1": dict(T=23, H=512, I=256, E=16, K=4, align=1, score_fn="sqrt_softplus", e_bias=True, seed=43),
    "K1_H384": dict(T=5, H=384, I=128, E=64, K=1, align=4, score_fn="sqrt_softplus", e_bias=True, seed=44),
    "decode_dims_E32": dict(T=8, H=7168, I=2048, E=32, K=6, align=16, score_fn="sqrt_softplus", e_bias=True, seed=45),
    "T40_align64": dict(T=40, H=1024, I=512, E=32, K=6, align=64, score_fn="sqrt_softplus", e_bias=True, seed=46),
    "E1024_T16": dict(T=16, H=256, I=256, E=1024, K=8, align=16, score_fn="sqrt_softplus", e_bias=True, seed=47),
    "T300_align256": dict(T=300, H=512, I=256, E=8, K=2, align=256, score_fn="softmax", seed=48),
}


def _forward(M, w, inp, stack):
    T = inp["hidden"].shape[0]
    w13, w2 = device_weights(M, stack, "int8")
    ws = M.new_workspace_i8(T, w.H, w.I, w.E, w.K, w.align)
    U = M.msum_upper(T, w.K, w.E, w.align)
    o = dict(topk_ids=torch.empty(T, w.K, **I32), topk_w=torch.empty(T, w.K, **F32),
             sorted_token_ids=torch.empty(U, **I32), expert_ids=torch.empty(U, **I32),
             inv_perm=torch.empty(T, w.K, **I32), m_sum=torch.empty(1, **I32))
    out = torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda")
    M.forward_i8(*_args(inp), w.I, w.K, w.align, w.score_fn, w.renormalize, w13, w2, out, ws, **o)
    assert M.get_error(ws) == M.OK
    res = {k: v.cpu().numpy() for k, v in o.items()}
    res["out"] = host_bits(out)
    return res


@pytest.mark.parametrize("case", sorted(CASES))
def test_forward_i8_against_oracle(M, case):
    w = synth.custom(name=case, fmt="int8", **CASES[case])
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    g = _forward(M, w, inp, stack)
    ref = QI.forward_i8(inp, lambda e: {k: (v[e] if v is not None else None) for k, v in stack.items()}, w.K,
                        w.align, w.score_fn, w.renormalize, topk_w_dtype=np.float32)
    def rerun(toks, routing):
        return QI.forward_i8(inp, lambda e: {k: (v[e] if v is not None else None) for k, v in stack.items()}, w.K,
                             w.align, w.score_fn, w.renormalize, tokens=toks, topk_w_dtype=np.float32,
                             routing=routing)

    check_layer(M, w, inp, g, ref, rerun, perm_fn=lambda i: O.permute(i, w.E, w.align))


@pytest.mark.parametrize("case", ["tiny", "T77_tensor_gate", "T40_align64"])
def test_forward_i8_matches_stage_calls(M, case):
    w = synth.custom(name=case, fmt="int8", **CASES[case])
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    T = w.T
    a = _forward(M, w, inp, stack)
    w13, w2 = device_weights(M, stack, "int8")
    ws = M.new_workspace_i8(T, w.H, w.I, w.E, w.K, w.align)
    U, srt, eid, inv, ms = _permute(M, np.zeros((T, w.K), np.int32), w.E, w.align)
    ids, tw = torch.empty(T, w.K, **I32), torch.empty(T, w.K, **F32)
    hidden = _args(inp)
    M.route(*hidden, w.K, w.score_fn, w.renormalize, ids, tw, ws)
    xq, xs = torch.empty(T, w.H, **I8), torch.empty(T, **F32)
    M.act_quant_i8(hidden[0], xq, xs)
    M.permute(ids, w.E, w.align, srt, eid, inv, ms, ws)
    hq, hs = torch.zeros(U, w.I, **I8), torch.zeros(U, **F32)
    M.grouped_gemm_l1_swiglu_i8(xq, xs, srt, eid, ms, T, w.K, w.H, w.I, w.E, w.align, w13, hq, hs, ws)
    y = torch.zeros(U, w.H, dtype=torch.bfloat16, device="cuda")
    M.grouped_gemm_l2_i8(hq, hs, eid, ms, T, w.K, w.H, w.I, w.E, w.align, w2, y, ws)
    out = torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda")
    M.unpermute_reduce(y, inv, tw, out)
    assert M.get_error(ws) == M.OK
    assert np.array_equal(host_bits(out), a["out"])
    assert np.array_equal(ids.cpu().numpy(), a["topk_ids"])


def test_forward_i8_graph_replay(M):
    # no call of the INT8 path synchronises with the host or allocates: a captured forward replays
    w = synth.custom(name="graph", fmt="int8", **CASES["tiny"])
    stack = synth.all_expert_weights(w)
    w13, w2 = device_weights(M, stack, "int8")
    inps = [synth.layer_inputs(dataclasses.replace(w, seed=w.seed + 100 * i)) for i in range(3)]
    base = synth.layer_inputs(w)
    args = list(_args(base))
    hidden = dev_bf16(inps[0]["hidden"]).clone()
    args[0] = hidden
    out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    ws = M.new_workspace_i8(w.T, w.H, w.I, w.E, w.K, w.align)
    call = lambda: M.forward_i8(*args, w.I, w.K, w.align, w.score_fn, w.renormalize, w13, w2, out, ws)
    eager = []
    for inp in inps:
        hidden.copy_(dev_bf16(inp["hidden"]))
        call()
        eager.append(out.clone())
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for i, inp in enumerate(inps):
        hidden.copy_(dev_bf16(inp["hidden"]))
        out.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager[i].view(torch.int16)), f"input {i}"
    assert M.get_error(ws) == M.OK


@pytest.mark.parametrize("case,S", [("tiny", 16), ("decode_dims_E32", 16), ("T40_align64", 64), ("K1_H384", 8),
                                    ("T77_tensor_gate", 128)])
def test_forward_batched_i8_equals_forward_i8(M, case, S):
    # the BatchedExperts layout changes where a row sits, not its arithmetic: the same bits
    w = synth.custom(name=case, fmt="int8", **CASES[case])
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    T = w.T
    a = _forward(M, w, inp, stack)
    w13, w2 = device_weights(M, stack, "int8")
    ws = M.new_workspace_batched_i8(T, w.H, w.I, w.E, w.K, S)
    U = w.E * S
    o = dict(topk_ids=torch.empty(T, w.K, **I32), topk_w=torch.empty(T, w.K, **F32),
             sorted_token_ids=torch.empty(U, **I32), expert_ids=torch.empty(U, **I32),
             inv_perm=torch.empty(T, w.K, **I32), m_sum=torch.empty(1, **I32), expert_num_tokens=torch.empty(w.E, **I32))
    out = torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda")
    M.forward_batched_i8(*_args(inp), w.I, w.K, S, w.score_fn, w.renormalize, w13, w2, out, ws, **o)
    assert M.get_error(ws) == M.OK
    assert np.array_equal(host_bits(out), a["out"])
    ids = o["topk_ids"].cpu().numpy()
    assert np.array_equal(ids, a["topk_ids"])
    p = O.permute_batched(ids, w.E, S)
    for k in ("sorted_token_ids", "expert_ids", "inv_perm"):
        assert np.array_equal(o[k].cpu().numpy(), p[k]), k
    assert np.array_equal(o["expert_num_tokens"].cpu().numpy(), p["expert_num_tokens"])
