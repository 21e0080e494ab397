"""GPU parity of the INT8 variant with [256, 256] block-quantised weights (MOE_W_INT8_B256) through the
C ABI against the float64 oracle (oracle.int8, block = True).

Bars, from the arithmetic:
  * moe_act_quant_i8_b256: codes and scales bit-exact (every decision one IEEE float32 operation);
  * L1: each 256-deep block's integer dot product is exact in fp32 (256 products of two int8 codes
    sum to less than 2^24); the blocks are summed in fp32 after scaling, the oracle sums in float64,
    and h is rounded to bf16 by both, so h may differ by one bf16 step where the two straddle a
    rounding boundary: group scales within 2^-7 relative, codes within one, >= 98% identical, the
    dequantised h within half a quantisation step + 2^-7 |h|;
  * L2 on the GPU's own h: each y within one bf16 step, or within 2^-16 of the sum of its |terms|;
  * the layer: index outputs bit-exact, every token within 2e-2 x RMS, equal to its stage calls.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import bf16_ulp_diff, check_layer, dev, dev_bf16, device_weights, ensure_lib, host_bits
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


def _prov(stack):
    return lambda e: {k: (v[e] if v is not None else None) for k, v in stack.items()}


@pytest.mark.parametrize("R,C", [(1, 256), (5, 512), (77, 7168), (300, 1024)])
def test_act_quant_b256_bit_exact(M, R, C):
    rng = np.random.default_rng(R + C)
    bits = synth.bf16_rows(rng, R, C)
    bits[0, :8] = F.round_bf16_rne(np.array([127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, -126.5]))  # ties at inv = 1
    bits[0, 8:256] = 0
    if C >= 512:
        bits[0, 256:512] = 0                          # a zero group beside a non-zero one
    q = torch.empty(R, C, **I8)
    s = torch.empty(R, C // 256, **F32)
    M.act_quant_i8(dev_bf16(bits), q, s)
    rq, rs = QI.act_quant_i8_groups(bits)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy(), rs)


def _case(T, K, E, H, I, align, seed):
    rng = np.random.default_rng(seed)
    wl = synth.custom(T=T, H=H, I=I, E=E, K=K, align=align, seed=seed, fmt="int8b")
    return rng, synth.all_expert_weights(wl), synth.topk_ids_random(rng, T, E, K, 0.5)


def _permute(M, ids, E, align, ws):
    T, K = ids.shape
    U = M.msum_upper(T, K, E, align)
    srt, eid, inv, ms = torch.empty(U, **I32), torch.empty(U, **I32), torch.empty(T, K, **I32), torch.empty(1, **I32)
    M.permute(dev(ids), E, align, srt, eid, inv, ms, ws)
    return U, srt, eid, inv, ms


L1_CASES = [(8, 4, 16, 512, 256, 16), (37, 4, 16, 512, 256, 16), (200, 6, 32, 1024, 512, 64), (64, 4, 8, 512, 512, 1),
            (300, 2, 4, 256, 256, 128), (16, 6, 32, 7168, 2048, 16)]


@pytest.mark.parametrize("T,K,E,H,I,align", L1_CASES)
def test_l1_b256_parity(M, T, K, E, H, I, align):
    rng, stack, ids = _case(T, K, E, H, I, align, T + 7 * H + I)
    xq, xs = QI.act_quant_i8_groups(synth.bf16_rows(rng, T, H))
    w13, _ = device_weights(M, stack, "int8b")
    ws = M.new_workspace_i8(T, H, I, E, K, align)
    U, srt, eid, inv, ms = _permute(M, ids, E, align, ws)
    hq_d = torch.zeros(U, I, **I8)
    hs_d = torch.zeros(U, I // 256, **F32)
    M.grouped_gemm_l1_swiglu_i8(dev(xq), dev(xs), srt, eid, ms, T, K, H, I, E, align, w13, hq_d, hs_d, ws)
    assert M.get_error(ws) == M.OK
    p = O.permute(ids, E, align)
    hq, hs = hq_d.cpu().numpy(), hs_d.cpu().numpy()
    n_codes = n_same = 0
    for e in range(E):
        rows = np.where(p["expert_ids"] == e)[0]
        if rows.size == 0:
            continue
        toks = p["sorted_token_ids"][rows] // K
        h, hq_ref, hs_ref = QI.expert_l1_swiglu_i8_block(xq[toks], xs[toks], stack["w13_q"][e], stack["w13_sf"][e], I)
        got_q, got_s = hq[rows].astype(np.int64), hs[rows].astype(np.float64)
        assert (np.abs(got_s - hs_ref) <= hs_ref.astype(np.float64) * 2.0 ** -7).all(), f"expert {e}: h_s"
        assert (np.abs(got_q - hq_ref) <= 1).all(), f"expert {e}: codes off by more than one"
        deq = QI.dequant_i8_groups(got_q, got_s)
        step = np.repeat(got_s, 256, axis=1)
        bad = np.abs(deq - h) > step * (0.5 + 1e-5) + np.abs(h) * 2.0 ** -7 + 1e-30
        assert not bad.any(), f"expert {e}: {bad.sum()} values off"
        n_codes += hq_ref.size
        n_same += int((got_q == hq_ref).sum())
    assert n_same >= 0.98 * n_codes


@pytest.mark.parametrize("T,K,E,H,I,align", L1_CASES[:5] + [(8, 6, 64, 7168, 2048, 16)])
def test_l2_b256_parity(M, T, K, E, H, I, align):
    rng, stack, ids = _case(T, K, E, H, I, align, 3 * T + H + I)
    _, w2 = device_weights(M, stack, "int8b")
    ws = M.new_workspace_i8(T, H, I, E, K, align)
    U, srt, eid, inv, ms = _permute(M, ids, E, align, ws)
    hq = synth.i8_codes(rng, U, I)
    hs = rng.uniform(1e-3, 1e-1, size=(U, I // 256)).astype(np.float32)
    y = torch.zeros(U, H, dtype=torch.bfloat16, device="cuda")
    M.grouped_gemm_l2_i8(dev(hq), dev(hs), eid, ms, T, K, H, I, E, align, w2, y, ws)
    assert M.get_error(ws) == M.OK
    p = O.permute(ids, E, align)
    yb = host_bits(y)
    for e in range(E):
        rows = np.where(p["expert_ids"] == e)[0]
        if rows.size == 0:
            continue
        ref = QI.expert_l2_i8_block(hq[rows], hs[rows], stack["w2_q"][e], stack["w2_sf"][e])
        # sum of |terms|: the scale of the fp32 accumulation error
        terms = np.abs(QI.dequant_i8_groups(hq[rows], hs[rows])) @ np.abs(QI.dequant_i8_blocks(stack["w2_q"][e],
                                                                                                stack["w2_sf"][e])).T
        ulp = bf16_ulp_diff(yb[rows], ref)
        diff = np.abs(F.bf16_to_f64(yb[rows]) - F.bf16_to_f64(ref))
        ok = (ulp <= 1) | (diff <= terms * 2.0 ** -16)
        assert ok.all(), f"expert {e}: {(~ok).sum()} values off"


CASES = {
    "tiny": dict(T=8, H=512, I=256, E=16, K=4, align=16, score_fn="softmax", seed=51),
    "T77_tensor_gate": dict(T=77, H=512, I=256, E=16, K=4, align=16, score_fn="softmax", seed=52),
    "align1": dict(T=23, H=512, I=256, E=16, K=4, align=1, score_fn="sqrt_softplus", e_bias=True, seed=53),
    "decode_dims_E32": dict(T=8, H=7168, I=2048, E=32, K=6, align=16, score_fn="sqrt_softplus", e_bias=True, seed=55),
    "T40_align64": dict(T=40, H=1024, I=512, E=32, K=6, align=64, score_fn="sqrt_softplus", e_bias=True, seed=56),
    "E1024_T16": dict(T=16, H=256, I=256, E=1024, K=8, align=16, score_fn="sqrt_softplus", e_bias=True, seed=57),
    "T300_align256": dict(T=300, H=512, I=256, E=8, K=2, align=256, score_fn="softmax", seed=58),
}


def _forward(M, w, inp, stack, batched=None):
    T = inp["hidden"].shape[0]
    w13, w2 = device_weights(M, stack, "int8b")
    out = torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda")
    if batched:
        ws = M.new_workspace_batched_i8(T, w.H, w.I, w.E, w.K, batched)
        o = dict(topk_ids=torch.empty(T, w.K, **I32), topk_w=torch.empty(T, w.K, **F32))
        M.forward_batched_i8(*_args(inp), w.I, w.K, batched, w.score_fn, w.renormalize, w13, w2, out, ws, **o)
    else:
        ws = M.new_workspace_i8(T, w.H, w.I, w.E, w.K, w.align)
        U = M.msum_upper(T, w.K, w.E, w.align)
        o = dict(topk_ids=torch.empty(T, w.K, **I32), topk_w=torch.empty(T, w.K, **F32),
                 sorted_token_ids=torch.empty(U, **I32), expert_ids=torch.empty(U, **I32),
                 inv_perm=torch.empty(T, w.K, **I32), m_sum=torch.empty(1, **I32))
        M.forward_i8(*_args(inp), w.I, w.K, w.align, w.score_fn, w.renormalize, w13, w2, out, ws, **o)
    assert M.get_error(ws) == M.OK
    res = {k: v.cpu().numpy() for k, v in o.items()}
    res["out"] = host_bits(out)
    return res


@pytest.mark.parametrize("case", sorted(CASES))
def test_forward_b256_against_oracle(M, case):
    w = synth.custom(name=case, fmt="int8b", **CASES[case])
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    g = _forward(M, w, inp, stack)

    def oracle(toks, routing=None):
        return QI.forward_i8(inp, _prov(stack), w.K, w.align, w.score_fn, w.renormalize, tokens=toks,
                             topk_w_dtype=np.float32, routing=routing, block=True)

    check_layer(M, w, inp, g, oracle(None), oracle, perm_fn=lambda i: O.permute(i, w.E, w.align))


@pytest.mark.parametrize("case", ["tiny", "T77_tensor_gate", "T40_align64"])
def test_forward_b256_matches_stage_calls(M, case):
    w = synth.custom(name=case, fmt="int8b", **CASES[case])
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    T = w.T
    a = _forward(M, w, inp, stack)
    w13, w2 = device_weights(M, stack, "int8b")
    ws = M.new_workspace_i8(T, w.H, w.I, w.E, w.K, w.align)
    ids, tw = torch.empty(T, w.K, **I32), torch.empty(T, w.K, **F32)
    hidden = _args(inp)
    M.route(*hidden, w.K, w.score_fn, w.renormalize, ids, tw, ws)
    xq, xs = torch.empty(T, w.H, **I8), torch.empty(T, w.H // 256, **F32)
    M.act_quant_i8(hidden[0], xq, xs)
    U = M.msum_upper(T, w.K, w.E, w.align)
    srt, eid, inv, ms = torch.empty(U, **I32), torch.empty(U, **I32), torch.empty(T, w.K, **I32), torch.empty(1, **I32)
    M.permute(ids, w.E, w.align, srt, eid, inv, ms, ws)
    hq, hs = torch.empty(U, w.I, **I8), torch.empty(U, w.I // 256, **F32)
    M.grouped_gemm_l1_swiglu_i8(xq, xs, srt, eid, ms, T, w.K, w.H, w.I, w.E, w.align, w13, hq, hs, ws)
    y = torch.empty(U, w.H, dtype=torch.bfloat16, device="cuda")
    M.grouped_gemm_l2_i8(hq, hs, eid, ms, T, w.K, w.H, w.I, w.E, w.align, w2, y, ws)
    out = torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda")
    M.unpermute_reduce(y, inv, tw, out)
    assert M.get_error(ws) == M.OK
    assert np.array_equal(host_bits(out), a["out"])


@pytest.mark.parametrize("case,slot", [("tiny", 8), ("T40_align64", 64)])
def test_forward_batched_b256_equals_contiguous(M, case, slot):
    w = synth.custom(name=case, fmt="int8b", **CASES[case])
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    a = _forward(M, w, inp, stack)
    b = _forward(M, w, inp, stack, batched=slot)
    assert np.array_equal(a["out"], b["out"])


def test_b256_rejects_shapes_not_in_whole_blocks(M):
    # H = 384 is not a multiple of 256: the block format is refused before any launch
    w = synth.custom(name="bad", T=4, H=384, I=256, E=4, K=2, align=4, fmt="int8", seed=59)
    stack = synth.all_expert_weights(w)
    w13 = M.Weight(dev(stack["w13_q"]), None, torch.ones(4, 2, 2, **F32), "int8b", pair=2)
    w2 = M.Weight(dev(stack["w2_q"]), None, torch.ones(4, 2, 1, **F32), "int8b", pair=1)
    inp = synth.layer_inputs(w)
    ws = M.new_workspace_i8(w.T, w.H, w.I, w.E, w.K, w.align)
    out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(M.MoeError):
        M.forward_i8(*_args(inp), w.I, w.K, w.align, w.score_fn, w.renormalize, w13, w2, out, ws)
