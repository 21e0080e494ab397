"""Pins for the oracle's expert FFN, FP8 requant, weight dequant, weighted reduce and whole layer."""
import math

import numpy as np
import torch

import synth
from conftest import load_golden
from oracle import formats as F
from oracle import moe


def test_silu_matches_torch():
    x = np.linspace(-40, 40, 2001)
    ref = torch.nn.functional.silu(torch.from_numpy(x)).numpy()
    assert np.allclose(moe.silu(x), ref, rtol=1e-15, atol=1e-300)


def test_swiglu_closed_form_and_gate_up_order():
    # one-hot x picks column j of W13, so gate_i = W13[i, j] and up_i = W13[I + i, j]
    # (MegaMoE page, 第三步: rows 0..I-1 of W13 are the gate projection, rows I..2I-1 the up projection)
    I, H = 128, 128
    rng = np.random.default_rng(0)
    w13 = rng.standard_normal((2 * I, H))
    j = 5
    x = np.zeros((1, H))
    x[0, j] = 1.0
    h, hq, hsf = moe.expert_l1_swiglu(x, w13, I)
    for i in range(I):
        g, u = w13[i, j], w13[I + i, j]
        ref = g / (1.0 + math.exp(-g)) * u
        assert abs(h[0, i] - ref) <= 1e-15 * (1 + abs(ref))
    swapped = np.array([w13[I + i, j] / (1 + math.exp(-w13[I + i, j])) * w13[i, j] for i in range(I)])
    assert not np.allclose(h[0], swapped)


def test_fp8_group_quant_properties():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((6, 512)) * np.array([1e-3, 1, 30, 1e4, 0, 1])[:, None]
    x[5, 128:256] = 0.0
    q, sf = moe.quantize_fp8_groups(x, 128)
    assert q.shape == (6, 512) and sf.shape == (6, 4)
    deq = moe.dequant_fp8_groups(q, sf, 128)
    for r in range(6):
        for g in range(4):
            blk = x[r, g * 128:(g + 1) * 128]
            e = int(sf[r, g]) - 127
            amax = np.abs(blk).max()
            if amax == 0:
                assert e == 0 and (q[r, g * 128:(g + 1) * 128] & 0x7F == 0).all()
                continue
            assert amax <= 448 * 2.0 ** e and amax > 448 * 2.0 ** (e - 1)     # smallest non-saturating scale
            scaled = blk * 2.0 ** -e
            # each code is the nearest E4M3 value: error at most half the local spacing (<= 2**-4 relative or 2**-10 abs)
            err = np.abs(deq[r, g * 128:(g + 1) * 128] * 2.0 ** -e - scaled)
            assert (err <= np.maximum(np.abs(scaled) * 2.0 ** -4, 2.0 ** -10) + 1e-300).all()


def test_mxfp4_dequant_by_hand():
    rng = np.random.default_rng(2)
    N, Kd = 3, 64
    q = rng.integers(0, 256, size=(N, Kd // 2), dtype=np.uint8)
    sf = rng.integers(100, 140, size=(N, Kd // 32), dtype=np.uint8)
    w = moe.dequant_mxfp4(q, sf)
    for n in range(N):
        for k in range(Kd):
            code = (int(q[n, k // 2]) >> (4 * (k % 2))) & 15
            assert w[n, k] == F.e2m1_value(code) * 2.0 ** (int(sf[n, k // 32]) - 127)


def test_nvfp4_dequant_by_hand():
    rng = np.random.default_rng(3)
    N, Kd = 2, 64
    q = rng.integers(0, 256, size=(N, Kd // 2), dtype=np.uint8)
    sf = rng.integers(0x20, 0x50, size=(N, Kd // 16), dtype=np.uint8)
    ts = np.float32(0.0061)
    w = moe.dequant_nvfp4(q, sf, ts)
    for n in range(N):
        for k in range(Kd):
            code = (int(q[n, k // 2]) >> (4 * (k % 2))) & 15
            ref = F.e2m1_value(code) * F.e4m3_value(int(sf[n, k // 16])) * float(ts)
            assert w[n, k] == ref


def test_l2_zero_weights_give_zero():
    hq = np.full((2, 256), 0x38, np.uint8)
    hsf = np.full((2, 2), 127, np.uint8)
    y = moe.expert_l2(hq, hsf, np.zeros((64, 256)))
    assert (y & 0x7FFF == 0).all()


def test_unpermute_reduce_brute_force():
    rng = np.random.default_rng(4)
    T, K, H, M = 4, 3, 16, 20
    y = synth.bf16_rows(rng, M, H)
    inv = np.array([rng.choice(M, K, replace=False) for _ in range(T)], dtype=np.int32)
    w = rng.uniform(0, 1, (T, K))
    out = F.bf16_to_f64(moe.unpermute_reduce(y, inv, w))
    yd = F.bf16_to_f64(y)
    for t in range(T):
        for h in range(H):
            s = math.fsum(w[t, k] * yd[inv[t, k], h] for k in range(K))
            assert out[t, h] == F.bf16_to_f64(F.round_bf16_rne(np.array([s])))[0]
    # one slot of weight 1 returns the row itself
    ident = moe.unpermute_reduce(y, inv[:, :1], np.ones((T, 1)))
    assert np.array_equal(ident, y[inv[:, 0]])


def _weights_from_stack(stack):
    def get(e):
        return {k: (v[e] if v is not None else None) for k, v in stack.items()}
    return get


def test_single_expert_layer_is_dense_swiglu_ffn():
    # E = 1, K = 1: routing weight 1, identity permute; the layer is one SwiGLU FFN.  Brute force by loops.
    w = synth.custom(T=3, H=128, I=128, E=1, K=1, align=4, score_fn="softmax")
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    res = moe.forward(inp, _weights_from_stack(stack), "mxfp4", 1, 4, "softmax")
    assert (res["route"]["topk_ids"] == 0).all() and np.allclose(res["route"]["topk_w"], 1.0)
    W13 = moe.dequant_mxfp4(stack["w13_q"][0], stack["w13_sf"][0])
    W2 = moe.dequant_mxfp4(stack["w2_q"][0], stack["w2_sf"][0])
    xq, xsf = res["x_q"], res["x_sf"]
    for t in range(3):
        x = [F.e4m3_value(int(xq[t, h])) * 2.0 ** (int(xsf[t, h // 128]) - 127) for h in range(128)]
        gu = [math.fsum(x[h] * W13[n, h] for h in range(128)) for n in range(256)]
        h = np.array([gu[i] / (1 + math.exp(-gu[i])) * gu[128 + i] for i in range(128)])
        hq, hsf = moe.quantize_fp8_groups(h[None, :], 128)
        hd = [F.e4m3_value(int(hq[0, i])) * 2.0 ** (int(hsf[0, 0]) - 127) for i in range(128)]
        y = np.array([math.fsum(hd[i] * W2[j, i] for i in range(128)) for j in range(128)])
        ref = F.round_bf16_rne(F.bf16_to_f64(F.round_bf16_rne(y)))
        assert np.array_equal(res["out"][t], ref)


def test_shape_chain_decode_dims():
    g = load_golden("shape_chain.txt")
    w = synth.WORKLOADS["decode"]
    assert (w.T, w.H, w.I, w.E, w.K) == (g["T"], g["H"], g["I"], g["E"], g["K"])
    inp = synth.layer_inputs(w)
    res = moe.forward(inp, lambda e: synth.expert_weights(w, e), w.fmt, w.K, w.align, w.score_fn, tokens=[2])
    assert list(res["route"]["logits"].shape) == g["gate"]
    assert list(res["route"]["topk_ids"].shape) == g["topk"]
    assert res["x_q"].shape == (1, g["H"])
    e = int(res["route"]["topk_ids"][2, 0])
    ew = synth.expert_weights(w, e)
    W13 = moe.dequant_mxfp4(ew["w13_q"], ew["w13_sf"])
    W2 = moe.dequant_mxfp4(ew["w2_q"], ew["w2_sf"])
    xd = moe.dequant_fp8_groups(res["x_q"], res["x_sf"])
    assert (xd @ W13.T).shape[1] == g["gate_up_per_row"]
    h, hq, hsf = moe.expert_l1_swiglu(xd, W13, w.I)
    assert h.shape[1] == g["h_act_per_row"] and hsf.shape[1] == w.I // 128
    assert moe.expert_l2(hq, hsf, W2).shape[1] == g["y_per_row"]
    assert res["out"].shape[1] == g["out"][1]
    assert np.array_equal(res["h_rows"][(2, e)][0], hq[0])


def test_tiny_layer_output_is_sane():
    w = synth.WORKLOADS["tiny"]
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    res = moe.forward(inp, _weights_from_stack(stack), w.fmt, w.K, w.align, w.score_fn)
    out = F.bf16_to_f64(res["out"])
    assert np.isfinite(out).all() and out.std() > 0
    assert res["perm"]["m_sum"] % w.align == 0


def test_l1_weight_power_of_two_commutes_with_requant_and_l2():
    # A power-of-two routing weight applied to h before the requant (MegaMoE page, 二、阶段 3) only
    # shifts the UE8M0 exponent: the E4M3 codes stay, the L2 row is scaled exactly, and the plain sum
    # of such rows equals the weighted sum of the unscaled ones, bit for bit.
    rng = np.random.default_rng(21)
    R, H, I = 5, 256, 256
    x = F.bf16_to_f64(synth.bf16_rows(rng, R, H))
    xq, xsf = moe.quantize_fp8_groups(x, 128)
    xd = moe.dequant_fp8_groups(xq, xsf)
    W13 = rng.normal(0, 0.05, (2 * I, H))
    W2 = rng.normal(0, 0.05, (H, I))
    w = np.array([1.0, 0.5, 0.25, 2.0, 0.125])
    _, hq0, hsf0 = moe.expert_l1_swiglu(xd, W13, I)
    _, hq1, hsf1 = moe.expert_l1_swiglu(xd, W13, I, w)
    assert np.array_equal(hq1, hq0)
    assert np.array_equal(hsf1.astype(int) - hsf0.astype(int), np.repeat(np.log2(w).astype(int)[:, None], I // 128, 1))
    y0 = moe.expert_l2(hq0, hsf0, W2)
    y1 = moe.expert_l2(hq1, hsf1, W2)
    assert np.array_equal(F.bf16_to_f64(y1), w[:, None] * F.bf16_to_f64(y0))
    inv = np.array([[0, 1], [2, 3], [4, 0]], dtype=np.int32)
    tw = w[inv]
    assert np.array_equal(moe.unpermute_reduce(y1, inv, None), moe.unpermute_reduce(y0, inv, tw))


def test_l1_weight_general_differs_only_by_requant_rounding():
    # general routing weights: the two placements agree to the FP8 requant error and no better
    w = synth.WORKLOADS["tiny"]
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    a = moe.forward(inp, _weights_from_stack(stack), w.fmt, w.K, w.align, w.score_fn)
    b = moe.forward(inp, _weights_from_stack(stack), w.fmt, w.K, w.align, w.score_fn, weights_in_l1=True)
    assert np.array_equal(a["route"]["topk_ids"], b["route"]["topk_ids"])
    oa, ob = F.bf16_to_f64(a["out"]), F.bf16_to_f64(b["out"])
    rms = np.sqrt(np.mean(oa * oa))
    # two independent E4M3 roundings of h (up to 2^-4 relative each) leave noise of a few percent of
    # the output's RMS; a weight dropped or applied twice moves it by tens of percent or more
    assert np.sqrt(np.mean((oa - ob) ** 2)) <= 0.08 * rms
    assert np.abs(oa - ob).max() <= 0.4 * rms
    assert not np.array_equal(a["out"], b["out"])       # the weights did move into L1
    # every y row of the L1 placement is its pair's weight times the reduce placement's row, up to
    # the same requant noise
    for (t, e), y_b in b["y_rows"].items():
        k = int(np.nonzero(a["route"]["topk_ids"][t] == e)[0][0])
        ya = a["route"]["topk_w"][t, k] * F.bf16_to_f64(a["y_rows"][(t, e)])
        yb = F.bf16_to_f64(y_b)
        assert np.sqrt(np.mean((yb - ya) ** 2)) <= 0.1 * np.sqrt(np.mean(ya * ya))


def test_routing_override_is_used_and_threads_change_nothing():
    # a routing given from outside replaces the computed one: a hand-made routing that sends every
    # token to one expert with weight 1 gives, per token, that expert's SwiGLU FFN alone (rows of
    # the layer with E = 1 computed by loops above); and experts computed on worker threads give the
    # same bits as one after another
    w = synth.custom(T=6, H=256, I=128, E=4, K=2, align=4, score_fn="softmax", seed=31)
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    get = _weights_from_stack(stack)
    ids = np.array([[2, 0]] * w.T, dtype=np.int32)
    tw = np.array([[1.0, 0.0]] * w.T)
    res = moe.forward(inp, get, "mxfp4", w.K, w.align, w.score_fn, routing=dict(topk_ids=ids, topk_w=tw))
    assert np.array_equal(res["route"]["topk_ids"], ids)
    W13 = moe.dequant_mxfp4(stack["w13_q"][2], stack["w13_sf"][2])
    W2 = moe.dequant_mxfp4(stack["w2_q"][2], stack["w2_sf"][2])
    xd = moe.dequant_fp8_groups(res["x_q"], res["x_sf"])
    _, hq, hsf = moe.expert_l1_swiglu(xd, W13, w.I)
    y2 = moe.expert_l2(hq, hsf, W2)
    assert np.array_equal(res["out"], F.round_bf16_rne(F.bf16_to_f64(y2)))
    # the permute follows the given routing: every token's two rows sit in the segments of 2 and 0
    assert res["perm"]["expert_counts"].tolist() == [w.T, 0, w.T, 0]
    a = moe.forward(inp, get, w.fmt, w.K, w.align, w.score_fn)
    b = moe.forward(inp, get, w.fmt, w.K, w.align, w.score_fn, workers=4)
    assert np.array_equal(a["out"], b["out"])
    assert all(np.array_equal(a["y_rows"][k], b["y_rows"][k]) for k in a["y_rows"])


def test_route_from_logits_matches_route_and_brute_force():
    # routing from given logits: softmax / sqrt(softplus) of those logits, selection by full sort
    rng = np.random.default_rng(32)
    logits = rng.standard_normal((5, 12))
    bias = rng.standard_normal(12) * 0.1
    r = moe.route_from_logits(logits, bias, 3, "sqrt_softplus")
    for t in range(5):
        s = [math.sqrt(math.log1p(math.exp(l))) for l in logits[t]]
        keys = [s[e] + float(np.float32(bias[e])) for e in range(12)]
        order = sorted(range(12), key=lambda e: (-keys[e], e))[:3]
        assert r["topk_ids"][t].tolist() == order
        tot = sum(s[e] for e in order)
        assert np.allclose(r["topk_w"][t], [s[e] / tot for e in order], rtol=1e-14)
