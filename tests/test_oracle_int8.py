"""Pins for the oracle's INT8 (W8A8) variant: per-row int8 quantisation, integer GEMMs with row and
channel scales, SwiGLU, and the whole layer's wiring (page "INT8 高吞吐/低延迟 EP 代码梳理", §2,
§3.1, §11.6.2; the readings are listed in the oracle's header)."""
import math

import numpy as np
import torch

import synth
from oracle import formats as F
from oracle import int8 as Q
from oracle import moe


def test_quantize_rows_by_hand():
    x = np.array([
        # amax 127: 127 / amax = 1 exactly, so q = RNE(x) (ties to even) and s = 1
        [127, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, -127, 0, 126.5],
        # amax 1: inv = 127 exactly; 0.5 * 127 = 63.5 -> 64 (even), -0.25 * 127 = -31.75 -> -32
        [1, 0.5, -0.25, 0.125, 0, 0, 0, 0, 0, 0],
        # all zero: q = 0, s = 0
        [0] * 10,
        # amax 3: inv = fp32(127/3) = 11097429 * 2^-18; 1.5 * inv = 16646143.5 * 2^-18 rounds (tie to
        # even) to 63.5 in float32, and RNE(63.5) = 64; in float64 the product 63.4999981 would give 63
        [3, 1.5, -1, 0, 0, 0, 0, 0, 0, 0],
    ], dtype=np.float64)
    q, s = Q.quantize_i8_rows(x)
    assert q.dtype == np.int8 and s.dtype == np.float32
    assert q[0].tolist() == [127, 2, 4, -2, 0, 0, 2, -127, 0, 126] and s[0] == 1.0
    assert q[1, :4].tolist() == [127, 64, -32, 16] and s[1] == np.float32(1.0 / 127.0)
    assert (q[2] == 0).all() and s[2] == 0.0
    assert q[3, :3].tolist() == [127, 64, -42] and s[3] == np.float32(3.0 / 127.0)


def test_quantize_rows_against_torch_float32():
    # the same rule through torch's float32 tensor ops (IEEE division and multiply, round half to even)
    rng = np.random.default_rng(3)
    bits = synth.bf16_rows(rng, 37, 640)
    bits[5] = 0                                            # a zero row
    bits[7, :] = synth.bf16_rows(rng, 1, 640, scale=1e-30)[0]   # tiny magnitudes
    x = F.bf16_to_f64(bits)
    q, s = Q.quantize_i8_rows(x)
    xt = torch.from_numpy(x.astype(np.float32))
    amax = xt.abs().amax(dim=1)
    inv = torch.where(amax > 0, torch.tensor(127.0) / amax, torch.zeros_like(amax))
    qt = torch.round(xt * inv[:, None]).clamp(-127, 127).to(torch.int8)
    assert np.array_equal(q, qt.numpy())
    assert np.array_equal(s, (amax / 127.0).numpy())


def test_quantize_rows_properties():
    rng = np.random.default_rng(4)
    x = F.bf16_to_f64(synth.bf16_rows(rng, 50, 256)) * rng.uniform(1e-3, 1e3, size=(50, 1))
    x = x.astype(np.float32).astype(np.float64)
    q, s = Q.quantize_i8_rows(x)
    amax = np.abs(x).max(axis=1)
    # the largest magnitude of each row maps to +-127, the sign is kept, the error is at most half a step
    assert (np.abs(q).max(axis=1) == 127).all()
    assert ((np.sign(q) == np.sign(x)) | (q == 0)).all()
    err = np.abs(Q.dequant_i8(q, s) - x)
    assert (err <= s[:, None].astype(np.float64) * (0.5 + 1e-5)).all()
    assert np.allclose(s, amax / 127.0, rtol=2.0 ** -23)


def test_integer_dot_brute_force():
    rng = np.random.default_rng(5)
    a = rng.integers(-127, 128, size=(3, 5)).astype(np.int8)
    w = rng.integers(-127, 128, size=(4, 5)).astype(np.int8)
    ref = [[sum(int(a[r, k]) * int(w[n, k]) for k in range(5)) for n in range(4)] for r in range(3)]
    assert Q.i8_dot(a, w).tolist() == ref
    # extreme codes over a long reduction: far beyond int32 per term count, exact in int64
    a = np.full((1, 4096), -127, np.int8)
    w = np.full((2, 4096), 127, np.int8)
    assert Q.i8_dot(a, w).tolist() == [[-127 * 127 * 4096] * 2]


def test_l1_swiglu_by_hand():
    # I = 1: W13 row 0 is the gate projection, row 1 the up projection
    x_q = np.array([[1, 2], [-3, 0]], np.int8)
    x_s = np.array([0.5, 2.0], np.float32)
    w13_q = np.array([[3, 4], [5, -6]], np.int8)
    w13_s = np.array([0.25, 2.0], np.float32)
    h, hq, hs = Q.expert_l1_swiglu_i8(x_q, x_s, w13_q, w13_s, 1)
    # row 0: gate = (3 + 8) * 0.5 * 0.25 = 1.375, up = (5 - 12) * 0.5 * 2 = -7
    # row 1: gate = -9 * 2 * 0.25 = -4.5, up = -15 * 2 * 2 = -60
    for r, (g, u) in enumerate([(1.375, -7.0), (-4.5, -60.0)]):
        exact = g / (1.0 + math.exp(-g)) * u
        assert h[r, 0] == F.bf16_to_f64(F.round_bf16_rne(np.array([exact])))[0]
        assert hq[r, 0] == (127 if exact > 0 else -127)
        assert hs[r] == np.float32(np.float32(abs(h[r, 0])) / np.float32(127))
    swapped = -7.0 / (1.0 + math.exp(7.0)) * 1.375
    assert abs(h[0, 0] - swapped) > 1.0


def test_l1_against_dequantised_float_gemm():
    # dequantise first, then a float64 GEMM: the same values up to float64 rounding
    rng = np.random.default_rng(6)
    R, H, I = 9, 256, 128
    x_q, x_s = Q.quantize_i8_rows(F.bf16_to_f64(synth.bf16_rows(rng, R, H)))
    w13_q = synth.i8_codes(rng, 2 * I, H)
    w13_s = synth.i8_channel_scales(rng, 2 * I)
    h, hq, hs = Q.expert_l1_swiglu_i8(x_q, x_s, w13_q, w13_s, I)
    gu = Q.dequant_i8(x_q, x_s) @ Q.dequant_i8(w13_q, w13_s).T
    ref = F.bf16_to_f64(F.round_bf16_rne(moe.silu(gu[:, :I]) * gu[:, I:]))
    assert np.abs(h - ref).max() <= np.abs(ref).max() * 2.0 ** -8
    assert (h == ref).mean() > 0.999
    q2, s2 = Q.quantize_i8_rows(h)
    assert np.array_equal(hq, q2) and np.array_equal(hs, s2)


def test_l2_by_hand():
    h_q = np.array([[2, -1]], np.int8)
    h_s = np.array([0.5], np.float32)
    w2_q = np.array([[1, 1], [4, 3], [-2, 5]], np.int8)     # H = 3 output channels, I = 2
    w2_s = np.array([1.0, 0.25, 2.0], np.float32)
    y = F.bf16_to_f64(Q.expert_l2_i8(h_q, h_s, w2_q, w2_s))
    # acc = [2 - 1, 8 - 3, -4 - 5] = [1, 5, -9]; y = acc * 0.5 * w2_s
    assert y.tolist() == [[0.5, 0.625, -9.0]]


def test_forward_wiring_against_per_token_loop():
    # the layer by explicit loops over tokens and their experts (no permute): the same bits
    w = synth.custom(T=11, H=256, I=128, E=8, K=3, align=4, fmt="int8", score_fn="sqrt_softplus", e_bias=True,
                     seed=31)
    inp = synth.layer_inputs(w)
    st = synth.all_expert_weights(w)
    wp = lambda e: {k: (v[e] if v is not None else None) for k, v in st.items()}
    res = Q.forward_i8(inp, wp, w.K, w.align, w.score_fn, w.renormalize)
    r = moe.route(inp["hidden"], inp["w_gate"], inp["gate_bias"], inp["e_score_bias"], w.K, w.score_fn, True)
    assert np.array_equal(res["route"]["topk_ids"], r["topk_ids"])
    for t in range(w.T):
        xq, xs = Q.quantize_i8_rows(F.bf16_to_f64(inp["hidden"][t:t + 1]))
        acc = np.zeros(w.H)
        for k in range(w.K):
            e = int(r["topk_ids"][t, k])
            _, hq, hs = Q.expert_l1_swiglu_i8(xq, xs, st["w13_q"][e], st["w13_sf"][e], w.I)
            acc += r["topk_w"][t, k] * F.bf16_to_f64(Q.expert_l2_i8(hq, hs, st["w2_q"][e], st["w2_sf"][e]))[0]
        assert np.array_equal(res["out"][t], F.round_bf16_rne(acc)), t
    # a token subset gives the same rows
    sub = Q.forward_i8(inp, wp, w.K, w.align, w.score_fn, w.renormalize, tokens=[7, 2])
    assert np.array_equal(sub["out"], res["out"][[7, 2]])


def test_quantize_rows_power_of_two_and_sign_symmetry():
    # scaling a row by 2^k leaves its codes unchanged and scales its scale by exactly 2^k (both
    # float32 divisions are exact under power-of-two scaling); negating a row negates its codes
    rng = np.random.default_rng(7)
    x = F.bf16_to_f64(synth.bf16_rows(rng, 20, 384))
    q, s = Q.quantize_i8_rows(x)
    for k in (-20, -3, 5, 30):
        qk, sk = Q.quantize_i8_rows(x * 2.0 ** k)
        assert np.array_equal(qk, q)
        assert np.array_equal(sk, (s * np.float32(2.0 ** k)).astype(np.float32))
    qn, sn = Q.quantize_i8_rows(-x)
    assert np.array_equal(qn, -q) and np.array_equal(sn, s)


def test_l2_linear_in_row_and_channel_scales():
    # doubling a row scale or a channel scale doubles those outputs exactly (bf16 rounding commutes
    # with a power of two); a dropped or misplaced scale fails this
    rng = np.random.default_rng(8)
    hq = synth.i8_codes(rng, 6, 256)
    hs = rng.uniform(1e-3, 1e-1, size=6).astype(np.float32)
    w2 = synth.i8_codes(rng, 128, 256)
    ws = synth.i8_channel_scales(rng, 128)
    y = F.bf16_to_f64(Q.expert_l2_i8(hq, hs, w2, ws))
    hs2 = hs.copy()
    hs2[2] *= 2
    y2 = F.bf16_to_f64(Q.expert_l2_i8(hq, hs2, w2, ws))
    assert np.array_equal(y2[2], 2 * y[2]) and np.array_equal(np.delete(y2, 2, 0), np.delete(y, 2, 0))
    ws2 = ws.copy()
    ws2[5] *= 2
    y3 = F.bf16_to_f64(Q.expert_l2_i8(hq, hs, w2, ws2))
    assert np.array_equal(y3[:, 5], 2 * y[:, 5]) and np.array_equal(np.delete(y3, 5, 1), np.delete(y, 5, 1))


# ---------------------------------------------------------------------------- [256, 256] block-quantised weights


def test_quantize_groups_by_hand():
    # two groups of 256 with their own amax: each group is quantised as a row of its own
    x = np.zeros((1, 512))
    x[0, 0], x[0, 1], x[0, 2] = 2.0, -1.0, 0.5           # group 0: amax 2 -> inv = fp32(127/2) = 63.5
    x[0, 256], x[0, 300] = 0.25, -0.125                   # group 1: amax 0.25 -> inv = 508
    q, s = Q.quantize_i8_groups(x)
    assert s.shape == (1, 2)
    assert s[0, 0] == np.float32(2.0) / np.float32(127) and s[0, 1] == np.float32(0.25) / np.float32(127)
    # 2 * 63.5 = 127; -1 * 63.5 = -63.5 -> -64 (ties to even); 0.5 * 63.5 = 31.75 -> 32
    assert q[0, :3].tolist() == [127, -64, 32]
    # 0.25 * 508 = 127; -0.125 * 508 = -63.5 -> -64
    assert q[0, 256] == 127 and q[0, 300] == -64
    assert (q[0, 3:256] == 0).all() and (np.delete(q[0, 256:], [0, 44]) == 0).all()
    # an all-zero group: codes 0, scale 0
    q0, s0 = Q.quantize_i8_groups(np.zeros((2, 256)))
    assert (q0 == 0).all() and (s0 == 0).all()


def test_dequant_blocks_by_hand():
    rng = np.random.default_rng(41)
    q = rng.integers(-127, 128, size=(512, 512)).astype(np.int8)
    s = np.array([[0.5, 2.0], [0.25, 3.0]], np.float32)
    w = Q.dequant_i8_blocks(q, s)
    for n, k in [(0, 0), (255, 255), (0, 256), (256, 0), (511, 511), (300, 17), (17, 300)]:
        assert w[n, k] == float(q[n, k]) * float(s[n // 256, k // 256])


def test_block_gemm_brute_force():
    rng = np.random.default_rng(42)
    R, N, Kd = 2, 256, 512
    a_q = rng.integers(-127, 128, size=(R, Kd)).astype(np.int8)
    a_s = rng.uniform(1e-3, 1e-2, size=(R, 2)).astype(np.float32)
    w_q = rng.integers(-127, 128, size=(N, Kd)).astype(np.int8)
    w_s = rng.uniform(1e-4, 1e-3, size=(1, 2)).astype(np.float32)
    out = Q.i8_block_gemm(a_q, a_s, w_q, w_s)
    for r in range(R):
        for n in (0, 77, 255):
            terms = [int(a_q[r, k]) * int(w_q[n, k]) * float(a_s[r, k // 256]) * float(w_s[0, k // 256])
                     for k in range(Kd)]
            assert math.isclose(out[r, n], math.fsum(terms), rel_tol=1e-13, abs_tol=1e-18)


def test_block_l1_against_dequantised_float_gemm():
    # dequantise activations and weights first, then a float64 GEMM: the same values up to float64 rounding
    rng = np.random.default_rng(43)
    R, H, I = 7, 512, 256
    x_q, x_s = Q.quantize_i8_groups(F.bf16_to_f64(synth.bf16_rows(rng, R, H)))
    w13_q = synth.i8_codes(rng, 2 * I, H)
    w13_s = synth.i8_block_scales(rng, 2 * I, H)
    h, hq, hs = Q.expert_l1_swiglu_i8_block(x_q, x_s, w13_q, w13_s, I)
    gu = Q.dequant_i8_groups(x_q, x_s) @ Q.dequant_i8_blocks(w13_q, w13_s).T
    ref = F.bf16_to_f64(F.round_bf16_rne(moe.silu(gu[:, :I]) * gu[:, I:]))
    assert np.abs(h - ref).max() <= np.abs(ref).max() * 2.0 ** -8
    assert (h == ref).mean() > 0.999
    assert hs.shape == (R, I // 256)
    q2, s2 = Q.quantize_i8_groups(h)
    assert np.array_equal(hq, q2) and np.array_equal(hs, s2)


def test_block_variant_reduces_to_channel_wise_with_uniform_scales():
    # one scale for every group of a row and one for every weight block: the block GEMM is the
    # channel-wise one with that row scale and a constant channel scale
    rng = np.random.default_rng(44)
    R, H, I = 5, 512, 256
    x_q = synth.i8_codes(rng, R, H)
    row_s = rng.uniform(1e-3, 1e-2, size=R).astype(np.float32)
    w13_q = synth.i8_codes(rng, 2 * I, H)
    c = np.float32(5e-4)
    hb, _, _ = Q.expert_l1_swiglu_i8_block(x_q, np.repeat(row_s[:, None], H // 256, 1), w13_q,
                                           np.full((2 * I // 256, H // 256), c, np.float32), I)
    hc, _, _ = Q.expert_l1_swiglu_i8(x_q, row_s, w13_q, np.full(2 * I, c, np.float32), I)
    assert np.abs(hb - hc).max() <= np.abs(hc).max() * 2.0 ** -8 and (hb == hc).mean() > 0.999


def test_block_l2_linear_in_block_scales():
    rng = np.random.default_rng(45)
    R, H, I = 4, 256, 512
    h_q = synth.i8_codes(rng, R, I)
    h_s = rng.uniform(1e-3, 1e-2, size=(R, I // 256)).astype(np.float32)
    w2_q = synth.i8_codes(rng, H, I)
    w2_s = synth.i8_block_scales(rng, H, I)
    y1 = F.bf16_to_f64(Q.expert_l2_i8_block(h_q, h_s, w2_q, w2_s))
    y2 = F.bf16_to_f64(Q.expert_l2_i8_block(h_q, h_s, w2_q, w2_s * np.float32(2)))
    assert np.array_equal(y2, 2 * y1)
    # a weight block's scale reaches only its own 256 reduction columns
    w2_z = w2_s.copy()
    w2_z[:, 1] = 0
    yz = F.bf16_to_f64(Q.expert_l2_i8_block(h_q, h_s, w2_q, w2_z))
    h0 = h_q.copy()
    h0[:, 256:] = 0
    assert np.array_equal(yz, F.bf16_to_f64(Q.expert_l2_i8_block(h0, h_s, w2_q, w2_s)))


def test_block_forward_wiring_against_per_token_loop():
    w = synth.custom(T=9, H=512, I=256, E=6, K=2, align=4, fmt="int8b", score_fn="sqrt_softplus", e_bias=True,
                     seed=46)
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    get = lambda e: {k: (v[e] if v is not None else None) for k, v in stack.items()}
    res = Q.forward_i8(inp, get, w.K, w.align, w.score_fn, w.renormalize, block=True)
    r = res["route"]
    xq, xs = Q.act_quant_i8_groups(inp["hidden"])
    assert np.array_equal(res["x_q"], xq) and np.array_equal(res["x_s"], xs)
    for t in range(w.T):
        acc = np.zeros(w.H)
        for k in range(w.K):
            e = int(r["topk_ids"][t, k])
            _, hq, hs = Q.expert_l1_swiglu_i8_block(xq[t:t + 1], xs[t:t + 1], stack["w13_q"][e], stack["w13_sf"][e], w.I)
            y = F.bf16_to_f64(Q.expert_l2_i8_block(hq, hs, stack["w2_q"][e], stack["w2_sf"][e]))[0]
            acc += r["topk_w"][t, k] * y
        assert np.array_equal(res["out"][t], F.round_bf16_rne(acc))
