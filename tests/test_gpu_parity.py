"""GPU parity: every hot-path call through the C ABI against the float64 oracle on the same seeded inputs.

Index outputs must match bit for bit; floating outputs within the stated tolerances:
  * routing weights: rtol 2e-5 (fp32 kernel vs float64 oracle);
  * x_q / x_sf: bit-exact (quantising bf16 inputs is exact arithmetic);
  * SwiGLU requant h: dequantised value within half an E4M3 step of the exact h (plus fp32 slack);
  * L2 rows and the reduce: within 1 bf16 step (fp32 accumulation vs float64, one rounding each);
  * layer output: max |err| <= 2e-2 x RMS(out).
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import (OUT_TOL, bf16_ulp_diff, check_layer, check_out, check_topk, dev, dev_bf16, device_weights,
                      ensure_lib, host_bits, oracle_route_on)
from oracle import formats as F
from oracle import moe as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_lib()


def _stack_provider(stack):
    return lambda e: {k: (v[e] if v is not None else None) for k, v in stack.items()}


# ------------------------------------------------------------------------------------------ route

@pytest.mark.parametrize("name,T", [("tiny", None), ("decode", None), ("batched", None), ("tiny", 1), ("tiny", 77),
                                    ("prefill", None)])
def test_route_parity(M, name, T):
    w = synth.WORKLOADS[name]
    inp = synth.layer_inputs(w, T)
    T = inp["hidden"].shape[0]
    r = O.route(inp["hidden"], inp["w_gate"], inp["gate_bias"], inp["e_score_bias"], w.K, w.score_fn, w.renormalize)
    ws = M.new_workspace(T, w.H, w.I, w.E, w.K, w.align)
    ids = torch.empty(T, w.K, dtype=torch.int32, device="cuda")
    tw = torch.empty(T, w.K, dtype=torch.float32, device="cuda")
    logits = torch.empty(T, w.E, dtype=torch.float32, device="cuda")
    xq = torch.empty(T, w.H, dtype=torch.uint8, device="cuda")
    xsf = torch.empty(T, w.H // 128, dtype=torch.uint8, device="cuda")
    M.route(dev_bf16(inp["hidden"]), dev(inp["w_gate"]), None if inp["gate_bias"] is None else dev(inp["gate_bias"]),
            None if inp["e_score_bias"] is None else dev(inp["e_score_bias"]), w.K, w.score_fn, w.renormalize,
            ids, tw, ws, logits_out=logits, x_q=xq, x_sf=xsf)
    assert M.get_error(ws) == M.OK
    lg = logits.cpu().numpy()
    assert np.allclose(lg, r["logits"], rtol=1e-4, atol=2e-5)
    counts = check_topk(ids.cpu().numpy(), tw.cpu().numpy(), r, w.K, oracle_route_on(lg, w, inp))
    print(f"routing parity {name} T={T}: {counts}")
    assert counts["unresolved"] <= max(2, T // 100)
    rows = np.arange(T) if T <= 512 else np.random.default_rng(0).choice(T, 256, replace=False)
    xq_ref, xsf_ref = O.act_quant(inp["hidden"][rows])
    assert np.array_equal(xq.cpu().numpy()[rows], xq_ref)
    assert np.array_equal(xsf.cpu().numpy()[rows], xsf_ref)


def test_act_quant_edge_values(M):
    # rows with exact scale boundaries, zeros, negative zeros, tiny and huge magnitudes
    H = 256
    x = np.zeros((6, H), np.float32)
    x[0, :128] = 448.0
    x[0, 5] = -448.0
    x[1, :] = np.float32(1.75)
    x[1, 200] = np.float32(1.76)
    x[2, :128] = -0.0
    x[3, :] = np.float32(2.0 ** -130)
    x[3, 7] = np.float32(-2.0 ** -133)
    x[4, :] = np.float32(3.0e38)
    x[5, :] = np.linspace(-1e-3, 1e-3, H, dtype=np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    E, K = 4, 1
    ws = M.new_workspace(6, H, 128, E, K, 1)
    ids = torch.empty(6, K, dtype=torch.int32, device="cuda")
    tw = torch.empty(6, K, dtype=torch.float32, device="cuda")
    xq = torch.empty(6, H, dtype=torch.uint8, device="cuda")
    xsf = torch.empty(6, H // 128, dtype=torch.uint8, device="cuda")
    M.route(dev_bf16(bits), torch.zeros(E, H, device="cuda"), None, None, K, "softmax", True, ids, tw, ws,
            x_q=xq, x_sf=xsf)
    q_ref, sf_ref = O.act_quant(bits)
    assert np.array_equal(xsf.cpu().numpy(), sf_ref)
    assert np.array_equal(xq.cpu().numpy(), q_ref)
    # all-zero logits: every key ties, the lowest id wins with weight 1
    assert (ids.cpu().numpy() == 0).all() and np.allclose(tw.cpu().numpy(), 1.0)


# ------------------------------------------------------------------------------------------ permute

@pytest.mark.parametrize("T,K,E,align,skew", [(8, 6, 256, 16, 0.0), (128, 6, 256, 64, 1.0), (3, 2, 3, 1, 0.0),
                                              (37, 4, 16, 16, 0.5), (500, 8, 64, 2, 1.5), (4096, 6, 256, 256, 0.0),
                                              (3000, 6, 256, 128, 1.2), (1, 1, 1, 1, 0.0), (171, 6, 32, 4, 0.7),
                                              (2000, 8, 1024, 16, 1.0),
                                              # kernel boundaries: row copy inside the small kernel up to
                                              # 128 pairs, the small kernel up to 1024 pairs
                                              (32, 4, 16, 16, 0.3), (43, 3, 16, 16, 0.3), (256, 4, 64, 8, 0.5),
                                              (205, 5, 64, 8, 0.5)])
def test_permute_parity(M, T, K, E, align, skew):
    rng = np.random.default_rng(T * 31 + E)
    ids = synth.topk_ids_random(rng, T, E, K, skew)
    H = 256
    xq = synth.e4m3_codes(rng, (T, H))
    xsf = synth.act_scale_codes(rng, (T, H // 128))
    p = O.permute(ids, E, align)
    U = M.msum_upper(T, K, E, align)
    assert U == p["U"]
    d_sorted = torch.empty(U, dtype=torch.int32, device="cuda")
    d_eids = torch.empty(U, dtype=torch.int32, device="cuda")
    d_inv = torch.empty(T, K, dtype=torch.int32, device="cuda")
    d_ms = torch.empty(1, dtype=torch.int32, device="cuda")
    d_cnt = torch.empty(E, dtype=torch.int32, device="cuda")
    d_xp = torch.full((U, H), 0xAA, dtype=torch.uint8, device="cuda")
    d_xpsf = torch.zeros(M.act_sf_tiled_bytes(U, H // 128, align), dtype=torch.uint8, device="cuda")
    ws = M.new_workspace(T, H, 256, E, K, align)
    M.permute(dev(ids), E, align, d_sorted, d_eids, d_inv, d_ms, ws, expert_counts=d_cnt, x_q=dev(xq),
              x_sf=dev(xsf), x_perm=d_xp, x_perm_sf=d_xpsf)
    assert M.get_error(ws) == M.OK
    assert int(d_ms.item()) == p["m_sum"]
    assert np.array_equal(d_sorted.cpu().numpy(), p["sorted_token_ids"])
    assert np.array_equal(d_eids.cpu().numpy(), p["expert_ids"])
    assert np.array_equal(d_cnt.cpu().numpy(), p["expert_counts"])
    inv = p["inv_perm"]
    assert np.array_equal(d_inv.cpu().numpy(), inv)
    xp = d_xp.cpu().numpy()
    assert np.array_equal(xp[inv.reshape(-1)], np.repeat(xq, K, axis=0))
    psf = M.act_sf_untile(d_xpsf.cpu().numpy(), U, H // 128, align)
    assert np.array_equal(psf[inv.reshape(-1)], np.repeat(xsf, K, axis=0))


def test_permute_empty_batch(M):
    T, K, E, align = 0, 4, 16, 16
    U = M.msum_upper(T, K, E, align)
    d_sorted = torch.zeros(U, dtype=torch.int32, device="cuda")
    d_eids = torch.zeros(U, dtype=torch.int32, device="cuda")
    d_ms = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    keep = torch.zeros(1, 1, dtype=torch.int32, device="cuda")   # non-null placeholders for the empty [0, K] arrays
    M.lib().moe_permute(keep.data_ptr(), T, K, E, align, d_sorted.data_ptr(), d_eids.data_ptr(), keep.data_ptr(),
                        d_ms.data_ptr(), None, None, None, 0, None, None, ws.data_ptr(), ws.numel(),
                        torch.cuda.current_stream().cuda_stream)
    assert M.get_error(ws) == M.OK
    assert int(d_ms.item()) == 0
    assert (d_eids.cpu().numpy() == -1).all() and (d_sorted.cpu().numpy() == 0).all()


def test_permute_reports_bad_expert_id(M):
    ids = np.array([[0, 1], [2, 9]], dtype=np.int32)        # 9 >= E
    E, K, align = 4, 2, 1
    U = M.msum_upper(2, K, E, align)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    bufs = [torch.empty(U, dtype=torch.int32, device="cuda") for _ in range(2)]
    M.permute(dev(ids), E, align, bufs[0], bufs[1], torch.empty(2, K, dtype=torch.int32, device="cuda"),
              torch.empty(1, dtype=torch.int32, device="cuda"), ws)
    assert M.get_error(ws) == M.ERR_DEVICE_INDEX
    assert M.get_error(ws) == M.OK                         # cleared by the read


# ------------------------------------------------------------------------------------------ grouped GEMMs

def _gemm_case(T, K, E, H, I, align, seed, skew=0.5, fmt="mxfp4", wide=False):
    rng = np.random.default_rng(seed)
    wl = synth.custom(T=T, H=H, I=I, E=E, K=K, align=align, seed=seed, fmt=fmt, wide_scales=wide)
    ids = synth.topk_ids_random(rng, T, E, K, skew)
    stack = synth.all_expert_weights(wl)
    return wl, rng, ids, stack


L1_CASES = [(8, 4, 16, 512, 256, 16), (37, 4, 16, 512, 256, 16), (200, 6, 32, 1024, 512, 64), (64, 4, 8, 512, 384, 1),
            (300, 2, 4, 256, 256, 128), (41, 3, 8, 640, 256, 32)]
# "wide": every E4M3 activation code (zeros, subnormals, the top binade), activation scales 2^-120 .. 2^10,
# MXFP4 block scales 2^-30 .. 2^4, NVFP4 scale codes 0x01 .. 0x7E
# NVFP4 with 128-row blocks runs on CTA pairs over quads of blocks: experts with one, two and more
# than four blocks (quads holding several experts, whole quads of one expert), padding-only blocks
# (align 256) and a single partial quad
PAIR_CASES = [(1200, 4, 8, 512, 256, 128), (600, 6, 16, 1024, 512, 256), (130, 1, 1, 256, 256, 128),
              (700, 4, 8, 384, 256, 128)]   # H = 384: W2's last tile is half a tile (the odd CTA's rows zero)
L1_PARAMS = ([c + ("mxfp4", False) for c in L1_CASES] + [c + ("nvfp4", False) for c in L1_CASES[:5]] +
             [L1_CASES[i] + (f, True) for i in (1, 2, 4) for f in ("mxfp4", "nvfp4")] +
             [c + ("nvfp4", False) for c in PAIR_CASES] + [PAIR_CASES[0] + ("nvfp4", True)])


@pytest.mark.parametrize("T,K,E,H,I,align,fmt,wide", L1_PARAMS)
def test_l1_swiglu_parity(M, T, K, E, H, I, align, fmt, wide):
    wl, rng, ids, stack = _gemm_case(T, K, E, H, I, align, seed=T + H, fmt=fmt, wide=wide)
    xq = synth.e4m3_codes(rng, (T, H), wide)
    xsf = synth.act_scale_codes(rng, (T, H // 128), wide)
    w13, _ = device_weights(M, stack, fmt)
    U = M.msum_upper(T, K, E, align)
    d_sorted = torch.empty(U, dtype=torch.int32, device="cuda")
    d_eids = torch.empty(U, dtype=torch.int32, device="cuda")
    d_inv = torch.empty(T, K, dtype=torch.int32, device="cuda")
    d_ms = torch.empty(1, dtype=torch.int32, device="cuda")
    d_xp = torch.zeros(U, H, dtype=torch.uint8, device="cuda")
    d_xpsf = torch.zeros(M.act_sf_tiled_bytes(U, H // 128, align), dtype=torch.uint8, device="cuda")
    ws = M.new_workspace(T, H, I, E, K, align)
    M.permute(dev(ids), E, align, d_sorted, d_eids, d_inv, d_ms, ws, x_q=dev(xq), x_sf=dev(xsf), x_perm=d_xp,
              x_perm_sf=d_xpsf)
    d_hq = torch.zeros(U, I, dtype=torch.uint8, device="cuda")
    d_hsf = torch.zeros(M.act_sf_tiled_bytes(U, I // 128, align), dtype=torch.uint8, device="cuda")
    M.grouped_gemm_l1_swiglu(d_xp, d_xpsf, d_eids, d_ms, T, K, H, I, E, align, w13, d_hq, d_hsf, ws)
    assert M.get_error(ws) == M.OK
    p = O.permute(ids, E, align)
    hq = d_hq.cpu().numpy()
    hsf = M.act_sf_untile(d_hsf.cpu().numpy(), U, I // 128, align)
    n_codes = n_same = 0
    for e in range(E):
        rows = np.where(p["expert_ids"] == e)[0]
        if rows.size == 0:
            continue
        toks = p["sorted_token_ids"][rows] // K
        W13 = O.dequant_weight(stack["w13_q"][e], stack["w13_sf"][e],
                               None if stack["w13_ts"] is None else stack["w13_ts"][e], fmt)
        h, hq_ref, hsf_ref = O.expert_l1_swiglu(O.dequant_fp8_groups(xq[toks], xsf[toks]), W13, I)
        got = O.dequant_fp8_groups(hq[rows], hsf[rows])
        gmax = np.abs(h).reshape(len(rows), I // 128, 128).max(axis=2).repeat(128, axis=1)
        bound = np.abs(h) * 2.0 ** -4 + gmax * 2.0 ** -12 + 1e-30
        bad = np.abs(got - h) > bound
        assert not bad.any(), f"expert {e}: {bad.sum()} values off; worst {np.abs(got - h).max():.3e}"
        # code identity over groups whose h is in fp32's normal range (below it the kernel's fp32 h
        # carries fewer bits than the codes; the absolute bound above covers those groups)
        normal = gmax >= 2.0 ** -90
        n_codes += int(normal.sum())
        n_same += int(((hq[rows] == hq_ref) & normal).sum())
    assert n_same >= 0.97 * n_codes, f"only {n_same}/{n_codes} E4M3 codes identical"


L2_CASES = [(8, 4, 16, 512, 256, 16), (37, 4, 16, 512, 256, 16), (200, 6, 32, 1024, 512, 64), (64, 4, 8, 384, 512, 1),
            (300, 2, 4, 256, 256, 128)]
L2_PARAMS = ([c + ("mxfp4", False) for c in L2_CASES] + [c + ("nvfp4", False) for c in L2_CASES] +
             [L2_CASES[i] + (f, True) for i in (1, 2, 3) for f in ("mxfp4", "nvfp4")] +
             [c + ("nvfp4", False) for c in PAIR_CASES] + [PAIR_CASES[1] + ("nvfp4", True)])


@pytest.mark.parametrize("T,K,E,H,I,align,fmt,wide", L2_PARAMS)
def test_l2_parity(M, T, K, E, H, I, align, fmt, wide):
    wl, rng, ids, stack = _gemm_case(T, K, E, H, I, align, seed=7 * T + I, fmt=fmt, wide=wide)
    _, w2 = device_weights(M, stack, fmt)
    U = M.msum_upper(T, K, E, align)
    hq = synth.e4m3_codes(rng, (U, I), wide)
    hsf = synth.act_scale_codes(rng, (U, I // 128), wide)
    d_sorted = torch.empty(U, dtype=torch.int32, device="cuda")
    d_eids = torch.empty(U, dtype=torch.int32, device="cuda")
    d_inv = torch.empty(T, K, dtype=torch.int32, device="cuda")
    d_ms = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = M.new_workspace(T, H, I, E, K, align)
    M.permute(dev(ids), E, align, d_sorted, d_eids, d_inv, d_ms, ws)
    d_y = torch.zeros(U, H, dtype=torch.bfloat16, device="cuda")
    M.grouped_gemm_l2(dev(hq), dev(M.act_sf_tile(hsf, align)), d_eids, d_ms, T, K, H, I, E, align, w2, d_y, ws)
    assert M.get_error(ws) == M.OK
    p = O.permute(ids, E, align)
    y = F.bf16_to_f64(host_bits(d_y))
    for e in range(E):
        rows = np.where(p["expert_ids"] == e)[0]
        if rows.size == 0:
            continue
        W2 = O.dequant_weight(stack["w2_q"][e], stack["w2_sf"][e],
                              None if stack["w2_ts"] is None else stack["w2_ts"][e], fmt)
        hd = O.dequant_fp8_groups(hq[rows], hsf[rows])
        exact = hd @ W2.T                      # float64, before the bf16 rounding
        terms = np.abs(hd) @ np.abs(W2).T      # sum of |products|: scale of the fp32 accumulation error
        # one bf16 step of the exact value (the final rounding) + fp32 accumulation error
        ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(exact), 1e-38))[1] - 8)
        bad = np.abs(y[rows] - exact) > ulp + 2.0 ** -16 * terms
        assert not bad.any(), f"expert {e}: {bad.sum()} outputs beyond tolerance"
        # rounding identity on outputs in the fp32/bf16 normal range (below it the absolute bound applies)
        normal = np.abs(exact) >= 2.0 ** -100
        ud = bf16_ulp_diff(host_bits(d_y)[rows], O.expert_l2(hq[rows], hsf[rows], W2))
        assert (ud[normal] <= 1).mean() > 0.999


def test_unpermute_reduce_parity(M):
    rng = np.random.default_rng(11)
    for T, K, H in [(8, 6, 7168), (129, 4, 512), (1, 1, 128)]:
        Mrows = T * K + 37
        y = synth.bf16_rows(rng, Mrows, H)
        inv = np.array([rng.choice(Mrows, K, replace=False) for _ in range(T)], dtype=np.int32)
        w = synth.topk_weights_random(rng, T, K)
        out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
        M.unpermute_reduce(dev_bf16(y), dev(inv), dev(w), out)
        ref = O.unpermute_reduce(y, inv, w.astype(np.float64))
        assert bf16_ulp_diff(host_bits(out), ref).max() <= 1


# ------------------------------------------------------------------------------------------ whole layer

def _run_forward(M, w, inp, stack):
    T = inp["hidden"].shape[0]
    w13, w2 = device_weights(M, stack, w.fmt)
    ws = M.new_workspace(T, w.H, w.I, w.E, w.K, w.align)
    U = M.msum_upper(T, w.K, w.E, w.align)
    # outputs poisoned, so that anything left unwritten shows
    o = dict(out=torch.full((T, w.H), float("nan"), dtype=torch.bfloat16, device="cuda"),
             topk_ids=torch.full((T, w.K), -1, dtype=torch.int32, device="cuda"),
             topk_w=torch.full((T, w.K), float("nan"), dtype=torch.float32, device="cuda"),
             sorted_token_ids=torch.full((U,), -7, dtype=torch.int32, device="cuda"),
             expert_ids=torch.full((U,), -7, dtype=torch.int32, device="cuda"),
             inv_perm=torch.full((T, w.K), -7, dtype=torch.int32, device="cuda"),
             m_sum=torch.full((1,), -7, dtype=torch.int32, device="cuda"))
    M.forward(dev_bf16(inp["hidden"]), dev(inp["w_gate"]),
              None if inp["gate_bias"] is None else dev(inp["gate_bias"]),
              None if inp["e_score_bias"] is None else dev(inp["e_score_bias"]), w.I, w.K, w.align, w.score_fn,
              w.renormalize, w13, w2, o["out"], ws, topk_ids=o["topk_ids"], topk_w=o["topk_w"],
              sorted_token_ids=o["sorted_token_ids"], expert_ids=o["expert_ids"], inv_perm=o["inv_perm"],
              m_sum=o["m_sum"])
    assert M.get_error(ws) == M.OK
    return {k: v.cpu() for k, v in o.items()}


def _check_perm_invariants(g, ids, E, align):
    """Properties of an expert-contiguous permute that hold for any routing."""
    T, K = ids.shape
    inv = g["inv_perm"].reshape(-1)
    ms = int(g["m_sum"].reshape(-1)[0])
    srt, eid = g["sorted_token_ids"], g["expert_ids"]
    assert len(set(inv.tolist())) == T * K and inv.max() < ms and ms % align == 0
    assert np.array_equal(srt[inv], np.arange(T * K)) and np.array_equal(eid[inv], ids.reshape(-1))
    real = eid[:ms][eid[:ms] >= 0]
    assert (np.diff(real) >= 0).all() and (eid >= 0).sum() == T * K


ORACLE_THREADS = 16


def _straddle_explainer(M, w, inp, stack, g):
    """Accounts for the tokens whose output misses the 2e-2 x RMS bound (the full workloads hold ~10^8
    outputs, and a few land there).  The kernel requantises h = silu(gate) * up from fp32 sums, the
    oracle from exact ones; where the exact h lies within the fp32 error of an E4M3 rounding
    boundary the two round to neighbouring codes, and the L2 row then differs by one code step times
    a column of W2.  For each such token this checks, on the kernel's own h codes (moe_forward
    equals the stage calls bit for bit, asserted here):
      * every h value of every one of the token's rows is within the L1 tolerance of the oracle's
        exact h (half an E4M3 step plus the fp32 accumulation slack), so each differing code is a
        legitimate rounding of the exact value;
      * the token's output equals the oracle's L2 and weighted reduce computed from those codes,
        within the 2e-2 x RMS bound."""
    st = _run_stages(M, w, inp, stack, keep=True)
    assert torch.equal(st["out"].view(torch.int16).cpu(), torch.from_numpy(g["out"].view(np.int16))), \
        "moe_forward and the stage calls disagree"
    U = M.msum_upper(w.T, w.K, w.E, w.align)
    hq = st["hq"].cpu().numpy()
    hsf = M.act_sf_untile(st["hsf"].cpu().numpy(), U, w.I // 128, w.align)
    xq, xsf = st["xq"].cpu().numpy(), st["xsf"].cpu().numpy()
    inv, tw = st["inv"].cpu().numpy(), st["tw"].cpu().numpy().astype(np.float64)
    ids = st["ids"].cpu().numpy()
    prov = _stack_provider(stack)

    def explain(tokens, rms):
        by_e = {}
        for t in tokens:
            for k in range(w.K):
                by_e.setdefault(int(ids[t, k]), []).append((int(t), k))
        y = {}
        flips = 0
        for e, pairs in by_e.items():
            ew = prov(e)
            W13 = O.dequant_weight(ew["w13_q"], ew["w13_sf"], ew["w13_ts"], w.fmt)
            W2 = O.dequant_weight(ew["w2_q"], ew["w2_sf"], ew["w2_ts"], w.fmt)
            ts = np.array([t for t, _ in pairs])
            rows = np.array([inv[t, k] for t, k in pairs])
            h, hq_ref, _ = O.expert_l1_swiglu(O.dequant_fp8_groups(xq[ts], xsf[ts]), W13, w.I)
            got = O.dequant_fp8_groups(hq[rows], hsf[rows])
            gmax = np.abs(h).reshape(len(rows), w.I // 128, 128).max(axis=2).repeat(128, axis=1)
            bad = np.abs(got - h) > np.abs(h) * 2.0 ** -4 + gmax * 2.0 ** -12 + 1e-30
            assert not bad.any(), f"expert {e}: h beyond the L1 tolerance"
            flips += int((hq[rows] != hq_ref).sum())
            yk = F.bf16_to_f64(O.expert_l2(hq[rows], hsf[rows], W2))
            for j, (t, k) in enumerate(pairs):
                y[(t, k)] = yk[j]
        for t in tokens:
            acc = sum(tw[t, k] * y[(int(t), k)] for k in range(w.K))
            ref_t = F.round_bf16_rne(acc)
            err = np.abs(F.bf16_to_f64(g["out"][t]) - F.bf16_to_f64(ref_t)).max()
            assert err <= OUT_TOL * rms, f"token {t}: {err / rms:.3e} x RMS even from the kernel's h codes"
        print(f"{w.name}: {len(tokens)} token(s) beyond 2e-2 x RMS, all from {flips} h code(s) rounded "
              f"the other way at an E4M3 rounding boundary")

    return explain


def _check_forward(M, w, T=None, tokens=None, explain_straddles=False):
    """The whole layer against the oracle: every token (or the given ones), every index output."""
    inp = synth.layer_inputs(w, T)
    T = inp["hidden"].shape[0]
    stack = synth.all_expert_weights(w)
    g = {k: (v.view(torch.int16) if v.dtype == torch.bfloat16 else v).numpy()
         for k, v in _run_forward(M, w, inp, stack).items()}
    g["out"] = g["out"].view(np.uint16)
    prov = _stack_provider(stack)

    def oracle(toks, routing=None):
        return O.forward(inp, prov, w.fmt, w.K, w.align, w.score_fn, w.renormalize, tokens=toks, routing=routing,
                         workers=ORACLE_THREADS)

    ref = oracle(tokens)
    explain = _straddle_explainer(M, w, inp, stack, g) if explain_straddles else None
    rel, counts = check_layer(M, w, inp, g, ref, oracle, perm_fn=lambda ids: O.permute(ids, w.E, w.align),
                              explain=explain)
    _check_perm_invariants(g, g["topk_ids"], w.E, w.align)
    return rel, g, inp, stack


@pytest.mark.parametrize("T", [None, 1, 5, 77])
def test_forward_tiny(M, T):
    _check_forward(M, synth.WORKLOADS["tiny"], T=T)


def test_forward_align_one_multi_expert_blocks(M):
    w = synth.custom(T=23, H=512, I=256, E=16, K=4, align=1, score_fn="sqrt_softplus", e_bias=True, seed=5)
    _check_forward(M, w)


def test_forward_deterministic(M):
    w = synth.WORKLOADS["tiny"]
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    a = _run_forward(M, w, inp, stack)
    b = _run_forward(M, w, inp, stack)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_forward_decode_full(M):
    # the pages' decode shape, every token checked against the full oracle
    rel, *_ = _check_forward(M, synth.WORKLOADS["decode"])
    assert rel < OUT_TOL


@pytest.mark.parametrize("T,E,K,H", [(20, 8, 4, 512), (32, 4, 4, 512), (9, 2, 1, 512), (24, 8, 4, 384)])
def test_forward_nvfp4_pair_fused_reduce(M, T, E, K, H):
    # NVFP4 with 128-row blocks runs on CTA pairs; up to 32 tokens every expert holds one block (a
    # lone block, split by rows over the pair as an M = 128 MMA) and the weighted reduce runs in
    # the L2 epilogue, after both halves of each row are stored
    w = synth.custom(T=T, H=H, I=256, E=E, K=K, align=128, score_fn="sqrt_softplus", e_bias=True, fmt="nvfp4",
                     seed=60 + T)
    _check_forward(M, w)
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    a = _run_forward(M, w, inp, stack)["out"]
    b = _run_stages(M, w, inp, stack)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_forward_tiny_nvfp4(M):
    w = synth.custom(T=40, H=512, I=256, E=16, K=4, align=16, score_fn="sqrt_softplus", e_bias=True, fmt="nvfp4",
                     gate_offset="zipf", seed=9)
    _check_forward(M, w)


@pytest.mark.parametrize("name", ["batched", "prefill", "skewed"])
def test_forward_full_workload(M, name):
    # every token of the workload against the oracle (every GEMM row block of every expert, and
    # the last items of the dynamic work queue, hold some checked token's rows)
    rel, g, _, _ = _check_forward(M, synth.WORKLOADS[name], explain_straddles=True)
    assert rel < OUT_TOL


def test_forward_pad_only_row_blocks(M):
    # align 256 gives 128-row GEMM blocks; experts with few rows leave blocks that hold only padding
    w = synth.custom(T=12, H=256, I=256, E=8, K=2, align=256, score_fn="sqrt_softplus", e_bias=True, seed=11)
    _check_forward(M, w)


def _run_stages(M, w, inp, stack, keep=False):
    """The layer as five separate C-ABI calls (route, permute, L1, L2, reduce); the output, or with
    ``keep`` every intermediate as device tensors."""
    T = inp["hidden"].shape[0]
    w13, w2 = device_weights(M, stack, w.fmt)
    ws = M.new_workspace(T, w.H, w.I, w.E, w.K, w.align)
    U = M.msum_upper(T, w.K, w.E, w.align)
    i32 = dict(dtype=torch.int32, device="cuda")
    u8 = dict(dtype=torch.uint8, device="cuda")
    ids, tw = torch.empty(T, w.K, **i32), torch.empty(T, w.K, dtype=torch.float32, device="cuda")
    xq, xsf = torch.empty(T, w.H, **u8), torch.empty(T, w.H // 128, **u8)
    M.route(dev_bf16(inp["hidden"]), dev(inp["w_gate"]), None if inp["gate_bias"] is None else dev(inp["gate_bias"]),
            None if inp["e_score_bias"] is None else dev(inp["e_score_bias"]), w.K, w.score_fn, w.renormalize,
            ids, tw, ws, x_q=xq, x_sf=xsf)
    srt, eid, inv, ms = torch.empty(U, **i32), torch.empty(U, **i32), torch.empty(T, w.K, **i32), torch.empty(1, **i32)
    xp = torch.zeros(U, w.H, **u8)
    xpsf = torch.zeros(M.act_sf_tiled_bytes(U, w.H // 128, w.align), **u8)
    M.permute(ids, w.E, w.align, srt, eid, inv, ms, ws, x_q=xq, x_sf=xsf, x_perm=xp, x_perm_sf=xpsf)
    hq = torch.zeros(U, w.I, **u8)
    hsf = torch.zeros(M.act_sf_tiled_bytes(U, w.I // 128, w.align), **u8)
    M.grouped_gemm_l1_swiglu(xp, xpsf, eid, ms, T, w.K, w.H, w.I, w.E, w.align, w13, hq, hsf, ws)
    y = torch.zeros(U, w.H, dtype=torch.bfloat16, device="cuda")
    M.grouped_gemm_l2(hq, hsf, eid, ms, T, w.K, w.H, w.I, w.E, w.align, w2, y, ws)
    out = torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda")
    M.unpermute_reduce(y, inv, tw, out)
    assert M.get_error(ws) == M.OK
    if keep:
        return dict(out=out, ids=ids, tw=tw, xq=xq, xsf=xsf, inv=inv, hq=hq, hsf=hsf, y=y)
    return out.cpu()


@pytest.mark.parametrize("case", ["tiny", "tiny77", "align1", "decode", "tiny_nvfp4"])
def test_forward_matches_stage_calls(M, case):
    # moe_forward fuses launches (one L1+L2 launch, the reduce in the L2 epilogue for small T); the
    # arithmetic is the same as the separate calls', so the outputs agree bit for bit
    T = None
    if case == "align1":
        w = synth.custom(T=23, H=512, I=256, E=16, K=4, align=1, score_fn="sqrt_softplus", e_bias=True, seed=5)
    elif case == "tiny_nvfp4":
        w = synth.custom(T=40, H=512, I=256, E=16, K=4, align=16, score_fn="sqrt_softplus", e_bias=True,
                         fmt="nvfp4", seed=9)
    else:
        w = synth.WORKLOADS["decode" if case == "decode" else "tiny"]
        T = 77 if case == "tiny77" else None
    inp = synth.layer_inputs(w, T)
    stack = synth.all_expert_weights(w)
    a = _run_forward(M, w, inp, stack)["out"]
    b = _run_stages(M, w, inp, stack)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("case", ["tiny", "align1", "pad_only", "nvfp4"])
def test_grouped_ffn_matches_separate_gemms(M, case):
    # moe_grouped_ffn = moe_grouped_gemm_l1_swiglu then moe_grouped_gemm_l2, bit for bit; called twice
    # in a row, since its per-row-block counters must be back at zero after each call
    if case == "align1":
        w = synth.custom(T=23, H=512, I=256, E=16, K=4, align=1, score_fn="sqrt_softplus", e_bias=True, seed=5)
    elif case == "pad_only":
        w = synth.custom(T=12, H=256, I=256, E=8, K=2, align=256, score_fn="sqrt_softplus", e_bias=True, seed=11)
    elif case == "nvfp4":
        w = synth.custom(T=40, H=512, I=256, E=16, K=4, align=16, score_fn="sqrt_softplus", e_bias=True,
                         fmt="nvfp4", seed=9)
    else:
        w = synth.WORKLOADS["tiny"]
    inp = synth.layer_inputs(w)
    T = inp["hidden"].shape[0]
    stack = synth.all_expert_weights(w)
    w13, w2 = device_weights(M, stack, w.fmt)
    ws = M.new_workspace(T, w.H, w.I, w.E, w.K, w.align)
    U = M.msum_upper(T, w.K, w.E, w.align)
    i32 = dict(dtype=torch.int32, device="cuda")
    u8 = dict(dtype=torch.uint8, device="cuda")
    ids, tw = torch.empty(T, w.K, **i32), torch.empty(T, w.K, dtype=torch.float32, device="cuda")
    xq, xsf = torch.empty(T, w.H, **u8), torch.empty(T, w.H // 128, **u8)
    M.route(dev_bf16(inp["hidden"]), dev(inp["w_gate"]), None if inp["gate_bias"] is None else dev(inp["gate_bias"]),
            None if inp["e_score_bias"] is None else dev(inp["e_score_bias"]), w.K, w.score_fn, w.renormalize,
            ids, tw, ws, x_q=xq, x_sf=xsf)
    srt, eid, inv, ms = torch.empty(U, **i32), torch.empty(U, **i32), torch.empty(T, w.K, **i32), torch.empty(1, **i32)
    xp = torch.zeros(U, w.H, **u8)
    xpsf = torch.zeros(M.act_sf_tiled_bytes(U, w.H // 128, w.align), **u8)
    M.permute(ids, w.E, w.align, srt, eid, inv, ms, ws, x_q=xq, x_sf=xsf, x_perm=xp, x_perm_sf=xpsf)
    sfb = M.act_sf_tiled_bytes(U, w.I // 128, w.align)
    hq0, hsf0 = torch.zeros(U, w.I, **u8), torch.zeros(sfb, **u8)
    y0 = torch.zeros(U, w.H, dtype=torch.bfloat16, device="cuda")
    M.grouped_gemm_l1_swiglu(xp, xpsf, eid, ms, T, w.K, w.H, w.I, w.E, w.align, w13, hq0, hsf0, ws)
    M.grouped_gemm_l2(hq0, hsf0, eid, ms, T, w.K, w.H, w.I, w.E, w.align, w2, y0, ws)
    ms_h = int(ms.item())
    real = (eid[:ms_h] >= 0).nonzero().flatten()
    for _ in range(2):
        hq, hsf = torch.full((U, w.I), 0x7F, **u8), torch.zeros(sfb, **u8)
        y = torch.zeros(U, w.H, dtype=torch.bfloat16, device="cuda")
        M.grouped_ffn(xp, xpsf, eid, ms, T, w.K, w.H, w.I, w.E, w.align, w13, w2, hq, hsf, y, ws)
        assert M.get_error(ws) == M.OK
        assert torch.equal(hq[real], hq0[real])
        assert torch.equal(y[real].view(torch.int16), y0[real].view(torch.int16))
        h_rows = M.act_sf_untile(hsf.cpu().numpy(), U, w.I // 128, w.align)
        h_rows0 = M.act_sf_untile(hsf0.cpu().numpy(), U, w.I // 128, w.align)
        assert np.array_equal(h_rows[real.cpu().numpy()], h_rows0[real.cpu().numpy()])


# ------------------------------------------------------------------------------------------ L1 token-order input

GATHER_CASES = [(8, 6, 32, 7168, 2048, 16, "mxfp4"), (37, 4, 16, 512, 256, 16, "mxfp4"),
                (300, 2, 4, 256, 256, 128, "mxfp4"), (64, 4, 8, 512, 384, 1, "mxfp4"), (41, 3, 8, 640, 256, 32, "mxfp4"),
                (600, 6, 16, 1024, 512, 256, "mxfp4"), (200, 6, 32, 1024, 512, 64, "nvfp4"),
                (37, 4, 16, 512, 256, 16, "nvfp4"), (1, 1, 4, 256, 256, 16, "mxfp4"),
                (1200, 4, 8, 512, 256, 128, "nvfp4")]


@pytest.mark.parametrize("T,K,E,H,I,align,fmt", GATHER_CASES)
def test_l1_token_order_input_matches_permuted_rows(M, T, K, E, H, I, align, fmt):
    # The L1 call with a_is_permuted = 0 reads each permuted row's activation through sorted_token_ids
    # (MegaMoE page, 路径 A) instead of from the x_perm copy: same rows, same arithmetic, same bits.
    # moe_permute with only the scales gives the same scale layout as with the row copy.
    wl, rng, ids, stack = _gemm_case(T, K, E, H, I, align, seed=3 * T + H, fmt=fmt)
    xq = synth.e4m3_codes(rng, (T, H))
    xsf = synth.act_scale_codes(rng, (T, H // 128))
    w13, w2 = device_weights(M, stack, fmt)
    U = M.msum_upper(T, K, E, align)
    i32 = dict(dtype=torch.int32, device="cuda")
    u8 = dict(dtype=torch.uint8, device="cuda")
    srt, eid, inv, ms = torch.empty(U, **i32), torch.empty(U, **i32), torch.empty(T, K, **i32), torch.empty(1, **i32)
    sfb = M.act_sf_tiled_bytes(U, H // 128, align)
    xp, xpsf = torch.zeros(U, H, **u8), torch.zeros(sfb, **u8)
    ws = M.new_workspace(T, H, I, E, K, align)
    d_xq, d_xsf = dev(xq), dev(xsf)
    M.permute(dev(ids), E, align, srt, eid, inv, ms, ws, x_q=d_xq, x_sf=d_xsf, x_perm=xp, x_perm_sf=xpsf)
    xpsf2 = torch.zeros(sfb, **u8)
    M.permute(dev(ids), E, align, srt, eid, inv, ms, ws, x_sf=d_xsf, x_perm_sf=xpsf2)
    assert torch.equal(xpsf, xpsf2)
    hsfb = M.act_sf_tiled_bytes(U, I // 128, align)
    hq0, hsf0 = torch.full((U, I), 0x7F, **u8), torch.zeros(hsfb, **u8)
    M.grouped_gemm_l1_swiglu(xp, xpsf, eid, ms, T, K, H, I, E, align, w13, hq0, hsf0, ws)
    hq1, hsf1 = torch.full((U, I), 0x7E, **u8), torch.zeros(hsfb, **u8)
    M.grouped_gemm_l1_swiglu(d_xq, d_xsf, eid, ms, T, K, H, I, E, align, w13, hq1, hsf1, ws, sorted_token_ids=srt)
    assert M.get_error(ws) == M.OK
    p = O.permute(ids, E, align)
    real = np.where(p["expert_ids"] >= 0)[0]
    assert np.array_equal(hq1.cpu().numpy()[real], hq0.cpu().numpy()[real])
    a0 = M.act_sf_untile(hsf0.cpu().numpy(), U, I // 128, align)[real]
    a1 = M.act_sf_untile(hsf1.cpu().numpy(), U, I // 128, align)[real]
    assert np.array_equal(a0, a1)
    # both GEMMs in one call from the token-order input, twice in a row
    y0 = torch.zeros(U, H, dtype=torch.bfloat16, device="cuda")
    M.grouped_gemm_l2(hq0, hsf0, eid, ms, T, K, H, I, E, align, w2, y0, ws)
    for _ in range(2):
        hq2, hsf2 = torch.full((U, I), 0x7D, **u8), torch.zeros(hsfb, **u8)
        y2 = torch.full((U, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        M.grouped_ffn(d_xq, d_xsf, eid, ms, T, K, H, I, E, align, w13, w2, hq2, hsf2, y2, ws, sorted_token_ids=srt)
        assert M.get_error(ws) == M.OK
        rr = torch.from_numpy(real).cuda()
        assert torch.equal(hq2[rr], hq0[rr])
        assert torch.equal(y2[rr].view(torch.int16), y0[rr].view(torch.int16))
