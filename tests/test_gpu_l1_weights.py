"""GPU parity of the routing-weight placement in the L1 epilogue (MegaMoE page, 二、阶段 3: the
SwiGLU output is silu(gate) * up * topk_weight before the requant; 阶段 5 then sums the rows
without weights) against the float64 oracle run with the same placement.

Tolerances as in test_gpu_parity: the requantised h within half an E4M3 step of the exact value
(plus fp32 slack), the layer output within 2e-2 x RMS, and bit-identity between moe_forward_l1_weighted
and the same path as separate C-ABI calls.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import OUT_TOL, bf16_ulp_diff, check_out, dev, dev_bf16, device_weights, ensure_lib, host_bits
from oracle import moe as O

pytestmark = pytest.mark.gpu

I32 = dict(dtype=torch.int32, device="cuda")
U8 = dict(dtype=torch.uint8, device="cuda")


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_lib()


CASES = [(8, 4, 16, 512, 256, 16, "mxfp4"), (37, 4, 16, 512, 256, 16, "mxfp4"), (200, 6, 32, 1024, 512, 64, "mxfp4"),
         (64, 4, 8, 512, 384, 1, "mxfp4"), (300, 2, 4, 256, 256, 128, "mxfp4"), (37, 4, 16, 512, 256, 16, "nvfp4"),
         (200, 6, 32, 1024, 512, 64, "nvfp4")]


@pytest.mark.parametrize("T,K,E,H,I,align,fmt", CASES)
def test_l1_weighted_parity(M, T, K, E, H, I, align, fmt):
    rng = np.random.default_rng(T + 3 * H)
    wl = synth.custom(T=T, H=H, I=I, E=E, K=K, align=align, seed=T + H, fmt=fmt)
    ids = synth.topk_ids_random(rng, T, E, K, 0.5)
    stack = synth.all_expert_weights(wl)
    xq = synth.e4m3_codes(rng, (T, H))
    xsf = synth.act_scale_codes(rng, (T, H // 128))
    tw = synth.topk_weights_random(rng, T, K)
    w13, _ = device_weights(M, stack, fmt)
    U = M.msum_upper(T, K, E, align)
    srt, eid, inv, ms = torch.empty(U, **I32), torch.empty(U, **I32), torch.empty(T, K, **I32), torch.empty(1, **I32)
    xp = torch.zeros(U, H, **U8)
    xpsf = torch.zeros(M.act_sf_tiled_bytes(U, H // 128, align), **U8)
    ws = M.new_workspace(T, H, I, E, K, align)
    M.permute(dev(ids), E, align, srt, eid, inv, ms, ws, x_q=dev(xq), x_sf=dev(xsf), x_perm=xp, x_perm_sf=xpsf)
    hq_d = torch.zeros(U, I, **U8)
    hsf_d = torch.zeros(M.act_sf_tiled_bytes(U, I // 128, align), **U8)
    M.grouped_gemm_l1_swiglu_weighted(xp, xpsf, eid, ms, srt, dev(tw), T, K, H, I, E, align, w13, hq_d, hsf_d, ws)
    assert M.get_error(ws) == M.OK
    p = O.permute(ids, E, align)
    hq = hq_d.cpu().numpy()
    hsf = M.act_sf_untile(hsf_d.cpu().numpy(), U, I // 128, align)
    n_codes = n_same = 0
    for e in range(E):
        rows = np.where(p["expert_ids"] == e)[0]
        if rows.size == 0:
            continue
        pairs = p["sorted_token_ids"][rows]
        W13 = O.dequant_weight(stack["w13_q"][e], stack["w13_sf"][e],
                               None if stack["w13_ts"] is None else stack["w13_ts"][e], fmt)
        rw = tw.reshape(-1)[pairs].astype(np.float64)
        h, hq_ref, _ = O.expert_l1_swiglu(O.dequant_fp8_groups(xq[pairs // K], xsf[pairs // K]), W13, I, rw)
        got = O.dequant_fp8_groups(hq[rows], hsf[rows])
        gmax = np.abs(h).reshape(len(rows), I // 128, 128).max(axis=2).repeat(128, axis=1)
        bad = np.abs(got - h) > np.abs(h) * 2.0 ** -4 + gmax * 2.0 ** -12 + 1e-30
        assert not bad.any(), f"expert {e}: {bad.sum()} values off"
        n_codes += hq_ref.size
        n_same += int((hq[rows] == hq_ref).sum())
    assert n_same >= 0.97 * n_codes


def test_unweighted_reduce_parity(M):
    rng = np.random.default_rng(12)
    for T, K, H in [(8, 6, 7168), (129, 4, 512), (1, 1, 128)]:
        R = T * K + 5
        y = synth.bf16_rows(rng, R, H)
        inv = np.stack([rng.choice(R, K, replace=False) for _ in range(T)]).astype(np.int32)
        out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
        M.unpermute_reduce(dev_bf16(y), dev(inv), None, out)
        assert bf16_ulp_diff(host_bits(out), O.unpermute_reduce(y, inv, None)).max() <= 1


def _case(name):
    T = None
    if name == "align1":
        w = synth.custom(T=23, H=512, I=256, E=16, K=4, align=1, score_fn="sqrt_softplus", e_bias=True, seed=5)
    elif name == "nvfp4":
        w = synth.custom(T=40, H=512, I=256, E=16, K=4, align=16, score_fn="sqrt_softplus", e_bias=True,
                         fmt="nvfp4", seed=9)
    elif name == "tiny77":
        w, T = synth.WORKLOADS["tiny"], 77
    else:
        w = synth.WORKLOADS[name]
    return w, T


def _forward(M, w, inp, stack, weights_in_l1):
    T = inp["hidden"].shape[0]
    w13, w2 = device_weights(M, stack, w.fmt)
    ws = M.new_workspace(T, w.H, w.I, w.E, w.K, w.align)
    out = torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(T, w.K, **I32)
    M.forward(dev_bf16(inp["hidden"]), dev(inp["w_gate"]), None if inp["gate_bias"] is None else dev(inp["gate_bias"]),
              None if inp["e_score_bias"] is None else dev(inp["e_score_bias"]), w.I, w.K, w.align, w.score_fn,
              w.renormalize, w13, w2, out, ws, topk_ids=ids, weights_in_l1=weights_in_l1)
    assert M.get_error(ws) == M.OK
    return out.cpu(), ids.cpu().numpy()


@pytest.mark.parametrize("case", ["tiny", "tiny77", "align1", "nvfp4", "decode"])
def test_forward_l1_weighted_against_oracle(M, case):
    w, T = _case(case)
    inp = synth.layer_inputs(w, T)
    stack = synth.all_expert_weights(w)
    out, ids = _forward(M, w, inp, stack, True)
    ref = O.forward(inp, lambda e: {k: (v[e] if v is not None else None) for k, v in stack.items()}, w.fmt, w.K,
                    w.align, w.score_fn, w.renormalize, topk_w_dtype=np.float32, weights_in_l1=True)
    agree = (ids == ref["route"]["topk_ids"]).all(axis=1)           # near-ties may pick another expert
    assert agree.sum() >= len(agree) - max(1, len(agree) // 100)
    assert check_out(host_bits(out)[agree], ref["out"][agree]) < OUT_TOL


@pytest.mark.parametrize("case", ["tiny", "tiny77", "nvfp4", "decode"])
def test_forward_l1_weighted_matches_stage_calls(M, case):
    # the fused launches (one L1+L2 launch; the unweighted reduce in the L2 epilogue up to 32 tokens)
    # against route -> permute -> weighted L1 -> L2 -> unweighted reduce as separate calls
    w, T = _case(case)
    inp = synth.layer_inputs(w, T)
    T = inp["hidden"].shape[0]
    stack = synth.all_expert_weights(w)
    a, _ = _forward(M, w, inp, stack, True)
    w13, w2 = device_weights(M, stack, w.fmt)
    ws = M.new_workspace(T, w.H, w.I, w.E, w.K, w.align)
    U = M.msum_upper(T, w.K, w.E, w.align)
    ids, tw = torch.empty(T, w.K, **I32), torch.empty(T, w.K, dtype=torch.float32, device="cuda")
    xq, xsf = torch.empty(T, w.H, **U8), torch.empty(T, w.H // 128, **U8)
    M.route(dev_bf16(inp["hidden"]), dev(inp["w_gate"]), None if inp["gate_bias"] is None else dev(inp["gate_bias"]),
            None if inp["e_score_bias"] is None else dev(inp["e_score_bias"]), w.K, w.score_fn, w.renormalize,
            ids, tw, ws, x_q=xq, x_sf=xsf)
    srt, eid, inv, ms = torch.empty(U, **I32), torch.empty(U, **I32), torch.empty(T, w.K, **I32), torch.empty(1, **I32)
    xp = torch.zeros(U, w.H, **U8)
    xpsf = torch.zeros(M.act_sf_tiled_bytes(U, w.H // 128, w.align), **U8)
    M.permute(ids, w.E, w.align, srt, eid, inv, ms, ws, x_q=xq, x_sf=xsf, x_perm=xp, x_perm_sf=xpsf)
    hq = torch.zeros(U, w.I, **U8)
    hsf = torch.zeros(M.act_sf_tiled_bytes(U, w.I // 128, w.align), **U8)
    M.grouped_gemm_l1_swiglu_weighted(xp, xpsf, eid, ms, srt, tw, T, w.K, w.H, w.I, w.E, w.align, w13, hq, hsf, ws)
    y = torch.zeros(U, w.H, dtype=torch.bfloat16, device="cuda")
    M.grouped_gemm_l2(hq, hsf, eid, ms, T, w.K, w.H, w.I, w.E, w.align, w2, y, ws)
    b = torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda")
    M.unpermute_reduce(y, inv, None, b)
    assert M.get_error(ws) == M.OK
    assert torch.equal(a.view(torch.int16), b.cpu().view(torch.int16))
