"""GPU parity of the tiny-batch path (no sort: pair p = t*K + k on row 16p of the permuted buffers)
through the C ABI.

Index outputs are compared with the oracle's tiny-batch layout bit for bit.  The layer output must
equal moe_forward's (align 16) bit for bit: every row's arithmetic is the same wherever it sits, and
the reduce sums the same rows in the same k order; moe_forward itself is checked against the float64
oracle in test_gpu_parity.
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
ROWS = 16


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_lib()


def _case(name):
    if name.startswith("tiny"):
        return synth.WORKLOADS["tiny"], int(name[4:])
    if name.startswith("decode"):
        return synth.WORKLOADS["decode"], int(name[6:])
    w = synth.custom(T=3, H=512, I=256, E=16, K=4, align=16, score_fn="sqrt_softplus", e_bias=True, fmt="nvfp4",
                     seed=9)
    return w, 3


def _args(inp):
    return (dev_bf16(inp["hidden"]), dev(inp["w_gate"]), None if inp["gate_bias"] is None else dev(inp["gate_bias"]),
            None if inp["e_score_bias"] is None else dev(inp["e_score_bias"]))


def _forward(M, w, inp, stack, naive):
    T = inp["hidden"].shape[0]
    w13, w2 = device_weights(M, stack, w.fmt)
    ws = M.new_workspace(T, w.H, w.I, w.E, w.K, ROWS)
    U = M.msum_upper(T, w.K, w.E, ROWS)
    o = dict(out=torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda"), topk_ids=torch.empty(T, w.K, **I32),
             topk_w=torch.empty(T, w.K, dtype=torch.float32, device="cuda"), sorted_token_ids=torch.empty(U, **I32),
             expert_ids=torch.empty(U, **I32), inv_perm=torch.empty(T, w.K, **I32), m_sum=torch.empty(1, **I32))
    idx = {k: o[k] for k in o if k != "out"}
    if naive:
        M.forward_naive(*_args(inp), w.I, w.K, w.score_fn, w.renormalize, w13, w2, o["out"], ws, **idx)
    else:
        M.forward(*_args(inp), w.I, w.K, ROWS, w.score_fn, w.renormalize, w13, w2, o["out"], ws, **idx)
    assert M.get_error(ws) == M.OK
    return {k: v.cpu() for k, v in o.items()}


@pytest.mark.parametrize("case", ["tiny1", "tiny2", "tiny4", "decode1", "decode2", "decode8", "decode16", "nvfp4"])
def test_forward_naive_equals_forward(M, case):
    w, T = _case(case)
    inp = synth.layer_inputs(w, T)
    stack = synth.all_expert_weights(w)
    a = _forward(M, w, inp, stack, False)
    b = _forward(M, w, inp, stack, True)
    assert torch.equal(a["out"].view(torch.int16), b["out"].view(torch.int16))
    assert torch.equal(a["topk_ids"], b["topk_ids"]) and torch.equal(a["topk_w"], b["topk_w"])
    p = O.permute_naive(b["topk_ids"].numpy(), w.E, ROWS)
    for k in ("sorted_token_ids", "expert_ids", "inv_perm"):
        assert np.array_equal(b[k].numpy(), p[k]), k
    assert int(b["m_sum"].item()) == p["m_sum"]


def test_forward_naive_tiny_against_oracle(M):
    w, T = _case("tiny2")
    inp = synth.layer_inputs(w, T)
    stack = synth.all_expert_weights(w)
    g = _forward(M, w, inp, stack, True)
    ref = O.forward(inp, lambda e: {k: (v[e] if v is not None else None) for k, v in stack.items()}, w.fmt, w.K,
                    ROWS, w.score_fn, w.renormalize)
    assert np.array_equal(g["topk_ids"].numpy(), ref["route"]["topk_ids"])
    check_out(host_bits(g["out"]), ref["out"])


@pytest.mark.parametrize("case", ["tiny3", "decode4"])
def test_route_naive_then_stage_calls(M, case):
    # moe_route_naive's buffers through moe_grouped_ffn (align 16) and the separate reduce give
    # moe_forward_naive's output bit for bit; the activation rows are the token's quantised row
    w, T = _case(case)
    inp = synth.layer_inputs(w, T)
    stack = synth.all_expert_weights(w)
    a = _forward(M, w, inp, stack, True)["out"]
    w13, w2 = device_weights(M, stack, w.fmt)
    ws = M.new_workspace(T, w.H, w.I, w.E, w.K, ROWS)
    U = M.msum_upper(T, w.K, w.E, ROWS)
    ids, tw = torch.empty(T, w.K, **I32), torch.empty(T, w.K, dtype=torch.float32, device="cuda")
    srt, eid, inv, ms = torch.empty(U, **I32), torch.empty(U, **I32), torch.empty(T, w.K, **I32), torch.empty(1, **I32)
    xp = torch.zeros(U, w.H, **U8)
    xpsf = torch.zeros(M.act_sf_tiled_bytes(U, w.H // 128, ROWS), **U8)
    M.route_naive(*_args(inp), w.K, w.score_fn, w.renormalize, ids, tw, srt, eid, inv, ms, xp, xpsf, ws)
    hq = torch.zeros(U, w.I, **U8)
    hsf = torch.zeros(M.act_sf_tiled_bytes(U, w.I // 128, ROWS), **U8)
    y = torch.zeros(U, w.H, dtype=torch.bfloat16, device="cuda")
    M.grouped_ffn(xp, xpsf, eid, ms, T, w.K, w.H, w.I, w.E, ROWS, w13, w2, hq, hsf, y, ws)
    b = torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda")
    M.unpermute_reduce(y, inv, tw, b)
    assert M.get_error(ws) == M.OK
    assert torch.equal(a.view(torch.int16), b.cpu().view(torch.int16))
    xq, xsf = O.act_quant(inp["hidden"])
    rows = inv.cpu().numpy().reshape(-1)
    toks = np.repeat(np.arange(T), w.K)
    assert np.array_equal(xp.cpu().numpy()[rows], xq[toks])
    sf = M.act_sf_untile(xpsf.cpu().numpy(), U, w.H // 128, ROWS)
    assert np.array_equal(sf[rows], xsf[toks])


def test_naive_rejects_large_batches(M):
    w = synth.WORKLOADS["tiny"]                    # E = 16, K = 4: T * K <= E needs T <= 4
    for T in (5, 17):
        inp = synth.layer_inputs(w, T)
        stack = synth.all_expert_weights(w)
        w13, w2 = device_weights(M, stack, w.fmt)
        ws = M.new_workspace(T, w.H, w.I, w.E, w.K, ROWS)
        out = torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(M.MoeError) as err:
            M.forward_naive(*_args(inp), w.I, w.K, w.score_fn, w.renormalize, w13, w2, out, ws)
        assert err.value.status == M.ERR_UNSUPPORTED
