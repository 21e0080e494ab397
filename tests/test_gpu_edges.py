"""GPU parity of the whole layer at the edges of the supported shapes, against the float64 oracle.

Each case checks the routing of every token (exact top-K, or a valid top-K for near-ties), the
permute's index outputs bit for bit where the routing agrees, and every token's output within
2e-2 x RMS (the same bars as test_gpu_parity):
  * E = 1024 (32 keys per lane in the top-K) at T = 16, the largest small-batch routing;
  * T = 17, the first batch through the tensor-core gate and the per-token top-K;
  * E = 3 (not a multiple of 32) with K = 2 and align 1;
  * K = 1, and H = 384 (the last W2 tile is a half tile of 128 rows), I = 128 (one W13 tile);
  * NVFP4 at H = 384;
  * T = 32 and 33, either side of the reduce moving out of the L2 epilogue;
plus the three variants (BatchedExperts, tiny batch, weights in L1) on the E = 1024 case.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import check_layer, dev, dev_bf16, device_weights, ensure_lib, host_bits
from oracle import moe as O

pytestmark = pytest.mark.gpu

I32 = dict(dtype=torch.int32, device="cuda")

CASES = {
    "E1024_T16": dict(T=16, H=256, I=256, E=1024, K=8, align=16, score_fn="sqrt_softplus", e_bias=True, seed=21),
    "E1024_T17": dict(T=17, H=256, I=256, E=1024, K=8, align=16, score_fn="softmax", seed=22),
    "E3_K2_align1": dict(T=19, H=128, I=128, E=3, K=2, align=1, score_fn="softmax", seed=23),
    "K1_H384_I128": dict(T=5, H=384, I=128, E=64, K=1, align=4, score_fn="sqrt_softplus", e_bias=True, seed=24),
    "nvfp4_H384": dict(T=9, H=384, I=256, E=32, K=4, align=8, score_fn="sqrt_softplus", e_bias=True, fmt="nvfp4",
                       seed=25),
    # the reduce runs in the L2 epilogue up to 32 tokens, as a separate kernel above
    "T32_fused_reduce": dict(T=32, H=512, I=256, E=16, K=4, align=16, score_fn="softmax", seed=26),
    "T33_separate_reduce": dict(T=33, H=512, I=256, E=16, K=4, align=16, score_fn="softmax", seed=27),
}


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_lib()


def _args(inp):
    return (dev_bf16(inp["hidden"]), dev(inp["w_gate"]), None if inp["gate_bias"] is None else dev(inp["gate_bias"]),
            None if inp["e_score_bias"] is None else dev(inp["e_score_bias"]))


def _oracle(w, inp, stack, weights_in_l1=False):
    return O.forward(inp, lambda e: {k: (v[e] if v is not None else None) for k, v in stack.items()}, w.fmt, w.K,
                     w.align, w.score_fn, w.renormalize, topk_w_dtype=np.float32, weights_in_l1=weights_in_l1)


def _compare(M, w, inp, stack, ids, tw, out, ref, perm=None, weights_in_l1=False, perm_fn=None):
    g = dict(topk_ids=ids, topk_w=tw, out=host_bits(out))
    if perm is not None:
        g.update(perm)

    def rerun(toks, routing):
        return O.forward(inp, lambda e: {k: (v[e] if v is not None else None) for k, v in stack.items()}, w.fmt,
                         w.K, w.align, w.score_fn, w.renormalize, tokens=toks, topk_w_dtype=np.float32,
                         weights_in_l1=weights_in_l1, routing=routing)

    check_layer(M, w, inp, g, ref, rerun, perm_fn=perm_fn or (lambda i: O.permute(i, w.E, w.align)))


@pytest.mark.parametrize("case", sorted(CASES))
def test_forward_edges(M, case):
    w = synth.custom(name=case, **CASES[case])
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    T = w.T
    w13, w2 = device_weights(M, stack, w.fmt)
    ws = M.new_workspace(T, w.H, w.I, w.E, w.K, w.align)
    U = M.msum_upper(T, w.K, w.E, w.align)
    out = torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda")
    o = dict(topk_ids=torch.empty(T, w.K, **I32), topk_w=torch.empty(T, w.K, dtype=torch.float32, device="cuda"),
             sorted_token_ids=torch.empty(U, **I32), expert_ids=torch.empty(U, **I32),
             inv_perm=torch.empty(T, w.K, **I32), m_sum=torch.empty(1, **I32))
    M.forward(*_args(inp), w.I, w.K, w.align, w.score_fn, w.renormalize, w13, w2, out, ws, **o)
    assert M.get_error(ws) == M.OK
    ref = _oracle(w, inp, stack)
    perm = {k: v.cpu().numpy() for k, v in o.items() if k in ("sorted_token_ids", "expert_ids", "inv_perm", "m_sum")}
    _compare(M, w, inp, stack, o["topk_ids"].cpu().numpy(), o["topk_w"].cpu().numpy(), out.cpu(), ref, perm)


@pytest.mark.parametrize("variant", ["batched", "naive", "weights_in_l1"])
def test_variants_on_1024_experts(M, variant):
    w = synth.custom(name="E1024_T16", **CASES["E1024_T16"])
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    T = w.T
    w13, w2 = device_weights(M, stack, w.fmt)
    out = torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(T, w.K, **I32)
    tw = torch.empty(T, w.K, dtype=torch.float32, device="cuda")
    if variant == "batched":
        ws = M.new_workspace_batched(T, w.H, w.I, w.E, w.K, 16)
        M.forward_batched(*_args(inp), w.I, w.K, 16, w.score_fn, w.renormalize, w13, w2, out, ws, topk_ids=ids,
                          topk_w=tw)
    elif variant == "naive":
        ws = M.new_workspace(T, w.H, w.I, w.E, w.K, M.NAIVE_ROWS)
        M.forward_naive(*_args(inp), w.I, w.K, w.score_fn, w.renormalize, w13, w2, out, ws, topk_ids=ids, topk_w=tw)
    else:
        ws = M.new_workspace(T, w.H, w.I, w.E, w.K, w.align)
        M.forward(*_args(inp), w.I, w.K, w.align, w.score_fn, w.renormalize, w13, w2, out, ws, topk_ids=ids,
                  topk_w=tw, weights_in_l1=True)
    assert M.get_error(ws) == M.OK
    ref = _oracle(w, inp, stack, weights_in_l1=variant == "weights_in_l1")
    _compare(M, w, inp, stack, ids.cpu().numpy(), tw.cpu().numpy(), out.cpu(), ref,
             weights_in_l1=variant == "weights_in_l1")
