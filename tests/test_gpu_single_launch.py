"""GPU parity of moe_forward_single_launch: the whole layer (routing, permute, L1, L2, weighted
reduce) as one cooperative launch, the single persistent kernel of page "DeepSeek V4 MegaMoE Kernel
深度解析", 一、架构概览 整体思路.  It runs the same routing, permute and GEMM code as moe_forward,
so every output (the layer output and each index output) must equal moe_forward's bit for bit;
moe_forward itself is checked against the float64 oracle in test_gpu_parity, and the tiny case is
checked against the oracle here as well.  Unsupported problems must be refused, not run.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import check_layer, dev, dev_bf16, device_weights, ensure_lib
from oracle import moe as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_lib()


def _run(M, w, inp, w13, w2, single, ws=None):
    T = inp["hidden"].shape[0]
    ws = M.new_workspace(T, w.H, w.I, w.E, w.K, w.align) if ws is None else ws
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
              m_sum=o["m_sum"], single_launch=single)
    assert M.get_error(ws) == M.OK
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in o.items()}


def _equal(a, b):
    for k in a:
        x, y = a[k], b[k]
        if x.dtype in (torch.bfloat16, torch.float32):
            x, y = x.view(torch.int16 if x.dtype == torch.bfloat16 else torch.int32), \
                y.view(torch.int16 if y.dtype == torch.bfloat16 else torch.int32)
        if k in ("sorted_token_ids", "expert_ids"):
            ms = int(a["m_sum"][0])
            x, y = x[:ms], y[:ms]
        assert torch.equal(x, y), f"{k} differs between moe_forward and moe_forward_single_launch"


CASES = {
    "decode": (synth.WORKLOADS["decode"], None),
    "tiny": (synth.WORKLOADS["tiny"], None),
    "one_token": (synth.WORKLOADS["decode"], 1),
    "odd_T": (synth.custom(T=5, H=1024, I=512, E=64, K=6, align=16, score_fn="sqrt_softplus", e_bias=True,
                           seed=21), None),
    "pairs_128": (synth.custom(T=16, H=512, I=256, E=32, K=8, align=16, score_fn="softmax", seed=22), None),
    "align_1": (synth.custom(T=11, H=512, I=384, E=16, K=4, align=1, score_fn="sqrt_softplus", e_bias=True,
                             seed=23), None),
    "h_384": (synth.custom(T=9, H=384, I=256, E=48, K=3, align=8, score_fn="softmax", seed=24), None),
    "gate_bias": (synth.custom(T=12, H=1024, I=256, E=128, K=6, align=16, score_fn="sqrt_softplus", e_bias=True,
                               gate_offset="normal", seed=25), None),
    "zipf_gate": (synth.custom(T=16, H=512, I=256, E=256, K=8, align=16, score_fn="sqrt_softplus", e_bias=True,
                               gate_offset="zipf", seed=26), None),
}


@pytest.mark.parametrize("case", list(CASES))
def test_single_launch_equals_forward(M, case):
    w, T = CASES[case]
    inp = synth.layer_inputs(w, T)
    stack = synth.all_expert_weights(w)
    w13, w2 = device_weights(M, stack, w.fmt)
    ref = _run(M, w, inp, w13, w2, single=False)
    got = _run(M, w, inp, w13, w2, single=True)
    _equal(ref, got)
    assert not torch.isnan(got["out"].float()).any()


def test_single_launch_repeated_calls(M):
    # the launch leaves its grid-barrier and work counters at zero: a second call on the same
    # workspace (and a moe_forward in between) gives the same bits
    w = synth.WORKLOADS["decode"]
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    w13, w2 = device_weights(M, stack, w.fmt)
    ws = M.new_workspace(8, w.H, w.I, w.E, w.K, w.align)
    a = _run(M, w, inp, w13, w2, single=True, ws=ws)
    b = _run(M, w, inp, w13, w2, single=False, ws=ws)
    c = _run(M, w, inp, w13, w2, single=True, ws=ws)
    _equal(a, b)
    _equal(a, c)


def test_single_launch_against_oracle(M):
    from test_gpu_parity import ORACLE_THREADS, _stack_provider
    w = synth.WORKLOADS["tiny"]
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    w13, w2 = device_weights(M, stack, w.fmt)
    got = _run(M, w, inp, w13, w2, single=True)
    g = {k: (v.view(torch.int16) if v.dtype == torch.bfloat16 else v).numpy() for k, v in got.items()}
    g["out"] = g["out"].view(np.uint16)
    prov = _stack_provider(stack)

    def oracle(toks, routing=None):
        return O.forward(inp, prov, w.fmt, w.K, w.align, w.score_fn, w.renormalize, tokens=toks, routing=routing,
                         workers=ORACLE_THREADS)

    check_layer(M, w, inp, g, oracle(None), oracle, perm_fn=lambda ids: O.permute(ids, w.E, w.align))


@pytest.mark.parametrize("what", ["T17", "nvfp4", "align32", "pairs_144"])
def test_single_launch_refuses_unsupported(M, what):
    if what == "T17":
        w, T = synth.custom(T=17, H=512, I=256, E=16, K=4, align=16, seed=31), None
    elif what == "nvfp4":
        w, T = synth.custom(T=8, H=512, I=256, E=16, K=4, align=16, fmt="nvfp4", seed=32), None
    elif what == "align32":
        w, T = synth.custom(T=8, H=512, I=256, E=16, K=4, align=32, seed=33), None
    else:
        w, T = synth.custom(T=16, H=512, I=256, E=16, K=9, align=16, seed=34), None
    inp = synth.layer_inputs(w, T)
    stack = synth.all_expert_weights(w)
    w13, w2 = device_weights(M, stack, w.fmt)
    with pytest.raises(M.MoeError) as e:
        _run(M, w, inp, w13, w2, single=True)
    assert e.value.status == M.ERR_UNSUPPORTED
