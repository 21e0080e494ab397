"""The whole layer captured into a CUDA graph.

No call of the hot path synchronises with the host or allocates (M_sum stays on the device and
the buffers are sized by its upper bound), so a captured moe_forward (and its variants) replays with
new inputs and gives the same bits as eager calls.
"""
import dataclasses

import pytest
import torch

import synth
from gpu_util import dev, dev_bf16, device_weights, ensure_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_lib()


@pytest.mark.parametrize("case", ["decode", "tiny77", "nvfp4", "naive", "batched_layout", "single_launch"])
def test_forward_graph_replay_matches_eager(M, case):
    if case == "nvfp4":
        w = synth.custom(T=40, H=512, I=256, E=16, K=4, align=16, score_fn="sqrt_softplus", e_bias=True,
                         fmt="nvfp4", seed=9)
        T = 40
    elif case == "tiny77":
        w, T = synth.WORKLOADS["tiny"], 77
    elif case == "naive":
        w, T = synth.WORKLOADS["decode"], 2
    else:
        w, T = synth.WORKLOADS["decode"], 8
    stack = synth.all_expert_weights(w)
    w13, w2 = device_weights(M, stack, w.fmt)
    inps = [synth.layer_inputs(dataclasses.replace(w, seed=w.seed + 100 * i), T) for i in range(3)]
    base = synth.layer_inputs(w, T)
    w_gate = dev(base["w_gate"])
    gate_bias = None if base["gate_bias"] is None else dev(base["gate_bias"])
    e_bias = None if base["e_score_bias"] is None else dev(base["e_score_bias"])
    hidden = dev_bf16(inps[0]["hidden"]).clone()
    out = torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda")
    if case == "naive":
        ws = M.new_workspace(T, w.H, w.I, w.E, w.K, M.NAIVE_ROWS)
        call = lambda: M.forward_naive(hidden, w_gate, gate_bias, e_bias, w.I, w.K, w.score_fn, w.renormalize, w13, w2,
                                       out, ws)
    elif case == "batched_layout":
        ws = M.new_workspace_batched(T, w.H, w.I, w.E, w.K, 16)
        call = lambda: M.forward_batched(hidden, w_gate, gate_bias, e_bias, w.I, w.K, 16, w.score_fn, w.renormalize,
                                         w13, w2, out, ws)
    else:
        ws = M.new_workspace(T, w.H, w.I, w.E, w.K, w.align)
        single = case == "single_launch"     # the whole layer as one cooperative launch
        call = lambda: M.forward(hidden, w_gate, gate_bias, e_bias, w.I, w.K, w.align, w.score_fn, w.renormalize, w13,
                                 w2, out, ws, single_launch=single)
    # eager reference outputs, one per input
    eager = []
    for inp in inps:
        hidden.copy_(dev_bf16(inp["hidden"]))
        call()
        eager.append(out.clone())
    assert M.get_error(ws) == M.OK
    # capture once (after a warm-up call on a side stream, as torch requires), replay per input
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
