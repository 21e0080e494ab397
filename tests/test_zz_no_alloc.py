"""The allocation-free routing call (moe_route_noalloc) against the regular one (moe_route) and the oracle.

moe_route_noalloc serves callers that can neither pass a workspace nor allocate device memory;
it keeps its scratch in a fixed array inside the library.  This file is collected last so that
a run stopping at the first failure has already run every other test.  It passes alone in a
fresh process (it loads the library itself) and after the other tests (the fixed array then
holds another call's partial sums, which must not leak into the results).

Every output buffer is filled with a poison pattern before each call (ids -1, weights and logits
NaN, codes and scales 0xFF), so a call that leaves an output unwritten cannot pass by inheriting
the bytes of an earlier call's freed buffer.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_util import check_topk, dev, dev_bf16, ensure_lib, oracle_route_on
from oracle import moe as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_lib()


def _outputs(T, w):
    nan = float("nan")
    return dict(ids=torch.full((T, w.K), -1, dtype=torch.int32, device="cuda"),
                tw=torch.full((T, w.K), nan, dtype=torch.float32, device="cuda"),
                logits=torch.full((T, w.E), nan, dtype=torch.float32, device="cuda"),
                xq=torch.full((T, w.H), 0xFF, dtype=torch.uint8, device="cuda"),
                xsf=torch.full((T, w.H // 128), 0xFF, dtype=torch.uint8, device="cuda"))


def _run(M, w, inp, noalloc):
    T = inp["hidden"].shape[0]
    o = _outputs(T, w)
    args = (dev_bf16(inp["hidden"]), dev(inp["w_gate"]),
            None if inp["gate_bias"] is None else dev(inp["gate_bias"]),
            None if inp["e_score_bias"] is None else dev(inp["e_score_bias"]), w.K, w.score_fn, w.renormalize,
            o["ids"], o["tw"])
    if noalloc:
        M.route_noalloc(*args, logits_out=o["logits"], x_q=o["xq"], x_sf=o["xsf"])
    else:
        ws = M.new_workspace(T, w.H, w.I, w.E, w.K, w.align)
        M.route(*args, ws, logits_out=o["logits"], x_q=o["xq"], x_sf=o["xsf"])
        assert M.get_error(ws) == M.OK
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in o.items()}


def _check_against_reference_and_oracle(M, w, inp):
    ref = _run(M, w, inp, noalloc=False)
    got = _run(M, w, inp, noalloc=True)
    T = inp["hidden"].shape[0]
    assert ((got["ids"] >= 0) & (got["ids"] < w.E)).all(), "topk_ids left unwritten or invalid"
    assert np.isfinite(got["tw"]).all() and np.isfinite(got["logits"]).all()
    assert np.array_equal(got["ids"], ref["ids"])
    assert np.allclose(got["tw"], ref["tw"], rtol=2e-5, atol=1e-7)
    assert np.allclose(got["logits"], ref["logits"], rtol=1e-5, atol=1e-6)
    assert np.array_equal(got["xq"], ref["xq"]) and np.array_equal(got["xsf"], ref["xsf"])
    r = O.route(inp["hidden"], inp["w_gate"], inp["gate_bias"], inp["e_score_bias"], w.K, w.score_fn,
                w.renormalize)
    counts = check_topk(got["ids"], got["tw"], r, w.K, oracle_route_on(got["logits"], w, inp))
    assert counts["unresolved"] <= max(2, T // 100)
    xq_ref, xsf_ref = O.act_quant(inp["hidden"])
    assert np.array_equal(got["xq"], xq_ref) and np.array_equal(got["xsf"], xsf_ref)


def _second_inputs(w, T):
    return synth.layer_inputs(synth.custom(name="second", T=w.T, H=w.H, I=w.I, E=w.E, K=w.K, align=w.align,
                                           score_fn=w.score_fn, e_bias=w.e_bias, gate_offset=w.gate_offset,
                                           seed=w.seed + 17), T)


# T = 64 and T = 77 at the small dims take the tensor-core gate (T > 16), whose three bf16 parts of
# the gate weight then also live in the fixed array
@pytest.mark.parametrize("name,T", [("decode", None), ("batched", 16), ("tiny", 3), ("tiny", 64), ("tiny", 77)])
def test_noalloc_route_matches_route_on_two_calls_in_a_row(M, name, T):
    w = synth.WORKLOADS[name]
    for inp in (synth.layer_inputs(w, T), _second_inputs(w, T)):    # two calls in a row on the shared scratch
        _check_against_reference_and_oracle(M, w, inp)


def test_noalloc_route_after_calls_of_other_shapes(M):
    # calls of different shapes one after another in one process: each finds the counter slot at
    # zero although the previous call left partial sums of another layout in the array
    seq = [("decode", None), ("batched", 16), ("tiny", 3), ("tiny", 77), ("tiny", 8), ("batched", 16),
           ("decode", 5)]
    for name, T in seq:
        w = synth.WORKLOADS[name]
        _check_against_reference_and_oracle(M, w, synth.layer_inputs(w, T))


def test_noalloc_route_rejects_problems_beyond_its_scratch(M):
    # the tiled gate GEMM for T = 16384 needs 16384 * 256 * 4 bytes (16 MiB) of partial sums: too big
    L = M.lib()
    buf = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(buf.data_ptr())
    st = L.moe_route_noalloc(p, p, None, None, 16384, 7168, 256, 6, 1, 1, None, p, p, None, None,
                             torch.cuda.current_stream().cuda_stream)
    assert st == M.ERR_UNSUPPORTED
