"""The allocation-free routing call (moe_route_noalloc) against the regular one (moe_route).

moe_route_noalloc serves callers that can neither pass a workspace nor allocate device memory;
it keeps its scratch in a fixed array inside the library.  This file is collected last so that
a run stopping at the first failure has already run every other test.  It passes alone in a
fresh process (it loads the library itself) and after the other tests (the fixed array then
holds another call's partial sums, which must not leak into the results).
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_util import dev, dev_bf16, ensure_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_lib()


def _outputs(T, w):
    return dict(ids=torch.empty(T, w.K, dtype=torch.int32, device="cuda"),
                tw=torch.empty(T, w.K, dtype=torch.float32, device="cuda"),
                logits=torch.empty(T, w.E, dtype=torch.float32, device="cuda"),
                xq=torch.empty(T, w.H, dtype=torch.uint8, device="cuda"),
                xsf=torch.empty(T, w.H // 128, dtype=torch.uint8, device="cuda"))


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
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in o.items()}


@pytest.mark.parametrize("name,T", [("decode", None), ("batched", 16), ("tiny", 3)])
def test_noalloc_route_matches_route_on_two_calls_in_a_row(M, name, T):
    w = synth.WORKLOADS[name]
    first = synth.layer_inputs(w, T)
    second = synth.layer_inputs(synth.custom(name="second", T=w.T, H=w.H, I=w.I, E=w.E, K=w.K, align=w.align,
                                             score_fn=w.score_fn, e_bias=w.e_bias, gate_offset=w.gate_offset,
                                             seed=w.seed + 17), T)
    for inp in (first, second):                      # two calls in a row on the shared scratch
        ref = _run(M, w, inp, noalloc=False)
        got = _run(M, w, inp, noalloc=True)
        assert np.array_equal(got["ids"], ref["ids"])
        assert np.allclose(got["tw"], ref["tw"], rtol=2e-5, atol=1e-7)
        assert np.allclose(got["logits"], ref["logits"], rtol=1e-5, atol=1e-6)
        assert np.array_equal(got["xq"], ref["xq"]) and np.array_equal(got["xsf"], ref["xsf"])


def test_noalloc_route_rejects_problems_beyond_its_scratch(M):
    # the tiled gate GEMM for T = 16384 needs 16384 * 256 * 4 bytes (16 MiB) of partial sums: too big
    L = M.lib()
    buf = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(buf.data_ptr())
    st = L.moe_route_noalloc(p, p, None, None, 16384, 7168, 256, 6, 1, 1, None, p, p, None, None,
                             torch.cuda.current_stream().cuda_stream)
    assert st == M.ERR_UNSUPPORTED
