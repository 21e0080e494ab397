"""Device failure path on the GPU without a fault: a bounded wait that nothing satisfies gives up,
records MOE_ERR_TIMEOUT in the workspace status word, and the context stays usable."""
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


def _forward(M, w, inp, stack):
    w13, w2 = device_weights(M, stack, w.fmt)
    ws = M.new_workspace(w.T, w.H, w.I, w.E, w.K, w.align)
    out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    M.forward(dev_bf16(inp["hidden"]), dev(inp["w_gate"]), None, None, w.I, w.K, w.align, w.score_fn, w.renormalize,
              w13, w2, out, ws)
    return out, ws


@pytest.mark.parametrize("mode", [0, 1])
def test_wait_timeout_is_reported_and_the_context_stays_usable(M, mode):
    w = synth.WORKLOADS["tiny"]
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    ref, ws_ref = _forward(M, w, inp, stack)
    assert M.get_error(ws_ref) == M.OK
    ws = M.new_workspace(w.T, w.H, w.I, w.E, w.K, w.align)
    M.selftest_wait_timeout(ws, mode)
    assert M.get_error(ws) == M.ERR_TIMEOUT
    assert M.get_error(ws) == M.OK                        # read and cleared
    out, ws2 = _forward(M, w, inp, stack)                 # the same context keeps working
    assert M.get_error(ws2) == M.OK
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_selftest_rejects_bad_arguments(M):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(M.MoeError):
        M.selftest_wait_timeout(ws, 2)
    with pytest.raises(M.MoeError):
        M.selftest_wait_timeout(ws[:128], 0)
