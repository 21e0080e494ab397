"""Helpers for the GPU parity tests: device upload, library build, and the comparison rules."""
import os

import numpy as np
import torch

from oracle import formats as F
from oracle import moe as O

# Output tolerance of the whole layer: max |gpu - oracle| <= OUT_TOL * RMS(oracle out).
OUT_TOL = 2e-2
# Relative key gap below which fp32 (kernel) and float64 (oracle) routing may legitimately
# order two experts differently; such tokens are checked for validity instead of equality.
TIE_DELTA = 1e-5


def ensure_lib():
    import moe_expert_ffn_sqrt_gb300 as M
    if not os.path.exists(M.LIB_PATH):
        from moe_expert_ffn_sqrt_gb300 import build
        build.build()
    M.lib()
    return M


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def device_weights(M, stack, fmt):
    if fmt == "int8":      # int8 codes; the per-channel scales travel as the weight's tscale
        return (M.Weight(dev(stack["w13_q"]), None, dev(stack["w13_sf"]), fmt, pair=2),
                M.Weight(dev(stack["w2_q"]), None, dev(stack["w2_sf"]), fmt, pair=1))
    w13 = M.Weight(dev(stack["w13_q"]), dev(stack["w13_sf"]),
                   None if stack["w13_ts"] is None else dev(stack["w13_ts"]), fmt, pair=2)
    w2 = M.Weight(dev(stack["w2_q"]), dev(stack["w2_sf"]),
                  None if stack["w2_ts"] is None else dev(stack["w2_ts"]), fmt, pair=1)
    return w13, w2


def near_tie_tokens(keys, K, delta=TIE_DELTA):
    """Tokens whose top-(K+1) keys (oracle, float64) contain a gap below delta * max|key|."""
    srt = -np.sort(-keys, axis=1)[:, : K + 1]
    gaps = srt[:, :-1] - srt[:, 1:]
    scale = np.abs(keys).max(axis=1)
    return np.where((gaps < delta * np.maximum(scale, 1e-30)[:, None]).any(axis=1))[0]


def check_topk(gpu_ids, gpu_w, r, K, delta=TIE_DELTA):
    """Exact ids / close weights on clear tokens; a valid top-K on near-tie tokens.  Returns #near-ties."""
    keys = r["keys"]
    ties = set(near_tie_tokens(keys, K, delta).tolist())
    T = keys.shape[0]
    for t in range(T):
        if t in ties:
            kth = -np.sort(-keys[t])[K - 1]
            tol = delta * np.abs(keys[t]).max()
            assert len(set(gpu_ids[t].tolist())) == K
            assert all(keys[t, e] >= kth - tol for e in gpu_ids[t]), f"token {t}: invalid top-K"
            continue
        assert np.array_equal(gpu_ids[t], r["topk_ids"][t]), f"token {t}: {gpu_ids[t]} vs {r['topk_ids'][t]}"
        assert np.allclose(gpu_w[t], r["topk_w"][t], rtol=2e-5, atol=1e-7), f"token {t} weights"
    return len(ties)


def check_out(gpu_bits, ref_bits, tol=OUT_TOL):
    g = F.bf16_to_f64(gpu_bits)
    r = F.bf16_to_f64(ref_bits)
    rms = float(np.sqrt(np.mean(r * r)))
    err = float(np.abs(g - r).max())
    assert np.isfinite(g).all()
    assert err <= tol * rms, f"max err {err:.3e} > {tol} x RMS {rms:.3e}"
    return err / rms


def bf16_ulp_diff(a_bits, b_bits):
    """|difference| in units of the bf16 grid (ordered-integer distance)."""
    def key(b):
        b = b.astype(np.int64)
        return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + b)
    return np.abs(key(a_bits) - key(b_bits))


def dequant_act(codes, sf, group=128):
    return O.dequant_fp8_groups(codes, sf, group)
