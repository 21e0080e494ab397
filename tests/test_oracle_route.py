"""Pins for the oracle's routing: gate GEMM, scoring functions, biased top-K, weights."""
import itertools
import math

import numpy as np
import scipy.special

from oracle import moe
from oracle.formats import bf16_to_f64


def _bf16(x):
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_gate_logits_brute_force():
    # gate = hidden @ W_gate^T with W_gate [E, H] (MegaMoE page, 第一步), summed term by term
    rng = np.random.default_rng(0)
    T, H, E = 3, 16, 5
    hid = _bf16(rng.standard_normal((T, H)))
    wg = rng.standard_normal((E, H)).astype(np.float32)
    gb = rng.standard_normal(E).astype(np.float32)
    got = moe.gate_logits(hid, wg, gb)
    x = bf16_to_f64(hid)
    for t in range(T):
        for e in range(E):
            ref = math.fsum(float(x[t, h]) * float(wg[e, h]) for h in range(H)) + float(gb[e])
            assert abs(got[t, e] - ref) <= 1e-12 * (1 + abs(ref))


def test_sqrt_softplus_closed_forms():
    x = np.array([0.0, 30.0, -30.0, 1.5, -2.25])
    got = moe.sqrt_softplus(x[None, :])[0]
    assert abs(got[0] - math.sqrt(math.log(2.0))) < 1e-15
    assert abs(got[1] - math.sqrt(30.0 + math.log1p(math.exp(-30.0)))) < 1e-14
    assert abs(got[2] - math.exp(-15.0)) < 1e-13 * math.exp(-15.0) + 1e-300   # sqrt(ln(1+e^-30)) ~ e^-15
    for i in (3, 4):
        assert abs(got[i] - math.sqrt(math.log(1.0 + math.exp(x[i])))) < 1e-15


def test_softmax_matches_scipy_and_sums_to_one():
    rng = np.random.default_rng(1)
    l = rng.standard_normal((7, 33)) * 4
    s = moe.softmax(l)
    assert np.allclose(s, scipy.special.softmax(l, axis=1), rtol=1e-14, atol=0)
    assert np.allclose(s.sum(axis=1), 1.0, rtol=0, atol=1e-15)


def _brute_topk(keys, K):
    out = []
    for row in keys:
        order = sorted(range(len(row)), key=lambda e: (-row[e], e))
        out.append(order[:K])
    return np.array(out)


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(2)
    for _ in range(200):
        E = int(rng.integers(2, 9))
        K = int(rng.integers(1, E + 1))
        keys = rng.integers(0, 4, size=(3, E)).astype(np.float64)   # many ties
        assert np.array_equal(moe.select_topk(keys, K), _brute_topk(keys, K))


def test_topk_exhaustive_small():
    # every ordering of 4 distinct keys: the top-2 are the two largest, larger first
    for perm in itertools.permutations(range(4)):
        keys = np.array([perm], dtype=np.float64)
        ids = moe.select_topk(keys, 2)[0]
        assert keys[0, ids[0]] == 3 and keys[0, ids[1]] == 2


def test_all_equal_keys_pick_lowest_ids():
    ids = moe.select_topk(np.zeros((2, 10)), 4)
    assert ids.tolist() == [[0, 1, 2, 3]] * 2


def test_weights_renormalised_and_softmax_invariant():
    rng = np.random.default_rng(3)
    T, H, E, K = 5, 64, 12, 3
    hid = _bf16(rng.standard_normal((T, H)))
    wg = (rng.standard_normal((E, H)) / 8).astype(np.float32)
    r = moe.route(hid, wg, None, None, K, "softmax")
    assert np.allclose(r["topk_w"].sum(axis=1), 1.0, atol=1e-15)
    # for softmax scoring the renormalised weights equal a softmax over the selected logits
    sel = np.take_along_axis(r["logits"], r["topk_ids"].astype(np.int64), axis=1)
    assert np.allclose(r["topk_w"], scipy.special.softmax(sel, axis=1), rtol=1e-13)


def test_score_bias_selects_but_does_not_weight():
    # e_score_correction_bias moves expert 0 into the selection; its weight uses the unbiased score
    rng = np.random.default_rng(4)
    T, H, E, K = 4, 32, 8, 2
    hid = _bf16(rng.standard_normal((T, H)))
    wg = (rng.standard_normal((E, H)) / 6).astype(np.float32)
    bias = np.zeros(E, np.float32)
    bias[0] = 100.0
    r = moe.route(hid, wg, None, bias, K, "sqrt_softplus")
    assert (r["topk_ids"][:, 0] == 0).all()
    s = r["scores"]
    for t in range(T):
        ids = r["topk_ids"][t]
        assert abs(r["topk_w"][t, 0] - s[t, 0] / (s[t, ids[0]] + s[t, ids[1]])) < 1e-15
    r0 = moe.route(hid, wg, None, None, K, "sqrt_softplus")
    assert np.array_equal(r0["scores"], r["scores"])


def test_not_renormalised_returns_raw_scores():
    rng = np.random.default_rng(5)
    hid = _bf16(rng.standard_normal((2, 32)))
    wg = rng.standard_normal((6, 32)).astype(np.float32)
    r = moe.route(hid, wg, None, None, 2, "sqrt_softplus", renormalize=False)
    assert np.array_equal(r["topk_w"], np.take_along_axis(r["scores"], r["topk_ids"].astype(np.int64), 1))
