"""Pins for the oracle's permute (align + scatter) against the printed example and brute force."""
import numpy as np
import pytest

import synth
from oracle import moe
from conftest import load_golden


def test_printed_permute_example():
    g = load_golden("permute_example.txt")
    ids = np.array(g["topk_ids"], dtype=np.int32).reshape(g["T"], g["K"])
    p = moe.permute(ids, g["E"], g["align"])
    assert p["inv_perm"].reshape(-1).tolist() == g["inv_perm"]
    assert p["m_sum"] == g["m_sum"]
    rows = p["sorted_token_ids"][: p["m_sum"]] // g["K"]
    assert rows.tolist() == g["row_token"]


def test_printed_example_aligned_to_four():
    # same routing, segments padded to multiples of 4: counts (1,3,2) -> 4+4+4 rows;
    # sorted_token_ids holds the flat index t*K + k (T*K = 6 on padding rows)
    g = load_golden("permute_example.txt")
    ids = np.array(g["topk_ids"], dtype=np.int32).reshape(3, 2)
    p = moe.permute(ids, 3, 4)
    assert p["m_sum"] == 12
    assert p["inv_perm"].tolist() == [[4, 8], [0, 5], [6, 9]]
    assert p["expert_ids"][:12].tolist() == [0, -1, -1, -1, 1, 1, 1, -1, 2, 2, -1, -1]
    assert p["sorted_token_ids"][:12].tolist() == [2, 6, 6, 6, 0, 3, 4, 6, 1, 5, 6, 6]


def test_unsorted_topk_rows_example():
    g = load_golden("topk_ids_example.txt")
    ids = np.array(g["topk_ids"], dtype=np.int32).reshape(3, 2)
    p = moe.permute(ids, 8, 1)
    # expert 1: tokens 1, 2; expert 3: tokens 0, 1; expert 7: tokens 0, 2
    assert p["inv_perm"].tolist() == [[2, 4], [3, 0], [5, 1]]


def _brute_permute(ids, E, A):
    T, K = ids.shape
    rows = []
    expert_of_row = []
    inv = np.zeros((T, K), dtype=np.int64)
    for e in range(E):
        start = len(rows)
        for t in range(T):
            for k in range(K):
                if ids[t, k] == e:
                    inv[t, k] = len(rows)
                    rows.append(t * K + k)
                    expert_of_row.append(e)
        while (len(rows) - start) % A:
            rows.append(T * K)
            expert_of_row.append(-1)
    return inv, rows, expert_of_row


@pytest.mark.parametrize("A", [1, 2, 4, 16, 64])
def test_permute_brute_force(A):
    rng = np.random.default_rng(A)
    for _ in range(20):
        E = int(rng.integers(1, 12))
        K = int(rng.integers(1, min(E, 4) + 1))
        T = int(rng.integers(0, 9))
        ids = np.array([rng.choice(E, K, replace=False) for _ in range(T)], dtype=np.int32).reshape(T, K)
        p = moe.permute(ids, E, A)
        inv, rows, er = _brute_permute(ids, E, A)
        assert np.array_equal(p["inv_perm"], inv)
        assert p["m_sum"] == len(rows)
        assert p["sorted_token_ids"][: len(rows)].tolist() == rows
        assert p["expert_ids"][: len(rows)].tolist() == er
        assert (p["expert_ids"][len(rows):] == -1).all()
        assert (p["sorted_token_ids"][len(rows):] == T * K).all()


@pytest.mark.parametrize("T,K,E,A", [(8, 6, 256, 16), (128, 6, 256, 64), (300, 4, 16, 256), (1, 1, 1, 1)])
def test_permute_invariants(T, K, E, A):
    rng = np.random.default_rng(T)
    ids = np.array([rng.choice(E, K, replace=False) for _ in range(T)], dtype=np.int32)
    p = moe.permute(ids, E, A)
    inv = p["inv_perm"].reshape(-1)
    M = p["m_sum"]
    assert len(set(inv.tolist())) == T * K and inv.min() >= 0 and inv.max() < M      # injective into [0, M_sum)
    assert np.array_equal(p["sorted_token_ids"][inv], np.arange(T * K))
    assert np.array_equal(p["expert_ids"][inv], ids.reshape(-1))
    assert M % A == 0
    assert T * K <= M <= moe.msum_upper(T, K, E, A)                                   # note §10 bound
    assert (p["expert_ids"] >= 0).sum() == T * K
    assert len(p["expert_ids"]) == moe.msum_upper(T, K, E, A)
    segs = [s for s, c in zip(p["seg_start"], p["expert_counts"]) if c > 0]
    assert all(s % A == 0 for s in segs)


def test_msum_upper_decode_shape():
    assert moe.msum_upper(8, 6, 256, 16) == 3888


def test_bad_expert_id_rejected():
    with pytest.raises(ValueError):
        moe.permute(np.array([[0, 5]], dtype=np.int32), 4, 1)


# ------------------------------------------------------------------------------------------ BatchedExperts layout

def test_batched_printed_example():
    g = load_golden("permute_batched_example.txt")
    ids = np.array(g["topk_ids"], dtype=np.int32).reshape(g["T"], g["K"])
    p = moe.permute_batched(ids, g["E"], g["max_tokens"])
    assert p["sorted_token_ids"].tolist() == g["sorted_token_ids"]
    assert p["expert_ids"].tolist() == g["expert_ids"]
    assert p["inv_perm"].reshape(-1).tolist() == g["inv_perm"]
    assert p["expert_num_tokens"].tolist() == g["expert_num_tokens"]
    assert p["m_sum"] == g["E"] * g["max_tokens"]


@pytest.mark.parametrize("T,K,E,S,seed", [(8, 6, 256, 16, 0), (37, 4, 16, 64, 1), (5, 2, 3, 8, 2), (128, 6, 64, 128, 3)])
def test_batched_slots_hold_the_contiguous_segments(T, K, E, S, seed):
    # each expert's slot holds exactly the pairs of that expert's contiguous segment, in the same
    # order (two independent constructions: per-expert boolean masks vs one stable sort)
    rng = np.random.default_rng(seed)
    ids = np.array([rng.choice(E, K, replace=False) for _ in range(T)], dtype=np.int32)
    b = moe.permute_batched(ids, E, S)
    c = moe.permute(ids, E, 1)
    for e in range(E):
        n = int(c["expert_counts"][e])
        seg = int(c["seg_start"][e])
        assert b["expert_num_tokens"][e] == n
        assert b["sorted_token_ids"][e * S: e * S + n].tolist() == c["sorted_token_ids"][seg: seg + n].tolist()
        assert (b["expert_ids"][e * S: e * S + n] == e).all() and (b["expert_ids"][e * S + n: (e + 1) * S] == -1).all()
        assert (b["sorted_token_ids"][e * S + n: (e + 1) * S] == T * K).all()
    flat = b["inv_perm"].reshape(-1)
    assert np.array_equal(b["sorted_token_ids"][flat], np.arange(T * K))
    assert np.array_equal(b["expert_ids"][flat], ids.reshape(-1))


def test_batched_rejects_an_overfull_slot():
    ids = np.array([[0, 1], [0, 2], [0, 1]], dtype=np.int32)     # expert 0 receives 3 tokens
    with pytest.raises(ValueError):
        moe.permute_batched(ids, 3, 2)


def test_naive_layout_by_hand():
    # token 0 picks experts 5 then 2 (K = 2, E = 8): pair 0 on row 0, pair 1 on row 16
    p = moe.permute_naive(np.array([[5, 2]]), 8)
    assert p["U"] == 2 + 8 * 15 and p["m_sum"] == 32
    assert p["inv_perm"].tolist() == [[0, 16]]
    assert p["expert_ids"][0] == 5 and p["expert_ids"][16] == 2
    assert (np.delete(p["expert_ids"], [0, 16]) == -1).all()
    assert p["sorted_token_ids"][0] == 0 and p["sorted_token_ids"][16] == 1
    assert (np.delete(p["sorted_token_ids"], [0, 16]) == 2).all()


@pytest.mark.parametrize("T,K,E", [(1, 6, 256), (4, 4, 16), (8, 6, 256), (3, 1, 3)])
def test_naive_layout_holds_the_same_pairs_as_the_contiguous_one(T, K, E):
    rng = np.random.default_rng(T * 7 + E)
    ids = synth.topk_ids_random(rng, T, E, K, 0.5)
    a = moe.permute_naive(ids, E)
    c = moe.permute(ids, E, 16)
    assert a["U"] == c["U"]                       # fits the contiguous layout's buffers (align 16)
    inv = a["inv_perm"].reshape(-1)
    assert np.array_equal(a["sorted_token_ids"][inv], np.arange(T * K))
    assert np.array_equal(a["expert_ids"][inv], ids.reshape(-1))
    assert (inv % 16 == 0).all() and len(set((inv // 16).tolist())) == T * K    # one pair per 16-row block
    real = a["expert_ids"] >= 0
    assert real.sum() == T * K and (a["sorted_token_ids"][~real] == T * K).all()
    # the same (token, expert) rows as the sorted layout, in another order
    pairs_a = sorted(zip(a["sorted_token_ids"][real] // K, a["expert_ids"][real]))
    rc = c["expert_ids"] >= 0
    pairs_c = sorted(zip(c["sorted_token_ids"][rc] // K, c["expert_ids"][rc]))
    assert pairs_a == pairs_c


def test_naive_layout_rejects_too_many_pairs():
    with pytest.raises(ValueError):
        moe.permute_naive(np.zeros((5, 4), dtype=np.int32) + np.arange(4), 16)
