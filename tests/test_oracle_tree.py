"""Pins for the oracle's tree builder (CPU only).

The oracle builds the tree with a heap; these tests check it against a
different algorithm (enumerate every node, sort by the total order, take the
first `budget`), against a hand-worked example, and against invariants the
best-first expansion must satisfy.
"""
import json
import os

import numpy as np
import pytest

from tests import _brute
from tree_speculative_decoding_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tree_worked_example.json")


def _single(oracle_mod, logp, ids, root, budget, max_depth, K):
    qo = np.array([0, budget + 1], np.int32)
    return oracle_mod.build_tree(np.asarray(logp, np.float32)[None], np.asarray(ids, np.int32)[None],
                                 np.array([root], np.int32), np.array([budget], np.int32), qo,
                                 max_depth, K)


def test_worked_example(oracle_mod):
    g = json.load(open(GOLDEN))
    tok, par, dep = _single(oracle_mod, g["topk_logp"], g["topk_ids"], g["root_id"], g["budget"],
                            g["max_depth"], g["K"])
    assert tok.tolist() == g["node_token"]
    assert par.tolist() == g["parent"]
    assert dep.tolist() == g["depth"]


def test_worked_tie_case(oracle_mod):
    g = json.load(open(GOLDEN))["tie_case"]
    tok, par, dep = _single(oracle_mod, g["topk_logp"], g["topk_ids"], g["root_id"], g["budget"],
                            g["max_depth"], g["K"])
    assert tok.tolist() == g["node_token"]
    assert par.tolist() == g["parent"]
    assert dep.tolist() == g["depth"]


def _random_topk(rng, max_depth, K, ties=False, vocab=1000):
    if ties:   # coarse grid of values: many exact fp32 ties
        lp = -rng.integers(0, 4, size=(max_depth, K)).astype(np.float32) * np.float32(0.5)
    else:
        lp = -rng.exponential(1.0, size=(max_depth, K)).astype(np.float32)
    lp = -np.sort(-lp, axis=1)
    ids = np.stack([rng.choice(vocab, size=K, replace=False) for _ in range(max_depth)]).astype(np.int32)
    return lp, ids


@pytest.mark.parametrize("max_depth,K", [(1, 5), (2, 3), (3, 3), (4, 4), (7, 2), (3, 1), (7, 1)])
@pytest.mark.parametrize("ties", [False, True])
def test_heap_equals_sorted_enumeration(oracle_mod, max_depth, K, ties):
    rng = np.random.default_rng(1000 * max_depth + 10 * K + int(ties))
    total = sum(K ** d for d in range(1, max_depth + 1))
    for trial in range(6):
        lp, ids = _random_topk(rng, max_depth, K, ties)
        for budget in sorted({0, 1, min(total, 3), min(total, 9), total // 2, total}):
            root = int(rng.integers(0, 1000))
            tok, par, dep = _single(oracle_mod, lp, ids, root, budget, max_depth, K)
            btok, bpar, bdep, _ = _brute.brute_tree(lp, ids, root, budget, max_depth, K)
            np.testing.assert_array_equal(tok, btok)
            np.testing.assert_array_equal(par, bpar)
            np.testing.assert_array_equal(dep, bdep)


def test_chain_when_topk_is_one(oracle_mod):
    lp = -np.arange(1, 8, dtype=np.float32)[:, None] / 4
    ids = np.arange(100, 107, dtype=np.int32)[:, None]
    for budget in range(0, 8):
        tok, par, dep = _single(oracle_mod, lp, ids, 3, budget, 7, 1)
        assert dep.tolist() == list(range(budget + 1))
        assert par.tolist() == [-1] + list(range(budget))
        assert tok.tolist() == [3] + list(range(100, 100 + budget))


def test_budget_beyond_implicit_tree_is_an_error(oracle_mod):
    lp = np.array([[-1.0, -2.0], [-1.0, -2.0]], np.float32)
    ids = np.array([[1, 2], [3, 4]], np.int32)
    _single(oracle_mod, lp, ids, 0, 6, 2, 2)
    with pytest.raises(oracle_mod.OracleError):
        _single(oracle_mod, lp, ids, 0, 7, 2, 2)


def test_unsorted_topk_is_rejected(oracle_mod):
    lp = np.array([[-2.0, -1.0]], np.float32)
    with pytest.raises(oracle_mod.OracleError):
        _single(oracle_mod, lp, np.array([[1, 2]], np.int32), 0, 1, 1, 2)


@pytest.mark.parametrize("name", ["tiny_p21_b8_h8", "mixed_bs32_b16or32_h16"])
def test_invariants_on_workloads(oracle_mod, name):
    wl = workloads.preset(name, fill_pool=False)
    tok, par, dep = oracle_mod.build_tree(wl.topk_logp, wl.topk_ids, wl.root_id, wl.budget,
                                          wl.qo_indptr, wl.max_depth, wl.K)
    for b in range(wl.B):
        lo, hi = wl.qo_indptr[b], wl.qo_indptr[b + 1]
        p, d, t = par[lo:hi], dep[lo:hi], tok[lo:hi]
        assert p[0] == -1 and d[0] == 0 and t[0] == wl.root_id[b]
        score = np.zeros(hi - lo, np.float32)
        rank = np.zeros(hi - lo, np.int64)
        for i in range(1, hi - lo):
            assert 0 <= p[i] < i                      # parent precedes child
            assert d[i] == d[p[i]] + 1 <= wl.max_depth
            row = wl.topk_ids[b, d[i] - 1]
            rank[i] = int(np.nonzero(row == t[i])[0][0])
            score[i] = np.float32(score[p[i]] + wl.topk_logp[b, d[i] - 1, rank[i]])
        assert np.all(np.diff(score[1:]) <= 0)        # popped in non-increasing score
        for i in range(1, hi - lo):                   # sibling-closed: rank r-1 present
            if rank[i] > 0:
                sib = [j for j in range(1, hi - lo) if p[j] == p[i] and rank[j] == rank[i] - 1]
                assert len(sib) == 1 and sib[0] < i
        # per depth, token ids are distinct under one parent
        for i in range(hi - lo):
            kids = t[1:][p[1:] == i]
            assert len(set(kids.tolist())) == len(kids)


def test_brute_force_on_tiny_workload_tree(oracle_mod):
    wl = workloads.preset("tiny_p21_b8_h8", fill_pool=False)
    tok, par, dep = oracle_mod.build_tree(wl.topk_logp, wl.topk_ids, wl.root_id, wl.budget,
                                          wl.qo_indptr, wl.max_depth, wl.K)
    # 4^1 + ... + 4^7 = 21844 nodes enumerated
    btok, bpar, bdep, _ = _brute.brute_tree(wl.topk_logp[0], wl.topk_ids[0], wl.root_id[0],
                                            int(wl.budget[0]), wl.max_depth, wl.K)
    np.testing.assert_array_equal(tok, btok)
    np.testing.assert_array_equal(par, bpar)
    np.testing.assert_array_equal(dep, bdep)
