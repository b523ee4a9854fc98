"""Pins for the oracle's greedy accept walk (CPU only)."""
import json
import os

import numpy as np
import pytest

from tests import _brute

GOLD = os.path.join(os.path.dirname(__file__), "golden", "tree_worked_example.json")


def test_worked_example(oracle_mod):
    g = json.load(open(GOLD))
    qo = np.array([0, len(g["parent"])], np.int32)
    alen, acc, com, bon = oracle_mod.accept(g["node_token"], g["parent"], qo, g["target_argmax"],
                                            g["max_depth"])
    assert alen.tolist() == [g["accept_len"]]
    assert acc[0].tolist() == g["accepted_nodes"]
    assert com[0].tolist() == g["commit_tokens"]
    assert bon.tolist() == [g["bonus"]]


def _tree(seed, K=3, D=4, budget=25):
    rng = np.random.default_rng(seed)
    lp = -np.sort(rng.exponential(1.0, size=(D, K)), axis=1).astype(np.float32)
    ids = np.stack([rng.choice(60, K, replace=False) for _ in range(D)]).astype(np.int32)
    return _brute.brute_tree(lp, ids, 9, budget, D, K)


@pytest.mark.parametrize("seed", range(6))
def test_never_matching_target_accepts_only_the_root(oracle_mod, seed):
    tok, par, dep, _ = _tree(seed)
    T = len(tok)
    argmax = np.full(T, -5, np.int32)
    argmax[0] = 12345
    alen, acc, com, bon = oracle_mod.accept(tok, par, np.array([0, T], np.int32), argmax, 4)
    assert alen[0] == 1 and bon[0] == 12345
    assert acc[0].tolist() == [0, -1, -1, -1, -1]
    assert com[0].tolist() == [12345, -1, -1, -1, -1]


@pytest.mark.parametrize("seed", range(6))
def test_chain_forcing_target_accepts_the_leftmost_path(oracle_mod, seed):
    tok, par, dep, paths = _tree(seed)
    T = len(tok)
    # the target always predicts the rank-0 child's token (the oracle drafter's
    # golden token), so the walk must follow rank paths (0), (0,0), (0,0,0), ...
    index = {p: n for n, p in enumerate(paths)}
    argmax = np.full(T, -7, np.int32)
    for n, p in enumerate(paths):
        child = p + (0,)
        if child in index:
            argmax[n] = tok[index[child]]
    leftmost = [n for n, p in enumerate(paths) if all(r == 0 for r in p)]
    alen, acc, com, bon = oracle_mod.accept(tok, par, np.array([0, T], np.int32), argmax, 4)
    assert alen[0] == len(leftmost)
    assert acc[0][: alen[0]].tolist() == leftmost
    assert com[0][: alen[0] - 1].tolist() == [int(tok[n]) for n in leftmost[1:]]
    assert bon[0] == argmax[leftmost[-1]]


@pytest.mark.parametrize("seed", range(10))
def test_random_targets_respect_bounds_and_follow_parent_links(oracle_mod, seed):
    rng = np.random.default_rng(100 + seed)
    tok, par, dep, _ = _tree(seed, K=2, D=5, budget=20)
    T = len(tok)
    # mix: half the nodes predict one of their children's tokens
    argmax = rng.integers(0, 60, T).astype(np.int32)
    alen, acc, com, bon = oracle_mod.accept(tok, par, np.array([0, T], np.int32), argmax, 5)
    n = int(alen[0])
    assert 1 <= n <= dep.max() + 1
    nodes = acc[0][:n]
    assert nodes[0] == 0
    for a, b in zip(nodes[:-1], nodes[1:]):
        assert par[b] == a and tok[b] == argmax[a]
    last = nodes[-1]
    assert not np.any((par == last) & (tok == argmax[last]))   # the walk stops only when stuck
    assert (acc[0][n:] == -1).all() and (com[0][n:] == -1).all()


def test_duplicate_child_tokens_take_the_lower_index(oracle_mod):
    tok = np.array([1, 5, 5, 6], np.int32)
    par = np.array([-1, 0, 0, 2], np.int32)
    argmax = np.array([5, 9, 6, 9], np.int32)
    alen, acc, com, bon = oracle_mod.accept(tok, par, np.array([0, 4], np.int32), argmax, 3)
    assert acc[0].tolist() == [0, 1, -1, -1] and bon[0] == 9


def test_budget_zero_is_autoregressive(oracle_mod):
    alen, acc, com, bon = oracle_mod.accept([3], [-1], np.array([0, 1], np.int32), [77], 7)
    assert alen[0] == 1 and com[0][0] == 77 and bon[0] == 77
