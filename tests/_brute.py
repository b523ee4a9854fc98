"""Independent brute-force references used to pin the oracle (tests only).

None of this shares code with ``oracle/``: trees are found by enumerating
every node of the implicit top-k tree and sorting, visibility by rank-path
prefixes, and attention by plain numpy softmax over an explicitly gathered
sequence.
"""
from __future__ import annotations

import itertools

import numpy as np

from tree_speculative_decoding_gb300.workloads import bf16_bits_to_f32


def enumerate_nodes(topk_logp_b: np.ndarray, max_depth: int, K: int):
    """All nodes (rank paths of length 1..max_depth) with fp32 root-to-leaf scores."""
    nodes = []
    for d in range(1, max_depth + 1):
        for path in itertools.product(range(K), repeat=d):
            s = np.float32(0.0)
            for level, r in enumerate(path):
                s = np.float32(s + np.float32(topk_logp_b[level, r]))
            nodes.append((path, s))
    return nodes


def brute_tree(topk_logp_b, topk_ids_b, root_id, budget, max_depth, K):
    """Top-`budget` nodes by (score desc, depth asc, rank path asc), in that
    order, as (node_token, parent, depth, paths)."""
    nodes = enumerate_nodes(topk_logp_b, max_depth, K)
    nodes.sort(key=lambda e: (-float(e[1]), len(e[0]), e[0]))
    chosen = [p for p, _ in nodes[:budget]]
    if len(chosen) < budget:
        raise ValueError("implicit tree too small")
    index = {(): 0}
    tok, par, dep, paths = [int(root_id)], [-1], [0], [()]
    for n, p in enumerate(chosen, start=1):
        index[p] = n
        tok.append(int(topk_ids_b[len(p) - 1, p[-1]]))
        par.append(index[p[:-1]])   # KeyError here would mean the set is not prefix-closed
        dep.append(len(p))
        paths.append(p)
    return np.array(tok, np.int32), np.array(par, np.int32), np.array(dep, np.int32), paths


def visible_from_paths(paths):
    """vis[i][j] = node j's rank path is a prefix of node i's (ancestor or self)."""
    T = len(paths)
    vis = np.zeros((T, T), bool)
    for i, pi in enumerate(paths):
        for j, pj in enumerate(paths):
            vis[i, j] = pi[: len(pj)] == pj
    return vis


def bf16_rows(bits: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


def attend(qvec: np.ndarray, keys: np.ndarray, scale: float):
    """softmax(scale * keys @ q) @ keys[:, :512] and its log-sum-exp, fp64."""
    s = scale * (keys @ qvec)
    m = s.max()
    w = np.exp(s - m)
    out = (w[:, None] * keys[:, :512]).sum(axis=0) / w.sum()
    return out, m + np.log(w.sum())
