"""Pins for the oracle's visibility mask and its fp64 attention (CPU only).

Checks against facts fixed independently of the oracle's code: the shapes
log printed on the pages (270 = 9 x (21 + 9) mask entries), popcounts,
rank-path ancestry from a brute-force tree, causal prefill for a chain,
per-node linearisation (plain attention over prefix ++ root-to-node path),
a single visible column, and uniform weights when all scores are equal.
"""
import json
import os

import numpy as np
import pytest

from tests import _brute
from tree_speculative_decoding_gb300 import workloads

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bits(mask, mip, b, i, N):
    W = (N + 31) // 32
    row = mask[mip[b] + i * W: mip[b] + (i + 1) * W]
    return np.array([(row[c // 32] >> (c % 32)) & 1 for c in range(N)], bool), row


def test_shapes_log_mask_size(oracle_mod):
    g = json.load(open(os.path.join(GOLD, "shapes_log_30_column_mask.json")))
    P, T = g["kv_len_max"], g["q_len"]
    parent = np.array([-1] + list(range(T - 1)), np.int32)      # a chain of 9 nodes
    qo = np.array([0, T], np.int32)
    mask, mip = oracle_mod.compile_visibility(parent, qo, np.array([P], np.int32))
    assert T * (P + T) == g["mask_elements"] and P + T == g["row_stride"]
    # one packed word per 30-column row
    assert mip.tolist() == [0, T]
    elements = 0
    for i in range(T):
        bits, row = _bits(mask, mip, 0, i, P + T)
        elements += bits.size
        # chain: ones over the 21 prefix columns and the first i+1 tree columns
        assert row[0] == (1 << (P + i + 1)) - 1
    assert elements == g["mask_elements"]


def test_worked_example_mask(oracle_mod):
    g = json.load(open(os.path.join(GOLD, "tree_worked_example.json")))
    qo = np.array([0, len(g["parent"])], np.int32)
    mask, mip = oracle_mod.compile_visibility(np.array(g["parent"], np.int32), qo,
                                              np.array([g["prefix_len"]], np.int32))
    assert mask.tolist() == g["mask_words"]


def test_mask_indptr_layout(oracle_mod):
    qo = np.array([0, 9, 42, 43], np.int32)
    P = np.array([21, 4096, 0], np.int32)
    mip = oracle_mod.mask_indptr(qo, P)
    # words per row = ceil((P + T) / 32)
    assert mip.tolist() == [0, 9, 9 + 33 * 130, 9 + 33 * 130 + 1]


@pytest.mark.parametrize("seed", range(4))
def test_mask_rows_match_rank_path_ancestry(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    K, D = 3, 4
    lp = -np.sort(rng.exponential(1.0, size=(D, K)), axis=1).astype(np.float32)
    ids = np.stack([rng.choice(50, K, replace=False) for _ in range(D)]).astype(np.int32)
    budget = int(rng.integers(1, 40))
    tok, par, dep, paths = _brute.brute_tree(lp, ids, 7, budget, D, K)
    vis = _brute.visible_from_paths(paths)
    T = budget + 1
    P = int(rng.integers(0, 70))
    mask, mip = oracle_mod.compile_visibility(par, np.array([0, T], np.int32), np.array([P], np.int32))
    W = (P + T + 31) // 32
    for i in range(T):
        bits, row = _bits(mask, mip, 0, i, P + T)
        assert bits[:P].all()
        np.testing.assert_array_equal(bits[P:], vis[i])
        assert bits.sum() == P + dep[i] + 1                 # prefix + ancestors + self
        pad = W * 32 - (P + T)                              # padding bits are zero
        if pad:
            assert (int(row[-1]) >> (32 - pad)) == 0


def _tiny_case(oracle_mod, seed, P, K, D, budget, H=2, pool_extra=7):
    """A small request with random paged slots; returns the pieces for attention."""
    rng = np.random.default_rng(seed)
    lp = -np.sort(rng.exponential(1.0, size=(D, K)), axis=1).astype(np.float32)
    ids = np.stack([rng.choice(100, K, replace=False) for _ in range(D)]).astype(np.int32)
    tok, par, dep, paths = _brute.brute_tree(lp, ids, 1, budget, D, K)
    T = budget + 1
    N = P + T
    pool_rows = N + pool_extra
    slots = rng.permutation(pool_rows)[:N].astype(np.int32)
    pool = workloads.to_bf16_bits(rng.standard_normal((pool_rows, 576)).astype(np.float32))
    q = workloads.to_bf16_bits(rng.standard_normal((T, H, 576)).astype(np.float32))
    qo = np.array([0, T], np.int32)
    kvp = np.array([0, N], np.int32)
    mask, mip = oracle_mod.compile_visibility(par, qo, np.array([P], np.int32))
    return dict(q=q, pool=pool, slots=slots, qo=qo, kvp=kvp, mask=mask, mip=mip, par=par,
                dep=dep, paths=paths, P=P, T=T, H=H)


@pytest.mark.parametrize("seed,P,K,D,budget", [(0, 5, 2, 3, 6), (1, 0, 3, 3, 10), (2, 40, 4, 2, 12),
                                               (3, 33, 1, 7, 7), (4, 17, 3, 4, 30)])
def test_attention_equals_linearised_causal_attention(oracle_mod, seed, P, K, D, budget):
    c = _tiny_case(oracle_mod, seed, P, K, D, budget)
    scale = 0.14468
    out, lse = oracle_mod.verify_attn(c["q"], c["pool"], c["slots"], c["kvp"], c["qo"], c["mask"],
                                      c["mip"], c["H"], scale)
    keys_all = _brute.bf16_rows(c["pool"])
    for i in range(c["T"]):
        # walk the rank path: node j is on i's path iff its path prefixes i's path
        path_nodes = [j for j in range(c["T"]) if c["paths"][i][: len(c["paths"][j])] == c["paths"][j]]
        path_nodes.sort(key=lambda j: len(c["paths"][j]))          # root -> node
        seq = list(c["slots"][: c["P"]]) + [c["slots"][c["P"] + j] for j in path_nodes]
        keys = keys_all[np.array(seq)]
        for h in range(c["H"]):
            qv = _brute.bf16_rows(c["q"][i, h])
            ref, ref_lse = _brute.attend(qv, keys, scale)
            r = i * c["H"] + h
            np.testing.assert_allclose(out[r], ref, rtol=1e-10, atol=1e-12)
            assert abs(lse[r] - ref_lse) < 1e-10


def test_chain_equals_causal_prefill(oracle_mod):
    c = _tiny_case(oracle_mod, 11, 23, 1, 7, 7, H=3)
    scale = 0.2
    out, lse = oracle_mod.verify_attn(c["q"], c["pool"], c["slots"], c["kvp"], c["qo"], c["mask"],
                                      c["mip"], c["H"], scale)
    keys = _brute.bf16_rows(c["pool"])[c["slots"]]          # P + T contiguous positions
    N = c["P"] + c["T"]
    Q = _brute.bf16_rows(c["q"])                            # [T, H, 576]
    S = scale * np.einsum("thd,nd->thn", Q, keys)
    causal = np.arange(N)[None, :] <= (c["P"] + np.arange(c["T"]))[:, None]   # [T, N]
    S = np.where(causal[:, None, :], S, -np.inf)
    m = S.max(-1, keepdims=True)
    w = np.exp(S - m)
    ref = np.einsum("thn,nd->thd", w, keys[:, :512]) / w.sum(-1, keepdims=True)
    np.testing.assert_allclose(out.reshape(c["T"], c["H"], 512), ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("prefix", [[0], [31, 33], [4096]])
def test_chain_of_128_gives_the_causal_mask(oracle_mod, prefix):
    # parent[i] = i - 1 over q_len 128 (the largest): row i sees columns [0, P + i]
    B, T = len(prefix), 128
    par = np.tile(np.arange(-1, T - 1, dtype=np.int32), B)
    qo = (np.arange(B + 1) * T).astype(np.int32)
    mask, mip = oracle_mod.compile_visibility(par, qo, np.array(prefix, np.int32))
    for b, P in enumerate(prefix):
        W = (P + T + 31) // 32
        words = np.ascontiguousarray(mask[mip[b]:mip[b + 1]]).astype("<u4")
        bits = np.unpackbits(words.view(np.uint8), bitorder="little").reshape(T, W * 32)
        causal = np.arange(W * 32)[None, :] <= (P + np.arange(T))[:, None]
        np.testing.assert_array_equal(bits.astype(bool), causal)


def test_single_visible_column_returns_its_value_row(oracle_mod):
    c = _tiny_case(oracle_mod, 5, 0, 2, 2, 3, H=4)     # prefix 0: the root sees only itself
    out, lse = oracle_mod.verify_attn(c["q"], c["pool"], c["slots"], c["kvp"], c["qo"], c["mask"],
                                      c["mip"], c["H"], 0.3, rows=np.arange(4))
    v = _brute.bf16_rows(c["pool"][c["slots"][0]])
    for h in range(4):
        assert np.array_equal(out[h], v[:512])             # exact: weight 1 on one row
        s = 0.3 * float(np.dot(_brute.bf16_rows(c["q"][0, h]), v))
        assert abs(lse[h] - s) < 1e-9


def test_equal_scores_give_the_mean_of_visible_values(oracle_mod):
    c = _tiny_case(oracle_mod, 6, 9, 3, 3, 8, H=1)
    zero_q = np.zeros_like(c["q"])                         # every score is 0
    out, lse = oracle_mod.verify_attn(zero_q, c["pool"], c["slots"], c["kvp"], c["qo"], c["mask"],
                                      c["mip"], 1, 0.14468)
    vals = _brute.bf16_rows(c["pool"])[c["slots"]][:, :512]
    for i in range(c["T"]):
        vis, _ = _bits(c["mask"], c["mip"], 0, i, c["P"] + c["T"])
        np.testing.assert_allclose(out[i], vals[vis].mean(axis=0), rtol=1e-12, atol=1e-13)
        assert abs(lse[i] - np.log(vis.sum())) < 1e-12


def test_ragged_batch_rows_match_single_request_calls(oracle_mod):
    a = _tiny_case(oracle_mod, 21, 12, 2, 3, 5, H=2, pool_extra=0)
    b = _tiny_case(oracle_mod, 22, 30, 3, 2, 9, H=2, pool_extra=0)
    pool = np.concatenate([a["pool"], b["pool"]])
    slots = np.concatenate([a["slots"], b["slots"] + a["pool"].shape[0]]).astype(np.int32)
    qo = np.array([0, a["T"], a["T"] + b["T"]], np.int32)
    kvp = np.array([0, a["P"] + a["T"], a["P"] + a["T"] + b["P"] + b["T"]], np.int32)
    par = np.concatenate([a["par"], b["par"]])
    mask, mip = oracle_mod.compile_visibility(par, qo, np.array([a["P"], b["P"]], np.int32))
    q = np.concatenate([a["q"], b["q"]])
    out, lse = oracle_mod.verify_attn(q, pool, slots, kvp, qo, mask, mip, 2, 0.14468)
    oa, la = oracle_mod.verify_attn(a["q"], a["pool"], a["slots"], a["kvp"], a["qo"], a["mask"],
                                    a["mip"], 2, 0.14468)
    ob, lb = oracle_mod.verify_attn(b["q"], b["pool"], b["slots"], b["kvp"], b["qo"], b["mask"],
                                    b["mip"], 2, 0.14468)
    np.testing.assert_array_equal(out, np.concatenate([oa, ob]))
    np.testing.assert_array_equal(lse, np.concatenate([la, lb]))


def test_thread_count_is_per_call(oracle_mod):
    # rows are independent, so one thread and all threads give the same bits; a
    # one-thread call leaves the default team size of later calls unchanged
    c = _tiny_case(oracle_mod, 8, 40, 3, 3, 12, H=8)
    before = oracle_mod.num_threads()
    one = oracle_mod.verify_attn(c["q"], c["pool"], c["slots"], c["kvp"], c["qo"], c["mask"],
                                 c["mip"], c["H"], 0.2, nthreads=1)
    assert oracle_mod.num_threads() == before
    every = oracle_mod.verify_attn(c["q"], c["pool"], c["slots"], c["kvp"], c["qo"], c["mask"],
                                   c["mip"], c["H"], 0.2)
    for a, b in zip(one, every):
        assert np.array_equal(a, b)
