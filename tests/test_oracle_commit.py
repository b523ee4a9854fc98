"""Pins for the oracle's KV commit (CPU only).

"The Architecture of a Speculative Decoding Engine" (the append-then-compact
scheme and "The Final Resolution: A Concrete Trace"): the step appended every
tree node's latent after the committed prefix; after acceptance only the
accepted nodes' latents are gathered into contiguous positions, and the cache
grows by accept_len.  The checks below restate that outcome through routes
that do not run the oracle's copy loop: a hand-worked example, the accepted
path re-derived from parent links, and the rows that must stay untouched.
"""
import numpy as np
import pytest

from tree_speculative_decoding_gb300 import workloads

D = 576


def _tagged_pool(rows):
    # row r holds the value r + 1 in every entry (r < 65535): rows are told apart by eye
    return np.repeat(np.arange(1, rows + 1, dtype=np.uint16)[:, None], D, axis=1)


def test_hand_worked_example(oracle_mod):
    # one request: prefix 3, tree of 6 nodes (positions 3..8), stored in
    # scattered pool rows; the accepted path is root -> node 2 -> node 5
    kv_indices = np.array([7, 0, 4, 9, 2, 8, 1, 5, 6], np.int32)  # position -> pool row
    kv_indptr = np.array([0, 9], np.int32)
    qo_indptr = np.array([0, 6], np.int32)
    pool = _tagged_pool(10)
    new_pool, new_len = oracle_mod.commit_kv(pool, kv_indices, kv_indptr, qo_indptr,
                                             np.array([3], np.int32),
                                             np.array([[0, 2, 5, -1]], np.int32), 3)
    # position 3 (row 9) keeps the root; position 4 (row 2) takes node 2's latent,
    # which was at position 5 (row 8), tag 9; position 5 (row 8) takes node 5's
    # latent, at position 8 (row 6), tag 7 -- row 8 is a destination and a
    # source at once, and position 4 gets its value from before the commit
    expect = pool.copy()
    expect[2] = 9
    expect[8] = 7
    np.testing.assert_array_equal(new_pool, expect)
    assert new_len.tolist() == [6]
    np.testing.assert_array_equal(pool, _tagged_pool(10))  # input untouched


def test_root_only_accept_is_a_no_op(oracle_mod):
    wl = workloads.preset("tiny_p21_b8_h8")
    pool = wl.kv_pool
    B = wl.B
    acc = np.full((B, wl.max_depth + 1), -1, np.int32)
    acc[:, 0] = 0
    new_pool, new_len = oracle_mod.commit_kv(pool, wl.kv_indices, wl.kv_indptr, wl.qo_indptr,
                                             np.ones(B, np.int32), acc, wl.max_depth)
    np.testing.assert_array_equal(new_pool, pool)
    assert new_len.tolist() == (wl.prefix_len + 1).tolist()


def test_chain_accepting_every_node_is_a_no_op(oracle_mod):
    # a chain tree accepted to the end: node k already sits at position P + k
    wl = workloads.make_workload("chain_commit", 91, 2, 4, [30, 7], [6, 3], 1, 300, 2.0)
    T = np.diff(wl.qo_indptr)
    acc = np.full((wl.B, wl.max_depth + 1), -1, np.int32)
    for b in range(wl.B):
        acc[b, :T[b]] = np.arange(T[b])
    new_pool, new_len = oracle_mod.commit_kv(wl.kv_pool, wl.kv_indices, wl.kv_indptr,
                                             wl.qo_indptr, T.astype(np.int32), acc, wl.max_depth)
    np.testing.assert_array_equal(new_pool, wl.kv_pool)
    assert new_len.tolist() == (wl.prefix_len + T).tolist()


@pytest.mark.parametrize("name", ["tiny_p21_b8_h8", "mixed_bs32_b16or32_h16"])
def test_committed_sequence_is_prefix_then_accepted_path(oracle_mod, name):
    # the committed sequence must read: the prefix rows as they were, then the
    # original latents of the root-to-leaf path that ends at the last accepted
    # node, found here by walking parent links up from that node
    if name.startswith("mixed"):  # the mixed recipe at a size the test reads quickly
        wl = workloads.make_workload("mixed_small", 17, 6, 4, [40, 3, 65, 0, 31, 128],
                                     [16, 32, 16, 32, 5, 9], 8, 500, 1.0, p_match=0.5)
        coin = wl.argmax_coin.astype(bool)
        coin[wl.qo_indptr[:-1]] = True  # every root's best child matches; deeper nodes by coin
    else:
        wl = workloads.preset(name)
        coin = np.ones(wl.total_q, bool)  # the target follows the best child everywhere
    tok, par, dep = oracle_mod.build_tree(wl.topk_logp, wl.topk_ids, wl.root_id, wl.budget,
                                          wl.qo_indptr, wl.max_depth, wl.K)
    argmax = oracle_mod.best_child_argmax(par, wl.qo_indptr, tok, coin, wl.argmax_random)
    alen, acc, com, bon = oracle_mod.accept(tok, par, wl.qo_indptr, argmax, wl.max_depth)
    assert alen.max() > 1  # some request accepts a draft
    new_pool, new_len = oracle_mod.commit_kv(wl.kv_pool, wl.kv_indices, wl.kv_indptr,
                                             wl.qo_indptr, alen, acc, wl.max_depth)
    written = np.zeros(len(wl.kv_pool), bool)
    for b in range(wl.B):
        q0 = int(wl.qo_indptr[b])
        P = int(wl.prefix_len[b])
        idx = wl.kv_indices[int(wl.kv_indptr[b]):int(wl.kv_indptr[b + 1])]
        n = int(alen[b])
        path = [int(acc[b, n - 1])]
        while path[-1] != 0:
            path.append(int(par[q0 + path[-1]]))
        path.reverse()
        assert path == acc[b, :n].tolist()
        for k, node in enumerate(path):
            np.testing.assert_array_equal(new_pool[idx[P + k]], wl.kv_pool[idx[P + node]])
            written[idx[P + k]] = True
        np.testing.assert_array_equal(new_pool[idx[:P]], wl.kv_pool[idx[:P]])
        assert new_len[b] == P + n
    np.testing.assert_array_equal(new_pool[~written], wl.kv_pool[~written])


@pytest.mark.parametrize("acc_row,alen", [
    ([1, 2, -1, -1], 2),     # does not start at the root
    ([0, 3, 3, -1], 3),      # not strictly increasing
    ([0, 2, 9, -1], 3),      # a node past q_len
    ([0, 1, 2, 3], 5),       # longer than max_depth + 1
    ([0, -1, -1, -1], 0),    # empty
])
def test_rejects_paths_that_are_not_accepted_paths(oracle_mod, acc_row, alen):
    kv_indices = np.arange(12, dtype=np.int32)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.commit_kv(_tagged_pool(12), kv_indices, np.array([0, 12], np.int32),
                             np.array([0, 6], np.int32), np.array([alen], np.int32),
                             np.array([acc_row], np.int32), 3)
