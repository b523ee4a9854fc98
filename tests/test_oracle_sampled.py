"""Pins for the oracle's sampling accept and tree links (CPU only).

"The DDTree CUDA Graph Fix ...", section "Temperature Support: Already Working
for Linear, Planned for DDTree": sampling accept runs tree rejection sampling
on the target distribution (temperature, top-k, top-p), with the tree given
as (retrieve_index, retrieve_next_token, retrieve_next_sibling).  The pages
give no algorithm text, so the reading (R15) is pinned by what any correct
reading must satisfy:
- every emitted token is distributed as the target distribution, a Monte Carlo
  check against a softmax computed here, and with top-p against a brute-force
  nucleus (every distinct logit tried as the threshold);
- at temperature 0, and for a vanishing top-p, it is the greedy walk; top-p of
  1 (or outside (0, 1)) is no top-p;
- hand-worked examples, one where the nucleus changes the walk and one where
  tied tokens at the threshold are all kept;
- the links agree with the children sets.
"""
import numpy as np
import pytest

from tests import _brute


def _tree(seed, K=3, D=4, budget=25):
    rng = np.random.default_rng(seed)
    lp = -np.sort(rng.exponential(1.0, size=(D, K)), axis=1).astype(np.float32)
    ids = np.stack([rng.choice(40, K, replace=False) for _ in range(D)]).astype(np.int32)
    return _brute.brute_tree(lp, ids, 9, budget, D, K)


@pytest.mark.parametrize("seed", range(5))
def test_tree_links_follow_the_children_sets(oracle_mod, seed):
    tok, par, dep, _ = _tree(seed)
    T = len(tok)
    qo = np.array([0, T], np.int32)
    fc, ns, ri = oracle_mod.tree_links(par, qo)
    children = {n: sorted(c for c in range(1, T) if par[c] == n) for n in range(T)}
    for n in range(T):
        assert fc[n] == (children[n][0] if children[n] else -1)
        sibs = children[par[n]] if n > 0 else [0]
        later = [c for c in sibs if c > n]
        assert ns[n] == (later[0] if later else -1)
    assert ri.tolist() == list(range(T))


def test_tree_links_ragged_rows_are_global(oracle_mod):
    par = np.array([-1, 0, 0, 1, -1, 0], np.int32)
    fc, ns, ri = oracle_mod.tree_links(par, np.array([0, 4, 6], np.int32))
    assert fc.tolist() == [1, 3, -1, -1, 1, -1]
    assert ns.tolist() == [-1, 2, -1, -1, -1, -1]
    assert ri.tolist() == [0, 1, 2, 3, 4, 5]


def _softmax_topk(l, T, k):
    l = l.astype(np.float64)
    keep = np.ones_like(l, bool) if k <= 0 or k >= len(l) else l >= np.sort(l)[::-1][k - 1]
    w = np.where(keep, np.exp((l - l.max()) / T), 0.0)
    return w / w.sum()


def test_hand_worked_example(oracle_mod):
    # vocab 4, T = 1, logits log([1, 2, 1, 4]) at both nodes: p = [1, 2, 1, 4] / 8.
    # root (token 7) has children 1 (token 3) and 2 (token 1).
    #  child 1: a = p(3) / 1 = 0.5, coin 0.6 -> rejected, residual mass 0.5
    #  child 2: a = p(1) / 0.5 = 0.5, coin 0.3 -> taken
    # node 2 has no children; bonus coin 0.5: residual p, cumulative
    #  0.125, 0.375, 0.5, 1.0 first exceeds 0.5 at token 3
    par = np.array([-1, 0, 0], np.int32)
    tok = np.array([7, 3, 1], np.int32)
    logits = np.tile(np.log(np.array([1, 2, 1, 4], np.float32)), (3, 1)).astype(np.float32)
    coins = np.array([[0.6, 0.3, 0.9], [0.9, 0.9, 0.9], [0.9, 0.9, 0.5]], np.float32)
    alen, acc, com, bon = oracle_mod.accept_sampled(tok, par, np.array([0, 3], np.int32), logits,
                                                    np.array([1.0], np.float32),
                                                    np.array([0], np.int32), coins, 3)
    assert alen.tolist() == [2]
    assert acc[0].tolist() == [0, 2, -1, -1]
    assert com[0].tolist() == [1, 3, -1, -1]
    assert bon.tolist() == [3]


@pytest.mark.parametrize("seed", range(6))
def test_temperature_zero_is_the_greedy_walk(oracle_mod, seed):
    tok, par, dep, _ = _tree(seed)
    T = len(tok)
    rng = np.random.default_rng(100 + seed)
    logits = rng.normal(size=(T, 40)).astype(np.float32)
    # make the argmax land on a child token often, so that walks go deep
    for n in range(T):
        kids = [c for c in range(1, T) if par[c] == n]
        if kids and rng.random() < 0.7:
            logits[n, tok[kids[rng.integers(len(kids))]]] = 9.0
    coins = rng.random((T, 4)).astype(np.float32)
    qo = np.array([0, T], np.int32)
    got = oracle_mod.accept_sampled(tok, par, qo, logits, np.array([0.0], np.float32),
                                    np.array([5], np.int32), coins, 4)
    ref = oracle_mod.accept(tok, par, qo, logits.argmax(axis=1).astype(np.int32), 4)
    for g, r in zip(got, ref):
        np.testing.assert_array_equal(g, r)
    # top_k = 1 keeps only the argmax token: the same walk at any temperature
    got1 = oracle_mod.accept_sampled(tok, par, qo, logits, np.array([0.8], np.float32),
                                     np.array([1], np.int32), coins, 4)
    for g, r in zip(got1, ref):
        np.testing.assert_array_equal(g, r)


@pytest.mark.parametrize("temp,top_k,kids", [(1.0, 0, [2, 5, 0]), (0.6, 4, [5, 1]), (1.3, 0, [])])
def test_emitted_tokens_follow_the_target_distribution(oracle_mod, temp, top_k, kids):
    # one root with children carrying tokens `kids` (each child a leaf); over many
    # coin draws, the first emitted token must follow p(root), and after taking
    # a child the second must follow p(child)
    V, n = 6, 20000
    rng = np.random.default_rng(7)
    T = 1 + len(kids)
    par = np.array([-1] + [0] * len(kids), np.int32)
    tok = np.array([9] + kids, np.int32)
    logits = rng.normal(scale=1.5, size=(T, V)).astype(np.float32)
    # n independent requests sharing the tree, coins drawn per request
    B = n
    par_b = np.tile(par, B)
    tok_b = np.tile(tok, B)
    logits_b = np.tile(logits, (B, 1))
    qo_b = np.arange(B + 1, dtype=np.int32) * T
    coins = rng.random((B * T, 4)).astype(np.float32)
    alen, acc, com, bon = oracle_mod.accept_sampled(
        tok_b, par_b, qo_b, logits_b, np.full(B, temp, np.float32), np.full(B, top_k, np.int32),
        coins, 2)
    p_root = _softmax_topk(logits[0], temp, top_k)
    first = com[:, 0]
    freq = np.bincount(first, minlength=V) / B
    assert np.abs(freq - p_root).max() < 4.5 * np.sqrt(p_root.max() * (1 - p_root.min()) / B) + 1e-9
    for ci, t in enumerate(kids):
        took = first == t
        if took.sum() < 2000:
            continue
        p_child = _softmax_topk(logits[1 + ci], temp, top_k)
        f2 = np.bincount(com[took, 1], minlength=V) / took.sum()
        assert np.abs(f2 - p_child).max() < 4.5 * np.sqrt(0.25 / took.sum())


def test_more_children_than_coins_is_rejected(oracle_mod):
    par = np.array([-1, 0, 0, 0], np.int32)
    tok = np.array([0, 1, 2, 3], np.int32)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.accept_sampled(tok, par, np.array([0, 4], np.int32),
                                  np.zeros((4, 5), np.float32), np.array([1.0], np.float32),
                                  np.array([0], np.int32), np.full((4, 3), 0.99, np.float32), 3)


def _deep_case(seed, V=40, T_bias=6.0):
    tok, par, dep, _ = _tree(seed)
    T = len(tok)
    rng = np.random.default_rng(200 + seed)
    logits = rng.normal(size=(T, V)).astype(np.float32)
    for n in range(T):
        kids = [c for c in range(1, T) if par[c] == n]
        if kids:
            logits[n, tok[kids[0]]] += T_bias
    coins = rng.random((T, 4)).astype(np.float32)
    return tok, par, np.array([0, T], np.int32), logits, coins


@pytest.mark.parametrize("seed", range(4))
def test_a_constant_added_to_the_logits_changes_nothing(oracle_mod, seed):
    # softmax is shift invariant; +8 is exact in fp32 for these magnitudes
    tok, par, qo, logits, coins = _deep_case(seed)
    t, k = np.array([0.9], np.float32), np.array([0], np.int32)
    a = oracle_mod.accept_sampled(tok, par, qo, logits, t, k, coins, 4)
    b = oracle_mod.accept_sampled(tok, par, qo, logits + np.float32(8.0), t, k, coins, 4)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("seed", range(4))
def test_top_k_of_the_whole_vocabulary_is_no_top_k(oracle_mod, seed):
    tok, par, qo, logits, coins = _deep_case(seed)
    t = np.array([1.1], np.float32)
    a = oracle_mod.accept_sampled(tok, par, qo, logits, t, np.array([0], np.int32), coins, 4)
    b = oracle_mod.accept_sampled(tok, par, qo, logits, t, np.array([40], np.int32), coins, 4)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("seed", range(4))
def test_a_vanishing_temperature_is_the_greedy_walk(oracle_mod, seed):
    # with distinct logits, T -> 0 puts all mass on the argmax
    tok, par, qo, logits, coins = _deep_case(seed)
    a = oracle_mod.accept_sampled(tok, par, qo, logits, np.array([1e-3], np.float32),
                                  np.array([0], np.int32), coins, 4)
    g = oracle_mod.accept(tok, par, qo, logits.argmax(axis=1).astype(np.int32), 4)
    for x, y in zip(a, g):
        np.testing.assert_array_equal(x, y)


def test_a_one_token_vocabulary_accepts_the_matching_child(oracle_mod):
    # p = 1 on token 0: the child carrying token 0 is always taken (coin < 1),
    # any child before it is rejected with zero mass removed, and the bonus is 0
    par = np.array([-1, 0, 0, 2], np.int32)
    tok = np.array([5, 3, 0, 0], np.int32)
    coins = np.full((4, 4), 0.999, np.float32)
    alen, acc, com, bon = oracle_mod.accept_sampled(tok, par, np.array([0, 4], np.int32),
                                                    np.zeros((4, 1), np.float32),
                                                    np.array([1.0], np.float32),
                                                    np.array([0], np.int32), coins, 3)
    assert alen.tolist() == [3]
    assert acc[0].tolist() == [0, 2, 3, -1]
    assert com[0].tolist() == [0, 0, 0, -1]
    assert bon.tolist() == [0]


# ------------------------------------------------------------------- top-p
def _nucleus(l, T, k, top_p):
    """Brute force of the top-p reading: tau is the largest logit x whose mass
    S(x) = p(logit >= x) reaches top_p; the tokens at or above tau, renormalised."""
    p = _softmax_topk(l, T, k)
    if not 0.0 < top_p < 1.0:
        return p
    lv = l.astype(np.float64)
    for x in sorted(set(lv[p > 0].tolist()), reverse=True):
        if p[lv >= x].sum() >= top_p:
            q = np.where(lv >= x, p, 0.0)
            return q / q.sum()
    raise AssertionError("the whole mass never reaches top_p")


@pytest.mark.parametrize("seed", range(4))
def test_top_p_of_one_or_outside_the_unit_interval_is_no_top_p(oracle_mod, seed):
    tok, par, qo, logits, coins = _deep_case(seed)
    t, k = np.array([1.1], np.float32), np.array([0], np.int32)
    ref = oracle_mod.accept_sampled(tok, par, qo, logits, t, k, coins, 4)
    for tp in (1.0, 1.5, 0.0, -0.5):
        got = oracle_mod.accept_sampled(tok, par, qo, logits, t, k, coins, 4,
                                        top_p=np.array([tp], np.float32))
        for x, y in zip(got, ref):
            np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("seed", range(4))
def test_a_vanishing_top_p_is_the_greedy_walk(oracle_mod, seed):
    # with distinct logits the nucleus of a tiny top_p is the argmax alone
    tok, par, qo, logits, coins = _deep_case(seed)
    got = oracle_mod.accept_sampled(tok, par, qo, logits, np.array([1.3], np.float32),
                                    np.array([0], np.int32), coins, 4,
                                    top_p=np.array([1e-6], np.float32))
    g = oracle_mod.accept(tok, par, qo, logits.argmax(axis=1).astype(np.int32), 4)
    for x, y in zip(got, g):
        np.testing.assert_array_equal(x, y)


def test_top_p_hand_worked_example(oracle_mod):
    # vocab 4, T = 1, logits log([1, 2, 1, 4]): p = [1, 2, 1, 4] / 8.  In logit
    # order the mass reaches 0.5 (token 3), 0.75 (token 1), 1.0 (tokens 0 and 2).
    # top_p 0.6: tau = log 2, the nucleus is {3, 1} with p = {3: 2/3, 1: 1/3}.
    # root (token 7): child 1 (token 0) has p 0 and is rejected, the residual
    # keeps mass 1; child 2 (token 1): a = 1/3, coin 0.3 -> taken.  Node 2 is a
    # leaf; bonus coin 0.5: cumulative 1/3 at id 1, 1 at id 3 -> token 3.
    # Without top-p child 1 leaves mass 7/8, child 2 gets a = 2/7 < 0.3 and is
    # rejected, so the nucleus changes the walk.
    par = np.array([-1, 0, 0], np.int32)
    tok = np.array([7, 0, 1], np.int32)
    logits = np.tile(np.log(np.array([1, 2, 1, 4], np.float32)), (3, 1)).astype(np.float32)
    coins = np.array([[0.6, 0.3, 0.9], [0.9, 0.9, 0.9], [0.9, 0.9, 0.5]], np.float32)
    args = (tok, par, np.array([0, 3], np.int32), logits, np.array([1.0], np.float32),
            np.array([0], np.int32), coins, 3)
    alen, acc, com, bon = oracle_mod.accept_sampled(*args, top_p=np.array([0.6], np.float32))
    assert alen.tolist() == [2] and acc[0].tolist() == [0, 2, -1, -1]
    assert com[0].tolist() == [1, 3, -1, -1] and bon.tolist() == [3]
    alen0, acc0, com0, bon0 = oracle_mod.accept_sampled(*args)
    assert alen0.tolist() == [1] and acc0[0].tolist() == [0, -1, -1, -1]
    # top_p 0.8 needs the tied tokens 0 and 2, and both are kept: no filter at all
    got = oracle_mod.accept_sampled(*args, top_p=np.array([0.8], np.float32))
    for x, y in zip(got, (alen0, acc0, com0, bon0)):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("temp,top_k,top_p,kids", [(1.0, 0, 0.7, [2, 5, 0]),
                                                   (0.8, 5, 0.6, [5, 1]),
                                                   (1.4, 0, 0.9, [])])
def test_emitted_tokens_follow_the_nucleus(oracle_mod, temp, top_k, top_p, kids):
    # as the temperature/top-k check: first and second emitted tokens against the
    # brute-force nucleus of the root's and the child's logits
    V, n = 8, 20000
    rng = np.random.default_rng(11)
    T = 1 + len(kids)
    par = np.array([-1] + [0] * len(kids), np.int32)
    tok = np.array([9] + kids, np.int32)
    logits = rng.normal(scale=1.5, size=(T, V)).astype(np.float32)
    B = n
    coins = rng.random((B * T, 4)).astype(np.float32)
    alen, acc, com, bon = oracle_mod.accept_sampled(
        np.tile(tok, B), np.tile(par, B), np.arange(B + 1, dtype=np.int32) * T,
        np.tile(logits, (B, 1)), np.full(B, temp, np.float32), np.full(B, top_k, np.int32),
        coins, 2, top_p=np.full(B, top_p, np.float32))
    p_root = _nucleus(logits[0], temp, top_k, top_p)
    assert (p_root == 0).any()  # the nucleus removes tokens
    first = com[:, 0]
    freq = np.bincount(first, minlength=V) / B
    assert np.all(freq[p_root == 0] == 0)
    assert np.abs(freq - p_root).max() < 4.5 * np.sqrt(0.25 / B)
    for ci, t in enumerate(kids):
        took = first == t
        if took.sum() < 2000:
            continue
        p_child = _nucleus(logits[1 + ci], temp, top_k, top_p)
        f2 = np.bincount(com[took, 1], minlength=V) / took.sum()
        assert np.all(f2[p_child == 0] == 0)
        assert np.abs(f2 - p_child).max() < 4.5 * np.sqrt(0.25 / took.sum())
