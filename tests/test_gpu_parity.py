"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Tree, mask and accept must match bit for bit.  Attention must satisfy
max|diff| <= 1e-2 * max|ref| and mean relative error (sum|diff| / sum|ref|)
<= 2e-3 against the fp64 oracle (bf16 inputs, fp32 accumulation and output),
over every row of every workload, the five full-size ones included; a few
extra cases at full size compare sampled rows the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
from tree_speculative_decoding_gb300 import ddt, workloads

pytestmark = pytest.mark.gpu

MAX_TOL = 1e-2
MEAN_TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tree_speculative_decoding_gb300 import _build
    _build.build()
    oracle.build()


def _step(wl, argmax=None, num_splits=0, fused=True):
    from tree_speculative_decoding_gb300.pipeline import VerifyStep
    st = VerifyStep(wl, "cuda:0", target_argmax=argmax, num_splits=num_splits,
                    fused_tree_mask=fused)
    st.run()
    torch.cuda.synchronize()
    st.check_device_errors()
    return st


def _oracle_tree(wl):
    return oracle.build_tree(wl.topk_logp, wl.topk_ids, wl.root_id, wl.budget, wl.qo_indptr,
                             wl.max_depth, wl.K)


def _sample_rows(wl, n, seed=0):
    rows_total = wl.total_q * wl.H
    if n >= rows_total:
        return np.arange(rows_total, dtype=np.int64)
    rng = np.random.default_rng(seed)
    picks = set()
    for b in range(wl.B):   # first and last node of every request, a random head
        for t in (wl.qo_indptr[b], wl.qo_indptr[b + 1] - 1):
            picks.add(int(t) * wl.H + int(rng.integers(wl.H)))
    while len(picks) < n:
        picks.add(int(rng.integers(rows_total)))
    return np.array(sorted(picks), dtype=np.int64)


def _check_attn(st, wl, mask, mip, rows):
    ref, ref_lse = oracle.verify_attn(wl.q, wl.kv_pool, wl.kv_indices, wl.kv_indptr,
                                      wl.qo_indptr, mask, mip, wl.H, wl.scale, rows=rows)
    out = st.out.reshape(-1, 512)
    got = out[torch.from_numpy(rows).to(out.device)].double().cpu().numpy()
    got_lse = st.lse.reshape(-1)[torch.from_numpy(rows).to(out.device)].double().cpu().numpy()
    diff = np.abs(got - ref)
    assert diff.max() <= MAX_TOL * np.abs(ref).max(), f"max|diff| {diff.max()}"
    assert diff.sum() / np.abs(ref).sum() <= MEAN_TOL, f"mean rel {diff.sum() / np.abs(ref).sum()}"
    np.testing.assert_allclose(got_lse, ref_lse, rtol=1e-4, atol=1e-3)
    full = st.out
    assert torch.isfinite(full).all() and torch.isfinite(st.lse).all()
    return diff.max() / np.abs(ref).max()


def _full_check(wl, n_rows, argmax=None, num_splits=0, fused=True):
    st = _step(wl, argmax=argmax, num_splits=num_splits, fused=fused)
    tok, par, dep = _oracle_tree(wl)
    np.testing.assert_array_equal(st.node_token.cpu().numpy(), tok)
    np.testing.assert_array_equal(st.parent.cpu().numpy(), par)
    np.testing.assert_array_equal(st.depth.cpu().numpy(), dep)
    mask, mip = oracle.compile_visibility(par, wl.qo_indptr, wl.prefix_len)
    np.testing.assert_array_equal(st.mask.cpu().numpy().view(np.uint32), mask)
    np.testing.assert_array_equal(st.mask_indptr_host.numpy(), mip)
    _check_attn(st, wl, mask, mip, _sample_rows(wl, n_rows))
    am = wl.argmax_random if argmax is None else argmax
    alen, acc, com, bon = oracle.accept(tok, par, wl.qo_indptr, am, wl.max_depth)
    np.testing.assert_array_equal(st.accept_len.cpu().numpy(), alen)
    np.testing.assert_array_equal(st.accepted_nodes.cpu().numpy(), acc)
    np.testing.assert_array_equal(st.commit_tokens.cpu().numpy(), com)
    np.testing.assert_array_equal(st.bonus.cpu().numpy(), bon)
    return st, (tok, par, dep)


def test_tiny_shapes_log_workload():
    _full_check(workloads.preset("tiny_p21_b8_h8"), n_rows=10 ** 9)


ALL = 10 ** 9   # every row


def test_single_request_full_heads():
    st, _ = _full_check(workloads.preset("single_p4096_b32_h64"), n_rows=ALL)
    assert st.launched_splits > 1   # the timed shape splits: the combine is covered


def test_ragged_batch():
    _full_check(workloads.preset("ragged_bs8_b32_h64"), n_rows=ALL)


def test_long_context_split_kv():
    # every one of the 4160 rows, with 1% of kv rows scaled by 8 (rescales)
    wl = workloads.preset("long_p131072_b64_h64")
    st, _ = _full_check(wl, n_rows=ALL)
    assert st.launched_splits > 1


def test_mixed_budgets_with_half_matching_targets():
    wl = workloads.preset("mixed_bs32_b16or32_h16")
    tok, par, _ = _oracle_tree(wl)
    argmax = oracle.best_child_argmax(par, wl.qo_indptr, tok, wl.argmax_coin, wl.argmax_random)
    st, _ = _full_check(wl, n_rows=ALL, argmax=argmax)
    assert st.accept_len.max().item() > 1   # the 50% matches do get accepted


def test_chain_forcing_targets_accept_deep_paths():
    wl = workloads.preset("single_p4096_b32_h64")
    tok, par, _ = _oracle_tree(wl)
    coin = np.ones(wl.total_q, np.uint8)
    argmax = oracle.best_child_argmax(par, wl.qo_indptr, tok, coin, wl.argmax_random)
    st, _ = _full_check(wl, n_rows=64, argmax=argmax)
    assert st.accept_len.item() >= 2


# requested -> launched: a split covers ceil(1506 / s) columns rounded up to
# whole 64-column tiles, and only the splits that then cover the 1506 columns
# of the longest request run
@pytest.mark.parametrize("splits,launched", [(1, 1), (2, 2), (3, 3), (7, 6), (16, 12), (24, 24)])
def test_forced_split_counts_agree(splits, launched):
    wl = workloads.make_workload("splits", 99, 2, 16, [700, 1500], [20, 5], 4, 1000, 2.0)
    st, _ = _full_check(wl, n_rows=10 ** 9, num_splits=splits)
    assert int(wl.kv_len.max()) == 1506 and st.launched_splits == launched


@pytest.mark.parametrize("H", [1, 3, 16, 17, 128])
def test_head_counts(H):
    wl = workloads.make_workload(f"h{H}", 500 + H, 2, H, [64, 33], [9, 3], 3, 200, 1.5)
    _full_check(wl, n_rows=10 ** 9)


def test_degenerate_requests_prefix0_budget0_and_max_qlen():
    # prefix 0 (the root sees only itself), budget 0 (plain autoregressive
    # verify: q_len 1) and the largest tree (budget 127, q_len 128)
    wl = workloads.make_workload("edge", 4242, 4, 8, [0, 57, 1, 300], [5, 0, 127, 31], 16, 5000,
                                 1.0)
    _full_check(wl, n_rows=10 ** 9)


@pytest.mark.parametrize("name", ["tiny_p21_b8_h8", "ragged_bs8_b32_h64", "mixed_bs32_b16or32_h16"])
def test_separate_tree_and_mask_launches(name):
    # ddt_build_tree + ddt_compile_visibility as two launches: the same
    # oracle outputs as the one-launch ddt_build_tree_visibility of the steps above
    _full_check(workloads.preset(name), n_rows=256, fused=False)


def test_fused_tree_mask_degenerate_requests():
    # both paths on prefix 0, budget 0, a prefix that is a multiple of 32 and
    # the largest tree, bit for bit against each other and the oracle
    wl = workloads.make_workload("edge2", 4243, 5, 4, [0, 64, 1, 300, 31], [5, 0, 127, 31, 2], 16,
                                 5000, 1.0)
    a, _ = _full_check(wl, n_rows=10 ** 9, fused=True)
    b, _ = _full_check(wl, n_rows=10 ** 9, fused=False)
    assert torch.equal(a.mask, b.mask) and torch.equal(a.parent, b.parent)


def _chain_forcing(wl, coin=None):
    tok, par, _ = _oracle_tree(wl)
    coin = np.ones(wl.total_q, bool) if coin is None else coin
    return oracle.best_child_argmax(par, wl.qo_indptr, tok, coin, wl.argmax_random)


def _commit_and_check(wl, argmax, full_pool):
    """Runs the step and the KV commit; checks the pool bit for bit."""
    st, _ = _full_check(wl, n_rows=64, argmax=argmax)
    alen = st.accept_len.cpu().numpy()
    acc = st.accepted_nodes.cpu().numpy()
    assert alen.max() > 1
    before = st.kv_pool.clone()
    st.commit_kv()
    torch.cuda.synchronize()
    st.check_device_errors()
    np.testing.assert_array_equal(st.new_len.cpu().numpy(), wl.prefix_len + alen)
    after = st.kv_pool.view(torch.int16)
    if full_pool:
        ref, ref_len = oracle.commit_kv(wl.kv_pool, wl.kv_indices, wl.kv_indptr, wl.qo_indptr,
                                        alen, acc, wl.max_depth)
        np.testing.assert_array_equal(after.cpu().numpy().view(np.uint16), ref)
        return
    # full size: each destination row holds its source's value from before the
    # commit, and no other row changed
    b16 = before.view(torch.int16)
    dst_all = []
    for b in range(wl.B):
        idx = wl.kv_indices[int(wl.kv_indptr[b]):int(wl.kv_indptr[b + 1])]
        P = int(wl.prefix_len[b])
        for k in range(int(alen[b])):
            d, src = int(idx[P + k]), int(idx[P + int(acc[b, k])])
            assert torch.equal(after[d], b16[src])
            dst_all.append(d)
    changed = (after != b16).any(dim=1).nonzero().flatten().cpu().numpy()
    assert set(changed.tolist()) <= set(dst_all)


@pytest.mark.parametrize("name", ["tiny_p21_b8_h8", "edge"])
def test_commit_kv_matches_oracle(name):
    if name == "edge":
        wl = workloads.make_workload("edge_commit", 4244, 5, 4, [0, 64, 1, 300, 31],
                                     [5, 0, 127, 31, 2], 16, 5000, 1.0)
    else:
        wl = workloads.preset(name)
    _commit_and_check(wl, _chain_forcing(wl), full_pool=True)
    # half-matching targets: paths stop at random depths
    coin = np.random.default_rng(7).random(wl.total_q) < 0.6
    coin[wl.qo_indptr[:-1]] = True
    _commit_and_check(wl, _chain_forcing(wl, coin), full_pool=True)


@pytest.mark.parametrize("name", ["single_p4096_b32_h64", "mixed_bs32_b16or32_h16"])
def test_commit_kv_full_size(name):
    wl = workloads.preset(name)
    _commit_and_check(wl, _chain_forcing(wl), full_pool=False)


def test_commit_kv_rejects_a_broken_path():
    from tree_speculative_decoding_gb300 import ddt
    wl = workloads.preset("tiny_p21_b8_h8")
    st = _step(wl, argmax=_chain_forcing(wl))
    before = st.kv_pool.clone()
    st.accepted_nodes[0, 1] = 0          # not increasing: made on the host, caught by the kernel
    st.commit_kv()
    torch.cuda.synchronize()
    status, bits = ddt.ddt_get_error()
    assert status == 5 and bits & 0x200
    assert torch.equal(st.kv_pool, before)


def _outputs(st):
    return [t.clone() for t in (st.node_token, st.parent, st.depth, st.mask, st.out, st.lse,
                                 st.accept_len, st.accepted_nodes, st.commit_tokens, st.bonus)]


@pytest.mark.parametrize("name", ["tiny_p21_b8_h8", "single_p4096_b32_h64", "edge"])
def test_one_call_step_and_step_graph_equal_the_staged_calls(name):
    from tree_speculative_decoding_gb300.pipeline import VerifyStep
    if name == "edge":
        wl = workloads.make_workload("edge_step", 4245, 5, 4, [0, 64, 1, 300, 31],
                                     [5, 0, 127, 31, 2], 16, 5000, 1.0)
    else:
        wl = workloads.preset(name)
    st, _ = _full_check(wl, n_rows=64)             # staged calls, checked against the oracle
    ref = _outputs(st)
    st2 = VerifyStep(wl, "cuda:0")
    st2.run_one_call()
    torch.cuda.synchronize()
    st2.check_device_errors()
    for a, b in zip(ref, _outputs(st2)):
        assert torch.equal(a, b)
    for t in (st2.node_token, st2.out, st2.accept_len):
        t.zero_()
    g = st2.step_graph()                           # captured once, replayed three times
    for _ in range(3):
        g.launch()
    torch.cuda.synchronize()
    st2.check_device_errors()
    for a, b in zip(ref, _outputs(st2)):
        assert torch.equal(a, b)
    g.close()


def test_step_graph_with_commit_equals_the_staged_commit():
    from tree_speculative_decoding_gb300.pipeline import VerifyStep
    wl = workloads.preset("tiny_p21_b8_h8")
    am = _chain_forcing(wl)
    st = _step(wl, argmax=am)
    st.commit_kv()
    torch.cuda.synchronize()
    st2 = VerifyStep(wl, "cuda:0", target_argmax=am)
    g = st2.step_graph(commit_kv=True)
    g.launch()
    torch.cuda.synchronize()
    st2.check_device_errors()
    assert torch.equal(st.kv_pool, st2.kv_pool) and torch.equal(st.new_len, st2.new_len)
    assert st.accept_len.max().item() > 1


def test_step_graph_with_host_copies_returns_the_step_in_host_memory():
    # ddt_step_graph_create_io: the inputs come from pinned host memory and the
    # results land there, equal to the staged calls' device results
    from tree_speculative_decoding_gb300.pipeline import VerifyStep
    wl = workloads.preset("tiny_p21_b8_h8")
    st, _ = _full_check(wl, n_rows=64)
    st2 = VerifyStep(wl, "cuda:0")
    h_in = st2.inputs.buf.cpu().pin_memory()
    h_out = torch.zeros_like(st2.outputs.buf, device="cpu").pin_memory()
    st2.inputs.buf.zero_()                         # the graph's own copy must bring them back
    g = st2.step_graph(host_io=(h_in, h_out))
    for _ in range(2):
        g.launch()
    torch.cuda.synchronize()
    st2.check_device_errors()
    for name in ("out", "lse", "accept_len", "accepted_nodes", "commit_tokens", "bonus"):
        v = st2.outputs.views[name]
        off = v.data_ptr() - st2.outputs.buf.data_ptr()
        got = h_out[off:off + v.numel() * v.element_size()].view(v.dtype).view(v.shape)
        assert torch.equal(got, getattr(st, name).cpu()), name
    g.close()
    with pytest.raises(ValueError):                # pageable host memory is refused
        st2.step_graph(host_io=(st2.inputs.buf.cpu(), h_out))


def test_step_graph_returns_only_the_accept_results_when_asked():
    # a host buffer of results_bytes takes the accept results alone (they lead the
    # output buffer); the attention output stays on the device
    from tree_speculative_decoding_gb300.pipeline import VerifyStep
    wl = workloads.preset("ragged_bs8_b32_h64")
    st, _ = _full_check(wl, n_rows=64)
    st2 = VerifyStep(wl, "cuda:0")
    assert st2.results_bytes == st2.outputs.offsets["out"] < st2.outputs.buf.numel()
    h_in = st2.inputs.buf.cpu().pin_memory()
    h_res = torch.full((st2.results_bytes,), 0x5A, dtype=torch.uint8).pin_memory()
    st2.inputs.buf.zero_()
    g = st2.step_graph(host_io=(h_in, h_res))
    g.launch()
    torch.cuda.synchronize()
    st2.check_device_errors()
    for name in ("accept_len", "accepted_nodes", "commit_tokens", "bonus"):
        v = st2.outputs.views[name]
        off = v.data_ptr() - st2.outputs.buf.data_ptr()
        assert off + v.numel() * v.element_size() <= st2.results_bytes
        got = h_res[off:off + v.numel() * v.element_size()].view(v.dtype).view(v.shape)
        assert torch.equal(got, getattr(st, name).cpu()), name
    assert torch.equal(st2.out, st.out)            # computed on the device all the same
    g.close()
    # a host buffer that is not whole 16-byte units takes the copy-engine path
    h_odd = torch.full((st2.results_bytes - 4,), 0x5A, dtype=torch.uint8).pin_memory()
    g = st2.step_graph(host_io=(h_in, h_odd))
    g.launch()
    torch.cuda.synchronize()
    st2.check_device_errors()
    assert torch.equal(h_odd, h_res[:st2.results_bytes - 4])
    g.close()


def test_step_graph_reports_a_host_check_and_makes_no_graph():
    from tree_speculative_decoding_gb300 import ddt
    from tree_speculative_decoding_gb300.pipeline import VerifyStep
    st = VerifyStep(workloads.preset("tiny_p21_b8_h8"), "cuda:0")
    a = st.step_args()
    a.max_depth = 8                                # unsupported: refused before any launch
    with pytest.raises(ddt.DDTError) as e:
        ddt.StepGraph(a)
    assert e.value.status == 2


@pytest.mark.parametrize("B", [256, 300])
def test_large_batches_cover_both_dispatch_orders(B):
    # up to 256 requests the kernel starts the longest first; beyond, block order
    rng = np.random.default_rng(B)
    prefix = rng.integers(0, 90, B)
    budget = rng.integers(0, 6, B)
    wl = workloads.make_workload(f"batch{B}", 7000 + B, B, 4, prefix, budget, 4, 300, 1.5)
    _full_check(wl, n_rows=600)


def test_chain_tree_equals_causal_prefill():
    wl = workloads.make_workload("chain", 77, 1, 4, [40], [7], 1, 300, 2.0)
    st, (tok, par, dep) = _full_check(wl, n_rows=10 ** 9)
    assert dep.tolist() == list(range(8))


def _causal_chunk(wl, one_call=True):
    """A prefill chunk of q_len tokens after each prefix: the tree replaced by
    the causal chain on the device, then the attention.  one_call: the whole
    chunk through ddt_prefill_step; else ddt_build_chain_visibility followed by
    the standalone ddt_verify_attn (every mask bit honoured)."""
    st = _step(wl)
    if one_call:
        st.run_prefill()
    else:
        st.build_chain_visibility()
        st.verify_attn()
    torch.cuda.synchronize()
    st.check_device_errors()
    # the chain, written on the device: parent[i] = i - 1, depth[i] = i per request
    par_ref = np.concatenate([np.arange(-1, T - 1) for T in wl.q_len]).astype(np.int32)
    dep_ref = np.concatenate([np.arange(T) for T in wl.q_len]).astype(np.int32)
    np.testing.assert_array_equal(st.parent.cpu().numpy(), par_ref)
    np.testing.assert_array_equal(st.depth.cpu().numpy(), dep_ref)
    mask, mip = oracle.compile_visibility(par_ref, wl.qo_indptr, wl.prefix_len)
    got = st.mask.cpu().numpy().view(np.uint32)
    np.testing.assert_array_equal(got, mask)
    # the chain's mask is the causal one: row i of request b sees columns [0, P_b + i]
    for b in range(wl.B):
        P, T = int(wl.prefix_len[b]), int(wl.q_len[b])
        W = (P + T + 31) // 32
        words = np.ascontiguousarray(got[mip[b]:mip[b + 1]]).astype("<u4")
        bits = np.unpackbits(words.view(np.uint8), bitorder="little").reshape(T, W * 32)
        causal = np.arange(W * 32)[None, :] <= (P + np.arange(T))[:, None]
        np.testing.assert_array_equal(bits.astype(bool), causal)
    return st, mask, mip


@pytest.mark.parametrize("one_call", [True, False])
@pytest.mark.parametrize("H", [1, 16])
def test_prefill_chunk_of_128_tokens_is_causal_attention(H, one_call):
    # q_len 128 after prefixes 300, 0 and 33 (a ragged word boundary), every row
    wl = workloads.make_workload(f"prefill{H}", 4250 + H, 3, H, [300, 0, 33], [127, 127, 60], 8,
                                 5000, 1.0)
    st, mask, mip = _causal_chunk(wl, one_call)
    _check_attn(st, wl, mask, mip, _sample_rows(wl, 10 ** 9))


def test_prefill_chunk_full_size():
    # the timed shape: 128 new tokens after a prefix of 4096, 64 heads, every row
    wl = workloads.preset("prefill_p4096_t128_h64")
    st, mask, mip = _causal_chunk(wl)
    _check_attn(st, wl, mask, mip, _sample_rows(wl, 10 ** 9))


def test_prefill_chunk_graph_replay_matches_the_direct_call():
    # the chunk is one capturable call: a CUDA graph of ddt_prefill_step replays
    # to the same bits as the direct call
    wl = workloads.make_workload("prefill_graph", 4270, 2, 8, [100, 7], [127, 40], 8, 2000, 1.0)
    st, _, _ = _causal_chunk(wl)
    ref = st.out.clone(), st.lse.clone(), st.mask.clone()
    for t in (st.out, st.lse, st.mask, st.parent, st.depth):
        t.fill_(0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            st.run_prefill(stream=s)
    torch.cuda.synchronize()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    st.check_device_errors()
    assert torch.equal(st.out, ref[0]) and torch.equal(st.lse, ref[1])
    assert torch.equal(st.mask, ref[2])


def test_chain_rejects_a_wrong_mask_range():
    # a mask_indptr that is not q_len * W words latches the mask bit; nothing faults
    wl = workloads.make_workload("chain_bad", 4280, 2, 4, [64, 10], [20, 9], 4, 300, 1.0)
    st = _step(wl)
    bad = st.mask_indptr.clone()
    bad[1] += 1
    st.mask.fill_(0x55)
    ddt.ddt_build_chain_visibility(st.qo_indptr, st.prefix_len, bad, st.parent, st.depth, st.mask)
    torch.cuda.synchronize()
    status, bits = ddt.ddt_get_error()
    assert status != 0 and bits & 0x8
    assert bool((st.mask == 0x55).all())  # neither request's mask range was written


def test_autoregressive_steps_budget_zero():
    # budget 0 everywhere: q_len 1, the plain decode step; the timed single
    # request at 64 heads, then a ragged batch of 64 at 8 heads
    st, (tok, par, dep) = _full_check(workloads.preset("ar_p4096_b0_h64"), n_rows=10 ** 9)
    assert st.accept_len.item() == 1 and par.tolist() == [-1]
    rng = np.random.default_rng(5)
    wl = workloads.make_workload("ar64", 4260, 64, 8, rng.integers(0, 3000, 64), np.zeros(64, int),
                                 4, 1000, 1.0)
    st, _ = _full_check(wl, n_rows=10 ** 9)
    assert (st.accept_len.cpu().numpy() == 1).all()


def test_cuda_graph_capture_and_replay():
    from tree_speculative_decoding_gb300.pipeline import VerifyStep
    wl = workloads.make_workload("graph", 31, 3, 16, [500, 20, 1100], [16, 9, 32], 8, 3000, 2.0)
    st = VerifyStep(wl, "cuda:0")
    st.run()
    torch.cuda.synchronize()
    ref_out = st.out.clone()
    ref_tok = st.node_token.clone()
    st.out.zero_()
    st.node_token.fill_(-9)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            st.run(stream=s)
    g.replay()
    torch.cuda.synchronize()
    st.check_device_errors()
    assert torch.equal(st.node_token, ref_tok)
    assert torch.equal(st.out, ref_out)


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    # failure detection without a fault: a kernel waits on a barrier nothing
    # arrives on; its bounded wait gives up, latches the timeout bit and exits
    from tree_speculative_decoding_gb300 import ddt
    assert ddt.ddt_get_error() == (0, 0)
    ddt.ddt_selftest_wait_timeout(1 << 12)
    torch.cuda.synchronize()
    status, bits = ddt.ddt_get_error()
    assert status == 6 and bits == 0x100
    assert ddt.ddt_get_error() == (0, 0)     # cleared
    # the context still runs a verify step, and correctly
    _full_check(workloads.preset("tiny_p21_b8_h8"), n_rows=10 ** 9)


def test_out_of_range_kv_index_is_latched_not_faulted():
    from tree_speculative_decoding_gb300 import ddt
    from tree_speculative_decoding_gb300.pipeline import VerifyStep
    wl = workloads.make_workload("bad", 5, 1, 8, [100], [4], 2, 100, 1.0)
    st = VerifyStep(wl, "cuda:0")
    st.kv_indices[7] = wl.pool_rows + 1000   # made on the host, caught by the kernel's check
    st.run()
    torch.cuda.synchronize()
    status, bits = ddt.ddt_get_error()
    assert status == 5 and bits & 0x4
    assert ddt.ddt_get_error() == (0, 0)     # cleared


def test_wrong_mask_stride_is_rejected():
    # the 30-column mask bug: a mask laid out with stride kv_len_max (prefix
    # only) instead of prefix + q_len must not be consumed silently
    from tree_speculative_decoding_gb300 import ddt
    from tree_speculative_decoding_gb300.pipeline import VerifyStep
    wl = workloads.make_workload("stride", 6, 1, 8, [21], [8], 4, 512, 2.0)
    st = VerifyStep(wl, "cuda:0")
    st.run()
    torch.cuda.synchronize()
    st.check_device_errors()
    T, P = 9, 21
    bad = torch.tensor([0, T * ((P + 31) // 32 + 1)], dtype=torch.int32, device="cuda:0")
    ddt.ddt_verify_attn(st.q, st.kv_pool, st.kv_indices, st.kv_indptr, st.qo_indptr, st.mask,
                        bad, wl.scale, st.out, st.lse, max_q_len=9, max_kv_len=30)
    torch.cuda.synchronize()
    status, bits = ddt.ddt_get_error()
    assert status == 5 and bits & 0x8


def _custom_mask_case(splits):
    """A visibility mask that is not a tree mask: every bit counts."""
    wl = workloads.make_workload("custom_mask", 909, 2, 8, [130, 61], [12, 20], 4, 3000, 2.0)
    st = _step(wl, num_splits=splits)
    tok, par, _ = _oracle_tree(wl)
    mask, mip = oracle.compile_visibility(par, wl.qo_indptr, wl.prefix_len)
    mask = mask.copy()

    def flip(b, i, c, on):
        W = (int(wl.kv_len[b]) + 31) // 32
        w = int(mip[b]) + i * W + c // 32
        if on:
            mask[w] |= np.uint32(1 << (c % 32))
        else:
            mask[w] &= np.uint32(~(1 << (c % 32)) & 0xFFFFFFFF)

    P0, P1 = int(wl.prefix_len[0]), int(wl.prefix_len[1])
    flip(0, 3, 5, False)          # a hidden prefix column
    for c in range(64, 128):      # a whole 64-column block of prefix hidden for node 4
        flip(0, 4, c, False)
    flip(0, 1, P0 + 7, True)      # a column after the row's own node made visible
    flip(1, 2, P1 + 19, True)     # the last tree column seen from an early node
    flip(1, 0, 0, False)          # the root of request 1 loses prefix column 0
    W1 = (int(wl.kv_len[1]) + 31) // 32
    row = int(mip[1]) + 5 * W1    # node 5 of request 1 sees nothing at all
    mask[row:row + W1] = 0
    return wl, st, mask, mip


@pytest.mark.parametrize("splits", [1, 3])
def test_verify_attn_honours_every_mask_bit(splits):
    # ddt_verify_attn takes any bit pattern: hidden prefix columns (one alone,
    # a whole block), visible columns after a row's own node, and a row that
    # sees nothing (out 0, lse -inf) all match the oracle, which honours every bit
    from tree_speculative_decoding_gb300 import ddt
    wl, st, mask, mip = _custom_mask_case(splits)
    dmask = torch.from_numpy(mask.view(np.int32)).to("cuda:0")
    out = torch.full_like(st.out, float("nan"))
    lse = torch.full_like(st.lse, float("nan"))
    ddt.ddt_verify_attn(st.q, st.kv_pool, st.kv_indices, st.kv_indptr, st.qo_indptr, dmask,
                        st.mask_indptr, wl.scale, out, lse, max_q_len=st.max_q_len,
                        max_kv_len=st.max_kv_len, num_splits=splits, workspace=st.workspace)
    torch.cuda.synchronize()
    assert ddt.ddt_get_error() == (0, 0)
    ref, ref_lse = oracle.verify_attn(wl.q, wl.kv_pool, wl.kv_indices, wl.kv_indptr,
                                      wl.qo_indptr, mask, mip, wl.H, wl.scale)
    got = out.reshape(-1, 512).double().cpu().numpy()
    got_lse = lse.reshape(-1).double().cpu().numpy()
    empty = np.isneginf(ref_lse)
    assert empty.sum() == wl.H                     # node 5 of request 1, every head
    assert np.array_equal(np.isneginf(got_lse), empty) and (got[empty] == 0).all()
    diff = np.abs(got - ref)
    assert diff.max() <= MAX_TOL * np.abs(ref).max()
    assert diff.sum() / np.abs(ref).sum() <= MEAN_TOL
    np.testing.assert_allclose(got_lse[~empty], ref_lse[~empty], rtol=1e-4, atol=1e-3)
    # the same step's own tree mask gives different rows where bits were flipped
    assert not np.allclose(got, st.out.reshape(-1, 512).double().cpu().numpy())


@pytest.mark.parametrize("splits", [1, 2])
def test_verify_attn_takes_a_random_mask(splits):
    # every bit of a ragged batch's mask drawn at random (70% set), so that almost
    # every 64-column block, prefix blocks included, takes the per-column select;
    # every row against the oracle, which honours every bit
    from tree_speculative_decoding_gb300 import ddt
    wl = workloads.make_workload("random_mask", 919, 3, 8, [300, 17, 129], [40, 127, 5], 8, 4000, 2.0)
    st = _step(wl, num_splits=splits)
    rng = np.random.default_rng(919)
    mask = np.zeros(int(st.mask_indptr_host[-1]), np.uint32)
    for b in range(wl.B):
        T, N = int(wl.q_len[b]), int(wl.kv_len[b])
        W = (N + 31) // 32
        bits = rng.random((T, W * 32)) < 0.7
        bits[:, N:] = False                       # padding bits stay zero
        words = np.packbits(bits.astype(np.uint8), axis=1, bitorder="little").view("<u4")
        m0 = int(st.mask_indptr_host[b])
        mask[m0:m0 + T * W] = words.reshape(-1)
    dmask = torch.from_numpy(mask.view(np.int32)).to("cuda:0")
    out = torch.full_like(st.out, float("nan"))
    lse = torch.full_like(st.lse, float("nan"))
    ddt.ddt_verify_attn(st.q, st.kv_pool, st.kv_indices, st.kv_indptr, st.qo_indptr, dmask,
                        st.mask_indptr, wl.scale, out, lse, max_q_len=st.max_q_len,
                        max_kv_len=st.max_kv_len, num_splits=splits, workspace=st.workspace)
    torch.cuda.synchronize()
    assert ddt.ddt_get_error() == (0, 0)
    assert st.launched_splits == splits
    ref, ref_lse = oracle.verify_attn(wl.q, wl.kv_pool, wl.kv_indices, wl.kv_indptr,
                                      wl.qo_indptr, mask, st.mask_indptr_host.numpy(), wl.H, wl.scale)
    got = out.reshape(-1, 512).double().cpu().numpy()
    diff = np.abs(got - ref)
    assert diff.max() <= MAX_TOL * np.abs(ref).max()
    assert diff.sum() / np.abs(ref).sum() <= MEAN_TOL
    np.testing.assert_allclose(lse.reshape(-1).double().cpu().numpy(), ref_lse, rtol=1e-4, atol=1e-3)


def test_prefill_chunk_with_forced_splits():
    # ddt_prefill_step through the split path (partials + combine), every row
    from tree_speculative_decoding_gb300.pipeline import VerifyStep
    wl = workloads.make_workload("prefill_split", 4290, 2, 8, [700, 250], [127, 90], 8, 4000, 1.0)
    st = VerifyStep(wl, "cuda:0", num_splits=3)
    assert st.launched_splits == 3
    st.run_prefill()
    torch.cuda.synchronize()
    st.check_device_errors()
    par = np.concatenate([np.arange(-1, T - 1) for T in wl.q_len]).astype(np.int32)
    mask, mip = oracle.compile_visibility(par, wl.qo_indptr, wl.prefix_len)
    assert np.array_equal(st.mask.cpu().numpy().view(np.uint32), mask)
    _check_attn(st, wl, mask, mip, _sample_rows(wl, 10 ** 9))


def test_step_graph_with_host_copies_and_commit():
    # the host-copy graph with the KV commit: the results in host memory and the
    # pool on the device equal the staged calls'
    from tree_speculative_decoding_gb300.pipeline import VerifyStep
    wl = workloads.preset("tiny_p21_b8_h8")
    am = _chain_forcing(wl)
    st = _step(wl, argmax=am)
    st.commit_kv()
    torch.cuda.synchronize()
    st2 = VerifyStep(wl, "cuda:0", target_argmax=am)
    h_in = st2.inputs.buf.cpu().pin_memory()
    h_out = torch.zeros_like(st2.outputs.buf, device="cpu").pin_memory()
    g = st2.step_graph(commit_kv=True, host_io=(h_in, h_out))
    g.launch()
    torch.cuda.synchronize()
    st2.check_device_errors()
    assert torch.equal(st.kv_pool, st2.kv_pool)
    for name in ("accept_len", "accepted_nodes", "commit_tokens", "bonus", "new_len"):
        v = st2.outputs.views[name]
        off = v.data_ptr() - st2.outputs.buf.data_ptr()
        got = h_out[off:off + v.numel() * v.element_size()].view(v.dtype).view(v.shape)
        assert torch.equal(got, getattr(st, name).cpu()), name
    assert st.accept_len.max().item() > 1
    g.close()


def test_inconsistent_offsets_are_latched_and_nothing_is_written():
    # qo_indptr past total_q, a negative qo_indptr and a negative mask_indptr,
    # each made on the host: the attention latches the bit and writes no row
    from tree_speculative_decoding_gb300 import ddt
    wl = workloads.make_workload("offsets", 31, 2, 8, [40, 70], [6, 9], 4, 500, 2.0)
    st = _step(wl, num_splits=1)
    cases = [("qo", torch.tensor([0, 7, st.total_q + 9], dtype=torch.int32), 0x1),
             ("qo", torch.tensor([-3, 7, st.total_q], dtype=torch.int32), 0x1),
             ("mask", torch.tensor([-1, st.mask_indptr_host[1].item(), st.mask_indptr_host[2].item()],
                                   dtype=torch.int32), 0x8)]
    for which, bad, bit in cases:
        qo = bad.to("cuda:0") if which == "qo" else st.qo_indptr
        mip = bad.to("cuda:0") if which == "mask" else st.mask_indptr
        out = torch.full_like(st.out, 7.0)
        ddt.ddt_verify_attn(st.q, st.kv_pool, st.kv_indices, st.kv_indptr, qo, st.mask, mip,
                            wl.scale, out, None, max_q_len=st.max_q_len, max_kv_len=st.max_kv_len,
                            num_splits=1)
        torch.cuda.synchronize()
        status, bits = ddt.ddt_get_error()
        assert status == 5 and bits & bit, (which, hex(bits))
        # request 0's rows: untouched when its own offsets are the bad ones
        if which == "mask" or bad[0] < 0:
            assert bool((out[:7] == 7.0).all())
    assert ddt.ddt_get_error() == (0, 0)


def test_bad_budget_indptr_is_latched():
    from tree_speculative_decoding_gb300 import ddt
    from tree_speculative_decoding_gb300.pipeline import VerifyStep
    wl = workloads.make_workload("budget", 8, 2, 4, [10, 10], [3, 3], 2, 50, 1.0)
    st = VerifyStep(wl, "cuda:0")
    st.budget[1] = 4                         # disagrees with qo_indptr
    st.build_tree()
    torch.cuda.synchronize()
    status, bits = ddt.ddt_get_error()
    assert status == 5 and bits & 0x1
    st.build_tree_visibility()               # the one-launch tree + mask checks the same
    torch.cuda.synchronize()
    status, bits = ddt.ddt_get_error()
    assert status == 5 and bits & 0x1
    assert ddt.ddt_get_error() == (0, 0)


# ---------------------------------------------------------------- sampling accept

def _links(st):
    from tree_speculative_decoding_gb300 import ddt
    T = st.node_token.numel()
    fc, ns, ri = (torch.empty(T, dtype=torch.int32, device="cuda:0") for _ in range(3))
    ddt.ddt_tree_links(st.parent, st.qo_indptr, fc, ns, ri)
    return fc, ns, ri


def _sampled(st, logits, temp, top_k, coins, top_p=None):
    from tree_speculative_decoding_gb300 import ddt
    fc, ns, _ = _links(st)
    B, W = st.accepted_nodes.shape
    out = [torch.empty(B, dtype=torch.int32, device="cuda:0"),
           torch.empty((B, W), dtype=torch.int32, device="cuda:0"),
           torch.empty((B, W), dtype=torch.int32, device="cuda:0"),
           torch.empty(B, dtype=torch.int32, device="cuda:0")]
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dt)).to("cuda:0")  # noqa: E731
    ddt.ddt_accept_sampled(st.node_token, fc, ns, st.qo_indptr, dev(logits, np.float32),
                           dev(temp, np.float32), dev(top_k, np.int32), dev(coins, np.float32),
                           st.wl.max_depth, *out,
                           top_p=None if top_p is None else dev(top_p, np.float32))
    torch.cuda.synchronize()
    st.check_device_errors()
    return [t.cpu().numpy() for t in out]


@pytest.mark.parametrize("name", ["tiny_p21_b8_h8", "mixed_bs32_b16or32_h16", "edge"])
def test_tree_links_match_oracle(name):
    if name == "edge":
        wl = workloads.make_workload("edge_links", 4246, 5, 4, [0, 64, 1, 300, 31],
                                     [5, 0, 127, 31, 2], 16, 5000, 1.0)
    else:
        wl = workloads.preset(name)
    st = _step(wl)
    fc, ns, ri = _links(st)
    torch.cuda.synchronize()
    st.check_device_errors()
    ref = oracle.tree_links(st.parent.cpu().numpy(), wl.qo_indptr)
    for g, r in zip((fc, ns, ri), ref):
        np.testing.assert_array_equal(g.cpu().numpy(), r)


def _sampling_case(wl, vocab, seed, chain_bias):
    # target logits whose argmax sits on a child token at most nodes, so that
    # walks go deep, plus uniform coins
    st = _step(wl)
    tok = st.node_token.cpu().numpy()
    par = st.parent.cpu().numpy()
    rng = np.random.default_rng(seed)
    logits = rng.normal(scale=1.5, size=(wl.total_q, vocab)).astype(np.float32)
    for b in range(wl.B):
        lo, hi = int(wl.qo_indptr[b]), int(wl.qo_indptr[b + 1])
        for n in range(lo, hi):
            kids = [c for c in range(n + 1, hi) if lo + par[c] == n]
            if kids:
                logits[n, tok[kids[0]] % vocab] += chain_bias
    coins = rng.random((wl.total_q, wl.K + 1)).astype(np.float32)
    return st, tok, par, logits, coins


@pytest.mark.parametrize("name,vocab", [("tiny_p21_b8_h8", 512), ("mixed_bs32_b16or32_h16", 32768)])
def test_sampled_accept_at_temperature_zero_is_greedy(name, vocab):
    wl = workloads.preset(name)
    st, tok, par, logits, coins = _sampling_case(wl, vocab, 5, 12.0)
    got = _sampled(st, logits, np.zeros(wl.B), np.full(wl.B, 50), coins)
    ref = oracle.accept(tok, par, wl.qo_indptr, logits.argmax(axis=1).astype(np.int32),
                        wl.max_depth)
    for g, r in zip(got, ref):
        np.testing.assert_array_equal(g, r)
    assert got[0].max() > 1


@pytest.mark.parametrize("name,vocab,temp,top_k,bias", [
    ("tiny_p21_b8_h8", 512, 0.8, 0, 10.0),
    ("mixed_bs32_b16or32_h16", 32768, 1.0, 0, 11.5),
    ("mixed_bs32_b16or32_h16", 32768, 0.7, 20, 7.0),
    # vocabularies that are not a multiple of 4: rows off the 16-byte grid
    # (scalar loads) and row tails, with and without top-k
    ("tiny_p21_b8_h8", 1001, 0.9, 0, 10.0),
    ("tiny_p21_b8_h8", 1001, 0.9, 5, 8.0),
    ("mixed_bs32_b16or32_h16", 20002, 1.0, 0, 11.5),
    ("mixed_bs32_b16or32_h16", 20002, 0.8, 12, 7.0),
])
def test_sampled_accept_matches_oracle(name, vocab, temp, top_k, bias):
    # probabilities are fp32 on the device and fp64 in the oracle: the seeds are
    # chosen with no coin within fp32 rounding of a threshold, so the decisions
    # (integers) must agree exactly
    wl = workloads.preset(name)
    st, tok, par, logits, coins = _sampling_case(wl, vocab, 11, bias)
    t = np.full(wl.B, temp)
    k = np.full(wl.B, top_k)
    got = _sampled(st, logits, t, k, coins)
    ref = oracle.accept_sampled(tok, par, wl.qo_indptr, logits, t, k, coins, wl.max_depth)
    for g, r in zip(got, ref):
        np.testing.assert_array_equal(g, r)
    assert got[0].max() > 1


def test_sampled_accept_emits_the_target_distribution():
    # 4096 copies of one root with three leaf children (tokens 2, 5, 0) over a
    # vocabulary of 8; the device's first emitted token must follow p(root)
    from tree_speculative_decoding_gb300 import ddt
    B, V, temp = 4096, 8, 0.9
    rng = np.random.default_rng(3)
    l = rng.normal(scale=1.2, size=V).astype(np.float32)
    p = np.exp((l - l.max()) / temp)
    p /= p.sum()
    T = 4
    par = np.tile(np.array([-1, 0, 0, 0], np.int32), B)
    tok = np.tile(np.array([9, 2, 5, 0], np.int32), B)
    qo = np.arange(B + 1, dtype=np.int32) * T
    fc = np.tile(np.array([1, -1, -1, -1], np.int32), B)
    ns = np.tile(np.array([-1, 2, 3, -1], np.int32), B)
    logits = np.tile(l, (B * T, 1))
    coins = rng.random((B * T, 4)).astype(np.float32)
    d = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dt)).to("cuda:0")  # noqa: E731
    out = [torch.empty(B, dtype=torch.int32, device="cuda:0"),
           torch.empty((B, 3), dtype=torch.int32, device="cuda:0"),
           torch.empty((B, 3), dtype=torch.int32, device="cuda:0"),
           torch.empty(B, dtype=torch.int32, device="cuda:0")]
    ddt.ddt_accept_sampled(d(tok, np.int32), d(fc, np.int32), d(ns, np.int32), d(qo, np.int32),
                           d(logits, np.float32), d(np.full(B, temp), np.float32),
                           d(np.zeros(B), np.int32), d(coins, np.float32), 2, *out)
    torch.cuda.synchronize()
    assert ddt.ddt_get_error() == (0, 0)
    first = out[2][:, 0].cpu().numpy()
    freq = np.bincount(first, minlength=V) / B
    assert np.abs(freq - p).max() < 4.5 * np.sqrt(0.25 / B)



@pytest.mark.parametrize("top_k", [0, 64])
def test_sampled_accept_at_the_largest_vocabulary(top_k):
    # vocab 262144 (the ABI's bound), a sharp temperature: each warp's segment
    # spans 64 steps of 256 ids.  The seed is one whose decisions do not move
    # when every coin moves by 3e-5, so fp32 and fp64 must agree.
    wl = workloads.preset("tiny_p21_b8_h8")
    st, tok, par, logits, coins = _sampling_case(wl, 262144, 16, 8.0)
    t = np.full(wl.B, 0.35)
    k = np.full(wl.B, top_k)
    got = _sampled(st, logits, t, k, coins)
    ref = oracle.accept_sampled(tok, par, wl.qo_indptr, logits, t, k, coins, wl.max_depth)
    for g, r in zip(got, ref):
        np.testing.assert_array_equal(g, r)
    assert got[0].max() > 1


def test_sampled_accept_residual_draw_over_many_steps():
    # 4096 copies of one root with three leaf children whose tokens sit in
    # different 256-id steps of a 4096-id vocabulary; the first emitted token
    # must follow p(root), checked per step and on the five likeliest tokens
    from tree_speculative_decoding_gb300 import ddt
    B, V, temp = 4096, 4096, 0.8
    rng = np.random.default_rng(21)
    l = rng.normal(scale=1.0, size=V).astype(np.float32)
    l[rng.choice(V, 24, replace=False)] += 4.0          # some mass in a few tokens
    kids = np.array([100, 1500, 3900], np.int32)
    l[kids] += 3.0
    p = np.exp((l.astype(np.float64) - l.max()) / temp)
    p /= p.sum()
    par = np.tile(np.array([-1, 0, 0, 0], np.int32), B)
    tok = np.tile(np.concatenate([[7], kids]).astype(np.int32), B)
    qo = np.arange(B + 1, dtype=np.int32) * 4
    fc = np.tile(np.array([1, -1, -1, -1], np.int32), B)
    ns = np.tile(np.array([-1, 2, 3, -1], np.int32), B)
    logits = np.tile(l, (B * 4, 1))
    coins = rng.random((B * 4, 4)).astype(np.float32)
    d = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dt)).to("cuda:0")  # noqa: E731
    out = [torch.empty(B, dtype=torch.int32, device="cuda:0"),
           torch.empty((B, 3), dtype=torch.int32, device="cuda:0"),
           torch.empty((B, 3), dtype=torch.int32, device="cuda:0"),
           torch.empty(B, dtype=torch.int32, device="cuda:0")]
    ddt.ddt_accept_sampled(d(tok, np.int32), d(fc, np.int32), d(ns, np.int32), d(qo, np.int32),
                           d(logits, np.float32), d(np.full(B, temp), np.float32),
                           d(np.zeros(B), np.int32), d(coins, np.float32), 2, *out)
    torch.cuda.synchronize()
    assert ddt.ddt_get_error() == (0, 0)
    first = out[2][:, 0].cpu().numpy()
    freq = np.bincount(first, minlength=V) / B
    f_step, p_step = freq.reshape(16, 256).sum(1), p.reshape(16, 256).sum(1)
    assert np.all(np.abs(f_step - p_step) < 4.5 * np.sqrt(p_step * (1 - p_step) / B) + 1e-3)
    top = np.argsort(p)[::-1][:5]
    assert np.all(np.abs(freq[top] - p[top]) < 4.5 * np.sqrt(p[top] * (1 - p[top]) / B) + 1e-3)


@pytest.mark.parametrize("name,vocab,temp,top_k,top_p,bias,seed", [
    ("tiny_p21_b8_h8", 512, 0.8, 0, 0.9, 6.0, 12),
    ("mixed_bs32_b16or32_h16", 32768, 0.5, 0, 0.6, 6.0, 11),
    ("mixed_bs32_b16or32_h16", 32768, 0.7, 20, 0.7, 5.0, 11),
    ("tiny_p21_b8_h8", 1001, 0.9, 5, 0.5, 3.0, 48),
    ("tiny_p21_b8_h8", 1001, 0.6, 0, 0.75, 4.0, 27),
    ("mixed_bs32_b16or32_h16", 20002, 0.5, 12, 0.8, 5.0, 11),
    ("tiny_p21_b8_h8", 262144, 0.35, 0, 0.8, 8.0, 12),
    ("tiny_p21_b8_h8", 262144, 0.35, 64, 0.7, 6.0, 35),
])
def test_sampled_accept_top_p_matches_oracle(name, vocab, temp, top_k, top_p, bias, seed):
    # the kept set is an integer decision taken from a sum of exponentials (fp64
    # in the oracle, 2^-40 fixed point over fp32 exponentials on the device): the
    # seeds are ones whose oracle decisions do not move when top_p moves by
    # +-3e-6 or every coin by +-3e-5, so both sides must decide alike.  In every
    # case a walk goes past the root and top-p changes some request's outcome.
    wl = workloads.preset(name)
    st, tok, par, logits, coins = _sampling_case(wl, vocab, seed, bias)
    t, k, tp = np.full(wl.B, temp), np.full(wl.B, top_k), np.full(wl.B, top_p, np.float32)
    ref = oracle.accept_sampled(tok, par, wl.qo_indptr, logits, t, k, coins, wl.max_depth,
                                top_p=tp)
    for moved in ([tp - np.float32(3e-6), coins], [tp + np.float32(3e-6), coins],
                  [tp, np.clip(coins - 3e-5, 0, 0.99999)], [tp, np.clip(coins + 3e-5, 0, 0.99999)]):
        r = oracle.accept_sampled(tok, par, wl.qo_indptr, logits, t, k, moved[1], wl.max_depth,
                                  top_p=moved[0])
        for a, b in zip(r, ref):
            np.testing.assert_array_equal(a, b)
    plain = oracle.accept_sampled(tok, par, wl.qo_indptr, logits, t, k, coins, wl.max_depth)
    assert ref[0].max() > 1
    assert (ref[0] != plain[0]).any() or (ref[3] != plain[3]).any()
    got = _sampled(st, logits, t, k, coins, top_p=tp)
    for g, r in zip(got, ref):
        np.testing.assert_array_equal(g, r)
    # top_p 1 (no filter) on the device is the plain sampling accept
    got1 = _sampled(st, logits, t, k, coins, top_p=np.ones(wl.B, np.float32))
    got0 = _sampled(st, logits, t, k, coins)
    for a, b in zip(got1, got0):
        np.testing.assert_array_equal(a, b)


def test_sampled_accept_top_p_emits_the_nucleus():
    # 4096 copies of one root with three leaf children over a vocabulary of 16;
    # the device's first emitted token must follow the nucleus of p(root) and
    # never be a token outside it
    from tree_speculative_decoding_gb300 import ddt
    B, V, temp, top_p = 4096, 16, 0.9, 0.75
    rng = np.random.default_rng(8)
    l = rng.normal(scale=1.3, size=V).astype(np.float32)
    p = np.exp((l.astype(np.float64) - l.max()) / temp)
    p /= p.sum()
    order = np.argsort(-l)
    csum = np.cumsum(p[order])
    keep = order[:int(np.searchsorted(csum, top_p)) + 1]     # distinct logits: no ties
    q = np.zeros(V)
    q[keep] = p[keep] / p[keep].sum()
    assert 2 < len(keep) < V
    T = 4
    par = np.tile(np.array([-1, 0, 0, 0], np.int32), B)
    kids = [int(order[0]), int(order[len(keep)]), int(order[1])]  # one outside the nucleus
    tok = np.tile(np.array([9] + kids, np.int32), B)
    qo = np.arange(B + 1, dtype=np.int32) * T
    fc = np.tile(np.array([1, -1, -1, -1], np.int32), B)
    ns = np.tile(np.array([-1, 2, 3, -1], np.int32), B)
    logits = np.tile(l, (B * T, 1))
    coins = rng.random((B * T, 4)).astype(np.float32)
    d = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dt)).to("cuda:0")  # noqa: E731
    out = [torch.empty(B, dtype=torch.int32, device="cuda:0"),
           torch.empty((B, 3), dtype=torch.int32, device="cuda:0"),
           torch.empty((B, 3), dtype=torch.int32, device="cuda:0"),
           torch.empty(B, dtype=torch.int32, device="cuda:0")]
    ddt.ddt_accept_sampled(d(tok, np.int32), d(fc, np.int32), d(ns, np.int32), d(qo, np.int32),
                           d(logits, np.float32), d(np.full(B, temp), np.float32),
                           d(np.zeros(B), np.int32), d(coins, np.float32), 2, *out,
                           top_p=d(np.full(B, top_p), np.float32))
    torch.cuda.synchronize()
    assert ddt.ddt_get_error() == (0, 0)
    first = out[2][:, 0].cpu().numpy()
    freq = np.bincount(first, minlength=V) / B
    assert np.all(freq[q == 0] == 0)
    assert np.abs(freq - q).max() < 4.5 * np.sqrt(0.25 / B)


def test_sampled_accept_latches_too_few_coins():
    # a root with three children but coins for two: a device check, no fault
    from tree_speculative_decoding_gb300 import ddt
    d = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dt)).to("cuda:0")  # noqa: E731
    out = [torch.full((1,), -7, dtype=torch.int32, device="cuda:0"),
           torch.empty((1, 3), dtype=torch.int32, device="cuda:0"),
           torch.empty((1, 3), dtype=torch.int32, device="cuda:0"),
           torch.empty(1, dtype=torch.int32, device="cuda:0")]
    assert ddt.ddt_get_error() == (0, 0)
    ddt.ddt_accept_sampled(d([0, 1, 2, 3], np.int32), d([1, -1, -1, -1], np.int32),
                           d([-1, 2, 3, -1], np.int32), d([0, 4], np.int32),
                           d(np.zeros((4, 16)), np.float32), d([1.0], np.float32),
                           d([0], np.int32), d(np.full((4, 3), 0.5), np.float32), 2, *out)
    torch.cuda.synchronize()
    assert ddt.ddt_get_error() == (5, 0x400)
    assert out[0].item() == -7                            # outputs left unset
