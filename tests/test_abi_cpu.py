"""The C ABI library without a GPU: it loads, exports every declared entry
point, and its host-side logic (mask layout, workspace sizing, argument
checks) behaves as documented.  No call here reaches a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ddt.h")


@pytest.fixture(scope="module")
def lib():
    from tree_speculative_decoding_gb300 import _build
    _build.build()
    from tree_speculative_decoding_gb300 import ddt
    return ddt.lib


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ddt_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    out = os.popen(f"nm -D --defined-only {lib._name}").read()
    exported = set(re.findall(r" T (ddt_\w+)", out))
    assert set(names) <= exported


def test_abi_version_and_status_strings(lib):
    assert lib.ddt_abi_version() == 3
    assert lib.ddt_status_string(0) == b"ok"
    assert b"workspace" in lib.ddt_status_string(3)


def test_mask_indptr_matches_oracle(lib, oracle_mod):
    from tree_speculative_decoding_gb300 import ddt
    import torch
    rng = np.random.default_rng(3)
    for _ in range(20):
        B = int(rng.integers(1, 40))
        T = rng.integers(1, 129, B)
        P = rng.integers(0, 20000, B)
        qo = np.concatenate([[0], np.cumsum(T)]).astype(np.int32)
        got = ddt.ddt_mask_indptr(torch.from_numpy(qo), torch.from_numpy(P.astype(np.int32)))
        ref = oracle_mod.mask_indptr(qo, P.astype(np.int32))
        assert got.numpy().tolist() == ref.tolist()


def test_mask_indptr_rejects_bad_sizes(lib):
    qo = (ctypes.c_int32 * 3)(0, 5, 5)          # second request has q_len 0
    pl = (ctypes.c_int32 * 2)(3, 4)
    out = (ctypes.c_int32 * 3)()
    assert lib.ddt_mask_indptr(qo, pl, 2, out) == 1
    assert lib.ddt_mask_indptr(None, pl, 2, out) == 1


def test_workspace_size_formula(lib):
    assert lib.ddt_verify_attn_workspace_size(33, 64, 1) == 0
    rows = 33 * 64
    a = (rows * 4 * 512 * 4 + 255) // 256 * 256
    b = (rows * 4 * 4 + 255) // 256 * 256
    assert lib.ddt_verify_attn_workspace_size(33, 64, 4) == a + b


def test_launched_splits_follow_the_tile_rounding(lib):
    # a split covers ceil(N / s) columns rounded up to whole 64-column tiles;
    # the splits launched are those that then cover N (no empty tail split)
    for N in (30, 64, 65, 309, 1520, 4129, 131137):
        for s in (1, 2, 3, 4, 7, 9, 16, 128):
            cols = -(-N // s)
            cols = -(-cols // 64) * 64
            assert lib.ddt_verify_attn_launched_splits(N, s) == -(-N // cols), (N, s)
    assert lib.ddt_verify_attn_launched_splits(1520, 7) == 6
    assert lib.ddt_verify_attn_launched_splits(1520, 16) == 12
    assert lib.ddt_verify_attn_launched_splits(30, 2) == 1      # one tile: nothing to split
    assert lib.ddt_verify_attn_launched_splits(309, 2) == 2
    assert lib.ddt_verify_attn_launched_splits(100, 0) == 1     # out of range: one split


def test_num_splits_is_bounded(lib):
    for B, H, T, N in [(1, 64, 33, 4129), (8, 64, 33, 16417), (1, 8, 9, 30), (1, 64, 65, 131137),
                       (32, 16, 33, 8225)]:
        s = lib.ddt_verify_attn_num_splits(B, H, T, N, 148)
        assert 1 <= s <= 128
        assert s == 1 or N // s >= 64


def _wave_model(B, H, T, N, sms):
    """The split choice as documented: one split for a batch that fills half the
    SMs with row tiles; else the count (>= 4 kv blocks of 64 per split) with the
    fewest waves x (blocks per split + 8), ties to fewer splits."""
    tiles = B * -(-(T * H) // 128)
    pairs = max(sms // 2, 1)
    if B > 1 and tiles >= pairs:
        return 1
    blocks = -(-N // 64)
    best, best_cost = 1, None
    smax = (blocks - 1) // 3 if blocks >= 4 else 1   # ceil(blocks / s) >= 4
    for s in range(1, max(1, min(smax, 128)) + 1):
        cost = -(-(tiles * s) // pairs) * (-(-blocks // s) + 8)
        if best_cost is None or cost < best_cost:
            best, best_cost = s, cost
    return best


def test_split_choice_for_the_timed_shapes(lib):
    # (batch, heads, max q_len, max kv_len) -> splits on 152 SMs
    cases = {(1, 64, 33, 4129): 4,        # one request, prefix 4096, budget 32
             (1, 64, 65, 131137): 9,      # long context
             (8, 64, 33, 16417): 1,       # ragged batch: the row tiles fill the SMs
             (32, 16, 33, 8225): 1,       # mixed batch of 32
             (1, 64, 1, 4097): 17,        # autoregressive step: 4 blocks per split
             (1, 64, 128, 4224): 1}       # prefill chunk of 128 tokens
    for (B, H, T, N), want in cases.items():
        assert lib.ddt_verify_attn_num_splits(B, H, T, N, 152) == want, (B, H, T, N)


def test_split_choice_follows_the_wave_model(lib):
    rng = __import__("numpy").random.default_rng(0)
    for _ in range(300):
        B = int(rng.choice([1, 1, 2, 3, 8, 40]))
        H = int(rng.choice([1, 8, 16, 64, 128]))
        T = int(rng.integers(1, 129))
        N = T + int(rng.integers(0, 300000))
        sms = int(rng.choice([148, 152, 20]))
        assert lib.ddt_verify_attn_num_splits(B, H, T, N, sms) == _wave_model(B, H, T, N, sms)


def test_host_argument_checks_launch_nothing(lib):
    dummy = ctypes.c_void_p(16)
    # null pointers -> invalid argument, returned before any CUDA call
    assert lib.ddt_build_tree(None, dummy, dummy, dummy, dummy, 1, 7, 8, dummy, dummy, dummy,
                              None) == 1
    # unsupported sizes
    assert lib.ddt_build_tree(dummy, dummy, dummy, dummy, dummy, 1, 8, 8, dummy, dummy, dummy,
                              None) == 2
    assert lib.ddt_build_tree(dummy, dummy, dummy, dummy, dummy, 1, 7, 17, dummy, dummy, dummy,
                              None) == 2
    assert lib.ddt_accept(dummy, dummy, dummy, dummy, 1, 0, dummy, dummy, dummy, dummy, None) == 2
    assert lib.ddt_compile_visibility(None, dummy, dummy, dummy, 1, 10, dummy, None) == 1
    assert lib.ddt_commit_kv(None, 10, dummy, dummy, dummy, dummy, dummy, 1, 7, None, None) == 1
    assert lib.ddt_commit_kv(ctypes.c_void_p(24), 10, dummy, dummy, dummy, dummy, dummy, 1, 7,
                             None, None) == 1  # pool not 16-byte aligned
    assert lib.ddt_commit_kv(dummy, 0, dummy, dummy, dummy, dummy, dummy, 1, 7, None, None) == 1
    assert lib.ddt_commit_kv(dummy, 10, dummy, dummy, dummy, dummy, dummy, 1, 8, None, None) == 2
    assert lib.ddt_commit_kv(dummy, 10, dummy, dummy, dummy, dummy, dummy, 0, 7, None, None) == 0
    assert lib.ddt_tree_links(None, dummy, 1, dummy, dummy, dummy, None) == 1
    sa = [dummy] * 5
    # (tree, links, qo, logits), vocab, temperature, top_k, top_p (may be NULL), coins,
    # coin_stride, batch, max_depth, four outputs, stream
    out4 = [dummy] * 4
    assert lib.ddt_accept_sampled(*sa, 0, dummy, dummy, None, dummy, 3, 1, 7, *out4,
                                  None) == 1   # vocab 0
    assert lib.ddt_accept_sampled(*sa, 100, dummy, dummy, None, dummy, 3, 1, 8, *out4,
                                  None) == 2  # max_depth 8
    assert lib.ddt_accept_sampled(*sa, 262145, dummy, dummy, None, dummy, 3, 1, 7, *out4,
                                  None) == 2  # vocab above DDT_MAX_VOCAB
    assert lib.ddt_accept_sampled(*sa, 100, dummy, dummy, None, dummy, 0, 1, 7, *out4,
                                  None) == 1  # no coins
    assert lib.ddt_accept_sampled(*sa, 100, dummy, dummy, dummy, dummy, 3, 0, 7, *out4,
                                  None) == 0  # empty batch: nothing to do
    # the allocation-free attention makes the same host checks before touching the device
    na = [dummy, dummy, 100, dummy, dummy, dummy, dummy, dummy]
    assert lib.ddt_verify_attn_noalloc(*na, 1, 8, 9, 9, 30, 0.1, 0, None, None, None) == 1
    assert lib.ddt_verify_attn_noalloc(*na, 1, 8, 9, 9, 30, 0.1, 129, dummy, None, None) == 2
    assert lib.ddt_verify_attn_noalloc(*na, 1, 8, 9, 9, 30, 0.1, -1, dummy, None, None) == 1
    assert lib.ddt_verify_attn_noalloc(*na, 1, 129, 9, 9, 30, 0.1, 0, dummy, None, None) == 2
    assert lib.ddt_verify_attn_noalloc(dummy, ctypes.c_void_p(18), *na[2:], 1, 8, 9, 9, 30, 0.1,
                                       0, dummy, None, None) == 1   # misaligned kv_pool
    assert lib.ddt_verify_step(None, None) == 1
    assert lib.ddt_prefill_step(None, None) == 1
    assert lib.ddt_build_chain_visibility(None, dummy, dummy, 1, dummy, dummy, dummy, None) == 1
    assert lib.ddt_build_chain_visibility(dummy, dummy, dummy, 1, dummy, dummy, None, None) == 1
    assert lib.ddt_build_chain_visibility(dummy, dummy, dummy, -1, dummy, dummy, dummy, None) == 1
    assert lib.ddt_build_chain_visibility(dummy, dummy, dummy, 0, dummy, dummy, dummy, None) == 0
    assert lib.ddt_step_graph_create(None, None) == 1
    assert lib.ddt_step_graph_launch(None, None) == 1
    assert lib.ddt_step_graph_destroy(None) == 1
    tv = [dummy] * 7
    assert lib.ddt_build_tree_visibility(*tv, 1, 7, 8, dummy, dummy, dummy, None, None) == 1
    assert lib.ddt_build_tree_visibility(*tv, 1, 8, 8, dummy, dummy, dummy, dummy, None) == 2
    assert lib.ddt_build_tree_visibility(*tv, 1, 7, 0, dummy, dummy, dummy, dummy, None) == 2
    assert lib.ddt_build_tree_visibility(*tv, 0, 7, 8, dummy, dummy, dummy, dummy, None) == 0
    args = [dummy, dummy, 100, dummy, dummy, dummy, dummy, dummy]
    #        B  H   total_q max_q max_kv scale splits
    bad = [(0, 8, 9, 9, 30, 0.1, 0), (1, 8, 9, 9, 5, 0.1, 0), (1, 8, 9, 9, 30, float("nan"), 0),
           (1, 8, 9, 9, 30, 0.1, -1)]
    for B, H, tq, mq, mk, sc, sp in bad:
        assert lib.ddt_verify_attn(*args, B, H, tq, mq, mk, sc, sp, dummy, None, None, 0,
                                   None) == 1
    assert lib.ddt_verify_attn(*args, 1, 8, 129, 129, 300, 0.1, 0, dummy, None, None, 0, None) == 2
    assert lib.ddt_verify_attn(*args, 1, 129, 9, 9, 30, 0.1, 0, dummy, None, None, 0, None) == 2
    # misaligned kv_pool
    a2 = [dummy, ctypes.c_void_p(18), 100, dummy, dummy, dummy, dummy, dummy]
    assert lib.ddt_verify_attn(*a2, 1, 8, 9, 9, 30, 0.1, 0, dummy, None, None, 0, None) == 1
    # the bounded-wait self test checks its poll limit before touching the device
    lib.ddt_selftest_wait_timeout.argtypes = [ctypes.c_uint32, ctypes.c_void_p]
    assert lib.ddt_selftest_wait_timeout(0, None) == 1
    assert lib.ddt_selftest_wait_timeout((1 << 24) + 1, None) == 1


def test_step_args_layout_matches_the_header(tmp_path):
    # the ctypes mirror of ddt_step_args must agree with the C compiler's layout
    import subprocess
    from tree_speculative_decoding_gb300 import ddt
    fields = [f[0] for f in ddt.StepArgs._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "ddt.h"\nint main(void) {\n'
                   '    printf("%zu\\n", sizeof(ddt_step_args));\n'
                   + "".join(f'    printf("%zu\\n", offsetof(ddt_step_args, {f}));\n' for f in fields)
                   + "    return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(os.path.dirname(__file__), "..", "include"),
                    "-o", str(exe), str(src)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    assert got[0] == ctypes.sizeof(ddt.StepArgs)
    assert got[1:] == [getattr(ddt.StepArgs, f).offset for f in fields]
