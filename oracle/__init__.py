"""Plain CPU oracle for the DDTree verify step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product path never does.
It shares no code with the CUDA library: the C source next to this file is
compiled on its own by ``build()`` (gcc, OpenMP) and loaded through ctypes.

The arithmetic lives in ``ddt_oracle.c``; this module only marshals numpy
arrays.  Each function cites the passage it follows in the C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ddt_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

DL, DR, D = 512, 64, 576


def build(force: bool = False) -> str:
    """Compile ddt_oracle.c into a shared library (gcc -O2, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_build_tree.argtypes = [P, P, P, P, P, i32, i32, i32, P, P, P]
            lib.oracle_mask_indptr.argtypes = [P, P, i32, P]
            lib.oracle_compile_visibility.argtypes = [P, P, P, P, i32, P]
            lib.oracle_verify_attn.argtypes = [P, P, i64, P, P, P, P, P, i32, i32, dbl,
                                               P, i64, P, P, i32]
            lib.oracle_accept.argtypes = [P, P, P, P, i32, i32, P, P, P, P]
            lib.oracle_commit_kv.argtypes = [P, i64, P, P, P, P, P, i32, i32, P]
            lib.oracle_tree_links.argtypes = [P, P, i32, P, P, P]
            lib.oracle_accept_sampled.argtypes = [P, P, P, P, i32, P, P, P, P, i32, i32, i32,
                                                  P, P, P, P]
            lib.oracle_num_threads.argtypes = []
            for f in (lib.oracle_build_tree, lib.oracle_mask_indptr,
                      lib.oracle_compile_visibility, lib.oracle_verify_attn,
                      lib.oracle_accept, lib.oracle_commit_kv, lib.oracle_tree_links,
                      lib.oracle_accept_sampled, lib.oracle_num_threads):
                f.restype = ctypes.c_int
            _lib = lib
        return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    pass


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def build_tree(topk_logp, topk_ids, root_id, budget, qo_indptr, max_depth, K):
    """Best-first tree; returns (node_token, parent, depth), ragged by qo_indptr."""
    lib = _load()
    topk_logp = _c(topk_logp, np.float32)
    topk_ids = _c(topk_ids, np.int32)
    root_id = _c(root_id, np.int32)
    budget = _c(budget, np.int32)
    qo_indptr = _c(qo_indptr, np.int32)
    B = budget.shape[0]
    total = int(qo_indptr[-1])
    tok = np.empty(total, np.int32)
    par = np.empty(total, np.int32)
    dep = np.empty(total, np.int32)
    rc = lib.oracle_build_tree(_ptr(topk_logp), _ptr(topk_ids), _ptr(root_id), _ptr(budget),
                               _ptr(qo_indptr), B, int(max_depth), int(K),
                               _ptr(tok), _ptr(par), _ptr(dep))
    if rc != 0:
        raise OracleError(f"oracle_build_tree failed ({rc})")
    return tok, par, dep


def mask_indptr(qo_indptr, prefix_len):
    lib = _load()
    qo_indptr = _c(qo_indptr, np.int32)
    prefix_len = _c(prefix_len, np.int32)
    B = prefix_len.shape[0]
    out = np.empty(B + 1, np.int64)
    rc = lib.oracle_mask_indptr(_ptr(qo_indptr), _ptr(prefix_len), B, _ptr(out))
    if rc != 0:
        raise OracleError(f"oracle_mask_indptr failed ({rc})")
    return out


def compile_visibility(parent, qo_indptr, prefix_len):
    """Bit-packed mask and its word offsets (int64)."""
    lib = _load()
    parent = _c(parent, np.int32)
    qo_indptr = _c(qo_indptr, np.int32)
    prefix_len = _c(prefix_len, np.int32)
    mip = mask_indptr(qo_indptr, prefix_len)
    mask = np.zeros(int(mip[-1]), np.uint32)
    rc = lib.oracle_compile_visibility(_ptr(parent), _ptr(qo_indptr), _ptr(prefix_len),
                                       _ptr(mip), prefix_len.shape[0], _ptr(mask))
    if rc != 0:
        raise OracleError(f"oracle_compile_visibility failed ({rc})")
    return mask, mip


def verify_attn(q, kv_pool, kv_indices, kv_indptr, qo_indptr, mask, mask_indptr_,
                num_heads, scale, rows=None, nthreads=0):
    """fp64 masked attention for the requested rows (row = token*H + head).

    q, kv_pool: uint16 arrays holding bf16 bits.  Returns (out [n,512], lse [n]).
    """
    lib = _load()
    q = _c(q, np.uint16)
    kv_pool = _c(kv_pool, np.uint16)
    kv_indices = _c(kv_indices, np.int32)
    kv_indptr = _c(kv_indptr, np.int32)
    qo_indptr = _c(qo_indptr, np.int32)
    mask = _c(mask, np.uint32)
    mip = _c(mask_indptr_, np.int64)
    B = qo_indptr.shape[0] - 1
    if rows is None:
        rows = np.arange(int(qo_indptr[-1]) * num_heads, dtype=np.int64)
    rows = _c(rows, np.int64)
    pool_rows = kv_pool.size // D
    out = np.empty((rows.shape[0], DL), np.float64)
    lse = np.empty(rows.shape[0], np.float64)
    rc = lib.oracle_verify_attn(_ptr(q), _ptr(kv_pool), pool_rows, _ptr(kv_indices),
                                _ptr(kv_indptr), _ptr(qo_indptr), _ptr(mask), _ptr(mip),
                                B, int(num_heads), float(scale), _ptr(rows), rows.shape[0],
                                _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise OracleError(f"oracle_verify_attn failed ({rc})")
    return out, lse


def accept(node_token, parent, qo_indptr, target_argmax, max_depth):
    """Greedy walk; returns (accept_len, accepted_nodes, commit_tokens, bonus)."""
    lib = _load()
    node_token = _c(node_token, np.int32)
    parent = _c(parent, np.int32)
    qo_indptr = _c(qo_indptr, np.int32)
    target_argmax = _c(target_argmax, np.int32)
    B = qo_indptr.shape[0] - 1
    W = int(max_depth) + 1
    alen = np.empty(B, np.int32)
    acc = np.empty((B, W), np.int32)
    com = np.empty((B, W), np.int32)
    bon = np.empty(B, np.int32)
    rc = lib.oracle_accept(_ptr(node_token), _ptr(parent), _ptr(qo_indptr), _ptr(target_argmax),
                           B, int(max_depth), _ptr(alen), _ptr(acc), _ptr(com), _ptr(bon))
    if rc != 0:
        raise OracleError(f"oracle_accept failed ({rc})")
    return alen, acc, com, bon


def commit_kv(kv_pool, kv_indices, kv_indptr, qo_indptr, accept_len, accepted_nodes, max_depth):
    """KV commit: returns (new pool, new_len).  kv_pool is uint16 (bf16 bits)
    [pool_rows, 576] and is not modified; the returned copy holds, at
    positions P_b .. P_b + accept_len - 1 of each request, the accepted
    nodes' latents in path order."""
    lib = _load()
    pool = np.array(kv_pool, dtype=np.uint16, copy=True, order="C")
    kv_indices = _c(kv_indices, np.int32)
    kv_indptr = _c(kv_indptr, np.int32)
    qo_indptr = _c(qo_indptr, np.int32)
    accept_len = _c(accept_len, np.int32)
    accepted_nodes = _c(accepted_nodes, np.int32)
    B = qo_indptr.shape[0] - 1
    new_len = np.empty(B, np.int32)
    rc = lib.oracle_commit_kv(_ptr(pool), int(pool.shape[0]), _ptr(kv_indices), _ptr(kv_indptr),
                              _ptr(qo_indptr), _ptr(accept_len), _ptr(accepted_nodes), B,
                              int(max_depth), _ptr(new_len))
    if rc != 0:
        raise OracleError(f"oracle_commit_kv failed ({rc})")
    return pool, new_len


def tree_links(parent, qo_indptr):
    """(first_child, next_sibling, retrieve_index) of the tree: local indices,
    -1 where there is none; retrieve_index is the node's global row."""
    lib = _load()
    parent = _c(parent, np.int32)
    qo_indptr = _c(qo_indptr, np.int32)
    n = parent.shape[0]
    fc, ns, ri = (np.empty(n, np.int32) for _ in range(3))
    rc = lib.oracle_tree_links(_ptr(parent), _ptr(qo_indptr), qo_indptr.shape[0] - 1, _ptr(fc),
                               _ptr(ns), _ptr(ri))
    if rc != 0:
        raise OracleError(f"oracle_tree_links failed ({rc})")
    return fc, ns, ri


def accept_sampled(node_token, parent, qo_indptr, logits, temperature, top_k, coins, max_depth,
                   top_p=None):
    """Sampling accept (reading R15).  logits float32 [rows, vocab]; temperature
    float32 [B]; top_k int32 [B]; coins float32 [rows, coin_stride]; top_p
    float32 [B] or None (no top-p).  Returns (accept_len, accepted_nodes,
    commit_tokens, bonus) as accept() does."""
    lib = _load()
    node_token = _c(node_token, np.int32)
    parent = _c(parent, np.int32)
    qo_indptr = _c(qo_indptr, np.int32)
    logits = _c(logits, np.float32)
    temperature = _c(temperature, np.float32)
    top_k = _c(top_k, np.int32)
    coins = _c(coins, np.float32)
    B = qo_indptr.shape[0] - 1
    top_p = None if top_p is None else _c(top_p, np.float32)
    W = int(max_depth) + 1
    alen = np.empty(B, np.int32)
    acc = np.empty((B, W), np.int32)
    com = np.empty((B, W), np.int32)
    bon = np.empty(B, np.int32)
    rc = lib.oracle_accept_sampled(_ptr(node_token), _ptr(parent), _ptr(qo_indptr), _ptr(logits),
                                   int(logits.shape[1]), _ptr(temperature), _ptr(top_k),
                                   None if top_p is None else _ptr(top_p), _ptr(coins),
                                   int(coins.shape[1]), B, int(max_depth), _ptr(alen), _ptr(acc),
                                   _ptr(com), _ptr(bon))
    if rc != 0:
        raise OracleError(f"oracle_accept_sampled failed ({rc})")
    return alen, acc, com, bon


def best_child_argmax(parent, qo_indptr, node_token, coin, fallback):
    """Compose a target argmax from an oracle tree: where coin[n] is set, the
    argmax at node n is the token of n's best child (its lowest-index child,
    the first one popped), else fallback[n].  A node without children always
    takes fallback[n].  Used to build chain-forcing and partly-matching
    argmax inputs for tests; it runs on oracle trees only."""
    parent = np.asarray(parent)
    out = np.array(fallback, dtype=np.int32, copy=True)
    for b in range(len(qo_indptr) - 1):
        lo, hi = int(qo_indptr[b]), int(qo_indptr[b + 1])
        first_child = {}
        for c in range(lo + 1, hi):
            p = lo + int(parent[c])
            if p not in first_child:
                first_child[p] = c
        for n in range(lo, hi):
            if coin[n] and n in first_child:
                out[n] = node_token[first_child[n]]
    return out
