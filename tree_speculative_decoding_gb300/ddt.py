"""Thin ctypes binding of libddt.so (``include/ddt.h``).

Argument marshalling only: torch tensors become device pointers, the current
torch stream becomes the ``cudaStream_t``; every step of the verify path runs
in the library's kernels.  There is no fallback: if the shared library is
missing or fails to load, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

DL, DR, D = 512, 64, 576
MAX_DEPTH, MAX_TOPK, MAX_Q_LEN, MAX_SPLITS = 7, 16, 128, 128

STATUS = {0: "DDT_OK", 1: "DDT_ERR_INVALID_ARG", 2: "DDT_ERR_UNSUPPORTED", 3: "DDT_ERR_WORKSPACE",
          4: "DDT_ERR_CUDA", 5: "DDT_ERR_DEVICE_CHECK", 6: "DDT_ERR_TIMEOUT"}


class DDTError(RuntimeError):
    def __init__(self, fn, status, detail=""):
        self.status = status
        super().__init__(f"{fn}: {STATUS.get(status, status)}{(' ' + detail) if detail else ''}")


def _load():
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"libddt.so not built at {path}; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
    sig = {
        "ddt_abi_version": ([], i32),
        "ddt_status_string": ([i32], ctypes.c_char_p),
        "ddt_build_tree": ([P, P, P, P, P, i32, i32, i32, P, P, P, P], i32),
        "ddt_mask_indptr": ([P, P, i32, P], i32),
        "ddt_compile_visibility": ([P, P, P, P, i32, i32, P, P], i32),
        "ddt_build_tree_visibility": ([P, P, P, P, P, P, P, i32, i32, i32, P, P, P, P, P], i32),
        "ddt_build_chain_visibility": ([P, P, P, i32, P, P, P, P], i32),
        "ddt_verify_attn_num_splits": ([i32, i32, i32, i32, i32], i32),
        "ddt_verify_attn_launched_splits": ([i32, i32], i32),
        "ddt_verify_attn_noalloc_splits": ([i32, i32, i32, i32, i32, i32], i32),
        "ddt_verify_attn_workspace_size": ([i32, i32, i32], sz),
        "ddt_verify_attn": ([P, P, i64, P, P, P, P, P, i32, i32, i32, i32, i32, f32, i32, P, P, P,
                             sz, P], i32),
        "ddt_verify_attn_noalloc": ([P, P, i64, P, P, P, P, P, i32, i32, i32, i32, i32, f32, i32, P,
                                     P, P], i32),
        "ddt_accept": ([P, P, P, P, i32, i32, P, P, P, P, P], i32),
        "ddt_commit_kv": ([P, i64, P, P, P, P, P, i32, i32, P, P], i32),
        "ddt_tree_links": ([P, P, i32, P, P, P, P], i32),
        "ddt_accept_sampled": ([P, P, P, P, P, i32, P, P, P, P, i32, i32, i32, P, P, P, P, P],
                               i32),
        "ddt_get_error": ([P, P], i32),
        "ddt_selftest_wait_timeout": ([ctypes.c_uint32, P], i32),
        "ddt_verify_step": ([P, P], i32),
        "ddt_prefill_step": ([P, P], i32),
        "ddt_step_graph_create": ([P, P], i32),
        "ddt_step_graph_create_io": ([P, P, P, sz, P, P, sz, P], i32),
        "ddt_step_graph_launch": ([P, P], i32),
        "ddt_step_graph_destroy": ([P], i32),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


lib = _load()


class StepArgs(ctypes.Structure):
    """ddt_step_args of include/ddt.h, field for field."""
    _P, _i32 = ctypes.c_void_p, ctypes.c_int32
    _fields_ = [
        ("topk_logp", _P), ("topk_ids", _P), ("root_id", _P), ("budget", _P),
        ("max_depth", _i32), ("topk", _i32),
        ("batch", _i32), ("total_q", _i32), ("max_q_len", _i32), ("max_kv_len", _i32),
        ("total_mask_words", _i32),
        ("qo_indptr", _P), ("kv_indptr", _P), ("prefix_len", _P), ("mask_indptr", _P),
        ("q", _P), ("kv_pool", _P), ("pool_rows", ctypes.c_int64), ("kv_indices", _P),
        ("num_heads", _i32), ("scale", ctypes.c_float), ("num_splits", _i32),
        ("workspace", _P), ("workspace_bytes", ctypes.c_size_t),
        ("target_argmax", _P),
        ("node_token", _P), ("parent", _P), ("depth", _P), ("mask", _P), ("out", _P), ("lse", _P),
        ("accept_len", _P), ("accepted_nodes", _P), ("commit_tokens", _P), ("bonus", _P),
        ("commit_kv", _i32), ("new_len", _P),
    ]


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, st):
    if st != 0:
        raise DDTError(fn, st)


def _dev(t, dtype, name):
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")
    return t


def abi_version() -> int:
    return lib.ddt_abi_version()


def ddt_build_tree(topk_logp, topk_ids, root_id, budget, qo_indptr, node_token, parent, depth,
                   stream=None):
    B, max_depth, K = topk_logp.shape
    _dev(topk_logp, torch.float32, "topk_logp")
    for n, t in (("topk_ids", topk_ids), ("root_id", root_id), ("budget", budget),
                 ("qo_indptr", qo_indptr), ("node_token", node_token), ("parent", parent),
                 ("depth", depth)):
        _dev(t, torch.int32, n)
    _check("ddt_build_tree", lib.ddt_build_tree(
        _p(topk_logp), _p(topk_ids), _p(root_id), _p(budget), _p(qo_indptr), B, max_depth, K,
        _p(node_token), _p(parent), _p(depth), _stream(stream)))


def ddt_mask_indptr(qo_indptr_host, prefix_len_host):
    """Host helper: int32 word offsets of the bit-packed mask (CPU tensors in/out)."""
    qo = qo_indptr_host.to(torch.int32).contiguous().cpu()
    pl = prefix_len_host.to(torch.int32).contiguous().cpu()
    out = torch.empty(pl.numel() + 1, dtype=torch.int32)
    _check("ddt_mask_indptr", lib.ddt_mask_indptr(_p(qo), _p(pl), pl.numel(), _p(out)))
    return out


def ddt_compile_visibility(parent, qo_indptr, prefix_len, mask_indptr, mask, stream=None):
    for n, t in (("parent", parent), ("qo_indptr", qo_indptr), ("prefix_len", prefix_len),
                 ("mask_indptr", mask_indptr)):
        _dev(t, torch.int32, n)
    if not (mask.is_cuda and mask.dtype in (torch.int32, torch.uint32) and mask.is_contiguous()):
        raise ValueError("mask must be a contiguous CUDA 32-bit tensor")
    B = prefix_len.numel()
    _check("ddt_compile_visibility", lib.ddt_compile_visibility(
        _p(parent), _p(qo_indptr), _p(prefix_len), _p(mask_indptr), B, mask.numel(), _p(mask),
        _stream(stream)))


def ddt_build_chain_visibility(qo_indptr, prefix_len, mask_indptr, parent, depth, mask,
                               stream=None):
    """A prefill chunk's chain (parent[i] = i - 1, depth[i] = i) and its causal mask."""
    for n, t in (("qo_indptr", qo_indptr), ("prefix_len", prefix_len), ("mask_indptr", mask_indptr),
                 ("parent", parent), ("depth", depth)):
        _dev(t, torch.int32, n)
    if not (mask.is_cuda and mask.dtype in (torch.int32, torch.uint32) and mask.is_contiguous()):
        raise ValueError("mask must be a contiguous CUDA 32-bit tensor")
    B = prefix_len.numel()
    if qo_indptr.numel() != B + 1 or mask_indptr.numel() != B + 1:
        raise ValueError("qo_indptr and mask_indptr must hold batch + 1 offsets")
    if parent.numel() != depth.numel():
        raise ValueError("parent and depth must have the same length")
    _check("ddt_build_chain_visibility", lib.ddt_build_chain_visibility(
        _p(qo_indptr), _p(prefix_len), _p(mask_indptr), B, _p(parent), _p(depth), _p(mask),
        _stream(stream)))


def ddt_build_tree_visibility(topk_logp, topk_ids, root_id, budget, qo_indptr, prefix_len,
                              mask_indptr, node_token, parent, depth, mask, stream=None):
    """ddt_build_tree and ddt_compile_visibility in one launch (same outputs)."""
    B, max_depth, K = topk_logp.shape
    _dev(topk_logp, torch.float32, "topk_logp")
    for n, t in (("topk_ids", topk_ids), ("root_id", root_id), ("budget", budget),
                 ("qo_indptr", qo_indptr), ("prefix_len", prefix_len), ("mask_indptr", mask_indptr),
                 ("node_token", node_token), ("parent", parent), ("depth", depth)):
        _dev(t, torch.int32, n)
    if not (mask.is_cuda and mask.dtype in (torch.int32, torch.uint32) and mask.is_contiguous()):
        raise ValueError("mask must be a contiguous CUDA 32-bit tensor")
    _check("ddt_build_tree_visibility", lib.ddt_build_tree_visibility(
        _p(topk_logp), _p(topk_ids), _p(root_id), _p(budget), _p(qo_indptr), _p(prefix_len),
        _p(mask_indptr), B, max_depth, K, _p(node_token), _p(parent), _p(depth), _p(mask),
        _stream(stream)))


def ddt_verify_attn_num_splits(batch, num_heads, max_q_len, max_kv_len, num_sms=0):
    return lib.ddt_verify_attn_num_splits(batch, num_heads, max_q_len, max_kv_len, num_sms)


def ddt_verify_attn_launched_splits(max_kv_len, num_splits):
    """Splits a ddt_verify_attn call with num_splits (>= 1) launches (the
    requested count rounded to whole 64-column tiles)."""
    return lib.ddt_verify_attn_launched_splits(int(max_kv_len), int(num_splits))


def ddt_verify_attn_noalloc_splits(batch, num_heads, total_q, max_q_len, max_kv_len, num_splits=0):
    """Splits a ddt_verify_attn_noalloc call with these sizes launches."""
    return lib.ddt_verify_attn_noalloc_splits(int(batch), int(num_heads), int(total_q),
                                              int(max_q_len), int(max_kv_len), int(num_splits))


def ddt_verify_attn_workspace_size(total_q, num_heads, num_splits):
    return lib.ddt_verify_attn_workspace_size(total_q, num_heads, num_splits)


def _attn_args(q, kv_pool, kv_indices, kv_indptr, qo_indptr, mask, mask_indptr, out, lse,
               max_q_len, max_kv_len):
    """The checks both attention entry points need (the C ABI cannot see tensor
    shapes): dtypes, contiguity, 576-wide rows, out [total_q, H, 512], lse
    [total_q, H]; returns (total_q, H, batch, max_q_len, max_kv_len)."""
    _dev(q, torch.bfloat16, "q")
    _dev(kv_pool, torch.bfloat16, "kv_pool")
    _dev(out, torch.float32, "out")
    for n, t in (("kv_indices", kv_indices), ("kv_indptr", kv_indptr), ("qo_indptr", qo_indptr),
                 ("mask_indptr", mask_indptr)):
        _dev(t, torch.int32, n)
    if not (mask.is_cuda and mask.dtype in (torch.int32, torch.uint32) and mask.is_contiguous()):
        raise ValueError("mask must be a contiguous CUDA 32-bit tensor")
    if q.dim() != 3 or kv_pool.dim() != 2:
        raise ValueError("q must be [total_q, H, 576] and kv_pool [pool_rows, 576]")
    total_q, H, d = q.shape
    if d != D or kv_pool.shape[-1] != D or tuple(out.shape) != (total_q, H, DL):
        raise ValueError("q/kv_pool rows must be 576 wide and out [total_q, H, 512]")
    if lse is not None:
        _dev(lse, torch.float32, "lse")
        if tuple(lse.shape) != (total_q, H):
            raise ValueError("lse must be [total_q, H]")
    B = qo_indptr.numel() - 1
    if kv_indptr.numel() != B + 1 or mask_indptr.numel() != B + 1:
        raise ValueError("qo_indptr, kv_indptr and mask_indptr must all hold batch + 1 entries")
    if max_q_len is None or max_kv_len is None:
        qo = qo_indptr.cpu()
        kv = kv_indptr.cpu()
        max_q_len = int((qo[1:] - qo[:-1]).max())
        max_kv_len = int((kv[1:] - kv[:-1]).max())
    return total_q, H, B, int(max_q_len), int(max_kv_len)


def ddt_verify_attn(q, kv_pool, kv_indices, kv_indptr, qo_indptr, mask, mask_indptr, scale,
                    out, lse=None, max_q_len=None, max_kv_len=None, num_splits=0,
                    workspace=None, stream=None):
    """q: [total_q, H, 576] bf16; kv_pool: [pool_rows, 576] bf16; out: [total_q, H, 512] f32.

    max_q_len / max_kv_len are host-side bounds used to size the grid; when
    omitted they are read from the indptrs (a device->host copy)."""
    total_q, H, B, max_q_len, max_kv_len = _attn_args(q, kv_pool, kv_indices, kv_indptr, qo_indptr,
                                                      mask, mask_indptr, out, lse, max_q_len,
                                                      max_kv_len)
    if workspace is None:
        splits = num_splits or ddt_verify_attn_num_splits(B, H, max_q_len, max_kv_len)
        nbytes = ddt_verify_attn_workspace_size(total_q, H, splits)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device) if nbytes else None
        num_splits = splits
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("ddt_verify_attn", lib.ddt_verify_attn(
        _p(q), _p(kv_pool), kv_pool.shape[0], _p(kv_indices), _p(kv_indptr), _p(qo_indptr),
        _p(mask), _p(mask_indptr), B, H, total_q, int(max_q_len), int(max_kv_len), float(scale),
        int(num_splits), _p(out), _p(lse), _p(workspace), ws_bytes, _stream(stream)))


NOALLOC_SCRATCH_BYTES = 32 << 20


def ddt_verify_attn_noalloc(q, kv_pool, kv_indices, kv_indptr, qo_indptr, mask, mask_indptr,
                            scale, out, lse=None, max_q_len=None, max_kv_len=None, num_splits=0,
                            stream=None):
    """ddt_verify_attn for callers that cannot allocate device memory (a
    pre-reserved engine pool, a host without an allocator, a loop where a
    device-synchronising cudaMalloc is not allowed): the split scratch is a
    fixed 32 MiB array inside libddt.so, so neither this wrapper nor the call
    allocates on the device.  Calls overlapping on the GPU race on that
    array.  num_splits = 0 takes the library's choice among the counts that
    fit the array; an explicit count that needs more scratch than the array
    holds raises DDTError(DDT_ERR_WORKSPACE)."""
    total_q, H, B, max_q_len, max_kv_len = _attn_args(q, kv_pool, kv_indices, kv_indptr, qo_indptr,
                                                      mask, mask_indptr, out, lse, max_q_len,
                                                      max_kv_len)
    _check("ddt_verify_attn_noalloc", lib.ddt_verify_attn_noalloc(
        _p(q), _p(kv_pool), kv_pool.shape[0], _p(kv_indices), _p(kv_indptr), _p(qo_indptr),
        _p(mask), _p(mask_indptr), B, H, total_q, int(max_q_len), int(max_kv_len), float(scale),
        int(num_splits), _p(out), _p(lse), _stream(stream)))


def ddt_accept(node_token, parent, qo_indptr, target_argmax, max_depth, accept_len,
               accepted_nodes, commit_tokens, bonus, stream=None):
    for n, t in (("node_token", node_token), ("parent", parent), ("qo_indptr", qo_indptr),
                 ("target_argmax", target_argmax), ("accept_len", accept_len),
                 ("accepted_nodes", accepted_nodes), ("commit_tokens", commit_tokens),
                 ("bonus", bonus)):
        _dev(t, torch.int32, n)
    B = qo_indptr.numel() - 1
    _check("ddt_accept", lib.ddt_accept(
        _p(node_token), _p(parent), _p(qo_indptr), _p(target_argmax), B, int(max_depth),
        _p(accept_len), _p(accepted_nodes), _p(commit_tokens), _p(bonus), _stream(stream)))


def ddt_commit_kv(kv_pool, kv_indices, kv_indptr, qo_indptr, accept_len, accepted_nodes, max_depth,
                  new_len=None, stream=None):
    """KV commit: gathers each request's accepted latents into positions
    P .. P + accept_len - 1 of its sequence, in place in kv_pool."""
    _dev(kv_pool, torch.bfloat16, "kv_pool")
    for n, t in (("kv_indices", kv_indices), ("kv_indptr", kv_indptr), ("qo_indptr", qo_indptr),
                 ("accept_len", accept_len), ("accepted_nodes", accepted_nodes)):
        _dev(t, torch.int32, n)
    if new_len is not None:
        _dev(new_len, torch.int32, "new_len")
    B = qo_indptr.numel() - 1
    _check("ddt_commit_kv", lib.ddt_commit_kv(
        _p(kv_pool), kv_pool.shape[0], _p(kv_indices), _p(kv_indptr), _p(qo_indptr),
        _p(accept_len), _p(accepted_nodes), B, int(max_depth), _p(new_len), _stream(stream)))


def ddt_verify_step(args: StepArgs, stream=None):
    """One verify step in one call (tree + mask, attention, accept, optional commit)."""
    _check("ddt_verify_step", lib.ddt_verify_step(ctypes.byref(args), _stream(stream)))


def ddt_prefill_step(args: StepArgs, stream=None):
    """One prefill chunk in one call (causal chain + mask, attention)."""
    _check("ddt_prefill_step", lib.ddt_prefill_step(ctypes.byref(args), _stream(stream)))


class StepGraph:
    """A library-owned CUDA graph of one ddt_verify_step; the tensors behind
    `args` must outlive it."""

    def __init__(self, args: StepArgs, keep_alive=(), io=None):
        """io = (h_in, d_in, h_out, d_out): pinned host and device uint8 buffers;
        the graph then copies h_in -> d_in before the step and d_out -> h_out
        after it (ddt_step_graph_create_io)."""
        self._keep = (args, tuple(keep_alive), io)
        h = ctypes.c_void_p()
        if io is None:
            _check("ddt_step_graph_create",
                   lib.ddt_step_graph_create(ctypes.byref(args), ctypes.byref(h)))
        else:
            h_in, d_in, h_out, d_out = io
            for t, dev, n in ((h_in, False, "h_in"), (d_in, True, "d_in"), (h_out, False, "h_out"),
                              (d_out, True, "d_out")):
                if t.is_cuda != dev or not t.is_contiguous() or (not dev and not t.is_pinned()):
                    raise ValueError(f"{n} must be a contiguous {'CUDA' if dev else 'pinned host'} "
                                     "tensor")
            nin = h_in.numel() * h_in.element_size()
            nout = h_out.numel() * h_out.element_size()
            if nin > d_in.numel() * d_in.element_size() or nout > d_out.numel() * d_out.element_size():
                raise ValueError("a host buffer is larger than its device buffer")
            _check("ddt_step_graph_create_io", lib.ddt_step_graph_create_io(
                ctypes.byref(args), _p(h_in), _p(d_in), nin, _p(h_out), _p(d_out), nout,
                ctypes.byref(h)))
        self._h = h

    def launch(self, stream=None):
        _check("ddt_step_graph_launch", lib.ddt_step_graph_launch(self._h, _stream(stream)))

    def close(self):
        if self._h:
            _check("ddt_step_graph_destroy", lib.ddt_step_graph_destroy(self._h))
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def ddt_tree_links(parent, qo_indptr, first_child, next_sibling, retrieve_index, stream=None):
    """The tree as (first_child, next_sibling, retrieve_index) links."""
    for n, t in (("parent", parent), ("qo_indptr", qo_indptr), ("first_child", first_child),
                 ("next_sibling", next_sibling), ("retrieve_index", retrieve_index)):
        _dev(t, torch.int32, n)
    _check("ddt_tree_links", lib.ddt_tree_links(
        _p(parent), _p(qo_indptr), qo_indptr.numel() - 1, _p(first_child), _p(next_sibling),
        _p(retrieve_index), _stream(stream)))


def ddt_accept_sampled(node_token, first_child, next_sibling, qo_indptr, target_logits,
                       temperature, top_k, coins, max_depth, accept_len, accepted_nodes,
                       commit_tokens, bonus, stream=None, top_p=None):
    """Sampling accept: tree rejection sampling with temperature, top-k and top-p.
    target_logits float32 [rows, vocab]; temperature float32 [B]; top_k int32 [B];
    coins float32 [rows, coin_stride] uniform in [0, 1); top_p float32 [B] or None."""
    _dev(target_logits, torch.float32, "target_logits")
    _dev(temperature, torch.float32, "temperature")
    _dev(coins, torch.float32, "coins")
    for n, t in (("node_token", node_token), ("first_child", first_child),
                 ("next_sibling", next_sibling), ("qo_indptr", qo_indptr), ("top_k", top_k),
                 ("accept_len", accept_len), ("accepted_nodes", accepted_nodes),
                 ("commit_tokens", commit_tokens), ("bonus", bonus)):
        _dev(t, torch.int32, n)
    B = qo_indptr.numel() - 1
    if top_p is not None:
        _dev(top_p, torch.float32, "top_p")
        if top_p.numel() != B:
            raise ValueError("top_p must hold one value per request")
    if temperature.numel() != B or top_k.numel() != B:
        raise ValueError("temperature and top_k must hold one value per request")
    _check("ddt_accept_sampled", lib.ddt_accept_sampled(
        _p(node_token), _p(first_child), _p(next_sibling), _p(qo_indptr), _p(target_logits),
        target_logits.shape[1], _p(temperature), _p(top_k), _p(top_p), _p(coins), coins.shape[1], B,
        int(max_depth), _p(accept_len), _p(accepted_nodes), _p(commit_tokens), _p(bonus),
        _stream(stream)))


def ddt_get_error(stream=None):
    """Returns (status, device_error_bits) and clears the device error word."""
    word = ctypes.c_uint32(0)
    st = lib.ddt_get_error(_stream(stream), ctypes.byref(word))
    return st, word.value


def ddt_selftest_wait_timeout(poll_limit=1 << 12, stream=None):
    """Launch the bounded-wait failure check: a kernel waiting on a barrier
    nobody arrives on gives up after `poll_limit` polls and latches the timeout
    bit (read it with ddt_get_error)."""
    _check("ddt_selftest_wait_timeout", lib.ddt_selftest_wait_timeout(int(poll_limit), _stream(stream)))
