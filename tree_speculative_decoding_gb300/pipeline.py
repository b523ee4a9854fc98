"""One DDTree verify step on the GPU through the C ABI.

``VerifyStep`` owns the device buffers of one batch and runs the four stages
in order on one stream: ddt_build_tree -> ddt_compile_visibility ->
ddt_verify_attn -> ddt_accept (the per-iteration data flow of "The Oracle
Drafter", section "The Engine Interface Design", with the mask and positions
built on the device instead of the host).  By default the first two run as
one launch (ddt_build_tree_visibility); ``fused_tree_mask=False`` calls them
separately.  It only allocates and calls the binding; all arithmetic runs in
libddt.so.
"""
from __future__ import annotations

import numpy as np
import torch

from . import ddt


def _i32(a, device):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def _bf16(a, device):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16).to(device)


class _Arena:
    """One contiguous device buffer holding several tensors at 256-byte-aligned
    offsets.  Each entry is (name, dtype, data or shape): numpy data (uint16
    holding bf16 bits for bfloat16) is copied in, a shape is left uninitialised."""

    def __init__(self, entries, device):
        layout, off = [], 0
        for name, dtype, src in entries:
            shape = tuple(src) if isinstance(src, tuple) else tuple(np.shape(src))
            nbytes = int(np.prod(shape, dtype=np.int64)) * torch.empty((), dtype=dtype).element_size()
            layout.append((name, dtype, shape, off, nbytes, None if isinstance(src, tuple) else src))
            off += (nbytes + 255) // 256 * 256
        self.buf = torch.empty(max(off, 256), dtype=torch.uint8, device=device)
        self.offsets = {name: o for name, _, _, o, _, _ in layout}
        self.views = {}
        for name, dtype, shape, o, nbytes, src in layout:
            v = self.buf[o:o + nbytes].view(dtype).view(shape)
            if src is not None:
                if dtype == torch.bfloat16:
                    host = torch.from_numpy(np.ascontiguousarray(src, np.uint16).view(np.int16)).view(torch.bfloat16)
                else:
                    host = torch.from_numpy(np.ascontiguousarray(src)).to(dtype)
                v.copy_(host.reshape(shape))
            self.views[name] = v


class VerifyStep:
    """Device-resident inputs and outputs of one verify step for a Workload."""

    def __init__(self, wl, device="cuda", target_argmax=None, num_splits=0, fused_tree_mask=True):
        self.wl = wl
        self.fused_tree_mask = fused_tree_mask
        self.device = torch.device(device)
        dev = self.device
        self.B, self.H = wl.B, wl.H
        self.total_q = wl.total_q
        self.max_q_len = int(wl.q_len.max())
        self.max_kv_len = int(wl.kv_len.max())
        mip = ddt.ddt_mask_indptr(torch.from_numpy(wl.qo_indptr.astype(np.int32)),
                                  torch.from_numpy(wl.prefix_len.astype(np.int32)))
        self.mask_indptr_host = mip
        self.total_words = int(mip[-1])
        argmax = wl.argmax_random if target_argmax is None else target_argmax
        T, W = self.total_q, wl.max_depth + 1
        # Per-step inputs in one device buffer and the step's results in another,
        # so that a host round trip is one copy each way.
        self.inputs = _Arena([
            ("topk_logp", torch.float32, np.ascontiguousarray(wl.topk_logp, np.float32)),
            ("topk_ids", torch.int32, wl.topk_ids), ("root_id", torch.int32, wl.root_id),
            ("budget", torch.int32, wl.budget), ("qo_indptr", torch.int32, wl.qo_indptr),
            ("kv_indptr", torch.int32, wl.kv_indptr), ("kv_indices", torch.int32, wl.kv_indices),
            ("prefix_len", torch.int32, wl.prefix_len), ("mask_indptr", torch.int32, mip.numpy()),
            ("target_argmax", torch.int32, argmax),
            ("q", torch.bfloat16, wl.q)], dev)
        for name, t in self.inputs.views.items():
            setattr(self, name, t)
        # The accept results come first: they are what a host reads back every
        # step (results_bytes from the start of the buffer); the attention output
        # and its lse follow, for a caller that wants them on the host too.
        self.outputs = _Arena([
            ("accept_len", torch.int32, (self.B,)), ("accepted_nodes", torch.int32, (self.B, W)),
            ("commit_tokens", torch.int32, (self.B, W)), ("bonus", torch.int32, (self.B,)),
            ("new_len", torch.int32, (self.B,)),
            ("out", torch.float32, (T, self.H, ddt.DL)), ("lse", torch.float32, (T, self.H))], dev)
        for name, t in self.outputs.views.items():
            setattr(self, name, t)
        self.results_bytes = self.outputs.offsets["out"]
        self.kv_pool = _bf16(wl.kv_pool, dev)  # the resident cache, not a per-step input
        self.node_token = torch.empty(T, dtype=torch.int32, device=dev)
        self.parent = torch.empty(T, dtype=torch.int32, device=dev)
        self.depth = torch.empty(T, dtype=torch.int32, device=dev)
        self.mask = torch.empty(self.total_words, dtype=torch.int32, device=dev)

        self.num_splits = num_splits or ddt.ddt_verify_attn_num_splits(
            self.B, self.H, self.max_q_len, self.max_kv_len)
        # what the attention launches: the requested count rounded to whole kv tiles
        self.launched_splits = ddt.ddt_verify_attn_launched_splits(self.max_kv_len, self.num_splits)
        nbytes = ddt.ddt_verify_attn_workspace_size(T, self.H, self.num_splits)
        self.workspace = (torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None)

    # -- stages -------------------------------------------------------------
    def build_tree(self, stream=None):
        ddt.ddt_build_tree(self.topk_logp, self.topk_ids, self.root_id, self.budget,
                           self.qo_indptr, self.node_token, self.parent, self.depth, stream)

    def compile_visibility(self, stream=None):
        ddt.ddt_compile_visibility(self.parent, self.qo_indptr, self.prefix_len, self.mask_indptr,
                                   self.mask, stream)

    def build_chain_visibility(self, stream=None):
        """Replaces the tree by a chain, parent[i] = i - 1 (depth i) within each
        request, and writes its mask, which is causal over the request's q_len
        new tokens (ddt_build_chain_visibility, one launch).  Engine page, "The
        Core Design Problem: A Unified Forward Pass": prefill, decode and tree
        verify are one forward that differs only in its mask, so verify_attn
        after it is a prefill chunk after the prefix."""
        ddt.ddt_build_chain_visibility(self.qo_indptr, self.prefix_len, self.mask_indptr,
                                       self.parent, self.depth, self.mask, stream)

    def run_prefill(self, stream=None):
        """A prefill chunk as one C call (ddt_prefill_step): chain + causal
        mask, then the attention."""
        ddt.ddt_prefill_step(self.step_args(), stream)

    def build_tree_visibility(self, stream=None):
        ddt.ddt_build_tree_visibility(self.topk_logp, self.topk_ids, self.root_id, self.budget,
                                      self.qo_indptr, self.prefix_len, self.mask_indptr,
                                      self.node_token, self.parent, self.depth, self.mask, stream)

    def verify_attn(self, stream=None):
        ddt.ddt_verify_attn(self.q, self.kv_pool, self.kv_indices, self.kv_indptr, self.qo_indptr,
                            self.mask, self.mask_indptr, self.wl.scale, self.out, self.lse,
                            max_q_len=self.max_q_len, max_kv_len=self.max_kv_len,
                            num_splits=self.num_splits, workspace=self.workspace, stream=stream)

    def accept(self, stream=None):
        ddt.ddt_accept(self.node_token, self.parent, self.qo_indptr, self.target_argmax,
                       self.wl.max_depth, self.accept_len, self.accepted_nodes,
                       self.commit_tokens, self.bonus, stream)

    def commit_kv(self, stream=None):
        """The step after accept: the accepted latents move to the positions after
        the prefix, in place in kv_pool; new_len = prefix + accept_len."""
        ddt.ddt_commit_kv(self.kv_pool, self.kv_indices, self.kv_indptr, self.qo_indptr,
                          self.accept_len, self.accepted_nodes, self.wl.max_depth, self.new_len,
                          stream)

    def step_args(self, commit_kv=False):
        """The step's buffers as one ddt_step_args (for ddt_verify_step and StepGraph)."""
        p = lambda t: None if t is None else t.data_ptr()  # noqa: E731
        a = ddt.StepArgs()
        a.topk_logp, a.topk_ids, a.root_id, a.budget = (p(self.topk_logp), p(self.topk_ids),
                                                        p(self.root_id), p(self.budget))
        a.max_depth, a.topk = self.wl.max_depth, self.wl.K
        a.batch, a.total_q, a.max_q_len, a.max_kv_len = self.B, self.total_q, self.max_q_len, self.max_kv_len
        a.total_mask_words = self.total_words
        a.qo_indptr, a.kv_indptr = p(self.qo_indptr), p(self.kv_indptr)
        a.prefix_len, a.mask_indptr = p(self.prefix_len), p(self.mask_indptr)
        a.q, a.kv_pool, a.pool_rows, a.kv_indices = (p(self.q), p(self.kv_pool), self.kv_pool.shape[0],
                                                     p(self.kv_indices))
        a.num_heads, a.scale, a.num_splits = self.H, self.wl.scale, self.num_splits
        a.workspace = p(self.workspace)
        a.workspace_bytes = 0 if self.workspace is None else self.workspace.numel()
        a.target_argmax = p(self.target_argmax)
        a.node_token, a.parent, a.depth, a.mask = p(self.node_token), p(self.parent), p(self.depth), p(self.mask)
        a.out, a.lse = p(self.out), p(self.lse)
        a.accept_len, a.accepted_nodes = p(self.accept_len), p(self.accepted_nodes)
        a.commit_tokens, a.bonus = p(self.commit_tokens), p(self.bonus)
        a.commit_kv, a.new_len = int(bool(commit_kv)), p(self.new_len)
        return a

    def run_one_call(self, stream=None, commit_kv=False):
        """The step as a single C call (ddt_verify_step)."""
        ddt.ddt_verify_step(self.step_args(commit_kv), stream)

    def step_graph(self, commit_kv=False, host_io=None):
        """A library-owned CUDA graph of the step (ddt_step_graph_*).  host_io =
        (h_in, h_out), pinned host buffers: the graph then copies h_in into the
        inputs before the step and the first len(h_out) bytes of the outputs
        into h_out after it (ddt_step_graph_create_io).  h_out of results_bytes
        brings back the accept results alone; of the whole output buffer, the
        attention output and lse as well."""
        io = None
        if host_io is not None:
            io = (host_io[0], self.inputs.buf, host_io[1], self.outputs.buf)
        return ddt.StepGraph(self.step_args(commit_kv), keep_alive=(self,), io=io)

    @property
    def launches_per_step(self):
        """Kernels one run() or run_one_call() launches: tree + mask (two launches
        for run() with fused_tree_mask=False), attention partial (+ combine when
        it splits), accept."""
        attn = 2 if self.launched_splits > 1 else 1
        return (1 if self.fused_tree_mask else 2) + attn + 1

    def run(self, stream=None):
        if self.fused_tree_mask:
            self.build_tree_visibility(stream)
        else:
            self.build_tree(stream)
            self.compile_visibility(stream)
        self.verify_attn(stream)
        self.accept(stream)

    def check_device_errors(self):
        st, bits = ddt.ddt_get_error()
        if st != 0:
            raise ddt.DDTError("device check", st, f"bits=0x{bits:x}")
