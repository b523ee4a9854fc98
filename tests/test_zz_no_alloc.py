"""ddt_verify_attn_noalloc: the verify attention for callers that cannot
allocate device memory (an engine whose memory is all pre-reserved by its own
pool, a plain C host without an allocator, a decode loop that must not risk
the device-wide synchronisation a cudaMalloc can cause).  Its split scratch is
a fixed array inside libddt.so.  Checked through the C ABI against
ddt_verify_attn (caller workspace) on two calls in a row, so the second call
runs on scratch the first one left behind.
"""
import pytest
import torch

from tree_speculative_decoding_gb300 import workloads

pytestmark = pytest.mark.gpu

MAX_TOL = 1e-2
MEAN_TOL = 2e-3


@pytest.fixture(scope="module")
def step():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tree_speculative_decoding_gb300 import _build
    _build.build()
    from tree_speculative_decoding_gb300.pipeline import VerifyStep
    # one request, prefix 2048, budget 32, 64 heads: the library splits the kv range
    wl = workloads.make_workload("noalloc", 0xA110C, 1, 64, [2048], [32], 8, 32768, 3.0)
    st = VerifyStep(wl, "cuda:0")
    st.run()
    torch.cuda.synchronize()
    st.check_device_errors()
    assert st.num_splits > 1
    return st


def _close(got, ref):
    diff = (got.double() - ref.double()).abs()
    assert diff.max().item() <= MAX_TOL * ref.abs().max().item()
    assert diff.sum().item() / ref.abs().sum().item() <= MEAN_TOL


def test_noalloc_matches_workspace_entry_point_twice(step):
    from tree_speculative_decoding_gb300 import ddt
    ref_out, ref_lse = step.out.clone(), step.lse.clone()
    # the explicit count splits here too, so the scratch is used
    assert ddt.ddt_verify_attn_noalloc_splits(1, step.H, step.total_q, step.max_q_len,
                                              step.max_kv_len, step.num_splits) > 1
    for call in range(2):
        out = torch.full_like(step.out, float("nan"))
        lse = torch.full_like(step.lse, float("nan"))
        ddt.ddt_verify_attn_noalloc(step.q, step.kv_pool, step.kv_indices, step.kv_indptr,
                                    step.qo_indptr, step.mask, step.mask_indptr, step.wl.scale,
                                    out, lse, max_q_len=step.max_q_len,
                                    max_kv_len=step.max_kv_len, num_splits=step.num_splits)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all() and torch.isfinite(lse).all(), f"call {call}"
        _close(out, ref_out)
        _close(lse, ref_lse)
    st, bits = ddt.ddt_get_error()
    assert st == 0, hex(bits)


def test_noalloc_rejects_scratch_beyond_its_capacity(step):
    from tree_speculative_decoding_gb300 import ddt
    need = ddt.ddt_verify_attn_workspace_size(step.total_q, step.H, 16)
    assert need > ddt.NOALLOC_SCRATCH_BYTES
    out = torch.zeros_like(step.out)
    with pytest.raises(ddt.DDTError) as e:
        ddt.ddt_verify_attn_noalloc(step.q, step.kv_pool, step.kv_indices, step.kv_indptr,
                                    step.qo_indptr, step.mask, step.mask_indptr, step.wl.scale,
                                    out, None, max_q_len=step.max_q_len,
                                    max_kv_len=step.max_kv_len, num_splits=16)
    assert e.value.status == 3            # DDT_ERR_WORKSPACE, nothing launched
    assert bool((out == 0).all())


def test_noalloc_own_split_choice_fits_its_scratch():
    # one request, prefix 131072, budget 64, 64 heads (4160 rows): the split
    # count the workspace entry point picks needs more than the fixed scratch
    # for any SM count from 132 to 160, so the allocation-free call must pick a
    # smaller count that fits, and here that count still splits the kv range
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tree_speculative_decoding_gb300 import ddt
    from tree_speculative_decoding_gb300.pipeline import VerifyStep
    wl = workloads.preset("long_p131072_b64_h64")
    st = VerifyStep(wl, "cuda:0")
    st.run()
    torch.cuda.synchronize()
    st.check_device_errors()
    assert ddt.ddt_verify_attn_workspace_size(st.total_q, st.H, st.num_splits) > \
        ddt.NOALLOC_SCRATCH_BYTES
    n = ddt.ddt_verify_attn_noalloc_splits(1, st.H, st.total_q, st.max_q_len, st.max_kv_len, 0)
    assert 1 < n < st.launched_splits
    assert ddt.ddt_verify_attn_workspace_size(st.total_q, st.H, n) <= ddt.NOALLOC_SCRATCH_BYTES
    for call in range(2):  # twice in a row, the second on what the first left behind
        out = torch.full_like(st.out, float("nan"))
        lse = torch.full_like(st.lse, float("nan"))
        ddt.ddt_verify_attn_noalloc(st.q, st.kv_pool, st.kv_indices, st.kv_indptr, st.qo_indptr,
                                    st.mask, st.mask_indptr, st.wl.scale, out, lse,
                                    max_q_len=st.max_q_len, max_kv_len=st.max_kv_len, num_splits=0)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all() and torch.isfinite(lse).all(), f"call {call}"
        _close(out, st.out)
        _close(lse, st.lse)
    status, bits = ddt.ddt_get_error()
    assert status == 0, hex(bits)


def test_noalloc_wrapper_checks_shapes(step):
    # the C ABI cannot see tensor shapes: the binding refuses what would make
    # the kernels read or write past a buffer, before any call
    from tree_speculative_decoding_gb300 import ddt
    q512 = step.q[..., :512].contiguous()
    with pytest.raises(ValueError):
        ddt.ddt_verify_attn_noalloc(q512, step.kv_pool, step.kv_indices, step.kv_indptr,
                                    step.qo_indptr, step.mask, step.mask_indptr, step.wl.scale,
                                    step.out, None)
    with pytest.raises(ValueError):
        ddt.ddt_verify_attn_noalloc(step.q, step.kv_pool, step.kv_indices, step.kv_indptr,
                                    step.qo_indptr, step.mask, step.mask_indptr, step.wl.scale,
                                    step.out[:-1], None)
    with pytest.raises(ValueError):
        ddt.ddt_verify_attn_noalloc(step.q, step.kv_pool, step.kv_indices.long(), step.kv_indptr,
                                    step.qo_indptr, step.mask, step.mask_indptr, step.wl.scale,
                                    step.out, None)
