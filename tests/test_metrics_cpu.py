"""Work and traffic counts used by the bench (host bookkeeping, CPU)."""
import numpy as np

from tree_speculative_decoding_gb300 import metrics


def test_flops_count_visible_pairs():
    # one request, prefix 4, a chain of three nodes (depths 0, 1, 2), one head:
    # node i sees the prefix and i + 1 tree columns -> 3 * 4 + (1 + 2 + 3) pairs
    f = metrics.attn_flops(np.array([4]), np.array([0, 1, 2]), np.array([0, 3]), 1)
    assert f == (12 + 6) * 2 * (576 + 512)
    # heads multiply
    assert metrics.attn_flops(np.array([4]), np.array([0, 1, 2]), np.array([0, 3]), 8) == 8 * f


def test_bytes_of_the_headline_shape():
    # one request, prefix 4096, 33 nodes, 64 heads: the KV stream and the total
    kv_indptr = np.array([0, 4096 + 33])
    assert metrics.kv_bytes(kv_indptr) == 4129 * 1152 == 4756608
    words = 33 * ((4096 + 33 + 31) // 32)
    total = metrics.algorithmic_bytes(kv_indptr, 33, 64, words)
    assert total == 4756608 + 2112 * 1152 + 2112 * 2048 + 4 * 4129 + 4 * words
    assert 11.5e6 < total < 11.6e6
