"""Work and traffic counts for one verify-attention call (bookkeeping for
throughput and roofline reporting; no part of the computation itself)."""
from __future__ import annotations

import numpy as np

DL, D = 512, 576


def attn_flops(prefix_len, depth, qo_indptr, H) -> float:
    """Algorithmic FLOPs of one verify-attention call: 2*(576+512) per visible
    (query-head, kv) pair; a node at depth d sees the prefix plus d+1 tree
    columns.  Counts visible pairs only (masked columns, softmax and the
    split combine are not counted).  `depth` comes from whichever tree the
    caller built."""
    total = 0
    for b in range(len(prefix_len)):
        lo, hi = int(qo_indptr[b]), int(qo_indptr[b + 1])
        T = hi - lo
        total += T * int(prefix_len[b]) + int(np.sum(np.asarray(depth[lo:hi]) + 1))
    return float(total) * H * 2 * (D + DL)


def kv_bytes(kv_indptr) -> float:
    """Each KV row (576 bf16 = 1152 B) read once per call."""
    return float(kv_indptr[-1]) * D * 2


def algorithmic_bytes(kv_indptr, total_q, H, mask_words) -> float:
    """All bytes one verify-attention call must move at least once: the KV rows,
    q (576 bf16 per row), the fp32 output (512 per row), the kv indices and the
    visibility mask words (4 B each)."""
    rows = float(total_q) * H
    return kv_bytes(kv_indptr) + rows * D * 2 + rows * DL * 4 + 4.0 * float(kv_indptr[-1]) + 4.0 * mask_words
