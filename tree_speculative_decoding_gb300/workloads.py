"""Seeded synthetic inputs for the DDTree verify step.

This module only draws inputs.  It holds none of the method's arithmetic (no
tree building, no masks, no attention, no accept walk), so both the CUDA path
and the CPU oracle can consume what it produces.

Random numbers come from one counter-based generator written from its
published definition: SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) -- the state advances by the
golden-ratio increment 0x9E3779B97F4A7C15 and each output is the state passed
through the variant-13 finaliser.  Output k of stream s under seed x is
``finalise(key(x, s) + (k + 1) * 0x9E3779B97F4A7C15)``, so any element can be
drawn without drawing the ones before it, and results do not depend on the
numpy version.

Workload shapes follow the five verify-step workloads of the target model's
verify call (absorbed MLA, 576-wide latent rows: 512 latent + 64 rope), with
the tiny one matching the shapes log printed on "The 30-Column Mask" page
(q=(9,8,576), prefix 21, scale 0.14468).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_STREAM_MUL = np.uint64(0xD1B54A32D192ED03)

DL, DR, D = 512, 64, 576
MAX_DEPTH = 7          # block size 8 minus the anchor: depth <= 7
DEFAULT_SCALE = 0.14468

# stream tags: one independent stream per drawn quantity
_S_PREFIX, _S_BUDGET, _S_PERM, _S_POOL, _S_HEAVY, _S_Q = 1, 2, 3, 4, 5, 6
_S_LOGITS, _S_ROOT, _S_ARGMAX, _S_COIN = 7, 8, 9, 10


def _finalise(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        x = np.array([np.uint64(seed & 0xFFFFFFFFFFFFFFFF) ^ (np.uint64(stream) * _STREAM_MUL)],
                     dtype=np.uint64)
        return _finalise(x)[0]


_CHUNK = 1 << 18   # work in small pieces: large temporaries are slow to fault in


def _u64_into(out: np.ndarray, k: np.uint64, start: int) -> None:
    n = out.shape[0]
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        idx = np.arange(start + lo + 1, start + hi + 1, dtype=np.uint64)
        with np.errstate(over="ignore"):
            out[lo:hi] = _finalise(k + idx * GOLDEN)


def u64(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs start .. start+n-1 of SplitMix64 stream `stream` under `seed`."""
    out = np.empty(n, np.uint64)
    _u64_into(out, _key(seed, stream), start)
    return out


def uniform(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """Doubles in [0, 1): top 53 bits of each output."""
    return (u64(seed, stream, n, start) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def integers(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    """Integers uniform in [lo, hi] (inclusive), via floor(u * span)."""
    span = hi - lo + 1
    return (lo + np.floor(uniform(seed, stream, n) * span)).astype(np.int64)


def normal(seed: int, stream: int, n: int, dtype=np.float64) -> np.ndarray:
    """Standard normals by Box-Muller on consecutive output pairs: output pair
    (2k, 2k+1) gives r*cos(a), r*sin(a) with r = sqrt(-2 ln u1), a = 2 pi u2."""
    out = np.empty(n, dtype)
    k = _key(seed, stream)
    pairs = (n + 1) // 2
    x = np.empty(2 * min(_CHUNK, max(pairs, 1)), np.uint64)
    for p0 in range(0, pairs, _CHUNK):
        m = min(_CHUNK, pairs - p0)
        xs = x[: 2 * m]
        _u64_into(xs, k, 2 * p0)
        u1 = ((xs[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
        u2 = (xs[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)          # [0, 1)
        r = np.sqrt(-2.0 * np.log(u1))
        a = 2.0 * math.pi * u2
        lo = 2 * p0
        hi = min(n, lo + 2 * m)
        z = np.empty(2 * m, np.float64)
        z[0::2] = r * np.cos(a)
        z[1::2] = r * np.sin(a)
        out[lo:hi] = z[: hi - lo]
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 round-to-nearest-even; returns the bf16 bit patterns (uint16)."""
    f = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.empty(f.shape[0], np.uint16)
    for lo in range(0, f.shape[0], _CHUNK):
        u = f[lo:lo + _CHUNK].view(np.uint32)
        bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
        out[lo:lo + _CHUNK] = ((u.astype(np.uint64) + bias) >> np.uint64(16)).astype(np.uint16)
    return out.reshape(np.shape(x))


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    B: int
    H: int
    scale: float
    K: int                      # top-k per draft depth
    max_depth: int
    vocab: int
    prefix_len: np.ndarray      # int32 [B]
    budget: np.ndarray          # int32 [B]
    qo_indptr: np.ndarray       # int32 [B+1], q_len = budget + 1
    kv_indptr: np.ndarray       # int32 [B+1], kv columns = prefix + q_len
    kv_indices: np.ndarray      # int32 [sum N]: prefix slots, then tree-node slots
    pool_rows: int
    kv_pool: np.ndarray         # uint16 bf16 bits [pool_rows, 576]
    q: np.ndarray               # uint16 bf16 bits [sum T, H, 576]
    topk_logp: np.ndarray       # float32 [B, max_depth, K], non-increasing along K
    topk_ids: np.ndarray        # int32 [B, max_depth, K]
    root_id: np.ndarray         # int32 [B]
    argmax_random: np.ndarray   # int32 [sum T]: uniform target tokens
    argmax_coin: np.ndarray     # uint8 [sum T]: 1 where the target should follow the best child
    p_match: float

    @property
    def total_q(self) -> int:
        return int(self.qo_indptr[-1])

    @property
    def q_len(self) -> np.ndarray:
        return np.diff(self.qo_indptr).astype(np.int32)

    @property
    def kv_len(self) -> np.ndarray:
        return np.diff(self.kv_indptr).astype(np.int32)


def make_workload(name: str, seed: int, B: int, H: int, prefix_len, budget, K: int,
                  vocab: int, logit_sigma: float, pool_rows: int | None = None,
                  heavy_frac: float = 0.0, heavy_mul: float = 8.0, p_match: float = 0.0,
                  scale: float = DEFAULT_SCALE, max_depth: int = MAX_DEPTH,
                  fill_pool: bool = True) -> Workload:
    prefix_len = np.asarray(prefix_len, dtype=np.int64).reshape(B)
    budget = np.asarray(budget, dtype=np.int64).reshape(B)
    T = budget + 1
    N = prefix_len + T
    qo_indptr = np.concatenate([[0], np.cumsum(T)]).astype(np.int32)
    kv_indptr = np.concatenate([[0], np.cumsum(N)]).astype(np.int32)
    total_kv = int(kv_indptr[-1])
    if pool_rows is None:
        pool_rows = total_kv
    if total_kv > pool_rows:
        raise ValueError(f"pool of {pool_rows} rows cannot hold {total_kv} kv rows")

    # paged slots: a seeded permutation of the pool, cut into disjoint chunks
    keys = u64(seed, _S_PERM, pool_rows)
    perm = np.argsort(keys, kind="stable")
    kv_indices = perm[:total_kv].astype(np.int32)

    # latent KV pool, N(0,1) -> bf16; optionally 1% of each request's rows x8
    if fill_pool:
        pool = normal(seed, _S_POOL, pool_rows * D, np.float32).reshape(pool_rows, D)
    else:
        pool = np.zeros((pool_rows, D), np.float32)
    if heavy_frac > 0.0:
        u = uniform(seed, _S_HEAVY, total_kv)
        heavy_slots = kv_indices[u < heavy_frac]
        pool[heavy_slots] *= np.float32(heavy_mul)
    kv_pool = to_bf16_bits(pool)
    del pool

    total_q = int(qo_indptr[-1])
    q = to_bf16_bits(normal(seed, _S_Q, total_q * H * D, np.float32)).reshape(total_q, H, D)

    # drafter output: per depth, log-softmax of N(0, sigma) logits over the vocab,
    # then the top K by value (ties to the lower token id)
    logits = normal(seed, _S_LOGITS, B * max_depth * vocab).reshape(B, max_depth, vocab) * logit_sigma
    mx = logits.max(axis=-1, keepdims=True)
    logp = logits - (mx + np.log(np.exp(logits - mx).sum(axis=-1, keepdims=True)))
    order = np.argsort(-logp, axis=-1, kind="stable")[..., :K]
    topk_ids = order.astype(np.int32)
    topk_logp = np.take_along_axis(logp, order, axis=-1).astype(np.float32)

    root_id = integers(seed, _S_ROOT, B, 0, vocab - 1).astype(np.int32)
    argmax_random = integers(seed, _S_ARGMAX, total_q, 0, vocab - 1).astype(np.int32)
    argmax_coin = (uniform(seed, _S_COIN, total_q) < p_match).astype(np.uint8)

    return Workload(name=name, seed=seed, B=B, H=H, scale=float(scale), K=K,
                    max_depth=max_depth, vocab=vocab,
                    prefix_len=prefix_len.astype(np.int32), budget=budget.astype(np.int32),
                    qo_indptr=qo_indptr, kv_indptr=kv_indptr, kv_indices=kv_indices,
                    pool_rows=pool_rows, kv_pool=kv_pool, q=q, topk_logp=topk_logp,
                    topk_ids=topk_ids, root_id=root_id, argmax_random=argmax_random,
                    argmax_coin=argmax_coin, p_match=p_match)


# The five verify-step workloads.  Seeds are 0xDD7E0000 + k.
PRESETS = {
    # shapes log of the custom verify kernel: bs 1, prefix 21, q_len 9, 8 heads
    "tiny_p21_b8_h8": dict(k=1, B=1, H=8, prefix=("fixed", 21), budget=("fixed", 8), K=4,
                           vocab=512, sigma=2.0, pool_rows=256),
    # one request, 64 heads, prefix 4096, budget 32
    "single_p4096_b32_h64": dict(k=2, B=1, H=64, prefix=("fixed", 4096), budget=("fixed", 32),
                                 K=8, vocab=32768, sigma=3.0, pool_rows=65536),
    # ragged batch of 8, prefixes U[1024, 16384], budget 32, 64 heads
    "ragged_bs8_b32_h64": dict(k=3, B=8, H=64, prefix=("uniform", 1024, 16384),
                               budget=("fixed", 32), K=8, vocab=32768, sigma=3.0,
                               pool_rows=200000),
    # long context, split-KV path: prefix 131072, budget 64, topk 16, 1% rows x8
    "long_p131072_b64_h64": dict(k=4, B=1, H=64, prefix=("fixed", 131072), budget=("fixed", 64),
                                 K=16, vocab=32768, sigma=3.0, pool_rows=262144,
                                 heavy_frac=0.01),
    # high concurrency: 32 requests, prefixes U[2048, 8192], budget 16 or 32, 16 heads
    "mixed_bs32_b16or32_h16": dict(k=5, B=32, H=16, prefix=("uniform", 2048, 8192),
                                   budget=("choice", 16, 32), K=8, vocab=32768, sigma=3.0,
                                   pool_rows=300000, p_match=0.5),
}


# The degenerate shapes of the same path, one request after a prefix of 4096
# at 64 heads: the autoregressive step (budget 0, q_len 1) and a prefill chunk
# of 128 new tokens (budget 127, whose tree the caller replaces by a causal
# chain).  Seeds continue the series above.
DEGENERATE = {
    "ar_p4096_b0_h64": dict(k=6, B=1, H=64, prefix=("fixed", 4096), budget=("fixed", 0), K=8,
                            vocab=32768, sigma=3.0, pool_rows=65536),
    "prefill_p4096_t128_h64": dict(k=7, B=1, H=64, prefix=("fixed", 4096),
                                   budget=("fixed", 127), K=8, vocab=32768, sigma=3.0,
                                   pool_rows=65536),
}


def preset_seed(name: str) -> int:
    return 0xDD7E0000 + {**PRESETS, **DEGENERATE}[name]["k"]


def preset(name: str, fill_pool: bool = True) -> Workload:
    p = {**PRESETS, **DEGENERATE}[name]
    seed = preset_seed(name)
    B = p["B"]
    kind = p["prefix"][0]
    if kind == "fixed":
        prefix = np.full(B, p["prefix"][1], np.int64)
    else:
        prefix = integers(seed, _S_PREFIX, B, p["prefix"][1], p["prefix"][2])
    kind = p["budget"][0]
    if kind == "fixed":
        budget = np.full(B, p["budget"][1], np.int64)
    else:
        pick = uniform(seed, _S_BUDGET, B) < 0.5
        budget = np.where(pick, p["budget"][1], p["budget"][2]).astype(np.int64)
    return make_workload(name, seed, B, p["H"], prefix, budget, p["K"], p["vocab"], p["sigma"],
                         pool_rows=p["pool_rows"], heavy_frac=p.get("heavy_frac", 0.0),
                         p_match=p.get("p_match", 0.0), fill_pool=fill_pool)
