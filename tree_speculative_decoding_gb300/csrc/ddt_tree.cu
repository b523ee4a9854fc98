// ddt_tree.cu -- the three small stages of the verify step: best-first tree
// build, visibility-mask compile and greedy accept.  One warp per request for
// the sequential walks, one thread per mask word for the mask.
//
// Page: "The DDTree CUDA Graph Fix: Unlocking Speculative Decoding at 109 tok/s
// on PCIe Blackwell", section "The DDTree Architecture: Confirming
// Multiple-Path Evaluation" (heap expansion, ancestor-plus-prefix visibility,
// follow-the-argmax acceptance with one bonus token).
#include <cuda_runtime.h>
#include <stdint.h>

#include "ddt_internal.cuh"

namespace ddt {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int SLOTS = 4;  // frontier slots per lane: 32 x 4 = 128 >= budget + 1

// Candidate key: larger key pops first.
//   bits 63..32  score mapped to an order-preserving uint32 (higher score first)
//   bits 31..29  7 - depth                    (shallower first on equal score)
//   bits 27..0   0x0FFFFFFF - rank path       (lexicographically smaller first)
// The rank path packs the sibling rank at depth k into bits 27-4(k-1)..24-4(k-1),
// so equal-depth paths compare lexicographically as integers.  Keys of distinct
// nodes are distinct, and 0 marks an empty slot (a real key is never 0: its
// high word is at least 0x007FFFFF).
__device__ __forceinline__ uint32_t order_score(float f) {
    f = f + 0.0f;  // -0 -> +0 so that equal scores give equal keys
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unorder_score(uint32_t u) {
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}
__device__ __forceinline__ uint64_t make_key(float score, int depth, uint32_t path) {
    return ((uint64_t)order_score(score) << 32) | ((uint64_t)(7 - depth) << 29) |
           (uint64_t)(0x0FFFFFFFu - path);
}
__device__ __forceinline__ int key_depth(uint64_t k) { return 7 - (int)((k >> 29) & 7u); }
__device__ __forceinline__ uint32_t key_path(uint64_t k) {
    return 0x0FFFFFFFu - (uint32_t)(k & 0x0FFFFFFFu);
}
__device__ __forceinline__ int path_rank(uint32_t path, int depth) {  // rank at `depth`
    return (int)((path >> (28 - 4 * depth)) & 0xFu);
}

// One warp per request.  The frontier (candidates not yet popped) lives in
// registers, SLOTS entries per lane, with the request's top-k log-probs and ids
// staged in shared memory.  Each pop is a warp-wide max over 64-bit keys.  To
// keep the sequential chain short, every lane prepares, before the reduction,
// what its best candidate would produce if it won (its token, its next
// sibling's key, its best child's key); the winner then refills its own slot
// with the child (or the sibling) and hands the remaining candidate to lane
// n % 32, which always has a free slot: lane k receives candidates only at pops
// n = k, k+32, k+64, k+96 (n <= budget <= 127), at most 4 including the seed.
// Builds request b's tree in shared memory (out_* [0, nb]) with one warp and
// returns 0, or the DDT_DEVERR_* bit to latch (the outputs are then unset).
// Reads only caller inputs, so it may run before the kernel's pdl_wait().
__device__ unsigned tree_warp(const float *__restrict__ topk_logp,
                              const int32_t *__restrict__ topk_ids, int b, int base, int end,
                              int nb, int rid, int max_depth, int K, float *lp, int32_t *ids,
                              int32_t *out_tok, int32_t *out_par, int32_t *out_dep) {
    const int lane = threadIdx.x & 31;
    const int total = max_depth * K;
    const float *lpb = topk_logp + (size_t)b * total;
    const int32_t *idb = topk_ids + (size_t)b * total;
    for (int e = lane; e < total; e += 32) {
        lp[e] = lpb[e];
        ids[e] = idb[e];
    }
    __syncwarp();
    bool sorted_ok = true;
    for (int e = lane; e < total; e += 32) {
        const float v = lp[e];
        if ((e % K) > 0 ? !(v <= lp[e - 1]) : (v != v)) sorted_ok = false;  // also rejects NaN
    }
    if (__any_sync(FULL, !sorted_ok)) return DDT_DEVERR_TOPK_ORDER;
    if (nb < 0 || nb > DDT_MAX_Q_LEN - 1 || end - base != nb + 1) return DDT_DEVERR_QO_INDPTR;
    if (lane == 0) {
        out_tok[0] = rid;
        out_par[0] = -1;
        out_dep[0] = 0;
    }
    if (nb == 0) {
        __syncwarp();
        return 0;
    }
    uint64_t key[SLOTS];
    float pscore[SLOTS];  // score of the candidate's parent (for its next sibling)
    int pout[SLOTS];      // output index of the candidate's parent
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) { key[s] = 0; pscore[s] = 0.f; pout[s] = 0; }
    if (lane == 0) key[0] = make_key(0.0f + lp[0], 1, 0u);  // seed: rank-0 child of the root

    // this lane's best candidate and what it yields if popped
    uint64_t best = 0, sib = 0, child = 0;
    int bs = 0, bd = 0, btok = 0, bpout = 0;
    float bpscore = 0.f, bscore = 0.f;
    auto prepare = [&]() {
        best = 0;
        bs = 0;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s)
            if (key[s] > best) { best = key[s]; bs = s; }
        sib = 0;
        child = 0;
        if (best != 0) {
#pragma unroll
            for (int s = 0; s < SLOTS; ++s)
                if (s == bs) { bpout = pout[s]; bpscore = pscore[s]; }
            bd = key_depth(best);
            const uint32_t path = key_path(best);
            const int r = path_rank(path, bd);
            bscore = unorder_score((uint32_t)(best >> 32));
            btok = ids[(bd - 1) * K + r];
            if (r + 1 < K)
                sib = make_key(bpscore + lp[(bd - 1) * K + r + 1], bd, path + (1u << (28 - 4 * bd)));
            if (bd < max_depth) child = make_key(bscore + lp[bd * K + 0], bd + 1, path);
        }
    };
    prepare();

    for (int n = 1; n <= nb; ++n) {
        const uint32_t hi = (uint32_t)(best >> 32);
        const uint32_t mhi = __reduce_max_sync(FULL, hi);
        if (mhi == 0u) return DDT_DEVERR_EXHAUSTED;  // frontier empty: budget exceeds the implicit tree
        unsigned who = __ballot_sync(FULL, hi == mhi);
        if (__popc(who) > 1) {  // equal scores: the rest of the key decides
            const uint32_t lo = (uint32_t)best;
            const uint32_t mlo = __reduce_max_sync(FULL, hi == mhi ? lo : 0u);
            who = __ballot_sync(FULL, hi == mhi && lo == mlo);
        }
        const int wl = __ffs(who) - 1;
        bool extra = false;  // the winner's sibling, when its child took the slot
        if (lane == wl) {  // outputs go to shared memory; one coalesced write at the end
            out_tok[n] = btok;
            out_par[n] = bpout;
            out_dep[n] = bd;
            extra = child != 0 && sib != 0;
#pragma unroll
            for (int s = 0; s < SLOTS; ++s)
                if (s == bs) {
                    if (child != 0) { key[s] = child; pscore[s] = bscore; pout[s] = n; }
                    else key[s] = sib;  // same parent: pscore / pout stay
                }
        }
        if (n == nb) break;
        if (__shfl_sync(FULL, extra ? 1 : 0, wl)) {
            const uint32_t xhi = __shfl_sync(FULL, (uint32_t)(sib >> 32), wl);
            const uint32_t xlo = __shfl_sync(FULL, (uint32_t)sib, wl);
            const float xps = __shfl_sync(FULL, bpscore, wl);
            const int xpo = __shfl_sync(FULL, bpout, wl);
            if (lane == (n & 31)) {
                int free_slot = 0;
#pragma unroll
                for (int s = SLOTS - 1; s >= 0; --s)
                    if (key[s] == 0) free_slot = s;
#pragma unroll
                for (int s = 0; s < SLOTS; ++s)
                    if (s == free_slot) {
                        key[s] = ((uint64_t)xhi << 32) | xlo;
                        pscore[s] = xps;
                        pout[s] = xpo;
                    }
            }
        }
        if (lane == wl || lane == (n & 31)) prepare();
    }
    __syncwarp();
    return 0;
}

__global__ void __launch_bounds__(32)
build_tree_kernel(const float *__restrict__ topk_logp, const int32_t *__restrict__ topk_ids,
                  const int32_t *__restrict__ root_id, const int32_t *__restrict__ budget,
                  const int32_t *__restrict__ qo_indptr, int max_depth, int K,
                  int32_t *__restrict__ node_token, int32_t *__restrict__ parent,
                  int32_t *__restrict__ depth, unsigned int *err) {
    __shared__ float lp[DDT_MAX_DEPTH * DDT_MAX_TOPK];
    __shared__ int32_t ids[DDT_MAX_DEPTH * DDT_MAX_TOPK];
    __shared__ int32_t out_tok[DDT_MAX_Q_LEN], out_par[DDT_MAX_Q_LEN], out_dep[DDT_MAX_Q_LEN];
    const int b = blockIdx.x;
    const int lane = threadIdx.x;
    pdl_trigger();
    // caller inputs only until the outputs are written: no wait needed before
    const int base = qo_indptr[b];
    const int end = qo_indptr[b + 1];
    const int nb = budget[b];
    const unsigned e = tree_warp(topk_logp, topk_ids, b, base, end, nb, root_id[b], max_depth, K,
                                 lp, ids, out_tok, out_par, out_dep);
    pdl_wait();  // the previous kernel may still read the tree buffers
    if (e) {
        if (lane == 0) latch(err, e);
        return;
    }
    for (int i = lane; i <= nb; i += 32) {
        node_token[base + i] = out_tok[i];
        parent[base + i] = out_par[i];
        depth[base + i] = out_dep[i];
    }
}

// Mask word k of row i of a request with prefix P and q_len T: prefix columns
// [32k, min(32k+32, P)) and the tree columns P + j for node i and its
// ancestors j (par: the request's parent links).  A broken parent chain
// latches DDT_DEVERR_PARENT and ends the walk.
__device__ __forceinline__ uint32_t mask_word(const int32_t *par, int P, int T, int i, int k,
                                              unsigned int *err) {
    const int c0 = k * 32;
    uint32_t bits = 0u;
    if (c0 < P) {
        const int n = min(32, P - c0);
        bits = (n == 32) ? 0xffffffffu : ((1u << n) - 1u);
    }
    if (c0 + 32 > P && c0 < P + T) {
        int j = i, guard = 0;
        while (j >= 0) {
            const int c = P + j;
            if (c >= c0 && c < c0 + 32) bits |= 1u << (c - c0);
            const int pj = par[j];
            if (pj >= j || ++guard > DDT_MAX_Q_LEN) {  // parents must precede
                if (pj >= 0) latch(err, DDT_DEVERR_PARENT);
                break;
            }
            j = pj;
        }
    }
    return bits;
}

// Tree build and visibility mask in one launch: one CTA per request.  Warp 0
// builds the tree while warps 1-7 write the all-ones prefix words of the mask
// (every word whose 32 columns are prefix columns); after a block barrier all
// eight warps write the remaining words from the tree in shared memory.
constexpr int kTreeVisThreads = 256;
__global__ void __launch_bounds__(kTreeVisThreads)
build_tree_visibility_kernel(const float *__restrict__ topk_logp,
                             const int32_t *__restrict__ topk_ids,
                             const int32_t *__restrict__ root_id,
                             const int32_t *__restrict__ budget,
                             const int32_t *__restrict__ qo_indptr, int max_depth, int K,
                             const int32_t *__restrict__ prefix_len,
                             const int32_t *__restrict__ mask_indptr,
                             int32_t *__restrict__ node_token, int32_t *__restrict__ parent,
                             int32_t *__restrict__ depth, uint32_t *__restrict__ mask,
                             unsigned int *err) {
    __shared__ float lp[DDT_MAX_DEPTH * DDT_MAX_TOPK];
    __shared__ int32_t ids[DDT_MAX_DEPTH * DDT_MAX_TOPK];
    __shared__ int32_t out_tok[DDT_MAX_Q_LEN], out_par[DDT_MAX_Q_LEN], out_dep[DDT_MAX_Q_LEN];
    __shared__ unsigned tree_err;
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    pdl_trigger();
    const int base = qo_indptr[b];
    const int end = qo_indptr[b + 1];
    const int T = end - base;
    const int P = prefix_len[b];
    const int W = (P + T + 31) >> 5;
    const int m0 = mask_indptr[b];
    const bool mask_ok = T >= 1 && T <= DDT_MAX_Q_LEN && P >= 0 && mask_indptr[b + 1] - m0 == T * W;
    const int full = mask_ok ? (P >> 5) : 0;  // leading all-ones words per row
    if (tid < 32) {
        const int nb = budget[b];
        const unsigned e = tree_warp(topk_logp, topk_ids, b, base, end, nb, root_id[b], max_depth,
                                     K, lp, ids, out_tok, out_par, out_dep);
        if (tid == 0) tree_err = e;
    } else {
        pdl_wait();  // the previous kernel may still read the mask
        for (int w = tid - 32; w < T * full; w += kTreeVisThreads - 32) {
            const int i = w / full;
            mask[m0 + i * W + (w - i * full)] = 0xffffffffu;
        }
    }
    __syncthreads();
    if (tid < 32) pdl_wait();  // the previous kernel may still read the tree buffers
    const unsigned e = tree_err;
    if (e) {
        if (tid == 0) latch(err, e);
    } else {
        for (int i = tid; i < T; i += kTreeVisThreads) {
            node_token[base + i] = out_tok[i];
            parent[base + i] = out_par[i];
            depth[base + i] = out_dep[i];
        }
    }
    if (!mask_ok) {
        if (tid == 0) latch(err, DDT_DEVERR_MASK_INDPTR);
        return;
    }
    const int rest = W - full;  // words per row that hold tree columns
    for (int w = tid; w < T * rest; w += kTreeVisThreads) {
        const int i = w / rest;
        const int k = full + (w - i * rest);
        mask[m0 + i * W + k] = e ? 0u : mask_word(out_par, P, T, i, k, err);
    }
}

// A prefill chunk's tree: the chain parent[i] = i - 1, depth[i] = i, and its
// mask, which is the causal one: row i sees columns [0, P + i].  Engine page,
// "The Core Design Problem: A Unified Forward Pass" (prefill, decode and tree
// verify are one forward that differs only in its mask).  One CTA per
// request; no parent walk is needed, each word follows from its row and
// column range alone.
constexpr int kChainThreads = 256;
__global__ void __launch_bounds__(kChainThreads)
build_chain_visibility_kernel(const int32_t *__restrict__ qo_indptr,
                              const int32_t *__restrict__ prefix_len,
                              const int32_t *__restrict__ mask_indptr,
                              int32_t *__restrict__ parent, int32_t *__restrict__ depth,
                              uint32_t *__restrict__ mask, unsigned int *err) {
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    pdl_trigger();
    const int base = qo_indptr[b];
    const int T = qo_indptr[b + 1] - base;
    const int P = prefix_len[b];
    const int W = (P + T + 31) >> 5;
    const int m0 = mask_indptr[b];
    const bool rows_ok = T >= 1 && T <= DDT_MAX_Q_LEN && base >= 0;
    const bool mask_ok = rows_ok && P >= 0 && mask_indptr[b + 1] - m0 == T * W;
    pdl_wait();  // the previous kernel may still read these buffers
    if (!mask_ok) {
        if (tid == 0) latch(err, DDT_DEVERR_MASK_INDPTR);
        if (!rows_ok) return;
    }
    for (int i = tid; i < T; i += kChainThreads) {
        parent[base + i] = i - 1;
        depth[base + i] = i;
    }
    if (!mask_ok) return;
    for (int w = tid; w < T * W; w += kChainThreads) {
        const int i = w / W;
        const int lo = (w - i * W) << 5;  // first column of the word
        const int last = P + i;           // last visible column of row i
        uint32_t bits;
        if (last >= lo + 31) bits = 0xffffffffu;
        else if (last < lo) bits = 0u;
        else bits = (2u << (last - lo)) - 1u;  // columns lo .. last
        mask[m0 + w] = bits;
    }
}

// One thread per mask word (grid-stride).  Word w of request b: row
// i = local / W_b, columns [32k, 32k+32) with k = local % W_b.
__global__ void compile_visibility_kernel(const int32_t *__restrict__ parent,
                                          const int32_t *__restrict__ qo_indptr,
                                          const int32_t *__restrict__ prefix_len,
                                          const int32_t *__restrict__ mask_indptr, int batch,
                                          int total_words, uint32_t *__restrict__ mask,
                                          unsigned int *err) {
    pdl_trigger();
    pdl_wait();  // parent comes from the tree build
    for (int w = blockIdx.x * blockDim.x + threadIdx.x; w < total_words;
         w += gridDim.x * blockDim.x) {
        // request owning word w: last b with mask_indptr[b] <= w
        int lo = 0, hi = batch - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (mask_indptr[mid] <= w) lo = mid; else hi = mid - 1;
        }
        const int b = lo;
        const int T = qo_indptr[b + 1] - qo_indptr[b];
        const int P = prefix_len[b];
        const int N = P + T;
        const int W = (N + 31) >> 5;
        if (T < 1 || T > DDT_MAX_Q_LEN || P < 0 ||
            mask_indptr[b + 1] - mask_indptr[b] != T * W) {
            latch(err, DDT_DEVERR_MASK_INDPTR);
            mask[w] = 0u;
            continue;
        }
        const int local = w - mask_indptr[b];
        const int i = local / W;
        const uint32_t bits = mask_word(parent + qo_indptr[b], P, T, i, local - i * W, err);
        mask[w] = bits;
    }
}

// One warp per request: walk from the root into the child carrying the
// target's argmax; lanes scan the nodes, the lowest matching index wins.  The
// request's argmax row (a caller input) is staged before the wait for the
// tree, its parents and tokens right after it, so the walk itself touches
// shared memory only.
__global__ void __launch_bounds__(32)
accept_kernel(const int32_t *__restrict__ node_token, const int32_t *__restrict__ parent,
              const int32_t *__restrict__ qo_indptr, const int32_t *__restrict__ target_argmax,
              int max_depth, int32_t *__restrict__ accept_len,
              int32_t *__restrict__ accepted_nodes, int32_t *__restrict__ commit_tokens,
              int32_t *__restrict__ bonus, unsigned int *err) {
    __shared__ int32_t s_want[DDT_MAX_Q_LEN], s_par[DDT_MAX_Q_LEN], s_tok[DDT_MAX_Q_LEN];
    const int b = blockIdx.x;
    const int lane = threadIdx.x;
    pdl_trigger();
    const int width = max_depth + 1;
    const int base = qo_indptr[b];
    const int T = qo_indptr[b + 1] - base;
    const bool bad = T < 1 || T > DDT_MAX_Q_LEN;
    if (!bad)
        for (int i = lane; i < T; i += 32) s_want[i] = target_argmax[base + i];
    pdl_wait();  // the tree comes from the tree build
    if (bad) {
        if (lane == 0) latch(err, DDT_DEVERR_QO_INDPTR);
        return;
    }
    for (int i = lane; i < T; i += 32) {
        s_par[i] = parent[base + i];
        s_tok[i] = node_token[base + i];
    }
    __syncwarp();
    int32_t *acc = accepted_nodes + (size_t)b * width;
    int32_t *com = commit_tokens + (size_t)b * width;
    int cur = 0, n = 1;
    int path[DDT_MAX_DEPTH + 1];  // the accepted nodes (the same in every lane)
    path[0] = 0;
    for (;;) {
        const int want = s_want[cur];
        int found = -1;
        for (int c0 = 1; c0 < T && found < 0; c0 += 32) {
            const int c = c0 + lane;
            const bool hit = c < T && s_par[c] == cur && s_tok[c] == want;
            const unsigned m = __ballot_sync(FULL, hit);
            if (m) found = c0 + __ffs(m) - 1;
        }
        if (found < 0) break;
        if (n >= width) {  // tree deeper than max_depth
            if (lane == 0) latch(err, DDT_DEVERR_DEPTH);
            break;
        }
        path[n] = found;
        ++n;
        cur = found;
    }
    const int bon = s_want[cur];
    if (lane == 0) {
        accept_len[b] = n;
        bonus[b] = bon;
    }
    for (int k = lane; k < width; k += 32) {
        acc[k] = (k < n) ? path[k] : -1;
        int t = -1;
        if (k < n - 1) t = s_tok[path[k + 1]];
        else if (k == n - 1) t = bon;
        com[k] = t;
    }
}

}  // namespace

// The attention kernel needs the SM's largest shared-memory carveout; a kernel
// that runs beside it must ask for the same, or the SM it lands on cannot take
// an attention CTA until it drains (measured: the last cluster of the verify
// step started ~15 us late).
cudaError_t tree_prepare_device() {
    cudaError_t e = cudaFuncSetAttribute(build_tree_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(build_tree_visibility_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(compile_visibility_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(accept_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(build_chain_visibility_kernel,
                                 cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    return e;
}

cudaError_t launch_build_chain_visibility(const int32_t *qo_indptr, const int32_t *prefix_len,
                                          const int32_t *mask_indptr, int batch, int32_t *parent,
                                          int32_t *depth, uint32_t *mask, unsigned int *err,
                                          cudaStream_t s) {
    return launch_pdl(build_chain_visibility_kernel, dim3(batch), dim3(kChainThreads), 0, s,
                      qo_indptr, prefix_len, mask_indptr, parent, depth, mask, err);
}

cudaError_t launch_build_tree(const float *topk_logp, const int32_t *topk_ids,
                              const int32_t *root_id, const int32_t *budget,
                              const int32_t *qo_indptr, int batch, int max_depth, int topk,
                              int32_t *node_token, int32_t *parent, int32_t *depth,
                              unsigned int *err, cudaStream_t s) {
    return launch_pdl(build_tree_kernel, dim3(batch), dim3(32), 0, s, topk_logp, topk_ids, root_id,
                      budget, qo_indptr, max_depth, topk, node_token, parent, depth, err);
}

cudaError_t launch_build_tree_visibility(const float *topk_logp, const int32_t *topk_ids,
                                         const int32_t *root_id, const int32_t *budget,
                                         const int32_t *qo_indptr, int batch, int max_depth, int topk,
                                         const int32_t *prefix_len, const int32_t *mask_indptr,
                                         int32_t *node_token, int32_t *parent, int32_t *depth,
                                         uint32_t *mask, unsigned int *err, cudaStream_t s) {
    return launch_pdl(build_tree_visibility_kernel, dim3(batch), dim3(kTreeVisThreads), 0, s, topk_logp,
                      topk_ids, root_id, budget, qo_indptr, max_depth, topk, prefix_len, mask_indptr,
                      node_token, parent, depth, mask, err);
}

cudaError_t launch_compile_visibility(const int32_t *parent, const int32_t *qo_indptr,
                                      const int32_t *prefix_len, const int32_t *mask_indptr,
                                      int batch, int total_words, uint32_t *mask,
                                      unsigned int *err, cudaStream_t s) {
    if (total_words <= 0) return cudaSuccess;
    const int threads = 256;
    int blocks = (total_words + threads - 1) / threads;
    if (blocks > 4096) blocks = 4096;
    return launch_pdl(compile_visibility_kernel, dim3(blocks), dim3(threads), 0, s, parent,
                      qo_indptr, prefix_len, mask_indptr, batch, total_words, mask, err);
}

cudaError_t launch_accept(const int32_t *node_token, const int32_t *parent,
                          const int32_t *qo_indptr, const int32_t *target_argmax, int batch,
                          int max_depth, int32_t *accept_len, int32_t *accepted_nodes,
                          int32_t *commit_tokens, int32_t *bonus, unsigned int *err,
                          cudaStream_t s) {
    return launch_pdl(accept_kernel, dim3(batch), dim3(32), 0, s, node_token, parent, qo_indptr,
                      target_argmax, max_depth, accept_len, accepted_nodes, commit_tokens, bonus, err);
}

}  // namespace ddt
