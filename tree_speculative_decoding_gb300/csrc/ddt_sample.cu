// ddt_sample.cu -- sampling accept: tree rejection sampling with temperature
// and top-k, and the tree links it walks.
//
// Page: "The DDTree CUDA Graph Fix: Unlocking Speculative Decoding at 109 tok/s
// on PCIe Blackwell", section "Temperature Support: Already Working for
// Linear, Planned for DDTree": sampling accept runs tree rejection sampling on
// the target distribution (temperature, top-k), with the tree given as
// (retrieve_index, retrieve_next_token, retrieve_next_sibling).  The pages
// give no algorithm text; the reading taken (target-only, deterministic
// drafts):
//   p(n)  = softmax(logits[n] / T) over the tokens whose logit is at least the
//           top_k-th largest (all of them for top_k <= 0 or >= vocab, ties
//           kept); T <= 0 means one-hot at the argmax (lowest id on ties);
//   at node n the children are tried in index order against the residual r
//   (p minus the tokens already rejected): child c with token t is taken when
//   coin[n][i] < r(t) / mass(r), else t leaves the residual;
//   with no child taken the bonus is the first token id whose cumulative
//   residual mass exceeds coin[n][last] * mass(r).
// Every emitted token is then distributed as p, and T <= 0 is the greedy walk.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ddt_internal.cuh"

namespace ddt {
namespace {

constexpr unsigned FULL = 0xffffffffu;

// ------------------------------------------------------------------ tree links
// One warp per request: node n's first child is the lowest index c > n with
// parent c == n; its next sibling the lowest index c > n with the same parent.
__global__ void __launch_bounds__(32)
tree_links_kernel(const int32_t *__restrict__ parent, const int32_t *__restrict__ qo_indptr,
                  int32_t *__restrict__ first_child, int32_t *__restrict__ next_sibling,
                  int32_t *__restrict__ retrieve_index, unsigned int *err) {
    __shared__ int32_t par[DDT_MAX_Q_LEN];
    const int b = blockIdx.x;
    const int lane = threadIdx.x;
    pdl_trigger();
    const int base = qo_indptr[b];
    const int T = qo_indptr[b + 1] - base;
    pdl_wait();  // the parents come from the tree build
    if (T < 1 || T > DDT_MAX_Q_LEN) {
        if (lane == 0) latch(err, DDT_DEVERR_QO_INDPTR);
        return;
    }
    for (int i = lane; i < T; i += 32) par[i] = parent[base + i];
    __syncwarp();
    for (int n = lane; n < T; n += 32) {
        int fc = -1, ns = -1;
        const int pn = n > 0 ? par[n] : -2;
        for (int c = n + 1; c < T; ++c) {
            const int pc = par[c];
            if (fc < 0 && pc == n) fc = c;
            if (ns < 0 && pc == pn) ns = c;
            if (fc >= 0 && ns >= 0) break;
        }
        first_child[base + n] = fc;
        next_sibling[base + n] = ns;
        retrieve_index[base + n] = base + n;
    }
}

// ------------------------------------------------------------- sampling accept
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ uint32_t order_key(float f) {  // larger float -> larger key
    const uint32_t u = __float_as_uint(f + 0.0f);  // -0 -> +0: equal floats, equal keys
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SampleSmem {
    float fred[kWarps];
    int ired[kWarps];
    unsigned hist[256];
    float chunk[kThreads];
    int removed[DDT_MAX_TOPK + 1];
    int nremoved;
    int decision;  // child taken, or -1
    float mass;
    int bonus;
    unsigned thr_key;
};

// block-wide max of (value, -index): the largest value, lowest index on ties
__device__ void block_argmax(float v, int idx, SampleSmem &sm, float &vmax, int &imax) {
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(FULL, v, o);
        const int oi = __shfl_xor_sync(FULL, idx, o);
        if (ov > v || (ov == v && oi < idx)) { v = ov; idx = oi; }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) { sm.fred[warp] = v; sm.ired[warp] = idx; }
    __syncthreads();
    v = sm.fred[0];
    idx = sm.ired[0];
    for (int w = 1; w < kWarps; ++w)
        if (sm.fred[w] > v || (sm.fred[w] == v && sm.ired[w] < idx)) { v = sm.fred[w]; idx = sm.ired[w]; }
    vmax = v;
    imax = idx;
}

// block-wide sum in a fixed order (warp shuffles, then warps 0..7)
__device__ float block_sum(float v, SampleSmem &sm) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) sm.fred[warp] = v;
    __syncthreads();
    float s = 0.f;
    for (int w = 0; w < kWarps; ++w) s += sm.fred[w];
    return s;
}

// key of the k-th largest logit (1 <= k <= vocab): four 8-bit radix passes
__device__ unsigned kth_largest_key(const float *row, int vocab, int k, SampleSmem &sm) {
    unsigned prefix = 0, mask = 0;
    int need = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += kThreads) sm.hist[i] = 0;
        __syncthreads();
        for (int v = threadIdx.x; v < vocab; v += kThreads) {
            const unsigned key = order_key(row[v]);
            if ((key & mask) == prefix) atomicAdd(&sm.hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int above = 0, d = 255;
            for (; d > 0; --d) {
                if (above + (int)sm.hist[d] >= need) break;
                above += (int)sm.hist[d];
            }
            sm.thr_key = (unsigned)d;
            sm.nremoved = need - above;  // reused as scratch: rank inside the bin
        }
        __syncthreads();
        prefix |= sm.thr_key << shift;
        mask |= 255u << shift;
        need = sm.nremoved;
        __syncthreads();
    }
    return prefix;
}

__global__ void __launch_bounds__(kThreads)
accept_sampled_kernel(const int32_t *__restrict__ node_token, const int32_t *__restrict__ first_child,
                      const int32_t *__restrict__ next_sibling, const int32_t *__restrict__ qo_indptr,
                      const float *__restrict__ logits, int vocab, const float *__restrict__ temperature,
                      const int32_t *__restrict__ top_k, const float *__restrict__ coins, int coin_stride,
                      int max_depth, int32_t *__restrict__ accept_len, int32_t *__restrict__ accepted_nodes,
                      int32_t *__restrict__ commit_tokens, int32_t *__restrict__ bonus, unsigned int *err) {
    __shared__ SampleSmem sm;
    __shared__ int path[DDT_MAX_DEPTH + 1];
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    pdl_trigger();
    const int base = qo_indptr[b];
    const int T = qo_indptr[b + 1] - base;
    const float temp = temperature[b];
    const int kk = top_k[b];
    const bool greedy = !(temp > 0.f);
    const bool use_topk = !greedy && kk > 0 && kk < vocab;
    const float inv_t = greedy ? 0.f : 1.f / temp;
    const int width = max_depth + 1;
    pdl_wait();  // the tree and its links come from earlier kernels
    if (T < 1 || T > DDT_MAX_Q_LEN) {
        if (tid == 0) latch(err, DDT_DEVERR_QO_INDPTR);
        return;
    }
    int cur = 0, n = 1;
    if (tid == 0) path[0] = 0;
    int bon = -1;
    for (;;) {
        const float *row = logits + (size_t)(base + cur) * vocab;
        const float *u = coins + (size_t)(base + cur) * coin_stride;
        // the argmax (and the max logit)
        float lv = -INFINITY;
        int li = vocab;
        for (int v = tid; v < vocab; v += kThreads) {
            const float x = row[v];
            if (x > lv) { lv = x; li = v; }
        }
        float lmax;
        int amax;
        block_argmax(lv, li, sm, lmax, amax);
        // kept set and normaliser
        unsigned thr = 0;
        if (use_topk) thr = kth_largest_key(row, vocab, kk, sm);
        float z = 1.f;
        if (!greedy) {
            float part = 0.f;
            for (int v = tid; v < vocab; v += kThreads) {
                const float x = row[v];
                if (order_key(x) >= thr) part += __expf((x - lmax) * inv_t);
            }
            z = block_sum(part, sm);
        }
        // p(v) of the target at this node (0 outside the kept set)
        auto prob = [&](int v) -> float {
            if (v < 0 || v >= vocab) return 0.f;
            if (greedy) return v == amax ? 1.f : 0.f;
            const float x = row[v];
            return order_key(x) >= thr ? __expf((x - lmax) * inv_t) / z : 0.f;
        };
        // the children against the residual (one thread: at most top-k children)
        if (tid == 0) {
            float mass = 1.f;
            int taken = -1, i = 0, nrem = 0;
            for (int c = first_child[base + cur]; c >= 0; c = next_sibling[base + c], ++i) {
                if (c <= cur || c >= T || i >= coin_stride - 1 || i > DDT_MAX_TOPK) {
                    latch(err, DDT_DEVERR_SAMPLE);  // links or coins do not fit the tree
                    taken = -2;
                    break;
                }
                const int t = node_token[base + c];
                const float pt = prob(t);
                if (u[i] < pt / mass) { taken = c; break; }
                mass -= pt;
                sm.removed[nrem++] = t;
            }
            sm.decision = taken;
            sm.nremoved = nrem;
            sm.mass = mass;
        }
        __syncthreads();
        const int taken = sm.decision;
        if (taken == -2) return;
        if (taken >= 0) {
            if (n >= width) {  // deeper than max_depth
                if (tid == 0) latch(err, DDT_DEVERR_DEPTH);
                return;
            }
            if (tid == 0) path[n] = taken;
            ++n;
            cur = taken;
            __syncthreads();
            continue;
        }
        // bonus: the first id whose cumulative residual mass exceeds coin * mass
        if (greedy) {
            bon = amax;
            break;
        }
        const int nrem = sm.nremoved;
        const float target = u[coin_stride - 1] * sm.mass;
        const int chunk = (vocab + kThreads - 1) / kThreads;
        const int v0 = tid * chunk, v1 = min(vocab, v0 + chunk);
        auto residual = [&](int v) -> float {
            for (int r = 0; r < nrem; ++r)
                if (sm.removed[r] == v) return 0.f;
            return prob(v);
        };
        float csum = 0.f;
        int last_pos = -1;
        for (int v = v0; v < v1; ++v) {
            const float pv = residual(v);
            csum += pv;
            if (pv > 0.f) last_pos = v;
        }
        sm.chunk[tid] = csum;
        __syncthreads();
        if (tid == 0) {  // exclusive scan over the chunks, in id order
            float acc = 0.f;
            for (int t = 0; t < kThreads; ++t) {
                const float s = sm.chunk[t];
                sm.chunk[t] = acc;
                acc += s;
            }
            sm.bonus = -1;
        }
        __syncthreads();
        float cum = sm.chunk[tid];
        if (cum <= target && cum + csum > target) {  // the one chunk where the prefix crosses
            int pick = -1;
            for (int v = v0; v < v1; ++v) {
                const float pv = residual(v);
                cum += pv;
                if (cum > target) {
                    pick = v;
                    break;
                }
            }
            sm.bonus = pick >= 0 ? pick : last_pos;  // rounding: the chunk's last id with mass
        }
        // rounding fallback: the last id with residual mass
        int lp = last_pos;
        for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(FULL, lp, o));
        if ((tid & 31) == 0) sm.ired[tid >> 5] = lp;
        __syncthreads();
        if (tid == 0) {
            int best = -1;
            for (int w = 0; w < kWarps; ++w) best = max(best, sm.ired[w]);
            if (sm.bonus < 0) sm.bonus = best >= 0 ? best : amax;
        }
        __syncthreads();
        bon = sm.bonus;
        break;
    }
    if (tid == 0) {
        accept_len[b] = n;
        bonus[b] = bon;
    }
    for (int k = tid; k < width; k += kThreads) {
        accepted_nodes[(size_t)b * width + k] = (k < n) ? path[k] : -1;
        int t = -1;
        if (k < n - 1) t = node_token[base + path[k + 1]];
        else if (k == n - 1) t = bon;
        commit_tokens[(size_t)b * width + k] = t;
    }
}

}  // namespace

cudaError_t sample_prepare_device() {
    cudaError_t e = cudaFuncSetAttribute(tree_links_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(accept_sampled_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    return e;
}

cudaError_t launch_tree_links(const int32_t *parent, const int32_t *qo_indptr, int batch,
                              int32_t *first_child, int32_t *next_sibling, int32_t *retrieve_index,
                              unsigned int *err, cudaStream_t s) {
    return launch_pdl(tree_links_kernel, dim3(batch), dim3(32), 0, s, parent, qo_indptr, first_child,
                      next_sibling, retrieve_index, err);
}

cudaError_t launch_accept_sampled(const int32_t *node_token, const int32_t *first_child,
                                  const int32_t *next_sibling, const int32_t *qo_indptr,
                                  const float *logits, int vocab, const float *temperature,
                                  const int32_t *top_k, const float *coins, int coin_stride, int batch,
                                  int max_depth, int32_t *accept_len, int32_t *accepted_nodes,
                                  int32_t *commit_tokens, int32_t *bonus, unsigned int *err,
                                  cudaStream_t s) {
    return launch_pdl(accept_sampled_kernel, dim3(batch), dim3(kThreads), 0, s, node_token, first_child,
                      next_sibling, qo_indptr, logits, vocab, temperature, top_k, coins, coin_stride,
                      max_depth, accept_len, accepted_nodes, commit_tokens, bonus, err);
}

}  // namespace ddt
