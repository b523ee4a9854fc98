// ddt_sample.cu -- sampling accept: tree rejection sampling with temperature,
// top-k and top-p, and the tree links it walks.
//
// Page: "The DDTree CUDA Graph Fix: Unlocking Speculative Decoding at 109 tok/s
// on PCIe Blackwell", section "Temperature Support: Already Working for
// Linear, Planned for DDTree": sampling accept runs tree rejection sampling on
// the target distribution (temperature, top-k, top-p), with the tree given as
// (retrieve_index, retrieve_next_token, retrieve_next_sibling).  The pages
// give no algorithm text; the reading taken (target-only, deterministic
// drafts):
//   p(n)  = softmax(logits[n] / T) over the tokens whose logit is at least the
//           top_k-th largest (all of them for top_k <= 0 or >= vocab, ties
//           kept); T <= 0 means one-hot at the argmax (lowest id on ties);
//   top-p then keeps the tokens whose logit is at least tau, the largest
//           logit x whose mass S(x) (of p over the tokens with logit >= x)
//           reaches top_p; tokens equal to tau are all kept and p is
//           renormalised over the kept set (top_p outside (0, 1): no filter);
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
#include "ddt_sm100.cuh"

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
constexpr int kThreads = 512;
// A visited node's logit row of up to this many ids is copied into shared
// memory once (one bulk copy per 32 KB), and every pass over it reads shared
// memory instead of L2; longer rows are read from global memory.
constexpr int kStageVocab = 45056;
constexpr uint32_t kStageChunk = 32768;
constexpr uint32_t kStageWaitLimit = 1u << 22;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxSteps = 64;  // 256-id steps per warp segment: vocabularies up to 16 * 64 * 256
static_assert(kWarps * kMaxSteps * 256 == DDT_MAX_VOCAB, "vocabulary bound of the ABI");

// Calls f(v, row[v]) for this thread's ids v = tid + k * kThreads with eight
// loads in flight, so that one CTA streaming a vocabulary row is not bound by
// one memory round trip per element.
template <class F>
__device__ __forceinline__ void for_each_logit(const float *row, int vocab, F f) {
    for (int v0 = threadIdx.x; v0 < vocab; v0 += 8 * kThreads) {
        float x[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int v = v0 + k * kThreads;
            x[k] = v < vocab ? row[v] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int v = v0 + k * kThreads;
            if (v < vocab) f(v, x[k]);
        }
    }
}

// the row into L2 ahead of its passes (bulk prefetch: 16-byte aligned, whole 16-byte units)
__device__ __forceinline__ void prefetch_row(const float *row, int vocab) {
    if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0 && (vocab & 3) == 0)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(row), "r"(vocab * 4) : "memory");
}

__device__ __forceinline__ uint32_t order_key(float f) {  // larger float -> larger key
    const uint32_t u = __float_as_uint(f + 0.0f);  // -0 -> +0: equal floats, equal keys
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SampleSmem {
    int tok[DDT_MAX_Q_LEN], fc[DDT_MAX_Q_LEN], ns[DDT_MAX_Q_LEN];  // the request's tree
    int kid[DDT_MAX_TOPK + 1];       // children of the current node, in order
    float kid_logit[DDT_MAX_TOPK + 1], kid_coin[DDT_MAX_TOPK + 1];
    int nkid;
    float fred[kWarps];
    int ired[kWarps];
    unsigned hist[256];
    unsigned long long hist64[256];  // top-p: bin masses in 2^-40 units
    unsigned long long topp_target, topp_above;
    float step[kWarps][kMaxSteps];  // mass of each 256-id step of each warp's segment
    float stepmax[kWarps][kMaxSteps];  // the step's max logit (the temperature pass)
    int removed[DDT_MAX_TOPK + 1];
    int nremoved;
    union {
        unsigned gone[DDT_MAX_VOCAB / 32];  // the removed tokens as a bit set, for the bonus pass
        unsigned long long whist[kWarps][256];  // top-p radix passes: each warp's bin masses
        struct {  // the same as two 32-bit halves (rows of at most kStageVocab ids)
            unsigned hi[kWarps][256], lo[kWarps][256];
        } wsplit;
        unsigned whist32[kWarps][256];          // top-k radix passes: each warp's bin counts
    };
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
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int shift = 24; shift >= 0; shift -= 8) {
        // each warp counts into a histogram of its own (atomics that only lanes of
        // one warp contend on: after the first pass nearly all keys share their
        // leading bits, and one histogram for the CTA would serialise all warps on
        // a handful of bins); the warps' counts are added per bin after the pass.
        // Eight loads in flight per thread.
        for (int i = lane; i < 256; i += 32) sm.whist32[warp][i] = 0u;
        __syncwarp();
        for (int v0 = threadIdx.x - lane; v0 < vocab; v0 += 8 * kThreads) {
            unsigned key[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int v = v0 + k * kThreads + lane;
                key[k] = v < vocab ? order_key(row[v]) : 0u;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int v = v0 + k * kThreads + lane;
                if (v < vocab && (key[k] & mask) == prefix)
                    atomicAdd(&sm.whist32[warp][(key[k] >> shift) & 255u], 1u);
            }
        }
        __syncthreads();
        for (int d = threadIdx.x; d < 256; d += kThreads) {
            unsigned t = 0u;
            for (int w = 0; w < kWarps; ++w) t += sm.whist32[w][d];
            sm.hist[d] = t;
        }
        __syncthreads();
        // Warp 0 walks the bins from the top (d = 255 down to 1) to the first whose
        // count, added to the count above it, reaches the rank; bin 0 if none does
        // (lane l holds bins 255 - 8l .. 248 - 8l, as in topp_key).
        if (warp == 0) {
            unsigned h[8], part = 0u;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                h[i] = sm.hist[255 - 8 * lane - i];
                part += h[i];
            }
            unsigned incl = part;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned t = __shfl_up_sync(FULL, incl, o);
                if (lane >= o) incl += t;
            }
            const unsigned cross = __ballot_sync(FULL, incl >= (unsigned)need);
            const int cl = cross ? __ffs(cross) - 1 : 31;
            if (lane == cl) {
                unsigned above = incl - part;
                int d = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int di = 255 - 8 * lane - i;
                    if (d == 0 && di > 0) {
                        if (above + h[i] >= (unsigned)need) d = di;
                        else above += h[i];
                    }
                }
                sm.thr_key = (unsigned)d;
                sm.nremoved = need - (int)above;  // reused as scratch: rank inside the bin
            }
        }
        __syncthreads();
        prefix |= sm.thr_key << shift;
        mask |= 255u << shift;
        need = sm.nremoved;
        __syncthreads();
    }
    return prefix;
}

// key of tau for top-p: the largest key kappa among the candidates (keys >= lo)
// whose mass S(kappa), the sum of e^{(x - lmax)/T} over candidate keys >=
// kappa, reaches top_p times the candidates' total.  Four 8-bit radix passes
// over the masses in fixed point (2^-40 units: integer sums, so the decision
// does not depend on any summation order).  Each warp adds its lanes' masses
// into a histogram of its own (shared-memory atomics that only lanes of the
// same warp contend on), and the warps' histograms are added per bin after
// the pass.  For rows of at most kStageVocab ids a warp adds at most 2816
// masses per bin, so each mass (at most 2^40) goes in as two 32-bit halves,
// bits 20 and up and the low 20 bits, whose per-warp sums stay below 2^32: two
// native 32-bit shared atomics instead of one 64-bit one.
__device__ unsigned topp_key(const float *row, int vocab, unsigned lo, float lmax, float inv_t,
                             float top_p, SampleSmem &sm) {
    static_assert(((kStageVocab + kThreads - 1) / kThreads) * 32 * (1ull << 20) < (1ull << 32),
                  "per-warp sums of the 32-bit halves fit");
    unsigned prefix = 0, mask = 0;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const bool halves = vocab <= kStageVocab;
    for (int shift = 24; shift >= 0; shift -= 8) {
        if (halves) {
            for (int i = lane; i < 256; i += 32) sm.wsplit.hi[warp][i] = sm.wsplit.lo[warp][i] = 0u;
        } else {
            for (int i = lane; i < 256; i += 32) sm.whist[warp][i] = 0ull;
        }
        __syncwarp();
        for (int v0 = threadIdx.x - lane; v0 < vocab; v0 += 8 * kThreads) {
            float x[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int v = v0 + k * kThreads + lane;
                x[k] = v < vocab ? row[v] : -INFINITY;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int v = v0 + k * kThreads + lane;
                const unsigned key = order_key(x[k]);
                const bool in = v < vocab && key >= lo && (key & mask) == prefix;
                if (in) {  // e <= 1 (x <= lmax), so the fixed-point mass is at most 2^40
                    const unsigned long long f =
                        __float2ull_rn(__expf((x[k] - lmax) * inv_t) * 1099511627776.0f);
                    const unsigned b = (key >> shift) & 255u;
                    if (halves) {
                        atomicAdd(&sm.wsplit.hi[warp][b], (unsigned)(f >> 20));
                        atomicAdd(&sm.wsplit.lo[warp][b], (unsigned)(f & 0xFFFFFull));
                    } else {
                        atomicAdd(&sm.whist[warp][b], f);
                    }
                }
            }
        }
        __syncthreads();
        for (int d = threadIdx.x; d < 256; d += kThreads) {
            unsigned long long t = 0ull;
            if (halves) {
                for (int w = 0; w < kWarps; ++w)
                    t += ((unsigned long long)sm.wsplit.hi[w][d] << 20) + sm.wsplit.lo[w][d];
            } else {
                for (int w = 0; w < kWarps; ++w) t += sm.whist[w][d];
            }
            sm.hist64[d] = t;
        }
        __syncthreads();
        // Warp 0 walks the bins from the top (d = 255 down to 1) to the first whose
        // mass, added to the mass above it, reaches the target; bin 0 if none does.
        // Lane l holds bins 255 - 8l .. 248 - 8l; a prefix sum over the lanes finds
        // the lane where the running mass crosses, which then walks its eight bins.
        if (warp == 0) {
            unsigned long long h[8], part = 0ull;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                h[i] = sm.hist64[255 - 8 * lane - i];
                part += h[i];
            }
            unsigned long long incl = part;  // bins of lanes 0..lane
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long t = __shfl_up_sync(FULL, incl, o);
                if (lane >= o) incl += t;
            }
            unsigned long long above = sm.topp_above, target = sm.topp_target;
            if (shift == 24) {
                const unsigned long long total = __shfl_sync(FULL, incl, 31);
                target = (unsigned long long)((double)top_p * (double)total);
                target = target < 1ull ? 1ull : target;
                above = 0ull;
            }
            const unsigned cross = __ballot_sync(FULL, above + incl >= target);
            const int cl = cross ? __ffs(cross) - 1 : 31;
            if (lane == cl) {
                unsigned long long run = above + (incl - part);
                int d = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int di = 255 - 8 * lane - i;
                    if (d == 0 && di > 0) {
                        if (run + h[i] >= target) d = di;
                        else run += h[i];
                    }
                }
                sm.thr_key = (unsigned)d;
                sm.topp_above = run;
                sm.topp_target = target;
            }
        }
        __syncthreads();
        prefix |= sm.thr_key << shift;
        mask |= 255u << shift;
        __syncthreads();
    }
    return prefix;
}

__global__ void __launch_bounds__(kThreads, 1)
accept_sampled_kernel(const int32_t *__restrict__ node_token, const int32_t *__restrict__ first_child,
                      const int32_t *__restrict__ next_sibling, const int32_t *__restrict__ qo_indptr,
                      const float *__restrict__ logits, int vocab, const float *__restrict__ temperature,
                      const int32_t *__restrict__ top_k, const float *__restrict__ top_p,
                      const float *__restrict__ coins, int coin_stride,
                      int max_depth, int32_t *__restrict__ accept_len, int32_t *__restrict__ accepted_nodes,
                      int32_t *__restrict__ commit_tokens, int32_t *__restrict__ bonus, int stage,
                      unsigned int *err) {
    __shared__ SampleSmem sm;
    __shared__ int path[DDT_MAX_DEPTH + 1];
    __shared__ __align__(8) uint64_t row_bar;
    extern __shared__ __align__(16) float srow[];  // the staged logit row (stage != 0)
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    pdl_trigger();
    const int base = qo_indptr[b];
    const int T = qo_indptr[b + 1] - base;
    const float temp = temperature[b];
    const int kk = top_k[b];
    const bool greedy = !(temp > 0.f);
    const bool use_topk = !greedy && kk > 0 && kk < vocab;
    const float tp = top_p ? top_p[b] : 1.f;
    const bool use_topp = !greedy && tp > 0.f && tp < 1.f;
    const bool use_filter = use_topk || use_topp;
    const float inv_t = greedy ? 0.f : 1.f / temp;
    const int width = max_depth + 1;
    if (tid == 0 && T >= 1 && T <= DDT_MAX_Q_LEN) prefetch_row(logits + (size_t)base * vocab, vocab);
    pdl_wait();  // the tree and its links come from earlier kernels
    if (T < 1 || T > DDT_MAX_Q_LEN) {
        if (tid == 0) latch(err, DDT_DEVERR_QO_INDPTR);
        return;
    }
    // the tree, once: every later walk step reads shared memory
    for (int i = tid; i < T; i += kThreads) {
        sm.tok[i] = node_token[base + i];
        sm.fc[i] = first_child[base + i];
        sm.ns[i] = next_sibling[base + i];
    }
    // warp w owns ids [w * seg, (w + 1) * seg) in steps of 256 ids, lane l
    // holding ids [8l, 8l+8) of a step
    const int warp = tid >> 5, lane = tid & 31;
    const int seg = ((vocab + kWarps - 1) / kWarps + 255) & ~255;
    const int s0 = warp * seg, s1 = min(vocab, s0 + seg);
    const int nsteps = s1 > s0 ? (s1 - s0 + 255) / 256 : 0;
    // at temperature > 0 without top-k the first pass also keeps, per step, the
    // sum of e^{(x - m)/T} and its max m, so the bonus draw needs no second pass
    const bool step_pass = !greedy && !use_filter;
    int cur = 0, n = 1;
    if (tid == 0) {
        path[0] = 0;
        if (stage) {
            sm100::mbar_init(sm100::smem_u32(&row_bar), 1);
            sm100::fence_barrier_init();
        }
    }
    int bon = -1;
    uint32_t visit = 0;  // staged rows so far: the parity of the row barrier
    for (;;) {
        __syncthreads();
        const float *row = logits + (size_t)(base + cur) * vocab;
        const float *u = coins + (size_t)(base + cur) * coin_stride;
        // the children of cur, from the links; then their logits and coins, in parallel
        if (tid == 0) {
            if (stage) {  // the row into shared memory; the previous row's readers are past the barrier
                const uint32_t bar = sm100::smem_u32(&row_bar);
                const uint32_t bytes = (uint32_t)vocab * 4u;
                sm100::fence_proxy_async_smem();
                sm100::mbar_arrive_expect_tx(bar, bytes);
                for (uint32_t off = 0; off < bytes; off += kStageChunk)
                    sm100::bulk_load_global(sm100::smem_u32(srow) + off, reinterpret_cast<const char *>(row) + off,
                                            min(kStageChunk, bytes - off), bar);
            }
            int nk = 0;
            for (int c = sm.fc[cur]; c >= 0; c = sm.ns[c]) {
                if (c <= cur || c >= T || nk >= coin_stride - 1 || nk > DDT_MAX_TOPK) {
                    nk = -1;  // links or coins do not fit the tree
                    break;
                }
                sm.kid[nk++] = c;
            }
            sm.nkid = nk;
        }
        __syncthreads();
        if (stage) {  // every thread waits for the row itself (bounded), and all agree
            const bool got = sm100::mbar_wait(sm100::smem_u32(&row_bar), visit & 1u, kStageWaitLimit);
            if (!__syncthreads_and(got)) {  // the copy never completed: give up on this request
                if (tid == 0) latch(err, DDT_DEVERR_TIMEOUT);
                return;
            }
            row = srow;
            ++visit;
        }
        const int nkid = sm.nkid;
        if (nkid < 0) {
            if (tid == 0) latch(err, DDT_DEVERR_SAMPLE);
            return;
        }
        if (tid < nkid) {
            const int t = sm.tok[sm.kid[tid]];
            sm.kid_logit[tid] = (t >= 0 && t < vocab) ? row[t] : -INFINITY;
            sm.kid_coin[tid] = u[tid];
            prefetch_row(logits + (size_t)(base + sm.kid[tid]) * vocab, vocab);  // the next level's candidates
        }
        // the argmax and the max logit; at temperature > 0 also the normaliser
        float lv = -INFINITY;
        int li = vocab;
        if (step_pass) {
            for (int st = 0; st < nsteps; ++st) {
                const int b0 = s0 + 256 * st + 8 * lane;
                float x[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) x[k] = b0 + k < s1 ? row[b0 + k] : -INFINITY;
                float m = -INFINITY;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if (b0 + k < s1 && (x[k] > lv || (x[k] == lv && b0 + k < li))) {
                        lv = x[k];
                        li = b0 + k;
                    }
                    m = fmaxf(m, x[k]);
                }
                for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
                float e = 0.f;
                if (m != -INFINITY) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) e += __expf((x[k] - m) * inv_t);
                }
                for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(FULL, e, o);
                if (lane == 0) {
                    sm.step[warp][st] = e;
                    sm.stepmax[warp][st] = m;
                }
            }
        } else {
            for_each_logit(row, vocab, [&](int v, float x) {
                if (x > lv || (x == lv && v < li)) {
                    lv = x;
                    li = v;
                }
            });
        }
        float lmax;
        int amax;
        block_argmax(lv, li, sm, lmax, amax);  // (its barriers publish the step sums)
        unsigned thr = 0;
        float z = 1.f;
        if (step_pass) {  // the step sums rescaled to lmax; z is their total
            float part = 0.f;
            for (int st = lane; st < nsteps; st += 32) {
                const float m = sm.stepmax[warp][st];
                const float e = m == -INFINITY ? 0.f : sm.step[warp][st] * __expf((m - lmax) * inv_t);
                sm.step[warp][st] = e;
                part += e;
            }
            z = block_sum(part, sm);
        } else if (use_filter) {  // kept set first (top-k, then top-p), then its mass per step
            if (use_topk) thr = kth_largest_key(row, vocab, kk, sm);
            if (use_topp) thr = topp_key(row, vocab, thr, lmax, inv_t, tp, sm);
            // the kept mass of each 256-id step of this warp's segment, as the
            // temperature pass keeps it, so that the bonus draw recomputes only
            // the steps of removed tokens; z is the total
            float part = 0.f;
            for (int st = 0; st < nsteps; ++st) {
                const int b0 = s0 + 256 * st + 8 * lane;
                float x[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) x[k] = b0 + k < s1 ? row[b0 + k] : -INFINITY;
                float e = 0.f;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    if (b0 + k < s1 && order_key(x[k]) >= thr) e += __expf((x[k] - lmax) * inv_t);
                part += e;
                for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(FULL, e, o);
                if (lane == 0) sm.step[warp][st] = e;
            }
            z = block_sum(part, sm);
        }
        // p(v) of the target at this node (0 outside the kept set), from its logit
        const float inv_z = 1.f / z;
        auto prob_of = [&](int v, float x) -> float {
            if (v < 0 || v >= vocab) return 0.f;
            if (greedy) return v == amax ? 1.f : 0.f;
            if (use_filter && order_key(x) < thr) return 0.f;
            return __expf((x - lmax) * inv_t) * inv_z;
        };
        // the children against the residual (one thread, shared-memory values)
        if (tid == 0) {
            float mass = 1.f;
            int taken = -1, nrem = 0;
            for (int i = 0; i < nkid; ++i) {
                const int t = sm.tok[sm.kid[i]];
                const float pt = prob_of(t, sm.kid_logit[i]);
                if (sm.kid_coin[i] < pt / mass) { taken = sm.kid[i]; break; }
                mass -= pt;
                sm.removed[nrem++] = t;
            }
            sm.decision = taken;
            sm.nremoved = nrem;
            sm.mass = mass;
        }
        __syncthreads();
        const int taken = sm.decision;
        if (taken >= 0) {
            if (n >= width) {  // deeper than max_depth
                if (tid == 0) latch(err, DDT_DEVERR_DEPTH);
                return;
            }
            if (tid == 0) path[n] = taken;
            ++n;
            cur = taken;
            continue;
        }
        // bonus: the first id whose cumulative residual mass exceeds coin * mass
        if (greedy) {
            bon = amax;
            break;
        }
        const int nrem = sm.nremoved;
        const float target = u[coin_stride - 1] * sm.mass;
        for (int i = tid; i < (vocab + 31) >> 5; i += kThreads) sm.gone[i] = 0u;
        for (int st = lane; st < nsteps; st += 32) sm.step[warp][st] *= inv_z;  // step masses as probabilities
        __syncthreads();
        if (tid < nrem) {
            const int t = sm.removed[tid];
            if (t >= 0 && t < vocab) atomicOr(&sm.gone[t >> 5], 1u << (t & 31));
        }
        __syncthreads();
        auto residual_of = [&](int v, float x) -> float {
            return (sm.gone[v >> 5] >> (v & 31)) & 1u ? 0.f : prob_of(v, x);
        };
        // step st of warp w's segment, per element: this lane's running sums (loc),
        // its total and its last id with mass
        auto step_sums = [&](int w, int st, float (&loc)[8], float &lsum, int &llast) {
            const int w1 = min(vocab, w * seg + seg);
            const int b0 = w * seg + 256 * st + 8 * lane;
            float x[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) x[k] = b0 + k < w1 ? row[b0 + k] : 0.f;
            lsum = 0.f;
            llast = -1;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float pv = b0 + k < w1 ? residual_of(b0 + k, x[k]) : 0.f;
                lsum += pv;
                loc[k] = lsum;
                if (pv > 0.f) llast = b0 + k;
            }
        };
        auto warp_total = [&](float lsum) {
            for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(FULL, lsum, o);
            return lsum;
        };
        // only the steps holding a removed token change (every step's mass is known
        // from the temperature pass or the kept-set pass): warp j recomputes the
        // step of removed token j per element, once per step (steps are the
        // id blocks [256i, 256i + 256), since seg is a multiple of 256)
        for (int j = warp; j < nrem; j += kWarps) {
            const int t = sm.removed[j];
            bool first = t >= 0 && t < vocab;
            for (int r = 0; r < j && first; ++r) {
                const int q = sm.removed[r];
                if (q >= 0 && q < vocab && q >> 8 == t >> 8) first = false;
            }
            if (first) {
                const int w = t / seg, st = (t - w * seg) >> 8;
                float loc[8], lsum;
                int llast;
                step_sums(w, st, loc, lsum, llast);
                lsum = warp_total(lsum);
                if (lane == 0) sm.step[w][st] = lsum;
            }
        }
        __syncthreads();
        // warp 0: the crossing step from running prefixes over (warp, step) in id
        // order (the same numbers in every lane), or, if rounding left the target
        // above the total, the last step with mass; then that step per element
        if (warp == 0) {
            // Step g in id order is step g % nsw of warp g / nsw's segment (nsw = seg /
            // 256 steps each; the last segments hold fewer or none).  Lane l sums the
            // steps [c l, c l + c); a prefix sum over the lanes finds the lane where
            // the running mass passes the target, and that lane walks its steps.
            const int nsw = seg >> 8;
            const int nst = kWarps * nsw;
            const int c = (nst + 31) >> 5;
            auto step_mass = [&](int g) -> float {
                if (g >= nst) return 0.f;
                const int w = g / nsw, st = g - w * nsw;
                const int ws0 = w * seg, ws1 = min(vocab, ws0 + seg);
                const int wn = ws1 > ws0 ? (ws1 - ws0 + 255) / 256 : 0;
                return st < wn ? sm.step[w][st] : 0.f;
            };
            float part = 0.f;
            for (int i = 0; i < c; ++i) part += step_mass(lane * c + i);
            float incl = part;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(FULL, incl, o);
                if (lane >= o) incl += y;
            }
            float excl = __shfl_up_sync(FULL, incl, 1);
            if (lane == 0) excl = 0.f;
            // the lane to walk: the crossing one, or, if rounding left the target at
            // or above the total, the last lane with mass (then its last step with mass)
            const unsigned over = __ballot_sync(FULL, target < incl);
            const unsigned has = __ballot_sync(FULL, part > 0.f);
            const int wl = over ? __ffs(over) - 1 : (has ? 31 - __clz(has) : -1);
            int cw = -1, cs = -1;
            float cpre = 0.f;
            if (wl >= 0) {
                if (lane == wl) {
                    float pre = excl;
                    int fw = -1, fs = -1;
                    float fpre = 0.f;
                    for (int i = 0; i < c; ++i) {
                        const int g = lane * c + i;
                        const float m = step_mass(g);
                        if (over && pre <= target && target < pre + m) {
                            cw = g / nsw;
                            cs = g - cw * nsw;
                            cpre = pre;
                            break;
                        }
                        if (m > 0.f) {
                            fw = g / nsw;
                            fs = g - fw * nsw;
                            fpre = pre;
                        }
                        pre += m;
                    }
                    if (cw < 0) {  // rounding: the lane's last step with mass
                        cw = fw;
                        cs = fs;
                        cpre = fpre;
                    }
                }
                cw = __shfl_sync(FULL, cw, wl);
                cs = __shfl_sync(FULL, cs, wl);
                cpre = __shfl_sync(FULL, cpre, wl);
            }
            int pick = amax;  // no residual mass at all
            if (cw >= 0) {
                float loc[8], lsum;
                int llast;
                step_sums(cw, cs, loc, lsum, llast);
                float incl = lsum;
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(FULL, incl, o);
                    if (lane >= o) incl += y;
                }
                const float base_l = cpre + incl - lsum;  // this lane's prefix
                const int b0 = cw * seg + 256 * cs + 8 * lane;
                const int w1 = min(vocab, cw * seg + seg);
                int mine = -1;  // the lane's first id with mass whose running sum passes the target
                if (base_l + lsum > target)
#pragma unroll
                    for (int k = 7; k >= 0; --k) {
                        const bool mass_k = k == 0 ? loc[0] > 0.f : loc[k] > loc[k - 1];
                        if (b0 + k < w1 && mass_k && base_l + loc[k] > target) mine = b0 + k;
                    }
                const unsigned hit = __ballot_sync(FULL, mine >= 0);
                int lastw = llast;
                for (int o = 16; o > 0; o >>= 1) lastw = max(lastw, __shfl_xor_sync(FULL, lastw, o));
                const int first = __shfl_sync(FULL, mine, hit ? __ffs(hit) - 1 : 0);
                pick = hit ? first : (lastw >= 0 ? lastw : amax);  // rounding: the step's last id with mass
            }
            if (lane == 0) sm.bonus = pick;
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
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(accept_sampled_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kStageVocab * (int)sizeof(float));
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
                                  const int32_t *top_k, const float *top_p, const float *coins,
                                  int coin_stride, int batch,
                                  int max_depth, int32_t *accept_len, int32_t *accepted_nodes,
                                  int32_t *commit_tokens, int32_t *bonus, unsigned int *err,
                                  cudaStream_t s) {
    // rows that fit are staged in shared memory: whole 16-byte units at 16-byte aligned starts
    const int stage = vocab <= kStageVocab && (vocab & 3) == 0 &&
                      (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
    return launch_pdl(accept_sampled_kernel, dim3(batch), dim3(kThreads),
                      stage ? (size_t)vocab * sizeof(float) : 0, s, node_token, first_child, next_sibling,
                      qo_indptr, logits, vocab, temperature, top_k, top_p, coins, coin_stride, max_depth,
                      accept_len, accepted_nodes, commit_tokens, bonus, stage, err);
}

}  // namespace ddt
