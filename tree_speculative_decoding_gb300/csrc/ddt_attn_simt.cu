// ddt_attn_simt.cu -- CUDA-core tree-verify attention (bring-up and
// cross-check path).  One CTA = one tree node (query), 16 heads, one kv split.
// The 16 heads share the node's mask row and every staged KV row.
//
// Computes, per row (node i, head h), over kv columns j visible in mask row i:
//   s_j = scale * <q[i,h,0:576], kv[idx_j, 0:576]>,  out = softmax(s) @ kv[idx, 0:512]
// ("The Architecture of a Speculative Decoding Engine", section "The Forward
// Pass Pseudocode"; "The 30-Column Mask", sections "The Message: Tensor Shapes
// as Evidence" and "The Fix: Building Combined Indices").
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ddt_internal.cuh"

namespace ddt {
namespace {

constexpr int kHeads = 16;         // heads per CTA
constexpr int kTile = 32;          // kv rows staged per step
constexpr int kThreads = 256;
constexpr int kWords = DDT_D / 2;  // 288 bf16x2 words per row
constexpr int kKvStride = kWords + 1;  // odd word stride: conflict-free column reads
constexpr float kLog2e = 1.4426950408889634f;
constexpr size_t kSmemBytes =
    sizeof(uint32_t) * (kHeads * kWords + kTile * kKvStride + kHeads * (kTile + 1) + kTile);

__device__ __forceinline__ float2 bf2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__global__ void __launch_bounds__(kThreads)
attn_simt_kernel(AttnArgs a) {
    extern __shared__ __align__(16) uint32_t smem_simt[];
    auto q_s = reinterpret_cast<uint32_t(*)[kWords]>(smem_simt);
    auto kv_s = reinterpret_cast<uint32_t(*)[kKvStride]>(smem_simt + kHeads * kWords);
    auto s_s = reinterpret_cast<float(*)[kTile + 1]>(smem_simt + kHeads * kWords + kTile * kKvStride);
    int *slot_s = reinterpret_cast<int *>(smem_simt + kHeads * kWords + kTile * kKvStride +
                                          kHeads * (kTile + 1));

    const int tid = threadIdx.x;
    const int b = blockIdx.z;
    const int hgroups = (a.num_heads + kHeads - 1) / kHeads;
    const int i = blockIdx.y / hgroups;
    const int h0 = (blockIdx.y % hgroups) * kHeads;
    const int split = blockIdx.x;

    const int qo0 = a.qo_indptr[b];
    const int T = a.qo_indptr[b + 1] - qo0;
    if (i >= T) return;
    const int kv0 = a.kv_indptr[b];
    const int N = a.kv_indptr[b + 1] - kv0;
    if (T > a.max_q_len || N < T || N > a.max_kv_len) {
        if (tid == 0) latch(a.err, T > a.max_q_len ? DDT_DEVERR_QO_INDPTR : DDT_DEVERR_KV_INDPTR);
        return;
    }
    const int P = N - T;
    const int W = (N + 31) >> 5;
    if (a.mask_indptr[b + 1] - a.mask_indptr[b] != T * W) {
        if (tid == 0) latch(a.err, DDT_DEVERR_MASK_INDPTR);
        return;
    }
    const uint32_t *mrow = a.mask + a.mask_indptr[b] + (int64_t)i * W;
    // node i sees nothing beyond its own column P + i (ancestors precede it)
    const int kv_end = P + i + 1;
    const int c_begin = split * a.split_cols;
    const int c_end = min(kv_end, c_begin + a.split_cols);

    const int t = qo0 + i;
    for (int e = tid; e < kHeads * kWords; e += kThreads) {
        const int hh = e / kWords, w = e % kWords;
        const int h = h0 + hh;
        q_s[hh][w] = (h < a.num_heads)
            ? reinterpret_cast<const uint32_t *>(a.q + ((int64_t)t * a.num_heads + h) * DDT_D)[w]
            : 0u;
    }

    // PV mapping: thread owns head hh2 and words sub + 16k (k < 16) of the latent
    const int hh2 = tid >> 4;
    const int sub = tid & 15;
    float acc[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) acc[k] = 0.f;
    float m = -INFINITY, l = 0.f;
    const float sc = a.scale * kLog2e;

    for (int c0 = c_begin; c0 < c_end; c0 += kTile) {
        __syncthreads();
        if (tid < kTile) {
            const int c = c0 + tid;
            int slot = 0;
            if (c < c_end) {
                slot = a.kv_indices[kv0 + c];
                if (slot < 0 || (int64_t)slot >= a.pool_rows) {
                    latch(a.err, DDT_DEVERR_KV_INDEX);
                    slot = -1;
                }
            } else {
                slot = -1;
            }
            slot_s[tid] = slot;
        }
        __syncthreads();
        for (int e = tid; e < kTile * kWords; e += kThreads) {
            const int j = e / kWords, w = e % kWords;
            const int slot = slot_s[j];
            kv_s[j][w] = (slot >= 0)
                ? reinterpret_cast<const uint32_t *>(a.kv_pool + (int64_t)slot * DDT_D)[w]
                : 0u;
        }
        __syncthreads();
        // scores: pair p -> head p/32, kv row p%32
        const uint32_t mword = (c0 < P && c0 + kTile <= P) ? 0xffffffffu : mrow[c0 >> 5];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int p = tid + e * kThreads;
            const int hh = p >> 5, j = p & 31;
            float dot = 0.f;
#pragma unroll 8
            for (int w = 0; w < kWords; ++w) {
                const float2 qa = bf2(q_s[hh][w]);
                const float2 kb = bf2(kv_s[j][w]);
                dot = fmaf(qa.x, kb.x, dot);
                dot = fmaf(qa.y, kb.y, dot);
            }
            const int c = c0 + j;
            const bool vis = c < c_end && slot_s[j] >= 0 && ((mword >> (c & 31)) & 1u);
            s_s[hh][j] = vis ? dot * sc : -INFINITY;
        }
        __syncthreads();
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < kTile; ++j) mt = fmaxf(mt, s_s[hh2][j]);
        const float m_new = fmaxf(m, mt);
        if (m_new == -INFINITY) continue;  // nothing visible yet
        const float alpha = exp2f(m - m_new);
        m = m_new;
        l *= alpha;
#pragma unroll
        for (int k = 0; k < 32; ++k) acc[k] *= alpha;
        for (int j = 0; j < kTile; ++j) {
            const float pj = exp2f(s_s[hh2][j] - m);
            l += pj;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float2 v = bf2(kv_s[j][sub + 16 * k]);
                acc[2 * k] = fmaf(pj, v.x, acc[2 * k]);
                acc[2 * k + 1] = fmaf(pj, v.y, acc[2 * k + 1]);
            }
        }
    }

    const int h = h0 + hh2;
    if (h >= a.num_heads) return;
    const int64_t row = (int64_t)t * a.num_heads + h;
    const int64_t rows = (int64_t)a.total_q * a.num_heads;
    const bool any = (m != -INFINITY);
    const float inv = any ? 1.f / l : 0.f;
    const float lse_v = any ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
    float *o;
    float *lp;
    if (a.num_splits > 1) {
        o = a.o_part + ((int64_t)split * rows + row) * DDT_DL;
        lp = a.lse_part + (int64_t)split * rows + row;
    } else {
        o = a.out + row * DDT_DL;
        lp = a.lse ? a.lse + row : nullptr;
    }
#pragma unroll
    for (int k = 0; k < 16; ++k)
        reinterpret_cast<float2 *>(o)[sub + 16 * k] = make_float2(acc[2 * k] * inv, acc[2 * k + 1] * inv);
    if (sub == 0 && lp) *lp = lse_v;
}

}  // namespace

cudaError_t attn_simt_prepare_device() {
    return cudaFuncSetAttribute(attn_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemBytes);
}

cudaError_t launch_attn_simt(const AttnArgs &a, cudaStream_t s) {
    const int hgroups = (a.num_heads + kHeads - 1) / kHeads;
    dim3 grid(a.num_splits, a.max_q_len * hgroups, a.batch);
    attn_simt_kernel<<<grid, kThreads, kSmemBytes, s>>>(a);
    return cudaGetLastError();
}

}  // namespace ddt
