// ddt_attn_combine.cu -- log-sum-exp merge of split-KV partial results.
//
// Each split s wrote, for every row (token, head), its normalised partial
// output o_s = sum_j e^{s_j - m_s} v_j / sum_j e^{s_j - m_s} and
// lse_s = log sum_j e^{s_j} over its own kv columns.  The full softmax over
// the union of the splits is  out = sum_s e^{lse_s - LSE} o_s  with
// LSE = log sum_s e^{lse_s}.  A split that saw no visible column carries
// lse_s = -inf and contributes nothing.
// Split-KV with a partial reduction follows "The 30-Column Mask", section
// "The Context: Building a Custom Verify Attention Kernel" (a KV-split
// flash-decode design with partial reduction for occupancy).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ddt_internal.cuh"

namespace ddt {
namespace {

constexpr int kThreads = 128;  // 4 output dims per thread

__global__ void __launch_bounds__(kThreads)
attn_combine_kernel(const float *__restrict__ o_part, const float *__restrict__ lse_part,
                    int num_splits, int64_t rows, float *__restrict__ out,
                    float *__restrict__ lse) {
    pdl_trigger();
    pdl_wait();  // the partials come from the partial pass
    const int64_t row = blockIdx.x;
    if (row >= rows) return;
    // Online merge over groups of four splits: a group's lse values and partial
    // rows are loaded together (one memory round trip per group), then folded
    // into the running max m, weight sum den and weighted sum acc.
    float m = -INFINITY, den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < num_splits; s0 += 4) {
        float ls[4];
        float4 o[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int s = s0 + t;
            ls[t] = (s < num_splits) ? lse_part[(int64_t)s * rows + row] : -INFINITY;
            o[t] = (s < num_splits)
                ? reinterpret_cast<const float4 *>(o_part + ((int64_t)s * rows + row) * DDT_DL)[threadIdx.x]
                : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mg = m;
#pragma unroll
        for (int t = 0; t < 4; ++t) mg = fmaxf(mg, ls[t]);
        if (mg == -INFINITY) continue;  // nothing visible so far
        const float c = (m == -INFINITY) ? 0.f : __expf(m - mg);  // rescale of the running sums
        den *= c;
        acc.x *= c; acc.y *= c; acc.z *= c; acc.w *= c;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            if (ls[t] == -INFINITY) continue;  // a split that saw no column
            const float w = __expf(ls[t] - mg);
            den += w;
            acc.x += w * o[t].x; acc.y += w * o[t].y; acc.z += w * o[t].z; acc.w += w * o[t].w;
        }
        m = mg;
    }
    if (m != -INFINITY) {
        const float inv = 1.f / den;
        acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
    }
    reinterpret_cast<float4 *>(out + row * DDT_DL)[threadIdx.x] = acc;
    if (lse && threadIdx.x == 0) lse[row] = (m == -INFINITY) ? -INFINITY : m + logf(den);
}

}  // namespace

// same shared-memory carveout as the partial pass it overlaps (see tree_prepare_device)
cudaError_t attn_combine_prepare_device() {
    return cudaFuncSetAttribute(attn_combine_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                (int)cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_attn_combine(const AttnArgs &a, cudaStream_t s) {
    const int64_t rows = (int64_t)a.total_q * a.num_heads;
    if (rows == 0) return cudaSuccess;
    return launch_pdl(attn_combine_kernel, dim3((unsigned)rows), dim3(kThreads), 0, s, a.o_part,
                      a.lse_part, a.num_splits, rows, a.out, a.lse);
}

}  // namespace ddt
