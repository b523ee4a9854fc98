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

constexpr int kThreads = 128;    // 4 output dims per thread
constexpr int kRowsPerCta = 2;   // rows merged by one CTA, their loads issued together

// Online merge over groups of four splits: a group's lse values and partial
// rows (for all of the CTA's rows) are loaded together -- one memory round
// trip per group -- then folded into the running max m, weight sum den and
// weighted sum acc of each row.
__global__ void __launch_bounds__(kThreads)
attn_combine_kernel(const float *__restrict__ o_part, const float *__restrict__ lse_part,
                    int num_splits, int64_t rows, float *__restrict__ out,
                    float *__restrict__ lse) {
    pdl_trigger();
    pdl_wait();  // the partials come from the partial pass
    const int64_t row0 = (int64_t)blockIdx.x * kRowsPerCta;
    float m[kRowsPerCta], den[kRowsPerCta];
    float4 acc[kRowsPerCta];
#pragma unroll
    for (int r = 0; r < kRowsPerCta; ++r) {
        m[r] = -INFINITY;
        den[r] = 0.f;
        acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int s0 = 0; s0 < num_splits; s0 += 4) {
        float ls[kRowsPerCta][4];
        float4 o[kRowsPerCta][4];
#pragma unroll
        for (int r = 0; r < kRowsPerCta; ++r) {
            const int64_t row = row0 + r;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int s = s0 + t;
                const bool in = s < num_splits && row < rows;
                ls[r][t] = in ? lse_part[(int64_t)s * rows + row] : -INFINITY;
                o[r][t] = in ? reinterpret_cast<const float4 *>(o_part + ((int64_t)s * rows + row) * DDT_DL)[threadIdx.x]
                             : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int r = 0; r < kRowsPerCta; ++r) {
            float mg = m[r];
#pragma unroll
            for (int t = 0; t < 4; ++t) mg = fmaxf(mg, ls[r][t]);
            if (mg == -INFINITY) continue;  // nothing visible so far
            const float c = (m[r] == -INFINITY) ? 0.f : __expf(m[r] - mg);  // rescale of the running sums
            den[r] *= c;
            acc[r].x *= c; acc[r].y *= c; acc[r].z *= c; acc[r].w *= c;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                if (ls[r][t] == -INFINITY) continue;  // a split that saw no column
                const float w = __expf(ls[r][t] - mg);
                den[r] += w;
                acc[r].x += w * o[r][t].x; acc[r].y += w * o[r][t].y;
                acc[r].z += w * o[r][t].z; acc[r].w += w * o[r][t].w;
            }
            m[r] = mg;
        }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerCta; ++r) {
        const int64_t row = row0 + r;
        if (row >= rows) break;
        float4 v = acc[r];
        if (m[r] != -INFINITY) {
            const float inv = 1.f / den[r];
            v.x *= inv; v.y *= inv; v.z *= inv; v.w *= inv;
        }
        reinterpret_cast<float4 *>(out + row * DDT_DL)[threadIdx.x] = v;
        if (lse && threadIdx.x == 0) lse[row] = (m[r] == -INFINITY) ? -INFINITY : m[r] + logf(den[r]);
    }
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
    const int64_t ctas = (rows + kRowsPerCta - 1) / kRowsPerCta;
    return launch_pdl(attn_combine_kernel, dim3((unsigned)ctas), dim3(kThreads), 0, s, a.o_part,
                      a.lse_part, a.num_splits, rows, a.out, a.lse);
}

}  // namespace ddt
