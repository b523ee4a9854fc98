// ddt_commit.cu -- KV commit after acceptance.
//
// Page: "The Architecture of a Speculative Decoding Engine", the
// append-then-compact scheme and section "The Final Resolution: A Concrete
// Trace": every tree node's latent was appended after the committed prefix
// (node j at position P + j); after acceptance the accepted nodes' latents
// are gathered into positions P .. P + accept_len - 1 and the cache grows by
// accept_len.  Position c of request b lives in pool row
// kv_indices[kv_indptr[b] + c].
//
// One CTA per request.  At most max_depth + 1 <= 8 rows of 1152 bytes move,
// so the CTA reads every source row into shared memory first and only then
// writes the destinations: a row that is both (node 2 -> position 1 while
// node 5 -> position 2) moves its value from before the commit.  Rows whose
// source and destination coincide (the root, a chain) are not rewritten.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ddt_internal.cuh"

namespace ddt {
namespace {

constexpr int kThreads = 128;
constexpr int kRowVecs = DDT_D * 2 / 16;  // 16-byte pieces per pool row

__global__ void __launch_bounds__(kThreads)
commit_kv_kernel(uint16_t *__restrict__ kv_pool, int64_t pool_rows,
                 const int32_t *__restrict__ kv_indices, const int32_t *__restrict__ kv_indptr,
                 const int32_t *__restrict__ qo_indptr, const int32_t *__restrict__ accept_len,
                 const int32_t *__restrict__ accepted_nodes, int max_depth,
                 int32_t *__restrict__ new_len, unsigned int *err) {
    __shared__ uint4 rows[DDT_MAX_DEPTH + 1][kRowVecs];
    __shared__ int64_t src_row[DDT_MAX_DEPTH + 1], dst_row[DDT_MAX_DEPTH + 1];
    __shared__ int s_n;
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    pdl_trigger();
    // caller inputs first; the accepted path comes from the accept kernel
    const int q0 = qo_indptr[b];
    const int T = qo_indptr[b + 1] - q0;
    const int k0 = kv_indptr[b];
    const int P = kv_indptr[b + 1] - k0 - T;
    const int width = max_depth + 1;
    pdl_wait();
    if (tid < 32) {  // lane k checks and resolves path entry k: three memory round trips in all
        const int lane = tid;
        const unsigned full = 0xffffffffu;
        const int n = accept_len[b];
        const int ak = lane < width ? accepted_nodes[(size_t)b * width + lane] : 0;
        const int aprev = __shfl_up_sync(full, ak, 1);
        const bool bad_entry = lane < n && (lane == 0 ? ak != 0 : (ak <= aprev || ak >= T));
        bool ok = T >= 1 && P >= 0 && n >= 1 && n <= width && n <= T && !__any_sync(full, bad_entry);
        if (!ok && lane == 0) latch(err, DDT_DEVERR_ACCEPTED);
        int64_t sr = 0, dr = 0;
        if (ok && lane < n) {
            sr = kv_indices[k0 + P + ak];
            dr = kv_indices[k0 + P + lane];
        }
        const bool bad_row = ok && lane < n && (sr < 0 || sr >= pool_rows || dr < 0 || dr >= pool_rows);
        if (__any_sync(full, bad_row)) {
            if (lane == 0) latch(err, DDT_DEVERR_KV_INDEX);
            ok = false;
        }
        if (ok && lane < n) {
            src_row[lane] = sr;
            dst_row[lane] = dr;
        }
        if (lane == 0) {
            s_n = ok ? n : 0;
            if (ok && new_len) new_len[b] = P + n;
        }
    }
    __syncthreads();
    const int n = s_n;
    const uint4 *pool_in = reinterpret_cast<const uint4 *>(kv_pool);
    uint4 *pool_out = reinterpret_cast<uint4 *>(kv_pool);
    for (int e = tid; e < n * kRowVecs; e += kThreads) {
        const int k = e / kRowVecs, c = e - k * kRowVecs;
        if (src_row[k] != dst_row[k]) rows[k][c] = pool_in[src_row[k] * kRowVecs + c];
    }
    __syncthreads();
    for (int e = tid; e < n * kRowVecs; e += kThreads) {
        const int k = e / kRowVecs, c = e - k * kRowVecs;
        if (src_row[k] != dst_row[k]) pool_out[dst_row[k] * kRowVecs + c] = rows[k][c];
    }
}

}  // namespace

// the same carveout as the other small kernels (see tree_prepare_device)
cudaError_t commit_prepare_device() {
    return cudaFuncSetAttribute(commit_kv_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                (int)cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_commit_kv(uint16_t *kv_pool, int64_t pool_rows, const int32_t *kv_indices,
                             const int32_t *kv_indptr, const int32_t *qo_indptr,
                             const int32_t *accept_len, const int32_t *accepted_nodes, int batch,
                             int max_depth, int32_t *new_len, unsigned int *err, cudaStream_t s) {
    return launch_pdl(commit_kv_kernel, dim3(batch), dim3(kThreads), 0, s, kv_pool, pool_rows,
                      kv_indices, kv_indptr, qo_indptr, accept_len, accepted_nodes, max_depth,
                      new_len, err);
}

}  // namespace ddt
