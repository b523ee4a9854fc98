// ddt_abi.cu -- the extern "C" entry points of libddt.so: host-side argument
// checks, split-KV sizing, launches, and the per-device error word.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <new>

#include "ddt_internal.cuh"

namespace {

// Per-device error word: kernels atomicOr DDT_DEVERR_* bits into it.
__device__ unsigned int g_ddt_error_word;

constexpr int kMaxDevices = 64;

struct DeviceState {
    // set (release) after err and num_sms are written; read (acquire) before
    // they are used, so a thread that sees it set also sees them
    std::atomic<bool> ready{false};
    unsigned int *err = nullptr;  // device address of g_ddt_error_word
    int num_sms = 0;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

// Set up (once per device, with that device current) the error-word address,
// the SM count and kernel attributes.  The first entry-point call on a device
// performs this set-up, so it should come before any stream capture.  Returns
// null on failure.
DeviceState *device_state() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    DeviceState &st = g_dev[dev];
    if (st.ready.load(std::memory_order_acquire)) return &st;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!st.ready.load(std::memory_order_relaxed)) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ddt_error_word) != cudaSuccess) return nullptr;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return nullptr;
        if (ddt::attn_prepare_device() != cudaSuccess) return nullptr;
        st.err = static_cast<unsigned int *>(p);
        st.num_sms = sms;
        st.ready.store(true, std::memory_order_release);
    }
    return &st;
}

inline cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int choose_splits(int batch, int num_heads, int max_q_len, int max_kv_len, int num_sms) {
    return ddt::attn_choose_splits(batch, num_heads, max_q_len, max_kv_len, num_sms);
}

}  // namespace

extern "C" {

const char *ddt_status_string(ddt_status s) {
    switch (s) {
        case DDT_OK: return "ok";
        case DDT_ERR_INVALID_ARG: return "invalid argument";
        case DDT_ERR_UNSUPPORTED: return "unsupported size";
        case DDT_ERR_WORKSPACE: return "workspace missing or too small";
        case DDT_ERR_CUDA: return "CUDA error";
        case DDT_ERR_DEVICE_CHECK: return "device-side data check failed";
        case DDT_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

int32_t ddt_abi_version(void) { return DDT_ABI_VERSION; }

ddt_status ddt_build_tree(const float *topk_logp, const int32_t *topk_ids,
                          const int32_t *root_id, const int32_t *budget,
                          const int32_t *qo_indptr, int32_t batch, int32_t max_depth,
                          int32_t topk, int32_t *node_token, int32_t *parent, int32_t *depth,
                          void *stream) {
    if (!topk_logp || !topk_ids || !root_id || !budget || !qo_indptr || !node_token ||
        !parent || !depth || batch < 0)
        return DDT_ERR_INVALID_ARG;
    if (max_depth < 1 || max_depth > DDT_MAX_DEPTH || topk < 1 || topk > DDT_MAX_TOPK)
        return DDT_ERR_UNSUPPORTED;
    if (batch == 0) return DDT_OK;
    DeviceState *st = device_state();
    if (!st) return DDT_ERR_CUDA;
    cudaError_t e = ddt::launch_build_tree(topk_logp, topk_ids, root_id, budget, qo_indptr, batch,
                                           max_depth, topk, node_token, parent, depth, st->err,
                                           as_stream(stream));
    return e == cudaSuccess ? DDT_OK : DDT_ERR_CUDA;
}

ddt_status ddt_mask_indptr(const int32_t *qo_indptr, const int32_t *prefix_len, int32_t batch,
                           int32_t *mask_indptr) {
    if (!qo_indptr || !prefix_len || !mask_indptr || batch < 0) return DDT_ERR_INVALID_ARG;
    int64_t off = 0;
    for (int b = 0; b < batch; ++b) {
        const int64_t T = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
        const int64_t P = prefix_len[b];
        if (T < 1 || P < 0) return DDT_ERR_INVALID_ARG;
        mask_indptr[b] = (int32_t)off;
        off += T * ((P + T + 31) / 32);
        if (off > INT32_MAX) return DDT_ERR_INVALID_ARG;
    }
    mask_indptr[batch] = (int32_t)off;
    return DDT_OK;
}

ddt_status ddt_compile_visibility(const int32_t *parent, const int32_t *qo_indptr,
                                  const int32_t *prefix_len, const int32_t *mask_indptr,
                                  int32_t batch, int32_t total_words, uint32_t *mask,
                                  void *stream) {
    if (!parent || !qo_indptr || !prefix_len || !mask_indptr || !mask || batch < 0 ||
        total_words < 0)
        return DDT_ERR_INVALID_ARG;
    if (batch == 0 || total_words == 0) return DDT_OK;
    DeviceState *st = device_state();
    if (!st) return DDT_ERR_CUDA;
    cudaError_t e = ddt::launch_compile_visibility(parent, qo_indptr, prefix_len, mask_indptr,
                                                   batch, total_words, mask, st->err,
                                                   as_stream(stream));
    return e == cudaSuccess ? DDT_OK : DDT_ERR_CUDA;
}

ddt_status ddt_build_tree_visibility(const float *topk_logp, const int32_t *topk_ids,
                                     const int32_t *root_id, const int32_t *budget,
                                     const int32_t *qo_indptr, const int32_t *prefix_len,
                                     const int32_t *mask_indptr, int32_t batch, int32_t max_depth,
                                     int32_t topk, int32_t *node_token, int32_t *parent,
                                     int32_t *depth, uint32_t *mask, void *stream) {
    if (!topk_logp || !topk_ids || !root_id || !budget || !qo_indptr || !prefix_len ||
        !mask_indptr || !node_token || !parent || !depth || !mask || batch < 0)
        return DDT_ERR_INVALID_ARG;
    if (max_depth < 1 || max_depth > DDT_MAX_DEPTH || topk < 1 || topk > DDT_MAX_TOPK)
        return DDT_ERR_UNSUPPORTED;
    if (batch == 0) return DDT_OK;
    DeviceState *st = device_state();
    if (!st) return DDT_ERR_CUDA;
    cudaError_t e = ddt::launch_build_tree_visibility(topk_logp, topk_ids, root_id, budget,
                                                      qo_indptr, batch, max_depth, topk, prefix_len,
                                                      mask_indptr, node_token, parent, depth, mask,
                                                      st->err, as_stream(stream));
    return e == cudaSuccess ? DDT_OK : DDT_ERR_CUDA;
}

ddt_status ddt_build_chain_visibility(const int32_t *qo_indptr, const int32_t *prefix_len,
                                      const int32_t *mask_indptr, int32_t batch, int32_t *parent,
                                      int32_t *depth, uint32_t *mask, void *stream) {
    if (!qo_indptr || !prefix_len || !mask_indptr || !parent || !depth || !mask || batch < 0)
        return DDT_ERR_INVALID_ARG;
    if (batch == 0) return DDT_OK;
    DeviceState *st = device_state();
    if (!st) return DDT_ERR_CUDA;
    cudaError_t e = ddt::launch_build_chain_visibility(qo_indptr, prefix_len, mask_indptr, batch,
                                                       parent, depth, mask, st->err,
                                                       as_stream(stream));
    return e == cudaSuccess ? DDT_OK : DDT_ERR_CUDA;
}

int32_t ddt_verify_attn_num_splits(int32_t batch, int32_t num_heads, int32_t max_q_len,
                                   int32_t max_kv_len, int32_t num_sms) {
    if (batch < 1 || num_heads < 1 || max_q_len < 1 || max_kv_len < 1) return 1;
    if (num_sms <= 0) {
        DeviceState *st = device_state();
        num_sms = st ? st->num_sms : 148;
    }
    return choose_splits(batch, num_heads, max_q_len, max_kv_len, num_sms);
}

int32_t ddt_verify_attn_launched_splits(int32_t max_kv_len, int32_t num_splits) {
    if (max_kv_len < 1 || num_splits < 1) return 1;
    return ddt::attn_launched_splits(max_kv_len, num_splits);
}

size_t ddt_verify_attn_workspace_size(int32_t total_q, int32_t num_heads, int32_t num_splits) {
    if (total_q < 1 || num_heads < 1 || num_splits <= 1) return 0;
    const size_t rows = (size_t)total_q * num_heads;
    return align256(rows * num_splits * DDT_DL * sizeof(float)) +
           align256(rows * num_splits * sizeof(float));
}

}  // extern "C"

namespace {
// ddt_verify_attn with the mask's provenance: tree_mask = 1 only where the
// mask was built by this library's tree + visibility kernel earlier in the
// same step (ddt_verify_step), so that its prefix columns are known visible.
ddt_status verify_attn_impl(const uint16_t *q, const uint16_t *kv_pool, int64_t pool_rows,
                            const int32_t *kv_indices, const int32_t *kv_indptr,
                            const int32_t *qo_indptr, const uint32_t *mask,
                            const int32_t *mask_indptr, int32_t batch, int32_t num_heads,
                            int32_t total_q, int32_t max_q_len, int32_t max_kv_len, float scale,
                            int32_t num_splits, float *out, float *lse, void *workspace,
                            size_t workspace_bytes, void *stream, int tree_mask) {
    if (!q || !kv_pool || !kv_indices || !kv_indptr || !qo_indptr || !mask || !mask_indptr ||
        !out)
        return DDT_ERR_INVALID_ARG;
    if (batch < 1 || num_heads < 1 || total_q < batch || pool_rows < 1 || max_q_len < 1 ||
        max_kv_len < max_q_len || !isfinite(scale) || num_splits < 0)
        return DDT_ERR_INVALID_ARG;
    if (max_q_len > DDT_MAX_Q_LEN || num_heads > 128 || num_splits > DDT_MAX_SPLITS)
        return DDT_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(kv_pool) & 15u) || (reinterpret_cast<uintptr_t>(q) & 15u) ||
        (reinterpret_cast<uintptr_t>(out) & 15u))
        return DDT_ERR_INVALID_ARG;
    DeviceState *st = device_state();
    if (!st) return DDT_ERR_CUDA;

    const int requested = num_splits > 0
        ? num_splits
        : choose_splits(batch, num_heads, max_q_len, max_kv_len, st->num_sms);
    int split_cols = 0, splits = 1;
    ddt::attn_split_layout(max_kv_len, requested, &split_cols, &splits);

    ddt::AttnArgs a;
    memset(&a, 0, sizeof a);
    a.q = q;
    a.kv_pool = kv_pool;
    a.pool_rows = pool_rows;
    a.kv_indices = kv_indices;
    a.kv_indptr = kv_indptr;
    a.qo_indptr = qo_indptr;
    a.mask = mask;
    a.mask_indptr = mask_indptr;
    a.batch = batch;
    a.num_heads = num_heads;
    a.total_q = total_q;
    a.max_q_len = max_q_len;
    a.max_kv_len = max_kv_len;
    a.scale = scale;
    a.num_splits = splits;
    a.split_cols = split_cols;
    a.tree_mask = tree_mask;
    a.out = out;
    a.lse = lse;
    a.err = st->err;
    if (splits > 1) {
        const size_t need = ddt_verify_attn_workspace_size(total_q, num_heads, splits);
        if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
            return DDT_ERR_WORKSPACE;
        const size_t rows = (size_t)total_q * num_heads;
        a.o_part = static_cast<float *>(workspace);
        a.lse_part = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                               align256(rows * splits * DDT_DL * sizeof(float)));
    }
    cudaStream_t s = as_stream(stream);
    cudaError_t e = ddt::launch_attn_partial(a, s);
    if (e == cudaSuccess && splits > 1) e = ddt::launch_attn_combine(a, s);
    return e == cudaSuccess ? DDT_OK : DDT_ERR_CUDA;
}
}  // namespace

extern "C" {

ddt_status ddt_verify_attn(const uint16_t *q, const uint16_t *kv_pool, int64_t pool_rows,
                           const int32_t *kv_indices, const int32_t *kv_indptr,
                           const int32_t *qo_indptr, const uint32_t *mask,
                           const int32_t *mask_indptr, int32_t batch, int32_t num_heads,
                           int32_t total_q, int32_t max_q_len, int32_t max_kv_len, float scale,
                           int32_t num_splits, float *out, float *lse, void *workspace,
                           size_t workspace_bytes, void *stream) {
    return verify_attn_impl(q, kv_pool, pool_rows, kv_indices, kv_indptr, qo_indptr, mask,
                            mask_indptr, batch, num_heads, total_q, max_q_len, max_kv_len, scale,
                            num_splits, out, lse, workspace, workspace_bytes, stream, 0);
}

ddt_status ddt_accept(const int32_t *node_token, const int32_t *parent,
                      const int32_t *qo_indptr, const int32_t *target_argmax, int32_t batch,
                      int32_t max_depth, int32_t *accept_len, int32_t *accepted_nodes,
                      int32_t *commit_tokens, int32_t *bonus, void *stream) {
    if (!node_token || !parent || !qo_indptr || !target_argmax || !accept_len ||
        !accepted_nodes || !commit_tokens || !bonus || batch < 0)
        return DDT_ERR_INVALID_ARG;
    if (max_depth < 1 || max_depth > DDT_MAX_DEPTH) return DDT_ERR_UNSUPPORTED;
    if (batch == 0) return DDT_OK;
    DeviceState *st = device_state();
    if (!st) return DDT_ERR_CUDA;
    cudaError_t e = ddt::launch_accept(node_token, parent, qo_indptr, target_argmax, batch,
                                       max_depth, accept_len, accepted_nodes, commit_tokens,
                                       bonus, st->err, as_stream(stream));
    return e == cudaSuccess ? DDT_OK : DDT_ERR_CUDA;
}

ddt_status ddt_commit_kv(uint16_t *kv_pool, int64_t pool_rows, const int32_t *kv_indices,
                         const int32_t *kv_indptr, const int32_t *qo_indptr,
                         const int32_t *accept_len, const int32_t *accepted_nodes, int32_t batch,
                         int32_t max_depth, int32_t *new_len, void *stream) {
    if (!kv_pool || !kv_indices || !kv_indptr || !qo_indptr || !accept_len || !accepted_nodes ||
        batch < 0 || pool_rows < 1 || (reinterpret_cast<uintptr_t>(kv_pool) & 15u))
        return DDT_ERR_INVALID_ARG;
    if (max_depth < 1 || max_depth > DDT_MAX_DEPTH) return DDT_ERR_UNSUPPORTED;
    if (batch == 0) return DDT_OK;
    DeviceState *st = device_state();
    if (!st) return DDT_ERR_CUDA;
    cudaError_t e = ddt::launch_commit_kv(kv_pool, pool_rows, kv_indices, kv_indptr, qo_indptr,
                                          accept_len, accepted_nodes, batch, max_depth, new_len,
                                          st->err, as_stream(stream));
    return e == cudaSuccess ? DDT_OK : DDT_ERR_CUDA;
}

ddt_status ddt_tree_links(const int32_t *parent, const int32_t *qo_indptr, int32_t batch,
                          int32_t *first_child, int32_t *next_sibling, int32_t *retrieve_index,
                          void *stream) {
    if (!parent || !qo_indptr || !first_child || !next_sibling || !retrieve_index || batch < 0)
        return DDT_ERR_INVALID_ARG;
    if (batch == 0) return DDT_OK;
    DeviceState *st = device_state();
    if (!st) return DDT_ERR_CUDA;
    cudaError_t e = ddt::launch_tree_links(parent, qo_indptr, batch, first_child, next_sibling,
                                           retrieve_index, st->err, as_stream(stream));
    return e == cudaSuccess ? DDT_OK : DDT_ERR_CUDA;
}

ddt_status ddt_accept_sampled(const int32_t *node_token, const int32_t *first_child,
                              const int32_t *next_sibling, const int32_t *qo_indptr,
                              const float *target_logits, int32_t vocab, const float *temperature,
                              const int32_t *top_k, const float *top_p, const float *coins,
                              int32_t coin_stride,
                              int32_t batch, int32_t max_depth, int32_t *accept_len,
                              int32_t *accepted_nodes, int32_t *commit_tokens, int32_t *bonus,
                              void *stream) {
    if (!node_token || !first_child || !next_sibling || !qo_indptr || !target_logits ||
        !temperature || !top_k || !coins || !accept_len || !accepted_nodes || !commit_tokens ||
        !bonus || batch < 0 || vocab < 1 || coin_stride < 1)
        return DDT_ERR_INVALID_ARG;
    if (max_depth < 1 || max_depth > DDT_MAX_DEPTH || vocab > DDT_MAX_VOCAB) return DDT_ERR_UNSUPPORTED;
    if (batch == 0) return DDT_OK;
    DeviceState *st = device_state();
    if (!st) return DDT_ERR_CUDA;
    cudaError_t e = ddt::launch_accept_sampled(node_token, first_child, next_sibling, qo_indptr,
                                               target_logits, vocab, temperature, top_k, top_p,
                                               coins,
                                               coin_stride, batch, max_depth, accept_len,
                                               accepted_nodes, commit_tokens, bonus, st->err,
                                               as_stream(stream));
    return e == cudaSuccess ? DDT_OK : DDT_ERR_CUDA;
}

ddt_status ddt_get_error(void *stream, uint32_t *device_error) {
    DeviceState *st = device_state();
    if (!st) return DDT_ERR_CUDA;
    cudaStream_t s = as_stream(stream);
    unsigned int word = 0;
    if (cudaMemcpyAsync(&word, st->err, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(st->err, 0, sizeof word, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return DDT_ERR_CUDA;
    if (device_error) *device_error = word;
    if (word == 0) return DDT_OK;
    return (word & DDT_DEVERR_TIMEOUT) ? DDT_ERR_TIMEOUT : DDT_ERR_DEVICE_CHECK;
}

ddt_status ddt_selftest_wait_timeout(uint32_t poll_limit, void *stream) {
    if (poll_limit < 1 || poll_limit > (1u << 24)) return DDT_ERR_INVALID_ARG;
    DeviceState *st = device_state();
    if (!st) return DDT_ERR_CUDA;
    cudaError_t e = ddt::launch_wait_timeout_selftest(poll_limit, st->err, as_stream(stream));
    return e == cudaSuccess ? DDT_OK : DDT_ERR_CUDA;
}

// ---------------------------------------------------------------- one-call step

ddt_status ddt_verify_step(const ddt_step_args *a, void *stream) {
    if (!a) return DDT_ERR_INVALID_ARG;
    ddt_status st = ddt_build_tree_visibility(a->topk_logp, a->topk_ids, a->root_id, a->budget,
                                              a->qo_indptr, a->prefix_len, a->mask_indptr,
                                              a->batch, a->max_depth, a->topk, a->node_token,
                                              a->parent, a->depth, a->mask, stream);
    if (st != DDT_OK) return st;
    // the mask was just built by ddt_build_tree_visibility: a tree mask
    st = verify_attn_impl(a->q, a->kv_pool, a->pool_rows, a->kv_indices, a->kv_indptr,
                          a->qo_indptr, a->mask, a->mask_indptr, a->batch, a->num_heads,
                          a->total_q, a->max_q_len, a->max_kv_len, a->scale, a->num_splits,
                          a->out, a->lse, a->workspace, a->workspace_bytes, stream, 1);
    if (st != DDT_OK) return st;
    st = ddt_accept(a->node_token, a->parent, a->qo_indptr, a->target_argmax, a->batch,
                    a->max_depth, a->accept_len, a->accepted_nodes, a->commit_tokens, a->bonus,
                    stream);
    if (st != DDT_OK || !a->commit_kv) return st;
    return ddt_commit_kv(a->kv_pool, a->pool_rows, a->kv_indices, a->kv_indptr, a->qo_indptr,
                         a->accept_len, a->accepted_nodes, a->batch, a->max_depth, a->new_len,
                         stream);
}

ddt_status ddt_prefill_step(const ddt_step_args *a, void *stream) {
    if (!a) return DDT_ERR_INVALID_ARG;
    ddt_status st = ddt_build_chain_visibility(a->qo_indptr, a->prefix_len, a->mask_indptr,
                                               a->batch, a->parent, a->depth, a->mask, stream);
    if (st != DDT_OK) return st;
    // the causal chain's mask was just built here: every prefix column is
    // visible and no row sees a column after its own token
    return verify_attn_impl(a->q, a->kv_pool, a->pool_rows, a->kv_indices, a->kv_indptr,
                            a->qo_indptr, a->mask, a->mask_indptr, a->batch, a->num_heads,
                            a->total_q, a->max_q_len, a->max_kv_len, a->scale, a->num_splits,
                            a->out, a->lse, a->workspace, a->workspace_bytes, stream, 1);
}

struct ddt_step_graph {
    cudaGraphExec_t exec = nullptr;
};

}  // extern "C"

namespace {
struct StepIO {
    const void *h_in = nullptr;
    void *d_in = nullptr;
    size_t in_bytes = 0;
    void *h_out = nullptr;
    const void *d_out = nullptr;
    size_t out_bytes = 0;
};

bool is_pinned_host(const void *p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // pageable memory on older runtimes reports an error
        return false;
    }
    return at.type == cudaMemoryTypeHost;
}

// Host buffers are pinned host memory, which the GPU reads and writes over the
// host link through a device pointer (cudaHostGetDevicePointer).  A kernel with
// one 16-byte load per thread, all in flight at once, moves a step's inputs in a
// fraction of a copy-engine transfer's latency.  Each thread copies up to four
// 16-byte units, loads first.
__device__ unsigned int g_io_edge;  // target of the memset that orders the step after the copy
__global__ void __launch_bounds__(256) io_copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                      size_t n16) {
    ddt::pdl_trigger();
    ddt::pdl_wait();  // the output copy may start before the step's last kernel has finished
    const size_t i0 = (size_t)blockIdx.x * 1024 + threadIdx.x;
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (i0 + 256 * k < n16) v[k] = src[i0 + 256 * k];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (i0 + 256 * k < n16) dst[i0 + 256 * k] = v[k];
}

// The device view of a pinned host buffer for a kernel copy of `bytes`, or null
// when a copy engine transfer must do (no device pointer, 16-byte units only).
const void *io_device_view(const void *host, const void *dev, size_t bytes) {
    void *d = nullptr;
    if (cudaHostGetDevicePointer(&d, const_cast<void *>(host), 0) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if ((reinterpret_cast<uintptr_t>(d) | reinterpret_cast<uintptr_t>(dev) | bytes) & 15u) return nullptr;
    return d;
}

cudaError_t io_copy(const void *src, void *dst, size_t bytes, cudaStream_t s) {
    const size_t n16 = bytes / 16;
    const unsigned ctas = (unsigned)((n16 + 1023) / 1024);
    return ddt::launch_pdl(io_copy_kernel, dim3(ctas), dim3(256), 0, s, static_cast<const uint4 *>(src),
                           static_cast<uint4 *>(dst), n16);
}

// Captures [H2D copy] -> ddt_verify_step -> [D2H copy] on a private stream and
// instantiates it.  The copies are kernels over the host buffers' device views
// where possible (else copy-engine transfers).  A 4-byte memset node follows the
// input copy: the step's first kernel is launched for programmatic dependent
// launch and reads caller inputs before its wait, and an edge from a non-kernel
// node is an ordinary one, so the step starts only after the copy is complete.
// The output copy is launched like the step's kernels and waits on the device for
// the step's last kernel before it reads anything.
ddt_status step_graph_create(const ddt_step_args *a, const StepIO &io, ddt_step_graph **graph) {
    if (!a || !graph) return DDT_ERR_INVALID_ARG;
    *graph = nullptr;
    if (!device_state()) return DDT_ERR_CUDA;  // one-time set-up outside the capture
    cudaStream_t s = nullptr;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return DDT_ERR_CUDA;
    ddt_status st = DDT_ERR_CUDA;
    cudaGraph_t g = nullptr;
    const void *in_view = io.in_bytes ? io_device_view(io.h_in, io.d_in, io.in_bytes) : nullptr;
    const void *out_view = io.out_bytes ? io_device_view(io.h_out, io.d_out, io.out_bytes) : nullptr;
    void *edge = nullptr;
    if (in_view && cudaGetSymbolAddress(&edge, g_io_edge) != cudaSuccess) {
        cudaGetLastError();
        in_view = nullptr;
    }
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
        st = DDT_OK;
        if (io.in_bytes) {
            const bool ok = in_view ? (io_copy(in_view, io.d_in, io.in_bytes, s) == cudaSuccess &&
                                       cudaMemsetAsync(edge, 0, sizeof(unsigned int), s) == cudaSuccess)
                                    : cudaMemcpyAsync(io.d_in, io.h_in, io.in_bytes, cudaMemcpyHostToDevice,
                                                      s) == cudaSuccess;
            if (!ok) st = DDT_ERR_CUDA;
        }
        if (st == DDT_OK) st = ddt_verify_step(a, s);
        if (st == DDT_OK && io.out_bytes) {
            const bool ok = out_view ? io_copy(io.d_out, const_cast<void *>(out_view), io.out_bytes, s) == cudaSuccess
                                     : cudaMemcpyAsync(io.h_out, io.d_out, io.out_bytes, cudaMemcpyDeviceToHost,
                                                       s) == cudaSuccess;
            if (!ok) st = DDT_ERR_CUDA;
        }
        const cudaError_t e = cudaStreamEndCapture(s, &g);  // ends the capture on every path
        if (st == DDT_OK && e != cudaSuccess) st = DDT_ERR_CUDA;
    }
    cudaGraphExec_t exec = nullptr;
    if (st == DDT_OK && cudaGraphInstantiate(&exec, g, 0) != cudaSuccess) st = DDT_ERR_CUDA;
    if (g) cudaGraphDestroy(g);
    cudaStreamDestroy(s);
    if (st != DDT_OK) {
        if (exec) cudaGraphExecDestroy(exec);
        return st;
    }
    ddt_step_graph *h = new (std::nothrow) ddt_step_graph;
    if (!h) {
        cudaGraphExecDestroy(exec);
        return DDT_ERR_CUDA;
    }
    h->exec = exec;
    *graph = h;
    return DDT_OK;
}
}  // namespace

extern "C" {

ddt_status ddt_step_graph_create(const ddt_step_args *a, ddt_step_graph **graph) {
    return step_graph_create(a, StepIO{}, graph);
}

ddt_status ddt_step_graph_create_io(const ddt_step_args *a, const void *h_in, void *d_in,
                                    size_t in_bytes, void *h_out, const void *d_out,
                                    size_t out_bytes, ddt_step_graph **graph) {
    if (!a || !graph) return DDT_ERR_INVALID_ARG;
    *graph = nullptr;
    if ((in_bytes && (!h_in || !d_in)) || (out_bytes && (!h_out || !d_out)))
        return DDT_ERR_INVALID_ARG;
    if (!device_state()) return DDT_ERR_CUDA;
    if ((in_bytes && !is_pinned_host(h_in)) || (out_bytes && !is_pinned_host(h_out)))
        return DDT_ERR_INVALID_ARG;
    StepIO io;
    io.h_in = h_in;
    io.d_in = d_in;
    io.in_bytes = in_bytes;
    io.h_out = h_out;
    io.d_out = d_out;
    io.out_bytes = out_bytes;
    return step_graph_create(a, io, graph);
}

ddt_status ddt_step_graph_launch(ddt_step_graph *graph, void *stream) {
    if (!graph || !graph->exec) return DDT_ERR_INVALID_ARG;
    return cudaGraphLaunch(graph->exec, as_stream(stream)) == cudaSuccess ? DDT_OK : DDT_ERR_CUDA;
}

ddt_status ddt_step_graph_destroy(ddt_step_graph *graph) {
    if (!graph) return DDT_ERR_INVALID_ARG;
    const cudaError_t e = graph->exec ? cudaGraphExecDestroy(graph->exec) : cudaSuccess;
    delete graph;
    return e == cudaSuccess ? DDT_OK : DDT_ERR_CUDA;
}

}  // extern "C"

namespace ddt {
// Device address of the current device's error word (sets the device up on
// first use, like every entry point); null on failure.
unsigned int *device_error_word() {
    DeviceState *st = device_state();
    return st ? st->err : nullptr;
}
int device_sm_count() {
    DeviceState *st = device_state();
    return st ? st->num_sms : 148;
}
}  // namespace ddt

