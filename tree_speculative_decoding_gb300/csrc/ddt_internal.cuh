// ddt_internal.cuh -- declarations shared by the CUDA translation units of
// libddt.so (launchers defined in each .cu, called from ddt_abi.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ddt.h"

namespace ddt {

// Latch a device-side check into the per-device error word.
__device__ __forceinline__ void latch(unsigned int *err, unsigned int bit) {
    if (err) atomicOr(err, bit);
}

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialization and announces at its start that the next
// kernel in the stream may be scheduled.  A kernel therefore may run while the
// previous one is still running, and it calls pdl_wait() -- which returns once
// the previous kernel (and, transitively, everything before it) has finished
// and its writes are visible -- before it reads anything an earlier kernel of
// the step wrote, and before its first global write.  Work on the caller's
// inputs (q, the kv pool and indices, top-k) may happen before the wait; a
// kernel that does not itself trigger early is complete before any of ours
// starts.  Dependents are scheduled only after every CTA of the previous
// kernel has started, so no wait can hold resources the previous kernel needs.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Launchers (host functions; each enqueues on `s` and returns the launch error).
cudaError_t launch_build_tree(const float *topk_logp, const int32_t *topk_ids,
                              const int32_t *root_id, const int32_t *budget,
                              const int32_t *qo_indptr, int batch, int max_depth, int topk,
                              int32_t *node_token, int32_t *parent, int32_t *depth,
                              unsigned int *err, cudaStream_t s);

cudaError_t launch_build_tree_visibility(const float *topk_logp, const int32_t *topk_ids,
                                         const int32_t *root_id, const int32_t *budget,
                                         const int32_t *qo_indptr, int batch, int max_depth, int topk,
                                         const int32_t *prefix_len, const int32_t *mask_indptr,
                                         int32_t *node_token, int32_t *parent, int32_t *depth,
                                         uint32_t *mask, unsigned int *err, cudaStream_t s);
cudaError_t launch_build_chain_visibility(const int32_t *qo_indptr, const int32_t *prefix_len,
                                          const int32_t *mask_indptr, int batch, int32_t *parent,
                                          int32_t *depth, uint32_t *mask, unsigned int *err,
                                          cudaStream_t s);
cudaError_t launch_compile_visibility(const int32_t *parent, const int32_t *qo_indptr,
                                      const int32_t *prefix_len, const int32_t *mask_indptr,
                                      int batch, int total_words, uint32_t *mask,
                                      unsigned int *err, cudaStream_t s);

cudaError_t launch_accept(const int32_t *node_token, const int32_t *parent,
                          const int32_t *qo_indptr, const int32_t *target_argmax, int batch,
                          int max_depth, int32_t *accept_len, int32_t *accepted_nodes,
                          int32_t *commit_tokens, int32_t *bonus, unsigned int *err,
                          cudaStream_t s);

cudaError_t launch_commit_kv(uint16_t *kv_pool, int64_t pool_rows, const int32_t *kv_indices,
                             const int32_t *kv_indptr, const int32_t *qo_indptr,
                             const int32_t *accept_len, const int32_t *accepted_nodes, int batch,
                             int max_depth, int32_t *new_len, unsigned int *err, cudaStream_t s);

cudaError_t launch_tree_links(const int32_t *parent, const int32_t *qo_indptr, int batch,
                              int32_t *first_child, int32_t *next_sibling, int32_t *retrieve_index,
                              unsigned int *err, cudaStream_t s);
cudaError_t launch_accept_sampled(const int32_t *node_token, const int32_t *first_child,
                                  const int32_t *next_sibling, const int32_t *qo_indptr,
                                  const float *logits, int vocab, const float *temperature,
                                  const int32_t *top_k, const float *top_p, const float *coins,
                                  int coin_stride, int batch,
                                  int max_depth, int32_t *accept_len, int32_t *accepted_nodes,
                                  int32_t *commit_tokens, int32_t *bonus, unsigned int *err,
                                  cudaStream_t s);

// Arguments of one verify-attention call as seen by the kernels.
struct AttnArgs {
    const uint16_t *q;
    const uint16_t *kv_pool;
    int64_t pool_rows;
    const int32_t *kv_indices;
    const int32_t *kv_indptr;
    const int32_t *qo_indptr;
    const uint32_t *mask;
    const int32_t *mask_indptr;
    int batch;
    int num_heads;
    int total_q;
    int max_q_len;
    int max_kv_len;
    float scale;
    int num_splits;
    int split_cols;       // kv columns per split (multiple of the kv tile)
    // 1 when the mask is a tree mask this library built in the same step (every
    // prefix column visible, no column after the row's own node): prefix-only
    // blocks then read no mask word.  0: every mask bit is honoured.
    int tree_mask;
    float *out;           // [total_q, H, 512]
    float *lse;           // [total_q, H] or null
    float *o_part;        // [splits, total_q*H, 512] when num_splits > 1
    float *lse_part;      // [splits, total_q*H]
    unsigned int *err;
};

// Split-KV partial pass (tensor-core kernel) and its sizing rules.
cudaError_t launch_attn_partial(const AttnArgs &a, cudaStream_t s);
// the split count for these bounds, at most max_splits (>= 1)
int attn_choose_splits(int batch, int num_heads, int max_q_len, int max_kv_len, int num_sms,
                       int max_splits = DDT_MAX_SPLITS);
cudaError_t attn_tc_prepare_device();
// CUDA-core kernel of the same pass (same arguments and outputs)
cudaError_t launch_attn_combine(const AttnArgs &a, cudaStream_t s);
cudaError_t attn_combine_prepare_device();
// shared-memory carveout of the small stages' kernels (they overlap the attention)
cudaError_t tree_prepare_device();
cudaError_t commit_prepare_device();
cudaError_t sample_prepare_device();

// A kernel whose bounded mbarrier wait can never succeed: it latches
// DDT_DEVERR_TIMEOUT and exits (the failure path, exercised without a fault).
cudaError_t launch_wait_timeout_selftest(uint32_t poll_limit, unsigned int *err, cudaStream_t s);

// kv columns per split must be a multiple of this (the attention kv tile)
int attn_kv_tile();
// The split layout a requested count (>= 1) gives: kv columns per split,
// rounded up to whole kv tiles, and the number of splits that then cover
// max_kv_len (no empty tail split), which can be fewer than requested.
void attn_split_layout(int max_kv_len, int requested, int *split_cols, int *splits);
int attn_launched_splits(int max_kv_len, int requested);

// Once per device, with that device current and before any stream capture:
// kernel attributes (dynamic shared memory opt-in).
cudaError_t attn_prepare_device();

// Device address of the current device's error word (null on failure).
unsigned int *device_error_word();
// the current device's SM count (after the same one-time set-up)
int device_sm_count();

}  // namespace ddt
