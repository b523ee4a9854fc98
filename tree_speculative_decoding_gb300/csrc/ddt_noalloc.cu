// ddt_noalloc.cu -- ddt_verify_attn for callers that cannot allocate device
// memory.
//
// ddt_verify_attn needs a caller-provided workspace whenever it splits the kv
// range (the split partial results and their log-sum-exps).  Some callers
// cannot obtain one: an engine that has handed all device memory to its own
// pool up front, a plain C host with no allocator of its own, or a decode loop
// where a cudaMalloc (which may synchronise the whole device) is not allowed.
// ddt_verify_attn_noalloc serves them: its split scratch is a fixed array in
// this library's device memory, so the call itself allocates nothing.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "ddt_internal.cuh"

namespace {

// The scratch array.  Every GPU that loads libddt.so holds these bytes until
// the process exits.  In host code `g_noalloc_scratch` only names a host-side
// stand-in; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DDT_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];  // device address per device, once set up
bool g_scratch_ready[kMaxDevices];
std::mutex g_scratch_mu;

// Once per device, with that device current: look up the array's device
// address.  Runs inside the first ddt_verify_attn_noalloc call on a device.
void *scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ready[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return nullptr;
        g_scratch_ptr[dev] = p;
        g_scratch_ready[dev] = true;
    }
    return g_scratch_ptr[dev];
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// The split count asked of the kernels: num_splits as given, or for 0 the
// library's choice among the counts whose partials fit the scratch.
int noalloc_requested_splits(int32_t batch, int32_t num_heads, int32_t total_q, int32_t max_q_len,
                             int32_t max_kv_len, int32_t num_splits) {
    if (num_splits > 0) return num_splits;
    int cap = DDT_MAX_SPLITS;
    while (cap > 1 &&
           ddt_verify_attn_workspace_size(total_q, num_heads, cap) > (size_t)DDT_NOALLOC_SCRATCH_BYTES)
        --cap;
    return ddt::attn_choose_splits(batch, num_heads, max_q_len, max_kv_len, ddt::device_sm_count(), cap);
}

}  // namespace

extern "C" int32_t ddt_verify_attn_noalloc_splits(int32_t batch, int32_t num_heads, int32_t total_q,
                                                  int32_t max_q_len, int32_t max_kv_len,
                                                  int32_t num_splits) {
    if (batch < 1 || num_heads < 1 || total_q < 1 || max_q_len < 1 || max_kv_len < 1 || num_splits < 0)
        return 1;
    return ddt::attn_launched_splits(
        max_kv_len, noalloc_requested_splits(batch, num_heads, total_q, max_q_len, max_kv_len, num_splits));
}

extern "C" ddt_status ddt_verify_attn_noalloc(
    const uint16_t *q, const uint16_t *kv_pool, int64_t pool_rows, const int32_t *kv_indices,
    const int32_t *kv_indptr, const int32_t *qo_indptr, const uint32_t *mask,
    const int32_t *mask_indptr, int32_t batch, int32_t num_heads, int32_t total_q,
    int32_t max_q_len, int32_t max_kv_len, float scale, int32_t num_splits, float *out,
    float *lse, void *stream) {
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
    unsigned int *err = ddt::device_error_word();  // also prepares the device
    void *scratch = scratch_address();
    if (!err || !scratch) return DDT_ERR_CUDA;

    int split_cols = 0, splits = 1;
    ddt::attn_split_layout(max_kv_len, noalloc_requested_splits(batch, num_heads, total_q, max_q_len,
                                                                max_kv_len, num_splits),
                           &split_cols, &splits);

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
    a.out = out;
    a.lse = lse;
    a.err = err;
    if (splits > 1) {
        // The partial pass writes every (split, row) entry before the combine
        // reads it, so nothing left by an earlier call needs clearing.
        const size_t need = ddt_verify_attn_workspace_size(total_q, num_heads, splits);
        if (need > (size_t)DDT_NOALLOC_SCRATCH_BYTES) return DDT_ERR_WORKSPACE;
        const size_t rows = (size_t)total_q * num_heads;
        a.o_part = static_cast<float *>(scratch);
        a.lse_part = reinterpret_cast<float *>(static_cast<char *>(scratch) +
                                               align256(rows * splits * DDT_DL * sizeof(float)));
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = ddt::launch_attn_partial(a, s);
    if (e == cudaSuccess && splits > 1) e = ddt::launch_attn_combine(a, s);
    return e == cudaSuccess ? DDT_OK : DDT_ERR_CUDA;
}
