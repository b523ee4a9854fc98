// ddt_attn_tc.cu -- tree-verify MLA attention on the sm_103a tensor cores.
//
// What it computes, per row (tree node i of request b, head h), over the kv
// columns j of the request that mask row i makes visible:
//   s_j = scale * <q[i,h,0:576], kv[idx_j, 0:576]>,
//   out[i,h,:] = sum_j softmax(s)_j kv[idx_j, 0:512],  lse = log sum_j e^{s_j}
// ("The Architecture of a Speculative Decoding Engine", section "The Forward
// Pass Pseudocode": absorbed MLA, scores over latent + rope, output in the
// latent space; "The 30-Column Mask", sections "The Message: Tensor Shapes as
// Evidence" and "The Fix: Building Combined Indices": kv columns = prefix slots
// then the tree nodes' slots, one 576-wide row per token shared by all heads).
//
// Tiling (GB300-specific, measured on the part):
//   * A tile is 128 consecutive (node, head) rows of one request, e.g. two
//     nodes x 64 heads.  A thread-block cluster of two CTAs owns one tile and
//     one kv split.  CTA c keeps in tensor memory the fp32 output for latent
//     half c (128 lanes x 256 columns), its latent half of Q as bf16 pairs
//     (128 columns) and two 64-column score blocks; its 32 rope dims of Q
//     ([512+32c, 512+32c+32)) sit in shared memory.  A full-width output tile
//     (512 columns) would leave no room for scores, which is why the latent
//     dimension is split across the pair.
//   * Per kv block of 64 columns: two producer warps gather this CTA's half of
//     the 64 kv rows with 16-byte cp.async copies into a 128-byte-swizzled
//     stage (four stages); the MMA warp computes partial scores over the dim
//     half (tcgen05.mma, M=128, N=64: 16 K-steps with A = Q from tensor memory,
//     2 with A = rope Q from shared memory) into alternate score blocks.  The
//     pair swaps fp32 partials through distributed shared memory: CTA c owns
//     the softmax of rows [64c, 64c+64).  The owner adds the two partials,
//     applies the mask, runs the online softmax (the running max moves only
//     when a block max exceeds it by more than a factor 2^48), writes P (bf16) locally
//     and bulk-copies its rows to the partner with the rows' rescale factors.
//     Each CTA then accumulates O_c += P V_c (tcgen05.mma, M=128, N=256, K=64,
//     V read as an MN-major operand straight from the gathered stage).  P and
//     the partner-partial buffer are double-buffered, so the owner writes
//     P_{j+1} while PV_j still reads P_j and the partner sends partials one
//     block ahead.
//   * Epilogue: after the single commit that follows the last PV, the softmax
//     warps read O out of tensor memory, scale by 1/l, stage the rows in the
//     idle gather stages and write each 1 KB row with one bulk copy.
//   * Distributed-shared-memory traffic moves at ~20 B/clk per direction only
//     when a warp's stores cover contiguous 512-byte runs (scattered 16-byte
//     pieces measured 8-9 B/clk), hence the chunk-major partial buffer and the
//     bulk-copied P rows.
//   * Warp roles: warps 0-3 softmax / epilogue (thread = row = TMEM lane);
//     of warps 4-6, one issues the MMAs (placed next to a non-owner softmax
//     warp) and two are producers.
//   * Q: the tile's rows are one contiguous block of q, so the MMA warp loads
//     this CTA's half with TMA tensor tiles as soon as the request's offsets
//     are known: the rope box lands in its 64-byte-swizzled operand layout,
//     the latent boxes are staged from the third kv stage on and moved into
//     tensor memory with tcgen05.cp.
//   * The visibility mask: by default every mask bit is honoured (a block
//     whose bits are all ones skips the per-column test).  A row's two words
//     for a block are loaded one block ahead by the warp that sends the row's
//     partial scores to the owner, and travel with them.  When the caller
//     states that the mask is a tree mask built by this library in the same
//     step (every prefix column visible, no column after the row's own node),
//     prefix-only blocks read no mask word, so the attention streams the prefix
//     while the tree build is still running, and columns after the tile's last
//     node are skipped.
//   * Every wait is bounded; on timeout the CTA latches DDT_DEVERR_TIMEOUT,
//     stops, and still meets its partner at the final cluster barrier.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include "ddt_internal.cuh"
#include "ddt_sm100.cuh"

namespace ddt {
namespace {

using namespace sm100;

constexpr int kRows = 128;            // rows per tile (TMEM lanes)
constexpr int kNb = 64;               // kv columns per block
constexpr int kThreads = 224;         // 7 warps
constexpr int kBoxBytes = kNb * 128;  // 64 rows x 64 bf16, 128-byte swizzle
constexpr int kRopeBytes = kNb * 64;  // 64 rows x this CTA's 32 rope dims, 64-byte swizzle
constexpr int kStageBytes = 4 * kBoxBytes + kRopeBytes;  // 4 latent boxes + rope half
constexpr int kStages = 4;
// ring depths of the partner-partial buffers (X) and the P buffers; block j
// uses buffer j % depth with barrier phase (j / depth) & 1
constexpr int kXBufs = 2;
constexpr int kPBufs = 2;
// P (128 rows x 64 kv, bf16): one 128-byte-swizzle atom column; the 32 rows of
// one warp are 4 contiguous KB and go to the partner as one bulk copy.
constexpr int kPBytes = kRows * 128;
// partner partial scores: [16 chunks of 4 columns][64 rows] x 16 bytes, so one
// warp's 16-byte stores for a chunk are 512 contiguous bytes; then the two mask
// words of the block for each of the 64 rows (8 bytes per row)
constexpr int kXScoreBytes = (kNb / 4) * 64 * 16;
constexpr int kXBytes = kXScoreBytes + 64 * 8;

constexpr int kOffStage = 0;
constexpr int kORowStride = 1040;  // epilogue staging of O rows in the idle stages (16 B of padding)
constexpr int kOffP = kOffStage + kStages * kStageBytes;  // two P buffers
constexpr int kOffX = kOffP + kPBufs * kPBytes;          // partner-partial buffers
constexpr int kOffQr = kOffX + kXBufs * kXBytes;          // Q rope half: 128 rows x 64 B, 64-byte swizzle
constexpr int kOffAlpha = kOffQr + kRows * 64;             // 64 rescale factors per P buffer
constexpr int kOffLinv = kOffAlpha + kPBufs * 64 * 4;     // 64 floats
constexpr int kOffBar = kOffLinv + 64 * 4;
// barrier slots
enum {
    B_FULL0 = 0, B_EMPTY0 = B_FULL0 + kStages, B_SFULL0 = B_EMPTY0 + kStages, B_SFULL1, B_SFREE0, B_SFREE1,
    B_XFULL0, B_XEMPTY0 = B_XFULL0 + kXBufs, B_PIN0 = B_XEMPTY0 + kXBufs, B_PEMPTY0 = B_PIN0 + kPBufs,
    B_PFULL0 = B_PEMPTY0 + kPBufs, B_PVDONE = B_PFULL0 + kPBufs, B_FIN, B_ODONE, B_QLD, B_QFREE, B_COUNT
};
constexpr int kOffXsig = kOffBar + B_COUNT * 8;  // per X buffer, 2 owner warps: 4-byte "read" signals
constexpr int kOffHolder = kOffXsig + 8 * kXBufs;
constexpr int kOffAbort = kOffHolder + 4;
constexpr int kSmemUsed = kOffAbort + 4;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment

// tensor memory columns
constexpr uint32_t kColO = 0;    // 256: output, latent half
constexpr uint32_t kColQ = 256;  // 128: Q latent half, bf16 pairs (the rope half is in shared memory)
constexpr uint32_t kColS = 384;  // 2 x 64: partial scores, double-buffered
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kWaitLimit = 1u << 22;
constexpr int kOrderMaxBatch = 256;  // longest-first dispatch order up to this many requests
// Lazy rescale: the running max m (log2 units) moves only when a block's max
// exceeds it by more than this, so p = 2^(s - m) <= 2^48.  P (bf16) and the
// fp32 sums keep their relative precision at any scale; the sums stay finite
// while N * 2^48 * max|v| < 2^128, i.e. for |v| below ~2^59 at a million kv
// columns.  A rescale of O (a serial 256-column TMEM read-modify-write after
// waiting for the previous PV) costs ~1-2 us, so it should stay rare: with 1%
// of kv rows scaled by 8, a threshold of 20 measured 1.3% slower.
constexpr float kRescaleLog2 = 48.0f;
constexpr float kLog2e = 1.4426950408889634f;

constexpr uint32_t kIdescS = idesc_bf16(kRows, kNb, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16(kRows, 256, 0, 1);

static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kColS + 2 * kNb <= kTmemCols, "tensor memory budget");
static_assert(kOffP % 1024 == 0 && kPBytes % 1024 == 0 && kStageBytes % 1024 == 0, "swizzle atoms");
static_assert(kOffQr % 512 == 0, "64-byte swizzle atom of the rope box");
static_assert(kXBufs >= 1 && kXBufs <= 3 && kPBufs >= 1 && kPBufs <= 3, "ring depths");

__device__ __forceinline__ int xbuf(int j) { return j % kXBufs; }
__device__ __forceinline__ uint32_t xphase(int j) { return (uint32_t)(j / kXBufs) & 1u; }
__device__ __forceinline__ int pbuf_of(int j) { return j % kPBufs; }
__device__ __forceinline__ uint32_t pphase(int j) { return (uint32_t)(j / kPBufs) & 1u; }
// the epilogue stages O rows over the kv stages, P and X buffers, all idle once the last PV is done
static_assert(kRows * kORowStride <= kOffQr - kOffStage, "epilogue staging fits before the rope of Q");

struct TcParams {
    // q viewed as [total_q * num_heads rows][576] bf16: boxes of 128 rows x 64
    // latent dims (128-byte swizzle) and 128 rows x 32 rope dims (64-byte swizzle)
    CUtensorMap q_lat;
    CUtensorMap q_rope;
    AttnArgs a;
    int tiles_per_req;
};
// The tile's Q latent half is staged by TMA in stages 2 and 3 (4 boxes of 16
// KB), copied into tensor memory by tcgen05.cp, and the two stages are then
// handed to the producers.
constexpr int kOffQStage = kOffStage + 2 * kStageBytes;
constexpr uint32_t kQBytes = 4 * kRows * 128 + kRows * 64;
// Q's latent boxes are staged from stage 2 on: over the later stages and the P
// buffers, which nothing writes before Q is in tensor memory, but not the X buffers
static_assert(kOffQStage + 4 * kRows * 128 <= kOffX, "Q staging ends before the X buffers");

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int *abort,
                                              unsigned int *err) {
    if (*abort) return false;
    if (mbar_wait(bar, parity, kWaitLimit)) return true;
    *abort = 1;
    latch(err, DDT_DEVERR_TIMEOUT);
    return false;
}
// The same wait for a whole warp: it succeeds for every lane or for none, so
// the warp stays converged for the warp-collective instructions after it.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          unsigned int *err) {
    return __all_sync(0xffffffffu, wait_or_abort(bar, parity, abort, err));
}

__device__ __forceinline__ float max64(const float (&v)[kNb]) {
    float m[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) m[i] = fmaxf(fmaxf(v[4 * i], v[4 * i + 1]), fmaxf(v[4 * i + 2], v[4 * i + 3]));
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
    return m[0];
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ TcParams prm) {
    const AttnArgs &a = prm.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + kOffBar + 8u * i; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffAbort);
    uint32_t *holder = reinterpret_cast<uint32_t *>(smem + kOffHolder);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    // The next kernel (the combine) may be scheduled now.  This kernel reads only
    // caller inputs until it needs mask words (the visibility compile may still be
    // running: prefix blocks never read the mask) or writes its outputs; both
    // happen after pdl_wait().
    pdl_trigger();
    const uint32_t rank = cluster_ctarank();  // 0 or 1: latent half
    const uint32_t peer = rank ^ 1u;
    // Clusters run tile-fastest: the row tiles that share a split's kv columns
    // are dispatched together, so that one wave reads those rows from HBM once.
    const int tile = blockIdx.x >> 1;
    const int split = blockIdx.y;
    const int mma_warp = rank ? 4 : 6;
    // The MMA warp's first lane sets up the barriers at once, so that it can
    // start the Q copies as soon as the request's offsets are known; the other
    // threads use the barriers only after the set-up's block barrier.
    if (warp == mma_warp && lane == 0) {
        for (int i = 0; i < B_COUNT; ++i) {
            // one arrival: stage empties, score full, PV done, O done, Q (MMA
            // commits or a TMA)
            uint32_t count = 1;
            if (i < B_EMPTY0) count = 64;                       // stage full: 64 producer lanes
            else if (i == B_SFREE0 || i == B_SFREE1 || (i >= B_PFULL0 && i < B_PFULL0 + kPBufs))
                count = 4;  // softmax warps
            else if (i >= B_XFULL0 && i < B_PFULL0) count = 2;  // two warps / two CTAs
            else if (i == B_FIN) count = 2;
            mbar_init(bar(i), count);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    // Clusters are dispatched in block-index order, request by request.  With
    // several requests, blockIdx.z = k takes the request with the k-th most kv
    // columns (ties by index), so the longest requests start first and a long
    // one never waits for the last wave.  Every CTA derives the same order from
    // kv_indptr; the idle stage memory is the scratch.
    int b = blockIdx.z;
    if (a.batch > 1 && a.batch <= kOrderMaxBatch) {
        int *s_len = reinterpret_cast<int *>(smem + kOffStage);
        int *s_req = s_len + kOrderMaxBatch;
        for (int i = tid; i < a.batch; i += kThreads) s_len[i] = a.kv_indptr[i + 1] - a.kv_indptr[i];
        __syncthreads();
        for (int r = tid; r < a.batch; r += kThreads) {
            const int len = s_len[r];
            int k = 0;
            for (int o = 0; o < a.batch; ++o) k += (s_len[o] > len) || (s_len[o] == len && o < r);
            if (k == (int)blockIdx.z) *s_req = r;
        }
        __syncthreads();
        b = *s_req;
    }

    // ---- work of this tile / split (identical in both CTAs of the pair) ----
    // All six offsets of the request are loaded in one round of independent
    // loads: after an L2 flush each dependent round trip costs ~1.6 us.
    const int H = a.num_heads;
    const int qo0 = a.qo_indptr[b], qo1 = a.qo_indptr[b + 1];
    const int kv0 = a.kv_indptr[b], kv1 = a.kv_indptr[b + 1];
    const int m0 = a.mask_indptr[b], m1 = a.mask_indptr[b + 1];
    const int T = qo1 - qo0;
    const int N = kv1 - kv0;
    const int W = (N + 31) >> 5;
    // rows of q and out: [qo0, qo1) within [0, total_q); kv columns [kv0, kv1);
    // mask words [m0, m1) as q_len rows of ceil(kv_len / 32) words
    const bool bad_qo = T < 1 || T > a.max_q_len || qo0 < 0 || qo1 > a.total_q;
    const bool bad_kv = N < T || N > a.max_kv_len || kv0 < 0;
    const bool bad_mask = !bad_qo && !bad_kv && (m0 < 0 || m1 - m0 != T * W);
    if (bad_qo || bad_kv || bad_mask) {  // uniform in the pair: no cluster interaction yet
        if (tid == 0 && rank == 0)
            latch(a.err, (bad_qo ? DDT_DEVERR_QO_INDPTR : 0u) | (bad_kv ? DDT_DEVERR_KV_INDPTR : 0u) |
                             (bad_mask ? DDT_DEVERR_MASK_INDPTR : 0u));
        pdl_wait();
        return;
    }
    const int rows_req = T * H;
    const int row0 = tile * kRows;
    if (row0 >= rows_req) { pdl_wait(); return; }  // uniform in the pair
    const int P = N - T;
    const int rows_valid = min(kRows, rows_req - row0);
    const int i_max = (row0 + rows_valid - 1) / H;   // last node in the tile
    // A library-built tree mask shows no column after the row's own node, so
    // nothing beyond P + i_max is visible to the tile; any other mask may set
    // any bit of the row.
    const int kv_end = a.tree_mask ? P + i_max + 1 : N;
    const int c_begin = split * a.split_cols;
    const int c_end = min(kv_end, c_begin + a.split_cols);
    const int nblk = (c_end > c_begin) ? (c_end - c_begin + kNb - 1) / kNb : 0;
    const int64_t rows_total = (int64_t)a.total_q * H;

    if (nblk == 0) {  // empty split: neutral partial result (only happens with splits > 1)
        pdl_wait();
        if (warp < 4) {
            const int r = tid;
            if (r < rows_valid && a.num_splits > 1) {
                const int rr = row0 + r;
                const int64_t grow = (int64_t)(qo0 + rr / H) * H + (rr % H);
                float *o = a.o_part + ((int64_t)split * rows_total + grow) * DDT_DL + 256 * rank;
                for (int q = 0; q < 64; ++q) reinterpret_cast<float4 *>(o)[q] = make_float4(0, 0, 0, 0);
                if (rank == 0) a.lse_part[(int64_t)split * rows_total + grow] = -INFINITY;
            }
        }
        return;
    }

    // ---- loads that need no set-up, issued before it so that the tensor-memory
    // allocation and the cluster sync run under their latency: the tile's Q
    // (TMA, by the MMA warp) and the producers' first kStages blocks of kv slots ----
    if (warp == mma_warp && lane == 0) {
        const int y = (qo0 * H) + row0;  // first (node, head) row of the tile in q
        mbar_arrive_expect_tx(bar(B_QLD), kQBytes);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            tma_load_2d(sbase + kOffQStage + k * kRows * 128, &prm.q_lat, 256 * (int)rank + 64 * k, y, bar(B_QLD));
        tma_load_2d(sbase + kOffQr, &prm.q_rope, 512 + 32 * (int)rank, y, bar(B_QLD));
    }
    const bool producer = warp >= 4 && warp != mma_warp;
    const int half = (warp == (rank ? 5 : 4)) ? 0 : 1;  // producers: kv rows [32 half, 32 half + 32)
    // slot of this producer lane's kv row of block j
    auto fetch_slot = [&](int j) {
        return a.kv_indices[kv0 + min(c_begin + j * kNb + 32 * half + lane, c_end - 1)];  // rows past the end reuse a valid one
    };
    int slot_ahead[kStages];
    if (producer) {
#pragma unroll
        for (int s = 0; s < kStages; ++s) slot_ahead[s] = (s < nblk) ? fetch_slot(s) : 0;
    }
    const int r = tid;  // row within the tile for warps 0-3

    // ---- setup ----
    if (warp == 5) tmem_alloc(smem_u32(holder), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;
    // both CTAs' barriers exist before any remote access: the inits were
    // published by fence.mbarrier_init, so the arrive can be relaxed and the
    // producers' kv slot loads in flight do not hold it up
    cluster_sync_relaxed_arrive();

    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    // Every MMA accumulates (enable-input-D set): an MMA that overwrites its
    // accumulator right behind a tcgen05.commit waits for the committed MMAs to
    // drain, which measured ~700-950 cycles per score block on the part.  The
    // score columns are therefore cleared by the warps that read them, and O
    // once at the start.
    auto zero_scores = [&](int sb) {
        const uint32_t z[32] = {};
#pragma unroll
        for (int q = 0; q < kNb / 32; ++q) tmem_st32(tmem + lane_off + kColS + kNb * sb + 32 * q, z);
        tmem_wait_st();
    };
    if (warp < 4) {  // O and both score blocks start at zero
        const uint32_t z[32] = {};
#pragma unroll
        for (int q = 0; q < 8; ++q) tmem_st32(tmem + lane_off + kColO + 32 * q, z);
        zero_scores(0);
        zero_scores(1);
    }
    // Q's latent half from the staging boxes into tensor memory (columns kColQ +
    // 8 ks hold dims [16 ks, 16 ks + 16) as bf16 pairs, the layout of an MMA A
    // operand); the commit hands stages 2 and 3 to the producers.
    bool q_in = true;
    if (warp == mma_warp) {
        if (lane == 0) {
            q_in = wait_or_abort(bar(B_QLD), 0, abort_flag, a.err);
            if (q_in) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 16; ++ks)
                    tmem_cp_128x256b(tmem + kColQ + 8 * ks,
                                     smem_desc(sbase + kOffQStage + (ks >> 2) * kRows * 128 + (ks & 3) * 32, 16, 1024));
                mma_commit(bar(B_QFREE));
            }
        }
        __syncwarp();
    }
    // Q / O / S in tensor memory before the first MMA: the softmax warps and the
    // MMA warp meet on a named barrier; the producers start gathering at once.
    // Warp w issues on sub-partition w % 4.  The MMA warp spins on barriers, so
    // it goes next to a non-owner softmax warp: warp 6 (with warp 2) in rank 0,
    // where warps 0-1 own rows, and warp 4 (with warp 0) in rank 1.
    if (warp < 4 || warp == mma_warp) {
        tc_fence_before();
        named_barrier(1, 160);
        tc_fence_after();
    }

    if (producer) {
        // ================= producers: gather this CTA's five boxes per kv row =================
        // Warp 4 moves kv rows [0, 32) of each block, warp 6 rows [32, 64).  One
        // warp instruction moves one 128-byte box line of four kv rows: lane =
        // 8 * (row within the group of four) + 16-byte chunk.  Chunks land with
        // the 128-byte swizzle (chunk ^ (row & 7)) that the MMA descriptors
        // expect.  Each lane arrives on the stage barrier once its own copies
        // have landed (64 arrivals per stage).
        const int sub = lane >> 3, chunk = lane & 7;
        const char *pool = reinterpret_cast<const char *>(a.kv_pool);
        // slot_ahead[s] holds block j's slot while stage s gathers block
        // j - kStages: each slot is loaded one stage ring ahead (the first
        // kStages before the set-up), so index loads overlap the stage waits.
        bool run = true;
        for (int j0 = 0; run && j0 < nblk; j0 += kStages) {
#pragma unroll
            for (int s = 0; s < kStages; ++s) {
                const int j = j0 + s, u = j0 / kStages;
                if (j >= nblk) break;
                if (__any_sync(0xffffffffu, *abort_flag != 0)) { run = false; break; }
                if (u >= 1 && !warp_wait(bar(B_EMPTY0 + s), (u - 1) & 1, abort_flag, a.err)) { run = false; break; }
                // stages 2 and 3 hold the staged Q until it is in tensor memory
                if (u == 0 && s == 2 && !warp_wait(bar(B_QFREE), 0, abort_flag, a.err)) { run = false; break; }
                const uint32_t stage = sbase + kOffStage + s * kStageBytes;
                int mine = slot_ahead[s];
                if (mine < 0 || (int64_t)mine >= a.pool_rows) {
                    latch(a.err, DDT_DEVERR_KV_INDEX);
                    mine = 0;
                }
                if (j + kStages < nblk) slot_ahead[s] = fetch_slot(j + kStages);
#pragma unroll 4
                for (int g = 0; g < 8; ++g) {
                    const int kk = 4 * g + sub;          // row within this warp's 32
                    const int k = 32 * half + kk;        // kv row within the block
                    const int slot = __shfl_sync(0xffffffffu, mine, kk);
                    const char *src = pool + (int64_t)slot * (DDT_D * 2) + chunk * 16;
                    const uint32_t dst = stage + (k >> 3) * 1024 + (k & 7) * 128 + ((chunk ^ (k & 7)) << 4);
#pragma unroll
                    for (int bx = 0; bx < 4; ++bx)
                        cp_async_16(dst + bx * kBoxBytes, src + (256 * rank + 64 * bx) * 2);
                    if (chunk < 4)  // rope: this CTA's 32 dims, 64-byte rows
                        cp_async_16(stage + 4 * kBoxBytes + k * 64 + ((chunk ^ ((k >> 1) & 3)) << 4),
                                    src + (512 + 32 * rank) * 2);
                }
                cp_async_arrive(bar(B_FULL0 + s));
            }
        }
    } else if (warp == mma_warp) {
        // ================= MMA issuer =================
        // Issues S_j as soon as block j is loaded and the score buffer is free,
        // and PV_j as soon as P_j is in place -- whichever is ready first.
        if (lane == 0) {
            auto issue_s = [&](int j) {
                const uint32_t stage = sbase + kOffStage + (j % kStages) * kStageBytes;
                const uint32_t sd = tmem + kColS + kNb * (j & 1);
                fence_proxy_async_smem();  // stage written by cp.async, read by the tensor core
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 16; ++ks) {  // latent half: 256 dims, A = Q from tensor memory
                    const uint64_t bd = smem_desc(stage + (ks >> 2) * kBoxBytes + (ks & 3) * 32, 16, 1024);
                    mma_ts(sd, tmem + kColQ + 8 * ks, bd, kIdescS, 1u);
                }
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {  // rope half: 32 dims, A = Q rope from shared memory
                    const uint64_t ad = smem_desc(sbase + kOffQr + 32 * ks, 16, 512, kSwizzle64B);
                    const uint64_t bd = smem_desc(stage + 4 * kBoxBytes + 32 * ks, 16, 512, kSwizzle64B);
                    mma_ss(sd, ad, bd, kIdescS, 1u);
                }
                mma_commit(bar(B_SFULL0 + (j & 1)));
            };
            auto issue_pv = [&](int k) {
                const int s = k % kStages, pb = pbuf_of(k);
                tc_fence_after();
                const uint32_t pbuf = sbase + kOffP + pb * kPBytes;
                const uint32_t stage = sbase + kOffStage + s * kStageBytes;
#pragma unroll
                for (int ks = 0; ks < kNb / 16; ++ks) {
                    const uint64_t ad = smem_desc(pbuf + ks * 32, 16, 1024);
                    const uint64_t bd = smem_desc(stage + ks * 2048, kBoxBytes, 1024);
                    mma_ss(tmem + kColO, ad, bd, kIdescPV, 1u);
                }
                mma_commit(bar(B_EMPTY0 + s));
                mma_commit_multicast(bar(B_PEMPTY0 + pb), (uint16_t)0x3);
                mma_commit(bar(B_PVDONE));
            };
            int ns = 0, np = 0;  // next S block, next PV block
            uint32_t idle = 0;
            while (np < nblk) {
                if (*abort_flag) break;
                bool did = false;
                if (ns < nblk && mbar_test_wait(bar(B_FULL0 + ns % kStages), (ns / kStages) & 1) &&
                    (ns < 2 || mbar_test_wait(bar(B_SFREE0 + (ns & 1)), ((ns - 2) >> 1) & 1))) {
                    issue_s(ns++);
                    did = true;
                }
                if (np < ns && mbar_test_wait(bar(B_PFULL0 + pbuf_of(np)), pphase(np))) {
                    issue_pv(np++);
                    did = true;
                }
                if (did) {
                    idle = 0;
                } else if (++idle > kWaitLimit) {
                    *abort_flag = 1;
                    latch(a.err, DDT_DEVERR_TIMEOUT);
                    break;
                }  // busy polling measured faster than a nanosleep backoff
            }
            if (np == nblk) mma_commit(bar(B_ODONE));  // O complete (single phase)
        }
        __syncwarp();
    } else {
        // ================= softmax / epilogue (warps 0-3, thread = row) =================
        const bool owner = (uint32_t)(warp >> 1) == rank;
        const int xrow = r & 63;
        const bool row_valid = r < rows_valid;
        const int rr = row0 + r;
        const int node = row_valid ? rr / H : 0;
        const int head = row_valid ? rr % H : 0;
        const uint32_t *mrow = a.mask + m0 + (int64_t)node * W;
        const float sc = a.scale * kLog2e;
        // cluster addresses of the partner's buffers / barriers
        const uint32_t peer_base = map_to_cta(sbase, peer);
        const uint32_t p_fin = map_to_cta(bar(B_FIN), peer);
        const uint32_t p_linv = map_to_cta(sbase + kOffLinv + xrow * 4, peer);
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        // Visibility words of a row for block j: its two words (64 columns from
        // c0, a multiple of 64).  Prefix-only blocks of a library-built tree mask
        // read none.  The mask may be the previous kernel's output: it is waited
        // for once, before the first word is read.  The sender of a row's
        // partial scores (the partner's non-owner warp) loads them one block
        // ahead and ships them with the partials, so the owner reads them from
        // its own shared memory.
        auto all_prefix = [&](int j) {
            const int c0 = c_begin + j * kNb;
            return a.tree_mask && c0 + kNb <= min(P, c_end);
        };
        bool mask_ready = false;
        auto mask_words = [&](int j, uint32_t &w0, uint32_t &w1) {
            if (all_prefix(j)) {
                w0 = w1 = 0xffffffffu;
                return;
            }
            if (!mask_ready) {
                pdl_wait();
                mask_ready = true;
            }
            const int w = (c_begin + j * kNb) >> 5;
            w0 = (w < W) ? mrow[w] : 0u;
            w1 = (w + 1 < W) ? mrow[w + 1] : 0u;
        };

        // read S_j into registers, clear it, and hand the score buffer back to the MMA warp
        auto take_scores = [&](int j, float (&sv)[kNb]) {
            tc_fence_after();
            uint32_t t32[32];
#pragma unroll
            for (int q = 0; q < kNb / 32; ++q) {
                tmem_ld32(tmem + lane_off + kColS + kNb * (j & 1) + 32 * q, t32);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) sv[32 * q + e] = __uint_as_float(t32[e]);
            }
            zero_scores(j & 1);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_SFREE0 + (j & 1)));
        };
        // O row *= alpha before PV_j (only when a row of this warp rescales, which
        // needs PV_{j-1} finished); then this warp's part of P_j is in place.
        auto finish_block = [&](int j, float alpha) -> bool {
            if (__any_sync(0xffffffffu, alpha != 1.0f)) {
                if (j > 0 && !wait_or_abort(bar(B_PVDONE), (j - 1) & 1, abort_flag, a.err)) return false;
                tc_fence_after();
                uint32_t t32[32];
#pragma unroll 1
                for (int q = 0; q < 8; ++q) {
                    tmem_ld32(tmem + lane_off + kColO + 32 * q, t32);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) t32[e] = __float_as_uint(__uint_as_float(t32[e]) * alpha);
                    tmem_st32(tmem + lane_off + kColO + 32 * q, t32);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PFULL0 + pbuf_of(j)));
            return true;
        };

        if (!owner) {
            // Rows owned by the partner: send each block's partial scores as soon as
            // they exist (two partial buffers: up to two sends ahead) and take the
            // partner's P rows (and rescale factors) as soon as they land.
            const uint32_t px_row = map_to_cta(sbase + kOffX + xrow * 16, peer);
            const uint32_t px_mask = map_to_cta(sbase + kOffX + kXScoreBytes + xrow * 8, peer);
            int nsend = 0, nfin = 0;
            int pj = -1;  // the block whose mask words pw0 / pw1 hold
            uint32_t pw0 = 0u, pw1 = 0u;
            bool pin_armed = false;
            uint32_t idle = 0;
            while (nfin < nblk && ok) {
                if (*abort_flag) { ok = false; break; }
                bool did = false;
                // uniform readiness tests (tcgen05.ld below is warp-collective)
                bool can_send = false;
                if (nsend < nblk && nsend <= nfin + kXBufs) {
                    bool t = mbar_test_wait(bar(B_SFULL0 + (nsend & 1)), (nsend >> 1) & 1) &&
                             (nsend < kXBufs ||
                              mbar_test_wait(bar(B_XEMPTY0 + xbuf(nsend)), xphase(nsend - kXBufs)));
                    can_send = __shfl_sync(0xffffffffu, t, 0);
                }
                if (can_send) {
                    const int j = nsend++;
                    float sv[kNb];
                    take_scores(j, sv);
                    const uint32_t dst = px_row + xbuf(j) * kXBytes;
                    const uint32_t p_xfull = map_to_cta(bar(B_XFULL0 + xbuf(j)), peer);
#pragma unroll
                    for (int q = 0; q < kNb / 4; ++q)
                        st_async_v4(dst + 64 * 16 * q, __float_as_uint(sv[4 * q]), __float_as_uint(sv[4 * q + 1]),
                                    __float_as_uint(sv[4 * q + 2]), __float_as_uint(sv[4 * q + 3]), p_xfull);
                    // the row's mask words of block j with them, the next block's loaded now
                    uint32_t w0, w1;
                    if (pj == j) {
                        w0 = pw0;
                        w1 = pw1;
                    } else {
                        mask_words(j, w0, w1);
                    }
                    st_async_v2(px_mask + xbuf(j) * kXBytes, w0, w1, p_xfull);
                    if (j + 1 < nblk) {
                        mask_words(j + 1, pw0, pw1);
                        pj = j + 1;
                    }
                    // the owner signals "read" with a 4-byte store per owner warp
                    if (lane == 0) mbar_arrive_expect_tx(bar(B_XEMPTY0 + xbuf(j)), 4);
                    did = true;
                }
                if (nfin < nsend) {
                    const int s = pbuf_of(nfin);
                    if (!pin_armed) {
                        if (lane == 0) mbar_arrive_expect_tx(bar(B_PIN0 + s), 32 * ((kNb / 8) * 16 + 4));
                        pin_armed = true;
                    }
                    const bool t = __shfl_sync(0xffffffffu, mbar_test_wait(bar(B_PIN0 + s), pphase(nfin)), 0);
                    if (t) {
                        const float alpha = reinterpret_cast<volatile float *>(smem + kOffAlpha)[s * 64 + xrow];
                        if (!finish_block(nfin, alpha)) { ok = false; break; }
                        ++nfin;
                        pin_armed = false;
                        did = true;
                    }
                }
                if (did) {
                    idle = 0;
                } else if (++idle > kWaitLimit) {
                    *abort_flag = 1;
                    latch(a.err, DDT_DEVERR_TIMEOUT);
                    ok = false;
                }
            }
            // The partner's "read" signals of the last sends are the only remote
            // writes into this CTA that nothing else waits for: take them in before
            // teardown, so that no store of the partner's can land after this CTA
            // has left.
            for (int j = max(0, nsend - kXBufs); j < nsend && ok; ++j)
                if (!warp_wait(bar(B_XEMPTY0 + xbuf(j)), xphase(j), abort_flag, a.err)) ok = false;
        } else {
            for (int j = 0; j < nblk && ok; ++j) {
                const int xs = xbuf(j), s = pbuf_of(j);
                float sv[kNb];
                if (!wait_or_abort(bar(B_SFULL0 + (j & 1)), (j >> 1) & 1, abort_flag, a.err)) { ok = false; break; }
                take_scores(j, sv);
                const int c0 = c_begin + j * kNb;
                const bool pre_only = all_prefix(j);
                // owner: partner partial + own partial -> softmax -> P for both CTAs;
                // the partner's partials come with this row's mask words
                if (lane == 0) mbar_arrive_expect_tx(bar(B_XFULL0 + xs), 32 * (kNb * 4 + 8));
                if (!wait_or_abort(bar(B_XFULL0 + xs), xphase(j), abort_flag, a.err)) { ok = false; break; }
                uint32_t mw0 = 0xffffffffu, mw1 = 0xffffffffu;
                if (!pre_only) {
                    const uint2 w = reinterpret_cast<const uint2 *>(smem + kOffX + xs * kXBytes + kXScoreBytes)[xrow];
                    mw0 = w.x;
                    mw1 = w.y;
                }
                {
                    const float4 *x = reinterpret_cast<const float4 *>(smem + kOffX + xs * kXBytes) + xrow;
#pragma unroll
                    for (int q = 0; q < kNb / 4; ++q) {
                        const float4 v = x[64 * q];
                        const float2 a = f2add(make_float2(sv[4 * q], sv[4 * q + 1]), make_float2(v.x, v.y));
                        const float2 c = f2add(make_float2(sv[4 * q + 2], sv[4 * q + 3]), make_float2(v.z, v.w));
                        sv[4 * q] = a.x; sv[4 * q + 1] = a.y; sv[4 * q + 2] = c.x; sv[4 * q + 3] = c.y;
                    }
                }
                __syncwarp();
                if (lane == 0)
                    st_async_b32(map_to_cta(sbase + kOffXsig + 4 * (2 * xs + (warp & 1)), peer), 0u,
                                 map_to_cta(bar(B_XEMPTY0 + xs), peer));
                // visibility of the block's 64 columns: the mask bits (for a tree mask,
                // or-ed with the prefix), and-ed with the split's range.  Rows past
                // the tile's last valid row are never stored; their scores are finite
                // (q rows of the next request, or zeros past the end of q).
                if (!pre_only) {
                    const int npre = a.tree_mask ? max(0, min(kNb, P - c0)) : 0;  // leading prefix columns
                    const int nin = max(0, min(kNb, c_end - c0));                 // columns inside the split
                    uint32_t vbits[2];
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const int lo = 32 * t;
                        const uint32_t pre = npre >= lo + 32 ? 0xffffffffu : (npre > lo ? (1u << (npre - lo)) - 1u : 0u);
                        const uint32_t in = nin >= lo + 32 ? 0xffffffffu : (nin > lo ? (1u << (nin - lo)) - 1u : 0u);
                        vbits[t] = ((t ? mw1 : mw0) | pre) & in;
                    }
                    if ((vbits[0] & vbits[1]) != 0xffffffffu) {
#pragma unroll
                        for (int k = 0; k < kNb; ++k) sv[k] = ((vbits[k >> 5] >> (k & 31)) & 1u) ? sv[k] : -INFINITY;
                    }
                }
                float mb = max64(sv);
                mb *= sc;  // scores in log2 units: s * scale * log2(e)
                float alpha = 1.0f;
                if (mb > m_ref + kRescaleLog2) {  // also true for the first visible block (m_ref = -inf)
                    alpha = ex2(m_ref - mb);  // 0 when nothing was seen before
                    l *= alpha;
                    m_ref = mb;
                }
                uint32_t pw[kNb / 2];
                const float mref = (m_ref == -INFINITY) ? 0.f : m_ref;  // all -inf rows give p = 0
                const float2 scv = make_float2(sc, sc), nmv = make_float2(-mref, -mref);
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < kNb; k += 2) {
                    const float2 t = f2fma(make_float2(sv[k], sv[k + 1]), scv, nmv);
                    const float p0 = ex2(t.x), p1 = ex2(t.y);
                    acc = f2add(acc, make_float2(p0, p1));
                    pw[k / 2] = pack_bf16(p0, p1);
                }
                l += acc.x + acc.y;
                // both CTAs' P buffer s must be free (PV_{j-2} done in both)
                if (j >= kPBufs && !wait_or_abort(bar(B_PEMPTY0 + s), pphase(j - kPBufs), abort_flag, a.err)) {
                    ok = false;
                    break;
                }
                const uint32_t p_pin = map_to_cta(bar(B_PIN0 + s), peer);
                const uint32_t poff = kOffP + s * kPBytes;
#pragma unroll
                for (int q = 0; q < kNb / 8; ++q) {  // chunks of 8 kv, 128-byte swizzle
                    const uint32_t off = poff + (r >> 3) * 1024 + (r & 7) * 128 + ((q ^ (r & 7)) << 4);
                    *reinterpret_cast<uint4 *>(smem + off) =
                        make_uint4(pw[4 * q], pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]);
                }
                st_async_b32(peer_base + kOffAlpha + (s * 64 + xrow) * 4,
                             __float_as_uint(j == 0 ? 1.0f : alpha), p_pin);
                fence_proxy_async_smem();  // P rows: read by the tensor core and the bulk copy
                __syncwarp();
                if (lane == 0) {  // this warp's 32 rows to the partner
                    const uint32_t off = poff + (uint32_t)(warp * 32) * 128;
                    bulk_copy_to_cta(peer_base + off, sbase + off, 32 * 128, p_pin);
                }
                if (!finish_block(j, j == 0 ? 1.0f : alpha)) { ok = false; break; }  // O starts at zero
            }
        }

        // ---- epilogue: O_c / l into the output (or this split's partial) ----
        // A parity wait only tells apart phases one apart, and this point may be
        // reached before, between or after the last two PV completions (the
        // owner's own PV_{nblk-1} can finish before its thread gets here); the
        // MMA warp's single commit after the last PV is unambiguous.
        if (ok && wait_or_abort(bar(B_ODONE), 0, abort_flag, a.err)) {
            pdl_wait();  // the previous kernel may still read this step's output buffers
            float linv = 0.f;
            float lse_v = -INFINITY;
            bool have = true;
            if (owner) {
                linv = (l > 0.f) ? 1.f / l : 0.f;
                lse_v = (l > 0.f) ? (m_ref + log2f(l)) * 0.6931471805599453f : -INFINITY;
                st_async_b32(p_linv, __float_as_uint(linv), p_fin);
            } else {
                if (lane == 0) mbar_arrive_expect_tx(bar(B_FIN), 32 * 4);
                have = wait_or_abort(bar(B_FIN), 0, abort_flag, a.err);
                linv = reinterpret_cast<volatile float *>(smem + kOffLinv)[xrow];
            }
            tc_fence_after();
            if (have) {
                float *o = nullptr;
                float *lp = nullptr;
                if (row_valid) {
                    const int64_t grow = (int64_t)(qo0 + node) * H + head;
                    if (a.num_splits > 1) {
                        o = a.o_part + ((int64_t)split * rows_total + grow) * DDT_DL;
                        lp = a.lse_part + (int64_t)split * rows_total + grow;
                    } else {
                        o = a.out + grow * DDT_DL;
                        lp = a.lse ? a.lse + grow : nullptr;
                    }
                    o += 256 * rank;
                }
                // The row (1 KB of fp32) goes through the idle kv stages and leaves
                // as one bulk copy: per-thread 16-byte global stores of 128 rows at a
                // 2 KB stride measured ~5 us per CTA.  The 1040-byte row stride spreads
                // a warp's 16-byte shared-memory stores over all banks.
                uint8_t *srow = smem + kOffStage + r * kORowStride;
                uint32_t t32[32];
#pragma unroll 1
                for (int q = 0; q < 8; ++q) {
                    tmem_ld32(tmem + lane_off + kColO + 32 * q, t32);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        reinterpret_cast<float4 *>(srow)[8 * q + e] =
                            make_float4(__uint_as_float(t32[4 * e]) * linv, __uint_as_float(t32[4 * e + 1]) * linv,
                                        __uint_as_float(t32[4 * e + 2]) * linv, __uint_as_float(t32[4 * e + 3]) * linv);
                }
                fence_proxy_async_smem();  // the row is read by the bulk copy
                if (row_valid) {
                    bulk_store_global(o, smem_u32(srow), 256 * 4);
                    bulk_commit();
                    bulk_wait_read_all();  // the staged row must outlive the copy's read
                }
                if (owner && row_valid && lp) *lp = lse_v;
            }
        }
    }

    // ---- teardown: nobody leaves while the partner may still write here ----
    if (warp == mma_warp && lane == 0 && !q_in) mbar_wait(bar(B_QLD), 0, kWaitLimit);  // Q copies in flight
    pdl_wait();  // every path waits once, so this grid ends after the previous one
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// One warp waits on a barrier that expects one arrival nobody makes, with the
// same bounded wait as the verify kernel; it gives up after `limit` polls.
__global__ void __launch_bounds__(32) wait_timeout_selftest_kernel(uint32_t limit, unsigned int *err) {
    __shared__ __align__(8) uint64_t never;
    const uint32_t bar = smem_u32(&never);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    if (!mbar_wait(bar, 0, limit) && threadIdx.x == 0) latch(err, DDT_DEVERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint32_t poll_limit, unsigned int *err, cudaStream_t s) {
    wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(poll_limit, err);
    return cudaGetLastError();
}

cudaError_t attn_tc_prepare_device() {
    return cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemBytes);
}

int attn_kv_tile() { return kNb; }

void attn_split_layout(int max_kv_len, int requested, int *split_cols, int *splits) {
    const int want = requested < 1 ? 1 : requested;
    int cols = (max_kv_len + want - 1) / want;
    cols = (cols + kNb - 1) / kNb * kNb;
    *split_cols = cols;
    *splits = (max_kv_len + cols - 1) / cols;
}

int attn_launched_splits(int max_kv_len, int requested) {
    int cols = 0, splits = 1;
    attn_split_layout(max_kv_len, requested, &cols, &splits);
    return splits;
}

cudaError_t attn_prepare_device() {
    cudaError_t e = attn_combine_prepare_device();
    if (e == cudaSuccess) e = tree_prepare_device();
    if (e == cudaSuccess) e = commit_prepare_device();
    if (e == cudaSuccess) e = sample_prepare_device();
    if (e != cudaSuccess) return e;
    return attn_tc_prepare_device();
}

// Split count from host-side bounds only (no per-request lengths).  Several
// requests that already fill a wave of clusters (num_sms / 2 of them) take
// one split: the kernel starts the longest requests first, which balances the
// waves better than splitting did (a mixed batch of 32: 209 us with one split,
// 259-300 us with 2-4; a ragged batch of 8: 329 us against 358-379 us).
// Otherwise the grid runs in waves of num_sms / 2 clusters, and a cluster
// costs its kv blocks plus a fixed fill / epilogue share worth ~8 blocks.  The
// count minimising waves x (blocks per split + 8) wins, the smallest on ties,
// with at least 4 blocks per split.  For one request this picks the best count
// measured (4 at prefix 4096, 9 at prefix 131072, where 297 clusters fill four
// waves almost exactly).
int attn_choose_splits(int batch, int num_heads, int max_q_len, int max_kv_len, int num_sms,
                       int max_splits) {
    const long long tiles = (long long)batch * (((long long)max_q_len * num_heads + kRows - 1) / kRows);
    const long long pairs = num_sms / 2 > 0 ? num_sms / 2 : 1;
    if (batch > 1 && tiles >= pairs) return 1;
    const long long blocks = ((long long)max_kv_len + kNb - 1) / kNb;
    // every split keeps >= 4 blocks as launched (ceil(blocks / s) >= 4): the launch
    // gives each split a whole number of blocks, so a cap of blocks / 4 would leave
    // 4.x-block counts that round up to 5
    long long smax = blocks >= 4 ? (blocks - 1) / 3 : 1;
    if (smax > DDT_MAX_SPLITS) smax = DDT_MAX_SPLITS;
    if (smax > max_splits) smax = max_splits;
    if (smax < 1) smax = 1;
    constexpr long long kFixedBlocks = 8;
    long long best = 1, best_cost = -1;
    for (long long sp = 1; sp <= smax; ++sp) {
        const long long waves = (tiles * sp + pairs - 1) / pairs;
        const long long cost = waves * ((blocks + sp - 1) / sp + kFixedBlocks);
        if (best_cost < 0 || cost < best_cost) {
            best = sp;
            best_cost = cost;
        }
    }
    return (int)best;
}

namespace {
// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// q as a [rows][576] bf16 tensor with boxes of kRows rows x box_cols columns
bool encode_q_map(CUtensorMap *map, const uint16_t *q, int64_t rows, uint32_t box_cols,
                  CUtensorMapSwizzle swizzle) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)DDT_D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)DDT_D * 2};
    const cuuint32_t box[2] = {box_cols, (cuuint32_t)kRows};
    const cuuint32_t elem[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(q), dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

cudaError_t launch_attn_partial(const AttnArgs &a, cudaStream_t s) {
    TcParams prm;
    const int64_t rows = (int64_t)a.total_q * a.num_heads;
    if (!encode_q_map(&prm.q_lat, a.q, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_q_map(&prm.q_rope, a.q, rows, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    prm.a = a;
    prm.tiles_per_req = (a.max_q_len * a.num_heads + kRows - 1) / kRows;
    dim3 grid(2 * prm.tiles_per_req, a.num_splits, a.batch);
    return launch_pdl(attn_tc_kernel, grid, dim3(kThreads), kSmemBytes, s, prm);
}

}  // namespace ddt
