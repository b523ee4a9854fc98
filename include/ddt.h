/*
 * ddt.h -- C ABI of the GB300 (sm_103a) DDTree verify step.
 *
 * The stages of one speculative-decoding verify step, as defined on the pages
 * "The DDTree CUDA Graph Fix: Unlocking Speculative Decoding at 109 tok/s on
 * PCIe Blackwell" (section "The DDTree Architecture: Confirming Multiple-Path
 * Evaluation"), "The Architecture of a Speculative Decoding Engine" (sections
 * "The Final Resolution: A Concrete Trace" and "The Forward Pass Pseudocode")
 * and "The 30-Column Mask" (sections "The Message: Tensor Shapes as Evidence",
 * "The Fix: Building Combined Indices", "Mask Stride Formula"):
 *
 *   ddt_build_tree          best-first expansion of per-depth top-k log-probs
 *   ddt_compile_visibility  bit-packed [q_len, prefix + q_len] visibility mask
 *   ddt_build_tree_visibility  the two above in one launch
 *   ddt_verify_attn         tree-verify MLA attention in absorbed form
 *                           (ddt_verify_attn_noalloc: without a caller workspace)
 *   ddt_accept              greedy walk: longest accepted chain + bonus token
 *   ddt_commit_kv           gather the accepted latents after the committed prefix
 *   ddt_tree_links          the tree as first-child / next-sibling links
 *   ddt_accept_sampled      tree rejection sampling with temperature, top-k, top-p
 *   ddt_verify_step         tree + mask, attention, accept (+ commit) in one call;
 *                           ddt_step_graph_* hold the same as one CUDA graph
 *                           (ddt_step_graph_create_io: with the step's host copies)
 *   ddt_build_chain_visibility  a prefill chunk's chain and its causal mask
 *   ddt_prefill_step        chain + causal mask, then the attention, in one call
 *
 * Conventions for every entry point:
 *   - Pointers marked (device) must be device memory of the current CUDA
 *     device; pointers marked (host) are host memory.  The caller owns all
 *     memory.  No entry point allocates device memory; split-KV scratch is a
 *     caller-provided workspace sized by ddt_verify_attn_workspace_size()
 *     (ddt_verify_attn_noalloc uses a fixed array inside the library, and an
 *     instantiated step graph holds CUDA's own graph resources).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Launches are
 *     asynchronous on that stream; no entry point synchronises the host except
 *     ddt_get_error().
 *   - Every kernel is launched with programmatic dependent launch, so it may
 *     start while the previous kernel on the stream is still running.  A
 *     kernel waits for that kernel before it reads anything that an earlier
 *     stage of this ABI writes (tree, mask, split partials) and before its
 *     first write.  Arguments that only the caller writes (q, kv_pool,
 *     kv_indices, the indptr arrays, top-k inputs, target_argmax, and the
 *     sampling accept's temperature, top_k, top_p and logits) may be read before
 *     that wait.  Producing them in a kernel that signals early
 *     completion (cudaTriggerProgrammaticLaunchCompletion) and then calling
 *     an entry point right after it is therefore unsupported.  An ordinary
 *     kernel, a copy or an event between the producer and the call is
 *     enough.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - Arguments checkable on the host are checked before any launch; a failure
 *     returns DDT_ERR_INVALID_ARG / DDT_ERR_UNSUPPORTED / DDT_ERR_WORKSPACE and
 *     launches nothing.  Inconsistencies only visible in device data (indptr
 *     not matching budgets, a kv index outside the pool, a tree deeper than
 *     max_depth, unsorted top-k) are latched by the kernels into a per-device
 *     error word read back by ddt_get_error(); the offending access is skipped
 *     (never performed out of bounds) and the affected outputs are unspecified.
 *   - Launch failures return DDT_ERR_CUDA.
 */
#ifndef DDT_H_
#define DDT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DDT_ABI_VERSION 3

/* Sizes fixed by the absorbed-MLA layout ("The 30-Column Mask", shapes log:
 * Dl=512, Dr=64; "The Forward Pass Pseudocode": scores over c_kv and k_pe,
 * output in the latent space). */
#define DDT_DL 512          /* latent width: values, first part of the keys */
#define DDT_DR 64           /* rope width: second part of the keys */
#define DDT_D 576           /* row width of q and of the latent KV pool */
#define DDT_MAX_DEPTH 7     /* draft block of 8 minus the anchor */
#define DDT_MAX_TOPK 16
#define DDT_MAX_Q_LEN 128   /* budget + 1 */
#define DDT_MAX_SPLITS 128
#define DDT_MAX_VOCAB 262144 /* ddt_accept_sampled */

typedef enum {
    DDT_OK = 0,
    DDT_ERR_INVALID_ARG = 1,   /* bad pointer / size / shape, found on the host */
    DDT_ERR_UNSUPPORTED = 2,   /* valid but outside the supported sizes */
    DDT_ERR_WORKSPACE = 3,     /* workspace missing or too small */
    DDT_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    DDT_ERR_DEVICE_CHECK = 5,  /* a kernel latched a data check (ddt_get_error) */
    DDT_ERR_TIMEOUT = 6        /* a bounded device wait gave up (ddt_get_error) */
} ddt_status;

/* Bits of the device error word (see ddt_get_error). */
#define DDT_DEVERR_QO_INDPTR    0x001u  /* qo_indptr not matching budget+1, q_len limits or [0, total_q] */
#define DDT_DEVERR_KV_INDPTR    0x002u  /* kv_len < q_len or kv_len > max_kv_len */
#define DDT_DEVERR_KV_INDEX     0x004u  /* a kv_indices entry outside [0, pool_rows) */
#define DDT_DEVERR_MASK_INDPTR  0x008u  /* mask_indptr negative or not matching q_len*ceil(kv_len/32) */
#define DDT_DEVERR_TOPK_ORDER   0x010u  /* top-k log-probs not non-increasing (or NaN) */
#define DDT_DEVERR_EXHAUSTED    0x020u  /* budget larger than the implicit tree */
#define DDT_DEVERR_PARENT       0x040u  /* a parent link that is not an earlier node */
#define DDT_DEVERR_DEPTH        0x080u  /* accepted chain longer than max_depth + 1 */
#define DDT_DEVERR_TIMEOUT      0x100u  /* a bounded wait inside a kernel ran out */
#define DDT_DEVERR_ACCEPTED     0x200u  /* accept_len / accepted_nodes not an accepted path */
#define DDT_DEVERR_SAMPLE       0x400u  /* sampling accept: links not a tree, or too few coins */

const char *ddt_status_string(ddt_status s);
int32_t ddt_abi_version(void);

/*
 * ddt_build_tree -- best-first tree from per-depth top-k log-probs.
 * Page: "The DDTree CUDA Graph Fix ..." section "The DDTree Architecture":
 * pop the highest cumulative-log-prob node, add it, push its best child and
 * its next sibling, until `budget` nodes are selected; the tree has
 * budget + 1 nodes (node 0 is the root, the last verified token).
 *
 *   topk_logp  (device) float [batch][max_depth][topk]: log-probs of the
 *              drafter's top-k at draft depth d+1, non-increasing along topk.
 *   topk_ids   (device) int32 [batch][max_depth][topk]: their token ids.
 *   root_id    (device) int32 [batch]: token of node 0.
 *   budget     (device) int32 [batch]: draft nodes to select (0 .. 127).
 *   qo_indptr  (device) int32 [batch+1]: node offsets, q_len_b = budget_b + 1.
 *   node_token, parent, depth
 *              (device) int32 [qo_indptr[batch]] outputs, ragged by qo_indptr:
 *              parent[root] = -1, depth[root] = 0; nodes appear in pop order,
 *              so parent[n] < n.
 * Order among equal scores: smaller depth first, then the path of sibling
 * ranks compared lexicographically.  Scores are fp32 sums root to leaf.
 * Supported: 1 <= topk <= 16, 1 <= max_depth <= 7, budget <= 127.
 */
ddt_status ddt_build_tree(const float *topk_logp, const int32_t *topk_ids,
                          const int32_t *root_id, const int32_t *budget,
                          const int32_t *qo_indptr, int32_t batch, int32_t max_depth,
                          int32_t topk, int32_t *node_token, int32_t *parent,
                          int32_t *depth, void *stream);

/*
 * ddt_mask_indptr -- (host helper) word offsets of the bit-packed mask.
 * Request b's mask is q_len_b rows of W_b = ceil((prefix_b + q_len_b) / 32)
 * uint32 words; mask_indptr[b] = sum over b' < b of q_len_b' * W_b'.
 *   qo_indptr (host) int32 [batch+1]; prefix_len (host) int32 [batch];
 *   mask_indptr (host) int32 [batch+1] output; returns DDT_ERR_INVALID_ARG on
 *   negative sizes or int32 overflow.
 */
ddt_status ddt_mask_indptr(const int32_t *qo_indptr, const int32_t *prefix_len,
                           int32_t batch, int32_t *mask_indptr);

/*
 * ddt_compile_visibility -- the verify mask.
 * Page: "The DDTree CUDA Graph Fix ..." section "The DDTree Architecture"
 * (each node attends to its ancestors plus the shared prefix; all prefix
 * columns visible) and "The 30-Column Mask" section "Mask Stride Formula"
 * (a row spans prefix + q_len columns: prefix first, then tree node j at
 * column prefix + j).
 *
 *   parent      (device) int32 [qo_indptr[batch]] from ddt_build_tree.
 *   qo_indptr   (device) int32 [batch+1].
 *   prefix_len  (device) int32 [batch].
 *   mask_indptr (device) int32 [batch+1] as given by ddt_mask_indptr.
 *   total_words = mask_indptr[batch] (host value: the size of `mask`).
 *   mask        (device) uint32 [total_words] output.  Bit (c mod 32) of word
 *               c / 32 of row i is column c (LSB first); padding bits are 0.
 */
ddt_status ddt_compile_visibility(const int32_t *parent, const int32_t *qo_indptr,
                                  const int32_t *prefix_len, const int32_t *mask_indptr,
                                  int32_t batch, int32_t total_words, uint32_t *mask,
                                  void *stream);

/*
 * ddt_build_tree_visibility -- ddt_build_tree and ddt_compile_visibility in one
 * launch, with the outputs of both: the same tree (node_token, parent, depth)
 * and the same mask words, bit for bit.  One CTA per request: one warp builds
 * the tree while the others write the all-ones prefix words, then the words
 * holding tree columns are written from the tree.  The arguments are those of
 * the two calls (qo_indptr, prefix_len and mask_indptr as for
 * ddt_compile_visibility; `mask` holds mask_indptr[batch] words).  Saving one
 * launch lets a following ddt_verify_attn start earlier.  Device errors are
 * those of the two calls; when the tree cannot be built, its outputs are not
 * written and the mask words that hold tree columns are written as 0.
 */
ddt_status ddt_build_tree_visibility(const float *topk_logp, const int32_t *topk_ids,
                                     const int32_t *root_id, const int32_t *budget,
                                     const int32_t *qo_indptr, const int32_t *prefix_len,
                                     const int32_t *mask_indptr, int32_t batch, int32_t max_depth,
                                     int32_t topk, int32_t *node_token, int32_t *parent,
                                     int32_t *depth, uint32_t *mask, void *stream);

/*
 * ddt_build_chain_visibility -- the tree of a prefill chunk and its mask.
 * Page: "The Architecture of a Speculative Decoding Engine", section "The Core
 * Design Problem: A Unified Forward Pass": prefill, decode and tree verify are
 * one forward that differs only in its mask.  For a chunk of q_len_b new
 * tokens after prefix_len_b cached ones, the tree is the chain
 * parent[i] = i - 1 (parent[0] = -1), depth[i] = i, request-local indices as
 * in ddt_build_tree, and its visibility mask is the causal one: row i sees
 * columns 0 .. prefix_len_b + i.  The mask equals, bit for bit, what
 * ddt_compile_visibility writes for that chain.
 *
 *   qo_indptr, prefix_len, mask_indptr (device) as for ddt_compile_visibility;
 *              1 <= q_len_b <= 128.
 *   parent, depth (device) int32 [qo_indptr[batch]] outputs.
 *   mask       (device) uint32 [mask_indptr[batch]] output.
 * One launch, no host synchronisation: it can be captured in a CUDA graph.
 * A request whose q_len is out of range or whose mask range is not
 * q_len * W words latches DDT_DEVERR_MASK_INDPTR and its mask is not written
 * (its chain is still written when q_len is in range).
 */
ddt_status ddt_build_chain_visibility(const int32_t *qo_indptr, const int32_t *prefix_len,
                                      const int32_t *mask_indptr, int32_t batch, int32_t *parent,
                                      int32_t *depth, uint32_t *mask, void *stream);

/*
 * Split-KV sizing.  ddt_verify_attn_num_splits() returns the split count the
 * library would pick for this shape on `num_sms` SMs (num_sms <= 0: query the
 * current device).  A split covers ceil(max_kv_len / num_splits) kv columns
 * rounded up to whole 64-column tiles, so fewer splits than asked may cover
 * the range: ddt_verify_attn_launched_splits() returns how many splits a call
 * with `num_splits` (>= 1) actually launches (1 = no combine kernel).
 * ddt_verify_attn_workspace_size() returns the workspace bytes ddt_verify_attn
 * needs for `num_splits` splits (0 bytes for one split): num_splits * total_q
 * * num_heads * (512 + 1) * 4 bytes, 256-byte aligned.
 */
int32_t ddt_verify_attn_num_splits(int32_t batch, int32_t num_heads, int32_t max_q_len,
                                   int32_t max_kv_len, int32_t num_sms);
int32_t ddt_verify_attn_launched_splits(int32_t max_kv_len, int32_t num_splits);
size_t ddt_verify_attn_workspace_size(int32_t total_q, int32_t num_heads, int32_t num_splits);

/*
 * ddt_verify_attn -- tree-verify MLA attention, absorbed form.
 * Pages: "The Architecture of a Speculative Decoding Engine" section "The
 * Forward Pass Pseudocode" (verify_attn(q_abs, q_pe, c_kv, k_pe, mask, scale)
 * returning out_latent); "The 30-Column Mask" sections "The Message: Tensor
 * Shapes as Evidence" and "The Fix: Building Combined Indices" (q = [tokens,
 * heads, 576], one 576-wide latent row per token shared by all heads, indices
 * = prefix slots ++ the tree nodes' slots, mask row stride prefix + q_len);
 * the split-KV partial pass + log-sum-exp combine follows "The 30-Column
 * Mask" section "The Context: Building a Custom Verify Attention Kernel".
 *
 * For row (token t of request b = tree node i, head h):
 *   s_j  = scale * <q[t,h,0:576], kv_pool[kv_indices[kv_indptr[b]+j], 0:576]>
 *          over the columns j in [0, kv_len_b) whose mask bit (i, j) is set,
 *   out[t,h,:] = sum_j softmax(s)_j * kv_pool[...same row..., 0:512],
 *   lse[t,h]   = log(sum_j exp(s_j))   (natural log).
 * Every mask bit is honoured: any bit pattern is valid, not only the
 * ancestors-plus-prefix masks of a tree.  A row with no visible column gets
 * out = 0 and lse = -inf.
 *
 *   q           (device) bf16 [total_q][num_heads][576] (absorbed q_nope ++ roped q_pe).
 *   kv_pool     (device) bf16 [pool_rows][576] (c_kv ++ k_pe), 16-byte aligned.
 *   kv_indices  (device) int32 [kv_indptr[batch]]: per request prefix_len_b
 *               prefix slots followed by q_len_b tree-node slots in node order.
 *   kv_indptr   (device) int32 [batch+1]; kv_len_b = prefix_len_b + q_len_b.
 *   qo_indptr   (device) int32 [batch+1]; q_len_b <= max_q_len <= 128.
 *   mask, mask_indptr (device) bit-packed as ddt_compile_visibility writes it:
 *               request b's rows start at word mask_indptr[b], each
 *               ceil(kv_len_b / 32) words, bit (j mod 32) of word j / 32 is
 *               column j.  The mask may be the output of the kernel launched
 *               just before on the same stream.
 *   total_q     = qo_indptr[batch] (host value); max_q_len / max_kv_len are
 *               host-side upper bounds used to size the grid.
 *   num_splits  0 = choose (ddt_verify_attn_num_splits), else 1..128.
 *   out         (device) float [total_q][num_heads][512].
 *   lse         (device) float [total_q][num_heads] or NULL.
 *   workspace   (device) >= ddt_verify_attn_workspace_size(total_q, num_heads,
 *               splits) bytes, 256-byte aligned; may be NULL when one split.
 * Supported: num_heads >= 1 (up to 128).
 * Device checks (latched, the request's rows left unwritten): q_len outside
 * [1, max_q_len] or qo_indptr outside [0, total_q] (DDT_DEVERR_QO_INDPTR),
 * kv_len outside [q_len, max_kv_len] or a negative kv_indptr
 * (DDT_DEVERR_KV_INDPTR), a negative mask_indptr or a request whose words do
 * not number q_len * ceil(kv_len / 32) (DDT_DEVERR_MASK_INDPTR), a kv_indices
 * entry outside the pool (DDT_DEVERR_KV_INDEX: row 0 is read instead).
 */
ddt_status ddt_verify_attn(const uint16_t *q, const uint16_t *kv_pool, int64_t pool_rows,
                           const int32_t *kv_indices, const int32_t *kv_indptr,
                           const int32_t *qo_indptr, const uint32_t *mask,
                           const int32_t *mask_indptr, int32_t batch, int32_t num_heads,
                           int32_t total_q, int32_t max_q_len, int32_t max_kv_len, float scale,
                           int32_t num_splits, float *out, float *lse, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * ddt_verify_attn_noalloc -- ddt_verify_attn without a caller workspace.
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory: an engine that reserved all device
 * memory for its own pool up front, a plain C host without an allocator, or
 * a decode loop in which a cudaMalloc (which may synchronise the whole
 * device) is not allowed.  The call allocates nothing: when it splits the kv
 * range, the split results live in a fixed array of
 * DDT_NOALLOC_SCRATCH_BYTES inside libddt.so's device memory, which every GPU
 * that loads the library holds until the process exits.
 *
 * Arguments, outputs and errors are those of ddt_verify_attn minus the
 * workspace.  ddt_verify_attn_noalloc_splits() returns the number of splits a
 * call with these sizes and `num_splits` launches.  With num_splits = 0 the library picks the split count as
 * ddt_verify_attn does, but only among the counts whose split results fit
 * DDT_NOALLOC_SCRATCH_BYTES (see ddt_verify_attn_workspace_size), down to 1,
 * which needs no scratch; so a long kv range over many rows may run with
 * fewer splits here than through ddt_verify_attn.  An explicit num_splits
 * that needs more scratch than that returns DDT_ERR_WORKSPACE and launches
 * nothing.
 * The first call on a device looks up the array's device address for that
 * device; make that first call before any stream capture.  All calls share
 * the one array: calls that overlap on the GPU (other streams, other
 * threads) race on it and must be serialised by the caller.  Every scratch
 * entry a call reads is written earlier in the same call, so nothing has to
 * be cleared between calls.
 */
#define DDT_NOALLOC_SCRATCH_BYTES (32u << 20)
int32_t ddt_verify_attn_noalloc_splits(int32_t batch, int32_t num_heads, int32_t total_q,
                                       int32_t max_q_len, int32_t max_kv_len, int32_t num_splits);
ddt_status ddt_verify_attn_noalloc(const uint16_t *q, const uint16_t *kv_pool, int64_t pool_rows,
                                   const int32_t *kv_indices, const int32_t *kv_indptr,
                                   const int32_t *qo_indptr, const uint32_t *mask,
                                   const int32_t *mask_indptr, int32_t batch, int32_t num_heads,
                                   int32_t total_q, int32_t max_q_len, int32_t max_kv_len,
                                   float scale, int32_t num_splits, float *out, float *lse,
                                   void *stream);

/*
 * ddt_accept -- greedy tree acceptance (follow_verified_tree).
 * Page: "The DDTree CUDA Graph Fix ..." section "The DDTree Architecture"
 * (walk from the root following the target's argmax into the matching child
 * until none matches; return the longest accepted chain plus one bonus
 * token); "The Oracle Drafter" section "The Engine Interface Design"
 * (outputs: accepted path, accept length, commit tokens, bonus);
 * "The Architecture of a Speculative Decoding Engine" section "The Final
 * Resolution" (the cache grows by accept_len, which counts the root).
 *
 *   node_token, parent (device) int32 [qo_indptr[batch]] (a ddt_build_tree tree).
 *   qo_indptr     (device) int32 [batch+1].
 *   target_argmax (device) int32 [qo_indptr[batch]]: target model's argmax at each node.
 *   accept_len    (device) int32 [batch]: accepted nodes incl. the root (1 .. max_depth+1).
 *   accepted_nodes(device) int32 [batch][max_depth+1]: node indices, -1 padded.
 *   commit_tokens (device) int32 [batch][max_depth+1]: accepted draft tokens then
 *                 the bonus token (accept_len entries), -1 padded.
 *   bonus         (device) int32 [batch]: target argmax at the last accepted node.
 * Among children carrying the same token the lowest node index is followed.
 */
ddt_status ddt_accept(const int32_t *node_token, const int32_t *parent,
                      const int32_t *qo_indptr, const int32_t *target_argmax, int32_t batch,
                      int32_t max_depth, int32_t *accept_len, int32_t *accepted_nodes,
                      int32_t *commit_tokens, int32_t *bonus, void *stream);

/*
 * ddt_tree_links -- the tree in the format of a tree-sampling kernel.
 * Page: "The DDTree CUDA Graph Fix ...", section "Temperature Support:
 * Already Working for Linear, Planned for DDTree" (the parent lists become
 * retrieve_index, retrieve_next_token and retrieve_next_sibling).
 *
 *   parent        (device) int32 [qo_indptr[batch]] from ddt_build_tree.
 *   qo_indptr     (device) int32 [batch+1].
 *   first_child   (device) int32 [qo_indptr[batch]] out: node n's lowest-index
 *                 child (request-local index) or -1 (retrieve_next_token).
 *   next_sibling  (device) int32 [qo_indptr[batch]] out: the next higher-index
 *                 child of n's parent or -1 (retrieve_next_sibling).
 *   retrieve_index(device) int32 [qo_indptr[batch]] out: qo_indptr[b] + n.
 */
ddt_status ddt_tree_links(const int32_t *parent, const int32_t *qo_indptr, int32_t batch,
                          int32_t *first_child, int32_t *next_sibling, int32_t *retrieve_index,
                          void *stream);

/*
 * ddt_accept_sampled -- sampling accept: tree rejection sampling on the
 * target distribution, the planned temperature support of "The DDTree CUDA
 * Graph Fix ..." (section "Temperature Support: Already Working for Linear,
 * Planned for DDTree").  The pages give no algorithm; the reading taken
 * (target-only, deterministic drafts) is:
 *   - p(n) = softmax(target_logits[n] / temperature[b]) over the tokens whose
 *     logit is at least the top_k[b]-th largest (ties kept; all tokens when
 *     top_k[b] <= 0 or >= vocab); temperature[b] <= 0 gives one-hot at the
 *     argmax (lowest id on ties);
 *   - top-p, after top-k: tau is the largest logit x whose mass S(x), the
 *     mass of p over the tokens with logit >= x, reaches top_p[b]; the tokens
 *     with logit >= tau are kept (ties at tau all kept) and p is renormalised
 *     over them.  top_p == NULL, or top_p[b] outside (0, 1), applies none;
 *   - at node n the children are tried in index order against the residual r
 *     (p minus the tokens already rejected at n): child i, with token t, is
 *     taken when coins[n][i] < r(t) / mass(r), otherwise t leaves r;
 *   - if no child is taken, the bonus is the first token id whose cumulative
 *     mass in r exceeds coins[n][coin_stride-1] * mass(r), and the walk stops.
 * Every emitted token is then distributed as p.  At temperature 0 (or top_k
 * 1) this is exactly ddt_accept with target_argmax = the logits' argmax.
 * Probabilities are fp32 on the device, so a coin within ~1e-6 of a threshold
 * may decide differently from an fp64 evaluation.  The top-p set is found
 * with masses summed in 2^-40 fixed point (the same set on every run); it can
 * differ from an fp64 evaluation only when S crosses top_p within ~1e-6.  If rounding leaves the
 * bonus target at or above the residual's total, the bonus is a token with
 * residual mass near the end of the id range (the argmax if r is empty).
 *
 *   node_token, first_child, next_sibling, qo_indptr
 *                 (device) the tree (ddt_build_tree) and its links (ddt_tree_links).
 *   target_logits (device) float [qo_indptr[batch]][vocab]: target logits at each node.
 *   temperature   (device) float [batch]; top_k (device) int32 [batch];
 *   top_p         (device) float [batch], or NULL.
 *   coins         (device) float [qo_indptr[batch]][coin_stride], uniform in [0,1):
 *                 coin i for the i-th child tried at a node, the last for the
 *                 bonus; coin_stride >= 1 + the largest number of children.
 *   outputs       as for ddt_accept.
 * Supported: 1 <= vocab <= DDT_MAX_VOCAB.
 * Device checks: links that do not form the tree, or a node with more
 * children than coin_stride - 1 or than DDT_MAX_TOPK + 1 (DDT_DEVERR_SAMPLE;
 * outputs unset), a walk deeper than max_depth (DDT_DEVERR_DEPTH).
 */
ddt_status ddt_accept_sampled(const int32_t *node_token, const int32_t *first_child,
                              const int32_t *next_sibling, const int32_t *qo_indptr,
                              const float *target_logits, int32_t vocab, const float *temperature,
                              const int32_t *top_k, const float *top_p, const float *coins,
                              int32_t coin_stride,
                              int32_t batch, int32_t max_depth, int32_t *accept_len,
                              int32_t *accepted_nodes, int32_t *commit_tokens, int32_t *bonus,
                              void *stream);

/*
 * ddt_commit_kv -- KV commit after acceptance (compaction of the accepted
 * latents).
 * Page: "The Architecture of a Speculative Decoding Engine", sections "The
 * Final Resolution: A Concrete Trace" and the compaction scheme before it:
 * the step appended every tree node's latent after the committed prefix
 * (node j at position P_b + j, the root at P_b); after acceptance the
 * accepted nodes' latents are gathered into contiguous positions
 * P_b .. P_b + accept_len - 1, the cache grows by accept_len, and the bonus
 * token becomes the next step's root at position P_b + accept_len.
 *
 * With the slot layout of ddt_verify_attn (position c of request b lives in
 * pool row kv_indices[kv_indptr[b] + c]), for k = 0 .. accept_len[b]-1:
 *   row(P_b + k) <- row(P_b + accepted_nodes[b][k])   (all 576 entries)
 * where every source row is read before any destination row is written, so
 * a destination that is also a later source (node 2 -> position 1 while
 * node 5 -> position 2) moves the original latent.  No other pool row is
 * written.
 *
 *   kv_pool       (device) bf16 [pool_rows][576], updated in place.
 *   kv_indices, kv_indptr, qo_indptr
 *                 (device) as for ddt_verify_attn (P_b = kv_len_b - q_len_b).
 *   accept_len, accepted_nodes
 *                 (device) as written by ddt_accept (max_depth+1 entries per request).
 *   new_len       (device) int32 [batch] or NULL: P_b + accept_len[b], the
 *                 committed cache length.
 * Device checks: accept_len in [1, min(q_len, max_depth+1)], accepted_nodes
 * starting at 0, strictly increasing and below q_len (DDT_DEVERR_ACCEPTED);
 * pool rows in range (DDT_DEVERR_KV_INDEX).  A request that fails a check is
 * left unchanged.
 */
ddt_status ddt_commit_kv(uint16_t *kv_pool, int64_t pool_rows, const int32_t *kv_indices,
                         const int32_t *kv_indptr, const int32_t *qo_indptr,
                         const int32_t *accept_len, const int32_t *accepted_nodes, int32_t batch,
                         int32_t max_depth, int32_t *new_len, void *stream);

/*
 * ddt_get_error -- read and clear the current device's error word.
 * Synchronises `stream`, copies the word to *device_error (host; may be NULL)
 * and resets it.  Returns DDT_OK when the word was 0, DDT_ERR_TIMEOUT when the
 * timeout bit was set, DDT_ERR_DEVICE_CHECK for any other bit, DDT_ERR_CUDA
 * when the copy failed.
 */
ddt_status ddt_get_error(void *stream, uint32_t *device_error);

/*
 * ddt_verify_step -- one verify step in one call: ddt_build_tree_visibility,
 * ddt_verify_attn, ddt_accept and, when `commit_kv` is set, ddt_commit_kv,
 * launched in that order on `stream`.  It is the whole per-iteration data flow
 * of "The Oracle Drafter" (section "The Engine Interface Design"), with every
 * stage on the GPU so that the step can be captured and replayed as one CUDA
 * graph ("The DDTree CUDA Graph Fix ...", section "Implications and the Path
 * Forward": graphs were the largest single gain on the pages).
 *
 * Each field has the meaning, layout and ownership it has in the call that
 * consumes it; `total_mask_words` = mask_indptr[batch] is the size of `mask`.
 * The step's attention uses the mask the step has just built, a tree mask
 * (every prefix column visible, no column after the row's own node): it reads
 * no mask word for blocks of prefix columns, so it streams the prefix while
 * the tree build is still running, and it skips the columns after each row
 * tile's last node.
 * Returns the first non-OK status of the four calls; nothing after that call
 * is launched.
 */
typedef struct {
    /* tree inputs */
    const float *topk_logp;
    const int32_t *topk_ids;
    const int32_t *root_id;
    const int32_t *budget;
    int32_t max_depth;
    int32_t topk;
    /* layout: batch, indptrs and host-side bounds */
    int32_t batch;
    int32_t total_q;
    int32_t max_q_len;
    int32_t max_kv_len;
    int32_t total_mask_words;
    const int32_t *qo_indptr;
    const int32_t *kv_indptr;
    const int32_t *prefix_len;
    const int32_t *mask_indptr;
    /* attention inputs */
    const uint16_t *q;
    uint16_t *kv_pool; /* read by the attention, written by the commit */
    int64_t pool_rows;
    const int32_t *kv_indices;
    int32_t num_heads;
    float scale;
    int32_t num_splits; /* 0: the library's choice */
    void *workspace;
    size_t workspace_bytes;
    /* accept input */
    const int32_t *target_argmax;
    /* outputs */
    int32_t *node_token;
    int32_t *parent;
    int32_t *depth;
    uint32_t *mask;
    float *out;
    float *lse; /* may be NULL */
    int32_t *accept_len;
    int32_t *accepted_nodes;
    int32_t *commit_tokens;
    int32_t *bonus;
    /* KV commit: skipped when commit_kv is 0 */
    int32_t commit_kv;
    int32_t *new_len; /* may be NULL */
} ddt_step_args;

ddt_status ddt_verify_step(const ddt_step_args *args, void *stream);

/*
 * ddt_prefill_step -- one prefill chunk as one call: ddt_build_chain_visibility
 * then the attention of ddt_verify_attn under that causal mask, on `stream`.
 * Page: "The Architecture of a Speculative Decoding Engine", section "The Core
 * Design Problem: A Unified Forward Pass" (prefill is the verify forward with
 * a causal mask).  It reads the fields of `args` that those two calls take
 * (layout, indptrs, attention inputs, workspace) and writes parent, depth,
 * mask, out and lse; the tree inputs, target_argmax and the accept and commit
 * outputs are not read.  The new tokens' latents must already sit at kv
 * columns prefix_len_b .. prefix_len_b + q_len_b - 1 (the chunk's own cache
 * rows); no commit follows, because a chain's accepted path is the identity.
 * Like the verify step, the attention knows the mask's shape (every prefix
 * column visible, none after the row's own token) and reads no mask word for
 * prefix blocks.  Returns the first non-OK status of the two calls.
 */
ddt_status ddt_prefill_step(const ddt_step_args *args, void *stream);

/*
 * A CUDA graph of one ddt_verify_step, owned by the library: create captures
 * the step's launches once (the buffers in `args` must then stay allocated and
 * keep their sizes: the verify buffers are sized for budget+1 tokens per
 * request, "The DDTree CUDA Graph Fix ...", section "The CUDA Graph Crash: A
 * Tale of Two Token Counts"); launch replays them on `stream`; destroy frees
 * the graph.
 * Create makes no launch of its own; it returns the status of the captured
 * ddt_verify_step, or DDT_ERR_CUDA if capture or instantiation fails.
 */
typedef struct ddt_step_graph ddt_step_graph;
ddt_status ddt_step_graph_create(const ddt_step_args *args, ddt_step_graph **graph);
/*
 * ddt_step_graph_create_io -- the same graph with the step's host traffic in
 * it: a copy of `in_bytes` from h_in to d_in before the step and a copy of
 * `out_bytes` from d_out to h_out after it, so that one launch takes a step's
 * inputs from host memory and returns its results there.  h_in and h_out are
 * pinned host memory (cudaHostAlloc or registered), d_in and d_out device
 * memory that the caller lays out so that the step's inputs and results fall
 * inside them (one packed buffer each way); all four stay allocated for the
 * graph's life.  A size of 0 omits that copy.  Where a host buffer has a device
 * pointer (cudaHostGetDevicePointer), both addresses are 16-byte aligned and the
 * size is whole 16-byte units, the copy is a kernel reading or writing the host
 * memory through that pointer; otherwise it is a copy-engine transfer.  Returns
 * DDT_ERR_INVALID_ARG for a null or unpinned host buffer, else as
 * ddt_step_graph_create.
 */
ddt_status ddt_step_graph_create_io(const ddt_step_args *args, const void *h_in, void *d_in,
                                    size_t in_bytes, void *h_out, const void *d_out,
                                    size_t out_bytes, ddt_step_graph **graph);
ddt_status ddt_step_graph_launch(ddt_step_graph *graph, void *stream);
ddt_status ddt_step_graph_destroy(ddt_step_graph *graph);

/*
 * ddt_selftest_wait_timeout -- exercise the failure path of the bounded device
 * waits without faulting the GPU.  Launches one 32-thread kernel on `stream`
 * that waits, with the same bounded mbarrier wait the verify kernels use (but
 * a limit of `poll_limit` polls, 1 .. 2^24), on a barrier that nothing ever
 * arrives on.  The wait gives up, the kernel latches DDT_DEVERR_TIMEOUT into
 * the device error word and exits; ddt_get_error() then reports
 * DDT_ERR_TIMEOUT and the context stays usable.  Returns DDT_ERR_INVALID_ARG
 * for a limit out of range, DDT_ERR_CUDA if the launch fails, else DDT_OK.
 */
ddt_status ddt_selftest_wait_timeout(uint32_t poll_limit, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* DDT_H_ */
