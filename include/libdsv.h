/*
 * libdsv -- C ABI of the DSV hot path on one GB300 (sm_103a).
 *
 * DSV ("DSV: Exploiting Dynamic Sparsity to Accelerate Large-Scale Video DiT
 * Training", summarised on gist.science, arXiv 2502.07590) trains video DiTs
 * with per-head, per-step sparse attention: a rank-r predictor (W_lr^Q,
 * W_lr^K) approximates QK^T, a fused low-rank MatMul + Top-K picks each query
 * group's critical keys without ever storing the S x S scores, and attention
 * (forward and backward) runs on the selected keys only.
 *
 * Conventions shared by every call:
 *  - Tensors Q, K, V, O, dO, dQ, dK, dV are bf16, layout [B][H][S][d],
 *    contiguous, device memory, 16-byte aligned. S = T*Y*X tokens of a
 *    T x Y x X latent grid, token s = (t*Y + y)*X + x.
 *  - W_lr^Q, W_lr^K are bf16 [H][d][r] (row-major d x r per head), device.
 *  - A query group is one gt x gy x gx cube of the grid; groups are numbered
 *    row-major over the (T/gt, Y/gy, X/gx) grid of cubes. n_groups = S/G.
 *  - "Problem" p = b*H + h indexes the B*H independent (batch, head) pairs.
 *  - Index sets: row (p, g) holds k_p ascending int32 key positions at
 *    idx + idx_offset[p] + g*k_p (device memory).
 *  - Every buffer is owned by the caller; libdsv allocates nothing and keeps
 *    no state between calls (dsv_lowrank_topk_noalloc, below, instead uses a
 *    fixed array inside the library). Scratch space is the caller's `workspace`
 *    (device, 256-byte aligned) of at least the size the matching
 *    dsv_*_workspace_size() call reports.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*).
 *    Argument errors are returned synchronously before anything is launched.
 *    Launch failures return DSV_ERR_CUDA. Conditions found on the device
 *    (a wait that ran out) are written to the caller's device word `dev_status`
 *    (int32, zero it before the call; libdsv only ever raises it), which the
 *    caller reads after synchronising (dsv_read_status does both). After a
 *    wait ran out, the call's later kernels see incomplete data; their
 *    consistency checks then leave the word at DSV_ERR_TIMEOUT.
 *  - Supported sizes: d in {64, 128}; r in {16, 32, 64}; G = gt*gy*gx in
 *    {64, 128}; S a multiple of 128 and < 2^31; 1 <= k <= S; B*H <= 256.
 */
#ifndef LIBDSV_H
#define LIBDSV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSV_OK = 0,
  DSV_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or shape */
  DSV_ERR_UNSUPPORTED = 2,   /* valid request outside the supported sizes */
  DSV_ERR_WORKSPACE = 3,     /* workspace missing or too small */
  DSV_ERR_CUDA = 4,          /* a CUDA launch or API call failed */
  DSV_ERR_TIMEOUT = 5,       /* device: a bounded wait ran out */
  DSV_ERR_OVERFLOW = 6,      /* reserved (no current call raises it) */
  DSV_ERR_CANDIDATES = 7     /* device: a top-k row failed its internal consistency check (it did not come
                                out with exactly k keys); no valid input raises it */
} dsv_status;

/* Problem shape: B batches x H heads, latent grid T x Y x X, head dim d. */
typedef struct {
  int64_t B, H, T, Y, X, d;
} dsv_shape;

/* Query-group cube gt x gy x gx; it must divide the grid. */
typedef struct {
  int32_t gt, gy, gx;
} dsv_group;

/* Human-readable name of a status code (static string, never NULL). */
const char* dsv_status_string(dsv_status s);

/* Synchronises `stream`, then copies the device status word to *host_out.
 * Returns DSV_ERR_CUDA if either step fails. */
dsv_status dsv_read_status(const int32_t* dev_status, int32_t* host_out, void* stream);

/* ------------------------------------------------------------------------
 * dsv_set_wait_limit_ns -- how long a kernel's pipeline waits before giving up.
 * Not part of the DSV method (the pages have no counterpart): it sets the
 * failure path that guards every wait inside the libdsv kernels. A wait that
 * runs out raises DSV_ERR_TIMEOUT in the call's dev_status word and the block
 * unwinds: it waits for the copies and MMAs it has already issued (those
 * complete by themselves, under a fixed 2 s limit), releases its tensor
 * memory and exits, so the call's outputs are incomplete but the context
 * stays usable. The default is 2,000,000,000 ns (2 s). The value applies to
 * every call launched after this returns, from any host thread of the
 * process; the previous value is returned. 0 makes every wait that has not
 * already completed give up at once, which is how the tests run the failure
 * path; production code has no reason to lower it.
 * ---------------------------------------------------------------------- */
uint64_t dsv_set_wait_limit_ns(uint64_t ns);

/* ------------------------------------------------------------------------
 * dsv_lowrank_topk -- fused low-rank MatMul + per-group Top-K.
 * Passage: technical summary section 2.2 ("efficient kernels": the low-rank
 * MatMul and the Top-K selection are fused so the O(S^2) score matrix is
 * never stored) with section 2.1 (per-head low-rank predictors W_lr^Q,
 * W_lr^K approximating QK^T; critical KV estimation) and the query grouping
 * of section 2.2.
 *
 * For every problem p with idx_offset[p] >= 0 and every group g:
 *   q_lr = Q W_lr^Q, k_lr = K W_lr^K (fp32 accumulate of exact bf16 products)
 *   s_gj = mean over the group's queries i of q_lr,i . k_lr,j
 *   idx row (p, g) = the k_p keys j with the largest s_gj, ties to the lower
 *   j, written in ascending order.
 * Problems with idx_offset[p] < 0 are skipped (dense heads).
 * The selection is exact for every input with finite scores, however the
 * scores cluster: the k-th score's histogram bin is narrowed by radix
 * rounds over the score's bits until it holds at most 4096 keys (the ones
 * completing the row found by a radix select over score and key) or a
 * single value (taken lowest key first).
 * k_per_head, idx_offset: HOST arrays of B*H entries (read during the call).
 * Device errors: DSV_ERR_TIMEOUT on a stalled pipeline (the rows are then
 * incomplete); DSV_ERR_CANDIDATES only if an internal consistency check
 * fails.
 * ---------------------------------------------------------------------- */
size_t dsv_lowrank_topk_workspace_size(dsv_shape shape, int32_t r, dsv_group group);
dsv_status dsv_lowrank_topk(const void* Q, const void* K, const void* Wq_lr, const void* Wk_lr, dsv_shape shape,
                            int32_t r, dsv_group group, const int32_t* k_per_head, const int64_t* idx_offset,
                            int32_t* idx, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                            void* stream);

/* ------------------------------------------------------------------------
 * dsv_lowrank_topk_noalloc -- dsv_lowrank_topk for callers that cannot
 * allocate device memory.
 * The DSV pages have no counterpart to this call; it exists for callers such
 * as a plugin whose enqueue step may not allocate, a serving loop with a
 * device memory budget fixed at start-up, or a host runtime that owns every
 * allocation and cannot lend a workspace.
 *
 * Same inputs, outputs and results as dsv_lowrank_topk, but the scratch space
 * is a fixed 64 MiB array compiled into libdsv (reserved on every GPU that
 * loads this part of the library, until the process exits). No workspace is
 * passed and nothing is allocated: the call makes no cudaMalloc/cudaFree and
 * no allocating library call.
 *  - Shapes whose dsv_lowrank_topk_workspace_size() exceeds 64 MiB are
 *    rejected with DSV_ERR_WORKSPACE before anything is launched.
 *  - The first call on a device looks up the array's device address (and
 *    loads the module there); make that first call before any stream capture.
 *    The address is kept per device and CUDA context: after a device reset
 *    (a new context) the next call looks it up again, so it too should come
 *    before any capture.
 *  - Every call uses the same array. The call clears what must start at zero
 *    itself, but calls whose work overlaps on the GPU (different streams, or
 *    several host threads) race on it: serialise them.
 * ---------------------------------------------------------------------- */
dsv_status dsv_lowrank_topk_noalloc(const void* Q, const void* K, const void* Wq_lr, const void* Wk_lr,
                                    dsv_shape shape, int32_t r, dsv_group group, const int32_t* k_per_head,
                                    const int64_t* idx_offset, int32_t* idx, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * dsv_coverage -- smallest k per problem covering `mass` of the predicted
 * softmax mass.
 * Passage: technical summary section 2.1 (critical KV are the pairs that
 * carry over 90% of the attention score; the OP dispatcher decides per block
 * from the current sparsity level).
 *
 * With the group scores s_gj of dsv_lowrank_topk and logits scale*s_gj, let
 * m_g(k) be the total softmax probability of group g's k most probable keys
 * and C(k) the mean of m_g(k) over all groups. k_cov[p] = min{k : C(k) >=
 * mass}. Per group the probabilities are binned (128 bins of width
 * range/128 over the group's logit range, 64 bins when r = 64) and m_g is
 * interpolated inside a bin assuming log-probabilities spread evenly across
 * it.
 * k_cov: DEVICE int32 [B*H]. curve (optional, may be NULL): DEVICE float
 * [B*H][n_curve] (n_curve <= 1024), C(k) sampled at k = ceil((i+1)*S/n_curve).
 * S <= 4186112 (64 key chunks of at most 65535 keys; DSV_ERR_UNSUPPORTED
 * otherwise).
 * ---------------------------------------------------------------------- */
size_t dsv_coverage_workspace_size(dsv_shape shape, int32_t r, dsv_group group);
dsv_status dsv_coverage(const void* Q, const void* K, const void* Wq_lr, const void* Wk_lr, dsv_shape shape,
                        int32_t r, dsv_group group, float scale, float mass, int32_t* k_cov, float* curve,
                        int32_t n_curve, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        void* stream);

/* ------------------------------------------------------------------------
 * dsv_coverage_topk -- dsv_coverage and dsv_lowrank_topk in one call.
 * Passage: technical summary sections 2.1 and 2.2, as for the two calls.
 *
 * Same arguments, outputs and device errors as dsv_coverage (scale, mass,
 * k_cov, curve, n_curve) followed by dsv_lowrank_topk (k_per_head,
 * idx_offset, idx); k_cov, curve and idx hold exactly the values the two
 * separate calls write. When every problem takes a top-k with 1 <= k < S
 * (no dense entry, no k = S), the key projection, the group-mean
 * projection and the per-row score range are computed once and serve both,
 * and the coverage pass's per-row bin counts locate each row's k-th score,
 * so the top-k runs no histogram pass of its own; otherwise the two calls
 * run one after the other. The workspace is at least
 * dsv_coverage_topk_workspace_size() bytes (the two calls' buffers side by
 * side); S <= 4186112 as for dsv_coverage.
 * ---------------------------------------------------------------------- */
size_t dsv_coverage_topk_workspace_size(dsv_shape shape, int32_t r, dsv_group group);
dsv_status dsv_coverage_topk(const void* Q, const void* K, const void* Wq_lr, const void* Wk_lr, dsv_shape shape,
                             int32_t r, dsv_group group, float scale, float mass, int32_t* k_cov, float* curve,
                             int32_t n_curve, const int32_t* k_per_head, const int64_t* idx_offset, int32_t* idx,
                             void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * dsv_plan_heads -- the OP dispatcher, per head (host only, no GPU).
 * Passage: technical summary section 2.1 (the OP dispatcher activates sparse
 * attention per block according to the current sparsity level).
 *
 * For each of n entries: dense[p] = k_cov[p] > dense_frac*S (then k_h[p] = S
 * and idx_offset[p] = -1); otherwise k_h[p] = clamp(k_cov[p], lo, hi) with
 * lo = round-half-up(lo_frac*S), hi = round-half-up(hi_frac*S), and the
 * sparse rows are packed back to back: idx_offset[p] = sum over earlier
 * sparse p' of n_groups*k_h[p']. *idx_total = total int32 entries needed.
 * All pointers are HOST memory.
 * ---------------------------------------------------------------------- */
dsv_status dsv_plan_heads(const int32_t* k_cov, int32_t n, int64_t S, int64_t n_groups, double lo_frac,
                          double hi_frac, double dense_frac, int32_t* k_h, uint8_t* dense, int64_t* idx_offset,
                          int64_t* idx_total);

/* ------------------------------------------------------------------------
 * dsv_plan_gpus -- sparse head-wise context parallelism: heads to GPUs by
 * their cost (host only, no GPU).
 * Passage: technical summary section 2.3 (head-wise CP re-balancing: each
 * head's assignment to a GPU follows its sparsity so that the compute load
 * balances across GPUs).
 *
 * cost[p] >= 0 is head p's work (its k_h for a sparse head, S for a dense
 * one: attention work is proportional to S k_h d). Longest processing time
 * first: heads in order of decreasing cost (ties: lower head first), each to
 * the GPU with the least load so far (ties: lower GPU); with equal_counts != 0
 * only GPUs holding fewer than ceil(n / n_gpus) heads take one (an equal split
 * of the heads, as head-wise parallelism lays them out). gpu_of[p] receives
 * the GPU of head p; load (optional, may be NULL) the total cost per GPU.
 * The largest load is within 4/3 of the best possible when equal_counts = 0.
 * All pointers are HOST memory: cost [n], gpu_of [n], load [n_gpus].
 * DSV_ERR_INVALID_ARG for n < 1, n_gpus < 1, a NULL cost/gpu_of or a
 * negative cost.
 * ---------------------------------------------------------------------- */
dsv_status dsv_plan_gpus(const int64_t* cost, int32_t n, int32_t n_gpus, int32_t equal_counts, int32_t* gpu_of,
                         int64_t* load);

/* ------------------------------------------------------------------------
 * dsv_sparse_attn_fwd -- query-grouped sparse attention, forward.
 * Passage: technical summary section 2.1 (full attention computed on the
 * critical KV pairs only) and section 2.2 (query grouping: a group of
 * adjacent queries shares one key index set).
 *
 * For query i of group g of problem p, with I = idx row (p, g) (or all S keys
 * when idx == NULL or idx_offset[p] < 0, the dense case):
 *   O_i = sum_{j in I} softmax_j(scale q_i.k_j) v_j      (bf16 out)
 *   LSE_i = ln sum_{j in I} exp(scale q_i.k_j)           (fp32 [B][H][S])
 * k_per_head, idx_offset: HOST arrays of B*H entries, or NULL with idx NULL.
 * ---------------------------------------------------------------------- */
size_t dsv_sparse_attn_fwd_workspace_size(dsv_shape shape, dsv_group group);
dsv_status dsv_sparse_attn_fwd(const void* Q, const void* K, const void* V, const int32_t* idx,
                               const int32_t* k_per_head, const int64_t* idx_offset, dsv_shape shape,
                               dsv_group group, float scale, void* O, float* LSE, void* workspace,
                               size_t workspace_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * dsv_attn_mass -- share of each query's true attention mass that its
 * group's selected keys carry.
 * Passage: technical summary section 2.1 (critical KV are the pairs that
 * carry over 90% of the attention score), measured on the real scores
 * q_i.k_j instead of the predictor's.
 *
 * For query i: m_i = sum_{j in I_g} exp(scale q_i.k_j) / sum_{all j} exp(scale
 * q_i.k_j) = exp(LSE_sel,i - LSE_all,i), with LSE_sel from
 * dsv_sparse_attn_fwd on the index sets and LSE_all from the same call with
 * idx = NULL (dense). mass[p] = mean over the problem's S queries of m_i
 * (fp64 sum in a fixed order: the same bits on every run).
 * LSE_sel, LSE_all: DEVICE float [P][S]; mass: DEVICE float [P]; per_query
 * (optional, may be NULL): DEVICE float [P][S] of m_i. No workspace.
 * P <= 256 problems, S >= 1; DSV_ERR_INVALID_ARG otherwise.
 * ---------------------------------------------------------------------- */
dsv_status dsv_attn_mass(const float* LSE_sel, const float* LSE_all, int64_t S, int32_t P, float* mass,
                         float* per_query, void* stream);

/* ------------------------------------------------------------------------
 * dsv_predicted_mass -- share of each query's own predicted softmax mass
 * that its group's selected keys carry.
 * Passage: technical summary section 2.1 (critical KV are the pairs that
 * carry over 90% of the attention score), read per query on the low-rank
 * predictor's logits; dsv_coverage is the pooled, group-level reading.
 *
 * For query i of group g of problem p, with the predictor's logits
 * l_ij = scale q_lr,i . k_lr,j over all S keys (q_lr = Q W_lr^Q,
 * k_lr = K W_lr^K as in dsv_lowrank_topk, the score to about 2^-21
 * relative): m_i = sum_{j in I_g} softmax_j(l_ij). idx, k_per_head and
 * idx_offset are as for dsv_sparse_attn_fwd (idx == NULL or
 * idx_offset[p] < 0: every key is selected and m_i = 1).
 * mass: DEVICE float [B*H], the mean of m_i over the problem's S queries
 * (fp64 sums in a fixed order: the same bits on every run). per_query
 * (optional, may be NULL): DEVICE float [B*H][S] of m_i in token order.
 * It scores every (query, key) pair, 3 tf32 products of rank r each: a
 * diagnostic, not part of a training step. S <= 262144
 * (DSV_ERR_UNSUPPORTED otherwise).
 * ---------------------------------------------------------------------- */
size_t dsv_predicted_mass_workspace_size(dsv_shape shape, int32_t r, dsv_group group);
dsv_status dsv_predicted_mass(const void* Q, const void* K, const void* Wq_lr, const void* Wk_lr, dsv_shape shape,
                              int32_t r, dsv_group group, const int32_t* idx, const int32_t* k_per_head,
                              const int64_t* idx_offset, float scale, float* mass, float* per_query, void* workspace,
                              size_t workspace_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * dsv_sparse_attn_bwd -- query-grouped sparse attention, backward.
 * Passage: technical summary section 2.1 (stage 2 trains with sparse
 * attention over the critical KV, so gradients flow through the selected
 * pairs only; the index sets are constants of the step).
 *
 * Given O, LSE from the forward and dO: P = exp(scale q.k - LSE),
 * dP = dO v^T, Delta_i = sum_c dO_ic O_ic, dS = P (dP - Delta):
 *   dQ_i = scale sum_{j in I} dS_ij k_j
 *   dK_j = scale sum over (group, query i) pairs that selected j of dS_ij q_i
 *   dV_j = sum over the same pairs of P_ij dO_i
 * dK and dV are reduced in a fixed order: every (group, key) pair writes its
 * bf16 partial rows to a slot ordered by (key, group), and each key's slots
 * are summed in ascending group order in fp32, so the result does not depend
 * on scheduling. dQ, dK, dV are fully overwritten.
 * k_per_head, idx_offset: HOST arrays (NULL with idx NULL: every problem
 * dense). The workspace size depends on the plan: pass the same k_per_head
 * and idx_offset to dsv_sparse_attn_bwd_workspace_size (it holds the bf16
 * partials of up to 48 GiB worth of (group, key) pairs at a time, a key x group
 * selection bitmap and per-key slot offsets; a head with more
 * pairs is split over several launches with fp32 running sums). A smaller
 * workspace is accepted: the call then keeps fewer pairs in flight per launch
 * (the largest power-of-two fraction of 48 GiB that fits, down to one query
 * group per launch), which changes no result bit; below that minimum it
 * returns DSV_ERR_WORKSPACE. Sparse problems need S <= 262144
 * (DSV_ERR_UNSUPPORTED otherwise); dense problems do not.
 * ---------------------------------------------------------------------- */
size_t dsv_sparse_attn_bwd_workspace_size(dsv_shape shape, dsv_group group, const int32_t* k_per_head,
                                          const int64_t* idx_offset);
/* The smallest workspace dsv_sparse_attn_bwd accepts: the least of its plans
 * (pairs in flight per launch halving from 48 GiB down to one query group);
 * every workspace at least this large is accepted (0 on invalid arguments). */
size_t dsv_sparse_attn_bwd_min_workspace_size(dsv_shape shape, dsv_group group, const int32_t* k_per_head,
                                              const int64_t* idx_offset);
dsv_status dsv_sparse_attn_bwd(const void* Q, const void* K, const void* V, const void* O, const float* LSE,
                               const void* dO, const int32_t* idx, const int32_t* k_per_head,
                               const int64_t* idx_offset, dsv_shape shape, dsv_group group, float scale, void* dQ,
                               void* dK, void* dV, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                               void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LIBDSV_H */
