/*
 * tv.h — C ABI of libtreeverify: batched speculative-tree verification on one
 * GB300 (sm_103a).
 *
 * The library implements the data-parallel step shared by tree and block
 * speculative decoding: after a drafter (and, for Graft, a successor table)
 * proposes candidate tokens, the target model verifies all of them in one
 * forward pass and the longest path it agrees with is accepted.
 *
 * Sources (web write-ups of four 2026 preprints), cited by short name:
 *   Graft page      — 浙江大学、阿里巴巴联手破解AI推理瓶颈 (arXiv:2605.20104)
 *   BlockPilot page — 阿里AMAP团队的AI提速新招："动态换挡"让大模型推理快4.2倍
 *                     (arXiv:2606.31315)
 *   D-cut page      — D-cut: Adaptive Verification Depth Pruning for Batched
 *                     Speculative Decoding
 *   SpecOPD page    — 【论文分享】给大模型推理安上"并发预读器": 解密阿里通义新作
 *                     SpecOPD ... (arXiv:2611.02846)
 *
 * Conventions for every entry point
 *   - Returns an int status (TV_OK = 0, negative on error).  Arguments are
 *     validated on the host before anything is launched; on an error nothing
 *     is launched.  No entry point allocates memory, synchronises, or reads
 *     device memory on the host; all work is ordered on `stream`.
 *   - Array arguments are DEVICE pointers owned by the caller, unless a
 *     comment says "host".  Scalars are passed by value.
 *   - A "workspace" is caller-owned device scratch of at least the size that
 *     the matching *_workspace_size() call returns; its contents on entry do
 *     not matter.  Calls that share one workspace must not overlap on the GPU.
 *   - Flattened trees: request r owns nodes node_off[r] .. node_off[r+1]-1;
 *     parent[] holds REQUEST-LOCAL indices, parents precede children, -1 marks
 *     a root.  Prefix (KV cache) tokens of request r are pre_off[r] ..
 *     pre_off[r+1]-1.
 *   - Attention tensors are token-major, contiguous: [tokens, heads, d].
 *   - dtype is TV_F32 or TV_BF16 (bf16 = the upper 16 bits of an IEEE float).
 *   - Results are deterministic: no floating-point atomics; integer results
 *     are bit-reproducible.
 */
#ifndef TREEVERIFY_TV_H
#define TREEVERIFY_TV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* tv_stream_t;

enum tv_status {
  TV_OK = 0,
  TV_EINVAL = -1,        /* bad pointer, size or shape                         */
  TV_EUNSUPPORTED = -2,  /* valid but outside what the kernels implement       */
  TV_ECUDA = -3,         /* a CUDA launch or runtime call failed               */
  TV_EWORKSPACE = -4     /* workspace pointer NULL/misaligned or too small     */
};

enum tv_dtype { TV_F32 = 0, TV_BF16 = 1 };

/* Limits of the library. */
#define TV_MAX_NODES 1024   /* nodes per request (tree_prep, attention, acceptance) */
#define TV_MAX_TOPK 16      /* k of vocab_argmax_topk / graft tables               */

/* Human-readable name of a status code (static storage). */
const char* tv_status_str(int status);
/* Library version, major*10000 + minor*100 + patch. */
int tv_version(void);

/* --------------------------------------------------------------------------
 * tv_tree_prep — flatten the candidate tree: depth, position ids, ancestor
 * bitmask, visible prefix.
 * Graft page §2 (third gear): the hybrid tree is flattened and its tree
 * position encoding and mask rebuilt.  SpecOPD page §02 (architecture table,
 * full-attention row): the mask is the ancestor relation — a node sees its
 * own ancestor path and the shared trunk, never siblings or later trunk tokens.
 *
 *   parent      int32 [n]   request-local parent, -1 = root (n = node_off[B])
 *   node_off    int32 [B+1]
 *   prefix_len  int32 [B]   prefix tokens of each request
 *   vis_prefix  int32 [n]   visible prefix per node, or NULL (= whole prefix).
 *                           Values are clamped to [0, prefix_len[r]].
 *   max_nodes   upper bound of node_off[r+1]-node_off[r]   (<= TV_MAX_NODES)
 *   anc_words   u64 words per ancestor row, >= ceil(max_nodes/64)
 * Outputs: depth int32 [n] (root 0), pos int32 [n] = vis + depth,
 *   anc uint64 [n, anc_words] (bit j%64 of word j/64 set iff node j is the
 *   node itself or one of its ancestors), vis_out int32 [n].
 * A parent index outside [-1, i) is reported by writing 1 to *err (device
 * int32, may be NULL); the node is then treated as a root.
 * -------------------------------------------------------------------------- */
int tv_tree_prep(const int32_t* parent, const int32_t* node_off, const int32_t* prefix_len,
                 const int32_t* vis_prefix, int B, int max_nodes, int anc_words,
                 int32_t* depth, int32_t* pos, uint64_t* anc, int32_t* vis_out,
                 int32_t* err, tv_stream_t stream);

/* --------------------------------------------------------------------------
 * tree_verify_attn — tree-masked grouped-query attention of the candidate
 * nodes over a shared KV prefix.
 * Graft page §2 (third gear) and SpecOPD page §02 (proposal-tree stage and
 * the tree attention mask): all candidates are verified in one forward pass
 * sharing the prefix/trunk KV; node i attends to prefix[0, vis_i) plus the
 * nodes set in its ancestor row (its root path, itself included):
 *   o[i,h] = sum_j softmax_j(scale * q[i,h].k[j,h/g]) v[j,h/g],  g = Hq/Hkv.
 *
 *   q        [n, Hq, d]       dtype
 *   k_pre/v_pre [P_total, Hkv, d] dtype; request r's prefix at pre_off[r]..
 *   pre_off  int32 [B+1]      several requests may point at the same prefix
 *   k_tree/v_tree [n, Hkv, d] the candidate nodes' own key/value rows
 *   node_off int32 [B+1]
 *   node_cnt int32 [B] or NULL: only the first node_cnt[r] nodes of request r
 *            are computed (D-cut packing); other rows of out/lse are untouched
 *   anc      uint64 [n, anc_words] from tv_tree_prep
 *   vis_prefix int32 [n] or NULL (= whole prefix); clamped to the prefix
 *   max_nodes, max_prefix  upper bounds over requests (launch geometry)
 *   total_nodes   rows of q / k_tree / v_tree (= node_off[B]; the tensor size)
 *   total_prefix  rows of k_pre / v_pre (>= max_prefix)
 *   d ∈ {64, 128}; Hq % Hkv == 0; scale > 0 is applied to q.k
 * bf16 with d = 128 (and Hq/Hkv dividing 128) runs on the tensor cores
 * (tcgen05 MMA, TMA-loaded K/V tiles, TMEM accumulators); other shapes on a
 * SIMT kernel with fp32 arithmetic.
 * Outputs: out [n, Hq, d] dtype; lse float [n, Hq] (natural log of the sum of
 *   exp(scale*q.k) over visible keys) or NULL.
 * Workspace: tree_verify_attn_workspace_size(...) bytes, 256-byte aligned.
 *   Its first int32 is a status word, set to 0 by the call and to a nonzero
 *   code if a pipeline wait inside the tensor-core kernel ran out (about 2 s;
 *   the outputs are then invalid).  The rest holds the key-split partials.
 * -------------------------------------------------------------------------- */
size_t tree_verify_attn_workspace_size(int B, int max_nodes, int max_prefix, int Hq, int Hkv,
                                       int d, int dtype);
int tree_verify_attn(const void* q, const void* k_pre, const void* v_pre, const int32_t* pre_off,
                     const void* k_tree, const void* v_tree, const int32_t* node_off,
                     const int32_t* node_cnt, const uint64_t* anc, int anc_words,
                     const int32_t* vis_prefix, int B, int max_nodes, int max_prefix,
                     long long total_nodes, long long total_prefix, int Hq, int Hkv, int d,
                     int dtype, float scale, void* out, float* lse, void* ws, size_t ws_bytes,
                     tv_stream_t stream);

/* --------------------------------------------------------------------------
 * vocab_argmax_topk — per-row reductions over next-token logits.
 * Graft page §2 (second and third gears): table rows hold the top-k next
 * tokens by probability and are refreshed from every verified position;
 * greedy verification accepts a token iff it is the target's choice (argmax).
 * §5: width about 8.
 *   argmax   = smallest index attaining the row maximum
 *   top-k    = first k of (value desc, index asc)
 *   row_max  = maximum;  row_lse = max + ln(sum exp(x - max))
 *
 *   logits  [*, ld] dtype, V valid entries per row, in device memory or in
 *           page-locked host memory the device addresses directly (e.g.
 *           cudaHostAlloc; with unified addressing the host pointer is the
 *           device pointer).  Host-resident rows are read in place over the
 *           host link, so with row_idx only the selected rows cross it; the
 *           call then uses a quarter of the SMs.
 *   rows    rows to reduce; row t reads logits row src(t) and writes outputs
 *           at index src(t), where src(t) = row_idx[t] (int32, device) or t
 *   k       0..TV_MAX_TOPK (topk_* may be NULL when k == 0)
 * Outputs (each may be NULL except argmax): argmax int32, topk_idx int32
 *   [*, k], topk_val float [*, k] (the logit values), row_max float,
 *   row_lse float.
 * Failure: the streaming kernels wait on shared-memory barriers with a bound
 *   of about 2 s.  If a wait runs out (only possible when the GPU stalls
 *   for seconds), every reduced row is written as argmax -1, top-k indices
 *   -1, and NaN for the top-k values, row_max and row_lse, and the first
 *   int32 of the workspace is nonzero.  The host return value cannot report
 *   it (the work is asynchronous).
 * Workspace: vocab_argmax_topk_workspace_size(rows, V, k) bytes, 16-byte
 *   aligned; contents need not persist between calls.
 * -------------------------------------------------------------------------- */
size_t vocab_argmax_topk_workspace_size(int rows, int V, int k);
int vocab_argmax_topk(const void* logits, int dtype, int rows, int V, int64_t ld,
                      const int32_t* row_idx, int k, int32_t* argmax, int32_t* topk_idx,
                      float* topk_val, float* row_max, float* row_lse, void* ws, size_t ws_bytes,
                      tv_stream_t stream);

/* --------------------------------------------------------------------------
 * vocab_argmax_topk_noalloc — vocab_argmax_topk for callers that cannot
 * allocate device memory.  (No counterpart in the source pages: this is an
 * interface convenience, not part of the method.)
 *
 * Some callers may not call cudaMalloc at all: runtimes with a fixed device
 * memory budget planned at start-up, allocators that forbid allocation on the
 * serving hot path (cudaMalloc can synchronise the device and can fail under
 * memory pressure), and code that must not change allocator state.  This
 * entry point needs no workspace: its scratch is a file-scope device array of
 * TV_NOALLOC_SCRATCH_BYTES (32 MiB), which every GPU that loads the library
 * holds until the process exits.  Arguments and outputs are those of
 * vocab_argmax_topk; the caller still provides the inputs and outputs.
 *   - Sizes whose scratch need (vocab_argmax_topk_workspace_size) exceeds
 *     TV_NOALLOC_SCRATCH_BYTES are rejected with TV_EWORKSPACE (for V = 151936:
 *     up to 24528 rows with k <= 8, 12985 with k <= 16).
 *   - The first call on a device looks up the array's device address (one
 *     runtime query, no allocation); make that first call before any stream
 *     capture on that device.
 *   - All calls share the one array and it keeps the last call's contents.
 *     Nothing in it needs to start at zero: each call on the streaming path
 *     resets the small header it uses with a one-thread kernel on the given
 *     stream, and the fallback path (rows that are not 16-byte multiples)
 *     overwrites every chunk record it later reads.  Calls that overlap on
 *     the GPU (different streams without ordering) race on it: order them.
 *   - An expired wait gives the same failure outputs as vocab_argmax_topk
 *     (argmax -1, NaN values); the caller cannot read the status word here.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * -------------------------------------------------------------------------- */
#define TV_NOALLOC_SCRATCH_BYTES (32u << 20)
int vocab_argmax_topk_noalloc(const void* logits, int dtype, int rows, int V, int64_t ld,
                              const int32_t* row_idx, int k, int32_t* argmax, int32_t* topk_idx,
                              float* topk_val, float* row_max, float* row_lse, tv_stream_t stream);

/* --------------------------------------------------------------------------
 * tree_tv_alpha — alpha = 1 - TV(p, q) = sum_v min(p_v, q_v) per row, its
 * running product along each branch, and the target's softmax mass of a
 * given token.
 * SpecOPD page §03: under exact rejection sampling the acceptance probability
 * of a draft token is the overlap of the target and draft distributions; the
 * E2E-TV objective multiplies these along a branch.  Graft page §3: coverage
 * gain is target probability mass.
 *
 *   p_logits, q_logits [rows, ld] dtype (target, draft), V entries per row
 *   branch_off int32 [nb+1] or NULL: alpha_prefix[r] = prod of alpha over the
 *              rows of r's branch up to r (rows outside every branch: 1)
 *   mass_tok   int32 [rows] or NULL: p_mass[r] = softmax(p)[mass_tok[r]]
 *              (0 when the token is outside [0, V))
 * Outputs: alpha float [rows]; alpha_prefix float [rows] (NULL allowed, needs
 *   branch_off); p_mass float [rows] (NULL allowed, needs mass_tok).
 * -------------------------------------------------------------------------- */
size_t tree_tv_alpha_workspace_size(int rows, int V);
int tree_tv_alpha(const void* p_logits, const void* q_logits, int dtype, int rows, int V,
                  int64_t ld, const int32_t* branch_off, int nb, const int32_t* mass_tok,
                  float* alpha, float* alpha_prefix, float* p_mass, void* ws, size_t ws_bytes,
                  tv_stream_t stream);

/* --------------------------------------------------------------------------
 * accept_longest_path — greedy (temperature 0) acceptance.
 * Graft page §2 (third gear): draft and retrieved nodes face the same rule;
 * BlockPilot page introduction / SpecOPD page §01: accept up to the first
 * disagreement with the target and truncate there; SpecOPD page §03 worked
 * example (acceptance lengths 0 and 3).
 *   acc(root) = valid(root);  acc(i) = acc(parent) && tok[i] == argmax[parent] && valid(i)
 *   best = deepest accepted node (lowest index on ties), accept_len = depth(best),
 *   path = root..best (request-local, -1 padded), bonus = argmax[best].
 *   path_acc[i] = depth of the deepest accepted node on root..i (-1 if none):
 *   the acceptance length had the draft been the path to i (read at a leaf,
 *   this is the acceptance of that branch; used for block-size sweeps).
 *
 *   parent, tok, argmax int32 [n]; valid uint8 [n] or NULL (all valid)
 *   max_depth  path has max_depth+1 columns; deeper paths are truncated
 * Outputs: accept_len, best_node, bonus int32 [B] (-1 when the root is not
 *   valid); path int32 [B, max_depth+1]; path_acc int32 [n] or NULL.
 * -------------------------------------------------------------------------- */
int accept_longest_path(const int32_t* parent, const int32_t* tok, const int32_t* argmax,
                        const uint8_t* valid, const int32_t* node_off, int B, int max_nodes,
                        int max_depth, int32_t* accept_len, int32_t* best_node, int32_t* path,
                        int32_t* bonus, int32_t* path_acc, tv_stream_t stream);

/* --------------------------------------------------------------------------
 * accept_rejection_sampling — lossless temperature-1 verification.
 * SpecOPD page §03: under exact rejection sampling the acceptance
 * probability of a draft token is the draft/target overlap; D-cut page §4
 * and SpecOPD page §04 report temperature-1 results but give no tree
 * procedure.  Reading (the standard multi-candidate scheme): from the root,
 * the children of the current node are tried in index order; child c with
 * token x is accepted iff u_node[c] < min(1, p'(x) / q(x)), p' = softmax of
 * the target logits at the current node, q = softmax of the draft logits
 * there; after each rejection p' becomes max(0, p' - q) renormalised; with
 * no child accepted the bonus token is the smallest j with
 * sum_{v <= j} p'(v) > u_final (inverse CDF in token order).
 *   parent, tok int32 [n] (request-local parents, parents before children)
 *   p_logits, q_logits [n, ld] dtype: target and draft logits at each node
 *   u_node float [n] (u of the test that accepts or rejects node i),
 *   u_final float [B]: uniforms in [0, 1) supplied by the caller
 *   ws accept_rejection_sampling_workspace_size(B, V) bytes (fp32 residual
 *   rows), 16-byte aligned
 * Outputs: accept_len, best_node, bonus int32 [B]; path int32
 *   [B, max_depth+1] (-1 padded; node indices request-local).
 * Arithmetic: fp32 throughout (exponentials, sums, the cross-CTA combines of
 * the 8-CTA cluster that serves each request); a decision whose uniform lies
 * within ~1e-5 of its threshold may differ from an exact-arithmetic
 * evaluation.
 * -------------------------------------------------------------------------- */
size_t accept_rejection_sampling_workspace_size(int B, int V);
int accept_rejection_sampling(const int32_t* parent, const int32_t* tok, const void* p_logits,
                              const void* q_logits, int dtype, int V, int64_t ld, const int32_t* node_off,
                              int B, int max_nodes, int max_depth, const float* u_node, const float* u_final,
                              int32_t* accept_len, int32_t* best_node, int32_t* path, int32_t* bonus, void* ws,
                              size_t ws_bytes, tv_stream_t stream);

/* --------------------------------------------------------------------------
 * graft_adj_update — online update of Graft's V x k successor table.
 * Graft page §2 (second/third gear) and §6: after verification, every
 * verified position, accepted or rejected, rewrites the row of its token with
 * the target's top-k next tokens.  Several nodes with the same token: the
 * last in index order wins; rows are overwritten, never merged.  The result
 * does not depend on scheduling: up to TV_ADJ_SCAN_MAX nodes an ordered scan
 * per table slice picks each row's last node; larger batches (a whole-table
 * refresh) record each token's last node with an integer maximum in the
 * workspace, then copy once per row.
 *
 *   adj       int32 [V, k], updated in place
 *   tok       int32 [n] tokens of the verified nodes
 *   topk_idx  int32 [n, topk_ld], first k used (topk_ld >= k)
 *   valid     uint8 [n] or NULL: nodes with valid == 0 are skipped
 *   n_bad     int32 (device, may be NULL): receives the number of valid nodes
 *             whose token lies outside [0, V) (those are skipped)
 *   ws        graft_adj_update_workspace_size(V, n) bytes (0 when n <=
 *             TV_ADJ_SCAN_MAX: ws may then be NULL), 16-byte aligned
 * -------------------------------------------------------------------------- */
#define TV_ADJ_SCAN_MAX 4096
size_t graft_adj_update_workspace_size(int V, int n);
int graft_adj_update(int32_t* adj, int V, int k, const int32_t* tok, const int32_t* topk_idx,
                     int topk_ld, const uint8_t* valid, int n, int32_t* n_bad, void* ws,
                     size_t ws_bytes, tv_stream_t stream);

/* --------------------------------------------------------------------------
 * graft_retrieve — expand retrieval candidates from the successor table by a
 * stage template.
 * Graft page §2 (second gear): rooted at the current token, follow the
 * stage-adaptive template through the table (one row/column lookup per
 * node); the number of retrieval slots depends on the pruning stage
 * (52/36/20/0 of a 60-slot budget).
 *   slot s of request b (template of stage[b], slots tmpl_off[st]..):
 *     rtok[b,s] = adj[ src, trank[s] ],  src = root_tok[b] if tparent[s] < 0
 *                                              else rtok[b, tparent[s]]
 *   tparent is slot-local (-1 = the root token) and must be < s.
 *
 *   adj int32 [V, k]; root_tok, stage int32 [B]; tparent, trank int32 [tmpl_off[n_stage]]
 *   tmpl_off int32 [n_stage+1] (device)
 * Outputs: rtok, rparent int32 [B, max_slots] (-1 padded), nslots int32 [B].
 * A template entry or table value out of range makes that slot and its
 * descendants -1 and writes 1 to *err (device int32, may be NULL).
 * -------------------------------------------------------------------------- */
int graft_retrieve(const int32_t* adj, int V, int k, const int32_t* root_tok, const int32_t* stage,
                   int B, const int32_t* tparent, const int32_t* trank, const int32_t* tmpl_off,
                   int n_stage, int max_slots, int32_t* rtok, int32_t* rparent, int32_t* nslots,
                   int32_t* err, tv_stream_t stream);

/* --------------------------------------------------------------------------
 * dcut_select — D-cut prefix-product scores and batch-global budget selection.
 * D-cut page, technical summary §2: score each position by the prefix product
 * of draft confidences (the probability the block survives to that depth),
 * rank all positions of the batch globally, keep the top K (a contiguous
 * prefix per request) and pack them; rho ∈ {0.25, 0.5, 0.75, 1.0}; §1: a step
 * verifies B x (D+1) positions.
 *   s[r,0] = 1, s[r,j] = fp32(s[r,j-1] * conf[r,j-1]) sequentially
 *   K(rho) = floor(rho * B*(D+1) + 0.5)   (computed in double)
 *   keep = first K in the order (s desc, r asc, j asc)
 *
 *   conf float [B, D] in [0, 1]; rho float [n_rho] (host array) in [0, 1]
 *   B*(D+1) <= 8192
 * Outputs: score float [B, D+1]; keep uint8 [n_rho, B, D+1];
 *   keep_len int32 [n_rho, B]; pack_off int32 [n_rho, B+1] or NULL;
 *   pack_idx int32 [n_rho, B*(D+1)] or NULL (flat r*(D+1)+j of kept positions
 *   in order, -1 padded).
 * -------------------------------------------------------------------------- */
size_t dcut_select_workspace_size(int B, int D, int n_rho);
int dcut_select(const float* conf, int B, int D, const float* rho, int n_rho, float* score,
                uint8_t* keep, int32_t* keep_len, int32_t* pack_off, int32_t* pack_idx, void* ws,
                size_t ws_bytes, tv_stream_t stream);

/* --------------------------------------------------------------------------
 * dcut_choose_rho — expected tokens per budget and the run-time budget choice.
 * D-cut page, technical summary §2 (runtime adaptive depth selection, budget
 * selection): the expected gain of a budget, estimated from the drafter's
 * confidences, over the hardware-profiled cost of a step at that budget;
 * rho* maximises it.  Reading: the expected gain is the sum of the kept
 * positions' survival probabilities (a kept root counts 1: the target's own
 * next token); the cost table is an input (its profiling is not done here).
 *   score float [B*(D+1)] and keep uint8 [n_rho, B*(D+1)] from dcut_select
 *   cost  host float [n_rho] > 0: profiled step cost of each budget
 * Outputs: exp_tok double [n_rho] (NULL allowed): the sum in 2^-50 fixed
 *   point, within B*(D+1) * 2^-51 of the exact sum; rho_star int32 (device,
 *   NULL allowed): the budget index maximising exp_tok / cost, lowest on ties.
 * -------------------------------------------------------------------------- */
int dcut_choose_rho(const float* score, const uint8_t* keep, int B, int D, int n_rho, const float* cost,
                    double* exp_tok, int32_t* rho_star, tv_stream_t stream);

/* --------------------------------------------------------------------------
 * graft_stage_decide — Graft's calibrated pruning checkpoints.
 * Graft page §2 (first gear): the best path's cumulative confidence is
 * checked at draft layers 0, 1 and 5 only; below the calibrated threshold
 * the tree stops there and the freed slots go to retrieval (stages 8/52,
 * 24/36, 40/20; no pruning 60/0).  Readings: a node's draft layer is its
 * depth - 1 (the root is the current token); its cumulative confidence is
 * the fp32 product of conf along its path, root excluded, in root-to-node
 * order; a layer the draft does not reach counts as 0.
 *   parent int32 [n] request-local (-1 = root), conf float [n] (root unused)
 *   node_off int32 [B+1]; tau host float [3] thresholds of layers 0, 1, 5
 * Outputs: stage int32 [B]: first checkpoint whose best value is below its
 *   threshold (0, 1, 2), else 3; best float [B, 3] or NULL; err (device
 *   int32, may be NULL) <- 1 for a malformed parent chain (node skipped).
 * -------------------------------------------------------------------------- */
int graft_stage_decide(const int32_t* parent, const float* conf, const int32_t* node_off, int B,
                       int max_nodes, const float* tau, int32_t* stage, float* best, int32_t* err,
                       tv_stream_t stream);

/* --------------------------------------------------------------------------
 * graft_replace — fixed-slot tree: replace low-confidence draft nodes by
 * retrieval nodes.
 * Graft page §4 (batched serving: the per-request slot count stays fixed,
 * low-confidence nodes of a static tree become retrieval nodes) with
 * attach = 0; §7 (Graft-TAIL: keep a block draft's confident prefix, replace
 * its tail by retrieval) with attach = 1 on a chain.
 * Readings: a draft node is kept when its cumulative confidence (as in
 * graft_stage_decide) is >= tau and its parent is kept; the S - kept freed
 * slots take the first slots of a best-first retrieval template, rooted at
 * the root token (attach 0) or at the deepest kept node (attach 1; ties:
 * larger cumulative confidence, then lower index).
 *   Request r's tree is nodes r*S .. r*S+S-1, node 0 of each its root:
 *   parent int32 [B*S] request-local, tok int32 [B*S], conf float [B*S]
 *   adj int32 [V, k]; tparent, trank int32 [n_tmpl] best-first template
 *   (tparent slot-local, -1 = the anchor, < the slot's own index)
 * Outputs: tok_out, parent_out int32 [B*S] (kept nodes in order, then the
 *   retrieval slots; -1 padded when the template is shorter), n_kept int32
 *   [B]; err (device int32, may be NULL) <- 1 for a bad template or table
 *   entry (that slot is -1) or a malformed parent chain.
 * -------------------------------------------------------------------------- */
int graft_replace(const int32_t* parent, const int32_t* tok, const float* conf, int B, int S, float tau,
                  int attach, const int32_t* adj, int V, int k, const int32_t* tparent, const int32_t* trank,
                  int n_tmpl, int32_t* tok_out, int32_t* parent_out, int32_t* n_kept, int32_t* err,
                  tv_stream_t stream);

/* --------------------------------------------------------------------------
 * blockpilot_mlp — BlockPilot's block-size predictor, run once per request.
 * BlockPilot page §3: the full next-token distribution at the last prefill
 * position feeds a two-layer MLP that picks the block size; §7: raw
 * probabilities are the input; §4: hidden 2048; §2: candidates B-3..B+3.
 *   x = exp(last_logits - row_lse)  (softmax, using row_lse from vocab_argmax_topk)
 *   h = ReLU(x W1 + b1);  z = h W2 + b2;  choice = argmax z (lowest index on ties)
 *   bsize = block - (C-1)/2 + choice
 *
 *   last_logits [B, ld] bf16; row_lse float [B]; W1 bf16 [V, H]; W2 bf16 [H, C];
 *   b1 float [H] or NULL; b2 float [C] or NULL.  H % 256 == 0, C <= 32, B <= 16.
 *   Up to 8 requests with H % 128 == 0 run layer 1 on the tensor cores: x is
 *   split into bf16 x_hi + x_lo (about 16 mantissa bits) against bf16 W1,
 *   fp32 accumulation; otherwise a CUDA-core GEMV in fp32.
 * Outputs: z float [B, C], choice int32 [B], bsize int32 [B].
 * -------------------------------------------------------------------------- */
size_t blockpilot_mlp_workspace_size(int B, int V, int H);
int blockpilot_mlp(const void* last_logits, int64_t ld, const float* row_lse, const void* W1,
                   const float* b1, const void* W2, const float* b2, int B, int V, int H, int C,
                   int block, float* z, int32_t* choice, int32_t* bsize, void* ws,
                   size_t ws_bytes, tv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TREEVERIFY_TV_H */
