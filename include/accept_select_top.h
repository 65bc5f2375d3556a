/*
 * accept_select_top.h -- C ABI of the GB300 (sm_103a) verify/accept step of
 * EAGLE-style speculative decoding.
 *
 * One verify step is, in order:
 *   spec_select_topk  x num_steps   draft-tree growth (select_top_k_tokens)
 *   spec_build_tree                 organize_draft_results + build_tree
 *   spec_verify_attention           tree-masked attention of the verify queries
 *   spec_verify_greedy | spec_verify_sampling   accept
 *   spec_commit_kv                  move accepted KV, release the rest
 *
 * Sources (web pages), cited below as [KEY section]:
 *   [SGL-XI]  "SGLang 源码完全拆解(十一):投机解码——草稿生成、批量验证与 token 接受如何接进同一条前向"
 *   [ACCEPT]  "投机解码 Accept从 Verify 行到最终输出路径"
 *   [EVOL]    "SGLang 设计演进投机解码、PD 分离与大规模 EP（2025 上半年）", chapter "EAGLE 投机解码四部曲"
 *   [INTERN]  "Speculative Decoding" (SGLang internals, part 3, execution model)
 *   [EAGLE2]  "把投机采样讲透：以 SGLang 中的 EAGLE-2 为例"
 *
 * Conventions for every call:
 *   - Every array pointer is a DEVICE pointer allocated and owned by the caller;
 *     the library keeps no pointer after a call returns and allocates nothing.
 *   - `stream` is a cudaStream_t passed as void*; every call is asynchronous on
 *     it and never synchronises the host (except spec_last_error).
 *   - `ws` / `ws_bytes` is caller-provided scratch memory sized by
 *     spec_workspace_size() and zero-filled once (spec_workspace_init) before its
 *     first use.  Every call leaves it zero again apart from the error word, so
 *     one workspace serves any sequence of calls on one stream.  Calls that may
 *     run concurrently (different streams) need separate workspaces.  Every
 *     kernel is launched with programmatic dependent launch: by default it
 *     waits for the kernel before it on the stream -- whichever library or
 *     framework launched that kernel -- before it reads any input, and only
 *     then lets the next kernel start, so inputs written by any earlier work
 *     on the stream are safe to read.  spec_workspace_set_overlap lets a
 *     caller allow two calls to start reading earlier (see there).
 *   - Return codes: SPEC_OK, SPEC_ERR_ARG (null pointer, bad size or shape, a
 *     limit below exceeded), SPEC_ERR_WORKSPACE (ws too small or misaligned),
 *     SPEC_ERR_LAUNCH (the CUDA launch failed; cudaGetLastError is consumed),
 *     SPEC_ERR_UNSUPPORTED (dtype or head size not built).
 *   - b == 0 (an idle batch) is a no-op that returns SPEC_OK [SGL-XI eagle_sample].
 *   - Indices read from device arrays are bounds-checked on the device; a bad
 *     one sets a bit in the workspace error word and the access is skipped (no
 *     trap).  spec_last_error() reads and clears that word.
 *   - Tree arrays use -1 for "none"; a verify row is the flattened index
 *     b*n + i of request b's tree node i [ACCEPT section 3].
 *   - Limits: 1 <= k <= 16, k <= V, 1 <= n <= 64, n - 1 <= k + (S-1)*k*k,
 *     S >= 1, head_dim D in {64, 128}, Hq a multiple of Hkv; spec_select_topk
 *     and spec_verify_sampling take V <= 262144 (larger returns
 *     SPEC_ERR_UNSUPPORTED).
 *   - Ties in every top-k / argmax go to the lowest index.
 */
#ifndef ACCEPT_SELECT_TOP_H
#define ACCEPT_SELECT_TOP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_OK 0
#define SPEC_ERR_ARG (-1)
#define SPEC_ERR_WORKSPACE (-2)
#define SPEC_ERR_LAUNCH (-3)
#define SPEC_ERR_UNSUPPORTED (-4)

/* logits dtypes */
#define SPEC_F32 0
#define SPEC_BF16 1

/* bits of the device error word */
#define SPEC_DEV_INDEX 1u      /* an index read from an input array was out of range */
#define SPEC_DEV_INVARIANT 2u  /* a selected node's parent was not selected (build_tree) */
#define SPEC_DEV_LENGTH 4u     /* a length (seq_len, accept_len) outside its valid range */
#define SPEC_DEV_TIMEOUT 8u    /* a bounded device-side wait ran out; the kernel stopped cleanly */

/* operation ids for spec_workspace_size */
#define SPEC_OP_SELECT_TOPK 0
#define SPEC_OP_BUILD_TREE 1
#define SPEC_OP_VERIFY_ATTENTION 2
#define SPEC_OP_VERIFY_GREEDY 3
#define SPEC_OP_VERIFY_SAMPLING 4
#define SPEC_OP_COMMIT_KV 5
#define SPEC_OP_VERIFY_TARGET_ONLY 6
#define SPEC_OP_LAST SPEC_OP_VERIFY_TARGET_ONLY

/* Bytes of workspace the operation needs for these sizes (b requests, n tree
 * nodes, k = topk, V vocabulary, Hq query heads, Hkv kv heads, max_seq_len an
 * upper bound on seq_lens).  Sizes an operation does not use are ignored.
 * Returns 0 for an unknown op or invalid sizes. */
size_t spec_workspace_size(int op, int b, int n, int k, int V, int Hq, int Hkv, int max_seq_len);

/* Zero-fills a workspace (cudaMemsetAsync on `stream`) and forgets what the
 * library recorded for this address (overlap back to off). */
int spec_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Overlap with the call before (off by default; enable = 0 or 1).  The pages
 * have no counterpart: it is a scheduling permission.  With overlap on, two
 * calls may read their main input before the kernel ahead of them on the
 * stream has finished (programmatic dependent launch):
 *   - spec_select_topk reads draft_logits early when the last call enqueued
 *     on this workspace (same batch size) was spec_select_topk or
 *     spec_commit_kv;
 *   - spec_verify_greedy reads logits early when the last call enqueued on
 *     this workspace (same batch size) was spec_verify_attention.
 * By enabling it the caller asserts that, for every call on this workspace,
 * that input was complete before the previous library call on the stream
 * was enqueued: no kernel that writes it sits between the two calls on the
 * stream (in an EAGLE loop the draft forward runs between two selects and the
 * target's MLP and LM head between the attention and the accept, so overlap
 * must stay off there).  The library records, per workspace address and
 * under a mutex, which call was last enqueued on it; that record is the only
 * host state of the library.  Returns SPEC_ERR_WORKSPACE for a NULL ws and
 * SPEC_ERR_ARG for another enable value. */
int spec_workspace_set_overlap(void* ws, int enable);

/* Synchronises `stream`, returns the device error word (SPEC_DEV_* bits, 0 if
 * clean) and clears it; a negative SPEC_ERR_* on failure. */
int spec_last_error(void* ws, void* stream);

/* Number of streaming multiprocessors of the current device (0 on failure). */
int spec_device_sm_count(void);

/* ---------------------------------------------------------------------------
 * spec_select_topk -- one step of select_top_k_tokens, with the draft
 * distribution's softmax and top-k fused in.
 * [SGL-XI organize_draft_results] (_select_top_k_tokens_first / _later) and
 * [SGL-XI 草稿主循环: draft()].
 *
 * draft_logits: [b * rows, V] (rows = 1 at step 0, k after), dtype SPEC_F32 or
 *   SPEC_BF16, row-major.  Per row: p = softmax(logits / temperature)
 *   (temperature > 0), topk_p = the k largest p in descending order, with
 *   their token ids.
 * step 0:  score block [b, k] = topk_p; token block [b, k] = ids;
 *          parent block [b, k+1] = -1, 0, .., k-1; scores_out = topk_p;
 *          next_input_ids = ids.
 * step i>0: scores_in [b, k] are the path scores of the current rows;
 *          expand[r*k+j] = scores_in[r] * topk_p[r][j] (one fp32 multiply);
 *          score block [b, k*k] = expand; token block [b, k*k] = ids;
 *          the k best expand values (value desc, flat index asc) sel[0..k-1]
 *          give parent block [b, k] = sel + k*k*(i-1) + k, scores_out [b, k]
 *          = expand[sel], next_input_ids [b*k] = ids[sel].
 * score_blk / token_blk rows are `score_ld` elements apart and parent_blk rows
 * `parent_ld` apart, so the blocks can be written straight into the
 * concatenated score / token space and parent list that spec_build_tree reads
 * (score_ld = k + (S-1)*k*k, parent_ld = 1 + (S-1)*k).  parent_blk may be NULL
 * (the last step's parent block is not part of the parent list).  topk_p_out
 * [b*rows, k] is optional (NULL).
 * Consecutive selects on one workspace alternate between two halves of the
 * select's workspace area.  With overlap on (spec_workspace_set_overlap) and
 * the last call on the workspace a select or a KV commit, the pass over
 * draft_logits starts before that call has finished; only the step's outputs
 * wait for it.  With overlap off (the default) the kernel waits first.
 * ------------------------------------------------------------------------- */
int spec_select_topk(int step, int b, int k, int V, int dtype,
                     const void* draft_logits, float temperature,
                     const float* scores_in,
                     float* score_blk, int32_t* token_blk, int score_ld,
                     int32_t* parent_blk, int parent_ld,
                     float* scores_out, int32_t* next_input_ids,
                     float* topk_p_out,
                     void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * spec_build_tree -- organize_draft_results followed by build_tree.
 * [SGL-XI organize_draft_results], [SGL-XI build_tree_kernel_efficient],
 * [ACCEPT section 2], [EAGLE2 sections 4.3, 5.3].
 *
 * score_space, token_space: [b, C], C = k + (S-1)*k*k; parent_space: [b, P],
 *   P = 1 + (S-1)*k; bonus, seq_lens: [b].
 * The n-1 best scores (value desc, index asc), re-sorted by position, become
 * nodes 1..n-1; node 0 is the bonus token.  The parent of the node at position
 * p is the node at position parent_space[p / k] (-1 = the root).
 * Outputs, [b*n] each: draft_tokens; positions = seq_len + depth;
 *   retrieve_index = b*n + i; next_token = first (smallest) child;
 *   next_sibling = next larger child of the same parent; mask_bits (uint64,
 *   bit j of row b*n+i set iff node j is an ancestor of node i or i itself).
 * A selected node whose parent is not selected sets SPEC_DEV_INVARIANT and is
 * attached to the root.
 * ------------------------------------------------------------------------- */
int spec_build_tree(int b, int k, int S, int n,
                    const float* score_space, const int32_t* token_space,
                    const int32_t* parent_space,
                    const int32_t* bonus, const int32_t* seq_lens,
                    int32_t* draft_tokens, int32_t* positions,
                    int32_t* retrieve_index, int32_t* next_token,
                    int32_t* next_sibling, uint64_t* mask_bits,
                    void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * spec_verify_attention -- tree-masked attention of the verify queries.
 * [EAGLE2 sections 4.2, 4.3], [SGL-XI 三种 mask 形态 (QLEN_ONLY)].
 *
 * q: [b*n, Hq, D] bf16; k_pool, v_pool: [num_slots, Hkv, D] bf16 (post-RoPE);
 * req_to_token: [req_rows, row_w] int32 slots; req_pool_idx, seq_lens: [b];
 * verify_loc: [b*n] slots of the tree nodes; mask_bits: [b*n] from
 * spec_build_tree.  For row b*n+i and q head h (kv head g = h / (Hq/Hkv)):
 *   keys = prefix positions 0..seq_len[b]-1 (all visible), then tree nodes j
 *   with mask bit (i, j) set;  out = softmax(scale * q.K^T) V.
 * out: [b*n, Hq, D] bf16; lse: [b*n, Hq] fp32 natural-log sum-exp of the
 * scaled scores (optional, NULL).  max_seq_len bounds every seq_len (a larger
 * one sets SPEC_DEV_LENGTH and is clamped).  page_size is the KV page size (1
 * or 16); slots of one page are consecutive.  One launch: the key lists are
 * spread evenly over one CTA per SM, and a (request, kv head) split between
 * CTAs is merged by the CTA that finishes it last.  The workspace holds the
 * merge slots (about 26 MB, independent of the sizes).
 * ------------------------------------------------------------------------- */
int spec_verify_attention(int b, int n, int Hq, int Hkv, int D, int page_size,
                          const void* q, const void* k_pool, const void* v_pool,
                          int64_t num_slots,
                          const int32_t* req_to_token, int req_rows, int row_w,
                          const int32_t* req_pool_idx, const int32_t* seq_lens,
                          int max_seq_len,
                          const int32_t* verify_loc, const uint64_t* mask_bits,
                          float scale, void* out, float* lse,
                          void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * spec_verify_greedy -- greedy accept.
 * [SGL-XI eagle_sample (路径一:贪心验证)], [ACCEPT section 3], [EAGLE2 5.3].
 *
 * logits: [b*n, V] (SPEC_F32 or SPEC_BF16).  target_predict = per-row argmax.
 * Walk per request: cur = node 0, accept_index[b,0] = row(0); up to S times,
 * the first child c of cur in sibling order with draft_tokens[b*n+c] ==
 * target_predict[b*n+cur] is accepted: predict[row(cur)] = its token,
 * accept_index[b,d] = row(c), cur = c; stop when no child matches.  Then
 * predict[row(cur)] = target_predict[b*n+cur].  row(i) = retrieve_index[b*n+i].
 * Outputs: predict [b*n] (0 on rows not on the path), accept_index [b, S+1]
 * (-1 padded), accept_lens [b] = accepted drafts + 1; optional (NULL):
 * accepted_tokens [b, S+1] = predict[accept_index] (-1 padded), next_root [b]
 * = the last accepted token.
 * Overlap: with overlap on (spec_workspace_set_overlap) and the last call
 * enqueued on the workspace spec_verify_attention, the argmax pass over
 * logits starts before that call has finished; the walk and the outputs wait
 * for it.  With overlap off (the default) the kernel waits first.  The
 * workspace keeps the attention's merge area untouched for this, so
 * spec_workspace_size(SPEC_OP_VERIFY_GREEDY, ...) includes it (about 26 MB).
 * ------------------------------------------------------------------------- */
int spec_verify_greedy(int b, int n, int S, int V, int dtype, const void* logits,
                       const int32_t* draft_tokens, const int32_t* retrieve_index,
                       const int32_t* next_token, const int32_t* next_sibling,
                       int32_t* predict, int32_t* accept_index,
                       int32_t* accept_lens, int32_t* accepted_tokens,
                       int32_t* next_root,
                       void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * spec_verify_sampling -- rejection-sampling accept with residual and bonus.
 * [ACCEPT section 4], [INTERN 接受/拒绝], [EAGLE2 5.6], [SGL-XI eagle_sample].
 *
 * p = softmax(logits_row / T_b) (T_b = temperatures[b] > 0; T_b <= 0 means
 * greedy: p is one-hot at the argmax).  draft_probs q: [b*n, V] fp32, row of
 * node i = the distribution i's children were proposed from.  At node cur each
 * child c (sibling order) with token x is accepted iff u[b*n+c] * q(x) < p(x)
 * (fp32); the first accepted child is descended into.  When every child of cur
 * is rejected the terminal token is the smallest v with
 * u_final[b] * Z < sum_{w<=v} max(0, p_w - q_w) (Z = the total; from p itself
 * when Z == 0); when cur has no child or S drafts were accepted it is drawn
 * from p the same way.  Outputs as spec_verify_greedy.
 * ------------------------------------------------------------------------- */
int spec_verify_sampling(int b, int n, int S, int V, int dtype, const void* logits,
                         const float* draft_probs, const float* temperatures,
                         const float* u, const float* u_final,
                         const int32_t* draft_tokens, const int32_t* retrieve_index,
                         const int32_t* next_token, const int32_t* next_sibling,
                         int32_t* predict, int32_t* accept_index,
                         int32_t* accept_lens, int32_t* accepted_tokens,
                         int32_t* next_root,
                         void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * spec_verify_target_only -- target-only tree sampling, the second sampler of
 * EAGLE trees (it uses the target distribution alone, no draft proposal q).
 * [ACCEPT section 4, "Target-only Tree Sampling"].
 *
 * p = softmax(logits_row / T_b) (T_b <= 0: one-hot at the argmax).  coins:
 * [b*n] fp32 in [0, 1), one per node: the coin used when that node's
 * children are scanned (the root's first).  At the current node the children
 * are scanned in sibling order with prob_acc = 0 (fp32): prob_acc += p(x), and
 * child c of token x is accepted iff
 *     p(x) > 0 and (coin < prob_acc / threshold_acc or p(x) >= threshold_single);
 * the accepted child becomes the current node and its own coin is used next.
 * At most S levels.  The terminal token is the smallest v with
 * u_final[b] * Z < sum_{w<=v} r_w, r = p with the tokens of the current
 * node's children removed when they were all rejected (relu(p - buffer), the
 * buffer holding the rejected children's p), else r = p; from p when Z == 0.
 * Thresholds in (0, 1] (else SPEC_ERR_ARG).  Outputs as spec_verify_greedy;
 * workspace: spec_workspace_size(SPEC_OP_VERIFY_TARGET_ONLY, ...).
 * ------------------------------------------------------------------------- */
int spec_verify_target_only(int b, int n, int S, int V, int dtype, const void* logits,
                            const float* temperatures, const float* coins, const float* u_final,
                            float threshold_single, float threshold_acc,
                            const int32_t* draft_tokens, const int32_t* retrieve_index,
                            const int32_t* next_token, const int32_t* next_sibling,
                            int32_t* predict, int32_t* accept_index,
                            int32_t* accept_lens, int32_t* accepted_tokens,
                            int32_t* next_root,
                            void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Relaxed penalties and the top-k / top-p renormalisation before the accept.
 * [SGL-XI eagle_sample 的骨架 (acc_additive_penalties repeated over
 * draft_token_num: the relaxed penalties)], [SGL-XI 路径三, ACCEPT section 4
 * (temperature softmax, then top-k, then top-p, then renormalisation: the p
 * the accept consumes)].
 *
 * spec_add_penalties -- in place: logits[b*n + i][v] += penalties[b][v] for
 * each of request b's n verify rows (fp32 sum; bf16 logits store it rounded
 * to nearest even).  logits [b*n, V] and penalties [b, V] fp32 16-byte
 * aligned with V a multiple of 8 (else SPEC_ERR_UNSUPPORTED).  HBM-bound.
 *
 * spec_renorm_probs -- probs [b*n, V] fp32, the target distribution of every
 * verify row: softmax(logits / T_b) (T_b <= 0: one-hot at the argmax); with
 * 0 < top_k[b] < V the tokens whose logit is at least the k-th largest logit
 * (ties at the cut all kept), renormalised; with top_p[b] < 1, in descending
 * order, the shortest prefix whose mass reaches top_p of the kept mass,
 * widened to the last kept logit's ties, renormalised.  No workspace.
 *
 * spec_verify_sampling_probs / spec_verify_target_only_probs -- the two
 * samplers with the target distribution given (probs from spec_renorm_probs):
 * p at a verify row is that row; no softmax, no temperature.  Otherwise as
 * spec_verify_sampling / spec_verify_target_only, with workspaces of
 * SPEC_OP_VERIFY_SAMPLING / SPEC_OP_VERIFY_TARGET_ONLY.
 * ------------------------------------------------------------------------- */
int spec_add_penalties(int b, int n, int V, int dtype, void* logits, const float* penalties, void* stream);
int spec_renorm_probs(int b, int n, int V, int dtype, const void* logits, const float* temperatures,
                      const int32_t* top_k, const float* top_p, float* probs, void* stream);
int spec_verify_sampling_probs(int b, int n, int S, int V, const float* probs, const float* draft_probs,
                               const float* u, const float* u_final, const int32_t* draft_tokens,
                               const int32_t* retrieve_index, const int32_t* next_token,
                               const int32_t* next_sibling, int32_t* predict, int32_t* accept_index,
                               int32_t* accept_lens, int32_t* accepted_tokens, int32_t* next_root,
                               void* ws, size_t ws_bytes, void* stream);
int spec_verify_target_only_probs(int b, int n, int S, int V, const float* probs, const float* coins,
                                  const float* u_final, float threshold_single, float threshold_acc,
                                  const int32_t* draft_tokens, const int32_t* retrieve_index,
                                  const int32_t* next_token, const int32_t* next_sibling, int32_t* predict,
                                  int32_t* accept_index, int32_t* accept_lens, int32_t* accepted_tokens,
                                  int32_t* next_root, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * The chain fast path: topk == 1 with num_draft_tokens == num_steps + 1.
 * [SGL-XI 平台分派与 chain 特化 (build_chain_tree)], [ACCEPT section 5 (DSpark
 * correct_len, commit_lens, BuildOutTokens)].
 *
 * spec_build_chain_tree -- the tree of b chains of S draft tokens without the
 * generic ranking (its structure is constant): n = S + 1 nodes per request,
 * node 0 = bonus[b], node i = draft_tokens[b*draft_ld + i - 1] (for topk = 1
 * the concatenated token space of the select steps, draft_ld = S); parent of
 * node i = node i - 1; positions = seq_lens[b] + i; mask row i = nodes 0..i
 * (lower triangular); next_token[i] = i + 1 (-1 for the last); next_sibling
 * = -1; retrieve_index = b*n + i.  Outputs [b*n] as spec_build_tree's.  No
 * workspace; waits for the kernel before it like every call.
 * ------------------------------------------------------------------------- */
int spec_build_chain_tree(int b, int S, const int32_t* bonus, const int32_t* draft_tokens, int draft_ld,
                          const int32_t* seq_lens, int32_t* tree_tokens, int32_t* positions,
                          int32_t* retrieve_index, int32_t* next_token, int32_t* next_sibling,
                          uint64_t* mask_bits, void* stream);

/* spec_verify_chain_greedy -- the greedy accept of b chains in DSpark's
 * counts.  logits: [b*(S+1), V] (row b*(S+1)+j = chain position j, the root
 * first); target_predict = per-row argmax (lowest index on ties).
 *   correct_len[b] = number of leading positions j < S with draft_tokens[b, j]
 *                    == target_predict[j] (the first mismatch ends it);
 *   bonus[b]       = target_predict[correct_len];
 *   out_tokens     [b, S+1] = the draft tokens then -1, with the bonus written
 *                    at position correct_len (only the first commit_lens are
 *                    output);
 *   commit_lens[b] = correct_len + 1;  new_seq_lens[b] = prefix_lens[b] +
 *                    commit_lens (the accepted drafts and the root get KV;
 *                    the bonus gets its KV next step);
 *   accept_index   [b, S+1] (nullable) = b*(S+1) + j for j < commit_lens,
 *                    -1 after: with commit_lens as accept_lens it feeds
 *                    spec_commit_kv.
 * Workspace and overlap as spec_verify_greedy (n = S + 1).
 * ------------------------------------------------------------------------- */
int spec_verify_chain_greedy(int b, int S, int V, int dtype, const void* logits,
                             const int32_t* draft_tokens, int draft_ld, const int32_t* prefix_lens,
                             int32_t* correct_len, int32_t* bonus, int32_t* out_tokens,
                             int32_t* commit_lens, int32_t* new_seq_lens, int32_t* accept_index,
                             void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * The draft side of the KV, and the materialised verify mask.
 * [SGL-XI draft 前向的输入准备:prepare_for_draft], [EVOL 草稿、验证与槽位 (the
 * last partial page is duplicated)], [SGL-XI 三种 mask 形态].
 * Each takes a workspace for its error word only (spec_workspace_size of any
 * op is enough; SPEC_DEV_INDEX / SPEC_DEV_LENGTH as for the other calls).
 *
 * spec_assign_draft_locs -- out_cache_loc [b, topk, S] (flattened): the slots
 * the S draft steps of each of the topk branches write.  With L = seq_lens[b]
 * and row = req_to_token[req_pool_idx[b]] (req_rows rows of row_w entries):
 *   page_size == 1 or topk == 1: branch t, step s -> row[L + t*S + s] (each
 *     branch's steps are contiguous positions after the prefix);
 *   page_size > 1 and topk > 1: last_page = L % page_size, prefix_base =
 *     L - last_page, R = ceil((last_page + S) / page_size) * page_size; branch
 *     t's region is the page-aligned positions [prefix_base + t*R, +R); its
 *     first last_page positions are holes over the prefix tail (branch 0's
 *     are the real tail) and step s -> row[prefix_base + t*R + last_page + s].
 * The caller has allocated those positions in req_to_token.  positions [b]
 * (nullable, topk == 1 only) receives L, the first draft row's position.  A
 * position past row_w or a slot outside [0, num_slots) writes -1 and sets
 * SPEC_DEV_INDEX.
 * ------------------------------------------------------------------------- */
int spec_assign_draft_locs(int b, int topk, int S, int page_size, const int32_t* req_to_token, int req_rows,
                           int row_w, const int32_t* req_pool_idx, const int32_t* seq_lens, int64_t num_slots,
                           int32_t* out_cache_loc, int32_t* positions, void* ws, size_t ws_bytes, void* stream);

/* spec_duplicate_prefix_tail -- for page_size > 1 and topk > 1, copies the KV of
 * the real prefix tail (row[prefix_base + j], j < last_page) into the hole
 * slots of branches 1..topk-1 (row[prefix_base + t*R + j]), every layer, K and
 * V [Hkv, D] bf16, so that a kernel reading whole pages sees the prefix tail
 * in every branch.  A no-op for page_size == 1 or topk == 1.  page_size <= 64;
 * k_layers / v_layers: HOST arrays of num_layers (<= 128) device pointers,
 * 16-byte aligned. */
int spec_duplicate_prefix_tail(int b, int topk, int S, int page_size, int Hkv, int D, int num_layers,
                               void* const* k_layers, void* const* v_layers, int64_t num_slots,
                               const int32_t* req_to_token, int req_rows, int row_w, const int32_t* req_pool_idx,
                               const int32_t* seq_lens, void* ws, size_t ws_bytes, void* stream);

/* spec_build_full_mask -- the FULL_MASK verify mask: one block per request in
 * request order, request b's block = n rows of L_b + n bytes (L_b =
 * seq_lens[b]); row i = L_b prefix bytes (1: every verify row sees the whole
 * prefix), then n tree bytes (byte j = bit j of mask_bits[b*n + i]).
 * fill_prefix (0/1, the pages' fill_prefix_mask): 0 writes the tree bytes only
 * and leaves the prefix bytes as the reused buffer holds them.  mask_bytes is
 * the buffer's size, at least sum_b n*(L_b + n) (else nothing is written and
 * SPEC_DEV_LENGTH is set); b <= 16384.  HBM-bound: 16-byte stores. */
int spec_build_full_mask(int b, int n, const int32_t* seq_lens, const uint64_t* mask_bits, int fill_prefix,
                         uint8_t* mask, size_t mask_bytes, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * spec_commit_kv -- move the accepted rows' KV into the sequence, release the rest.
 * [SGL-XI KV 回写 (move_accept_tokens_to_target_kvcache)], [ACCEPT section 3
 * (input/output shift)], [EVOL 草稿、验证与槽位].
 *
 * For request b, L = accept_lens[b], k < L:
 *   dst_k = req_to_token[req_pool_idx[b], seq_lens[b] + k],
 *   src_k = verify_loc[accept_index[b, k]]   (accept_index is [b, W], global rows);
 * K and V rows [Hkv, D] bf16 of every layer move src -> dst, every source row
 * of a request being read before any of its targets is written.
 * new_seq_lens[b] = seq_lens[b] + L.
 * Free list (request order, then ascending node order): page_size == 1: each
 * verify slot of the request that is no dst slot; page_size > 1: each page id
 * (slot / page_size) holding a verify slot of the request and no dst slot of
 * it, once.  free_ids: [b*n] capacity; n_free: one int32.
 * k_layers / v_layers: HOST arrays of num_layers (<= 128) device pointers to
 * [num_slots, Hkv, D] bf16 pools.
 * ------------------------------------------------------------------------- */
int spec_commit_kv(int b, int n, int W, int Hkv, int D, int num_layers, int page_size,
                   void* const* k_layers, void* const* v_layers, int64_t num_slots,
                   const int32_t* req_to_token, int req_rows, int row_w,
                   const int32_t* req_pool_idx, const int32_t* seq_lens,
                   const int32_t* verify_loc, const int32_t* accept_index,
                   const int32_t* accept_lens, int32_t* new_seq_lens,
                   int32_t* free_ids, int32_t* n_free,
                   void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * spec_verify_greedy_noalloc -- spec_verify_greedy without a caller workspace.
 * The pages have no counterpart: this exists for callers that cannot allocate
 * device memory when they verify -- an engine whose allocator owns all device
 * memory, a latency-critical path that must not pay cudaMalloc's implicit
 * device synchronisation, or a plugin host that forbids allocation after
 * start-up.
 *
 * Arguments, outputs and semantics are those of spec_verify_greedy.  The
 * scratch memory is a fixed array of SPEC_NOALLOC_SCRATCH_BYTES inside the
 * library's device image; every GPU that loads the library holds it until the
 * process exits.  The entry point allocates nothing (no cudaMalloc, no
 * allocating library call).
 *   - The first call on a device looks the array's device address up
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - The first call on a device caches the address for the life of the
 *     process; it assumes the device's primary context lives that long (do
 *     not call this entry point after a cudaDeviceReset of that device).
 *   - Each call checks every argument before it enqueues anything, zeroes the
 *     array's arrival counters on `stream`, then runs the greedy kernel with
 *     the array as its workspace.
 *   - Every call shares the one array per device: calls that overlap on the
 *     GPU (different streams, or concurrent host threads) race.  Serialise them.
 *   - Returns SPEC_ERR_WORKSPACE when b, n and V need more scratch than the
 *     array holds.  The array is laid out for greedy accept alone (no room
 *     kept for the attention's merge area, so the pass never overlaps the
 *     call before it): 256 bytes of header, the arrival counters
 *     (4 * max(256, 2b+1) + 4b bytes, rounded up to 256) and 8 bytes per
 *     verify row and row chunk (about 9 chunks per row for 128 rows of 128K).
 *   - Device index errors (a tree pointer out of range) are handled as in
 *     spec_verify_greedy: the access is skipped and clamped, and a bit is set
 *     in the array's error word.  The word is not cleared between calls;
 *     spec_noalloc_last_error reads and clears it.
 * ------------------------------------------------------------------------- */
#define SPEC_NOALLOC_SCRATCH_BYTES (1u << 20)

int spec_verify_greedy_noalloc(int b, int n, int S, int V, int dtype, const void* logits,
                               const int32_t* draft_tokens, const int32_t* retrieve_index,
                               const int32_t* next_token, const int32_t* next_sibling,
                               int32_t* predict, int32_t* accept_index,
                               int32_t* accept_lens, int32_t* accepted_tokens,
                               int32_t* next_root, void* stream);

/* Synchronises `stream`, returns the SPEC_DEV_* bits that calls of
 * spec_verify_greedy_noalloc on the current device have set since the last
 * read (0 if clean) and clears them; a negative SPEC_ERR_* on failure.  Like
 * the entry point it serves, it allocates nothing. */
int spec_noalloc_last_error(void* stream);

#ifdef __cplusplus
}
#endif
#endif /* ACCEPT_SELECT_TOP_H */
