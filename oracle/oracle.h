/*
 * oracle.h -- plain, slow CPU oracle for one EAGLE-style verify/accept step.
 *
 * TEST INFRASTRUCTURE ONLY.  This library is loaded by the test suite, by the
 * package smoke check and by the CPU-baseline leg of the benchmark, and by
 * nothing else.  It shares no code, header, table or helper with the GPU
 * library: it includes none of its headers and the GPU library includes none
 * of these.  Both sides meet only at the seeded input generator.
 *
 * Sources (web pages), cited in this file as [KEY section]:
 *   [SGL-XI]  "SGLang 源码完全拆解(十一):投机解码——草稿生成、批量验证与 token 接受如何接进同一条前向"
 *   [ACCEPT]  "投机解码 Accept从 Verify 行到最终输出路径"
 *   [EVOL]    "SGLang 设计演进投机解码、PD 分离与大规模 EP（2025 上半年）", chapter "EAGLE 投机解码四部曲"
 *   [INTERN]  "Speculative Decoding" (SGLang internals, part 3, execution model)
 *   [EAGLE2]  "把投机采样讲透：以 SGLang 中的 EAGLE-2 为例"
 *
 * Arithmetic is fp64 except where the method itself hands values over in a
 * narrower type: probabilities leave the softmax as fp32, a path score is one
 * correctly rounded fp32 product, and the accept test compares fp32 values.
 *
 * Conventions shared by every function:
 *   - every pointer is a host pointer owned by the caller; nothing is kept;
 *   - "row" of a request b and tree node i is the flattened verify row b*n+i;
 *   - -1 means "none" in every tree pointer and in accept_index padding;
 *   - return value 0 = success; ORC_EARG = bad argument; ORC_EBOUNDS = an index
 *     read from an input array is out of range; ORC_EINVARIANT = an input breaks
 *     an invariant of the method (for example a selected node whose parent was
 *     not selected).
 *
 * Parity status: every function is pinned by tests against values the pages
 * print, closed forms, library routines or brute force.  The rejection sampler
 * on trees with several children per node follows a reading of the pages (p
 * and q fixed across siblings, one coin per child), which the pages give no
 * numbers for; it is pinned against that reading's closed-form law for one
 * sibling level (each sibling's acceptance probability and the residual's
 * share, by a chi-square test), besides the single-candidate values the pages
 * print and the T=0 == greedy identity.
 */
#ifndef ACCEPT_SELECT_TOP_ORACLE_H
#define ACCEPT_SELECT_TOP_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_F32 0
#define ORC_BF16 1

#define ORC_OK 0
#define ORC_EARG 1
#define ORC_EBOUNDS 2
#define ORC_EINVARIANT 3

/* c1 -- per-row softmax and top-k of the draft distribution.
 * [SGL-XI select_top_k_tokens]: each draft row yields topk_p (its top-k
 * probabilities) and topk_index (their token ids).
 * p_v = exp((l_v - max l)/T) / sum_w exp((l_w - max l)/T), fp64, rounded to fp32.
 * The k tokens are the k largest logits ordered by (logit desc, token id asc).
 * logits: [rows, V] of dtype (ORC_F32 or ORC_BF16 bit patterns).
 * topk_p, topk_idx: [rows, k]. */
int oracle_softmax_topk(int rows, int V, int dtype, const void* logits,
                        double temperature, int k, float* topk_p, int32_t* topk_idx);

/* c2 -- one step of select_top_k_tokens given the rows' top-k.
 * [SGL-XI organize_draft_results] (_select_top_k_tokens_first / _later).
 * step 0: rows = 1 per request; score block = topk_p [b,k]; tokens = topk_idx
 *   [b,k]; parent block = [-1, 0, .., k-1] [b,k+1]; next scores = topk_p.
 * step i>=1: rows = k per request; expand[r*k+j] = fp32(scores_in[r]*topk_p[r,j]);
 *   score block = expand [b,k*k]; tokens = topk_idx [b,k*k]; the k best expand
 *   values by (value desc, flat index asc), in that order, give
 *   parent block = sel + k*k*(i-1) + k [b,k], next scores = expand[sel],
 *   next input ids = tokens[sel]. */
int oracle_path_step(int step, int b, int k, const float* topk_p,
                     const int32_t* topk_idx, const float* scores_in,
                     float* score_blk, int32_t* token_blk, int32_t* parent_blk,
                     float* scores_out, int32_t* next_ids);

/* c1 followed by c2 on draft logits [b*(step ? k : 1), V]; topk_p_out may be NULL. */
int oracle_select_topk(int step, int b, int k, int V, int dtype,
                       const void* draft_logits, double temperature,
                       const float* scores_in, float* score_blk,
                       int32_t* token_blk, int32_t* parent_blk,
                       float* scores_out, int32_t* next_ids, float* topk_p_out);

/* c3..c5 -- organize_draft_results followed by build_tree_kernel_efficient.
 * [SGL-XI organize_draft_results], [SGL-XI build_tree_kernel_efficient],
 * [ACCEPT section 2], [EAGLE2 sections 4.3, 5.3, 5.4].
 * score_space, token_space: [b, C], C = k + (S-1)*k*k (all S blocks, in step order);
 * parent_space: [b, 1 + (S-1)*k] (the parent blocks of steps 0..S-2).
 * Outputs (all [b*n] unless stated): draft_tokens, positions, retrieve_index,
 * next_token, next_sibling (node indices local to the request), mask_bits
 * (one uint64 per row, bit j set iff node j is an ancestor of the row's node or
 * the node itself), parent_node (optional, may be NULL). n <= 64. */
int oracle_build_tree(int b, int k, int S, int n, const float* score_space,
                      const int32_t* token_space, const int32_t* parent_space,
                      const int32_t* bonus, const int32_t* seq_lens,
                      int32_t* draft_tokens, int32_t* positions,
                      int32_t* retrieve_index, int32_t* next_token,
                      int32_t* next_sibling, uint64_t* mask_bits,
                      int32_t* parent_node);

/* c6 -- tree-masked verify attention, fp64.
 * [EAGLE2 sections 4.2-4.3]: the queries are the tree nodes; the keys are the
 * request's cached prefix (positions 0..seq_len-1 through req_to_token, all
 * visible) followed by the tree nodes whose mask bit is set (through verify_loc).
 * q: [b*n, Hq, D] bf16 bits; k_pool, v_pool: [num_slots, Hkv, D] bf16 bits;
 * q head h reads kv head h / (Hq/Hkv).  out: [b*n, Hq, D] fp64 and lse:
 * [b*n, Hq] fp64 (natural log), both optional.  With pairs != NULL only the
 * n_pairs (row, head) pairs listed are computed and written (pairs is
 * [n_pairs, 2]); other outputs are left untouched. */
int oracle_verify_attention(int b, int n, int Hq, int Hkv, int D,
                            const uint16_t* q, const uint16_t* k_pool,
                            const uint16_t* v_pool, int64_t num_slots,
                            const int32_t* req_to_token, int row_w,
                            const int32_t* req_pool_idx, const int32_t* seq_lens,
                            const int32_t* verify_loc, const uint64_t* mask_bits,
                            double scale, int n_pairs, const int32_t* pairs,
                            double* out, double* lse);

/* c7 -- greedy accept.  [SGL-XI eagle_sample], [ACCEPT section 3], [EAGLE2 5.3].
 * logits: [b*n, V]; accept_index, accepted_tokens: [b, S+1]; predict: [b*n];
 * accept_lens, next_root: [b].  accepted_tokens and next_root may be NULL. */
int oracle_verify_greedy(int b, int n, int S, int V, int dtype, const void* logits,
                         const int32_t* draft_tokens, const int32_t* retrieve_index,
                         const int32_t* next_token, const int32_t* next_sibling,
                         int32_t* predict, int32_t* accept_index,
                         int32_t* accept_lens, int32_t* accepted_tokens,
                         int32_t* next_root);

/* c8 -- rejection-sampling accept.  [ACCEPT section 4], [INTERN accept/reject],
 * [EAGLE2 5.6], [SGL-XI eagle_sample].
 * draft_probs: [b*n, V] fp32, row of node i = the distribution node i's children
 * were proposed from; temperatures: [b] (<= 0 means greedy); u: [b*n] (one coin
 * per child node, u[b*n+0] unused); u_final: [b].  Outputs as c7. */
int oracle_verify_sampling(int b, int n, int S, int V, int dtype, const void* logits,
                           const float* draft_probs, const float* temperatures,
                           const float* u, const float* u_final,
                           const int32_t* draft_tokens, const int32_t* retrieve_index,
                           const int32_t* next_token, const int32_t* next_sibling,
                           int32_t* predict, int32_t* accept_index,
                           int32_t* accept_lens, int32_t* accepted_tokens,
                           int32_t* next_root);

/* f1 -- target-only tree sampling (the second sampler of EAGLE trees).
 * [ACCEPT section 4, "Target-only Tree Sampling"].
 * p_cur = softmax(logits_row(cur) / T_b), rounded to fp32 (T_b <= 0: one-hot
 * at the argmax).  The walk starts at the root with coin = u[b*n + 0]; at the
 * current node the children are scanned in sibling order with an fp32
 * accumulator prob_acc (zero at each node): prob_acc += p_cur(x) for child c
 * of token x, and c is accepted iff
 *     p_cur(x) > 0  and  (coin < prob_acc / threshold_acc  or  p_cur(x) >= threshold_single)
 * (fp32 arithmetic).  An accepted child becomes the current node and its own
 * coin u[b*n + c] is used for the next level; a rejected child writes p_cur(x)
 * into the buffer row of the current node.  At most S levels.  The terminal
 * token is drawn with u_final[b] from relu(p_cur - buffer_cur) (the current
 * node's rejected siblings removed; from p_cur itself when that mass is 0), as
 * the smallest v with u_final * Z < running sum (fp64, vocabulary order).
 * Thresholds in (0, 1].  Outputs as oracle_verify_greedy. */
int oracle_verify_target_only(int b, int n, int S, int V, int dtype, const void* logits,
                              const float* temperatures, const float* u, const float* u_final,
                              float threshold_single, float threshold_acc,
                              const int32_t* draft_tokens, const int32_t* retrieve_index,
                              const int32_t* next_token, const int32_t* next_sibling,
                              int32_t* predict, int32_t* accept_index,
                              int32_t* accept_lens, int32_t* accepted_tokens,
                              int32_t* next_root);

/* f2 -- the chain fast path for topk == 1 (num_draft_tokens = num_steps + 1).
 * [SGL-XI 平台分派与 chain 特化 (build_chain_tree)], [ACCEPT section 5 (DSpark
 * correct_len)].
 *
 * oracle_build_chain_tree: the tree of a chain of S draft tokens per request,
 * n = S + 1 nodes: node 0 = bonus[b], node i = draft_tokens[b*draft_ld + i-1];
 * the parent of node i is node i-1; positions = seq_len + i; mask row i =
 * nodes 0..i (lower triangular); next_token[i] = i + 1 (-1 for the last);
 * next_sibling = -1; retrieve_index = b*n + i.  Outputs [b*n]. */
int oracle_build_chain_tree(int b, int S, const int32_t* bonus, const int32_t* draft_tokens,
                            int draft_ld, const int32_t* seq_lens,
                            int32_t* tree_tokens, int32_t* positions, int32_t* retrieve_index,
                            int32_t* next_token, int32_t* next_sibling, uint64_t* mask_bits);

/* oracle_chain_accept_greedy: the chain's greedy accept in the counts DSpark
 * uses.  logits: [b*(S+1), V], row b*(S+1)+j = the target at chain position
 * j (the root is position 0).  target_predict[j] = argmax (lowest index on
 * ties).  correct_len = the number of leading positions j < S with
 * draft_tokens[b, j] == target_predict[j] (the first mismatch ends it);
 * bonus = target_predict[correct_len]; out_tokens [b, S+1] = the draft tokens
 * then -1, with the bonus written at position correct_len (only the first
 * commit_lens entries are output); commit_lens = correct_len + 1;
 * new_seq_lens = prefix_lens + commit_lens; accept_index [b, S+1] (nullable)
 * = b*(S+1) + j for j < commit_lens, -1 after. */
int oracle_chain_accept_greedy(int b, int S, int V, int dtype, const void* logits,
                               const int32_t* draft_tokens, int draft_ld, const int32_t* prefix_lens,
                               int32_t* correct_len, int32_t* bonus, int32_t* out_tokens,
                               int32_t* commit_lens, int32_t* new_seq_lens, int32_t* accept_index);

/* f4 -- the draft side of the KV: slots for the draft writes, the prefix-tail
 * copy of paged branches, and the materialised verify mask.
 * [SGL-XI draft 前向的输入准备:prepare_for_draft], [EVOL 草稿、验证与槽位 (the
 * last partial page is duplicated)], [SGL-XI 三种 mask 形态 (FULL_MASK,
 * fill_prefix_mask)].
 *
 * oracle_assign_draft_locs: out_cache_loc [b, topk, S] (flattened) = the slots
 * the S draft steps of each of the topk branches write.  With L = seq_lens[b]
 * and row = req_to_token row req_pool_idx[b]:
 *   page_size == 1 or topk == 1: branch t, step s -> row[L + t*S + s] (each
 *     branch writes contiguous positions after the prefix);
 *   page_size > 1 and topk > 1: last_page = L % page_size, prefix_base = L -
 *     last_page, R = ceil((last_page + S) / page_size) * page_size; branch t's
 *     page-aligned region is positions [prefix_base + t*R, prefix_base +
 *     (t+1)*R), its first last_page positions are holes (branch 0's are the
 *     real prefix tail) and step s -> row[prefix_base + t*R + last_page + s].
 * positions [b] (nullable; topk == 1 only) = L, the position of the first
 * draft row.  ORC_EBOUNDS when a position passes row_w or a slot is out of
 * [0, num_slots). */
int oracle_assign_draft_locs(int b, int topk, int S, int page_size, const int32_t* req_to_token,
                             int row_w, const int32_t* req_pool_idx, const int32_t* seq_lens,
                             int64_t num_slots, int32_t* out_cache_loc, int32_t* positions);

/* oracle_duplicate_prefix_tail: for page_size > 1 and topk > 1, copies the KV
 * of the real prefix tail (row[prefix_base + j], j < last_page) into the hole
 * slots of branches 1..topk-1 (row[prefix_base + t*R + j]), every layer, K and
 * V, so that a kernel reading whole pages sees the prefix tail in every
 * branch.  Does nothing for page_size == 1 or topk == 1. */
int oracle_duplicate_prefix_tail(int b, int topk, int S, int page_size, int Hkv, int D, int num_layers,
                                 uint16_t* const* k_layers, uint16_t* const* v_layers, int64_t num_slots,
                                 const int32_t* req_to_token, int row_w, const int32_t* req_pool_idx,
                                 const int32_t* seq_lens);

/* oracle_full_mask: the FULL_MASK verify mask, one block per request, blocks
 * concatenated in request order: request b's block is n rows of L_b + n bytes
 * (L_b = seq_lens[b]), row i = L_b prefix columns (1, visible; written only
 * when fill_prefix, else left as they are) then n tree columns, column j = 1
 * iff bit j of mask_bits[b*n + i] is set.  mask: uint8, sum_b n*(L_b + n)
 * bytes. */
int oracle_full_mask(int b, int n, const int32_t* seq_lens, const uint64_t* mask_bits, int fill_prefix,
                     uint8_t* mask);

/* f3 -- relaxed penalties and top-k / top-p renormalisation before the accept.
 * [SGL-XI eagle_sample 的骨架 (acc_additive_penalties, repeat_interleave over
 * draft_token_num: the relaxed penalties)], [SGL-XI 路径三 and ACCEPT section 4
 * (temperature softmax, then top-k, then top-p, then renormalisation; p is the
 * distribution the accept consumes)].
 *
 * oracle_add_penalties: logits[b*n + i][v] += penalties[b][v] for every verify
 * row i of request b, the sum formed in fp32 and stored in the logits' type
 * (bf16: rounded to nearest, ties to even). */
int oracle_add_penalties(int b, int n, int V, int dtype, void* logits, const float* penalties);

/* oracle_renorm_probs: probs [b*n, V] fp32 = the target distribution of every
 * verify row: p = softmax(l / T_b) in fp64 (T_b <= 0: one-hot at the argmax);
 * top-k (0 < top_k[b] < V): the tokens whose logit is at least the k-th
 * largest logit (ties at the cut all kept), renormalised; top-p (top_p[b] <
 * 1): in descending order of p (index ascending among equals) the shortest
 * prefix whose mass reaches top_p, widened to every token whose logit equals
 * the last one kept, renormalised; each probability rounded to fp32. */
int oracle_renorm_probs(int b, int n, int V, int dtype, const void* logits, const float* temperatures,
                        const int32_t* top_k, const float* top_p, float* probs);

/* The two samplers on a given target distribution (probs [b*n, V] fp32, the
 * output of oracle_renorm_probs): p at a verify row is that row, no softmax
 * and no temperature; everything else as oracle_verify_sampling and
 * oracle_verify_target_only. */
int oracle_verify_sampling_probs(int b, int n, int S, int V, const float* probs, const float* draft_probs,
                                 const float* u, const float* u_final,
                                 const int32_t* draft_tokens, const int32_t* retrieve_index,
                                 const int32_t* next_token, const int32_t* next_sibling,
                                 int32_t* predict, int32_t* accept_index,
                                 int32_t* accept_lens, int32_t* accepted_tokens,
                                 int32_t* next_root);
int oracle_verify_target_only_probs(int b, int n, int S, int V, const float* probs, const float* u,
                                    const float* u_final, float threshold_single, float threshold_acc,
                                    const int32_t* draft_tokens, const int32_t* retrieve_index,
                                    const int32_t* next_token, const int32_t* next_sibling,
                                    int32_t* predict, int32_t* accept_index,
                                    int32_t* accept_lens, int32_t* accepted_tokens,
                                    int32_t* next_root);

/* c9 -- KV commit.  [SGL-XI KV 回写], [ACCEPT section 3 (input/output shift)],
 * [EVOL 草稿、验证与槽位].
 * For request b with L = accept_lens[b] and k < L:
 *   dst_k = req_to_token[req_pool_idx[b]*row_w + seq_lens[b] + k],
 *   src_k = verify_loc[accept_index[b*W + k]];
 * every src row is read (all layers, K and V, [Hkv, D]) before any dst row is
 * written.  new_seq_lens[b] = seq_lens[b] + L.
 * Free list, request order, then ascending node order:
 *   page_size == 1: every verify slot of the request that is no dst slot;
 *   page_size  > 1: every page (slot / page_size) that holds a verify slot of
 *   the request and no dst slot of the request, listed once, at its first node.
 * k_layers, v_layers: arrays of num_layers host pointers to [num_slots, Hkv, D]
 * bf16 pools (modified in place); free_ids: [>= b*n]; n_free: one int. */
int oracle_commit_kv(int b, int n, int W, int Hkv, int D, int num_layers,
                     int page_size, uint16_t* const* k_layers,
                     uint16_t* const* v_layers, int64_t num_slots,
                     const int32_t* req_to_token, int row_w,
                     const int32_t* req_pool_idx, const int32_t* seq_lens,
                     const int32_t* verify_loc, const int32_t* accept_index,
                     const int32_t* accept_lens, int32_t* new_seq_lens,
                     int32_t* free_ids, int32_t* n_free);

#ifdef __cplusplus
}
#endif
#endif
