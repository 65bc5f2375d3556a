/*
 * oracle.c -- plain, slow CPU oracle for one EAGLE-style verify/accept step.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h for who may load it, the sources
 * cited as [KEY section], and the conventions).  Every function follows the
 * pages' statement of the step in their order, one request at a time, with no
 * blocking or fusion beyond what that statement implies.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- helpers */

/* A logit as fp64: fp32 directly, bf16 by placing its 16 bits on top of an
 * fp32 (exact widening). */
static double logit_at(const void* base, int dtype, size_t i) {
  if (dtype == ORC_F32) return (double)((const float*)base)[i];
  uint32_t w = (uint32_t)((const uint16_t*)base)[i] << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

static double bf16_at(const uint16_t* base, size_t i) {
  uint32_t w = (uint32_t)base[i] << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* Ordering used by every top-k / argmax of the method: a ranks before b when
 * its value is larger, or equal with the smaller index.  The pages leave ties
 * open; the lowest index wins everywhere. */
static int ranks_before(double va, long ia, double vb, long ib) {
  return va > vb || (va == vb && ia < ib);
}

/* Index of the largest logit of one row, ties to the lowest index. */
static int row_argmax(const void* logits, int dtype, size_t off, int V) {
  int best = 0;
  double bv = logit_at(logits, dtype, off);
  for (int v = 1; v < V; ++v) {
    double x = logit_at(logits, dtype, off + (size_t)v);
    if (ranks_before(x, v, bv, best)) {
      bv = x;
      best = v;
    }
  }
  return best;
}

/* Softmax of one row at temperature T > 0, fp64, each probability rounded to
 * fp32 (the type in which probabilities are handed on). */
static void row_softmax(const void* logits, int dtype, size_t off, int V,
                        double T, float* p) {
  double m = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double x = logit_at(logits, dtype, off + (size_t)v);
    if (x > m) m = x;
  }
  double s = 0.0;
  for (int v = 0; v < V; ++v) s += exp((logit_at(logits, dtype, off + (size_t)v) - m) / T);
  for (int v = 0; v < V; ++v)
    p[v] = (float)(exp((logit_at(logits, dtype, off + (size_t)v) - m) / T) / s);
}

/* ------------------------------------------------------- c1 softmax/top-k */

int oracle_softmax_topk(int rows, int V, int dtype, const void* logits,
                        double temperature, int k, float* topk_p,
                        int32_t* topk_idx) {
  if (rows < 0 || V <= 0 || k <= 0 || k > V || !(temperature > 0.0)) return ORC_EARG;
  if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_EARG;
  double* best = (double*)malloc(sizeof(double) * (size_t)k);
  long* bidx = (long*)malloc(sizeof(long) * (size_t)k);
  for (int r = 0; r < rows; ++r) {
    size_t off = (size_t)r * (size_t)V;
    /* softmax denominator */
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
      double x = logit_at(logits, dtype, off + (size_t)v);
      if (x > m) m = x;
    }
    double s = 0.0;
    for (int v = 0; v < V; ++v) s += exp((logit_at(logits, dtype, off + (size_t)v) - m) / temperature);
    /* the k best logits, kept sorted by insertion */
    int have = 0;
    for (int v = 0; v < V; ++v) {
      double x = logit_at(logits, dtype, off + (size_t)v);
      if (have == k && !ranks_before(x, v, best[k - 1], bidx[k - 1])) continue;
      int pos = have < k ? have++ : k - 1;
      while (pos > 0 && ranks_before(x, v, best[pos - 1], bidx[pos - 1])) {
        best[pos] = best[pos - 1];
        bidx[pos] = bidx[pos - 1];
        --pos;
      }
      best[pos] = x;
      bidx[pos] = v;
    }
    for (int j = 0; j < k; ++j) {
      topk_idx[(size_t)r * k + j] = (int32_t)bidx[j];
      topk_p[(size_t)r * k + j] = (float)(exp((best[j] - m) / temperature) / s);
    }
  }
  free(best);
  free(bidx);
  return ORC_OK;
}

/* ---------------------------------------------------- c2 path-score step */

int oracle_path_step(int step, int b, int k, const float* topk_p,
                     const int32_t* topk_idx, const float* scores_in,
                     float* score_blk, int32_t* token_blk, int32_t* parent_blk,
                     float* scores_out, int32_t* next_ids) {
  if (step < 0 || b < 0 || k <= 0) return ORC_EARG;
  if (step == 0) {
    /* _select_top_k_tokens_first: the root's top-k is the first block; the
     * parent block is arange(-1, k). */
    for (int r = 0; r < b; ++r) {
      for (int j = 0; j < k; ++j) {
        size_t i = (size_t)r * k + j;
        score_blk[i] = topk_p[i];
        token_blk[i] = topk_idx[i];
        scores_out[i] = topk_p[i];
        next_ids[i] = topk_idx[i];
      }
      for (int j = 0; j <= k; ++j) parent_blk[(size_t)r * (k + 1) + j] = j - 1;
    }
    return ORC_OK;
  }
  if (!scores_in) return ORC_EARG;
  const int kk = k * k;
  float* expand = (float*)malloc(sizeof(float) * (size_t)kk);
  char* taken = (char*)malloc((size_t)kk);
  for (int r = 0; r < b; ++r) {
    /* _select_top_k_tokens_later: expand_scores = scores[:, :, None] * topk_p */
    for (int row = 0; row < k; ++row) {
      for (int j = 0; j < k; ++j) {
        /* the fp64 product of two fp32 values is exact, so this is the
         * correctly rounded fp32 product */
        double prod = (double)scores_in[(size_t)r * k + row] *
                      (double)topk_p[((size_t)r * k + row) * k + j];
        expand[row * k + j] = (float)prod;
      }
    }
    for (int f = 0; f < kk; ++f) {
      score_blk[(size_t)r * kk + f] = expand[f];
      token_blk[(size_t)r * kk + f] = topk_idx[(size_t)r * kk + f];
      taken[f] = 0;
    }
    /* fast_topk over the k*k flattened scores, best first */
    for (int j = 0; j < k; ++j) {
      int sel = -1;
      for (int f = 0; f < kk; ++f) {
        if (taken[f]) continue;
        if (sel < 0 || ranks_before(expand[f], f, expand[sel], sel)) sel = f;
      }
      taken[sel] = 1;
      parent_blk[(size_t)r * k + j] = sel + kk * (step - 1) + k;
      scores_out[(size_t)r * k + j] = expand[sel];
      next_ids[(size_t)r * k + j] = topk_idx[(size_t)r * kk + sel];
    }
  }
  free(expand);
  free(taken);
  return ORC_OK;
}

int oracle_select_topk(int step, int b, int k, int V, int dtype,
                       const void* draft_logits, double temperature,
                       const float* scores_in, float* score_blk,
                       int32_t* token_blk, int32_t* parent_blk,
                       float* scores_out, int32_t* next_ids, float* topk_p_out) {
  if (step < 0 || b < 0 || k <= 0) return ORC_EARG;
  int rows = b * (step ? k : 1);
  float* p = (float*)malloc(sizeof(float) * ((size_t)rows * k + 1));
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * ((size_t)rows * k + 1));
  int rc = oracle_softmax_topk(rows, V, dtype, draft_logits, temperature, k, p, idx);
  if (rc == ORC_OK)
    rc = oracle_path_step(step, b, k, p, idx, scores_in, score_blk, token_blk,
                          parent_blk, scores_out, next_ids);
  if (rc == ORC_OK && topk_p_out) memcpy(topk_p_out, p, sizeof(float) * (size_t)rows * k);
  free(p);
  free(idx);
  return rc;
}

/* -------------------------------------------- c3..c5 organize + build tree */

int oracle_build_tree(int b, int k, int S, int n, const float* score_space,
                      const int32_t* token_space, const int32_t* parent_space,
                      const int32_t* bonus, const int32_t* seq_lens,
                      int32_t* draft_tokens, int32_t* positions,
                      int32_t* retrieve_index, int32_t* next_token,
                      int32_t* next_sibling, uint64_t* mask_bits,
                      int32_t* parent_node) {
  if (b < 0 || k <= 0 || S <= 0 || n <= 0 || n > 64) return ORC_EARG;
  const int C = k + (S - 1) * k * k;  /* score space == token space length */
  const int P = 1 + (S - 1) * k;      /* parent_list length */
  if (n - 1 > C) return ORC_EARG;
  int rc = ORC_OK;
  char* taken = (char*)malloc((size_t)C + 1);
  int sel[64], par[64];
  for (int r = 0; r < b && rc == ORC_OK; ++r) {
    const float* sc = score_space + (size_t)r * C;
    /* organize_draft_results: torch.topk(score_list, n-1) ... */
    memset(taken, 0, (size_t)C);
    for (int t = 0; t < n - 1; ++t) {
      int best = -1;
      for (int p = 0; p < C; ++p) {
        if (taken[p]) continue;
        if (best < 0 || ranks_before(sc[p], p, sc[best], best)) best = p;
      }
      taken[best] = 1;
      sel[t] = best;
    }
    /* ... then torch.sort(top_scores_index): ascending positions */
    for (int t = 1; t < n - 1; ++t) {
      int v = sel[t], j = t;
      while (j > 0 && sel[j - 1] > v) {
        sel[j] = sel[j - 1];
        --j;
      }
      sel[j] = v;
    }
    /* build_tree: node 0 is the bonus token (the root), node j >= 1 is the
     * j-th selected position.  The parent of position p is parent_list[p / k]
     * (a global position, -1 = root); its node is 1 + its rank among the
     * selected positions. */
    par[0] = -1;
    for (int j = 1; j < n; ++j) {
      int p = sel[j - 1];
      int t = p / k;
      if (t < 0 || t >= P) { rc = ORC_EBOUNDS; break; }
      int ppos = parent_space[(size_t)r * P + t];
      if (ppos < 0) {
        par[j] = 0;
      } else {
        int found = -1;
        for (int q = 0; q < n - 1; ++q)
          if (sel[q] == ppos) found = q + 1;
        if (found < 0) { rc = ORC_EINVARIANT; break; }
        par[j] = found;
      }
    }
    if (rc != ORC_OK) break;
    const size_t base = (size_t)r * n;
    for (int i = 0; i < n; ++i) {
      /* ancestors-or-self by walking the parent pointers */
      uint64_t m = 0;
      int depth = -1, a = i, guard = 0;
      while (a != -1 && guard <= n) {
        m |= (uint64_t)1 << a;
        ++depth;
        a = par[a];
        ++guard;
      }
      if (guard > n) { rc = ORC_EINVARIANT; break; }
      mask_bits[base + i] = m;
      positions[base + i] = seq_lens[r] + depth;
      retrieve_index[base + i] = (int32_t)(base + i);
      draft_tokens[base + i] = i == 0 ? bonus[r] : token_space[(size_t)r * C + sel[i - 1]];
      /* first child = smallest node whose parent is i */
      int first = -1;
      for (int c = 0; c < n && first < 0; ++c)
        if (par[c] == i) first = c;
      next_token[base + i] = first;
      /* next sibling = smallest larger node with the same parent */
      int sib = -1;
      if (i > 0)
        for (int c = i + 1; c < n && sib < 0; ++c)
          if (par[c] == par[i]) sib = c;
      next_sibling[base + i] = sib;
      if (parent_node) parent_node[base + i] = par[i];
    }
  }
  free(taken);
  return rc;
}

/* ------------------------------------------------------- c6 attention */

static int attend_one(int b, int i, int h, int n, int Hq, int Hkv, int D,
                      const uint16_t* q, const uint16_t* k_pool,
                      const uint16_t* v_pool, int64_t num_slots,
                      const int32_t* req_to_token, int row_w,
                      const int32_t* req_pool_idx, const int32_t* seq_lens,
                      const int32_t* verify_loc, const uint64_t* mask_bits,
                      double scale, double* o, double* lse_out) {
  const int g = h / (Hq / Hkv);
  const size_t row = (size_t)b * n + i;
  const int L = seq_lens[b];
  const int req = req_pool_idx[b];
  if (L < 0 || L > row_w) return ORC_EBOUNDS;
  /* key list: prefix positions, then the visible tree nodes */
  int nkeys = 0;
  int64_t* slots = (int64_t*)malloc(sizeof(int64_t) * ((size_t)L + (size_t)n));
  for (int t = 0; t < L; ++t) slots[nkeys++] = req_to_token[(size_t)req * row_w + t];
  for (int j = 0; j < n; ++j)
    if ((mask_bits[row] >> j) & 1u) slots[nkeys++] = verify_loc[(size_t)b * n + j];
  for (int t = 0; t < nkeys; ++t)
    if (slots[t] < 0 || slots[t] >= num_slots) {
      free(slots);
      return ORC_EBOUNDS;
    }
  double* s = (double*)malloc(sizeof(double) * (size_t)(nkeys + 1));
  double m = -INFINITY;
  const size_t qoff = (row * Hq + h) * (size_t)D;
  for (int t = 0; t < nkeys; ++t) {
    const size_t koff = ((size_t)slots[t] * Hkv + g) * (size_t)D;
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += bf16_at(q, qoff + d) * bf16_at(k_pool, koff + d);
    s[t] = scale * dot;
    if (s[t] > m) m = s[t];
  }
  double l = 0.0;
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  for (int t = 0; t < nkeys; ++t) {
    double w = exp(s[t] - m);
    l += w;
    const size_t voff = ((size_t)slots[t] * Hkv + g) * (size_t)D;
    for (int d = 0; d < D; ++d) o[d] += w * bf16_at(v_pool, voff + d);
  }
  for (int d = 0; d < D; ++d) o[d] /= l;
  *lse_out = m + log(l);
  free(s);
  free(slots);
  return ORC_OK;
}

int oracle_verify_attention(int b, int n, int Hq, int Hkv, int D,
                            const uint16_t* q, const uint16_t* k_pool,
                            const uint16_t* v_pool, int64_t num_slots,
                            const int32_t* req_to_token, int row_w,
                            const int32_t* req_pool_idx, const int32_t* seq_lens,
                            const int32_t* verify_loc, const uint64_t* mask_bits,
                            double scale, int n_pairs, const int32_t* pairs,
                            double* out, double* lse) {
  if (b < 0 || n <= 0 || n > 64 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0) return ORC_EARG;
  double* o = (double*)malloc(sizeof(double) * (size_t)D);
  int rc = ORC_OK;
  const long total = pairs ? n_pairs : (long)b * n * Hq;
  for (long t = 0; t < total && rc == ORC_OK; ++t) {
    long row, h;
    if (pairs) {
      row = pairs[2 * t];
      h = pairs[2 * t + 1];
      if (row < 0 || row >= (long)b * n || h < 0 || h >= Hq) { rc = ORC_EARG; break; }
    } else {
      row = t / Hq;
      h = t % Hq;
    }
    double l;
    rc = attend_one((int)(row / n), (int)(row % n), (int)h, n, Hq, Hkv, D, q, k_pool,
                    v_pool, num_slots, req_to_token, row_w, req_pool_idx, seq_lens,
                    verify_loc, mask_bits, scale, o, &l);
    if (rc != ORC_OK) break;
    if (out) memcpy(out + ((size_t)row * Hq + h) * D, o, sizeof(double) * (size_t)D);
    if (lse) lse[(size_t)row * Hq + h] = l;
  }
  free(o);
  return rc;
}

/* ------------------------------------------------------- c7 greedy accept */

/* Fills accepted_tokens / next_root from predict and accept_index:
 * accept_tokens = predict[accept_index], the next root is the last one. */
static void gather_outputs(int b, int W, const int32_t* predict,
                           const int32_t* accept_index, const int32_t* accept_lens,
                           int32_t* accepted_tokens, int32_t* next_root) {
  for (int r = 0; r < b; ++r) {
    int L = accept_lens[r];
    if (accepted_tokens)
      for (int d = 0; d < W; ++d)
        accepted_tokens[(size_t)r * W + d] = d < L ? predict[accept_index[(size_t)r * W + d]] : -1;
    if (next_root) next_root[r] = predict[accept_index[(size_t)r * W + L - 1]];
  }
}

int oracle_verify_greedy(int b, int n, int S, int V, int dtype, const void* logits,
                         const int32_t* draft_tokens, const int32_t* retrieve_index,
                         const int32_t* next_token, const int32_t* next_sibling,
                         int32_t* predict, int32_t* accept_index,
                         int32_t* accept_lens, int32_t* accepted_tokens,
                         int32_t* next_root) {
  if (b < 0 || n <= 0 || S <= 0 || V <= 0) return ORC_EARG;
  if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_EARG;
  const int W = S + 1;
  const size_t rows = (size_t)b * n;
  /* target_predict = argmax over every verify row */
  int32_t* tp = (int32_t*)malloc(sizeof(int32_t) * (rows + 1));
  for (size_t r = 0; r < rows; ++r) tp[r] = row_argmax(logits, dtype, r * (size_t)V, V);
  /* predict starts as zeros, accept_index as -1 */
  for (size_t r = 0; r < rows; ++r) predict[r] = 0;
  for (size_t i = 0; i < (size_t)b * W; ++i) accept_index[i] = -1;
  int rc = ORC_OK;
  for (int r = 0; r < b && rc == ORC_OK; ++r) {
    const size_t base = (size_t)r * n;
    int cur = 0, ncd = 0;
    accept_index[(size_t)r * W] = retrieve_index[base];
    for (int d = 1; d <= S; ++d) {
      int c = next_token[base + cur], hit = -1, guard = 0;
      while (c != -1) {
        if (c < 0 || c >= n || ++guard > n) { rc = ORC_EBOUNDS; break; }
        if (draft_tokens[base + c] == tp[base + cur]) { hit = c; break; }
        c = next_sibling[base + c];
      }
      if (rc != ORC_OK || hit < 0) break;
      predict[retrieve_index[base + cur]] = draft_tokens[base + hit];
      accept_index[(size_t)r * W + d] = retrieve_index[base + hit];
      ++ncd;
      cur = hit;
    }
    if (rc != ORC_OK) break;
    /* terminal Target token at the last accepted row */
    predict[retrieve_index[base + cur]] = tp[base + cur];
    accept_lens[r] = ncd + 1;
  }
  if (rc == ORC_OK) gather_outputs(b, W, predict, accept_index, accept_lens, accepted_tokens, next_root);
  free(tp);
  return rc;
}

/* ------------------------------------------------ c8 rejection sampling */

/* Smallest v with u*Z < sum_{w<=v} r_w, accumulated in fp64 in vocab order. */
static int sample_from(const double* r, int V, double Z, float u) {
  const double target = (double)u * Z;
  double acc = 0.0;
  int last = -1;
  for (int v = 0; v < V; ++v) {
    if (r[v] > 0.0) last = v;
    acc += r[v];
    if (target < acc) return v;
  }
  return last;
}

/* The target distribution at a verify row: given (probs, the renormalised
 * distribution), or softmax(logits / T) (one-hot at the argmax for T <= 0). */
static void target_p(const float* probs, const void* logits, int dtype, size_t row, int V, double T, float* p) {
  const size_t loff = row * (size_t)V;
  if (probs) {
    memcpy(p, probs + loff, sizeof(float) * (size_t)V);
  } else if (T > 0.0) {
    row_softmax(logits, dtype, loff, V, T, p);
  } else {
    int a = row_argmax(logits, dtype, loff, V);
    for (int v = 0; v < V; ++v) p[v] = v == a ? 1.0f : 0.0f;
  }
}

static int sampling_walk(int b, int n, int S, int V, int dtype, const void* logits, const float* probs,
                         const float* draft_probs, const float* temperatures,
                         const float* u, const float* u_final,
                         const int32_t* draft_tokens, const int32_t* retrieve_index,
                         const int32_t* next_token, const int32_t* next_sibling,
                         int32_t* predict, int32_t* accept_index,
                         int32_t* accept_lens, int32_t* accepted_tokens,
                         int32_t* next_root) {
  if (b < 0 || n <= 0 || S <= 0 || V <= 0) return ORC_EARG;
  if (!probs && dtype != ORC_F32 && dtype != ORC_BF16) return ORC_EARG;
  const int W = S + 1;
  const size_t rows = (size_t)b * n;
  float* p = (float*)malloc(sizeof(float) * (size_t)V);
  double* res = (double*)malloc(sizeof(double) * (size_t)V);
  for (size_t r = 0; r < rows; ++r) predict[r] = 0;
  for (size_t i = 0; i < (size_t)b * W; ++i) accept_index[i] = -1;
  int rc = ORC_OK;
  for (int r = 0; r < b && rc == ORC_OK; ++r) {
    const size_t base = (size_t)r * n;
    const double T = probs ? 1.0 : temperatures[r];
    int cur = 0, ncd = 0, all_rejected = 0;
    accept_index[(size_t)r * W] = retrieve_index[base];
    for (int d = 0; d <= S; ++d) {
      /* p = the target distribution at the current node: softmax(logits / T),
       * or the one-hot argmax when T <= 0 (greedy), or the given one */
      target_p(probs, logits, dtype, base + cur, V, T, p);
      if (d == S) break; /* depth exhausted: bonus from p */
      const float* q = draft_probs + (base + cur) * (size_t)V;
      /* try the children in sibling order; accept x when u*q(x) < p(x), i.e.
       * u < min(1, p(x)/q(x)) without the division */
      int c = next_token[base + cur], hit = -1, guard = 0, had_child = c != -1;
      while (c != -1) {
        if (c < 0 || c >= n || ++guard > n) { rc = ORC_EBOUNDS; break; }
        int x = draft_tokens[base + c];
        if (x < 0 || x >= V) { rc = ORC_EBOUNDS; break; }
        float lhs = u[base + c] * q[x]; /* one fp32 multiply */
        if (lhs < p[x]) { hit = c; break; }
        c = next_sibling[base + c];
      }
      if (rc != ORC_OK) break;
      if (hit < 0) {
        all_rejected = had_child;
        break;
      }
      predict[retrieve_index[base + cur]] = draft_tokens[base + hit];
      accept_index[(size_t)r * W + d + 1] = retrieve_index[base + hit];
      ++ncd;
      cur = hit;
    }
    if (rc != ORC_OK) break;
    /* terminal token: from the residual max(0, p - q)/Z when every child of
     * the current node was rejected (from p when Z == 0), else from p */
    const float* q = draft_probs + (base + cur) * (size_t)V;
    double Z = 0.0;
    if (all_rejected) {
      for (int v = 0; v < V; ++v) {
        double rv = (double)p[v] - (double)q[v];
        res[v] = rv > 0.0 ? rv : 0.0;
        Z += res[v];
      }
    }
    if (!(Z > 0.0)) {
      Z = 0.0;
      for (int v = 0; v < V; ++v) {
        res[v] = (double)p[v];
        Z += res[v];
      }
    }
    predict[retrieve_index[base + cur]] = sample_from(res, V, Z, u_final[r]);
    accept_lens[r] = ncd + 1;
  }
  if (rc == ORC_OK) gather_outputs(b, W, predict, accept_index, accept_lens, accepted_tokens, next_root);
  free(p);
  free(res);
  return rc;
}

int oracle_verify_sampling(int b, int n, int S, int V, int dtype, const void* logits,
                           const float* draft_probs, const float* temperatures,
                           const float* u, const float* u_final,
                           const int32_t* draft_tokens, const int32_t* retrieve_index,
                           const int32_t* next_token, const int32_t* next_sibling,
                           int32_t* predict, int32_t* accept_index,
                           int32_t* accept_lens, int32_t* accepted_tokens,
                           int32_t* next_root) {
  return sampling_walk(b, n, S, V, dtype, logits, NULL, draft_probs, temperatures, u, u_final, draft_tokens,
                       retrieve_index, next_token, next_sibling, predict, accept_index, accept_lens,
                       accepted_tokens, next_root);
}

int oracle_verify_sampling_probs(int b, int n, int S, int V, const float* probs, const float* draft_probs,
                                 const float* u, const float* u_final,
                                 const int32_t* draft_tokens, const int32_t* retrieve_index,
                                 const int32_t* next_token, const int32_t* next_sibling,
                                 int32_t* predict, int32_t* accept_index,
                                 int32_t* accept_lens, int32_t* accepted_tokens,
                                 int32_t* next_root) {
  if (!probs) return ORC_EARG;
  return sampling_walk(b, n, S, V, ORC_F32, NULL, probs, draft_probs, NULL, u, u_final, draft_tokens,
                       retrieve_index, next_token, next_sibling, predict, accept_index, accept_lens,
                       accepted_tokens, next_root);
}

/* -------------------------------------- f1 target-only tree sampling */

static int target_only_walk(int b, int n, int S, int V, int dtype, const void* logits, const float* probs,
                            const float* temperatures, const float* u, const float* u_final,
                            float threshold_single, float threshold_acc,
                            const int32_t* draft_tokens, const int32_t* retrieve_index,
                            const int32_t* next_token, const int32_t* next_sibling,
                            int32_t* predict, int32_t* accept_index,
                            int32_t* accept_lens, int32_t* accepted_tokens,
                            int32_t* next_root) {
  if (b < 0 || n <= 0 || S <= 0 || V <= 0) return ORC_EARG;
  if (!probs && dtype != ORC_F32 && dtype != ORC_BF16) return ORC_EARG;
  if (!(threshold_single > 0.0f && threshold_single <= 1.0f)) return ORC_EARG;
  if (!(threshold_acc > 0.0f && threshold_acc <= 1.0f)) return ORC_EARG;
  const int W = S + 1;
  const size_t rows = (size_t)b * n;
  float* p = (float*)malloc(sizeof(float) * (size_t)V);
  float* buf = (float*)malloc(sizeof(float) * (size_t)V); /* the current node's buffer row */
  double* r = (double*)malloc(sizeof(double) * (size_t)V);
  for (size_t i = 0; i < rows; ++i) predict[i] = 0;
  for (size_t i = 0; i < (size_t)b * W; ++i) accept_index[i] = -1;
  int rc = ORC_OK;
  for (int q = 0; q < b && rc == ORC_OK; ++q) {
    const size_t base = (size_t)q * n;
    const double T = probs ? 1.0 : temperatures[q];
    int cur = 0, ncd = 0;
    float coin = u[base + 0];
    accept_index[(size_t)q * W] = retrieve_index[base];
    for (int d = 0; d <= S; ++d) {
      /* the target distribution at the current node, and its empty buffer row */
      target_p(probs, logits, dtype, base + cur, V, T, p);
      for (int v = 0; v < V; ++v) buf[v] = 0.0f;
      if (d == S) break; /* depth exhausted */
      /* siblings in order, accumulating their target mass */
      float prob_acc = 0.0f;
      int c = next_token[base + cur], hit = -1, guard = 0;
      while (c != -1) {
        if (c < 0 || c >= n || ++guard > n) { rc = ORC_EBOUNDS; break; }
        int x = draft_tokens[base + c];
        if (x < 0 || x >= V) { rc = ORC_EBOUNDS; break; }
        const float px = p[x];
        prob_acc += px; /* fp32 accumulation */
        if (px > 0.0f && (coin < prob_acc / threshold_acc || px >= threshold_single)) {
          hit = c;
          break;
        }
        buf[x] = px; /* rejected: its mass is kept out of the terminal draw here */
        c = next_sibling[base + c];
      }
      if (rc != ORC_OK || hit < 0) break;
      predict[retrieve_index[base + cur]] = draft_tokens[base + hit];
      accept_index[(size_t)q * W + d + 1] = retrieve_index[base + hit];
      ++ncd;
      cur = hit;
      coin = u[base + hit]; /* the accepted child's own coin for the next level */
    }
    if (rc != ORC_OK) break;
    /* terminal token from relu(p - buffer) at the current node */
    double Z = 0.0;
    for (int v = 0; v < V; ++v) {
      double rv = (double)p[v] - (double)buf[v];
      r[v] = rv > 0.0 ? rv : 0.0;
      Z += r[v];
    }
    if (!(Z > 0.0)) {
      Z = 0.0;
      for (int v = 0; v < V; ++v) {
        r[v] = (double)p[v];
        Z += r[v];
      }
    }
    predict[retrieve_index[base + cur]] = sample_from(r, V, Z, u_final[q]);
    accept_lens[q] = ncd + 1;
  }
  if (rc == ORC_OK) gather_outputs(b, W, predict, accept_index, accept_lens, accepted_tokens, next_root);
  free(p);
  free(buf);
  free(r);
  return rc;
}

int oracle_verify_target_only(int b, int n, int S, int V, int dtype, const void* logits,
                              const float* temperatures, const float* u, const float* u_final,
                              float threshold_single, float threshold_acc,
                              const int32_t* draft_tokens, const int32_t* retrieve_index,
                              const int32_t* next_token, const int32_t* next_sibling,
                              int32_t* predict, int32_t* accept_index,
                              int32_t* accept_lens, int32_t* accepted_tokens,
                              int32_t* next_root) {
  return target_only_walk(b, n, S, V, dtype, logits, NULL, temperatures, u, u_final, threshold_single,
                          threshold_acc, draft_tokens, retrieve_index, next_token, next_sibling, predict,
                          accept_index, accept_lens, accepted_tokens, next_root);
}

int oracle_verify_target_only_probs(int b, int n, int S, int V, const float* probs, const float* u,
                                    const float* u_final, float threshold_single, float threshold_acc,
                                    const int32_t* draft_tokens, const int32_t* retrieve_index,
                                    const int32_t* next_token, const int32_t* next_sibling,
                                    int32_t* predict, int32_t* accept_index,
                                    int32_t* accept_lens, int32_t* accepted_tokens,
                                    int32_t* next_root) {
  if (!probs) return ORC_EARG;
  return target_only_walk(b, n, S, V, ORC_F32, NULL, probs, NULL, u, u_final, threshold_single, threshold_acc,
                          draft_tokens, retrieve_index, next_token, next_sibling, predict, accept_index,
                          accept_lens, accepted_tokens, next_root);
}

/* ------------------------------------------------------ f2 chain fast path */

int oracle_build_chain_tree(int b, int S, const int32_t* bonus, const int32_t* draft_tokens,
                            int draft_ld, const int32_t* seq_lens,
                            int32_t* tree_tokens, int32_t* positions, int32_t* retrieve_index,
                            int32_t* next_token, int32_t* next_sibling, uint64_t* mask_bits) {
  if (b < 0 || S < 1 || S + 1 > 64 || draft_ld < S) return ORC_EARG;
  const int n = S + 1;
  for (int q = 0; q < b; ++q) {
    const size_t base = (size_t)q * n;
    for (int i = 0; i < n; ++i) {
      /* a chain: node i hangs below node i-1 and sees nodes 0..i */
      tree_tokens[base + i] = i == 0 ? bonus[q] : draft_tokens[(size_t)q * draft_ld + i - 1];
      positions[base + i] = seq_lens[q] + i;
      retrieve_index[base + i] = (int32_t)(base + i);
      next_token[base + i] = i + 1 < n ? i + 1 : -1;
      next_sibling[base + i] = -1;
      uint64_t m = 0;
      for (int j = 0; j <= i; ++j) m |= (uint64_t)1 << j;
      mask_bits[base + i] = m;
    }
  }
  return ORC_OK;
}

int oracle_chain_accept_greedy(int b, int S, int V, int dtype, const void* logits,
                               const int32_t* draft_tokens, int draft_ld, const int32_t* prefix_lens,
                               int32_t* correct_len, int32_t* bonus, int32_t* out_tokens,
                               int32_t* commit_lens, int32_t* new_seq_lens, int32_t* accept_index) {
  if (b < 0 || S < 1 || V <= 0 || draft_ld < S) return ORC_EARG;
  if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_EARG;
  const int n = S + 1;
  for (int q = 0; q < b; ++q) {
    /* compute_dflash_correct_drafts_and_bonus: leading matches of the chain */
    int c = 0;
    while (c < S) {
      int tp = row_argmax(logits, dtype, ((size_t)q * n + c) * (size_t)V, V);
      if (draft_tokens[(size_t)q * draft_ld + c] != tp) break;
      ++c;
    }
    correct_len[q] = c;
    bonus[q] = row_argmax(logits, dtype, ((size_t)q * n + c) * (size_t)V, V);
    /* BuildOutTokens: the draft tokens, then the bonus scattered at correct_len */
    for (int j = 0; j < n; ++j) out_tokens[(size_t)q * n + j] = j < S ? draft_tokens[(size_t)q * draft_ld + j] : -1;
    out_tokens[(size_t)q * n + c] = bonus[q];
    /* FinalizeAcceptLens */
    commit_lens[q] = c + 1;
    new_seq_lens[q] = prefix_lens[q] + c + 1;
    if (accept_index)
      for (int j = 0; j < n; ++j) accept_index[(size_t)q * n + j] = j <= c ? (int32_t)((size_t)q * n + j) : -1;
  }
  return ORC_OK;
}

/* ------------------------------------------- f4 the draft side of the KV */

/* The region geometry of paged branches: hole count, page-aligned base and
 * the positions one branch region spans. */
static void branch_region(int L, int S, int page_size, int* last_page, int* prefix_base, int* R) {
  *last_page = L % page_size;
  *prefix_base = L - *last_page;
  *R = (*last_page + S + page_size - 1) / page_size * page_size;
}

int oracle_assign_draft_locs(int b, int topk, int S, int page_size, const int32_t* req_to_token,
                             int row_w, const int32_t* req_pool_idx, const int32_t* seq_lens,
                             int64_t num_slots, int32_t* out_cache_loc, int32_t* positions) {
  if (b < 0 || topk < 1 || S < 1 || page_size < 1 || row_w < 1) return ORC_EARG;
  for (int q = 0; q < b; ++q) {
    const int L = seq_lens[q];
    const int32_t* row = req_to_token + (size_t)req_pool_idx[q] * row_w;
    for (int t = 0; t < topk; ++t) {
      for (int s = 0; s < S; ++s) {
        long pos;
        if (page_size == 1 || topk == 1) {
          pos = (long)L + (long)t * S + s; /* contiguous after the prefix */
        } else {
          int last_page, prefix_base, R;
          branch_region(L, S, page_size, &last_page, &prefix_base, &R);
          pos = (long)prefix_base + (long)t * R + last_page + s;
        }
        if (L < 0 || pos >= row_w) return ORC_EBOUNDS;
        const int32_t slot = row[pos];
        if (slot < 0 || slot >= num_slots) return ORC_EBOUNDS;
        out_cache_loc[((size_t)q * topk + t) * S + s] = slot;
      }
    }
    if (positions && topk == 1) positions[q] = L;
  }
  return ORC_OK;
}

int oracle_duplicate_prefix_tail(int b, int topk, int S, int page_size, int Hkv, int D, int num_layers,
                                 uint16_t* const* k_layers, uint16_t* const* v_layers, int64_t num_slots,
                                 const int32_t* req_to_token, int row_w, const int32_t* req_pool_idx,
                                 const int32_t* seq_lens) {
  if (b < 0 || topk < 1 || S < 1 || page_size < 1 || Hkv < 1 || D < 1 || num_layers < 1) return ORC_EARG;
  if (page_size == 1 || topk == 1) return ORC_OK;
  const size_t rowlen = (size_t)Hkv * D;
  for (int q = 0; q < b; ++q) {
    int last_page, prefix_base, R;
    branch_region(seq_lens[q], S, page_size, &last_page, &prefix_base, &R);
    const int32_t* row = req_to_token + (size_t)req_pool_idx[q] * row_w;
    for (int t = 1; t < topk; ++t) {
      for (int j = 0; j < last_page; ++j) {
        const long sp = (long)prefix_base + j, dp = (long)prefix_base + (long)t * R + j;
        if (dp >= row_w) return ORC_EBOUNDS;
        const int64_t src = row[sp], dst = row[dp];
        if (src < 0 || src >= num_slots || dst < 0 || dst >= num_slots) return ORC_EBOUNDS;
        for (int l = 0; l < num_layers; ++l) {
          memcpy(k_layers[l] + (size_t)dst * rowlen, k_layers[l] + (size_t)src * rowlen, rowlen * 2);
          memcpy(v_layers[l] + (size_t)dst * rowlen, v_layers[l] + (size_t)src * rowlen, rowlen * 2);
        }
      }
    }
  }
  return ORC_OK;
}

int oracle_full_mask(int b, int n, const int32_t* seq_lens, const uint64_t* mask_bits, int fill_prefix,
                     uint8_t* mask) {
  if (b < 0 || n < 1 || n > 64) return ORC_EARG;
  size_t off = 0;
  for (int q = 0; q < b; ++q) {
    const int L = seq_lens[q];
    if (L < 0) return ORC_EBOUNDS;
    for (int i = 0; i < n; ++i) {
      uint8_t* row = mask + off + (size_t)i * (L + n);
      if (fill_prefix)
        for (int j = 0; j < L; ++j) row[j] = 1; /* every verify row sees the whole prefix */
      for (int j = 0; j < n; ++j) row[L + j] = (uint8_t)((mask_bits[(size_t)q * n + i] >> j) & 1u);
    }
    off += (size_t)n * (L + n);
  }
  return ORC_OK;
}

/* ------------------------- f3 relaxed penalties, top-k / top-p renorm */

/* fp32 -> bf16 bits, round to nearest with ties to even (NaN kept quiet). */
static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x40u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

int oracle_add_penalties(int b, int n, int V, int dtype, void* logits, const float* penalties) {
  if (b < 0 || n <= 0 || V <= 0) return ORC_EARG;
  if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_EARG;
  for (int q = 0; q < b; ++q)
    for (int i = 0; i < n; ++i)
      for (int v = 0; v < V; ++v) {
        const size_t e = ((size_t)q * n + i) * (size_t)V + v;
        /* the same penalty row for every verify row of the request, added in fp32 */
        const float sum = (float)logit_at(logits, dtype, e) + penalties[(size_t)q * V + v];
        if (dtype == ORC_F32) ((float*)logits)[e] = sum;
        else ((uint16_t*)logits)[e] = to_bf16(sum);
      }
  return ORC_OK;
}

typedef struct {
  double l;
  int v;
} LogitAt;

/* descending logit, ascending index among equals */
static int by_logit_desc(const void* pa, const void* pb) {
  const LogitAt* a = (const LogitAt*)pa;
  const LogitAt* b = (const LogitAt*)pb;
  if (a->l != b->l) return a->l > b->l ? -1 : 1;
  return a->v < b->v ? -1 : (a->v > b->v);
}

int oracle_renorm_probs(int b, int n, int V, int dtype, const void* logits, const float* temperatures,
                        const int32_t* top_k, const float* top_p, float* probs) {
  if (b < 0 || n <= 0 || V <= 0) return ORC_EARG;
  if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_EARG;
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  char* keep = (char*)malloc((size_t)V);
  LogitAt* order = (LogitAt*)malloc(sizeof(LogitAt) * (size_t)V);
  for (int q = 0; q < b; ++q) {
    const double T = temperatures[q];
    for (int i = 0; i < n; ++i) {
      const size_t off = ((size_t)q * n + i) * (size_t)V;
      /* the temperature softmax (one-hot at the argmax for T <= 0) */
      if (T > 0.0) {
        double m = -INFINITY, s = 0.0;
        for (int v = 0; v < V; ++v) {
          double x = logit_at(logits, dtype, off + v);
          if (x > m) m = x;
        }
        for (int v = 0; v < V; ++v) s += (p[v] = exp((logit_at(logits, dtype, off + v) - m) / T));
        for (int v = 0; v < V; ++v) p[v] /= s;
      } else {
        int a = row_argmax(logits, dtype, off, V);
        for (int v = 0; v < V; ++v) p[v] = v == a ? 1.0 : 0.0;
      }
      for (int v = 0; v < V; ++v) {
        keep[v] = 1;
        order[v].l = logit_at(logits, dtype, off + v);
        order[v].v = v;
      }
      qsort(order, (size_t)V, sizeof(LogitAt), by_logit_desc);
      /* top-k: every token at or above the k-th largest logit */
      const int k = top_k[q];
      if (k > 0 && k < V) {
        const double cut = order[k - 1].l;
        for (int v = 0; v < V; ++v) keep[v] = logit_at(logits, dtype, off + v) >= cut;
      }
      double z = 0.0;
      for (int v = 0; v < V; ++v) z += keep[v] ? p[v] : 0.0;
      for (int v = 0; v < V; ++v) p[v] = keep[v] ? p[v] / z : 0.0;
      /* top-p on the renormalised distribution: the shortest prefix (in
       * descending order) whose mass reaches top_p, widened to ties */
      const double tp = top_p[q];
      if (tp < 1.0) {
        double acc = 0.0, cut = order[0].l;
        for (int r = 0; r < V; ++r) {
          const int v = order[r].v;
          if (!keep[v]) continue;
          acc += p[v];
          cut = order[r].l;
          if (acc >= tp) break;
        }
        for (int v = 0; v < V; ++v) keep[v] = keep[v] && logit_at(logits, dtype, off + v) >= cut;
        z = 0.0;
        for (int v = 0; v < V; ++v) z += keep[v] ? p[v] : 0.0;
        for (int v = 0; v < V; ++v) p[v] = keep[v] ? p[v] / z : 0.0;
      }
      for (int v = 0; v < V; ++v) probs[off + v] = (float)p[v];
    }
  }
  free(p);
  free(keep);
  free(order);
  return ORC_OK;
}

/* ------------------------------------------------------------ c9 commit */

int oracle_commit_kv(int b, int n, int W, int Hkv, int D, int num_layers,
                     int page_size, uint16_t* const* k_layers,
                     uint16_t* const* v_layers, int64_t num_slots,
                     const int32_t* req_to_token, int row_w,
                     const int32_t* req_pool_idx, const int32_t* seq_lens,
                     const int32_t* verify_loc, const int32_t* accept_index,
                     const int32_t* accept_lens, int32_t* new_seq_lens,
                     int32_t* free_ids, int32_t* n_free) {
  if (b < 0 || n <= 0 || W <= 0 || Hkv <= 0 || D <= 0 || num_layers <= 0 || page_size <= 0)
    return ORC_EARG;
  const size_t rowlen = (size_t)Hkv * D; /* elements of one slot */
  int64_t* src = (int64_t*)malloc(sizeof(int64_t) * (size_t)W);
  int64_t* dst = (int64_t*)malloc(sizeof(int64_t) * (size_t)W);
  uint16_t* tmp = (uint16_t*)malloc(sizeof(uint16_t) * rowlen * (size_t)W * 2);
  int nf = 0, rc = ORC_OK;
  for (int r = 0; r < b && rc == ORC_OK; ++r) {
    const int L = accept_lens[r];
    const int s0 = seq_lens[r];
    const int req = req_pool_idx[r];
    if (L < 1 || L > W || s0 < 0 || s0 + L > row_w) { rc = ORC_EBOUNDS; break; }
    for (int k = 0; k < L; ++k) {
      int ai = accept_index[(size_t)r * W + k];
      if (ai < 0 || ai >= b * n) { rc = ORC_EBOUNDS; break; }
      src[k] = verify_loc[ai];
      dst[k] = req_to_token[(size_t)req * row_w + s0 + k];
      if (src[k] < 0 || src[k] >= num_slots || dst[k] < 0 || dst[k] >= num_slots) { rc = ORC_EBOUNDS; break; }
    }
    if (rc != ORC_OK) break;
    /* move_kv_cache(tgt, src): every source row is read before any target is
     * written, so a target that is also a later source cannot be clobbered */
    for (int layer = 0; layer < num_layers; ++layer) {
      for (int k = 0; k < L; ++k) {
        memcpy(tmp + (size_t)(2 * k) * rowlen, k_layers[layer] + (size_t)src[k] * rowlen, rowlen * 2);
        memcpy(tmp + (size_t)(2 * k + 1) * rowlen, v_layers[layer] + (size_t)src[k] * rowlen, rowlen * 2);
      }
      for (int k = 0; k < L; ++k) {
        memcpy(k_layers[layer] + (size_t)dst[k] * rowlen, tmp + (size_t)(2 * k) * rowlen, rowlen * 2);
        memcpy(v_layers[layer] + (size_t)dst[k] * rowlen, tmp + (size_t)(2 * k + 1) * rowlen, rowlen * 2);
      }
    }
    new_seq_lens[r] = s0 + L;
    /* release what the accepted path does not keep */
    for (int j = 0; j < n; ++j) {
      int64_t slot = verify_loc[(size_t)r * n + j];
      if (slot < 0 || slot >= num_slots) { rc = ORC_EBOUNDS; break; }
      int64_t unit = slot / page_size;
      int kept = 0;
      for (int k = 0; k < L && !kept; ++k) kept = dst[k] / page_size == unit;
      if (kept) continue;
      int listed = 0; /* a page is listed once, at its first node */
      for (int jj = 0; jj < j && !listed; ++jj) listed = verify_loc[(size_t)r * n + jj] / page_size == unit;
      if (listed) continue;
      free_ids[nf++] = (int32_t)unit;
    }
  }
  if (rc == ORC_OK) *n_free = nf;
  free(src);
  free(dst);
  free(tmp);
  return rc;
}
