// kernels.cuh -- launch parameters of the verify/accept kernels (device side of
// the C ABI in accept_select_top.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace spec {

constexpr int kMaxLayers = 128;

struct SelectParams {
  int step, b, k, V, dtype;
  const void* logits;
  float temperature;
  const float* scores_in;
  float* score_blk;
  int32_t* token_blk;
  int score_ld;
  int32_t* parent_blk;
  int parent_ld;
  float* scores_out;
  int32_t* next_ids;
  float* topk_p_out;
  int rows, chunks, chunk_elems;
  bool vec_ok;
  // The chunk pass may run before the launch waits on the kernel ahead of
  // it (early): only with overlap allowed on the workspace, and only when
  // that kernel is the previous select on it, which uses the other half
  // (1 - half) of the partials and counters, or the KV commit, which uses
  // neither.
  bool early;
  int half;
  // streaming pass (rows of whole 16-byte vectors, at least one unit long,
  // at least kStreamMinBytes of logits): stream_ctas persistent CTAs taking
  // the stream_nb units of 256 vectors from a queue, group records
  // [stream_nb][2 row parities][32 lanes] in the partials, then each row's k
  // best [rows][kMaxK]; 0 selects the chunked kernel
  int stream_ctas, stream_nb;
  uint32_t* error;
  uint32_t* counters;    // this call's half: b counters
  uint32_t* queue;       // this call's half: the streaming kernel's batch queue
  unsigned char* partials;  // this call's half
};

struct ChainParams {
  int b, S, draft_ld;
  const int32_t* bonus;
  const int32_t* draft_tokens;
  const int32_t* seq_lens;
  int32_t* tree_tokens;
  int32_t* positions;
  int32_t* retrieve_index;
  int32_t* next_token;
  int32_t* next_sibling;
  uint64_t* mask_bits;
};

struct BuildParams {
  int b, k, S, n;
  const float* score_space;
  const int32_t* token_space;
  const int32_t* parent_space;
  const int32_t* bonus;
  const int32_t* seq_lens;
  int32_t* draft_tokens;
  int32_t* positions;
  int32_t* retrieve_index;
  int32_t* next_token;
  int32_t* next_sibling;
  uint64_t* mask_bits;
  uint32_t* error;
};

struct GreedyParams {
  int b, n, S, V, dtype;
  const void* logits;
  // chain: the DSpark counts of a topk = 1 chain (n = S + 1; no tree arrays):
  // draft tokens [b, S] with row stride draft_ld, prefix_lens in, and
  // correct_len / bonus / out_tokens [b, n] / commit_lens / new_seq_lens out;
  // accept_index [b, n] is written too (nullable in this mode)
  int chain;
  int draft_ld;
  const int32_t* chain_drafts;
  const int32_t* prefix_lens;
  int32_t* correct_len;
  int32_t* bonus;
  int32_t* out_tokens;
  int32_t* commit_lens;
  int32_t* new_seq_lens;
  const int32_t* draft_tokens;
  const int32_t* retrieve_index;
  const int32_t* next_token;
  const int32_t* next_sibling;
  int32_t* predict;
  int32_t* accept_index;
  int32_t* accept_lens;
  int32_t* accepted_tokens;
  int32_t* next_root;
  int chunks, chunk_elems;
  bool vec_ok;
  // The scan may run before the launch waits on the kernel ahead of it
  // (early): only with overlap allowed on the workspace, and only when that
  // kernel is the verify attention on it, whose merge slots and counters the
  // scan's partials and counters do not share.
  bool early;
  uint32_t* error;
  uint32_t* counters;
  unsigned char* partials;
};

struct SamplingParams {
  int b, n, S, V, dtype;
  const void* logits;
  // probabilities mode: probs [b*n, V] fp32 is the target distribution of
  // every verify row (no softmax, no temperature; logits unused)
  const float* probs;
  // target_only: the target-only tree sampler (coin of the scanned node,
  // sibling mass against the thresholds; draft_probs unused, may be null)
  int target_only;
  float thr_single, thr_acc;
  const float* draft_probs;
  const float* temperatures;
  const float* u;
  const float* u_final;
  const int32_t* draft_tokens;
  const int32_t* retrieve_index;
  const int32_t* next_token;
  const int32_t* next_sibling;
  int32_t* predict;
  int32_t* accept_index;
  int32_t* accept_lens;
  int32_t* accepted_tokens;
  int32_t* next_root;
  int chunks, chunk_elems;    // pass 1 split of a verify row
  int chunks2, chunk2_elems;  // pass 2 split of the terminal row
  int term_ctas;              // pass 2 CTAs a request (each takes chunks term_ctas apart)
  bool vec_ok;
  // pass 2 may read a thread's 16 tokens (logits and q) with 16-byte loads:
  // logits mode, V % 16 == 0, 16-byte aligned rows
  bool vec_term;
  // the streaming pass (logit rows of whole 16-byte vectors): stream_ctas
  // CTAs over stream_nu units, unit summaries usum; 0: the chunked pass 1
  int stream_ctas, stream_nu;
  float2* usum;
  uint32_t* queue;
  uint32_t* error;
  uint32_t* counters;
  unsigned char* partials;   // pass 1 partials (a row's statistics after the streaming pass)
  unsigned char* state;      // per-request state handed from pass 1 to pass 2
  unsigned char* partials2;  // pass 2 partials
};

struct AttentionParams {
  int b, n, Hq, Hkv, D, page_size;
  const void* q;
  const void* k_pool;
  const void* v_pool;
  long long num_slots;
  const int32_t* req_to_token;
  int req_rows, row_w;
  const int32_t* req_pool_idx;
  const int32_t* seq_lens;
  int max_seq_len;
  const int32_t* verify_loc;
  const uint64_t* mask_bits;
  float scale;
  void* out;
  float* lse;
  int splits;
  uint32_t* error;
  uint32_t* counters;
  unsigned char* partials;
};

struct CommitParams {
  int b, n, W, Hkv, D, num_layers, page_size;
  void* k_layers[kMaxLayers];
  void* v_layers[kMaxLayers];
  long long num_slots;
  const int32_t* req_to_token;
  int req_rows, row_w;
  const int32_t* req_pool_idx;
  const int32_t* seq_lens;
  const int32_t* verify_loc;
  const int32_t* accept_index;
  const int32_t* accept_lens;
  int32_t* new_seq_lens;
  int32_t* free_ids;
  int32_t* n_free;
  uint32_t* error;
  uint32_t* counters;
  unsigned char* partials;
};

struct DraftLocParams {
  int b, topk, S, page_size;
  const int32_t* req_to_token;
  int req_rows, row_w;
  const int32_t* req_pool_idx;
  const int32_t* seq_lens;
  long long num_slots;
  int32_t* out_cache_loc;
  int32_t* positions;
  uint32_t* error;
};

struct DupTailParams {
  int b, topk, S, page_size, Hkv, D, num_layers;
  void* k_layers[kMaxLayers];
  void* v_layers[kMaxLayers];
  long long num_slots;
  const int32_t* req_to_token;
  int req_rows, row_w;
  const int32_t* req_pool_idx;
  const int32_t* seq_lens;
  uint32_t* error;
};

struct FullMaskParams {
  int b, n, fill_prefix;
  const int32_t* seq_lens;
  const uint64_t* mask_bits;
  uint8_t* mask;
  size_t mask_bytes;
  uint32_t* error;
};

struct PenaltyParams {
  int b, n, V, dtype;
  void* logits;
  const float* penalties;
};

struct RenormParams {
  int b, n, V, dtype;
  const void* logits;
  const float* temperatures;
  const int32_t* top_k;
  const float* top_p;
  float* probs;
};

int launch_add_penalties(const PenaltyParams& p, cudaStream_t stream);
int launch_renorm(const RenormParams& p, cudaStream_t stream);

int launch_assign_draft_locs(const DraftLocParams& p, cudaStream_t stream);
int launch_duplicate_prefix_tail(const DupTailParams& p, cudaStream_t stream);
int launch_full_mask(const FullMaskParams& p, cudaStream_t stream);

int launch_select_topk(const SelectParams& p, cudaStream_t stream);
int launch_build_tree(const BuildParams& p, cudaStream_t stream);
int launch_build_chain_tree(const ChainParams& p, cudaStream_t stream);
int launch_verify_greedy(const GreedyParams& p, cudaStream_t stream);
int launch_verify_sampling(const SamplingParams& p, cudaStream_t stream);
int launch_commit_kv(const CommitParams& p, cudaStream_t stream);

size_t select_partial_bytes(int rows, int chunks);
// The logits streaming pass (stream_records.cu): per group of a lane's 8
// vectors of a 4 KB unit inside one row, the group maximum and the sum of
// 2^((x - max) c), c = log2(e) / T of the row.
struct StreamRecParams {
  const void* logits;
  int rows, V;
  float temperature;          // one temperature for every row, or
  const float* temperatures;  // one a request of rows_per_temp rows (0: greedy)
  int rows_per_temp;
  int nu;                     // units
  int cu;                     // units a queue answer hands out (set by launch_stream_records)
  float2* rec;                // records [nu][2 row parities][32 lanes], or null
  float2* usum;               // unit summaries [nu][2 row parities], or null
  uint32_t* queue;            // the unit queue (0 at launch)
  bool early;                 // reads may start before the grid before is done
};
struct StreamGeometry {
  int ctas, nb;    // CTAs (0: the streaming pass does not apply) and units
  size_t bytes;    // the records
};
// Records of a row that a request step holds at most (shared memory).
constexpr int kRowRecordsMax = 8192;
// The select takes the streaming pass from this many bytes of logits a call
// (measured crossover with the chunked kernel: about 30 MB on GB300).
constexpr size_t kStreamMinBytes = size_t(32) << 20;
// The streaming split of `rows` rows of V logits (vec per 16-byte vector) on a
// device of `sms` SMs.
StreamGeometry stream_geometry(long rows, int V, int vec, int sms);
int launch_stream_records(const StreamRecParams& p, int ctas, int dtype, cudaStream_t stream);
// The select's streaming layout: the records and then the rows' k best.
StreamGeometry select_stream_geometry(long rows, int V, int vec, int sms);
size_t build_tree_smem_bytes(int k, int S);
size_t sampling_partial_bytes(int rows, int chunks);
size_t sampling_state_bytes(int b);
size_t sampling_partial2_bytes(int b, int chunks2);
size_t commit_partial_bytes(int b, int n);

// Geometry of the tensor-core attention: m_tiles units of 128 query rows per
// (request, kv head); splits is always 1 (units split over CTAs are merged
// inside the kernel, in the same launch).
struct TcGeometry {
  int m_tiles, split_tiles, splits;
};
TcGeometry attention_tc_geometry(int b, int n, int Hq, int Hkv, int max_seq_len);
int launch_attention_tc(const AttentionParams& p, const TcGeometry& geo, cudaStream_t stream);
size_t attention_partial_bytes();  // merge slots and counters, any D <= 128

// spec_verify_greedy on a workspace laid out for greedy accept alone (the
// partials straight after the counters; never overlaps the kernel before):
// the no-allocation entry point's fixed scratch.
size_t greedy_compact_bytes(int b, int n, int V);
int verify_greedy_compact(int b, int n, int S, int V, int dtype, const void* logits, const int32_t* draft_tokens,
                          const int32_t* retrieve_index, const int32_t* next_token, const int32_t* next_sibling,
                          int32_t* predict, int32_t* accept_index, int32_t* accept_lens, int32_t* accepted_tokens,
                          int32_t* next_root, void* ws, size_t ws_bytes, void* stream);

}  // namespace spec
