// spec_api.cu -- the C ABI declared in accept_select_top.h: argument checks,
// workspace sizing and layout, and kernel dispatch.  No call allocates memory
// or synchronises the host, except spec_last_error.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <unordered_map>

#include "accept_select_top.h"
#include "common.cuh"
#include "kernels.cuh"

using namespace spec;

namespace {

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline int elem_bytes(int dtype) { return dtype == SPEC_F32 ? 4 : 2; }
inline int vec_elems(int dtype) { return dtype == SPEC_F32 ? 4 : 8; }

// Upper bound on the chunk count pick_split() returns for `rows` rows of V.
inline int chunk_bound(long rows, int V) { return pick_split(rows, V, 1).chunks; }

inline bool vec_ok(const void* logits, int V, int dtype) {
  return aligned(logits, 16) && (size_t(V) * elem_bytes(dtype)) % 16 == 0;
}

// Pass 1 partials of the sampling accept over `rows` rows: the chunked
// partials, or a row's statistics and the streaming pass's records.
size_t sampling_pass1_bytes(long rows, int V) {
  size_t bytes = sampling_partial_bytes(int(rows), chunk_bound(rows, V));
  for (int vec : {4, 8}) {  // fp32 and bf16 rows
    if (V % vec) continue;
    const StreamGeometry g = stream_geometry(rows, V, vec, 152);  // (the records do not depend on the SM count)
    const size_t s = g.ctas > 0 ? sampling_partial_bytes(int(rows), 1) + g.bytes : 0;
    if (s > bytes) bytes = s;
  }
  return bytes;
}

// Greedy accept's per-chunk argmax partials.
size_t greedy_part_bytes(int b, int n, int V) { return align256(size_t(b) * n * greedy_split(long(b) * n, V, 1).chunks * 8); }

// The select's partials start past the largest area the KV commit uses (its
// staged free lists and counts, for any tree of at most kMaxN nodes), so that
// a select may also overlap a commit before it.
size_t select_base_bytes(int b) { return align256(size_t(b) * (kMaxN + 1) * 4); }

// SMs of the current device (152, a GB300's, when no device answers: the
// workspace size is then computed for that part).
int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
    cudaGetLastError();  // leave no sticky error behind
    return 152;
  }
  return sms;
}

// Partials of one select launch of `rows` rows: the chunked layout, or the
// streaming layout (rows x pieces) when the rows are 16-byte vectors.
size_t select_launch_bytes(long rows, int V) {
  const size_t chunked = select_partial_bytes(int(rows), select_split(rows, V, 1).chunks);
  size_t streamed = 0;
  for (int vec : {4, 8}) {  // fp32 and bf16 rows
    if (V % vec) continue;
    const StreamGeometry g = select_stream_geometry(rows, V, vec, device_sms());
    if (g.bytes > streamed) streamed = g.bytes;
  }
  return chunked > streamed ? chunked : streamed;
}

// One half of the select partials: the larger of step 0 (b rows) and a
// later step (b*k rows).
size_t select_half_bytes(int b, int k, int V) {
  const size_t a = select_launch_bytes(b, V);
  const size_t c = select_launch_bytes(long(b) * k, V);
  return a > c ? a : c;
}

size_t partial_bytes(int op, int b, int n, int k, int V, int Hq, int Hkv, int max_seq_len) {
  switch (op) {
    case SPEC_OP_SELECT_TOPK:
      return select_base_bytes(b) + 2 * select_half_bytes(b, k, V);
    case SPEC_OP_BUILD_TREE:
      return 0;
    case SPEC_OP_VERIFY_GREEDY:  // after the attention's merge region (see spec_verify_greedy)
      return attention_partial_bytes() + greedy_part_bytes(b, n, V);
    case SPEC_OP_VERIFY_SAMPLING:
    case SPEC_OP_VERIFY_TARGET_ONLY:
      return sampling_pass1_bytes(long(b) * n, V) + sampling_state_bytes(b) +
             sampling_partial2_bytes(b, terminal_split(V).chunks);
    case SPEC_OP_VERIFY_ATTENTION:
      return attention_partial_bytes();
    case SPEC_OP_COMMIT_KV:
      return commit_partial_bytes(b, n);
    default:
      return 0;
  }
}

// Per workspace: whether the caller has allowed overlap with the call before
// (spec_workspace_set_overlap; off by default), whether the last call enqueued
// on it was a select, and the half (of the select partials and counters) that
// select used.  With overlap allowed, a select enqueued right after another
// select, or after a KV commit, on the same workspace takes the other half and
// runs its chunk pass before waiting on that call (programmatic dependent
// launch; neither touches the select's area), and greedy accept right after
// the verify attention scans its logits before waiting.  Otherwise every
// kernel waits for the kernel before it -- whatever produced it -- before it
// reads anything.  The workspace layout depends on the batch size, so a call
// overlaps the one before it only when both have the same b.  Every kernel
// lets its successor start only after its own wait, so a kernel overlaps only
// the one kernel before it.
struct WsState {
  bool overlap = false;
  bool last_select = false;
  bool last_attention = false;
  bool last_commit = false;
  int half = 1;
  int b = -1;  // batch size of the last call
};
std::mutex g_ws_mu;
std::unordered_map<const void*, WsState> g_ws_state;

enum class Call { kOther, kAttention, kCommit };
void note_other(const void* ws, Call call = Call::kOther, int b = -1) {
  std::lock_guard<std::mutex> lock(g_ws_mu);
  if (call == Call::kOther) {
    auto it = g_ws_state.find(ws);
    if (it != g_ws_state.end()) it->second.last_select = it->second.last_attention = it->second.last_commit = false;
    return;
  }
  WsState& st = g_ws_state[ws];
  st.last_select = false;
  st.last_attention = call == Call::kAttention;
  st.last_commit = call == Call::kCommit;
  st.b = b;
}

// whether greedy accept of batch size b may scan before waiting: overlap is
// allowed and the last call enqueued on ws was the verify attention with the
// same batch size (the record is cleared either way)
bool take_after_attention(const void* ws, int b) {
  std::lock_guard<std::mutex> lock(g_ws_mu);
  auto it = g_ws_state.find(ws);
  if (it == g_ws_state.end()) return false;
  const bool r = it->second.overlap && it->second.last_attention && it->second.b == b;
  it->second.last_select = it->second.last_attention = it->second.last_commit = false;
  return r;
}

// (early, half) for a select of batch size b about to be enqueued on ws
std::pair<bool, int> take_select(const void* ws, int b) {
  std::lock_guard<std::mutex> lock(g_ws_mu);
  WsState& st = g_ws_state[ws];
  const bool early = st.overlap && (st.last_select || st.last_commit) && st.b == b;
  st.half ^= 1;
  st.last_select = true;
  st.last_attention = st.last_commit = false;
  st.b = b;
  return {early, st.half};
}

// forget everything recorded for ws (overlap back to off)
void reset_state(const void* ws) {
  std::lock_guard<std::mutex> lock(g_ws_mu);
  g_ws_state.erase(ws);
}

int check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws || !aligned(ws, 256)) return SPEC_ERR_WORKSPACE;
  if (ws_bytes < need) return SPEC_ERR_WORKSPACE;
  return SPEC_OK;
}

// compact: the no-allocation layout (partials straight after the counters,
// never early).  Otherwise the partials sit after the attention's merge
// region, and the scan runs before waiting on the kernel ahead when that
// kernel is the verify attention on this workspace.
int greedy_call(bool compact, int b, int n, int S, int V, int dtype, const void* logits,
                const int32_t* draft_tokens, const int32_t* retrieve_index, const int32_t* next_token,
                const int32_t* next_sibling, int32_t* predict, int32_t* accept_index, int32_t* accept_lens,
                int32_t* accepted_tokens, int32_t* next_root, void* ws, size_t ws_bytes, void* stream) {
  if (b < 0 || n < 1 || n > kMaxN || S < 1 || V < 1) return SPEC_ERR_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (b == 0) return SPEC_OK;
  if (!logits || !draft_tokens || !retrieve_index || !next_token || !next_sibling || !predict || !accept_index ||
      !accept_lens)
    return SPEC_ERR_ARG;
  const size_t need = compact ? kHeaderBytes + counters_bytes(b) + greedy_part_bytes(b, n, V)
                              : spec_workspace_size(SPEC_OP_VERIFY_GREEDY, b, n, 1, V, 0, 0, 0);
  if (int rc = check_ws(ws, ws_bytes, need)) return rc;
  const bool early = !compact && take_after_attention(ws, b);
  if (compact) note_other(ws);
  const WsView v = ws_view(ws, b);
  GreedyParams p{};
  p.b = b;
  p.n = n;
  p.S = S;
  p.V = V;
  p.dtype = dtype;
  p.logits = logits;
  p.draft_tokens = draft_tokens;
  p.retrieve_index = retrieve_index;
  p.next_token = next_token;
  p.next_sibling = next_sibling;
  p.predict = predict;
  p.accept_index = accept_index;
  p.accept_lens = accept_lens;
  p.accepted_tokens = accepted_tokens;
  p.next_root = next_root;
  const RowSplit sp = greedy_split(long(b) * n, V, vec_elems(dtype));
  p.chunks = sp.chunks;
  p.chunk_elems = sp.chunk_elems;
  p.vec_ok = vec_ok(logits, V, dtype);
  p.early = early;
  p.error = v.error;
  p.counters = v.counters + greedy_counter_base(b);
  p.partials = v.partials + (compact ? 0 : attention_partial_bytes());
  return launch_verify_greedy(p, as_stream(stream));
}

// The chain's greedy accept (DSpark counts), on greedy accept's workspace
// layout and overlap rule.
int chain_call(int b, int S, int V, int dtype, const void* logits, const int32_t* draft_tokens, int draft_ld,
               const int32_t* prefix_lens, int32_t* correct_len, int32_t* bonus, int32_t* out_tokens,
               int32_t* commit_lens, int32_t* new_seq_lens, int32_t* accept_index, void* ws, size_t ws_bytes,
               void* stream) {
  const int n = S + 1;
  if (b < 0 || S < 1 || n > kMaxN || V < 1 || draft_ld < S) return SPEC_ERR_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (b == 0) return SPEC_OK;
  if (!logits || !draft_tokens || !prefix_lens || !correct_len || !bonus || !out_tokens || !commit_lens ||
      !new_seq_lens)
    return SPEC_ERR_ARG;
  const size_t need = spec_workspace_size(SPEC_OP_VERIFY_GREEDY, b, n, 1, V, 0, 0, 0);
  if (int rc = check_ws(ws, ws_bytes, need)) return rc;
  const bool early = take_after_attention(ws, b);
  const WsView v = ws_view(ws, b);
  GreedyParams p{};
  p.b = b;
  p.n = n;
  p.S = S;
  p.V = V;
  p.dtype = dtype;
  p.logits = logits;
  p.chain = 1;
  p.draft_ld = draft_ld;
  p.chain_drafts = draft_tokens;
  p.prefix_lens = prefix_lens;
  p.correct_len = correct_len;
  p.bonus = bonus;
  p.out_tokens = out_tokens;
  p.commit_lens = commit_lens;
  p.new_seq_lens = new_seq_lens;
  p.accept_index = accept_index;
  const RowSplit sp = greedy_split(long(b) * n, V, vec_elems(dtype));
  p.chunks = sp.chunks;
  p.chunk_elems = sp.chunk_elems;
  p.vec_ok = vec_ok(logits, V, dtype);
  p.early = early;
  p.error = v.error;
  p.counters = v.counters + greedy_counter_base(b);
  p.partials = v.partials + attention_partial_bytes();
  return launch_verify_greedy(p, as_stream(stream));
}

}  // namespace

extern "C" {

int spec_build_chain_tree(int b, int S, const int32_t* bonus, const int32_t* draft_tokens, int draft_ld,
                          const int32_t* seq_lens, int32_t* tree_tokens, int32_t* positions, int32_t* retrieve_index,
                          int32_t* next_token, int32_t* next_sibling, uint64_t* mask_bits, void* stream) {
  if (b < 0 || S < 1 || S + 1 > kMaxN || draft_ld < S) return SPEC_ERR_ARG;
  if (b == 0) return SPEC_OK;
  if (!bonus || !draft_tokens || !seq_lens || !tree_tokens || !positions || !retrieve_index || !next_token ||
      !next_sibling || !mask_bits)
    return SPEC_ERR_ARG;
  ChainParams p{};
  p.b = b;
  p.S = S;
  p.draft_ld = draft_ld;
  p.bonus = bonus;
  p.draft_tokens = draft_tokens;
  p.seq_lens = seq_lens;
  p.tree_tokens = tree_tokens;
  p.positions = positions;
  p.retrieve_index = retrieve_index;
  p.next_token = next_token;
  p.next_sibling = next_sibling;
  p.mask_bits = mask_bits;
  return launch_build_chain_tree(p, as_stream(stream));
}

int spec_verify_chain_greedy(int b, int S, int V, int dtype, const void* logits, const int32_t* draft_tokens,
                             int draft_ld, const int32_t* prefix_lens, int32_t* correct_len, int32_t* bonus,
                             int32_t* out_tokens, int32_t* commit_lens, int32_t* new_seq_lens,
                             int32_t* accept_index, void* ws, size_t ws_bytes, void* stream) {
  return chain_call(b, S, V, dtype, logits, draft_tokens, draft_ld, prefix_lens, correct_len, bonus, out_tokens,
                    commit_lens, new_seq_lens, accept_index, ws, ws_bytes, stream);
}

int spec_add_penalties(int b, int n, int V, int dtype, void* logits, const float* penalties, void* stream) {
  if (b < 0 || n < 1 || V < 1) return SPEC_ERR_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (b == 0) return SPEC_OK;
  if (!logits || !penalties) return SPEC_ERR_ARG;
  // 16-byte vectors of logits and of penalties
  if (!vec_ok(logits, V, dtype) || !aligned(penalties, 16) || V % 8) return SPEC_ERR_UNSUPPORTED;
  PenaltyParams p{};
  p.b = b;
  p.n = n;
  p.V = V;
  p.dtype = dtype;
  p.logits = logits;
  p.penalties = penalties;
  return launch_add_penalties(p, as_stream(stream));
}

int spec_renorm_probs(int b, int n, int V, int dtype, const void* logits, const float* temperatures,
                      const int32_t* top_k, const float* top_p, float* probs, void* stream) {
  if (b < 0 || n < 1 || V < 1 || int64_t(b) * n >= (int64_t(1) << 31)) return SPEC_ERR_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (b == 0) return SPEC_OK;
  if (!logits || !temperatures || !top_k || !top_p || !probs) return SPEC_ERR_ARG;
  RenormParams p{};
  p.b = b;
  p.n = n;
  p.V = V;
  p.dtype = dtype;
  p.logits = logits;
  p.temperatures = temperatures;
  p.top_k = top_k;
  p.top_p = top_p;
  p.probs = probs;
  return launch_renorm(p, as_stream(stream));
}

int spec_assign_draft_locs(int b, int topk, int S, int page_size, const int32_t* req_to_token, int req_rows,
                           int row_w, const int32_t* req_pool_idx, const int32_t* seq_lens, int64_t num_slots,
                           int32_t* out_cache_loc, int32_t* positions, void* ws, size_t ws_bytes, void* stream) {
  if (b < 0 || topk < 1 || topk > kMaxK || S < 1 || page_size < 1 || req_rows < 1 || row_w < 1 || num_slots < 1)
    return SPEC_ERR_ARG;
  if (int64_t(b) * topk * S >= (int64_t(1) << 31)) return SPEC_ERR_ARG;
  if (b == 0) return SPEC_OK;
  if (!req_to_token || !req_pool_idx || !seq_lens || !out_cache_loc) return SPEC_ERR_ARG;
  if (int rc = check_ws(ws, ws_bytes, kHeaderBytes)) return rc;
  note_other(ws);
  DraftLocParams p{};
  p.b = b;
  p.topk = topk;
  p.S = S;
  p.page_size = page_size;
  p.req_to_token = req_to_token;
  p.req_rows = req_rows;
  p.row_w = row_w;
  p.req_pool_idx = req_pool_idx;
  p.seq_lens = seq_lens;
  p.num_slots = num_slots;
  p.out_cache_loc = out_cache_loc;
  p.positions = topk == 1 ? positions : nullptr;
  p.error = ws_view(ws, b).error;
  return launch_assign_draft_locs(p, as_stream(stream));
}

int spec_duplicate_prefix_tail(int b, int topk, int S, int page_size, int Hkv, int D, int num_layers,
                               void* const* k_layers, void* const* v_layers, int64_t num_slots,
                               const int32_t* req_to_token, int req_rows, int row_w, const int32_t* req_pool_idx,
                               const int32_t* seq_lens, void* ws, size_t ws_bytes, void* stream) {
  if (b < 0 || topk < 1 || topk > kMaxK || S < 1 || page_size < 1 || Hkv < 1) return SPEC_ERR_ARG;
  if (page_size > 64) return SPEC_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return SPEC_ERR_UNSUPPORTED;
  if (num_layers < 1 || num_layers > kMaxLayers || num_slots < 1 || req_rows < 1 || row_w < 1) return SPEC_ERR_ARG;
  if (b == 0 || topk == 1 || page_size == 1) return SPEC_OK;  // no holes to fill
  if (!k_layers || !v_layers || !req_to_token || !req_pool_idx || !seq_lens) return SPEC_ERR_ARG;
  if (int rc = check_ws(ws, ws_bytes, kHeaderBytes)) return rc;
  DupTailParams p{};
  p.b = b;
  p.topk = topk;
  p.S = S;
  p.page_size = page_size;
  p.Hkv = Hkv;
  p.D = D;
  p.num_layers = num_layers;
  for (int i = 0; i < num_layers; ++i) {
    if (!k_layers[i] || !v_layers[i] || !aligned(k_layers[i], 16) || !aligned(v_layers[i], 16)) return SPEC_ERR_ARG;
    p.k_layers[i] = k_layers[i];
    p.v_layers[i] = v_layers[i];
  }
  note_other(ws);
  p.num_slots = num_slots;
  p.req_to_token = req_to_token;
  p.req_rows = req_rows;
  p.row_w = row_w;
  p.req_pool_idx = req_pool_idx;
  p.seq_lens = seq_lens;
  p.error = ws_view(ws, b).error;
  return launch_duplicate_prefix_tail(p, as_stream(stream));
}

int spec_build_full_mask(int b, int n, const int32_t* seq_lens, const uint64_t* mask_bits, int fill_prefix,
                         uint8_t* mask, size_t mask_bytes, void* ws, size_t ws_bytes, void* stream) {
  if (b < 0 || b > 16384 || n < 1 || n > kMaxN || (fill_prefix != 0 && fill_prefix != 1)) return SPEC_ERR_ARG;
  if (b == 0) return SPEC_OK;
  if (!seq_lens || !mask_bits || !mask) return SPEC_ERR_ARG;
  if (int rc = check_ws(ws, ws_bytes, kHeaderBytes)) return rc;
  note_other(ws);
  FullMaskParams p{};
  p.b = b;
  p.n = n;
  p.fill_prefix = fill_prefix;
  p.seq_lens = seq_lens;
  p.mask_bits = mask_bits;
  p.mask = mask;
  p.mask_bytes = mask_bytes;
  p.error = ws_view(ws, b).error;
  return launch_full_mask(p, as_stream(stream));
}

size_t spec_workspace_size(int op, int b, int n, int k, int V, int Hq, int Hkv, int max_seq_len) {
  if (b < 0 || op < 0 || op > SPEC_OP_LAST) return 0;
  if (b == 0) return kHeaderBytes + counters_bytes(0);
  if (n < 1 || n > kMaxN || k < 1 || k > kMaxK || V < 1) return 0;
  if (op == SPEC_OP_VERIFY_ATTENTION && (Hq < 1 || Hkv < 1 || Hq % Hkv || max_seq_len < 0)) return 0;
  return kHeaderBytes + counters_bytes(b) + partial_bytes(op, b, n, k, V, Hq, Hkv, max_seq_len);
}

int spec_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws) return SPEC_ERR_WORKSPACE;
  reset_state(ws);
  return cudaMemsetAsync(ws, 0, ws_bytes, as_stream(stream)) == cudaSuccess ? SPEC_OK : SPEC_ERR_LAUNCH;
}

int spec_workspace_set_overlap(void* ws, int enable) {
  if (!ws) return SPEC_ERR_WORKSPACE;
  if (enable != 0 && enable != 1) return SPEC_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_ws_mu);
  g_ws_state[ws].overlap = enable != 0;
  return SPEC_OK;
}

int spec_last_error(void* ws, void* stream) {
  if (!ws) return SPEC_ERR_WORKSPACE;
  uint32_t word = 0;
  cudaStream_t s = as_stream(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return SPEC_ERR_LAUNCH;
  if (cudaMemcpy(&word, ws, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return SPEC_ERR_LAUNCH;
  if (cudaMemsetAsync(ws, 0, sizeof word, s) != cudaSuccess) return SPEC_ERR_LAUNCH;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SPEC_ERR_LAUNCH;
  return int(word & 0x7fffffffu);
}

int spec_device_sm_count(void) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

int spec_select_topk(int step, int b, int k, int V, int dtype, const void* draft_logits, float temperature,
                     const float* scores_in, float* score_blk, int32_t* token_blk, int score_ld,
                     int32_t* parent_blk, int parent_ld, float* scores_out, int32_t* next_input_ids,
                     float* topk_p_out, void* ws, size_t ws_bytes, void* stream) {
  if (b < 0 || step < 0 || k < 1 || k > kMaxK || V < k) return SPEC_ERR_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (!(temperature > 0.f)) return SPEC_ERR_ARG;
  if (b == 0) return SPEC_OK;
  if (!draft_logits || !score_blk || !token_blk || !scores_out || !next_input_ids) return SPEC_ERR_ARG;
  if (step > 0 && !scores_in) return SPEC_ERR_ARG;
  if (score_ld < (step ? k * k : k)) return SPEC_ERR_ARG;
  if (parent_blk && parent_ld < (step ? k : k + 1)) return SPEC_ERR_ARG;
  const size_t need = spec_workspace_size(SPEC_OP_SELECT_TOPK, b, 1, k, V, 0, 0, 0);
  if (int rc = check_ws(ws, ws_bytes, need)) return rc;
  const WsView v = ws_view(ws, b);
  SelectParams p{};
  p.step = step;
  p.b = b;
  p.k = k;
  p.V = V;
  p.dtype = dtype;
  p.logits = draft_logits;
  p.temperature = temperature;
  p.scores_in = scores_in;
  p.score_blk = score_blk;
  p.token_blk = token_blk;
  p.score_ld = score_ld;
  p.parent_blk = parent_blk;
  p.parent_ld = parent_ld;
  p.scores_out = scores_out;
  p.next_ids = next_input_ids;
  p.topk_p_out = topk_p_out;
  p.rows = b * (step ? k : 1);
  const RowSplit sp = select_split(p.rows, V, vec_elems(dtype));
  if (sp.chunks > kMaxChunks || sp.chunk_elems > kSelectChunkMax) return SPEC_ERR_UNSUPPORTED;
  p.chunks = sp.chunks;
  p.chunk_elems = sp.chunk_elems;
  p.vec_ok = vec_ok(draft_logits, V, dtype);
  // rows of whole 16-byte vectors, at least kStreamMinBytes of them: the
  // streaming pass and the request step (below that the chunked kernel, one
  // launch with its finalize inside, is faster)
  if (p.vec_ok && size_t(p.rows) * size_t(V) * elem_bytes(dtype) >= kStreamMinBytes) {
    const StreamGeometry g = select_stream_geometry(p.rows, V, vec_elems(dtype), device_sms());
    p.stream_ctas = g.ctas;
    p.stream_nb = g.nb;
  }
  p.error = v.error;
  const std::pair<bool, int> eh = take_select(ws, b);
  p.early = eh.first;
  p.half = eh.second;
  p.counters = v.counters + 1 + size_t(eh.second) * b;  // word 0 is the commit's
  p.queue = v.counters + 1 + 2 * size_t(b) + eh.second;
  p.partials = v.partials + select_base_bytes(b) + size_t(eh.second) * select_half_bytes(b, k, V);
  return launch_select_topk(p, as_stream(stream));
}

int spec_build_tree(int b, int k, int S, int n, const float* score_space, const int32_t* token_space,
                    const int32_t* parent_space, const int32_t* bonus, const int32_t* seq_lens,
                    int32_t* draft_tokens, int32_t* positions, int32_t* retrieve_index, int32_t* next_token,
                    int32_t* next_sibling, uint64_t* mask_bits, void* ws, size_t ws_bytes, void* stream) {
  if (b < 0 || k < 1 || k > kMaxK || S < 1 || n < 1 || n > kMaxN) return SPEC_ERR_ARG;
  const long C = long(k) + long(S - 1) * k * k;
  if (n - 1 > C || C > 16384) return SPEC_ERR_ARG;
  if (b == 0) return SPEC_OK;
  if (!score_space || !token_space || !parent_space || !bonus || !seq_lens || !draft_tokens || !positions ||
      !retrieve_index || !next_token || !next_sibling || !mask_bits)
    return SPEC_ERR_ARG;
  if (int rc = check_ws(ws, ws_bytes, kHeaderBytes)) return rc;
  note_other(ws);
  BuildParams p{};
  p.b = b;
  p.k = k;
  p.S = S;
  p.n = n;
  p.score_space = score_space;
  p.token_space = token_space;
  p.parent_space = parent_space;
  p.bonus = bonus;
  p.seq_lens = seq_lens;
  p.draft_tokens = draft_tokens;
  p.positions = positions;
  p.retrieve_index = retrieve_index;
  p.next_token = next_token;
  p.next_sibling = next_sibling;
  p.mask_bits = mask_bits;
  p.error = ws_view(ws, b).error;
  return launch_build_tree(p, as_stream(stream));
}

int spec_verify_attention(int b, int n, int Hq, int Hkv, int D, int page_size, const void* q, const void* k_pool,
                          const void* v_pool, int64_t num_slots, const int32_t* req_to_token, int req_rows,
                          int row_w, const int32_t* req_pool_idx, const int32_t* seq_lens, int max_seq_len,
                          const int32_t* verify_loc, const uint64_t* mask_bits, float scale, void* out,
                          float* lse, void* ws, size_t ws_bytes, void* stream) {
  if (b < 0 || n < 1 || n > kMaxN || Hq < 1 || Hkv < 1 || Hq % Hkv || page_size < 1) return SPEC_ERR_ARG;
  if (D != 64 && D != 128) return SPEC_ERR_UNSUPPORTED;
  if (num_slots < 1 || req_rows < 1 || row_w < 1 || max_seq_len < 0) return SPEC_ERR_ARG;
  // TMA row coordinates of the gathers (slot * Hkv + head, node rows * Hq) are int32
  if (num_slots * Hkv >= (int64_t(1) << 31) || int64_t(b) * n * Hq >= (int64_t(1) << 31)) return SPEC_ERR_ARG;
  if (b == 0) return SPEC_OK;
  if (!q || !k_pool || !v_pool || !req_to_token || !req_pool_idx || !seq_lens || !verify_loc || !mask_bits || !out)
    return SPEC_ERR_ARG;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16)) return SPEC_ERR_ARG;
  const size_t need = spec_workspace_size(SPEC_OP_VERIFY_ATTENTION, b, n, 1, 1, Hq, Hkv, max_seq_len);
  if (int rc = check_ws(ws, ws_bytes, need)) return rc;
  note_other(ws, Call::kAttention, b);
  const WsView v = ws_view(ws, b);
  AttentionParams p{};
  p.b = b;
  p.n = n;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.D = D;
  p.page_size = page_size;
  p.q = q;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.num_slots = num_slots;
  p.req_to_token = req_to_token;
  p.req_rows = req_rows;
  p.row_w = row_w;
  p.req_pool_idx = req_pool_idx;
  p.seq_lens = seq_lens;
  p.max_seq_len = max_seq_len;
  p.verify_loc = verify_loc;
  p.mask_bits = mask_bits;
  p.scale = scale;
  p.out = out;
  p.lse = lse;
  const TcGeometry geo = attention_tc_geometry(b, n, Hq, Hkv, max_seq_len);
  p.splits = geo.splits;
  p.error = v.error;
  p.counters = v.counters;
  p.partials = v.partials;
  return launch_attention_tc(p, geo, as_stream(stream));
}

int spec_verify_greedy(int b, int n, int S, int V, int dtype, const void* logits, const int32_t* draft_tokens,
                       const int32_t* retrieve_index, const int32_t* next_token, const int32_t* next_sibling,
                       int32_t* predict, int32_t* accept_index, int32_t* accept_lens, int32_t* accepted_tokens,
                       int32_t* next_root, void* ws, size_t ws_bytes, void* stream) {
  return greedy_call(false, b, n, S, V, dtype, logits, draft_tokens, retrieve_index, next_token, next_sibling,
                     predict, accept_index, accept_lens, accepted_tokens, next_root, ws, ws_bytes, stream);
}

}  // extern "C"

namespace {

// Both samplers: the classic p/q rejection sampler (draft_probs given) or the
// target-only tree sampler (thresholds given, draft_probs unused).
int sampling_call(bool target_only, int b, int n, int S, int V, int dtype, const void* logits, const float* probs,
                  const float* draft_probs, const float* temperatures, const float* u, const float* u_final,
                  float thr_single, float thr_acc, const int32_t* draft_tokens, const int32_t* retrieve_index,
                  const int32_t* next_token, const int32_t* next_sibling, int32_t* predict, int32_t* accept_index,
                  int32_t* accept_lens, int32_t* accepted_tokens, int32_t* next_root, void* ws, size_t ws_bytes,
                  void* stream) {
  if (b < 0 || n < 1 || n > kMaxN || S < 1 || V < 1) return SPEC_ERR_ARG;
  if (target_only && !(thr_single > 0.f && thr_single <= 1.f && thr_acc > 0.f && thr_acc <= 1.f))
    return SPEC_ERR_ARG;
  if (probs) dtype = SPEC_F32;  // the probabilities mode reads fp32 probabilities, no logits
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (b == 0) return SPEC_OK;
  if ((!logits && !probs) || (!target_only && !draft_probs) || (!probs && !temperatures) || !u || !u_final ||
      !draft_tokens || !retrieve_index || !next_token || !next_sibling || !predict || !accept_index || !accept_lens)
    return SPEC_ERR_ARG;
  const size_t need = spec_workspace_size(target_only ? SPEC_OP_VERIFY_TARGET_ONLY : SPEC_OP_VERIFY_SAMPLING, b,
                                          n, 1, V, 0, 0, 0);
  if (int rc = check_ws(ws, ws_bytes, need)) return rc;
  note_other(ws);
  const WsView v = ws_view(ws, b);
  SamplingParams p{};
  p.b = b;
  p.n = n;
  p.S = S;
  p.V = V;
  p.dtype = dtype;
  p.logits = probs ? static_cast<const void*>(probs) : logits;  // (not read in the probabilities mode)
  p.probs = probs;
  p.target_only = target_only ? 1 : 0;
  p.thr_single = thr_single;
  p.thr_acc = thr_acc;
  p.draft_probs = target_only ? nullptr : draft_probs;
  p.temperatures = temperatures;
  p.u = u;
  p.u_final = u_final;
  p.draft_tokens = draft_tokens;
  p.retrieve_index = retrieve_index;
  p.next_token = next_token;
  p.next_sibling = next_sibling;
  p.predict = predict;
  p.accept_index = accept_index;
  p.accept_lens = accept_lens;
  p.accepted_tokens = accepted_tokens;
  p.next_root = next_root;
  // the probabilities mode has no row statistics to gather: one CTA a row
  const RowSplit s1 = probs ? RowSplit{1, V} : pick_split(long(b) * n, V, vec_elems(dtype));
  const RowSplit s2 = terminal_split(V);
  if (s2.chunks > kMaxChunks2) return SPEC_ERR_UNSUPPORTED;
  p.chunks = s1.chunks;
  p.chunk_elems = s1.chunk_elems;
  p.chunks2 = s2.chunks;
  p.chunk2_elems = s2.chunk_elems;
  {  // terminal-pass CTAs a request: a CTA a chunk up to four waves of two
     // CTAs a SM; past that one wave, each CTA looping over its chunks
     // (measured: 32 requests x 32 chunks faster as 1024 CTAs, 256 x 32
     // as 512)
    const long wave = 2L * device_sms();
    const long per = long(b) * s2.chunks <= 4 * wave ? s2.chunks : (wave + b - 1) / b;
    p.term_ctas = int(per < 1 ? 1 : per > s2.chunks ? s2.chunks : per);
  }
  p.vec_ok = vec_ok(logits, V, dtype);
  p.vec_term = !probs && V % 16 == 0 && s2.chunk_elems % 16 == 0 && aligned(logits, 16) &&
               (target_only || aligned(draft_probs, 16));
  if (!probs && p.vec_ok) {  // logit rows of whole 16-byte vectors: the streaming pass, where it applies
    const StreamGeometry g = stream_geometry(long(b) * n, V, vec_elems(dtype), device_sms());
    if (g.ctas > 0) {
      p.stream_ctas = g.ctas;
      p.stream_nu = g.nb;
      p.usum = reinterpret_cast<float2*>(v.partials + sampling_partial_bytes(b * n, 1));
      p.queue = v.counters + sampling_queue_word(b);
    }
  }
  p.error = v.error;
  p.counters = v.counters;
  p.partials = v.partials;
  p.state = v.partials + sampling_pass1_bytes(long(b) * n, V);
  p.partials2 = p.state + sampling_state_bytes(b);
  return launch_verify_sampling(p, as_stream(stream));
}

}  // namespace

extern "C" {

int spec_verify_sampling(int b, int n, int S, int V, int dtype, const void* logits, const float* draft_probs,
                         const float* temperatures, const float* u, const float* u_final,
                         const int32_t* draft_tokens, const int32_t* retrieve_index, const int32_t* next_token,
                         const int32_t* next_sibling, int32_t* predict, int32_t* accept_index,
                         int32_t* accept_lens, int32_t* accepted_tokens, int32_t* next_root, void* ws,
                         size_t ws_bytes, void* stream) {
  return sampling_call(false, b, n, S, V, dtype, logits, nullptr, draft_probs, temperatures, u, u_final, 1.f, 1.f,
                       draft_tokens, retrieve_index, next_token, next_sibling, predict, accept_index, accept_lens,
                       accepted_tokens, next_root, ws, ws_bytes, stream);
}

int spec_verify_target_only(int b, int n, int S, int V, int dtype, const void* logits, const float* temperatures,
                            const float* coins, const float* u_final, float threshold_single, float threshold_acc,
                            const int32_t* draft_tokens, const int32_t* retrieve_index, const int32_t* next_token,
                            const int32_t* next_sibling, int32_t* predict, int32_t* accept_index,
                            int32_t* accept_lens, int32_t* accepted_tokens, int32_t* next_root, void* ws,
                            size_t ws_bytes, void* stream) {
  return sampling_call(true, b, n, S, V, dtype, logits, nullptr, nullptr, temperatures, coins, u_final, threshold_single,
                       threshold_acc, draft_tokens, retrieve_index, next_token, next_sibling, predict, accept_index,
                       accept_lens, accepted_tokens, next_root, ws, ws_bytes, stream);
}

int spec_verify_sampling_probs(int b, int n, int S, int V, const float* probs, const float* draft_probs,
                               const float* u, const float* u_final, const int32_t* draft_tokens,
                               const int32_t* retrieve_index, const int32_t* next_token, const int32_t* next_sibling,
                               int32_t* predict, int32_t* accept_index, int32_t* accept_lens,
                               int32_t* accepted_tokens, int32_t* next_root, void* ws, size_t ws_bytes,
                               void* stream) {
  if (!probs && b > 0) return SPEC_ERR_ARG;
  return sampling_call(false, b, n, S, V, SPEC_F32, nullptr, probs, draft_probs, nullptr, u, u_final, 1.f, 1.f,
                       draft_tokens, retrieve_index, next_token, next_sibling, predict, accept_index, accept_lens,
                       accepted_tokens, next_root, ws, ws_bytes, stream);
}

int spec_verify_target_only_probs(int b, int n, int S, int V, const float* probs, const float* coins,
                                  const float* u_final, float threshold_single, float threshold_acc,
                                  const int32_t* draft_tokens, const int32_t* retrieve_index,
                                  const int32_t* next_token, const int32_t* next_sibling, int32_t* predict,
                                  int32_t* accept_index, int32_t* accept_lens, int32_t* accepted_tokens,
                                  int32_t* next_root, void* ws, size_t ws_bytes, void* stream) {
  if (!probs && b > 0) return SPEC_ERR_ARG;
  return sampling_call(true, b, n, S, V, SPEC_F32, nullptr, probs, nullptr, nullptr, coins, u_final,
                       threshold_single, threshold_acc, draft_tokens, retrieve_index, next_token, next_sibling,
                       predict, accept_index, accept_lens, accepted_tokens, next_root, ws, ws_bytes, stream);
}


int spec_commit_kv(int b, int n, int W, int Hkv, int D, int num_layers, int page_size, void* const* k_layers,
                   void* const* v_layers, int64_t num_slots, const int32_t* req_to_token, int req_rows, int row_w,
                   const int32_t* req_pool_idx, const int32_t* seq_lens, const int32_t* verify_loc,
                   const int32_t* accept_index, const int32_t* accept_lens, int32_t* new_seq_lens,
                   int32_t* free_ids, int32_t* n_free, void* ws, size_t ws_bytes, void* stream) {
  if (b < 0 || n < 1 || n > kMaxN || W < 1 || W > kMaxN + 1 || Hkv < 1 || page_size < 1) return SPEC_ERR_ARG;
  if (D != 64 && D != 128) return SPEC_ERR_UNSUPPORTED;
  if (num_layers < 1 || num_layers > kMaxLayers || num_slots < 1 || req_rows < 1 || row_w < 1) return SPEC_ERR_ARG;
  if (b == 0) return SPEC_OK;
  if (!k_layers || !v_layers || !req_to_token || !req_pool_idx || !seq_lens || !verify_loc || !accept_index ||
      !accept_lens || !new_seq_lens || !free_ids || !n_free)
    return SPEC_ERR_ARG;
  const size_t need = spec_workspace_size(SPEC_OP_COMMIT_KV, b, n, 1, 1, 0, 0, 0);
  if (int rc = check_ws(ws, ws_bytes, need)) return rc;
  note_other(ws, Call::kCommit, b);
  const WsView v = ws_view(ws, b);
  CommitParams p{};
  p.b = b;
  p.n = n;
  p.W = W;
  p.Hkv = Hkv;
  p.D = D;
  p.num_layers = num_layers;
  p.page_size = page_size;
  for (int i = 0; i < num_layers; ++i) {
    if (!k_layers[i] || !v_layers[i] || !aligned(k_layers[i], 16) || !aligned(v_layers[i], 16)) return SPEC_ERR_ARG;
    p.k_layers[i] = k_layers[i];
    p.v_layers[i] = v_layers[i];
  }
  p.num_slots = num_slots;
  p.req_to_token = req_to_token;
  p.req_rows = req_rows;
  p.row_w = row_w;
  p.req_pool_idx = req_pool_idx;
  p.seq_lens = seq_lens;
  p.verify_loc = verify_loc;
  p.accept_index = accept_index;
  p.accept_lens = accept_lens;
  p.new_seq_lens = new_seq_lens;
  p.free_ids = free_ids;
  p.n_free = n_free;
  p.error = v.error;
  p.counters = v.counters;
  p.partials = v.partials;
  return launch_commit_kv(p, as_stream(stream));
}

}  // extern "C"

namespace spec {

size_t greedy_compact_bytes(int b, int n, int V) {
  if (b < 1 || n < 1 || V < 1) return kHeaderBytes + counters_bytes(0);
  return kHeaderBytes + counters_bytes(b) + greedy_part_bytes(b, n, V);
}

int verify_greedy_compact(int b, int n, int S, int V, int dtype, const void* logits, const int32_t* draft_tokens,
                          const int32_t* retrieve_index, const int32_t* next_token, const int32_t* next_sibling,
                          int32_t* predict, int32_t* accept_index, int32_t* accept_lens, int32_t* accepted_tokens,
                          int32_t* next_root, void* ws, size_t ws_bytes, void* stream) {
  return greedy_call(true, b, n, S, V, dtype, logits, draft_tokens, retrieve_index, next_token, next_sibling,
                     predict, accept_index, accept_lens, accepted_tokens, next_root, ws, ws_bytes, stream);
}

}  // namespace spec
