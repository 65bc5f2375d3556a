"""Thin Python binding of libspecdec.so: one function per C-ABI entry point,
with the same names.  Argument marshalling only -- every step runs in the CUDA
kernels behind the C ABI.  Tensors are torch CUDA tensors (torch provides the
device memory and the stream); the current torch stream is used unless a
stream is given.

Importing this module loads the library and raises ``RuntimeError`` if it is
missing: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libspecdec.so")

SPEC_OK = 0
SPEC_F32, SPEC_BF16 = 0, 1
(OP_SELECT_TOPK, OP_BUILD_TREE, OP_VERIFY_ATTENTION, OP_VERIFY_GREEDY, OP_VERIFY_SAMPLING, OP_COMMIT_KV,
 OP_VERIFY_TARGET_ONLY) = range(7)
DEV_INDEX, DEV_INVARIANT, DEV_LENGTH = 1, 2, 4
_ERRORS = {-1: "bad argument", -2: "workspace too small or misaligned", -3: "CUDA launch failed",
           -4: "unsupported dtype or head size"}

EXPORTS = ["spec_workspace_size", "spec_workspace_init", "spec_workspace_set_overlap", "spec_last_error",
           "spec_device_sm_count", "spec_select_topk", "spec_build_tree", "spec_verify_attention",
           "spec_verify_greedy", "spec_verify_sampling", "spec_verify_target_only", "spec_build_chain_tree",
           "spec_verify_chain_greedy", "spec_assign_draft_locs", "spec_duplicate_prefix_tail",
           "spec_build_full_mask", "spec_add_penalties", "spec_renorm_probs", "spec_verify_sampling_probs",
           "spec_verify_target_only_probs", "spec_commit_kv", "spec_verify_greedy_noalloc",
           "spec_noalloc_last_error"]


class SpecError(RuntimeError):
    pass


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libspecdec.so is not built ({LIB_PATH}); run `python -m accept_select_top_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, Z, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_int64
    sig = {
        "spec_workspace_size": (Z, [I, I, I, I, I, I, I, I]),
        "spec_workspace_init": (I, [P, Z, P]),
        "spec_workspace_set_overlap": (I, [P, I]),
        "spec_last_error": (I, [P, P]),
        "spec_device_sm_count": (I, []),
        "spec_select_topk": (I, [I, I, I, I, I, P, F, P, P, P, I, P, I, P, P, P, P, Z, P]),
        "spec_build_tree": (I, [I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, P, Z, P]),
        "spec_verify_attention": (I, [I, I, I, I, I, I, P, P, P, L, P, I, I, P, P, I, P, P, F, P, P, P, Z, P]),
        "spec_verify_greedy": (I, [I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, Z, P]),
        "spec_verify_sampling": (I, [I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, Z, P]),
        "spec_verify_target_only": (I, [I, I, I, I, I, P, P, P, P, F, F, P, P, P, P, P, P, P, P, P, P, Z, P]),
        "spec_build_chain_tree": (I, [I, I, P, P, I, P, P, P, P, P, P, P, P]),
        "spec_verify_chain_greedy": (I, [I, I, I, I, P, P, I, P, P, P, P, P, P, P, P, Z, P]),
        "spec_assign_draft_locs": (I, [I, I, I, I, P, I, I, P, P, L, P, P, P, Z, P]),
        "spec_duplicate_prefix_tail": (I, [I, I, I, I, I, I, I, P, P, L, P, I, I, P, P, P, Z, P]),
        "spec_build_full_mask": (I, [I, I, P, P, I, P, Z, P, Z, P]),
        "spec_add_penalties": (I, [I, I, I, I, P, P, P]),
        "spec_renorm_probs": (I, [I, I, I, I, P, P, P, P, P, P]),
        "spec_verify_sampling_probs": (I, [I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, P, P, P, Z, P]),
        "spec_verify_target_only_probs": (I, [I, I, I, I, P, P, P, F, F, P, P, P, P, P, P, P, P, P, P, Z, P]),
        "spec_commit_kv": (I, [I, I, I, I, I, I, I, P, P, L, P, I, I, P, P, P, P, P, P, P, P, P, Z, P]),
        "spec_verify_greedy_noalloc": (I, [I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P]),
        "spec_noalloc_last_error": (I, [P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = _load()


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise SpecError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise SpecError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, what: str):
    if rc != SPEC_OK:
        raise SpecError(f"{what}: {_ERRORS.get(rc, rc)}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise SpecError(f"logits must be float32 or bfloat16, got {t.dtype}")


class Workspace:
    """Caller-owned scratch memory for the C ABI (a zero-filled uint8 tensor)."""

    def __init__(self, nbytes: int, device=None, stream=None):
        self.nbytes = max(int(nbytes), 256)
        self.tensor = torch.empty(self.nbytes, dtype=torch.uint8, device=device or "cuda")
        # zero-filled through the C ABI, which also forgets any earlier
        # workspace that lived at this address
        _check(LIB.spec_workspace_init(self.ptr, ctypes.c_size_t(self.nbytes), _stream(stream)),
               "spec_workspace_init")

    @property
    def ptr(self):
        return ctypes.c_void_p(self.tensor.data_ptr())

    def set_overlap(self, enable: bool):
        """Allow (or forbid) a select or greedy accept on this workspace to read
        its main input before the kernel ahead of it has finished.  Off by
        default; see spec_workspace_set_overlap for what the caller asserts."""
        _check(LIB.spec_workspace_set_overlap(self.ptr, 1 if enable else 0), "spec_workspace_set_overlap")

    def last_error(self, stream=None) -> int:
        rc = LIB.spec_last_error(self.ptr, _stream(stream))
        if rc < 0:
            _check(rc, "spec_last_error")
        return rc


def spec_workspace_size(op: int, b: int, n: int, k: int, V: int, Hq: int = 0, Hkv: int = 0,
                        max_seq_len: int = 0) -> int:
    return int(LIB.spec_workspace_size(op, b, n, k, V, Hq, Hkv, max_seq_len))


def spec_device_sm_count() -> int:
    return int(LIB.spec_device_sm_count())


def spec_select_topk(step: int, b: int, k: int, draft_logits: torch.Tensor, temperature: float,
                     scores_in: Optional[torch.Tensor], score_blk: torch.Tensor, token_blk: torch.Tensor,
                     score_ld: int, parent_blk: Optional[torch.Tensor], parent_ld: int,
                     scores_out: torch.Tensor, next_input_ids: torch.Tensor,
                     topk_p_out: Optional[torch.Tensor], ws: Workspace, stream=None):
    V = draft_logits.shape[-1]
    _check(LIB.spec_select_topk(step, b, k, V, _dtype_code(draft_logits), _ptr(draft_logits), float(temperature),
                                _ptr(scores_in), _ptr(score_blk), _ptr(token_blk), score_ld, _ptr(parent_blk),
                                parent_ld, _ptr(scores_out), _ptr(next_input_ids), _ptr(topk_p_out), ws.ptr,
                                ws.nbytes, _stream(stream)), "spec_select_topk")


def spec_build_tree(b: int, k: int, S: int, n: int, score_space, token_space, parent_space, bonus, seq_lens,
                    draft_tokens, positions, retrieve_index, next_token, next_sibling, mask_bits,
                    ws: Workspace, stream=None):
    _check(LIB.spec_build_tree(b, k, S, n, _ptr(score_space), _ptr(token_space), _ptr(parent_space), _ptr(bonus),
                               _ptr(seq_lens), _ptr(draft_tokens), _ptr(positions), _ptr(retrieve_index),
                               _ptr(next_token), _ptr(next_sibling), _ptr(mask_bits), ws.ptr, ws.nbytes,
                               _stream(stream)), "spec_build_tree")


def spec_verify_attention(b: int, n: int, Hq: int, Hkv: int, D: int, page_size: int, q, k_pool, v_pool,
                          req_to_token, req_pool_idx, seq_lens, max_seq_len: int, verify_loc, mask_bits,
                          scale: float, out, lse, ws: Workspace, stream=None):
    num_slots = k_pool.shape[0]
    _check(LIB.spec_verify_attention(b, n, Hq, Hkv, D, page_size, _ptr(q), _ptr(k_pool), _ptr(v_pool), num_slots,
                                     _ptr(req_to_token), req_to_token.shape[0], req_to_token.shape[1],
                                     _ptr(req_pool_idx), _ptr(seq_lens), int(max_seq_len), _ptr(verify_loc),
                                     _ptr(mask_bits), float(scale), _ptr(out), _ptr(lse), ws.ptr, ws.nbytes,
                                     _stream(stream)), "spec_verify_attention")


def spec_verify_greedy(b: int, n: int, S: int, logits, draft_tokens, retrieve_index, next_token, next_sibling,
                       predict, accept_index, accept_lens, accepted_tokens, next_root, ws: Workspace, stream=None):
    V = logits.shape[-1]
    _check(LIB.spec_verify_greedy(b, n, S, V, _dtype_code(logits), _ptr(logits), _ptr(draft_tokens),
                                  _ptr(retrieve_index), _ptr(next_token), _ptr(next_sibling), _ptr(predict),
                                  _ptr(accept_index), _ptr(accept_lens), _ptr(accepted_tokens), _ptr(next_root),
                                  ws.ptr, ws.nbytes, _stream(stream)), "spec_verify_greedy")


def spec_verify_sampling(b: int, n: int, S: int, logits, draft_probs, temperatures, u, u_final, draft_tokens,
                         retrieve_index, next_token, next_sibling, predict, accept_index, accept_lens,
                         accepted_tokens, next_root, ws: Workspace, stream=None):
    V = logits.shape[-1]
    _check(LIB.spec_verify_sampling(b, n, S, V, _dtype_code(logits), _ptr(logits), _ptr(draft_probs),
                                    _ptr(temperatures), _ptr(u), _ptr(u_final), _ptr(draft_tokens),
                                    _ptr(retrieve_index), _ptr(next_token), _ptr(next_sibling), _ptr(predict),
                                    _ptr(accept_index), _ptr(accept_lens), _ptr(accepted_tokens), _ptr(next_root),
                                    ws.ptr, ws.nbytes, _stream(stream)), "spec_verify_sampling")


def spec_verify_target_only(b: int, n: int, S: int, logits, temperatures, coins, u_final, threshold_single: float,
                            threshold_acc: float, draft_tokens, retrieve_index, next_token, next_sibling, predict,
                            accept_index, accept_lens, accepted_tokens, next_root, ws: Workspace, stream=None):
    V = logits.shape[-1]
    _check(LIB.spec_verify_target_only(b, n, S, V, _dtype_code(logits), _ptr(logits), _ptr(temperatures),
                                       _ptr(coins), _ptr(u_final), float(threshold_single), float(threshold_acc),
                                       _ptr(draft_tokens), _ptr(retrieve_index), _ptr(next_token),
                                       _ptr(next_sibling), _ptr(predict), _ptr(accept_index), _ptr(accept_lens),
                                       _ptr(accepted_tokens), _ptr(next_root), ws.ptr, ws.nbytes, _stream(stream)),
           "spec_verify_target_only")


def spec_build_chain_tree(b: int, S: int, bonus, draft_tokens, draft_ld: int, seq_lens, tree_tokens, positions,
                          retrieve_index, next_token, next_sibling, mask_bits, stream=None):
    _check(LIB.spec_build_chain_tree(b, S, _ptr(bonus), _ptr(draft_tokens), int(draft_ld), _ptr(seq_lens),
                                     _ptr(tree_tokens), _ptr(positions), _ptr(retrieve_index), _ptr(next_token),
                                     _ptr(next_sibling), _ptr(mask_bits), _stream(stream)), "spec_build_chain_tree")


def spec_verify_chain_greedy(b: int, S: int, logits, draft_tokens, draft_ld: int, prefix_lens, correct_len, bonus,
                             out_tokens, commit_lens, new_seq_lens, accept_index, ws: Workspace, stream=None):
    V = logits.shape[-1]
    _check(LIB.spec_verify_chain_greedy(b, S, V, _dtype_code(logits), _ptr(logits), _ptr(draft_tokens),
                                        int(draft_ld), _ptr(prefix_lens), _ptr(correct_len), _ptr(bonus),
                                        _ptr(out_tokens), _ptr(commit_lens), _ptr(new_seq_lens), _ptr(accept_index),
                                        ws.ptr, ws.nbytes, _stream(stream)), "spec_verify_chain_greedy")


def spec_assign_draft_locs(b: int, topk: int, S: int, page_size: int, req_to_token, req_pool_idx, seq_lens,
                           num_slots: int, out_cache_loc, positions, ws: Workspace, stream=None):
    _check(LIB.spec_assign_draft_locs(b, topk, S, page_size, _ptr(req_to_token), req_to_token.shape[0],
                                      req_to_token.shape[1], _ptr(req_pool_idx), _ptr(seq_lens), int(num_slots),
                                      _ptr(out_cache_loc), _ptr(positions), ws.ptr, ws.nbytes, _stream(stream)),
           "spec_assign_draft_locs")


def spec_duplicate_prefix_tail(b: int, topk: int, S: int, page_size: int, Hkv: int, D: int,
                               k_layers: Sequence[torch.Tensor], v_layers: Sequence[torch.Tensor], req_to_token,
                               req_pool_idx, seq_lens, ws: Workspace, stream=None):
    L = len(k_layers)
    for t in list(k_layers) + list(v_layers):
        _ptr(t)
    kp = (ctypes.c_void_p * L)(*[t.data_ptr() for t in k_layers])
    vp = (ctypes.c_void_p * L)(*[t.data_ptr() for t in v_layers])
    _check(LIB.spec_duplicate_prefix_tail(b, topk, S, page_size, Hkv, D, L, ctypes.cast(kp, ctypes.c_void_p),
                                          ctypes.cast(vp, ctypes.c_void_p), k_layers[0].shape[0],
                                          _ptr(req_to_token), req_to_token.shape[0], req_to_token.shape[1],
                                          _ptr(req_pool_idx), _ptr(seq_lens), ws.ptr, ws.nbytes, _stream(stream)),
           "spec_duplicate_prefix_tail")


def spec_build_full_mask(b: int, n: int, seq_lens, mask_bits, fill_prefix: bool, mask, ws: Workspace,
                         stream=None):
    """mask: a uint8 tensor of at least sum_b n*(L_b + n) bytes."""
    _check(LIB.spec_build_full_mask(b, n, _ptr(seq_lens), _ptr(mask_bits), 1 if fill_prefix else 0, _ptr(mask),
                                    ctypes.c_size_t(mask.numel()), ws.ptr, ws.nbytes, _stream(stream)),
           "spec_build_full_mask")


def spec_add_penalties(b: int, n: int, logits, penalties, stream=None):
    """In place: each request's penalty row [b, V] fp32 added to its n verify rows."""
    V = logits.shape[-1]
    _check(LIB.spec_add_penalties(b, n, V, _dtype_code(logits), _ptr(logits), _ptr(penalties), _stream(stream)),
           "spec_add_penalties")


def spec_renorm_probs(b: int, n: int, logits, temperatures, top_k, top_p, probs, stream=None):
    V = logits.shape[-1]
    _check(LIB.spec_renorm_probs(b, n, V, _dtype_code(logits), _ptr(logits), _ptr(temperatures), _ptr(top_k),
                                 _ptr(top_p), _ptr(probs), _stream(stream)), "spec_renorm_probs")


def spec_verify_sampling_probs(b: int, n: int, S: int, probs, draft_probs, u, u_final, draft_tokens, retrieve_index,
                               next_token, next_sibling, predict, accept_index, accept_lens, accepted_tokens,
                               next_root, ws: Workspace, stream=None):
    V = probs.shape[-1]
    _check(LIB.spec_verify_sampling_probs(b, n, S, V, _ptr(probs), _ptr(draft_probs), _ptr(u), _ptr(u_final),
                                          _ptr(draft_tokens), _ptr(retrieve_index), _ptr(next_token),
                                          _ptr(next_sibling), _ptr(predict), _ptr(accept_index), _ptr(accept_lens),
                                          _ptr(accepted_tokens), _ptr(next_root), ws.ptr, ws.nbytes,
                                          _stream(stream)), "spec_verify_sampling_probs")


def spec_verify_target_only_probs(b: int, n: int, S: int, probs, coins, u_final, threshold_single: float,
                                  threshold_acc: float, draft_tokens, retrieve_index, next_token, next_sibling,
                                  predict, accept_index, accept_lens, accepted_tokens, next_root, ws: Workspace,
                                  stream=None):
    V = probs.shape[-1]
    _check(LIB.spec_verify_target_only_probs(b, n, S, V, _ptr(probs), _ptr(coins), _ptr(u_final),
                                             float(threshold_single), float(threshold_acc), _ptr(draft_tokens),
                                             _ptr(retrieve_index), _ptr(next_token), _ptr(next_sibling),
                                             _ptr(predict), _ptr(accept_index), _ptr(accept_lens),
                                             _ptr(accepted_tokens), _ptr(next_root), ws.ptr, ws.nbytes,
                                             _stream(stream)), "spec_verify_target_only_probs")


def spec_commit_kv(b: int, n: int, W: int, Hkv: int, D: int, page_size: int, k_layers: Sequence[torch.Tensor],
                   v_layers: Sequence[torch.Tensor], req_to_token, req_pool_idx, seq_lens, verify_loc,
                   accept_index, accept_lens, new_seq_lens, free_ids, n_free, ws: Workspace, stream=None):
    L = len(k_layers)
    kp = (ctypes.c_void_p * L)(*[t.data_ptr() for t in k_layers])
    vp = (ctypes.c_void_p * L)(*[t.data_ptr() for t in v_layers])
    for t in list(k_layers) + list(v_layers):
        _ptr(t)
    _check(LIB.spec_commit_kv(b, n, W, Hkv, D, L, page_size, ctypes.cast(kp, ctypes.c_void_p),
                              ctypes.cast(vp, ctypes.c_void_p), k_layers[0].shape[0], _ptr(req_to_token),
                              req_to_token.shape[0], req_to_token.shape[1], _ptr(req_pool_idx), _ptr(seq_lens),
                              _ptr(verify_loc), _ptr(accept_index), _ptr(accept_lens), _ptr(new_seq_lens),
                              _ptr(free_ids), _ptr(n_free), ws.ptr, ws.nbytes, _stream(stream)), "spec_commit_kv")


def spec_verify_greedy_noalloc(b: int, n: int, S: int, logits, draft_tokens, retrieve_index, next_token,
                               next_sibling, predict, accept_index, accept_lens, accepted_tokens, next_root,
                               stream=None):
    """spec_verify_greedy for callers that cannot allocate device memory: the
    library's fixed device scratch array stands in for the workspace."""
    V = logits.shape[-1]
    _check(LIB.spec_verify_greedy_noalloc(b, n, S, V, _dtype_code(logits), _ptr(logits), _ptr(draft_tokens),
                                          _ptr(retrieve_index), _ptr(next_token), _ptr(next_sibling), _ptr(predict),
                                          _ptr(accept_index), _ptr(accept_lens), _ptr(accepted_tokens),
                                          _ptr(next_root), _stream(stream)), "spec_verify_greedy_noalloc")


def spec_noalloc_last_error(stream=None) -> int:
    """Reads and clears the SPEC_DEV_* bits set by spec_verify_greedy_noalloc
    calls on the current device (synchronises the stream)."""
    rc = LIB.spec_noalloc_last_error(_stream(stream))
    if rc < 0:
        _check(rc, "spec_noalloc_last_error")
    return rc
