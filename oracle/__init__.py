"""CPU oracle for one EAGLE-style verify/accept step (test infrastructure).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The GPU path never
imports, links or calls it, and it never imports the GPU path.

The arithmetic lives in ``oracle.c`` (plain C11, fp64, compiled with gcc and
``-ffp-contract=off`` so that x86-64 and aarch64 round alike).  This module only
marshals numpy arrays in and out.  bf16 tensors travel as ``uint16`` arrays of
their bit patterns.  Each function returns a dict of numpy arrays and raises
``OracleError`` when the C routine reports a bad argument, an out-of-range
index or a broken invariant.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_SOURCES = [os.path.join(_HERE, "oracle.c"), os.path.join(_HERE, "oracle.h")]

F32, BF16 = 0, 1
_ERRORS = {1: "bad argument", 2: "index out of range", 3: "input breaks an invariant of the method"}

_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` (gcc, portable flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and all(
        os.path.getmtime(_LIB_PATH) >= os.path.getmtime(s) for s in _SOURCES)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
           os.path.join(_HERE, "oracle.c"), "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            for name in ("oracle_softmax_topk", "oracle_path_step", "oracle_select_topk",
                         "oracle_build_tree", "oracle_verify_attention", "oracle_verify_greedy",
                         "oracle_verify_sampling", "oracle_verify_target_only", "oracle_build_chain_tree",
                         "oracle_chain_accept_greedy", "oracle_assign_draft_locs", "oracle_duplicate_prefix_tail",
                         "oracle_full_mask", "oracle_add_penalties", "oracle_renorm_probs",
                         "oracle_verify_sampling_probs", "oracle_verify_target_only_probs", "oracle_commit_kv"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a):
    """Pointer to a contiguous numpy array (or NULL for None).  ``data_as``
    keeps a reference to the array, so a temporary converted array stays alive
    for as long as the pointer object does (the duration of the call)."""
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what}: {_ERRORS.get(rc, rc)}")


def _logits(x: np.ndarray):
    """(array, dtype code) for fp32 logits or bf16 bit patterns."""
    if x.dtype == np.float32:
        return np.ascontiguousarray(x), F32
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x), BF16
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {x.dtype}")


def _i32(x, shape=None):
    a = np.ascontiguousarray(np.asarray(x, dtype=np.int32))
    if shape is not None:
        a = a.reshape(shape)
    return a


def softmax_topk(logits: np.ndarray, k: int, temperature: float = 1.0):
    x, dt = _logits(logits)
    rows, V = x.shape
    p = np.empty((rows, k), np.float32)
    idx = np.empty((rows, k), np.int32)
    _check(_load().oracle_softmax_topk(rows, V, dt, _p(x), ctypes.c_double(temperature), k,
                                       _p(p), _p(idx)), "softmax_topk")
    return {"topk_p": p, "topk_idx": idx}


def _step_shapes(step, b, k):
    if step == 0:
        return (b, k), (b, k + 1)
    return (b, k * k), (b, k)


def path_step(step: int, b: int, k: int, topk_p, topk_idx, scores_in=None):
    blk, pblk = _step_shapes(step, b, k)
    out = {"score_blk": np.empty(blk, np.float32), "token_blk": np.empty(blk, np.int32),
           "parent_blk": np.empty(pblk, np.int32), "scores_out": np.empty((b, k), np.float32),
           "next_ids": np.empty((b, k), np.int32)}
    tp = np.ascontiguousarray(topk_p, np.float32)
    ti = _i32(topk_idx)
    si = None if scores_in is None else np.ascontiguousarray(scores_in, np.float32)
    _check(_load().oracle_path_step(step, b, k, _p(tp), _p(ti), _p(si), _p(out["score_blk"]),
                                    _p(out["token_blk"]), _p(out["parent_blk"]),
                                    _p(out["scores_out"]), _p(out["next_ids"])), "path_step")
    return out


def select_topk(step: int, b: int, k: int, draft_logits, temperature: float = 1.0, scores_in=None):
    x, dt = _logits(draft_logits)
    rows = b * (k if step else 1)
    assert x.shape[0] == rows, (x.shape, rows)
    V = x.shape[1]
    blk, pblk = _step_shapes(step, b, k)
    out = {"score_blk": np.empty(blk, np.float32), "token_blk": np.empty(blk, np.int32),
           "parent_blk": np.empty(pblk, np.int32), "scores_out": np.empty((b, k), np.float32),
           "next_ids": np.empty((b, k), np.int32), "topk_p": np.empty((rows, k), np.float32)}
    si = None if scores_in is None else np.ascontiguousarray(scores_in, np.float32)
    _check(_load().oracle_select_topk(step, b, k, V, dt, _p(x), ctypes.c_double(temperature),
                                      _p(si), _p(out["score_blk"]), _p(out["token_blk"]),
                                      _p(out["parent_blk"]), _p(out["scores_out"]),
                                      _p(out["next_ids"]), _p(out["topk_p"])), "select_topk")
    return out


def build_tree(b, k, S, n, score_space, token_space, parent_space, bonus, seq_lens):
    C = k + (S - 1) * k * k
    P = 1 + (S - 1) * k
    sc = np.ascontiguousarray(score_space, np.float32).reshape(b, C)
    tk = _i32(token_space, (b, C))
    pa = _i32(parent_space, (b, P))
    bo = _i32(bonus, (b,))
    sl = _i32(seq_lens, (b,))
    out = {name: np.empty(b * n, np.int32) for name in
           ("draft_tokens", "positions", "retrieve_index", "next_token", "next_sibling", "parent_node")}
    out["mask_bits"] = np.empty(b * n, np.uint64)
    _check(_load().oracle_build_tree(b, k, S, n, _p(sc), _p(tk), _p(pa), _p(bo), _p(sl),
                                     _p(out["draft_tokens"]), _p(out["positions"]),
                                     _p(out["retrieve_index"]), _p(out["next_token"]),
                                     _p(out["next_sibling"]), _p(out["mask_bits"]),
                                     _p(out["parent_node"])), "build_tree")
    return out


def verify_attention(b, n, Hq, Hkv, D, q, k_pool, v_pool, req_to_token, req_pool_idx, seq_lens,
                     verify_loc, mask_bits, scale, pairs=None):
    """Returns out [b*n, Hq, D] fp64 and lse [b*n, Hq] fp64.  With ``pairs`` (an
    [m, 2] array of (row, head)) only those entries are computed; the others
    are NaN."""
    q = np.ascontiguousarray(q, np.uint16)
    k_pool = np.ascontiguousarray(k_pool, np.uint16)
    v_pool = np.ascontiguousarray(v_pool, np.uint16)
    num_slots = k_pool.size // (Hkv * D)
    r2t = _i32(req_to_token)
    row_w = r2t.shape[-1]
    out = np.full((b * n, Hq, D), np.nan)
    lse = np.full((b * n, Hq), np.nan)
    pr = None if pairs is None else _i32(pairs).reshape(-1, 2)
    _check(_load().oracle_verify_attention(
        b, n, Hq, Hkv, D, _p(q), _p(k_pool), _p(v_pool), ctypes.c_int64(num_slots), _p(r2t), row_w,
        _p(_i32(req_pool_idx)), _p(_i32(seq_lens)), _p(_i32(verify_loc)),
        _p(np.ascontiguousarray(mask_bits, np.uint64)), ctypes.c_double(scale),
        0 if pr is None else pr.shape[0], _p(pr), _p(out), _p(lse)), "verify_attention")
    return {"out": out, "lse": lse}


def _accept_outputs(b, n, S):
    W = S + 1
    return {"predict": np.empty(b * n, np.int32), "accept_index": np.empty((b, W), np.int32),
            "accept_lens": np.empty(b, np.int32), "accepted_tokens": np.empty((b, W), np.int32),
            "next_root": np.empty(b, np.int32)}


def verify_greedy(b, n, S, logits, draft_tokens, retrieve_index, next_token, next_sibling):
    x, dt = _logits(logits)
    V = x.shape[-1]
    out = _accept_outputs(b, n, S)
    _check(_load().oracle_verify_greedy(
        b, n, S, V, dt, _p(x), _p(_i32(draft_tokens)), _p(_i32(retrieve_index)),
        _p(_i32(next_token)), _p(_i32(next_sibling)), _p(out["predict"]), _p(out["accept_index"]),
        _p(out["accept_lens"]), _p(out["accepted_tokens"]), _p(out["next_root"])), "verify_greedy")
    return out


def verify_sampling(b, n, S, logits, draft_probs, temperatures, u, u_final, draft_tokens,
                    retrieve_index, next_token, next_sibling):
    x, dt = _logits(logits)
    V = x.shape[-1]
    out = _accept_outputs(b, n, S)
    _check(_load().oracle_verify_sampling(
        b, n, S, V, dt, _p(x), _p(np.ascontiguousarray(draft_probs, np.float32)),
        _p(np.ascontiguousarray(temperatures, np.float32)), _p(np.ascontiguousarray(u, np.float32)),
        _p(np.ascontiguousarray(u_final, np.float32)), _p(_i32(draft_tokens)),
        _p(_i32(retrieve_index)), _p(_i32(next_token)), _p(_i32(next_sibling)),
        _p(out["predict"]), _p(out["accept_index"]), _p(out["accept_lens"]),
        _p(out["accepted_tokens"]), _p(out["next_root"])), "verify_sampling")
    return out


def verify_target_only(b, n, S, logits, temperatures, u, u_final, threshold_single, threshold_acc, draft_tokens,
                       retrieve_index, next_token, next_sibling):
    """Target-only tree sampling: u [b*n] holds one coin per node (the coin used
    to scan that node's children), u_final [b] the terminal draw's."""
    x, dt = _logits(logits)
    V = x.shape[-1]
    out = _accept_outputs(b, n, S)
    _check(_load().oracle_verify_target_only(
        b, n, S, V, dt, _p(x), _p(np.ascontiguousarray(temperatures, np.float32)),
        _p(np.ascontiguousarray(u, np.float32)), _p(np.ascontiguousarray(u_final, np.float32)),
        ctypes.c_float(threshold_single), ctypes.c_float(threshold_acc), _p(_i32(draft_tokens)),
        _p(_i32(retrieve_index)), _p(_i32(next_token)), _p(_i32(next_sibling)),
        _p(out["predict"]), _p(out["accept_index"]), _p(out["accept_lens"]),
        _p(out["accepted_tokens"]), _p(out["next_root"])), "verify_target_only")
    return out


def build_chain_tree(b, S, bonus, draft_tokens, seq_lens):
    """Tree arrays of b chains; draft_tokens [b, S] (row stride = its width)."""
    dt = _i32(draft_tokens)
    dt = dt.reshape(b, -1)
    n = S + 1
    out = {name: np.empty(b * n, np.int32) for name in
           ("draft_tokens", "positions", "retrieve_index", "next_token", "next_sibling")}
    out["mask_bits"] = np.empty(b * n, np.uint64)
    _check(_load().oracle_build_chain_tree(b, S, _p(_i32(bonus, (b,))), _p(dt), dt.shape[1],
                                           _p(_i32(seq_lens, (b,))), _p(out["draft_tokens"]), _p(out["positions"]),
                                           _p(out["retrieve_index"]), _p(out["next_token"]),
                                           _p(out["next_sibling"]), _p(out["mask_bits"])), "build_chain_tree")
    return out


def chain_accept_greedy(b, S, logits, draft_tokens, prefix_lens):
    x, dt = _logits(logits)
    V = x.shape[-1]
    d = _i32(draft_tokens).reshape(b, -1)
    n = S + 1
    out = {"correct_len": np.empty(b, np.int32), "bonus": np.empty(b, np.int32),
           "out_tokens": np.empty((b, n), np.int32), "commit_lens": np.empty(b, np.int32),
           "new_seq_lens": np.empty(b, np.int32), "accept_index": np.empty((b, n), np.int32)}
    _check(_load().oracle_chain_accept_greedy(
        b, S, V, dt, _p(x), _p(d), d.shape[1], _p(_i32(prefix_lens, (b,))), _p(out["correct_len"]),
        _p(out["bonus"]), _p(out["out_tokens"]), _p(out["commit_lens"]), _p(out["new_seq_lens"]),
        _p(out["accept_index"])), "chain_accept_greedy")
    return out


def assign_draft_locs(b, topk, S, page_size, req_to_token, req_pool_idx, seq_lens, num_slots):
    r2t = _i32(req_to_token)
    out = np.empty(b * topk * S, np.int32)
    pos = np.empty(b, np.int32)
    _check(_load().oracle_assign_draft_locs(b, topk, S, page_size, _p(r2t), r2t.shape[-1], _p(_i32(req_pool_idx)),
                                            _p(_i32(seq_lens)), ctypes.c_int64(num_slots), _p(out), _p(pos)),
           "assign_draft_locs")
    return {"out_cache_loc": out, "positions": pos if topk == 1 else None}


def duplicate_prefix_tail(b, topk, S, page_size, Hkv, D, k_layers, v_layers, req_to_token, req_pool_idx, seq_lens):
    """Copies in place into the uint16 pool arrays of k_layers / v_layers."""
    L = len(k_layers)
    for a in list(k_layers) + list(v_layers):
        assert a.dtype == np.uint16 and a.flags["C_CONTIGUOUS"]
    num_slots = k_layers[0].size // (Hkv * D)
    kp = (ctypes.c_void_p * L)(*[a.ctypes.data for a in k_layers])
    vp = (ctypes.c_void_p * L)(*[a.ctypes.data for a in v_layers])
    r2t = _i32(req_to_token)
    _check(_load().oracle_duplicate_prefix_tail(b, topk, S, page_size, Hkv, D, L, kp, vp, ctypes.c_int64(num_slots),
                                                _p(r2t), r2t.shape[-1], _p(_i32(req_pool_idx)), _p(_i32(seq_lens))),
           "duplicate_prefix_tail")


def full_mask(b, n, seq_lens, mask_bits, fill_prefix=True, out=None):
    """The FULL_MASK verify mask (uint8, one [n, L_b + n] block per request);
    with fill_prefix False the prefix columns keep the values of ``out``."""
    sl = _i32(seq_lens, (b,))
    total = int(np.sum(n * (sl.astype(np.int64) + n)))
    m = np.zeros(total, np.uint8) if out is None else np.ascontiguousarray(out, np.uint8).copy()
    assert m.size == total
    _check(_load().oracle_full_mask(b, n, _p(sl), _p(np.ascontiguousarray(mask_bits, np.uint64)),
                                    1 if fill_prefix else 0, _p(m)), "full_mask")
    return m


def add_penalties(b, n, logits, penalties):
    """A copy of the logits (fp32, or bf16 bits as uint16) with each request's
    penalty row [b, V] fp32 added to its n verify rows."""
    x, dt = _logits(logits)
    out = x.copy()
    V = out.shape[-1]
    _check(_load().oracle_add_penalties(b, n, V, dt, _p(out), _p(np.ascontiguousarray(penalties, np.float32))),
           "add_penalties")
    return out


def renorm_probs(b, n, logits, temperatures, top_k, top_p):
    x, dt = _logits(logits)
    V = x.shape[-1]
    out = np.empty((b * n, V), np.float32)
    _check(_load().oracle_renorm_probs(b, n, V, dt, _p(x), _p(np.ascontiguousarray(temperatures, np.float32)),
                                       _p(_i32(top_k, (b,))), _p(np.ascontiguousarray(top_p, np.float32)),
                                       _p(out)), "renorm_probs")
    return out


def verify_sampling_probs(b, n, S, probs, draft_probs, u, u_final, draft_tokens, retrieve_index, next_token,
                          next_sibling):
    pr = np.ascontiguousarray(probs, np.float32)
    V = pr.shape[-1]
    out = _accept_outputs(b, n, S)
    _check(_load().oracle_verify_sampling_probs(
        b, n, S, V, _p(pr), _p(np.ascontiguousarray(draft_probs, np.float32)),
        _p(np.ascontiguousarray(u, np.float32)), _p(np.ascontiguousarray(u_final, np.float32)),
        _p(_i32(draft_tokens)), _p(_i32(retrieve_index)), _p(_i32(next_token)), _p(_i32(next_sibling)),
        _p(out["predict"]), _p(out["accept_index"]), _p(out["accept_lens"]), _p(out["accepted_tokens"]),
        _p(out["next_root"])), "verify_sampling_probs")
    return out


def verify_target_only_probs(b, n, S, probs, u, u_final, threshold_single, threshold_acc, draft_tokens,
                             retrieve_index, next_token, next_sibling):
    pr = np.ascontiguousarray(probs, np.float32)
    V = pr.shape[-1]
    out = _accept_outputs(b, n, S)
    _check(_load().oracle_verify_target_only_probs(
        b, n, S, V, _p(pr), _p(np.ascontiguousarray(u, np.float32)), _p(np.ascontiguousarray(u_final, np.float32)),
        ctypes.c_float(threshold_single), ctypes.c_float(threshold_acc), _p(_i32(draft_tokens)),
        _p(_i32(retrieve_index)), _p(_i32(next_token)), _p(_i32(next_sibling)), _p(out["predict"]),
        _p(out["accept_index"]), _p(out["accept_lens"]), _p(out["accepted_tokens"]), _p(out["next_root"])),
        "verify_target_only_probs")
    return out


def commit_kv(b, n, W, Hkv, D, page_size, k_layers, v_layers, req_to_token, req_pool_idx, seq_lens,
              verify_loc, accept_index, accept_lens):
    """Commits in place into the uint16 pool arrays in ``k_layers``/``v_layers``
    (lists of [num_slots, Hkv, D] arrays) and returns new_seq_lens and the free list."""
    L = len(k_layers)
    for a in list(k_layers) + list(v_layers):
        assert a.dtype == np.uint16 and a.flags["C_CONTIGUOUS"]
    num_slots = k_layers[0].size // (Hkv * D)
    kp = (ctypes.c_void_p * L)(*[a.ctypes.data for a in k_layers])
    vp = (ctypes.c_void_p * L)(*[a.ctypes.data for a in v_layers])
    r2t = _i32(req_to_token)
    new_seq = np.empty(b, np.int32)
    free_ids = np.empty(max(1, b * n), np.int32)
    n_free = np.zeros(1, np.int32)
    _check(_load().oracle_commit_kv(
        b, n, W, Hkv, D, L, page_size, kp, vp, ctypes.c_int64(num_slots), _p(r2t), r2t.shape[-1],
        _p(_i32(req_pool_idx)), _p(_i32(seq_lens)), _p(_i32(verify_loc)), _p(_i32(accept_index)),
        _p(_i32(accept_lens)), _p(new_seq), _p(free_ids), _p(n_free)), "commit_kv")
    return {"new_seq_lens": new_seq, "free_ids": free_ids[: int(n_free[0])].copy()}
