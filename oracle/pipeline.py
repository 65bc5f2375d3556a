"""The oracle's verify/accept step over a generated workload (test infrastructure).

TEST INFRASTRUCTURE ONLY, like the rest of this package.  It chains the oracle
functions in the order of one verify step:
select_top_k_tokens x S -> organize_draft_results + build_tree -> verify
attention -> accept (greedy or rejection sampling) -> KV commit,
on host copies of inputs drawn by ``accept_select_top_gb300.workloads``.
"""
from __future__ import annotations

from typing import Dict, List, Optional

import numpy as np

import oracle
from accept_select_top_gb300 import workloads as wlmod


def select_chain(wl: wlmod.Workload, drafts: List[np.ndarray], temperature: float = 1.0) -> Dict:
    """Runs select_top_k_tokens for steps 0..S-1 on host draft logits and
    concatenates the blocks into the score / token space and the parent list."""
    b, k, S = wl.b, wl.k, wl.S
    steps = []
    scores = None
    for i in range(S):
        o = oracle.select_topk(i, b, k, drafts[i], temperature, scores)
        steps.append(o)
        scores = o["scores_out"]
    score_space = np.concatenate([s["score_blk"] for s in steps], axis=1)
    token_space = np.concatenate([s["token_blk"] for s in steps], axis=1)
    parent_space = np.concatenate([s["parent_blk"] for s in steps[:-1]], axis=1) if S > 1 \
        else np.full((b, 1), -1, np.int32)
    return {"steps": steps, "score_space": np.ascontiguousarray(score_space),
            "token_space": np.ascontiguousarray(token_space),
            "parent_space": np.ascontiguousarray(parent_space)}


def tree_from_chain(wl: wlmod.Workload, chain: Dict, bonus: np.ndarray, seq_lens: np.ndarray) -> Dict:
    return oracle.build_tree(wl.b, wl.k, wl.S, wl.n, chain["score_space"], chain["token_space"],
                             chain["parent_space"], bonus, seq_lens)


def accept(wl: wlmod.Workload, mode: str, tree: Dict, logits: np.ndarray,
           q: Optional[np.ndarray] = None, temps=None, u=None, u_final=None) -> Dict:
    args = (tree["draft_tokens"], tree["retrieve_index"], tree["next_token"], tree["next_sibling"])
    if mode == "greedy":
        return oracle.verify_greedy(wl.b, wl.n, wl.S, logits, *args)
    return oracle.verify_sampling(wl.b, wl.n, wl.S, logits, q, temps, u, u_final, *args)


def commit(wl: wlmod.Workload, layout: Dict, k_pool: np.ndarray, v_pool: np.ndarray, acc: Dict) -> Dict:
    return oracle.commit_kv(wl.b, wl.n, wl.W, wl.Hkv, wl.D, wl.page_size, [k_pool], [v_pool],
                            layout["req_to_token"], layout["req_pool_idx"], layout["seq_lens"],
                            layout["verify_loc"], acc["accept_index"], acc["accept_lens"])
