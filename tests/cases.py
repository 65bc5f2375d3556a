"""Parity cases: seeded inputs drawn on the device, host copies for the oracle,
and the oracle's own chain of results (test infrastructure)."""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np
import torch

from accept_select_top_gb300 import workloads as W
from oracle import pipeline as OP


@dataclasses.dataclass
class Case:
    wl: W.Workload
    mode: str
    layout: Dict
    drafts: list            # device tensors per step
    host_drafts: list
    bonus: torch.Tensor
    chain: Dict             # oracle select chain
    tree: Dict              # oracle tree
    node_rows: np.ndarray
    logits: torch.Tensor    # target logits (device)
    q: Optional[torch.Tensor]
    temps: np.ndarray
    u: torch.Tensor
    u_final: torch.Tensor
    att: Dict               # q, k_pool, v_pool (device)

    def device_inputs(self, device="cuda"):
        from accept_select_top_gb300.pipeline import DeviceInputs
        lay = self.layout
        t = lambda a: torch.as_tensor(np.ascontiguousarray(a)).to(device)
        return DeviceInputs(
            drafts=self.drafts, bonus=self.bonus, seq_lens=t(lay["seq_lens"]), req_pool_idx=t(lay["req_pool_idx"]),
            req_to_token=t(lay["req_to_token"]), verify_loc=t(lay["verify_loc"]), q=self.att["q"],
            k_pool=self.att["k_pool"], v_pool=self.att["v_pool"], max_seq_len=int(lay["seq_lens"].max()),
            target_logits=self.logits, draft_probs=self.q,
            temperatures=t(self.temps.astype(np.float32)), u=self.u, u_final=self.u_final)


def make_case(wl: W.Workload, mode: str, device="cuda", seed: int = 0, temps_mode: Optional[str] = None,
              with_attention: bool = True) -> Case:
    drafts = [W.draft_logits(wl, i, device, seed) for i in range(wl.S)]
    host_drafts = [W.host(d) for d in drafts]
    lay = W.kv_layout(wl, seed)
    bonus = W.bonus_tokens(wl, device, seed)
    chain = OP.select_chain(wl, host_drafts)
    tree = OP.tree_from_chain(wl, chain, W.host(bonus), lay["seq_lens"])
    rows = W.draft_rows_of_nodes(wl, tree["draft_tokens"], tree["next_token"], tree["next_sibling"],
                                 chain["token_space"], chain["parent_space"])
    all_d = torch.cat(drafts, 0)
    logits = W.target_logits(wl, rows, all_d, device, seed)
    if wl.agreement == "planted":
        logits = W.plant_agreement(wl, logits, tree["draft_tokens"], tree["next_token"], tree["next_sibling"], seed)
    if temps_mode is None:
        temps_mode = {"greedy": "greedy", "sampling": "sampling", "mixed": "mixed", "both": "sampling"}[
            wl.accept if mode == "sampling" else "greedy"]
    temps = W.request_temperatures(wl, temps_mode)
    q = W.draft_probs(wl, rows, all_d, temps, device) if mode == "sampling" else None
    u, uf = W.coins(wl, device, seed)
    att = W.attention_tensors(wl, int(lay["num_slots"]), device, seed) if with_attention else {}
    return Case(wl, mode, lay, drafts, host_drafts, bonus, chain, tree, rows, logits, q, temps, u, uf, att)


# --------------------------------------------------------- certification

def certified_topk_difference(values: np.ndarray, sel_a, sel_b, k: int, rtol: float = 4e-6) -> bool:
    """Two top-k selections over the same candidates differ only among values
    within ``rtol`` of the k-th best value (a near tie that ulp-level
    differences in the inputs may flip)."""
    a, b = set(int(x) for x in sel_a), set(int(x) for x in sel_b)
    if a == b:
        return True
    kth = np.sort(values)[::-1][k - 1]
    return all(abs(values[i] - kth) <= rtol * abs(kth) for i in a ^ b)


def sampling_margin(logits_row: np.ndarray, T: float, q_row: np.ndarray, x: int, u: float) -> float:
    """Relative margin of one accept test u*q(x) < p(x) with p in fp64."""
    z = logits_row.astype(np.float64) / T
    z -= z.max()
    p = np.exp(z)
    p /= p.sum()
    return abs(u * float(q_row[x]) - p[x]) / max(p[x], 1e-30)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
