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
    p = _softmax64(logits_row, T)
    return abs(u * float(q_row[x]) - p[x]) / max(p[x], 1e-30)


def _softmax64(row: np.ndarray, T: float) -> np.ndarray:
    z = row.astype(np.float64) / T
    z -= z.max()
    p = np.exp(z)
    return p / p.sum()


# Bounds of a near tie.  An accept test is a near tie when u*q(x) and p(x)
# are within SAMPLING_ACCEPT_RTOL of p(x): the device's fp32 p has a relative
# error of about 1e-6 (hardware exp2 of each term, fp32 row sum), the
# oracle's is exact to fp32 rounding.  A terminal draw is a near tie when
# u_final lies within SAMPLING_CDF_ATOL of the normalised cumulative mass at
# the boundary between the two tokens and no mass above that bound lies
# between them.
SAMPLING_ACCEPT_RTOL = 2e-6
SAMPLING_CDF_ATOL = 1e-6

# The select's top-k probabilities p = exp((v - M)/T) / S against the
# oracle's fp64 softmax: the bar is 1e-6 relative.  The device keeps the
# denominator's error systematic-free: each term's exponent is (x - g) c with
# x - g exact (bf16) and c = log2(e)/T carried as hi + lo from fp64, so no
# error proportional to the row maximum or to c's rounding enters (over a
# 128K vocabulary, where most of the mass sits 10-15 binary orders below the
# maximum, those alone reach 1e-6); each term then goes through the hardware
# ex2 (2^-22 relative), a group's 64 terms are added as a tree, the groups of a
# thread with compensation, and the CTA in fp64; the numerator is expf (2 ulp).
# A path score is one more fp32 product of p.
SELECT_P_RTOL = 1e-6
SELECT_SCORE_RTOL = SELECT_P_RTOL + 2.0 ** -24


def sampling_divergence(lg_rows: np.ndarray, q_rows: np.ndarray, T: float, u: np.ndarray, u_final: float,
                        tok: np.ndarray, nt: np.ndarray, ns: np.ndarray, n: int, r: int,
                        o_idx: np.ndarray, o_len: int, o_term: int, g_idx: np.ndarray, g_len: int,
                        g_term: int):
    """Where the oracle's and the device's accept of request r part, and
    whether that one decision is a near tie.

    Both sides walk the same tree from the root, testing the children of the
    current node in sibling order.  The first child that one side accepts
    and the other rejects is the decision that parted them: it is certified
    when its test u*q(x) < p(x) is a near tie.  When the two paths agree, the
    terminal draw at the last node parted them: it is certified when u_final
    sits at the boundary between the two tokens (see the bounds above).

    lg_rows / q_rows: fp64 logits and fp32 q of request r's n rows; u: its n
    coins; tok / nt / ns: its tree arrays (local node ids); *_idx: accept_index
    rows of r (global), *_len: accept_lens, *_term: the terminal token.
    Returns (kind, certified, margin): kind is "same", "accept" or "terminal"
    ("greedy" for T <= 0, where every decision is exact and nothing can be
    certified)."""
    if T <= 0:
        return "greedy", False, float("inf")
    o_path = [int(x) - r * n for x in o_idx[:o_len]]
    g_path = [int(x) - r * n for x in g_idx[:g_len]]
    cur, d = 0, 0
    while True:
        oc = o_path[d + 1] if d + 1 < len(o_path) else -1
        gc = g_path[d + 1] if d + 1 < len(g_path) else -1
        if oc == gc:
            if oc == -1:
                break
            cur, d = oc, d + 1
            continue
        # the first child in sibling order that one side accepted
        c = nt[cur]
        while c != -1 and c != oc and c != gc:
            c = ns[c]
        p = _softmax64(lg_rows[cur], T)
        x = int(tok[c])
        margin = abs(float(u[c]) * float(q_rows[cur][x]) - p[x]) / max(p[x], 1e-300)
        return "accept", margin <= SAMPLING_ACCEPT_RTOL, margin
    if o_term == g_term:
        return "same", True, 0.0
    # the terminal draw at node cur: from the residual when cur's children
    # were all rejected, else from p
    p = _softmax64(lg_rows[cur], T)
    had_child = nt[cur] != -1 and len(o_path) - 1 < (len(o_idx) - 1)
    dist = p
    if had_child:
        res = np.maximum(p - q_rows[cur].astype(np.float64), 0.0)
        if res.sum() > 0:
            dist = res
    cdf = np.cumsum(dist) / dist.sum()
    lo, hi = min(o_term, g_term), max(o_term, g_term)
    margin = max(abs(float(u_final) - cdf[lo]), abs(float(u_final) - cdf[hi - 1]))
    return "terminal", margin <= SAMPLING_CDF_ATOL, margin


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def target_only_divergence(lg_rows: np.ndarray, T: float, coins: np.ndarray, u_final: float, t_single: float,
                           t_acc: float, tok: np.ndarray, nt: np.ndarray, ns: np.ndarray, S: int, n: int, r: int,
                           o_idx: np.ndarray, o_len: int, o_term: int, g_idx: np.ndarray, g_len: int,
                           g_term: int):
    """As sampling_divergence, for the target-only sampler: the first child
    one side accepts and the other rejects is certified when either of its
    tests is a near tie (the coin against prob_acc / threshold_acc, or p(x)
    against threshold_single, within SAMPLING_ACCEPT_RTOL), the terminal draw
    as in sampling_divergence with the rejected children's tokens removed."""
    if T <= 0:
        return "greedy", False, float("inf")
    o_path = [int(x) - r * n for x in o_idx[:o_len]]
    g_path = [int(x) - r * n for x in g_idx[:g_len]]
    cur, d = 0, 0
    while True:
        oc = o_path[d + 1] if d + 1 < len(o_path) else -1
        gc = g_path[d + 1] if d + 1 < len(g_path) else -1
        if oc == gc:
            if oc == -1:
                break
            cur, d = oc, d + 1
            continue
        p = _softmax64(lg_rows[cur], T)
        coin = float(coins[cur])
        acc = 0.0
        c = nt[cur]
        while c != -1:
            acc += p[int(tok[c])]
            if c == oc or c == gc:
                break
            c = ns[c]
        x = int(tok[c])
        m1 = abs(coin - acc / t_acc) / max(acc / t_acc, 1e-300)
        m2 = abs(p[x] - t_single) / t_single
        margin = min(m1, m2)
        return "accept", margin <= SAMPLING_ACCEPT_RTOL, margin
    if o_term == g_term:
        return "same", True, 0.0
    p = _softmax64(lg_rows[cur], T)
    dist = p
    if nt[cur] != -1 and len(o_path) - 1 < S:  # every child of cur was rejected
        dist = p.copy()
        c = nt[cur]
        while c != -1:
            dist[int(tok[c])] = 0.0
            c = ns[c]
        if dist.sum() <= 0:
            dist = p
    cdf = np.cumsum(dist) / dist.sum()
    lo, hi = min(o_term, g_term), max(o_term, g_term)
    margin = max(abs(float(u_final) - cdf[lo]), abs(float(u_final) - cdf[hi - 1]))
    return "terminal", margin <= SAMPLING_CDF_ATOL, margin
