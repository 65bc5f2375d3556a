"""Seeded synthetic inputs for one verify/accept step.

This module is the only code that the GPU path and the CPU oracle share: it
draws the inputs, lays out the paged KV cache, and says which draft row proposed
the children of each tree node.  It computes none of the method's steps (no
top-k, no tree building, no attention, no accept decision).  Its callers run
those steps on the device or in the oracle and hand the results back where a
recipe depends on them (the target logits of a node are correlated with the
draft row that expanded it).

Every draw comes from a ``torch.Generator`` seeded by a stable hash of
(seed, workload name, tensor name), so a tensor does not depend on the order in
which the others are drawn.  Draws on a device use that device's generator; a
run uses one device for all its draws and hands the same tensors to both sides.

The five workloads follow the shapes of the method's published settings:
topk / num_steps / num_draft_tokens, a Llama-3 vocabulary, GQA heads, page
sizes 1 and 16.  No public dataset is involved; every input is synthetic.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    b: int                 # requests in the batch
    k: int                 # topk per draft step
    S: int                 # num_steps
    n: int                 # num_draft_tokens (tree nodes, root included)
    V: int                 # vocabulary
    logits_dtype: str      # "f32" or "bf16"
    Hq: int
    Hkv: int
    D: int
    ctx: tuple             # ("fixed", L) | ("uniform", lo, hi) | ("list", (L0, L1, ..))
    page_size: int
    verify_layout: str     # "inplace": verify slots = the request's next positions;
                           # "scratch": verify slots in fresh pages (first seq_len % page holes)
    slot_order: str        # "contiguous" | "permuted" (scattered slots / pages)
    accept: str            # "greedy" | "sampling" | "both" | "mixed"
    agreement: str         # "noise": target = a*draft + N(0, s); "planted": see plant_agreement
    draft_std: float
    noise_a: float
    noise_std: float
    target_std: float      # target rows with no draft row behind them
    alpha: float = 0.0     # planted hit probability
    sample_temperature: float = 1.0
    draft_peak: tuple = ()  # (lo, hi): one token per draft row gets + U(lo, hi) (confident drafts)

    @property
    def C(self) -> int:
        """Length of the score (== token) space of one request."""
        return self.k + (self.S - 1) * self.k * self.k

    @property
    def P(self) -> int:
        """Length of the parent list of one request."""
        return 1 + (self.S - 1) * self.k

    @property
    def W(self) -> int:
        """Width of accept_index (max accepted rows, root included)."""
        return self.S + 1

    def rows(self, step: int) -> int:
        return self.b * (self.k if step else 1)

    @property
    def torch_logits_dtype(self):
        return torch.float32 if self.logits_dtype == "f32" else torch.bfloat16


_SQ5 = math.sqrt(5.0)

WORKLOADS: Dict[str, Workload] = {
    # bs=4 topk=2 steps=3 ndt=6 V=1024; draft N(0,1) fp32, target = draft + N(0,0.5);
    # 4 q / 1 kv heads, D=64, context 128, page 1, contiguous slots.
    "tiny": Workload("tiny", 4, 2, 3, 6, 1024, "f32", 4, 1, 64, ("fixed", 128), 1, "inplace",
                     "contiguous", "both", "noise", 1.0, 1.0, 0.5, math.sqrt(1.25)),
    # Llama-3-8B shape, greedy: bs=8 topk=4 steps=5 ndt=16 V=128256, bf16 N(0,2) logits,
    # agreement planted for ~3 accepted tokens; 32/8 heads, D=128, ctx U[512,4096], page 1.
    "llama8b_greedy": Workload("llama8b_greedy", 8, 4, 5, 16, 128256, "bf16", 32, 8, 128,
                               ("uniform", 512, 4096), 1, "inplace", "permuted", "greedy",
                               "planted", 2.0, 0.0, 0.0, 2.0, alpha=0.85, draft_peak=(8.0, 16.0)),
    # sampling-heavy: bs=32 topk=8 steps=6 ndt=64, T=1; target N(0,2), draft = target + N(0,1)
    # (drawn draft-first: d ~ N(0, sqrt 5), t = 0.8 d + N(0, sqrt 0.8)); ctx 2048, page 16.
    "sampling_heavy": Workload("sampling_heavy", 32, 8, 6, 64, 128256, "bf16", 32, 8, 128,
                               ("fixed", 2048), 16, "scratch", "permuted", "sampling", "noise",
                               _SQ5, 0.8, math.sqrt(0.8), 2.0),
    # long context, 70B shape: bs=2 topk=8 steps=8 ndt=64, greedy; 64/8 heads; ctx 32K and 128K.
    "long_context": Workload("long_context", 2, 8, 8, 64, 128256, "bf16", 64, 8, 128,
                             ("list", (32768, 131072)), 16, "scratch", "permuted", "greedy",
                             "planted", 2.0, 0.0, 0.0, 2.0, alpha=0.8, draft_peak=(8.0, 16.0)),
    # MTP-style chain: topk=1 steps=3 ndt=4 bs=256 V=129280, half greedy, half T=0.7.
    "mtp_chain": Workload("mtp_chain", 256, 1, 3, 4, 129280, "bf16", 32, 8, 128,
                          ("uniform", 256, 4096), 1, "inplace", "permuted", "mixed", "noise",
                          _SQ5, 0.8, math.sqrt(0.8), 2.0, sample_temperature=0.7),
}

ORDER = ["tiny", "llama8b_greedy", "sampling_heavy", "long_context", "mtp_chain"]


def scaled(wl: Workload, **changes) -> Workload:
    """A copy of a workload with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(wl, **changes)


# ----------------------------------------------------------------- seeding

def seed_for(seed: int, workload: str, tensor: str) -> int:
    h = hashlib.blake2b(f"{seed}/{workload}/{tensor}".encode(), digest_size=8).digest()
    return int.from_bytes(h, "little") & ((1 << 63) - 1)


def _gen(device, seed: int, wl: Workload, tensor: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed_for(seed, wl.name, tensor))
    return g


def _np_rng(seed: int, wl: Workload, tensor: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed_for(seed, wl.name, tensor)))


def normal(shape, std: float, device, gen: torch.Generator) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std


def uniform(shape, device, gen: torch.Generator) -> torch.Tensor:
    return torch.rand(shape, generator=gen, device=device, dtype=torch.float32)


# ------------------------------------------------------------- draft side

def draft_logits(wl: Workload, step: int, device="cpu", seed: int = 0) -> torch.Tensor:
    """Draft-model logits of step ``step``: [b*(1 or k), V] in the workload dtype."""
    x = normal((wl.rows(step), wl.V), wl.draft_std, device, _gen(device, seed, wl, f"draft{step}"))
    if wl.draft_peak:
        # a confident draft head: one random token per row is lifted by U(lo, hi)
        g = _gen(device, seed, wl, f"draft_peak{step}")
        tok = torch.randint(0, wl.V, (wl.rows(step),), generator=g, device=device)
        lift = wl.draft_peak[0] + (wl.draft_peak[1] - wl.draft_peak[0]) * uniform((wl.rows(step),), device, g)
        x[torch.arange(wl.rows(step), device=device), tok] += lift
    return x.to(wl.torch_logits_dtype)


def bonus_tokens(wl: Workload, device="cpu", seed: int = 0) -> torch.Tensor:
    g = _gen("cpu", seed, wl, "bonus")
    return torch.randint(0, wl.V, (wl.b,), generator=g, dtype=torch.int32).to(device)


# ------------------------------------------------------- paged KV layout

def kv_layout(wl: Workload, seed: int = 0, spare_slots: int = 64) -> Dict[str, np.ndarray]:
    """Host-side layout of the paged KV cache for the verify step.

    req_to_token[req, pos] is the slot of position ``pos`` of request ``req``;
    rows cover the prefix and the positions the commit may write
    (seq_len .. seq_len + W - 1); with the in-place verify layout they also
    cover the n verify positions.  verify_loc[b*n + j] is the slot holding
    tree node j of request b.  Slots never overlap between requests.
    """
    rng = _np_rng(seed, wl, "layout")
    b, n, ps = wl.b, wl.n, wl.page_size
    kind = wl.ctx[0]
    if kind == "fixed":
        seq = np.full(b, wl.ctx[1], np.int64)
    elif kind == "uniform":
        seq = rng.integers(wl.ctx[1], wl.ctx[2] + 1, size=b)
    else:
        vals = np.array(wl.ctx[1], np.int64)
        seq = vals[np.arange(b) % len(vals)]
    # positions each request owns in its req_to_token row
    own = seq + (n if wl.verify_layout == "inplace" else wl.W)
    own_pages = -(-own // ps)
    hole = seq % ps
    scratch_pages = -(-(hole + n) // ps) if wl.verify_layout == "scratch" else np.zeros(b, np.int64)
    total_pages = int(own_pages.sum() + scratch_pages.sum()) + -(-spare_slots // ps)
    if wl.slot_order == "permuted":
        page_ids = rng.permutation(total_pages)
    else:
        page_ids = np.arange(total_pages)
    row_w = int(own_pages.max()) * ps
    # request b lives in req_to_token row req_pool_idx[b] (a permutation, so the
    # indirection matters); one unused row is left in the table.
    max_req = b + 1
    req_pool_idx = rng.permutation(max_req)[:b].astype(np.int32)
    req_to_token = np.full((max_req, row_w), -1, np.int64)
    verify_loc = np.empty(b * n, np.int64)
    cursor = 0
    for r in range(b):
        pages = page_ids[cursor: cursor + own_pages[r]]
        cursor += own_pages[r]
        pos = np.arange(own_pages[r] * ps)
        slots = pages[pos // ps] * ps + pos % ps
        req_to_token[req_pool_idx[r], : len(slots)] = slots
        if wl.verify_layout == "inplace":
            verify_loc[r * n:(r + 1) * n] = slots[seq[r]: seq[r] + n]
        else:
            sp = page_ids[cursor: cursor + scratch_pages[r]]
            cursor += scratch_pages[r]
            off = hole[r] + np.arange(n)
            verify_loc[r * n:(r + 1) * n] = sp[off // ps] * ps + off % ps
    num_slots = total_pages * ps
    return {
        "seq_lens": seq.astype(np.int32),
        "req_pool_idx": req_pool_idx,
        "req_to_token": np.where(req_to_token < 0, 0, req_to_token).astype(np.int32),
        "verify_loc": verify_loc.astype(np.int32),
        "num_slots": np.int64(num_slots),
        "row_w": np.int32(row_w),
    }


def attention_tensors(wl: Workload, num_slots: int, device="cpu", seed: int = 0) -> Dict[str, torch.Tensor]:
    """q [b*n, Hq, D] and the K/V pools [num_slots, Hkv, D], bf16 N(0,1)
    (post-RoPE values: RoPE is outside the step)."""
    q = normal((wl.b * wl.n, wl.Hq, wl.D), 1.0, device, _gen(device, seed, wl, "q")).to(torch.bfloat16)
    k = normal((num_slots, wl.Hkv, wl.D), 1.0, device, _gen(device, seed, wl, "k")).to(torch.bfloat16)
    v = normal((num_slots, wl.Hkv, wl.D), 1.0, device, _gen(device, seed, wl, "v")).to(torch.bfloat16)
    return {"q": q, "k_pool": k, "v_pool": v}


# ----------------------------------------------- which draft row is whose

def tree_parents(next_token: np.ndarray, next_sibling: np.ndarray, b: int, n: int) -> np.ndarray:
    """Parent node of every node, read off the first-child / next-sibling arrays."""
    nt = next_token.reshape(b, n)
    ns = next_sibling.reshape(b, n)
    par = np.full((b, n), -1, np.int64)
    for r in range(b):
        for i in range(n):
            c = nt[r, i]
            while c != -1:
                par[r, c] = i
                c = ns[r, c]
    return par


def draft_rows_of_nodes(wl: Workload, draft_tokens: np.ndarray, next_token: np.ndarray,
                        next_sibling: np.ndarray, token_space: np.ndarray,
                        parent_space: np.ndarray) -> np.ndarray:
    """For each tree node, the draft row whose distribution proposed the node's
    children: an index into the concatenation of all steps' draft logits
    (step 0 rows first), or -1 when the node was never expanded.

    The root was expanded by step 0's row of its request.  A node at depth d
    came from step d-1; it was expanded at step d when its position in the
    token space is one of the rows of step d, i.e. listed in the parent block
    of step d-1.  A node's position is found from its parent's position and its
    token (the k tokens of one draft row are distinct).
    """
    b, n, k, S = wl.b, wl.n, wl.k, wl.S
    C, P = wl.C, wl.P
    tok = draft_tokens.reshape(b, n)
    ts = token_space.reshape(b, C)
    ps = parent_space.reshape(b, P)
    par = tree_parents(next_token, next_sibling, b, n)
    step_row0 = np.cumsum([0] + [wl.rows(s) for s in range(S)])  # first row of each step
    out = np.full((b, n), -1, np.int64)
    for r in range(b):
        pos = np.full(n, -1, np.int64)
        depth = np.zeros(n, np.int64)
        out[r, 0] = step_row0[0] + r
        for j in range(1, n):
            pj = par[r, j]
            depth[j] = depth[pj] + 1
            d = depth[j]
            if d == 1:
                cand = np.arange(k)
            else:
                rows_prev = ps[r, 1 + (d - 2) * k: 1 + (d - 1) * k]   # rows of step d-1
                rr = int(np.nonzero(rows_prev == pos[pj])[0][0])
                cand = k + (d - 2) * k * k + rr * k + np.arange(k)
            pos[j] = int(cand[np.nonzero(ts[r, cand] == tok[r, j])[0][0]])
            if d <= S - 1:
                rows_d = ps[r, 1 + (d - 1) * k: 1 + d * k]             # rows of step d
                hit = np.nonzero(rows_d == pos[j])[0]
                if len(hit):
                    out[r, j] = step_row0[d] + r * k + int(hit[0])
    return out.reshape(-1)


# ---------------------------------------------------------- verify side

def target_logits(wl: Workload, node_rows: np.ndarray, all_draft: torch.Tensor,
                  device="cpu", seed: int = 0) -> torch.Tensor:
    """Target logits [b*n, V] for the "noise" agreement recipe: the row of an
    expanded node is a*draft_row + N(0, noise_std); other rows are N(0, target_std)."""
    rows = wl.b * wl.n
    fresh = normal((rows, wl.V), wl.target_std, device, _gen(device, seed, wl, "target"))
    if wl.agreement != "noise":
        return fresh.to(wl.torch_logits_dtype)
    noise = normal((rows, wl.V), wl.noise_std, device, _gen(device, seed, wl, "target_noise"))
    idx = torch.as_tensor(node_rows, device=device)
    has = idx >= 0
    src = all_draft.index_select(0, idx.clamp_min(0)).float()
    t = torch.where(has[:, None], wl.noise_a * src + noise, fresh)
    return t.to(wl.torch_logits_dtype)


def plant_agreement(wl: Workload, logits: torch.Tensor, draft_tokens: np.ndarray,
                    next_token: np.ndarray, next_sibling: np.ndarray, seed: int = 0) -> torch.Tensor:
    """Planted greedy agreement: at every verify row whose node has children,
    with probability alpha the token of the node's first child (the draft's own
    top choice at that node) gets the row's largest logit plus 1, so the
    target's argmax is that child; otherwise every child token gets the largest
    non-child logit minus 1, so no child is the argmax.  Rows without children
    keep their random logits."""
    rng = _np_rng(seed, wl, "plant")
    b, n = wl.b, wl.n
    tok = draft_tokens.reshape(b, n)
    par = tree_parents(next_token, next_sibling, b, n)
    out = logits.clone()
    f = out.float()
    for r in range(b):
        for i in range(n):
            kids = np.nonzero(par[r] == i)[0]
            if len(kids) == 0:
                continue
            row = r * n + i
            ktoks = torch.as_tensor(tok[r, kids].astype(np.int64), device=out.device)
            if rng.random() < wl.alpha:
                f[row, ktoks[0]] = f[row].max() + 1.0
            else:
                others = f[row].clone()
                others[ktoks] = -float("inf")
                f[row, ktoks] = others.max() - 1.0
    return f.to(logits.dtype)


def request_temperatures(wl: Workload, mode: str) -> np.ndarray:
    """Per-request temperature; <= 0 means greedy."""
    if mode == "greedy":
        return np.zeros(wl.b, np.float32)
    if mode == "sampling":
        return np.full(wl.b, wl.sample_temperature, np.float32)
    if mode == "mixed":  # first half greedy, second half sampled
        t = np.full(wl.b, wl.sample_temperature, np.float32)
        t[: wl.b // 2] = 0.0
        return t
    raise ValueError(mode)


def draft_probs(wl: Workload, node_rows: np.ndarray, all_draft: torch.Tensor,
                temperatures: np.ndarray, device="cpu") -> torch.Tensor:
    """q [b*n, V] fp32: the draft model's distribution at each expanded node,
    softmax(draft_row / T) in fp32 (T = 1 for greedy requests); zero rows for
    nodes that were never expanded.  This stands in for the draft model's own
    output distribution, which the draft forward pass would provide."""
    rows = wl.b * wl.n
    idx = torch.as_tensor(node_rows, device=device)
    has = idx >= 0
    t = torch.as_tensor(temperatures, device=device).float()
    t = torch.where(t > 0, t, torch.ones_like(t)).repeat_interleave(wl.n)
    q = torch.zeros((rows, wl.V), device=device, dtype=torch.float32)
    sel = torch.nonzero(has).flatten()
    for chunk in torch.split(sel, 256):
        src = all_draft.index_select(0, idx[chunk]).float() / t[chunk, None]
        q[chunk] = torch.softmax(src, dim=-1)
    return q


def coins(wl: Workload, device="cpu", seed: int = 0):
    """u [b*n] (one coin per child node) and u_final [b], uniform in [0, 1)."""
    u = uniform((wl.b * wl.n,), device, _gen(device, seed, wl, "u"))
    uf = uniform((wl.b,), device, _gen(device, seed, wl, "u_final"))
    return u, uf


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor, on the host."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def host(t) -> np.ndarray:
    """A host numpy array for an fp32 / int tensor, or bf16 bit patterns."""
    if isinstance(t, np.ndarray):
        return t
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.detach().cpu().contiguous().numpy()
