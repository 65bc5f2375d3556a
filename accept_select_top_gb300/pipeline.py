"""One verify step on the GPU: buffers for a workload and the call sequence

    spec_select_topk x S -> spec_build_tree -> spec_verify_attention ->
    spec_verify_greedy | spec_verify_sampling -> spec_commit_kv

Every call goes through the C ABI (``ops``); this module only allocates the
caller-owned buffers (torch) and passes pointers.  The select steps write their
score / token blocks straight into the concatenated score and token spaces and
their parent blocks into the parent list, so no concatenation runs between the
steps.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional

import torch

from . import ops
from .workloads import Workload


class DeviceInputs:
    """Device tensors of one step's inputs."""

    def __init__(self, drafts: List[torch.Tensor], bonus: torch.Tensor, seq_lens: torch.Tensor,
                 req_pool_idx: torch.Tensor, req_to_token: torch.Tensor, verify_loc: torch.Tensor,
                 q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, max_seq_len: int,
                 target_logits: Optional[torch.Tensor] = None, draft_probs: Optional[torch.Tensor] = None,
                 temperatures: Optional[torch.Tensor] = None, u: Optional[torch.Tensor] = None,
                 u_final: Optional[torch.Tensor] = None):
        self.drafts = drafts
        self.bonus = bonus
        self.seq_lens = seq_lens
        self.req_pool_idx = req_pool_idx
        self.req_to_token = req_to_token
        self.verify_loc = verify_loc
        self.q = q
        self.k_pool = k_pool
        self.v_pool = v_pool
        self.max_seq_len = int(max_seq_len)
        self.target_logits = target_logits
        self.draft_probs = draft_probs
        self.temperatures = temperatures
        self.u = u
        self.u_final = u_final


class VerifyStep:
    def __init__(self, wl: Workload, inp: DeviceInputs, mode: str = "greedy", device="cuda",
                 draft_temperature: float = 1.0, with_lse: bool = True, overlap: bool = False,
                 chain: Optional[bool] = None):
        assert mode in ("greedy", "sampling")
        self.wl, self.inp, self.mode = wl, inp, mode
        # the chain fast path: topk = 1 with num_draft_tokens = num_steps + 1
        # (the tree is the chain of the S selected tokens)
        is_chain = wl.k == 1 and wl.n == wl.S + 1
        self.chain = is_chain if chain is None else bool(chain)
        if self.chain and not is_chain:
            raise ValueError("the chain fast path needs topk = 1 and num_draft_tokens = num_steps + 1")
        self.draft_temperature = draft_temperature
        b, k, S, n, W = wl.b, wl.k, wl.S, wl.n, wl.W
        i32, f32 = torch.int32, torch.float32
        z = lambda shape, dt: torch.zeros(shape, dtype=dt, device=device)
        self.score_space = z((b, wl.C), f32)
        self.token_space = z((b, wl.C), i32)
        self.parent_space = z((b, wl.P), i32)
        self.last_parent = z((b, k + 1), i32)  # k+1 columns: the last step may be step 0
        self.scores = [z((b, k), f32), z((b, k), f32)]
        self.next_ids = z((b * k,), i32)
        self.draft_tokens = z((b * n,), i32)
        self.positions = z((b * n,), i32)
        self.retrieve_index = z((b * n,), i32)
        self.next_token = z((b * n,), i32)
        self.next_sibling = z((b * n,), i32)
        self.mask_bits = z((b * n,), torch.int64)  # uint64 bit patterns
        self.out = z((b * n, wl.Hq, wl.D), torch.bfloat16)
        self.lse = z((b * n, wl.Hq), f32) if with_lse else None
        self.predict = z((b * n,), i32)
        self.accept_index = z((b, W), i32)
        self.accept_lens = z((b,), i32)
        self.accepted_tokens = z((b, W), i32)
        self.next_root = z((b,), i32)
        self.new_seq_lens = z((b,), i32)
        self.correct_len = z((b,), i32)  # chain greedy accept: leading matches
        self.free_ids = z((max(1, b * n),), i32)
        self.n_free = z((1,), i32)
        nbytes = max(ops.spec_workspace_size(op, b, n, k, wl.V, wl.Hq, wl.Hkv, inp.max_seq_len)
                     for op in range(6))
        self.ws = ops.Workspace(nbytes, device=device)
        # overlap asserts that every draft-logits / target-logits input is
        # complete before the previous call is enqueued (true when all inputs
        # are resident up front, as in a benchmark; false in an EAGLE loop,
        # where the draft forward and the target's LM head run in between)
        self.overlap = bool(overlap)
        self.ws.set_overlap(self.overlap)
        # select step i writes its blocks at these offsets of the score / parent spaces
        self.score_off = [0 if i == 0 else k + (i - 1) * k * k for i in range(S)]
        # parent list = [-1, 0..k-1] (step 0, k+1 entries), then k entries per later step
        self.parent_off = [0 if i == 0 else 1 + i * k for i in range(S)]

    # ----------------------------------------------------------- the calls
    def select_step(self, i: int, stream=None):
        """Draft step i of select_top_k_tokens (one spec_select_topk call)."""
        wl, k = self.wl, self.wl.k
        last = i == wl.S - 1
        pblk = _view_from(self.last_parent, 0) if last else _view_from(self.parent_space, self.parent_off[i])
        ops.spec_select_topk(
            i, wl.b, k, self.inp.drafts[i], self.draft_temperature,
            None if i == 0 else self.scores[(i - 1) % 2],
            _view_from(self.score_space, self.score_off[i]), _view_from(self.token_space, self.score_off[i]),
            wl.C, pblk, (k + 1 if i == 0 else k) if last else wl.P,
            self.scores[i % 2], self.next_ids, None, self.ws, stream)

    def select(self, stream=None):
        for i in range(self.wl.S):
            self.select_step(i, stream)

    def build(self, stream=None):
        wl = self.wl
        if self.chain:
            # for topk = 1 the token space holds the S chain tokens, in order
            ops.spec_build_chain_tree(wl.b, wl.S, self.inp.bonus, self.token_space, wl.C, self.inp.seq_lens,
                                      self.draft_tokens, self.positions, self.retrieve_index, self.next_token,
                                      self.next_sibling, self.mask_bits, stream)
            return
        ops.spec_build_tree(wl.b, wl.k, wl.S, wl.n, self.score_space, self.token_space, self.parent_space,
                            self.inp.bonus, self.inp.seq_lens, self.draft_tokens, self.positions,
                            self.retrieve_index, self.next_token, self.next_sibling, self.mask_bits, self.ws, stream)

    def attention(self, stream=None):
        wl, inp = self.wl, self.inp
        ops.spec_verify_attention(wl.b, wl.n, wl.Hq, wl.Hkv, wl.D, wl.page_size, inp.q, inp.k_pool, inp.v_pool,
                                  inp.req_to_token, inp.req_pool_idx, inp.seq_lens, inp.max_seq_len,
                                  inp.verify_loc, self.mask_bits, 1.0 / math.sqrt(wl.D), self.out, self.lse,
                                  self.ws, stream)

    def accept(self, stream=None):
        wl, inp = self.wl, self.inp
        tree = (self.draft_tokens, self.retrieve_index, self.next_token, self.next_sibling)
        outs = (self.predict, self.accept_index, self.accept_lens, self.accepted_tokens, self.next_root)
        if self.mode == "greedy" and self.chain:
            # DSpark counts: commit_lens is accept_lens, the out tokens are the
            # accepted tokens, the bonus is the next root
            ops.spec_verify_chain_greedy(wl.b, wl.S, inp.target_logits, self.token_space, wl.C, inp.seq_lens,
                                         self.correct_len, self.next_root, self.accepted_tokens, self.accept_lens,
                                         self.new_seq_lens, self.accept_index, self.ws, stream)
        elif self.mode == "greedy":
            ops.spec_verify_greedy(wl.b, wl.n, wl.S, inp.target_logits, *tree, *outs, self.ws, stream)
        else:
            ops.spec_verify_sampling(wl.b, wl.n, wl.S, inp.target_logits, inp.draft_probs, inp.temperatures,
                                     inp.u, inp.u_final, *tree, *outs, self.ws, stream)

    def commit(self, stream=None):
        wl, inp = self.wl, self.inp
        ops.spec_commit_kv(wl.b, wl.n, wl.W, wl.Hkv, wl.D, wl.page_size, [inp.k_pool], [inp.v_pool],
                           inp.req_to_token, inp.req_pool_idx, inp.seq_lens, inp.verify_loc, self.accept_index,
                           self.accept_lens, self.new_seq_lens, self.free_ids, self.n_free, self.ws, stream)

    def run(self, stream=None):
        self.select(stream)
        self.build(stream)
        self.attention(stream)
        self.accept(stream)
        self.commit(stream)

    def launches_per_step(self) -> int:
        return launches_per_step(self.wl, self.mode)


STREAM_MIN_BYTES = 32 << 20  # the select's streaming pass from this many bytes of logits a call


def select_launches(wl: Workload, step: int) -> int:
    """Kernels spec_select_topk launches at draft step `step`: rows of whole
    16-byte vectors, at least one streaming unit (256 vectors) and at most 254
    units long, and at least 32 MiB of logits in the call (the buffers here
    are aligned), take the streaming pass and its request step; other calls
    the chunked kernel alone."""
    elem = 4 if wl.logits_dtype == "f32" else 2
    vecs = wl.V * elem // 16
    rows = wl.b * (wl.k if step else 1)
    ok = (wl.V * elem) % 16 == 0 and 256 <= vecs and (vecs // 256 + 2) <= 256
    return 2 if ok and rows * wl.V * elem >= STREAM_MIN_BYTES else 1


def sampling_launches(wl: Workload) -> int:
    """Kernels the sampling accept launches: the streaming pass, the row
    statistics and the terminal pass where its logit rows take the streaming
    pass, else the chunked statistics pass and the terminal pass."""
    elem = 4 if wl.logits_dtype == "f32" else 2
    vecs = wl.V * elem // 16
    ok = (wl.V * elem) % 16 == 0 and 256 <= vecs and (vecs // 256 + 2) <= 256
    return 3 if ok else 2


def launches_per_step(wl: Workload, mode: str) -> int:
    """Kernels one VerifyStep.run() launches: S selects, the tree build (the
    generic or the chain kernel), the attention (one launch: split key lists
    are merged inside it), the accept (greedy one launch, sampling two or
    three) and the KV commit."""
    selects = sum(select_launches(wl, i) for i in range(wl.S))
    return selects + 1 + 1 + (1 if mode == "greedy" else sampling_launches(wl)) + 1


def _view_from(t: torch.Tensor, offset: int) -> torch.Tensor:
    """A flat view of ``t`` starting ``offset`` elements into its first row
    (the callee addresses rows with its own leading dimension)."""
    flat = t.view(-1)
    return flat[offset:]
