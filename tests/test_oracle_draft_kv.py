"""Oracle pins for the draft side of the KV (CPU only).

[SGL-XI prepare_for_draft]: with page_size 1 or topk 1 every draft branch
writes contiguous slots after the prefix (and with topk 1 the first draft
row's position comes out of the same call); with page_size > 1 and topk > 1
each branch gets a page-aligned region whose first slots are holes over the
prefix's last partial page, and the real prefix-tail KV is copied into them
"so whole-page reads stay coherent".  [SGL-XI, the three mask forms]: the
FULL_MASK verify mask gives each verify row the whole prefix plus its tree
columns, and fill_prefix_mask controls whether the prefix columns are written.

The pins check the purposes the pages state, not the index formulas: a reader
of whole pages sees, for every branch, the prefix followed by that branch's
draft rows; the FULL_MASK, used as a dense mask by a plain attention, gives the
oracle's tree attention.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _paged_request(L, S, topk, page, rng, extra_pages=2):
    """One request's req_to_token row over randomly permuted pages: the
    prefix, then room for topk page-aligned branch regions."""
    last = L % page
    base = L - last
    R = -(-(last + S) // page) * page
    need = base + topk * R if (page > 1 and topk > 1) else L + topk * S
    pages = -(-need // page) + extra_pages
    perm = rng.permutation(pages + 5)[:pages]
    row = (perm[np.arange(pages * page) // page] * page + np.arange(pages * page) % page).astype(np.int32)
    return row[None, :], (pages + 5) * page, base, last, R


@pytest.mark.parametrize("L,S,topk,page", [(37, 5, 3, 16), (48, 3, 4, 16), (5, 20, 2, 16), (33, 4, 2, 8)])
def test_paged_branches_read_whole_pages_coherently(L, S, topk, page):
    """After assign + duplicate, reading branch t's pages whole -- the
    prefix's full pages, then the branch's region -- yields the prefix's KV
    for positions 0..L-1 followed by the branch's own draft slots; regions are
    page-aligned, disjoint, and the draft slots distinct."""
    rng = np.random.default_rng(L + S)
    Hkv, D = 2, 8
    r2t, num_slots, base, last, R = _paged_request(L, S, topk, page, rng)
    k = rng.integers(0, 60000, (num_slots, Hkv, D)).astype(np.uint16)
    v = rng.integers(0, 60000, (num_slots, Hkv, D)).astype(np.uint16)
    k0, v0 = k.copy(), v.copy()
    o = oracle.assign_draft_locs(1, topk, S, page, r2t, [0], [L], num_slots)
    loc = o["out_cache_loc"].reshape(topk, S)
    oracle.duplicate_prefix_tail(1, topk, S, page, Hkv, D, [k], [v], r2t, [0], [L])
    assert len(set(loc.ravel().tolist())) == topk * S
    row = r2t[0]
    prefix_slots = row[:L]
    for t in range(topk):
        start = base + t * R
        assert start % page == 0
        region = row[start:start + R]
        # whole pages of the branch: the prefix's full pages, then the region's pages
        seen = np.concatenate([row[:base], region])
        kv_k = k[seen]
        expect_prefix = k0[prefix_slots]
        np.testing.assert_array_equal(kv_k[:L], expect_prefix, err_msg=f"branch {t}: prefix as read by pages")
        np.testing.assert_array_equal(v[seen][:L], v0[prefix_slots])
        # then the branch's draft slots, in step order
        np.testing.assert_array_equal(seen[L:L + S], loc[t])
    # the regions do not overlap one another, nor the prefix
    regions = [set(row[base + t * R: base + (t + 1) * R].tolist()) for t in range(topk)]
    for t in range(1, topk):
        assert not (regions[t] & set(prefix_slots.tolist()))
        for u in range(t):
            assert not (regions[t] & regions[u])
    # nothing outside the holes of branches 1.. changed
    changed = np.nonzero((k != k0).any(axis=(1, 2)))[0]
    holes = {int(row[base + t * R + j]) for t in range(1, topk) for j in range(last)}
    assert set(changed.tolist()) <= holes


@pytest.mark.parametrize("topk,page", [(1, 16), (4, 1), (1, 1)])
def test_contiguous_branches_after_the_prefix(topk, page):
    """page_size 1 or topk 1: every branch writes a contiguous run of the
    request's own positions after the prefix, the runs side by side; topk 1
    returns the first draft row's position, the prefix length.  No prefix
    slot is ever handed out, no slot twice."""
    rng = np.random.default_rng(topk * 10 + page)
    b, S = 3, 5
    L = np.array([7, 16, 30], np.int32)
    row_w = 64
    slots = rng.permutation(b * row_w).astype(np.int32).reshape(b, row_w)
    req_pool_idx = np.array([2, 0, 1], np.int32)
    r2t = np.empty_like(slots)
    r2t[req_pool_idx] = slots
    o = oracle.assign_draft_locs(b, topk, S, page, r2t, req_pool_idx, L, b * row_w)
    loc = o["out_cache_loc"].reshape(b, topk, S)
    assert len(set(loc.ravel().tolist())) == loc.size
    for q in range(b):
        pos_of = {int(s): p for p, s in enumerate(r2t[req_pool_idx[q]])}
        pos = np.array([[pos_of[int(s)] for s in loc[q, t]] for t in range(topk)])
        assert pos.min() == L[q]                                   # right after the prefix
        assert (np.diff(pos.ravel()) == 1).all()                   # contiguous, branch after branch
    if topk == 1:
        np.testing.assert_array_equal(o["positions"], L)


def test_assign_rejects_rows_too_short():
    r2t = np.arange(20, dtype=np.int32)[None, :]
    with pytest.raises(oracle.OracleError):
        oracle.assign_draft_locs(1, 2, 8, 1, r2t, [0], [10], 20)


def _matrug():
    from tests.helpers import golden
    fx = golden("matrug_draft.json")
    return fx


def test_full_mask_matrug_rows():
    """The mat/rug tree (mask rows 0x01, 0x03, 0x05, 0x0B, 0x13, 0x25): each verify
    row sees the whole prefix and exactly its ancestors and itself."""
    bits = np.array([0x01, 0x03, 0x05, 0x0B, 0x13, 0x25], np.uint64)
    L, n = 7, 6
    m = oracle.full_mask(1, n, [L], bits).reshape(n, L + n)
    assert (m[:, :L] == 1).all()
    expect = [[1, 0, 0, 0, 0, 0], [1, 1, 0, 0, 0, 0], [1, 0, 1, 0, 0, 0],
              [1, 1, 0, 1, 0, 0], [1, 1, 0, 0, 1, 0], [1, 0, 1, 0, 0, 1]]
    assert m[:, L:].tolist() == expect


def test_full_mask_without_prefix_fill_keeps_the_prefix_columns():
    """fill_prefix_mask off: the prefix columns keep what the reused buffer
    held; every tree column is written."""
    bits = np.array([1, 3, 5, 1, 3, 7], np.uint64)
    L = [4, 2]
    n = 3
    total = sum(n * (x + n) for x in L)
    buf = np.full(total, 9, np.uint8)
    m = oracle.full_mask(2, n, L, bits, fill_prefix=False, out=buf)
    off = 0
    for q in range(2):
        blk = m[off: off + n * (L[q] + n)].reshape(n, L[q] + n)
        assert (blk[:, :L[q]] == 9).all()
        assert set(blk[:, L[q]:].ravel().tolist()) <= {0, 1}
        off += n * (L[q] + n)


def test_full_mask_as_a_dense_mask_gives_the_tree_attention():
    """Used as a dense boolean mask over [prefix keys, tree keys] by a plain
    masked softmax attention (torch, fp64), the FULL_MASK blocks reproduce the
    oracle's tree attention for every row and head."""
    from accept_select_top_gb300 import workloads as W
    from oracle import pipeline as P
    wl = W.scaled(W.WORKLOADS["tiny"], name="fullmask", b=3, V=256, ctx=("uniform", 9, 30))
    drafts = [W.host(W.draft_logits(wl, i)) for i in range(wl.S)]
    lay = W.kv_layout(wl)
    tree = P.tree_from_chain(wl, P.select_chain(wl, drafts), W.host(W.bonus_tokens(wl)), lay["seq_lens"])
    att = W.attention_tensors(wl, int(lay["num_slots"]))
    q, kp, vp = (W.host(att[x]) for x in ("q", "k_pool", "v_pool"))
    ref = oracle.verify_attention(wl.b, wl.n, wl.Hq, wl.Hkv, wl.D, q, kp, vp, lay["req_to_token"],
                                  lay["req_pool_idx"], lay["seq_lens"], lay["verify_loc"], tree["mask_bits"],
                                  1.0 / math.sqrt(wl.D))["out"]
    m = oracle.full_mask(wl.b, wl.n, lay["seq_lens"], tree["mask_bits"])
    f = lambda bits: torch.from_numpy((bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    Q, K, Vv = f(q), f(kp), f(vp)
    G = wl.Hq // wl.Hkv
    off = 0
    for r in range(wl.b):
        L = int(lay["seq_lens"][r])
        blk = torch.from_numpy(m[off: off + wl.n * (L + wl.n)].reshape(wl.n, L + wl.n).astype(bool))
        off += wl.n * (L + wl.n)
        keys = np.concatenate([lay["req_to_token"][lay["req_pool_idx"][r], :L],
                               lay["verify_loc"][r * wl.n:(r + 1) * wl.n]])
        for h in range(wl.Hq):
            qq = Q[r * wl.n:(r + 1) * wl.n, h]                     # [n, D]
            kk = K[keys, h // G]
            vv = Vv[keys, h // G]
            s = (qq @ kk.T) / math.sqrt(wl.D)
            s = s.masked_fill(~blk, float("-inf"))
            out = torch.softmax(s, dim=-1) @ vv
            np.testing.assert_allclose(out.numpy(), ref[r * wl.n:(r + 1) * wl.n, h], rtol=1e-9, atol=1e-12)
