"""Oracle pins for tree-masked verify attention and the KV commit (CPU only)."""
import numpy as np
import pytest
import torch

import oracle
from accept_select_top_gb300 import workloads as W
from oracle import pipeline as P
from tests.helpers import golden


def _bits_to_f64(a):
    return torch.from_numpy(np.ascontiguousarray(a).astype(np.uint32) << 16).view(torch.float32).double()


def _case(Hq=4, Hkv=2, D=64, seed=0, k=2, S=3, n=6, ctx=("uniform", 20, 60), page=1, layout="inplace"):
    wl = W.scaled(W.WORKLOADS["tiny"], name=f"att{seed}", Hq=Hq, Hkv=Hkv, D=D, k=k, S=S, n=n, ctx=ctx,
                  page_size=page, verify_layout=layout, slot_order="permuted")
    drafts = [W.host(W.draft_logits(wl, i, seed=seed)) for i in range(wl.S)]
    lay = W.kv_layout(wl, seed=seed)
    ch = P.select_chain(wl, drafts)
    tree = P.tree_from_chain(wl, ch, np.zeros(wl.b, np.int32), lay["seq_lens"])
    att = W.attention_tensors(wl, int(lay["num_slots"]), seed=seed)
    return wl, lay, tree, {k_: W.host(v) for k_, v in att.items()}


def _sdpa_reference(wl, lay, tree, att, row, h):
    """torch SDPA (fp64) over an explicit key list: the request's prefix slots
    and the slots of the node's ancestors (walked from parent pointers) and
    itself."""
    n = wl.n
    b, i = divmod(row, n)
    g = h // (wl.Hq // wl.Hkv)
    req = lay["req_pool_idx"][b]
    slots = list(lay["req_to_token"][req, : lay["seq_lens"][b]])
    par = tree["parent_node"]
    chain, a = [], i
    while a != -1:
        chain.append(a)
        a = par[b * n + a]
    slots += [lay["verify_loc"][b * n + j] for j in sorted(chain)]
    kp = _bits_to_f64(att["k_pool"])
    vp = _bits_to_f64(att["v_pool"])
    q = _bits_to_f64(att["q"][row, h])[None, None, None, :]
    K = kp[slots, g][None, None]
    V = vp[slots, g][None, None]
    return torch.nn.functional.scaled_dot_product_attention(q, K, V, scale=1.0 / np.sqrt(wl.D))[0, 0, 0].numpy()


@pytest.mark.parametrize("seed", range(3))
def test_attention_matches_sdpa_on_ancestor_keys(seed):
    wl, lay, tree, att = _case(seed=seed)
    o = oracle.verify_attention(wl.b, wl.n, wl.Hq, wl.Hkv, wl.D, att["q"], att["k_pool"], att["v_pool"],
                                lay["req_to_token"], lay["req_pool_idx"], lay["seq_lens"], lay["verify_loc"],
                                tree["mask_bits"], 1.0 / np.sqrt(wl.D))
    for row in range(wl.b * wl.n):
        for h in range(wl.Hq):
            ref = _sdpa_reference(wl, lay, tree, att, row, h)
            np.testing.assert_allclose(o["out"][row, h], ref, rtol=1e-10, atol=1e-12)


def test_attention_chain_is_causal_and_n1_is_decode():
    """topk=1 chain: the tree mask is causal over prefix + chain (torch SDPA
    with a boolean causal mask); n=1: plain decode attention over the prefix
    and the node itself."""
    wl, lay, tree, att = _case(k=1, S=3, n=4, seed=5)
    o = oracle.verify_attention(wl.b, wl.n, wl.Hq, wl.Hkv, wl.D, att["q"], att["k_pool"], att["v_pool"],
                                lay["req_to_token"], lay["req_pool_idx"], lay["seq_lens"], lay["verify_loc"],
                                tree["mask_bits"], 1.0 / np.sqrt(wl.D))
    kp, vp = _bits_to_f64(att["k_pool"]), _bits_to_f64(att["v_pool"])
    for b in range(wl.b):
        L = lay["seq_lens"][b]
        slots = list(lay["req_to_token"][lay["req_pool_idx"][b], :L]) + list(lay["verify_loc"][b * 4:(b + 1) * 4])
        mask = torch.ones(4, L + 4, dtype=torch.bool)
        mask[:, L:] = torch.tril(torch.ones(4, 4, dtype=torch.bool))
        for h in range(wl.Hq):
            g = h // (wl.Hq // wl.Hkv)
            q = _bits_to_f64(att["q"][b * 4:(b + 1) * 4, h])[None, None]
            ref = torch.nn.functional.scaled_dot_product_attention(
                q, kp[slots, g][None, None], vp[slots, g][None, None], attn_mask=mask, scale=1 / np.sqrt(wl.D))
            np.testing.assert_allclose(o["out"][b * 4:(b + 1) * 4, h], ref[0, 0].numpy(), rtol=1e-10, atol=1e-12)
    # n = 1: the verify step degenerates to one decode query per request
    wl1, lay1, tree1, att1 = _case(k=1, S=1, n=1, seed=6)
    assert tree1["mask_bits"].tolist() == [1] * wl1.b
    o1 = oracle.verify_attention(wl1.b, 1, wl1.Hq, wl1.Hkv, wl1.D, att1["q"], att1["k_pool"], att1["v_pool"],
                                 lay1["req_to_token"], lay1["req_pool_idx"], lay1["seq_lens"],
                                 lay1["verify_loc"], tree1["mask_bits"], 1.0 / np.sqrt(wl1.D))
    kp1, vp1 = _bits_to_f64(att1["k_pool"]), _bits_to_f64(att1["v_pool"])
    for b in range(wl1.b):
        slots = list(lay1["req_to_token"][lay1["req_pool_idx"][b], :lay1["seq_lens"][b]]) + [lay1["verify_loc"][b]]
        for h in range(wl1.Hq):
            g = h // (wl1.Hq // wl1.Hkv)
            ref = torch.nn.functional.scaled_dot_product_attention(
                _bits_to_f64(att1["q"][b, h])[None, None, None], kp1[slots, g][None, None], vp1[slots, g][None, None],
                scale=1 / np.sqrt(wl1.D))
            np.testing.assert_allclose(o1["out"][b, h], ref[0, 0, 0].numpy(), rtol=1e-10, atol=1e-12)


def test_attention_pairs_subset_and_lse():
    wl, lay, tree, att = _case(seed=2)
    args = (wl.b, wl.n, wl.Hq, wl.Hkv, wl.D, att["q"], att["k_pool"], att["v_pool"], lay["req_to_token"],
            lay["req_pool_idx"], lay["seq_lens"], lay["verify_loc"], tree["mask_bits"], 1.0 / np.sqrt(wl.D))
    full = oracle.verify_attention(*args)
    pairs = np.array([[0, 0], [7, 3], [wl.b * wl.n - 1, 1]])
    part = oracle.verify_attention(*args, pairs=pairs)
    for r, h in pairs:
        np.testing.assert_array_equal(part["out"][r, h], full["out"][r, h])
        assert part["lse"][r, h] == full["lse"][r, h]
    assert np.isnan(part["out"][1, 0]).all()
    # lse = log sum exp of the scaled scores (torch.logsumexp over the same keys)
    kp = _bits_to_f64(att["k_pool"])
    row, h = 7, 3
    b, i = divmod(row, wl.n)
    g = h // (wl.Hq // wl.Hkv)
    slots = list(lay["req_to_token"][lay["req_pool_idx"][b], :lay["seq_lens"][b]])
    slots += [lay["verify_loc"][b * wl.n + j] for j in range(wl.n) if (int(tree["mask_bits"][row]) >> j) & 1]
    s = (kp[slots, g] @ _bits_to_f64(att["q"][row, h])) / np.sqrt(wl.D)
    assert abs(torch.logsumexp(s, 0).item() - full["lse"][row, h]) < 1e-10


# ------------------------------------------------------------------ commit

def _pools(num_slots, Hkv=1, D=4):
    """Pools whose every slot holds its own id, so moved rows are recognisable."""
    k = np.repeat(np.arange(num_slots, dtype=np.uint16)[:, None, None], Hkv * D, 2).reshape(num_slots, Hkv, D).copy()
    v = (k + 30000).astype(np.uint16)
    return k, v


def test_commit_rabcd_prefix_10():
    """R/A/B/C/D in the next positions 10..14 of an in-place layout; accepted
    rows R, A, C land at positions 10, 11, 12; new length 13; the slots of C and
    D are released (C's KV now lives in B's old slot)."""
    fx = golden("rabcd_greedy.json")
    chain = golden("chain_commit.json")
    slots = np.array([7, 3, 9, 2, 8, 5, 1, 0, 6, 4, 15, 11, 14, 10, 13, 12], np.int32)
    r2t = slots[None, :]
    verify_loc = slots[10:15]
    k, v = _pools(16)
    k0 = k.copy()
    acc_rows = np.array([fx["expect"]["accept_rows"] + [-1]], np.int32)
    o = oracle.commit_kv(1, 5, 4, 1, 4, 1, [k], [v], r2t, [0], [10], verify_loc, acc_rows, [3])
    assert o["new_seq_lens"].tolist() == [chain["expect"]["new_seq_len"]]
    names = fx["nodes"]
    committed = [names[list(verify_loc).index(int(k[slots[10 + j], 0, 0]))] for j in range(3)]
    assert committed == fx["expect"]["committed_rows"]
    assert o["free_ids"].tolist() == [verify_loc[3], verify_loc[4]]
    untouched = np.setdiff1d(np.arange(16), slots[10:13])
    np.testing.assert_array_equal(k[untouched], k0[untouched])


def test_commit_gather_before_scatter():
    """dst of the first accepted row is the src of the second: the rows must
    swap, which a row-by-row copy would not do."""
    slots = np.arange(8, dtype=np.int32)
    r2t = slots[None, :]
    # verify node 0 sits at position 5's slot, node 1 at position 4's slot
    verify_loc = np.array([5, 4, 6], np.int32)
    k, v = _pools(8)
    o = oracle.commit_kv(1, 3, 3, 1, 4, 1, [k], [v], r2t, [0], [4], verify_loc, np.array([[0, 1, -1]]), [2])
    assert k[4, 0, 0] == 5 and k[5, 0, 0] == 4
    assert v[4, 0, 0] == 30005 and v[5, 0, 0] == 30004
    assert o["free_ids"].tolist() == [6]


def test_commit_page16_scratch_pages():
    """Page size 16: seq_len 20 leaves 4 hole slots at the head of the verify
    scratch page; the accepted rows are copied into the request's own tail page
    and the scratch pages are released whole, once each."""
    ps = 16
    own_pages = [3, 0]          # positions 0..31 -> pages 3, 0
    scratch = [5, 2]            # verify nodes: offsets 4..19 of the scratch pages
    r2t = np.array([[p * ps + o for p in own_pages for o in range(ps)]], np.int32)
    n = 14
    off = 4 + np.arange(n)
    verify_loc = (np.array(scratch)[off // ps] * ps + off % ps).astype(np.int32)
    k, v = _pools(6 * ps)
    acc = np.array([[0, 2, 9, -1, -1]], np.int32)
    o = oracle.commit_kv(1, n, 5, 1, 4, ps, [k], [v], r2t, [0], [20], verify_loc, acc, [3])
    assert o["new_seq_lens"].tolist() == [23]
    assert [int(k[r2t[0, 20 + j], 0, 0]) for j in range(3)] == [int(verify_loc[a]) for a in (0, 2, 9)]
    assert o["free_ids"].tolist() == scratch


def test_commit_layers_and_free_invariant():
    """Every layer moves the same rows; free list + committed slots cover the
    verify slots of each request (page size 1, in-place layout)."""
    wl = W.scaled(W.WORKLOADS["tiny"], name="commit", Hkv=2, D=8)
    lay = W.kv_layout(wl)
    rng = np.random.default_rng(3)
    ns = int(lay["num_slots"])
    layers_k = [rng.integers(0, 65535, (ns, 2, 8)).astype(np.uint16) for _ in range(3)]
    layers_v = [rng.integers(0, 65535, (ns, 2, 8)).astype(np.uint16) for _ in range(3)]
    before_k = [x.copy() for x in layers_k]
    # a valid accept path per request: root then nodes 1, 3 (depth-ordered ids)
    acc = np.full((wl.b, wl.W), -1, np.int32)
    lens = np.array([1, 2, 3, 2], np.int32)
    for r in range(wl.b):
        path = [0, 1, 3][: lens[r]]
        acc[r, : lens[r]] = [r * wl.n + x for x in path]
    o = oracle.commit_kv(wl.b, wl.n, wl.W, 2, 8, 1, layers_k, layers_v, lay["req_to_token"], lay["req_pool_idx"],
                         lay["seq_lens"], lay["verify_loc"], acc, lens)
    for L in range(3):
        for r in range(wl.b):
            for j in range(lens[r]):
                dst = lay["req_to_token"][lay["req_pool_idx"][r], lay["seq_lens"][r] + j]
                src = lay["verify_loc"][acc[r, j]]
                np.testing.assert_array_equal(layers_k[L][dst], before_k[L][src])
    fr = set(o["free_ids"].tolist())
    for r in range(wl.b):
        vs = set(lay["verify_loc"][r * wl.n:(r + 1) * wl.n].tolist())
        dsts = {int(lay["req_to_token"][lay["req_pool_idx"][r], lay["seq_lens"][r] + j]) for j in range(lens[r])}
        assert (fr & vs) | dsts >= vs
        assert not (fr & dsts)
    assert o["new_seq_lens"].tolist() == (lay["seq_lens"] + lens).tolist()


def test_commit_rejects_bad_index():
    k, v = _pools(8)
    with pytest.raises(oracle.OracleError):
        oracle.commit_kv(1, 2, 2, 1, 4, 1, [k], [v], np.arange(8)[None], [0], [4], np.array([4, 5]),
                         np.array([[0, 7]]), [2])  # accept row 7 is outside the batch's 2 rows
