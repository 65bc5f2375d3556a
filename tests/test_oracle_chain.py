"""Oracle pins for the chain fast path (topk = 1), CPU only.

build_chain_tree writes the constant structure of a chain (a lower-triangular
mask, linear parents) [SGL-XI, platform dispatch and the chain
specialisation]; the DSpark greedy accept counts correct_len, the bonus, the
fixed-width out tokens and commit_lens = correct_len + 1 [ACCEPT section 5].
The chain tree is pinned against the generic organize + build on topk = 1
select chains and the pages' chain example; the chain accept against the
pages' DSpark counts, the stop-at-first-mismatch rule, and the tree walk.
"""
import numpy as np
import pytest

import oracle
from accept_select_top_gb300 import workloads as W
from oracle import pipeline as P
from tests.helpers import golden, onehot_logits


@pytest.mark.parametrize("S", [1, 3, 5])
def test_chain_tree_equals_generic_build_for_topk1(S):
    """With topk = 1 the generic path selects all S candidates and builds a
    chain; the chain fast path must give the same arrays."""
    wl = W.scaled(W.WORKLOADS["mtp_chain"], name=f"chain{S}", b=6, S=S, n=S + 1, V=300, logits_dtype="f32")
    drafts = [W.host(W.draft_logits(wl, i)) for i in range(S)]
    lay = W.kv_layout(wl)
    bonus = W.host(W.bonus_tokens(wl))
    ch = P.select_chain(wl, drafts)
    gen = P.tree_from_chain(wl, ch, bonus, lay["seq_lens"])
    assert ch["token_space"].shape == (wl.b, S)  # the chain's draft tokens
    fast = oracle.build_chain_tree(wl.b, S, bonus, ch["token_space"], lay["seq_lens"])
    for k in ("draft_tokens", "positions", "retrieve_index", "next_token", "next_sibling", "mask_bits"):
        np.testing.assert_array_equal(fast[k], gen[k], err_msg=k)


def test_chain_example_positions_and_mask():
    """The/cat/sat/on at positions L..L+3, each row seeing itself and every
    node before it (a lower-triangular mask)."""
    fx = golden("chain_topk1.json")
    tok = fx["tokens"]
    t = oracle.build_chain_tree(1, fx["S"], [tok[fx["root"]]], [[tok[x] for x in fx["draft_chain"]]], [fx["L"]])
    assert (t["positions"] - fx["L"]).tolist() == fx["expect"]["positions_offset"]
    assert t["mask_bits"].tolist() == [0b1, 0b11, 0b111, 0b1111]
    assert t["next_token"].tolist() == [1, 2, 3, -1] and t["next_sibling"].tolist() == [-1] * 4
    assert t["draft_tokens"].tolist() == [tok[x] for x in [fx["root"]] + fx["draft_chain"]]


def _dspark():
    fx = golden("chain_commit.json")
    tok = fx["tokens"]
    drafts = [[tok[x] for x in fx["nodes"][1:]]]
    logits = onehot_logits([tok[x] for x in fx["target_argmax"]], 8)
    return fx, tok, drafts, logits


def test_dspark_counts():
    fx, tok, drafts, logits = _dspark()
    o = oracle.chain_accept_greedy(1, 3, logits, drafts, [fx["prefix"]])
    ex = fx["expect"]
    assert o["correct_len"][0] == ex["correct_len"]
    assert o["commit_lens"][0] == ex["commit_lens"]
    assert o["new_seq_lens"][0] == ex["new_seq_len"]
    assert o["bonus"][0] == tok["X"]
    # out tokens: A, B, then the bonus X scattered at correct_len; only the first commit_lens are output
    assert o["out_tokens"][0, : ex["commit_lens"]].tolist() == [tok[x] for x in ex["accepted_tokens"]]
    assert o["out_tokens"][0].tolist() == [tok["A"], tok["B"], tok["X"], -1]
    rows = o["accept_index"][0, : ex["commit_lens"]]
    assert [fx["nodes"][r] for r in rows] == ex["committed_rows"]
    assert o["accept_index"][0, ex["commit_lens"]:].tolist() == [-1]


def test_a_later_match_does_not_resume():
    """Draft A, Y, C against target A, B, C: the mismatch at position 1 ends the
    accept although position 2 would match."""
    V = 8
    o = oracle.chain_accept_greedy(1, 3, onehot_logits([2, 3, 4, 5], V), [[2, 7, 4]], [0])
    assert o["correct_len"][0] == 1 and o["bonus"][0] == 3
    assert o["out_tokens"][0].tolist() == [2, 3, 4, -1]
    # every position matches: the bonus is the target at the last row
    o = oracle.chain_accept_greedy(1, 3, onehot_logits([2, 3, 4, 5], V), [[2, 3, 4]], [7])
    assert o["correct_len"][0] == 3 and o["bonus"][0] == 5 and o["new_seq_lens"][0] == 11
    assert o["out_tokens"][0].tolist() == [2, 3, 4, 5]


@pytest.mark.parametrize("seed", range(3))
def test_chain_accept_equals_tree_walk(seed):
    """On a chain tree the greedy tree walk and the DSpark counts agree:
    accept_lens = commit_lens, accepted tokens = the first commit_lens out
    tokens, the same accept_index, next_root = bonus."""
    rng = np.random.default_rng(seed)
    b, S, V = 20, 4, 16
    n = S + 1
    logits = rng.normal(0, 1, (b * n, V)).astype(np.float32)
    tp = logits.argmax(-1).reshape(b, n)
    drafts = rng.integers(0, V, (b, S)).astype(np.int32)
    agree = rng.random((b, S)) < 0.7
    drafts[agree] = tp[:, :S][agree]  # mostly matching chains
    bonus = rng.integers(0, V, b).astype(np.int32)
    tree = oracle.build_chain_tree(b, S, bonus, drafts, np.zeros(b, np.int32))
    g = oracle.verify_greedy(b, n, S, logits, tree["draft_tokens"], tree["retrieve_index"], tree["next_token"],
                             tree["next_sibling"])
    o = oracle.chain_accept_greedy(b, S, logits, drafts, np.arange(b))
    np.testing.assert_array_equal(g["accept_lens"], o["commit_lens"])
    np.testing.assert_array_equal(g["accept_index"], o["accept_index"])
    np.testing.assert_array_equal(g["next_root"], o["bonus"])
    for r in range(b):
        L = o["commit_lens"][r]
        assert g["accepted_tokens"][r, :L].tolist() == o["out_tokens"][r, :L].tolist()
    np.testing.assert_array_equal(o["new_seq_lens"], np.arange(b) + o["commit_lens"])
