"""Oracle pins for draft-tree assembly: softmax/top-k, path scores,
organize_draft_results and build_tree (CPU only)."""
import numpy as np
import pytest
import scipy.special

import oracle
from accept_select_top_gb300 import workloads as W
from oracle import pipeline as P
from tests.helpers import golden


def _ranked_topk(x, k):
    """Library reference: stable sort by descending value keeps the lowest
    index first among equal values."""
    return np.argsort(-x, kind="stable")[:k]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_softmax_topk_matches_library(dtype, T):
    wl = W.scaled(W.WORKLOADS["tiny"], logits_dtype=dtype, b=6)
    x = W.draft_logits(wl, 1)
    xh = W.host(x)
    o = oracle.softmax_topk(xh, 5, T)
    xf = x.float().numpy().astype(np.float64)
    ref = scipy.special.softmax(xf / T, axis=-1)
    for r in range(xf.shape[0]):
        idx = _ranked_topk(xf[r], 5)
        np.testing.assert_array_equal(o["topk_idx"][r], idx)
        np.testing.assert_allclose(o["topk_p"][r], ref[r, idx], rtol=1e-6)


def test_topk_ties_go_to_lowest_index():
    x = np.zeros((1, 16), np.float32)
    x[0, [3, 7, 9, 12]] = 2.0
    o = oracle.softmax_topk(x, 3)
    assert o["topk_idx"].tolist() == [[3, 7, 9]]
    np.testing.assert_allclose(o["topk_p"], np.full((1, 3), np.exp(2) / (12 + 4 * np.exp(2))), rtol=1e-7)


def _fixture_topk(fx):
    """topk_p / topk_idx per step, as the fixture lists them."""
    tok = fx["tokens"]
    out = []
    for st in fx["steps"]:
        p = np.array([[pv for _, pv in row] for row in st["rows"]], np.float32)
        i = np.array([[tok[t] for t, _ in row] for row in st["rows"]], np.int32)
        out.append((p, i))
    return out


def test_matrug_path_scores_and_tree():
    fx = golden("matrug_draft.json")
    k, S, n = fx["k"], fx["S"], fx["n"]
    tok = fx["tokens"]
    steps = []
    scores = None
    for i, (p, idx) in enumerate(_fixture_topk(fx)):
        o = oracle.path_step(i, 1, k, p, idx, scores)
        steps.append(o)
        scores = o["scores_out"]
    score_space = np.concatenate([s["score_blk"] for s in steps], axis=1)
    token_space = np.concatenate([s["token_blk"] for s in steps], axis=1)
    parent_space = np.concatenate([s["parent_blk"] for s in steps[:-1]], axis=1)
    ex = fx["expect"]
    np.testing.assert_allclose(score_space[0], np.array(ex["score_space"], np.float32), rtol=1e-6)
    assert score_space.shape[1] == k + (S - 1) * k * k  # token / score space isomorphism
    assert parent_space[0].tolist() == ex["parent_list"]
    assert parent_space.shape[1] == 1 + (S - 1) * k
    t = oracle.build_tree(1, k, S, n, score_space, token_space, parent_space,
                          np.array([tok["bonus"]]), np.array([fx["seq_len"]]))
    assert t["draft_tokens"].tolist() == [tok[x] for x in ex["draft_tokens"]]
    assert t["parent_node"].tolist() == ex["parents"]
    assert t["next_token"].tolist() == ex["next_token"]
    assert t["next_sibling"].tolist() == ex["next_sibling"]
    assert t["mask_bits"].tolist() == ex["mask_rows"]
    assert t["positions"].tolist() == [fx["seq_len"] + d for d in ex["depth"]]
    assert t["retrieve_index"].tolist() == list(range(n))


def test_matrug_matches_eagle2_pages():
    """The same tree against the pointer table and the visibility the EAGLE-2
    page prints for it."""
    fx = golden("matrug_draft.json")
    pg = golden("eagle2_child_sibling.json")
    k, S, n = fx["k"], fx["S"], fx["n"]
    steps, scores = [], None
    for i, (p, idx) in enumerate(_fixture_topk(fx)):
        o = oracle.path_step(i, 1, k, p, idx, scores)
        steps.append(o)
        scores = o["scores_out"]
    t = oracle.build_tree(1, k, S, n, np.concatenate([s["score_blk"] for s in steps], 1),
                          np.concatenate([s["token_blk"] for s in steps], 1),
                          np.concatenate([s["parent_blk"] for s in steps[:-1]], 1),
                          np.array([fx["tokens"]["bonus"]]), np.array([0]))
    assert t["next_token"].tolist() == pg["next_token"]
    assert t["next_sibling"].tolist() == pg["next_sibling"]
    names = pg["mat_rug"]["nodes"]
    for i, name in enumerate(names):
        seen = {names[j] for j in range(n) if (int(t["mask_bits"][i]) >> j) & 1}
        assert seen == set(pg["mat_rug"]["visible"][name]), name


def test_positions_example():
    """depths [0,1,1,2] with prompt length 7 -> positions [7,8,8,9]."""
    fx = golden("positions_example.json")
    # step 0: a 0.6, b 0.3; step 1: a -> c 0.5, d 0.1; b -> e 0.1, f 0.05
    p0 = np.array([[0.6, 0.3]], np.float32)
    i0 = np.array([[10, 11]], np.int32)
    s0 = oracle.path_step(0, 1, 2, p0, i0)
    p1 = np.array([[0.5, 0.1], [0.1, 0.05]], np.float32)
    i1 = np.array([[12, 13, 14, 15]], np.int32)
    s1 = oracle.path_step(1, 1, 2, p1, i1, s0["scores_out"])
    t = oracle.build_tree(1, 2, 2, 4, np.concatenate([s0["score_blk"], s1["score_blk"]], 1),
                          np.concatenate([s0["token_blk"], s1["token_blk"]], 1), s0["parent_blk"],
                          np.array([9]), np.array([fx["prompt_len"]]))
    depth = [bin(int(m)).count("1") - 1 for m in t["mask_bits"]]
    assert depth == fx["depths"]
    assert t["positions"].tolist() == fx["positions"]


def test_path_step_against_numpy():
    """Library reference for one later step: fp32 products (numpy float32
    multiply) ranked by a stable sort."""
    rng = np.random.default_rng(1)
    b, k = 5, 3
    for step in (1, 2, 4):
        p = np.sort(rng.random((b * k, k)).astype(np.float32), axis=1)[:, ::-1].copy()
        idx = rng.integers(0, 1000, (b * k, k)).astype(np.int32)
        sc = rng.random((b, k)).astype(np.float32)
        p[0, 1] = p[0, 0]  # a tie inside one row
        o = oracle.path_step(step, b, k, p, idx, sc)
        for r in range(b):
            expand = (sc[r][:, None] * p[r * k:(r + 1) * k]).astype(np.float32).reshape(-1)
            np.testing.assert_array_equal(o["score_blk"][r], expand)
            sel = _ranked_topk(expand.astype(np.float64), k)
            assert o["parent_blk"][r].tolist() == (sel + k * k * (step - 1) + k).tolist()
            np.testing.assert_array_equal(o["scores_out"][r], expand[sel])
            assert o["next_ids"][r].tolist() == idx[r * k:(r + 1) * k].reshape(-1)[sel].tolist()


def _random_chain(seed, b=3, k=3, S=4, n=10, V=64):
    wl = W.scaled(W.WORKLOADS["tiny"], name=f"rand{seed}", b=b, k=k, S=S, n=n, V=V)
    drafts = [W.host(W.draft_logits(wl, i, seed=seed)) for i in range(S)]
    return wl, drafts


@pytest.mark.parametrize("seed", range(6))
def test_tree_invariants_random(seed):
    wl, drafts = _random_chain(seed)
    ch = P.select_chain(wl, drafts)
    seq = np.arange(wl.b, dtype=np.int32) * 10 + 5
    t = P.tree_from_chain(wl, ch, np.arange(wl.b) + 900, seq)
    b, n = wl.b, wl.n
    for r in range(b):
        sc = ch["score_space"][r].astype(np.float64)
        sel = np.sort(_ranked_topk(sc, n - 1))
        # draft tokens are the selected positions' tokens, bonus first
        assert t["draft_tokens"][r * n] == 900 + r
        assert t["draft_tokens"][r * n + 1:(r + 1) * n].tolist() == ch["token_space"][r][sel].tolist()
        par = t["parent_node"][r * n:(r + 1) * n]
        assert par[0] == -1
        for j in range(1, n):
            pj = par[j]
            assert 0 <= pj < j
            if pj > 0:  # a child never outscores its parent
                assert sc[sel[j - 1]] <= sc[sel[pj - 1]]
            # mask row = parent's row plus the node itself
            assert int(t["mask_bits"][r * n + j]) == int(t["mask_bits"][r * n + pj]) | (1 << j)
        # the sibling chains visit each node's children in ascending order, once
        nt = t["next_token"][r * n:(r + 1) * n]
        ns = t["next_sibling"][r * n:(r + 1) * n]
        for i in range(n):
            kids, c = [], nt[i]
            while c != -1:
                kids.append(int(c))
                c = ns[c]
            assert kids == [c for c in range(n) if par[c] == i]
        depth = [bin(int(m)).count("1") - 1 for m in t["mask_bits"][r * n:(r + 1) * n]]
        assert t["positions"][r * n:(r + 1) * n].tolist() == [seq[r] + d for d in depth]


@pytest.mark.parametrize("seed", range(4))
def test_parent_recovery_by_provenance(seed):
    """Independent of the parent_list formula: draft rows whose top-k tokens
    are unique to (step, row) let the test read every node's true parent off
    the token that was fed as that row's input."""
    rng = np.random.default_rng(100 + seed)
    b, k, S, n, V = 2, 3, 4, 11, 4096
    drafts = []
    for i in range(S):
        rows = b * (k if i else 1)
        x = rng.normal(size=(rows, V)).astype(np.float32)
        for row in range(rows):
            base = 64 + (i * 64 + row) * 8
            x[row, base:base + k] = 6.0 + rng.random(k).astype(np.float32) * 3
        drafts.append(x)
    wl = W.scaled(W.WORKLOADS["tiny"], name="prov", b=b, k=k, S=S, n=n, V=V)
    ch = P.select_chain(wl, drafts)
    t = P.tree_from_chain(wl, ch, np.array([1, 2]), np.zeros(b, np.int32))

    def origin(token):
        j = (token - 64) // 8
        return j // 64, j % 64  # (step, row)

    for r in range(b):
        toks = t["draft_tokens"][r * n:(r + 1) * n]
        par = t["parent_node"][r * n:(r + 1) * n]
        for j in range(1, n):
            step, row = origin(int(toks[j]))
            if step == 0:
                assert par[j] == 0
                continue
            # the row's input token at this step = next_ids of the previous step
            fed = int(ch["steps"][step - 1]["next_ids"].reshape(-1)[row])
            assert int(toks[par[j]]) == fed
            assert row // k == r


def test_chain_topk1_tree():
    fx = golden("chain_topk1.json")
    tok = fx["tokens"]
    steps, scores = [], None
    for i, name in enumerate(fx["draft_chain"]):
        o = oracle.path_step(i, 1, 1, np.array([[0.9 - 0.1 * i]], np.float32),
                             np.array([[tok[name]]], np.int32), scores)
        steps.append(o)
        scores = o["scores_out"]
    t = oracle.build_tree(1, 1, fx["S"], fx["n"], np.concatenate([s["score_blk"] for s in steps], 1),
                          np.concatenate([s["token_blk"] for s in steps], 1),
                          np.concatenate([s["parent_blk"] for s in steps[:-1]], 1),
                          np.array([tok[fx["root"]]]), np.array([fx["L"]]))
    assert t["positions"].tolist() == [fx["L"] + d for d in fx["expect"]["positions_offset"]]
    assert t["parent_node"].tolist() == [-1, 0, 1, 2]
    assert t["mask_bits"].tolist() == [1, 3, 7, 15]  # lower-triangular


def test_build_tree_rejects_orphan():
    """A selected node whose parent was not selected breaks the method's
    invariant and must be reported, not silently attached."""
    # k=1, S=2: positions 0 (step 0) and 1 (step 1, parent position 0)
    with pytest.raises(oracle.OracleError):
        oracle.build_tree(1, 1, 2, 2, np.array([[0.1, 0.5]], np.float32), np.array([[5, 6]]),
                          np.array([[-1, 0]]), np.array([1]), np.array([0]))
