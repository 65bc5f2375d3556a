"""Oracle pins for the accept step: greedy walk and rejection sampling (CPU only)."""
import numpy as np
import pytest
import scipy.stats

import oracle
from accept_select_top_gb300 import workloads as W
from oracle import pipeline as P
from tests.helpers import golden, onehot_logits, pointers_from_parents


def _rabcd():
    fx = golden("rabcd_greedy.json")
    tok = fx["tokens"]
    nodes = fx["nodes"]
    n = len(nodes)
    draft = np.array([tok[x] for x in nodes], np.int32)
    nt, ns = pointers_from_parents(fx["parents"])
    logits = onehot_logits([tok[fx["target_argmax"][x]] for x in nodes], fx["V"])
    return fx, n, draft, nt, ns, logits


def test_rabcd_greedy():
    fx, n, draft, nt, ns, logits = _rabcd()
    tok, ex = fx["tokens"], fx["expect"]
    S = 2
    o = oracle.verify_greedy(1, n, S, logits, draft, np.arange(n), nt, ns)
    W_ = S + 1
    assert o["accept_index"][0, : ex["accept_lens"]].tolist() == ex["accept_rows"]
    assert (o["accept_index"][0, ex["accept_lens"]:] == -1).all()
    assert o["accept_lens"].tolist() == [ex["num_correct_drafts"] + 1] == [ex["accept_lens"]]
    expect_pred = np.zeros(n, np.int32)
    for row, name in ex["predict"].items():
        expect_pred[int(row)] = tok[name]
    assert o["predict"].tolist() == expect_pred.tolist()
    assert o["accepted_tokens"][0, : ex["accept_lens"]].tolist() == [tok[x] for x in ex["accepted_tokens"]]
    assert o["next_root"].tolist() == [tok[ex["next_root"]]]
    # the rows that feed the KV commit are the input rows R, A, C, not the output X
    rows = o["accept_index"][0, : o["accept_lens"][0]]
    assert [fx["nodes"][r] for r in rows] == ex["committed_rows"]
    assert W_ == o["accept_index"].shape[1]


def test_rabcd_greedy_batched_rows_are_global():
    """accept_index holds flattened rows b*n+i of the whole batch."""
    fx, n, draft, nt, ns, logits = _rabcd()
    b = 3
    o = oracle.verify_greedy(b, n, 2, np.tile(logits, (b, 1)), np.tile(draft, b),
                             np.arange(b * n), np.tile(nt, b), np.tile(ns, b))
    for r in range(b):
        assert o["accept_index"][r].tolist() == [r * n + x for x in fx["expect"]["accept_rows"]]


def test_eagle2_walk_root_a_d():
    fx = golden("eagle2_child_sibling.json")
    nodes = fx["nodes"]
    n = len(nodes)
    tok = {x: 10 + i for i, x in enumerate(nodes)}
    tok["bonus"] = 30
    draft = np.array([tok[x] for x in nodes], np.int32)
    want = {"root": tok["A"], "A": tok["D"], "D": tok["bonus"]}
    logits = onehot_logits([want.get(x, 31) for x in nodes], 32)
    o = oracle.verify_greedy(1, n, 3, logits, draft, np.arange(n), np.array(fx["next_token"]),
                             np.array(fx["next_sibling"]))
    L = o["accept_lens"][0]
    assert [nodes[i] for i in o["accept_index"][0, :L]] == fx["walk"]["accepted"]
    assert L - 1 == fx["walk"]["num_correct_drafts"]


def test_chain_the_cat_sat():
    fx = golden("chain_topk1.json")
    tok = fx["tokens"]
    names = [fx["root"]] + fx["draft_chain"]
    draft = np.array([tok[x] for x in names], np.int32)
    nt, ns = pointers_from_parents([-1, 0, 1, 2])
    logits = onehot_logits([tok[x] for x in fx["target_argmax"]], 8)
    o = oracle.verify_greedy(1, 4, fx["S"], logits, draft, np.arange(4), nt, ns)
    ex = fx["expect"]
    assert o["accept_lens"][0] == ex["accept_lens"] == ex["num_correct_drafts"] + 1
    assert o["accepted_tokens"][0, :3].tolist() == [tok[x] for x in ex["accepted_tokens"]]
    assert o["accepted_tokens"][0, 3] == -1


def test_dspark_chain_counts():
    fx = golden("chain_commit.json")
    tok = fx["tokens"]
    draft = np.array([tok[x] for x in fx["nodes"]], np.int32)
    nt, ns = pointers_from_parents([-1, 0, 1, 2])
    logits = onehot_logits([tok[x] for x in fx["target_argmax"]], 8)
    o = oracle.verify_greedy(1, 4, 3, logits, draft, np.arange(4), nt, ns)
    ex = fx["expect"]
    assert o["accept_lens"][0] - 1 == ex["correct_len"]
    assert o["accept_lens"][0] == ex["commit_lens"]
    assert o["accepted_tokens"][0, :3].tolist() == [tok[x] for x in ex["accepted_tokens"]]


def test_greedy_first_sibling_wins_and_root_only():
    """Two siblings with the same token: the first in sibling order is taken.
    No matching child: only the root row, accept_lens 1, output = target at root."""
    draft = np.array([1, 5, 5, 6], np.int32)
    nt, ns = pointers_from_parents([-1, 0, 0, 1])
    o = oracle.verify_greedy(1, 4, 3, onehot_logits([5, 6, 7, 7], 8), draft, np.arange(4), nt, ns)
    assert o["accept_index"][0].tolist() == [0, 1, 3, -1]
    o = oracle.verify_greedy(1, 4, 3, onehot_logits([4, 6, 7, 7], 8), draft, np.arange(4), nt, ns)
    assert o["accept_index"][0].tolist() == [0, -1, -1, -1]
    assert o["accept_lens"][0] == 1 and o["predict"].tolist() == [4, 0, 0, 0]


def test_greedy_argmax_ties_lowest_index():
    draft = np.array([1, 3, 2], np.int32)
    nt, ns = pointers_from_parents([-1, 0, 0])
    x = np.zeros((3, 8), np.float32)
    x[0, [2, 3]] = 1.0  # tie between tokens 2 and 3: token 2 wins -> node 2
    o = oracle.verify_greedy(1, 3, 1, x, draft, np.arange(3), nt, ns)
    assert o["accept_index"][0].tolist() == [0, 2]


def _tiny_case(seed=0, mode="sampling"):
    wl = W.WORKLOADS["tiny"]
    drafts_t = [W.draft_logits(wl, i, seed=seed) for i in range(wl.S)]
    drafts = [W.host(d) for d in drafts_t]
    lay = W.kv_layout(wl, seed=seed)
    ch = P.select_chain(wl, drafts)
    tree = P.tree_from_chain(wl, ch, W.host(W.bonus_tokens(wl, seed=seed)), lay["seq_lens"])
    rows = W.draft_rows_of_nodes(wl, tree["draft_tokens"], tree["next_token"], tree["next_sibling"],
                                 ch["token_space"], ch["parent_space"])
    all_d = torch_cat(drafts_t)
    logits = W.target_logits(wl, rows, all_d, seed=seed)
    temps = W.request_temperatures(wl, mode)
    q = W.draft_probs(wl, rows, all_d, temps)
    u, uf = W.coins(wl, seed=seed)
    return wl, tree, W.host(logits), W.host(q), temps, W.host(u), W.host(uf)


def torch_cat(ts):
    import torch
    return torch.cat(ts, 0)


@pytest.mark.parametrize("seed", range(5))
def test_t0_sampling_equals_greedy(seed):
    wl, tree, logits, q, temps, u, uf = _tiny_case(seed, "greedy")
    g = P.accept(wl, "greedy", tree, logits)
    s = P.accept(wl, "sampling", tree, logits, q, np.zeros(wl.b, np.float32), u, uf)
    for key in g:
        np.testing.assert_array_equal(g[key], s[key], err_msg=key)


@pytest.mark.parametrize("mode", ["greedy", "sampling"])
@pytest.mark.parametrize("seed", range(5))
def test_accept_invariants(mode, seed):
    """accept_lens = drafts + 1; the valid prefix of accept_index is a root-to-
    node path through parent -> child links; predict[accept_index] = accepted
    draft tokens followed by the terminal token."""
    wl, tree, logits, q, temps, u, uf = _tiny_case(seed, mode)
    o = P.accept(wl, mode, tree, logits, q, temps, u, uf)
    b, n = wl.b, wl.n
    par = tree["parent_node"].reshape(b, n)
    for r in range(b):
        L = o["accept_lens"][r]
        rows = o["accept_index"][r, :L]
        assert (o["accept_index"][r, L:] == -1).all()
        assert rows[0] == r * n
        for d in range(1, L):
            assert par[r, rows[d] - r * n] == rows[d - 1] - r * n
        toks = o["predict"][rows]
        assert toks[:-1].tolist() == tree["draft_tokens"][rows[1:]].tolist()
        assert o["accepted_tokens"][r, :L].tolist() == toks.tolist()
        assert o["next_root"][r] == toks[-1]
        visited = set(rows.tolist())
        for i in range(r * n, (r + 1) * n):
            if i not in visited:
                assert o["predict"][i] == 0
        if mode == "greedy":
            assert toks[-1] == np.argmax(logits[rows[-1]])


def _single_candidate(p, q, u, uf, x, leaf_logits=None, T=1.0):
    """b single-candidate chains: root (target logits log p, draft q) with one
    child x, every request at temperature T."""
    b = len(u)
    V = len(p)
    logits = np.empty((b * 2, V), np.float32)
    logits[0::2] = np.log(np.asarray(p, np.float64)).astype(np.float32)
    logits[1::2] = leaf_logits if leaf_logits is not None else np.log(np.full(V, 1.0 / V)).astype(np.float32)
    qq = np.zeros((b * 2, V), np.float32)
    qq[0::2] = np.asarray(q, np.float32)
    draft = np.empty(b * 2, np.int32)
    draft[0::2] = 0
    draft[1::2] = x
    uu = np.zeros(b * 2, np.float32)
    uu[1::2] = u
    nt = np.tile(np.array([1, -1], np.int32), b)
    ns = np.full(b * 2, -1, np.int32)
    return oracle.verify_sampling(b, 2, 1, logits, qq, np.full(b, T, np.float32), uu,
                                  np.asarray(uf, np.float32), draft, np.arange(b * 2), nt, ns)


def _tempered(p, T):
    """The target distribution at temperature T when the logits are the fp32
    log-probabilities: p_T(v) = p(v)^(1/T) / sum_w p(w)^(1/T) (closed form)."""
    lp = np.log(np.asarray(p, np.float64)).astype(np.float32).astype(np.float64)
    w = np.power(np.exp(lp), 1.0 / T)
    return w / w.sum()


@pytest.mark.parametrize("T", [0.7, 2.0])
def test_rejection_temperature_closed_form(T):
    """The sampler's p is the softmax of logits / T.  With logits = log p the
    tempered target is p^(1/T) normalised.  Quadrature over (x ~ q, u,
    u_final): candidate x is accepted with probability min(1, p_T(x)/q(x)), a
    rejected candidate's mass goes to max(0, p_T - q)/Z, and the first output
    token is distributed as p_T.  A temperature multiplied instead of divided,
    or left out, moves every one of these."""
    fx = golden("rejection_example.json")
    p, q = np.array(fx["p"]), np.array(fx["q"], np.float32).astype(np.float64)
    pT = _tempered(p, T)
    assert np.abs(pT - p).max() > 0.02  # the temperature matters for this p
    G = 300
    grid = (np.arange(G) + 0.5) / G
    uu, ff = np.meshgrid(grid, grid, indexing="ij")
    uu, ff = uu.ravel(), ff.ravel()
    dist = np.zeros(3)
    res = np.maximum(pT - q, 0.0)
    res /= res.sum()
    for x in range(3):
        o = _single_candidate(p, q, uu, ff, x, T=T)
        first = o["accepted_tokens"][:, 0]
        acc = o["accept_lens"] == 2
        assert abs(acc.mean() - min(1.0, pT[x] / q[x])) < 2.0 / G, (x, acc.mean())
        if (~acc).sum() > G:
            frac = np.bincount(first[~acc], minlength=3) / (~acc).sum()
            np.testing.assert_allclose(frac, res, atol=2.0 / G)
        dist += q[x] * np.bincount(first, minlength=3) / len(first)
    np.testing.assert_allclose(dist, pT, atol=2.0 / G)


def test_rejection_chi_square_temperature():
    """V=16 at T=0.7, 1e5 single-candidate trials with x drawn from q: the
    output follows p_T = softmax(log p / 0.7) and the acceptance rate is
    sum(min(p_T, q))."""
    rng = np.random.default_rng(17)
    V, N, T = 16, 100_000, 0.7
    p = rng.dirichlet(np.full(V, 0.8))
    q = rng.dirichlet(np.full(V, 0.8))
    pT = _tempered(p, T)
    x = np.searchsorted(np.cumsum(q), rng.random(N), side="right").clip(0, V - 1)
    u = rng.random(N).astype(np.float32)
    uf = rng.random(N).astype(np.float32)
    o = _single_candidate(p, q.astype(np.float32), u, uf, x, T=T)
    counts = np.bincount(o["accepted_tokens"][:, 0], minlength=V)
    stat, pval = scipy.stats.chisquare(counts, pT * N)
    assert pval > 1e-3, (stat, pval)
    acc = (o["accept_lens"] == 2).mean()
    a = np.minimum(pT, q.astype(np.float32)).sum()
    assert abs(acc - a) < 4 * np.sqrt(a * (1 - a) / N)


def test_terminal_draw_past_the_total_mass_takes_the_last_positive_token():
    """The draw takes the smallest v with u_final * Z < the running sum.  A
    coin u_final = 1 (outside [0, 1): the running sum never passes u*Z = Z)
    falls through to the last token with positive mass: C for the rejected
    residual (0, 0.1, 0.2); with target logits -inf past token 2 of 6 (zero
    probability there), token 2 for a draw from p itself."""
    fx = golden("rejection_example.json")
    o = _single_candidate(fx["p"], fx["q"], [0.9], [1.0], 0)
    assert o["accept_lens"][0] == 1 and o["accepted_tokens"][0, 0] == 2
    # a leaf root (no child): the bonus is drawn from p; p is zero past token 2
    V = 6
    logits = np.full((1, V), -np.inf, np.float32)
    logits[0, :3] = np.log([0.2, 0.5, 0.3])
    o = oracle.verify_sampling(1, 1, 1, logits, np.zeros((1, V), np.float32), np.ones(1, np.float32),
                               np.zeros(1, np.float32), np.ones(1, np.float32), np.zeros(1, np.int32),
                               np.arange(1), np.full(1, -1, np.int32), np.full(1, -1, np.int32))
    assert o["accept_lens"][0] == 1 and o["accepted_tokens"][0, 0] == 2
    # and just below 1 the draw is the last positive-mass token by the running sum as well
    o = oracle.verify_sampling(1, 1, 1, logits, np.zeros((1, V), np.float32), np.ones(1, np.float32),
                               np.zeros(1, np.float32), np.full(1, np.float32(1) - np.float32(2 ** -24)),
                               np.zeros(1, np.int32), np.arange(1), np.full(1, -1, np.int32),
                               np.full(1, -1, np.int32))
    assert o["accepted_tokens"][0, 0] == 2


def test_rejection_example_points():
    fx = golden("rejection_example.json")
    p, q = fx["p"], fx["q"]
    leaf = np.log(np.array([0.2, 0.5, 0.3])).astype(np.float32)
    o = _single_candidate(p, q, [0.49, 0.49, 0.51, 0.51, 0.51], [0.1, 0.5, 0.3, 0.34, 0.99], 0, leaf)
    # u < 0.5 accepts A; then A is a leaf and the bonus comes from its own p
    assert o["accept_lens"].tolist() == [2, 2, 1, 1, 1]
    assert o["accepted_tokens"][:2, :2].tolist() == [[0, 0], [0, 1]]
    # rejected: residual (0, 0.1, 0.2)/0.3 -> B below 1/3, C above
    assert o["accepted_tokens"][2:, 0].tolist() == [1, 2, 2]


def test_rejection_example_distribution_closed_form():
    """Quadrature over (x ~ q, u, u_final) on a midpoint grid: the first output
    token is distributed as p, the accept probability of A is 0.5 and the
    rejected mass lands on B and C as 1/3, 2/3."""
    fx = golden("rejection_example.json")
    p, q = np.array(fx["p"]), np.array(fx["q"])
    G = 300
    grid = (np.arange(G) + 0.5) / G
    uu, ff = np.meshgrid(grid, grid, indexing="ij")
    uu, ff = uu.ravel(), ff.ravel()
    dist = np.zeros(3)
    for x in range(3):
        o = _single_candidate(p, q, uu, ff, x)
        first = o["accepted_tokens"][:, 0]
        acc = o["accept_lens"] == 2
        if x == 0:
            assert abs(acc.mean() - fx["expect"]["accept_prob_A"]) < 2.0 / G
            rej = first[~acc]
            frac = np.bincount(rej, minlength=3) / len(rej)
            np.testing.assert_allclose(frac, fx["expect"]["residual_normalised"], atol=2.0 / G)
        dist += q[x] * np.bincount(first, minlength=3) / len(first)
    np.testing.assert_allclose(dist, fx["expect"]["combined"], atol=2.0 / G)


def test_rejection_chi_square():
    """V=16, 1e5 single-candidate trials with x drawn from q: the output is
    distributed as p and the acceptance rate is sum(min(p, q))."""
    rng = np.random.default_rng(7)
    V, N = 16, 100_000
    p = rng.dirichlet(np.full(V, 0.8))
    q = rng.dirichlet(np.full(V, 0.8))
    pf = np.exp(np.log(p).astype(np.float32).astype(np.float64))
    pf /= pf.sum()
    x = np.searchsorted(np.cumsum(q), rng.random(N), side="right").clip(0, V - 1)
    u = rng.random(N).astype(np.float32)
    uf = rng.random(N).astype(np.float32)
    o = _single_candidate(p, q.astype(np.float32), u, uf, x)
    first = o["accepted_tokens"][:, 0]
    counts = np.bincount(first, minlength=V)
    stat, pval = scipy.stats.chisquare(counts, pf * N)
    assert pval > 1e-3, (stat, pval)
    acc = (o["accept_lens"] == 2).mean()
    a = np.minimum(pf, q).sum()
    assert abs(acc - a) < 4 * np.sqrt(a * (1 - a) / N)


def _one_level_siblings(p, q, xs, u, uf):
    """b requests, each a root (target p, draft q) with len(xs) leaf children
    in sibling order carrying tokens xs; u[b, m] are the children's coins."""
    b, m = u.shape
    V = len(p)
    n = m + 1
    logits = np.zeros((b * n, V), np.float32)  # leaves: uniform p (their bonus draws)
    logits[0::n] = np.log(np.asarray(p, np.float64)).astype(np.float32)
    qq = np.zeros((b * n, V), np.float32)
    qq[0::n] = np.asarray(q, np.float32)
    draft = np.tile(np.array([0] + list(xs), np.int32), b)
    uu = np.zeros((b, n), np.float32)
    uu[:, 1:] = u
    nt = np.tile(np.array([1] + [-1] * m, np.int32), b)
    ns = np.tile(np.array([-1] + list(range(2, n)) + [-1], np.int32), b)
    return oracle.verify_sampling(b, n, 1, logits, qq, np.ones(b, np.float32), uu.ravel(),
                                  np.asarray(uf, np.float32), draft, np.arange(b * n), nt, ns)


def test_rejection_siblings_closed_form():
    """One level, three sibling leaves with distinct tokens, p and q fixed
    across siblings, one coin per child.  With a_i = min(1, p(x_i)/q(x_i)),
    sibling i is accepted with probability prod_{j<i}(1 - a_j) a_i, and with
    prod_j (1 - a_j) every child is rejected and the output token follows
    max(0, p - q)/Z.  1e5 seeded trials against that law (chi-square over the
    outcomes: accepted sibling, or the residual token), which fixes the
    sibling order, the per-child coin and the node the residual is taken at."""
    rng = np.random.default_rng(11)
    V, m, N = 12, 3, 100_000
    p = rng.dirichlet(np.full(V, 0.7))
    q = rng.dirichlet(np.full(V, 0.7))
    pf = np.exp(np.log(p).astype(np.float32).astype(np.float64))
    pf /= pf.sum()  # the oracle's p: softmax of the fp32 log-probabilities
    qf = q.astype(np.float32).astype(np.float64)
    # siblings on tokens with p < q, so that every one can be rejected and
    # every outcome (each sibling, the residual) has a fair share
    xs = [int(v) for v in rng.choice(np.flatnonzero(pf < 0.8 * qf), size=m, replace=False)]
    a = np.minimum(1.0, pf[xs] / qf[xs])
    reach = np.concatenate([[1.0], np.cumprod(1.0 - a)])  # reach[i]: all of the first i rejected
    p_acc = reach[:m] * a
    res = np.maximum(pf - qf, 0.0)
    res /= res.sum()
    expect = np.concatenate([p_acc, reach[m] * res])  # outcomes: sibling 0..m-1, then residual token v
    assert p_acc.min() > 0.02 and reach[m] > 0.05  # a non-degenerate case
    u = rng.random((N, m)).astype(np.float32)
    uf = rng.random(N).astype(np.float32)
    o = _one_level_siblings(p, q, xs, u, uf)
    acc = o["accept_lens"] == 2
    idx = o["accept_index"][:, 1] - np.arange(N) * (m + 1) - 1  # accepted sibling, -1 / -(..) if none
    outcome = np.where(acc, idx, m + o["accepted_tokens"][:, 0])
    counts = np.bincount(outcome, minlength=m + V)
    keep = expect > 0
    assert counts[~keep].sum() == 0
    stat, pval = scipy.stats.chisquare(counts[keep], expect[keep] * N)
    assert pval > 1e-3, (stat, pval)
    # an accepted sibling's token is the first output; the leaf's bonus is uniform
    first = o["accepted_tokens"][:, 0]
    np.testing.assert_array_equal(first[acc], np.array(xs)[idx[acc]])


def test_residual_zero_falls_back_to_p():
    """q == p at the only child's row and the child rejected: Z would be 0 only
    if p <= q everywhere; here q puts all mass on x, p does not, so the
    residual is p without x."""
    p = np.array([0.5, 0.25, 0.25])
    q = np.array([1.0, 0.0, 0.0], np.float32)
    o = _single_candidate(p, q, [0.9], [0.0], 0)
    assert o["accept_lens"][0] == 1 and o["accepted_tokens"][0, 0] == 1
    # q == p with the child on a zero-probability token: u*0 < 0 fails, the
    # residual max(0, p - q) is zero everywhere (Z == 0) and the bonus comes from p
    p = np.array([0.5, 0.5, 0.0])
    o = _single_candidate(p, p.astype(np.float32), [0.3], [0.74], 2)
    assert o["accept_lens"][0] == 1 and o["accepted_tokens"][0, 0] == 1
    # with q == p > 0 at the child, u*q < p holds for every u < 1: always accepted
    p = np.array([0.25, 0.25, 0.5])
    o = _single_candidate(p, p.astype(np.float32), [0.999999], [0.74], 2)
    assert o["accept_lens"][0] == 2
