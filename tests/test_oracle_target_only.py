"""Oracle pins for target-only tree sampling (CPU only).

The accept page's section 4 (Target-only Tree Sampling) states the rule: the
siblings of the current node are scanned in order, their target mass is
accumulated, and a sibling is accepted when its target probability is positive
and the coin lies below the accumulated mass over threshold_acc, or its own
probability reaches threshold_single; a rejected sibling's probability goes
into the current row's buffer, and the terminal token is drawn from
relu(p - buffer).  These tests pin the oracle to cases worked by hand from that
rule, to the closed-form law the rule implies for one sibling level (by a
chi-square test), to the greedy walk at T = 0, and to the accept invariants.
"""
import numpy as np
import pytest
import scipy.stats

import oracle
from tests.helpers import golden, onehot_logits, pointers_from_parents


def _logp(p):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, np.float64)).astype(np.float32)


def _one_level(p, xs, coins, uf, t_single, t_acc, T=1.0):
    """b requests, each a root (target logits log p) with leaf children
    carrying tokens xs in sibling order; coins [b] are the roots' coins."""
    b = len(coins)
    m = len(xs)
    n = m + 1
    V = len(p)
    logits = np.zeros((b * n, V), np.float32)  # the leaves' rows: uniform p (their terminal draws)
    logits[0::n] = _logp(p)
    draft = np.tile(np.array([0] + list(xs), np.int32), b)
    u = np.zeros((b, n), np.float32)
    u[:, 0] = coins
    nt = np.tile(np.array([1] + [-1] * m, np.int32), b)
    ns = np.tile(np.array([-1] + list(range(2, n)) + [-1], np.int32), b)
    return oracle.verify_target_only(b, n, 1, logits, np.full(b, T, np.float32), u.ravel(),
                                     np.asarray(uf, np.float32), t_single, t_acc, draft, np.arange(b * n),
                                     nt, ns)


def test_hand_worked_threshold_cases():
    fx = golden("target_only_example.json")
    names = list(fx["children"])
    xs = [fx["children"][k] for k in names]
    for case in fx["cases"]:
        o = _one_level(fx["p_root"], xs, [case["coin"]], [case["u_final"]], case["threshold_single"],
                       case["threshold_acc"])
        if case["accepted"] is None:
            assert o["accept_lens"][0] == 1, case
            assert o["accepted_tokens"][0, 0] == case["terminal"], case
        else:
            assert o["accept_lens"][0] == 2, case
            assert o["accept_index"][0, 1] == 1 + names.index(case["accepted"]), case
            assert o["accepted_tokens"][0, 0] == fx["children"][case["accepted"]], case


def test_accepted_child_coin_and_per_row_buffer():
    """Two levels: the accumulator restarts at the accepted child, whose own
    coin decides its children; a sibling rejected at the root stays in the
    terminal draw at a deeper node (the buffer is per row)."""
    fx = golden("target_only_example.json")["two_levels"]
    V = len(fx["p_root"])
    tok = fx["tokens"]
    draft = np.array([0, tok["X"], tok["A"], tok["A1"]], np.int32)
    nt, ns = pointers_from_parents(fx["parents"])
    logits = np.zeros((4, V), np.float32)
    logits[0] = _logp(fx["p_root"])
    logits[2] = _logp(fx["p_A"])
    u = np.array([fx["coin_root"], 0.0, fx["coin_A"], 0.0], np.float32)
    o = oracle.verify_target_only(1, 4, 2, logits, np.ones(1, np.float32), u,
                                  np.array([fx["u_final"]], np.float32), 1.0, 1.0, draft, np.arange(4), nt, ns)
    L = o["accept_lens"][0]
    assert L == fx["expect_accept_lens"]
    assert o["accepted_tokens"][0, :L].tolist() == fx["expect_tokens"]
    assert o["accept_index"][0, :L].tolist() == [0, 2]


def _law(p, xs, t_single, t_acc):
    """Exact law of one sibling level: the probability that sibling i is the
    first accepted (over the coin c ~ U[0, 1)), and the probability that all
    are rejected times relu(p - buffer) normalised."""
    p = np.asarray(p, np.float64)
    m = len(xs)
    lo = 0.0  # every coin below lo was accepted by an earlier sibling
    acc = np.zeros(m)
    cum = 0.0
    for i, x in enumerate(xs):
        cum += p[x]
        if p[x] <= 0:
            continue
        if p[x] >= t_single:
            acc[i] = max(0.0, 1.0 - lo)
            lo = 1.0
            break
        hi = min(1.0, cum / t_acc)
        if hi > lo:
            acc[i] = hi - lo
            lo = hi
    rest = max(0.0, 1.0 - lo)
    r = p.copy()
    r[list(xs)] = 0.0
    if r.sum() <= 0:
        r = p.copy()
    return acc, rest * r / r.sum()


@pytest.mark.parametrize("t_single,t_acc", [(1.0, 1.0), (None, 0.6)])
def test_one_level_law_chi_square(t_single, t_acc):
    """1e5 seeded trials of one sibling level against the exact law: outcome
    = the accepted sibling, or the terminal token when none is accepted.  With
    both thresholds at 1 the first output token follows p exactly (the coin
    picks a sibling by its own mass, and the rest of the mass is drawn with the
    siblings removed)."""
    rng = np.random.default_rng(23)
    V, m, N = 12, 3, 100_000
    p = rng.dirichlet(np.full(V, 0.6))
    pf = np.exp(_logp(p).astype(np.float64))
    pf /= pf.sum()  # the oracle's p: softmax of the fp32 log-probabilities
    xs = [int(v) for v in rng.choice(V, size=m, replace=False, p=pf)]
    if t_single is None:
        # the second sibling carries the argmax and reaches threshold_single,
        # the first does not: the first is accepted only below prob_acc /
        # threshold_acc, the second by its own mass, the third never
        big = int(np.argmax(pf))
        xs = [v for v in xs if v != big][:1] + [big] + [v for v in xs if v != big][1:2]
        t_single = float(0.5 * (pf[xs[0]] + pf[big]))
        assert pf[big] >= t_single > pf[xs[0]]
    acc, term = _law(pf, xs, t_single, t_acc)
    coins = rng.random(N).astype(np.float32)
    uf = rng.random(N).astype(np.float32)
    o = _one_level(p, xs, coins, uf, t_single, t_acc)
    accepted = o["accept_lens"] == 2
    sib = o["accept_index"][:, 1] - np.arange(N) * (m + 1) - 1
    outcome = np.where(accepted, sib, m + o["accepted_tokens"][:, 0])
    expect = np.concatenate([acc, term])
    counts = np.bincount(outcome, minlength=m + V)
    keep = expect > 0
    assert counts[~keep].sum() == 0
    stat, pval = scipy.stats.chisquare(counts[keep], expect[keep] / expect.sum() * N)
    assert pval > 1e-3, (stat, pval)
    if (t_single, t_acc) == (1.0, 1.0):
        first = o["accepted_tokens"][:, 0]
        stat, pval = scipy.stats.chisquare(np.bincount(first, minlength=V), pf * N)
        assert pval > 1e-3, (stat, pval)


def test_t0_equals_greedy():
    """T <= 0 makes p one-hot at the argmax: with thresholds in (0, 1] the walk
    accepts exactly the child carrying the argmax token, and the terminal
    token is the argmax -- the greedy accept."""
    fx = golden("rabcd_greedy.json")
    tok = fx["tokens"]
    nodes = fx["nodes"]
    n = len(nodes)
    draft = np.array([tok[x] for x in nodes], np.int32)
    nt, ns = pointers_from_parents(fx["parents"])
    logits = onehot_logits([tok[fx["target_argmax"][x]] for x in nodes], fx["V"])
    g = oracle.verify_greedy(1, n, 2, logits, draft, np.arange(n), nt, ns)
    rng = np.random.default_rng(3)
    for t_single, t_acc in ((1.0, 1.0), (0.5, 0.2)):
        o = oracle.verify_target_only(1, n, 2, logits, np.zeros(1, np.float32), rng.random(n).astype(np.float32),
                                      rng.random(1).astype(np.float32), t_single, t_acc, draft, np.arange(n), nt, ns)
        for k in g:
            np.testing.assert_array_equal(o[k], g[k], err_msg=k)


@pytest.mark.parametrize("seed", range(4))
def test_invariants_on_random_trees(seed):
    """accept_lens = drafts + 1; the accepted rows form a root-to-node path;
    predict on the path = the accepted tokens then the terminal token; 0 off
    the path."""
    rng = np.random.default_rng(seed)
    b, n, V, S = 6, 9, 40, 4
    parents = [-1] + [int(rng.integers(0, i)) for i in range(1, n)]
    depth = [0] * n
    for i in range(1, n):
        depth[i] = depth[parents[i]] + 1
    nt, ns = pointers_from_parents(parents)
    logits = rng.normal(0, 2, (b * n, V)).astype(np.float32)
    draft = rng.integers(0, V, b * n).astype(np.int32)
    # make a child's token likely: the parent's argmax
    for r in range(b):
        for c in range(1, n):
            if rng.random() < 0.6:
                draft[r * n + c] = int(np.argmax(logits[r * n + parents[c]]))
    o = oracle.verify_target_only(b, n, S, logits, rng.uniform(0.5, 1.5, b).astype(np.float32),
                                  rng.random(b * n).astype(np.float32), rng.random(b).astype(np.float32), 0.8, 0.9,
                                  draft, np.arange(b * n), np.tile(nt, b), np.tile(ns, b))
    for r in range(b):
        L = o["accept_lens"][r]
        rows = o["accept_index"][r, :L]
        assert 1 <= L <= S + 1 and (o["accept_index"][r, L:] == -1).all()
        assert rows[0] == r * n
        for d in range(1, L):
            assert parents[rows[d] - r * n] == rows[d - 1] - r * n
        assert depth[rows[-1] - r * n] == L - 1
        toks = o["predict"][rows]
        assert toks[:-1].tolist() == draft[rows[1:]].tolist()
        assert o["accepted_tokens"][r, :L].tolist() == toks.tolist()
        assert o["next_root"][r] == toks[-1]
        off = np.setdiff1d(np.arange(r * n, (r + 1) * n), rows)
        assert (o["predict"][off] == 0).all()


def test_rejects_thresholds_outside_unit_interval():
    logits = np.zeros((2, 4), np.float32)
    args = (np.array([0, 1], np.int32), np.arange(2), np.array([1, -1], np.int32), np.array([-1, -1], np.int32))
    for ts, ta in ((0.0, 1.0), (1.0, 0.0), (1.5, 1.0), (1.0, 1.01)):
        with pytest.raises(oracle.OracleError):
            oracle.verify_target_only(1, 2, 1, logits, np.ones(1, np.float32), np.zeros(2, np.float32),
                                      np.zeros(1, np.float32), ts, ta, *args)
