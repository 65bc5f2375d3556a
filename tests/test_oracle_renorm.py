"""Oracle pins for the relaxed penalties and the top-k / top-p
renormalisation before the accept (CPU only).

[SGL-XI eagle_sample]: each request's accumulated additive penalty row is
repeated over its draft_token_num verify rows and added to the logits (the
relaxed penalties); on the sampling path the target softmax by temperature is
filtered by top-k, then top-p, and renormalised, and that distribution is what
the accept consumes [ACCEPT section 4].
"""
import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import oracle
from tests.helpers import pointers_from_parents


def test_penalties_fp32_and_bf16_rounding():
    """fp32: the fp32 sum; bf16: the fp32 sum rounded to nearest-even bf16
    (torch's conversion); each request's row is added to its n verify rows."""
    rng = np.random.default_rng(5)
    b, n, V = 3, 4, 37
    pen = rng.normal(0, 3, (b, V)).astype(np.float32)
    x = rng.normal(0, 2, (b * n, V)).astype(np.float32)
    out = oracle.add_penalties(b, n, x, pen)
    np.testing.assert_array_equal(out, x + np.repeat(pen, n, axis=0))
    xb = torch.from_numpy(x).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    out = oracle.add_penalties(b, n, bits, pen)
    want = (xb.float() + torch.from_numpy(np.repeat(pen, n, axis=0))).to(torch.bfloat16)
    np.testing.assert_array_equal(out, want.view(torch.int16).numpy().view(np.uint16))


def _renorm(logp, k, p, T=1.0):
    lg = np.asarray(logp, np.float32)[None, :]
    return oracle.renorm_probs(1, 1, lg, [T], [k], [p])[0].astype(np.float64)


def test_top_k_then_top_p_worked_example():
    """p = (0.5, 0.3, 0.15, 0.05): top-k 2 keeps (0.625, 0.375); top-p 0.75
    keeps the same two (0.5 < 0.75 <= 0.8); top-p 0.85 keeps three; top-k 3
    then top-p 0.7 renormalises to (0.526, 0.316, 0.158) first, whose first
    two reach 0.7."""
    lp = np.log([0.5, 0.3, 0.15, 0.05])
    np.testing.assert_allclose(_renorm(lp, 2, 1.0), [0.625, 0.375, 0, 0], rtol=1e-6)
    np.testing.assert_allclose(_renorm(lp, -1, 0.75), [0.625, 0.375, 0, 0], rtol=1e-6)
    np.testing.assert_allclose(_renorm(lp, 0, 0.85), np.array([0.5, 0.3, 0.15, 0]) / 0.95, rtol=1e-6)
    np.testing.assert_allclose(_renorm(lp, 3, 0.7), [0.625, 0.375, 0, 0], rtol=1e-6)
    # top-p below the largest probability keeps the largest alone
    np.testing.assert_allclose(_renorm(lp, -1, 0.3), [1, 0, 0, 0], rtol=1e-6)


def test_ties_at_the_cut_are_kept():
    lg = [2.0, 1.0, 1.0, 0.0]
    e = np.exp(np.array(lg) - 2.0)
    np.testing.assert_allclose(_renorm(lg, 2, 1.0), np.r_[e[:3], 0] / e[:3].sum(), rtol=1e-6)
    # top-p: the prefix reaching the mass ends inside the tied pair: both kept
    p = e / e.sum()
    tp = float(p[0] + 0.5 * p[1])
    np.testing.assert_allclose(_renorm(lg, -1, tp), np.r_[e[:3], 0] / e[:3].sum(), rtol=1e-6)


def test_disabled_filters_give_the_tempered_softmax_and_t0_one_hot():
    rng = np.random.default_rng(9)
    lg = rng.normal(0, 2, 50).astype(np.float32)
    for T in (1.0, 0.7, 2.0):
        Tf = float(np.float32(T))  # temperatures travel as fp32
        want = scipy.special.softmax(lg.astype(np.float64) / Tf)
        np.testing.assert_allclose(_renorm(lg, -1, 1.0, T), want, rtol=1e-7)
        np.testing.assert_allclose(_renorm(lg, 50, 1.0, T), want, rtol=1e-7)
    h = _renorm(lg, 5, 0.5, 0.0)
    assert h.sum() == 1.0 and h[int(np.argmax(lg))] == 1.0


def test_temperature_then_filters():
    """Temperature first: T = 0.5 sharpens (0.6, 0.3, 0.1) to (0.78, 0.20, 0.02),
    so top-p 0.75 keeps one token, while at T = 1 it keeps two."""
    lp = np.log([0.6, 0.3, 0.1])
    np.testing.assert_allclose(_renorm(lp, -1, 0.75, 0.5), [1, 0, 0], rtol=1e-6)
    np.testing.assert_allclose(_renorm(lp, -1, 0.75, 1.0), [2 / 3, 1 / 3, 0], rtol=1e-6)


def _tree_case(seed, b=5, n=7, V=30):
    rng = np.random.default_rng(seed)
    parents = [-1] + [int(rng.integers(0, i)) for i in range(1, n)]
    nt, ns = pointers_from_parents(parents)
    logits = rng.normal(0, 2, (b * n, V)).astype(np.float32)
    draft = rng.integers(0, V, b * n).astype(np.int32)
    q = rng.dirichlet(np.full(V, 0.5), b * n).astype(np.float32)
    return rng, parents, np.tile(nt, b), np.tile(ns, b), logits, draft, q


@pytest.mark.parametrize("seed", range(3))
def test_probs_samplers_equal_logit_samplers_without_filters(seed):
    """Fed the temperature softmax as its distribution (both filters off), the
    probabilities-mode samplers give exactly what the logit samplers give."""
    rng, parents, nt, ns, logits, draft, q = _tree_case(seed)
    b, n, S = 5, 7, 3
    T = rng.uniform(0.5, 1.5, b).astype(np.float32)
    probs = oracle.renorm_probs(b, n, logits, T, np.full(b, -1), np.ones(b, np.float32))
    u = rng.random(b * n).astype(np.float32)
    uf = rng.random(b).astype(np.float32)
    ri = np.arange(b * n)
    a = oracle.verify_sampling(b, n, S, logits, q, T, u, uf, draft, ri, nt, ns)
    c = oracle.verify_sampling_probs(b, n, S, probs, q, u, uf, draft, ri, nt, ns)
    for k in a:
        np.testing.assert_array_equal(a[k], c[k], err_msg=k)
    a = oracle.verify_target_only(b, n, S, logits, T, u, uf, 0.8, 0.9, draft, ri, nt, ns)
    c = oracle.verify_target_only_probs(b, n, S, probs, u, uf, 0.8, 0.9, draft, ri, nt, ns)
    for k in a:
        np.testing.assert_array_equal(a[k], c[k], err_msg=k)


def test_rejection_on_a_renormalised_target_follows_it():
    """The p/q rule keeps any target law: single-candidate trials with x ~ q
    against the top-k-3 renormalised target produce that renormalised law
    (chi-square of 1e5 trials) and never a filtered-out token."""
    rng = np.random.default_rng(31)
    V, N = 10, 100_000
    lg = rng.normal(0, 1.5, V).astype(np.float32)
    pr = oracle.renorm_probs(1, 1, lg[None, :], [1.0], [3], [1.0])[0]
    q = rng.dirichlet(np.full(V, 0.8)).astype(np.float32)
    x = np.searchsorted(np.cumsum(q.astype(np.float64)), rng.random(N), side="right").clip(0, V - 1)
    probs = np.zeros((2 * N, V), np.float32)
    probs[0::2] = pr
    probs[1::2] = 1.0 / V
    qq = np.zeros((2 * N, V), np.float32)
    qq[0::2] = q
    draft = np.zeros(2 * N, np.int32)
    draft[1::2] = x
    u = np.zeros(2 * N, np.float32)
    u[1::2] = rng.random(N)
    o = oracle.verify_sampling_probs(N, 2, 1, probs, qq, u, rng.random(N).astype(np.float32), draft,
                                     np.arange(2 * N), np.tile(np.array([1, -1], np.int32), N),
                                     np.full(2 * N, -1, np.int32))
    first = o["accepted_tokens"][:, 0]
    counts = np.bincount(first, minlength=V)
    keep = pr > 0
    assert keep.sum() == 3 and counts[~keep].sum() == 0
    stat, pval = scipy.stats.chisquare(counts[keep], pr[keep].astype(np.float64) / pr[keep].sum() * N)
    assert pval > 1e-3, (stat, pval)
