"""GPU-vs-oracle parity of the relaxed penalties, the top-k / top-p
renormalisation and the samplers on a given distribution, through the C ABI.

Bars: the penalty add bit-exact; the renormalised support exact at the top-k
cut (an integer count on exact keys) and at the top-p cut unless the
cumulative mass there is within 1e-6 of top_p (a near tie, reported);
probabilities within 1e-5 relative (fp32 exp of a correctly rounded quotient
against the oracle's fp64); the samplers, fed the oracle's distribution,
bit-exact apart from certified terminal near ties."""
import numpy as np
import pytest
import torch

import oracle
from accept_select_top_gb300 import workloads as W
from tests.cases import bf16_to_f64, make_case

pytestmark = pytest.mark.gpu


def _ops():
    from accept_select_top_gb300 import ops
    return ops


@pytest.mark.parametrize("name", ["tiny", "sampling_heavy"])
def test_add_penalties_parity(name):
    ops = _ops()
    wl = W.WORKLOADS[name]
    g = torch.Generator(device="cuda").manual_seed(3)
    logits = (torch.randn(wl.b * wl.n, wl.V, device="cuda", generator=g) * 2).to(wl.torch_logits_dtype)
    pen = torch.randn(wl.b, wl.V, device="cuda", generator=g)
    host = W.host(logits).copy()
    ops.spec_add_penalties(wl.b, wl.n, logits, pen)
    o = oracle.add_penalties(wl.b, wl.n, host, W.host(pen))
    np.testing.assert_array_equal(W.host(logits), o)


def _settings(b, rng):
    """Per-request temperature, top_k and top_p: both filters, each alone,
    neither, and a greedy request."""
    T = rng.uniform(0.6, 1.4, b).astype(np.float32)
    k = rng.choice([-1, 1, 20, 50, 4000], b).astype(np.int32)
    p = rng.choice([1.0, 0.9, 0.95, 0.5], b).astype(np.float32)
    T[0], k[0], p[0] = 1.0, 50, 0.9
    if b > 1:
        T[1] = 0.0
    if b > 2:
        k[2], p[2] = -1, 1.0
    return T, k, p


def _check_rows(lg, T, k, p, got, want, rows):
    """Support and values of the sampled rows; returns how many rows differ
    at a certified top-p near tie."""
    certified = 0
    for j, r in enumerate(rows):
        g, o = got[r], want[j]
        gs, os_ = g > 0, o > 0
        if not np.array_equal(gs, os_):
            # only the top-p cut may move, and only at a near tie of the mass
            assert p[j] < 1.0 and T[j] > 0, (r, "support differs without a top-p cut")
            x = lg[r].astype(np.float64)
            e = np.exp((x - x.max()) / np.float64(np.float32(T[j])))
            kept_k = np.ones_like(gs) if not (0 < k[j] < x.size) else x >= np.sort(x)[::-1][k[j] - 1]
            e = np.where(kept_k, e, 0.0)
            zk = e.sum()
            for cut in (x[gs].min(), x[os_].min()):
                assert abs(e[x > cut].sum() / zk - p[j]) <= 1e-6 or abs(e[x >= cut].sum() / zk - p[j]) <= 1e-6, \
                    (r, "top-p cut moved without a near tie")
            certified += 1
            continue
        np.testing.assert_allclose(g[gs], o[gs], rtol=1e-5, err_msg=f"row {r}")
    return certified


@pytest.mark.parametrize("name", ["tiny", "sampling_heavy", "mtp_chain"])
def test_renorm_parity(name, record_property):
    ops = _ops()
    wl = W.WORKLOADS[name]
    rng = np.random.default_rng(11)
    g = torch.Generator(device="cuda").manual_seed(5)
    logits = (torch.randn(wl.b * wl.n, wl.V, device="cuda", generator=g) * 2).to(wl.torch_logits_dtype)
    T, k, p = _settings(wl.b, rng)
    probs = torch.empty(wl.b * wl.n, wl.V, device="cuda")
    t = lambda a: torch.as_tensor(a).cuda()
    ops.spec_renorm_probs(wl.b, wl.n, logits, t(T), t(k), t(p), probs)
    got = probs.cpu().numpy()
    lgh = W.host(logits)
    lg = bf16_to_f64(lgh) if lgh.dtype == np.uint16 else lgh.astype(np.float64)
    # the oracle on a sample of rows: every row of the first three requests, then a spread
    rows = sorted(set(list(range(min(wl.b, 3) * wl.n)) + list(rng.choice(wl.b * wl.n, min(40, wl.b * wl.n), replace=False))))
    req = np.array(rows) // wl.n
    want = oracle.renorm_probs(len(rows), 1, np.ascontiguousarray(lgh[rows]), T[req], k[req], p[req])
    n_cert = _check_rows(lg, T[req], k[req], p[req], got, want, rows)
    record_property("certified_top_p_cuts", n_cert)
    assert n_cert <= 2
    np.testing.assert_allclose(got.sum(axis=1), 1.0, rtol=1e-5)


@pytest.mark.parametrize("sampler", ["classic", "target_only"])
@pytest.mark.parametrize("name", ["tiny", "mtp_chain"])
def test_probs_samplers_parity(name, sampler):
    """Both samplers fed the oracle's renormalised target distribution (top-k
    and top-p per request): bit-exact accept on the same probabilities."""
    ops = _ops()
    c = make_case(W.WORKLOADS[name], "sampling", with_attention=False)
    wl = c.wl
    rng = np.random.default_rng(2)
    T, k, p = _settings(wl.b, rng)
    probs_h = oracle.renorm_probs(wl.b, wl.n, W.host(c.logits), T, k, p)
    probs = torch.as_tensor(probs_h).cuda()
    tree = [torch.as_tensor(np.ascontiguousarray(c.tree[x])).cuda()
            for x in ("draft_tokens", "retrieve_index", "next_token", "next_sibling")]
    z = lambda *s_: torch.zeros(s_, dtype=torch.int32, device="cuda")
    out = [z(wl.b * wl.n), z(wl.b, wl.W), z(wl.b), z(wl.b, wl.W), z(wl.b)]
    args = (c.tree["draft_tokens"], c.tree["retrieve_index"], c.tree["next_token"], c.tree["next_sibling"])
    if sampler == "classic":
        ws = ops.Workspace(ops.spec_workspace_size(ops.OP_VERIFY_SAMPLING, wl.b, wl.n, 1, wl.V))
        ops.spec_verify_sampling_probs(wl.b, wl.n, wl.S, probs, c.q, c.u, c.u_final, *tree, *out, ws)
        o = oracle.verify_sampling_probs(wl.b, wl.n, wl.S, probs_h, W.host(c.q), W.host(c.u), W.host(c.u_final),
                                         *args)
    else:
        ws = ops.Workspace(ops.spec_workspace_size(ops.OP_VERIFY_TARGET_ONLY, wl.b, wl.n, 1, wl.V))
        ops.spec_verify_target_only_probs(wl.b, wl.n, wl.S, probs, c.u, c.u_final, 0.6, 0.8, *tree, *out, ws)
        o = oracle.verify_target_only_probs(wl.b, wl.n, wl.S, probs_h, W.host(c.u), W.host(c.u_final), 0.6, 0.8,
                                            *args)
    assert ws.last_error() == 0
    names = ("predict", "accept_index", "accept_lens", "accepted_tokens", "next_root")
    g = {n_: x.cpu().numpy() for n_, x in zip(names, out)}
    # the walk decisions compare the same fp32 probabilities on both sides
    np.testing.assert_array_equal(g["accept_lens"], o["accept_lens"])
    np.testing.assert_array_equal(g["accept_index"], o["accept_index"])
    bad = []
    for r in range(wl.b):
        L = o["accept_lens"][r]
        if g["accepted_tokens"][r, L - 1] != o["accepted_tokens"][r, L - 1]:
            # the terminal draw: certified only at the boundary between the two tokens
            row = int(o["accept_index"][r, L - 1])
            pr = probs_h[row].astype(np.float64)
            if L - 1 < wl.S and c.tree["next_token"][row] != -1:  # every child of the terminal node rejected
                if sampler == "classic":
                    res = np.maximum(pr - W.host(c.q)[row].astype(np.float64), 0)
                else:  # target-only: the rejected children's tokens left out
                    res = pr.copy()
                    ch = int(c.tree["next_token"][row])
                    base = r * wl.n
                    while ch != -1:
                        res[int(c.tree["draft_tokens"][base + ch])] = 0.0
                        ch = int(c.tree["next_sibling"][base + ch])
                pr = res if res.sum() > 0 else pr
            cdf = np.cumsum(pr) / pr.sum()
            lo, hi = sorted((int(g["accepted_tokens"][r, L - 1]), int(o["accepted_tokens"][r, L - 1])))
            if abs(cdf[lo] - float(W.host(c.u_final)[r])) > 1e-6:
                bad.append(r)
    assert not bad, bad
