"""GPU-vs-oracle parity of the draft side of the KV and the FULL_MASK verify
mask, through the C ABI: bit-exact slots, positions, pools and mask bytes."""
import numpy as np
import pytest
import torch

import oracle
from accept_select_top_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _ops():
    from accept_select_top_gb300 import ops
    return ops


def _layout(b, L, S, topk, page, rng):
    """req_to_token rows over permuted pages with room for the prefix and
    every branch region (paged branches) or contiguous branch runs."""
    rows = []
    for q in range(b):
        last = L[q] % page
        base = L[q] - last
        R = -(-(last + S) // page) * page
        need = base + topk * R if (page > 1 and topk > 1) else L[q] + topk * S
        rows.append(-(-need // page) + 1)
    row_w = max(rows) * page
    total_pages = sum(rows) + 3
    perm = rng.permutation(total_pages)
    req_pool_idx = rng.permutation(b + 1)[:b].astype(np.int32)
    r2t = np.zeros((b + 1, row_w), np.int32)
    cur = 0
    for q in range(b):
        pages = perm[cur:cur + rows[q]]
        cur += rows[q]
        pos = np.arange(rows[q] * page)
        r2t[req_pool_idx[q], :len(pos)] = pages[pos // page] * page + pos % page
    return r2t, req_pool_idx, total_pages * page


CASES = [(8, 4, 5, 1), (8, 1, 5, 16), (32, 8, 6, 16), (2, 8, 8, 16), (256, 1, 3, 1), (5, 3, 7, 8)]


@pytest.mark.parametrize("b,topk,S,page", CASES)
def test_assign_draft_locs_parity(b, topk, S, page):
    ops = _ops()
    rng = np.random.default_rng(b * 100 + topk * 10 + S)
    L = rng.integers(1, 3000, b).astype(np.int32)
    r2t, rpi, num_slots = _layout(b, L, S, topk, page, rng)
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a)).cuda()
    out = torch.full((b * topk * S,), 7, dtype=torch.int32, device="cuda")
    pos = torch.full((b,), 7, dtype=torch.int32, device="cuda")
    ws = ops.Workspace(1024)
    ops.spec_assign_draft_locs(b, topk, S, page, t(r2t), t(rpi), t(L), num_slots, out, pos, ws)
    o = oracle.assign_draft_locs(b, topk, S, page, r2t, rpi, L, num_slots)
    assert ws.last_error() == 0
    np.testing.assert_array_equal(out.cpu().numpy(), o["out_cache_loc"])
    if topk == 1:
        np.testing.assert_array_equal(pos.cpu().numpy(), o["positions"])


@pytest.mark.parametrize("b,topk,S,page,layers", [(4, 4, 5, 16, 3), (3, 8, 6, 16, 1), (6, 2, 9, 8, 2)])
def test_duplicate_prefix_tail_parity(b, topk, S, page, layers):
    ops = _ops()
    rng = np.random.default_rng(b + topk + S)
    L = rng.integers(1, 500, b).astype(np.int32)
    L[0] = 32  # a prefix ending on a page boundary: no holes for that request
    r2t, rpi, num_slots = _layout(b, L, S, topk, page, rng)
    Hkv, D = 8, 128
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a)).cuda()
    kl = [torch.randn(num_slots, Hkv, D, device="cuda").to(torch.bfloat16) for _ in range(layers)]
    vl = [torch.randn(num_slots, Hkv, D, device="cuda").to(torch.bfloat16) for _ in range(layers)]
    hk = [W.host(x).copy() for x in kl]
    hv = [W.host(x).copy() for x in vl]
    ws = ops.Workspace(1024)
    ops.spec_duplicate_prefix_tail(b, topk, S, page, Hkv, D, kl, vl, t(r2t), t(rpi), t(L), ws)
    oracle.duplicate_prefix_tail(b, topk, S, page, Hkv, D, hk, hv, r2t, rpi, L)
    assert ws.last_error() == 0
    for i in range(layers):
        np.testing.assert_array_equal(W.host(kl[i]), hk[i], err_msg=f"K layer {i}")
        np.testing.assert_array_equal(W.host(vl[i]), hv[i], err_msg=f"V layer {i}")


@pytest.mark.parametrize("fill", [True, False])
@pytest.mark.parametrize("name", ["tiny", "sampling_heavy", "long_context", "mtp_chain"])
def test_full_mask_parity(name, fill):
    """The FULL_MASK of each workload's tree (from the oracle's select chain),
    written at an odd offset of the buffer so that the head and tail bytes
    take the byte path; without the prefix fill the prefix bytes keep the
    buffer's sentinel."""
    from oracle import pipeline as P
    ops = _ops()
    wl = W.WORKLOADS[name]
    lay = W.kv_layout(wl)
    if wl.k == 1 or name == "tiny":
        drafts = [W.host(W.draft_logits(wl, i)) for i in range(wl.S)]
        bits = P.tree_from_chain(wl, P.select_chain(wl, drafts), W.host(W.bonus_tokens(wl)),
                                 lay["seq_lens"])["mask_bits"]
    else:  # a random ancestor structure of the same size (the mask writer only reads the bits)
        rng = np.random.default_rng(1)
        par = [[-1] + [int(rng.integers(0, i)) for i in range(1, wl.n)] for _ in range(wl.b)]
        bits = np.zeros(wl.b * wl.n, np.uint64)
        for q in range(wl.b):
            for i in range(wl.n):
                m, x = 0, i
                while x != -1:
                    m |= 1 << x
                    x = par[q][x]
                bits[q * wl.n + i] = m
    L = lay["seq_lens"]
    total = int(np.sum(wl.n * (L.astype(np.int64) + wl.n)))
    sentinel = 9
    buf = torch.full((total + 19,), sentinel, dtype=torch.uint8, device="cuda")
    view = buf[3:3 + total]  # an unaligned start
    ws = ops.Workspace(1024)
    ops.spec_build_full_mask(wl.b, wl.n, torch.as_tensor(L).cuda(), torch.as_tensor(bits.view(np.int64)).cuda(),
                             fill, view, ws)
    assert ws.last_error() == 0
    got = buf.cpu().numpy()
    o = oracle.full_mask(wl.b, wl.n, L, bits, fill_prefix=fill, out=np.full(total, sentinel, np.uint8))
    np.testing.assert_array_equal(got[3:3 + total], o)
    assert (got[:3] == sentinel).all() and (got[3 + total:] == sentinel).all()  # nothing outside the mask


def test_full_mask_too_small_buffer_writes_nothing():
    ops = _ops()
    L = torch.tensor([5, 6], dtype=torch.int32, device="cuda")
    bits = torch.tensor([1, 3, 1, 3], dtype=torch.int64, device="cuda")
    buf = torch.full((10,), 9, dtype=torch.uint8, device="cuda")  # needs 2*(5+2) + 2*(6+2) = 30
    ws = ops.Workspace(1024)
    ops.spec_build_full_mask(2, 2, L, bits, True, buf, ws)
    assert ws.last_error() & 4  # SPEC_DEV_LENGTH
    assert (buf.cpu().numpy() == 9).all()
