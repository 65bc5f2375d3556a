"""spec_verify_greedy_noalloc: the greedy accept for callers that cannot
allocate device memory (an engine allocator that owns all device memory, a
latency path that must avoid cudaMalloc's implicit synchronisation, a plugin
host that forbids allocation after start-up).  It must give exactly what
spec_verify_greedy gives with a caller workspace, on consecutive calls that
reuse the library's fixed scratch array, including the clamped outputs of a
tree with an out-of-range index, whose error bit spec_noalloc_last_error
reports.  This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

from accept_select_top_gb300 import workloads as W
from tests.cases import make_case

pytestmark = pytest.mark.gpu


def _bufs(wl):
    z = lambda *s: torch.full(s, 7, dtype=torch.int32, device="cuda")  # not zero: outputs must be written
    return [z(wl.b * wl.n), z(wl.b, wl.W), z(wl.b), z(wl.b, wl.W), z(wl.b)]


@pytest.mark.parametrize("name", ["llama8b_greedy", "tiny"])
def test_noalloc_matches_workspace_entry_point_twice(name):
    from accept_select_top_gb300 import ops
    c = make_case(W.WORKLOADS[name], "greedy", with_attention=False)
    wl = c.wl
    tree = [torch.as_tensor(np.ascontiguousarray(c.tree[k])).cuda()
            for k in ("draft_tokens", "retrieve_index", "next_token", "next_sibling")]
    ws = ops.Workspace(ops.spec_workspace_size(ops.OP_VERIFY_GREEDY, wl.b, wl.n, 1, wl.V))
    ref = _bufs(wl)
    ops.spec_verify_greedy(wl.b, wl.n, wl.S, c.logits, *tree, *ref, ws)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    V = wl.V
    dtype = ops.SPEC_F32 if c.logits.dtype == torch.float32 else ops.SPEC_BF16
    for _ in range(2):  # the second call reuses the scratch the first one left behind
        out = _bufs(wl)
        rc = ops.LIB.spec_verify_greedy_noalloc(wl.b, wl.n, wl.S, V, dtype, P(c.logits), *[P(t) for t in tree],
                                                *[P(t) for t in out], stream)
        assert rc == 0
        torch.cuda.synchronize()
        for a, b in zip(out, ref):
            assert torch.equal(a, b)
    assert ws.last_error() == 0
    assert ops.spec_noalloc_last_error() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from accept_select_top_gb300 import ops
    x = torch.zeros(1, device="cuda")
    i = torch.zeros(1, dtype=torch.int32, device="cuda")
    # 4096 requests x 64 nodes need one 8-byte partial per verify row: 2 MiB > the 1 MiB scratch
    need = ops.spec_workspace_size(ops.OP_VERIFY_GREEDY, 4096, 64, 1, 128256)
    assert need > (1 << 20)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = ops.LIB.spec_verify_greedy_noalloc(4096, 64, 4, 128256, ops.SPEC_BF16, P(x), P(i), P(i), P(i), P(i), P(i),
                                            P(i), P(i), P(i), P(i), None)
    assert rc == -2


def test_noalloc_bad_index_clamps_like_the_workspace_entry_point():
    """A next_token pointing outside the tree: both entry points skip the bad
    pointer the same way and give the same outputs; the no-allocation entry
    point still returns SPEC_OK, and its error bit stays set across calls until
    spec_noalloc_last_error reads and clears it."""
    from accept_select_top_gb300 import ops
    c = make_case(W.WORKLOADS["tiny"], "greedy", with_attention=False)
    wl = c.wl
    tree = [torch.as_tensor(np.ascontiguousarray(c.tree[k])).cuda()
            for k in ("draft_tokens", "retrieve_index", "next_token", "next_sibling")]
    tree[2] = tree[2].clone()
    tree[2][0] = 1000  # the root's first child: out of range
    ws = ops.Workspace(ops.spec_workspace_size(ops.OP_VERIFY_GREEDY, wl.b, wl.n, 1, wl.V))
    ref = _bufs(wl)
    ops.spec_verify_greedy(wl.b, wl.n, wl.S, c.logits, *tree, *ref, ws)
    assert ws.last_error() & ops.DEV_INDEX
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dtype = ops.SPEC_F32 if c.logits.dtype == torch.float32 else ops.SPEC_BF16
    ops.spec_noalloc_last_error()  # start from a clean word, whatever ran before
    for _ in range(2):
        out = _bufs(wl)
        rc = ops.LIB.spec_verify_greedy_noalloc(wl.b, wl.n, wl.S, wl.V, dtype, P(c.logits), *[P(t) for t in tree],
                                                *[P(t) for t in out], stream)
        assert rc == 0
        torch.cuda.synchronize()
        for a, b in zip(out, ref):
            assert torch.equal(a, b)
    assert ops.spec_noalloc_last_error() & ops.DEV_INDEX
    assert ops.spec_noalloc_last_error() == 0  # read-and-clear


def test_noalloc_rejects_null_pointers_before_enqueueing():
    """A NULL input is refused with SPEC_ERR_ARG before anything is put on the
    stream (no device pointer here is ever dereferenced)."""
    from accept_select_top_gb300 import ops
    i = torch.zeros(64, dtype=torch.int32, device="cuda")
    x = torch.zeros(16, 1024, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = ops.LIB.spec_verify_greedy_noalloc(4, 4, 3, 1024, ops.SPEC_F32, None, P(i), P(i), P(i), P(i), P(i),
                                            P(i), P(i), None, None, None)
    assert rc == -1
    rc = ops.LIB.spec_verify_greedy_noalloc(4, 4, 3, 1024, ops.SPEC_F32, P(x), P(i), P(i), None, P(i), P(i),
                                            P(i), P(i), None, None, None)
    assert rc == -1
