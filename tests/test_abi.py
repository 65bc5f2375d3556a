"""The C-ABI library loads on a machine without a GPU, exports every entry
point the header declares, and validates arguments on the host (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"^\s*(?:size_t|int)\s+(spec_\w+)\s*\(", text, re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from accept_select_top_gb300 import build
    return ctypes.CDLL(build.build())


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10, names
    for name in names:
        assert hasattr(lib, name), name


def test_binding_names_match_header():
    from accept_select_top_gb300 import ops
    assert sorted(ops.EXPORTS) == _declared()
    for name in _declared():
        assert hasattr(ops.LIB, name)


def test_workspace_sizes_host_only():
    from accept_select_top_gb300 import ops
    for op in range(6):
        s = ops.spec_workspace_size(op, 8, 16, 4, 128256, 32, 8, 4096)
        assert s >= 256 + 64
    assert ops.spec_workspace_size(ops.OP_VERIFY_GREEDY, 0, 16, 4, 1000) > 0  # idle batch
    assert ops.spec_workspace_size(ops.OP_VERIFY_GREEDY, 8, 65, 4, 1000) == 0  # n > 64
    assert ops.spec_workspace_size(ops.OP_SELECT_TOPK, 8, 16, 17, 1000) == 0   # k > 16
    assert ops.spec_workspace_size(99, 8, 16, 4, 1000) == 0


def test_workspace_layout_keeps_overlapping_calls_apart_host_only():
    """Greedy accept may scan while the attention before it finishes, so its
    partials lie past the attention's merge area: its workspace need covers that
    area plus its own partials, for any batch.  The select keeps two halves of
    its partials (a select may overlap the previous one), past the commit's
    area."""
    from accept_select_top_gb300 import ops
    for b, n in ((1, 4), (8, 16), (32, 64), (256, 4)):
        att = ops.spec_workspace_size(ops.OP_VERIFY_ATTENTION, b, n, 1, 1, 32, 8, 4096)
        gre = ops.spec_workspace_size(ops.OP_VERIFY_GREEDY, b, n, 1, 128256)
        assert gre > att, (b, n)
    base = ops.spec_workspace_size(ops.OP_BUILD_TREE, 8, 16, 4, 128256)  # header + counters only
    sel = ops.spec_workspace_size(ops.OP_SELECT_TOPK, 8, 16, 4, 128256)
    # two halves of 32 rows x 19 chunks x 144-byte partials, past the commit's area
    assert sel - base >= 2 * 32 * 19 * 144


def test_overlap_switch_host_only(lib):
    """Overlap is a per-workspace permission: it takes 0 or 1 and a non-NULL
    workspace, and needs no device (nothing is enqueued)."""
    f = lib.spec_workspace_set_overlap
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int]
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: the call only records a flag
    assert f(fake, 1) == 0
    assert f(fake, 0) == 0
    assert f(fake, 2) == -1
    assert f(None, 1) == -2


def test_launches_per_step_host_only():
    """S selects (two launches each where a call streams at least 32 MiB of
    whole 16-byte vectors), the tree build, one attention launch, the accept
    (two or three when sampling) and the commit."""
    import dataclasses
    from accept_select_top_gb300 import workloads as W
    from accept_select_top_gb300.pipeline import launches_per_step
    wl = W.WORKLOADS["llama8b_greedy"]  # 8 MiB a select call: the chunked select
    assert launches_per_step(wl, "greedy") == wl.S + 4
    sh = W.WORKLOADS["sampling_heavy"]  # step 0: 8 MiB; later steps: 66 MB, streamed
    assert launches_per_step(sh, "sampling") == 1 + 2 * (sh.S - 1) + 3 + 3
    odd = dataclasses.replace(sh, V=sh.V + 1)  # bf16 rows of an odd length: chunked select and accept
    assert launches_per_step(odd, "sampling") == sh.S + 3 + 2


def test_host_argument_checks_without_gpu(lib):
    """Rejected arguments and the idle batch return before any CUDA call."""
    P = ctypes.c_void_p
    f = lib.spec_select_topk
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 5 + [P, ctypes.c_float, P, P, P, ctypes.c_int, P, ctypes.c_int, P, P, P, P,
                                       ctypes.c_size_t, P]
    args = lambda step, b, k, V, dt, T: (step, b, k, V, dt, None, T, None, None, None, 4, None, 5, None, None,
                                         None, None, 0, None)
    assert f(*args(0, 0, 4, 100, 1, 1.0)) == 0        # b == 0: no-op
    assert f(*args(0, 2, 17, 100, 1, 1.0)) == -1      # k > 16
    assert f(*args(0, 2, 4, 3, 1, 1.0)) == -1         # V < k
    assert f(*args(0, 2, 4, 100, 7, 1.0)) == -4       # dtype
    assert f(*args(0, 2, 4, 100, 1, 0.0)) == -1       # temperature
    assert f(*args(0, 2, 4, 100, 1, 1.0)) == -1       # null pointers
    g = lib.spec_verify_attention
    g.restype = ctypes.c_int
    g.argtypes = [ctypes.c_int] * 6 + [P, P, P, ctypes.c_int64, P, ctypes.c_int, ctypes.c_int, P, P,
                                       ctypes.c_int, P, P, ctypes.c_float, P, P, P, ctypes.c_size_t, P]
    base = [2, 4, 8, 2, 128, 1, None, None, None, 10, None, 1, 10, None, None, 10, None, None, 0.1, None, None,
            None, 0, None]
    bad_d = list(base)
    bad_d[4] = 96
    assert g(*bad_d) == -4
    bad_g = list(base)
    bad_g[3] = 3
    assert g(*bad_g) == -1
    assert g(*base) == -1  # null pointers
