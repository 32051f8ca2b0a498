"""Host-side checks of the C ABI (no GPU compute): the library loads, exports
every symbol include/detffn.h declares, builds its SiLU tables identically to
the oracle's, sizes workspaces consistently, and rejects bad arguments before
launching anything."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from gemm_deterministic_bf16_gb300 import build, detffn
    build.build()
    return detffn.lib()


def _declared():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"DETFFN_API\s+[\w\s\*]+?\b(detffn_\w+)\s*\(", txt)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n


def test_library_silu_tables_equal_oracle(L, oracle_mod):
    from gemm_deterministic_bf16_gb300 import detffn_silu_tables
    s, d = detffn_silu_tables(host_only=True)
    os_, od = oracle_mod.silu_tables()
    nan = (os_ & 0x7FFF) > 0x7F80
    assert np.array_equal(s[~nan], os_[~nan])
    assert np.array_equal((s[nan] & 0x7FFF) > 0x7F80, np.ones(nan.sum(), bool))
    fin = np.isfinite(od)
    assert np.array_equal(d[fin].view(np.uint32), od[fin].view(np.uint32))


def test_status_strings(L):
    for s in range(8):
        assert L.detffn_status_string(s)


def _ws(L, op, M, H, I, k=1):
    from gemm_deterministic_bf16_gb300.detffn import Options
    n = ctypes.c_size_t()
    st = L.detffn_workspace_size(None, op, M, H, I, k, ctypes.byref(Options(64, 0, 1, 0)), ctypes.byref(n))
    return st, n.value


def test_workspace_sizes(L):
    st, n1 = _ws(L, 0, 32, 4096, 12288)
    assert st == 0 and n1 >= 3 * 32 * 12288 * 2
    st, n2 = _ws(L, 1, 32, 4096, 12288, 8)
    assert st == 0 and n2 >= 3 * 32 * 12288 * 2 + 8 * 32 * 4096 * 2   # stage tensors + shard partials
    assert _ws(L, 1, 32, 4096, 12288, 3)[0] == 1          # k not in {1,2,4,8}
    assert _ws(L, 9, 32, 4096, 12288)[0] == 1             # unknown op
    assert _ws(L, 0, 32, 0, 12288)[0] == 2                # H = 0


def test_argument_errors_launch_nothing(L):
    from gemm_deterministic_bf16_gb300.detffn import Options
    opts = ctypes.byref(Options(64, 0, 1, 0))
    # No handle.
    assert L.detffn_forward(None, 16, 16, 16, 16, 16, None, None, 1, 64, 64, None, 0, None, opts) == 1
    # Rank tree: n = 3, bad dtype, misaligned fp32 output, partial overlap.
    p = (ctypes.c_void_p * 8)(*([4096] * 8))
    assert L.detffn_rank_tree_reduce(p, 3, 8192, 16, 2, None) == 1
    assert L.detffn_rank_tree_reduce(p, 2, 8192, 16, 7, None) == 1
    assert L.detffn_rank_tree_reduce(p, 2, 8194, 16, 0, None) == 3
    q = (ctypes.c_void_p * 2)(4096, 8192)
    assert L.detffn_rank_tree_reduce(q, 2, 4100, 16, 2, None) == 1
    # Unsupported leaf width.
    bad = ctypes.byref(Options(32, 0, 1, 0))
    n = ctypes.c_size_t()
    assert L.detffn_workspace_size(None, 0, 1, 64, 64, 1, bad, ctypes.byref(n)) == 4
    # Unknown option flag bits and a negative poll limit are argument errors.
    for fl in (16, 32, 1 << 30, -1):
        assert L.detffn_workspace_size(None, 0, 1, 64, 64, 1, ctypes.byref(Options(64, 0, 1, fl, 0)),
                                       ctypes.byref(n)) == 1
    for fl in (2, 4, 6, 8):  # dHidden overlap, two-launch forward, host buffers: valid flags
        assert L.detffn_workspace_size(None, 0, 1, 64, 64, 1, ctypes.byref(Options(64, 0, 1, fl, 0)),
                                       ctypes.byref(n)) == 0
    # Host buffers (flag 8): the forward's workspace holds the staged x and
    # out (two 256-byte-aligned blocks of M*H BF16 here); the backward and
    # the chunked weight gradients do not take the flag.
    plain, hio = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.detffn_workspace_size(None, 0, 1, 64, 64, 1, ctypes.byref(Options(64, 0, 1, 0, 0)),
                                   ctypes.byref(plain)) == 0
    assert L.detffn_workspace_size(None, 0, 1, 64, 64, 1, ctypes.byref(Options(64, 0, 1, 8, 0)),
                                   ctypes.byref(hio)) == 0
    assert hio.value == plain.value + 512
    assert L.detffn_workspace_size(None, 1, 1, 64, 128, 2, ctypes.byref(Options(64, 0, 1, 8, 0)),
                                   ctypes.byref(hio)) == 0
    for op in (2, 3):
        assert L.detffn_workspace_size(None, op, 1, 64, 64, 1, ctypes.byref(Options(64, 0, 1, 8, 0)),
                                       ctypes.byref(n)) == 1
    assert L.detffn_workspace_size(None, 0, 1, 64, 64, 1, ctypes.byref(Options(64, 0, 1, 0, -5)),
                                   ctypes.byref(n)) == 1
    assert L.detffn_workspace_size(None, 0, 1, 64, 64, 1, ctypes.byref(Options(64, 0, 1, 1, 100)),
                                   ctypes.byref(n)) == 0
    # Leaf dump and conversion diagnostics: argument errors before any launch.
    L.detffn_tree_gemm_leaves.argtypes = [ctypes.c_void_p] * 1 + [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_longlong,
                                          ctypes.c_void_p, ctypes.c_longlong, ctypes.c_longlong, ctypes.c_longlong,
                                          ctypes.c_longlong, ctypes.c_longlong, ctypes.c_void_p, ctypes.c_longlong,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert L.detffn_tree_gemm_leaves(None, 16, 64, 1, 16, 64, 1, 1, 1, 64, 16, 1, 16, None, None) == 1
    L.detffn_cvt_f32_bf16.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong,
                                      ctypes.c_void_p]
    assert L.detffn_cvt_f32_bf16(None, 16, 32, 4, None) == 1


def test_header_names_readings():
    txt = open(os.path.join(ROOT, "include", "detffn.h")).read()
    for needle in ["leaf", "midpoint", "rne_bf16", "PR #325", "PR #357"]:
        assert needle in txt


def test_piece_decomposition_and_fold_selfcheck():
    """The few-token tensor kernels split each tile's tree into pieces (maximal
    aligned blocks of bottom groups) by a closed form and fold them with
    per-piece codes; the library's host check compares the closed form with
    the greedy decomposition on every range of every tile of up to 256 groups
    and replays the fold symbolically on every three-way split of each tile
    (the pieces of each right child must meet their own left sibling and end
    in the root once).  No GPU is needed."""
    from gemm_deterministic_bf16_gb300 import build, detffn
    build.build()
    assert detffn.detffn_selfcheck_pieces(8) == 0
    L = detffn.lib()
    n = ctypes.c_ulonglong()
    L.detffn_selfcheck_pieces.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_ulonglong)]
    assert L.detffn_selfcheck_pieces(9, ctypes.byref(n)) != 0          # out of range: an argument error
    assert L.detffn_selfcheck_pieces(8, None) != 0


def test_fused_forward_schedule_selfcheck():
    """The one-launch decode forward's schedule, checked on the host over a
    grid of shapes and SM counts: every down block on one CTA, each range of
    I counting exactly the gate/up tiles its blocks read, the waiter counts,
    and the fold's room in the pipeline stages.  The benchmark shape (H = 4096,
    I = 12288) is among the covered ones.  No GPU is needed."""
    from gemm_deterministic_bf16_gb300 import build, detffn
    build.build()
    cases, failures = detffn.detffn_selfcheck_fused_schedule()
    assert failures == 0
    assert cases >= 50, cases
    L = detffn.lib()
    L.detffn_selfcheck_fused_schedule.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    assert L.detffn_selfcheck_fused_schedule(None, None) != 0
