"""The allocation-free decode forward, checked against detffn_forward.

detffn_forward_decode_noalloc serves callers that cannot call cudaMalloc (for
example when a caching allocator's pool already holds the device's memory):
it keeps its scratch in fixed arrays inside the library instead of a
caller-provided workspace.  This file is collected last, so that a run that
stops at the first failure has already run every other test.  It checks, on
two calls in a row, that the output equals detffn_forward's on the exact path
bit for bit (the tolerance of the exact path is 0 mismatching elements) and
that the call's status word reports no timeout; that the output equals the
CPU oracle's; that a bounded wait that runs out (a test setting, no fault)
is reported by the call's status word; and that sizes beyond its limits are
refused before anything is launched.
"""
import numpy as np
import pytest
import torch

from gemm_deterministic_bf16_gb300.inputs import ffn_inputs
from tests.gpu_util import dev, host, mismatches

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    import gemm_deterministic_bf16_gb300 as G
    from gemm_deterministic_bf16_gb300 import build
    build.build()
    return G


@pytest.mark.parametrize("M,H,I", [(8, 4096, 12288), (1, 4096, 12288), (5, 1024, 3072)])
def test_noalloc_matches_forward_twice(G, M, H, I):
    d = ffn_inputs(M, H, I, seed=40 + M, with_dout=False)
    t = {n: dev(v) for n, v in d.items()}
    ref = host(G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], path=G.PATH_EXACT))
    out = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    for _ in range(2):
        out.fill_(0)
        G.detffn_forward_decode_noalloc(t["x"], t["Wg"], t["Wu"], t["Wd"], out=out)
        torch.cuda.synchronize()
        assert mismatches(host(out), ref) == 0
        # No bounded wait ran out (the call's own status word, read and cleared).
        assert G.detffn_forward_decode_noalloc_status() == 0


def test_noalloc_matches_oracle(G, oracle_mod):
    """Against the CPU oracle directly: the allocation-free call gives the
    oracle's bits (its leaves follow the oracle's stated in-leaf order)."""
    M, H, I = 4, 1024, 3072
    d = ffn_inputs(M, H, I, seed=77, with_dout=False)
    t = {n: dev(v) for n, v in d.items()}
    out = G.detffn_forward_decode_noalloc(t["x"], t["Wg"], t["Wu"], t["Wd"])
    torch.cuda.synchronize()
    ref = oracle_mod.ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"])
    assert mismatches(host(out), ref["out"]) == 0
    assert G.detffn_forward_decode_noalloc_status() == 0


def test_noalloc_reports_a_wait_that_ran_out(G):
    """The failure path, without any fault: with the test setting that makes
    the kernels issue no copies and a short poll limit, the first wait of the
    gate/up launch runs out; the call's status word reports DETFFN_ERR_TIMEOUT
    (the down launch returns at entry, leaving out untouched), reading it
    clears it, and the next normal call is bit-identical to detffn_forward."""
    M, H, I = 2, 1024, 3072
    d = ffn_inputs(M, H, I, seed=81, with_dout=False)
    t = {n: dev(v) for n, v in d.items()}
    ref = host(G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], path=G.PATH_EXACT))
    out = torch.zeros(M, H, dtype=torch.bfloat16, device="cuda")
    assert G.detffn_forward_decode_noalloc_status() == 0
    G.detffn_forward_decode_noalloc_test_waits(spin_limit=4096, stall=1)
    try:
        G.detffn_forward_decode_noalloc(t["x"], t["Wg"], t["Wu"], t["Wd"], out=out)
        torch.cuda.synchronize()
        assert G.detffn_forward_decode_noalloc_status() == 7           # DETFFN_ERR_TIMEOUT
        assert G.detffn_forward_decode_noalloc_status() == 0           # read and cleared
        assert not torch.any(out.view(torch.int16) != 0).item()        # the down launch did nothing
    finally:
        G.detffn_forward_decode_noalloc_test_waits(0, 0)
    G.detffn_forward_decode_noalloc(t["x"], t["Wg"], t["Wu"], t["Wd"], out=out)
    torch.cuda.synchronize()
    assert G.detffn_forward_decode_noalloc_status() == 0
    assert mismatches(host(out), ref) == 0
    with pytest.raises(G.DetFFNError):
        G.detffn_forward_decode_noalloc_test_waits(spin_limit=-1)


def test_noalloc_rejects_sizes_beyond_limits(G):
    x = torch.zeros(9, 256, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(768, 256, dtype=torch.bfloat16, device="cuda")
    wd = torch.zeros(256, 768, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(G.DetFFNError) as e:
        G.detffn_forward_decode_noalloc(x, w, w, wd)   # M = 9 > 8
    assert e.value.status == 2
    big = torch.zeros(32768, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(G.DetFFNError) as e:
        G.detffn_forward_decode_noalloc(x[:1], big, big,
                                        torch.zeros(256, 32768, dtype=torch.bfloat16, device="cuda"))
    assert e.value.status == 2                           # I = 32768 > 12288
    xh = torch.zeros(1, 8192, dtype=torch.bfloat16, device="cuda")
    wh = torch.zeros(768, 8192, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(G.DetFFNError) as e:
        G.detffn_forward_decode_noalloc(xh, wh, wh, torch.zeros(8192, 768, dtype=torch.bfloat16, device="cuda"))
    assert e.value.status == 2                           # H = 8192: 128 leaves, not covered
