"""The bounded-wait failure path, exercised without faulting or hanging a GPU.

Every mbarrier wait in the streaming kernels is bounded; when one runs out
the CTA records DETFFN_ERR_TIMEOUT in the handle's status word, drains the
copies it issued and exits.  A test makes a wait run out by withholding
work (the test-only DETFFN_FLAG_TEST_STALL: the kernels issue no copies, so
the barrier they wait on is never completed) together with a small poll
limit.  Checked for each kernel family that waits (exact weight streaming,
few-token and many-token tensor kernels):

* the call returns (no hang) and detffn_get_status reports the timeout;
* the status word is sticky: a normal call made before it is read launches
  kernels that return at entry and leave the output untouched;
* after the status is read (and cleared), a normal call is bit-identical to
  a call that never saw a timeout, and the status reads OK.

The failure-detection model follows the pages' bounded collectives
(RL-Kernel PR #357, "Design": ready/done generations) restated for waits
inside one GPU.
"""
import numpy as np
import pytest
import torch

from gemm_deterministic_bf16_gb300.inputs import ffn_inputs
from tests.gpu_util import dev, host, mismatches

pytestmark = pytest.mark.gpu
OK, TIMEOUT = 0, 7


@pytest.fixture(scope="module")
def G():
    import gemm_deterministic_bf16_gb300 as G
    from gemm_deterministic_bf16_gb300 import build
    build.build()
    assert G.detffn_get_status() == OK
    return G


@pytest.mark.parametrize("path,M,H,I", [(1, 8, 1024, 3072),      # exact weight streaming (k_decode)
                                        (2, 8, 1024, 3072),      # few-token tensor kernels (k_tcs), top kernel
                                        (2, 8, 1024, 1536),      # k_tcs, trees folded by their last CTA
                                        (2, 256, 512, 1536)])    # many-token tensor kernel (k_tc)
def test_stalled_wait_times_out_and_recovers(G, path, M, H, I):
    d = ffn_inputs(M, H, I, seed=90 + M, with_dout=False)
    t = {n: dev(v) for n, v in d.items()}
    ref = host(G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], path=path))
    assert G.detffn_get_status() == OK
    sentinel = torch.full((M, H), 7.0, dtype=torch.bfloat16, device="cuda")
    out = sentinel.clone()
    # A call whose waits cannot complete: it returns, and reports the timeout.
    G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], out=out, path=path, spin_limit=2048,
                     flags=G.FLAG_TEST_STALL)
    torch.cuda.synchronize()
    # Sticky: a normal call before the status is read does nothing to `out`.
    out2 = sentinel.clone()
    G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], out=out2, path=path)
    torch.cuda.synchronize()
    assert mismatches(host(out2), host(sentinel)) == 0
    assert G.detffn_get_status() == TIMEOUT
    assert G.detffn_get_status() == OK                 # reading it cleared it
    # Recovered: the same call gives the bits of a call that never timed out.
    got = host(G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], path=path))
    assert G.detffn_get_status() == OK
    assert mismatches(got, ref) == 0


def test_small_poll_limit_without_stall_is_harmless(G):
    """A poll limit that legitimate waits may or may not exceed: either the
    call completes with the right bits, or it reports a timeout; it never
    hangs, and a normal call afterwards is bit-identical."""
    M, H, I = 8, 1024, 3072
    d = ffn_inputs(M, H, I, seed=97, with_dout=False)
    t = {n: dev(v) for n, v in d.items()}
    ref = host(G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], path=2))
    got = host(G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], path=2, spin_limit=64))
    st = G.detffn_get_status()
    assert st in (OK, TIMEOUT)
    if st == OK:
        assert mismatches(got, ref) == 0
    again = host(G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], path=2))
    assert G.detffn_get_status() == OK
    assert mismatches(again, ref) == 0


def test_unknown_flag_is_rejected(G):
    x = torch.zeros(1, 256, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(768, 256, dtype=torch.bfloat16, device="cuda")
    wd = torch.zeros(256, 768, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(G.DetFFNError) as e:
        G.detffn_forward(x, w, w, wd, flags=16)
    assert e.value.status == 1
    with pytest.raises(G.DetFFNError) as e:
        G.detffn_forward(x, w, w, wd, spin_limit=-1)
    assert e.value.status == 1
    assert np.asarray(G.detffn_get_status()) == OK
