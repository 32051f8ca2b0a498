"""The two-stream dHidden option (RL-Kernel PR #325, "Communication overlap
assessment"): with k > 1 shards, the gate contribution's rank tree runs on a
second stream while the up contribution is computed.  It is accepted only if
every result is the same bits as the one-stream call, so each case compares
dX (and the weight gradients, which follow it on the same stream) element by
element, with zero mismatches allowed."""
import numpy as np
import pytest
import torch

from gemm_deterministic_bf16_gb300.inputs import ffn_inputs
from tests.gpu_util import dev, empty_bf16, host, mismatches

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    import gemm_deterministic_bf16_gb300 as G
    from gemm_deterministic_bf16_gb300 import build
    build.build()
    return G


def _bwd(G, t, g, u, k, path, flags, stream=None):
    res = G.detffn_backward(t["x"], t["Wg"], t["Wu"], t["Wd"], g, u, t["dOut"], shards=k, path=path,
                            flags=flags, stream=stream)
    torch.cuda.synchronize()
    return [host(r) for r in res]


@pytest.mark.parametrize("M,H,I,path,ks", [(32, 4096, 12288, 2, (2, 4, 8)), (4096, 4096, 12288, 0, (2,)),
                                           (8, 256, 1024, 1, (2, 4)), (200, 384, 1536, 2, (2, 4))])
def test_overlap_same_bits_as_one_stream(G, M, H, I, path, ks):
    d = ffn_inputs(M, H, I, seed=11)
    t = {n: dev(v) for n, v in d.items()}
    g, u = empty_bf16(M, I), empty_bf16(M, I)
    G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], gate_save=g, up_save=u, path=path)
    for k in ks:
        one = _bwd(G, t, g, u, k, path, 0)
        # A stream of the caller's own, so that the fork and join are taken
        # from a stream other than the default one.
        s = torch.cuda.Stream()
        two = _bwd(G, t, g, u, k, path, G.FLAG_OVERLAP_DHIDDEN, stream=s)
        for n, a, b in zip(("dX", "dWg", "dWu", "dWd"), two, one):
            assert mismatches(a, b) == 0, (k, n)


def test_overlap_repeated_calls_and_no_shards(G):
    """Back-to-back overlapped calls on one stream reuse the same workspace
    (each call's side work must be joined before the next begins), and the
    flag changes nothing without shards."""
    M, H, I = 32, 1024, 4096
    d = ffn_inputs(M, H, I, seed=12)
    t = {n: dev(v) for n, v in d.items()}
    g, u = empty_bf16(M, I), empty_bf16(M, I)
    G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], gate_save=g, up_save=u)
    ref = _bwd(G, t, g, u, 4, 0, 0)
    ws = G.workspace(G.OP_BACKWARD, M, H, I, 4, 0, t["x"].device)
    outs = []
    for _ in range(5):
        dX = empty_bf16(M, H)
        G.detffn_backward(t["x"], t["Wg"], t["Wu"], t["Wd"], g, u, t["dOut"], dX=dX, ws=ws, shards=4,
                          flags=G.FLAG_OVERLAP_DHIDDEN)
        outs.append(dX)
    torch.cuda.synchronize()
    for dX in outs:
        assert mismatches(host(dX), ref[0]) == 0
    a = _bwd(G, t, g, u, 1, 0, 0)
    b = _bwd(G, t, g, u, 1, 0, G.FLAG_OVERLAP_DHIDDEN)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
