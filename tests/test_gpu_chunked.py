"""Weight gradients from token chunks on the tensor family (RL-Kernel PR
#325, "Design": complete CP token sequences gathered before the weight-
gradient GEMMs).  Whatever the chunking, the three weight gradients must be
the same bits as the one-shot backward's: chunks of whole leaves (64 tokens)
are read in place as one K axis (a tensor map per chunk), other chunkings,
more than eight chunks and unaligned chunks are gathered first, and gate/up
chunks are read in place where aligned.  Every case compares element by
element, with zero mismatches allowed."""
import pytest
import torch

from gemm_deterministic_bf16_gb300.inputs import ffn_inputs
from tests.gpu_util import dev, empty_bf16, host, mismatches

pytestmark = pytest.mark.gpu
TENSOR = 2


@pytest.fixture(scope="module")
def G():
    import gemm_deterministic_bf16_gb300 as G
    from gemm_deterministic_bf16_gb300 import build
    build.build()
    return G


_CASES = {}


def _case(G, M):
    """Inputs, forward saves and the one-shot backward's weight gradients at
    M tokens (H = 256, I = 512): 32 tokens are one leaf, 384 tokens a tree of
    6 leaves (bottom groups of three), 512 tokens one of 8 leaves (pairs)."""
    if M not in _CASES:
        H, I = 256, 512
        d = ffn_inputs(M, H, I, seed=23 + M)
        t = {n: dev(v) for n, v in d.items()}
        g, u = empty_bf16(M, I), empty_bf16(M, I)
        G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], gate_save=g, up_save=u, path=TENSOR)
        _, dWg, dWu, dWd = G.detffn_backward(t["x"], t["Wg"], t["Wu"], t["Wd"], g, u, t["dOut"], path=TENSOR)
        torch.cuda.synchronize()
        _CASES[M] = (t, g, u, [host(dWg), host(dWu), host(dWd)])
    return _CASES[M]


def _misaligned(v):
    """The same values at a 2-byte (not 16-byte) aligned address."""
    buf = torch.empty(v.numel() + 1, dtype=v.dtype, device=v.device)
    out = buf[1:].view(v.shape)
    out.copy_(v)
    return out


# M = 32: the few-token kernels for dh, whole and in chunks of 16, 8 and 24.
@pytest.mark.parametrize("M,sizes", [(32, [32]), (32, [16, 16]), (32, [8, 24]),
                                     (384, [128, 256]), (384, [64] * 6), (384, [64, 320]), (384, [192, 192]),
                                     (384, [0, 384, 0]), (384, [100, 284]), (384, [32] * 12), (384, [1, 63, 320]),
                                     (512, [256, 256]), (512, [64] * 8), (512, [448, 64]), (512, [200, 312])])
@pytest.mark.parametrize("aligned", [True, False])
def test_chunked_wgrad_tensor_same_bits(G, M, sizes, aligned):
    t, g, u, ref = _case(G, M)
    edges = [0]
    for s in sizes:
        edges.append(edges[-1] + s)
    sl = [slice(a, b) for a, b in zip(edges[:-1], edges[1:])]
    prep = (lambda v: v.contiguous()) if aligned else (lambda v: _misaligned(v.contiguous()))  # noqa: E731
    got = G.detffn_wgrad_chunked([prep(t["x"][s]) for s in sl], [prep(g[s]) for s in sl],
                                 [prep(u[s]) for s in sl], [prep(t["dOut"][s]) for s in sl], t["Wd"],
                                 path=TENSOR)
    torch.cuda.synchronize()
    for n, a, b in zip(("dWg", "dWu", "dWd"), got, ref):
        assert mismatches(host(a), b) == 0, (M, sizes, aligned, n)
