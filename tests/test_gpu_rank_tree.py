"""GPU parity of detffn_rank_tree_reduce against the oracle: bit-exact for
n in {1,2,4,8} buffers of 4 KiB, 64 KiB, 1 MiB and 16 MiB in FP32, FP16 and
BF16, with misaligned offset views, odd tails and in-place output.
Arithmetic: ((b0+b1)+(b2+b3))+... with every node rounded to the dtype
(RL-Kernel PR #357, "Design"; PR #356, "Design").  The max-abs difference from
an unordered float64 sum is reported, as the pages' collective report does,
but the oracle is the arithmetic authority."""
import numpy as np
import pytest
import torch

from gemm_deterministic_bf16_gb300.inputs import rank_tree_inputs
from tests.gpu_util import host, mismatches

pytestmark = pytest.mark.gpu

DT = {"f32": (torch.float32, 4, 0), "f16": (torch.float16, 2, 1), "bf16": (torch.bfloat16, 2, 2)}


@pytest.fixture(scope="module")
def G():
    import gemm_deterministic_bf16_gb300 as G
    from gemm_deterministic_bf16_gb300 import build
    build.build()
    return G


def _to_dev(buf, tdt):
    if tdt == torch.float32:
        return torch.from_numpy(buf).cuda()
    return torch.from_numpy(buf.view(np.int16)).view(tdt).cuda()


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("n", [1, 2, 4, 8])
@pytest.mark.parametrize("size", [4096, 65536, 1 << 20, 16 << 20])
def test_sweep(G, oracle_mod, dt, n, size):
    tdt, esz, odt = DT[dt]
    count = size // esz
    bufs = rank_tree_inputs(n, count, dt, seed=size + n)
    ins = [_to_dev(b, tdt) for b in bufs]
    out = G.detffn_rank_tree_reduce(ins)
    ref = oracle_mod.rank_tree(bufs, odt)
    assert mismatches(host(out), ref) == 0


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("offset", [1, 2, 3])
def test_offset_views_and_tails(G, oracle_mod, dt, offset):
    tdt, esz, odt = DT[dt]
    n, count = 4, (1 << 16) - 1 - offset       # odd tail, start off the 16-byte grid
    bufs = rank_tree_inputs(n, count + 8, dt, seed=offset)
    ins = [_to_dev(b, tdt)[offset:offset + count] for b in bufs]
    out_base = torch.zeros(count + 8, dtype=tdt, device="cuda")
    out = out_base[offset:offset + count]
    G.detffn_rank_tree_reduce(ins, out=out)
    ref = oracle_mod.rank_tree([b[offset:offset + count] for b in bufs], odt)
    assert mismatches(host(out), ref) == 0
    assert not host(out_base[:offset]).any() and not host(out_base[offset + count:]).any()


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("offsets,count", [((1, 1, 1, 1, 0), 4093), ((2, 3, 2), 70001), ((3, 3, 3), 3),
                                           ((1, 1, 1, 1, 1), 9), ((0, 1, 2, 3, 3), 1027)])
def test_mixed_offsets_and_short_heads(G, oracle_mod, dt, offsets, count):
    """Buffers at different offsets from the 16-byte grid (no common boundary:
    element by element or 4-byte steps), and counts shorter than the head
    that a common offset would take one element at a time."""
    tdt, esz, odt = DT[dt]
    n = len(offsets) - 1  # input offsets, then the output's
    bufs = rank_tree_inputs(n, count + 8, dt, seed=count)
    ins = [_to_dev(b, tdt)[o:o + count] for b, o in zip(bufs, offsets)]
    oo = offsets[-1]
    out_base = torch.zeros(count + 8, dtype=tdt, device="cuda")
    out = out_base[oo:oo + count]
    G.detffn_rank_tree_reduce(ins, out=out)
    ref = oracle_mod.rank_tree([b[o:o + count] for b, o in zip(bufs, offsets)], odt)
    assert mismatches(host(out), ref) == 0
    assert not host(out_base[:oo]).any() and not host(out_base[oo + count:]).any()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_in_place(G, oracle_mod, dt):
    tdt, esz, odt = DT[dt]
    bufs = rank_tree_inputs(8, 100003, dt, seed=9)
    ins = [_to_dev(b, tdt) for b in bufs]
    G.detffn_rank_tree_reduce(ins, out=ins[3])
    assert mismatches(host(ins[3]), oracle_mod.rank_tree(bufs, odt)) == 0


def test_empty_and_repeat(G):
    a = torch.randn(0, device="cuda")
    G.detffn_rank_tree_reduce([a, a])
    xs = [torch.randn(1 << 20, device="cuda").bfloat16() for _ in range(8)]
    r1 = host(G.detffn_rank_tree_reduce(xs))
    r2 = host(G.detffn_rank_tree_reduce(xs))
    assert mismatches(r1, r2) == 0
    exact = torch.stack([x.double() for x in xs]).sum(0)
    maxabs = (G.detffn_rank_tree_reduce(xs).double() - exact).abs().max().item()
    assert maxabs < 0.25   # BF16 rounding at three levels of magnitude ~ sqrt(8)
