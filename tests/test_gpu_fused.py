"""The decode forward in one launch (tensor family, at most 32 tokens).

One kernel takes the stacked gate/up tiles (SiLU * up in their epilogue) and
then the down projection's aligned blocks, each block waiting only for the
gate/up tiles of its K range (RL-Kernel PR #325, "Communication overlap
assessment": the gate/up -> down dependency).  It computes the same leaves and
trees as the two-launch form, so every output -- out, and gate and up where
kept -- must be the same bits, call after call.  Shapes outside its cover
(here 32 pieces per down tree at I = 3072) take the two-launch form.
"""
import pytest
import torch

from gemm_deterministic_bf16_gb300.inputs import ffn_inputs
from tests.gpu_util import dev, empty_bf16, host, mismatches

pytestmark = pytest.mark.gpu
TENSOR = 2

_INPUTS = {}


@pytest.fixture(scope="module")
def G():
    import gemm_deterministic_bf16_gb300 as G
    from gemm_deterministic_bf16_gb300 import build
    build.build()
    return G


def _inputs(H, I):
    """32 tokens of seeded inputs for (H, I); a test takes the first M."""
    if (H, I) not in _INPUTS:
        d = ffn_inputs(32, H, I, seed=60 + H // 256 + I // 768, with_dout=False)
        _INPUTS[(H, I)] = {n: dev(v) for n, v in d.items()}
    return _INPUTS[(H, I)]


def _forward(G, t, M, saves, flags):
    H, I = t["x"].shape[1], t["Wg"].shape[0]
    out = empty_bf16(M, H)
    g = empty_bf16(M, I) if saves else None
    u = empty_bf16(M, I) if saves else None
    G.detffn_forward(t["x"][:M], t["Wg"], t["Wu"], t["Wd"], out=out, gate_save=g, up_save=u, path=TENSOR,
                     flags=flags)
    torch.cuda.synchronize()
    return [host(v) for v in (out, g, u) if v is not None]


@pytest.mark.parametrize("M,H,I,one_launch", [(32, 4096, 12288, True), (8, 4096, 12288, True),
                                              (1, 4096, 12288, True), (8, 1024, 1536, True),
                                              (17, 1024, 1536, True), (8, 1024, 3072, False)])
@pytest.mark.parametrize("saves", [False, True])
def test_one_launch_forward_same_bits_as_two(G, M, H, I, one_launch, saves):
    t = _inputs(H, I)
    G.detffn_profiling(True)
    fused = _forward(G, t, M, saves, 0)
    ops = G.detffn_profile_read()
    G.detffn_profiling(False)
    # The one-launch form ran exactly where it covers the shape.
    assert ("tcs_forward" in ops) == one_launch, sorted(ops)
    if one_launch:
        assert ops["tcs_forward"]["launches"] == 1 and len(ops) == 1, ops
    split = _forward(G, t, M, saves, G.FLAG_SPLIT_FORWARD)
    again = _forward(G, t, M, saves, 0)
    assert G.detffn_get_status() == 0
    for name, a, b, c in zip(("out", "gate", "up"), fused, split, again):
        assert mismatches(a, b) == 0, (M, H, I, saves, name)
        assert mismatches(a, c) == 0, (M, H, I, saves, name, "repeat")


def test_one_launch_forward_after_other_calls(G):
    """Calls of other shapes in between (they use the same tree tickets and
    range counters of the handle) leave the next one-launch forward's bits
    unchanged."""
    t = _inputs(1024, 1536)
    ref = _forward(G, t, 8, True, 0)
    big = _inputs(4096, 12288)
    _forward(G, big, 32, False, 0)
    _forward(G, t, 17, False, G.FLAG_SPLIT_FORWARD)
    _forward(G, big, 1, True, 0)
    got = _forward(G, t, 8, True, 0)
    assert G.detffn_get_status() == 0
    for a, b in zip(ref, got):
        assert mismatches(a, b) == 0
