"""Exhaustive GPU checks of the element operations the kernels rely on.

The tree node is rne_bf16(fp32(left) + fp32(right)) (RL-Kernel PR #325,
"Design": BF16 nodes, round to nearest even).  Since binary32 carries more
than 2*8 + 2 significand bits, that equals the correctly rounded BF16 sum, so
the device's packed add.rn.bf16x2 must agree with it on every one of the
2^32 pairs of BF16 values; the tensor-core epilogue relies on that."""
import pytest

pytestmark = pytest.mark.gpu


def test_packed_node_add_exhaustive():
    import gemm_deterministic_bf16_gb300 as G
    from gemm_deterministic_bf16_gb300 import build
    build.build()
    assert G.detffn_selfcheck_node_add() == 0
