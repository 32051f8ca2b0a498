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


def test_fp32_to_bf16_rounding_exhaustive(oracle_mod):
    """Every FP32 bit pattern (2^32 of them, in chunks of 2^28): the device
    conversion the kernels use for leaves, nodes and stage boundaries equals
    the oracle's round-to-nearest-even rule (BF16 nodes rounded to nearest
    even: RL-Kernel PR #325, "Design"); NaNs compare as one class."""
    import numpy as np
    import torch

    import gemm_deterministic_bf16_gb300 as G
    from gemm_deterministic_bf16_gb300 import build
    build.build()
    chunk = 1 << 28
    bad = 0
    for lo in range(-(1 << 31), 1 << 31, chunk):
        bits = torch.arange(lo, lo + chunk, dtype=torch.int32, device="cuda")
        got = G.detffn_cvt_f32_bf16(bits.view(torch.float32)).view(torch.int16).cpu().numpy().view(np.uint16)
        del bits
        x = np.arange(lo, lo + chunk, dtype=np.int64).astype(np.int32).view(np.float32)
        ref = oracle_mod.rne_bf16(x)
        nan_g = (got & 0x7FFF) > 0x7F80
        nan_r = (ref & 0x7FFF) > 0x7F80
        bad += int(np.count_nonzero((got != ref) & ~(nan_g & nan_r)))
        del got, ref, x
    assert bad == 0
