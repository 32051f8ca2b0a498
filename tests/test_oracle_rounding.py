"""Pins of the oracle's element rounding (RNE to BF16 and FP16, the BF16 node add).

The node rule -- an FP32 add then rounding to BF16 with round-to-nearest-even --
is the "BF16-node" of the canonical tree (RL-Kernel PR #325, "Design"); the
FP16 node is the rank tree's rounding for FP16 buffers (PR #357, "Design").
Pins: hand-worked ties, and library conversions (PyTorch / NumPy) that are
themselves round-to-nearest-even, on every tie and near-tie pattern.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from tests import exact


def _torch_bf16_bits(f32):
    return torch.from_numpy(np.ascontiguousarray(f32, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _is_nan_bf16(b):
    b = b.astype(np.uint32)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)


def test_hand_ties(oracle_mod):
    lib = oracle_mod.lib()
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties to the even one, 1.0.
    assert lib.or_rne_bf16(np.float32(1 + 2 ** -8)) == 0x3F80
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: ties to 1 + 2^-6.
    assert lib.or_rne_bf16(np.float32(1 + 3 * 2 ** -8)) == 0x3F82
    # Just above the first tie rounds up.
    assert lib.or_rne_bf16(np.float32(1 + 2 ** -8 + 2 ** -20)) == 0x3F81
    # Largest finite BF16 plus half an ulp overflows to +inf.
    assert lib.or_rne_bf16(np.float32(np.uint32(0x7F7F8000).view(np.float32))) == 0x7F80
    assert lib.or_rne_bf16(np.float32(-0.0)) == 0x8000


def _tie_patterns():
    hi = np.arange(65536, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint32)
    return (hi[:, None] | lows[None, :]).reshape(-1)


def test_rne_bf16_matches_torch_on_every_tie(oracle_mod):
    rng = np.random.default_rng(1)
    pats = np.concatenate([_tie_patterns(),
                           rng.integers(0, 2 ** 32, 1 << 21, dtype=np.uint64).astype(np.uint32)])
    f = pats.view(np.float32)
    ours = oracle_mod.rne_bf16(f)
    ref = _torch_bf16_bits(f)
    nan = _is_nan_bf16(ref)
    assert np.array_equal(_is_nan_bf16(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_bf16_widening_is_exact(oracle_mod):
    b = np.arange(65536, dtype=np.uint16)
    ours = oracle_mod.bf16_to_f32(b)
    ref = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


def test_rne_f16_matches_numpy(oracle_mod):
    rng = np.random.default_rng(2)
    # Every FP16 value, the FP32 midpoints between neighbours and one FP32 ulp
    # either side of each midpoint, plus random patterns.
    h = np.arange(0, 0x7C00, dtype=np.uint16)
    v = h.view(np.float16).astype(np.float64)
    mids = (v[:-1] + v[1:]) / 2
    mids32 = mids.astype(np.float32)
    near = np.concatenate([mids32, np.nextafter(mids32, np.float32(np.inf)),
                           np.nextafter(mids32, np.float32(0)), v.astype(np.float32)])
    near = np.concatenate([near, -near, np.float32([65504, 65519.99, 65520, 1e6, np.inf, -np.inf, 0.0])])
    rnd = rng.integers(0, 2 ** 32, 1 << 20, dtype=np.uint64).astype(np.uint32).view(np.float32)
    f = np.concatenate([near, rnd[np.isfinite(rnd)]])
    ours = oracle_mod.rne_f16(f)
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)
    back = oracle_mod.f16_to_f32(np.arange(0, 0x7C00, dtype=np.uint16))
    assert np.array_equal(back, np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float32))


def test_bf16_node_add_is_correctly_rounded(oracle_mod):
    """rne_bf16(fp32(a) + fp32(b)) equals the correctly rounded BF16 sum
    (double rounding through binary32 is innocuous for BF16: 24 >= 2*8 + 2)."""
    rng = np.random.default_rng(3)
    n = 1 << 20
    a = rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16)
    b = rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16)
    # Also operands of close magnitude, where cancellation and ties are common.
    b[: n // 2] = (a[: n // 2].astype(np.int32) + rng.integers(-300, 300, n // 2)).clip(0, 65535).astype(np.uint16)
    fa, fb = oracle_mod.bf16_to_f32(a), oracle_mod.bf16_to_f32(b)
    ok = np.isfinite(fa) & np.isfinite(fb)
    ours = oracle_mod.add_bf16(a[ok], b[ok])
    s = fa[ok].astype(np.float64) + fb[ok].astype(np.float64)
    ref = torch.from_numpy(s).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = _is_nan_bf16(ref)
    assert not nan.any()
    assert np.array_equal(ours, ref)


def test_exact_helper_is_rne(oracle_mod):
    """The exact-rational rounding used by the brute-force pins agrees with
    NumPy's float64 -> float32 conversion (itself round-to-nearest-even)."""
    rng = np.random.default_rng(4)
    d = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-40, 38, 2000),
                        np.float64([1 + 2 ** -24, 1 + 3 * 2 ** -24, 2 ** -149, 2 ** -150, 3 * 2 ** -150])])
    for x in d:
        assert float(exact.rn(Fraction(float(x)), exact.F32)) == float(np.float32(x))
