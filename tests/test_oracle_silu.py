"""Pins of the oracle's SiLU stage-boundary tables.

The FFN is the bias-free gated Qwen3 MLP, down(SiLU(gate) * up) (RL-Kernel
PR #325, "Design").  Reading (the page gives no formula): silu_bf16(g) =
rne_bf16(rne_f32(g*sigma(g))) and dsilu(g) = rne_f32(sigma(g)*(1+g*(1-sigma(g)))),
both functions of the 16-bit gate.  Pin: every one of the 2^16 entries
against a 40-digit evaluation rounded exactly, plus the limits at +-inf.
"""
from fractions import Fraction

import numpy as np
import pytest

from tests import exact

mpmath = pytest.importorskip("mpmath")


TINY = Fraction(1, 2 ** 160)   # far below half the least binary32 subnormal (2^-150)


def _mpf_to_fraction(v):
    """Exact value of an mpmath number; magnitudes below 2^-160 become a
    signed zero stand-in (they round to zero in binary32 whatever they are)."""
    sign, man, exp, bc = v._mpf_
    if man == 0 or exp + bc < -160:
        return Fraction(0)
    f = Fraction(int(man)) * (Fraction(2) ** int(exp))
    return -f if sign else f


def test_silu_tables_exhaustive(oracle_mod):
    silu, dsilu = oracle_mod.silu_tables()
    bits = np.arange(65536, dtype=np.uint32)
    g32 = (bits << 16).view(np.float32)
    mpmath.mp.dps = 40
    bad = []
    for i in range(65536):
        g = float(g32[i])
        if not np.isfinite(g):
            continue
        gm = mpmath.mpf(g)
        s = 1 / (1 + mpmath.exp(-gm))
        y = _mpf_to_fraction(gm * s)
        d = _mpf_to_fraction(s * (1 + gm * (1 - s)))
        y_b = exact.rn(exact.rn(y, exact.F32), exact.BF16)
        d_f = exact.rn(d, exact.F32)
        got_y = exact.bf16_value(int(silu[i]))
        got_d = Fraction(float(dsilu[i]))
        if got_y != y_b or got_d != d_f:
            bad.append(i)
    assert not bad, [hex(b) for b in bad[:10]]


def test_silu_limits(oracle_mod):
    silu, dsilu = oracle_mod.silu_tables()
    assert silu[0x7F80] == 0x7F80 and dsilu[0x7F80] == 1.0     # +inf
    assert silu[0xFF80] == 0x8000 and dsilu[0xFF80] == 0.0     # -inf -> -0
    assert silu[0x0000] == 0x0000 and dsilu[0x0000] == 0.5     # SiLU(0) = 0, SiLU'(0) = 1/2


def test_stage_boundaries(oracle_mod):
    """h, dU, dA, dG follow the definitions from the tables (hand-checked values)."""
    from gemm_deterministic_bf16_gb300.inputs import to_bf16_bits
    g = to_bf16_bits(np.float32([0.0, 40.0, 1.0]))
    u = to_bf16_bits(np.float32([3.0, 2.0, 1.0]))
    dh = to_bf16_bits(np.float32([5.0, 0.5, 2.0]))
    h = oracle_mod.silu_mul(g, u)
    # SiLU(0)*3 = 0; SiLU(40) = 40 in BF16 (40*sigma(40) differs from 40 by ~1e-16), 40*2 = 80.
    assert list(h[:2]) == [0x0000, int(to_bf16_bits(np.float32([80.0]))[0])]
    dU, dA, dG = oracle_mod.silu_bwd(dh, g, u)
    # dA = dh*u exactly here: 15, 1, 2; dU = dh*a: 0, 20, 2*silu(1).
    assert list(oracle_mod.bf16_to_f32(dA)) == [15.0, 1.0, 2.0]
    assert oracle_mod.bf16_to_f32(dU)[:2].tolist() == [0.0, 20.0]
    # dG = dA * SiLU'(g): at g=0 SiLU' = 1/2 -> 7.5; at g=40 SiLU' = 1 -> 1.
    assert oracle_mod.bf16_to_f32(dG)[:2].tolist() == [7.5, 1.0]
