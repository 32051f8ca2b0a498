"""Unrounded binary64 FFN -- checks the oracle only (test infrastructure).

Computes the bias-free gated FFN (RL-Kernel PR #325, "Design" and "Operator
test matrix": gate/up/down projections with Hugging Face [out, in] weights)
and its exact-arithmetic backward in float64 from the same BF16 inputs, with
no intermediate rounding.  The rounded oracle must agree with it to a
relative L2 error of 1e-2 or better on every output.
"""
import numpy as np


def _w(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ffn_fp64(x, Wg, Wu, Wd, dOut=None):
    """Returns a dict with gate, up, h, out and, when dOut is given, dh, dG,
    dU, dX, dWg, dWu, dWd, all float64."""
    x, Wg, Wu, Wd = _w(x), _w(Wg), _w(Wu), _w(Wd)
    gate = x @ Wg.T
    up = x @ Wu.T
    sig = 1.0 / (1.0 + np.exp(-gate))
    a = gate * sig
    h = a * up
    out = h @ Wd.T
    res = dict(gate=gate, up=up, h=h, out=out)
    if dOut is not None:
        dO = _w(dOut)
        dh = dO @ Wd
        dU = dh * a
        dA = dh * up
        dG = dA * sig * (1.0 + gate * (1.0 - sig))
        res.update(dh=dh, dU=dU, dG=dG,
                   dX=dG @ Wg + dU @ Wu,
                   dWd=dO.T @ h, dWg=dG.T @ x, dWu=dU.T @ x)
    return res


def rel_l2(approx, exact):
    """||approx - exact||_2 / ||exact||_2 in float64."""
    approx = np.asarray(approx, np.float64)
    exact = np.asarray(exact, np.float64)
    den = np.linalg.norm(exact.ravel())
    return float(np.linalg.norm((approx - exact).ravel()) / (den if den else 1.0))
