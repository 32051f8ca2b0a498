"""Seeded synthetic inputs shared by the tests, the oracle checks and the benchmark.

This module draws random numbers and converts them to the storage types; it
holds none of the method's arithmetic.  Rounding to BF16/FP16 uses PyTorch's
own CPU conversion (round to nearest even).

Recipe (the pages use "seeded tensors" only -- RL-Kernel PR #325, "Note"):
  * ``numpy.random.default_rng`` on ``SeedSequence(seed).spawn(5)`` children, used
    in the fixed order x, Wg, Wu, Wd, dOut;
  * float64 standard normals times the scale (x, dOut: 1; weights: 0.02),
    cast to float32, then rounded to BF16;
  * weights in the Hugging Face ``[out, in]`` layout: Wg, Wu ``[I, H]``, Wd ``[H, I]``.
BF16/FP16 arrays are returned as ``numpy.uint16`` bit patterns.
"""
import numpy as np
import torch

W_STD = 0.02


def _to16(f32: np.ndarray, dtype) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32)).to(dtype)
    return t.view(torch.int16).numpy().view(np.uint16)


def to_bf16_bits(f32: np.ndarray) -> np.ndarray:
    return _to16(f32, torch.bfloat16)


def to_f16_bits(f32: np.ndarray) -> np.ndarray:
    return _to16(f32, torch.float16)


def ffn_inputs(M: int, H: int, I: int, seed: int = 0, w_std: float = W_STD,
               with_dout: bool = True) -> dict:
    """x [M,H], Wg [I,H], Wu [I,H], Wd [H,I], dOut [M,H] as BF16 bit patterns."""
    rngs = [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(5)]
    shapes = {"x": (M, H), "Wg": (I, H), "Wu": (I, H), "Wd": (H, I), "dOut": (M, H)}
    scales = {"x": 1.0, "Wg": w_std, "Wu": w_std, "Wd": w_std, "dOut": 1.0}
    out = {}
    for rng, name in zip(rngs, ["x", "Wg", "Wu", "Wd", "dOut"]):
        if name == "dOut" and not with_dout:
            continue
        v = rng.standard_normal(shapes[name]) * scales[name]
        out[name] = to_bf16_bits(v.astype(np.float32))
    return out


def rank_tree_inputs(n: int, count: int, dtype: str, seed: int = 0) -> list:
    """n buffers of ``count`` N(0,1) values in 'f32' (float32), 'f16' or 'bf16'
    (uint16 bit patterns)."""
    rngs = [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]
    bufs = []
    for rng in rngs:
        v = rng.standard_normal(count).astype(np.float32)
        if dtype == "f32":
            bufs.append(v)
        elif dtype == "f16":
            bufs.append(to_f16_bits(v))
        elif dtype == "bf16":
            bufs.append(to_bf16_bits(v))
        else:
            raise ValueError(dtype)
    return bufs


def sample_indices(n: int, count: int, seed: int) -> np.ndarray:
    """``count`` distinct sorted indices in [0, n), seeded."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, n, count]))
    return np.sort(rng.choice(n, size=min(count, n), replace=False))
