"""Helpers for the GPU tests: move BF16 bit patterns between numpy and CUDA
tensors, and compare results element by element."""
import numpy as np
import torch


def dev(u16, device="cuda"):
    """numpy uint16 BF16 bits -> contiguous CUDA bfloat16 tensor."""
    t = torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16)
    return t.to(device).contiguous()


def host(t):
    """CUDA bfloat16/float16 tensor -> numpy uint16 bits (float32 -> float32)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def mismatches(a, b):
    """Number of differing elements (bit patterns)."""
    a = np.asarray(a)
    b = np.asarray(b)
    assert a.shape == b.shape, (a.shape, b.shape)
    return int(np.count_nonzero(a != b))


def ulp_key(u16):
    """Order-preserving integer map of BF16 bit patterns (+0 and -0 equal)."""
    v = np.asarray(u16).astype(np.int32)
    return np.where(v & 0x8000, -(v & 0x7FFF), v)


def ulp_dist(a, b):
    return np.abs(ulp_key(a) - ulp_key(b))


def empty_bf16(*shape):
    return torch.empty(shape, dtype=torch.bfloat16, device="cuda")
