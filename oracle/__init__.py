"""CPU oracle of the deterministic gated BF16 FFN -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library and never calls it.

Arrays: BF16 and FP16 tensors are ``numpy.uint16`` bit patterns, FP32 is
``numpy.float32``; 2-D arrays are row-major ``[rows, cols]`` unless a
function says otherwise.  Weights use the Hugging Face ``[out, in]`` layout
(RL-Kernel PR #325, "Operator test matrix").

Method source: RL-Kernel PR #325 "feat(ffn): add deterministic distributed
Triton FFN for ROCm", section "Design" (canonical FP32-leaf/BF16-node
midpoint reduction tree, BF16 stage boundaries, TP K shards as subtrees, CP
token gathering before weight gradients) and section "Communication overlap
assessment" (gate-then-up dHidden addition); PR #357 / PR #356 "Design"
(fixed balanced rank tree).

Parity status of each function is stated in its docstring; the pins live in
``tests/test_oracle_*.py``.
"""
import ctypes

import numpy as np

from ._lib import lib

SEQ, LANE = 0, 1
F32, F16, BF16 = 0, 1, 2
LEAF_WIDTH = 64

__all__ = [
    "SEQ", "LANE", "F32", "F16", "BF16", "LEAF_WIDTH",
    "rne_bf16", "bf16_to_f32", "rne_f16", "f16_to_f32",
    "leaf", "tree_from_leaves", "tree_node", "tree_gemm", "tree_leaves", "tree_replay",
    "silu_tables", "silu_mul", "silu_bwd", "add_bf16", "rank_tree",
    "ffn_forward", "ffn_backward", "ffn_forward_sharded", "dhidden_sharded",
    "wgrad_chunked", "wgrad_chunk_roots", "n_leaves",
]


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def n_leaves(K, lw=LEAF_WIDTH):
    """L(K) = ceil(K / lw) leaves; the last one may be partial."""
    return (K + lw - 1) // lw


# --------------------------------------------------------------------------
# Element rounding (round to nearest, ties to even)
# --------------------------------------------------------------------------

def rne_bf16(x):
    """binary32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    x = _f32(x)
    out = np.empty(x.shape, np.uint16)
    lib().or_cvt_f32_bf16(x.reshape(-1), out.reshape(-1), x.size)
    return out


def bf16_to_f32(b):
    """Exact widening of bfloat16 bit patterns to binary32."""
    return (_u16(b).astype(np.uint32) << 16).view(np.float32)


def rne_f16(x):
    """binary32 -> binary16 bit patterns (uint16), round to nearest even."""
    x = _f32(x)
    out = np.empty(x.shape, np.uint16)
    lib().or_cvt_f32_f16(x.reshape(-1), out.reshape(-1), x.size)
    return out


def f16_to_f32(h):
    """Exact widening of binary16 bit patterns to binary32."""
    h = _u16(h)
    out = np.empty(h.shape, np.float32)
    lib().or_cvt_f16_f32(h.reshape(-1), out.reshape(-1), h.size)
    return out


# --------------------------------------------------------------------------
# Leaves and the canonical tree (PR #325, Design: "canonical FP32-leaf/BF16-node
# midpoint reduction tree in deterministic GEMM")
# --------------------------------------------------------------------------

def leaf(a, b, lw=LEAF_WIDTH, order=LANE):
    """One FP32 leaf of a contraction: the partial dot product of two BF16
    vectors of length <= lw, in the stated in-leaf order (SEQ or LANE).
    Parity: pinned (closed forms on integer data, exact-rational brute force)."""
    a, b = _u16(a), _u16(b)
    assert a.shape == b.shape and a.ndim == 1 and a.size <= lw
    return float(lib().or_leaf(a.ctypes.data, 1, b.ctypes.data, 1, a.size, lw, order))


def tree_from_leaves(leaves):
    """Output element of the tree over FP32 leaves: rne_bf16(root); +0 if empty.
    Parity: pinned (integer closed form, explicit parenthesisations)."""
    lv = _f32(leaves).reshape(-1)
    return int(lib().or_tree_from_leaves(lv, lv.size))


def tree_node(leaves, lo, hi):
    """Raw value of the subtree node over leaves [lo, hi) (FP32 leaf if single)."""
    lv = _f32(leaves).reshape(-1)
    return float(lib().or_tree_node(lv, lo, hi))


def _gemm(A, B, want_out, want_leaves, lw, order, nthreads):
    A = _u16(A)
    B = _u16(B)
    assert A.ndim == 2 and B.ndim == 2 and A.shape[1] == B.shape[1]
    R, K = A.shape
    C = B.shape[0]
    out = np.zeros((R, C), np.uint16) if want_out else None
    L = n_leaves(K, lw)
    lv = np.zeros((R, C, L), np.float32) if want_leaves else None
    if R == 0 or C == 0:
        return out, lv
    lib().or_tree_gemm(A.ctypes.data, K, 1, B.ctypes.data, K, 1, R, C, K,
                       out.ctypes.data if want_out else None, C, 1,
                       lv.ctypes.data if want_leaves else None, lw, order, nthreads)
    return out, lv


def tree_gemm(A, B, lw=LEAF_WIDTH, order=LANE, nthreads=0):
    """out[r, c] = T_K(A[r, :], B[c, :]) in BF16, A [R, K] and B [C, K].
    Any strided view is accepted (it is copied to a contiguous array first;
    copying reorders no arithmetic).  Parity: pinned through leaf and tree."""
    return _gemm(A, B, True, False, lw, order, nthreads)[0]


def tree_leaves(A, B, lw=LEAF_WIDTH, order=LANE, nthreads=0):
    """The FP32 leaves [R, C, L] of tree_gemm(A, B)."""
    return _gemm(A, B, False, True, lw, order, nthreads)[1]


def tree_replay(leaves):
    """Applies the tree to leaves [..., L] (FP32), giving BF16 outputs [...]."""
    lv = _f32(leaves)
    L = lv.shape[-1]
    n = lv.size // L if L else int(np.prod(lv.shape[:-1]))
    out = np.zeros(lv.shape[:-1], np.uint16)
    if n and L:
        lib().or_tree_replay(lv.reshape(-1), n, L, out.reshape(-1))
    return out


# --------------------------------------------------------------------------
# Stage boundaries (PR #325, Design: "preserve BF16 stage boundaries in forward
# and backward")
# --------------------------------------------------------------------------

def silu_tables():
    """(silu_bf16[65536], dsilu_f32[65536]) indexed by the gate's bit pattern.
    Parity: pinned against a 60-digit evaluation of g*sigma(g)."""
    s = np.zeros(65536, np.uint16)
    d = np.zeros(65536, np.float32)
    lib().or_silu_tables(s, d)
    return s, d


def silu_mul(gate, up):
    """h = rne_bf16(silu_bf16(gate) * up) elementwise."""
    g, u = _u16(gate), _u16(up)
    assert g.shape == u.shape
    h = np.empty(g.shape, np.uint16)
    lib().or_silu_mul(g.reshape(-1), u.reshape(-1), g.size, h.reshape(-1))
    return h


def silu_bwd(dh, gate, up):
    """(dU, dA, dG): dU = rne_bf16(dh*a), dA = rne_bf16(dh*u),
    dG = rne_bf16(rne_f32(dA * dsilu(g))) with a = silu_bf16(g)."""
    d, g, u = _u16(dh), _u16(gate), _u16(up)
    assert d.shape == g.shape == u.shape
    dU = np.empty(d.shape, np.uint16)
    dA = np.empty(d.shape, np.uint16)
    dG = np.empty(d.shape, np.uint16)
    lib().or_silu_bwd(d.reshape(-1), g.reshape(-1), u.reshape(-1), d.size,
                      dU.ctypes.data, dA.ctypes.data, dG.ctypes.data)
    return dU, dA, dG


def add_bf16(a, b):
    """rne_bf16(a + b) elementwise; the first operand is the gate contribution."""
    a, b = _u16(a), _u16(b)
    out = np.empty(a.shape, np.uint16)
    lib().or_add_bf16(a.reshape(-1), b.reshape(-1), a.size, out.reshape(-1))
    return out


def rank_tree(bufs, dtype):
    """Balanced rank tree ((b0+b1)+(b2+b3))+... over n in {1,2,4,8} buffers,
    each node an FP32 add rounded to ``dtype`` (F32, F16 or BF16; F32 buffers
    are float32 arrays, the others uint16).  PR #357 / PR #356, Design."""
    n = len(bufs)
    want = np.float32 if dtype == F32 else np.uint16
    bufs = [np.ascontiguousarray(b, dtype=want).reshape(-1) for b in bufs]
    count = bufs[0].size
    assert all(b.size == count for b in bufs)
    out = np.empty(count, want)
    ptrs = (ctypes.c_void_p * n)(*[b.ctypes.data for b in bufs])
    rc = lib().or_rank_tree(ptrs, n, count, dtype, out.ctypes.data)
    if rc != 0:
        raise ValueError("rank_tree supports n in {1,2,4,8} and dtype F32/F16/BF16")
    return out


# --------------------------------------------------------------------------
# The FFN (PR #325, Design; weights [out, in])
# --------------------------------------------------------------------------

def ffn_forward(x, Wg, Wu, Wd, lw=LEAF_WIDTH, order=LANE, nthreads=0):
    """Forward of the bias-free gated FFN (PR #325, Design / Operator test matrix):
    gate = T(x, Wg), up = T(x, Wu) over K=H; h = rne_bf16(silu_bf16(gate)*up);
    out = T(h, Wd) over K=I.  Returns dict(gate, up, h, out).  ``nthreads``
    (0 = all host cores) only splits output rows over threads; the result
    does not depend on it."""
    gate = tree_gemm(x, Wg, lw, order, nthreads)
    up = tree_gemm(x, Wu, lw, order, nthreads)
    h = silu_mul(gate, up)
    out = tree_gemm(h, Wd, lw, order, nthreads)
    return dict(gate=gate, up=up, h=h, out=out)


def ffn_backward(x, Wg, Wu, Wd, gate, up, dOut, lw=LEAF_WIDTH, order=LANE):
    """Backward (PR #325, Design and "Communication overlap assessment"):
      dh = T(dOut, Wd^T) over K=H
      dU = rne(dh*a), dA = rne(dh*u), dG = rne(rne_f32(dA*dsilu(g)))
      cg = T(dG, Wg^T), cu = T(dU, Wu^T) over K=I; dX = rne(cg + cu) (gate first)
      dWd = T(dOut^T, h^T), dWg = T(dG^T, x^T), dWu = T(dU^T, x^T) over K=tokens.
    Returns a dict with every stage."""
    dh = tree_gemm(dOut, np.ascontiguousarray(np.asarray(Wd).T), lw, order)
    dU, dA, dG = silu_bwd(dh, gate, up)
    cg = tree_gemm(dG, np.ascontiguousarray(np.asarray(Wg).T), lw, order)
    cu = tree_gemm(dU, np.ascontiguousarray(np.asarray(Wu).T), lw, order)
    dX = add_bf16(cg, cu)
    h = silu_mul(gate, up)
    dWd = tree_gemm(np.ascontiguousarray(np.asarray(dOut).T), np.ascontiguousarray(h.T), lw, order)
    dWg = tree_gemm(np.ascontiguousarray(dG.T), np.ascontiguousarray(np.asarray(x).T), lw, order)
    dWu = tree_gemm(np.ascontiguousarray(dU.T), np.ascontiguousarray(np.asarray(x).T), lw, order)
    return dict(dh=dh, dU=dU, dA=dA, dG=dG, cg=cg, cu=cu, dX=dX, h=h,
                dWd=dWd, dWg=dWg, dWu=dWu)


def _shard_slices(I, k, lw):
    if I % k or (I // k) % lw or (I // k) // lw < 2:
        raise ValueError("shard preconditions: I % k == 0, (I/k) % lw == 0, (I/k)/lw >= 2")
    w = I // k
    return [slice(s * w, (s + 1) * w) for s in range(k)]


def ffn_forward_sharded(x, Wg, Wu, Wd, k, lw=LEAF_WIDTH, order=LANE):
    """TP emulation (PR #325, Design: "each contiguous TP K shard the same subtree
    used by TP=1" and the fixed balanced BF16 rank tree): shard s owns rows s of
    Wg/Wu and columns s of Wd (I/k each), computes its own gate/up/h and the
    down-projection subtree root p_s over its I/k slice; out = rank_tree(p_*)."""
    parts = []
    for sl in _shard_slices(np.asarray(Wg).shape[0], k, lw):
        g = tree_gemm(x, np.asarray(Wg)[sl], lw, order)
        u = tree_gemm(x, np.asarray(Wu)[sl], lw, order)
        h = silu_mul(g, u)
        parts.append(tree_gemm(h, np.asarray(Wd)[:, sl], lw, order))
    return rank_tree(parts, BF16).reshape(parts[0].shape), parts


def dhidden_sharded(dG, dU, Wg, Wu, k, lw=LEAF_WIDTH, order=LANE):
    """Sharded dHidden: per-shard subtree roots cg_s, cu_s over I/k, each rank
    tree separately, then dX = rne(cg + cu) in gate-then-up order."""
    cgs, cus = [], []
    for sl in _shard_slices(np.asarray(Wg).shape[0], k, lw):
        cgs.append(tree_gemm(np.asarray(dG)[:, sl], np.ascontiguousarray(np.asarray(Wg)[sl].T), lw, order))
        cus.append(tree_gemm(np.asarray(dU)[:, sl], np.ascontiguousarray(np.asarray(Wu)[sl].T), lw, order))
    shape = cgs[0].shape
    cg = rank_tree(cgs, BF16).reshape(shape)
    cu = rank_tree(cus, BF16).reshape(shape)
    return add_bf16(cg, cu)


def _chunk_stages(x_chunks, gate_chunks, up_chunks, dOut_chunks, Wd, lw, order):
    WdT = np.ascontiguousarray(np.asarray(Wd).T)
    xs, hs, dGs, dUs, dOs = [], [], [], [], []
    for x, g, u, dO in zip(x_chunks, gate_chunks, up_chunks, dOut_chunks):
        dh = tree_gemm(dO, WdT, lw, order)
        dU, _, dG = silu_bwd(dh, g, u)
        xs.append(np.asarray(x)); hs.append(silu_mul(g, u)); dGs.append(dG)
        dUs.append(dU); dOs.append(np.asarray(dO))
    return xs, hs, dGs, dUs, dOs


def wgrad_chunked(x_chunks, gate_chunks, up_chunks, dOut_chunks, Wd,
                  lw=LEAF_WIDTH, order=LANE):
    """CP emulation (PR #325, Design: "Gather complete CP token sequences before
    weight-gradient GEMMs so their K tree matches CP=1"): the row-wise stages run
    per chunk, the chunks are concatenated in logical token order, and the
    weight gradients are one tree over all tokens.  Returns (dWg, dWu, dWd)."""
    xs, hs, dGs, dUs, dOs = _chunk_stages(x_chunks, gate_chunks, up_chunks,
                                          dOut_chunks, Wd, lw, order)
    x = np.concatenate(xs, 0); h = np.concatenate(hs, 0)
    dG = np.concatenate(dGs, 0); dU = np.concatenate(dUs, 0); dO = np.concatenate(dOs, 0)
    dWd = tree_gemm(np.ascontiguousarray(dO.T), np.ascontiguousarray(h.T), lw, order)
    dWg = tree_gemm(np.ascontiguousarray(dG.T), np.ascontiguousarray(x.T), lw, order)
    dWu = tree_gemm(np.ascontiguousarray(dU.T), np.ascontiguousarray(x.T), lw, order)
    return dWg, dWu, dWd


def wgrad_chunk_roots(x_chunks, gate_chunks, up_chunks, dOut_chunks, Wd,
                      lw=LEAF_WIDTH, order=LANE):
    """Stricter CP reading: when every chunk is an aligned subtree of the token
    tree (equal power-of-two counts of whole leaves, each >= 2), each chunk's
    subtree root combined by the balanced rank tree equals the one-shot tree.
    Returns (dWg, dWu, dWd) computed that way."""
    xs, hs, dGs, dUs, dOs = _chunk_stages(x_chunks, gate_chunks, up_chunks,
                                          dOut_chunks, Wd, lw, order)
    roots = {"dWd": [], "dWg": [], "dWu": []}
    for x, h, dG, dU, dO in zip(xs, hs, dGs, dUs, dOs):
        if x.shape[0] % lw or x.shape[0] // lw < 2:
            raise ValueError("chunk roots need whole leaves, at least two per chunk")
        roots["dWd"].append(tree_gemm(np.ascontiguousarray(dO.T), np.ascontiguousarray(h.T), lw, order))
        roots["dWg"].append(tree_gemm(np.ascontiguousarray(dG.T), np.ascontiguousarray(x.T), lw, order))
        roots["dWu"].append(tree_gemm(np.ascontiguousarray(dU.T), np.ascontiguousarray(x.T), lw, order))
    res = {k: rank_tree(v, BF16).reshape(v[0].shape) for k, v in roots.items()}
    return res["dWg"], res["dWu"], res["dWd"]
