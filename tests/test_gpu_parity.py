"""Parity of the tensor-core family (the default for more than one token)
against the oracle, at the benchmark's own sizes.

A tensor-core leaf is the hardware's sum of its 64 products, not the oracle's
stated in-leaf order, so a leaf may differ from the oracle's by FP32 rounding;
the canonical tree over the leaves (RL-Kernel PR #325, "Design") must still
be applied exactly.  Three kinds of evidence:

* Leaf dump: the tensor kernels write their FP32 leaves; the oracle's tree
  over those leaves must give the GPU's output bit for bit (this pins the
  tree, the piece folds and the stores on the hardware's own leaves), and
  every leaf -- the GPU's and the oracle's -- must lie within the FP32
  summation bound 64 * 2^-24 * sum|a_k b_k| of the exact dot product.
* Stage-wise comparison with the oracle (each contraction fed the GPU's own
  BF16 stage inputs): element-wise stages are bit-exact; contractions meet
  relative L2 <= 1e-3, and the elements more than one BF16 ulp away are
  counted.  Where a count is not zero, the leaf dump of the same contraction
  shows that the tree over the GPU's leaves reproduces them exactly, i.e.
  they come from leaf rounding amplified by cancellation (their condition
  number sum|a b| / |result| is reported next to the count).
* Invariance (PR #325, "Correctness results"): shards k = 2, 4, 8 and token
  chunks c = 2, 4 give 0 mismatches against the unsharded, one-shot call.

Setting DETFFN_PARITY_LOG to a file path appends one JSON line of statistics
per checked stage (used for the written parity summary).
"""
import json
import os

import numpy as np
import pytest
import torch

from gemm_deterministic_bf16_gb300.inputs import ffn_inputs, sample_indices, to_bf16_bits
from tests.gpu_util import dev, empty_bf16, host, mismatches, ulp_dist

pytestmark = pytest.mark.gpu
TENSOR = 2
LEAF_BOUND = 64 * 2.0 ** -24


@pytest.fixture(scope="module")
def G():
    import gemm_deterministic_bf16_gb300 as G
    from gemm_deterministic_bf16_gb300 import build
    build.build()
    return G


def _f64(u16):
    return (np.asarray(u16, np.uint32) << 16).view(np.float32).astype(np.float64)


def _t(a):
    return np.ascontiguousarray(np.asarray(a).T)


def record(name, got, ref, cond=None):
    """Compares BF16 arrays; logs rel-L2, max ulp and the >1-ulp count."""
    g, r = _f64(got), _f64(ref)
    d = ulp_dist(got, ref)
    rl2 = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300))
    rec = {"stage": name, "elements": int(d.size), "rel_l2": rl2, "max_ulp": int(d.max()) if d.size else 0,
           "within_1ulp": int(np.count_nonzero(d <= 1)), "over_1ulp": int(np.count_nonzero(d > 1)),
           "mismatches": int(np.count_nonzero(np.asarray(got) != np.asarray(ref)))}
    if cond is not None and rec["over_1ulp"]:
        rec["cond_median_over_1ulp"] = float(np.median(cond[d > 1]))
        rec["cond_median_all"] = float(np.median(cond))
    print(json.dumps(rec))
    path = os.environ.get("DETFFN_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")
    return rec, d


def _exact_leaves(A, B):
    """Exact (float64) leaf sums and sums of |a b| per leaf, [R, C, L]."""
    a, b = _f64(A), _f64(B)
    R, K = a.shape
    C = b.shape[0]
    L = (K + 63) // 64
    ex = np.empty((R, C, L))
    ab = np.empty((R, C, L))
    for j in range(L):
        sa, sb = a[:, 64 * j:64 * j + 64], b[:, 64 * j:64 * j + 64]
        ex[:, :, j] = sa @ sb.T
        ab[:, :, j] = np.abs(sa) @ np.abs(sb).T
    return ex, ab


def _rand(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return to_bf16_bits((scale * rng.standard_normal(shape)).astype(np.float32))


# Few-token shapes cover the three ways a tree's root is formed: its last
# CTA folds the pieces of a tree split over several CTAs (2, 4, 8 per tree at
# the first three; 4 at (16, 8192, 1536)), a top kernel does (32 pieces at
# (1, 1024, 4096)), or each CTA takes whole trees (two each at
# (4, 40960, 128)).
@pytest.mark.parametrize("R,C,K", [(32, 12288, 4096), (32, 4096, 12288), (8, 3072, 768), (1, 1024, 4096),
                                   (4, 40960, 128), (16, 8192, 1536),
                                   (256, 256, 4096), (256, 128, 12288), (200, 296, 40), (130, 72, 64),
                                   (96, 384, 128)])
def test_leaf_dump_replay_and_bound(G, oracle_mod, R, C, K):
    A, B = _rand((R, K), R + K), _rand((C, K), C + K + 1, 0.02)
    out, lv = G.detffn_tree_gemm_leaves(dev(A), dev(B))
    out, lv = host(out), lv.cpu().numpy()
    # The dump instance computes what the plain contraction computes.
    assert mismatches(host(G.detffn_tree_gemm(dev(A), dev(B), path=TENSOR)), out) == 0
    # The canonical tree over the GPU's own leaves is the GPU's output.
    assert mismatches(oracle_mod.tree_replay(lv), out) == 0
    # Every leaf is within the FP32 summation bound of the exact dot product.
    ex, ab = _exact_leaves(A, B)
    tiny = 2.0 ** -140
    ratio_gpu = np.abs(lv.astype(np.float64) - ex) / (2.0 ** -24 * ab + tiny)
    olv = oracle_mod.tree_leaves(A, B)
    ratio_or = np.abs(olv.astype(np.float64) - ex) / (2.0 ** -24 * ab + tiny)
    print("leaf error / (2^-24 sum|ab|): gpu max %.3f, oracle max %.3f" % (ratio_gpu.max(), ratio_or.max()))
    assert np.all(np.abs(lv - ex) <= LEAF_BOUND * ab + tiny)
    assert np.all(np.abs(olv - ex) <= LEAF_BOUND * ab + tiny)
    ref = oracle_mod.tree_gemm(A, B)
    cond = ab.sum(-1) / np.maximum(np.abs(_f64(ref)), 1e-30)
    rec, d = record("tree_gemm R=%d C=%d K=%d" % (R, C, K), out, ref, cond)
    assert rec["rel_l2"] <= 1e-3
    # Where the leaves agree with the oracle's, so do the outputs.
    same = np.all(lv == olv, axis=-1)
    assert mismatches(out[same], ref[same]) == 0


def _fwd_bwd_saves(G, t, path=TENSOR, k=1):
    M, H = t["x"].shape
    I = t["Wg"].shape[0]
    g, u = empty_bf16(M, I), empty_bf16(M, I)
    if k == 1:
        out = G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], gate_save=g, up_save=u, path=path)
    else:
        out = G.detffn_forward_sharded(t["x"], t["Wg"], t["Wu"], t["Wd"], k, gate_save=g, up_save=u, path=path)
    dh, dU, dG = empty_bf16(M, I), empty_bf16(M, I), empty_bf16(M, I)
    dX, dWg, dWu, dWd = G.detffn_backward(t["x"], t["Wg"], t["Wu"], t["Wd"], g, u, t["dOut"], dh_save=dh,
                                          dU_save=dU, dG_save=dG, shards=k, path=path)
    torch.cuda.synchronize()
    return {n: host(v) for n, v in dict(out=out, gate=g, up=u, dh=dh, dU=dU, dG=dG, dX=dX, dWg=dWg,
                                        dWu=dWu, dWd=dWd).items()}


def _cond(A, B):
    """sum_k |a_k b_k| for every (row of A, row of B), float64."""
    return np.abs(_f64(A)) @ np.abs(_f64(B)).T


def test_m32_tensor_forward_backward_stagewise(G, oracle_mod):
    """M=32, H=4096, I=12288 (the training shape of the benchmark) on the
    tensor family, every stage against the oracle fed the GPU's own stage
    inputs; shards k = 2, 4, 8 give the same bits."""
    M, H, I = 32, 4096, 12288
    d = ffn_inputs(M, H, I, seed=2)
    t = {n: dev(v) for n, v in d.items()}
    got = _fwd_bwd_saves(G, t)
    x, Wg, Wu, Wd, dO = d["x"], d["Wg"], d["Wu"], d["Wd"], d["dOut"]
    for name, ref, cond in [("M32 gate", oracle_mod.tree_gemm(x, Wg), _cond(x, Wg)),
                            ("M32 up", oracle_mod.tree_gemm(x, Wu), _cond(x, Wu))]:
        rec, _ = record(name, got[name.split()[1]], ref, cond)
        assert rec["rel_l2"] <= 1e-3
    h = oracle_mod.silu_mul(got["gate"], got["up"])
    rec, _ = record("M32 out", got["out"], oracle_mod.tree_gemm(h, Wd), _cond(h, Wd))
    assert rec["rel_l2"] <= 1e-3
    WdT = _t(Wd)
    rec, _ = record("M32 dh", got["dh"], oracle_mod.tree_gemm(dO, WdT), _cond(dO, WdT))
    assert rec["rel_l2"] <= 1e-3
    dU, _, dG = oracle_mod.silu_bwd(got["dh"], got["gate"], got["up"])
    assert mismatches(got["dU"], dU) == 0          # element-wise stages: bit-exact
    assert mismatches(got["dG"], dG) == 0
    dX = oracle_mod.add_bf16(oracle_mod.tree_gemm(got["dG"], _t(Wg)), oracle_mod.tree_gemm(got["dU"], _t(Wu)))
    rec, _ = record("M32 dX", got["dX"], dX)
    assert rec["rel_l2"] <= 1e-3
    ri, rn = sample_indices(I, 64, 20), sample_indices(H, 64, 21)
    xT, hT = _t(x), _t(h)
    for name, rows, A, B in [("M32 dWg", ri, _t(got["dG"])[ri], xT), ("M32 dWu", ri, _t(got["dU"])[ri], xT),
                             ("M32 dWd", rn, _t(dO)[rn], hT)]:
        rec, _ = record(name + " (64 rows)", got[name.split()[1]][rows], oracle_mod.tree_gemm(A, B), _cond(A, B))
        assert rec["rel_l2"] <= 1e-3
    # The elements of gate more than 1 ulp from the oracle: the tree over the
    # GPU's own leaves reproduces them (leaf dump of the same contraction).
    g_l, lv = G.detffn_tree_gemm_leaves(t["x"], t["Wg"])
    assert mismatches(host(g_l), got["gate"]) == 0
    assert mismatches(oracle_mod.tree_replay(lv.cpu().numpy()), got["gate"]) == 0
    del lv
    # Shards: 0 mismatches on out, dHidden and every dW.
    for k in [2, 4, 8]:
        sh = _fwd_bwd_saves(G, t, k=k)
        for n in ["out", "gate", "up", "dh", "dX", "dWg", "dWu", "dWd"]:
            assert mismatches(sh[n], got[n]) == 0, (k, n)


def test_m4096_forward_backward_sampled_and_chunks(G, oracle_mod):
    """M=4096 (2 x 2048 tokens), H=4096, I=12288 on the default family: 64
    seeded token rows of every row-wise stage and 64 seeded rows of each
    weight gradient against the oracle (fed the GPU's own stage inputs), and
    the weight gradients from c = 2 and c = 4 token chunks bit-equal to the
    one-shot backward (PR #325, "Design": CP token sequences gathered before
    the weight-gradient GEMMs)."""
    M, H, I = 4096, 4096, 12288
    d = ffn_inputs(M, H, I, seed=7)
    t = {n: dev(v) for n, v in d.items()}
    got = _fwd_bwd_saves(G, t, path=0)
    x, Wg, Wu, Wd, dO = d["x"], d["Wg"], d["Wu"], d["Wd"], d["dOut"]
    rm = sample_indices(M, 64, 30)
    xr = x[rm]
    for name, W in [("gate", Wg), ("up", Wu)]:
        rec, _ = record("M4096 %s (64 rows)" % name, got[name][rm], oracle_mod.tree_gemm(xr, W), _cond(xr, W))
        assert rec["rel_l2"] <= 1e-3
    hr = oracle_mod.silu_mul(got["gate"][rm], got["up"][rm])
    rec, _ = record("M4096 out (64 rows)", got["out"][rm], oracle_mod.tree_gemm(hr, Wd), _cond(hr, Wd))
    assert rec["rel_l2"] <= 1e-3
    WdT = _t(Wd)
    rec, _ = record("M4096 dh (64 rows)", got["dh"][rm], oracle_mod.tree_gemm(dO[rm], WdT), _cond(dO[rm], WdT))
    assert rec["rel_l2"] <= 1e-3
    del WdT
    dU, _, dG = oracle_mod.silu_bwd(got["dh"][rm], got["gate"][rm], got["up"][rm])
    assert mismatches(got["dU"][rm], dU) == 0
    assert mismatches(got["dG"][rm], dG) == 0
    dX = oracle_mod.add_bf16(oracle_mod.tree_gemm(got["dG"][rm], _t(Wg)), oracle_mod.tree_gemm(got["dU"][rm], _t(Wu)))
    rec, _ = record("M4096 dX (64 rows)", got["dX"][rm], dX)
    assert rec["rel_l2"] <= 1e-3
    ri, rn = sample_indices(I, 64, 31), sample_indices(H, 64, 32)
    xT = _t(x)
    for name, src in [("dWg", "dG"), ("dWu", "dU")]:
        A = _t(got[src])[ri]
        rec, _ = record("M4096 %s (64 rows)" % name, got[name][ri], oracle_mod.tree_gemm(A, xT), _cond(A, xT))
        assert rec["rel_l2"] <= 1e-3
    del xT
    hT = _t(oracle_mod.silu_mul(got["gate"], got["up"]))
    A = _t(dO)[rn]
    rec, _ = record("M4096 dWd (64 rows)", got["dWd"][rn], oracle_mod.tree_gemm(A, hT), _cond(A, hT))
    assert rec["rel_l2"] <= 1e-3
    del hT
    # Chunks in logical order: the same bits as the one-shot weight gradients.
    g, u = dev(got["gate"]), dev(got["up"])
    for c in (2, 4):
        sl = [slice(j * M // c, (j + 1) * M // c) for j in range(c)]
        dWg, dWu, dWd = G.detffn_wgrad_chunked([t["x"][s] for s in sl], [g[s] for s in sl],
                                               [u[s] for s in sl], [t["dOut"][s] for s in sl], t["Wd"])
        assert mismatches(host(dWg), got["dWg"]) == 0, c
        assert mismatches(host(dWu), got["dWu"]) == 0, c
        assert mismatches(host(dWd), got["dWd"]) == 0, c


def test_token_results_do_not_depend_on_token_count(G):
    """Batch invariance on the tensor family: token 0's gate, up and output
    (and tokens 0-7's) are the same bits at M = 1, 8, 32 (few-token kernels,
    weights on the MMA's 128-row side) and M = 4096 (many-token kernel,
    tokens on that side)."""
    M, H, I = 4096, 4096, 12288
    d = ffn_inputs(M, H, I, seed=5, with_dout=False)
    t = {n: dev(v) for n, v in d.items()}
    res = {}
    for m in (1, 8, 32, 4096):
        g, u = empty_bf16(m, I), empty_bf16(m, I)
        out = G.detffn_forward(t["x"][:m], t["Wg"], t["Wu"], t["Wd"], gate_save=g, up_save=u, path=TENSOR)
        torch.cuda.synchronize()
        res[m] = {"gate": host(g[:8]), "up": host(u[:8]), "out": host(out[:8])}
    for m in (8, 32, 4096):
        for n in ("gate", "up", "out"):
            assert mismatches(res[m][n][:1], res[1][n]) == 0, (m, n)
            if m > 8:
                assert mismatches(res[m][n][:8], res[8][n]) == 0, (m, n)
