"""GPU parity of the tensor-core (tcgen05) path.

Each 64-wide leaf is summed by the tensor core in the hardware's own order,
so on general data the leaves (and through them the outputs) may differ from
the oracle's LANE8x8 leaves; that is the tolerance branch of the contract.
Two kinds of checks:

* Integer-valued operands (entries in {-2, ..., 2}): every leaf is an exact
  integer below 2^24 whatever the summation order, so the tensor path must
  equal the oracle bit for bit.  This pins the TMA/descriptor layout, the
  leaf boundaries, the tree shapes (G = 1, 2, 3 bottom groups) and the
  stores, including partial leaves and ragged tiles.
* Random data: relative L2 <= 1e-3 against the oracle and the distribution
  of BF16 ulp distances, plus bitwise determinism and shard/chunk invariance
  within the tensor path (RL-Kernel PR #325, "Design"; "Correctness results").
"""
import numpy as np
import pytest
import torch

from gemm_deterministic_bf16_gb300.inputs import ffn_inputs, to_bf16_bits
from oracle.fp64 import rel_l2
from tests.gpu_util import dev, empty_bf16, host, mismatches, ulp_dist

pytestmark = pytest.mark.gpu
TENSOR = 2


@pytest.fixture(scope="module")
def G():
    import gemm_deterministic_bf16_gb300 as G
    from gemm_deterministic_bf16_gb300 import build
    build.build()
    return G


def _ints(shape, seed):
    rng = np.random.default_rng(seed)
    return to_bf16_bits(rng.integers(-2, 3, shape).astype(np.float32))


@pytest.mark.parametrize("R,C,K", [(128, 128, 64), (256, 128, 128), (128, 256, 256), (200, 300, 104),
                                   (130, 129, 192), (256, 256, 768), (128, 128, 4096),
                                   (256, 128, 12288), (384, 384, 3072),
                                   # block folds of short trees: three-leaf groups Q = 2, two-leaf Q = 4
                                   (200, 136, 384), (130, 200, 512)])
def test_tc_integer_inputs_bit_exact(G, oracle_mod, R, C, K):
    A, B = _ints((R, K), R + K), _ints((C, K), C + 7 * K)
    got = host(G.detffn_tree_gemm(dev(A), dev(B), path=TENSOR))
    assert mismatches(got, oracle_mod.tree_gemm(A, B)) == 0


@pytest.mark.parametrize("R,C,K", [(200, 296, 40), (130, 72, 64), (33, 1000, 24), (4096, 136, 32), (200, 300, 48)])
def test_tc_one_leaf_ragged_bit_exact(G, oracle_mod, R, C, K):
    """One-leaf trees (K <= 64) with more than 32 rows: the output leaves
    through TMA tensor stores of 32 x 64 boxes, clipped at ragged edges (or,
    with a row length that is not a multiple of 8, through plain stores)."""
    A, B = _ints((R, K), R + 3 * K), _ints((C, K), C + 5 * K)
    got = host(G.detffn_tree_gemm(dev(A), dev(B), path=TENSOR))
    assert mismatches(got, oracle_mod.tree_gemm(A, B)) == 0


@pytest.mark.parametrize("R,C,K", [(1, 256, 4096), (8, 384, 768), (32, 1024, 12288), (17, 200, 256)])
def test_tc_few_rows_swapped_bit_exact(G, oracle_mod, R, C, K):
    """R <= 32: weights on the 128-row MMA side, tokens as the 32-wide tile."""
    A, B = _ints((R, K), R + K + 1), _ints((C, K), C + K + 2)
    got = host(G.detffn_tree_gemm(dev(A), dev(B), path=TENSOR))
    assert mismatches(got, oracle_mod.tree_gemm(A, B)) == 0


def _stats(got, ref):
    f = lambda u: (np.asarray(u, np.uint32) << 16).view(np.float32)  # noqa: E731
    d = ulp_dist(got, ref)
    return rel_l2(f(got), f(ref)), float(np.mean(d <= 1)), int(d.max())


@pytest.mark.parametrize("R,C,K", [(256, 256, 4096), (256, 128, 12288)])
def test_tc_random_within_tolerance(G, oracle_mod, R, C, K):
    rng = np.random.default_rng(R + C + K)
    A = to_bf16_bits(rng.standard_normal((R, K)).astype(np.float32))
    B = to_bf16_bits((0.02 * rng.standard_normal((C, K))).astype(np.float32))
    got = host(G.detffn_tree_gemm(dev(A), dev(B), path=TENSOR))
    rl2, within1, mx = _stats(got, oracle_mod.tree_gemm(A, B))
    print("tensor vs oracle: rel-L2 %.3g, within 1 ulp %.6f, max ulp %d" % (rl2, within1, mx))
    assert rl2 <= 1e-3
    assert within1 >= 0.999


def _fwd_bwd(G, t, path, k=1):
    M, H = t["x"].shape
    I = t["Wg"].shape[0]
    g, u = empty_bf16(M, I), empty_bf16(M, I)
    if k == 1:
        out = G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], gate_save=g, up_save=u, path=path)
    else:
        out = G.detffn_forward_sharded(t["x"], t["Wg"], t["Wu"], t["Wd"], k, gate_save=g, up_save=u, path=path)
    dh = empty_bf16(M, I)
    dX, dWg, dWu, dWd = G.detffn_backward(t["x"], t["Wg"], t["Wu"], t["Wd"], g, u, t["dOut"],
                                          dh_save=dh, shards=k, path=path)
    torch.cuda.synchronize()
    return {n: host(v) for n, v in dict(out=out, gate=g, up=u, dh=dh, dX=dX, dWg=dWg, dWu=dWu,
                                        dWd=dWd).items()}


def test_tc_ffn_integer_inputs_bit_exact(G, oracle_mod):
    """Forward+backward on the tensor path with integer-valued x, dOut and
    weights: the contractions whose operands are integers (gate, up, dh) have
    exact leaves and must equal the oracle bit for bit; h and everything after
    it are not integers, so those stages are checked with the tolerance."""
    M, H, I = 128, 256, 768
    d = {"x": _ints((M, H), 1), "Wg": _ints((I, H), 2), "Wu": _ints((I, H), 3),
         "Wd": _ints((H, I), 4), "dOut": _ints((M, H), 5)}
    got = _fwd_bwd(G, {n: dev(v) for n, v in d.items()}, TENSOR)
    f = oracle_mod.ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"])
    assert mismatches(got["gate"], f["gate"]) == 0
    assert mismatches(got["up"], f["up"]) == 0
    b = oracle_mod.ffn_backward(d["x"], d["Wg"], d["Wu"], d["Wd"], got["gate"], got["up"], d["dOut"])
    assert mismatches(got["dh"], b["dh"]) == 0
    for n in ["out"]:
        assert _stats(got[n], f[n])[0] <= 1e-3, n
    for n in ["dX", "dWg", "dWu", "dWd"]:
        assert _stats(got[n], b[n])[0] <= 1e-3, n


def test_tc_ffn_random_tolerance_and_invariance(G, oracle_mod):
    M, H, I = 256, 512, 1536
    d = ffn_inputs(M, H, I, seed=21)
    t = {n: dev(v) for n, v in d.items()}
    base = _fwd_bwd(G, t, TENSOR)
    again = _fwd_bwd(G, t, TENSOR)
    for n in base:
        assert mismatches(base[n], again[n]) == 0, n            # repeat: bitwise
    for k in [2, 4, 8]:
        sh = _fwd_bwd(G, t, TENSOR, k)
        for n in ["out", "dX", "dWg", "dWu", "dWd"]:
            assert mismatches(base[n], sh[n]) == 0, (k, n)      # shards: bitwise
    f = oracle_mod.ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"])
    b = oracle_mod.ffn_backward(d["x"], d["Wg"], d["Wu"], d["Wd"], f["gate"], f["up"], d["dOut"])
    for n, ref in [("out", f["out"]), ("dX", b["dX"]), ("dWg", b["dWg"]), ("dWu", b["dWu"]), ("dWd", b["dWd"])]:
        rl2, within1, mx = _stats(base[n], ref)
        print("%s: rel-L2 %.3g, within 1 ulp %.5f, max ulp %d" % (n, rl2, within1, mx))
        assert rl2 <= 1e-3, n


def test_tc_chunked_wgrad_invariance(G):
    M, H, I = 512, 256, 768
    d = ffn_inputs(M, H, I, seed=22)
    t = {n: dev(v) for n, v in d.items()}
    base = _fwd_bwd(G, t, TENSOR)
    g, u = dev(base["gate"]), dev(base["up"])
    for sizes in ([256, 256], [128, 128, 128, 128], [100, 412], [16, 496]):
        e = np.cumsum([0] + sizes)
        sl = [slice(int(a), int(b)) for a, b in zip(e[:-1], e[1:])]
        dWg, dWu, dWd = G.detffn_wgrad_chunked([t["x"][s].contiguous() for s in sl],
                                               [g[s].contiguous() for s in sl],
                                               [u[s].contiguous() for s in sl],
                                               [t["dOut"][s].contiguous() for s in sl], t["Wd"],
                                               path=TENSOR)
        assert mismatches(host(dWg), base["dWg"]) == 0
        assert mismatches(host(dWu), base["dWu"]) == 0
        assert mismatches(host(dWd), base["dWd"]) == 0


@pytest.mark.parametrize("M", [1, 8, 32])
def test_tc_decode_split_k_same_bits(G, oracle_mod, M):
    """The tensor forward at decode sizes splits K into aligned subtrees (block
    roots combined by the top of the tree); gate and up must equal the
    unsplit contraction bit for bit, and the output stays within tolerance
    of the oracle; sharded forwards agree bitwise."""
    H, I = 4096, 12288
    d = ffn_inputs(M, H, I, seed=30 + M, with_dout=False)
    t = {n: dev(v) for n, v in d.items()}
    g, u = empty_bf16(M, I), empty_bf16(M, I)
    out = G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], gate_save=g, up_save=u, path=TENSOR)
    g_direct = G.detffn_tree_gemm(t["x"], t["Wg"], path=TENSOR)    # no scratch: one block per tile
    assert mismatches(host(g), host(g_direct)) == 0
    for k in [2, 4, 8]:
        o2 = G.detffn_forward_sharded(t["x"], t["Wg"], t["Wu"], t["Wd"], k, path=TENSOR)
        assert mismatches(host(o2), host(out)) == 0, k
    ref = oracle_mod.ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"])
    rl2, within1, mx = _stats(host(out), ref["out"])
    print("decode M=%d tensor out: rel-L2 %.3g, within 1 ulp %.5f, max ulp %d" % (M, rl2, within1, mx))
    assert rl2 <= 1e-3


@pytest.mark.parametrize("M,H,I", [(32, 4096, 1536), (1, 768, 200), (17, 64, 384), (32, 12288, 256),
                                   (8, 192, 136), (32, 8192, 1024)])
def test_tcs_forward_integer_inputs_bit_exact(G, oracle_mod, M, H, I):
    """Few-token forward (balanced K ranges folded from pieces, SiLU * up fused
    into the top of the trees): with integer-valued x and weights every leaf is
    exact, so gate and up equal the oracle bit for bit -- this pins the piece
    split and fold for bottom groups of 1, 2 and 3 leaves, ragged row tiles
    and single tokens; h and out follow the tolerance."""
    d = {"x": _ints((M, H), M + 3), "Wg": _ints((I, H), 4), "Wu": _ints((I, H), 5), "Wd": _ints((H, I), 6)}
    t = {n: dev(v) for n, v in d.items()}
    g, u = empty_bf16(M, I), empty_bf16(M, I)
    out = G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], gate_save=g, up_save=u, path=TENSOR)
    out_inf = G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], path=TENSOR)
    f = oracle_mod.ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"])
    assert mismatches(host(g), f["gate"]) == 0
    assert mismatches(host(u), f["up"]) == 0
    assert mismatches(host(out), host(out_inf)) == 0          # training and inference forward agree
    assert _stats(host(out), f["out"])[0] <= 1e-3


@pytest.mark.parametrize("M,H,I", [(32, 4096, 1536), (5, 768, 1000), (32, 3072, 128)])
def test_tcs_pieces_equal_whole_tiles(G, M, H, I):
    """The forward's gate (pieces from balanced ranges, folded by the top
    kernel) equals the stand-alone contraction, which forms whole tiles in one
    CTA (no scratch): the same canonical tree either way."""
    d = ffn_inputs(M, H, I, seed=40 + M, with_dout=False)
    t = {n: dev(v) for n, v in d.items()}
    g, u = empty_bf16(M, I), empty_bf16(M, I)
    G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], gate_save=g, up_save=u, path=TENSOR)
    assert mismatches(host(g), host(G.detffn_tree_gemm(t["x"], t["Wg"], path=TENSOR))) == 0
    assert mismatches(host(u), host(G.detffn_tree_gemm(t["x"], t["Wu"], path=TENSOR))) == 0


@pytest.mark.parametrize("M", [32, 17, 8])
def test_tc_backward_few_tokens(G, oracle_mod, M):
    """Tensor-family backward with few tokens: the few-token contractions
    (dh, cg, cu), the weight and token transposes (vector tiles for 32 and 8
    tokens, element-wise for 17) and the one-leaf weight gradients.  With
    integer-valued operands dh is exact in any leaf order and must equal the
    oracle bit for bit; the rest follows the tolerance."""
    H, I = 512, 1536
    d = {"x": _ints((M, H), 11), "Wg": _ints((I, H), 12), "Wu": _ints((I, H), 13),
         "Wd": _ints((H, I), 14), "dOut": _ints((M, H), 15)}
    got = _fwd_bwd(G, {n: dev(v) for n, v in d.items()}, TENSOR)
    f = oracle_mod.ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"])
    b = oracle_mod.ffn_backward(d["x"], d["Wg"], d["Wu"], d["Wd"], got["gate"], got["up"], d["dOut"])
    assert mismatches(got["dh"], b["dh"]) == 0
    for n in ["dX", "dWg", "dWu", "dWd"]:
        assert _stats(got[n], b[n])[0] <= 1e-3, n


@pytest.mark.parametrize("R,C,K", [(1, 256, 4096), (32, 200, 768), (17, 384, 256), (200, 296, 1024), (256, 128, 64)])
def test_tc_weights_mn_major_bit_exact(G, oracle_mod, R, C, K):
    """B given as a column view of a [K, C] matrix (C contiguous, as the
    backward reads Wd, Wg and Wu) is read MN-major by the tensor core, with no
    transposed copy: with integer-valued operands the result must equal the
    oracle bit for bit (few-token and many-token kernels, ragged C)."""
    A = _ints((R, K), R + 5)
    Bt = _ints((K, C), C + 9)                   # stored [K, C]
    B_view = dev(Bt).t()                        # logical [C, K], strides (1, C)
    assert B_view.stride() == (1, C)
    got = host(G.detffn_tree_gemm(dev(A), B_view, path=TENSOR))
    assert mismatches(got, oracle_mod.tree_gemm(A, np.ascontiguousarray(Bt.T))) == 0
