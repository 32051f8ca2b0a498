"""Pins of the oracle's FFN forward/backward, sharding and chunking.

* Against the unrounded binary64 FFN: relative L2 <= 1e-2 on every output
  (a dropped term, wrong sign or transposed operand moves it far above that).
* Shard invariance: K-shards of the down projection (and of dHidden) combined
  by the balanced rank tree reproduce the unsharded result bit for bit
  (RL-Kernel PR #325, "Design": "Make each contiguous TP K shard the same
  subtree used by TP=1"; fixed balanced BF16 rank reduction tree).
* Chunk invariance: weight gradients from chunked token sets equal the
  one-shot result (PR #325, "Design": "Gather complete CP token sequences
  before weight-gradient GEMMs so their K tree matches CP=1").
"""
import numpy as np
import pytest

from gemm_deterministic_bf16_gb300.inputs import ffn_inputs
from oracle.fp64 import ffn_fp64, rel_l2


@pytest.fixture(scope="module")
def tiny(oracle_mod):
    # The tiny configuration: M=8, H=256, I=768, one seed.
    d = ffn_inputs(8, 256, 768, seed=0)
    fwd = oracle_mod.ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"])
    bwd = oracle_mod.ffn_backward(d["x"], d["Wg"], d["Wu"], d["Wd"], fwd["gate"], fwd["up"], d["dOut"])
    return d, fwd, bwd


def test_against_fp64(oracle_mod, tiny):
    d, fwd, bwd = tiny
    ref = ffn_fp64(d["x"], d["Wg"], d["Wu"], d["Wd"], d["dOut"])
    f = oracle_mod.bf16_to_f32
    errs = {k: rel_l2(f(fwd[k]), ref[k]) for k in ["gate", "up", "h", "out"]}
    errs.update({k: rel_l2(f(bwd[k]), ref[k]) for k in ["dh", "dU", "dG", "dX", "dWg", "dWu", "dWd"]})
    assert max(errs.values()) <= 1e-2, errs
    # A planted transposition of the weights is far outside the bound.
    bad = oracle_mod.ffn_forward(d["x"], d["Wu"], d["Wg"], d["Wd"])["out"]
    assert rel_l2(f(bad), ref["out"]) > 0.1


def test_against_fp64_medium(oracle_mod):
    d = ffn_inputs(4, 512, 1536, seed=5)
    fwd = oracle_mod.ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"])
    bwd = oracle_mod.ffn_backward(d["x"], d["Wg"], d["Wu"], d["Wd"], fwd["gate"], fwd["up"], d["dOut"])
    ref = ffn_fp64(d["x"], d["Wg"], d["Wu"], d["Wd"], d["dOut"])
    f = oracle_mod.bf16_to_f32
    for k in ["out"]:
        assert rel_l2(f(fwd[k]), ref[k]) <= 1e-2
    for k in ["dX", "dWg", "dWu", "dWd"]:
        assert rel_l2(f(bwd[k]), ref[k]) <= 1e-2


@pytest.mark.parametrize("k", [1, 2, 4])
def test_shard_invariance_tiny(oracle_mod, tiny, k):
    d, fwd, bwd = tiny
    out_k, parts = oracle_mod.ffn_forward_sharded(d["x"], d["Wg"], d["Wu"], d["Wd"], k)
    assert len(parts) == k
    assert np.array_equal(out_k, fwd["out"])
    dX_k = oracle_mod.dhidden_sharded(bwd["dG"], bwd["dU"], d["Wg"], d["Wu"], k)
    assert np.array_equal(dX_k, bwd["dX"])


@pytest.mark.parametrize("k", [2, 4, 8])
def test_shard_invariance_k8_shape(oracle_mod, k):
    # I=1536 -> 24 leaves: 12/6/3 leaves per shard (the 3-leaf subtrees test the odd split).
    d = ffn_inputs(3, 128, 1536, seed=7)
    fwd = oracle_mod.ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"])
    out_k, _ = oracle_mod.ffn_forward_sharded(d["x"], d["Wg"], d["Wu"], d["Wd"], k)
    assert np.array_equal(out_k, fwd["out"])


def test_shard_preconditions(oracle_mod, tiny):
    d, _, _ = tiny
    with pytest.raises(ValueError):   # 768/8 = 96 is not a whole number of leaves
        oracle_mod.ffn_forward_sharded(d["x"], d["Wg"], d["Wu"], d["Wd"], 8)


def test_sharding_changes_nothing_only_because_of_the_tree(oracle_mod):
    """Planted mistake: combining shard roots sequentially instead of with the
    balanced tree breaks bitwise equality on some element, so the invariance
    test above is sensitive to the rank-tree shape."""
    d = ffn_inputs(16, 128, 2048, seed=9)
    fwd = oracle_mod.ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"])
    _, parts = oracle_mod.ffn_forward_sharded(d["x"], d["Wg"], d["Wu"], d["Wd"], 4)
    f = oracle_mod.bf16_to_f32
    seq = parts[0]
    for p in parts[1:]:
        seq = oracle_mod.rne_bf16(f(seq) + f(p))
    assert not np.array_equal(seq, fwd["out"])


def _chunks(d, M, sizes):
    from oracle import ffn_forward
    fwd = ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"])
    edges = np.cumsum([0] + list(sizes))
    assert edges[-1] == M
    sl = [slice(a, b) for a, b in zip(edges[:-1], edges[1:])]
    return fwd, [d["x"][s] for s in sl], [fwd["gate"][s] for s in sl], \
        [fwd["up"][s] for s in sl], [d["dOut"][s] for s in sl]


@pytest.mark.parametrize("sizes", [[256], [128, 128], [64, 64, 64, 64], [100, 156], [1, 200, 55]])
def test_chunk_invariance(oracle_mod, sizes):
    M = 256
    d = ffn_inputs(M, 64, 128, seed=11)
    fwd, xs, gs, us, ds = _chunks(d, M, sizes)
    one = oracle_mod.ffn_backward(d["x"], d["Wg"], d["Wu"], d["Wd"], fwd["gate"], fwd["up"], d["dOut"])
    dWg, dWu, dWd = oracle_mod.wgrad_chunked(xs, gs, us, ds, d["Wd"])
    assert np.array_equal(dWg, one["dWg"])
    assert np.array_equal(dWu, one["dWu"])
    assert np.array_equal(dWd, one["dWd"])


@pytest.mark.parametrize("c", [2, 4])
def test_chunk_roots_equal_one_shot(oracle_mod, c):
    """Stricter reading: per-chunk subtree roots (512 tokens = 8 leaves, split
    into c aligned subtrees) combined by the rank tree equal the one-shot tree."""
    M = 512
    d = ffn_inputs(M, 32, 64, seed=12)
    fwd, xs, gs, us, ds = _chunks(d, M, [M // c] * c)
    one = oracle_mod.wgrad_chunked([d["x"]], [fwd["gate"]], [fwd["up"]], [d["dOut"]], d["Wd"])
    roots = oracle_mod.wgrad_chunk_roots(xs, gs, us, ds, d["Wd"])
    for a, b in zip(roots, one):
        assert np.array_equal(a, b)
