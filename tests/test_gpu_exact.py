"""GPU parity of the exact (CUDA-core, LANE8x8 leaves) path against the oracle:
bit-exact, i.e. 0 mismatching elements, on every output and stage.

Configurations: the tiny FFN (M=8, H=256, I=768) with shards k=1,2,4; ragged
shapes (partial leaves, M=1, odd sizes); decode forward M in {1, 8, 32} at
H=4096, I=12288; the M=32 training shape with k=2,4,8 shards.
Determinism (RL-Kernel PR #325, "Correctness results"): repeated runs,
training vs inference forward, sharded vs unsharded (forward output and
dHidden) must all show 0 mismatches.
"""
import numpy as np
import pytest
import torch

from gemm_deterministic_bf16_gb300.inputs import ffn_inputs, sample_indices
from tests.gpu_util import dev, empty_bf16, host, mismatches

pytestmark = pytest.mark.gpu
EXACT = 1


@pytest.fixture(scope="module")
def G():
    import gemm_deterministic_bf16_gb300 as G
    from gemm_deterministic_bf16_gb300 import build
    build.build()
    return G


def _run_fwd_bwd(G, d, path=EXACT, shards=1, k_fwd=1):
    M, H = d["x"].shape
    I = d["Wg"].shape[0]
    t = {n: dev(v) for n, v in d.items()}
    gate, up = empty_bf16(M, I), empty_bf16(M, I)
    if k_fwd == 1:
        out = G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], gate_save=gate, up_save=up, path=path)
    else:
        out = G.detffn_forward_sharded(t["x"], t["Wg"], t["Wu"], t["Wd"], k_fwd, gate_save=gate,
                                       up_save=up, path=path)
    dh, dU, dG = empty_bf16(M, I), empty_bf16(M, I), empty_bf16(M, I)
    dX, dWg, dWu, dWd = G.detffn_backward(t["x"], t["Wg"], t["Wu"], t["Wd"], gate, up, t["dOut"],
                                          dh_save=dh, dU_save=dU, dG_save=dG, shards=shards,
                                          path=path)
    torch.cuda.synchronize()
    return {k: host(v) for k, v in dict(out=out, gate=gate, up=up, dh=dh, dU=dU, dG=dG, dX=dX,
                                        dWg=dWg, dWu=dWu, dWd=dWd).items()}


def _oracle(oracle_mod, d):
    f = oracle_mod.ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"])
    b = oracle_mod.ffn_backward(d["x"], d["Wg"], d["Wu"], d["Wd"], f["gate"], f["up"], d["dOut"])
    return {**f, **b}


def test_silu_tables_on_device(G, oracle_mod):
    s, d = G.detffn_silu_tables()
    os_, od = oracle_mod.silu_tables()
    fin = np.isfinite(od)
    assert np.array_equal(d[fin].view(np.uint32), od[fin].view(np.uint32))
    nan = (os_ & 0x7FFF) > 0x7F80
    assert np.array_equal(s[~nan], os_[~nan])


def test_tiny_config_bit_exact(G, oracle_mod):
    d = ffn_inputs(8, 256, 768, seed=0)
    got = _run_fwd_bwd(G, d)
    ref = _oracle(oracle_mod, d)
    for k in ["gate", "up", "out", "dh", "dU", "dG", "dX", "dWg", "dWu", "dWd"]:
        assert mismatches(got[k], ref[k]) == 0, k


@pytest.mark.parametrize("k", [1, 2, 4])
def test_tiny_shards_and_repeat(G, k):
    d = ffn_inputs(8, 256, 768, seed=0)
    base = _run_fwd_bwd(G, d)
    again = _run_fwd_bwd(G, d, shards=k, k_fwd=k)
    for name in base:
        assert mismatches(base[name], again[name]) == 0, name


@pytest.mark.parametrize("M,H,I", [(1, 64, 128), (3, 200, 328), (5, 130, 190), (17, 96, 256),
                                   (70, 64, 192)])
def test_ragged_shapes_bit_exact(G, oracle_mod, M, H, I):
    d = ffn_inputs(M, H, I, seed=M + H + I)
    got = _run_fwd_bwd(G, d)
    ref = _oracle(oracle_mod, d)
    for k in ["gate", "up", "out", "dh", "dU", "dG", "dX", "dWg", "dWu", "dWd"]:
        assert mismatches(got[k], ref[k]) == 0, k


def test_training_and_inference_forward_agree(G):
    d = ffn_inputs(8, 512, 1024, seed=3)
    t = {n: dev(v) for n, v in d.items()}
    a = G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], path=EXACT)
    g, u = empty_bf16(8, 1024), empty_bf16(8, 1024)
    b = G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], gate_save=g, up_save=u, path=EXACT)
    assert mismatches(host(a), host(b)) == 0


@pytest.mark.parametrize("M", [1, 8, 32])
def test_decode_forward_bit_exact(G, oracle_mod, M):
    d = ffn_inputs(M, 4096, 12288, seed=1, with_dout=False)
    t = {n: dev(v) for n, v in d.items()}
    gate, up = empty_bf16(M, 12288), empty_bf16(M, 12288)
    out = G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], gate_save=gate, up_save=up, path=EXACT)
    ref = oracle_mod.ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"])
    assert mismatches(host(gate), ref["gate"]) == 0
    assert mismatches(host(up), ref["up"]) == 0
    assert mismatches(host(out), ref["out"]) == 0


def test_m32_training_shards(G, oracle_mod):
    """M=32, H=4096, I=12288 forward+backward; shards k=2,4,8 give 0
    mismatches on out, dHidden and every dW; dX and sampled dW rows match
    the oracle bit for bit (stage-wise: the oracle takes the GPU's dG/dU)."""
    d = ffn_inputs(32, 4096, 12288, seed=2)
    base = _run_fwd_bwd(G, d)
    for k in [2, 4, 8]:
        sh = _run_fwd_bwd(G, d, shards=k, k_fwd=k)
        for name in ["out", "dX", "dWg", "dWu", "dWd"]:
            assert mismatches(base[name], sh[name]) == 0, (k, name)
    ref = oracle_mod.ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"])
    assert mismatches(base["out"], ref["out"]) == 0
    cg = oracle_mod.tree_gemm(base["dG"], np.ascontiguousarray(d["Wg"].T))
    cu = oracle_mod.tree_gemm(base["dU"], np.ascontiguousarray(d["Wu"].T))
    assert mismatches(base["dX"], oracle_mod.add_bf16(cg, cu)) == 0
    rows_i = sample_indices(12288, 64, 20)
    rows_n = sample_indices(4096, 64, 21)
    h = oracle_mod.silu_mul(base["gate"], base["up"])
    dWg = oracle_mod.tree_gemm(np.ascontiguousarray(base["dG"].T[rows_i]), np.ascontiguousarray(d["x"].T))
    dWu = oracle_mod.tree_gemm(np.ascontiguousarray(base["dU"].T[rows_i]), np.ascontiguousarray(d["x"].T))
    dWd = oracle_mod.tree_gemm(np.ascontiguousarray(d["dOut"].T[rows_n]), np.ascontiguousarray(h.T))
    assert mismatches(base["dWg"][rows_i], dWg) == 0
    assert mismatches(base["dWu"][rows_i], dWu) == 0
    assert mismatches(base["dWd"][rows_n], dWd) == 0
    dh = oracle_mod.tree_gemm(d["dOut"], np.ascontiguousarray(d["Wd"].T))
    assert mismatches(base["dh"], dh) == 0


@pytest.mark.parametrize("sizes", [[128, 128], [64, 64, 64, 64], [100, 156], [1, 200, 55], [0, 256]])
def test_chunked_wgrad(G, oracle_mod, sizes):
    M, H, I = 256, 128, 384
    d = ffn_inputs(M, H, I, seed=4)
    base = _run_fwd_bwd(G, d)
    edges = np.cumsum([0] + sizes)
    t = {n: dev(v) for n, v in d.items()}
    g, u = dev(base["gate"]), dev(base["up"])
    sl = [slice(int(a), int(b)) for a, b in zip(edges[:-1], edges[1:])]
    dWg, dWu, dWd = G.detffn_wgrad_chunked([t["x"][s].contiguous() for s in sl],
                                           [g[s].contiguous() for s in sl],
                                           [u[s].contiguous() for s in sl],
                                           [t["dOut"][s].contiguous() for s in sl], t["Wd"], path=EXACT)
    assert mismatches(host(dWg), base["dWg"]) == 0
    assert mismatches(host(dWu), base["dWu"]) == 0
    assert mismatches(host(dWd), base["dWd"]) == 0
    ref = _oracle(oracle_mod, d)
    assert mismatches(host(dWd), ref["dWd"]) == 0


def test_tree_gemm_layouts(G, oracle_mod):
    rng = np.random.default_rng(5)
    from gemm_deterministic_bf16_gb300.inputs import to_bf16_bits
    A = to_bf16_bits(rng.standard_normal((70, 300)).astype(np.float32))
    B = to_bf16_bits(rng.standard_normal((90, 300)).astype(np.float32))
    ref = oracle_mod.tree_gemm(A, B)
    At, Bt = dev(np.ascontiguousarray(A.T)), dev(np.ascontiguousarray(B.T))
    got = G.detffn_tree_gemm(At.t(), Bt.t(), path=EXACT)      # both K-strided views
    assert mismatches(host(got), ref) == 0
    got = G.detffn_tree_gemm(dev(A), Bt.t(), path=EXACT)
    assert mismatches(host(got), ref) == 0
    z = G.detffn_tree_gemm(dev(A)[:, :0], dev(B)[:, :0], path=EXACT)   # K = 0 -> +0
    assert not host(z).any()


def test_status_word_ok(G):
    assert G.detffn_get_status() == 0


@pytest.mark.parametrize("M,H,I", [(2, 1024, 3072), (3, 256, 768), (5, 1024, 3072), (7, 512, 1536),
                                   (13, 1024, 3072), (24, 256, 768), (1, 4096, 1536)])
def test_decode_kernel_shapes_bit_exact(G, oracle_mod, M, H, I):
    """The weight-streaming decode kernel (leaf blocks of 4, 8, 12 and 24
    leaves, 1 to 4 token passes) against the oracle, forward and sharded."""
    d = ffn_inputs(M, H, I, seed=M * 7 + H, with_dout=False)
    t = {n: dev(v) for n, v in d.items()}
    gate, up = empty_bf16(M, I), empty_bf16(M, I)
    out = G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], gate_save=gate, up_save=up, path=EXACT)
    ref = oracle_mod.ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"])
    assert mismatches(host(gate), ref["gate"]) == 0
    assert mismatches(host(up), ref["up"]) == 0
    assert mismatches(host(out), ref["out"]) == 0
    for k in [2, 4]:
        if (I // k) % 64 == 0 and (I // k) // 64 >= 2:
            o2 = G.detffn_forward_sharded(t["x"], t["Wg"], t["Wu"], t["Wd"], k, path=EXACT)
            assert mismatches(host(o2), ref["out"]) == 0, k


def test_decode_repeat_and_stream(G):
    """Repeated decode forwards on a side stream are bitwise identical."""
    d = ffn_inputs(8, 4096, 12288, seed=11, with_dout=False)
    t = {n: dev(v) for n, v in d.items()}
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for _ in range(3):
            outs.append(G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], path=EXACT).clone())
    s.synchronize()
    assert mismatches(host(outs[0]), host(outs[1])) == 0
    assert mismatches(host(outs[0]), host(outs[2])) == 0
