"""Forward on host buffers (DETFFN_FLAG_HOST_IO): x and out in page-locked
host memory, moved by the call's own copy kernels in stream order.

The arithmetic is the device-buffer forward's (RL-Kernel PR #325, "Design"),
so out must be the same bits -- on the one-launch few-token forward, the
two-launch form, the many-token tiles, the exact family and the sharded
forward -- and a sequence of calls on changing host inputs, issued without a
host synchronization between them, must give each call's own result.
"""

import numpy as np
import pytest
import torch

from gemm_deterministic_bf16_gb300.inputs import ffn_inputs
from tests.gpu_util import dev, empty_bf16, host, mismatches

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    import gemm_deterministic_bf16_gb300 as G
    from gemm_deterministic_bf16_gb300 import build
    build.build()
    return G


def _pinned(u16):
    t = torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory()


def _case(M, H, I, seed):
    d = ffn_inputs(M, H, I, seed=seed, with_dout=False)
    return d, {n: dev(v) for n, v in d.items()}


@pytest.mark.parametrize("M,H,I,path,flags", [
    (32, 4096, 12288, 0, 0),   # one-launch decode forward
    (8, 1024, 1536, 0, 0),
    (17, 1024, 1536, 2, 4),    # two-launch form (DETFFN_FLAG_SPLIT_FORWARD)
    (1, 256, 768, 1, 0),       # exact family
    (96, 512, 1536, 2, 0),     # many-token tiles
])
def test_host_buffers_same_bits(G, M, H, I, path, flags):
    d, t = _case(M, H, I, seed=70 + M)
    ref = G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], path=path, flags=flags)
    torch.cuda.synchronize()
    xh = _pinned(d["x"])
    oh = torch.empty((M, H), dtype=torch.bfloat16).pin_memory()
    got = G.detffn_forward(xh, t["Wg"], t["Wu"], t["Wd"], out=oh, path=path, flags=flags | G.FLAG_HOST_IO)
    assert got.data_ptr() == oh.data_ptr()
    torch.cuda.synchronize()
    assert G.detffn_get_status() == 0
    assert mismatches(host(ref), host(oh)) == 0


def test_host_buffers_with_saves_and_shards(G):
    M, H, I = 8, 1024, 1536
    d, t = _case(M, H, I, seed=81)
    g, u = empty_bf16(M, I), empty_bf16(M, I)
    ref = G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"])
    G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], gate_save=g, up_save=u)
    rg, ru = host(g), host(u)
    xh = _pinned(d["x"])
    g.zero_()
    u.zero_()
    oh = G.detffn_forward(xh, t["Wg"], t["Wu"], t["Wd"], gate_save=g, up_save=u, flags=G.FLAG_HOST_IO)
    sh = G.detffn_forward_sharded(xh, t["Wg"], t["Wu"], t["Wd"], 2, flags=G.FLAG_HOST_IO)
    torch.cuda.synchronize()
    assert G.detffn_get_status() == 0
    assert mismatches(host(ref), host(oh)) == 0
    assert mismatches(host(ref), host(sh)) == 0
    assert mismatches(rg, host(g)) == 0 and mismatches(ru, host(u)) == 0


def test_host_buffers_unaligned_and_in_stream_order(G):
    """x and out at 2-byte offsets into pinned buffers (the copies then move
    2-byte elements), and several calls with different inputs issued back to
    back on one stream before a single synchronization."""
    M, H, I = 8, 1024, 1536
    cases = [_case(M, H, I, seed=90 + i) for i in range(3)]
    refs = []
    for d, t in cases:
        refs.append(host(G.detffn_forward(t["x"], cases[0][1]["Wg"], cases[0][1]["Wu"], cases[0][1]["Wd"])))
    torch.cuda.synchronize()
    w = cases[0][1]
    xbuf = torch.empty(3 * M * H + 1, dtype=torch.bfloat16).pin_memory()
    obuf = torch.empty(3 * M * H + 1, dtype=torch.bfloat16).pin_memory()
    outs = []
    for i, (d, _) in enumerate(cases):
        xv = xbuf[1 + i * M * H: 1 + (i + 1) * M * H].view(M, H)
        xv.copy_(torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16))
        ov = obuf[1 + i * M * H: 1 + (i + 1) * M * H].view(M, H)
        outs.append(G.detffn_forward(xv, w["Wg"], w["Wu"], w["Wd"], out=ov, flags=G.FLAG_HOST_IO))
    torch.cuda.synchronize()
    assert G.detffn_get_status() == 0
    for r, o in zip(refs, outs):
        assert mismatches(r, host(o)) == 0


def test_host_flag_rejects_other_memory(G):
    """The flag with device or pageable host buffers, and on calls that do not
    take it: DETFFN_ERR_INVALID_ARG, nothing launched."""
    from gemm_deterministic_bf16_gb300 import detffn as D
    L = D.lib()
    M, H, I = 1, 256, 768
    _, t = _case(M, H, I, seed=99)
    out = empty_bf16(M, H)
    ws = G.workspace(G.OP_FORWARD, M, H, I, flags=G.FLAG_HOST_IO)
    pageable = torch.zeros(M, H, dtype=torch.bfloat16)
    pinned = torch.zeros(M, H, dtype=torch.bfloat16).pin_memory()
    h = D.handle()
    opts = D._opts(0, 1, 0, G.FLAG_HOST_IO)
    for xp, op in ((t["x"], out), (pageable, pinned), (pinned, pageable), (pinned, out)):
        st = L.detffn_forward(h, xp.data_ptr(), t["Wg"].data_ptr(), t["Wu"].data_ptr(), t["Wd"].data_ptr(),
                              op.data_ptr(), None, None, M, H, I, ws.data_ptr(), ws.numel(), None, opts)
        assert st == 1
    # A workspace sized without the flag is too small for the staged copies.
    ws0 = G.workspace(G.OP_FORWARD, M, H, I)
    pinned_out = torch.zeros(M, H, dtype=torch.bfloat16).pin_memory()
    assert ws0.numel() < ws.numel()
    st = L.detffn_forward(h, pinned.data_ptr(), t["Wg"].data_ptr(), t["Wu"].data_ptr(), t["Wd"].data_ptr(),
                          pinned_out.data_ptr(), None, None, M, H, I, ws0.data_ptr(), ws0.numel(), None, opts)
    assert st == D.ERR_WORKSPACE
    with pytest.raises(G.DetFFNError) as e:
        G.detffn_backward(t["x"], t["Wg"], t["Wu"], t["Wd"], empty_bf16(M, I), empty_bf16(M, I),
                          empty_bf16(M, H), flags=G.FLAG_HOST_IO)
    assert e.value.status == 1
    with pytest.raises(ValueError):
        G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], flags=G.FLAG_HOST_IO)
    torch.cuda.synchronize()
    assert G.detffn_get_status() == 0
