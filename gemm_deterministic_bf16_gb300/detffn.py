"""ctypes binding of libdetffn (argument marshalling only).

Every function here has the name of the C call it wraps and does nothing but
check tensor properties, pass ``data_ptr()`` values, sizes and the current
CUDA stream, and raise ``DetFFNError`` on a non-OK status.  All computation
happens in the library's CUDA kernels; there is no fallback.  Tensors are
``torch.bfloat16`` (rank tree: float32/float16/bfloat16) on a CUDA device.
"""
import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdetffn.so")

OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_ALIGN, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(8)
F32, F16, BF16 = 0, 1, 2
PATH_AUTO, PATH_EXACT, PATH_TENSOR = 0, 1, 2
OP_FORWARD, OP_FORWARD_SHARDED, OP_BACKWARD, OP_WGRAD_CHUNKED = 0, 1, 2, 3

_vp, _ll, _int = ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int


class DetFFNError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        msg = "%s: %s (status %d)" % (what, _status_string(status), status)
        if status == ERR_CUDA:
            try:
                L = lib()
                L.detffn_last_cuda_error.restype = ctypes.c_char_p
                msg += ": " + L.detffn_last_cuda_error().decode()
            except Exception:  # noqa: BLE001 - only used to format an error message
                pass
        super().__init__(msg)


FLAG_TEST_STALL = 1
FLAG_OVERLAP_DHIDDEN = 2
FLAG_SPLIT_FORWARD = 4
FLAG_HOST_IO = 8


class Options(ctypes.Structure):
    _fields_ = [("leaf_width", ctypes.c_int), ("path", ctypes.c_int),
                ("shards", ctypes.c_int), ("flags", ctypes.c_int), ("spin_limit", ctypes.c_longlong)]


_LOCK = threading.Lock()
_LIB = None
_HANDLES = {}


def lib():
    """The loaded libdetffn.so; raises if it has not been built."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libdetffn.so is missing (build it with "
                                   "gemm_deterministic_bf16_gb300.build.build())")
            L = ctypes.CDLL(LIB_PATH)
            st = ctypes.c_int
            L.detffn_status_string.argtypes = [st]
            L.detffn_status_string.restype = ctypes.c_char_p
            L.detffn_create.argtypes = [ctypes.POINTER(_vp), _int]
            L.detffn_destroy.argtypes = [_vp]
            L.detffn_workspace_size.argtypes = [_vp, _int, _ll, _ll, _ll, _int, ctypes.POINTER(Options),
                                                ctypes.POINTER(ctypes.c_size_t)]
            L.detffn_forward.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _ll, _ll, _ll,
                                         _vp, ctypes.c_size_t, _vp, ctypes.POINTER(Options)]
            L.detffn_forward_sharded.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _ll, _ll,
                                                 _ll, _int, _vp, ctypes.c_size_t, _vp,
                                                 ctypes.POINTER(Options)]
            L.detffn_backward.argtypes = [_vp] + [_vp] * 7 + [_vp] * 4 + [_vp] * 3 + \
                [_ll, _ll, _ll, _vp, ctypes.c_size_t, _vp, ctypes.POINTER(Options)]
            L.detffn_wgrad_chunked.argtypes = [_vp, _int, ctypes.POINTER(_ll), ctypes.POINTER(_vp),
                                               ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                               ctypes.POINTER(_vp), _vp, _vp, _vp, _vp, _ll, _ll,
                                               _vp, ctypes.c_size_t, _vp, ctypes.POINTER(Options)]
            L.detffn_rank_tree_reduce.argtypes = [ctypes.POINTER(_vp), _int, _vp, _ll, _int, _vp]
            L.detffn_tree_gemm.argtypes = [_vp, _vp, _ll, _ll, _vp, _ll, _ll, _ll, _ll, _ll, _vp,
                                           _ll, _vp, ctypes.POINTER(Options)]
            L.detffn_silu_tables.argtypes = [_vp, _vp, _vp]
            L.detffn_get_status.argtypes = [_vp, _vp]
            for name in ["detffn_create", "detffn_destroy", "detffn_workspace_size", "detffn_forward",
                         "detffn_forward_sharded", "detffn_backward", "detffn_wgrad_chunked",
                         "detffn_rank_tree_reduce", "detffn_tree_gemm", "detffn_silu_tables",
                         "detffn_get_status"]:
                getattr(L, name).restype = st
            _LIB = L
    return _LIB


def _status_string(s):
    try:
        return lib().detffn_status_string(s).decode()
    except Exception:  # noqa: BLE001 - only used to format an error message
        return "status %d" % s


def _check(status, what):
    if status != OK:
        raise DetFFNError(status, what)


def handle(device=None):
    """The per-device handle (created on first use)."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else
                       torch.device(device).index or 0)
    key = dev.index
    with _LOCK:
        h = _HANDLES.get(key)
    if h is None:
        hv = _vp()
        _check(lib().detffn_create(ctypes.byref(hv), key), "detffn_create")
        with _LOCK:
            h = _HANDLES.setdefault(key, hv.value)
    return h


def _opts(path=PATH_AUTO, shards=1, spin_limit=0, flags=0):
    return ctypes.byref(Options(64, path, shards, flags, spin_limit))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(dev, stream):
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    return s.cuda_stream


def _bf16(*ts):
    for t in ts:
        if t is not None:
            if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
                raise ValueError("expected contiguous CUDA bfloat16 tensors")


def _bf16_host(*ts):
    for t in ts:
        if t.dtype != torch.bfloat16 or t.is_cuda or not t.is_pinned() or not t.is_contiguous():
            raise ValueError("FLAG_HOST_IO: expected contiguous pinned (page-locked) CPU bfloat16 tensors")


def _io(x, out, M, H, device, flags):
    """x and out of a forward: device tensors, or pinned host tensors under
    FLAG_HOST_IO (out allocated where it is None)."""
    if flags & FLAG_HOST_IO:
        if out is None:
            out = torch.empty((M, H), dtype=torch.bfloat16).pin_memory()
        _bf16_host(x, out)
    else:
        if out is None:
            out = torch.empty((M, H), dtype=torch.bfloat16, device=device)
        _bf16(x, out)
    return out


def detffn_workspace_size(op, M, H, I, k=1, path=PATH_AUTO, device=None, flags=0):
    n = ctypes.c_size_t()
    _check(lib().detffn_workspace_size(handle(device), op, M, H, I, k, _opts(path, 1, 0, flags),
                                       ctypes.byref(n)), "detffn_workspace_size")
    return n.value


def workspace(op, M, H, I, k=1, path=PATH_AUTO, device=None, flags=0):
    """A caller-owned scratch buffer of the size the call needs (flags:
    FLAG_HOST_IO for forwards on host buffers)."""
    n = detffn_workspace_size(op, M, H, I, k, path, device, flags)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def detffn_forward(x, Wg, Wu, Wd, out=None, gate_save=None, up_save=None, ws=None,
                   path=PATH_AUTO, stream=None, spin_limit=0, flags=0):
    """out = down(silu(gate) * up); x [M,H], Wg/Wu [I,H], Wd [H,I].  Pass
    gate_save/up_save ([M,I]) to keep gate and up (training mode).
    spin_limit and flags go to detffn_options (flags: FLAG_TEST_STALL for
    tests of the failure path only; FLAG_HOST_IO: x and out are pinned CPU
    tensors, moved by the call itself; out is complete once the stream has
    passed the call)."""
    _bf16(Wg, Wu, Wd, gate_save, up_save)
    M, H = x.shape
    I = Wg.shape[0]
    dev = Wg.device
    out = _io(x, out, M, H, dev, flags)
    if ws is None:
        ws = workspace(OP_FORWARD, M, H, I, 1, path, dev, flags & FLAG_HOST_IO)
    _check(lib().detffn_forward(handle(dev), _ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(out),
                                _ptr(gate_save), _ptr(up_save), M, H, I, _ptr(ws), ws.numel(),
                                _stream(dev, stream), _opts(path, 1, spin_limit, flags)),
           "detffn_forward")
    return out


def detffn_forward_sharded(x, Wg, Wu, Wd, k, out=None, gate_save=None, up_save=None, ws=None,
                           path=PATH_AUTO, stream=None, flags=0):
    """Forward with k in {1,2,4,8} tensor-parallel shards of I emulated on one
    GPU; the same bits as detffn_forward (flags as there)."""
    _bf16(Wg, Wu, Wd, gate_save, up_save)
    M, H = x.shape
    I = Wg.shape[0]
    dev = Wg.device
    out = _io(x, out, M, H, dev, flags)
    if ws is None:
        ws = workspace(OP_FORWARD_SHARDED, M, H, I, k, path, dev, flags & FLAG_HOST_IO)
    _check(lib().detffn_forward_sharded(handle(dev), _ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd),
                                        _ptr(out), _ptr(gate_save), _ptr(up_save), M, H, I, k,
                                        _ptr(ws), ws.numel(), _stream(dev, stream),
                                        _opts(path, 1, 0, flags)), "detffn_forward_sharded")
    return out


def detffn_backward(x, Wg, Wu, Wd, gate, up, dOut, dX=None, dWg=None, dWu=None, dWd=None,
                    dh_save=None, dU_save=None, dG_save=None, ws=None, shards=1,
                    path=PATH_AUTO, stream=None, spin_limit=0, flags=0):
    """Returns (dX, dWg, dWu, dWd)."""
    _bf16(x, Wg, Wu, Wd, gate, up, dOut, dX, dWg, dWu, dWd, dh_save, dU_save, dG_save)
    M, H = x.shape
    I = Wg.shape[0]
    e = lambda *s: torch.empty(s, dtype=torch.bfloat16, device=x.device)  # noqa: E731
    dX = e(M, H) if dX is None else dX
    dWg = e(I, H) if dWg is None else dWg
    dWu = e(I, H) if dWu is None else dWu
    dWd = e(H, I) if dWd is None else dWd
    if ws is None:
        ws = workspace(OP_BACKWARD, M, H, I, shards, path, x.device)
    _check(lib().detffn_backward(handle(x.device), _ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd),
                                 _ptr(gate), _ptr(up), _ptr(dOut), _ptr(dX), _ptr(dWg), _ptr(dWu),
                                 _ptr(dWd), _ptr(dh_save), _ptr(dU_save), _ptr(dG_save), M, H, I,
                                 _ptr(ws), ws.numel(), _stream(x.device, stream),
                                 _opts(path, shards, spin_limit, flags)), "detffn_backward")
    return dX, dWg, dWu, dWd


def detffn_wgrad_chunked(x_chunks, gate_chunks, up_chunks, dOut_chunks, Wd, dWg=None, dWu=None,
                         dWd=None, ws=None, path=PATH_AUTO, stream=None):
    """Weight gradients from token chunks given in logical order; returns
    (dWg, dWu, dWd), equal to detffn_backward's for any chunking."""
    n = len(x_chunks)
    _bf16(Wd, dWg, dWu, dWd, *x_chunks, *gate_chunks, *up_chunks, *dOut_chunks)
    H, I = Wd.shape
    M = sum(int(t.shape[0]) for t in x_chunks)
    dev = Wd.device
    e = lambda *s: torch.empty(s, dtype=torch.bfloat16, device=dev)  # noqa: E731
    dWg = e(I, H) if dWg is None else dWg
    dWu = e(I, H) if dWu is None else dWu
    dWd = e(H, I) if dWd is None else dWd
    if ws is None:
        ws = workspace(OP_WGRAD_CHUNKED, M, H, I, 1, path, dev)
    toks = (_ll * n)(*[int(t.shape[0]) for t in x_chunks])
    arr = lambda ts: (_vp * n)(*[t.data_ptr() for t in ts])  # noqa: E731
    _check(lib().detffn_wgrad_chunked(handle(dev), n, toks, arr(x_chunks), arr(gate_chunks),
                                      arr(up_chunks), arr(dOut_chunks), _ptr(Wd), _ptr(dWg),
                                      _ptr(dWu), _ptr(dWd), H, I, _ptr(ws), ws.numel(),
                                      _stream(dev, stream), _opts(path)), "detffn_wgrad_chunked")
    return dWg, dWu, dWd


_DT = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}


def detffn_rank_tree_reduce(inputs, out=None, stream=None):
    """out = ((b0+b1)+(b2+b3))+... over 1, 2, 4 or 8 same-sized tensors (any
    alignment; out may be one of the inputs)."""
    n = len(inputs)
    dt = inputs[0].dtype
    count = inputs[0].numel()
    for t in inputs:
        if t.dtype != dt or t.numel() != count or not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors of one dtype and size")
    if out is None:
        out = torch.empty_like(inputs[0])
    ptrs = (_vp * n)(*[t.data_ptr() for t in inputs])
    with torch.cuda.device(inputs[0].device):
        _check(lib().detffn_rank_tree_reduce(ptrs, n, _ptr(out), count, _DT[dt],
                                             _stream(inputs[0].device, stream)),
               "detffn_rank_tree_reduce")
    return out


def detffn_tree_gemm(A, B, out=None, path=PATH_AUTO, stream=None, spin_limit=0, flags=0):
    """out[r, c] = T_K(A[r, :], B[c, :]) for 2-D strided bfloat16 views A [R,K], B [C,K]."""
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise ValueError("bfloat16 operands expected")
    R, K = A.shape
    C = B.shape[0]
    if out is None:
        out = torch.empty((R, C), dtype=torch.bfloat16, device=A.device)
    _check(lib().detffn_tree_gemm(handle(A.device), _ptr(A), A.stride(0), A.stride(1), _ptr(B),
                                  B.stride(0), B.stride(1), R, C, K, _ptr(out), out.stride(0),
                                  _stream(A.device, stream), _opts(path, 1, spin_limit, flags)),
           "detffn_tree_gemm")
    return out


def detffn_tree_gemm_leaves(A, B, out=None, leaves=None, stream=None):
    """The tensor family's contraction of detffn_tree_gemm, plus its FP32
    leaves: returns (out [R,C] bfloat16, leaves [R,C,L] float32)."""
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise ValueError("bfloat16 operands expected")
    R, K = A.shape
    C = B.shape[0]
    L = (K + 63) // 64
    if out is None:
        out = torch.empty((R, C), dtype=torch.bfloat16, device=A.device)
    if leaves is None:
        leaves = torch.empty((R, C, L), dtype=torch.float32, device=A.device)
    L_ = lib()
    L_.detffn_tree_gemm_leaves.argtypes = [_vp, _vp, _ll, _ll, _vp, _ll, _ll, _ll, _ll, _ll, _vp, _ll,
                                           _vp, _vp, ctypes.POINTER(Options)]
    L_.detffn_tree_gemm_leaves.restype = ctypes.c_int
    _check(L_.detffn_tree_gemm_leaves(handle(A.device), _ptr(A), A.stride(0), A.stride(1), _ptr(B),
                                      B.stride(0), B.stride(1), R, C, K, _ptr(out), out.stride(0),
                                      _ptr(leaves), _stream(A.device, stream), _opts(PATH_TENSOR)),
           "detffn_tree_gemm_leaves")
    return out, leaves


def detffn_cvt_f32_bf16(x, out=None, stream=None):
    """The kernels' own FP32 -> BF16 rounding applied to a float32 CUDA tensor
    (returns a bfloat16 tensor of the same shape)."""
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("contiguous CUDA float32 tensor expected")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    L = lib()
    L.detffn_cvt_f32_bf16.argtypes = [_vp, _vp, _vp, _ll, _vp]
    L.detffn_cvt_f32_bf16.restype = ctypes.c_int
    _check(L.detffn_cvt_f32_bf16(handle(x.device), _ptr(x), _ptr(out), x.numel(),
                                 _stream(x.device, stream)), "detffn_cvt_f32_bf16")
    return out


def detffn_silu_tables(device=None, host_only=False):
    """(silu_bf16 uint16 [65536], dsilu float32 [65536]) as numpy arrays; with
    host_only=True the library builds them without touching a GPU."""
    import numpy as np
    s = np.zeros(65536, np.uint16)
    d = np.zeros(65536, np.float32)
    h = None if host_only else handle(device)
    _check(lib().detffn_silu_tables(h, s.ctypes.data, d.ctypes.data), "detffn_silu_tables")
    return s, d


def detffn_get_status(device=None, stream=None):
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    return lib().detffn_get_status(handle(dev), _stream(dev, stream))


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int), ("ms", ctypes.c_double),
                ("bytes", ctypes.c_double), ("flops", ctypes.c_double)]


def detffn_profiling(enable, device=None):
    """Starts (clearing old records) or stops per-launch event timing."""
    L = lib()
    L.detffn_profiling.argtypes = [_vp, _int]
    L.detffn_profiling.restype = ctypes.c_int
    _check(L.detffn_profiling(handle(device), 1 if enable else 0), "detffn_profiling")


def detffn_profile_read(device=None):
    """{kernel name: dict(launches, ms, bytes, flops)} summed since profiling began."""
    L = lib()
    L.detffn_profile_read.argtypes = [_vp, _int, ctypes.POINTER(KernelTime), ctypes.POINTER(_int)]
    L.detffn_profile_read.restype = ctypes.c_int
    buf = (KernelTime * 64)()
    n = _int()
    _check(L.detffn_profile_read(handle(device), 64, buf, ctypes.byref(n)), "detffn_profile_read")
    return {buf[i].name.decode(): dict(launches=buf[i].launches, ms=buf[i].ms, bytes=buf[i].bytes,
                                       flops=buf[i].flops) for i in range(n.value)}


def detffn_forward_decode_noalloc(x, Wg, Wu, Wd, out=None, stream=None):
    """The decode forward (1 <= M <= 8) for callers that cannot allocate device
    memory: the library uses its own fixed scratch, so this call makes no
    allocation of its own (pass `out` to avoid the one for the result).
    Same bits as detffn_forward(path=PATH_EXACT).  Calls must not overlap on
    the GPU; the first call on a device does a one-time set-up."""
    _bf16(x, Wg, Wu, Wd, out)
    M, H = x.shape
    I = Wg.shape[0]
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    L = lib()
    L.detffn_forward_decode_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _ll, _ll, _ll, _vp]
    L.detffn_forward_decode_noalloc.restype = ctypes.c_int
    with torch.cuda.device(x.device):
        _check(L.detffn_forward_decode_noalloc(_ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(out),
                                               M, H, I, _stream(x.device, stream)),
               "detffn_forward_decode_noalloc")
    return out


def detffn_forward_decode_noalloc_status(device=None, stream=None):
    """Status of the last allocation-free decode forward on the device (OK or
    ERR_TIMEOUT); reading it clears it."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    L = lib()
    L.detffn_forward_decode_noalloc_status.argtypes = [_vp]
    L.detffn_forward_decode_noalloc_status.restype = ctypes.c_int
    with torch.cuda.device(dev):
        return L.detffn_forward_decode_noalloc_status(_stream(dev, stream))


def detffn_forward_decode_noalloc_test_waits(spin_limit=0, stall=0):
    """Test-only settings of the allocation-free decode forward's bounded
    waits: (0, 0) is the normal path; stall=1 makes its waits run out."""
    L = lib()
    L.detffn_forward_decode_noalloc_test_waits.argtypes = [_ll, ctypes.c_int]
    L.detffn_forward_decode_noalloc_test_waits.restype = ctypes.c_int
    _check(L.detffn_forward_decode_noalloc_test_waits(spin_limit, stall), "detffn_forward_decode_noalloc_test_waits")


def detffn_selfcheck_fused_schedule():
    """(shapes covered, failed cases) of the host check of the one-launch
    forward's schedule (no GPU needed)."""
    L = lib()
    L.detffn_selfcheck_fused_schedule.argtypes = [ctypes.POINTER(ctypes.c_ulonglong)] * 2
    L.detffn_selfcheck_fused_schedule.restype = ctypes.c_int
    c, n = ctypes.c_ulonglong(), ctypes.c_ulonglong()
    _check(L.detffn_selfcheck_fused_schedule(ctypes.byref(c), ctypes.byref(n)), "detffn_selfcheck_fused_schedule")
    return c.value, n.value


def detffn_selfcheck_pieces(max_levels=8):
    """Failed cases of the host check of the few-token kernels' piece
    decomposition and fold codes (no GPU needed)."""
    L = lib()
    L.detffn_selfcheck_pieces.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_ulonglong)]
    L.detffn_selfcheck_pieces.restype = ctypes.c_int
    n = ctypes.c_ulonglong()
    _check(L.detffn_selfcheck_pieces(int(max_levels), ctypes.byref(n)), "detffn_selfcheck_pieces")
    return n.value


def detffn_selfcheck_node_add(device=None):
    """Number of BF16 pairs where the device's packed add differs from the
    tree node rne_bf16(fp32(a) + fp32(b)) (exhaustive over 2^32 pairs)."""
    L = lib()
    L.detffn_selfcheck_node_add.argtypes = [_vp, ctypes.POINTER(ctypes.c_ulonglong)]
    L.detffn_selfcheck_node_add.restype = ctypes.c_int
    n = ctypes.c_ulonglong()
    _check(L.detffn_selfcheck_node_add(handle(device), ctypes.byref(n)), "detffn_selfcheck_node_add")
    return n.value
