#!/usr/bin/env python
"""Benchmark of the deterministic gated BF16 FFN on GB300 (libdetffn).

Step: one decode-shaped forward, M=32 tokens, H=4096, I=12288 (weights
~302 MB, larger than the 129 MB L2; two weight copies alternate between steps
so every step streams its weights from HBM).  `value` is the forward latency
in microseconds (max over ranks; lower is better).  The same run also reports
the M=1 and M=8 forward latencies and the M=32 forward+backward latency.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the only reference this build has:
the pages hold no code) on the same workload, the whole forward per step.  Under torchrun (N>1) each rank runs
an independent replica (the FFN itself runs on one GPU); rank 0 prints one
JSON line.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M_DEC, H, I = 32, 4096, 12288
METRIC = "det. FFN fwd / fwd+bwd latency (µs) and HBM GB/s, M=1/8/32, H=4096, I=12288"
WEIGHT_BYTES = 3 * H * I * 2
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {
    "tree_gemm_exact": "k_exact.cu",
    "decode_gateup": "k_decode.cu",
    "decode_down": "k_decode.cu",
    "tc_tree_gemm": "k_tc.cu",
    "tcs_gateup": "k_tcs.cu",
    "tcs_tree_gemm": "k_tcs.cu",
    "tcs_forward": "k_tcs.cu",
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK, "fallback"


def fwd_bytes(M):
    return WEIGHT_BYTES + 2 * M * H * 2


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            self.proc.wait(timeout=5)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def traffic_for(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None when the kernel source changed since the capture."""
    src = KERNEL_SOURCES.get(kernel)
    summ = os.path.join(ROOT, "profiles", "ncu_%s_%s.txt" % (kernel, workload))
    if not src or not os.path.exists(summ):
        return None
    with open(os.path.join(ROOT, "gemm_deterministic_bf16_gb300", "csrc", src), "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    rec = {}
    with open(summ) as f:
        for ln in f:
            if ":" in ln:
                k, v = ln.split(":", 1)
                rec[k.strip()] = v.strip()
    if rec.get("kernel_source_sha256") != sha:
        return None
    try:
        return float(rec["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def dist_setup(n_gpus):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, v):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


_ORACLE_INPUTS = {}


def _oracle_inputs(seed=0):
    from gemm_deterministic_bf16_gb300.inputs import ffn_inputs
    if seed not in _ORACLE_INPUTS:
        _ORACLE_INPUTS[seed] = ffn_inputs(M_DEC, H, I, seed=seed, with_dout=False)
    return _ORACLE_INPUTS[seed]


def oracle_forward_rows(rows, seed=0, nthreads=0):
    """Times the CPU oracle's forward on the first `rows` token rows of the
    M=32 decode workload (rows are independent); returns (seconds, out)."""
    import oracle
    d = _oracle_inputs(seed)
    t0 = time.perf_counter()
    r = oracle.ffn_forward(d["x"][:rows], d["Wg"], d["Wu"], d["Wd"], nthreads=nthreads)
    return time.perf_counter() - t0, r["out"]


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part", "processor\t: 0")) and ":" in ln:
                    v = ln.split(":", 1)[1].strip()
                    if v:
                        return v
    except OSError:
        pass
    return "unknown"


def run_reference(args):
    """The reference arm: the CPU oracle (the only reference the pages allow:
    they hold no code) running the whole M=32, H=4096, I=12288 forward each
    step on all host cores."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.lib()
    for _ in range(args.warmup):
        oracle_forward_rows(M_DEC)
    times = [oracle_forward_rows(M_DEC)[0] for _ in range(args.steps)]
    us = statistics.median(times) * 1e6
    sample = ("oracle (plain C, LANE8x8 leaves, all %d host threads): the whole M=32, H=4096, "
              "I=12288 forward each step (no extrapolation); CPU %s" % (host_cores(), cpu_model()))
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": "us", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) x, N(0,0.02) weights)",
            "config": {"workload": "decode forward M=32 H=4096 I=12288", "M": M_DEC, "H": H, "I": I},
            "cpu_baseline": {"value": us, "unit": "us", "cores": host_cores(), "kind": "oracle",
                             "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": us, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def bits_mismatch(a, b):
    """Elements whose bit patterns differ (two CUDA tensors of one shape)."""
    import torch
    ia = a.view(torch.int16) if a.element_size() == 2 else a.view(torch.int32)
    ib = b.view(torch.int16) if b.element_size() == 2 else b.view(torch.int32)
    return int((ia != ib).sum().item())


def large_training(G, args, ws_n, timed):
    """M=4096 (2 x 2048 tokens) forward and forward+backward on the default
    (tensor-core) family: TFLOP/s against 6*M*H*I and 18*M*H*I; the weight
    gradients from c = 2 and 4 token chunks, timed and compared bit for bit
    with the one-shot backward's."""
    import numpy as np
    import torch
    from gemm_deterministic_bf16_gb300.inputs import ffn_inputs
    M = 4096
    d = ffn_inputs(M, H, I, seed=7)
    t = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).cuda() for k, v in d.items()}
    e = lambda *s: torch.empty(s, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    out, g, u, dX = e(M, H), e(M, I), e(M, I), e(M, H)
    dWg, dWu, dWd = e(I, H), e(I, H), e(H, I)
    wsf = G.workspace(G.OP_FORWARD, M, H, I)
    wsb = G.workspace(G.OP_BACKWARD, M, H, I)

    def fwd(i):
        G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], out=out, gate_save=g, up_save=u, ws=wsf)

    def train(i):
        fwd(i)
        G.detffn_backward(t["x"], t["Wg"], t["Wu"], t["Wd"], g, u, t["dOut"], dX=dX, dWg=dWg, dWu=dWu,
                          dWd=dWd, ws=wsb)

    steps = max(3, args.steps // 4)
    fwd_ms = max_over_ranks(ws_n, timed(fwd, steps, 3))
    trn_ms = max_over_ranks(ws_n, timed(train, steps, 3))
    ref = [dWg.clone(), dWu.clone(), dWd.clone()]
    res = {}
    # Backward with the I axis in k = 2 shards, one stream and two-stream
    # dHidden (the gate contribution's rank tree beside the up shards).
    dX1 = dX.clone()
    wsk = G.workspace(G.OP_BACKWARD, M, H, I, 2)
    dXk = e(M, H)
    for name, fl in (("", 0), ("_overlap", G.FLAG_OVERLAP_DHIDDEN)):
        def bwd_k(i, fl=fl):
            G.detffn_backward(t["x"], t["Wg"], t["Wu"], t["Wd"], g, u, t["dOut"], dX=dXk, dWg=dWg, dWu=dWu,
                              dWd=dWd, ws=wsk, shards=2, flags=fl)
        res["bwd_ms_M4096_k2" + name] = max_over_ranks(ws_n, timed(bwd_k, steps, 3))
        torch.cuda.synchronize()
        res["dX_mismatches_M4096_k2" + name] = bits_mismatch(dXk, dX1)
    del wsk, dXk, dX1
    for c in (2, 4):
        sl = [slice(j * M // c, (j + 1) * M // c) for j in range(c)]
        xs, gs, us, ds = ([v[q] for q in sl] for v in (t["x"], g, u, t["dOut"]))
        wsc = G.workspace(G.OP_WGRAD_CHUNKED, M, H, I)
        cw = [e(I, H), e(I, H), e(H, I)]
        res["wgrad_chunked_ms_M4096_c%d" % c] = max_over_ranks(ws_n, timed(
            lambda i: G.detffn_wgrad_chunked(xs, gs, us, ds, t["Wd"], dWg=cw[0], dWu=cw[1], dWd=cw[2], ws=wsc),
            steps, 3))
        res["chunk_mismatches_M4096_c%d" % c] = sum(bits_mismatch(a, b) for a, b in zip(cw, ref))
        del xs, gs, us, ds, wsc, cw
    G.detffn_profiling(True)
    train(0)
    prof = G.detffn_profile_read()
    G.detffn_profiling(False)
    res.update({"fwd_ms_M4096": fwd_ms, "fwd_tflops_M4096": 6 * M * H * I / (fwd_ms * 1e-3) / 1e12,
                "fwd_bwd_ms_M4096": trn_ms,
                "fwd_bwd_tflops_M4096": 18 * M * H * I / (trn_ms * 1e-3) / 1e12,
                "kernels_M4096": {k: {"launches": v["launches"], "ms": v["ms"],
                                      "tflops": (v["flops"] / (v["ms"] * 1e-3) / 1e12) if v["flops"] else None,
                                      "gbs": v["bytes"] / (v["ms"] * 1e-3) / 1e9}
                                  for k, v in prof.items()}})
    del t, out, g, u, dX, dWg, dWu, dWd, wsf, wsb, ref
    torch.cuda.empty_cache()
    return res


L2_BYTES = 129 << 20


def rank_tree_rows(G, args):
    """The balanced rank tree over n in {2, 4, 8} buffers of 4 KiB, 64 KiB,
    1 MiB and 16 MiB in FP32, FP16 and BF16, plus 16 MiB offset views
    (+1, +2, +3 elements) with odd tails.  Each row replays a CUDA graph of
    `reps` calls, cycling over enough buffer sets that a 16 MiB row's sets
    exceed twice the L2 (so they stream from HBM); the time per call is the
    kernel's plus the graph's launch gap, free of the host's per-call cost.
    16 MiB rows report GB/s of (n+1)*S bytes and the fraction of HBM peak."""
    import torch
    pk, _ = peaks()
    rows = {}
    reps = 24
    cases = [(dt, S, n, 0, 0) for dt in ("f32", "f16", "bf16") for S in (4 << 10, 64 << 10, 1 << 20, 16 << 20)
             for n in (2, 4, 8)]
    cases += [(dt, 16 << 20, 8, off, 1) for dt in ("f16", "bf16") for off in (1, 2, 3)]
    cases += [("f32", 16 << 20, 8, 1, 1)]
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
    for dt, S, n, off, tail in cases:
        esz = 4 if dt == "f32" else 2
        count = S // esz - tail
        nsets = 2
        if S >= 16 << 20:
            nsets = max(2, -(-2 * L2_BYTES // ((n + 1) * S)))
        sets = []
        for _ in range(nsets):
            ins = [torch.randn(count + off, device="cuda").to(tdt[dt])[off:] for _ in range(n)]
            out = torch.empty(count + off, dtype=tdt[dt], device="cuda")[off:]
            sets.append((ins, out))
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for ins, out in sets:
                G.detffn_rank_tree_reduce(ins, out=out)
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(reps):
                G.detffn_rank_tree_reduce(sets[i % nsets][0], out=sets[i % nsets][1])
        graph.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        nrep = 4
        a.record()
        for _ in range(nrep):
            graph.replay()
        b.record()
        torch.cuda.synchronize()
        us = 1e3 * a.elapsed_time(b) / (nrep * reps)
        row = {"us": us}
        if S >= 16 << 20:
            gbs = (n + 1) * count * esz / (us * 1e-6) / 1e9
            row.update({"gbs": gbs, "frac_hbm": gbs / pk["hbm_gbs"], "buffer_sets": nsets})
        name = "%s_n%d_%dKiB" % (dt, n, S >> 10) + ("_off%d_tail" % off if off or tail else "")
        rows[name] = row
        del sets, graph
    torch.cuda.empty_cache()
    return rows


def run_ours(args):
    import numpy as np
    import torch

    import gemm_deterministic_bf16_gb300 as G
    from gemm_deterministic_bf16_gb300 import build as libbuild
    from gemm_deterministic_bf16_gb300.inputs import ffn_inputs

    ws_n, rank, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    # One rank compiles (the others would race on the same object files);
    # the rest load the library once it is there.
    if rank == 0:
        libbuild.build()
    barrier(ws_n)
    path = {"auto": G.PATH_AUTO, "exact": G.PATH_EXACT, "tensor": G.PATH_TENSOR}[args.path]

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    # Two weight copies, alternated per step: every step streams 302 MB from HBM.
    copies = []
    for c in range(2):
        d = ffn_inputs(M_DEC, H, I, seed=100 * rank + c)
        copies.append({k: dev(v) for k, v in d.items()})
    stream = torch.cuda.current_stream()

    def fwd(M, c, out, ws, pth=None, flags=0):
        t = copies[c]
        G.detffn_forward(t["x"][:M], t["Wg"], t["Wu"], t["Wd"], out=out, ws=ws, path=path if pth is None else pth,
                         flags=flags)

    def timed(fn, steps, warmup):
        for i in range(warmup):
            fn(i)
        torch.cuda.synchronize()
        barrier(ws_n)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(steps):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps  # ms per step

    outs = {M: torch.empty(M, H, dtype=torch.bfloat16, device="cuda") for M in (1, 8, 32)}
    wss = {M: G.workspace(G.OP_FORWARD, M, H, I, 1, path) for M in (1, 8, 32)}

    # Headline: M=32 forward.
    with Clocks(local) as clk:
        ms = timed(lambda i: fwd(M_DEC, i & 1, outs[M_DEC], wss[M_DEC]), args.steps, args.warmup)
    ms = max_over_ranks(ws_n, ms)
    us = ms * 1e3

    # Per-op durations from events on the launching stream (the same loop
    # with per-op event pairs: each op is then timed alone, without the
    # programmatic-dependent overlap of the chained launches).
    G.detffn_profiling(True)
    for i in range(args.steps):
        fwd(M_DEC, i & 1, outs[M_DEC], wss[M_DEC])
    prof = G.detffn_profile_read()
    G.detffn_profiling(False)
    launches = sum(v["launches"] for v in prof.values()) // max(1, args.steps)
    top = max(prof.items(), key=lambda kv: kv[1]["ms"])
    pk, how = peaks()
    kname, kv = top
    op_ms = kv["ms"] / args.steps
    op_bytes = kv["bytes"] / args.steps
    step_gbs = fwd_bytes(M_DEC) / (us * 1e-6) / 1e9
    if len(prof) == 1 and launches == 1:
        # The step is this one kernel: its average duration over the timed
        # region is the step time (consecutive launches chained as in use).
        duration_ms, source = ms, "timed_region"
    else:
        # Several kernels per step: this kernel's time from its own event pair.
        duration_ms, source = op_ms, "op_alone"
    achieved = op_bytes / (duration_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                "traffic": traffic_for(kname, "decode_m32"), "peak_source": how,
                "duration_us": duration_ms * 1e3, "duration_source": source,
                "op_us_alone": op_ms * 1e3, "algorithmic_bytes_per_op": op_bytes,
                "share": kv["ms"] / sum(v["ms"] for v in prof.values()),
                "step_achieved": step_gbs, "step_frac": step_gbs / pk["hbm_gbs"]}

    extra = {}
    # Other decode sizes, and each family at every decode size.
    for M in (1, 8):
        extra["fwd_us_M%d" % M] = 1e3 * max_over_ranks(
            ws_n, timed(lambda i, M=M: fwd(M, i & 1, outs[M], wss[M]), args.steps, args.warmup))
        extra["fwd_gbs_M%d" % M] = fwd_bytes(M) / (extra["fwd_us_M%d" % M] * 1e-6) / 1e9
    for M in (1, 8, 32):
        for name, pth in (("tensor", G.PATH_TENSOR), ("exact", G.PATH_EXACT)):
            wsm = G.workspace(G.OP_FORWARD, M, H, I, 1, pth)
            extra["fwd_us_M%d_%s" % (M, name)] = 1e3 * max_over_ranks(ws_n, timed(
                lambda i, M=M, pth=pth, wsm=wsm: fwd(M, i & 1, outs[M], wsm, pth), args.steps, args.warmup))
            del wsm
        # The tensor family's two-launch form of the same forward (same bits).
        extra["fwd_us_M%d_two_launch" % M] = 1e3 * max_over_ranks(ws_n, timed(
            lambda i, M=M: fwd(M, i & 1, outs[M], wss[M], G.PATH_TENSOR, G.FLAG_SPLIT_FORWARD), args.steps,
            args.warmup))

    # The M=32 training step (forward with saves + backward), unsharded and
    # with the I axis in k = 2, 4, 8 shards (tensor-parallel emulation: shard
    # partials combined by the rank tree); the shards' outputs are compared
    # bit for bit with the unsharded call's.
    e = lambda *s: torch.empty(s, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    tsteps = max(3, args.steps // 4)
    base = None
    for k in (1, 2, 4, 8):
        gs, us_, outk, dXk = e(M_DEC, I), e(M_DEC, I), e(M_DEC, H), e(M_DEC, H)
        grads = [e(I, H), e(I, H), e(H, I)]
        wsf = G.workspace(G.OP_FORWARD_SHARDED if k > 1 else G.OP_FORWARD, M_DEC, H, I, k, path)
        wsb = G.workspace(G.OP_BACKWARD, M_DEC, H, I, k, path)

        def train_step(i, k=k, gs=gs, us_=us_, outk=outk, dXk=dXk, grads=grads, wsf=wsf, wsb=wsb, flags=0):
            t = copies[i & 1]
            if k == 1:
                G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], out=outk, gate_save=gs, up_save=us_, ws=wsf,
                                 path=path)
            else:
                G.detffn_forward_sharded(t["x"], t["Wg"], t["Wu"], t["Wd"], k, out=outk, gate_save=gs,
                                         up_save=us_, ws=wsf, path=path)
            G.detffn_backward(t["x"], t["Wg"], t["Wu"], t["Wd"], gs, us_, t["dOut"], dX=dXk, dWg=grads[0],
                              dWu=grads[1], dWd=grads[2], ws=wsb, shards=k, path=path, flags=flags)

        key = "fwd_bwd_us_M32" + ("" if k == 1 else "_k%d" % k)
        if k > 1:
            # The same step with the gate contribution's rank tree on a second
            # stream (two-stream dHidden); its results are compared below too.
            ov = lambda i, ts=train_step: ts(i, flags=G.FLAG_OVERLAP_DHIDDEN)  # noqa: E731
            extra[key + "_overlap"] = 1e3 * max_over_ranks(ws_n, timed(ov, tsteps, 3))
            ov(0)
            torch.cuda.synchronize()
            extra["overlap_mismatches_M32_k%d" % k] = {
                n: bits_mismatch(a, b) for n, a, b in zip(["out", "dX", "dWg", "dWu", "dWd"], [outk, dXk] + grads,
                                                          base)}
        extra[key] = 1e3 * max_over_ranks(ws_n, timed(train_step, tsteps, 3))
        train_step(0)   # copy 0 last, for the comparison
        torch.cuda.synchronize()
        res = [outk, dXk] + grads
        if base is None:
            base = [r.clone() for r in res]
            extra["fwd_bwd_gbs_M32"] = 3 * WEIGHT_BYTES / (extra[key] * 1e-6) / 1e9
        else:
            extra["shard_mismatches_M32_k%d" % k] = {n: bits_mismatch(a, b) for n, a, b in
                                                     zip(["out", "dX", "dWg", "dWu", "dWd"], res, base)}
        del gs, us_, outk, dXk, grads, wsf, wsb, res
    del base
    torch.cuda.empty_cache()
    extra["rank_tree"] = rank_tree_rows(G, args)
    if not args.no_large:
        extra.update(large_training(G, args, ws_n, timed))

    # End to end through the public API: every step's x comes from pinned
    # host memory and its out goes back to pinned host memory.  The headline
    # is the C-ABI call on the host buffers themselves (DETFFN_FLAG_HOST_IO:
    # the library's copy kernels move x in and out over the host link); the
    # same step with the copies made by torch around a device-buffer call is
    # reported beside it.
    xh = torch.empty(M_DEC, H, dtype=torch.bfloat16).pin_memory()
    xh.copy_(copies[0]["x"].cpu())
    oh = torch.empty(M_DEC, H, dtype=torch.bfloat16).pin_memory()
    xd = torch.empty(M_DEC, H, dtype=torch.bfloat16, device="cuda")
    ws_hio = G.workspace(G.OP_FORWARD, M_DEC, H, I, 1, path, flags=G.FLAG_HOST_IO)

    def e2e_step(i):
        t = copies[i & 1]
        G.detffn_forward(xh, t["Wg"], t["Wu"], t["Wd"], out=oh, ws=ws_hio, path=path, flags=G.FLAG_HOST_IO)

    def e2e_torch_step(i):
        t = copies[i & 1]
        xd.copy_(xh, non_blocking=True)
        G.detffn_forward(xd, t["Wg"], t["Wu"], t["Wd"], out=outs[M_DEC], ws=wss[M_DEC], path=path)
        oh.copy_(outs[M_DEC], non_blocking=True)

    e2e_us = 1e3 * max_over_ranks(ws_n, timed(e2e_step, args.steps, args.warmup))
    torch.cuda.synchronize()
    e2e_out = oh.clone()
    extra["e2e_torch_copies_us"] = 1e3 * max_over_ranks(ws_n, timed(e2e_torch_step, args.steps, args.warmup))
    torch.cuda.synchronize()
    extra["e2e_host_io_mismatches"] = bits_mismatch(e2e_out, oh)

    cpu = None
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        # The oracle on the same workload: the whole M=32 forward on all host
        # cores, and one token row on one core (scaled by 32, labelled so).
        # Its output rows are compared with this run's (the default family).
        t_all, ref_out = oracle_forward_rows(M_DEC, seed=0)
        t_one, _ = oracle_forward_rows(1, seed=0, nthreads=1)
        fwd(M_DEC, 0, outs[M_DEC], wss[M_DEC])
        got = outs[M_DEC].cpu().view(torch.int16).numpy().view(np.uint16)
        key = lambda u: np.where(u & 0x8000, -(u.astype(np.int32) & 0x7FFF), u.astype(np.int32))  # noqa: E731
        dist = np.abs(key(got) - key(ref_out))
        cpu = {"value": t_all * 1e6, "unit": "us", "cores": host_cores(), "kind": "oracle",
               "sample": "the whole M=32, H=4096, I=12288 forward, once, on all host cores",
               "cpu_model": cpu_model(),
               "single_thread_us_extrapolated": t_one * 1e6 * M_DEC,
               "single_thread_sample": "one token row on one core, scaled by 32",
               "gpu_vs_oracle": {"family": args.path, "elements": int(dist.size),
                                 "mismatches": int(np.count_nonzero(dist)),
                                 "over_1ulp": int(np.count_nonzero(dist > 1)), "max_ulp": int(dist.max())}}

    if rank == 0:
        line = {"metric": METRIC, "value": us, "unit": "us", "n_gpus": ws_n, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic (seeded N(0,1) x and dOut, N(0,0.02) weights, [out,in] layout)",
                "config": {"workload": "decode forward M=32 H=4096 I=12288", "M": M_DEC, "H": H,
                           "I": I, "path": args.path,
                           "l2": "weights 302 MB > 129 MB L2, two copies alternated per step",
                           "replicas": ws_n},
                "hbm_gbs": step_gbs,
                "roofline": roofline, "cpu_baseline": cpu,
                "e2e": {"value": e2e_us, "unit": "us", "h2d_bytes_per_step": M_DEC * H * 2,
                        "d2h_bytes_per_step": M_DEC * H * 2},
                "gpu_launches": launches * args.steps, "clocks": clk.summary(),
                "kernels": {k: {"launches_per_step": v["launches"] // max(1, args.steps),
                                "us_per_step": 1e3 * v["ms"] / max(1, args.steps)}
                            for k, v in prof.items()},
                "extra": extra}
        print(json.dumps(line))
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_profile_case(args):
    """A few forwards of one size and nothing else: the command ncu captures."""
    import numpy as np
    import torch

    import gemm_deterministic_bf16_gb300 as G
    from gemm_deterministic_bf16_gb300 import build as libbuild
    from gemm_deterministic_bf16_gb300.inputs import ffn_inputs
    libbuild.build()
    if args.profile_case.startswith("rt"):
        # Rank tree: n = int(suffix) BF16 buffers of 16 MiB, --steps calls.
        n = int(args.profile_case[2:])
        bufs = [torch.randn(8 << 20, device="cuda").to(torch.bfloat16) for _ in range(n)]
        out = torch.empty_like(bufs[0])
        for _ in range(args.steps):
            G.detffn_rank_tree_reduce(bufs, out=out)
        torch.cuda.synchronize()
        print("profile case %s done" % args.profile_case)
        return 0
    kind, M = args.profile_case[:3], int(args.profile_case[3:])
    path = {"auto": G.PATH_AUTO, "exact": G.PATH_EXACT, "tensor": G.PATH_TENSOR}[args.path]
    d = ffn_inputs(M, H, I, seed=0, with_dout=(kind == "trn"))
    t = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).cuda() for k, v in d.items()}
    for _ in range(args.steps):
        if kind == "fwd":
            G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], path=path)
        else:
            g = torch.empty(M, I, dtype=torch.bfloat16, device="cuda")
            u = torch.empty_like(g)
            G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], gate_save=g, up_save=u, path=path)
            G.detffn_backward(t["x"], t["Wg"], t["Wu"], t["Wd"], g, u, t["dOut"], path=path)
    torch.cuda.synchronize()
    print("profile case %s done" % args.profile_case)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--path", choices=["auto", "exact", "tensor"], default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-large", action="store_true", help="skip the M=4096 training measurement")
    ap.add_argument("--profile-case", default=None,
                    help="fwdM or trnM (e.g. fwd8): run --steps forwards (or training steps) "
                         "of M tokens only; rtN: --steps rank-tree calls over N 16 MiB BF16 "
                         "buffers; for profiler captures")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.profile_case:
        return run_profile_case(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
