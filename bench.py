#!/usr/bin/env python
"""Benchmark of the deterministic gated BF16 FFN on GB300 (libdetffn).

Step: one decode-shaped forward, M=32 tokens, H=4096, I=12288 (weights
~302 MB, larger than the 129 MB L2; two weight copies alternate between steps
so every step streams its weights from HBM).  `value` is the forward latency
in microseconds (max over ranks; lower is better).  The same run also reports
the M=1 and M=8 forward latencies and the M=32 forward+backward latency.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the only reference this build has) on
a bounded sample of the same workload.  Under torchrun (N>1) each rank runs
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


def oracle_forward_rows(rows, seed=0):
    """Times the CPU oracle on `rows` token rows of the M=32 decode forward
    (rows are independent, so the M=32 latency scales by 32/rows)."""
    import oracle
    from gemm_deterministic_bf16_gb300.inputs import ffn_inputs
    if seed not in _ORACLE_INPUTS:
        _ORACLE_INPUTS[seed] = ffn_inputs(M_DEC, H, I, seed=seed, with_dout=False)
    d = _ORACLE_INPUTS[seed]
    t0 = time.perf_counter()
    oracle.ffn_forward(d["x"][:rows], d["Wg"], d["Wu"], d["Wd"])
    return time.perf_counter() - t0


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.lib()
    rows = args.ref_rows
    for _ in range(args.warmup):
        oracle_forward_rows(rows)
    times = [oracle_forward_rows(rows) for _ in range(args.steps)]
    us = statistics.median(times) * 1e6 * M_DEC / rows
    sample = ("oracle (plain C, LANE8x8 leaves, all host threads) on %d of the 32 token rows of "
              "the M=32, H=4096, I=12288 forward per step, scaled by 32/%d" % (rows, rows))
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": "us", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) x, N(0,0.02) weights)",
            "config": {"workload": "decode forward M=32 H=4096 I=12288", "M": M_DEC, "H": H, "I": I},
            "cpu_baseline": {"value": us, "unit": "us", "cores": host_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": us, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def large_training(G, args, ws_n, timed):
    """M=4096 (2 x 2048 tokens) forward and forward+backward on the default
    (tensor-core) family: TFLOP/s against 6*M*H*I and 18*M*H*I."""
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
    # Weight gradients with the tokens given as c chunks in logical order (the
    # same bits as the one-shot backward's).
    chunked = {}
    for c in (2, 4):
        sl = [slice(j * M // c, (j + 1) * M // c) for j in range(c)]
        xs, gs, us, ds = ([v[q].contiguous() for q in sl] for v in (t["x"], g, u, t["dOut"]))
        wsc = G.workspace(G.OP_WGRAD_CHUNKED, M, H, I)
        chunked["wgrad_chunked_ms_M4096_c%d" % c] = max_over_ranks(ws_n, timed(
            lambda i: G.detffn_wgrad_chunked(xs, gs, us, ds, t["Wd"], dWg=dWg, dWu=dWu, dWd=dWd, ws=wsc),
            steps, 3))
        del xs, gs, us, ds, wsc
    G.detffn_profiling(True)
    train(0)
    prof = G.detffn_profile_read()
    G.detffn_profiling(False)
    res = dict(chunked)
    res.update({"fwd_ms_M4096": fwd_ms, "fwd_tflops_M4096": 6 * M * H * I / (fwd_ms * 1e-3) / 1e12,
           "fwd_bwd_ms_M4096": trn_ms, "fwd_bwd_tflops_M4096": 18 * M * H * I / (trn_ms * 1e-3) / 1e12,
           "kernels_M4096": {k: {"launches": v["launches"], "ms": v["ms"],
                                 "tflops": (v["flops"] / (v["ms"] * 1e-3) / 1e12) if v["flops"] else None,
                                 "gbs": v["bytes"] / (v["ms"] * 1e-3) / 1e9}
                             for k, v in prof.items()}})
    del t, out, g, u, dX, dWg, dWu, dWd, wsf, wsb
    torch.cuda.empty_cache()
    return res


def rank_tree_rows(G, args, ws_n, timed):
    """The balanced rank tree over n buffers of S bytes: microseconds per call,
    and for 16 MiB buffers (larger than L2 in total) GB/s of (n+1)*S bytes."""
    import torch
    pk, _ = peaks()
    rows = {}
    steps = max(5, args.steps)
    for dt, name in ((torch.float32, "f32"), (torch.bfloat16, "bf16")):
        esz = torch.tensor([], dtype=dt).element_size()
        for S in (4 << 10, 1 << 20, 16 << 20):
            for n in (2, 4, 8):
                bufs = [torch.randn(S // esz, device="cuda").to(dt) for _ in range(n)]
                out = torch.empty_like(bufs[0])
                us = 1e3 * max_over_ranks(ws_n, timed(lambda i: G.detffn_rank_tree_reduce(bufs, out=out), steps, 3))
                row = {"us": us}
                if S >= 16 << 20:
                    gbs = (n + 1) * S / (us * 1e-6) / 1e9
                    row.update({"gbs": gbs, "frac_hbm": gbs / pk["hbm_gbs"]})
                rows["%s_n%d_%dKiB" % (name, n, S >> 10)] = row
                del bufs, out
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

    def fwd(M, c, out, ws):
        t = copies[c]
        G.detffn_forward(t["x"][:M], t["Wg"], t["Wu"], t["Wd"], out=out, ws=ws, path=path)

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

    # Per-kernel durations from events on the launching stream (same loop, profiling on).
    G.detffn_profiling(True)
    for i in range(args.steps):
        fwd(M_DEC, i & 1, outs[M_DEC], wss[M_DEC])
    prof = G.detffn_profile_read()
    G.detffn_profiling(False)
    launches = sum(v["launches"] for v in prof.values()) // max(1, args.steps)
    top = max(prof.items(), key=lambda kv: kv[1]["ms"])
    pk, how = peaks()
    kname, kv = top
    per_launch_ms = kv["ms"] / kv["launches"]
    bytes_per_launch = kv["bytes"] / kv["launches"]
    achieved = bytes_per_launch / (per_launch_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                "traffic": traffic_for(kname, "decode_m32"), "peak_source": how,
                "share": kv["ms"] / sum(v["ms"] for v in prof.values()),
                "algorithmic_bytes_per_launch": bytes_per_launch}

    # Other decode sizes and the M=32 training step (forward with saves + backward).
    extra = {}
    for M in (1, 8):
        extra["fwd_us_M%d" % M] = 1e3 * max_over_ranks(
            ws_n, timed(lambda i, M=M: fwd(M, i & 1, outs[M], wss[M]), args.steps, args.warmup))
        extra["fwd_gbs_M%d" % M] = fwd_bytes(M) / (extra["fwd_us_M%d" % M] * 1e-6) / 1e9
    gsave = torch.empty(M_DEC, I, dtype=torch.bfloat16, device="cuda")
    usave = torch.empty_like(gsave)
    grads = [torch.empty(I, H, dtype=torch.bfloat16, device="cuda") for _ in range(2)] + \
        [torch.empty(H, I, dtype=torch.bfloat16, device="cuda")]
    dX = torch.empty(M_DEC, H, dtype=torch.bfloat16, device="cuda")
    wsb = G.workspace(G.OP_BACKWARD, M_DEC, H, I, 1, path)
    wsf = G.workspace(G.OP_FORWARD, M_DEC, H, I, 1, path)

    def train_step(i):
        t = copies[i & 1]
        G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], out=outs[M_DEC], gate_save=gsave,
                         up_save=usave, ws=wsf, path=path)
        G.detffn_backward(t["x"], t["Wg"], t["Wu"], t["Wd"], gsave, usave, t["dOut"], dX=dX,
                          dWg=grads[0], dWu=grads[1], dWd=grads[2], ws=wsb, path=path)

    tsteps = max(3, args.steps // 4)
    extra["fwd_bwd_us_M32"] = 1e3 * max_over_ranks(ws_n, timed(train_step, tsteps, 3))
    extra["fwd_bwd_gbs_M32"] = 3 * WEIGHT_BYTES / (extra["fwd_bwd_us_M32"] * 1e-6) / 1e9

    # The M=32 forward on the tensor-core family (leaves in the hardware's order).
    wst = G.workspace(G.OP_FORWARD, M_DEC, H, I, 1, G.PATH_TENSOR)

    def fwd_tc(i):
        t = copies[i & 1]
        G.detffn_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], out=outs[M_DEC], ws=wst, path=G.PATH_TENSOR)

    extra["fwd_us_M32_tensor"] = 1e3 * max_over_ranks(ws_n, timed(fwd_tc, args.steps, args.warmup))
    extra["fwd_gbs_M32_tensor"] = fwd_bytes(M_DEC) / (extra["fwd_us_M32_tensor"] * 1e-6) / 1e9
    # Each family at the other decode sizes (AUTO takes one of them by M).
    for M in (1, 8):
        for name, pth in (("tensor", G.PATH_TENSOR), ("exact", G.PATH_EXACT)):
            wsm = G.workspace(G.OP_FORWARD, M, H, I, 1, pth)
            us_m = 1e3 * max_over_ranks(ws_n, timed(
                lambda i, M=M, pth=pth, wsm=wsm: G.detffn_forward(copies[i & 1]["x"][:M], copies[i & 1]["Wg"],
                                                                  copies[i & 1]["Wu"], copies[i & 1]["Wd"],
                                                                  out=outs[M], ws=wsm, path=pth),
                args.steps, args.warmup))
            extra["fwd_us_M%d_%s" % (M, name)] = us_m
    # The M=32 training step with the I axis in k=8 shards (tensor-parallel
    # emulation: shard partials combined by the rank tree; the same bits).
    wsf8 = G.workspace(G.OP_FORWARD_SHARDED, M_DEC, H, I, 8, path)
    wsb8 = G.workspace(G.OP_BACKWARD, M_DEC, H, I, 8, path)

    def train_step_k8(i):
        t = copies[i & 1]
        G.detffn_forward_sharded(t["x"], t["Wg"], t["Wu"], t["Wd"], 8, out=outs[M_DEC], gate_save=gsave,
                                 up_save=usave, ws=wsf8, path=path)
        G.detffn_backward(t["x"], t["Wg"], t["Wu"], t["Wd"], gsave, usave, t["dOut"], dX=dX,
                          dWg=grads[0], dWu=grads[1], dWd=grads[2], ws=wsb8, shards=8, path=path)

    extra["fwd_bwd_us_M32_k8"] = 1e3 * max_over_ranks(ws_n, timed(train_step_k8, tsteps, 3))
    extra["rank_tree"] = rank_tree_rows(G, args, ws_n, timed)
    if not args.no_large:
        extra.update(large_training(G, args, ws_n, timed))

    # End to end through the public API: pinned host x in, host out back, every step.
    xh = torch.empty(M_DEC, H, dtype=torch.bfloat16).pin_memory()
    xh.copy_(copies[0]["x"].cpu())
    oh = torch.empty(M_DEC, H, dtype=torch.bfloat16).pin_memory()
    xd = torch.empty(M_DEC, H, dtype=torch.bfloat16, device="cuda")

    def e2e_step(i):
        t = copies[i & 1]
        xd.copy_(xh, non_blocking=True)
        G.detffn_forward(xd, t["Wg"], t["Wu"], t["Wd"], out=outs[M_DEC], ws=wss[M_DEC], path=path)
        oh.copy_(outs[M_DEC], non_blocking=True)

    e2e_us = 1e3 * max_over_ranks(ws_n, timed(e2e_step, args.steps, args.warmup))

    cpu = None
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        t = oracle_forward_rows(args.ref_rows)
        cpu = {"value": t * 1e6 * M_DEC / args.ref_rows, "unit": "us", "cores": host_cores(),
               "kind": "oracle",
               "sample": "one oracle forward on %d of the 32 token rows, scaled by 32/%d"
                         % (args.ref_rows, args.ref_rows)}

    if rank == 0:
        line = {"metric": METRIC, "value": us, "unit": "us", "n_gpus": ws_n, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic (seeded N(0,1) x and dOut, N(0,0.02) weights, [out,in] layout)",
                "config": {"workload": "decode forward M=32 H=4096 I=12288", "M": M_DEC, "H": H,
                           "I": I, "path": args.path,
                           "l2": "weights 302 MB > 129 MB L2, two copies alternated per step",
                           "replicas": ws_n},
                "hbm_gbs": fwd_bytes(M_DEC) / (us * 1e-6) / 1e9,
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
    ap.add_argument("--ref-rows", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-large", action="store_true", help="skip the M=4096 training measurement")
    ap.add_argument("--profile-case", default=None,
                    help="fwdM or trnM (e.g. fwd8): run --steps forwards (or training steps) "
                         "of M tokens only, for profiler captures")
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
