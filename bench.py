#!/usr/bin/env python3
"""Benchmark of the dropless MoE layer forward on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                [--config mixtral|dsv3|qwen|skew|tiny] [--precision bf16|mxfp8]

One step = one pass of the whole forward (router logits, top-K routing +
histogram/scan/dispatch order, permute, grouped GEMM1 + SwiGLU, grouped GEMM2,
weighted unpermute/combine) over one batch of T tokens, through the C ABI.
Default workload: the Mixtral-8x7B-shaped layer (T=8192, d=4096, E=8, K=2,
f=14336), seeded synthetic bf16 data.  Under torchrun every rank runs an
independent replica on its own tokens (the forward has no cross-token
dependency, so there is no collective): weak scaling.

Prints one JSON line (rank 0).  `value` is useful TFLOP/s = 6*T*K*d*f per
step (only the valid rows of the two grouped GEMMs count), aggregated over
ranks; per-kernel durations come from CUDA events on the launching stream
inside the timed region.  `--impl reference` times the oracle (plain CPU
implementation, fp64) on a bounded sample of the same workload.

`--precision mxfp8` runs the expert matmuls with MXFP8 block scaling (E4M3
elements, one UE8M0 scale per 32 along K): the expert weights are quantised
once before the timed region (as a training step reuses them), the token
activations inside every step (fused into the permute), and h inside GEMM1's
epilogue.  Its roofline peak is the measured bf16 peak times the nominal
fp8 / bf16 tensor ratio (2).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import DESCRIPTIONS, make_tokens, make_weights, shape  # noqa: E402

STEP_NAMES = ["router_logits", "route", "permute", "grouped_gemm1_swiglu", "grouped_gemm2", "unpermute"]
KERNELS_PER_STEP = 9


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def _traffic_record(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    this workload and the kernel's source has not changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    rec = d.get(kernel)
    if not rec or rec.get("workload") != workload:
        return None
    # the hash covers every source file the kernel is built from
    srcs = rec["source"] if isinstance(rec["source"], list) else [rec["source"]]
    digest = hashlib.sha256()
    for src in srcs:
        with open(os.path.join(ROOT, src), "rb") as fh:
            digest.update(fh.read())
    if digest.hexdigest()[:16] != rec.get("source_sha256_16"):
        return None
    return rec


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        reasons = set()
        for r in rows:
            for name, val in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"],
                                 r[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(v: float, ws: int, device="cuda") -> float:
    """The slowest rank's time: the whole job is done when every replica is."""
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(rank: int) -> int:
    """Token seed of a replica: every rank forwards its own batch of T tokens
    (the weights, seed 0, are the same on every rank)."""
    return rank


def aggregate(work_per_step: float, ws: int, steps: int, elapsed_ms_max: float) -> float:
    """Whole-job rate: the work of all ranks' steps over the slowest rank's time."""
    return work_per_step * ws * steps / (elapsed_ms_max * 1e-3)


# ------------------------------------------------------------------ oracle timing
def _oracle_sample_run(s, x_np, Wr_np, bias_np, W1_np, W2_np, n_tok: int, nthreads: int):
    import oracle
    t0 = time.perf_counter()
    oracle.forward(x_np[:n_tok], Wr_np, bias_np, W1_np, W2_np, s.K, nthreads=nthreads)
    return time.perf_counter() - t0


def _oracle_inputs(s, x, w):
    """Host copies of the layer (weights in fp64 when host memory allows, which
    the oracle then uses as they are)."""
    try:
        avail = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError, AttributeError):
        avail = 0
    f64_bytes = 8 * s.E * 3 * s.d * s.f
    wdtype = np.float64 if avail > 3 * f64_bytes else np.float32
    x_np = x.float().cpu().numpy()
    Wr_np = w.Wr.cpu().numpy()
    bias_np = w.bias.cpu().numpy()
    W1_np = np.empty((s.E, 2 * s.f, s.d), wdtype)
    W2_np = np.empty((s.E, s.d, s.f), wdtype)
    for e in range(s.E):
        W1_np[e] = w.W1[e].float().cpu().numpy()
        W2_np[e] = w.W2[e].float().cpu().numpy()
    return x_np, Wr_np, bias_np, W1_np, W2_np, np.dtype(wdtype).name


def _oracle_rate(s, inputs, budget_s: float, nthreads: int):
    """Times the oracle on the first n tokens, n sized for about budget_s."""
    x_np, Wr_np, bias_np, W1_np, W2_np, _ = inputs
    n = min(16, s.T)
    t = _oracle_sample_run(s, x_np, Wr_np, bias_np, W1_np, W2_np, n, nthreads)
    # grow the sample until one run takes about the budget (the oracle has a
    # fixed cost per expert, so a single small run underestimates the rate)
    while t < 0.5 * budget_s and n < s.T:
        n = int(min(s.T, max(2 * n, n * 0.8 * budget_s / max(t, 1e-9))))
        t = _oracle_sample_run(s, x_np, Wr_np, bias_np, W1_np, W2_np, n, nthreads)
    return n, t


def run_reference(args):
    ws, rank, local = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return
    import oracle
    s = shape(args.config)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = make_weights(s, seed=0, device=dev)
    x = make_tokens(s, seed=0, device=dev)
    inputs = _oracle_inputs(s, x, w)
    del w, x
    nthreads = oracle.host_threads()
    steps, warm = args.steps, args.warmup
    budget = max(1.0, 90.0 / max(1, steps + warm))
    x_np, Wr_np, bias_np, W1_np, W2_np, wdt = inputs
    # size the per-step sample from one calibration run
    n0 = min(16, s.T)
    t0 = _oracle_sample_run(s, x_np, Wr_np, bias_np, W1_np, W2_np, n0, nthreads)
    n = int(max(1, min(s.T, budget / max(t0 / n0, 1e-9))))
    for _ in range(warm):
        _oracle_sample_run(s, x_np, Wr_np, bias_np, W1_np, W2_np, n, nthreads)
    times = [_oracle_sample_run(s, x_np, Wr_np, bias_np, W1_np, W2_np, n, nthreads) for _ in range(steps)]
    total = sum(times)
    flops = 6.0 * n * s.K * s.d * s.f
    value = flops * steps / total / 1e12
    sample = f"first {n} of {s.T} tokens per step (all {s.E} experts' weights as {wdt}), oracle.forward"
    line = {
        "impl": "reference", "metric": _metric(s), "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": steps, "warmup": warm, "ms_per_step": total / steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": _config(args.config, s, ws),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _metric(s):
    return "MoE layer fwd useful TFLOPS (6*T*K*d*f per layer) at 1 GB300"


def _config(name, s, ws):
    return {"workload": DESCRIPTIONS.get(name, f"MoE layer fwd T={s.T} d={s.d} E={s.E} K={s.K} f={s.f}"),
            "T": s.T, "d": s.d, "E": s.E, "K": s.K, "f": s.f, "bias": s.bias,
            "tokens_per_gpu": s.T, "parallelism": f"replicas{ws}" if ws > 1 else "single",
            "l2": "inputs larger than L2 (expert weights stream from HBM every step)"}


# ------------------------------------------------------------------ GPU arm
def run_gpu(args):
    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    import __graft_entry__
    if rank == 0 or ws == 1:
        __graft_entry__.build()
    _barrier(ws)
    import dropless_moe_expert_gb300 as moe

    s = shape(args.config)
    s_name = args.config
    T, d, E, K, f = s.T, s.d, s.E, s.K, s.f
    TK = T * K
    dev = torch.device("cuda", local)
    w = make_weights(s, seed=0, device=dev)
    x = make_tokens(s, seed=replica_seed(rank), device=dev)

    # persistent buffers of the step (granular C-ABI calls so that each
    # kernel can be bracketed by events on the launching stream)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    route_ws = torch.empty((max(4, moe.route_workspace_size(T, E, K)),), dtype=torch.uint8, device=dev)
    router_ws = torch.empty((moe.router_workspace_size(d, E),), dtype=torch.uint8, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    topk_idx, row_of = torch.empty((T, K), **i32), torch.empty((T, K), **i32)
    topk_w = torch.empty((T, K), dtype=torch.float32, device=dev)
    counts, offsets, src_tok = torch.empty((E,), **i32), torch.empty((E + 1,), **i32), torch.empty((TK,), **i32)
    mxfp8 = args.precision == "mxfp8"
    if mxfp8:
        W1q, W1s = moe.mxfp8_quantize(w.W1)
        W2q, W2s = moe.mxfp8_quantize(w.W2)
        x_perm = torch.empty((TK, d), dtype=torch.uint8, device=dev)
        sfa = torch.empty((moe.mxfp8_act_scales_size(TK, E, d),), dtype=torch.uint8, device=dev)
        h = torch.empty((TK, f), dtype=torch.uint8, device=dev)
        sfh = torch.empty((moe.mxfp8_act_scales_size(TK, E, f),), dtype=torch.uint8, device=dev)
    else:
        x_perm = torch.empty((TK, d), dtype=torch.bfloat16, device=dev)
        h = torch.empty((TK, f), dtype=torch.bfloat16, device=dev)
    y_perm = torch.empty((TK, d), dtype=torch.bfloat16, device=dev)
    y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    counters = torch.empty((max(1, int(moe.lib.moe_combine_counters_size(T, d)) // 4),), dtype=torch.int32,
                           device=dev)
    if args.fused_combine and args.precision != "bf16":
        raise SystemExit("--fused-combine is a bf16-path option")
    L = moe.lib
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    P = lambda t: t.data_ptr()  # noqa: E731
    bias_p = P(w.bias)

    def step(ev=None):
        def rec(i):
            if ev is not None:
                ev[i].record(stream)
        rec(0)
        st = L.moe_router_logits(P(x), P(w.Wr), bias_p, T, d, E, P(logits), P(router_ws), router_ws.numel(), sp)
        rec(1)
        st |= L.moe_route(P(logits), T, E, K, P(topk_idx), P(topk_w), P(counts), P(offsets), P(row_of),
                          P(src_tok), P(route_ws), route_ws.numel(), sp)
        rec(2)
        if mxfp8:
            st |= L.moe_permute_mxfp8(P(x), P(topk_idx), P(row_of), P(offsets), T, K, d, E, P(x_perm), P(sfa),
                                      sfa.numel(), sp)
            rec(3)
            st |= L.moe_grouped_gemm1_swiglu_mxfp8(P(x_perm), P(sfa), sfa.numel(), P(offsets), E, TK, d, f, P(W1q),
                                                   P(W1s), P(h), P(sfh), sfh.numel(), sp)
            rec(4)
            st |= L.moe_grouped_gemm2_mxfp8(P(h), P(sfh), sfh.numel(), P(offsets), E, TK, d, f, P(W2q), P(W2s),
                                            P(y_perm), sp)
            rec(5)
        else:
            st |= L.moe_permute(P(x), P(row_of), T, K, d, P(x_perm), sp)
            rec(3)
            st |= L.moe_grouped_gemm1_swiglu(P(x_perm), P(offsets), E, TK, d, f, P(w.W1), P(h), sp)
            rec(4)
            if args.fused_combine:
                # GEMM2 and the combine in one kernel; the combine step below is empty
                st |= L.moe_grouped_gemm2_combine(P(h), P(offsets), E, TK, d, f, P(w.W2), P(src_tok), P(row_of),
                                                  P(topk_w), T, K, P(y_perm), P(counters), counters.numel() * 4,
                                                  P(y), sp)
            else:
                st |= L.moe_grouped_gemm2(P(h), P(offsets), E, TK, d, f, P(w.W2), P(y_perm), sp)
            rec(5)
        if not args.fused_combine:
            st |= L.moe_unpermute(P(y_perm), P(row_of), P(topk_w), T, K, d, P(y), sp)
        rec(6)
        if st != 0:
            raise RuntimeError(f"C ABI returned {st}")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert moe.device_status() == 0

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(args.steps)]
    sampler = ClockSampler(local) if rank == 0 else None
    _barrier(ws)
    torch.cuda.synchronize()
    l0 = moe.launch_count()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    _barrier(ws)
    launches = moe.launch_count() - l0
    clocks = sampler.stop() if sampler else None
    assert moe.device_status() == 0
    elapsed_ms = start.elapsed_time(end)
    elapsed_ms = _max_over_ranks(elapsed_ms, ws)
    per_kernel = {n: [] for n in STEP_NAMES}
    for ev in evs:
        for j, n in enumerate(STEP_NAMES):
            per_kernel[n].append(ev[j].elapsed_time(ev[j + 1]))
    kmean = {n: sum(v) / len(v) for n, v in per_kernel.items()}
    ms_per_step = elapsed_ms / args.steps
    flops_step = 6.0 * TK * d * f
    value = aggregate(flops_step, ws, args.steps, elapsed_ms) / 1e12
    tokens_s = aggregate(T, ws, args.steps, elapsed_ms)

    # ---- end to end through the public API with host buffers (pinned): every
    # batch's host->device copy of x and device->host copy of y run inside
    # the timed region, on the library's copy streams, overlapped with the
    # compute of the neighbouring batches (moe_forward_host_pipelined).  Two
    # host input and two host output buffers are cycled over the K batches.
    x_hosts_buf = [x.cpu().pin_memory(),
                   make_tokens(s, seed=replica_seed(rank) + 1, device="cpu").pin_memory()]
    y_hosts_buf = [torch.empty((T, d), dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    if mxfp8:
        del x_perm, h, sfa, sfh
        nbytes = int(L.moe_forward_mxfp8_host_pipelined_workspace_size(T, d, E, K, f))
        ws_pipe = torch.empty((nbytes,), dtype=torch.uint8, device=dev)

        def e2e_run(n):
            moe.forward_mxfp8_host_pipelined([x_hosts_buf[i % 2] for i in range(n)],
                                             [y_hosts_buf[i % 2] for i in range(n)], w.Wr, w.bias, W1q, W1s, W2q,
                                             W2s, K, workspace=ws_pipe)
    else:
        nbytes = int(L.moe_forward_host_pipelined_workspace_size(T, d, E, K, f))
        ws_pipe = torch.empty((nbytes,), dtype=torch.uint8, device=dev)

        def e2e_run(n):
            moe.forward_host_pipelined([x_hosts_buf[i % 2] for i in range(n)],
                                       [y_hosts_buf[i % 2] for i in range(n)], w.Wr, w.bias, w.W1, w.W2, K,
                                       workspace=ws_pipe)
    e2e_run(max(3, args.warmup))
    torch.cuda.synchronize()
    _barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1), ws)
    e2e_value = aggregate(flops_step, ws, args.steps, e2e_ms) / 1e12

    # ---- the whole layer (one moe_forward call) captured once as a CUDA graph
    # and replayed: the launch-overhead-free time of a step
    graph = None
    if not mxfp8 and not args.fused_combine:
        # The graph reads its tokens from one static buffer; before every
        # replay a fresh batch is copied into it (two seeded batches,
        # alternating), so each replay routes differently and the graph is
        # never captured again.  Only the replays are timed, each between its
        # own pair of events; the copies fall outside those intervals.
        layer_g = moe.MoELayer(w.Wr, w.bias, w.W1, w.W2, K, T)
        y_g = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
        pool = [x, make_tokens(s, seed=replica_seed(rank) + 2, device=dev)]
        x_g = x.clone()
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            layer_g(x_g, out=y_g)  # warm the library's per-device state outside capture
        gs.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            layer_g(x_g, out=y_g)
        for i in range(max(3, args.warmup)):
            x_g.copy_(pool[i % 2])
            g.replay()
        torch.cuda.synchronize()
        _barrier(ws)
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.steps):
            x_g.copy_(pool[i % 2])
            gev[i][0].record(stream)
            g.replay()
            gev[i][1].record(stream)
        torch.cuda.synchronize()
        assert moe.device_status() == 0
        g_ms = _max_over_ranks(sum(a.elapsed_time(b) for a, b in gev), ws)
        graph = {"value": aggregate(flops_step, ws, args.steps, g_ms) / 1e12, "unit": "TFLOP/s",
                 "ms_per_step": g_ms / args.steps,
                 "note": "moe_forward captured once and replayed K times; before each replay a new token batch "
                         "(two seeds, alternating) is copied into the graph's input, so every replay routes "
                         "differently; only the replays are timed"}
        del g, layer_g, pool, x_g

    # ---- roofline of the dominant kernel
    peaks, peak_src = _peaks()
    dom = max(("grouped_gemm1_swiglu", "grouped_gemm2"), key=lambda n: kmean[n])
    dom_flops = (4.0 if dom == "grouped_gemm1_swiglu" else 2.0) * TK * d * f
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    peak_src_note = f"{peak_src} bf16_tflops_sustained"
    eb = 1.0 if mxfp8 else 2.0  # bytes per weight / activation element
    if mxfp8:
        peak *= 2.0
        peak_src_note += " x 2 (nominal fp8 / bf16 dense tensor ratio, 4.5 / 2.25 PFLOP/s)"
    # algorithmic bytes of one launch: the live experts' weights, the
    # activations read and the output written (scales of the MXFP8 operands
    # add 1/32 of their codes)
    live = int((counts > 0).sum().item())
    sc = (1.0 + 1.0 / 32.0) if mxfp8 else 1.0
    if dom == "grouped_gemm1_swiglu":
        dom_bytes = sc * eb * (live * 2.0 * f * d + TK * d) + sc * eb * TK * f
    else:
        dom_bytes = sc * eb * (live * 1.0 * d * f + TK * f) + 2.0 * TK * d
    t_dom = kmean[dom] * 1e-3
    hbm_peak = float(peaks["hbm_gbs"])
    # the binding resource: the larger of the two floors
    tensor_floor, hbm_floor = dom_flops / (peak * 1e12), dom_bytes / (hbm_peak * 1e9)
    tr = _traffic_record(dom + ("_mxfp8" if mxfp8 else ""), s_name)
    common = {"kernel": dom + ("_mxfp8" if mxfp8 else ""),
              "traffic": (tr["dram_bytes_per_launch"] if tr else None),
              "traffic_note": (tr.get("note") if tr else
                               "no ncu counters for this kernel source on this workload"),
              "algorithmic": {"flop": dom_flops, "bytes": dom_bytes, "live_experts": live,
                              "tensor_floor_ms": tensor_floor * 1e3, "hbm_floor_ms": hbm_floor * 1e3}}
    if hbm_floor > tensor_floor:
        achieved = dom_bytes / t_dom / 1e9
        roofline = dict(bound="hbm", achieved=achieved, peak=hbm_peak, unit="GB/s", frac=achieved / hbm_peak,
                        peak_source=f"{peak_src} hbm_gbs", **common)
    else:
        achieved = dom_flops / t_dom / 1e12
        roofline = dict(bound="tensor", achieved=achieved, peak=peak, unit="TFLOP/s", frac=achieved / peak,
                        peak_source=peak_src_note, **common)
    share = {n: kmean[n] / sum(kmean.values()) for n in STEP_NAMES}
    chunks = (T + 63) // 64
    hbm_bytes = {
        # logits read; topk_idx, topk_w, row_of written; two [chunks, E] tables written and read
        "route": 4.0 * T * E + 12.0 * TK + 16.0 * chunks * E,
        "permute": 2.0 * T * d + 2.0 * TK * d + 4.0 * TK,
        "unpermute": 2.0 * TK * d + 2.0 * T * d + 8.0 * TK,
    }
    kernels = {n: {"ms": kmean[n], "share": share[n]} for n in STEP_NAMES}
    for n, b in hbm_bytes.items():
        kernels[n]["GB/s"] = b / (kmean[n] * 1e-3) / 1e9
        kernels[n]["frac_of_hbm"] = kernels[n]["GB/s"] / float(peaks["hbm_gbs"])
    # router: bf16 tensor-core work of the three-piece split, 3 x 2*T*d*E
    kernels["router_logits"]["TFLOP/s"] = 6.0 * T * d * E / (kmean["router_logits"] * 1e-3) / 1e12
    if mxfp8:
        # E4M3 codes: x read as bf16 once, codes written K times, scales beside them
        hbm_bytes["permute"] = 2.0 * T * d + 1.0 * TK * d + TK * d / 32.0 + 8.0 * TK
        kernels["permute"]["GB/s"] = hbm_bytes["permute"] / (kmean["permute"] * 1e-3) / 1e9
        kernels["permute"]["frac_of_hbm"] = kernels["permute"]["GB/s"] / float(peaks["hbm_gbs"])
    for n in ("grouped_gemm1_swiglu", "grouped_gemm2"):
        fl = (4.0 if n == "grouped_gemm1_swiglu" else 2.0) * TK * d * f
        kernels[n]["TFLOP/s"] = fl / (kmean[n] * 1e-3) / 1e12

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N=1 only)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and not mxfp8:
        import oracle
        inputs = _oracle_inputs(s, x, w)
        nthreads = oracle.host_threads()
        n, t = _oracle_rate(s, inputs, args.cpu_budget, nthreads)
        cpu = {"value": 6.0 * n * K * d * f / t / 1e12, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
               "sample": f"first {n} of {T} tokens, oracle.forward (all {E} experts' weights as {inputs[5]}), "
                         f"{t:.1f} s"}

    if rank == 0:
        line = {
            "metric": _metric(s), "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "mxfp8" if mxfp8 else "bf16",
            "data": "synthetic (seeded N(0,1) tokens, N(0,1/fan_in) weights)",
            "config": dict(_config(s_name, s, ws), fused_combine=bool(args.fused_combine), precision=(
                "mxfp8: E4M3 elements, UE8M0 scale per 32 along K, fp32 accumulate; expert weights quantised "
                "once before the timed region" if mxfp8 else "bf16, fp32 accumulate")),
            "tokens_per_s": tokens_s, "kernels": kernels, "roofline": roofline, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": T * d * 2,
                    "d2h_bytes_per_step": T * d * 2, "ms_per_step": e2e_ms / args.steps,
                    "copies": "every batch's copies inside the timed region, overlapped with the neighbouring "
                              "batches' compute (moe_forward_host_pipelined)"},
            "gpu_launches": launches, "clocks": clocks, "graph": graph,
            "routing": {"empty_experts": int((counts == 0).sum().item()), "max_group": int(counts.max().item())},
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_train_step(args):
    """One training step of the layer: moe_forward then moe_backward with a
    seeded output gradient, timed together (kernels: forward, backward)."""
    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    import __graft_entry__
    if rank == 0 or ws == 1:
        __graft_entry__.build()
    _barrier(ws)
    import dropless_moe_expert_gb300 as moe

    s = shape(args.config)
    T, d, E, K, f = s.T, s.d, s.E, s.K, s.f
    TK = T * K
    dev = torch.device("cuda", local)
    w = make_weights(s, seed=0, device=dev)
    x = make_tokens(s, seed=replica_seed(rank), device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(7 + rank)
    dy = torch.randn((T, d), generator=g, device=dev).to(torch.bfloat16)
    layer = moe.MoELayer(w.Wr, w.bias, w.W1, w.W2, K, T)
    y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    layer(x, out=y, save_preact=True)
    grads = layer.backward(x, dy)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        # the forward keeps GEMM1's pre-activations for the backward (as a
        # training framework stores its saved activations)
        if ev is not None:
            ev[0].record(stream)
        layer(x, out=y, save_preact=True)
        if ev is not None:
            ev[1].record(stream)
        layer.backward(x, dy, grads=grads, workspace=layer.bw_workspace)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local) if rank == 0 else None
    _barrier(ws)
    torch.cuda.synchronize()
    l0 = moe.launch_count()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    _barrier(ws)
    launches = moe.launch_count() - l0
    clocks = sampler.stop() if sampler else None
    assert moe.device_status() == 0
    elapsed_ms = _max_over_ranks(start.elapsed_time(end), ws)
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    bwd_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps
    # useful work: forward 6 TK d f, backward 12 TK d f (data and weight
    # gradients of both GEMMs); the recomputed pre-activations do not count
    flops_step = 18.0 * TK * d * f
    value = aggregate(flops_step, ws, args.steps, elapsed_ms) / 1e12
    if rank == 0:
        line = {
            "metric": "MoE layer training step (fwd + bwd) useful TFLOPS (18*T*K*d*f per step) at 1 GB300",
            "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) tokens and output gradient)",
            "config": dict(_config(args.config, s, ws), step="forward + backward",
                           grads="dx bf16; dWr, dbias, dW1, dW2 fp32",
                           saved="GEMM1 pre-activations [T*K, 2f] bf16, stored by the forward"),
            "kernels": {"forward": {"ms": fwd_ms, "TFLOP/s": 6.0 * TK * d * f / (fwd_ms * 1e-3) / 1e12},
                        "backward": {"ms": bwd_ms, "TFLOP/s": 12.0 * TK * d * f / (bwd_ms * 1e-3) / 1e12}},
            "gpu_launches": launches, "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", default="mixtral")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fused-combine", action="store_true",
                    help="fuse the combine into GEMM2's epilogue (bf16 path)")
    ap.add_argument("--backward", action="store_true",
                    help="time a training step of the layer (forward + backward) instead of the forward")
    ap.add_argument("--precision", default="bf16", choices=["bf16", "mxfp8"],
                    help="expert matmuls in bf16 or MXFP8 (E4M3, UE8M0 scale per 32)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.backward:
        run_train_step(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
