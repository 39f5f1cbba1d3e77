#!/usr/bin/env python3
"""Benchmark of the dropless MoE layer forward on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                [--config skew|mixtral|dsv3|qwen|tiny] [--extra-configs LIST]
                [--precision bf16|mxfp8] [--backward] [--fused-combine]

One step = one pass of the whole forward (router logits, top-K routing +
histogram/scan/dispatch order, permute, grouped GEMM1 + SwiGLU, grouped GEMM2,
weighted unpermute/combine) over one batch of T tokens, through the C ABI.
The steps alternate between two resident token batches, so consecutive steps
route differently.  Default workload: the extreme-skew layer (T=32768,
d=4096, E=64, K=6, f=1536), the one with the most work per step; the
Mixtral-, DeepSeek-V3- and Qwen-shaped layers are then timed on the device in
the same run and reported under `other_configs`.  Seeded synthetic bf16
data.  Under torchrun every rank runs an independent replica on its own
tokens (the forward has no cross-token dependency, so there is no
collective): weak scaling.

Prints one JSON line (rank 0).  `value` is useful TFLOP/s = 6*T*K*d*f per
step (only the valid rows of the two grouped GEMMs count), aggregated over
ranks; per-kernel durations come from CUDA events on the launching stream
inside the timed region.  Clocks are sampled through NVML's query calls
inside the timed region.  The roofline fraction of the dominant GEMM is
given against both measured bf16 peaks; `frac` takes the burst figure for a
timed region under one second and the sustained one otherwise.  `--impl reference` times the oracle (plain CPU
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
    rec = d.get(f"{kernel}@{workload}")
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
    """SM clock, power and clock-event reasons sampled DURING the timed region.

    A background thread queries NVML (libnvidia-ml, the driver's library)
    every `period_s` through read-only calls: nvmlDeviceGetClockInfo,
    nvmlDeviceGetMaxClockInfo, nvmlDeviceGetPowerUsage and the current
    clock-event reasons.  No setting of the GPU is changed.  The device is
    found by its UUID (else PCI bus id, else index), so the sample is of the
    GPU this process runs on whatever CUDA_VISIBLE_DEVICES holds.  Without
    NVML it falls back to polling nvidia-smi every 100 ms."""

    # clock-event reason bits (nvml.h): the ones a timing must record
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, cuda_index: int, period_s: float = 0.004):
        import ctypes
        import threading
        self.period = period_s
        self.rows = []          # (sm_mhz, power_w, reason_bits)
        self.max_mhz = None
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self._nvml = None
        self._h = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit_v2 failed")
            h = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(cuda_index)
            ok = False
            uuid = getattr(props, "uuid", None)
            if uuid is not None:
                key = str(uuid)
                key = key if key.startswith("GPU-") else "GPU-" + key
                ok = nv.nvmlDeviceGetHandleByUUID(key.encode(), ctypes.byref(h)) == 0
            if not ok and hasattr(props, "pci_bus_id"):
                bus = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                            getattr(props, "pci_device_id", 0))
                ok = nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
            if not ok:
                ok = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(cuda_index), ctypes.byref(h)) == 0
            if not ok:
                raise OSError("no NVML handle for the device")
            self._reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint(0)
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # NVML_CLOCK_SM
                self.max_mhz = float(mx.value)
            self._nvml, self._h, self._ct = nv, h, ctypes
            self.source = f"NVML query every {period_s * 1e3:.0f} ms in a thread of the bench process"
        except Exception:
            self._nvml = None

    def _sample_nvml(self):
        ct, nv, h = self._ct, self._nvml, self._h
        mhz, mw, bits = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(mhz)) == 0:
                p = mw.value / 1e3 if nv.nvmlDeviceGetPowerUsage(h, ct.byref(mw)) == 0 else None
                r = bits.value if self._reasons_fn(h, ct.byref(bits)) == 0 else 0
                self.rows.append((float(mhz.value), p, int(r)))
            self._stop.wait(self.period)

    def start(self):
        import threading
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._sample_nvml, daemon=True)
            self._thread.start()
            return self
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi -lms 100"
        except Exception:
            self._proc = None
        return self

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        elif self._proc is not None:
            self._proc.terminate()
            try:
                out, _ = self._proc.communicate(timeout=5)
            except Exception:
                self._proc.kill()
                out = ""
            for line in out.splitlines():
                parts = [q.strip() for q in line.split(",")]
                try:
                    self.max_mhz = float(parts[1])
                    self.rows.append((float(parts[0]), float(parts[2]), int(parts[3], 16)))
                except (ValueError, IndexError):
                    continue
        else:
            return None
        if not self.rows:
            return None
        sm = [r[0] for r in self.rows]
        pw = [r[1] for r in self.rows if r[1] is not None]
        reasons = sorted({name for r in self.rows for bit, name in self.REASONS.items() if r[2] & bit})
        counts = {name: sum(1 for r in self.rows if r[2] & bit) for bit, name in self.REASONS.items()}
        return {"sm_mhz": statistics.median(sm), "sm_mhz_min": min(sm), "sm_max_mhz": self.max_mhz,
                "power_w_max": max(pw) if pw else None, "reasons": reasons,
                "reason_samples": {k: v for k, v in counts.items() if v}, "samples": len(self.rows),
                "source": self.source}


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
        "config": _config(args.config, s, ws, args),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _metric(s):
    return "MoE layer fwd useful TFLOPS (6*T*K*d*f per layer) at 1 GB300"


def _config(name, s, ws, args):
    mxfp8 = getattr(args, "precision", "bf16") == "mxfp8"
    return {"workload": DESCRIPTIONS.get(name, f"MoE layer fwd T={s.T} d={s.d} E={s.E} K={s.K} f={s.f}"),
            "T": s.T, "d": s.d, "E": s.E, "K": s.K, "f": s.f, "bias": s.bias,
            "tokens_per_gpu": s.T, "parallelism": f"replicas{ws}" if ws > 1 else "single",
            "l2": "inputs larger than L2 (expert weights stream from HBM every step)",
            "fused_combine": bool(getattr(args, "fused_combine", False)),
            "permute": getattr(args, "permute", "auto"),
            "precision": ("mxfp8: E4M3 elements, UE8M0 scale per 32 along K, fp32 accumulate; expert weights "
                          "quantised once before the timed region" if mxfp8 else "bf16, fp32 accumulate")}


# ------------------------------------------------------------------ GPU arm
# A timed region shorter than this runs at the clocks of a burst (the bench's
# regions are tens of ms); longer ones settle where the sustained peak was
# measured (a seconds-long loop under the power cap).
BURST_REGION_S = 1.0


def _dominant_roofline(s, s_name, kmean, counts, mxfp8, region_s, fused_permute=False):
    """Roofline of the dominant grouped GEMM: its binding resource (the
    larger of the tensor and HBM floors), achieved rate from the event-timed
    mean launch, and the fraction of both measured bf16 peaks, the one that
    applies named by the length of the timed region."""
    T, d, E, K, f = s.T, s.d, s.E, s.K, s.f
    TK = T * K
    peaks, peak_src = _peaks()
    dom = max(("grouped_gemm1_swiglu", "grouped_gemm2"), key=lambda n: kmean[n])
    dom_flops = (4.0 if dom == "grouped_gemm1_swiglu" else 2.0) * TK * d * f
    burst = float(peaks.get("bf16_tflops", 1900.0))
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    ratio = 2.0 if mxfp8 else 1.0      # nominal dense fp8 / bf16 tensor ratio (4.5 / 2.25 PFLOP/s)
    use_burst = region_s < BURST_REGION_S
    peak = (burst if use_burst else sustained) * ratio
    peak_src_note = (f"{peak_src} bf16_tflops ({'burst' if use_burst else 'sustained'}: the timed region "
                     f"lasted {region_s:.3f} s, {'under' if use_burst else 'over'} {BURST_REGION_S:.0f} s)")
    if not use_burst:
        peak_src_note = peak_src_note.replace("bf16_tflops (", "bf16_tflops_sustained (")
    if mxfp8:
        peak_src_note += " x 2 (nominal fp8 / bf16 dense tensor ratio, 4.5 / 2.25 PFLOP/s)"
    eb = 1.0 if mxfp8 else 2.0  # bytes per weight / activation element
    # algorithmic bytes of one launch: the live experts' weights, the
    # activations read and the output written (scales of the MXFP8 operands
    # add 1/32 of their codes)
    live = int((counts > 0).sum().item())
    sc = (1.0 + 1.0 / 32.0) if mxfp8 else 1.0
    if dom == "grouped_gemm1_swiglu":
        # A: the permuted rows, or (permute fused) each token row once
        a_rows = T if fused_permute else TK
        dom_bytes = sc * eb * (live * 2.0 * f * d + a_rows * d) + sc * eb * TK * f
    else:
        dom_bytes = sc * eb * (live * 1.0 * d * f + TK * f) + 2.0 * TK * d
    t_dom = kmean[dom] * 1e-3
    hbm_peak = float(peaks["hbm_gbs"])
    tensor_floor, hbm_floor = dom_flops / (peak * 1e12), dom_bytes / (hbm_peak * 1e9)
    tr = _traffic_record(dom + ("_mxfp8" if mxfp8 else ""), s_name)
    tflops = dom_flops / t_dom / 1e12
    common = {"kernel": dom + ("_mxfp8" if mxfp8 else ""),
              "traffic": (tr["dram_bytes_per_launch"] if tr else None),
              "traffic_note": (tr.get("note") if tr else
                               "no ncu counters for this kernel source on this workload"),
              "algorithmic": {"flop": dom_flops, "bytes": dom_bytes, "live_experts": live,
                              "tensor_floor_ms": tensor_floor * 1e3, "hbm_floor_ms": hbm_floor * 1e3},
              "frac_of_bf16_burst": tflops / (burst * ratio),
              "frac_of_bf16_sustained": tflops / (sustained * ratio),
              "frac_of_hbm": dom_bytes / t_dom / 1e9 / hbm_peak}
    if hbm_floor > tensor_floor:
        achieved = dom_bytes / t_dom / 1e9
        return dict(bound="hbm", achieved=achieved, peak=hbm_peak, unit="GB/s", frac=achieved / hbm_peak,
                    peak_source=f"{peak_src} hbm_gbs", **common)
    return dict(bound="tensor", achieved=tflops, peak=peak, unit="TFLOP/s", frac=tflops / peak,
                peak_source=peak_src_note, **common)


def _kernel_table(s, kmean, mxfp8, fused_permute=False):
    T, d, E, K, f = s.T, s.d, s.E, s.K, s.f
    TK = T * K
    peaks, _ = _peaks()
    share = {n: kmean[n] / sum(kmean.values()) for n in STEP_NAMES}
    chunks = (T + 63) // 64
    hbm_bytes = {
        # logits read; topk_idx, topk_w, row_of written; two [chunks, E] tables written and read
        "route": 4.0 * T * E + 12.0 * TK + 16.0 * chunks * E,
        "permute": 2.0 * T * d + 2.0 * TK * d + 4.0 * TK,
        "unpermute": 2.0 * TK * d + 2.0 * T * d + 8.0 * TK,
    }
    if mxfp8:
        # E4M3 codes: x read as bf16 once, codes written K times, scales beside them
        hbm_bytes["permute"] = 2.0 * T * d + 1.0 * TK * d + TK * d / 32.0 + 8.0 * TK
    kernels = {n: {"ms": kmean[n], "share": share[n]} for n in STEP_NAMES}
    if fused_permute:
        # no permute kernel: GEMM1 gathers its rows from x
        del hbm_bytes["permute"]
        kernels["permute"]["fused_into"] = "grouped_gemm1_swiglu"
    for n, b in hbm_bytes.items():
        kernels[n]["GB/s"] = b / (kmean[n] * 1e-3) / 1e9
        kernels[n]["frac_of_hbm"] = kernels[n]["GB/s"] / float(peaks["hbm_gbs"])
    # router: bf16 tensor-core work of the three-piece split, 3 x 2*T*d*E
    kernels["router_logits"]["TFLOP/s"] = 6.0 * T * d * E / (kmean["router_logits"] * 1e-3) / 1e12
    for n in ("grouped_gemm1_swiglu", "grouped_gemm2"):
        fl = (4.0 if n == "grouped_gemm1_swiglu" else 2.0) * TK * d * f
        kernels[n]["TFLOP/s"] = fl / (kmean[n] * 1e-3) / 1e12
    return kernels


def measure_forward(moe, s_name, args, ws, rank, local, full=True):
    """Times K steps of the layer forward on workload `s_name` through the C
    ABI (one event pair per kernel on the launching stream).  The steps
    alternate between two resident token batches (two seeds), so that
    consecutive steps route differently.  With `full`, also the end-to-end
    host-buffer rate, the graph replays and the CPU baseline."""
    s = shape(s_name)
    T, d, E, K, f = s.T, s.d, s.E, s.K, s.f
    TK = T * K
    dev = torch.device("cuda", local)
    w = make_weights(s, seed=0, device=dev)
    xs = [make_tokens(s, seed=replica_seed(rank), device=dev),
          make_tokens(s, seed=replica_seed(rank) + 1, device=dev)]

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
    L = moe.lib
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    P = lambda t: t.data_ptr()  # noqa: E731
    bias_p = P(w.bias)
    fuse_permute = not mxfp8 and (args.permute == "fused" or (
        args.permute == "auto" and moe.forward_fuses_permute(T, d, E, K, f)))

    def step(i, ev=None):
        x = xs[i % 2]

        def rec(j):
            if ev is not None:
                ev[j].record(stream)
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
            if fuse_permute:
                # the permute fused into GEMM1's operand load; the permute step is empty
                rec(3)
                st |= L.moe_grouped_gemm1_swiglu_gather(P(x), P(src_tok), P(offsets), T, E, TK, d, f, P(w.W1), P(h),
                                                        sp)
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

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert moe.device_status() == 0

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(args.steps)]
    sampler = ClockSampler(local).start() if rank == 0 else None
    _barrier(ws)
    torch.cuda.synchronize()
    l0 = moe.launch_count()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(i, evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    _barrier(ws)
    launches = moe.launch_count() - l0
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
    res = {
        "config": s_name, "s": s, "value": aggregate(flops_step, ws, args.steps, elapsed_ms) / 1e12,
        "fused_permute": bool(fuse_permute),
        "tokens_per_s": aggregate(T, ws, args.steps, elapsed_ms), "ms_per_step": ms_per_step,
        "launches": launches, "clocks": clocks, "timed_region_s": elapsed_ms * 1e-3,
        "kernels": _kernel_table(s, kmean, mxfp8, fuse_permute),
        "roofline": _dominant_roofline(s, s_name, kmean, counts, mxfp8, elapsed_ms * 1e-3, fuse_permute),
        "routing": {"empty_experts": int((counts == 0).sum().item()), "max_group": int(counts.max().item()),
                    "batches": "two resident token batches (seeds r, r+1), alternating step by step"},
    }
    if not full:
        return res

    # ---- end to end through the public API with host buffers (pinned): every
    # batch's host->device copy of x and device->host copy of y run inside
    # the timed region, on the library's copy streams, overlapped with the
    # compute of the neighbouring batches (moe_forward_host_pipelined).  Two
    # host input and two host output buffers are cycled over the K batches.
    x_hosts_buf = [xs[0].cpu().pin_memory(), xs[1].cpu().pin_memory()]
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
    e2e_sampler = ClockSampler(local).start() if rank == 0 else None
    e0.record(stream)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_clocks = e2e_sampler.stop() if e2e_sampler else None
    assert moe.device_status() == 0
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1), ws)
    res["e2e"] = {"value": aggregate(flops_step, ws, args.steps, e2e_ms) / 1e12, "unit": "TFLOP/s",
                  "h2d_bytes_per_step": T * d * 2, "d2h_bytes_per_step": T * d * 2,
                  "ms_per_step": e2e_ms / args.steps,
                  "copies": "every batch's copies inside the timed region, overlapped with the neighbouring "
                            "batches' compute (moe_forward_host_pipelined)",
                  "clocks": e2e_clocks}
    del ws_pipe

    # ---- the whole layer (one moe_forward call) captured once as a CUDA graph
    # and replayed: the launch-overhead-free time of a step
    res["graph"] = None
    if not mxfp8 and not args.fused_combine and args.permute == "auto":
        # The graph reads its tokens from one static buffer; before every
        # replay a fresh batch is copied into it (two seeded batches,
        # alternating), so each replay routes differently and the graph is
        # never captured again.  Only the replays are timed, each between its
        # own pair of events; the copies fall outside those intervals.
        layer_g = moe.MoELayer(w.Wr, w.bias, w.W1, w.W2, K, T)
        y_g = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
        pool = [xs[0], make_tokens(s, seed=replica_seed(rank) + 2, device=dev)]
        x_g = xs[0].clone()
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
        res["graph"] = {"value": aggregate(flops_step, ws, args.steps, g_ms) / 1e12, "unit": "TFLOP/s",
                        "ms_per_step": g_ms / args.steps,
                        "note": "moe_forward captured once and replayed K times; before each replay a new token "
                                "batch (two seeds, alternating) is copied into the graph's input, so every replay "
                                "routes differently; only the replays are timed"}
        del g, layer_g, pool, x_g

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N=1 only)
    res["cpu_baseline"] = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and not mxfp8:
        import oracle
        inputs = _oracle_inputs(s, xs[0], w)
        nthreads = oracle.host_threads()
        n, t = _oracle_rate(s, inputs, args.cpu_budget, nthreads)
        res["cpu_baseline"] = {
            "value": 6.0 * n * K * d * f / t / 1e12, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
            "sample": f"first {n} of {T} tokens, oracle.forward (all {E} experts' weights as {inputs[5]}), "
                      f"{t:.1f} s"}
    return res


def run_gpu(args):
    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    import __graft_entry__
    if rank == 0 or ws == 1:
        __graft_entry__.build()
    _barrier(ws)
    import dropless_moe_expert_gb300 as moe

    mxfp8 = args.precision == "mxfp8"
    r = measure_forward(moe, args.config, args, ws, rank, local, full=True)
    # the other large workloads, device-timed the same way (no e2e or
    # baseline legs), so that one run reports every configuration
    others = {}
    for name in [c for c in args.extra_configs.split(",") if c and c != args.config]:
        torch.cuda.empty_cache()
        o = measure_forward(moe, name, args, ws, rank, local, full=False)
        others[name] = {"workload": DESCRIPTIONS.get(name, name), "value": o["value"], "unit": "TFLOP/s",
                        "tokens_per_s": o["tokens_per_s"], "ms_per_step": o["ms_per_step"],
                        "kernels": {n: {"ms": k["ms"], **({"TFLOP/s": k["TFLOP/s"]} if "TFLOP/s" in k else {}),
                                        **({"frac_of_hbm": k["frac_of_hbm"]} if "frac_of_hbm" in k else {})}
                                    for n, k in o["kernels"].items()},
                        "roofline": {kk: o["roofline"][kk] for kk in (
                            "bound", "kernel", "achieved", "peak", "unit", "frac", "frac_of_bf16_burst",
                            "frac_of_bf16_sustained", "frac_of_hbm")},
                        "routing": o["routing"], "clocks": o["clocks"], "gpu_launches": o["launches"],
                        "fused_permute": o["fused_permute"]}
    s = r["s"]
    if rank == 0:
        line = {
            "metric": _metric(s), "value": r["value"], "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "mxfp8" if mxfp8 else "bf16",
            "data": "synthetic (seeded N(0,1) tokens, N(0,1/fan_in) weights)",
            "config": _config(args.config, s, ws, args),
            "tokens_per_s": r["tokens_per_s"], "kernels": r["kernels"], "roofline": r["roofline"],
            "cpu_baseline": r["cpu_baseline"], "e2e": r["e2e"], "gpu_launches": r["launches"],
            "clocks": r["clocks"], "timed_region_s": r["timed_region_s"], "graph": r["graph"],
            "routing": r["routing"], "fused_permute": r["fused_permute"], "other_configs": others or None,
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
    sampler = ClockSampler(local).start() if rank == 0 else None
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
            "config": dict(_config(args.config, s, ws, args), step="forward + backward",
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
    ap.add_argument("--config", default="skew",
                    help="headline workload (default: the extreme-skew layer, the most work per step)")
    ap.add_argument("--extra-configs", default="mixtral,dsv3,qwen",
                    help="other workloads timed on the device in the same run (comma list, '' for none)")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fused-combine", action="store_true",
                    help="fuse the combine into GEMM2's epilogue (bf16 path)")
    ap.add_argument("--permute", default="auto", choices=["auto", "fused", "separate"],
                    help="bf16 path: fuse the permute into GEMM1's operand load, or run it as its own kernel; "
                         "auto = moe_forward's choice for the shape (moe_forward_fuses_permute)")
    ap.add_argument("--backward", action="store_true",
                    help="time a training step of the layer (forward + backward) instead of the forward")
    ap.add_argument("--precision", default="bf16", choices=["bf16", "mxfp8"],
                    help="expert matmuls in bf16 or MXFP8 (E4M3, UE8M0 scale per 32)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if (args.permute == "fused" or args.fused_combine) and args.precision != "bf16":
        raise SystemExit("--permute fused and --fused-combine are bf16-path options")
    if args.impl == "reference":
        run_reference(args)
    elif args.backward:
        run_train_step(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
