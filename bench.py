"""Benchmark: one step = the whole MXFP8 hot path of a Qwen3-8B linear layer set at one
micro-batch of 4096 tokens ("End-to-End MXFP8 RL on Blackwell", sections "The pipeline"
and "Where the time goes": per linear layer, the operands X, W and dY are quantized
row-wise and column-wise, then the fprop, dgrad and wgrad block-scaled GEMMs run).

Per step and layer (qkv 4096->6144, o 4096->4096, gate_up 4096->24576, down 12288->4096):
two dual quantize launches (X and W together, as the forward pass has them; dY alone, as
the backward pass has it), each giving both copies from one read, and 3 GEMM launches;
20 launches per step (--quant separate: 6 single-axis quantizes per layer). A layer's
wgrad needs only the quantized copies, not the fprop or dgrad results, so it runs on a
second stream beside them (--streams 1 keeps every launch on one stream); the per-launch
split is measured with every launch on one stream. Inputs are synthetic
(seeded, BF16) and live in HBM before the timed region; the step's working set (453 MB
of BF16 inputs) is larger than L2, so no flush is needed between steps.

Output: one JSON line (rank 0). `value` is the step's MXFP8 GEMM FLOPs divided by the
step time (quantization included), in TFLOP/s, with the step's 20 launches issued as
above (`cuda_graph` gives the same step replayed from a CUDA graph). The `quantize` and
`gemm` objects split the time, from CUDA events around every launch of further steps;
`roofline` is for the dominant kernel (the GEMM) and `roofline_quantize` for the quantizer.
`secondary` measures the other configurations after the headline, on the same GPU: the
Qwen3-30B-A3B expert layer (grouped GEMMs), the Qwen3-8B weight-synchronization pass and
the micro-batch sweep.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --workload moe|sync|sweep     # one of the other configurations alone
  python bench.py --workload gemm --shapes 4096,4096,4096[;M,N,K...]   # single GEMMs
  python bench.py --workload quantize --shapes 4096,4096 --mode dual   # single quantizes
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantize GB/s + MXFP8 GEMM TFLOP/s on Qwen3-8B linears, % of GB300 roofline"
FP8_OVER_BF16 = 2.0   # nominal dense FP8 : BF16 tensor rate (4.5 : 2.25 PFLOP/s)
QBYTES_PER_ELEM = 2.0 + 1.0 + 1.0 / 32.0   # BF16 read + E4M3 + E8M0/32 written
DUAL_BYTES_PER_ELEM = 2.0 + 2 * (1.0 + 1.0 / 32.0)   # one BF16 read, two quantized copies
REF_ROW_FRAC = 1.0 / 8192   # reference arm: 32 rows of every operand per step
REF_BLOCK = (8, 16)         # reference arm: output block sampled per GEMM


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ----------------------------------------------------------------------- distributed

def dist_setup(n_gpus):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, ws


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()


def max_over_ranks(x: float, ws: int) -> float:
    """The slowest rank's value (timing only; no data-path collective)."""
    if ws == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self, busy_mhz_floor: float = 0.0):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), power=float(f[3]),
                                 hw=f[5], hwt=f[6], swt=f[7], pcap=f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        load = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(load),
                "power_w_max": max(r["power"] for r in rows)}


# --------------------------------------------------------------------------- workload

def layer_flops(t, n, k):
    return 3 * 2.0 * t * n * k


def layer_quant_elems(t, n, k):
    # X [t,k], W [n,k], dY [t,n], each row-wise and column-wise
    return 2 * (t * k + n * k + t * n)


class DenseStep:
    """Buffers and launches of one step over dense linear layers (name, N, K, X, W, dY);
    every launch goes through the C ABI."""

    def __init__(self, m, layers, dev, dual: bool = True, streams: int = 1):
        self.m = m
        self.dual = dual
        # streams == 2: each layer's wgrad runs on a second stream, beside its fprop and dgrad
        # (they only share the quantized inputs), so that one GEMM's partial last wave of
        # clusters overlaps the next GEMM's first one
        self.side = torch.cuda.Stream(device=dev) if streams == 2 else None
        self.layers = []
        for name, n, k, x, w, dy in layers:
            t = x.shape[0]
            L = dict(name=name, t=t, n=n, k=k, x=x, w=w, dy=dy)
            for key, src, axis in (("xr", x, m.ROW), ("xc", x, m.COL), ("wr", w, m.ROW),
                                   ("wc", w, m.COL), ("dyr", dy, m.ROW), ("dyc", dy, m.COL)):
                r, c = src.shape
                shape = (r, c) if axis == m.ROW else (c, r)
                L[key] = (torch.empty(shape, dtype=torch.uint8, device=dev),
                          torch.empty(m.scale_bytes(r, c, axis, m.SWIZZLED), dtype=torch.uint8,
                                      device=dev), src, axis)
            L["y"] = torch.empty((t, n), dtype=torch.bfloat16, device=dev)
            L["dx"] = torch.empty((t, k), dtype=torch.bfloat16, device=dev)
            L["dw"] = torch.empty((n, k), dtype=torch.bfloat16, device=dev)
            self.layers.append(L)
        # split-K workspaces for the GEMMs whose last wave runs as K pieces (zero-filled once;
        # one per stream, since a workspace serves one GEMM at a time)
        need = max([m.gemm_workspace_bytes(*mnk) for L in self.layers
                    for mnk in ((L["t"], L["n"], L["k"]), (L["t"], L["k"], L["n"]),
                                (L["n"], L["k"], L["t"]))] + [0])
        self.ws = [torch.zeros(need, dtype=torch.uint8, device=dev) if need else None
                   for _ in range(2)]
        self.flops = sum(layer_flops(L["t"], L["n"], L["k"]) for L in self.layers)
        self.qelems = sum(layer_quant_elems(L["t"], L["n"], L["k"]) for L in self.layers)
        self.launches = (5 if dual else 9) * len(self.layers)

    def run(self, stream, events=None):
        """Enqueues one step. With `events` (a list), appends (kind, units, start, end); the
        per-launch events keep every launch on `stream`."""
        side = self.side if events is None else None
        done = None
        for L in self.layers:
            self.run_quantize(L, stream, events)
            done = self.run_gemms(L, stream, events, side=side) or done
        if done is not None:
            stream.wait_event(done)  # the side stream rejoins before the step ends

    def run_quantize(self, L, stream, events=None):
        """The layer's quantize launches (they read x, w and dy)."""
        m = self.m
        if self.dual:
            # One read of each BF16 tensor gives both of its quantized copies. The forward
            # operands (x and w) go in one launch; dy, which a training step only has in
            # the backward pass, in another.
            x, w = L["x"], L["w"]
            ev = self._ev(events, stream, "quantize",
                          (x.numel() + w.numel()) * DUAL_BYTES_PER_ELEM,
                          f"{L['name']}.x+w dual {x.shape[0]}x{x.shape[1]} + {w.shape[0]}x{w.shape[1]}")
            m.quantize_dual_multi([x, w], m.SWIZZLED,
                                  outs=[(L["xr"][0], L["xr"][1], L["xc"][0], L["xc"][1]),
                                        (L["wr"][0], L["wr"][1], L["wc"][0], L["wc"][1])],
                                  stream=stream)
            self._end(events, stream, ev)
            dy = L["dy"]
            ev = self._ev(events, stream, "quantize", dy.numel() * DUAL_BYTES_PER_ELEM,
                          f"{L['name']}.dy dual {dy.shape[0]}x{dy.shape[1]}")
            m.quantize_dual(dy, m.SWIZZLED, row_out=L["dyr"][0], row_scales=L["dyr"][1],
                            col_out=L["dyc"][0], col_scales=L["dyc"][1], stream=stream)
            self._end(events, stream, ev)
        else:
            for key in ("xr", "xc", "wr", "wc", "dyr", "dyc"):
                q, s, src, axis = L[key]
                ev = self._ev(events, stream, "quantize", src.numel() * QBYTES_PER_ELEM,
                              f"{L['name']}.{key} {src.shape[0]}x{src.shape[1]}")
                m.quantize(src, axis, m.SWIZZLED, out=q, scales=s, stream=stream)
                self._end(events, stream, ev)

    def run_gemms(self, L, stream, events=None, side=None):
        """The layer's three GEMMs (they write y, dx and dw). With a `side` stream the wgrad
        runs there, after the layer's quantize launches; returns the event that marks its
        end (None without a side stream)."""
        m = self.m
        t, n, k = L["t"], L["n"], L["k"]
        done = None
        if side is not None:
            quantized = torch.cuda.Event()
            quantized.record(stream)
            side.wait_event(quantized)
        for op, a, b, out, mnk in ((m.FPROP, "xr", "wr", L["y"], (t, n, k)),
                                   (m.DGRAD, "dyr", "wc", L["dx"], (t, k, n)),
                                   (m.WGRAD, "dyc", "xc", L["dw"], (n, k, t))):
            st = side if (side is not None and op == m.WGRAD) else stream
            ev = self._ev(events, st, "gemm", 2.0 * mnk[0] * mnk[1] * mnk[2],
                          f"{L['name']}.{('fprop', 'dgrad', 'wgrad')[op]} {mnk[0]}x{mnk[1]}x{mnk[2]}")
            m.gemm(L[a][0], L[a][1], L[b][0], L[b][1], op, m.OUT_BF16, out=out, stream=st,
                   workspace=self.ws[1 if st is side else 0])
            self._end(events, st, ev)
            if st is side:
                done = torch.cuda.Event()
                done.record(side)
        return done

    @staticmethod
    def _ev(events, stream, kind, units, label=""):
        if events is None:
            return None
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        return (kind, units, s, e, label)

    @staticmethod
    def _end(events, stream, ev):
        if ev is not None:
            ev[3].record(stream)
            events.append(ev)


KERNEL_SOURCES = {"mxfp8_gemm": ("gemm.cu", "device.cuh"),
                  "quantize_dual": ("quantize.cu", "device.cuh")}


def source_sha(kernel_key: str):
    """Short hash of the sources a kernel is built from."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel_key]:
        with open(os.path.join(ROOT, "mxfp8_block_scaled_05_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key: str):
    """DRAM bytes per launch (step average) from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    sha = source_sha(kernel_key)
    for line in open(p):
        if line.startswith("#"):
            continue
        f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if (f.get("kernel") == kernel_key and f.get("source_sha") == sha
                and f.get("workload") == "step_average"):
            return float(f["dram_bytes_per_launch"])
    return None


# ------------------------------------------------------------------------- CPU oracle

def oracle_step_sample(seed: int = 0, row_frac: float = 1.0 / 512, block=(32, 64)):
    """Times the CPU oracle on a bounded sample of one step: a fraction of the rows of
    every quantized operand and one 32 x 64 output block per GEMM. Returns (seconds for
    the sampled work, seconds extrapolated to a full step, description)."""
    import oracle.mxfp8_oracle as O
    from mxfp8_block_scaled_05_gb300 import workloads as W
    rng = np.random.default_rng(seed)
    q_sec, q_elems, g_sec, g_flops = 0.0, 0, 0.0, 0.0
    total_q, total_f = 0, 0.0
    for name, n, k in W.QWEN3_8B_LINEARS:
        t = 4096
        total_q += layer_quant_elems(t, n, k)
        total_f += layer_flops(t, n, k)
        for rows, cols in ((t, k), (n, k), (t, n)):
            r = max(32, int(rows * row_frac) // 32 * 32)
            x = (rng.standard_normal((r, cols)).astype(np.float32).view(np.uint32) >> 16
                 ).astype(np.uint16)
            t0 = time.perf_counter()
            O.quantize(x, O.ROW)
            O.quantize(x, O.COL)
            q_sec += time.perf_counter() - t0
            q_elems += 2 * r * cols
        for mm, nn, kk in ((t, n, k), (t, k, n), (n, k, t)):
            a = (rng.standard_normal((block[0], kk)).astype(np.float32).view(np.uint32) >> 16
                 ).astype(np.uint16)
            b = (rng.standard_normal((block[1], kk)).astype(np.float32).view(np.uint32) >> 16
                 ).astype(np.uint16)
            qa, sa = O.quantize(a, O.ROW)
            qb, sb = O.quantize(b, O.ROW)
            t0 = time.perf_counter()
            O.gemm(qa, sa, qb, sb)
            O.gemm_abs(qa, sa, qb, sb)
            g_sec += time.perf_counter() - t0
            g_flops += 2.0 * block[0] * block[1] * kk
    est = q_sec * total_q / q_elems + g_sec * total_f / g_flops
    desc = (f"{row_frac:.4g} of every operand's rows quantized row+col ({q_elems} elems) and a "
            f"{block[0]}x{block[1]} output block of each of the 12 GEMMs ({g_flops / 1e9:.3f} GFLOP), "
            "extrapolated to the full step")
    return q_sec + g_sec, est, desc, total_f


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------- arms

def run_reference(args, rank, ws):
    """The oracle as it stands, on the host cores (a deliberately slow program)."""
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_step_sample(0, REF_ROW_FRAC, REF_BLOCK)
    secs, ests, desc, flops = [], [], "", 0.0
    for i in range(args.steps):
        s, est, desc, flops = oracle_step_sample(i + 1, REF_ROW_FRAC, REF_BLOCK)
        secs.append(s)
        ests.append(est)
    step_s = float(np.mean(ests))
    value = flops / step_s / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_obj(),
        "cpu_baseline": {"kind": "oracle", "value": value, "unit": "TFLOP/s",
                         "cores": cpu_cores(), "sample": desc,
                         "sample_seconds_per_step": float(np.mean(secs))},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_obj(tokens=4096):
    return {"workload": f"Qwen3-8B dense linear layer set at {tokens} tokens: qkv 4096->6144, "
                        "o 4096->4096, gate_up 4096->24576, down 12288->4096; X, W, dY "
                        "quantized row- and column-wise (swizzled scales), then fprop, dgrad "
                        "and wgrad MXFP8 GEMMs (BF16 out) per layer",
            "tokens": tokens, "layers": 4,
            "l2": "inputs larger than L2 (453 MB BF16 per step), no flush"}


def run_ours(args, rank, ws):
    import mxfp8_block_scaled_05_gb300 as m
    dev = torch.device("cuda", torch.cuda.current_device())
    pk = peaks()
    from mxfp8_block_scaled_05_gb300 import workloads as W
    step = DenseStep(m, W.qwen3_8b_layer_set(args.tokens, dev, seed=1 + rank), dev,
                     dual=args.quant == "dual", streams=args.streams)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step.run(stream)
    torch.cuda.synchronize()
    if m.device_status() != m.OK:
        raise RuntimeError("device status set during warm-up")

    # The K timed steps: the 20 launches of each step issued on one stream, nothing else
    # enqueued between them (the host stays ahead of the GPU).
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier(ws)
        start.record(stream)
        for _ in range(args.steps):
            step.run(stream)
        end.record(stream)
        barrier(ws)
    ms = start.elapsed_time(end)
    ms_max = max_over_ranks(ms, ws)
    status = m.device_status()
    if status != m.OK:
        raise RuntimeError(f"device status {status} after the timed region")

    # The split between quantize and GEMM time, per launch: further steps with CUDA events
    # around every launch.
    split_steps = max(10, args.steps // 4)
    events = []
    for _ in range(split_steps):
        step.run(stream, events)
    torch.cuda.synchronize()
    q_ms = sum(s.elapsed_time(e) for k, _, s, e, _ in events if k == "quantize")
    g_ms = sum(s.elapsed_time(e) for k, _, s, e, _ in events if k == "gemm")
    g_units = sum(u for k, u, _, _, _ in events if k == "gemm")
    g_launches = sum(1 for k, *_ in events if k == "gemm")
    q_units = sum(u for k, u, _, _, _ in events if k == "quantize")
    q_launches = sum(1 for k, *_ in events if k == "quantize")
    per = {}
    for k, u, s, e, label in events:
        d = per.setdefault(label, [k, u, 0.0, 0])
        d[2] += s.elapsed_time(e)
        d[3] += 1
    breakdown = {}
    for label, (k, u, tot, cnt) in per.items():
        ms = tot / cnt
        breakdown[label] = ({"us": round(ms * 1e3, 1), "TFLOP/s": round(u / (ms * 1e-3) / 1e12, 1)}
                            if k == "gemm" else
                            {"us": round(ms * 1e3, 1), "GB/s": round(u / (ms * 1e-3) / 1e9, 1)})
    step_ms = ms_max / args.steps
    value = ws * step.flops / (step_ms * 1e-3) / 1e12
    gemm_tflops = g_units / (g_ms * 1e-3) / 1e12
    quant_gbs = q_units / (q_ms * 1e-3) / 1e9
    # The GEMM launches are timed one by one with CUDA events (tens to hundreds of us each,
    # inside a region of tens of ms), so the burst peak is the denominator; the sustained
    # one (seconds under the power cap) is reported beside it.
    fp8_peak = pk["bf16"] * FP8_OVER_BF16
    fp8_sus = pk["bf16_sus"] * FP8_OVER_BF16
    traffic = recorded_traffic("mxfp8_gemm")
    e2e = run_e2e(args, m, step, dev, stream, ws)
    graph_ms = run_graph(step, stream, split_steps)
    cal = calibrate(dev)
    # the end-to-end step cannot beat moving its bytes over the host link in both directions
    link_ms = (e2e["h2d_bytes_per_step"] + e2e["d2h_bytes_per_step"]) / (cal["h2d+d2h_GB/s"] * 1e6)
    e2e["host_link_bound_ms_per_step"] = link_ms
    e2e["frac_of_host_link_bound"] = link_ms / e2e["ms_per_step"]
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic (seeded N(0,1) activations with 0.5% x30 outlier channels, "
                "N(0,0.02) weights, N(0,1) gradients; BF16)",
        "config": config_obj(args.tokens),
        "gpu_launches": step.launches * args.steps,
        "quantize": {"GB/s": quant_gbs, "frac_of_hbm": quant_gbs / pk["hbm"],
                     "ms_per_step": q_ms / split_steps,
                     "mode": ("dual (one read, both copies; X and W of a layer in one launch)"
                              if step.dual else "separate"),
                     "bytes_per_elem": DUAL_BYTES_PER_ELEM if step.dual else QBYTES_PER_ELEM,
                     "bytes_per_step": q_units / split_steps,
                     "peak_GB/s": pk["hbm"], "peak_src": pk["src"],
                     "frac_of_copy_this_run": quant_gbs / cal["d2d_GB/s"]},
        "gemm": {"TFLOP/s": gemm_tflops, "frac_of_mxfp8": gemm_tflops / fp8_peak,
                 "frac_of_mxfp8_sustained": gemm_tflops / fp8_sus,
                 "ms_per_step": g_ms / split_steps, "flops_per_step": step.flops},
        "roofline": {"bound": "tensor", "achieved": gemm_tflops, "peak": fp8_peak,
                     "unit": "TFLOP/s", "frac": gemm_tflops / fp8_peak,
                     "traffic": traffic,
                     "kernel": "mxfp8_gemm_2sm_kernel (12 launches per step; 256x384, 256x256 or 256x192 tiles)",
                     "peak_note": f"{pk['src']} bf16 burst {pk['bf16']} x {FP8_OVER_BF16} "
                                  "(nominal FP8:BF16 ratio); burst because every launch is "
                                  "event-timed alone (tens to hundreds of us)",
                     "frac_of_sustained": gemm_tflops / fp8_sus,
                     "flops_per_launch": g_units / g_launches},
        "roofline_quantize": {"bound": "hbm", "achieved": quant_gbs, "peak": pk["hbm"],
                              "unit": "GB/s", "frac": quant_gbs / pk["hbm"],
                              "traffic": recorded_traffic("quantize_dual"),
                              "kernel": "quantize_tile_kernel (dual: one BF16 read, row- and "
                                        "column-wise copies; 8 launches per step)",
                              "peak_note": f"{pk['src']} HBM copy bandwidth",
                              "bytes_per_launch": q_units / q_launches},
        "clocks": clk.summary(),
        "e2e": e2e,
        "per_launch": breakdown,
        "calibration": cal,
        "execution": ("20 launches per step; each layer's wgrad on a second stream beside its "
                      "fprop and dgrad" if args.streams == 2 else
                      "20 launches per step issued on one stream")
                     + ("; programmatic dependent launch off (MXFP8_PDL=0)"
                        if os.environ.get("MXFP8_PDL", "1").startswith("0") else
                        "; kernels launched with programmatic stream serialization"),
        "cuda_graph": {"ms_per_step": graph_ms,
                       "value": ws * step.flops / (graph_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                       "note": "the same step captured once in a CUDA graph and replayed"},
    }
    if rank == 0:
        if not args.no_secondary:
            del step
            torch.cuda.empty_cache()
            line["secondary"] = secondary_obj(m, dev, stream, pk)
        if ws == 1:  # the oracle baseline is timed at N = 1 only
            line["cpu_baseline"] = cpu_baseline_obj()
        print(json.dumps(line), flush=True)


def calibrate(dev, nbytes=512 << 20, reps=10):
    """Copy bandwidths on this GPU in the same run: device to device (read + write bytes, the
    HBM bound of the quantizer) and pinned host memory to and from the device, each way and
    both at once (the bound of the end-to-end step). torch copies, CUDA events, buffers larger
    than L2."""
    a = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    b = torch.empty_like(a)
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def timed_ms(fn):
        # the fastest of three regions: a bound is what the link does at its best (the host
        # link is shared with the rest of the machine, and a region now and then runs slow)
        fn()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) / reps)
        return best

    def both():
        cur = torch.cuda.current_stream()
        s1.wait_stream(cur)
        s2.wait_stream(cur)
        with torch.cuda.stream(s1):
            b.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s2):
            h_out.copy_(a, non_blocking=True)
        cur.wait_stream(s1)
        cur.wait_stream(s2)

    d2d = timed_ms(lambda: b.copy_(a))
    h2d = timed_ms(lambda: b.copy_(h_in, non_blocking=True))
    d2h = timed_ms(lambda: h_out.copy_(a, non_blocking=True))
    bidir = timed_ms(both)
    out = {"d2d_GB/s": 2 * nbytes / (d2d * 1e-3) / 1e9,
           "h2d_GB/s": nbytes / (h2d * 1e-3) / 1e9,
           "d2h_GB/s": nbytes / (d2h * 1e-3) / 1e9,
           "h2d+d2h_GB/s": 2 * nbytes / (bidir * 1e-3) / 1e9,
           "bytes": nbytes, "reps": reps}
    del a, b, h_in, h_out
    torch.cuda.empty_cache()
    return out


def run_e2e(args, m, step, dev, stream, ws):
    """Same step through the public API, with the BF16 inputs copied in from pinned host
    memory and the BF16 results copied back inside the timed region. Copies run on their
    own streams, layer by layer, so that host-to-device copies, compute and device-to-host
    copies of different layers (and of consecutive steps) overlap, as a training loop with
    asynchronous input and output transfers would run them. Events keep every dependency:
    a layer's inputs are overwritten only after the previous step's quantize read them,
    and its outputs only after the previous step's copy-out read them."""
    host_in, host_out = [], []
    for L in step.layers:
        host_in.append([(torch.empty_like(L[key], device="cpu").pin_memory(), L[key])
                        for key in ("x", "w", "dy")])
        host_out.append([(L[key], torch.empty_like(L[key], device="cpu").pin_memory())
                         for key in ("y", "dx", "dw")])
    for layer in host_in:
        for h, d in layer:
            h.copy_(d)
    h2d = sum(h.numel() * h.element_size() for layer in host_in for h, _ in layer)
    d2h = sum(h.numel() * h.element_size() for layer in host_out for _, h in layer)
    # the copies of consecutive steps overlap (see above), so the timed steps include one
    # pipeline fill and drain: enough steps keep that a small part of the region (each is
    # about 6 ms, bound by the host link)
    steps = max(20, args.steps)
    n = len(step.layers)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    in_ready, q_done = [ev() for _ in range(n)], [ev() for _ in range(n)]
    g_done, out_done = [ev() for _ in range(n)], [ev() for _ in range(n)]

    def one():
        for i in range(n):
            s_in.wait_event(q_done[i])  # the previous step has read this layer's inputs
            with torch.cuda.stream(s_in):
                for h, d in host_in[i]:
                    d.copy_(h, non_blocking=True)
            in_ready[i].record(s_in)
        for i, L in enumerate(step.layers):
            stream.wait_event(in_ready[i])
            step.run_quantize(L, stream)
            q_done[i].record(stream)
            stream.wait_event(out_done[i])  # the previous step's outputs have left
            step.run_gemms(L, stream)
            g_done[i].record(stream)
            s_out.wait_event(g_done[i])
            with torch.cuda.stream(s_out):
                for d, h in host_out[i]:
                    h.copy_(d, non_blocking=True)
            out_done[i].record(s_out)

    for _ in range(2):
        one()
    torch.cuda.synchronize()
    # three timed regions of `steps` steps each; the median is reported (the host link is
    # shared with the rest of the machine, and a region now and then runs far slower)
    runs = []
    for _ in range(3):
        barrier(ws)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for _ in range(steps):
            one()
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
        e.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        runs.append(max_over_ranks(s.elapsed_time(e), ws) / steps)
    ms = sorted(runs)[1]
    return {"value": ws * step.flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "steps": steps, "regions_ms_per_step": runs,
            "overlap": "per-layer copy-in, compute and copy-out on three streams"}


def capture_step(step, stream):
    """One step captured in a CUDA graph on a side stream (its buffers stay with `step`)."""
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        step.run(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            step.run(side)
    torch.cuda.synchronize()
    return graph


def run_graph(step, stream, steps):
    """The step captured once in a CUDA graph and replayed `steps` times; ms per step."""
    graph = capture_step(step, stream)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(steps):
        graph.replay()
    e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / steps

def cpu_baseline_obj():
    budget, t0 = 15.0, time.perf_counter()
    ests, secs, desc, flops = [], [], "", 0.0
    i = 0
    while time.perf_counter() - t0 < budget and i < 50:
        s, est, desc, flops = oracle_step_sample(100 + i)
        ests.append(est)
        secs.append(s)
        i += 1
    step_s = float(np.mean(ests))
    return {"value": flops / step_s / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(),
            "kind": "oracle", "sample": f"{i} samples of: {desc}",
            "seconds": time.perf_counter() - t0, "ms_per_step_extrapolated": step_s * 1e3,
            "single_core": cpu_baseline_single_core()}


SINGLE_CORE_CHILD = """
import json, os, sys, time
os.sched_setaffinity(0, {min(os.sched_getaffinity(0))})
sys.path.insert(0, sys.argv[1])
import numpy as np
import bench
t0, ests, flops = time.perf_counter(), [], 0.0
while time.perf_counter() - t0 < 5.0 and len(ests) < 20:
    s, est, desc, flops = bench.oracle_step_sample(200 + len(ests))
    ests.append(est)
step_s = float(np.mean(ests))
print(json.dumps({"value": flops / step_s / 1e12, "samples": len(ests),
                  "ms_per_step_extrapolated": step_s * 1e3}))
"""


def cpu_baseline_single_core():
    """The same oracle sample on one host core (a child process pinned to one CPU, with the
    BLAS and OpenMP pools at one thread), for about 5 s; None if it could not run."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    try:
        r = subprocess.run([sys.executable, "-c", SINGLE_CORE_CHILD, ROOT], env=env,
                           capture_output=True, text=True, timeout=120)
        out = json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.TimeoutExpired, ValueError, IndexError, OSError):
        return None
    return {"value": out["value"], "unit": "TFLOP/s", "cores": 1, "samples": out["samples"],
            "ms_per_step_extrapolated": out["ms_per_step_extrapolated"]}


# ------------------------------------------------------------ other configurations

def _timed_ms(fn, stream, reps, warm=3):
    """Mean ms of `fn` over `reps` back-to-back calls on `stream` (CUDA events)."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(reps):
        fn()
    e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / reps


def _split(run, stream, reps):
    """Runs `run(events)` `reps` times with CUDA events around every launch; returns
    {kind: (ms per rep, units per rep)} and {label: (kind, units, ms)}."""
    run(None)
    torch.cuda.synchronize()
    events = []
    for _ in range(reps):
        run(events)
    torch.cuda.synchronize()
    kinds, labels = {}, {}
    for k, u, s, e, label in events:
        ms = s.elapsed_time(e)
        a = kinds.setdefault(k, [0.0, 0.0])
        a[0] += ms / reps
        a[1] += u / reps
        b = labels.setdefault(label, [k, u, 0.0])
        b[2] += ms / reps
    return kinds, labels


def _gemm_roof(flops, nbytes, ms, pk):
    """TFLOP/s of a GEMM and its fraction of min(tensor peak, arithmetic intensity x HBM)."""
    ai = flops / nbytes
    roof = min(pk["bf16"] * FP8_OVER_BF16, ai * pk["hbm"] * 1e-3)
    tf = flops / (ms * 1e-3) / 1e12
    return {"ms": ms, "TFLOP/s": tf, "flop_per_byte": ai, "roof_TFLOP/s": roof,
            "frac_of_roof": tf / roof}


def measure_moe(m, dev, stream, pk, reps=10):
    """Qwen3-30B-A3B expert layer: 128 experts, 8192 tokens routed top-8 (Zipf 1.1 counts,
    segments padded to 32). Per projection (gate_up 2048 -> 1536, down 768 -> 2048): the
    grouped dual quantize of the routed activations and of the upstream gradient, the
    batched row- and column-wise quantize of the expert weights, and the grouped fprop,
    dgrad and wgrad GEMMs (BF16 out). FLOPs count routed rows only (not the padding)."""
    from mxfp8_block_scaled_05_gb300 import workloads as W
    d = W.moe_expert_layer(dev)
    offs = d["offsets"].to(dev)
    real = int(d["counts"].sum())
    t_rows = int(d["offsets"][-1])
    out = {"experts": int(d["counts"].numel()), "routed_rows": real, "padded_rows": t_rows}
    for proj, x, w, dy in (("gate_up", d["x"], d["w_gate_up"], d["dy_gate_up"]),
                           ("down", d["h"], d["w_down"], d["dy_down"])):
        E, n, k = w.shape
        xq = m.quantize_grouped_dual(x, offs)
        dyq = m.quantize_grouped_dual(dy, offs)
        wr = m.quantize_batched(w, m.ROW)
        wc = m.quantize_batched(w, m.COL)
        y = torch.empty((t_rows, n), dtype=torch.bfloat16, device=dev)
        dx = torch.empty((t_rows, k), dtype=torch.bfloat16, device=dev)
        dw = torch.empty((E, n, k), dtype=torch.bfloat16, device=dev)
        flops = 2.0 * real * n * k
        gemm_bytes = {  # E4M3 operands (+1/32 scales) and the BF16 output
            "fprop": (t_rows * k + E * n * k) * (1 + 1 / 32) + t_rows * n * 2,
            "dgrad": (t_rows * n + E * n * k) * (1 + 1 / 32) + t_rows * k * 2,
            "wgrad": (n + k) * t_rows * (1 + 1 / 32) + E * n * k * 2}

        def run(events, x=x, dy=dy, w=w, xq=xq, dyq=dyq, wr=wr, wc=wc, y=y, dx=dx, dw=dw,
                flops=flops):
            for label, units, fn in (
                    ("quantize x", x.numel() * DUAL_BYTES_PER_ELEM,
                     lambda: m.quantize_grouped_dual(x, offs, *xq, stream=stream)),
                    ("quantize w", w.numel() * 2 * QBYTES_PER_ELEM,
                     lambda: (m.quantize_batched(w, m.ROW, out=wr[0], scales=wr[1], stream=stream),
                              m.quantize_batched(w, m.COL, out=wc[0], scales=wc[1], stream=stream))),
                    ("quantize dy", dy.numel() * DUAL_BYTES_PER_ELEM,
                     lambda: m.quantize_grouped_dual(dy, offs, *dyq, stream=stream)),
                    ("fprop", flops, lambda: m.grouped_gemm(xq[0], xq[1], wr[0], wr[1], offs,
                                                            m.FPROP, out=y, stream=stream)),
                    ("dgrad", flops, lambda: m.grouped_gemm(dyq[0], dyq[1], wc[0], wc[1], offs,
                                                            m.DGRAD, out=dx, stream=stream)),
                    ("wgrad", flops, lambda: m.grouped_gemm(dyq[2], dyq[3], xq[2], xq[3], offs,
                                                            m.WGRAD, out=dw, stream=stream))):
                ev = DenseStep._ev(events, stream, "gemm" if label in gemm_bytes else "quantize",
                                   units, label)
                fn()
                DenseStep._end(events, stream, ev)

        kinds, labels = _split(run, stream, reps)
        res = {"shape": f"{E} x {n} x {k}"}
        for label, (kind, units, ms) in labels.items():
            if kind == "gemm":
                res[label] = _gemm_roof(units, gemm_bytes[label], ms, pk)
            else:
                res[label] = {"ms": ms, "GB/s": units / (ms * 1e-3) / 1e9}
        qms, qb = kinds["quantize"]
        gms, gf = kinds["gemm"]
        res["quantize_GB/s"] = qb / (qms * 1e-3) / 1e9
        res["gemm_TFLOP/s"] = gf / (gms * 1e-3) / 1e12
        res["ms_per_step"] = qms + gms
        out[proj] = res
        del xq, dyq, wr, wc, y, dx, dw
    del d
    torch.cuda.empty_cache()
    return out


def measure_sync(m, dev, stream, pk, reps=3):
    """Weight-synchronization pass of a Qwen3-8B-shaped model: 36 layers x {qkv, o, gate_up,
    down} weights quantized row-wise into the swizzled scale layout, one launch per weight
    (144 launches, 6.95 G elements). One buffer per distinct shape is reused across layers;
    each is larger than L2."""
    from mxfp8_block_scaled_05_gb300 import workloads as W
    shapes = W.sync_weight_shapes()
    bufs = {}
    for _, name, n, k in shapes[:4]:
        w = W.sync_weight(0, name, n, k, dev)
        bufs[name] = (w, torch.empty_like(w, dtype=torch.uint8),
                      torch.empty(m.scale_bytes(n, k), dtype=torch.uint8, device=dev))

    def sync_pass():
        for _, name, n, k in shapes:
            w, q, sc = bufs[name]
            m.quantize(w, m.ROW, m.SWIZZLED, out=q, scales=sc, stream=stream)

    ms = _timed_ms(sync_pass, stream, reps, warm=1)
    elems = sum(n * k for _, _, n, k in shapes)
    gbs = elems * QBYTES_PER_ELEM / (ms * 1e-3) / 1e9
    del bufs
    torch.cuda.empty_cache()
    return {"weights": len(shapes), "elements": elems, "ms": ms, "GB/s": gbs,
            "frac_of_hbm": gbs / pk["hbm"], "launches": len(shapes)}


def measure_sweep(m, dev, stream, pk, reps=5, tokens=None):
    """Micro-batch sweep on the Qwen3-8B gate_up and down shapes: per token count, the same
    step as the headline (dual quantize of X+W and of dY, fprop, dgrad, wgrad) for the two
    layers, with the quantize and GEMM time split by CUDA events around every launch."""
    from mxfp8_block_scaled_05_gb300 import workloads as W
    rows = []
    for t in (tokens or W.SWEEP_TOKENS):
        step = DenseStep(m, W.sweep_layers(t, dev), dev)
        kinds, _ = _split(lambda ev: step.run(stream, ev), stream, reps)
        qms, qb = kinds["quantize"]
        gms, gf = kinds["gemm"]
        rows.append({"tokens": t, "quantize_ms": qms, "gemm_ms": gms,
                     "quantize_GB/s": qb / (qms * 1e-3) / 1e9,
                     "gemm_TFLOP/s": gf / (gms * 1e-3) / 1e12,
                     "gemm_frac_of_mxfp8": gf / (gms * 1e-3) / 1e12 / (pk["bf16"] * FP8_OVER_BF16),
                     "quantize_share": qms / (qms + gms)})
        del step
        torch.cuda.empty_cache()
    return rows


def secondary_obj(m, dev, stream, pk):
    """The other configurations, measured after the headline on the same GPU."""
    t0 = time.perf_counter()
    out = {"moe_qwen3_30b_a3b": measure_moe(m, dev, stream, pk),
           "weight_sync_qwen3_8b": measure_sync(m, dev, stream, pk),
           "microbatch_sweep": measure_sweep(m, dev, stream, pk)}
    out["seconds"] = time.perf_counter() - t0
    out["note"] = ("GEMM fractions against the burst MXFP8 peak (measured bf16 burst x 2); "
                   "MoE GEMMs against min(peak, arithmetic intensity x HBM)")
    return out


def _parse_shapes(text):
    return [tuple(int(v) for v in part.split(",")) for part in text.split(";") if part.strip()]


def measure_gemm_shapes(m, dev, stream, pk, shapes, reps=20, op_name="fprop"):
    """Single dense GEMMs (C = A . B^T, BF16 out) on random operands quantized by the
    library: per shape, the mean launch time back to back and with events around every
    launch; TFLOP/s from 2 M N K."""
    op = {"fprop": m.FPROP, "dgrad": m.DGRAD, "wgrad": m.WGRAD}[op_name]
    g = torch.Generator(device=dev).manual_seed(7)
    rows = []
    for mm, nn, kk in shapes:
        a = torch.randn((mm, kk), generator=g, device=dev).to(torch.bfloat16)
        b = (torch.randn((nn, kk), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        qa, sa = m.quantize(a, m.ROW)
        qb, sb = m.quantize(b, m.ROW)
        c = torch.empty((mm, nn), dtype=torch.bfloat16, device=dev)
        nws = m.gemm_workspace_bytes(mm, nn, kk, op)
        ws = torch.zeros(nws, dtype=torch.uint8, device=dev) if nws else None
        fn = lambda: m.gemm(qa, sa, qb, sb, op, out=c, stream=stream, workspace=ws)
        ms = _timed_ms(fn, stream, reps)
        evs = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        ev_ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)
        flops = 2.0 * mm * nn * kk
        rows.append({"M": mm, "N": nn, "K": kk, "op": op_name, "workspace_bytes": nws,
                     "us_back_to_back": ms * 1e3, "us_event_median": ev_ms * 1e3,
                     "TFLOP/s": flops / (ms * 1e-3) / 1e12,
                     "frac_of_burst": flops / (ms * 1e-3) / 1e12 / (pk["bf16"] * FP8_OVER_BF16)})
        del a, b, qa, sa, qb, sb, c, ws
    torch.cuda.empty_cache()
    return rows


def measure_quantize_shapes(m, dev, stream, pk, shapes, reps=20, mode="dual"):
    """Single quantize launches on N(0,1) BF16 inputs: mean launch time back to back and
    GB/s over the algorithmic bytes (dual: 2 + 2 x 1.03125 B per element; row or col:
    3.03125 B per element)."""
    g = torch.Generator(device=dev).manual_seed(8)
    rows = []
    for r, c in shapes:
        x = torch.randn((r, c), generator=g, device=dev).to(torch.bfloat16)
        if mode == "dual":
            outs = m.quantize_dual(x)
            fn = lambda: m.quantize_dual(x, m.SWIZZLED, *outs, stream=stream)
            per = DUAL_BYTES_PER_ELEM
        else:
            axis = m.ROW if mode == "row" else m.COL
            q, sc = m.quantize(x, axis)
            fn = lambda: m.quantize(x, axis, m.SWIZZLED, out=q, scales=sc, stream=stream)
            per = QBYTES_PER_ELEM
        ms = _timed_ms(fn, stream, reps)
        gbs = r * c * per / (ms * 1e-3) / 1e9
        rows.append({"rows": r, "cols": c, "mode": mode, "us_back_to_back": ms * 1e3,
                     "GB/s": gbs, "frac_of_hbm": gbs / pk["hbm"]})
        del x
    torch.cuda.empty_cache()
    return rows


def run_workload(args):
    """One secondary configuration alone, one JSON line (or one line per shape)."""
    import mxfp8_block_scaled_05_gb300 as m
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    pk = peaks()
    if args.workload == "gemm":
        for row in measure_gemm_shapes(m, dev, stream, pk, _parse_shapes(args.shapes),
                                       reps=args.reps, op_name=args.op):
            print(json.dumps(row), flush=True)
        return
    if args.workload == "quantize":
        for row in measure_quantize_shapes(m, dev, stream, pk, _parse_shapes(args.shapes),
                                           reps=args.reps, mode=args.mode):
            print(json.dumps(row), flush=True)
        return
    if args.workload == "sync":
        line = measure_sync(m, dev, stream, pk, reps=5)
        from mxfp8_block_scaled_05_gb300 import workloads as W
        shapes = W.sync_weight_shapes()
        elems = line["elements"]
        # the same pass with the FP8 block-wise recipe (128 x 128 blocks): 2 B read + 1 B
        # written per element, plus one float per block
        bw_bytes = elems * (3.0 + 4.0 / (128 * 128))
        ws = {name: W.sync_weight(0, name, n, k, dev) for _, name, n, k in shapes[:4]}
        for key, st in (("blockwise_pow2", m.BW_POW2), ("blockwise_fp32", m.BW_FP32)):
            outs = {name: (torch.empty_like(w, dtype=torch.uint8),
                           torch.empty(((w.shape[0] + 127) // 128, (w.shape[1] + 127) // 128),
                                       dtype=torch.float32, device=dev))
                    for name, w in ws.items()}

            def bw_pass(st=st, outs=outs):
                for _, name, n, k in shapes:
                    q, si = outs[name]
                    m.quantize_blockwise(ws[name], st, out=q, scale_inv=si, stream=stream)

            bms = _timed_ms(bw_pass, stream, 5)
            line[key] = {"ms": bms, "GB/s": bw_bytes / (bms * 1e-3) / 1e9,
                         "frac_of_hbm": bw_bytes / (bms * 1e-3) / 1e9 / pk["hbm"]}
        print(json.dumps({"workload": "weight-sync quantize pass, Qwen3-8B shapes", **line}),
              flush=True)
    elif args.workload == "moe":
        print(json.dumps({"workload": "Qwen3-30B-A3B expert layer",
                          **measure_moe(m, dev, stream, pk, reps=20)}), flush=True)
    elif args.workload == "sweep":
        for row in measure_sweep(m, dev, stream, pk, reps=10):
            print(json.dumps(row), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--tokens", type=int, default=4096)
    ap.add_argument("--workload", choices=("dense", "moe", "sync", "sweep", "gemm", "quantize"),
                    default="dense")
    ap.add_argument("--shapes", default="4096,4096,4096",
                    help="--workload gemm: M,N,K[;M,N,K...]; --workload quantize: R,C[;R,C...]")
    ap.add_argument("--op", choices=("fprop", "dgrad", "wgrad"), default="fprop")
    ap.add_argument("--mode", choices=("dual", "row", "col"), default="dual")
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--quant", choices=("dual", "separate"), default="dual",
                    help="quantize each tensor once for both copies (dual) or per copy")
    ap.add_argument("--streams", type=int, choices=(1, 2), default=2,
                    help="2 (default): each layer's wgrad on a second stream beside its fprop "
                         "and dgrad; 1: every launch on one stream")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the secondary configurations after the headline line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, rank, int(os.environ.get("WORLD_SIZE", "1")))
        return
    import __graft_entry__
    __graft_entry__.build()
    rank, ws = dist_setup(args.gpus)
    try:
        if args.workload != "dense":
            if rank == 0:
                run_workload(args)
        else:
            run_ours(args, rank, ws)
    finally:
        if ws > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
