#!/usr/bin/env python
"""Benchmark of the decode-step linear set on GB300.

One step = the decode linears of a Qwen2-7B-shaped model: 28 layers x
(fused QKV 4608x3584, O 3584x3584, fused gate/up 37888x3584, down 3584x18944)
plus the lm_head 152064x3584, per-row INT4 weights, M tokens (default 1),
each linear one fused quantize + GEMV launch of libw4a8.so.  The 113
launches are chained with programmatic dependent launch and replayed from a
CUDA graph.  As in a decoder, each linear reads what the previous one wrote:
its x[M][K] is the first M*K values of the previous linear's output (the
attention, norm and activation between them are not part of this path);
the first linear reads the step's input x[M][3584] ~ N(0, 1).  Weights
(3.5 GB) are synthetic (seeded N(0, 0.02) draws quantized on the GPU) and
resident in HBM; they exceed L2, so no L2 flush is needed between steps.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle
instead (host cores, bounded sample per step).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from bit_quantized_decode_gb300 import workloads as wl  # noqa: E402

METRIC = "W4A8 GEMV achieved HBM GB/s (% of GB300 peak); 7B decode-step linear ms"
FALLBACK_PEAK_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0          # GB300 HBM3e, nominal (~8 TB/s)
READ_PEAK_BYTES = 4 << 30         # the pure-read probe streams this many bytes per launch


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--M", type=int, default=1, help="tokens sharing one weight pass (1..16)")
    p.add_argument("--layers", type=int, default=wl.QWEN7B_LAYERS, help="layers in the step (28 = full model)")
    p.add_argument("--no-lm-head", action="store_true")
    p.add_argument("--no-pdl", action="store_true")
    p.add_argument("--chain", action="store_true",
                   help="one chained launch per step (w4a8_linear_chain) instead of one PDL launch per linear")
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--weights", choices=("w4", "w4a32", "w8a32"), default="w4",
                   help="the step's linear path: per-row INT4 x INT8 activations on DP4A (default), or a "
                        "weight-only path on float activations (INT4 unpacked to float, per-row INT8; M <= 2)")
    p.add_argument("--decoder", choices=("off", "fused", "unfused"), default="off",
                   help="run the step with the RMSNorm, SwiGLU and residual adds of a decoder layer around "
                        "the linears: fused into them, or as separate kernels")
    p.add_argument("--suite", action="store_true",
                   help="instead of the step line: every GEMV of the single, 7B-layer, Gemma Q4_0 and lm_head "
                        "workloads on its own, then the full step at M = 1, 2, 4, 8, 16 (one JSON line each)")
    p.add_argument("--suite-ms", default="1,2,4,8,16", help="token counts of the suite's full-step lines")
    p.add_argument("--suite-only-steps", action="store_true", help="suite: skip the single-GEMV lines")
    p.add_argument("--suite-gemvs", default="",
                   help="suite: only these single GEMVs, comma-separated, each a workload (gemma_q4_0) or "
                        "workload:linear (lm_head:lm_head_q6g32); default all")
    p.add_argument("--suite-gemv-ms", default="1",
                   help="token counts of the suite's single-GEMV lines (the multi-token verify case: M tokens "
                        "sharing one pass over the weights)")
    p.add_argument("--suite-ablation-ms", default="1",
                   help="token counts of the suite's weight-only ablation lines (INT4 DP4A, INT4 float unpack, "
                        "INT8 weight-only; at most 2 tokens: the float activations of the K = 18944 linear "
                        "live in shared memory)")
    p.add_argument("--suite-decoder-ms", default="1,16",
                   help="token counts of the suite's decoder-step lines (operators unfused, then fused)")
    p.add_argument("--independent-x", action="store_true",
                   help="every linear reads its own static input buffer instead of the previous output")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--per-linear", action="store_true", help="also time each linear kind on its own")
    p.add_argument("--ref-budget-s", type=float, default=120.0, help="reference arm: total CPU seconds")
    p.add_argument("--tune", action="append", default=[], metavar="KEY=VALUE",
                   help="launch tuning passed to w4_set_tuning: blocks_per_sm, max_stages, grid_blocks")
    p.add_argument("--profile", action="store_true",
                   help="profiler mode: eager step, graph warm-up and timed replays only (no e2e, no CPU "
                        "baseline, no clock sampling); the launch order is fixed: one eager step, then "
                        "warmup + steps graph replays")
    return p.parse_args(argv)


# ----------------------------------------------------------------- workload
def step_linears(layers: int, lm_head: bool):
    seq = [(layer, lin) for layer in range(layers) for lin in wl.qwen7b_layer()]
    if lm_head:
        seq.append((layers, wl.qwen7b_lm_head()))
    return seq


def algorithmic_bytes(lin, M: int) -> int:
    """Bytes one decode linear must move: its weights in their packed format
    (per-row INT4: 0.5 B a weight + a 4-byte scale a row; Q4_0: 18 B per 32
    weights; i8g32: 1 B a weight + 2 B per 32; q6g32: 26 B per 32), the bias,
    fp32 x and fp32 y."""
    if lin.fmt in ("w4", "w4a32"):
        w = lin.N * lin.K // 2 + 4 * lin.N
    elif lin.fmt == "w8a32":
        w = lin.N * lin.K + 4 * lin.N
    elif lin.fmt == "q4_0":
        w = lin.N * (lin.K // 32) * 18
    elif lin.fmt == "q6g32":
        w = lin.N * (lin.K // 32) * 26
    else:
        w = lin.N * lin.K + lin.N * (lin.K // 32) * 2
    return w + (4 * lin.N if lin.bias else 0) + 4 * M * lin.K + 4 * M * lin.N


def workload_config(args, n_gpus):
    return {
        "workload": (f"qwen2-7b decode-step linear set: {args.layers} layers x (fused QKV 4608x3584, "
                     f"O 3584x3584, fused gate/up 37888x3584, down 3584x18944)"
                     + ("" if args.no_lm_head else " + lm_head 152064x3584")
                     + {"w4": ", per-row INT4 weights, INT8 per-token activations",
                        "w4a32": ", per-row INT4 weights unpacked to float, float activations",
                        "w8a32": ", per-row INT8 weights, float activations"}[args.weights]
                     + f", M={args.M}"),
        "M": args.M,
        "layers": args.layers,
        "lm_head": not args.no_lm_head,
        "linears_per_step": 4 * args.layers + (0 if args.no_lm_head else 1),
        "l2": "inputs larger than L2 (3.5 GB of weights per step), no flush",
        "dataflow": ("independent static inputs" if args.independent_x else
                     "each linear reads the previous linear's output (first M*K values)"),
        "parallelism": f"replicas x{n_gpus}",
    } | ({} if args.decoder == "off" else {
        "decoder": args.decoder,
        "dataflow": ("decoder layers: RMSNorm -> QKV -> O (+ residual) -> RMSNorm -> gate/up -> SwiGLU -> down "
                     "(+ residual); final RMSNorm -> lm_head; O reads the first M*3584 QKV outputs"),
        "operators": ("fused into the linears (norm prologue, SwiGLU and residual epilogues)"
                      if args.decoder == "fused" else "separate kernels (w4_rmsnorm, w4_glu, w4_add)"),
    })


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_PEAK_GBS, "fallback"


def read_peak(device, stream, reps: int = 10):
    """Pure-read HBM bandwidth of this device, GB/s: the best of `reps`
    launches of the library's read probe (w4_hbm_read) over a 4 GiB buffer,
    timed with CUDA events on `stream`.  [310B-Gemma4] §4.1 bounds a weight
    stream by the measured pure read bandwidth, which differs from a copy."""
    import torch

    from bit_quantized_decode_gb300 import _lib
    buf = torch.empty(READ_PEAK_BYTES, dtype=torch.uint8, device=device)
    sink = torch.zeros(1, dtype=torch.int32, device=device)
    best = 0.0
    with torch.cuda.stream(stream):
        for _ in range(2):
            _lib.hbm_read(buf, sink, stream)
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            _lib.hbm_read(buf, sink, stream)
            e1.record(stream)
            e1.synchronize()
            best = max(best, READ_PEAK_BYTES / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del buf
    return best


def roofline_fracs(achieved: float, peak_copy: float, peak_read) -> dict:
    """The achieved rate against the three denominators: the driver's measured
    copy peak (read+write bytes), the pure-read peak measured in this run, and
    the nominal HBM rate."""
    out = {"frac": round(achieved / peak_copy, 4), "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
           "nominal": NOMINAL_HBM_GBS}
    if peak_read:
        out["peak_read"] = round(peak_read, 1)
        out["frac_read"] = round(achieved / peak_read, 4)
    return out


def profiled_traffic(alg_bytes_per_launch: float, chain: bool):
    """DRAM bytes per launch from the committed ncu summary of this path: the
    measured traffic / algorithmic ratio times this launch's algorithmic
    bytes, if the summary was taken on the current kernel sources (else None)."""
    try:
        from bit_quantized_decode_gb300 import build
        digest = build.kernel_digest()
        name = "stream_chain_w4_qwen7b_step.md" if chain else "stream_linear_w4_fused_qwen7b_step.md"
        vals = {}
        with open(os.path.join(ROOT, "profiles", name)) as f:
            for line in f:
                if line.startswith("- ") and ":" in line:
                    k, v = line[2:].split(":", 1)
                    vals[k.strip()] = v.strip().strip("`")
        if vals.get("source_digest") != digest:
            return None
        return round(float(vals["traffic_over_algorithmic"]) * alg_bytes_per_launch)
    except Exception:
        return None


# ------------------------------------------------------------- clock sampler
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 10:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]),
                             "util": float(parts[4]) if parts[4] not in ("[N/A]", "N/A") else 100.0,
                             "hw": parts[6], "hwt": parts[7], "swt": parts[8], "pcap": parts[9]})
            except ValueError:
                continue
        if not rows:
            return None
        loaded = [r for r in rows if r["util"] >= 50] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": max(r["max"] for r in loaded),
                "reasons": sorted(reasons), "samples": len(loaded)}


# --------------------------------------------------------- oracle baseline
def oracle_layer_sample(M: int, seed: int = 1, row_fraction: float = 1.0):
    """Host-side inputs for the first rows of each linear of one Qwen2-7B
    layer, N(0, 0.02) weights quantized by the oracle."""
    import oracle
    g = wl.rng(seed)
    layer = []
    for lin in wl.qwen7b_layer():
        n = max(8, int(lin.N * row_fraction))
        W = wl.weights(g, n, lin.K)
        q, sw = oracle.quantize_rows_int4(W)
        del W
        layer.append((lin, oracle.pack_int4(q), sw, wl.activations(g, M, lin.K), wl.bias(g, n)))
    return layer


def time_oracle(layer, M: int, min_seconds: float, row_fraction: float = 1.0):
    """Run the oracle's decode linear over (a row slice of) the layer until
    min_seconds of CPU time have passed.  Returns (GB/s, seconds, reps)."""
    import oracle
    work = []
    for lin, packed, sw, x, b in layer:
        n = min(packed.shape[0], max(8, int(lin.N * row_fraction)))
        work.append((packed[:n], sw[:n], x, b[:n], n, lin))
    nbytes = sum(n * lin.K // 2 + 8 * n + 4 * M * lin.K + 4 * M * n for _, _, _, _, n, lin in work)
    reps, t0 = 0, time.perf_counter()
    while True:
        for packed, sw, x, b, n, lin in work:
            oracle.w4a8_linear(packed, sw, x, b)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    return nbytes * reps / dt / 1e9, dt, reps


def oracle_gemv_baseline(lin, M: int, seconds: float = 1.5, seed: int = 3) -> dict:
    """The oracle (single-threaded C) on a row slice of one decode linear of
    the suite: N(0, sigma) weights drawn on the host and quantized by the
    oracle in the linear's format, x ~ N(0, 1); the timed work is the whole
    linear (activation quantization, integer GEMV, epilogue).  GB/s counts the
    slice's algorithmic bytes.  A baseline only."""
    import dataclasses

    import oracle
    g = wl.rng(seed)
    n = min(lin.N, 256)
    while True:
        sl = dataclasses.replace(lin, shards=(n,))
        W = wl.weights(g, n, lin.K, lin.sigma)
        x = wl.activations(g, M, lin.K)
        b = wl.bias(g, n) if lin.bias else None
        if lin.fmt == "w4":
            q, sw = oracle.quantize_rows_int4(W)
            packed = oracle.pack_int4(q)

            def run():
                oracle.w4a8_linear(packed, sw, x, b)
        elif lin.fmt == "q4_0":
            blocks = oracle.quantize_q4_0(W)

            def run():
                qx, sx = oracle.quantize_act_int8(x)
                oracle.gemv_q4_0(blocks, qx, sx, b)
        else:                            # i8g32, and q6g32 (the same values and arithmetic)
            qi, d = oracle.quantize_i8g32(W)

            def run():
                qx, sx = oracle.quantize_act_int8(x)
                oracle.gemv_i8g32(qi, d, qx, sx, b)
        t0 = time.perf_counter()
        run()
        dt = time.perf_counter() - t0
        cap = min(lin.N, max(256, (1 << 25) // lin.K))     # at most ~32 M weights drawn on the host
        if dt * 4 >= seconds or n >= cap:
            break
        n = min(cap, n * min(16, max(2, int(seconds / 4 / max(dt, 1e-6)))))
    reps, t0 = 0, time.perf_counter()
    while True:
        run()
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    gbs = algorithmic_bytes(sl, M) * reps / dt / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "host_cpus": os.cpu_count(), "kind": "oracle",
            "sample": f"rows 0..{n} of {lin.N} ({lin.fmt}, K={lin.K}), M={M}, {reps} passes in {dt:.2f} s"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: host cores, bounded sample per step."""
    if rank != 0:
        return 0
    M = max(1, min(16, args.M))
    layer_bytes = sum(algorithmic_bytes(lin, M) for lin in wl.qwen7b_layer())
    # size each step so that warmup + steps fit the budget at the oracle's speed
    gbs_est, _, _ = time_oracle(oracle_layer_sample(M, row_fraction=0.005), M, 0.0, row_fraction=0.005)
    per_step_s = args.ref_budget_s / max(1, args.steps + args.warmup)
    frac = min(1.0, max(0.002, per_step_s * gbs_est * 1e9 / layer_bytes))
    layer = oracle_layer_sample(M, row_fraction=frac)
    for _ in range(args.warmup):
        time_oracle(layer, M, 0.0, frac)
    times, nbytes = [], 0
    for _ in range(args.steps):
        gbs, dt, reps = time_oracle(layer, M, 0.0, frac)
        times.append(dt)
        nbytes = gbs * dt * 1e9
    total = sum(times)
    value = nbytes * len(times) / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / len(times), 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32 (int4 x int8)",
        "data": "synthetic", "config": workload_config(args, args.gpus),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"rows 0..{frac:.4f}*N of each linear of one Qwen2-7B layer (QKV, O, gate/up, "
                                   f"down), M={M}, through the single-threaded C oracle, per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- our arm
def build_weights(args, device, fmt: str = "w4"):
    """The step's linears with resident repacked weights: [(layer, lin, QuantLinear)]."""
    import dataclasses

    import torch

    from bit_quantized_decode_gb300 import QuantLinear
    out = []
    seed = 1000
    for layer, lin in step_linears(args.layers, not args.no_lm_head):
        lin = dataclasses.replace(lin, fmt=fmt)
        shards = []
        for rows in lin.shards:
            shards.append(wl.torch_normal((rows, lin.K), lin.sigma, seed, device))
            seed += 1
        biases = [wl.torch_normal((rows,), 0.01, seed + i, device) for i, rows in enumerate(lin.shards)]
        seed += len(lin.shards)
        out.append((layer, lin, QuantLinear.from_float(fmt, shards, biases)))
        del shards
    torch.cuda.synchronize()
    return out


def make_buffers(weights, M: int, independent_x: bool, device, seed: int = 5000):
    """Per-linear activation buffers for M tokens.  Returns (items, x_in, y_out):
    x_in is the step's input, y_out the last linear's output (the logits with
    the lm_head); with independent_x, x_in and y_out hold every linear's input
    and output instead.  items: (layer, lin, ql, x, y, qx, sx)."""
    import torch
    if independent_x:
        x_all = torch.empty(sum(M * lin.K for _, lin, _ in weights), dtype=torch.float32, device=device)
        y_all = torch.empty(sum(M * lin.N for _, lin, _ in weights), dtype=torch.float32, device=device)
    else:
        x_all = torch.empty(M * weights[0][1].K, dtype=torch.float32, device=device)
    items = []
    xo = yo = 0
    prev_y = None
    for layer, lin, ql in weights:
        if independent_x or prev_y is None:
            x = x_all[xo: xo + M * lin.K].view(M, lin.K)
            x.copy_(wl.torch_normal((M, lin.K), 1.0, seed, device))
            xo += M * lin.K
        else:
            if prev_y.numel() < M * lin.K:
                raise ValueError(f"{lin.name}: the previous output has fewer than M*K values")
            x = prev_y.view(-1)[: M * lin.K].view(M, lin.K)
        seed += 1
        if independent_x:
            y = y_all[yo: yo + M * lin.N].view(M, lin.N)
            yo += M * lin.N
        else:
            y = torch.empty((M, lin.N), dtype=torch.float32, device=device)
        qx = torch.empty((M, lin.K), dtype=torch.int8, device=device)
        sx = torch.empty(M, dtype=torch.float32, device=device)
        items.append((layer, lin, ql, x, y, qx, sx))
        prev_y = y
    torch.cuda.synchronize()
    y_out = y_all if independent_x else prev_y.view(-1)
    return items, x_all, y_out


def build_step(args, device):
    return make_buffers(build_weights(args, device, args.weights), args.M, args.independent_x, device)


NORM_EPS = 1e-6


def build_decoder(args, device):
    """The step with the operators a decoder layer runs around its linears:
    per layer h += O(QKV(RMSNorm(h))[:, :3584]) and h += down(SiLU(gate) * up
    of RMSNorm(h)), then logits = lm_head(RMSNorm(h)); attention is out of the
    path (O reads the first M*3584 values of the QKV output in its place).
    decoder="fused": RMSNorm in the quantize prologue, SwiGLU and the residual
    add in the epilogue (gate/up paired per tile): 4 launches a layer + 1.
    decoder="unfused": the same arithmetic with w4_rmsnorm, w4_glu and w4_add
    as separate kernels between plain linears: 9 launches a layer + 2.
    The step input h_in (residual stream, N(0, 4^2)) is read, never written,
    so replays are identical.  Returns (ops, h_in, logits, bytes_per_step);
    each op takes the launch flags."""
    import torch

    from bit_quantized_decode_gb300 import QuantLinear, _lib
    fused = args.decoder == "fused"
    M = args.M
    H = wl.QWEN7B_HIDDEN
    seed = 1000
    F32 = torch.float32

    def norm_weight():
        nonlocal seed
        seed += 1
        return (1.0 + wl.torch_normal((H,), 0.1, seed, device)).contiguous()

    def linear(lin, paired=False):
        nonlocal seed
        shards = [wl.torch_normal((rows, lin.K), lin.sigma, seed + i, device) for i, rows in enumerate(lin.shards)]
        seed += len(lin.shards)
        biases = [wl.torch_normal((rows,), 0.01, seed + i, device) for i, rows in enumerate(lin.shards)]
        seed += len(lin.shards)
        return QuantLinear.from_float("w4", shards, biases, glu_pairs=paired)

    def buf(*shape, dtype=F32):
        return torch.empty(*shape, dtype=dtype, device=device)

    h_in = wl.torch_normal((M, H), 4.0, 4999, device).contiguous()
    h = buf(M, H)
    xn = buf(M, H)
    ops = []
    bytes_per_step = 0
    for layer in range(args.layers):
        qkv_l, o_l, gu_l, down_l = wl.qwen7b_layer()
        g_attn, g_mlp = norm_weight(), norm_weight()
        qkv, o, down = linear(qkv_l), linear(o_l), linear(down_l)
        gu = linear(gu_l, paired=fused)
        h_src = h_in if layer == 0 else h
        y_qkv = buf(M, qkv_l.N)
        x_o = y_qkv.view(-1)[: M * H].view(M, H)
        act = buf(M, wl.QWEN7B_INTERMEDIATE)
        q1, q2, q3, q4 = buf(M, H, dtype=torch.int8), buf(M, H, dtype=torch.int8), \
            buf(M, H, dtype=torch.int8), buf(M, down_l.K, dtype=torch.int8)
        s1, s2, s3, s4 = buf(M), buf(M), buf(M), buf(M)
        if fused:
            ops += [
                lambda f, a=h_src, y=y_qkv, q=q1, s=s1, L=qkv, g=g_attn: L(a, y, q, s, f, norm=g, eps=NORM_EPS),
                lambda f, a=x_o, r=h_src, q=q2, s=s2, L=o: L(a, h, q, s, f, residual=r),
                lambda f, y=act, q=q3, s=s3, L=gu, g=g_mlp: L(h, y, q, s, f, norm=g, eps=NORM_EPS,
                                                               glu=_lib.W4_GLU_SILU),
                lambda f, a=act, q=q4, s=s4, L=down: L(a, h, q, s, f, residual=h),
            ]
        else:
            y_o = buf(M, H)
            y_gu = buf(M, gu_l.N)
            y_d = buf(M, H)
            ops += [
                lambda f, a=h_src, g=g_attn: _lib.w4_rmsnorm(a, g, NORM_EPS, xn, f),
                lambda f, y=y_qkv, q=q1, s=s1, L=qkv: L(xn, y, q, s, f),
                lambda f, y=y_o, a=x_o, q=q2, s=s2, L=o: L(a, y, q, s, f),
                lambda f, a=h_src, y=y_o: _lib.w4_add(a, y, h, f),
                lambda f, g=g_mlp: _lib.w4_rmsnorm(h, g, NORM_EPS, xn, f),
                lambda f, y=y_gu, q=q3, s=s3, L=gu: L(xn, y, q, s, f),
                lambda f, y=y_gu: _lib.w4_glu(y, _lib.W4_GLU_SILU, act, f),
                lambda f, y=y_d, q=q4, s=s4, L=down: L(act, y, q, s, f),
                lambda f, y=y_d: _lib.w4_add(h, y, h, f),
            ]
        # the linears' bytes, plus what the fused operators must read: the norm
        # weights and the residual stream (the gated output is I values, not 2I)
        for lin in (qkv_l, o_l, gu_l, down_l):
            bytes_per_step += algorithmic_bytes(lin, M)
        bytes_per_step += 2 * 4 * H + 2 * 4 * M * H - 4 * M * wl.QWEN7B_INTERMEDIATE
    head_l = wl.qwen7b_lm_head()
    head = linear(head_l)
    g_final = norm_weight()
    logits = buf(M, head_l.N)
    qh, sh = buf(M, H, dtype=torch.int8), buf(M)
    h_last = h if args.layers > 0 else h_in
    if not args.no_lm_head:
        if fused:
            ops.append(lambda f: head(h_last, logits, qh, sh, f, norm=g_final, eps=NORM_EPS))
        else:
            ops.append(lambda f: _lib.w4_rmsnorm(h_last, g_final, NORM_EPS, xn, f))
            ops.append(lambda f: head(xn, logits, qh, sh, f))
        bytes_per_step += algorithmic_bytes(head_l, M) + 4 * H
    torch.cuda.synchronize()
    return ops, h_in.view(-1), (logits if not args.no_lm_head else h).view(-1), bytes_per_step


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest of every rank's value (identity on one process)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step: int, steps: int, world: int, t_max_ms: float) -> float:
    """Weak scaling: every rank streams its own copy of the step."""
    return world * bytes_per_step * steps / (t_max_ms / 1e3) / 1e9


def run_ours(args, rank, world, local_rank):
    import torch

    from bit_quantized_decode_gb300 import W4_FLAG_PDL, LinearChain, W4Error, _lib
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    _lib.load()
    _lib.clear_device_error()
    tuning = {}
    for kv in args.tune:
        k, v = kv.split("=")
        _lib.set_tuning(k, int(v))
        tuning[k] = int(v)
    M = args.M
    pdl_flag = 0 if args.no_pdl else W4_FLAG_PDL
    if args.decoder != "off":
        ops, x_all, y_all, bytes_per_step = build_decoder(args, dev)
        items = []
        launches = len(ops)
    else:
        items, x_all, y_all = build_step(args, dev)
        bytes_per_step = sum(algorithmic_bytes(lin, M) for _, lin, *_ in items)
        launches = len(items)
        ops = [lambda f, it=it: it[2](it[3], it[4], it[5], it[6], flags=f) for it in items]

    stream = torch.cuda.Stream(device=dev)

    def step_per_linear():
        for i, op in enumerate(ops):
            op(pdl_flag if i > 0 else 0)

    # one chained launch per step (at most W4_MAX_CHAIN linears per launch)
    chains = []
    if args.chain and args.decoder == "off" and args.weights == "w4":
        try:
            for c0 in range(0, len(items), _lib.W4_MAX_CHAIN):
                part = items[c0: c0 + _lib.W4_MAX_CHAIN]
                chains.append(LinearChain([(ql, x, y, qx, sx) for _, _, ql, x, y, qx, sx in part], M))
            with torch.cuda.stream(stream):
                for ch in chains:
                    ch()
            torch.cuda.synchronize()
        except W4Error as e:
            if e.status != 2:          # anything but "does not fit" is a real failure
                raise
            chains = []
    launches = len(chains) if chains else launches

    def step():
        if chains:
            for ch in chains:
                ch()
        else:
            step_per_linear()

    with torch.cuda.stream(stream):
        step()                     # eager run: sets kernel attributes, checks the path
    torch.cuda.synchronize()
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        torch.cuda.synchronize()

    def replay():
        if graph is not None:
            graph.replay()
        else:
            step()

    def barrier():
        if dist is not None:
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank)
    if not args.profile:
        sampler.start()
        time.sleep(0.3)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    elapsed_ms = ev0.elapsed_time(ev1)
    if elapsed_ms < 400 and not args.profile:
        time.sleep(0.2)
    clocks = sampler.stop()
    err = _lib.device_error()
    if err:
        raise RuntimeError(f"device error word {err:#x} after the timed region")

    t_max = max_over_ranks(elapsed_ms, dist, dev)
    ms_per_step = t_max / args.steps
    value = whole_job_gbs(bytes_per_step, args.steps, world, t_max)

    if args.profile:
        if rank == 0:
            print(json.dumps({"profile": True, "chain": bool(chains), "tuning": tuning or "auto",
                              "ms_per_step": elapsed_ms / args.steps,
                              "GB/s": bytes_per_step * args.steps / (elapsed_ms / 1e3) / 1e9,
                              "launches_per_step": launches}), flush=True)
        return 0

    # ---- end to end: pinned host inputs in, results out, every step
    e2e_steps = args.e2e_steps or max(3, min(args.steps, 200))
    x_host = torch.empty(x_all.numel(), dtype=torch.float32, pin_memory=True)
    x_host.copy_(x_all.cpu())
    y_host = torch.empty(y_all.numel(), dtype=torch.float32, pin_memory=True)
    with torch.cuda.stream(stream):
        for _ in range(2):
            x_all.copy_(x_host, non_blocking=True)
            replay()
            y_host.copy_(y_all, non_blocking=True)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            x_all.copy_(x_host, non_blocking=True)
            replay()
            y_host.copy_(y_all, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    e2e_value = whole_job_gbs(bytes_per_step, e2e_steps, world, e2e_ms)

    # ---- optional: each linear kind on its own (rotating over the layers' copies)
    per_linear = None
    if args.per_linear and rank == 0:
        per_linear = {}
        for name in ("qkv", "o", "gate_up", "down", "lm_head"):
            sel = [it for it in items if it[1].name == name]
            if not sel:
                continue
            reps = max(1, 200 // len(sel))
            with torch.cuda.stream(stream):
                for it in sel:
                    it[2](it[3], it[4], it[5], it[6])
                a0 = torch.cuda.Event(enable_timing=True)
                a1 = torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                for _ in range(reps):
                    for it in sel:
                        it[2](it[3], it[4], it[5], it[6])
                a1.record(stream)
            torch.cuda.synchronize()
            us = a0.elapsed_time(a1) * 1e3 / (reps * len(sel))
            b = algorithmic_bytes(sel[0][1], M)
            per_linear[name] = {"us": round(us, 3), "GB/s": round(b / us / 1e3, 1), "bytes": b}

    if rank != 0:
        return 0

    cpu_baseline = None
    if not args.no_cpu_baseline:
        layer = oracle_layer_sample(M)
        gbs, dt, reps = time_oracle(layer, M, 10.0)
        cpu_baseline = {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "host_cpus": os.cpu_count(),
                        "kind": "oracle",
                        "sample": (f"one Qwen2-7B layer (QKV, O, gate/up, down; N(0,0.02) weights drawn on the "
                                   f"host and quantized by the oracle), M={M}, single-threaded C oracle, "
                                   f"{reps} passes in {dt:.1f} s")}

    peak, peak_kind = measured_peak()
    peak_rd = read_peak(dev, stream)
    achieved = value / world
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"w4": "int32 (int4 x int8 dp4a)", "w4a32": "f32 (int4 weights unpacked to float)",
                  "w8a32": "f32 (int8 weights, float activations)"}[args.weights],
        "data": "synthetic",
        "config": workload_config(args, world),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     **roofline_fracs(achieved, peak, peak_rd),
                     "traffic": profiled_traffic(bytes_per_step / launches, bool(chains)),
                     "peak_kind": peak_kind,
                     "peak_read_kind": "measured in this run: best of 10 w4_hbm_read launches over 4 GiB",
                     "kernel": ("stream_linear_kernel<W4, M, fused, chain> (one launch per step: the whole linear set)"
                                if chains else
                                "stream_linear_kernel<W4, M, fused> (one launch per linear; bytes and time per launch "
                                "averaged over the step)")},
        "cpu_baseline": cpu_baseline,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(x_all.numel() * 4), "d2h_bytes_per_step": int(y_all.numel() * 4)},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
        "bytes_per_step": bytes_per_step,
        "tuning": tuning or "auto",
        "path": "chain" if chains else "per-linear launches (PDL)",
    }
    if per_linear is not None:
        line["per_linear"] = per_linear
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------- suite
L2_BYTES = 129e6


def _timed_graph(fn, stream, steps: int, warmup: int) -> float:
    """ms per replay of a CUDA graph of fn() on `stream` (CUDA events)."""
    import torch
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    with torch.cuda.stream(stream):
        for _ in range(max(3, warmup)):
            g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def suite_gemv(wname: str, lin, M: int, device, stream, steps: int, warmup: int, peak: float,
               peak_read=None) -> dict:
    """One decode linear timed on its own: back-to-back fused launches (PDL)
    rotating over enough distinct weight copies (>= 4, > 2.5x L2 in all)
    that L2 cannot serve the weights."""
    import math

    import torch

    from bit_quantized_decode_gb300 import W4_FLAG_PDL, QuantLinear
    b = algorithmic_bytes(lin, M)
    wbytes = b - 4 * M * (lin.K + lin.N)
    copies = max(4, math.ceil(2.5 * L2_BYTES / wbytes))
    qls = []
    seed = 7000 + lin.N + lin.K
    for c in range(copies):
        shards = [wl.torch_normal((rows, lin.K), lin.sigma, seed + 31 * c + i, device) for i, rows in enumerate(lin.shards)]
        biases = ([wl.torch_normal((rows,), 0.01, seed + 31 * c + 17 + i, device) for i, rows in enumerate(lin.shards)]
                  if lin.bias else None)
        qls.append(QuantLinear.from_float(lin.fmt, shards, biases))
        del shards
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn((M, lin.K), generator=g, device=device, dtype=torch.float32)
    if wname == "w4a8_single":           # 0.1% of the entries scaled by 20 (seeded choice)
        n_out = max(1, (M * lin.K) // 1000)
        idx = torch.randperm(M * lin.K, generator=g, device=device)[:n_out]
        x.view(-1)[idx] *= 20.0
    y, qx, sx = qls[0].buffers(M)

    def run():
        for i, ql in enumerate(qls):
            ql(x, y, qx, sx, flags=W4_FLAG_PDL if i else 0)

    reps = max(3, min(steps, int(2e5 / copies)))
    ms = _timed_graph(run, stream, reps, warmup)
    us = ms * 1e3 / copies
    gbs = b / us / 1e3
    del qls
    torch.cuda.synchronize()
    return {"suite": wname, "linear": lin.name, "fmt": lin.fmt, "N": lin.N, "K": lin.K, "M": M,
            "us_per_gemv": round(us, 3), "GB/s": round(gbs, 1), **roofline_fracs(gbs, peak, peak_read),
            "bytes": b, "weight_copies": copies, "replays": reps}


def suite_selected(spec: str, wname: str, lname: str) -> bool:
    """--suite-gemvs: an empty list selects every GEMV; an entry is a workload
    name or workload:linear."""
    sel = [e.strip() for e in spec.split(",") if e.strip()]
    return not sel or wname in sel or f"{wname}:{lname}" in sel


def run_suite(args, local_rank):
    """Configs 1-4 GEMV by GEMV, then the full step at M = 1, 2, 4, 8, 16.
    One JSON line per entry."""
    import torch

    from bit_quantized_decode_gb300 import W4_FLAG_PDL, _lib
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    _lib.load()
    _lib.clear_device_error()
    for kv in args.tune:                       # launch tuning applies to every line of the suite
        k, v = kv.split("=")
        _lib.set_tuning(k, int(v))
    peak, _ = measured_peak()
    stream = torch.cuda.Stream(device=dev)
    peak_rd = read_peak(dev, stream)
    print(json.dumps({"suite": "hbm_read_peak", "GB/s": round(peak_rd, 1), "bytes": READ_PEAK_BYTES,
                      "copy_peak": peak, "nominal": NOMINAL_HBM_GBS}), flush=True)

    def baseline(lin, M):
        return None if args.no_cpu_baseline else oracle_gemv_baseline(lin, M)

    gemv_ms = [int(m) for m in args.suite_gemv_ms.split(",") if m]
    for M in (() if args.suite_only_steps else gemv_ms):
        for wname in ("w4a8_single", "qwen7b_layer", "gemma_q4_0", "lm_head"):
            lins = list(wl.workload(wname).linears)
            if wname == "lm_head":
                lins.append(wl.gemma_lm_head_q6g32())   # the same values packed in 6 bits
            for lin in lins:
                if suite_selected(args.suite_gemvs, wname, lin.name):
                    line = suite_gemv(wname, lin, M, dev, stream, args.steps, args.warmup, peak, peak_rd)
                    line["cpu_baseline"] = baseline(lin, M)
                    print(json.dumps(line), flush=True)
    step_ms = [int(m) for m in args.suite_ms.split(",") if m]
    weights = build_weights(args, dev) if step_ms else None
    for M in step_ms:
        items, _, _ = make_buffers(weights, M, args.independent_x, dev)

        def step():
            for i, (_, lin, ql, x, y, qx, sx) in enumerate(items):
                ql(x, y, qx, sx, flags=W4_FLAG_PDL if i else 0)

        ms = _timed_graph(step, stream, max(3, min(args.steps, 400)), args.warmup)
        b = sum(algorithmic_bytes(lin, M) for _, lin, *_ in items)
        gbs = b / (ms / 1e3) / 1e9
        cpu = None
        if not args.no_cpu_baseline:
            layer = oracle_layer_sample(M, row_fraction=0.02)
            cgbs, cdt, creps = time_oracle(layer, M, 2.0, row_fraction=0.02)
            cpu = {"value": round(cgbs, 4), "unit": "GB/s", "cores": 1, "host_cpus": os.cpu_count(),
                   "kind": "oracle", "sample": f"rows 0..0.02*N of each linear of one Qwen2-7B layer, M={M}, "
                                               f"{creps} passes in {cdt:.2f} s"}
        print(json.dumps({"suite": "qwen7b_step", "M": M, "linears": len(items), "ms_per_step": round(ms, 5),
                          "GB/s": round(gbs, 1), **roofline_fracs(gbs, peak, peak_rd), "bytes": b,
                          "ms_per_token": round(ms / M, 5), "cpu_baseline": cpu}), flush=True)
        del items
    del weights
    # the decoder step: RMSNorm / SwiGLU / residual as separate kernels, then fused
    for M in (int(m) for m in args.suite_decoder_ms.split(",") if m):
        for mode in ("unfused", "fused"):
            a2 = argparse.Namespace(**vars(args))
            a2.decoder, a2.M = mode, M
            ops, _, _, b = build_decoder(a2, dev)

            def dstep(ops=ops):
                for i, op in enumerate(ops):
                    op(W4_FLAG_PDL if i else 0)

            ms = _timed_graph(dstep, stream, max(3, min(args.steps, 400)), args.warmup)
            gbs = b / (ms / 1e3) / 1e9
            print(json.dumps({"suite": "qwen7b_decoder_step", "operators": mode, "M": M, "launches": len(ops),
                              "ms_per_step": round(ms, 5), "GB/s": round(gbs, 1),
                              **roofline_fracs(gbs, peak, peak_rd), "bytes": b}), flush=True)
            del ops
            torch.cuda.empty_cache()
    # [Orin-INT4] §"为什么 INT4 float 解包不快": the same step on the weight-only
    # paths with float activations (INT4 unpacked to float, INT8 weight-only)
    for M in (int(m) for m in args.suite_ablation_ms.split(",") if m):
        for fmt, label in (("w4", "int4_dp4a_int8_activations"), ("w4a32", "int4_float_unpack"),
                           ("w8a32", "int8_weight_only")):
            weights = build_weights(args, dev, fmt)
            items, _, _ = make_buffers(weights, M, args.independent_x, dev)

            def astep(items=items):
                for i, (_, lin, ql, x, y, qx, sx) in enumerate(items):
                    ql(x, y, qx, sx, flags=W4_FLAG_PDL if i else 0)

            ms = _timed_graph(astep, stream, max(3, min(args.steps, 400)), args.warmup)
            b = sum(algorithmic_bytes(lin, M) for _, lin, *_ in items)
            gbs = b / (ms / 1e3) / 1e9
            print(json.dumps({"suite": "qwen7b_step_ablation", "path": label, "M": M, "ms_per_step": round(ms, 5),
                              "steps_per_s": round(1e3 / ms, 1), "GB/s": round(gbs, 1),
                              **roofline_fracs(gbs, peak, peak_rd), "bytes": b}), flush=True)
            del items, weights
            torch.cuda.empty_cache()
    err = _lib.device_error()
    if err:
        raise RuntimeError(f"device error word {err:#x}")
    return 0


def main(argv=None):
    args = parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if not 1 <= args.M <= 16:
        raise SystemExit("--M must be in 1..16")
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.suite:
        return run_suite(args, local_rank) if rank == 0 else 0
    return run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
