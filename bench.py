"""Benchmark of the block-scaled FP8 linear layer on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--tokens M]
                    [--impl reference] [--variant mx]

One step is one pass of the whole hot path over one batch.  On the default
workload: the weight-block quantizer over all of the layer's weights (codes
and the transposed copy, one launch), then for every linear one pass over X
producing its row-wise (Fprop) and column-wise (Wgrad) codes, Fprop, one pass
over dY producing its row-wise (Dgrad) and column-wise (Wgrad) codes, Dgrad
and Wgrad.  The other workloads run the launches of their configuration
(--workload; see WORKLOAD_GEMMS).

Metric: FP8 block-scaled GEMM TFLOP/s including quantization = sum of 2*M*N*K
over the step's GEMMs divided by the step time (quantizers included), plus
that number as a fraction of the FP8 tensor peak.  FLOPs count only the
GEMMs.  Inputs are synthetic BF16 tensors resident in HBM; the step's working
set (several GB) is far larger than the 126 MB L2, so no flush is needed.

Default workload (layer_3p8b): one 3.8B-shaped transformer layer at 32768
tokens (hidden 3072, 32 q / 8 kv heads of 96, SwiGLU FFN 8192): QKV
3072->4608, O 3072->3072, gate+up 3072->16384, down 8192->3072.

On one GPU the step's launches are captured once into a CUDA graph and the
timed steps replay it (--no-graph times eager launches instead).

Also reported: per-launch CUDA-event times (the roofline of the GEMM kernel
against the FP8 tensor peak, the quantizers against HBM), the same metric
end to end through the Python API with pinned host buffers (host->device
copies of X, W, dY and device->host copies of Y, dX, dW inside the timed
region), and the CPU oracle timed on a bounded sample on the host cores.

--variant mx times the MX variant of the same step instead: every operand
quantized with a power-of-two scale per 1x32 block along its GEMM's reduction
dimension (one pass over each of X, W and dY emits both layouts) and the three
GEMMs on the block-scaled MMA, which applies the scales itself.

Multi-GPU (torchrun): data parallel with weak scaling.  Every rank runs the
step on its own batch of the workload's size; Fprop and Dgrad need nothing
from other ranks, each linear's Wgrad is computed in FP32
(fp8bq_gemm_wgrad_f32) and that FP32 dW is summed over the ranks with an NCCL
all-reduce inside the timed step (the only exchange of the path).  The timed
region is bracketed by barriers and the max over ranks is reported.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 block-scaled GEMM TFLOP/s (incl. quantize) and % of B300 FP8 peak"
UNIT = "TFLOP/s"
TOKENS = {"layer_3p8b": 32768, "swiglu": 16384, "up_bwd": 16384, "qkv_1p7b": 8192, "tiny": 256}
# the GEMMs each linear of a workload runs in one step
WORKLOAD_GEMMS = {"layer_3p8b": ("fprop", "dgrad", "wgrad"), "swiglu": ("fprop",), "up_bwd": ("dgrad", "wgrad"),
                  "qkv_1p7b": ("fprop",), "tiny": ("fprop",)}
FP8_OVER_BF16 = 2.0  # nominal dense ratio (4.5 / 2.25 PFLOP/s)
NOMINAL_FP8_TFLOPS = 4500.0
VARIANTS = {
    "fp32-scale": "FP32 scale amax/448 per 1x128 tile (X, dY) and 128x128 block (W); per-128-chunk promotion",
    "mx": ("MX variant: power-of-two (E8M0) scale per 1x32 block along each GEMM's reduction dim, "
           "applied inside the block-scaled MMA; every operand quantized in both layouts"),
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="layer_3p8b", choices=sorted(TOKENS))
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the token count M of the workload (e.g. a smaller case for ncu)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--variant", default="fp32-scale", choices=["fp32-scale", "mx"],
                    help="fp32-scale: the layer's FP32 amax/448 scales per 1x128 tile / 128x128 block with "
                         "per-chunk promotion; mx: power-of-two scale per 1x32 block applied inside the MMA")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager launches instead of a CUDA graph of the step (one GPU)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# workload description (shapes only; tensors come from synth)
# ---------------------------------------------------------------------------

def workload_shapes(name, tokens=None):
    from fp8_precision_pretraining_amax_b300 import synth
    M = tokens or TOKENS[name]
    if name == "layer_3p8b":
        return [(n, M, K, N) for n, K, N in synth.LAYER_3P8B]
    if name == "swiglu":
        return [("gate_up", M, 2048, 12288), ("down", M, 6144, 2048)]
    if name == "up_bwd":
        return [("up", M, 2048, 6144)]
    if name == "qkv_1p7b":
        return [("qkv", M, 2048, 4096)]
    return [("tiny", M, 512, 384)]


def workload_config(name, tokens=None):
    shapes = workload_shapes(name, tokens)
    desc = {
        "layer_3p8b": "3.8B-shaped layer: QKV 3072->4608, O 3072->3072, gate+up 3072->16384, down 8192->3072; "
                      "Fprop+Dgrad+Wgrad each with all quantizers",
        "swiglu": "SwiGLU MLP forward: gate+up 2048->12288 Fprop, SwiGLU fused into the down projection's "
                  "row+column quantizer, down 6144->2048 Fprop; weight and input quantizers included",
        "up_bwd": "backward of the 2048->6144 up-projection: row+column pass over dY, column-wise pass over X, "
                  "Dgrad (reduce 6144) and Wgrad (reduce over the tokens); the weight codes come from the "
                  "forward pass and are not re-quantized in the step",
        "qkv_1p7b": "Qwen3-1.7B QKV Fprop 2048->4096: weight-block and row-wise quantizers, Fprop",
        "tiny": "tiny Fprop: FP32 A 256x512, B 512x384 (W = B^T): weight-block and row-wise quantizers, Fprop",
    }[name]
    return {"workload": name, "description": desc, "tokens": shapes[0][1], "gemms": list(WORKLOAD_GEMMS[name]),
            "linears": {n: {"M": M, "K": K, "N": N} for n, M, K, N in shapes}}


def step_flops(shapes, gemms=("fprop", "dgrad", "wgrad")):
    return sum(len(gemms) * 2 * M * N * K for _, M, K, N in shapes)


def make_inputs(name, device, tokens=None):
    """Input tensors per linear (X, W, dY as the workload needs), generated on `device`."""
    from fp8_precision_pretraining_amax_b300 import synth
    M = tokens or TOKENS[name]
    if name == "layer_3p8b":
        return synth.layer_3p8b(device, M=M)
    if name == "swiglu":
        return list(synth.swiglu(device, M=M))
    if name == "up_bwd":
        return [synth.up_bwd(device, M=M)]
    if name == "qkv_1p7b":
        return [synth.qkv_1p7b(device, M=M)]
    lin = synth.tiny(device)
    gen = synth.generator(10, device)
    lin.dy = synth.grads(lin.M, lin.N, gen, device)   # used by the layer step of the MX variant / CPU sample
    return [lin]


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def nvsmi_id(local_rank):
    """nvidia-smi --id of the CUDA device this rank uses (its UUID when known)."""
    try:
        import torch
        u = str(torch.cuda.get_device_properties(local_rank).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[local_rank].strip()
        return str(local_rank)


class ClockSampler:
    def __init__(self, local_rank):
        self.gpu = nvsmi_id(local_rank)
        self.proc = None
        self.path = os.path.join("/tmp", f"fp8bq_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows), "reasons": reasons}


# ---------------------------------------------------------------------------
# peaks and the committed ncu traffic record
# ---------------------------------------------------------------------------

def peaks():
    try:
        mp = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return {"hbm_gbs": mp["hbm_gbs"], "bf16_burst": mp["bf16_tflops"],
                "bf16_sustained": mp.get("bf16_tflops_sustained", mp["bf16_tflops"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6400.0, "bf16_burst": 1800.0, "bf16_sustained": 1400.0, "source": "fallback"}


def gemm_traffic_record(variant="fp32-scale"):
    """DRAM bytes per GEMM launch from the committed ncu summary; valid only
    while the kernel source is unchanged (its sha256 is recorded there)."""
    name, key = {"fp32-scale": ("gemm.cuh", "gemm_block_scaled_layer_3p8b_traffic.txt"),
                 "mx": ("mx.cuh", "mx_gemm_layer_3p8b_traffic.txt")}[variant]
    src = os.path.join(ROOT, "fp8_precision_pretraining_amax_b300", "csrc", name)
    rec = os.path.join(ROOT, "profiles", key)
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        kv = {}
        for line in open(rec):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        return kv if kv.get(name.replace(".", "_") + "_sha256") == sha else None
    except OSError:
        return None


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def rowcol_bytes(R, C):
    """Row+column pass over BF16 [R, C]: one read, two code layouts, two scale sets."""
    return 2 * R * C + 2 * R * C + 4 * R * (C // 128) + 4 * (R // 128) * C


def rowwise_bytes(R, C, in_bytes=2):
    return in_bytes * R * C + R * C + 4 * R * (C // 128)


def colwise_bytes(R, C, in_bytes=2):
    return in_bytes * R * C + R * C + 4 * (R // 128) * C


def weight_bytes(N, K, transposed=True, in_bytes=2):
    return in_bytes * N * K + (2 if transposed else 1) * N * K + 4 * (N // 128) * (K // 128)


def swiglu_bytes(M, F):
    """SwiGLU-fused quantizer: reads g and u (BF16), writes H's row-wise and
    column-wise codes and scales."""
    return 4 * M * F + 2 * M * F + 4 * M * (F // 128) + 4 * (M // 128) * F


def step_launches(fp8bq, L, lin):
    """(kind, algorithmic work, call) for one linear's 6 launches, in step order.
    Work: FLOPs for GEMMs, bytes read + written for quantizers (BF16 in, one
    code byte per layout, one FP32 scale per 128 elements and layout)."""
    M, K, N = L.M, L.K, L.N
    return [
        ("quant_weight", weight_bytes(N, K), lambda: fp8bq.fp8bq_quantize_weight_block(lin.w, L.wq, L.wqT, L.sw)),
        ("quant_rowcol", rowcol_bytes(M, K), lambda: fp8bq.fp8bq_quantize_rowcol(lin.x, L.xq, L.sx, L.xqT, L.sxT)),
        ("gemm_fprop", 2 * M * N * K, lambda: fp8bq.fp8bq_gemm_fprop(L.xq, L.sx, L.wq, L.sw, L.y)),
        ("quant_rowcol", rowcol_bytes(M, N),
         lambda: fp8bq.fp8bq_quantize_rowcol(lin.dy, L.dyq, L.sdy, L.dyqT, L.sdyT)),
        ("gemm_dgrad", 2 * M * N * K, lambda: fp8bq.fp8bq_gemm_dgrad(L.dyq, L.sdy, L.wqT, L.sw, L.dx)),
        ("gemm_wgrad", 2 * M * N * K,
         lambda: fp8bq.fp8bq_gemm_wgrad_balanced(L.dyqT, L.sdyT, L.xqT, L.sxT, L.dw, L.wscratch)),
    ]


def step_launches_mx(fp8bq, L, lin):
    """The MX variant's 6 launches per linear, in step order.  Quantizer bytes:
    BF16 in once, one code byte and 1/32 exponent byte per element and layout."""
    M, K, N = L.M, L.K, L.N
    both = lambda R, C: 2 * R * C + 2 * (R * C + R * C // 32)
    return [
        ("quant_mx_rowcol", both(N, K), lambda: fp8bq.fp8bq_mx_quantize_rowcol(lin.w, L.wq, L.ew, L.wqT, L.ewT)),
        ("quant_mx_rowcol", both(M, K), lambda: fp8bq.fp8bq_mx_quantize_rowcol(lin.x, L.xq, L.ex, L.xqT, L.exT)),
        ("gemm_mx_fprop", 2 * M * N * K, lambda: fp8bq.fp8bq_mx_gemm(L.xq, L.ex, L.wq, L.ew, L.y)),
        ("quant_mx_rowcol", both(M, N),
         lambda: fp8bq.fp8bq_mx_quantize_rowcol(lin.dy, L.dyq, L.edy, L.dyqT, L.edyT)),
        ("gemm_mx_dgrad", 2 * M * N * K, lambda: fp8bq.fp8bq_mx_gemm(L.dyq, L.edy, L.wqT, L.ewT, L.dx)),
        ("gemm_mx_wgrad", 2 * M * N * K, lambda: fp8bq.fp8bq_mx_gemm(L.dyqT, L.edyT, L.xqT, L.exT, L.dw)),
    ]


class Unit:
    """One part of the step: its launches, the input tensors a user would
    bring from the host and the outputs a user would take back (the
    end-to-end leg moves exactly these).  reads[j] = (first, last): the
    launches that first and last read input j; ready[j]: the launch after
    which output j is complete (defaults: every launch reads every input,
    outputs are complete after the last launch)."""

    def __init__(self, name, launches, inputs, outputs, setup=(), reads=None, ready=None):
        self.name, self.launches, self.inputs, self.outputs = name, launches, list(inputs), list(outputs)
        self.setup = list(setup)   # calls made once before the first step (not timed)
        n = len(launches)
        self.reads = list(reads) if reads is not None else [(0, n - 1)] * len(self.inputs)
        self.ready = list(ready) if ready is not None else [n - 1] * len(self.outputs)
        assert len(self.reads) == len(self.inputs) and len(self.ready) == len(self.outputs)
        assert all(0 <= f <= l < n for f, l in self.reads) and all(0 <= r < n for r in self.ready)


def launch_index(launches, kind, nth=0):
    """Index of the nth launch of `kind` in a launch list."""
    return [i for i, (k, _, _) in enumerate(launches) if k == kind][nth]


def data_parallel_wgrad(fp8bq, L, launches, dist):
    """N > 1: the rank's Wgrad in FP32 (fp8bq_gemm_wgrad_f32) and one NCCL
    all-reduce of it, in place of the BF16 Wgrad.  Returns the FP32 dW."""
    import torch
    dw32 = torch.empty((L.N, L.K), dtype=torch.float32, device=L.dw.device)
    i = [k for k, _, _ in launches].index("gemm_wgrad")
    launches[i] = ("gemm_wgrad", launches[i][1],
                   lambda: fp8bq.fp8bq_gemm_wgrad_f32(L.dyqT, L.sdyT, L.xqT, L.sxT, dw32))
    launches.insert(i + 1, ("comm_allreduce_dw", 4 * L.N * L.K,
                            lambda: dist.all_reduce(dw32, op=dist.ReduceOp.SUM)))
    return dw32


def build_units(fp8bq, name, lins, dev, world, variant="fp32-scale"):
    """The step of workload `name` as a list of Units."""
    import torch
    import torch.distributed as dist
    from fp8_precision_pretraining_amax_b300.linear import LinearFP8, LinearMX, SwiGLUMLPFP8
    mx = variant == "mx"
    if mx and name != "layer_3p8b":
        raise SystemExit("the MX variant is benchmarked on the layer_3p8b workload only")
    units = []
    if name == "layer_3p8b":
        layers = [(LinearMX if mx else LinearFP8)(lin.M, lin.K, lin.N, device=dev) for lin in lins]
        if not mx:
            # every weight of the layer in one launch (the step quantizes them
            # all once, as after an optimizer update)
            wl = [(lin.w, L.wq, L.wqT, L.sw) for L, lin in zip(layers, lins)]
            units.append(Unit("weights", [("quant_weight", sum(weight_bytes(l.N, l.K) for l in lins),
                                           lambda: fp8bq.fp8bq_quantize_weight_blocks(wl))],
                              [lin.w for lin in lins], [], reads=[(0, 0)] * len(lins)))
        for L, lin in zip(layers, lins):
            launches = step_launches_mx(fp8bq, L, lin) if mx else step_launches(fp8bq, L, lin)[1:]
            dw = L.dw
            if world > 1 and mx:  # the MX variant has no FP32 Wgrad: its BF16 dW is summed
                launches.append(("comm_allreduce_dw", 2 * L.N * L.K,
                                 lambda L=L: dist.all_reduce(L.dw, op=dist.ReduceOp.SUM)))
            elif world > 1:
                dw = data_parallel_wgrad(fp8bq, L, launches, dist)
            last = len(launches) - 1
            if mx:
                q = "quant_mx_rowcol"
                reads = [(launch_index(launches, q, 1),) * 2, (launch_index(launches, q, 0),) * 2,
                         (launch_index(launches, q, 2),) * 2]
                ready = [launch_index(launches, "gemm_mx_fprop"), launch_index(launches, "gemm_mx_dgrad"), last]
            else:
                reads = [(launch_index(launches, "quant_rowcol", 0),) * 2, (launch_index(launches, "quant_rowcol", 1),) * 2]
                ready = [launch_index(launches, "gemm_fprop"), launch_index(launches, "gemm_dgrad"), last]
            units.append(Unit(lin.name, launches, (lin.x, lin.w, lin.dy) if mx else (lin.x, lin.dy), (L.y, L.dx, dw),
                              reads=reads, ready=ready))
    elif name == "swiglu":
        gu_lin, down_lin = lins
        M, D, F = gu_lin.M, gu_lin.K, down_lin.K
        mlp = SwiGLUMLPFP8(M, D, F, device=dev)
        g = mlp.gate_up
        launches = [
            ("quant_weight", weight_bytes(2 * F, D, transposed=False),
             lambda: fp8bq.fp8bq_quantize_weight_block(gu_lin.w, g.wq, None, g.sw)),
            ("quant_rowwise", rowwise_bytes(M, D), lambda: fp8bq.fp8bq_quantize_rowwise(gu_lin.x, g.xq, g.sx)),
            ("gemm_fprop", 2 * M * 2 * F * D, lambda: fp8bq.fp8bq_gemm_fprop(g.xq, g.sx, g.wq, g.sw, g.y)),
            ("quant_swiglu", swiglu_bytes(M, F),
             lambda: fp8bq.fp8bq_swiglu_quantize(g.y, None, mlp.hq, mlp.sh, mlp.hqT, mlp.shT)),
            ("quant_weight", weight_bytes(D, F, transposed=False),
             lambda: fp8bq.fp8bq_quantize_weight_block(down_lin.w, mlp.wdq, None, mlp.swd)),
            ("gemm_fprop", 2 * M * D * F, lambda: fp8bq.fp8bq_gemm_fprop(mlp.hq, mlp.sh, mlp.wdq, mlp.swd, mlp.out)),
        ]
        units.append(Unit("mlp", launches, (gu_lin.x, gu_lin.w, down_lin.w), (mlp.out,),
                          reads=[(1, 1), (0, 0), (4, 4)]))
    elif name == "up_bwd":
        lin = lins[0]
        M, K, N = lin.M, lin.K, lin.N
        L = LinearFP8(M, K, N, device=dev)
        launches = [
            ("quant_colwise", colwise_bytes(M, K), lambda: fp8bq.fp8bq_quantize_colwise(lin.x, L.xqT, L.sxT)),
            ("quant_rowcol", rowcol_bytes(M, N),
             lambda: fp8bq.fp8bq_quantize_rowcol(lin.dy, L.dyq, L.sdy, L.dyqT, L.sdyT)),
            ("gemm_dgrad", 2 * M * N * K, lambda: fp8bq.fp8bq_gemm_dgrad(L.dyq, L.sdy, L.wqT, L.sw, L.dx)),
            ("gemm_wgrad", 2 * M * N * K,
             lambda: fp8bq.fp8bq_gemm_wgrad_balanced(L.dyqT, L.sdyT, L.xqT, L.sxT, L.dw, L.wscratch)),
        ]
        dw = data_parallel_wgrad(fp8bq, L, launches, dist) if world > 1 else L.dw
        # the weight's codes (and transposed codes) come from the forward pass
        setup = [lambda: fp8bq.fp8bq_quantize_weight_block(lin.w, L.wq, L.wqT, L.sw)]
        units.append(Unit(lin.name, launches, (lin.x, lin.dy), (L.dx, dw), setup=setup,
                          reads=[(0, 0), (1, 1)], ready=[launch_index(launches, "gemm_dgrad"), len(launches) - 1]))
    else:  # Fprop only: qkv_1p7b, tiny
        lin = lins[0]
        M, K, N = lin.M, lin.K, lin.N
        L = LinearFP8(M, K, N, device=dev)
        eb = lin.x.element_size()
        launches = [
            ("quant_weight", weight_bytes(N, K, transposed=False, in_bytes=eb),
             lambda: fp8bq.fp8bq_quantize_weight_block(lin.w, L.wq, None, L.sw)),
            ("quant_rowwise", rowwise_bytes(M, K, in_bytes=eb), lambda: fp8bq.fp8bq_quantize_rowwise(lin.x, L.xq, L.sx)),
            ("gemm_fprop", 2 * M * N * K, lambda: fp8bq.fp8bq_gemm_fprop(L.xq, L.sx, L.wq, L.sw, L.y)),
        ]
        units.append(Unit(lin.name, launches, (lin.x, lin.w), (L.y,), reads=[(1, 1), (0, 0)]))
    return units


def run_ours(args, rank, world, local_rank):
    import torch
    from fp8_precision_pretraining_amax_b300 import fp8bq

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    shapes = workload_shapes(args.workload, args.tokens)
    lins = make_inputs(args.workload, dev, args.tokens)
    mx = args.variant == "mx"
    units = build_units(fp8bq, args.workload, lins, dev, world, args.variant)
    for u in units:
        for fn in u.setup:
            fn()
    plan = [u.launches for u in units]
    torch.cuda.synchronize()
    flops = step_flops(shapes, WORKLOAD_GEMMS[args.workload])
    launches_per_step = sum(1 for p in plan for kind, _, _ in p if not kind.startswith("comm"))

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    def step(record=None):
        for launches in plan:
            for kind, work, fn in launches:
                if record is None:
                    fn()
                else:
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record()
                    fn()
                    e1.record()
                    record.append((kind, work, e0, e1))

    # One GPU: the step's launches are captured once into a CUDA graph and
    # the timed steps replay it (no host launch overhead between kernels).
    # Several GPUs: eager launches (the NCCL all-reduce stays outside graphs).
    run_step = step
    if world == 1 and not args.no_graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            step()                      # first calls (descriptor encoding, attributes) outside capture
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        run_step = graph.replay
    for _ in range(args.warmup):
        run_step()
    fp8bq.check(dev)
    torch.cuda.synchronize()

    # timed region: K steps on the launching (current) stream
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(args.steps):
            run_step()
        t1.record()
        torch.cuda.synchronize()
    barrier()
    dev_ms = t0.elapsed_time(t1)
    fp8bq.check(dev)

    # per-launch CUDA events on the same stream (kernel durations for the roofline)
    rec = []
    torch.cuda.synchronize()
    for _ in range(args.steps):
        step(rec)
    torch.cuda.synchronize()
    per_kind = {}
    for kind, work, e0, e1 in rec:
        d = per_kind.setdefault(kind, {"launches": 0, "ms": 0.0, "work": 0})
        d["launches"] += 1
        d["ms"] += e0.elapsed_time(e1)
        d["work"] += work

    if world > 1:
        t = torch.tensor([dev_ms], device=dev, dtype=torch.float64)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        dev_ms = float(t.item())
    ms_per_step = dev_ms / args.steps
    value = flops * world * args.steps / (dev_ms * 1e-3) / 1e12

    e2e = None if args.no_e2e else run_e2e(args, units, dev, flops, world, barrier)

    if rank != 0:
        return None
    pk = peaks()
    fp8_burst = pk["bf16_burst"] * FP8_OVER_BF16
    fp8_sus = pk["bf16_sustained"] * FP8_OVER_BF16
    gk = [v for k, v in per_kind.items() if k.startswith("gemm")]
    qk = [v for k, v in per_kind.items() if k.startswith("quant")]
    g_ms, g_fl, g_n = sum(v["ms"] for v in gk), sum(v["work"] for v in gk), sum(v["launches"] for v in gk)
    q_ms, q_by = sum(v["ms"] for v in qk), sum(v["work"] for v in qk)
    achieved = g_fl / (g_ms * 1e-3) / 1e12
    tr = gemm_traffic_record(args.variant)
    traffic = None
    if tr is not None and tr.get("workload") == args.workload and args.tokens in (None, TOKENS[args.workload]):
        traffic = float(tr["dram_bytes_per_launch"])
    breakdown = {}
    for k, v in sorted(per_kind.items()):
        b = {"launches_per_step": v["launches"] // args.steps, "ms_per_step": v["ms"] / args.steps}
        if k.startswith("gemm"):
            b["tflops"] = v["work"] / (v["ms"] * 1e-3) / 1e12
            b["frac_of_fp8_peak"] = b["tflops"] / fp8_burst
        elif k.startswith("quant"):
            b["gbs"] = v["work"] / (v["ms"] * 1e-3) / 1e9
            b["frac_of_hbm"] = b["gbs"] / pk["hbm_gbs"]
        breakdown[k] = b
    breakdown["gemm_only_tflops"] = achieved
    if qk:
        breakdown["quantizers"] = {"gbs": q_by / (q_ms * 1e-3) / 1e9,
                                   "frac_of_hbm": q_by / (q_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                                   "ms_per_step": q_ms / args.steps}
    cfg = workload_config(args.workload, args.tokens)
    cfg["variant"] = VARIANTS[args.variant]
    if world > 1:
        cfg["parallelism"] = (f"data parallel x{world}: own batch per rank"
                              + (", FP32 dW all-reduced each step" if "wgrad" in WORKLOAD_GEMMS[args.workload]
                                 else " (replicas: no exchange on this path)"))
    else:
        cfg["parallelism"] = "single GPU"
    cfg["l2"] = "inputs larger than L2 (no flush)" if args.workload != "tiny" else "inputs fit in L2"
    cfg["launch"] = ("timed steps replay a CUDA graph of the step's launches" if world == 1 and not args.no_graph
                     else "eager launches")
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("e4m3 (e8m0 block scales) x e4m3 -> f32 accumulate -> bf16" if mx
                  else "e4m3 x e4m3 -> f32 accumulate -> bf16"), "data": "synthetic",
        "config": cfg,
        "pct_of_fp8_peak": 100.0 * value / fp8_burst,
        "pct_of_nominal_fp8_peak": 100.0 * value / NOMINAL_FP8_TFLOPS,
        "roofline": {"bound": "tensor",
                     "kernel": ("mx_gemm_kernel (Fprop/Dgrad/Wgrad)" if mx
                                else "gemm_block_scaled_kernel (Fprop/Dgrad/Wgrad)"),
                     "achieved": achieved, "peak": fp8_burst, "unit": "TFLOP/s", "frac": achieved / fp8_burst,
                     "traffic": traffic,
                     "peak_note": (f"FP8 = 2 x {pk['source']} burst cuBLAS bf16 ({pk['bf16_burst']} TFLOP/s; "
                                   f"the timed region is well under a second at near-maximum SM clock); "
                                   f"sustained-based {fp8_sus:.0f}, nominal dense FP8 {NOMINAL_FP8_TFLOPS:.0f}: "
                                   f"frac {achieved / fp8_sus:.3f} and {achieved / NOMINAL_FP8_TFLOPS:.3f}"),
                     "launches_per_step": g_n // args.steps},
        "breakdown": breakdown,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if e2e is not None:
        out["e2e"] = e2e
    if not args.no_cpu_baseline and world == 1:
        out["cpu_baseline"] = cpu_baseline(args.workload, lins, variant=args.variant)
    return out


def run_e2e(args, units, dev, flops, world, barrier):
    """The same step from pinned host buffers and back: every step copies each
    unit's inputs host -> device into the tensors its launches read and its
    outputs device -> host."""
    import torch
    from fp8_precision_pretraining_amax_b300 import fp8bq

    host_in = [[t.cpu().pin_memory() for t in u.inputs] for u in units]
    host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in u.outputs] for u in units]
    h2d = sum(t.numel() * t.element_size() for hs in host_in for t in hs)
    d2h = sum(t.numel() * t.element_size() for hs in host_out for t in hs)

    # Three streams.  Host->device copies run ahead on their own stream, each
    # into a buffer as soon as the previous step's last reader of it has run;
    # the compute stream waits for an input just before its first reader;
    # each output goes device->host on the third stream as soon as the
    # launch that completes it has run, while the rest of the step computes
    # (PCIe is full duplex).  Events keep each buffer's reuse in order
    # across units and steps.
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_free = [[torch.cuda.Event() for _ in u.inputs] for u in units]    # last reader of the input ran
    ev_in = [[torch.cuda.Event() for _ in u.inputs] for u in units]      # the input is on the device
    ev_ready = [[torch.cuda.Event() for _ in u.outputs] for u in units]  # the output is complete
    ev_out = [[torch.cuda.Event() for _ in u.outputs] for u in units]    # the output is on the host
    for i in range(len(units)):  # everything starts free
        for e in ev_free[i]:
            e.record(comp)
        for e in ev_out[i]:
            e.record(s_out)

    def e2e_step():
        for i, (u, hin, hout) in enumerate(zip(units, host_in, host_out)):
            with torch.cuda.stream(s_in):
                for j, (d, h) in enumerate(zip(u.inputs, hin)):
                    s_in.wait_event(ev_free[i][j])
                    d.copy_(h, non_blocking=True)
                    ev_in[i][j].record(s_in)
            for e in ev_out[i]:                      # last step's outputs have left the device
                comp.wait_event(e)
            for k, (_, _, fn) in enumerate(u.launches):
                for j, (first, _) in enumerate(u.reads):
                    if first == k:
                        comp.wait_event(ev_in[i][j])
                fn()
                for j, (_, last) in enumerate(u.reads):
                    if last == k:
                        ev_free[i][j].record(comp)
                for j, r in enumerate(u.ready):
                    if r == k:
                        ev_ready[i][j].record(comp)
                        with torch.cuda.stream(s_out):
                            s_out.wait_event(ev_ready[i][j])
                            hout[j].copy_(u.outputs[j], non_blocking=True)
                            ev_out[i][j].record(s_out)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, 5))
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        e2e_step()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    barrier()
    fp8bq.check(dev)
    if world > 1:
        t = torch.tensor([dt], device=dev, dtype=torch.float64)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        dt = float(t.item())
    return {"value": flops * world * steps / dt / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": 1e3 * dt / steps,
            "path": ("pinned host -> device copies of every input, the C-ABI launches, device -> pinned host "
                     "copies of every output; each input is copied as soon as its buffer is free and each output "
                     "as soon as it is complete, on two copy streams that overlap compute")}


# ---------------------------------------------------------------------------
# CPU oracle: the baseline leg and the reference arm
# ---------------------------------------------------------------------------

def host_slices(lins, tile):
    """The operand slices the oracle sample needs, copied to the host (a
    missing operand of the workload gives None)."""
    from fp8_precision_pretraining_amax_b300 import synth

    def bits(t):
        if t is None:
            return None
        return synth.bf16_bits(t) if t.dtype == synth.torch.bfloat16 else t.detach().cpu().contiguous().numpy()
    out = []
    for l in lins:
        dy = getattr(l, "dy", None)
        out.append(((l.name, l.M, l.K, l.N), (
            bits(l.x[:tile]),                                         # tile rows of X, all K
            bits(l.x[:, :128].contiguous()),                          # 128 columns of X, all tokens
            bits(l.w[:128]),                                          # one N block of W, all K
            bits(l.w[:, :128].contiguous()),                          # one K block of W, all N
            None if dy is None else bits(dy[:tile]),                  # tile rows of dY
            None if dy is None else bits(dy[:, :128].contiguous())))) # 128 columns of dY, all tokens
    return out


def quantized_elements(workload, lin_name, M, K, N):
    """Elements the step's quantizers process for one linear, one layout pass
    each (the oracle quantizes every layout separately)."""
    if workload == "layer_3p8b":
        return 2 * M * K + 2 * M * N + N * K      # X rows+cols, dY rows+cols, W
    if workload == "up_bwd":
        return M * K + 2 * M * N                  # X cols, dY rows+cols
    if workload == "swiglu" and lin_name == "down":
        return 2 * M * K + N * K                  # H rows+cols, W
    return M * K + N * K                          # X rows, W


def oracle_sample(slices, tile, variant="fp32-scale", workload="layer_3p8b"):
    """Time the oracle on a bounded sample of one step and extrapolate.

    For each linear: quantize the operand slices that one tile x tile output
    block of each of the workload's GEMMs needs, then compute those blocks.
    Quantizer seconds per element and GEMM seconds per multiply-add are
    scaled to the full step's element and multiply-add counts."""
    import numpy as np
    import oracle

    gemms = WORKLOAD_GEMMS[workload]
    q_time = g_time = 0.0
    q_elems = g_macs = full_q = full_macs = 0
    for (name, M, K, N), (xr, xc, wr, wc, dyr, dyc) in slices:
        full_macs += len(gemms) * M * N * K
        idx = np.arange(tile)
        if variant == "mx":
            full_q += 2 * M * K + 2 * M * N + 2 * N * K  # every operand in both layouts
            t = time.perf_counter()
            xq = oracle.mx_quantize_rowwise(xr)
            wq = oracle.mx_quantize_rowwise(wr)
            dyq = oracle.mx_quantize_rowwise(dyr)
            wqT = oracle.mx_quantize_colwise(wc)
            dyqT = oracle.mx_quantize_colwise(dyc)
            xqT = oracle.mx_quantize_colwise(xc)
            q_time += time.perf_counter() - t
            q_elems += xr.size + wr.size + dyr.size + wc.size + dyc.size + xc.size
            t = time.perf_counter()
            oracle.mx_gemm(*xq, *wq, rows=idx, cols=idx)
            oracle.mx_gemm(*dyq, *wqT, rows=idx, cols=idx)
            oracle.mx_gemm(*dyqT, *xqT, rows=idx, cols=idx)
            g_time += time.perf_counter() - t
            g_macs += tile * tile * (K + N + M)
            continue
        full_q += quantized_elements(workload, name, M, K, N)
        if "fprop" in gemms:
            t = time.perf_counter()
            xq, sx = oracle.quantize_rowwise(xr)
            wq, _, sw = oracle.quantize_weight_block(wr)
            q_time += time.perf_counter() - t
            q_elems += xr.size + wr.size
            t = time.perf_counter()
            oracle.gemm_fprop(xq, sx, wq, sw, rows=idx, cols=idx)
            g_time += time.perf_counter() - t
            g_macs += tile * tile * K
        if "dgrad" in gemms:
            t = time.perf_counter()
            dyq, sdy = oracle.quantize_rowwise(dyr)
            wq2, _, sw2 = oracle.quantize_weight_block(wc)
            q_time += time.perf_counter() - t
            q_elems += dyr.size + wc.size
            t = time.perf_counter()
            oracle.gemm_dgrad(dyq, sdy, wq2, sw2, rows=idx, cols=idx)
            g_time += time.perf_counter() - t
            g_macs += tile * tile * N
        if "wgrad" in gemms:
            t = time.perf_counter()
            dyqT, sdyT = oracle.quantize_colwise(dyc)
            xqT, sxT = oracle.quantize_colwise(xc)
            q_time += time.perf_counter() - t
            q_elems += dyc.size + xc.size
            t = time.perf_counter()
            oracle.gemm_wgrad(dyqT, sdyT, xqT, sxT, rows=idx, cols=idx)
            g_time += time.perf_counter() - t
            g_macs += tile * tile * M
    est = full_q * (q_time / q_elems) + full_macs * (g_time / g_macs)
    return {"tflops": 2 * full_macs / est / 1e12, "sample_seconds": q_time + g_time, "step_seconds": est,
            "parts": (q_time, q_elems, g_time, g_macs, full_q, full_macs)}


def cpu_baseline(workload, lins, tile=64, variant="fp32-scale", min_seconds=10.0, max_reps=200):
    """The oracle's rate on repeated samples of the step (at least
    min_seconds of CPU work in all), extrapolated to the full step."""
    import oracle
    sl = host_slices(lins, tile)
    tot = [0.0, 0, 0.0, 0]
    reps = 0
    while reps < max_reps and tot[0] + tot[2] < min_seconds:
        q_time, q_elems, g_time, g_macs, full_q, full_macs = oracle_sample(sl, tile, variant, workload)["parts"]
        tot = [tot[0] + q_time, tot[1] + q_elems, tot[2] + g_time, tot[3] + g_macs]
        reps += 1
    est = full_q * (tot[0] / tot[1]) + full_macs * (tot[2] / tot[3])
    gem = "/".join(g.capitalize() for g in WORKLOAD_GEMMS[workload])
    return {"value": 2 * full_macs / est / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": (f"per linear one {tile}x{tile} output block of {gem} plus the quantization of the "
                       f"operand slices it needs, {reps} times ({tot[0] + tot[2]:.1f} s of CPU work), "
                       f"extrapolated to the full step ({est:.3g} s)")}


def run_reference(args):
    """The oracle as it stands on the host cores, same metric and config."""
    import oracle
    import torch
    device = "cuda" if torch.cuda.is_available() else "cpu"  # input generation only
    tile = 64
    lins = make_inputs(args.workload, device, args.tokens)
    sl = host_slices(lins, tile)
    del lins
    vals = [oracle_sample(sl, tile, args.variant, args.workload) for _ in range(args.warmup + args.steps)]
    vals = vals[args.warmup:]
    value = statistics.median(v["tflops"] for v in vals)
    est = statistics.median(v["step_seconds"] for v in vals)
    cfg = workload_config(args.workload, args.tokens)
    cfg["variant"] = VARIANTS[args.variant]
    cfg["parallelism"] = "host cores (oracle)"
    gem = "/".join(g.capitalize() for g in WORKLOAD_GEMMS[args.workload])
    sample = (f"each step: per linear one {tile}x{tile} output block of {gem} plus the quantization of the "
              f"operand slices it needs; time extrapolated to the full step")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": est * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": ("f64 oracle (E4M3 codes, E8M0 block exponents)" if args.variant == "mx"
                      else "f64 oracle (E4M3 codes, FP32 scales)"),
            "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------------

def main(argv=None):
    args = parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0

    import torch
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
