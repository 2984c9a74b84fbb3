"""Host-side pieces of bench.py: workload bookkeeping, the launch plans, the
committed ncu traffic records, and the reference arm (the oracle on the host
cores), which runs without a GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_layer_workload_shapes_and_flops():
    shapes = bench.workload_shapes("layer_3p8b")
    assert [(n, M, K, N) for n, M, K, N in shapes] == [
        ("qkv", 32768, 3072, 4608), ("o", 32768, 3072, 3072), ("gate_up", 32768, 3072, 16384),
        ("down", 32768, 8192, 3072)]
    # Fprop, Dgrad and Wgrad of every linear, 2 M N K each
    assert bench.step_flops(shapes) == sum(3 * 2 * M * N * K for _, M, K, N in shapes)
    assert abs(bench.step_flops(shapes) / 1e12 - 19.48) < 0.01
    assert bench.workload_shapes("layer_3p8b", tokens=8192)[0][1] == 8192


class _Layer:
    def __init__(self, M, K, N):
        self.M, self.K, self.N = M, K, N


def test_launch_plans_count_the_work_once():
    from fp8_precision_pretraining_amax_b300 import fp8bq  # loads the library; no CUDA call
    M, K, N = 256, 384, 640
    L, lin = _Layer(M, K, N), None
    plan = bench.step_launches(fp8bq, L, lin)
    kinds = [k for k, _, _ in plan]
    assert kinds == ["quant_weight", "quant_rowcol", "gemm_fprop", "quant_rowcol", "gemm_dgrad", "gemm_wgrad"]
    assert sum(w for k, w, _ in plan if k.startswith("gemm")) == 3 * 2 * M * N * K
    mx = bench.step_launches_mx(fp8bq, L, lin)
    assert [k for k, _, _ in mx] == ["quant_mx_rowcol", "quant_mx_rowcol", "gemm_mx_fprop", "quant_mx_rowcol",
                                    "gemm_mx_dgrad", "gemm_mx_wgrad"]
    # one BF16 read, two code layouts, one exponent byte per 32 codes of each layout
    assert mx[0][1] == 2 * N * K + 2 * (N * K + N * K // 32)


@pytest.mark.parametrize("variant,src", [("fp32-scale", "gemm.cuh"), ("mx", "mx.cuh")])
def test_committed_traffic_records(variant, src):
    """A record is used only while its sha256 matches the kernel source; a
    stale one makes bench.py report traffic as null (not a wrong number)."""
    rec = bench.gemm_traffic_record(variant)
    if rec is None:
        pytest.skip(f"the DRAM record for {src} predates the current source: bench.py reports null")
    assert rec["workload"] == "layer_3p8b"
    assert float(rec["dram_bytes_per_launch"]) > float(rec["algorithmic_bytes_per_launch"]) > 0


@pytest.mark.parametrize("variant", ["fp32-scale", "mx"])
def test_reference_arm_prints_one_json_line(variant):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "tiny", "--steps", "1", "--warmup", "1", "--variant", variant],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny" and d["config"]["variant"] == bench.VARIANTS[variant]


class _Lin:
    def __init__(self, name, M, K, N, x=True, dy=True):
        import torch
        self.name, self.M, self.K, self.N = name, M, K, N
        self.x = torch.zeros((M, K), dtype=torch.bfloat16)
        self.w = torch.zeros((N, K), dtype=torch.bfloat16)
        self.dy = torch.zeros((M, N), dtype=torch.bfloat16) if dy else None


@pytest.mark.parametrize("workload", ["layer_3p8b", "swiglu", "up_bwd", "qkv_1p7b", "tiny"])
def test_every_workload_plan_does_its_gemms_once(workload):
    """Each workload's step runs exactly the GEMMs its configuration names
    (2 M N K each), and the end-to-end leg moves the inputs and outputs of
    every unit.  Plans are built on CPU tensors; no launch is made."""
    from fp8_precision_pretraining_amax_b300 import fp8bq
    shapes = bench.workload_shapes(workload, tokens=256)
    lins = [_Lin(n, M, K, N) for n, M, K, N in shapes]
    units = bench.build_units(fp8bq, workload, lins, "cpu", 1)
    kinds = [k for u in units for k, _, _ in u.launches]
    gemm_flops = sum(w for u in units for k, w, _ in u.launches if k.startswith("gemm"))
    assert gemm_flops == bench.step_flops(shapes, bench.WORKLOAD_GEMMS[workload])
    want = {"layer_3p8b": 12, "swiglu": 2, "up_bwd": 2, "qkv_1p7b": 1, "tiny": 1}[workload]
    assert sum(k.startswith("gemm") for k in kinds) == want
    assert not any(k.startswith("comm") for k in kinds)
    assert all(u.inputs for u in units) and all(u.outputs for u in units if u.name != "weights")
    if workload == "layer_3p8b":
        assert units[0].name == "weights" and [k for k, _, _ in units[0].launches] == ["quant_weight"]
        assert sum(k == "quant_weight" for k in kinds) == 1     # one launch for all four weights
    if workload == "swiglu":
        assert kinds == ["quant_weight", "quant_rowwise", "gemm_fprop", "quant_swiglu", "quant_weight", "gemm_fprop"]
    if workload == "up_bwd":
        assert kinds == ["quant_colwise", "quant_rowcol", "gemm_dgrad", "gemm_wgrad"]
        assert len(units[0].setup) == 1    # the weight codes come from the forward pass, outside the step


def test_data_parallel_plan_all_reduces_the_fp32_wgrad():
    """N > 1: every Wgrad is computed in FP32 and all-reduced right after
    (the same arithmetic as dp.LinearFP8DP); the GEMM count is unchanged."""
    import torch
    from fp8_precision_pretraining_amax_b300 import fp8bq
    shapes = bench.workload_shapes("layer_3p8b", tokens=256)
    lins = [_Lin(n, M, K, N) for n, M, K, N in shapes]
    units = bench.build_units(fp8bq, "layer_3p8b", lins, "cpu", 2)
    for u in units[1:]:          # units[0] quantizes the weights
        kinds = [k for k, _, _ in u.launches]
        i = kinds.index("gemm_wgrad")
        assert kinds[i + 1] == "comm_allreduce_dw"
        assert u.outputs[-1].dtype == torch.float32
    assert sum(k.startswith("gemm") for u in units for k, _, _ in u.launches) == 12


@pytest.mark.parametrize("workload,world,variant", [("layer_3p8b", 1, "fp32-scale"), ("layer_3p8b", 2, "fp32-scale"),
                                                    ("layer_3p8b", 1, "mx"), ("swiglu", 1, "fp32-scale"),
                                                    ("up_bwd", 1, "fp32-scale"), ("qkv_1p7b", 1, "fp32-scale")])
def test_end_to_end_copy_schedule_points_at_the_right_launches(workload, world, variant):
    """The end-to-end leg copies an input in once its previous reader ran and
    an output out once its producer ran: every input's readers are the
    quantizers that consume it, and every output is ready after the GEMM (or
    all-reduce) that writes it."""
    from fp8_precision_pretraining_amax_b300 import fp8bq
    shapes = bench.workload_shapes(workload, tokens=256)
    lins = [_Lin(n, M, K, N) for n, M, K, N in shapes]
    units = bench.build_units(fp8bq, workload, lins, "cpu", world, variant)
    for u in units:
        kinds = [k for k, _, _ in u.launches]
        assert len(u.reads) == len(u.inputs) and len(u.ready) == len(u.outputs)
        for first, last in u.reads:
            assert first <= last and kinds[first].startswith("quant") and kinds[last].startswith("quant")
        if u.name == "weights" or workload != "layer_3p8b":
            continue
        fprop, dgrad = ("gemm_mx_fprop", "gemm_mx_dgrad") if variant == "mx" else ("gemm_fprop", "gemm_dgrad")
        y, dx, dw = u.ready
        assert kinds[y] == fprop and kinds[dx] == dgrad and dw == len(kinds) - 1
        assert kinds[dw] == ("comm_allreduce_dw" if world > 1 else kinds[dw])
        # X is read by the pass that quantizes it, dY by the pass over dY, before the GEMMs that need them
        x_first = u.reads[0][0]
        dy_first = u.reads[-1][0]
        assert x_first < y and dy_first < dx
