"""The balanced Wgrad's work split, checked on the host: tests/schedule_check.cu
includes the kernel header and calls the same __host__ __device__ schedule
functions the kernel's warps call, over about 3000 grid and problem sizes
(every chunk of every tile owned once, whole-tile rounds in tile order, chunk
counts equal to the MMA thread's, slot and counter indexes inside the host's
scratch, and the parts a finishing warp sums equal to the parts written).
Needs nvcc, not a GPU."""
import os
import shutil
import subprocess

from fp8_precision_pretraining_amax_b300 import build as fbuild

HERE = os.path.dirname(os.path.abspath(__file__))


def test_balanced_wgrad_schedule_covers_every_chunk_once(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    assert os.path.exists(nvcc), "nvcc is needed to compile the schedule check"
    exe = str(tmp_path / "schedule_check")
    subprocess.run([nvcc, *fbuild.ARCH, "-std=c++17", "-O1", "-I", os.path.join(fbuild.ROOT, "include"),
                    "-I", fbuild.CSRC, "-o", exe, os.path.join(HERE, "schedule_check.cu")],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.startswith("schedule ok:"), out.stdout
    assert int(out.stdout.split()[2]) > 1000   # cases checked
