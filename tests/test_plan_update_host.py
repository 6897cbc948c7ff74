"""okc_attn_plan_update on the host (no GPU): compiles tests/plan_update_host.cu
(the library's planner source with host fakes for its CUDA runtime calls) and
runs it: in-place updates equal fresh plans byte for byte, and refused or failed
updates leave the plan unchanged."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plan_update_equals_fresh_plans_and_failures_leave_it_unchanged(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "plan_update_host")
    cmd = [nvcc, "-O1", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "fp8_kv_paged_gb300", "csrc"),
           "-o", exe, os.path.join(ROOT, "tests", "plan_update_host.cu"), "-lcudart"]
    subprocess.run(cmd, check=True, capture_output=True, text=True, timeout=600)
    r = subprocess.run([exe, "1500"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok:"), r.stdout
