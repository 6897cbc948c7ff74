"""Host-side logic of the library without a GPU: each harness compiles the
library's own source with host fakes for its CUDA runtime calls and runs it.
tests/plan_update_host.cu: okc_attn_plan_update's in-place updates equal fresh
plans byte for byte, and refused or failed updates leave the plan unchanged.
tests/noalloc_host.cu: okc_attn_decode_combine_noalloc uploads the plan's split
and launches over it inside its static array, and refuses exactly the calls
past its documented limits. tests/step_host_routing.cu: okc_attn_step_host
reads each mapped, aligned host buffer in place and copies every other one
with its exact byte count, for every combination. tests/arg_validation_host.cu:
the launching calls refuse missing or misaligned buffers, unusable RoPE
tables, missing scales and bad eps before any launch. tests/c_abi_host.c: the header compiles as strict
C99 without CUDA headers, and a C program linked against libokc_attn.so runs the
host-only entry points."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run_harness(tmp_path, name, iters):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path / name)
    cmd = [nvcc, "-O1", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "fp8_kv_paged_gb300", "csrc"),
           "-o", exe, os.path.join(ROOT, "tests", name + ".cu"), "-lcudart"]
    subprocess.run(cmd, check=True, capture_output=True, text=True, timeout=600)
    r = subprocess.run([exe, str(iters)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok:"), r.stdout


def test_plan_update_equals_fresh_plans_and_failures_leave_it_unchanged(tmp_path):
    _run_harness(tmp_path, "plan_update_host", 1500)


def test_noalloc_uploads_the_plans_split_within_its_array(tmp_path):
    _run_harness(tmp_path, "noalloc_host", 2000)


def test_step_host_routes_every_buffer_as_documented(tmp_path):
    _run_harness(tmp_path, "step_host_routing", 0)


def test_launching_calls_refuse_bad_arguments_before_any_launch(tmp_path):
    _run_harness(tmp_path, "arg_validation_host", 0)


def test_header_is_plain_c_and_the_library_links_from_c(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    import fp8_kv_paged_gb300 as okc
    lib = okc.build()
    exe = str(tmp_path / "c_abi_host")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           "-o", exe, os.path.join(ROOT, "tests", "c_abi_host.c"), lib, "-Wl,-rpath," + os.path.dirname(lib)]
    subprocess.run(cmd, check=True, capture_output=True, text=True, timeout=300)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
