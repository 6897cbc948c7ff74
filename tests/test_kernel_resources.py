"""Per-kernel resources as ptxas reports them for sm_103a (-Xptxas -v; no GPU):
the hot kernels keep the register counts their occupancy rests on (the decode
kernels for q_len 1 at 80 registers x 256 threads: three CTAs per SM; the
two-group tcgen05 decode (verify blocks) at 120 x 352 as allocated: one CTA per
SM with room for a prepare and two combine CTAs beside it; its one-kernel step
form, which also derives q and the new rows, within one CTA per SM (at most
136 registers on TMA-fed tiles, 184 on cp.async-fed ones); the per-KV-head
tcgen05 decode (extends) at 120 x 352: one CTA per SM with room for two combine
CTAs beside it; the combine for blocks of several
tokens under 64 x 128, so that two of its CTAs fit beside a tcgen05 decode CTA)
and spill nothing beyond the fused step's known 16-byte frame."""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "fp8_kv_paged_gb300", "csrc")

# kernel (substring of the mangled name) -> (max registers, max spill bytes stored)
LIMITS = {
    "decode_kernelILi2ELi1ELi4ELb1E": (80, 16),   # the fused step (sliding, mixed)
    "decode_kernelILi2ELi1ELi4ELb0E": (80, 0),    # q_len-1 decode of the three-call step
    "decode_tc_kernelILb1ELi2ELb0E": (120, 0),    # verify block, TMA gather (allocated as 120)
    "decode_tc_kernelILb0ELi2ELb0E": (120, 0),    # verify block on pages of < 8 rows, cp.async gather (allocated as 120)
    "decode_tc_kernelILb1ELi2ELb1E": (136, 0),    # the verify block's one-kernel step, TMA gather
    "decode_tc_kernelILb0ELi2ELb1E": (184, 0),    # the same on pages of < 8 rows (one CTA per SM: 184 x 352 fits)
    "decode_tc_kernelILb1ELi3ELb0E": (120, 0),    # extend (one group per KV head), TMA gather
    "decode_tc_kernelILb0ELi3ELb0E": (120, 0),    # extend, cp.async gather
    "prepare_kernel": (64, 0),
    "combine_kernel": (128, 0),
    "combine_kernelILi4E": (64, 0),               # verify and extend steps (4 splits per round trip)
}


def _ptxas_report(src):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-Xptxas", "-v",
           "-I", os.path.join(ROOT, "include"), "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", os.devnull]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    report, name = {}, None
    for line in r.stderr.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            name = m.group(1)
            report[name] = {"spill": 0, "regs": None}
            continue
        if name is None:
            continue
        m = re.search(r"(\d+) bytes spill stores", line)
        if m:
            report[name]["spill"] = int(m.group(1))
        m = re.search(r"Used (\d+) registers", line)
        if m:
            report[name]["regs"] = int(m.group(1))
    return report


@pytest.mark.parametrize("src", ["decode.cu", "decode_tc.cu", "prepare.cu", "combine.cu"])
def test_hot_kernels_keep_their_register_budget(src):
    report = _ptxas_report(src)
    checked = 0
    for key, (max_regs, max_spill) in LIMITS.items():
        for name, r in report.items():
            if key in name:
                assert r["regs"] is not None and r["regs"] <= max_regs, (key, r)
                assert r["spill"] <= max_spill, (key, r)
                checked += 1
    assert checked > 0, sorted(report)
