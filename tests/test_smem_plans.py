"""Host-side check of the Gated DeltaNet step kernel's shared-memory plans.

tests/smem_plans.cu includes the kernel's layout headers and checks, for every
ring length and a range of items per CTA, the plan the launcher picks: it fits
in 227 KiB, the tensor-core operand regions are 1024-byte aligned (128-byte
swizzle atoms), the Gram MMA's 128-row read past the projection operand stays
inside the fold phase's plan, and the fold phase is used exactly up to 512
items per CTA.  Compiled with nvcc and run on the CPU (no GPU needed).
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gdn_step_smem_plans(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "smem_plans")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17",
           "-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(ROOT, "ssm_decode_state_gb300", "csrc"),
           os.path.join(ROOT, "tests", "smem_plans.cu"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip().endswith("ok"), out.stdout[-3000:]
    # the serving shape (ring 16, batch 256 x 32 heads on 152 SMs: 54 items per CTA)
    assert "L 16 items/CTA   54: stages 5 fold phase 1" in out.stdout
