"""The launch planners' invariants, on the CPU: tests/plan_invariants.cu calls
the inline host planners of the kernel headers (decode warp-MMA kernel, dp4a
GEMV, streaming warp-MMA kernel, tcgen05 GEMM) over a grid of shapes and
checks every plan against the device limits it was made for (GB300: 152 SMs,
227 KB of shared memory per block) and the layout rules its kernel relies on.
No GPU is touched."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_every_plan_fits_and_keeps_its_layout_rules(tmp_path):
    from gguf_block_quantized_qmatmul_gb300 import build
    try:
        nvcc = build._nvcc()
    except RuntimeError:
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "plan_invariants")
    cmd = [nvcc, *build.ARCH, "-std=c++17", "-O1", "-I", build.CSRC, "-o", exe,
           os.path.join(ROOT, "tests", "plan_invariants.cu")]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-4000:]
    last = r.stdout.strip().splitlines()[-1]
    assert last.startswith("ok ") and int(last.split()[1]) > 5000, last
