"""Exhaustive GPU checks of the 8-bit Adam step's own arithmetic, by the
program tests/gpu_adam8_math_check.cu (compiled here for sm_103a):

- the bucket-table nearest-code search against a search written from the
  definition (the nearer of the two neighbouring map values, exact double
  distances, ties to the smaller), for every float in [0, 1], both maps;
- the constant-divisor division (correctly rounded reciprocal, two residual
  corrections) against CUDA's IEEE division, bit for bit, for every float
  2^-100 <= |x| < 2^100 and 40 divisors 1 - beta^t;
- the normalization of a block by its scale (the same division by the
  block's largest magnitude) against the IEEE quotient: equal codes under
  both maps for every |x| <= scale, equal quotients wherever they reach a
  code threshold, for 40 scales over [2^-64, 2^64];
- the mixed-precision accumulation of an fp16 contribution (PTX
  add.rn.f32.f16) against widening and __fadd_rn, for every fp16 value."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_adam8_math_exhaustive(cuda_device, tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "adam8_math_check")
    csrc = os.path.join(ROOT, "zero_partitioned_mixed_partition_gb300", "csrc")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-Xcompiler", "-ffp-contract=off", "-I", csrc, "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "gpu_adam8_math_check.cu"), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("all equal")
    assert r.stdout.count("0 mismatches") == 4 + 40 + 40 + 1
