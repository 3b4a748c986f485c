"""The debug build (libzeroshard_checked.so: the same sources compiled with
the kernels' index checks) runs the element-by-element GPU parity suites --
every entry point, layout, edge case and the 256-shard step -- and no kernel
may record an index-check failure (the conftest checks the record after each
test).  compute-sanitizer is not available on this machine; this is the
read-and-write-side check of every kernel's indexing, next to the canary
bands that check writes against the real allocations."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["test_gpu_step.py", "test_gpu_layout.py", "test_gpu_clip.py", "test_gpu_sgd.py", "test_gpu_qwz.py",
          "test_gpu_fast_math.py", "test_gpu_many_shards.py", "test_gpu_group.py", "test_gpu_guard.py",
          "test_gpu_checkpoint.py", "test_gpu_adam8.py", "test_zz_no_alloc.py"]


def test_parity_suites_under_index_checks(zs, cuda_device):
    from zero_partitioned_mixed_partition_gb300 import build
    build.build(checked=True)
    env = dict(os.environ, ZS_CHECKED="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           *[os.path.join(ROOT, "tests", f) for f in SUITES]]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = "\n".join((r.stdout + r.stderr).strip().splitlines()[-15:])
    assert r.returncode == 0, tail
    assert " passed" in tail and "failed" not in tail, tail
