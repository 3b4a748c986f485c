"""zero_shard_step_noalloc, the entry point for callers that may not allocate
device memory (for example a plugin inside an application whose allocator has
already reserved the device, where a cudaMalloc of its own would bypass that
pool or fail).  It keeps its overflow words in an array compiled into the
library instead of a caller buffer.

Checked here through the C ABI, on several calls in a row (a normal step, an
overflow step, then a normal step again, which also shows the shared array is
cleared between calls), against both the existing zero_shard_step on the same
inputs and the oracle, within the parity tolerances of the other tests.  The
three shards of a call share one grouped launch, as in zero_shard_step.  This
file is named to be collected last, and it needs nothing from the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth
from parity_util import OracleShard, assert_f16_close, assert_f32_close, f16_bits, oracle_group_step, to_np

pytestmark = pytest.mark.gpu


def _shards(zs, dev, sizes, n_d, seed):
    """Device buffers of several shards of one step (same values every call)."""
    views, keep = [], []
    for i, n in enumerate(sizes):
        grads = [synth.random_fp16(n, seed * 100 + i * 10 + k, scale=200.0, device=dev) for k in range(n_d)]
        master = (synth.random_f32(n, seed * 100 + i, scale=0.02, device=dev), torch.zeros(n, device=dev))
        m = (torch.zeros(n, device=dev), torch.zeros(n, device=dev))
        v = (torch.zeros(n, device=dev), torch.zeros(n, device=dev))
        params = torch.zeros(n, dtype=torch.float16, device=dev)
        zs.zero_params_from_master(master[0], params, n)
        views.append(zs.ShardView(grads, master, m, v, params, n))
        keep.append((grads, master, m, v, params))
    return views, keep


class _Hp:
    """The hyper-parameters in the form the oracle helpers read."""
    lr, beta1, beta2, eps, weight_decay = 1e-3, 0.9, 0.999, 1e-8, 0.01


def test_noalloc_matches_zero_shard_step_and_oracle(zs, oracle, cuda_device):
    sizes, n_d, loss_scale = [4099, 2048 * 6 + 3, 17], 4, 256.0
    hp = zs.adam(_Hp.lr, _Hp.beta1, _Hp.beta2, _Hp.eps, _Hp.weight_decay)
    ref_views, ref_keep = _shards(zs, cuda_device, sizes, n_d, seed=5)
    new_views, new_keep = _shards(zs, cuda_device, sizes, n_d, seed=5)
    orc = [OracleShard(oracle, to_np(keep[1][0])) for keep in new_keep]
    flag = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    cur, step, ls, applied = 0, 1, loss_scale, 0
    for call, inject in enumerate([False, True, False]):
        if inject:
            for keep in (ref_keep, new_keep):
                keep[1][0][2][sizes[1] - 2] = float("inf")    # shard 1, rank 2, a tail element
        host = [[synth.fp16_bits(g) for g in keep[0]] for keep in new_keep]
        a = zs.zero_shard_step(ref_views, n_d, hp, loss_scale, step, cur, flag)
        b = zs.zero_shard_step_noalloc(new_views, n_d, hp, loss_scale, step, cur)
        ovf, ls, applied = oracle_group_step(oracle, orc, host, _Hp, ls, applied)
        assert a == b == ovf == int(inject), (call, a, b, ovf)
        if inject:
            for keep in (ref_keep, new_keep):
                keep[1][0][2][sizes[1] - 2] = 0.0
            loss_scale = max(loss_scale / 2, 1.0)
        else:
            cur, step = cur ^ 1, step + 1
        assert (ls, applied) == (loss_scale, step - 1)
        for i, ((_, rm, rmm, rv, rp), (_, nm, nmm, nv, np_)) in enumerate(zip(ref_keep, new_keep)):
            for x, y, nm_ in ((rm, nm, "master"), (rmm, nmm, "m"), (rv, nv, "v")):
                assert_f32_close(to_np(y[cur]), to_np(x[cur]), f"call {call} {nm_}")
            assert_f16_close(f16_bits(np_), f16_bits(rp), f"call {call} params")
            orc[i].compare(to_np(nm[cur]), to_np(nmm[cur]), to_np(nv[cur]), f16_bits(np_),
                           f"call {call} shard {i} vs oracle")


def test_noalloc_refuses_too_many_shards(zs, cuda_device):
    n = 64
    views, keep = _shards(zs, cuda_device, [n] * (zs.ZS_NOALLOC_MAX_SHARDS + 1), 2, seed=9)
    launches = zs.zero_kernel_launches()
    with pytest.raises(zs.ZeroShardError) as e:
        zs.zero_shard_step_noalloc(views, 2, zs.adam(1e-3), 1.0, 1, 0)
    assert e.value.status == zs.ZS_ERR_ARG and "ZS_NOALLOC_MAX_SHARDS" in str(e.value)
    assert zs.zero_kernel_launches() == launches
    # the largest allowed call works
    assert zs.zero_shard_step_noalloc(views[: zs.ZS_NOALLOC_MAX_SHARDS], 2, zs.adam(1e-3), 1.0, 1, 0) == 0
