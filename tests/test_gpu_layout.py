"""The partition/indexing kernel against the oracle, bit for bit: the five
workload tensor lists (one tensor of 1.5e9, 110 GPT-2 tensors, 4096 ragged
tensors straddling shard boundaries, the padded 7.5e9 list) and random tiny
lists with empty tensors."""
import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth

pytestmark = pytest.mark.gpu


def _device_layout(zs, numels, n_d, align, cap=None, dev="cuda"):
    t = len(numels)
    cap = t + n_d if cap is None else cap
    numels_dev = torch.tensor(list(numels), dtype=torch.int64, device=dev)
    scalars = torch.full((5,), -7, dtype=torch.int64, device=dev)
    toff = torch.empty(max(t, 1), dtype=torch.int64, device=dev)
    soff = torch.empty(n_d + 1, dtype=torch.int64, device=dev)
    frags = torch.zeros(max(cap, 1) * 4, dtype=torch.int64, device=dev)
    zs.zero_partition_layout_device(numels_dev, n_d, align, scalars, toff, soff, frags, cap)
    sc = scalars.cpu().numpy()
    nf = int(sc[3])
    table = zs.fragments_from_bytes(frags.cpu().numpy(), min(nf, cap)) if nf >= 0 else None
    return sc, toff.cpu().numpy()[:t], soff.cpu().numpy(), table


def _check(zs, oracle, numels, n_d, align):
    sc, toff, soff, table = _device_layout(zs, numels, n_d, align)
    ref = oracle.layout(list(numels), n_d, align)
    assert sc[4] == 0
    assert (sc[0], sc[1], sc[2], sc[3]) == (ref["psi"], ref["psi_pad"], ref["shard_numel"], len(ref["fragments"]))
    assert np.array_equal(toff, ref["tensor_offsets"])
    assert np.array_equal(soff, ref["shard_offsets"])
    for name in ("tensor", "shard", "tensor_offset", "shard_offset", "length"):
        assert np.array_equal(table[name], ref["fragments"][name]), name


@pytest.mark.parametrize("name", ["tiny", "gpt2s", "ragged", "xl", "7b5"])
def test_device_layout_workloads(zs, oracle, cuda_device, name):
    w = synth.WORKLOADS[name]
    _check(zs, oracle, w.numels, w.n_d, w.align)


def test_device_layout_random(zs, oracle, cuda_device):
    rng = np.random.Generator(np.random.PCG64(12))
    for _ in range(60):
        t = int(rng.integers(1, 3000))
        numels = rng.integers(0, 3000, size=t)
        numels[rng.random(t) < 0.1] = 0
        n_d = int(rng.choice([1, 2, 3, 7, 16, 64, 1000]))
        align = int(rng.choice([1, 4, 128]))
        _check(zs, oracle, list(numels), n_d, align)
    _check(zs, oracle, [0, 0, 0], 4, 1)          # empty model: every shard empty


def test_device_layout_errors_and_capacity(zs, oracle, cuda_device):
    sc, _, _, _ = _device_layout(zs, [5, -1, 3], 2, 1)
    assert sc[4] == zs.ZS_ERR_ARG
    ref = oracle.layout([100, 100, 100], 4, 1)
    sc, _, _, table = _device_layout(zs, [100, 100, 100], 4, 1, cap=2)
    assert sc[3] == len(ref["fragments"]) and len(table) == 2
    assert np.array_equal(table["length"], ref["fragments"]["length"][:2])
