"""The driver's device-memory arena (one allocation, every buffer on a 2 MiB
boundary, handed out in order with its dtype checked), on CPU memory."""
import pytest
import torch

from zero_partitioned_mixed_partition_gb300.runner import _Arena


def test_arena_offsets_alignment_and_order():
    specs = [(1000, torch.float16), (3, torch.float16), ((2 << 20) // 4 + 1, torch.float32), (7, torch.float32)]
    a = _Arena("cpu", specs)
    bufs = [a.take(dt) for _, dt in specs]
    base = a.storage.data_ptr()
    for (n, dt), b in zip(specs, bufs):
        assert b.dtype == dt and b.numel() == n
        assert (b.data_ptr() - base) % _Arena.ALIGN == 0
    # the 2 MiB + 4 byte buffer takes two slots; no buffer overlaps the next
    ends = [b.data_ptr() + b.numel() * b.element_size() for b in bufs]
    assert all(e <= nb.data_ptr() for e, nb in zip(ends, bufs[1:]))
    assert a.storage.numel() == 5 * _Arena.ALIGN
    # distinct memory: writing one buffer leaves its neighbours as they were
    bufs[1].fill_(2.0)
    bufs[0].fill_(1.0)
    bufs[2].zero_()
    assert float(bufs[0].float().sum()) == 1000.0 and float(bufs[1].float().sum()) == 6.0


def test_arena_refuses_wrong_dtype():
    a = _Arena("cpu", [(4, torch.float32)])
    with pytest.raises(RuntimeError, match="float32"):
        a.take(torch.float16)
