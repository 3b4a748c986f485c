"""Out-of-range writes: every device buffer of every entry point sits between
4 KiB canary bands, sized exactly to the elements the call may touch, with
ragged lengths, the three access widths, overflow steps (restore), the qwZ
copy, clipping, SGD, the partition kernel, the casts and N_d at its maximum.
After the calls every band must still hold its pattern.  (compute-sanitizer
is not available on this machine; this is the write-side check.)"""
import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side
PATTERN = 0x5A


class Guarded:
    """Device buffers with canary bands; the views start `offset` elements in."""

    def __init__(self, dev):
        self.dev = dev
        self.raw = []

    def buf(self, n, dtype, offset=0, fill=None):
        esz = torch.tensor([], dtype=dtype).element_size()
        g = GUARD // esz
        raw = torch.empty((g * 2 + n + offset) * esz, dtype=torch.uint8, device=self.dev)
        raw.fill_(PATTERN)
        view = raw.view(dtype)[g + offset:g + offset + n]
        if fill is not None:
            view.copy_(fill)
        elif dtype.is_floating_point:
            view.zero_()
        self.raw.append((raw, (g + offset) * esz, (g + offset + n) * esz))
        return view

    def check(self, what):
        torch.cuda.synchronize()
        for raw, lo, hi in self.raw:
            host = raw.cpu().numpy()
            bad_lo = np.flatnonzero(host[:lo] != PATTERN)
            bad_hi = np.flatnonzero(host[hi:] != PATTERN)
            assert bad_lo.size == 0 and bad_hi.size == 0, (
                f"{what}: write outside the buffer ({bad_lo.size} bytes before, {bad_hi.size} after)")


def _shard(zs, gd, n, n_d, offset=0, qwz=False, seed=0):
    grads = [gd.buf(n, torch.float16, offset, synth.random_fp16(n, seed + k, 100.0, device=gd.dev))
             for k in range(n_d)]
    master = (gd.buf(n, torch.float32, offset, synth.random_f32(n, seed, 0.02, device=gd.dev)),
              gd.buf(n, torch.float32, offset))
    m = (gd.buf(n, torch.float32, offset), gd.buf(n, torch.float32, offset))
    v = (gd.buf(n, torch.float32, offset), gd.buf(n, torch.float32, offset))
    params = gd.buf(n, torch.float16, offset)
    q = {}
    if qwz:
        q = dict(qcodes=gd.buf(n, torch.int8, offset), qscales=gd.buf((n + 255) // 256, torch.float32))
    return zs.ShardView(grads, master, m, v, params, n, **q)


@pytest.mark.parametrize("n", [1, 7, 255, 256 * 7 + 13, 2048 * 5 + 9])
@pytest.mark.parametrize("n_d,offset", [(4, 0), (8, 0), (64, 0), (3, 4), (5, 1)])
def test_steps_write_inside_their_buffers(zs, cuda_device, n, n_d, offset):
    gd = Guarded(cuda_device)
    shards = [_shard(zs, gd, n, n_d, offset, qwz=(offset != 1), seed=7),
              _shard(zs, gd, n + 3, n_d, offset, qwz=(offset != 1), seed=9)]
    ctrl = gd.buf(zs.CTRL_BYTES // 8 + 1, torch.int64)
    flag = gd.buf(1, torch.int32)
    hp = zs.adam(1e-3, weight_decay=0.01)
    zs.zero_ctrl_init(ctrl, 1024.0)
    for step in range(1, 4):
        if step == 2:
            shards[1].grads[0][n // 2] = float("inf")          # overflow: restore paths
        zs.zero_shard_step_async(shards, n_d, hp, ctrl)
        ovf = zs.zero_shard_step(shards, n_d, hp, 1024.0, 1, 0, flag)
        ovf2 = zs.zero_shard_step_noalloc(shards, n_d, hp, 1024.0, 1, 0)
        assert ovf == ovf2 == int(step == 2)
        if step == 2:
            shards[1].grads[0][n // 2] = 0.0
    gd.check(f"adam n={n} n_d={n_d} offset={offset}")


@pytest.mark.parametrize("n,n_d,offset", [(2048 * 3 + 5, 4, 0), (777, 16, 0), (300, 64, 0), (1000, 5, 1)])
@pytest.mark.parametrize("keep_g", [False, True])
def test_clipped_and_sgd_steps_write_inside(zs, cuda_device, n, n_d, offset, keep_g):
    gd = Guarded(cuda_device)
    shards = [_shard(zs, gd, n, n_d, offset, qwz=(offset == 0), seed=3)]
    ctrl = gd.buf(zs.CTRL_BYTES // 8 + 1, torch.int64)
    sq = gd.buf(1, torch.float64)
    g = [gd.buf(n, torch.float32, offset)] if keep_g else None
    zs.zero_ctrl_init(ctrl, 256.0)
    for _ in range(2):
        zs.zero_shard_step_clipped_async(shards, n_d, zs.adam(1e-3), 0.5, sq, ctrl, g_dev=g)
    sgd_shards = [_shard(zs, gd, n, n_d, offset, seed=5)]
    for _ in range(2):
        zs.zero_shard_step_sgd_async(sgd_shards, n_d, zs.sgd(0.01, 0.9, 1e-4), ctrl)
    gd.check(f"clip/sgd n={n} n_d={n_d}")


def test_max_contributions(zs, oracle, cuda_device):
    """N_d at its maximum (1024 contributions, the largest address table)."""
    n, n_d = 300, zs.ZS_MAX_ND
    gd = Guarded(cuda_device)
    sh = _shard(zs, gd, n, n_d, 0, seed=11)
    flag = gd.buf(1, torch.int32)
    assert zs.zero_shard_step([sh], n_d, zs.adam(1e-3), 1.0, 1, 0, flag) == 0
    gd.check("n_d = 1024")
    contribs = [synth.fp16_bits(g) for g in sh.grads]
    master = sh.master[0].cpu().numpy().copy()
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    params = np.zeros(n, np.uint16)
    assert oracle.shard_step(contribs, master, m, v, params, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                             weight_decay=0.0, loss_scale=1.0, step=1) == 0
    assert np.array_equal(sh.master[1].cpu().numpy(), master)
    assert np.array_equal(sh.params.cpu().view(torch.int16).numpy().view(np.uint16), params)


def test_layout_cast_and_qwz_kernels_write_inside(zs, cuda_device):
    gd = Guarded(cuda_device)
    numels = [5, 0, 3000, 17, 1 << 16]
    n_d = 7
    numels_dev = gd.buf(len(numels), torch.int64, 0, torch.tensor(numels, dtype=torch.int64))
    scalars = gd.buf(5, torch.int64)
    toff = gd.buf(len(numels), torch.int64)
    soff = gd.buf(n_d + 1, torch.int64)
    cap = 3
    frags = gd.buf(cap * 4, torch.int64)
    zs.zero_partition_layout_device(numels_dev, n_d, 128, scalars, toff, soff, frags, cap)
    for n, off in ((1, 0), (4097, 1), (256 * 9 + 7, 0)):
        master = gd.buf(n, torch.float32, off, synth.random_f32(n, n, 1.0, device=cuda_device))
        params = gd.buf(n, torch.float16, off)
        zs.zero_params_from_master(master, params, n)
        codes = gd.buf(n, torch.int8, off)
        scales = gd.buf((n + 255) // 256, torch.float32)
        zs.zero_qwz_quantize(params, n, codes, scales)
        back = gd.buf(n, torch.float16, off)
        zs.zero_qwz_dequantize(codes, scales, n, back)
    gd.check("layout / cast / qwz")


@pytest.mark.parametrize("n", [1, 7, 2047, 2049, 2048 * 3 + 9])
@pytest.mark.parametrize("n_d,offset", [(4, 0), (8, 0), (64, 0), (5, 1)])
def test_adam8_writes_inside_its_buffers(zs, cuda_device, n, n_d, offset):
    """8-bit Adam: codes, block scales, master and params of two shards (one
    with an overflow step) between canary bands, every access width."""
    gd = Guarded(cuda_device)

    def shard(n, seed):
        grads = [gd.buf(n, torch.float16, offset, synth.random_fp16(n, seed + k, 100.0, device=gd.dev))
                 for k in range(n_d)]
        master = (gd.buf(n, torch.float32, offset, synth.random_f32(n, seed, 0.02, device=gd.dev)),
                  gd.buf(n, torch.float32, offset))
        nb = (n + 2047) // 2048
        codes = lambda: gd.buf(n, torch.uint8, offset, torch.zeros(n, dtype=torch.uint8, device=gd.dev))
        scales = lambda: gd.buf(nb, torch.float32, offset)
        params = gd.buf(n, torch.float16, offset)
        return zs.Adam8View(grads, master, (codes(), codes()), (codes(), codes()), (scales(), scales()),
                            (scales(), scales()), params, n)

    shards = [shard(n, 7), shard(n + 3, 9)]
    ctrl = gd.buf(zs.CTRL_BYTES // 8 + 1, torch.int64)
    hp = zs.adam(1e-3, weight_decay=0.01, math=zs.ZS_MATH_FAST)
    zs.zero_ctrl_init(ctrl, 1024.0)
    for step in range(1, 4):
        if step == 2:
            shards[1].grads[0][n // 2] = float("inf")          # overflow: the commit's restore path
        zs.zero_shard_step_adam8_async(shards, n_d, hp, ctrl)
        torch.cuda.synchronize()
        assert zs.read_ctrl(ctrl)["last_overflow"] == int(step == 2)
        if step == 2:
            shards[1].grads[0][n // 2] = 0.0
    gd.check(f"adam8 n={n} n_d={n_d} offset={offset}")
