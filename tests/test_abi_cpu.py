"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every entry point the header declares, the host functions agree with
the oracle, and invalid arguments are refused before anything is enqueued."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

from zero_partitioned_mixed_partition_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    text = open(os.path.join(ROOT, "include", "zero_shard.h")).read()
    return sorted(set(re.findall(r"ZS_API\s+[\w\s\*]+?\b(zero_\w+)\s*\(", text)))


def test_header_symbols_exported(zs):
    names = _header_functions()
    assert len(names) >= 12
    lib = ctypes.CDLL(zs.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(zs.EXPORTED) == names


def test_missing_library_raises(zs, monkeypatch, tmp_path):
    monkeypatch.setattr(zs, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(zs, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        zs.lib()


def test_status_strings(zs):
    assert zs.status_string(0) == "ok"
    assert zs.status_string(-1) == "invalid argument"
    assert zs.status_string(-2) == "misaligned pointer"
    assert zs.status_string(-3) == "CUDA error"


@pytest.mark.parametrize("psi", [1.5e9, 7.5e9, 7e9, 70e9, 3e9, 124_419_840, 1.0])
@pytest.mark.parametrize("n_d", [1, 4, 8, 64, 1000])
def test_state_bytes_matches_oracle(zs, oracle, psi, n_d):
    for stage in range(4):
        for k in (12.0, 4.0, 6.0):
            a, b = zs.zero_state_bytes(psi, n_d, stage, k), oracle.state_bytes(psi, n_d, stage, k)
            assert math.isclose(a, b, rel_tol=1e-14), (stage, k, a, b)
    assert math.isnan(zs.zero_state_bytes(psi, n_d, 4, 12.0))
    assert math.isnan(zs.zero_state_bytes(psi, 0, 1, 12.0))


def _same_layout(a, b):
    for key in ("psi", "psi_pad", "shard_numel"):
        assert a[key] == b[key], key
    assert np.array_equal(a["tensor_offsets"], b["tensor_offsets"])
    assert np.array_equal(a["shard_offsets"], b["shard_offsets"])
    fa, fb = a["fragments"], b["fragments"]
    assert len(fa) == len(fb)
    for name in ("tensor", "shard", "tensor_offset", "shard_offset", "length"):
        assert np.array_equal(fa[name], fb[name]), name


@pytest.mark.parametrize("name", ["tiny", "gpt2s", "ragged", "xl", "7b5"])
def test_host_layout_matches_oracle_workloads(zs, oracle, name):
    w = synth.WORKLOADS[name]
    _same_layout(zs.zero_partition_layout(w.numels, w.n_d, w.align), oracle.layout(w.numels, w.n_d, w.align))


def test_host_layout_matches_oracle_random(zs, oracle):
    rng = np.random.Generator(np.random.PCG64(77))
    for _ in range(200):
        t = int(rng.integers(0, 40))
        numels = rng.integers(0, 5000, size=t)
        numels[rng.random(t) < 0.2] = 0
        n_d = int(rng.choice([1, 2, 3, 5, 8, 16, 64, 1024]))
        align = int(rng.choice([1, 2, 8, 128]))
        _same_layout(zs.zero_partition_layout(list(numels), n_d, align),
                     oracle.layout(list(numels), n_d, align))


def test_host_layout_errors(zs):
    for args in (([1], 0, 1), ([1], 1025, 1), ([1], 2, 3), ([1], 2, 0), ([1, -1], 2, 1)):
        with pytest.raises(zs.ZeroShardError) as e:
            zs.zero_partition_layout(*args)
        assert e.value.status == zs.ZS_ERR_ARG
    # frag_cap smaller than needed: error, count still reported
    L = zs.lib()
    numels = np.array([10, 10], np.int64)
    nf = ctypes.c_int64()
    frags = (zs.Fragment * 1)()
    rc = L.zero_partition_layout(numels.ctypes.data, 2, 4, 1, None, None, None, None, None, frags, 1,
                                 ctypes.byref(nf))
    assert rc == zs.ZS_ERR_ARG and nf.value == 4


def _fake_shard(n=16, n_d=2, base=0x10000, grads_ok=True, shift=0):
    table = (ctypes.c_void_p * n_d)(*[base + 0x1000 * (k + 1) + shift for k in range(n_d)])
    s = zs_struct = None
    from zero_partitioned_mixed_partition_gb300 import binding as b
    s = b.Shard()
    s.grads = ctypes.cast(table, ctypes.POINTER(ctypes.c_void_p)) if grads_ok else None
    for i in range(2):
        s.master[i] = base + 0x100000 + 0x10000 * i
        s.m[i] = base + 0x200000 + 0x10000 * i
        s.v[i] = base + 0x300000 + 0x10000 * i
    s.params = base + 0x400000
    s.n = n
    return s, table


def test_step_argument_checks_refuse_before_cuda(zs):
    """Every refusal below happens in the host checks: no CUDA call is made
    (on a machine without a GPU a call that got further would report a CUDA
    error instead)."""
    L = zs.lib()
    hp = zs.adam(1e-3)
    flag = ctypes.c_void_p(0x20000)
    ovf = ctypes.c_int32()
    s, keep = _fake_shard()
    arr = (zs.Shard * 1)(s)
    good = dict(n_shards=1, n_d=2, loss_scale=1.0, step=1, cur=0)

    def call(**kw):
        a = dict(good, **kw)
        return L.zero_shard_step(kw.get("arr", arr), a["n_shards"], a["n_d"], ctypes.byref(kw.get("hp", hp)),
                                 a["loss_scale"], a["step"], a["cur"], kw.get("flag", flag), None,
                                 ctypes.byref(ovf))

    assert call(n_d=0) == zs.ZS_ERR_ARG
    assert call(n_d=zs.ZS_MAX_ND + 1) == zs.ZS_ERR_ARG
    assert call(n_shards=0) == zs.ZS_ERR_ARG
    assert call(n_shards=zs.ZS_MAX_SHARDS + 1) == zs.ZS_ERR_ARG
    assert call(loss_scale=0.0) == zs.ZS_ERR_ARG
    assert call(loss_scale=float("nan")) == zs.ZS_ERR_ARG
    assert call(step=0) == zs.ZS_ERR_ARG
    assert call(cur=2) == zs.ZS_ERR_ARG
    assert call(flag=None) == zs.ZS_ERR_ARG
    assert call(flag=ctypes.c_void_p(0x20002)) == zs.ZS_ERR_ALIGN
    assert call(hp=zs.adam(1e-3, beta1=1.0)) == zs.ZS_ERR_ARG
    assert call(hp=zs.adam(float("nan"))) == zs.ZS_ERR_ARG
    assert call(hp=zs.adam(1e-3, math=2)) == zs.ZS_ERR_ARG        # no such arithmetic mode
    assert call(hp=zs.adam(1e-3, math=-1)) == zs.ZS_ERR_ARG
    odd = zs.adam(1e-3, math=zs.ZS_MATH_FAST)
    odd.reserved = 1
    assert call(hp=odd) == zs.ZS_ERR_ARG
    bad, k1 = _fake_shard(n=-1)
    assert call(arr=(zs.Shard * 1)(bad)) == zs.ZS_ERR_ARG
    bad, k2 = _fake_shard(grads_ok=False)
    assert call(arr=(zs.Shard * 1)(bad)) == zs.ZS_ERR_ARG
    bad, k3 = _fake_shard(shift=1)              # fp16 contribution on an odd address
    assert call(arr=(zs.Shard * 1)(bad)) == zs.ZS_ERR_ALIGN
    bad, k4 = _fake_shard()
    bad.master[1] = 0x100002                    # fp32 state on a 2-byte boundary
    assert call(arr=(zs.Shard * 1)(bad)) == zs.ZS_ERR_ALIGN
    bad, k5 = _fake_shard()
    bad.params = None
    assert call(arr=(zs.Shard * 1)(bad)) == zs.ZS_ERR_ARG

    ctrl = ctypes.c_void_p(0x30000)
    assert L.zero_shard_step_async(arr, 1, 0, ctypes.byref(hp), ctrl, None) == zs.ZS_ERR_ARG
    assert L.zero_shard_step_async(arr, 1, 2, ctypes.byref(hp), None, None) == zs.ZS_ERR_ARG
    assert L.zero_shard_step_async(arr, 1, 2, ctypes.byref(hp), ctypes.c_void_p(0x30004), None) == zs.ZS_ERR_ALIGN
    assert L.zero_shard_reduce_adam_async(None, 2, ctypes.byref(hp), ctrl, None) == zs.ZS_ERR_ARG
    assert L.zero_step_commit_async(arr, 0, ctypes.byref(hp), ctrl, None) == zs.ZS_ERR_ARG
    assert L.zero_ctrl_init(None, 1.0, None) == zs.ZS_ERR_ARG
    assert L.zero_ctrl_init(ctrl, 0.0, None) == zs.ZS_ERR_ARG
    assert L.zero_params_from_master(None, None, 5, None) == zs.ZS_ERR_ARG
    assert L.zero_params_from_master(ctypes.c_void_p(0x40001), ctypes.c_void_p(0x50000), 5, None) == zs.ZS_ERR_ALIGN
    assert L.zero_partition_layout_device(None, 3, 2, 1, ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000),
                                          ctypes.c_void_p(0x3000), None, 0, None) == zs.ZS_ERR_ARG
    assert L.zero_partition_layout_device(ctypes.c_void_p(0x1004), 3, 2, 1, ctypes.c_void_p(0x1000),
                                          ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000), None, 0,
                                          None) == zs.ZS_ERR_ALIGN
    assert zs.zero_kernel_launches() == 0


def test_adam_struct_layout(zs):
    """zs_adam: five doubles, then the int32 arithmetic mode and a reserved
    int32, 48 bytes; the binding's default is the IEEE mode."""
    assert ctypes.sizeof(zs.Adam) == 48
    assert zs.Adam.math.offset == 40 and zs.Adam.reserved.offset == 44
    assert zs.adam(1e-3).math == zs.ZS_MATH_IEEE == 0
    assert zs.adam(1e-3, math=zs.ZS_MATH_FAST).math == zs.ZS_MATH_FAST == 1
    text = open(os.path.join(ROOT, "include", "zero_shard.h")).read()
    assert re.search(r"#define ZS_MATH_IEEE 0\b", text) and re.search(r"#define ZS_MATH_FAST 1\b", text)


def test_debug_checks_absent_from_ordinary_build(zs):
    """The ordinary library has no index checks: zero_debug_checks reports so
    without touching the device; a NULL output pointer is refused."""
    if os.environ.get("ZS_CHECKED") == "1":
        pytest.skip("the debug build is loaded")
    assert zs.zero_debug_checks() == (False, 0)
    assert zs.lib().zero_debug_checks(None) == zs.ZS_ERR_ARG


def test_adam8_maps_match_oracle(zs, oracle):
    """The library builds its code maps on the host from the same definition as
    the oracle, in code of its own: the tables agree bit for bit."""
    mag7, mag8 = zs.zero_adam8_maps()
    o7, o8 = oracle.adam8_maps()
    assert np.array_equal(mag7.view(np.uint32), o7.view(np.uint32))
    assert np.array_equal(mag8.view(np.uint32), o8.view(np.uint32))
    assert zs.lib().zero_adam8_maps(None, None) == zs.ZS_ERR_ARG


def _fake_adam8(n=1000, n_d=2):
    from zero_partitioned_mixed_partition_gb300 import binding
    table = (ctypes.c_void_p * n_d)(*[0x100000 * (k + 1) for k in range(n_d)])
    s = binding.Adam8Shard()
    s.grads = ctypes.cast(table, ctypes.POINTER(ctypes.c_void_p))
    for i in range(2):
        s.master[i] = 0x1000000 + 0x100000 * i
        s.m_codes[i] = 0x2000000 + 0x100000 * i
        s.v_codes[i] = 0x3000000 + 0x100000 * i
        s.m_scale[i] = 0x4000000 + 0x100000 * i
        s.v_scale[i] = 0x5000000 + 0x100000 * i
    s.params = 0x6000000
    s.n = n
    return s, table


def test_adam8_argument_checks_refuse_before_cuda(zs):
    L = zs.lib()
    hp = zs.adam(1e-3)
    ctrl = ctypes.c_void_p(0x30000)
    s, keep = _fake_adam8()
    arr = (zs.Adam8Shard * 1)(s)

    def call(a=arr, n_shards=1, n_d=2, h=hp, c=ctrl):
        return L.zero_shard_step_adam8_async(a, n_shards, n_d, ctypes.byref(h), c, None)

    assert call(n_d=0) == zs.ZS_ERR_ARG
    assert call(n_d=zs.ZS_MAX_ND + 1) == zs.ZS_ERR_ARG
    assert call(n_shards=0) == zs.ZS_ERR_ARG
    assert call(c=None) == zs.ZS_ERR_ARG
    assert call(c=ctypes.c_void_p(0x30004)) == zs.ZS_ERR_ALIGN
    assert call(h=zs.adam(1e-3, beta2=1.0)) == zs.ZS_ERR_ARG
    assert call(h=zs.adam(1e-3, math=3)) == zs.ZS_ERR_ARG
    for field, value, status in (("n", -1, zs.ZS_ERR_ARG), ("params", None, zs.ZS_ERR_ARG),
                                 ("params", 0x6000001, zs.ZS_ERR_ALIGN)):
        bad, k = _fake_adam8()
        setattr(bad, field, value)
        assert call(a=(zs.Adam8Shard * 1)(bad)) == status, field
    bad, k = _fake_adam8()
    bad.v_codes[1] = None
    assert call(a=(zs.Adam8Shard * 1)(bad)) == zs.ZS_ERR_ARG
    bad, k = _fake_adam8()
    bad.m_scale[0] = 0x4000002                  # fp32 scales on a 2-byte boundary
    assert call(a=(zs.Adam8Shard * 1)(bad)) == zs.ZS_ERR_ALIGN
    bad, k = _fake_adam8()
    bad.master[0] = 0x1000002
    assert call(a=(zs.Adam8Shard * 1)(bad)) == zs.ZS_ERR_ALIGN
    assert zs.zero_kernel_launches() == 0


def test_adam8_struct_layout(zs):
    """zs_adam8_shard: the contribution table, five pointer pairs, params, n."""
    assert ctypes.sizeof(zs.Adam8Shard) == 8 + 5 * 16 + 8 + 8
    assert zs.Adam8Shard.params.offset == 88 and zs.Adam8Shard.n.offset == 96
    text = open(os.path.join(ROOT, "include", "zero_shard.h")).read()
    assert re.search(r"#define ZS_ADAM8_BLOCK 2048\b", text) and zs.ZS_ADAM8_BLOCK == 2048


def test_offload_argument_checks_refuse_before_cuda(zs):
    """zero_shard_step_offload validates on the host before any CUDA call: a
    NULL shard, a chunk that is not a multiple of 16, a negative n, bad
    hyper-parameters; an empty shard returns at once with no overflow."""
    import ctypes
    L = zs.lib()
    ovf = ctypes.c_int32(-1)
    hp = zs.adam(1e-3)
    s = zs.OffloadShard()
    s.n = 0
    call = lambda shard, n_d=2, h=hp, ls=1.0, step=1, cur=0, threads=0, chunk=0: L.zero_shard_step_offload(
        shard, n_d, ctypes.byref(h), ls, step, cur, threads, chunk, None, None, ctypes.byref(ovf))
    assert call(None) == zs.ZS_ERR_ARG
    assert call(ctypes.byref(s), chunk=10) == zs.ZS_ERR_ARG
    assert call(ctypes.byref(s), n_d=0) == zs.ZS_ERR_ARG
    assert call(ctypes.byref(s), ls=0.0) == zs.ZS_ERR_ARG
    assert call(ctypes.byref(s), step=0) == zs.ZS_ERR_ARG
    assert call(ctypes.byref(s), cur=2) == zs.ZS_ERR_ARG
    assert call(ctypes.byref(s), threads=-1) == zs.ZS_ERR_ARG
    bad = zs.adam(1e-3, beta1=1.5)
    assert call(ctypes.byref(s), h=bad) == zs.ZS_ERR_ARG
    s.n = -1
    assert call(ctypes.byref(s)) == zs.ZS_ERR_ARG
    s.n = 8                                          # buffers missing
    assert call(ctypes.byref(s)) == zs.ZS_ERR_ARG
    s.n = 0
    ovf.value = -1
    assert call(ctypes.byref(s)) == zs.ZS_OK and ovf.value == 0
