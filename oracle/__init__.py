"""Python handle on the C oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
never loads it, and this package imports nothing from the product package.

The oracle is a plain single-threaded C restatement of the ZeRO shard step
(see the header comment of ``oracle.c`` for the passages each function
follows).  This module only compiles it with gcc and marshals numpy arrays
through ctypes; it performs none of the method's arithmetic itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: every fp32 multiply and add rounds on its own (no fused
# multiply-add), which is how the oracle states the arithmetic.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to the source (gcc, no CUDA)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Fragment(ctypes.Structure):
    _fields_ = [
        ("tensor", ctypes.c_int32),
        ("shard", ctypes.c_int32),
        ("tensor_offset", ctypes.c_int64),
        ("shard_offset", ctypes.c_int64),
        ("length", ctypes.c_int64),
    ]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F64 = ctypes.c_double


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f32.restype = ctypes.c_float
            lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_f16.restype = ctypes.c_uint16
            lib.oracle_f16_to_f32_array.argtypes = [_P, _P, _I64]
            lib.oracle_f32_to_f16_array.argtypes = [_P, _P, _I64]
            lib.oracle_state_bytes.argtypes = [_F64, _I32, _I32, _F64]
            lib.oracle_state_bytes.restype = _F64
            lib.oracle_layout.argtypes = [_P, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _I64, _P]
            lib.oracle_layout.restype = _I32
            lib.oracle_grad_reduce.argtypes = [_P, _I32, _I64, _F64, _P, _P]
            lib.oracle_grad_reduce.restype = _I32
            lib.oracle_adam_apply.argtypes = [_P, _I64, _P, _P, _P, _P, _F64, _F64, _F64, _F64, _F64, _I64]
            lib.oracle_adam_apply.restype = _I32
            lib.oracle_shard_step.argtypes = [_P, _I32, _I64, _P, _P, _P, _P, _F64, _F64, _F64,
                                              _F64, _F64, _F64, _I64, _P, _P]
            lib.oracle_shard_step.restype = _I32
            lib.oracle_commit.argtypes = [_I32, _P, _P]
            lib.oracle_commit.restype = None
            lib.oracle_grad_sqnorm.argtypes = [_P, _I64, _P]
            lib.oracle_grad_sqnorm.restype = None
            lib.oracle_clip_factor.argtypes = [_F64, _F64]
            lib.oracle_clip_factor.restype = ctypes.c_float
            lib.oracle_scale.argtypes = [_P, _I64, ctypes.c_float]
            lib.oracle_scale.restype = None
            lib.oracle_sgd_apply.argtypes = [_P, _I64, _P, _P, _P, _F64, _F64, _F64]
            lib.oracle_sgd_apply.restype = _I32
            lib.oracle_qwz_quantize.argtypes = [_P, _I64, _P, _P]
            lib.oracle_qwz_quantize.restype = None
            lib.oracle_qwz_dequantize.argtypes = [_P, _P, _I64, _P]
            lib.oracle_qwz_dequantize.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _contig(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


# ----------------------------------------------------------------- fp16 ---

def f16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Decode uint16 binary16 bit patterns to float32."""
    bits = _contig(bits, np.uint16)
    out = np.empty(bits.shape, np.float32)
    _load().oracle_f16_to_f32_array(_ptr(bits), _ptr(out), bits.size)
    return out


def f32_to_f16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to binary16 (ties to even); returns uint16 bits."""
    x = _contig(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().oracle_f32_to_f16_array(_ptr(x), _ptr(out), x.size)
    return out


# --------------------------------------------------------- state bytes ---

def state_bytes(psi: float, n_d: int, stage: int, k: float = 12.0) -> float:
    """Model-state bytes per device (NaN for a stage outside 0..3 or n_d < 1)."""
    return _load().oracle_state_bytes(float(psi), int(n_d), int(stage), float(k))


# -------------------------------------------------------------- layout ---

def layout(numels, n_d: int, align: int):
    """Partition a tensor list; returns a dict of psi, psi_pad, shard_numel,
    tensor_offsets, shard_offsets and the fragment table (structured array).
    Raises ValueError on invalid arguments."""
    lib = _load()
    numels = _contig(np.asarray(numels, dtype=np.int64), np.int64)
    t = numels.size
    psi, psi_pad, s, nf = _I64(), _I64(), _I64(), _I64()
    toff = np.empty(t, np.int64)
    soff = np.empty(max(n_d, 0) + 1, np.int64)
    rc = lib.oracle_layout(_ptr(numels), t, n_d, align, ctypes.byref(psi), ctypes.byref(psi_pad),
                           ctypes.byref(s), _ptr(toff), _ptr(soff), None, 0, ctypes.byref(nf))
    if rc != 0:
        raise ValueError("oracle_layout: invalid arguments")
    frags = (Fragment * max(nf.value, 1))()
    rc = lib.oracle_layout(_ptr(numels), t, n_d, align, ctypes.byref(psi), ctypes.byref(psi_pad),
                           ctypes.byref(s), _ptr(toff), _ptr(soff), frags, nf.value, ctypes.byref(nf))
    if rc != 0:
        raise ValueError("oracle_layout: fragment table")
    table = np.array([(f.tensor, f.shard, f.tensor_offset, f.shard_offset, f.length)
                      for f in frags[: nf.value]],
                     dtype=[("tensor", np.int32), ("shard", np.int32), ("tensor_offset", np.int64),
                            ("shard_offset", np.int64), ("length", np.int64)])
    return {"psi": psi.value, "psi_pad": psi_pad.value, "shard_numel": s.value,
            "tensor_offsets": toff, "shard_offsets": soff, "fragments": table}


# ---------------------------------------------------------- shard step ---

def _contrib_table(contribs):
    arrs = [_contig(c, np.uint16) for c in contribs]
    table = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    return arrs, table


def grad_reduce(contribs, loss_scale: float, n: int | None = None):
    """Reduced fp32 gradient and the non-finite flag of N_d fp16 contributions
    (each a uint16 array of the shard's bit patterns)."""
    arrs, table = _contrib_table(contribs)
    n = arrs[0].size if n is None else n
    g = np.empty(n, np.float32)
    bad = _I32()
    rc = _load().oracle_grad_reduce(table, len(arrs), n, float(loss_scale), _ptr(g), ctypes.byref(bad))
    if rc != 0:
        raise ValueError("oracle_grad_reduce: invalid arguments")
    return g, int(bad.value)


def adam_apply(g, master, m, v, params, *, lr, beta1, beta2, eps, weight_decay, step):
    """In-place Adam/AdamW update of float32 master/m/v and uint16 params."""
    g = _contig(g, np.float32)
    for a in (master, m, v):
        if a.dtype != np.float32 or not a.flags.c_contiguous:
            raise TypeError("state arrays must be contiguous float32")
    if params is not None and (params.dtype != np.uint16 or not params.flags.c_contiguous):
        raise TypeError("params must be contiguous uint16")
    rc = _load().oracle_adam_apply(_ptr(g), g.size, _ptr(master), _ptr(m), _ptr(v), _ptr(params),
                                   lr, beta1, beta2, eps, weight_decay, int(step))
    if rc != 0:
        raise ValueError("oracle_adam_apply: invalid arguments")


def shard_step(contribs, master, m, v, params, *, lr, beta1, beta2, eps, weight_decay,
               loss_scale, step, n: int | None = None) -> int:
    """One shard step in place (nothing written on overflow); returns the flag."""
    arrs, table = _contrib_table(contribs)
    n = master.size if n is None else n
    for a in (master, m, v):
        if a.dtype != np.float32 or not a.flags.c_contiguous:
            raise TypeError("state arrays must be contiguous float32")
    scratch = np.empty(max(n, 1), np.float32)
    ovf = _I32()
    rc = _load().oracle_shard_step(table, len(arrs), n, _ptr(master), _ptr(m), _ptr(v), _ptr(params),
                                   lr, beta1, beta2, eps, weight_decay, float(loss_scale), int(step),
                                   _ptr(scratch), ctypes.byref(ovf))
    if rc != 0:
        raise ValueError("oracle_shard_step: invalid arguments")
    return int(ovf.value)


def commit(overflow: int, loss_scale: float, applied_steps: int):
    """Skip/commit bookkeeping; returns (loss_scale, applied_steps)."""
    ls, st = _F64(loss_scale), _I64(applied_steps)
    _load().oracle_commit(int(overflow), ctypes.byref(ls), ctypes.byref(st))
    return ls.value, st.value


# ------------------------------------------------------------ clipping ---

def grad_sqnorm(g, start: float = 0.0) -> float:
    """start + sum of g_j^2 (float64, index order) over float32 gradients."""
    g = _contig(g, np.float32)
    acc = _F64(start)
    _load().oracle_grad_sqnorm(_ptr(g), g.size, ctypes.byref(acc))
    return acc.value


def clip_factor(sqnorm: float, max_norm: float) -> float:
    """min(1, max_norm / (sqrt(sqnorm) + 1e-6)) rounded to float32."""
    return float(_load().oracle_clip_factor(float(sqnorm), float(max_norm)))


def scale(g, c: float):
    """g *= c in float32, in place."""
    if g.dtype != np.float32 or not g.flags.c_contiguous:
        raise TypeError("g must be contiguous float32")
    _load().oracle_scale(_ptr(g), g.size, ctypes.c_float(c))


# -------------------------------------------------- quantized weights ---

QWZ_BLOCK = 256


def qwz_quantize(params_bits):
    """int8 codes and float32 per-block scales of uint16 fp16 parameters."""
    p = _contig(params_bits, np.uint16)
    codes = np.empty(p.size, np.int8)
    scales = np.empty((p.size + QWZ_BLOCK - 1) // QWZ_BLOCK, np.float32)
    _load().oracle_qwz_quantize(_ptr(p), p.size, _ptr(codes), _ptr(scales))
    return codes, scales


def qwz_dequantize(codes, scales):
    """uint16 fp16 parameters rebuilt from codes and scales."""
    c = _contig(codes, np.int8)
    s = _contig(scales, np.float32)
    out = np.empty(c.size, np.uint16)
    _load().oracle_qwz_dequantize(_ptr(c), _ptr(s), c.size, _ptr(out))
    return out


# ----------------------------------------------------- SGD with momentum ---

def sgd_apply(g, master, mom, params, *, lr, momentum, weight_decay):
    """In-place SGD-with-momentum update of float32 master / momentum and
    uint16 params."""
    g = _contig(g, np.float32)
    for a in (master, mom):
        if a.dtype != np.float32 or not a.flags.c_contiguous:
            raise TypeError("state arrays must be contiguous float32")
    rc = _load().oracle_sgd_apply(_ptr(g), g.size, _ptr(master), _ptr(mom), _ptr(params), lr, momentum,
                                  weight_decay)
    if rc != 0:
        raise ValueError("oracle_sgd_apply: invalid arguments")


# ----------------------------------------------------------- 8-bit Adam ---

ADAM8_BLOCK = 2048


def _lib_adam8():
    lib = _load()
    if not getattr(lib, "_adam8_typed", False):
        lib.oracle_adam8_maps.argtypes = [_P, _P]
        lib.oracle_adam8_maps.restype = None
        lib.oracle_adam8_code_signed.argtypes = [ctypes.c_float, _P]
        lib.oracle_adam8_code_signed.restype = ctypes.c_uint8
        lib.oracle_adam8_code_unsigned.argtypes = [ctypes.c_float, _P]
        lib.oracle_adam8_code_unsigned.restype = ctypes.c_uint8
        lib.oracle_adam8_apply.argtypes = [_P, _I64, _P, _P, _P, _P, _P, _P, _F64, _F64, _F64, _F64, _F64, _I64]
        lib.oracle_adam8_apply.restype = _I32
        lib._adam8_typed = True
    return lib


def adam8_maps():
    """The two code tables of 8-bit Adam: (mag7[128] signed-map magnitudes,
    mag8[256] unsigned map), float32."""
    mag7 = np.empty(128, np.float32)
    mag8 = np.empty(256, np.float32)
    _lib_adam8().oracle_adam8_maps(_ptr(mag7), _ptr(mag8))
    return mag7, mag8


def adam8_code_signed(x: float) -> int:
    """Signed-map code of one float32 x in [-1, 1]."""
    mag7, _ = adam8_maps()
    return int(_lib_adam8().oracle_adam8_code_signed(ctypes.c_float(x), _ptr(mag7)))


def adam8_code_unsigned(x: float) -> int:
    """Unsigned-map code of one float32 x in [0, 1]."""
    _, mag8 = adam8_maps()
    return int(_lib_adam8().oracle_adam8_code_unsigned(ctypes.c_float(x), _ptr(mag8)))


def adam8_apply(g, master, m_codes, v_codes, m_scale, v_scale, params, *, lr, beta1, beta2, eps, weight_decay,
                step):
    """In-place 8-bit Adam update of float32 master, uint8 codes, float32
    per-2048 scales and uint16 params."""
    g = _contig(g, np.float32)
    for a, dt in ((master, np.float32), (m_codes, np.uint8), (v_codes, np.uint8), (m_scale, np.float32),
                  (v_scale, np.float32)):
        if a.dtype != dt or not a.flags.c_contiguous:
            raise TypeError(f"expected contiguous {dt}")
    rc = _lib_adam8().oracle_adam8_apply(_ptr(g), g.size, _ptr(master), _ptr(m_codes), _ptr(v_codes),
                                         _ptr(m_scale), _ptr(v_scale), _ptr(params), lr, beta1, beta2, eps,
                                         weight_decay, int(step))
    if rc != 0:
        raise ValueError("oracle_adam8_apply: invalid arguments")
