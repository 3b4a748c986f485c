"""ctypes binding of ``libzeroshard.so`` (C ABI in ``include/zero_shard.h``).

Argument marshalling only: every function has the name of the C entry point it
wraps, turns torch tensors into device pointers and Python values into C
structs, and raises :class:`ZeroShardError` on a non-zero status.  Every step
of the computation runs in the library's CUDA kernels.  There is no fallback:
if the library has not been built, :func:`lib` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Iterable, List, Optional, Sequence

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# ZS_CHECKED=1 in the environment selects the debug build (kernel index checks)
LIB_PATH = os.path.join(_PKG, "libzeroshard_checked.so" if os.environ.get("ZS_CHECKED") == "1"
                        else "libzeroshard.so")

ZS_OK, ZS_ERR_ARG, ZS_ERR_ALIGN, ZS_ERR_CUDA, ZS_ERR_TIMEOUT = 0, -1, -2, -3, -4
ZS_MAX_ND = 1024
ZS_MAX_SHARDS = 256
ZS_NOALLOC_MAX_SHARDS = 64
ZS_QWZ_BLOCK = 256
ZS_ADAM8_BLOCK = 2048
ZS_MATH_IEEE, ZS_MATH_FAST = 0, 1

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F64 = ctypes.c_double


class ZeroShardError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})" + (f": {detail}" if detail else ""))


class Fragment(ctypes.Structure):
    _fields_ = [("tensor", _I32), ("shard", _I32), ("tensor_offset", _I64),
                ("shard_offset", _I64), ("length", _I64)]


class Adam(ctypes.Structure):
    _fields_ = [("lr", _F64), ("beta1", _F64), ("beta2", _F64), ("eps", _F64), ("weight_decay", _F64),
                ("math", _I32), ("reserved", _I32)]


class Shard(ctypes.Structure):
    _fields_ = [("grads", ctypes.POINTER(_P)), ("master", _P * 2), ("m", _P * 2), ("v", _P * 2),
                ("params", _P), ("n", _I64), ("qcodes", _P), ("qscales", _P)]


class Adam8Shard(ctypes.Structure):
    _fields_ = [("grads", ctypes.POINTER(_P)), ("master", _P * 2), ("m_codes", _P * 2), ("v_codes", _P * 2),
                ("m_scale", _P * 2), ("v_scale", _P * 2), ("params", _P), ("n", _I64)]


class OffloadShard(ctypes.Structure):
    _fields_ = [("grads_dev", ctypes.POINTER(_P)), ("params_dev", _P), ("grads_host", ctypes.POINTER(_P)),
                ("params_host", _P), ("master", _P * 2), ("m", _P * 2), ("v", _P * 2), ("n", _I64)]


class Sgd(ctypes.Structure):
    _fields_ = [("lr", _F64), ("momentum", _F64), ("weight_decay", _F64)]


class Ctrl(ctypes.Structure):
    _fields_ = [("loss_scale", _F64), ("beta1_pow", _F64), ("beta2_pow", _F64), ("step", _I64),
                ("skipped", _I64), ("cur", _I32), ("overflow", _I32), ("last_overflow", _I32),
                ("arrivals", ctypes.c_uint32)]


FRAGMENT_DTYPE = np.dtype([("tensor", np.int32), ("shard", np.int32), ("tensor_offset", np.int64),
                           ("shard_offset", np.int64), ("length", np.int64)])
assert FRAGMENT_DTYPE.itemsize == ctypes.sizeof(Fragment) == 32
CTRL_BYTES = ctypes.sizeof(Ctrl)

_lock = threading.Lock()
_lib = None

_SIGNATURES = {
    "zero_partition_layout": (_I32, [_P, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _I64, _P]),
    "zero_partition_layout_device": (_I32, [_P, _I32, _I32, _I32, _P, _P, _P, _P, _I64, _P]),
    "zero_state_bytes": (_F64, [_F64, _I32, _I32, _F64]),
    "zero_shard_step": (_I32, [_P, _I32, _I32, _P, _F64, _I64, _I32, _P, _P, _P]),
    "zero_shard_step_noalloc": (_I32, [_P, _I32, _I32, _P, _F64, _I64, _I32, _P, _P]),
    "zero_ctrl_init": (_I32, [_P, _F64, _P]),
    "zero_shard_step_async": (_I32, [_P, _I32, _I32, _P, _P, _P]),
    "zero_shard_step_host": (_I32, [_P, _I32, _P, _P, _P, _P]),
    "zero_shard_reduce_adam_async": (_I32, [_P, _I32, _P, _P, _P]),
    "zero_shard_reduce_adam_all_async": (_I32, [_P, _I32, _I32, _P, _P, _P]),
    "zero_shard_grad_sqnorm_async": (_I32, [_P, _I32, _P, _P, _P, _P]),
    "zero_shard_clipped_adam_async": (_I32, [_P, _I32, _P, _F64, _P, _P, _P, _P]),
    "zero_shard_step_clipped_async": (_I32, [_P, _I32, _I32, _P, _F64, _P, _P, _P, _P]),
    "zero_shard_grad_sqnorm_all_async": (_I32, [_P, _I32, _I32, _P, _P, _P, _P]),
    "zero_shard_clipped_adam_all_async": (_I32, [_P, _I32, _I32, _P, _F64, _P, _P, _P, _P]),
    "zero_step_commit_async": (_I32, [_P, _I32, _P, _P, _P]),
    "zero_params_from_master": (_I32, [_P, _P, _I64, _P]),
    "zero_shard_step_cpu": (_I32, [_P, _I32, _I32, _P, _F64, _I64, _I32, _I32, _P]),
    "zero_shard_step_offload": (_I32, [_P, _I32, _P, _F64, _I64, _I32, _I32, _I64, _P, _P, _P]),
    "zero_shard_step_sgd_async": (_I32, [_P, _I32, _I32, _P, _P, _P]),
    "zero_shard_step_adam8_async": (_I32, [_P, _I32, _I32, _P, _P, _P]),
    "zero_adam8_maps": (_I32, [_P, _P]),
    "zero_qwz_quantize": (_I32, [_P, _I64, _P, _P, _P]),
    "zero_qwz_dequantize": (_I32, [_P, _P, _I64, _P, _P]),
    "zero_status_string": (ctypes.c_char_p, [_I32]),
    "zero_last_error": (ctypes.c_char_p, []),
    "zero_kernel_launches": (_I64, []),
    "zero_debug_checks": (_I32, [_P]),
}
EXPORTED = tuple(_SIGNATURES)


def lib():
    """The loaded library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                                   "(there is no CPU fallback)")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def status_string(status: int) -> str:
    if _lib is None and not os.path.exists(LIB_PATH):
        return str(status)
    return lib().zero_status_string(int(status)).decode()


def zero_last_error() -> str:
    return lib().zero_last_error().decode()


def zero_kernel_launches() -> int:
    return int(lib().zero_kernel_launches())


def zero_debug_checks():
    """(built with index checks, first recorded failure or 0); clears the
    record and synchronises the device."""
    out = ctypes.c_uint64(0)
    rc = int(lib().zero_debug_checks(ctypes.byref(out)))
    if rc < 0:
        _check(rc, "zero_debug_checks")
    return rc == 1, int(out.value)


def _check(rc: int, what: str):
    if rc != ZS_OK:
        raise ZeroShardError(rc, what, zero_last_error() if rc == ZS_ERR_CUDA else "")


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev_ptr(t: Optional[torch.Tensor], dtype, what: str) -> Optional[int]:
    if t is None:
        return None
    if t.dtype != dtype:
        raise TypeError(f"{what}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{what}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise TypeError(f"{what}: expected a contiguous tensor")
    return t.data_ptr()


# ------------------------------------------------------------------ layout ---

def zero_partition_layout(numels: Sequence[int], n_d: int, align: int) -> dict:
    """Host partition; returns psi, psi_pad, shard_numel, tensor_offsets,
    shard_offsets (numpy int64) and fragments (numpy structured array)."""
    L = lib()
    arr = np.ascontiguousarray(np.asarray(numels, dtype=np.int64))
    t = arr.size
    psi, psi_pad, s, nf = _I64(), _I64(), _I64(), _I64()
    toff = np.empty(t, np.int64)
    soff = np.empty(max(int(n_d), 0) + 1, np.int64)
    rc = L.zero_partition_layout(arr.ctypes.data if t else None, t, int(n_d), int(align),
                                 ctypes.byref(psi), ctypes.byref(psi_pad), ctypes.byref(s),
                                 toff.ctypes.data if t else None, soff.ctypes.data, None, 0,
                                 ctypes.byref(nf))
    _check(rc, "zero_partition_layout")
    frags = np.zeros(nf.value, FRAGMENT_DTYPE)
    rc = L.zero_partition_layout(arr.ctypes.data if t else None, t, int(n_d), int(align),
                                 ctypes.byref(psi), ctypes.byref(psi_pad), ctypes.byref(s),
                                 toff.ctypes.data if t else None, soff.ctypes.data,
                                 frags.ctypes.data if nf.value else None, nf.value, ctypes.byref(nf))
    _check(rc, "zero_partition_layout")
    return {"psi": psi.value, "psi_pad": psi_pad.value, "shard_numel": s.value,
            "tensor_offsets": toff, "shard_offsets": soff, "fragments": frags}


def zero_partition_layout_device(numels_dev: torch.Tensor, n_d: int, align: int, scalars_dev: torch.Tensor,
                                 tensor_offsets_dev: torch.Tensor, shard_offsets_dev: torch.Tensor,
                                 frags_dev: Optional[torch.Tensor], frag_cap: int, stream=None):
    """Device partition (stream-ordered).  ``frags_dev`` is a byte or int64
    tensor of at least 32 * frag_cap bytes, or None."""
    fptr = None
    if frags_dev is not None:
        if frags_dev.numel() * frags_dev.element_size() < 32 * frag_cap:
            raise ValueError("frags_dev too small for frag_cap")
        fptr = _dev_ptr(frags_dev, frags_dev.dtype, "frags_dev")
    n = numels_dev.numel()
    rc = lib().zero_partition_layout_device(
        _dev_ptr(numels_dev, torch.int64, "numels_dev") if n else None, n, int(n_d), int(align),
        _dev_ptr(scalars_dev, torch.int64, "scalars_dev"),
        _dev_ptr(tensor_offsets_dev, torch.int64, "tensor_offsets_dev") if n else None,
        _dev_ptr(shard_offsets_dev, torch.int64, "shard_offsets_dev"), fptr, int(frag_cap), _stream(stream))
    _check(rc, "zero_partition_layout_device")


def fragments_from_bytes(raw: np.ndarray, count: int) -> np.ndarray:
    """View a host copy of a device fragment table as the structured dtype."""
    return np.frombuffer(np.ascontiguousarray(raw).tobytes(), dtype=FRAGMENT_DTYPE, count=count)


def zero_state_bytes(psi: float, n_d: int, stage: int, k: float = 12.0) -> float:
    return float(lib().zero_state_bytes(float(psi), int(n_d), int(stage), float(k)))


# ------------------------------------------------------------------ shards ---

class ShardView:
    """One shard's device buffers, and the C struct that describes them.

    grads: list of n_d fp16 CUDA tensors (each >= n elements);
    master, m, v: pairs (set 0, set 1) of fp32 CUDA tensors (the same tensor
    twice means in-place); params: fp16 CUDA tensor (the shard's slice of the
    full parameter buffer); n: elements stepped; qcodes / qscales: optional
    int8 / fp32 CUDA tensors for the qwZ copy of the fp16 slice."""

    def __init__(self, grads: Sequence[torch.Tensor], master, m, v, params: torch.Tensor, n: int,
                 qcodes: Optional[torch.Tensor] = None, qscales: Optional[torch.Tensor] = None):
        self.grads = list(grads)
        self.master, self.m, self.v = tuple(master), tuple(m), tuple(v)
        self.params = params
        self.n = int(n)
        self._table = (_P * max(len(self.grads), 1))(
            *[_dev_ptr(g, torch.float16, "grads") for g in self.grads])
        self.struct = Shard()
        self.struct.grads = ctypes.cast(self._table, ctypes.POINTER(_P))
        for i in range(2):
            self.struct.master[i] = _dev_ptr(self.master[i], torch.float32, "master")
            self.struct.m[i] = _dev_ptr(self.m[i], torch.float32, "m")
            self.struct.v[i] = _dev_ptr(self.v[i], torch.float32, "v")
        self.struct.params = _dev_ptr(params, torch.float16, "params")
        self.struct.n = self.n
        self.qcodes, self.qscales = qcodes, qscales
        if (qcodes is None) != (qscales is None):
            raise ValueError("qcodes and qscales go together")
        if qcodes is not None:
            if qcodes.numel() < self.n or qscales.numel() < (self.n + ZS_QWZ_BLOCK - 1) // ZS_QWZ_BLOCK:
                raise ValueError("qwZ buffers too small")
            self.struct.qcodes = _dev_ptr(qcodes, torch.int8, "qcodes")
            self.struct.qscales = _dev_ptr(qscales, torch.float32, "qscales")

    @property
    def n_d(self) -> int:
        return len(self.grads)


def _shard_array(shards: Sequence[ShardView]):
    arr = (Shard * len(shards))()
    for i, s in enumerate(shards):
        arr[i] = s.struct
    return arr


def adam(lr: float, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8,
         weight_decay: float = 0.0, math: int = None) -> Adam:
    """Adam hyper-parameters; math is ZS_MATH_IEEE (default) or ZS_MATH_FAST."""
    return Adam(float(lr), float(beta1), float(beta2), float(eps), float(weight_decay),
                ZS_MATH_IEEE if math is None else int(math), 0)


def sgd(lr: float, momentum: float = 0.9, weight_decay: float = 0.0) -> Sgd:
    return Sgd(float(lr), float(momentum), float(weight_decay))


def zero_shard_step_sgd_async(shards: Sequence[ShardView], n_d: int, hp: Sgd, ctrl_dev: torch.Tensor, stream=None):
    """Stream-ordered step with SGD with momentum (momentum in ShardView.m)."""
    arr = _shard_array(shards)
    rc = lib().zero_shard_step_sgd_async(arr, len(shards), int(n_d), ctypes.byref(hp),
                                         _dev_ptr(ctrl_dev, torch.int64, "ctrl_dev"), _stream(stream))
    _check(rc, "zero_shard_step_sgd_async")


# -------------------------------------------------------------- 8-bit Adam ---

class Adam8View:
    """One shard of 8-bit Adam state and the C struct that describes it.

    grads, params, n as ShardView; master: pair of fp32 CUDA tensors; m_codes,
    v_codes: pairs of uint8 CUDA tensors (>= n); m_scale, v_scale: pairs of
    fp32 CUDA tensors (>= ceil(n / ZS_ADAM8_BLOCK))."""

    def __init__(self, grads: Sequence[torch.Tensor], master, m_codes, v_codes, m_scale, v_scale,
                 params: torch.Tensor, n: int):
        self.grads = list(grads)
        self.master, self.m_codes, self.v_codes = tuple(master), tuple(m_codes), tuple(v_codes)
        self.m_scale, self.v_scale = tuple(m_scale), tuple(v_scale)
        self.params = params
        self.n = int(n)
        blocks = (self.n + ZS_ADAM8_BLOCK - 1) // ZS_ADAM8_BLOCK
        for pair in (self.m_codes, self.v_codes):
            if any(t.numel() < self.n for t in pair):
                raise ValueError("code buffers too small")
        for pair in (self.m_scale, self.v_scale):
            if any(t.numel() < blocks for t in pair):
                raise ValueError("scale buffers too small")
        self._table = (_P * max(len(self.grads), 1))(
            *[_dev_ptr(g, torch.float16, "grads") for g in self.grads])
        self.struct = Adam8Shard()
        self.struct.grads = ctypes.cast(self._table, ctypes.POINTER(_P))
        for i in range(2):
            self.struct.master[i] = _dev_ptr(self.master[i], torch.float32, "master")
            self.struct.m_codes[i] = _dev_ptr(self.m_codes[i], torch.uint8, "m_codes")
            self.struct.v_codes[i] = _dev_ptr(self.v_codes[i], torch.uint8, "v_codes")
            self.struct.m_scale[i] = _dev_ptr(self.m_scale[i], torch.float32, "m_scale")
            self.struct.v_scale[i] = _dev_ptr(self.v_scale[i], torch.float32, "v_scale")
        self.struct.params = _dev_ptr(params, torch.float16, "params")
        self.struct.n = self.n


def zero_shard_step_adam8_async(shards: Sequence[Adam8View], n_d: int, hp: Adam, ctrl_dev: torch.Tensor,
                                stream=None):
    """Stream-ordered step with 8-bit Adam states."""
    arr = (Adam8Shard * len(shards))()
    for i, s in enumerate(shards):
        arr[i] = s.struct
    rc = lib().zero_shard_step_adam8_async(arr, len(shards), int(n_d), ctypes.byref(hp),
                                           _dev_ptr(ctrl_dev, torch.int64, "ctrl_dev"), _stream(stream))
    _check(rc, "zero_shard_step_adam8_async")


def zero_adam8_maps():
    """The library's code maps: (mag7[128], mag8[256]) float32 numpy arrays."""
    mag7 = np.empty(128, np.float32)
    mag8 = np.empty(256, np.float32)
    _check(lib().zero_adam8_maps(mag7.ctypes.data, mag8.ctypes.data), "zero_adam8_maps")
    return mag7, mag8


def zero_shard_step(shards: Sequence[ShardView], n_d: int, hp: Adam, loss_scale: float, step: int, cur: int,
                    flag_dev: torch.Tensor, stream=None) -> int:
    """Synchronous step over ``shards``; returns the overflow flag (0/1)."""
    arr = _shard_array(shards)
    ovf = _I32(-1)
    rc = lib().zero_shard_step(arr, len(shards), int(n_d), ctypes.byref(hp), float(loss_scale), int(step),
                               int(cur), _dev_ptr(flag_dev, torch.int32, "flag_dev"), _stream(stream),
                               ctypes.byref(ovf))
    _check(rc, "zero_shard_step")
    return int(ovf.value)


def zero_shard_step_noalloc(shards: Sequence[ShardView], n_d: int, hp: Adam, loss_scale: float, step: int,
                            cur: int, stream=None) -> int:
    """zero_shard_step without the caller's flag buffer: for callers that may
    not allocate device memory, the overflow words live in a small array
    compiled into the library.  Returns the overflow flag (0/1)."""
    arr = _shard_array(shards)
    ovf = _I32(-1)
    rc = lib().zero_shard_step_noalloc(arr, len(shards), int(n_d), ctypes.byref(hp), float(loss_scale),
                                       int(step), int(cur), _stream(stream), ctypes.byref(ovf))
    if rc != ZS_OK:
        raise ZeroShardError(rc, "zero_shard_step_noalloc", zero_last_error())
    return int(ovf.value)


def new_ctrl(device="cuda") -> torch.Tensor:
    """Device memory for one zs_ctrl (int64-typed so it is 8-byte aligned)."""
    return torch.zeros((CTRL_BYTES + 7) // 8, dtype=torch.int64, device=device)


def zero_ctrl_init(ctrl_dev: torch.Tensor, loss_scale: float, stream=None):
    rc = lib().zero_ctrl_init(_dev_ptr(ctrl_dev, torch.int64, "ctrl_dev"), float(loss_scale), _stream(stream))
    _check(rc, "zero_ctrl_init")


def zero_shard_step_async(shards: Sequence[ShardView], n_d: int, hp: Adam, ctrl_dev: torch.Tensor, stream=None):
    arr = _shard_array(shards)
    rc = lib().zero_shard_step_async(arr, len(shards), int(n_d), ctypes.byref(hp),
                                     _dev_ptr(ctrl_dev, torch.int64, "ctrl_dev"), _stream(stream))
    _check(rc, "zero_shard_step_async")


def zero_shard_reduce_adam_all_async(shards: Sequence[ShardView], n_d: int, hp: Adam, ctrl_dev: torch.Tensor,
                                     stream=None):
    arr = _shard_array(shards)
    rc = lib().zero_shard_reduce_adam_all_async(arr, len(shards), int(n_d), ctypes.byref(hp),
                                                _dev_ptr(ctrl_dev, torch.int64, "ctrl_dev"), _stream(stream))
    _check(rc, "zero_shard_reduce_adam_all_async")


class HostShardView(ShardView):
    """A shard whose gradient contributions and fp16 slice (and optional qwZ
    copy) are page-locked HOST tensors (``tensor.pin_memory()``); master/m/v
    are CUDA tensors."""

    def __init__(self, grads, master, m, v, params, n, qcodes=None, qscales=None):
        for g in list(grads) + [params]:
            if g.is_cuda or not g.is_pinned() or g.dtype != torch.float16 or not g.is_contiguous():
                raise TypeError("host shard: grads and params must be contiguous pinned fp16 host tensors")
        self.grads = list(grads)
        self.master, self.m, self.v = tuple(master), tuple(m), tuple(v)
        self.params = params
        self.n = int(n)
        self._table = (_P * max(len(self.grads), 1))(*[g.data_ptr() for g in self.grads])
        self.struct = Shard()
        self.struct.grads = ctypes.cast(self._table, ctypes.POINTER(_P))
        for i in range(2):
            self.struct.master[i] = _dev_ptr(self.master[i], torch.float32, "master")
            self.struct.m[i] = _dev_ptr(self.m[i], torch.float32, "m")
            self.struct.v[i] = _dev_ptr(self.v[i], torch.float32, "v")
        self.struct.params = params.data_ptr()
        self.struct.n = self.n
        self.qcodes, self.qscales = qcodes, qscales
        if qcodes is not None:
            for t in (qcodes, qscales):
                if t.is_cuda or not t.is_pinned():
                    raise TypeError("host shard: qwZ buffers must be pinned host tensors")
            self.struct.qcodes = qcodes.data_ptr()
            self.struct.qscales = qscales.data_ptr()


class CpuShardView(ShardView):
    """A shard whose buffers all live in host memory (CPU torch tensors), for
    the step on the host cores."""

    def __init__(self, grads, master, m, v, params, n):
        def host(t, dtype, what):
            if t.is_cuda or t.dtype != dtype or not t.is_contiguous():
                raise TypeError(f"{what}: expected a contiguous host {dtype} tensor")
            return t.data_ptr()
        self.grads = list(grads)
        self.master, self.m, self.v = tuple(master), tuple(m), tuple(v)
        self.params = params
        self.n = int(n)
        self._table = (_P * max(len(self.grads), 1))(*[host(g, torch.float16, "grads") for g in self.grads])
        self.struct = Shard()
        self.struct.grads = ctypes.cast(self._table, ctypes.POINTER(_P))
        for i in range(2):
            self.struct.master[i] = host(self.master[i], torch.float32, "master")
            self.struct.m[i] = host(self.m[i], torch.float32, "m")
            self.struct.v[i] = host(self.v[i], torch.float32, "v")
        self.struct.params = host(params, torch.float16, "params")
        self.struct.n = self.n


def zero_shard_step_cpu(shards: Sequence[ShardView], n_d: int, hp: Adam, loss_scale: float, step: int, cur: int,
                        n_threads: int = 0) -> int:
    """The shard step on the host cores (every buffer in host memory); returns
    the overflow flag.  Same results as zero_shard_step, bit for bit."""
    arr = _shard_array(shards)
    ovf = _I32(-1)
    rc = lib().zero_shard_step_cpu(arr, len(shards), int(n_d), ctypes.byref(hp), float(loss_scale), int(step),
                                   int(cur), int(n_threads), ctypes.byref(ovf))
    _check(rc, "zero_shard_step_cpu")
    return int(ovf.value)


class OffloadShardView:
    """One rank's shard for the ZeRO-Offload step: the device contributions
    and fp16 slice, page-locked host staging buffers for both, and the host
    fp32 state (two sets each of master, m, v)."""

    def __init__(self, grads_dev, params_dev, grads_host, params_host, master, m, v, n):
        def host(t, dtype, what, pinned=False):
            if t.is_cuda or t.dtype != dtype or not t.is_contiguous():
                raise TypeError(f"{what}: expected a contiguous host {dtype} tensor")
            if pinned and not t.is_pinned():
                raise TypeError(f"{what}: expected page-locked host memory (pin_memory())")
            return t.data_ptr()
        self.n = int(n)
        self.grads_dev, self.grads_host = list(grads_dev), list(grads_host)
        self.params_dev, self.params_host = params_dev, params_host
        self.master, self.m, self.v = tuple(master), tuple(m), tuple(v)
        self._dev = (_P * max(len(self.grads_dev), 1))(*[_dev_ptr(g, torch.float16, "grads_dev")
                                                          for g in self.grads_dev])
        self._host = (_P * max(len(self.grads_host), 1))(*[host(g, torch.float16, "grads_host", True)
                                                           for g in self.grads_host])
        self.struct = OffloadShard()
        self.struct.grads_dev = ctypes.cast(self._dev, ctypes.POINTER(_P))
        self.struct.grads_host = ctypes.cast(self._host, ctypes.POINTER(_P))
        self.struct.params_dev = _dev_ptr(params_dev, torch.float16, "params_dev")
        self.struct.params_host = host(params_host, torch.float16, "params_host", True)
        for i in range(2):
            self.struct.master[i] = host(self.master[i], torch.float32, "master")
            self.struct.m[i] = host(self.m[i], torch.float32, "m")
            self.struct.v[i] = host(self.v[i], torch.float32, "v")
        self.struct.n = self.n


def zero_shard_step_offload(shard: OffloadShardView, n_d: int, hp: Adam, loss_scale: float, step: int, cur: int,
                            n_threads: int = 0, chunk: int = 0, d2h_stream=None, h2d_stream=None) -> int:
    """ZeRO-Offload step: contributions to the host, the step on the host
    cores, fp16 parameters back to the device, overlapped by chunks; returns
    the overflow flag (synchronous)."""
    ovf = _I32(-1)
    rc = lib().zero_shard_step_offload(ctypes.byref(shard.struct), int(n_d), ctypes.byref(hp), float(loss_scale),
                                       int(step), int(cur), int(n_threads), int(chunk), _stream(d2h_stream),
                                       _stream(h2d_stream), ctypes.byref(ovf))
    _check(rc, "zero_shard_step_offload")
    return int(ovf.value)


def zero_shard_step_host(shard: HostShardView, n_d: int, hp: Adam, ctrl_dev: torch.Tensor, stream=None) -> int:
    """Step with host-resident contributions and fp16 shard; returns the flag."""
    ovf = _I32(-1)
    rc = lib().zero_shard_step_host(ctypes.byref(shard.struct), int(n_d), ctypes.byref(hp),
                                    _dev_ptr(ctrl_dev, torch.int64, "ctrl_dev"), _stream(stream),
                                    ctypes.byref(ovf))
    _check(rc, "zero_shard_step_host")
    return int(ovf.value)


def zero_shard_reduce_adam_async(shard: ShardView, n_d: int, hp: Adam, ctrl_dev: torch.Tensor, stream=None):
    rc = lib().zero_shard_reduce_adam_async(ctypes.byref(shard.struct), int(n_d), ctypes.byref(hp),
                                            _dev_ptr(ctrl_dev, torch.int64, "ctrl_dev"), _stream(stream))
    _check(rc, "zero_shard_reduce_adam_async")


def zero_step_commit_async(shards: Sequence[ShardView], hp: Adam, ctrl_dev: torch.Tensor, stream=None):
    arr = _shard_array(shards)
    rc = lib().zero_step_commit_async(arr, len(shards), ctypes.byref(hp),
                                      _dev_ptr(ctrl_dev, torch.int64, "ctrl_dev"), _stream(stream))
    _check(rc, "zero_step_commit_async")


def new_sqnorm(device="cuda") -> torch.Tensor:
    """Device accumulator for the squared gradient norm (one float64)."""
    return torch.zeros(1, dtype=torch.float64, device=device)


def zero_shard_grad_sqnorm_async(shard: ShardView, n_d: int, sqnorm_dev: torch.Tensor, ctrl_dev: torch.Tensor,
                                 g_dev: Optional[torch.Tensor] = None, stream=None):
    """Clipping pass 1 for one shard: adds its sum of squares to sqnorm_dev."""
    rc = lib().zero_shard_grad_sqnorm_async(ctypes.byref(shard.struct), int(n_d),
                                            _dev_ptr(g_dev, torch.float32, "g_dev"),
                                            _dev_ptr(sqnorm_dev, torch.float64, "sqnorm_dev"),
                                            _dev_ptr(ctrl_dev, torch.int64, "ctrl_dev"), _stream(stream))
    _check(rc, "zero_shard_grad_sqnorm_async")


def zero_shard_clipped_adam_async(shard: ShardView, n_d: int, hp: Adam, max_norm: float, sqnorm_dev: torch.Tensor,
                                  ctrl_dev: torch.Tensor, g_dev: Optional[torch.Tensor] = None, stream=None):
    """Clipping pass 2 for one shard: clipped update and fp16 cast."""
    rc = lib().zero_shard_clipped_adam_async(ctypes.byref(shard.struct), int(n_d), ctypes.byref(hp),
                                             float(max_norm), _dev_ptr(g_dev, torch.float32, "g_dev"),
                                             _dev_ptr(sqnorm_dev, torch.float64, "sqnorm_dev"),
                                             _dev_ptr(ctrl_dev, torch.int64, "ctrl_dev"), _stream(stream))
    _check(rc, "zero_shard_clipped_adam_async")


def zero_shard_step_clipped_async(shards: Sequence[ShardView], n_d: int, hp: Adam, max_norm: float,
                                  sqnorm_dev: torch.Tensor, ctrl_dev: torch.Tensor,
                                  g_dev: Optional[Sequence[Optional[torch.Tensor]]] = None, stream=None):
    """Whole clipped step over shards that all live on this device."""
    arr = _shard_array(shards)
    table = None
    if g_dev is not None:
        table = (_P * len(shards))(*[_dev_ptr(g, torch.float32, "g_dev") for g in g_dev])
    rc = lib().zero_shard_step_clipped_async(arr, len(shards), int(n_d), ctypes.byref(hp), float(max_norm), table,
                                             _dev_ptr(sqnorm_dev, torch.float64, "sqnorm_dev"),
                                             _dev_ptr(ctrl_dev, torch.int64, "ctrl_dev"), _stream(stream))
    _check(rc, "zero_shard_step_clipped_async")


def _g_table(shards, g_dev):
    if g_dev is None:
        return None
    return (_P * len(shards))(*[_dev_ptr(g, torch.float32, "g_dev") for g in g_dev])


def zero_shard_grad_sqnorm_all_async(shards: Sequence[ShardView], n_d: int, sqnorm_dev: torch.Tensor,
                                     ctrl_dev: torch.Tensor, g_dev=None, stream=None):
    """Clipping pass 1 for a list of shards (grouped launches)."""
    arr = _shard_array(shards)
    rc = lib().zero_shard_grad_sqnorm_all_async(arr, len(shards), int(n_d), _g_table(shards, g_dev),
                                                _dev_ptr(sqnorm_dev, torch.float64, "sqnorm_dev"),
                                                _dev_ptr(ctrl_dev, torch.int64, "ctrl_dev"), _stream(stream))
    _check(rc, "zero_shard_grad_sqnorm_all_async")


def zero_shard_clipped_adam_all_async(shards: Sequence[ShardView], n_d: int, hp: Adam, max_norm: float,
                                      sqnorm_dev: torch.Tensor, ctrl_dev: torch.Tensor, g_dev=None, stream=None):
    """Clipping pass 2 for a list of shards (grouped launches)."""
    arr = _shard_array(shards)
    rc = lib().zero_shard_clipped_adam_all_async(arr, len(shards), int(n_d), ctypes.byref(hp), float(max_norm),
                                                 _g_table(shards, g_dev),
                                                 _dev_ptr(sqnorm_dev, torch.float64, "sqnorm_dev"),
                                                 _dev_ptr(ctrl_dev, torch.int64, "ctrl_dev"), _stream(stream))
    _check(rc, "zero_shard_clipped_adam_all_async")


def zero_params_from_master(master: torch.Tensor, params: torch.Tensor, n: int, stream=None):
    rc = lib().zero_params_from_master(_dev_ptr(master, torch.float32, "master"),
                                       _dev_ptr(params, torch.float16, "params"), int(n), _stream(stream))
    _check(rc, "zero_params_from_master")


def zero_qwz_quantize(params: torch.Tensor, n: int, codes: torch.Tensor, scales: torch.Tensor, stream=None):
    """int8 codes and per-256 fp32 scales of an fp16 slice (stream-ordered)."""
    rc = lib().zero_qwz_quantize(_dev_ptr(params, torch.float16, "params"), int(n),
                                 _dev_ptr(codes, torch.int8, "codes"), _dev_ptr(scales, torch.float32, "scales"),
                                 _stream(stream))
    _check(rc, "zero_qwz_quantize")


def zero_qwz_dequantize(codes: torch.Tensor, scales: torch.Tensor, n: int, params: torch.Tensor, stream=None):
    """fp16 slice rebuilt from int8 codes and scales (the all-gather receiver)."""
    rc = lib().zero_qwz_dequantize(_dev_ptr(codes, torch.int8, "codes"), _dev_ptr(scales, torch.float32, "scales"),
                                   int(n), _dev_ptr(params, torch.float16, "params"), _stream(stream))
    _check(rc, "zero_qwz_dequantize")


def read_ctrl(ctrl_dev: torch.Tensor) -> dict:
    """Host snapshot of a device control block (synchronises the copy)."""
    raw = ctrl_dev.detach().cpu().numpy().tobytes()[:CTRL_BYTES]
    c = Ctrl.from_buffer_copy(raw)
    return {name: getattr(c, name) for name, _ in Ctrl._fields_}
