"""CPU oracle for the KV-cache write path -- TEST INFRASTRUCTURE ONLY.

This package wraps ``kv_oracle.c`` (a plain C restatement of the write path,
compiled with gcc) for the tests, the package smoke check and the
benchmark's CPU-baseline leg. Nothing else may import it; the CUDA library
neither links nor calls it, and it shares no code with the library.

Functions follow sglang's ``kvcache.cuh`` (kernel ``store_kvcache``: byte copy
of each token's K and V row into slot ``indices[token]``, with the rule
``0 <= slot < size_limit``) and ``trtllm_fp8_kv_kernel.py`` (kernels
``_fused_fp8_set_kv_buffer_kernel`` / ``_process_kv_tensor``: page
decomposition of the slot, fp32 multiply by the inverse scale, conversion to
FP8 e4m3fn).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kv_oracle.c")
_SRC_THREADS = os.path.join(_HERE, "kv_oracle_threads.c")
_LIBDIR = os.path.join(_HERE, "lib")
_LIB = os.path.join(_LIBDIR, "libkvoracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/lib/libkvoracle.so``."""
    if (not force and os.path.exists(_LIB)
            and all(os.path.getmtime(_LIB) >= os.path.getmtime(s) for s in (_SRC, _SRC_THREADS))):
        return _LIB
    os.makedirs(_LIBDIR, exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, _SRC_THREADS, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        lib.kvo_e4m3fn_encode.argtypes = [ctypes.c_float]
        lib.kvo_e4m3fn_encode.restype = ctypes.c_uint8
        lib.kvo_e4m3fn_decode.argtypes = [ctypes.c_uint8]
        lib.kvo_e4m3fn_decode.restype = ctypes.c_double
        lib.kvo_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.kvo_bf16_to_f32.restype = ctypes.c_float
        lib.kvo_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.kvo_f16_to_f32.restype = ctypes.c_float
        lib.kvo_scale_f32.argtypes = [ctypes.c_float, ctypes.c_float]
        lib.kvo_scale_f32.restype = ctypes.c_float
        lib.kvo_encode_f32_array.argtypes = [P, P, I64]
        lib.kvo_decode_array.argtypes = [P, P, I64]
        lib.kvo_store_copy.argtypes = [P, P, P, P, P, I32, I64, I64, I64, I32, I32, I32,
                                       P, I64, P, P]
        lib.kvo_store_copy.restype = I32
        lib.kvo_store_fp8.argtypes = [P, P, P, P, P, I32, I64, I64, I64, I32, I32, I32,
                                      P, I64, I64, I64, I64, ctypes.c_float, ctypes.c_float,
                                      I32, P, P]
        lib.kvo_store_fp8.restype = I32
        lib.kvo_store_copy_paged.argtypes = [P, P, P, P, P, I32, I64, I64, I64, I32, I32, I32,
                                             P, I64, I64, I64, I64, P, P]
        lib.kvo_store_copy_paged.restype = I32
        lib.kvo_inv_scale.argtypes = [ctypes.c_float]
        lib.kvo_inv_scale.restype = ctypes.c_float
        lib.kvo_absmax_inv.argtypes = [P, P, I32, I64, I32, I32, P, ctypes.c_float, P, P]
        lib.kvo_e5m2_encode_array.argtypes = [P, P, I64]
        lib.kvo_e5m2_decode_array.argtypes = [P, P, I64]
        lib.kvo_store_fp8_ex.argtypes = [P, P, P, P, P, I32, I64, I64, I64, I32, I32, I32, P, I64,
                                         I64, I64, I64, I32, I32, ctypes.c_float, ctypes.c_float,
                                         P, P, I64, P, P]
        lib.kvo_store_fp8_ex.restype = I32
        lib.kvo_gather_fp8_ex.argtypes = [P, P, P, P, P, I32, I64, I64, I64, I32, I32, I32, P,
                                          I64, I64, I64, I64, I32, I32, ctypes.c_float,
                                          ctypes.c_float, P, P, I64, P, P]
        lib.kvo_gather_fp8_ex.restype = I32
        lib.kvo_gather_copy.argtypes = lib.kvo_store_copy.argtypes
        lib.kvo_gather_copy.restype = I32
        lib.kvo_gather_copy_paged.argtypes = lib.kvo_store_copy_paged.argtypes
        lib.kvo_gather_copy_paged.restype = I32
        lib.kvo_gather_fp8.argtypes = lib.kvo_store_fp8.argtypes
        lib.kvo_gather_fp8.restype = I32
        lib.kvo_run_threads.argtypes = [P, I64, I32, ctypes.c_double, I64, P, P, P]
        lib.kvo_run_threads.restype = I32
        lib.kvo_f32_to_bf16_array.argtypes = [P, P, I64]
        lib.kvo_f32_to_f16_array.argtypes = [P, P, I64]
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# -- number formats ---------------------------------------------------------

def e4m3fn_encode(x) -> np.ndarray:
    """e4m3fn codes (uint8) of float32 values: nearest, ties even, saturating."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().kvo_encode_f32_array(_ptr(x), _ptr(out), x.size)
    return out


def e4m3fn_decode(codes) -> np.ndarray:
    """Exact float64 values of e4m3fn codes (NaN for 0x7F / 0xFF)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().kvo_decode_array(_ptr(c), _ptr(out), c.size)
    return out


def f32_to_bf16(x) -> np.ndarray:
    """bf16 bits (uint16) of float32 values: nearest, ties even, NaN -> 0x7FFF."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().kvo_f32_to_bf16_array(_ptr(x), _ptr(out), x.size)
    return out


def f32_to_f16(x) -> np.ndarray:
    """IEEE fp16 bits (uint16) of float32 values: nearest, ties even, NaN -> 0x7FFF."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().kvo_f32_to_f16_array(_ptr(x), _ptr(out), x.size)
    return out


def bf16_to_f32(bits: int) -> float:
    return _load().kvo_bf16_to_f32(bits)


def f16_to_f32(bits: int) -> float:
    return _load().kvo_f16_to_f32(bits)


def scale_f32(x: float, inv: float) -> float:
    return _load().kvo_scale_f32(x, inv)


# -- the write path ---------------------------------------------------------

class Strides:
    """Byte strides of K, V and the two caches, in the library's order."""

    FIELDS = ("k_token", "k_head", "k_dim", "v_token", "v_head", "v_dim",
              "kc_slot", "kc_head", "kc_dim", "vc_slot", "vc_head", "vc_dim")

    def __init__(self, **kw):
        self.values = np.array([int(kw[f]) for f in self.FIELDS], dtype=np.int64)


def _check_buf(a: np.ndarray, name: str):
    if not (isinstance(a, np.ndarray) and a.flags.c_contiguous):
        raise TypeError(f"{name} must be a C-contiguous numpy array")


def store_copy(k, v, k_cache, v_cache, indices, strides: Strides, num_heads, head_dim,
               elem_bytes, size_limit, k_off=0, v_off=0, kc_off=0, vc_off=0,
               index_stride=1, t_begin=0, t_end=None):
    """Plain copy scatter into host caches (in place). Returns (bad_count, first_bad).

    ``k``/``v``/``k_cache``/``v_cache`` are host arrays; ``*_off`` are byte
    offsets of the first element inside them (views such as a fused QKV).
    """
    for a, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_buf(a, n)
    idx = np.ascontiguousarray(indices)
    if idx.dtype not in (np.int32, np.int64):
        raise TypeError("indices must be int32 or int64")
    T = idx.size // index_stride if t_end is None else t_end
    bad = np.zeros(1, np.int64)
    first = np.zeros(1, np.int64)
    rc = _load().kvo_store_copy(_ptr(k) + k_off, _ptr(v) + v_off, _ptr(k_cache) + kc_off,
                                _ptr(v_cache) + vc_off, _ptr(idx), int(idx.dtype == np.int64),
                                index_stride, t_begin, T, num_heads, head_dim, elem_bytes,
                                _ptr(strides.values), size_limit, _ptr(bad), _ptr(first))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return int(bad[0]), int(first[0])


def store_copy_paged(k, v, k_cache, v_cache, indices, strides: Strides, num_heads, head_dim,
                     elem_bytes, page_size, kc_page_stride, vc_page_stride, size_limit, k_off=0,
                     v_off=0, index_stride=1, t_end=None):
    """Paged plain copy (4-D cache). Returns (bad_count, first_bad)."""
    for a, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_buf(a, n)
    idx = np.ascontiguousarray(indices)
    T = idx.size // index_stride if t_end is None else t_end
    bad = np.zeros(1, np.int64)
    first = np.zeros(1, np.int64)
    rc = _load().kvo_store_copy_paged(_ptr(k) + k_off, _ptr(v) + v_off, _ptr(k_cache),
                                      _ptr(v_cache), _ptr(idx), int(idx.dtype == np.int64),
                                      index_stride, 0, T, num_heads, head_dim, elem_bytes,
                                      _ptr(strides.values), page_size, kc_page_stride,
                                      vc_page_stride, size_limit, _ptr(bad), _ptr(first))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return int(bad[0]), int(first[0])


def store_fp8(k, v, k_cache, v_cache, indices, strides: Strides, num_heads, head_dim,
              src_dtype, page_size, kc_page_stride, vc_page_stride, size_limit,
              inv_k=1.0, inv_v=1.0, use_scale=0, k_off=0, v_off=0, index_stride=1,
              t_begin=0, t_end=None):
    """Fused scale + e4m3fn scatter into host uint8 caches (in place).

    Returns (bad_count, first_bad)."""
    for a, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_buf(a, n)
    idx = np.ascontiguousarray(indices)
    if idx.dtype not in (np.int32, np.int64):
        raise TypeError("indices must be int32 or int64")
    if src_dtype not in ("bf16", "f16"):
        raise ValueError(src_dtype)
    T = idx.size // index_stride if t_end is None else t_end
    bad = np.zeros(1, np.int64)
    first = np.zeros(1, np.int64)
    rc = _load().kvo_store_fp8(_ptr(k) + k_off, _ptr(v) + v_off, _ptr(k_cache), _ptr(v_cache),
                               _ptr(idx), int(idx.dtype == np.int64), index_stride, t_begin, T,
                               num_heads, head_dim, int(src_dtype == "bf16"),
                               _ptr(strides.values), page_size, kc_page_stride,
                               vc_page_stride, size_limit, float(np.float32(inv_k)),
                               float(np.float32(inv_v)), int(use_scale), _ptr(bad), _ptr(first))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return int(bad[0]), int(first[0])


# -- the inverse path (cache rows back to token rows) -------------------------

def gather_copy(k_cache, v_cache, k_out, v_out, indices, strides: Strides, num_heads, head_dim,
                elem_bytes, size_limit, kc_off=0, vc_off=0, index_stride=1, t_end=None):
    """Row t of the outputs takes cache row indices[t] (byte copy); out-of-range
    slots leave the row untouched. ``strides``: k_*/v_* describe the outputs,
    kc_*/vc_* the caches. Returns (bad_count, first_bad)."""
    for a, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (k_out, "k_out"), (v_out, "v_out")):
        _check_buf(a, n)
    idx = np.ascontiguousarray(indices)
    T = idx.size // index_stride if t_end is None else t_end
    bad = np.zeros(1, np.int64)
    first = np.zeros(1, np.int64)
    rc = _load().kvo_gather_copy(_ptr(k_cache) + kc_off, _ptr(v_cache) + vc_off, _ptr(k_out),
                                 _ptr(v_out), _ptr(idx), int(idx.dtype == np.int64), index_stride,
                                 0, T, num_heads, head_dim, elem_bytes, _ptr(strides.values),
                                 size_limit, _ptr(bad), _ptr(first))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return int(bad[0]), int(first[0])


def gather_copy_paged(k_cache, v_cache, k_out, v_out, indices, strides: Strides, num_heads,
                      head_dim, elem_bytes, page_size, kc_page_stride, vc_page_stride,
                      size_limit, index_stride=1, t_end=None):
    """Gather from a paged cache (the inverse of store_copy_paged)."""
    for a, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (k_out, "k_out"), (v_out, "v_out")):
        _check_buf(a, n)
    idx = np.ascontiguousarray(indices)
    T = idx.size // index_stride if t_end is None else t_end
    bad = np.zeros(1, np.int64)
    first = np.zeros(1, np.int64)
    rc = _load().kvo_gather_copy_paged(_ptr(k_cache), _ptr(v_cache), _ptr(k_out), _ptr(v_out),
                                       _ptr(idx), int(idx.dtype == np.int64), index_stride, 0, T,
                                       num_heads, head_dim, elem_bytes, _ptr(strides.values),
                                       page_size, kc_page_stride, vc_page_stride, size_limit,
                                       _ptr(bad), _ptr(first))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return int(bad[0]), int(first[0])


def gather_fp8(k_cache, v_cache, k_out, v_out, indices, strides: Strides, num_heads, head_dim,
               out_dtype, page_size, kc_page_stride, vc_page_stride, size_limit, scale_k=1.0,
               scale_v=1.0, use_scale=0, index_stride=1, t_end=None):
    """Dequantising gather: e4m3fn -> fp32 (* scale) -> bf16 / fp16 rows."""
    for a, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (k_out, "k_out"), (v_out, "v_out")):
        _check_buf(a, n)
    if out_dtype not in ("bf16", "f16"):
        raise ValueError(out_dtype)
    idx = np.ascontiguousarray(indices)
    T = idx.size // index_stride if t_end is None else t_end
    bad = np.zeros(1, np.int64)
    first = np.zeros(1, np.int64)
    rc = _load().kvo_gather_fp8(_ptr(k_cache), _ptr(v_cache), _ptr(k_out), _ptr(v_out),
                                _ptr(idx), int(idx.dtype == np.int64), index_stride, 0, T,
                                num_heads, head_dim, int(out_dtype == "bf16"),
                                _ptr(strides.values), page_size, kc_page_stride, vc_page_stride,
                                size_limit, float(np.float32(scale_k)), float(np.float32(scale_v)),
                                int(use_scale), _ptr(bad), _ptr(first))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return int(bad[0]), int(first[0])


# -- scale preparation ---------------------------------------------------------

def inv_scale(scale) -> np.ndarray:
    """fl32(1 / scale) elementwise (correctly rounded fp32 reciprocal)."""
    sc = np.ascontiguousarray(scale, dtype=np.float32).ravel()
    return np.array([_load().kvo_inv_scale(float(x)) for x in sc], dtype=np.float32)


def absmax_inv(k, v, strides: Strides, num_tokens, num_heads, head_dim, src_dtype, fp8_max=448.0,
               k_off=0, v_off=0):
    """(amax[2], inv[2]) float32: per-tensor max |x| (NaN ignored) of K and V and
    fp8_max / amax (1.0 when amax is 0)."""
    for a, n in ((k, "k"), (v, "v")):
        _check_buf(a, n)
    amax = np.zeros(2, np.float32)
    inv = np.zeros(2, np.float32)
    _load().kvo_absmax_inv(_ptr(k) + k_off, _ptr(v) + v_off, int(src_dtype == "bf16"), num_tokens,
                           num_heads, head_dim, _ptr(strides.values), float(np.float32(fp8_max)),
                           _ptr(amax), _ptr(inv))
    return amax, inv


# -- e5m2 and the extended FP8 write / gather -------------------------------------

FMT = {"e4m3fn": 0, "e5m2": 1}
SCALE_MODE = {"none": 0, "tensor": 1, "token": 2, "token_head": 3, "page": 4}


def e5m2_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().kvo_e5m2_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def e5m2_decode(codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().kvo_e5m2_decode_array(_ptr(c), _ptr(out), c.size)
    return out


def _null_or(a):
    return None if a is None else _ptr(a)


def store_fp8_ex(k, v, k_cache, v_cache, indices, strides: Strides, num_heads, head_dim,
                 src_dtype, page_size, kc_page_stride, vc_page_stride, size_limit, fmt="e4m3fn",
                 scale_mode="none", inv_k=1.0, inv_v=1.0, k_scales=None, v_scales=None,
                 scales_slot_stride=1, k_off=0, v_off=0, index_stride=1, t_end=None):
    """Extended FP8 write (format, scale mode, per-slot scale caches); in place.
    With ``scale_mode="page"``, ``k_scales`` / ``v_scales`` hold one fp32
    INVERSE scale per cache page (index slot // page_size), read only.
    Returns (bad_count, first_bad)."""
    for a, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_buf(a, n)
    for a in (k_scales, v_scales):
        if a is not None:
            assert a.dtype == np.float32 and a.flags.c_contiguous
    idx = np.ascontiguousarray(indices)
    T = idx.size // index_stride if t_end is None else t_end
    bad = np.zeros(1, np.int64)
    first = np.zeros(1, np.int64)
    rc = _load().kvo_store_fp8_ex(_ptr(k) + k_off, _ptr(v) + v_off, _ptr(k_cache), _ptr(v_cache),
                                  _ptr(idx), int(idx.dtype == np.int64), index_stride, 0, T,
                                  num_heads, head_dim, int(src_dtype == "bf16"),
                                  _ptr(strides.values), page_size, kc_page_stride, vc_page_stride,
                                  size_limit, FMT[fmt], SCALE_MODE[scale_mode],
                                  float(np.float32(inv_k)), float(np.float32(inv_v)),
                                  _null_or(k_scales), _null_or(v_scales), scales_slot_stride,
                                  _ptr(bad), _ptr(first))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return int(bad[0]), int(first[0])


def gather_fp8_ex(k_cache, v_cache, k_out, v_out, indices, strides: Strides, num_heads, head_dim,
                  out_dtype, page_size, kc_page_stride, vc_page_stride, size_limit,
                  fmt="e4m3fn", scale_mode="none", scale_k=1.0, scale_v=1.0, k_scales=None,
                  v_scales=None, scales_slot_stride=1, index_stride=1, t_end=None):
    """Extended dequantising gather. With ``scale_mode="page"``, ``k_scales`` /
    ``v_scales`` hold one fp32 (forward) scale per cache page. Returns
    (bad_count, first_bad)."""
    for a, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (k_out, "k_out"), (v_out, "v_out")):
        _check_buf(a, n)
    idx = np.ascontiguousarray(indices)
    T = idx.size // index_stride if t_end is None else t_end
    bad = np.zeros(1, np.int64)
    first = np.zeros(1, np.int64)
    rc = _load().kvo_gather_fp8_ex(_ptr(k_cache), _ptr(v_cache), _ptr(k_out), _ptr(v_out),
                                   _ptr(idx), int(idx.dtype == np.int64), index_stride, 0, T,
                                   num_heads, head_dim, int(out_dtype == "bf16"),
                                   _ptr(strides.values), page_size, kc_page_stride,
                                   vc_page_stride, size_limit, FMT[fmt], SCALE_MODE[scale_mode],
                                   float(np.float32(scale_k)), float(np.float32(scale_v)),
                                   _null_or(k_scales), _null_or(v_scales), scales_slot_stride,
                                   _ptr(bad), _ptr(first))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return int(bad[0]), int(first[0])


# -- host-thread runner (CPU baseline timing) ---------------------------------

class _Job(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("index_is_i64", ctypes.c_int32),
                ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("indices", ctypes.c_void_p), ("index_stride", ctypes.c_int64),
                ("num_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("use_scale", ctypes.c_int32),
                ("strides", ctypes.c_void_p), ("page_size", ctypes.c_int64),
                ("kc_page_stride", ctypes.c_int64), ("vc_page_stride", ctypes.c_int64),
                ("size_limit", ctypes.c_int64), ("inv_k", ctypes.c_float),
                ("inv_v", ctypes.c_float)]


JOB_KINDS = {"copy": 0, "copy_paged": 1, "fp8": 2}


class ThreadedJob:
    """One write problem for ``kvo_run_threads``: the unchanged oracle loop
    (``store_copy``, ``store_copy_paged`` or ``store_fp8``) run over token
    ranges on POSIX threads, outside the interpreter lock.

    ``kind`` is ``"copy"``, ``"copy_paged"`` or ``"fp8"``; the keyword
    arguments are those of the matching function above (``elem_bytes`` or
    ``src_dtype``, page geometry, inverse scales)."""

    def __init__(self, kind, k, v, k_cache, v_cache, indices, strides: Strides, num_heads,
                 head_dim, size_limit, elem_bytes=2, src_dtype="bf16", page_size=1,
                 kc_page_stride=0, vc_page_stride=0, inv_k=1.0, inv_v=1.0, use_scale=0,
                 k_off=0, v_off=0, index_stride=1):
        for a, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
            _check_buf(a, n)
        self.idx = np.ascontiguousarray(indices)
        if self.idx.dtype not in (np.int32, np.int64):
            raise TypeError("indices must be int32 or int64")
        self.num_tokens = self.idx.size // index_stride
        self._keep = (k, v, k_cache, v_cache, strides)
        j = _Job()
        j.kind = JOB_KINDS[kind]
        j.index_is_i64 = int(self.idx.dtype == np.int64)
        j.k, j.v = _ptr(k) + k_off, _ptr(v) + v_off
        j.k_cache, j.v_cache = _ptr(k_cache), _ptr(v_cache)
        j.indices = _ptr(self.idx)
        j.index_stride = index_stride
        j.num_heads, j.head_dim = num_heads, head_dim
        j.dtype = int(src_dtype == "bf16") if kind == "fp8" else elem_bytes
        j.use_scale = int(use_scale)
        j.strides = _ptr(strides.values)
        j.page_size = page_size
        j.kc_page_stride, j.vc_page_stride = kc_page_stride, vc_page_stride
        j.size_limit = size_limit
        j.inv_k, j.inv_v = float(np.float32(inv_k)), float(np.float32(inv_v))
        self.job = j

    def run(self, threads: int, seconds: float = 0.0, min_reps: int = 1, num_tokens=None):
        """Thread i repeats tokens [T*i/n, T*(i+1)/n) until ``seconds`` have
        passed and it has made ``min_reps`` passes. Returns (tokens processed,
        elapsed seconds, out-of-range tokens met)."""
        T = self.num_tokens if num_tokens is None else num_tokens
        done = np.zeros(1, np.int64)
        el = np.zeros(1, np.float64)
        bad = np.zeros(1, np.int64)
        rc = _load().kvo_run_threads(ctypes.addressof(self.job), T, threads, seconds, min_reps,
                                     _ptr(done), _ptr(el), _ptr(bad))
        if rc != 0:
            raise ValueError("oracle rejected the arguments")
        return int(done[0]), float(el[0]), int(bad[0])
