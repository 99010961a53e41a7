"""GB300 KV-cache write path: Python binding of ``libkvstore.so``.

The library (the kernels in ``csrc/*.cu``, C ABI in ``include/kvstore.h``) does
all the work; this module only marshals arguments. It exposes the C entry points under
the same names:

* :func:`kv_store`      -- plain byte-exact scatter of K/V rows into cache slots
  (sglang ``kvcache.cuh``, ``store_kvcache``).
* :func:`kv_store_fp8`  -- fused fp32 scale + FP8 e4m3fn conversion + paged
  scatter (sglang ``trtllm_fp8_kv_kernel.py``, ``fused_fp8_set_kv_buffer``).
* :func:`kv_store_paged`, :func:`kv_store_fp8_ex` (e5m2; scales per tensor, or
  per token row / per (token, head) computed in the kernel),
  :func:`kv_gather`, :func:`kv_gather_fp8` (the inverse), :func:`kv_inv_scale`,
  :func:`kv_absmax_inv` (scale preparation), :func:`kv_store_fp8_dynamic_tensor`
  (per-tensor scales formed from the batch and the write, in one call).
* :func:`kv_error_poll`, :func:`kv_error_reset`, :func:`kv_status_str`.

The tensor-level functions take torch tensors (device memory and streams come
from PyTorch) and pass their data pointers and byte strides; the ``raw``
functions take plain integers exactly as the C ABI does. There is no CPU
fallback: if the compiled library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import enum
import os
import threading
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libkvstore.so")

__all__ = [
    "KVStatus", "KVError", "kv_store", "kv_store_fp8", "kv_store_paged", "kv_store_fp8_ex",
    "kv_gather", "kv_gather_fp8", "kv_inv_scale", "kv_absmax_inv", "kv_error_poll",
    "kv_error_reset", "kv_status_str", "error_record", "load_library", "raw", "STRIDE_FIELDS",
    "fused_fp8_set_kv_buffer", "kv_store_fp8_dynamic_tensor", "DYNAMIC_TENSOR_WORK_BYTES",
]


class KVStatus(enum.IntEnum):
    OK = 0
    ERR_INVALID_ARG = 1
    ERR_UNSUPPORTED = 2
    ERR_CUDA = 3
    ERR_INDEX_OOB = 4


class KVError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = KVStatus(status)
        super().__init__(f"{what}: {kv_status_str(status)}")


STRIDE_FIELDS = ("k_token", "k_head", "k_dim", "v_token", "v_head", "v_dim",
                 "kc_slot", "kc_head", "kc_dim", "vc_slot", "vc_head", "vc_dim")


class _Strides(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int64) for f in STRIDE_FIELDS]


_lock = threading.Lock()
_lib = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load ``libkvstore.so`` (built by ``fp8_quant_gb300.build``); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"CUDA library {p} is missing: build it with `python -m fp8_quant_gb300.build` "
                "(there is no CPU fallback)")
        lib = ctypes.CDLL(p)
        P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.kv_store.argtypes = [P, P, P, P, P, I32, I64, I64, I32, I32, I32,
                                 ctypes.POINTER(_Strides), I64, I32, P, P]
        lib.kv_store.restype = I32
        lib.kv_store_fp8.argtypes = [P, P, P, P, P, I32, I64, I64, I32, I32, I32,
                                     ctypes.POINTER(_Strides), I64, I64, I64, I64, P, P, I32, P, P]
        lib.kv_store_fp8.restype = I32
        lib.kv_store_paged.argtypes = [P, P, P, P, P, I32, I64, I64, I32, I32, I32,
                                       ctypes.POINTER(_Strides), I64, I64, I64, I64, I32, P, P]
        lib.kv_store_paged.restype = I32
        lib.kv_gather.argtypes = [P, P, P, P, P, I32, I64, I64, I32, I32, I32,
                                  ctypes.POINTER(_Strides), I64, P, P]
        lib.kv_gather.restype = I32
        lib.kv_gather_paged.argtypes = [P, P, P, P, P, I32, I64, I64, I32, I32, I32,
                                        ctypes.POINTER(_Strides), I64, I64, I64, I64, P, P]
        lib.kv_gather_paged.restype = I32
        lib.kv_gather_fp8.argtypes = [P, P, P, P, P, I32, I64, I64, I32, I32, I32,
                                      ctypes.POINTER(_Strides), I64, I64, I64, I64, P, P, I32, P,
                                      P]
        lib.kv_gather_fp8.restype = I32
        lib.kv_store_fp8_ex.argtypes = [P, P, P, P, P, I32, I64, I64, I32, I32, I32,
                                        ctypes.POINTER(_Strides), I64, I64, I64, I64, I32, I32,
                                        P, P, P, P, I64, P, P]
        lib.kv_store_fp8_ex.restype = I32
        lib.kv_gather_fp8_ex.argtypes = [P, P, P, P, P, I32, I64, I64, I32, I32, I32,
                                         ctypes.POINTER(_Strides), I64, I64, I64, I64, I32, I32,
                                         P, P, P, P, I64, P, P]
        lib.kv_gather_fp8_ex.restype = I32
        lib.kv_inv_scale.argtypes = [P, P, I64, P]
        lib.kv_inv_scale.restype = I32
        lib.kv_absmax_inv.argtypes = [P, P, I32, I64, I32, I32, ctypes.POINTER(_Strides),
                                      ctypes.c_float, P, P, P, P]
        lib.kv_absmax_inv.restype = I32
        lib.kv_store_fp8_dynamic_tensor.argtypes = [P, P, P, P, P, I32, I64, I64, I32, I32, I32,
                                                    ctypes.POINTER(_Strides), I64, I64, I64, I64,
                                                    I32, P, P, P, P, P]
        lib.kv_store_fp8_dynamic_tensor.restype = I32
        lib.kv_store_noalloc.argtypes = [P, P, P, P, P, I32, I64, I64, I32, I32, I32,
                                         ctypes.POINTER(_Strides), I64, I32,
                                         ctypes.POINTER(I64), ctypes.POINTER(I64), P]
        lib.kv_store_noalloc.restype = I32
        lib.kv_error_poll.argtypes = [P, P, ctypes.POINTER(I64), ctypes.POINTER(I64)]
        lib.kv_error_poll.restype = I32
        lib.kv_error_snapshot.argtypes = [P, P, P]
        lib.kv_error_snapshot.restype = I32
        lib.kv_launch_floor.argtypes = [I64, P]
        lib.kv_launch_floor.restype = I32
        lib.kv_error_reset.argtypes = [P, P]
        lib.kv_error_reset.restype = I32
        lib.kv_status_str.argtypes = [I32]
        lib.kv_status_str.restype = ctypes.c_char_p
        lib.kv_last_cuda_error.argtypes = []
        lib.kv_last_cuda_error.restype = ctypes.c_int
        lib.kv_abi_version.argtypes = []
        lib.kv_abi_version.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def kv_status_str(status: int) -> str:
    return load_library().kv_status_str(int(status)).decode()


# ---------------------------------------------------------------------------
# Raw entry points: integers in, status out (the C ABI one to one).
# ---------------------------------------------------------------------------

class raw:
    """The C ABI with plain integers (device addresses, byte strides, stream handle)."""

    @staticmethod
    def kv_store(k, v, k_cache, v_cache, indices, index_dtype, index_stride, num_tokens,
                 num_heads, head_dim, elem_bytes, strides: Sequence[int], size_limit,
                 num_split, d_err, stream) -> int:
        st = _Strides(*[int(x) for x in strides])
        return load_library().kv_store(k, v, k_cache, v_cache, indices, index_dtype,
                                       index_stride, num_tokens, num_heads, head_dim,
                                       elem_bytes, ctypes.byref(st), size_limit, num_split,
                                       d_err, stream)

    @staticmethod
    def kv_store_fp8(k, v, k_cache, v_cache, indices, index_dtype, index_stride, num_tokens,
                     num_heads, head_dim, src_dtype, strides: Sequence[int], page_size,
                     kc_page_stride, vc_page_stride, size_limit, inv_k_scale, inv_v_scale,
                     use_scale, d_err, stream) -> int:
        st = _Strides(*[int(x) for x in strides])
        return load_library().kv_store_fp8(k, v, k_cache, v_cache, indices, index_dtype,
                                           index_stride, num_tokens, num_heads, head_dim,
                                           src_dtype, ctypes.byref(st), page_size,
                                           kc_page_stride, vc_page_stride, size_limit,
                                           inv_k_scale, inv_v_scale, use_scale, d_err, stream)

    @staticmethod
    def kv_store_paged(k, v, k_cache, v_cache, indices, index_dtype, index_stride, num_tokens,
                       num_heads, head_dim, elem_bytes, strides: Sequence[int], page_size,
                       kc_page_stride, vc_page_stride, size_limit, num_split, d_err,
                       stream) -> int:
        st = _Strides(*[int(x) for x in strides])
        return load_library().kv_store_paged(k, v, k_cache, v_cache, indices, index_dtype,
                                             index_stride, num_tokens, num_heads, head_dim,
                                             elem_bytes, ctypes.byref(st), page_size,
                                             kc_page_stride, vc_page_stride, size_limit,
                                             num_split, d_err, stream)

    @staticmethod
    def kv_gather(k_cache, v_cache, k_out, v_out, indices, index_dtype, index_stride, num_tokens,
                  num_heads, head_dim, elem_bytes, strides: Sequence[int], size_limit, d_err,
                  stream) -> int:
        st = _Strides(*[int(x) for x in strides])
        return load_library().kv_gather(k_cache, v_cache, k_out, v_out, indices, index_dtype,
                                        index_stride, num_tokens, num_heads, head_dim, elem_bytes,
                                        ctypes.byref(st), size_limit, d_err, stream)

    @staticmethod
    def kv_gather_paged(k_cache, v_cache, k_out, v_out, indices, index_dtype, index_stride,
                        num_tokens, num_heads, head_dim, elem_bytes, strides: Sequence[int],
                        page_size, kc_page_stride, vc_page_stride, size_limit, d_err,
                        stream) -> int:
        st = _Strides(*[int(x) for x in strides])
        return load_library().kv_gather_paged(k_cache, v_cache, k_out, v_out, indices,
                                              index_dtype, index_stride, num_tokens, num_heads,
                                              head_dim, elem_bytes, ctypes.byref(st), page_size,
                                              kc_page_stride, vc_page_stride, size_limit, d_err,
                                              stream)

    @staticmethod
    def kv_gather_fp8(k_cache, v_cache, k_out, v_out, indices, index_dtype, index_stride,
                      num_tokens, num_heads, head_dim, out_dtype, strides: Sequence[int],
                      page_size, kc_page_stride, vc_page_stride, size_limit, k_scale, v_scale,
                      use_scale, d_err, stream) -> int:
        st = _Strides(*[int(x) for x in strides])
        return load_library().kv_gather_fp8(k_cache, v_cache, k_out, v_out, indices, index_dtype,
                                            index_stride, num_tokens, num_heads, head_dim,
                                            out_dtype, ctypes.byref(st), page_size,
                                            kc_page_stride, vc_page_stride, size_limit, k_scale,
                                            v_scale, use_scale, d_err, stream)

    @staticmethod
    def kv_store_fp8_ex(k, v, k_cache, v_cache, indices, index_dtype, index_stride, num_tokens,
                        num_heads, head_dim, src_dtype, strides: Sequence[int], page_size,
                        kc_page_stride, vc_page_stride, size_limit, fmt, scale_mode, inv_k_scale,
                        inv_v_scale, k_scales, v_scales, scales_slot_stride, d_err,
                        stream) -> int:
        st = _Strides(*[int(x) for x in strides])
        return load_library().kv_store_fp8_ex(k, v, k_cache, v_cache, indices, index_dtype,
                                              index_stride, num_tokens, num_heads, head_dim,
                                              src_dtype, ctypes.byref(st), page_size,
                                              kc_page_stride, vc_page_stride, size_limit, fmt,
                                              scale_mode, inv_k_scale, inv_v_scale, k_scales,
                                              v_scales, scales_slot_stride, d_err, stream)

    @staticmethod
    def kv_store_fp8_dynamic_tensor(k, v, k_cache, v_cache, indices, index_dtype, index_stride,
                                    num_tokens, num_heads, head_dim, src_dtype,
                                    strides: Sequence[int], page_size, kc_page_stride,
                                    vc_page_stride, size_limit, fmt, k_scale, v_scale, work,
                                    d_err, stream) -> int:
        st = _Strides(*[int(x) for x in strides])
        return load_library().kv_store_fp8_dynamic_tensor(
            k, v, k_cache, v_cache, indices, index_dtype, index_stride, num_tokens, num_heads,
            head_dim, src_dtype, ctypes.byref(st), page_size, kc_page_stride, vc_page_stride,
            size_limit, fmt, k_scale, v_scale, work, d_err, stream)

    @staticmethod
    def kv_gather_fp8_ex(k_cache, v_cache, k_out, v_out, indices, index_dtype, index_stride,
                         num_tokens, num_heads, head_dim, out_dtype, strides: Sequence[int],
                         page_size, kc_page_stride, vc_page_stride, size_limit, fmt, scale_mode,
                         k_scale, v_scale, k_scales, v_scales, scales_slot_stride, d_err,
                         stream) -> int:
        st = _Strides(*[int(x) for x in strides])
        return load_library().kv_gather_fp8_ex(k_cache, v_cache, k_out, v_out, indices,
                                               index_dtype, index_stride, num_tokens, num_heads,
                                               head_dim, out_dtype, ctypes.byref(st), page_size,
                                               kc_page_stride, vc_page_stride, size_limit, fmt,
                                               scale_mode, k_scale, v_scale, k_scales, v_scales,
                                               scales_slot_stride, d_err, stream)

    @staticmethod
    def kv_inv_scale(scale, inv, n, stream) -> int:
        return load_library().kv_inv_scale(scale, inv, n, stream)

    @staticmethod
    def kv_absmax_inv(k, v, src_dtype, num_tokens, num_heads, head_dim, strides: Sequence[int],
                      fp8_max, amax, inv, work, stream) -> int:
        st = _Strides(*[int(x) for x in strides])
        return load_library().kv_absmax_inv(k, v, src_dtype, num_tokens, num_heads, head_dim,
                                            ctypes.byref(st), float(fp8_max), amax, inv, work,
                                            stream)

    @staticmethod
    def kv_store_noalloc(k, v, k_cache, v_cache, indices, index_dtype, index_stride,
                         num_tokens, num_heads, head_dim, elem_bytes, strides: Sequence[int],
                         size_limit, num_split, stream):
        """kv_store without a caller-supplied error record (nothing is
        allocated; the record is a static array of the library). Blocks until
        the write is done; returns (status, oob_count, first_bad_token)."""
        st = _Strides(*[int(x) for x in strides])
        n = ctypes.c_int64(0)
        first = ctypes.c_int64(0)
        rc = load_library().kv_store_noalloc(k, v, k_cache, v_cache, indices, index_dtype,
                                             index_stride, num_tokens, num_heads, head_dim,
                                             elem_bytes, ctypes.byref(st), size_limit, num_split,
                                             ctypes.byref(n), ctypes.byref(first), stream)
        return rc, n.value, first.value

    @staticmethod
    def kv_error_poll(d_err, stream):
        n = ctypes.c_int64(0)
        first = ctypes.c_int64(0)
        rc = load_library().kv_error_poll(d_err, stream, ctypes.byref(n), ctypes.byref(first))
        return rc, n.value, first.value

    @staticmethod
    def kv_error_snapshot(d_err, dst, stream) -> int:
        return load_library().kv_error_snapshot(d_err, dst, stream)

    @staticmethod
    def kv_error_reset(d_err, stream) -> int:
        return load_library().kv_error_reset(d_err, stream)

    @staticmethod
    def kv_launch_floor(num_warps, stream) -> int:
        return load_library().kv_launch_floor(num_warps, stream)


# ---------------------------------------------------------------------------
# Tensor-level entry points
# ---------------------------------------------------------------------------

_default_records = {}


def error_record(device=None):
    """A zeroed device error record (two int64) owned by the caller."""
    import torch
    return torch.zeros(2, dtype=torch.int64, device=device or "cuda")


def _default_record(device):
    import torch
    dev = torch.device(device)
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    rec = _default_records.get(key)
    if rec is None:
        rec = _default_records[key] = error_record(torch.device("cuda", key))
    return rec


def _stream_handle(stream, device) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _rows3(x, H, D):
    """(token, head, dim) byte strides of a [T, H, D] or [T, H*D] tensor."""
    e = x.element_size()
    if x.dim() == 3:
        if tuple(x.shape[1:]) != (H, D):
            raise ValueError(f"row shape {tuple(x.shape)} != [T, {H}, {D}]")
        return x.stride(0) * e, x.stride(1) * e, x.stride(2) * e
    if x.dim() == 2:
        if x.shape[1] != H * D:
            raise ValueError(f"row width {x.shape[1]} != {H}*{D}")
        return x.stride(0) * e, D * x.stride(1) * e, x.stride(1) * e
    raise ValueError("rows must be 2-D or 3-D")


def _cache_shape(cache, num_heads=None, head_dim=None):
    """(slots, H, D) of a [slots, H, D] / [slots, H*D] / [pages, ps, H, D] cache."""
    if cache.dim() == 4:
        return cache.shape[0] * cache.shape[1], cache.shape[2], cache.shape[3]
    if cache.dim() == 3:
        return cache.shape[0], cache.shape[1], cache.shape[2]
    if cache.dim() == 2 and num_heads and head_dim:
        return cache.shape[0], num_heads, head_dim
    raise ValueError("cache must be [slots, H, D], [pages, page_size, H, D], or 2-D with "
                     "num_heads/head_dim given")


def _index_args(indices):
    import torch
    if indices.dim() != 1:
        raise ValueError("indices must be 1-D")
    if indices.dtype == torch.int32:
        return 0, indices.stride(0)
    if indices.dtype == torch.int64:
        return 1, indices.stride(0)
    raise TypeError("indices must be int32 or int64")


def _check(rc: int, what: str):
    if rc != KVStatus.OK:
        raise KVError(rc, what)


def kv_store(k, v, k_cache, v_cache, indices, *, size_limit: Optional[int] = None,
             num_split: int = 0, err=None, stream=None, num_heads: Optional[int] = None,
             head_dim: Optional[int] = None) -> None:
    """Plain copy of each token's K/V row into cache row ``indices[t]``.

    ``k``/``v``: [T, H, D] or [T, H*D] (any strides, any dtype); caches:
    [slots, H, D] or [slots, H*D] of the same element size. ``size_limit``
    defaults to the number of cache rows. Out-of-range slots are skipped and
    counted in ``err`` (a per-device default record if None); see
    :func:`kv_error_poll`.
    """
    slots, H, D = _cache_shape(k_cache, num_heads, head_dim)
    if k_cache.dim() == 4:
        raise ValueError("kv_store takes [slots, H, D] caches; use kv_store_fp8 for pages")
    e = k.element_size()
    if v.element_size() != e or k_cache.element_size() != e or v_cache.element_size() != e:
        raise TypeError("K, V and the caches must have the same element size")
    kt, kh, kd = _rows3(k, H, D)
    vt, vh, vd = _rows3(v, H, D)
    ks, khc, kdc = _rows3(k_cache, H, D)
    vs, vhc, vdc = _rows3(v_cache, H, D)
    idt, istride = _index_args(indices)
    T = indices.shape[0]
    if k.shape[0] < T or v.shape[0] < T:
        raise ValueError("fewer K/V rows than indices")
    rec = err if err is not None else _default_record(k.device)
    rc = raw.kv_store(k.data_ptr(), v.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                      indices.data_ptr(), idt, istride, T, H, D, e,
                      (kt, kh, kd, vt, vh, vd, ks, khc, kdc, vs, vhc, vdc),
                      slots if size_limit is None else size_limit, num_split, rec.data_ptr(),
                      _stream_handle(stream, k.device))
    _check(rc, "kv_store")


def kv_store_fp8(k, v, k_cache, v_cache, indices, *, page_size: int = 1,
                 inv_k_scale=None, inv_v_scale=None, size_limit: Optional[int] = None,
                 err=None, stream=None, num_heads: Optional[int] = None,
                 head_dim: Optional[int] = None) -> None:
    """Fused scale + e4m3fn conversion + paged write.

    ``k``/``v``: bf16 or fp16 [T, H, D] or [T, H*D]. Caches: uint8 /
    float8_e4m3fn, [slots, H, D] (3-D) or [pages, page_size, H, D] (4-D).
    ``inv_k_scale``/``inv_v_scale``: fp32 device scalars (0-D or 1-element
    tensors); the scale is used only when both are given.
    """
    import torch
    slots, H, D = _cache_shape(k_cache, num_heads, head_dim)
    if k.dtype not in (torch.bfloat16, torch.float16) or v.dtype != k.dtype:
        raise TypeError("K and V must both be bf16 or both fp16")
    if k_cache.element_size() != 1 or v_cache.element_size() != 1:
        raise TypeError("FP8 caches have 1-byte elements")
    kt, kh, kd = _rows3(k, H, D)
    vt, vh, vd = _rows3(v, H, D)
    if k_cache.dim() == 4:
        if k_cache.shape[1] != page_size or v_cache.shape[1] != page_size:
            raise ValueError("page_size does not match the cache")
        kp, ks, khc, kdc = k_cache.stride()
        vp, vs, vhc, vdc = v_cache.stride()
    else:
        ks, khc, kdc = _rows3(k_cache, H, D)
        vs, vhc, vdc = _rows3(v_cache, H, D)
        kp, vp = ks * page_size, vs * page_size
    idt, istride = _index_args(indices)
    T = indices.shape[0]
    if k.shape[0] < T or v.shape[0] < T:
        raise ValueError("fewer K/V rows than indices")
    use_scale = int(inv_k_scale is not None and inv_v_scale is not None)
    for s in (inv_k_scale, inv_v_scale) if use_scale else ():
        if s.dtype != torch.float32 or s.numel() != 1 or s.device.type != "cuda":
            raise TypeError("inverse scales must be 1-element fp32 device tensors")
    rec = err if err is not None else _default_record(k.device)
    rc = raw.kv_store_fp8(
        k.data_ptr(), v.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), indices.data_ptr(),
        idt, istride, T, H, D, 1 if k.dtype == torch.bfloat16 else 0,
        (kt, kh, kd, vt, vh, vd, ks, khc, kdc, vs, vhc, vdc), page_size, kp, vp,
        slots if size_limit is None else size_limit,
        inv_k_scale.data_ptr() if use_scale else None,
        inv_v_scale.data_ptr() if use_scale else None, use_scale, rec.data_ptr(),
        _stream_handle(stream, k.device))
    _check(rc, "kv_store_fp8")


def kv_error_poll(err=None, stream=None, device=None):
    """Synchronise, read and clear an error record: (status, oob_count, first_bad_token)."""
    import torch
    if err is None:
        err = _default_record(device or torch.device("cuda", torch.cuda.current_device()))
    rc, n, first = raw.kv_error_poll(err.data_ptr(), _stream_handle(stream, err.device))
    if rc not in (KVStatus.OK, KVStatus.ERR_INDEX_OOB):
        raise KVError(rc, "kv_error_poll")
    return KVStatus(rc), n, first


def kv_error_reset(err=None, stream=None, device=None) -> None:
    import torch
    if err is None:
        err = _default_record(device or torch.device("cuda", torch.cuda.current_device()))
    _check(raw.kv_error_reset(err.data_ptr(), _stream_handle(stream, err.device)),
           "kv_error_reset")


# ---------------------------------------------------------------------------
# Tensor-level wrappers of the other entry points
# ---------------------------------------------------------------------------

FP8_FORMATS = {"e4m3fn": 0, "e5m2": 1}
SCALE_MODES = {"none": 0, "tensor": 1, "token": 2, "token_head": 3, "page": 4}


def _paged_cache(cache, page_size, H, D):
    """(slot, head, dim, page) byte strides of a [slots, H, D] or [pages, ps, H, D] cache."""
    if cache.dim() == 4:
        if cache.shape[1] != page_size:
            raise ValueError("page_size does not match the cache")
        e = cache.element_size()
        sp, ss, sh, sd = (x * e for x in cache.stride())
        return ss, sh, sd, sp
    ss, sh, sd = _rows3(cache, H, D)
    return ss, sh, sd, ss * page_size


def _device_ptr_or_none(t):
    return None if t is None else t.data_ptr()


def kv_store_paged(k, v, k_cache, v_cache, indices, *, page_size: int, size_limit=None,
                   num_split: int = 0, err=None, stream=None) -> None:
    """Plain copy into [pages, page_size, H, D] caches (any page stride)."""
    slots, H, D = _cache_shape(k_cache)
    e = k.element_size()
    kt, kh, kd = _rows3(k, H, D)
    vt, vh, vd = _rows3(v, H, D)
    ks, khc, kdc, kp = _paged_cache(k_cache, page_size, H, D)
    vs, vhc, vdc, vp = _paged_cache(v_cache, page_size, H, D)
    idt, istride = _index_args(indices)
    rec = err if err is not None else _default_record(k.device)
    _check(raw.kv_store_paged(k.data_ptr(), v.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                              indices.data_ptr(), idt, istride, indices.shape[0], H, D, e,
                              (kt, kh, kd, vt, vh, vd, ks, khc, kdc, vs, vhc, vdc), page_size, kp,
                              vp, slots if size_limit is None else size_limit, num_split,
                              rec.data_ptr(), _stream_handle(stream, k.device)), "kv_store_paged")


def kv_store_fp8_ex(k, v, k_cache, v_cache, indices, *, page_size: int = 1,
                    fmt: str = "e4m3fn", scale_mode: str = "none", inv_k_scale=None,
                    inv_v_scale=None, k_scales=None, v_scales=None, size_limit=None, err=None,
                    stream=None) -> None:
    """FP8 write in e4m3fn / e5m2 with no, per-tensor, per-token or per-(token, head)
    scales. Dynamic modes write the dequantisation scale of slot s (head h) to
    k_scales[s, h] / v_scales[s, h] (fp32 device tensors [slots, >= groups])."""
    slots, H, D = _cache_shape(k_cache)
    kt, kh, kd = _rows3(k, H, D)
    vt, vh, vd = _rows3(v, H, D)
    ks, khc, kdc, kp = _paged_cache(k_cache, page_size, H, D)
    vs, vhc, vdc, vp = _paged_cache(v_cache, page_size, H, D)
    idt, istride = _index_args(indices)
    sstride = 0
    if k_scales is not None:
        if k_scales.dim() != 2 or k_scales.stride(1) != 1 or v_scales.stride() != k_scales.stride():
            raise ValueError("scale caches must be [slots, groups] with unit inner stride")
        sstride = k_scales.stride(0)
    rec = err if err is not None else _default_record(k.device)
    import torch
    _check(raw.kv_store_fp8_ex(
        k.data_ptr(), v.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), indices.data_ptr(),
        idt, istride, indices.shape[0], H, D, 1 if k.dtype == torch.bfloat16 else 0,
        (kt, kh, kd, vt, vh, vd, ks, khc, kdc, vs, vhc, vdc), page_size, kp, vp,
        slots if size_limit is None else size_limit, FP8_FORMATS[fmt], SCALE_MODES[scale_mode],
        _device_ptr_or_none(inv_k_scale), _device_ptr_or_none(inv_v_scale),
        _device_ptr_or_none(k_scales), _device_ptr_or_none(v_scales), sstride, rec.data_ptr(),
        _stream_handle(stream, k.device)), "kv_store_fp8_ex")


DYNAMIC_TENSOR_WORK_BYTES = 24  # KV_DYNAMIC_TENSOR_WORK_BYTES of the C header


def kv_store_fp8_dynamic_tensor(k, v, k_cache, v_cache, indices, *, page_size: int = 1,
                                fmt: str = "e4m3fn", scales=None, work=None, size_limit=None,
                                err=None, stream=None):
    """FP8 write with per-tensor scales formed from the batch, in one call:
    amax over all K (V) rows, inv = fmax / amax, codes fp8(x * inv).  Returns
    ``scales``: a 2-element fp32 device tensor receiving the forward scales
    amax / fmax (K, V).  ``work``: a device tensor of at least
    DYNAMIC_TENSOR_WORK_BYTES bytes, zero before its first use and reused
    across calls on one stream (a fresh zeroed one when None)."""
    import torch
    slots, H, D = _cache_shape(k_cache)
    kt, kh, kd = _rows3(k, H, D)
    vt, vh, vd = _rows3(v, H, D)
    ks, khc, kdc, kp = _paged_cache(k_cache, page_size, H, D)
    vs, vhc, vdc, vp = _paged_cache(v_cache, page_size, H, D)
    idt, istride = _index_args(indices)
    if k.dtype not in (torch.bfloat16, torch.float16) or v.dtype != k.dtype:
        raise TypeError("K and V must both be bf16 or both fp16")
    if scales is None:
        scales = torch.empty(2, dtype=torch.float32, device=k.device)
    if scales.dtype != torch.float32 or scales.numel() < 2 or not scales.is_contiguous():
        raise TypeError("scales must be a contiguous fp32 tensor of 2 elements")
    if work is None:
        work = torch.zeros(DYNAMIC_TENSOR_WORK_BYTES // 8, dtype=torch.int64, device=k.device)
    if work.numel() * work.element_size() < DYNAMIC_TENSOR_WORK_BYTES:
        raise ValueError(f"work holds fewer than {DYNAMIC_TENSOR_WORK_BYTES} bytes")
    rec = err if err is not None else _default_record(k.device)
    _check(raw.kv_store_fp8_dynamic_tensor(
        k.data_ptr(), v.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), indices.data_ptr(),
        idt, istride, indices.shape[0], H, D, 1 if k.dtype == torch.bfloat16 else 0,
        (kt, kh, kd, vt, vh, vd, ks, khc, kdc, vs, vhc, vdc), page_size, kp, vp,
        slots if size_limit is None else size_limit, FP8_FORMATS[fmt], scales.data_ptr(),
        scales.data_ptr() + 4, work.data_ptr(), rec.data_ptr(), _stream_handle(stream, k.device)),
        "kv_store_fp8_dynamic_tensor")
    return scales


def kv_gather(k_cache, v_cache, k_out, v_out, indices, *, page_size: int = 1, size_limit=None,
              err=None, stream=None) -> None:
    """Row t of k_out / v_out takes the cache row of indices[t] (byte copy)."""
    slots, H, D = _cache_shape(k_cache)
    e = k_out.element_size()
    kt, kh, kd = _rows3(k_out, H, D)
    vt, vh, vd = _rows3(v_out, H, D)
    ks, khc, kdc, kp = _paged_cache(k_cache, page_size, H, D)
    vs, vhc, vdc, vp = _paged_cache(v_cache, page_size, H, D)
    idt, istride = _index_args(indices)
    rec = err if err is not None else _default_record(k_cache.device)
    _check(raw.kv_gather_paged(k_cache.data_ptr(), v_cache.data_ptr(), k_out.data_ptr(),
                               v_out.data_ptr(), indices.data_ptr(), idt, istride,
                               indices.shape[0], H, D, e,
                               (kt, kh, kd, vt, vh, vd, ks, khc, kdc, vs, vhc, vdc), page_size,
                               kp, vp, slots if size_limit is None else size_limit,
                               rec.data_ptr(), _stream_handle(stream, k_cache.device)),
           "kv_gather")


def kv_gather_fp8(k_cache, v_cache, k_out, v_out, indices, *, page_size: int = 1,
                  fmt: str = "e4m3fn", scale_mode: str = "none", k_scale=None, v_scale=None,
                  k_scales=None, v_scales=None, size_limit=None, err=None, stream=None) -> None:
    """Dequantising gather into bf16 / fp16 rows (the dtype of k_out)."""
    import torch
    slots, H, D = _cache_shape(k_cache)
    kt, kh, kd = _rows3(k_out, H, D)
    vt, vh, vd = _rows3(v_out, H, D)
    ks, khc, kdc, kp = _paged_cache(k_cache, page_size, H, D)
    vs, vhc, vdc, vp = _paged_cache(v_cache, page_size, H, D)
    idt, istride = _index_args(indices)
    sstride = k_scales.stride(0) if k_scales is not None else 0
    rec = err if err is not None else _default_record(k_cache.device)
    _check(raw.kv_gather_fp8_ex(
        k_cache.data_ptr(), v_cache.data_ptr(), k_out.data_ptr(), v_out.data_ptr(),
        indices.data_ptr(), idt, istride, indices.shape[0], H, D,
        1 if k_out.dtype == torch.bfloat16 else 0,
        (kt, kh, kd, vt, vh, vd, ks, khc, kdc, vs, vhc, vdc), page_size, kp, vp,
        slots if size_limit is None else size_limit, FP8_FORMATS[fmt], SCALE_MODES[scale_mode],
        _device_ptr_or_none(k_scale), _device_ptr_or_none(v_scale),
        _device_ptr_or_none(k_scales), _device_ptr_or_none(v_scales), sstride, rec.data_ptr(),
        _stream_handle(stream, k_cache.device)), "kv_gather_fp8")


def kv_inv_scale(scale, out=None, stream=None):
    """1 / scale in fp32 on the device; returns `out` (a new tensor if None)."""
    import torch
    if scale.dtype != torch.float32 or not scale.is_contiguous():
        raise TypeError("scale must be a contiguous fp32 tensor")
    out = torch.empty_like(scale) if out is None else out
    _check(raw.kv_inv_scale(scale.data_ptr(), out.data_ptr(), scale.numel(),
                            _stream_handle(stream, scale.device)), "kv_inv_scale")
    return out


def fused_fp8_set_kv_buffer(k, v, k_cache, v_cache, cache_loc, k_scale=None, v_scale=None,
                            page_size: int = 16, *, err=None, stream=None) -> None:
    """The fused FP8 write with the argument list of sglang trtllm_fp8_kv_kernel.py
    (`fused_fp8_set_kv_buffer`, its wrapper): K and V rows ([T, H, D] or
    [T, H*D], bf16 or fp16) go to slots ``cache_loc`` of e4m3fn caches,
    [slots, H, D] (``slots`` a multiple of ``page_size``) or
    [pages, page_size, H, D].  ``k_scale`` / ``v_scale`` are the forward
    (dequantisation) scales, Python floats or fp32 tensors, used only when both
    are given; as in that wrapper, ``1 / scale`` is formed on the device
    (``kv_inv_scale``), so tensor scales cost no host synchronisation.  The
    write itself is ``kv_store_fp8``; there is no second, unfused path.  The
    scale staging runs on ``stream`` (torch's current stream when None)."""
    import contextlib
    import torch
    if k_cache.dim() == 3 and k_cache.shape[0] % page_size:
        raise ValueError("cache slots must be a multiple of page_size")
    inv = None
    if k_scale is not None and v_scale is not None:
        ctx = (torch.cuda.stream(stream) if isinstance(stream, torch.cuda.Stream)
               else contextlib.nullcontext())
        if stream is not None and not isinstance(stream, torch.cuda.Stream):
            raise TypeError("with scales, stream must be a torch.cuda.Stream or None")
        with ctx:
            sc = torch.empty(2, dtype=torch.float32, device=k.device)
            for i, x in enumerate((k_scale, v_scale)):
                if isinstance(x, torch.Tensor):
                    if x.numel() != 1:
                        raise ValueError("a scale tensor holds one value")
                    sc[i:i + 1].copy_(x.reshape(1))
                else:
                    sc[i:i + 1].fill_(float(x))
            inv = kv_inv_scale(sc, stream=stream)
    kv_store_fp8(k, v, k_cache, v_cache, cache_loc, page_size=page_size,
                 inv_k_scale=None if inv is None else inv[0:1],
                 inv_v_scale=None if inv is None else inv[1:2], err=err, stream=stream)


def kv_absmax_inv(k, v, *, fp8_max: float = 448.0, num_heads=None, head_dim=None, out=None,
                  work=None, stream=None):
    """Per-tensor max |K|, max |V| and fp8_max / amax on the device: returns a
    4-float tensor [amax_k, amax_v, inv_k, inv_v]. ``work``: an optional
    device workspace of at least 8 bytes, zero before first use, kept zero by
    the calls (two kernels per call instead of three)."""
    import torch
    if k.dim() == 3:
        H, D = k.shape[1], k.shape[2]
    else:
        H, D = num_heads, head_dim
    kt, kh, kd = _rows3(k, H, D)
    vt, vh, vd = _rows3(v, H, D)
    out = torch.empty(4, dtype=torch.float32, device=k.device) if out is None else out
    _check(raw.kv_absmax_inv(k.data_ptr(), v.data_ptr(), 1 if k.dtype == torch.bfloat16 else 0,
                             k.shape[0], H, D, (kt, kh, kd, vt, vh, vd, 0, 0, 0, 0, 0, 0), fp8_max,
                             out.data_ptr(), out.data_ptr() + 8,
                             None if work is None else work.data_ptr(),
                             _stream_handle(stream, k.device)),
           "kv_absmax_inv")
    return out
