"""Seeded synthetic inputs for the KV-cache write path.

This module is shared by the tests, ``bench.py`` and the smoke check. It draws
the K/V rows, the slot indices and the cache pre-fill for every workload, and
nothing else: it holds none of the write path's arithmetic (no scatter, no
scaling, no FP8 encoding). Both the CUDA path and the CPU oracle receive exactly
the arrays built here.

Random numbers come from one counter-based generator, SplitMix64 (Steele, Lea
and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014): the
i-th draw of a stream with key ``seed`` is ``mix(seed + (i + 1) * golden)``.
Normals use the Box-Muller transform in float64, then float32, then
round-to-nearest-even to bf16 or fp16. Distinct slots are the ``k`` slots with
the smallest random keys, listed in random order.

Workloads (sizes of the KV-cache write configurations this library is
measured on; ``T`` tokens, ``H`` KV heads, ``D`` head dim):

* ``tiny``     T=16,    H=2, D=64,  bf16, cache 256 slots, int32 indices.
* ``decode``   T=256,   H=8, D=128, bf16, cache 1,048,576 slots, int64.
* ``prefill``  T=32768, H=8, D=128, bf16, cache 4,194,304 slots, page 64,
               512 whole pages in random page order, int32.
* ``fp8``      T=8192,  H=8, D=128, bf16 4*N(0,1) with 0.1% outliers
               +-U(500,2000), e4m3fn cache 1,048,576 slots, page 32, int64.
* ``strided``  fp16 K/V as column views of a fused QKV [65536, 6144] tensor,
               cache 2,097,152 slots, int32.
* ``odd``      fp16 H=1, D=576 (1152-byte rows), 1280-byte slot stride,
               cache 2,097,152 slots, int32.
* ``paged``    the prefill batch into 4-D pages [65536, 64, 8, 128] padded by
               one slot per page (page stride 133,120 B).
* ``fp8_dynamic`` the fp8 batch with per-(token, head) scales computed in the
               kernel and stored per slot (``fp8_dynamic_token``: one scale
               per token row).
* ``fp8_e5m2`` the fp8 batch into an e5m2 cache, per-tensor scales 57344/amax.
* ``fp8_page`` the fp8 batch with one inverse scale per 32-slot cache page.

The gather workloads read these caches back (``gather_decode``,
``gather_prefill``, ``gather_fp8``), and ``absmax`` reads the fp8 batch once.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

BF16_SENTINEL = 0x7FC0   # cache pre-fill for 2-byte caches (a bf16 NaN pattern)
FP8_SENTINEL = 0x7F      # cache pre-fill for e4m3fn caches (the e4m3fn NaN code)


def splitmix64(seed: int, start: int, n: int) -> np.ndarray:
    """Draws ``start .. start+n-1`` of the SplitMix64 stream keyed by ``seed``."""
    with np.errstate(over="ignore"):
        ctr = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + ctr * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def uniform01(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Float64 uniforms in [0, 1) with 53 random bits each."""
    return (splitmix64(seed, start, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, n: int, chunk: int = 1 << 24) -> np.ndarray:
    """``n`` standard normals (float32), Box-Muller on pairs of uniforms."""
    out = np.empty(n, dtype=np.float32)
    half = (n + 1) // 2
    for p0 in range(0, half, chunk):
        m = min(chunk, half - p0)
        u = uniform01(seed, 2 * m, start=2 * p0)
        u1 = 1.0 - u[0::2]            # (0, 1]: log is finite
        u2 = u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        a = 2.0 * math.pi * u2
        z = np.empty(2 * m, dtype=np.float64)
        z[0::2] = r * np.cos(a)
        z[1::2] = r * np.sin(a)
        lo = 2 * p0
        hi = min(n, lo + 2 * m)
        out[lo:hi] = z[: hi - lo]
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns the uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (b & 0x7FFFFFFF) > 0x7F800000
    r = (b + np.uint32(0x7FFF) + ((b >> 16) & 1)) >> 16
    r = np.where(nan, (b >> 16) | 0x40, r)
    return r.astype(np.uint16)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to fp16 (IEEE, nearest even); returns the uint16 bits."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    if dtype == "f16":
        return f32_to_f16_bits(x)
    raise ValueError(dtype)


def distinct_slots(seed: int, n_slots: int, k: int) -> np.ndarray:
    """``k`` distinct slots of ``[0, n_slots)``, in random order (int64)."""
    if k > n_slots:
        raise ValueError("more tokens than slots")
    keys = splitmix64(seed, 0, n_slots)
    pick = np.argpartition(keys, k - 1)[:k] if k < n_slots else np.arange(n_slots)
    order = np.argsort(splitmix64(seed ^ 0x5A5A5A5A, 0, k), kind="stable")
    return pick[order].astype(np.int64)


def page_run_slots(seed: int, n_pages: int, page_size: int, k_pages: int) -> np.ndarray:
    """Whole pages in random page order, each filled with offsets 0..page_size-1."""
    pages = distinct_slots(seed, n_pages, k_pages)
    return (pages[:, None] * page_size + np.arange(page_size)[None, :]).reshape(-1)


@dataclass
class Workload:
    """One synthetic write problem, host side.

    ``k``/``v`` are uint16 bit arrays of shape ``src_shape`` (the input tensors);
    ``k_view``/``v_view`` describe the K and V rows inside them as
    (byte offset, token stride, head stride, dim stride), all in bytes. The cache
    is ``n_slots`` slots of ``slot_stride`` bytes, each slot holding ``H`` heads of
    ``D`` elements (``cache_elem`` bytes each, head stride ``cache_head_stride``).
    """

    name: str
    T: int
    H: int
    D: int
    src_dtype: str                  # "bf16" | "f16"
    kind: str                       # "copy" | "fp8" | "fp8_dyn" | "gather" | "gather_fp8" | "absmax"
    k: np.ndarray
    v: np.ndarray
    k_view: tuple
    v_view: tuple
    indices: np.ndarray             # int32 or int64
    n_slots: int
    slot_stride: int
    cache_head_stride: int
    cache_elem: int                 # 2 (copy) or 1 (fp8)
    sentinel: int                   # pre-fill byte pattern (uint16 for copy, uint8 for fp8)
    page_size: int
    page_stride: int
    inv_k: float = 1.0              # fp32 inverse scales (fp8 only)
    inv_v: float = 1.0
    use_scale: int = 0
    num_split: int = 0
    notes: dict = field(default_factory=dict)

    @property
    def row_bytes(self) -> int:
        return self.H * self.D * 2

    @property
    def paged(self) -> bool:
        """Pages padded beyond page_size slots (the 4-D [pages, page_size, H, D] layout)."""
        return self.page_stride != self.page_size * self.slot_stride

    @property
    def cache_bytes(self) -> int:
        pages = -(-self.n_slots // self.page_size)
        return pages * self.page_stride if self.paged else self.n_slots * self.slot_stride

    def algorithmic_bytes(self) -> int:
        """Bytes a call must move: K and V rows read, cache rows written, indices read
        (for the absmax pass: K and V rows read, four floats written; for the
        dynamic FP8 write also one fp32 scale per token and head, K and V; for
        the fused per-tensor dynamic write the rows once and two scales)."""
        if self.kind == "absmax":
            return self.T * 2 * self.row_bytes + 16
        out_row = self.H * self.D * self.cache_elem
        groups = self.H if self.notes.get("scale_mode", "token_head") == "token_head" else 1
        scales = 2 * groups * 4 if self.kind == "fp8_dyn" else 0
        if self.notes.get("scale_mode") == "page":
            scales = 2 * 4          # the page's inverse scale, K and V
        if self.notes.get("scale_mode") == "tensor_dynamic":
            # K and V counted once (the scale pass's read; the write's second
            # read of the same rows is served from L2), plus the two scales
            return self.T * (2 * self.row_bytes + 2 * out_row + self.indices.itemsize) + 8
        return self.T * (2 * self.row_bytes + 2 * out_row + self.indices.itemsize + scales)


def _contig_view(H: int, D: int, elem: int = 2):
    return (0, H * D * elem, D * elem, elem)


def _normal_rows(seed: int, T: int, H: int, D: int, dtype: str, scale: float = 1.0) -> np.ndarray:
    x = normal(seed, T * H * D)
    if scale != 1.0:
        x *= np.float32(scale)
    return to_bits(x, dtype).reshape(T, H, D)


def _amax_inv(bits: np.ndarray, dtype: str, fmax: float = 448.0) -> float:
    """Per-tensor inverse scale fmax/amax in fp32 (the fp8 workload's input
    recipe; fmax is 448 for e4m3fn caches, 57344 for e5m2)."""
    if dtype == "bf16":
        vals = (bits.astype(np.uint32) << 16).view(np.float32)
    else:
        vals = bits.view(np.float16).astype(np.float32)
    amax = np.float32(np.max(np.abs(vals)))
    return float(np.float32(fmax) / amax)


def make_copy(name, T, H, D, n_slots, seed, dtype="bf16", index_dtype=np.int32,
              slot_stride=None, slots=None, page_size=16, num_split=0) -> Workload:
    """A contiguous-row plain-copy problem with distinct random slots."""
    k = _normal_rows(seed * 4 + 1, T, H, D, dtype)
    v = _normal_rows(seed * 4 + 2, T, H, D, dtype)
    if slots is None:
        slots = distinct_slots(seed * 4 + 3, n_slots, T)
    ss = slot_stride if slot_stride is not None else H * D * 2
    return Workload(name=name, T=T, H=H, D=D, src_dtype=dtype, kind="copy", k=k, v=v,
                    k_view=_contig_view(H, D), v_view=_contig_view(H, D),
                    indices=slots.astype(index_dtype), n_slots=n_slots, slot_stride=ss,
                    cache_head_stride=D * 2, cache_elem=2, sentinel=BF16_SENTINEL,
                    page_size=page_size, page_stride=page_size * ss, num_split=num_split)


def make_fp8(name, T, H, D, n_slots, seed, dtype="bf16", index_dtype=np.int64,
             page_size=32, use_scale=1, scale=4.0, outlier_frac=0.001,
             slot_stride=None, page_stride=None) -> Workload:
    """An FP8 problem: scale*N(0,1) with a fraction of +-U(500, 2000) outliers."""
    ks = []
    for j in (1, 2):
        x = normal(seed * 8 + j, T * H * D) * np.float32(scale)
        u = uniform01(seed * 8 + 2 + j, 3 * x.size)
        hit = u[0::3] < outlier_frac
        mag = 500.0 + 1500.0 * u[1::3]
        sgn = np.where(u[2::3] < 0.5, -1.0, 1.0)
        x = np.where(hit, (sgn * mag).astype(np.float32), x)
        ks.append(to_bits(x, dtype).reshape(T, H, D))
    k, v = ks
    slots = distinct_slots(seed * 8 + 5, n_slots, T)
    ss = slot_stride if slot_stride is not None else H * D
    ps = page_stride if page_stride is not None else page_size * ss
    w = Workload(name=name, T=T, H=H, D=D, src_dtype=dtype, kind="fp8", k=k, v=v,
                 k_view=_contig_view(H, D), v_view=_contig_view(H, D),
                 indices=slots.astype(index_dtype), n_slots=n_slots, slot_stride=ss,
                 cache_head_stride=D, cache_elem=1, sentinel=FP8_SENTINEL,
                 page_size=page_size, page_stride=ps, use_scale=use_scale)
    w.inv_k = _amax_inv(k, dtype)
    w.inv_v = _amax_inv(v, dtype)
    return w


# ``n_slots`` overrides the cache size (smaller caches for profiler captures;
# the slot draws then differ from the full-size workload's).

def tiny(n_slots: int = 256) -> Workload:
    return make_copy("tiny", T=16, H=2, D=64, n_slots=n_slots, seed=0x5EED0000, page_size=16)


def decode(num_split: int = 0, n_slots: int = 1 << 20) -> Workload:
    return make_copy("decode", T=256, H=8, D=128, n_slots=n_slots, seed=0x5EED0001,
                     index_dtype=np.int64, num_split=num_split)


def prefill(n_slots: int = 1 << 22) -> Workload:
    slots = page_run_slots(0x5EED0002 * 4 + 3, n_pages=n_slots // 64, page_size=64, k_pages=512)
    w = make_copy("prefill", T=32768, H=8, D=128, n_slots=n_slots, seed=0x5EED0002,
                  slots=slots, page_size=64)
    w.notes["whole_pages"] = True
    return w


def fp8(use_scale: int = 1, n_slots: int = 1 << 20) -> Workload:
    return make_fp8("fp8", T=8192, H=8, D=128, n_slots=n_slots, seed=0x5EED0003,
                    page_size=32, use_scale=use_scale)


def strided(n_slots: int = 1 << 21) -> Workload:
    """fp16 K and V as views into a fused QKV tensor [T, (32 + 2*8) * 128].

    Only the K and V columns are ever read; the Q columns are filled with a
    constant pattern so that generating them costs nothing.
    """
    T, H, D, HQ = 65536, 8, 128, 32
    width = (HQ + 2 * H) * D
    qkv = np.full((T, width), 0x3C00, dtype=np.uint16)   # fp16 1.0 in the Q columns
    qkv[:, HQ * D:(HQ + H) * D] = _normal_rows(0x5EED0004 * 4 + 1, T, H, D, "f16").reshape(T, H * D)
    qkv[:, (HQ + H) * D:] = _normal_rows(0x5EED0004 * 4 + 2, T, H, D, "f16").reshape(T, H * D)
    slots = distinct_slots(0x5EED0004 * 4 + 3, n_slots, T)
    tok = width * 2
    w = Workload(name="strided", T=T, H=H, D=D, src_dtype="f16", kind="copy", k=qkv, v=qkv,
                 k_view=(HQ * D * 2, tok, D * 2, 2), v_view=((HQ + H) * D * 2, tok, D * 2, 2),
                 indices=slots.astype(np.int32), n_slots=n_slots, slot_stride=H * D * 2,
                 cache_head_stride=D * 2, cache_elem=2, sentinel=BF16_SENTINEL,
                 page_size=16, page_stride=16 * H * D * 2)
    w.notes["shared_source"] = True
    return w


def paged(n_slots: int = 1 << 22) -> Workload:
    """The prefill batch into a 4-D cache [pages, 64, 8, 128] whose pages are
    padded by one slot (page stride 133,120 B): kv_store_paged."""
    w = prefill(n_slots=n_slots)
    w.name = "paged"
    w.page_stride = w.page_size * w.slot_stride + w.slot_stride
    w.notes["whole_pages"] = True
    return w


def fp8_dynamic(n_slots: int = 1 << 20) -> Workload:
    """The ``fp8`` batch written with scales computed in the kernel per
    (token, head): amax of each head's 128 elements, codes of x * (448/amax),
    and amax/448 stored per slot and head in an fp32 scale cache."""
    w = fp8(n_slots=n_slots)
    w.name, w.kind = "fp8_dynamic", "fp8_dyn"
    return w


def fp8_dynamic_token(n_slots: int = 1 << 20) -> Workload:
    """As ``fp8_dynamic`` with one scale per token row (amax over all 1024
    elements of the K or V row)."""
    w = fp8_dynamic(n_slots=n_slots)
    w.name = "fp8_dynamic_token"
    w.notes["scale_mode"] = "token"
    return w


def fp8_e5m2(n_slots: int = 1 << 20) -> Workload:
    """The ``fp8`` batch into an e5m2 cache with per-tensor inverse scales
    57344/amax (kv_store_fp8_ex)."""
    w = fp8(n_slots=n_slots)
    w.name = "fp8_e5m2"
    w.notes["fmt"] = "e5m2"
    w.inv_k = _amax_inv(w.k, w.src_dtype, 57344.0)
    w.inv_v = _amax_inv(w.v, w.src_dtype, 57344.0)
    return w


def fp8_page(n_slots: int = 1 << 20) -> Workload:
    """The ``fp8`` batch written with one inverse scale per 32-slot cache page
    (scale mode "page"): page p of the K cache has inv_k * 2**e_p with e_p
    drawn from {-3, -2, -1, 0} (likewise V), so every page's scale keeps the
    batch's values within the e4m3fn range except the saturating outliers."""
    w = fp8(n_slots=n_slots)
    w.name = "fp8_page"
    w.notes["scale_mode"] = "page"
    n_pages = -(-n_slots // w.page_size)
    for j, inv in ((0, w.inv_k), (1, w.inv_v)):
        e = np.floor(uniform01(0x5EED0006 + j, n_pages) * 4) - 3
        w.notes["page_inv_" + "kv"[j]] = (np.float32(inv) * (2.0 ** e)).astype(np.float32)
    return w


def odd(n_slots: int = 1 << 21) -> Workload:
    """fp16 H=1, D=576 rows (1152 B) into 1280-byte slots."""
    return make_copy("odd", T=65536, H=1, D=576, n_slots=n_slots, seed=0x5EED0005,
                     dtype="f16", slot_stride=1280)


def gather_decode(n_slots: int = 1 << 20) -> Workload:
    """Inverse of ``decode``: 256 rows gathered from a 1,048,576-slot bf16 cache."""
    w = decode(n_slots=n_slots)
    w.name, w.kind = "gather_decode", "gather"
    return w


def gather_prefill(n_slots: int = 1 << 22) -> Workload:
    """Inverse of ``prefill``: 32768 rows (512 whole pages) gathered from a
    4,194,304-slot bf16 cache."""
    w = prefill(n_slots=n_slots)
    w.name, w.kind = "gather_prefill", "gather"
    return w


def gather_fp8(n_slots: int = 1 << 20) -> Workload:
    """Inverse of ``fp8``: 8192 e4m3fn rows dequantised (x 1/inv) to bf16."""
    w = fp8(n_slots=n_slots)
    w.name, w.kind = "gather_fp8", "gather_fp8"
    return w


def fp8_tensor_dynamic(n_slots: int = 1 << 20) -> Workload:
    """The ``fp8`` batch written with per-tensor scales formed from the batch
    in the same call (amax over K and over V, inv = 448 / amax, then the
    write): the fused dynamic per-tensor write."""
    w = fp8(n_slots=n_slots)
    w.name = "fp8_tensor_dynamic"
    w.notes["scale_mode"] = "tensor_dynamic"
    return w


def absmax(n_slots: int = 1 << 20) -> Workload:
    """Per-tensor scale pass over the ``fp8`` batch (K and V read once)."""
    w = fp8(n_slots=n_slots)
    w.name, w.kind = "absmax", "absmax"
    return w


WORKLOADS = {
    "tiny": tiny,
    "decode": decode,
    "prefill": prefill,
    "fp8": fp8,
    "strided": strided,
    "odd": odd,
    "paged": paged,
    "fp8_dynamic": fp8_dynamic,
    "fp8_dynamic_token": fp8_dynamic_token,
    "fp8_e5m2": fp8_e5m2,
    "fp8_page": fp8_page,
    "gather_decode": gather_decode,
    "gather_prefill": gather_prefill,
    "gather_fp8": gather_fp8,
    "absmax": absmax,
    "fp8_tensor_dynamic": fp8_tensor_dynamic,
}
