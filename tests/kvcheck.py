"""Test harness: run one write problem through the C ABI on the GPU and through
the CPU oracle on the host, on byte-identical inputs.

A problem is described in bytes: a source storage per input (K and V may share
one, e.g. a fused QKV tensor), a view of K and of V inside it as (byte offset,
token stride, head stride, dim stride), a cache storage size and the cache
view (slot, head, dim strides, plus a page stride for FP8). Both sides see
exactly these bytes; the GPU side passes device addresses and byte strides to
``raw.kv_store`` / ``raw.kv_store_fp8``.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np

import oracle
import workloads as wl


@dataclass
class View:
    offset: int
    token: int      # token stride (inputs) or slot stride (caches), bytes
    head: int
    dim: int


@dataclass
class Problem:
    kind: str                  # "copy" | "fp8"
    k_src: np.ndarray          # uint8 storage of K
    v_src: np.ndarray          # uint8 storage of V (may be the same object as k_src)
    k_view: View
    v_view: View
    kc_view: View
    vc_view: View
    cache_bytes: int           # bytes per cache storage
    sentinel: bytes            # pre-fill pattern repeated over the caches
    indices: np.ndarray        # int32 / int64, possibly with index_stride > 1 (raw storage)
    index_stride: int
    T: int
    H: int
    D: int
    elem: int                  # input element size (copy) / 2 (fp8)
    size_limit: int
    num_split: int = 0
    src_dtype: str = "bf16"    # fp8 only
    page_size: int = 1
    kc_page: int = 0
    vc_page: int = 0
    inv_k: float = 1.0
    inv_v: float = 1.0
    use_scale: int = 0
    paged: bool = False        # copy through kv_store_paged (page_size, kc_page, vc_page)

    def strides(self):
        return (self.k_view.token, self.k_view.head, self.k_view.dim,
                self.v_view.token, self.v_view.head, self.v_view.dim,
                self.kc_view.token, self.kc_view.head, self.kc_view.dim,
                self.vc_view.token, self.vc_view.head, self.vc_view.dim)


def filled(nbytes: int, pattern: bytes) -> np.ndarray:
    reps = -(-nbytes // len(pattern))
    return np.frombuffer(pattern * reps, dtype=np.uint8)[:nbytes].copy()


SENT16 = bytes([wl.BF16_SENTINEL & 0xFF, wl.BF16_SENTINEL >> 8])
SENT8 = bytes([wl.FP8_SENTINEL])


def run_oracle(p: Problem):
    """Returns (k_cache bytes, v_cache bytes, (bad_count, first_bad))."""
    kc = filled(p.cache_bytes, p.sentinel)
    vc = filled(p.cache_bytes, p.sentinel)
    st = oracle.Strides(**dict(zip(oracle.Strides.FIELDS, p.strides())))
    if p.kind == "copy" and p.paged:
        assert p.kc_view.offset == 0 and p.vc_view.offset == 0
        res = oracle.store_copy_paged(p.k_src, p.v_src, kc, vc, p.indices, st, p.H, p.D, p.elem,
                                      p.page_size, p.kc_page, p.vc_page, p.size_limit,
                                      k_off=p.k_view.offset, v_off=p.v_view.offset,
                                      index_stride=p.index_stride, t_end=p.T)
    elif p.kind == "copy":
        res = oracle.store_copy(p.k_src, p.v_src, kc, vc, p.indices, st, p.H, p.D, p.elem,
                                p.size_limit, k_off=p.k_view.offset, v_off=p.v_view.offset,
                                kc_off=p.kc_view.offset, vc_off=p.vc_view.offset,
                                index_stride=p.index_stride, t_end=p.T)
    else:
        assert p.kc_view.offset == 0 and p.vc_view.offset == 0
        res = oracle.store_fp8(p.k_src, p.v_src, kc, vc, p.indices, st, p.H, p.D, p.src_dtype,
                               p.page_size, p.kc_page, p.vc_page, p.size_limit, p.inv_k,
                               p.inv_v, p.use_scale, k_off=p.k_view.offset,
                               v_off=p.v_view.offset, index_stride=p.index_stride, t_end=p.T)
    return kc, vc, res


class DeviceRun:
    """Device copies of a problem's inputs and caches, and the C-ABI call."""

    def __init__(self, p: Problem, device="cuda"):
        import torch
        self.p = p
        self.torch = torch
        self.dev = torch.device(device)
        self.k_src = torch.from_numpy(p.k_src).to(self.dev)
        self.v_src = self.k_src if p.v_src is p.k_src else torch.from_numpy(p.v_src).to(self.dev)
        self.idx = torch.from_numpy(p.indices).to(self.dev)
        pat = torch.from_numpy(filled(p.cache_bytes, p.sentinel)) if p.cache_bytes <= (64 << 20) \
            else None
        if pat is not None:
            self.kc = pat.to(self.dev)
            self.vc = self.kc.clone()
        else:
            self.kc = self._fill_big(p.cache_bytes, p.sentinel)
            self.vc = self._fill_big(p.cache_bytes, p.sentinel)
        self.err = torch.zeros(2, dtype=torch.int64, device=self.dev)
        self.inv = torch.tensor([p.inv_k, p.inv_v], dtype=torch.float32, device=self.dev)

    def _fill_big(self, nbytes, pattern):
        torch = self.torch
        if len(pattern) == 1:
            return torch.full((nbytes,), pattern[0], dtype=torch.uint8, device=self.dev)
        assert len(pattern) == 2 and nbytes % 2 == 0
        val = int.from_bytes(pattern, "little")
        val = val - 65536 if val >= 32768 else val
        return torch.full((nbytes // 2,), val, dtype=torch.int16, device=self.dev).view(torch.uint8)

    def call(self, stream=None, num_split=None) -> int:
        import fp8_quant_gb300 as kv
        p = self.p
        s = stream if stream is not None else self.torch.cuda.current_stream(self.dev).cuda_stream
        idt = 1 if p.indices.dtype == np.int64 else 0
        kptr = self.k_src.data_ptr() + p.k_view.offset
        vptr = self.v_src.data_ptr() + p.v_view.offset
        if p.kind == "copy" and p.paged:
            return kv.raw.kv_store_paged(kptr, vptr, self.kc.data_ptr(), self.vc.data_ptr(),
                                         self.idx.data_ptr(), idt, p.index_stride, p.T, p.H, p.D,
                                         p.elem, p.strides(), p.page_size, p.kc_page, p.vc_page,
                                         p.size_limit,
                                         p.num_split if num_split is None else num_split,
                                         self.err.data_ptr(), s)
        if p.kind == "copy":
            return kv.raw.kv_store(kptr, vptr, self.kc.data_ptr() + p.kc_view.offset,
                                   self.vc.data_ptr() + p.vc_view.offset, self.idx.data_ptr(),
                                   idt, p.index_stride, p.T, p.H, p.D, p.elem, p.strides(),
                                   p.size_limit, p.num_split if num_split is None else num_split,
                                   self.err.data_ptr(), s)
        return kv.raw.kv_store_fp8(kptr, vptr, self.kc.data_ptr(), self.vc.data_ptr(),
                                   self.idx.data_ptr(), idt, p.index_stride, p.T, p.H, p.D,
                                   1 if p.src_dtype == "bf16" else 0, p.strides(), p.page_size,
                                   p.kc_page, p.vc_page, p.size_limit,
                                   self.inv.data_ptr() if p.use_scale else None,
                                   self.inv.data_ptr() + 4 if p.use_scale else None,
                                   p.use_scale, self.err.data_ptr(), s)

    def poll(self, stream=None):
        import fp8_quant_gb300 as kv
        s = stream if stream is not None else self.torch.cuda.current_stream(self.dev).cuda_stream
        return kv.raw.kv_error_poll(self.err.data_ptr(), s)

    def caches(self):
        self.torch.cuda.synchronize(self.dev)
        return self.kc.cpu().numpy(), self.vc.cpu().numpy()


def diff_report(got: np.ndarray, want: np.ndarray, row: int) -> str:
    bad = np.flatnonzero(got != want)
    if bad.size == 0:
        return "equal"
    b = bad[0]
    return (f"{bad.size} bytes differ; first at byte {b} (row {b // row}, byte {b % row}): "
            f"got {got[b]:#04x} want {want[b]:#04x}")


def assert_same(p: Problem, row_bytes: Optional[int] = None, num_split=None):
    """Run both sides; compare every cache byte and the error report."""
    g = DeviceRun(p)
    rc = g.call(num_split=num_split)
    assert rc == 0, f"launch status {rc}"
    prc, pn, pfirst = g.poll()
    kc, vc = g.caches()
    okc, ovc, (obad, ofirst) = run_oracle(p)
    rb = row_bytes or max(1, p.kc_view.token)
    assert np.array_equal(kc, okc), "K cache: " + diff_report(kc, okc, rb)
    assert np.array_equal(vc, ovc), "V cache: " + diff_report(vc, ovc, rb)
    assert (pn, pfirst) == (obad, ofirst), ((pn, pfirst), (obad, ofirst))
    assert prc == (4 if obad else 0)
    return g


# ---------------------------------------------------------------------------
# Problem builders
# ---------------------------------------------------------------------------

def rand_bytes(seed: int, n: int) -> np.ndarray:
    """Random 2-byte elements (N(0,1) as bf16) as bytes; n must be even."""
    return wl.f32_to_bf16_bits(wl.normal(seed, n // 2)).view(np.uint8)


def copy_problem(T, H, D, n_slots, seed, elem=2, idx_dtype=np.int64, index_stride=1,
                 slot_pad=0, head_pad_src=0, head_pad_dst=0, dim_stride_mult=1,
                 src_off=0, dst_off=0, token_pad=0, num_split=0, size_limit=None,
                 slots=None, qkv_shared=False, page_size=None, page_pad=0) -> Problem:
    """A copy problem with optional padding/offsets that exercise every path."""
    row_src_head = D * elem * dim_stride_mult + head_pad_src
    tok = H * row_src_head + token_pad
    nsrc = src_off + T * tok + 64
    if qkv_shared:
        # K and V interleaved in one storage: token = [K heads | V heads]
        tok2 = 2 * H * row_src_head + token_pad
        nsrc = src_off + T * tok2 + 64
        src = rand_bytes(seed, nsrc + nsrc % 2)[:nsrc].copy()
        kvw = View(src_off, tok2, row_src_head, elem * dim_stride_mult)
        vvw = View(src_off + H * row_src_head, tok2, row_src_head, elem * dim_stride_mult)
        ksrc = vsrc = src
    else:
        ksrc = rand_bytes(seed, nsrc + nsrc % 2)[:nsrc].copy()
        vsrc = rand_bytes(seed + 1, nsrc + nsrc % 2)[:nsrc].copy()
        kvw = View(src_off, tok, row_src_head, elem * dim_stride_mult)
        vvw = View(src_off, tok, row_src_head, elem * dim_stride_mult)
    dst_head = D * elem * dim_stride_mult + head_pad_dst
    slot = H * dst_head + slot_pad
    cache_bytes = dst_off + n_slots * slot
    paged = page_size is not None
    ps = page_size or 1
    page = ps * slot + page_pad
    if paged:
        assert dst_off == 0
        cache_bytes = -(-n_slots // ps) * page
    if slots is None:
        slots = wl.distinct_slots(seed + 2, n_slots, T)
    idx_store = np.zeros(T * index_stride, dtype=idx_dtype)
    idx_store[::index_stride] = slots
    return Problem(kind="copy", paged=paged, page_size=ps, kc_page=page, vc_page=page,
                   k_src=ksrc, v_src=vsrc, k_view=kvw, v_view=vvw,
                   kc_view=View(dst_off, slot, dst_head, elem * dim_stride_mult),
                   vc_view=View(dst_off, slot, dst_head, elem * dim_stride_mult),
                   cache_bytes=cache_bytes, sentinel=SENT16 if elem % 2 == 0 else SENT8,
                   indices=idx_store, index_stride=index_stride, T=T, H=H, D=D, elem=elem,
                   size_limit=n_slots if size_limit is None else size_limit,
                   num_split=num_split)


def fp8_problem(T, H, D, n_slots, seed, src_dtype="bf16", idx_dtype=np.int64, page_size=16,
                page_pad=0, use_scale=1, slot_pad=0, head_pad_src=0, head_pad_dst=0,
                src_dim_mult=1, dst_dim_mult=1, src_off=0, token_pad=0, index_stride=1,
                size_limit=None, scale=4.0, outlier_frac=0.001, src_bits=None,
                inv=None) -> Problem:
    """An FP8 problem; ``src_bits`` ([T, H, D] uint16 per K and V) overrides the data."""
    if src_bits is None:
        w = wl.make_fp8("t", T, H, D, max(n_slots, T), seed=seed, dtype=src_dtype,
                        page_size=page_size, scale=scale, outlier_frac=outlier_frac)
        kb, vb, ik, iv = w.k, w.v, w.inv_k, w.inv_v
    else:
        kb, vb = src_bits
        ik = iv = 1.0
    if inv is not None:
        ik, iv = inv
    e = 2
    row_head = D * e * src_dim_mult + head_pad_src
    tok = H * row_head + token_pad
    nsrc = src_off + T * tok + 64

    def place(bits):
        buf = np.zeros(nsrc, dtype=np.uint8)
        for h in range(H):
            for_d = np.arange(D) * e * src_dim_mult
            base = src_off + np.arange(T)[:, None] * tok + h * row_head + for_d[None, :]
            vals = bits[:, h, :].astype(np.uint16).view(np.uint8).reshape(T, D, 2)
            buf[base] = vals[..., 0]
            buf[base + 1] = vals[..., 1]
        return buf

    ksrc, vsrc = place(kb), place(vb)
    dst_head = D * dst_dim_mult + head_pad_dst
    slot = H * dst_head + slot_pad
    n_pages = -(-n_slots // page_size)
    page = page_size * slot + page_pad
    cache_bytes = n_pages * page
    slots = wl.distinct_slots(seed + 9, n_slots, T)
    idx_store = np.zeros(T * index_stride, dtype=idx_dtype)
    idx_store[::index_stride] = slots
    return Problem(kind="fp8", k_src=ksrc, v_src=vsrc,
                   k_view=View(src_off, tok, row_head, e * src_dim_mult),
                   v_view=View(src_off, tok, row_head, e * src_dim_mult),
                   kc_view=View(0, slot, dst_head, dst_dim_mult),
                   vc_view=View(0, slot, dst_head, dst_dim_mult),
                   cache_bytes=cache_bytes, sentinel=SENT8, indices=idx_store,
                   index_stride=index_stride, T=T, H=H, D=D, elem=2,
                   size_limit=n_slots if size_limit is None else size_limit,
                   src_dtype=src_dtype, page_size=page_size, kc_page=page, vc_page=page,
                   inv_k=ik, inv_v=iv, use_scale=use_scale)
