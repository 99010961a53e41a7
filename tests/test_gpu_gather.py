"""GPU parity of the inverse path (kv_gather, kv_gather_fp8) against the CPU
oracle, through the C ABI.

Each case fills a cache storage with seeded random bytes (so every e4m3fn
code, NaNs included, appears for the FP8 gather), pre-fills the outputs with
a sentinel, gathers, and compares every output byte and the out-of-range
report with the oracle. Layouts cover contiguous and padded rows, head
segments, strided dims (element kernels), misaligned views, 3-D and padded
4-D paged caches, both index types, index strides and out-of-range slots,
in launches small enough for one side per warp, large enough for the
paired K/V form, and larger than one wave of resident warps (look-ahead
prefetch).
"""

import zlib
from dataclasses import dataclass

import numpy as np
import pytest

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    yield


@dataclass
class G:
    kind: str              # "copy" | "fp8"
    T: int
    H: int
    D: int
    elem: int              # copy element size / 2 for fp8 outputs
    cache: np.ndarray      # K cache storage (V cache = a second random storage)
    vcache: np.ndarray
    cslot: int
    chead: int
    cdim: int
    page_size: int
    cpage: int
    out_bytes: int
    otok: int
    ohead: int
    odim: int
    ooff: int
    idx: np.ndarray
    index_stride: int
    size_limit: int
    out_dtype: str = "bf16"
    scale: float = 1.0
    use_scale: int = 0

    def strides(self):
        return (self.otok, self.ohead, self.odim, self.otok, self.ohead, self.odim,
                self.cslot, self.chead, self.cdim, self.cslot, self.chead, self.cdim)


def make(kind, T, H, D, n, seed, elem=2, idx_dtype=np.int64, index_stride=1, slot_pad=0,
         head_pad_c=0, head_pad_o=0, dim_mult=1, ooff=0, page_size=1, page_pad=0, out="bf16",
         scale=None, bad=()):
    ce = 1 if kind == "fp8" else elem
    oe = 2 if kind == "fp8" else elem
    chead = D * ce * dim_mult + head_pad_c
    cslot = H * chead + slot_pad
    n_pages = -(-n // page_size)
    cpage = page_size * cslot + page_pad
    cbytes = n_pages * cpage
    rnd = lambda s: (wl.splitmix64(s, 0, (cbytes + 7) // 8).view(np.uint8)[:cbytes]).copy()
    ohead = D * oe * dim_mult + head_pad_o
    otok = H * ohead
    out_bytes = ooff + T * otok
    slots = wl.distinct_slots(seed + 2, n, T)
    for i, b in bad:
        slots[i] = b
    idx = np.zeros(T * index_stride, dtype=idx_dtype)
    idx[::index_stride] = slots
    return G(kind=kind, T=T, H=H, D=D, elem=oe, cache=rnd(seed), vcache=rnd(seed + 1),
             cslot=cslot, chead=chead, cdim=ce * dim_mult, page_size=page_size, cpage=cpage,
             out_bytes=out_bytes, otok=otok, ohead=ohead, odim=oe * dim_mult, ooff=ooff, idx=idx,
             index_stride=index_stride, size_limit=n, out_dtype=out,
             scale=1.0 if scale is None else scale, use_scale=0 if scale is None else 1)


SENT = bytes([0xC0, 0x7F])


def run_both(g: G, host_out=False, host_idx=False):
    """host_out: the gathered rows are written straight into pinned host memory;
    host_idx: the slot ids are read from pinned host memory."""
    import torch
    import fp8_quant_gb300 as kv
    dev = torch.device("cuda")
    filled = np.frombuffer(SENT * (g.out_bytes // 2 + 1), np.uint8)[:g.out_bytes].copy()
    kc = torch.from_numpy(g.cache).to(dev)
    vc = torch.from_numpy(g.vcache).to(dev)
    if host_out:
        ko = torch.from_numpy(filled.copy()).pin_memory()
        vo = torch.from_numpy(filled.copy()).pin_memory()
    else:
        ko = torch.from_numpy(filled).to(dev)
        vo = ko.clone()
    idx = torch.from_numpy(g.idx).pin_memory() if host_idx else torch.from_numpy(g.idx).to(dev)
    err = torch.zeros(2, dtype=torch.int64, device=dev)
    sc = torch.tensor([g.scale, g.scale], dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    idt = 1 if g.idx.dtype == np.int64 else 0
    paged_copy = g.kind == "copy" and g.cpage != g.page_size * g.cslot
    if paged_copy:
        rc = kv.raw.kv_gather_paged(kc.data_ptr(), vc.data_ptr(), ko.data_ptr() + g.ooff,
                                    vo.data_ptr() + g.ooff, idx.data_ptr(), idt, g.index_stride,
                                    g.T, g.H, g.D, g.elem, g.strides(), g.page_size, g.cpage,
                                    g.cpage, g.size_limit, err.data_ptr(), s)
    elif g.kind == "copy":
        rc = kv.raw.kv_gather(kc.data_ptr(), vc.data_ptr(), ko.data_ptr() + g.ooff,
                              vo.data_ptr() + g.ooff, idx.data_ptr(), idt, g.index_stride, g.T,
                              g.H, g.D, g.elem, g.strides(), g.size_limit, err.data_ptr(), s)
    else:
        rc = kv.raw.kv_gather_fp8(kc.data_ptr(), vc.data_ptr(), ko.data_ptr() + g.ooff,
                                  vo.data_ptr() + g.ooff, idx.data_ptr(), idt, g.index_stride,
                                  g.T, g.H, g.D, 1 if g.out_dtype == "bf16" else 0, g.strides(),
                                  g.page_size, g.cpage, g.cpage, g.size_limit,
                                  sc.data_ptr() if g.use_scale else None,
                                  sc.data_ptr() + 4 if g.use_scale else None, g.use_scale,
                                  err.data_ptr(), s)
    assert rc == 0, kv.kv_status_str(rc)
    prc, pn, pfirst = kv.raw.kv_error_poll(err.data_ptr(), s)
    torch.cuda.synchronize()
    gk, gv = ko.cpu().numpy().copy(), vo.cpu().numpy().copy()

    ok, ov = filled.copy(), filled.copy()
    st = oracle.Strides(**dict(zip(oracle.Strides.FIELDS, g.strides())))
    okv, ovv = ok[g.ooff:], ov[g.ooff:]
    if paged_copy:
        res = oracle.gather_copy_paged(g.cache, g.vcache, okv, ovv, g.idx, st, g.H, g.D, g.elem,
                                       g.page_size, g.cpage, g.cpage, g.size_limit,
                                       index_stride=g.index_stride, t_end=g.T)
    elif g.kind == "copy":
        res = oracle.gather_copy(g.cache, g.vcache, okv, ovv, g.idx, st, g.H, g.D, g.elem,
                                 g.size_limit, index_stride=g.index_stride, t_end=g.T)
    else:
        res = oracle.gather_fp8(g.cache, g.vcache, okv, ovv, g.idx, st, g.H, g.D, g.out_dtype,
                                g.page_size, g.cpage, g.cpage, g.size_limit, g.scale, g.scale,
                                g.use_scale, index_stride=g.index_stride, t_end=g.T)
    # okv/ovv are views into ok/ov: the oracle wrote through them
    for got, want, what in ((gk, ok, "K"), (gv, ov, "V")):
        if not np.array_equal(got, want):
            b = np.flatnonzero(got != want)
            raise AssertionError(f"{what}: {b.size} bytes differ, first at {b[0]}: "
                                 f"got {got[b[0]]:#04x} want {want[b[0]]:#04x}")
    assert (pn, pfirst) == res and prc == (4 if res[0] else 0)


COPY = {
    "decode_shape": dict(T=777, H=8, D=128, n=4096),
    "odd_1152_in_1280": dict(T=900, H=1, D=576, n=3000, slot_pad=128, idx_dtype=np.int32),
    "head_segments": dict(T=500, H=8, D=64, n=2000, head_pad_c=64, head_pad_o=32),
    "strided_dims": dict(T=300, H=4, D=32, n=900, dim_mult=2),
    "misaligned_out": dict(T=400, H=4, D=64, n=1200, ooff=4),
    "bytes_odd": dict(T=300, H=3, D=7, n=900, elem=1, ooff=1),
    "fp32_rows": dict(T=300, H=2, D=96, n=900, elem=4),
    "index_stride2": dict(T=513, H=8, D=128, n=2000, index_stride=2, idx_dtype=np.int32),
    "small_batch": dict(T=3, H=8, D=128, n=64),
    "oob": dict(T=600, H=8, D=128, n=2000, bad=((0, -1), (17, 2000), (599, 2 ** 40))),
    # kv_gather_paged: padded pages
    "paged_padded_16": dict(T=700, H=8, D=128, n=4096, page_size=16, page_pad=512),
    "paged_odd_rows": dict(T=500, H=1, D=576, n=2048, page_size=32, page_pad=128, slot_pad=128,
                           idx_dtype=np.int32),
    "paged_page7_generic": dict(T=300, H=2, D=20, n=700, page_size=7, page_pad=12, dim_mult=2),
    # launches of at least 4096 warps pair the K and V rows of a slot in one warp
    "paired_rows_parts2": dict(T=1111, H=8, D=128, n=8192),
    "paired_oob": dict(T=3001, H=8, D=128, n=8192, bad=((0, -1), (1500, 8192), (3000, -5))),
    "paired_paged_i32": dict(T=2500, H=8, D=128, n=8192, page_size=16, page_pad=512,
                             idx_dtype=np.int32),
    # more units than resident warps: each warp also prefetches the rows of the
    # unit one resident wave ahead
    "multiwave_rows_oob": dict(T=20000, H=8, D=128, n=32768,
                               bad=((5, -1), (10000, 40000), (19999, 32768))),
    "multiwave_heads_paged": dict(T=3000, H=8, D=64, n=8192, head_pad_c=64, head_pad_o=32,
                                  page_size=16, page_pad=256),
}

FP8 = {
    "bf16_unscaled": dict(T=1000, H=8, D=128, n=4096),
    "bf16_scaled": dict(T=1000, H=8, D=128, n=4096, scale=0.0123),
    "f16_scaled": dict(T=700, H=8, D=128, n=2048, out="f16", scale=3.5),
    "f16_overflow": dict(T=300, H=4, D=64, n=1024, out="f16", scale=1000.0),
    "pages_4d_padded": dict(T=900, H=8, D=128, n=4096, page_size=32, page_pad=256, scale=0.5),
    "odd_page_size": dict(T=400, H=2, D=64, n=1000, page_size=7, page_pad=16, scale=2.0),
    "head_segments": dict(T=500, H=8, D=64, n=1500, head_pad_c=32, head_pad_o=64, scale=1.5),
    "in8_d24": dict(T=640, H=3, D=24, n=1500, scale=0.25),
    "in4_d20": dict(T=640, H=1, D=20, n=1500),
    "in2_d6": dict(T=640, H=1, D=6, n=1500, out="f16"),
    "generic_odd_d": dict(T=300, H=3, D=45, n=900, scale=1.25),
    "generic_strided": dict(T=300, H=2, D=32, n=900, dim_mult=2, scale=7.0),
    "misaligned_out": dict(T=300, H=4, D=64, n=900, ooff=2, scale=0.75),
    "oob_int32": dict(T=600, H=8, D=128, n=2000, idx_dtype=np.int32,
                      bad=((5, -9), (6, 2000)), scale=1.0),
    "paired_scaled_oob": dict(T=3001, H=8, D=128, n=8192, scale=0.37,
                              bad=((7, -1), (3000, 8192))),
    "paired_f16_pages": dict(T=2222, H=8, D=128, n=8192, out="f16", page_size=32, page_pad=256,
                             scale=2.5),
    "paired_parts2": dict(T=1111, H=8, D=128, n=4096, scale=1.0),
    "paired_in8_heads": dict(T=900, H=3, D=24, n=2048, scale=0.5),
    "multiwave_scaled_oob": dict(T=12000, H=8, D=128, n=16384, scale=0.3,
                                 bad=((1, -1), (6000, 16384), (11999, -7))),
    "multiwave_f16_heads": dict(T=3000, H=8, D=64, n=8192, head_pad_c=32, head_pad_o=64,
                                out="f16", scale=2.0),
}


@pytest.mark.parametrize("name", sorted(COPY))
def test_gather_copy_parity(name):
    run_both(make("copy", seed=zlib.crc32(name.encode()) % 9999, **COPY[name]))


@pytest.mark.parametrize("name", sorted(FP8))
def test_gather_fp8_parity(name):
    run_both(make("fp8", seed=zlib.crc32(name.encode()) % 9999, **FP8[name]))


def test_store_fp8_then_gather_round_trip():
    """kv_store_fp8 then kv_gather_fp8 on the GPU equals the oracle's store
    then gather, byte for byte."""
    import torch
    import fp8_quant_gb300 as kv
    T, H, D, n, ps = 1024, 8, 128, 4096, 16
    w = wl.make_fp8("rt", T, H, D, n, seed=901, page_size=ps)
    dev = torch.device("cuda")
    k = torch.from_numpy(w.k.view(np.int16)).to(dev).view(torch.bfloat16)
    v = torch.from_numpy(w.v.view(np.int16)).to(dev).view(torch.bfloat16)
    idx = torch.from_numpy(w.indices).to(dev)
    kc = torch.full((n, H, D), 0x7F, dtype=torch.uint8, device=dev)
    vc = kc.clone()
    inv = torch.tensor([w.inv_k, w.inv_v], dtype=torch.float32, device=dev)
    scale = torch.tensor([1.0, 1.0], dtype=torch.float32, device=dev) / inv
    err = kv.error_record(dev)
    kv.kv_store_fp8(k, v, kc, vc, idx, page_size=ps, inv_k_scale=inv[0:1], inv_v_scale=inv[1:2],
                    err=err)
    ko = torch.zeros(T, H, D, dtype=torch.bfloat16, device=dev)
    vo = torch.zeros_like(ko)
    s = torch.cuda.current_stream().cuda_stream
    R = H * D * 2
    strides = (R, D * 2, 2, R, D * 2, 2, H * D, D, 1, H * D, D, 1)
    assert kv.raw.kv_gather_fp8(kc.data_ptr(), vc.data_ptr(), ko.data_ptr(), vo.data_ptr(),
                                idx.data_ptr(), 1, 1, T, H, D, 1, strides, ps, ps * H * D,
                                ps * H * D, n, scale.data_ptr(), scale.data_ptr() + 4, 1,
                                err.data_ptr(), s) == 0
    assert kv.kv_error_poll(err)[1] == 0
    sk, sv = scale.cpu().numpy()
    okc = np.full(n * H * D, 0x7F, np.uint8)
    ovc = okc.copy()
    st = oracle.Strides(k_token=R, k_head=D * 2, k_dim=2, v_token=R, v_head=D * 2, v_dim=2,
                        kc_slot=H * D, kc_head=D, kc_dim=1, vc_slot=H * D, vc_head=D, vc_dim=1)
    oracle.store_fp8(w.k, w.v, okc, ovc, w.indices, st, H, D, "bf16", ps, ps * H * D, ps * H * D,
                     n, w.inv_k, w.inv_v, 1)
    ok = np.zeros(T * H * D, np.uint16)
    ov = ok.copy()
    oracle.gather_fp8(okc, ovc, ok, ov, w.indices, st, H, D, "bf16", ps, ps * H * D, ps * H * D,
                      n, float(sk), float(sv), 1)
    assert np.array_equal(ko.view(torch.int16).cpu().numpy().view(np.uint16).ravel(), ok)
    assert np.array_equal(vo.view(torch.int16).cpu().numpy().view(np.uint16).ravel(), ov)


@pytest.mark.parametrize("kind", ["copy", "fp8"])
def test_gather_into_pinned_host_memory(kind):
    """Swap-out: the gathered (and dequantised) rows are written straight into
    pinned host memory by the kernel."""
    if kind == "copy":
        g = make("copy", T=900, H=8, D=128, n=4096, seed=801)
    else:
        g = make("fp8", T=900, H=8, D=128, n=4096, seed=802, page_size=16, page_pad=64,
                 scale=0.05)
    run_both(g, host_out=True)


@pytest.mark.parametrize("kind", ["copy", "fp8"])
@pytest.mark.parametrize("tokens", [300, 3000])
def test_gather_offload_from_pinned_slots(kind, tokens):
    """Slot ids read from pinned host memory and rows written into pinned host
    memory (the zero-copy offload), one side per warp and paired."""
    if kind == "copy":
        g = make("copy", T=tokens, H=8, D=128, n=8192, seed=803, bad=((1, -1),))
    else:
        g = make("fp8", T=tokens, H=8, D=128, n=8192, seed=804, page_size=16, scale=0.1,
                 bad=((2, 8192),))
    run_both(g, host_out=True, host_idx=True)
