"""GPU parity of the extended FP8 write and gather (kv_store_fp8_ex,
kv_gather_fp8_ex) against the CPU oracle: e4m3fn and e5m2 caches; no scale,
per-tensor scales, and scales computed per token row or per (token, head),
whose per-slot scale caches are compared too, and caller-supplied scales
per cache page. Layouts: contiguous rows (the
row-layout kernel, one side or K and V paired per warp), head-segmented
rows, padded 4-D pages, odd head dims (narrow chunks), groups longer than a
warp holds in registers (two-pass), both index types and out-of-range
slots. All 65,536 bf16 and fp16 patterns go through the e5m2
conversion."""

import zlib

import numpy as np
import pytest

import oracle
import workloads as wl
from kvcheck import SENT8, filled, fp8_problem

pytestmark = pytest.mark.gpu

MODES = {"none": 0, "tensor": 1, "token": 2, "token_head": 3, "page": 4}


def page_inverse_scales(p, seed):
    """Per-page inverse scales around the problem's per-tensor ones: from a
    quarter of it (codes well inside the range) to 16 times it (outliers and
    large values saturate)."""
    n_pages = -(-p.size_limit // p.page_size)
    out = []
    for j, inv in enumerate((p.inv_k, p.inv_v)):
        u = wl.uniform01(seed + j, n_pages)
        out.append((np.float32(inv) * (2.0 ** np.floor(u * 7 - 2))).astype(np.float32))
    return out
FMTS = {"e4m3fn": 0, "e5m2": 1}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    yield


def run_store(p, fmt, mode, sstride=None, host=False):
    """kv_store_fp8_ex on the GPU and the oracle; compare caches, scales, errors.
    host: K, V and the slot ids in pinned host memory, read in place."""
    import torch
    import fp8_quant_gb300 as kv
    dev = torch.device("cuda")
    G = p.H if mode == "token_head" else 1
    sstride = sstride or G
    n = p.size_limit
    put = (lambda a: torch.from_numpy(a).pin_memory()) if host else (
        lambda a: torch.from_numpy(a).to(dev))
    k = put(p.k_src)
    v = put(p.v_src)
    idx = put(p.indices)
    kc = torch.from_numpy(filled(p.cache_bytes, SENT8)).to(dev)
    vc = kc.clone()
    ks = torch.full((n * sstride,), -1.0, dtype=torch.float32, device=dev)
    vs = ks.clone()
    inv = torch.tensor([p.inv_k, p.inv_v], dtype=torch.float32, device=dev)
    pages = page_inverse_scales(p, zlib.crc32(fmt.encode()) % 997) if mode == "page" else None
    if pages is not None:
        pk, pv = (torch.from_numpy(a).to(dev) for a in pages)
        inv_k_ptr, inv_v_ptr = pk.data_ptr(), pv.data_ptr()
    else:
        inv_k_ptr, inv_v_ptr = inv.data_ptr(), inv.data_ptr() + 4
    err = torch.zeros(2, dtype=torch.int64, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    rc = kv.raw.kv_store_fp8_ex(
        k.data_ptr() + p.k_view.offset, v.data_ptr() + p.v_view.offset, kc.data_ptr(),
        vc.data_ptr(), idx.data_ptr(), 1 if p.indices.dtype == np.int64 else 0, p.index_stride,
        p.T, p.H, p.D, 1 if p.src_dtype == "bf16" else 0, p.strides(), p.page_size, p.kc_page,
        p.vc_page, n, FMTS[fmt], MODES[mode], inv_k_ptr, inv_v_ptr,
        ks.data_ptr(), vs.data_ptr(), sstride, err.data_ptr(), s)
    assert rc == 0, kv.kv_status_str(rc)
    prc, pn, pfirst = kv.raw.kv_error_poll(err.data_ptr(), s)

    okc = filled(p.cache_bytes, SENT8)
    ovc = okc.copy()
    oks = np.full(n * sstride, -1.0, np.float32)
    ovs = oks.copy()
    st = oracle.Strides(**dict(zip(oracle.Strides.FIELDS, p.strides())))
    res = oracle.store_fp8_ex(p.k_src, p.v_src, okc, ovc, p.indices, st, p.H, p.D, p.src_dtype,
                              p.page_size, p.kc_page, p.vc_page, n, fmt=fmt, scale_mode=mode,
                              inv_k=p.inv_k, inv_v=p.inv_v,
                              k_scales=oks if pages is None else pages[0],
                              v_scales=ovs if pages is None else pages[1],
                              scales_slot_stride=sstride, k_off=p.k_view.offset,
                              v_off=p.v_view.offset, index_stride=p.index_stride, t_end=p.T)
    for got, want, what in ((kc, okc, "K"), (vc, ovc, "V")):
        g = got.cpu().numpy()
        if not np.array_equal(g, want):
            b = np.flatnonzero(g != want)
            raise AssertionError(f"{what} cache: {b.size} bytes differ, first {b[0]}: "
                                 f"got {g[b[0]]:#04x} want {want[b[0]]:#04x}")
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), oks.view(np.uint32))
    assert np.array_equal(vs.cpu().numpy().view(np.uint32), ovs.view(np.uint32))
    assert (pn, pfirst) == res and prc == (4 if res[0] else 0)
    return kc, vc, ks, vs, pages


CASES = {
    "rows_1024": dict(T=700, H=8, D=128, n_slots=2048, page_size=32),
    "pages_padded": dict(T=500, H=8, D=128, n_slots=2048, page_size=16, page_pad=256),
    "segmented_heads": dict(T=400, H=8, D=64, n_slots=1024, head_pad_src=64, head_pad_dst=32),
    "segmented_long_heads": dict(T=300, H=8, D=128, n_slots=1024, head_pad_src=64,
                                 head_pad_dst=32),
    "two_pass_2048": dict(T=200, H=16, D=128, n_slots=512),
    "odd_d_narrow": dict(T=300, H=3, D=45, n_slots=1024, src_dtype="f16"),
    "d24_i32": dict(T=300, H=2, D=24, n_slots=1024, idx_dtype=np.int32, index_stride=2),
    "single_head_576": dict(T=256, H=1, D=576, n_slots=1024),
    # at least 4096 rows: one warp converts the K and the V row of a token
    "paired_rows_pages": dict(T=2500, H=8, D=128, n_slots=8192, page_size=16, page_pad=256),
    "paired_long_rows_i32": dict(T=2100, H=16, D=128, n_slots=4096, idx_dtype=np.int32),
    # row-layout kernel: 512 / 1024 / 2048-byte rows, heads of 16 to 1024
    # elements (per-head groups from 2 lanes to whole multi-slab rows)
    "staged_d64_pages": dict(T=1000, H=8, D=64, n_slots=4096, page_size=16, page_pad=256),
    "staged_d32_i32": dict(T=777, H=8, D=32, n_slots=4096, idx_dtype=np.int32),
    "staged_d16": dict(T=333, H=16, D=16, n_slots=1024),
    "staged_h4_d256": dict(T=900, H=4, D=256, n_slots=4096, page_size=8),
    "staged_h2_d512": dict(T=700, H=2, D=512, n_slots=2048),
    "staged_h1_d1024_f16": dict(T=650, H=1, D=1024, n_slots=2048, src_dtype="f16"),
    "staged_many_tokens": dict(T=20000, H=8, D=128, n_slots=65536, page_size=32),
    # paired rows of one chunk per lane: per head the two divisions of a
    # group fit its 4 lanes (D=64), or not (D=32: the owner-lane form)
    "paired_h4_d64": dict(T=2500, H=4, D=64, n_slots=8192, page_size=16),
    "paired_h8_d32_i32": dict(T=2200, H=8, D=32, n_slots=8192, idx_dtype=np.int32),
    # paired rows of 2 and 4 chunks per lane with 16-lane heads (D=256)
    "paired_h4_d256": dict(T=2100, H=4, D=256, n_slots=4096, page_size=8),
    "paired_h8_d256_i32": dict(T=2100, H=8, D=256, n_slots=4096, idx_dtype=np.int32),
}


@pytest.mark.parametrize("fmt", sorted(FMTS))
@pytest.mark.parametrize("mode", sorted(MODES))
@pytest.mark.parametrize("case", sorted(CASES))
def test_store_fp8_ex_parity(case, mode, fmt):
    kw = dict(CASES[case])
    p = fp8_problem(seed=zlib.crc32((case + mode + fmt).encode()) % 9999, **kw)
    run_store(p, fmt, mode)


@pytest.mark.parametrize("mode", ["token", "token_head"])
def test_store_fp8_ex_dynamic_oob_and_scale_stride(mode):
    p = fp8_problem(T=300, H=4, D=64, n_slots=1000, seed=71, page_size=8)
    p.indices[[2, 150]] = [-1, 1000]
    run_store(p, "e4m3fn", mode, sstride=p.H + 3)


@pytest.mark.parametrize("mode", ["tensor", "token", "token_head"])
@pytest.mark.parametrize("tokens", [300, 3000])
def test_store_fp8_ex_pinned_host_inputs(mode, tokens):
    """K, V and the slot ids in pinned host memory (no L2 prefetch of host
    memory), one side per warp and paired."""
    p = fp8_problem(T=tokens, H=8, D=128, n_slots=8192, seed=79, page_size=16)
    run_store(p, "e4m3fn", mode, host=True)


@pytest.mark.parametrize("fmt", sorted(FMTS))
@pytest.mark.parametrize("mode", ["token", "token_head"])
def test_store_fp8_ex_dynamic_paired_oob(mode, fmt):
    p = fp8_problem(T=4000, H=8, D=64, n_slots=8192, seed=77, page_size=32)
    p.indices[[0, 1999, 3999]] = [-3, 8192, 2 ** 40]
    run_store(p, fmt, mode, sstride=p.H + 1)


@pytest.mark.parametrize("src", ["bf16", "f16"])
@pytest.mark.parametrize("inv", [None, 1.0, 0.001, 64.0])
def test_e5m2_exhaustive_input_patterns(src, inv):
    bits = np.arange(1 << 16, dtype=np.uint16).reshape(64, 8, 128)
    p = fp8_problem(T=64, H=8, D=128, n_slots=256, seed=72, src_dtype=src,
                    src_bits=(bits, bits[::-1].copy()), use_scale=0 if inv is None else 1,
                    inv=None if inv is None else (inv, inv))
    run_store(p, "e5m2", "none" if inv is None else "tensor")


@pytest.mark.parametrize("src", ["bf16", "f16"])
@pytest.mark.parametrize("fmt", sorted(FMTS))
@pytest.mark.parametrize("mode", ["token", "token_head"])
@pytest.mark.parametrize("tokens", [64, 2560])
def test_dynamic_exhaustive_input_patterns(src, fmt, mode, tokens):
    """Every 16-bit pattern (NaNs, infinities, subnormals, zeros) inside the
    dynamically scaled groups: groups whose amax is infinite, groups of only
    zeros or NaNs. 64 tokens run one side per warp, 2560 the paired form."""
    bits = np.arange(1 << 16, dtype=np.uint16)
    rep = tokens * 8 * 128 // bits.size
    kb = np.tile(bits, rep).reshape(tokens, 8, 128)
    vb = np.tile(bits[::-1], rep).reshape(tokens, 8, 128)
    p = fp8_problem(T=tokens, H=8, D=128, n_slots=4 * tokens, seed=78, src_dtype=src,
                    src_bits=(kb, vb))
    run_store(p, fmt, mode)


def _gather(kc, vc, p, fmt, mode, ks=None, vs=None, sstride=1, out="bf16", scale=(1.0, 1.0),
            pages=None):
    """kv_gather_fp8_ex on the GPU against the oracle.  pages: per-page forward
    scales (K, V) for the per-page mode."""
    import torch
    import fp8_quant_gb300 as kv
    dev = torch.device("cuda")
    T, H, D = p.T, p.H, p.D
    R = H * D * 2
    ko = torch.zeros(T * R, dtype=torch.uint8, device=dev)
    vo = torch.zeros_like(ko)
    sc = torch.tensor(scale, dtype=torch.float32, device=dev)
    if pages is not None:
        gk, gv = (torch.from_numpy(a).to(dev) for a in pages)
        sk_ptr, sv_ptr = gk.data_ptr(), gv.data_ptr()
    else:
        sk_ptr, sv_ptr = sc.data_ptr(), sc.data_ptr() + 4
    err = torch.zeros(2, dtype=torch.int64, device=dev)
    strides = (R, D * 2, 2, R, D * 2, 2) + p.strides()[6:]
    s = torch.cuda.current_stream().cuda_stream
    rc = kv.raw.kv_gather_fp8_ex(
        kc.data_ptr(), vc.data_ptr(), ko.data_ptr(), vo.data_ptr(),
        torch.from_numpy(p.indices).to(dev).data_ptr(), 1 if p.indices.dtype == np.int64 else 0,
        p.index_stride, T, H, D, 1 if out == "bf16" else 0, strides, p.page_size, p.kc_page,
        p.vc_page, p.size_limit, FMTS[fmt], MODES[mode], sk_ptr, sv_ptr,
        None if ks is None else ks.data_ptr(), None if vs is None else vs.data_ptr(), sstride,
        err.data_ptr(), s)
    assert rc == 0, kv.kv_status_str(rc)
    torch.cuda.synchronize()
    ok = np.zeros(T * R, np.uint8)
    ov = ok.copy()
    st = oracle.Strides(**dict(zip(oracle.Strides.FIELDS, strides)))
    oracle.gather_fp8_ex(kc.cpu().numpy(), vc.cpu().numpy(), ok, ov, p.indices, st, H, D, out,
                         p.page_size, p.kc_page, p.vc_page, p.size_limit, fmt=fmt,
                         scale_mode=mode, scale_k=scale[0], scale_v=scale[1],
                         k_scales=pages[0] if pages is not None else
                         None if ks is None else ks.cpu().numpy(),
                         v_scales=pages[1] if pages is not None else
                         None if vs is None else vs.cpu().numpy(),
                         scales_slot_stride=sstride, index_stride=p.index_stride, t_end=T)
    assert np.array_equal(ko.cpu().numpy(), ok) and np.array_equal(vo.cpu().numpy(), ov)


@pytest.mark.parametrize("fmt", sorted(FMTS))
@pytest.mark.parametrize("mode", sorted(MODES))
@pytest.mark.parametrize("out", ["bf16", "f16"])
def test_store_then_gather_fp8_ex(fmt, mode, out):
    p = fp8_problem(T=600, H=8, D=128, n_slots=2048, seed=73, page_size=16, page_pad=128)
    kc, vc, ks, vs, pages = run_store(p, fmt, mode)
    G = p.H if mode == "token_head" else 1
    scale = (1.0 / p.inv_k, 1.0 / p.inv_v)
    fwd = None if pages is None else [(np.float32(1.0) / a).astype(np.float32) for a in pages]
    _gather(kc, vc, p, fmt, mode, ks if mode in ("token", "token_head") else None,
            vs if mode in ("token", "token_head") else None, G, out, scale, pages=fwd)


@pytest.mark.parametrize("fmt", sorted(FMTS))
def test_gather_fp8_ex_every_code(fmt):
    """Random caches (every code, NaNs and infinities included) and random
    per-head scales through the dequantising gather."""
    import torch
    T, H, D, n = 512, 4, 64, 1024
    p = fp8_problem(T=T, H=H, D=D, n_slots=n, seed=74)
    dev = torch.device("cuda")
    raw = wl.splitmix64(75, 0, p.cache_bytes // 8 + 1).view(np.uint8)[:p.cache_bytes].copy()
    kc = torch.from_numpy(raw).to(dev)
    vc = torch.from_numpy(raw[::-1].copy()).to(dev)
    sc = (wl.uniform01(76, n * H) * 4 + 0.01).astype(np.float32)
    ks = torch.from_numpy(sc).to(dev)
    vs = torch.from_numpy(sc[::-1].copy()).to(dev)
    _gather(kc, vc, p, fmt, "token_head", ks, vs, H, "bf16")
    _gather(kc, vc, p, fmt, "token_head", ks, vs, H, "f16")


@pytest.mark.parametrize("tokens", [300, 3000])
def test_store_fp8_ex_per_page_oob_and_host_inputs(tokens):
    """Per-page scales with out-of-range slots (skipped before the scale load:
    no read past the scale arrays) and with K, V and slot ids in pinned host
    memory; one side per warp and paired."""
    p = fp8_problem(T=tokens, H=8, D=128, n_slots=8192, seed=81, page_size=16)
    p.indices[[1, tokens // 2, tokens - 1]] = [-1, 8192, 2 ** 40]
    run_store(p, "e4m3fn", "page")
    q = fp8_problem(T=tokens, H=8, D=128, n_slots=8192, seed=82, page_size=16)
    run_store(q, "e5m2", "page", host=True)


@pytest.mark.parametrize("fmt", sorted(FMTS))
def test_gather_fp8_ex_per_page_every_code(fmt):
    """Random caches (every code) through the dequantising gather with one
    random forward scale per page, paged layout with padding, both outputs."""
    import torch
    T, H, D, n = 3000, 8, 128, 8192
    p = fp8_problem(T=T, H=H, D=D, n_slots=n, seed=83, page_size=32, page_pad=512)
    dev = torch.device("cuda")
    raw = wl.splitmix64(84, 0, p.cache_bytes // 8 + 1).view(np.uint8)[:p.cache_bytes].copy()
    kc = torch.from_numpy(raw).to(dev)
    vc = torch.from_numpy(raw[::-1].copy()).to(dev)
    n_pages = -(-n // p.page_size)
    fk = (wl.uniform01(85, n_pages) * 4 + 0.01).astype(np.float32)
    fv = (wl.uniform01(86, n_pages) * 8 + 0.5).astype(np.float32)
    _gather(kc, vc, p, fmt, "page", out="bf16", pages=(fk, fv))
    _gather(kc, vc, p, fmt, "page", out="f16", pages=(fk, fv))
