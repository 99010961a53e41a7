"""Full-size parity: every benchmark workload at its full size, in exactly the
launch configuration ``bench.py`` times (its ``Pool.call`` on batch 0, which is
the workload's own seeded data).

For each call: every written cache row (gathered on the GPU at the batch's
slots, whole slot stride including padding) is compared byte for byte with
the CPU oracle run on the same inputs (slots renumbered 0..T-1 into a compact
host cache, which leaves the row contents unchanged); the number of cache rows
that differ from the pre-fill must equal T, so nothing else was touched; and
the error record must be clean.
"""

import numpy as np
import pytest

import oracle

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    yield


def _rows_changed(torch, cache, n_slots, slot_bytes, sentinel_bytes):
    """Rows of the cache whose bytes differ from the pre-fill (counted on the GPU)."""
    words = cache.view(torch.uint8).view(n_slots, slot_bytes)
    pat = torch.tensor(list(sentinel_bytes) * (slot_bytes // len(sentinel_bytes)),
                       dtype=torch.uint8, device=cache.device)
    total = 0
    step = max(1, (256 << 20) // slot_bytes)
    for r0 in range(0, n_slots, step):
        total += int((words[r0:r0 + step] != pat).any(dim=1).sum().item())
    return total


def _oracle_gather_compact(w, rows_k, rows_v):
    """Oracle gather from the T named cache rows (compact cache, slots 0..T-1)."""
    T = w.T
    idx = np.arange(T, dtype=w.indices.dtype)
    sb = w.slot_stride
    st = oracle.Strides(k_token=w.k_view[1], k_head=w.k_view[2], k_dim=w.k_view[3],
                        v_token=w.v_view[1], v_head=w.v_view[2], v_dim=w.v_view[3],
                        kc_slot=sb, kc_head=w.cache_head_stride, kc_dim=w.cache_elem,
                        vc_slot=sb, vc_head=w.cache_head_stride, vc_dim=w.cache_elem)
    ok = np.zeros(T * w.k_view[1], np.uint8)
    ov = np.zeros_like(ok)
    kc, vc = rows_k.reshape(-1).copy(), rows_v.reshape(-1).copy()
    if w.kind == "gather":
        bad = oracle.gather_copy(kc, vc, ok, ov, idx, st, w.H, w.D, 2, T)
    else:
        assert w.page_stride == w.page_size * sb
        bad = oracle.gather_fp8(kc, vc, ok, ov, idx, st, w.H, w.D, w.src_dtype, w.page_size,
                                w.page_stride, w.page_stride, T + (-T) % w.page_size,
                                float(np.float32(1.0) / np.float32(w.inv_k)),
                                float(np.float32(1.0) / np.float32(w.inv_v)), 1)
    assert bad == (0, -1)
    return ok, ov


@pytest.mark.parametrize("name", ["gather_decode", "gather_prefill", "gather_fp8"])
def test_full_size_gather(name):
    import torch
    import bench
    import fp8_quant_gb300 as kv
    dev = torch.device("cuda", 0)
    pool = bench.Pool(name, dev, pool_bytes=0)
    w = pool.w
    assert pool.call(0, torch.cuda.current_stream().cuda_stream) == 0
    assert kv.kv_error_poll(pool.err)[:2] == (kv.KVStatus.OK, 0)
    sb = w.slot_stride
    slots = torch.from_numpy(w.indices.astype(np.int64)).to(dev)
    rows = [c.view(torch.uint8).view(w.n_slots, sb).index_select(0, slots).cpu().numpy()
            for c in (pool.kc, pool.vc)]
    ok, ov = _oracle_gather_compact(w, *rows)
    gk = pool.k[0].view(torch.uint8).reshape(-1).cpu().numpy()
    gv = pool.v[0].view(torch.uint8).reshape(-1).cpu().numpy()
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)
    del pool
    torch.cuda.empty_cache()


def _oracle_compact(w):
    """Oracle over all tokens with slots renumbered 0..T-1 (compact caches)."""
    T = w.T
    idx = np.arange(T, dtype=w.indices.dtype)
    sb = w.slot_stride
    sent = (w.sentinel.to_bytes(2, "little") if w.cache_elem == 2 else bytes([w.sentinel]))
    kc = np.frombuffer(sent * (T * sb // len(sent)), dtype=np.uint8).copy()
    vc = kc.copy()
    st = oracle.Strides(k_token=w.k_view[1], k_head=w.k_view[2], k_dim=w.k_view[3],
                        v_token=w.v_view[1], v_head=w.v_view[2], v_dim=w.v_view[3],
                        kc_slot=sb, kc_head=w.cache_head_stride, kc_dim=w.cache_elem,
                        vc_slot=sb, vc_head=w.cache_head_stride, vc_dim=w.cache_elem)
    k = np.ascontiguousarray(w.k).view(np.uint8).reshape(-1)
    v = np.ascontiguousarray(w.v).view(np.uint8).reshape(-1)
    if w.kind == "copy":
        bad = oracle.store_copy(k, v, kc, vc, idx, st, w.H, w.D, 2, T,
                                k_off=w.k_view[0], v_off=w.v_view[0])
    elif w.notes.get("fmt") == "e5m2":
        assert w.page_stride == w.page_size * sb
        bad = oracle.store_fp8_ex(k, v, kc, vc, idx, st, w.H, w.D, w.src_dtype, w.page_size,
                                  w.page_stride, w.page_stride, T + (-T) % w.page_size,
                                  fmt="e5m2", scale_mode="tensor", inv_k=w.inv_k, inv_v=w.inv_v,
                                  k_off=w.k_view[0], v_off=w.v_view[0])
    else:
        # compact slot j sits at j * slot_stride for any page size when pages are dense
        assert w.page_stride == w.page_size * sb
        bad = oracle.store_fp8(k, v, kc, vc, idx, st, w.H, w.D, w.src_dtype, w.page_size,
                               w.page_stride, w.page_stride, T + (-T) % w.page_size,
                               w.inv_k, w.inv_v, w.use_scale,
                               k_off=w.k_view[0], v_off=w.v_view[0])
    assert bad == (0, -1)
    return kc.reshape(T, sb), vc.reshape(T, sb), sent


@pytest.mark.parametrize("name,split", [
    ("tiny", 0), ("decode", 0), ("decode", 1), ("decode", 2), ("decode", 4),
    ("prefill", 0), ("fp8", 0), ("fp8_noscale", 0), ("fp8_e5m2", 0), ("strided", 0), ("odd", 0),
])
def test_full_size_workload(name, split):
    import torch
    import bench
    import fp8_quant_gb300 as kv
    dev = torch.device("cuda", 0)
    pool = bench.Pool(name, dev, pool_bytes=0)
    w = pool.w
    w.num_split = split
    assert pool.num_batches == 1
    assert pool.call(0, torch.cuda.current_stream().cuda_stream) == 0
    st, nbad, first = kv.kv_error_poll(pool.err)
    assert (st, nbad, first) == (kv.KVStatus.OK, 0, -1)

    okc, ovc, sent = _oracle_compact(w)
    sb = w.slot_stride
    slots = torch.from_numpy(w.indices.astype(np.int64)).to(dev)
    for cache, want, what in ((pool.kc, okc, "K"), (pool.vc, ovc, "V")):
        rows = cache.view(torch.uint8).view(w.n_slots, sb).index_select(0, slots).cpu().numpy()
        if not np.array_equal(rows, want):
            bad = np.argwhere(rows != want)
            t, b = bad[0]
            raise AssertionError(f"{what} cache: {len(bad)} bytes differ; first token {t} "
                                 f"byte {b}: got {rows[t, b]:#04x} want {want[t, b]:#04x}")
        assert _rows_changed(torch, cache, w.n_slots, sb, sent) == w.T, f"{what}: stray rows"
    del pool
    torch.cuda.empty_cache()


def test_full_size_paged_copy():
    """The prefill batch into padded 4-D pages through kv_store_paged: the
    touched pages (pad bytes included) equal the oracle's, and no other page
    changed."""
    import torch
    import bench
    import fp8_quant_gb300 as kv
    dev = torch.device("cuda", 0)
    pool = bench.Pool("paged", dev, pool_bytes=0)
    w = pool.w
    assert w.paged and pool.num_batches == 1
    assert pool.call(0, torch.cuda.current_stream().cuda_stream) == 0
    assert kv.kv_error_poll(pool.err) == (kv.KVStatus.OK, 0, -1)
    ps, pstride = w.page_size, w.page_stride
    n_pages = w.cache_bytes // pstride
    slots = w.indices.astype(np.int64)
    pages = np.unique(slots // ps)
    compact = {int(p): j for j, p in enumerate(pages)}
    cidx = np.array([compact[int(s // ps)] * ps + int(s % ps) for s in slots], dtype=w.indices.dtype)
    sent = w.sentinel.to_bytes(2, "little")
    okc = np.frombuffer(sent * (len(pages) * pstride // 2), dtype=np.uint8).copy()
    ovc = okc.copy()
    st = oracle.Strides(k_token=w.k_view[1], k_head=w.k_view[2], k_dim=w.k_view[3],
                        v_token=w.v_view[1], v_head=w.v_view[2], v_dim=w.v_view[3],
                        kc_slot=w.slot_stride, kc_head=w.cache_head_stride, kc_dim=2,
                        vc_slot=w.slot_stride, vc_head=w.cache_head_stride, vc_dim=2)
    k = np.ascontiguousarray(w.k).view(np.uint8).reshape(-1)
    v = np.ascontiguousarray(w.v).view(np.uint8).reshape(-1)
    assert oracle.store_copy_paged(k, v, okc, ovc, cidx, st, w.H, w.D, 2, ps, pstride, pstride,
                                   len(pages) * ps) == (0, -1)
    sel = torch.from_numpy(pages).to(dev)
    pat = torch.tensor(list(sent) * (pstride // 2), dtype=torch.uint8, device=dev)
    for cache, want, what in ((pool.kc, okc, "K"), (pool.vc, ovc, "V")):
        view = cache.view(torch.uint8)[: n_pages * pstride].view(n_pages, pstride)
        got = view.index_select(0, sel).cpu().numpy().reshape(-1)
        assert np.array_equal(got, want), f"{what}: touched pages differ"
        changed = 0
        for p0 in range(0, n_pages, 2048):
            changed += int((view[p0:p0 + 2048] != pat).any(dim=1).sum().item())
        assert changed == len(pages), f"{what}: stray pages"
    del pool
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["fp8_dynamic", "fp8_dynamic_token"])
def test_full_size_dynamic_fp8(name):
    """The fp8 batch with scales computed in the kernel per (token, head) or
    per token row: every written row and scale equals the oracle's, nothing
    else changed."""
    import torch
    import bench
    import fp8_quant_gb300 as kv
    dev = torch.device("cuda", 0)
    pool = bench.Pool(name, dev, pool_bytes=0)
    w = pool.w
    assert not w.paged and pool.num_batches == 1
    assert pool.call(0, torch.cuda.current_stream().cuda_stream) == 0
    assert kv.kv_error_poll(pool.err) == (kv.KVStatus.OK, 0, -1)
    mode = w.notes.get("scale_mode", "token_head")
    T, H, sb = w.T, pool.groups, w.slot_stride
    idx = np.arange(T, dtype=w.indices.dtype)
    okc = np.full(T * sb, w.sentinel, np.uint8)
    ovc = okc.copy()
    oks = np.full(T * H, -1.0, np.float32)
    ovs = oks.copy()
    st = oracle.Strides(k_token=w.k_view[1], k_head=w.k_view[2], k_dim=w.k_view[3],
                        v_token=w.v_view[1], v_head=w.v_view[2], v_dim=w.v_view[3],
                        kc_slot=sb, kc_head=w.cache_head_stride, kc_dim=1,
                        vc_slot=sb, vc_head=w.cache_head_stride, vc_dim=1)
    k = np.ascontiguousarray(w.k).view(np.uint8).reshape(-1)
    v = np.ascontiguousarray(w.v).view(np.uint8).reshape(-1)
    assert w.page_stride == w.page_size * sb
    bad = oracle.store_fp8_ex(k, v, okc, ovc, idx, st, w.H, w.D, w.src_dtype, w.page_size,
                              w.page_stride, w.page_stride, T + (-T) % w.page_size,
                              fmt="e4m3fn", scale_mode=mode, k_scales=oks,
                              v_scales=ovs, scales_slot_stride=H)
    assert bad == (0, -1)
    slots = torch.from_numpy(w.indices.astype(np.int64)).to(dev)
    for cache, scales, want, wscale, what in ((pool.kc, pool.ks, okc, oks, "K"),
                                              (pool.vc, pool.vs, ovc, ovs, "V")):
        rows = cache.view(w.n_slots, sb).index_select(0, slots).cpu().numpy().reshape(-1)
        assert np.array_equal(rows, want), f"{what} cache rows differ"
        got_s = scales.view(w.n_slots, H).index_select(0, slots).cpu().numpy().reshape(-1)
        assert np.array_equal(got_s.view(np.uint32), wscale.view(np.uint32)), f"{what} scales"
        assert _rows_changed(torch, cache, w.n_slots, sb, bytes([w.sentinel])) == T
        assert int((scales != -1.0).sum().item()) == T * H
    del pool
    torch.cuda.empty_cache()


def test_full_size_per_page_scales():
    """The fp8 batch with one inverse scale per 32-slot page (32,768 pages):
    every written row equals the oracle's, nothing else changed.  The oracle
    runs on a compact cache (slot j for token j, pages of one slot) whose
    scale j is the scale of token j's real page, which leaves every code
    unchanged."""
    import torch
    import bench
    import fp8_quant_gb300 as kv
    dev = torch.device("cuda", 0)
    pool = bench.Pool("fp8_page", dev, pool_bytes=0)
    w = pool.w
    assert pool.num_batches == 1 and w.page_stride == w.page_size * w.slot_stride
    assert pool.call(0, torch.cuda.current_stream().cuda_stream) == 0
    assert kv.kv_error_poll(pool.err) == (kv.KVStatus.OK, 0, -1)
    T, sb = w.T, w.slot_stride
    idx = np.arange(T, dtype=w.indices.dtype)
    page = w.indices.astype(np.int64) // w.page_size
    ck = w.notes["page_inv_k"][page].copy()
    cv = w.notes["page_inv_v"][page].copy()
    okc = np.full(T * sb, w.sentinel, np.uint8)
    ovc = okc.copy()
    st = oracle.Strides(k_token=w.k_view[1], k_head=w.k_view[2], k_dim=w.k_view[3],
                        v_token=w.v_view[1], v_head=w.v_view[2], v_dim=w.v_view[3],
                        kc_slot=sb, kc_head=w.cache_head_stride, kc_dim=1,
                        vc_slot=sb, vc_head=w.cache_head_stride, vc_dim=1)
    k = np.ascontiguousarray(w.k).view(np.uint8).reshape(-1)
    v = np.ascontiguousarray(w.v).view(np.uint8).reshape(-1)
    assert oracle.store_fp8_ex(k, v, okc, ovc, idx, st, w.H, w.D, w.src_dtype, 1, sb, sb, T,
                               fmt="e4m3fn", scale_mode="page", k_scales=ck,
                               v_scales=cv) == (0, -1)
    slots = torch.from_numpy(w.indices.astype(np.int64)).to(dev)
    for cache, want, what in ((pool.kc, okc, "K"), (pool.vc, ovc, "V")):
        rows = cache.view(w.n_slots, sb).index_select(0, slots).cpu().numpy().reshape(-1)
        assert np.array_equal(rows, want), f"{what} cache rows differ"
        assert _rows_changed(torch, cache, w.n_slots, sb, bytes([w.sentinel])) == T
    del pool
    torch.cuda.empty_cache()


def test_full_size_fused_dynamic_tensor_write():
    """The fused dynamic per-tensor write on the fp8 batch at full size,
    through bench.Pool.call (the launch the bench times), twice in a row on
    the pool's one workspace: every written row equals the oracle's (absmax,
    inverse scale, per-tensor write), the forward scales are amax / 448 bit
    for bit, nothing else changed."""
    import torch
    import bench
    import fp8_quant_gb300 as kv
    dev = torch.device("cuda", 0)
    pool = bench.Pool("fp8_tensor_dynamic", dev, pool_bytes=0)
    w = pool.w
    assert pool.num_batches == 1
    s = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        assert pool.call(0, s) == 0
    assert kv.kv_error_poll(pool.err) == (kv.KVStatus.OK, 0, -1)
    assert int(pool.dyn_work.cpu()[0]) == 2
    T, sb = w.T, w.slot_stride
    st = oracle.Strides(k_token=w.k_view[1], k_head=w.k_view[2], k_dim=w.k_view[3],
                        v_token=w.v_view[1], v_head=w.v_view[2], v_dim=w.v_view[3],
                        kc_slot=sb, kc_head=w.cache_head_stride, kc_dim=1,
                        vc_slot=sb, vc_head=w.cache_head_stride, vc_dim=1)
    k = np.ascontiguousarray(w.k).view(np.uint8).reshape(-1)
    v = np.ascontiguousarray(w.v).view(np.uint8).reshape(-1)
    amax, inv = oracle.absmax_inv(k, v, st, T, w.H, w.D, w.src_dtype, 448.0)
    idx = np.arange(T, dtype=w.indices.dtype)          # compact oracle cache: slot j for token j
    okc = np.full(T * sb, w.sentinel, np.uint8)
    ovc = okc.copy()
    assert oracle.store_fp8_ex(k, v, okc, ovc, idx, st, w.H, w.D, w.src_dtype, 1, sb, sb, T,
                               fmt="e4m3fn", scale_mode="tensor", inv_k=float(inv[0]),
                               inv_v=float(inv[1])) == (0, -1)
    slots = torch.from_numpy(w.indices.astype(np.int64)).to(dev)
    for cache, want, what in ((pool.kc, okc, "K"), (pool.vc, ovc, "V")):
        rows = cache.view(w.n_slots, sb).index_select(0, slots).cpu().numpy().reshape(-1)
        assert np.array_equal(rows, want), f"{what} cache rows differ"
        assert _rows_changed(torch, cache, w.n_slots, sb, bytes([w.sentinel])) == T
    assert np.array_equal(pool.dyn_scale.cpu().numpy(), (amax / np.float32(448.0)).astype(np.float32))
    del pool
    torch.cuda.empty_cache()
