"""GPU parity: the CUDA library through its C ABI against the CPU oracle.

Every case compares every byte of both caches (pre-filled with a sentinel, so
stray writes show) and the out-of-range report. Sizes span many warps and
CTAs with ragged tails; the cases cover each kernel variant (16/8/4/2/1-byte
vectors, head-segmented rows, row splits, element-wise strided paths),
both index types, index strides, padded slots and pages, misaligned views,
out-of-range slots, empty calls, duplicates, and all 65,536 bf16 and fp16
input patterns of the FP8 conversion.
"""

import zlib

import numpy as np
import pytest

import workloads as wl
from kvcheck import Problem, View, DeviceRun, assert_same, copy_problem, fp8_problem, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()
    yield


# ---------------------------------------------------------------------------
# Plain copy
# ---------------------------------------------------------------------------

COPY_CASES = {
    # name: kwargs of copy_problem
    "tiny_cfg_shape": dict(T=16, H=2, D=64, n_slots=256, idx_dtype=np.int32),
    "decode_shape": dict(T=777, H=8, D=128, n_slots=4096),
    "split2": dict(T=301, H=8, D=128, n_slots=1024, num_split=2),
    "split4": dict(T=301, H=8, D=128, n_slots=1024, num_split=4, idx_dtype=np.int32),
    "split1": dict(T=301, H=8, D=128, n_slots=1024, num_split=1),
    "row1152_pad1280": dict(T=1000, H=1, D=576, n_slots=3000, slot_pad=128, idx_dtype=np.int32),
    "row4096_long": dict(T=90, H=16, D=128, n_slots=200),
    "row8192_multi_batch": dict(T=33, H=32, D=128, n_slots=100),
    "small_rows_h1_d8": dict(T=2049, H=1, D=8, n_slots=5000),
    "vec8_offset": dict(T=500, H=4, D=64, n_slots=1500, src_off=8, dst_off=8),
    "vec4_offset": dict(T=500, H=4, D=64, n_slots=1500, src_off=4),
    "vec2_offset": dict(T=500, H=4, D=64, n_slots=1500, dst_off=2),
    "vec1_bytes_odd": dict(T=300, H=3, D=7, n_slots=900, elem=1, src_off=1),
    "elem4_fp32": dict(T=400, H=2, D=96, n_slots=800, elem=4),
    "elem8": dict(T=200, H=2, D=20, n_slots=800, elem=8),
    "head_segments": dict(T=640, H=8, D=64, n_slots=2000, head_pad_src=32, head_pad_dst=64),
    "head_segments_odd_d": dict(T=333, H=5, D=80, n_slots=2000, head_pad_dst=16),
    "qkv_interleaved": dict(T=1024, H=8, D=128, n_slots=4096, qkv_shared=True),
    "token_pad_odd": dict(T=257, H=2, D=40, n_slots=700, token_pad=6),
    "dims_strided_generic": dict(T=200, H=4, D=32, n_slots=600, dim_stride_mult=2),
    "index_stride3_i32": dict(T=513, H=8, D=128, n_slots=2000, index_stride=3,
                              idx_dtype=np.int32),
    "single_token": dict(T=1, H=8, D=128, n_slots=8),
    # kv_store_paged: [pages, page_size, H, D] caches, dense and padded page strides
    "paged_dense_64": dict(T=700, H=8, D=128, n_slots=4096, page_size=64),
    "paged_padded_16": dict(T=700, H=8, D=128, n_slots=4096, page_size=16, page_pad=512),
    "paged_padded_odd_rows": dict(T=600, H=1, D=576, n_slots=2048, page_size=32, page_pad=128,
                                  slot_pad=128, idx_dtype=np.int32),
    "paged_page7_vec4": dict(T=400, H=2, D=40, n_slots=1000, page_size=7, page_pad=12),
    "paged_segments": dict(T=500, H=8, D=64, n_slots=2000, page_size=16, page_pad=64,
                           head_pad_dst=32),
    "paged_generic_dims": dict(T=200, H=4, D=32, n_slots=600, page_size=8, page_pad=32,
                               dim_stride_mult=2),
    "paged_split4": dict(T=300, H=8, D=128, n_slots=1024, page_size=32, page_pad=256,
                         num_split=4),
}


@pytest.mark.parametrize("name", sorted(COPY_CASES))
def test_copy_parity(name):
    kw = dict(COPY_CASES[name])
    p = copy_problem(seed=zlib.crc32(name.encode()) % 10000, **kw)
    assert_same(p)


@pytest.mark.parametrize("split", [0, 1, 2, 4])
def test_copy_split_invariance(split):
    p = copy_problem(T=256, H=8, D=128, n_slots=4096, seed=5, num_split=split)
    g = assert_same(p)
    if split:
        ref = assert_same(copy_problem(T=256, H=8, D=128, n_slots=4096, seed=5, num_split=0))
        a, b = g.caches(), ref.caches()
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_copy_out_of_range_slots():
    T, n = 600, 2000
    slots = wl.distinct_slots(77, n, T)
    bad_at = [3, 10, 11, 599]
    for i, val in zip(bad_at, [-1, n, 2 ** 62, -(2 ** 40)]):
        slots[i] = val
    p = copy_problem(T=T, H=8, D=128, n_slots=n, seed=78, slots=slots)
    g = assert_same(p)
    # the poll cleared the record
    rc, nbad, first = g.poll()
    assert (rc, nbad, first) == (0, 0, -1)


def test_copy_out_of_range_int32_extremes():
    T, n = 64, 128
    slots = wl.distinct_slots(79, n, T)
    slots[[0, 63]] = [np.iinfo(np.int32).min, np.iinfo(np.int32).max]
    p = copy_problem(T=T, H=2, D=64, n_slots=n, seed=80, slots=slots, idx_dtype=np.int32)
    assert_same(p)


def test_copy_size_limit_below_cache_rows():
    # slots in [size_limit, n) are out of range even though the cache has them
    p = copy_problem(T=300, H=2, D=64, n_slots=1000, seed=81, size_limit=500)
    assert_same(p)


def test_copy_size_limit_zero():
    p = copy_problem(T=50, H=2, D=64, n_slots=100, seed=82, size_limit=0)
    g = assert_same(p)
    kc, _ = g.caches()
    assert np.all(kc.view(np.uint16) == wl.BF16_SENTINEL)


def test_empty_calls_launch_nothing():
    import torch
    import fp8_quant_gb300 as kv
    s = torch.cuda.current_stream().cuda_stream
    zeros = (0,) * 12
    assert kv.raw.kv_store(None, None, None, None, None, 0, 1, 0, 8, 128, 2, zeros, 0, 0,
                           None, s) == 0
    assert kv.raw.kv_store_fp8(None, None, None, None, None, 0, 1, 0, 8, 128, 1, zeros, 1, 0, 0,
                               0, None, None, 0, None, s) == 0


def test_copy_duplicate_slots_take_a_candidate():
    """Duplicate slots: every element of the row equals that element of some
    candidate row (concurrent writes may mix candidates element by element)."""
    T, n, H, D = 512, 64, 4, 64
    slots = (wl.splitmix64(83, 0, T) % np.uint64(n)).astype(np.int64)
    p = copy_problem(T=T, H=H, D=D, n_slots=n, seed=84, slots=slots)
    g = DeviceRun(p)
    assert g.call() == 0
    kc, vc = g.caches()
    E = H * D
    for cache, src in ((kc, p.k_src), (vc, p.v_src)):
        rows = src[:T * E * 2].view(np.uint16).reshape(T, E)
        got = cache.view(np.uint16).reshape(n, E)
        for s in np.unique(slots):
            cands = rows[slots == s]
            assert np.all(np.any(cands == got[s][None, :], axis=0)), f"slot {s}"
    untouched = np.setdiff1d(np.arange(n), slots)
    assert np.all(kc.view(np.uint16).reshape(n, E)[untouched] == wl.BF16_SENTINEL)


def test_stream_order_with_preceding_kernels():
    """A torch kernel writes the indices right before the call; a second call
    overwrites the same slots. Both orderings must hold (programmatic launch
    waits for the preceding grid)."""
    import torch
    import fp8_quant_gb300 as kv
    T, H, D, n = 4096, 8, 128, 1 << 15
    dev = torch.device("cuda")
    k1 = torch.randn(T, H, D, device=dev, dtype=torch.bfloat16)
    k2 = torch.randn(T, H, D, device=dev, dtype=torch.bfloat16)
    kc = torch.zeros(n, H, D, device=dev, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    idx = torch.zeros(T, device=dev, dtype=torch.int64)
    err = kv.error_record(dev)
    perm = torch.randperm(n, device=dev)[:T]
    for _ in range(3):
        idx.zero_()
        idx.copy_(perm)                                   # producer kernel on the stream
        kv.kv_store(k1, k1, kc, vc, idx, err=err)
        kv.kv_store(k2, k1, kc, vc, idx, err=err)         # same slots, new K
    st, nbad, _ = kv.kv_error_poll(err)
    assert st == kv.KVStatus.OK and nbad == 0
    assert torch.equal(kc[perm], k2) and torch.equal(vc[perm], k1)


def test_graph_capture_replay():
    import torch
    import fp8_quant_gb300 as kv
    T, H, D, n = 1000, 8, 128, 8192
    dev = torch.device("cuda")
    k = torch.randn(T, H, D, device=dev, dtype=torch.bfloat16)
    kc = torch.zeros(n, H, D, device=dev, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    idx = torch.randperm(n, device=dev)[:T].to(torch.int32)
    err = kv.error_record(dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        kv.kv_store(k, k, kc, vc, idx, err=err)           # warm-up outside the graph
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kv.kv_store(k, k, kc, vc, idx, err=err)
    kc.zero_()
    vc.zero_()
    k.mul_(-1)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(kc[idx.long()], k) and torch.equal(vc[idx.long()], k)
    assert kv.kv_error_poll(err)[1] == 0


def test_tensor_binding_matches_raw():
    """The tensor-level binding (views, 2-D caches with padded slots) gives the
    oracle's bytes too."""
    import torch
    import fp8_quant_gb300 as kv
    T, H, D, n = 300, 1, 576, 1000
    p = copy_problem(T=T, H=H, D=D, n_slots=n, seed=85, slot_pad=128, idx_dtype=np.int32)
    okc, ovc, _ = run_oracle(p)
    dev = torch.device("cuda")
    k = torch.from_numpy(p.k_src[:T * 1152].copy()).to(dev).view(torch.float16).view(T, H, D)
    v = torch.from_numpy(p.v_src[:T * 1152].copy()).to(dev).view(torch.float16).view(T, H, D)
    kc_store = torch.from_numpy(np.full(n * 640, wl.BF16_SENTINEL, np.uint16).view(np.int16))
    kc_store = kc_store.to(dev).view(n, 640)
    vc_store = kc_store.clone()
    idx = torch.from_numpy(p.indices).to(dev)
    kv.kv_store(k, v, kc_store[:, :576].view(torch.float16), vc_store[:, :576].view(torch.float16),
                idx, num_heads=1, head_dim=576)
    assert np.array_equal(kc_store.cpu().numpy().view(np.uint8).ravel(), okc)
    assert np.array_equal(vc_store.cpu().numpy().view(np.uint8).ravel(), ovc)


# ---------------------------------------------------------------------------
# Fused FP8
# ---------------------------------------------------------------------------

FP8_CASES = {
    "cfg_shape_scaled": dict(T=1200, H=8, D=128, n_slots=4096, page_size=32),
    "cfg_shape_unscaled": dict(T=1200, H=8, D=128, n_slots=4096, page_size=32, use_scale=0),
    "fp16_scaled": dict(T=700, H=8, D=128, n_slots=2048, src_dtype="f16"),
    "fp16_unscaled": dict(T=700, H=4, D=64, n_slots=2048, src_dtype="f16", use_scale=0),
    "int32_index_stride2": dict(T=555, H=8, D=128, n_slots=2048, idx_dtype=np.int32,
                                index_stride=2),
    "padded_pages_4d": dict(T=900, H=8, D=128, n_slots=4096, page_size=64, page_pad=256),
    "page_size_one": dict(T=400, H=2, D=64, n_slots=1024, page_size=1),
    "odd_page_size": dict(T=400, H=2, D=64, n_slots=1000, page_size=7, page_pad=16),
    "segmented_heads": dict(T=500, H=8, D=64, n_slots=1500, head_pad_src=64, head_pad_dst=32),
    "out8_d24": dict(T=640, H=3, D=24, n_slots=1500),
    "out4_d20": dict(T=640, H=1, D=20, n_slots=1500),
    "out2_d6": dict(T=640, H=1, D=6, n_slots=1500),
    "misaligned_src": dict(T=300, H=4, D=64, n_slots=900, src_off=2),
    "slot_pad_8": dict(T=300, H=4, D=64, n_slots=900, slot_pad=8, page_size=4),
    "generic_odd_d": dict(T=300, H=3, D=45, n_slots=900),
    "generic_strided_dims": dict(T=300, H=2, D=32, n_slots=900, src_dim_mult=3,
                                 dst_dim_mult=2),
    "long_rows_d576": dict(T=200, H=1, D=576, n_slots=600),
    "many_heads_long": dict(T=64, H=64, D=128, n_slots=128),
    "single_token": dict(T=1, H=8, D=128, n_slots=16),
    # launches of at least 4096 warps: one warp writes the K and the V row of a token
    "paired_rows_parts2": dict(T=1111, H=8, D=128, n_slots=4096, page_size=32),
    "paired_pages_i32": dict(T=3000, H=8, D=128, n_slots=8192, page_size=16, page_pad=256,
                             idx_dtype=np.int32),
    "paired_heads_f16": dict(T=700, H=8, D=64, n_slots=2048, head_pad_src=64, head_pad_dst=32,
                             src_dtype="f16"),
    "paired_unscaled_odd_rows": dict(T=5000, H=1, D=576, n_slots=8192, use_scale=0),
}


@pytest.mark.parametrize("name", sorted(FP8_CASES))
def test_fp8_parity(name):
    p = fp8_problem(seed=zlib.crc32(name.encode()) % 10000, **FP8_CASES[name])
    assert_same(p)


def test_fp8_out_of_range():
    p = fp8_problem(T=300, H=8, D=128, n_slots=1000, seed=91, page_size=16)
    p.indices[[0, 5, 299]] = [-7, 1000, 2 ** 50]
    assert_same(p)


def test_fp8_out_of_range_paired():
    p = fp8_problem(T=3000, H=8, D=128, n_slots=8192, seed=94, page_size=16)
    p.indices[[0, 1500, 2999]] = [-1, 8192, 2 ** 40]
    assert_same(p)


def test_fp8_use_scale_off_equals_inv_one():
    a = DeviceRun(fp8_problem(T=512, H=8, D=128, n_slots=2048, seed=92, use_scale=0))
    b = DeviceRun(fp8_problem(T=512, H=8, D=128, n_slots=2048, seed=92, use_scale=1,
                           inv=(1.0, 1.0)))
    assert a.call() == 0 and b.call() == 0
    ka, va = a.caches()
    kb, vb = b.caches()
    assert np.array_equal(ka, kb) and np.array_equal(va, vb)


def _all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint16).reshape(64, 8, 128)
    return bits, bits[::-1].copy()


@pytest.mark.parametrize("src", ["bf16", "f16"])
@pytest.mark.parametrize("inv", [None, 1.0, 0.5, 3.0, 448.0 / 2.75, 2.0 ** -20, 1e30])
def test_fp8_exhaustive_input_patterns(src, inv):
    """All 65,536 input bit patterns (NaNs, infinities, subnormals included)
    through the conversion, unscaled and with several inverse scales."""
    kb, vb = _all_patterns()
    p = fp8_problem(T=64, H=8, D=128, n_slots=256, seed=93, src_dtype=src, src_bits=(kb, vb),
                    use_scale=0 if inv is None else 1,
                    inv=None if inv is None else (inv, inv))
    assert_same(p)


# ---------------------------------------------------------------------------
# Inputs in page-locked host memory (read by the kernels over NVLink-C2C)
# ---------------------------------------------------------------------------

def _pinned(a: np.ndarray):
    import torch
    return torch.from_numpy(a).pin_memory()


@pytest.mark.parametrize("kind", ["copy", "fp8"])
def test_pinned_host_inputs(kind):
    """K, V and the slot ids in pinned host memory, caches on the device: the
    same bytes as the oracle (the library reads the host buffers in place)."""
    import torch
    import fp8_quant_gb300 as kv
    if kind == "copy":
        p = copy_problem(T=700, H=8, D=128, n_slots=4096, seed=601)
    else:
        p = fp8_problem(T=700, H=8, D=128, n_slots=4096, seed=602, page_size=16)
    g = DeviceRun(p)
    hk, hv, hi = _pinned(p.k_src), _pinned(p.v_src), _pinned(p.indices)
    s = torch.cuda.current_stream().cuda_stream
    idt = 1 if p.indices.dtype == np.int64 else 0
    if kind == "copy":
        rc = kv.raw.kv_store(hk.data_ptr(), hv.data_ptr(), g.kc.data_ptr(), g.vc.data_ptr(),
                             hi.data_ptr(), idt, 1, p.T, p.H, p.D, 2, p.strides(), p.size_limit,
                             0, g.err.data_ptr(), s)
    else:
        rc = kv.raw.kv_store_fp8(hk.data_ptr(), hv.data_ptr(), g.kc.data_ptr(), g.vc.data_ptr(),
                                 hi.data_ptr(), idt, 1, p.T, p.H, p.D, 1, p.strides(), p.page_size,
                                 p.kc_page, p.vc_page, p.size_limit, g.inv.data_ptr(),
                                 g.inv.data_ptr() + 4, 1, g.err.data_ptr(), s)
    assert rc == 0, kv.kv_status_str(rc)
    assert g.poll()[:2] == (0, 0)
    kc, vc = g.caches()
    okc, ovc, _ = run_oracle(p)
    assert np.array_equal(kc, okc) and np.array_equal(vc, ovc)


def test_unregistered_host_memory_is_rejected():
    """Pageable host memory unknown to CUDA is an argument error, found before
    any launch."""
    import torch
    import fp8_quant_gb300 as kv
    p = copy_problem(T=64, H=2, D=64, n_slots=256, seed=603)
    g = DeviceRun(p)
    s = torch.cuda.current_stream().cuda_stream
    k_host = p.k_src.ctypes.data                      # plain numpy buffer
    rc = kv.raw.kv_store(k_host, g.v_src.data_ptr(), g.kc.data_ptr(), g.vc.data_ptr(),
                         g.idx.data_ptr(), 1, 1, p.T, p.H, p.D, 2, p.strides(), p.size_limit, 0,
                         g.err.data_ptr(), s)
    assert rc == kv.KVStatus.ERR_INVALID_ARG
    kc, _ = g.caches()
    assert np.all(kc.view(np.uint16) == wl.BF16_SENTINEL)


def test_error_snapshot_to_pinned_host_and_device():
    import torch
    import fp8_quant_gb300 as kv
    slots = wl.distinct_slots(611, 1000, 300)
    slots[[7, 9]] = [-1, 5000]
    p = copy_problem(T=300, H=2, D=64, n_slots=1000, seed=612, slots=slots)
    g = DeviceRun(p)
    assert g.call() == 0
    s = torch.cuda.current_stream().cuda_stream
    host = torch.zeros(2, dtype=torch.int64).pin_memory()
    dev = torch.zeros(2, dtype=torch.int64, device="cuda")
    assert kv.raw.kv_error_snapshot(g.err.data_ptr(), host.data_ptr(), s) == 0
    assert kv.raw.kv_error_snapshot(g.err.data_ptr(), dev.data_ptr(), s) == 0
    torch.cuda.synchronize()
    n, key = (int(x) for x in host.numpy().view(np.uint64))
    assert n == 2 and (~key & 0xFFFFFFFFFFFFFFFF) == 7
    assert torch.equal(dev.cpu(), host)
    assert g.poll()[:3] == (4, 2, 7)           # the snapshot left the record intact
    unregistered = np.zeros(2, np.int64)
    assert kv.raw.kv_error_snapshot(g.err.data_ptr(), unregistered.ctypes.data,
                                    s) == kv.KVStatus.ERR_INVALID_ARG


def test_concurrent_streams_disjoint_slots():
    """A copy and an FP8 write on two streams at once, into different caches
    with disjoint slots, each with its own error record: both equal the oracle."""
    import torch
    import fp8_quant_gb300 as kv
    pc = copy_problem(T=3000, H=8, D=128, n_slots=8192, seed=621)
    pf = fp8_problem(T=3000, H=8, D=128, n_slots=8192, seed=622, page_size=16)
    gc, gf = DeviceRun(pc), DeviceRun(pf)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(3):
        assert gc.call(stream=s1.cuda_stream) == 0
        assert gf.call(stream=s2.cuda_stream) == 0
    torch.cuda.synchronize()
    for g, p in ((gc, pc), (gf, pf)):
        kc, vc = g.caches()
        okc, ovc, _ = run_oracle(p)
        assert np.array_equal(kc, okc) and np.array_equal(vc, ovc)
        assert g.poll()[:2] == (0, 0)


def test_graph_of_dynamic_fp8_write_and_gather():
    """kv_store_fp8_ex (per-head dynamic scales) then kv_gather_fp8_ex captured
    in one CUDA graph and replayed on new data: equals the eager calls."""
    import torch
    import fp8_quant_gb300 as kv
    T, H, D, n, ps = 512, 8, 128, 4096, 16
    dev = torch.device("cuda")
    k = torch.randn(T, H, D, device=dev, dtype=torch.bfloat16)
    v = torch.randn(T, H, D, device=dev, dtype=torch.bfloat16)
    idx = torch.randperm(n, device=dev)[:T]
    kc = torch.zeros(n, H, D, dtype=torch.uint8, device=dev)
    vc = torch.zeros_like(kc)
    ks = torch.zeros(n, H, dtype=torch.float32, device=dev)
    vs = torch.zeros_like(ks)
    ko = torch.zeros(T, H, D, dtype=torch.bfloat16, device=dev)
    vo = torch.zeros_like(ko)
    err = kv.error_record(dev)
    R = H * D * 2
    st_in = (R, D * 2, 2, R, D * 2, 2, H * D, D, 1, H * D, D, 1)

    def step(stream):
        s = stream.cuda_stream
        assert kv.raw.kv_store_fp8_ex(k.data_ptr(), v.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                      idx.data_ptr(), 1, 1, T, H, D, 1, st_in, ps, ps * H * D,
                                      ps * H * D, n, 0, 3, None, None, ks.data_ptr(),
                                      vs.data_ptr(), H, err.data_ptr(), s) == 0
        assert kv.raw.kv_gather_fp8_ex(kc.data_ptr(), vc.data_ptr(), ko.data_ptr(), vo.data_ptr(),
                                       idx.data_ptr(), 1, 1, T, H, D, 1, st_in, ps, ps * H * D,
                                       ps * H * D, n, 0, 3, None, None, ks.data_ptr(),
                                       vs.data_ptr(), H, err.data_ptr(), s) == 0

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(side)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream())
    k.normal_()
    v.normal_()
    g.replay()
    torch.cuda.synchronize()
    got = (ko.clone(), vo.clone(), kc.clone(), ks.clone())
    step(torch.cuda.current_stream())            # eager on the same new data
    torch.cuda.synchronize()
    assert torch.equal(got[0], ko) and torch.equal(got[1], vo)
    assert torch.equal(got[2], kc) and torch.equal(got[3], ks)
    # and the dequantised rows are close to the inputs: half an e4m3fn step
    # (relative 2^-4 for normals, absolute 2^-10 of the head's scale for
    # subnormals) plus the bf16 rounding of the output
    x = k.float()
    sc = ks[idx][:, :, None]
    bound = x.abs() * (2 ** -4 + 2 ** -8) + sc * 2 ** -10 * 1.01
    assert bool(((ko.float() - x).abs() <= bound).all())
    assert kv.kv_error_poll(err)[1] == 0


def test_tensor_wrappers_round_trips():
    import torch
    import fp8_quant_gb300 as kv
    dev = torch.device("cuda")
    T, H, D, ps, pages = 300, 8, 128, 16, 64
    k = torch.randn(T, H, D, device=dev, dtype=torch.bfloat16)
    v = torch.randn(T, H, D, device=dev, dtype=torch.bfloat16)
    idx = torch.randperm(ps * pages, device=dev)[:T]
    # paged copy and paged gather give the rows back exactly
    big = torch.zeros(pages, ps * H * D + 256, dtype=torch.bfloat16, device=dev)
    kc = big[:, :ps * H * D].view(pages, ps, H, D)
    vc = torch.zeros_like(big)[:, :ps * H * D].view(pages, ps, H, D)
    kv.kv_store_paged(k, v, kc, vc, idx, page_size=ps)
    ko, vo = torch.empty_like(k), torch.empty_like(v)
    kv.kv_gather(kc, vc, ko, vo, idx, page_size=ps)
    assert torch.equal(ko, k) and torch.equal(vo, v)
    assert int((big[:, ps * H * D:] != 0).sum()) == 0          # page padding untouched
    # dynamic per-(token, head) e5m2 and back: within half an e5m2 step
    c8 = torch.zeros(pages * ps, H, D, dtype=torch.uint8, device=dev)
    c8v = torch.zeros_like(c8)
    ks = torch.zeros(pages * ps, H, dtype=torch.float32, device=dev)
    vs = torch.zeros_like(ks)
    kv.kv_store_fp8_ex(k, v, c8, c8v, idx, page_size=ps, fmt="e5m2", scale_mode="token_head",
                       k_scales=ks, v_scales=vs)
    kv.kv_gather_fp8(c8, c8v, ko, vo, idx, page_size=ps, fmt="e5m2", scale_mode="token_head",
                     k_scales=ks, v_scales=vs)
    x, sc = k.float(), ks[idx][:, :, None]
    assert bool(((ko.float() - x).abs() <= x.abs() * (2 ** -3 + 2 ** -8) + sc * 2 ** -17).all())
    # device absmax -> per-tensor write equals the host recipe's write
    s = kv.kv_absmax_inv(k, v)
    amax = torch.stack([k.float().abs().max(), v.float().abs().max()])
    assert torch.equal(s[:2], amax)
    assert torch.equal(s[2:], (torch.tensor(448.0, device=dev) / amax))
    inv = kv.kv_inv_scale(torch.tensor([2.0, 8.0], device=dev))
    assert inv.tolist() == [0.5, 0.125]
    assert kv.kv_error_poll()[1] == 0



@pytest.mark.parametrize("layout", ["3d_float_scales", "4d_tensor_scales", "4d_no_scale"])
def test_fused_fp8_set_kv_buffer_matches_oracle(layout):
    """The wrapper with the argument list of the fused FP8 write's page: float
    or device-tensor forward scales (reciprocal formed on the device) or none,
    [T, H*D] or [T, H, D] rows, 3-D or 4-D caches; every cache byte equals the
    oracle's write with fl32(1 / scale)."""
    import torch
    import fp8_quant_gb300 as kv
    import oracle
    dev = torch.device("cuda")
    T, H, D, ps, pages = 777, 8, 128, 16, 96
    seed = zlib.crc32(layout.encode()) % 10000
    kb = wl.f32_to_bf16_bits(wl.normal(seed, T * H * D) * 3.0).reshape(T, H, D)
    vb = wl.f32_to_bf16_bits(wl.normal(seed + 1, T * H * D) * 0.25).reshape(T, H, D)
    slots = wl.distinct_slots(seed, ps * pages, T).astype(np.int32)
    k = torch.from_numpy(kb.view(np.int16)).to(dev).view(torch.bfloat16)
    v = torch.from_numpy(vb.view(np.int16)).to(dev).view(torch.bfloat16)
    scales = (0.0234375, 0.00390625) if layout != "4d_no_scale" else (None, None)
    if layout == "3d_float_scales":
        shape = (ps * pages, H, D)
        k, v = k.reshape(T, H * D), v.reshape(T, H * D)
        ks, vs = scales
    else:
        shape = (pages, ps, H, D)
        ks, vs = (None, None) if scales[0] is None else (
            torch.tensor(scales[0], device=dev), torch.tensor(scales[1], device=dev))
    kc = torch.full(shape, 0x5A, dtype=torch.uint8, device=dev)
    vc = torch.full(shape, 0xA5, dtype=torch.uint8, device=dev)
    kv.fused_fp8_set_kv_buffer(k, v, kc, vc, torch.from_numpy(slots).to(dev), ks, vs,
                               page_size=ps)
    assert kv.kv_error_poll()[1] == 0
    R = H * D
    okc = np.full(ps * pages * R, 0x5A, np.uint8)
    ovc = np.full(ps * pages * R, 0xA5, np.uint8)
    st = oracle.Strides(k_token=2 * R, k_head=2 * D, k_dim=2, v_token=2 * R, v_head=2 * D,
                        v_dim=2, kc_slot=R, kc_head=D, kc_dim=1, vc_slot=R, vc_head=D, vc_dim=1)
    use = scales[0] is not None
    inv = oracle.inv_scale(scales) if use else (1.0, 1.0)
    bad, _ = oracle.store_fp8(kb, vb, okc, ovc, slots, st, H, D, "bf16", ps, ps * R, ps * R,
                              ps * pages, inv_k=inv[0], inv_v=inv[1], use_scale=int(use))
    assert bad == 0
    assert np.array_equal(kc.cpu().numpy().ravel(), okc)
    assert np.array_equal(vc.cpu().numpy().ravel(), ovc)



def test_fused_fp8_set_kv_buffer_on_a_side_stream():
    """Scales computed on a side stream and the wrapper called on that stream
    (the inverse scales are staged there too): the result equals the same
    call on the default stream, byte for byte."""
    import torch
    import fp8_quant_gb300 as kv
    dev = torch.device("cuda")
    T, H, D, ps, pages = 640, 8, 128, 16, 64
    kb = wl.f32_to_bf16_bits(wl.normal(901, T * H * D) * 2.0).reshape(T, H, D)
    k = torch.from_numpy(kb.view(np.int16)).to(dev).view(torch.bfloat16)
    v = (k.float() * 0.5).to(torch.bfloat16)
    idx = torch.from_numpy(wl.distinct_slots(902, ps * pages, T).astype(np.int64)).to(dev)
    caches = [torch.zeros(pages, ps, H, D, dtype=torch.uint8, device=dev) for _ in range(4)]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ks = k.float().abs().max() / 448.0          # produced on the side stream
        vs = v.float().abs().max() / 448.0
        kv.fused_fp8_set_kv_buffer(k, v, caches[0], caches[1], idx, ks, vs, page_size=ps,
                                   stream=s)
    torch.cuda.synchronize()
    kv.fused_fp8_set_kv_buffer(k, v, caches[2], caches[3], idx, ks, vs, page_size=ps)
    torch.cuda.synchronize()
    assert torch.equal(caches[0], caches[2]) and torch.equal(caches[1], caches[3])
    assert int((caches[0] != 0).sum()) > 0
    assert kv.kv_error_poll()[1] == 0

@pytest.mark.gpu
def test_launch_floor_runs_in_stream_order_and_in_a_graph():
    """kv_launch_floor (the measurement aid) launches, keeps stream order
    after a torch producer and replays from a CUDA graph; it writes nothing."""
    import torch
    import fp8_quant_gb300 as kv
    dev = torch.device("cuda", 0)
    x = torch.zeros(1 << 20, device=dev)
    st = torch.cuda.current_stream().cuda_stream
    x.fill_(3.0)
    assert kv.raw.kv_launch_floor(1024, st) == 0
    assert kv.raw.kv_launch_floor(1, st) == 0
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(8):
            assert kv.raw.kv_launch_floor(32768, s.cuda_stream) == 0
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert bool((x == 3.0).all())
