"""GPU parity of the fused dynamic per-tensor FP8 write
(kv_store_fp8_dynamic_tensor) against the CPU oracle's two steps: the
per-tensor absmax with its inverse scale, then the per-tensor FP8 write.
Every cache byte, the forward scales (amax / fmax, compared bit for bit) and
the out-of-range report are compared. Layouts: contiguous rows (one side per
warp and K/V paired), head-segmented rows, padded 4-D pages, strided cache
dims (the element kernel), narrow odd heads; both formats and source types;
out-of-range slots. Consecutive calls sharing one workspace (its generation
tag), also replayed from a CUDA graph; every 16-bit input pattern (NaN,
infinities); an all-zero batch (scale 1)."""

import zlib

import numpy as np
import pytest

import oracle
import workloads as wl
from kvcheck import SENT8, filled, fp8_problem

pytestmark = pytest.mark.gpu

FMTS = {"e4m3fn": 0, "e5m2": 1}
FMAX = {"e4m3fn": 448.0, "e5m2": 57344.0}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    yield


def expected(p, fmt):
    """The oracle: absmax -> inverse scale -> per-tensor write; returns the
    caches, the forward scales and the out-of-range report."""
    st = oracle.Strides(**dict(zip(oracle.Strides.FIELDS, p.strides())))
    amax, inv = oracle.absmax_inv(p.k_src, p.v_src, st, p.T, p.H, p.D, p.src_dtype, FMAX[fmt],
                                  k_off=p.k_view.offset, v_off=p.v_view.offset)
    okc = filled(p.cache_bytes, SENT8)
    ovc = okc.copy()
    res = oracle.store_fp8_ex(p.k_src, p.v_src, okc, ovc, p.indices, st, p.H, p.D, p.src_dtype,
                              p.page_size, p.kc_page, p.vc_page, p.size_limit, fmt=fmt,
                              scale_mode="tensor", inv_k=float(inv[0]), inv_v=float(inv[1]),
                              k_off=p.k_view.offset, v_off=p.v_view.offset,
                              index_stride=p.index_stride, t_end=p.T)
    fmax = np.float32(FMAX[fmt])
    scale = np.where(amax > 0, amax / fmax, np.float32(1.0)).astype(np.float32)
    return okc, ovc, scale, res


class Dev:
    """A problem's buffers on the device, for one or more calls."""

    def __init__(self, p):
        import torch
        dev = torch.device("cuda")
        self.p = p
        self.k = torch.from_numpy(p.k_src).to(dev)
        self.v = torch.from_numpy(p.v_src).to(dev)
        self.idx = torch.from_numpy(p.indices).to(dev)
        self.kc = torch.from_numpy(filled(p.cache_bytes, SENT8)).to(dev)
        self.vc = self.kc.clone()
        self.scale = torch.full((2,), -1.0, dtype=torch.float32, device=dev)
        self.err = torch.zeros(2, dtype=torch.int64, device=dev)

    def call(self, fmt, work, stream=None):
        import torch
        import fp8_quant_gb300 as kv
        p = self.p
        s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
        return kv.raw.kv_store_fp8_dynamic_tensor(
            self.k.data_ptr() + p.k_view.offset, self.v.data_ptr() + p.v_view.offset,
            self.kc.data_ptr(), self.vc.data_ptr(), self.idx.data_ptr(),
            1 if p.indices.dtype == np.int64 else 0, p.index_stride, p.T, p.H, p.D,
            1 if p.src_dtype == "bf16" else 0, p.strides(), p.page_size, p.kc_page, p.vc_page,
            p.size_limit, FMTS[fmt], self.scale.data_ptr(), self.scale.data_ptr() + 4,
            work.data_ptr(), self.err.data_ptr(), s)

    def check(self, fmt):
        import fp8_quant_gb300 as kv
        import torch
        okc, ovc, scale, res = expected(self.p, fmt)
        s = torch.cuda.current_stream().cuda_stream
        prc, pn, pfirst = kv.raw.kv_error_poll(self.err.data_ptr(), s)
        for got, want, what in ((self.kc, okc, "K"), (self.vc, ovc, "V")):
            g = got.cpu().numpy()
            if not np.array_equal(g, want):
                b = np.flatnonzero(g != want)
                raise AssertionError(f"{what} cache: {b.size} bytes differ, first {b[0]}: "
                                     f"got {g[b[0]]:#04x} want {want[b[0]]:#04x}")
        got_scale = self.scale.cpu().numpy()
        assert np.array_equal(got_scale.view(np.uint32), scale.view(np.uint32)), (got_scale, scale)
        assert (pn, pfirst) == res and prc == (4 if res[0] else 0)


def new_work():
    import torch
    import fp8_quant_gb300 as kv
    return torch.zeros(kv.DYNAMIC_TENSOR_WORK_BYTES // 8, dtype=torch.int64,
                       device=torch.device("cuda"))


CASES = {
    "rows_1024": dict(T=700, H=8, D=128, n_slots=2048, page_size=32),
    "paired_pages": dict(T=2500, H=8, D=128, n_slots=8192, page_size=16, page_pad=256),
    "segmented_heads": dict(T=400, H=8, D=64, n_slots=1024, head_pad_src=64, head_pad_dst=32),
    "strided_cache_dims": dict(T=300, H=4, D=32, n_slots=1024, dst_dim_mult=2),
    "odd_d_narrow_i32": dict(T=300, H=3, D=45, n_slots=1024, idx_dtype=np.int32, index_stride=2),
    "single_head_576": dict(T=256, H=1, D=576, n_slots=1024),
    # 32-byte rows, many of them
    "tiny_rows_many": dict(T=100000, H=1, D=16, n_slots=200000),
    # a batch beyond L2 (82 MB): the write's second read comes from HBM
    "large_batch": dict(T=20000, H=8, D=128, n_slots=32768, page_size=16),
}


@pytest.mark.parametrize("src", ["bf16", "f16"])
@pytest.mark.parametrize("fmt", sorted(FMTS))
@pytest.mark.parametrize("case", sorted(CASES))
def test_dynamic_tensor_parity(case, fmt, src):
    p = fp8_problem(seed=zlib.crc32((case + fmt + src).encode()) % 9999, src_dtype=src,
                    **CASES[case])
    d = Dev(p)
    assert d.call(fmt, new_work()) == 0
    d.check(fmt)


def test_dynamic_tensor_out_of_range_slots():
    """Bad slots skip their rows, are reported, and do not drop their rows
    from the maxima (those cover the whole batch)."""
    p = fp8_problem(T=3000, H=8, D=128, n_slots=8192, seed=515, page_size=16)
    p.indices[[0, 1234, 2999]] = [-1, 8192, 2 ** 40]
    d = Dev(p)
    assert d.call("e4m3fn", new_work()) == 0
    d.check("e4m3fn")


@pytest.mark.parametrize("src", ["bf16", "f16"])
@pytest.mark.parametrize("fmt", sorted(FMTS))
def test_dynamic_tensor_every_input_pattern(src, fmt):
    """All 65,536 16-bit patterns: the maxima meet infinities (inverse scale
    0) and ignore NaNs."""
    bits = np.arange(1 << 16, dtype=np.uint16)
    kb = bits.reshape(64, 8, 128)
    vb = bits[::-1].copy().reshape(64, 8, 128)
    p = fp8_problem(T=64, H=8, D=128, n_slots=256, seed=516, src_dtype=src, src_bits=(kb, vb))
    d = Dev(p)
    assert d.call(fmt, new_work()) == 0
    d.check(fmt)


def test_dynamic_tensor_finite_patterns_and_zero_batch():
    """Every finite bf16 pattern (no infinity, no NaN: a real inverse scale),
    and an all-zero batch (amax 0: inverse scale and stored scale 1)."""
    bits = np.arange(1 << 16, dtype=np.uint16)
    finite = bits[(bits & 0x7F80) != 0x7F80]
    rep = -(-64 * 8 * 128 // finite.size)
    kb = np.tile(finite, rep)[:64 * 8 * 128].reshape(64, 8, 128)
    vb = np.zeros_like(kb)
    p = fp8_problem(T=64, H=8, D=128, n_slots=256, seed=517, src_bits=(kb, vb))
    d = Dev(p)
    assert d.call("e4m3fn", new_work()) == 0
    d.check("e4m3fn")
    assert d.scale.cpu().numpy()[1] == 1.0


def _batches(n, T=2500, H=8, D=128):
    """n problems of one shape whose magnitudes differ by powers of 4, so a
    maximum left over from another call would change every code."""
    out = []
    for i in range(n):
        p = fp8_problem(T=T, H=H, D=D, n_slots=8192, seed=600 + i, page_size=16,
                        scale=4.0 * 4.0 ** (-i if i % 2 else i), outlier_frac=0.0)
        out.append(p)
    return out


def test_dynamic_tensor_consecutive_calls_share_a_workspace():
    """Calls on one stream share one workspace: large, small, large, small
    batches, each equal to its own oracle result (the generation tag makes a
    later call's maxima win without a clearing pass)."""
    work = new_work()
    for i, p in enumerate(_batches(4)):
        d = Dev(p)
        assert d.call("e4m3fn", work) == 0
        d.check("e4m3fn")
    import torch
    torch.cuda.synchronize()
    assert int(work.cpu()[0]) == 4          # one generation per call


def test_dynamic_tensor_from_a_cuda_graph():
    """Three calls on different batches captured into a CUDA graph and
    replayed twice: every replay leaves each call's caches and scales equal
    to its oracle result, and the workspace advances one generation per call."""
    import torch
    work = new_work()
    ds = [Dev(p) for p in _batches(3)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for d in ds:
            assert d.call("e5m2", work, stream=s.cuda_stream) == 0
    torch.cuda.current_stream().wait_stream(s)
    for rep in range(2):
        for d in ds:
            d.kc.fill_(SENT8[0])
            d.vc.fill_(SENT8[0])
            d.scale.fill_(-1.0)
        g.replay()
        torch.cuda.synchronize()
        for d in ds:
            d.check("e5m2")
    assert int(work.cpu()[0]) == 6


def test_dynamic_tensor_empty_batch_and_rejections():
    """num_tokens == 0 launches nothing and writes nothing; a workspace or a
    scale in host memory is rejected before anything runs."""
    import torch
    import fp8_quant_gb300 as kv
    p = fp8_problem(T=64, H=8, D=128, n_slots=256, seed=518)
    d = Dev(p)
    work = new_work()
    s = torch.cuda.current_stream().cuda_stream
    rc = kv.raw.kv_store_fp8_dynamic_tensor(
        d.k.data_ptr(), d.v.data_ptr(), d.kc.data_ptr(), d.vc.data_ptr(), d.idx.data_ptr(), 1, 1,
        0, p.H, p.D, 1, p.strides(), p.page_size, p.kc_page, p.vc_page, p.size_limit, 0,
        d.scale.data_ptr(), d.scale.data_ptr() + 4, work.data_ptr(), d.err.data_ptr(), s)
    assert rc == 0
    torch.cuda.synchronize()
    assert bool((d.scale == -1.0).all()) and int(work.abs().sum()) == 0
    host_work = torch.zeros(3, dtype=torch.int64).pin_memory()
    assert d.call("e4m3fn", host_work) == kv.KVStatus.ERR_INVALID_ARG
    host_scale = torch.zeros(2, dtype=torch.float32).pin_memory()
    rc = kv.raw.kv_store_fp8_dynamic_tensor(
        d.k.data_ptr(), d.v.data_ptr(), d.kc.data_ptr(), d.vc.data_ptr(), d.idx.data_ptr(), 1, 1,
        p.T, p.H, p.D, 1, p.strides(), p.page_size, p.kc_page, p.vc_page, p.size_limit, 0,
        host_scale.data_ptr(), host_scale.data_ptr() + 4, work.data_ptr(), d.err.data_ptr(), s)
    assert rc == kv.KVStatus.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(work.abs().sum()) == 0        # nothing ran


def test_dynamic_tensor_tensor_wrapper():
    """The binding's wrapper: [T, H, D] rows into a 4-D paged cache, scales
    returned; equal to the raw call's result."""
    import torch
    import fp8_quant_gb300 as kv
    dev = torch.device("cuda")
    T, H, D, ps, pages = 512, 8, 128, 16, 64
    kb = wl.f32_to_bf16_bits(wl.normal(77, T * H * D) * 3.0).reshape(T, H, D)
    vb = wl.f32_to_bf16_bits(wl.normal(78, T * H * D) * 0.5).reshape(T, H, D)
    slots = wl.distinct_slots(79, ps * pages, T)
    k = torch.from_numpy(kb.view(np.int16)).to(dev).view(torch.bfloat16)
    v = torch.from_numpy(vb.view(np.int16)).to(dev).view(torch.bfloat16)
    kc = torch.full((pages, ps, H, D), SENT8[0], dtype=torch.uint8, device=dev)
    vc = kc.clone()
    sc = kv.kv_store_fp8_dynamic_tensor(k, v, kc, vc, torch.from_numpy(slots).to(dev),
                                        page_size=ps)
    assert kv.kv_error_poll()[1] == 0
    R = H * D
    st = oracle.Strides(k_token=2 * R, k_head=2 * D, k_dim=2, v_token=2 * R, v_head=2 * D,
                        v_dim=2, kc_slot=R, kc_head=D, kc_dim=1, vc_slot=R, vc_head=D, vc_dim=1)
    amax, inv = oracle.absmax_inv(kb, vb, st, T, H, D, "bf16", 448.0)
    okc = np.full(ps * pages * R, SENT8[0], np.uint8)
    ovc = okc.copy()
    oracle.store_fp8_ex(kb, vb, okc, ovc, slots, st, H, D, "bf16", ps, ps * R, ps * R, ps * pages,
                        fmt="e4m3fn", scale_mode="tensor", inv_k=float(inv[0]),
                        inv_v=float(inv[1]), t_end=T)
    assert np.array_equal(kc.cpu().numpy().ravel(), okc)
    assert np.array_equal(vc.cpu().numpy().ravel(), ovc)
    assert np.array_equal(sc.cpu().numpy(), (amax / np.float32(448.0)).astype(np.float32))


def test_dynamic_tensor_concurrent_streams_separate_workspaces():
    """Two streams, each with its own workspace and batch, write at the same
    time (no synchronisation between them): both results equal their oracle
    results, and each workspace advances by its own calls only."""
    import torch
    ps = _batches(2)
    ds = [Dev(p) for p in ps]
    works = [new_work(), new_work()]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for rep in range(3):
        for d, w, s in zip(ds, works, streams):
            with torch.cuda.stream(s):
                assert d.call("e4m3fn", w, stream=s.cuda_stream) == 0
    torch.cuda.synchronize()
    for d in ds:
        d.check("e4m3fn")
    assert [int(w.cpu()[0]) for w in works] == [3, 3]
