"""GPU parity of the scale preparation (kv_inv_scale, kv_absmax_inv) against
the CPU oracle, bit for bit, and of the two-pass dynamic per-tensor FP8 write
(kv_absmax_inv then kv_store_fp8 with the device-computed inverse scales)."""

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


def _stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def test_inv_scale_bits():
    import torch
    import fp8_quant_gb300 as kv
    x = np.concatenate([wl.normal(11, 5000) * np.float32(50),
                        np.array([1.0, 3.0, 448.0, 1e-38, 3e-39, 1e38, -7.5, 0.1], np.float32)])
    x = x[x != 0].astype(np.float32)
    d = torch.from_numpy(x).cuda()
    out = torch.empty_like(d)
    assert kv.raw.kv_inv_scale(d.data_ptr(), out.data_ptr(), x.size, _stream()) == 0
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), oracle.inv_scale(x).view(np.uint32))
    # in place, and n = 0
    assert kv.raw.kv_inv_scale(d.data_ptr(), d.data_ptr(), x.size, _stream()) == 0
    assert np.array_equal(d.cpu().numpy().view(np.uint32), got.view(np.uint32))
    assert kv.raw.kv_inv_scale(None, None, 0, _stream()) == 0


def _absmax_case(T, H, D, src, seed, head_pad=0, nan_at=(), inf_at=(), zero=False, fp8_max=448.0,
                 host=False):
    import torch
    import fp8_quant_gb300 as kv
    w = wl.make_fp8("t", T, H, D, max(T, 64), seed=seed, dtype=src)
    kb, vb = w.k.copy(), w.v.copy()
    if zero:
        kb[:] = 0
        vb[:] = 0x8000            # -0.0
    nan = 0x7FC0 if src == "bf16" else 0x7E00
    inf = 0x7F80 if src == "bf16" else 0x7C00
    for i in nan_at:
        kb.reshape(-1)[i] = nan
    for i in inf_at:
        vb.reshape(-1)[i] = inf | 0x8000
    e = 2
    hs = D * e + head_pad
    tok = H * hs
    buf = np.zeros((2, T * tok), np.uint8)
    for j, bits in enumerate((kb, vb)):
        rows = buf[j].reshape(T, H, hs)
        rows[:, :, :D * e] = bits.reshape(T, H, D).view(np.uint8).reshape(T, H, D * e)
    st = oracle.Strides(k_token=tok, k_head=hs, k_dim=e, v_token=tok, v_head=hs, v_dim=e,
                        kc_slot=0, kc_head=0, kc_dim=0, vc_slot=0, vc_head=0, vc_dim=0)
    want_amax, want_inv = oracle.absmax_inv(buf[0].copy(), buf[1].copy(), st, T, H, D, src,
                                            fp8_max)
    dbuf = torch.from_numpy(buf).pin_memory() if host else torch.from_numpy(buf).cuda()
    # without a workspace (three kernels) and with one (two kernels; the
    # workspace is zero before the call and zero again after it)
    work = torch.zeros(2, dtype=torch.int32, device="cuda")
    for use_work in (False, True):
        out = torch.full((4,), 123.0, dtype=torch.float32, device="cuda")
        rc = kv.raw.kv_absmax_inv(dbuf[0].data_ptr(), dbuf[1].data_ptr(),
                                  1 if src == "bf16" else 0, T, H, D,
                                  tuple(int(x) for x in st.values), fp8_max, out.data_ptr(),
                                  out.data_ptr() + 8, work.data_ptr() if use_work else None,
                                  _stream())
        assert rc == 0, kv.kv_status_str(rc)
        got = out.cpu().numpy()
        assert np.array_equal(got[:2].view(np.uint32), want_amax.view(np.uint32)), (got, want_amax)
        assert np.array_equal(got[2:].view(np.uint32), want_inv.view(np.uint32)), (got, want_inv)
        assert work.cpu().tolist() == [0, 0]
    return w, got


@pytest.mark.parametrize("src", ["bf16", "f16"])
@pytest.mark.parametrize("shape", [(8192, 8, 128), (1, 8, 128), (777, 1, 576), (300, 3, 40),
                                   (129, 2, 7)])
def test_absmax_inv_bits(src, shape):
    T, H, D = shape
    _absmax_case(T, H, D, src, seed=T + H + D)


def test_absmax_inv_special_values():
    _absmax_case(500, 8, 128, "bf16", seed=3, nan_at=(0, 5, 9999), head_pad=64)
    _absmax_case(500, 8, 128, "f16", seed=4, inf_at=(77,))
    _, got = _absmax_case(64, 4, 64, "bf16", seed=5, zero=True)
    assert list(got) == [0.0, 0.0, 1.0, 1.0]
    _absmax_case(1000, 8, 128, "bf16", seed=6, fp8_max=57344.0)


def test_absmax_inv_host_rows():
    """Rows in pinned host memory are read in place (no L2 prefetch of host
    memory); pageable host memory is rejected before any launch."""
    import torch
    import fp8_quant_gb300 as kv
    _absmax_case(3000, 8, 128, "bf16", seed=7, host=True)
    _absmax_case(300, 3, 40, "f16", seed=8, host=True)
    rows = np.zeros(2 * 64 * 256, np.uint8)
    out = torch.full((4,), 123.0, dtype=torch.float32, device="cuda")
    st = (256, 128, 2, 256, 128, 2) + (0,) * 6
    rc = kv.raw.kv_absmax_inv(rows.ctypes.data, rows.ctypes.data + 64 * 256, 1, 64, 2, 64, st,
                              448.0, out.data_ptr(), out.data_ptr() + 8, None, _stream())
    assert rc == kv.KVStatus.ERR_INVALID_ARG
    assert out.cpu().tolist() == [123.0] * 4


def test_fp8_workload_recipe_on_device():
    """The fp8 workload's host recipe inv = 448/amax is what the device computes."""
    w, got = _absmax_case(8192, 8, 128, "bf16", seed=0x5EED0003 * 8 % 100000)
    assert got[2] == np.float32(w.inv_k) and got[3] == np.float32(w.inv_v)


def test_two_pass_dynamic_per_tensor_write():
    """kv_absmax_inv then kv_store_fp8 reading the device inv: byte-equal to the
    oracle's absmax_inv then store_fp8."""
    import torch
    import fp8_quant_gb300 as kv
    T, H, D, n, ps = 2048, 8, 128, 8192, 16
    w = wl.make_fp8("dyn", T, H, D, n, seed=44, page_size=ps)
    dev = torch.device("cuda")
    k = torch.from_numpy(w.k.view(np.int16)).to(dev).view(torch.bfloat16)
    v = torch.from_numpy(w.v.view(np.int16)).to(dev).view(torch.bfloat16)
    idx = torch.from_numpy(w.indices).to(dev)
    kc = torch.full((n, H, D), 0x7F, dtype=torch.uint8, device=dev)
    vc = kc.clone()
    scal = torch.empty(4, dtype=torch.float32, device=dev)
    R = H * D * 2
    strides = (R, D * 2, 2, R, D * 2, 2, H * D, D, 1, H * D, D, 1)
    work = torch.zeros(2, dtype=torch.int32, device=dev)
    assert kv.raw.kv_absmax_inv(k.data_ptr(), v.data_ptr(), 1, T, H, D, strides, 448.0,
                                scal.data_ptr(), scal.data_ptr() + 8, work.data_ptr(),
                                _stream()) == 0
    kv.kv_store_fp8(k, v, kc, vc, idx, page_size=ps, inv_k_scale=scal[2:3],
                    inv_v_scale=scal[3:4])
    st = oracle.Strides(k_token=R, k_head=D * 2, k_dim=2, v_token=R, v_head=D * 2, v_dim=2,
                        kc_slot=H * D, kc_head=D, kc_dim=1, vc_slot=H * D, vc_head=D, vc_dim=1)
    _, inv = oracle.absmax_inv(w.k, w.v, st, T, H, D, "bf16")
    okc = np.full(n * H * D, 0x7F, np.uint8)
    ovc = okc.copy()
    oracle.store_fp8(w.k, w.v, okc, ovc, w.indices, st, H, D, "bf16", ps, ps * H * D, ps * H * D,
                     n, float(inv[0]), float(inv[1]), 1)
    assert np.array_equal(kc.cpu().numpy().ravel(), okc)
    assert np.array_equal(vc.cpu().numpy().ravel(), ovc)


def test_scale_argument_errors():
    import fp8_quant_gb300 as kv
    s = _stream()
    z = (0,) * 12
    assert kv.raw.kv_inv_scale(None, None, -1, s) == kv.KVStatus.ERR_INVALID_ARG
    assert kv.raw.kv_inv_scale(0x1002, 0x2000, 4, s) == kv.KVStatus.ERR_INVALID_ARG
    st = (256, 128, 2, 256, 128, 2) + (0,) * 6
    assert kv.raw.kv_absmax_inv(0x1000, 0x1000, 1, 4, 2, 64, st, 0.0, 0x3000, 0x3008, None,
                                s) == kv.KVStatus.ERR_INVALID_ARG
    assert kv.raw.kv_absmax_inv(0x1000, 0x1000, 1, 4, 2, 64, st[:2] + (4,) + st[3:], 448.0,
                                0x3000, 0x3008, None, s) == kv.KVStatus.ERR_UNSUPPORTED
    assert kv.raw.kv_absmax_inv(0x1000, 0x1000, 5, 4, 2, 64, z, 448.0, 0x3000, 0x3008, None,
                                s) == kv.KVStatus.ERR_INVALID_ARG
    assert kv.raw.kv_absmax_inv(0x1000, 0x1000, 1, 4, 2, 64, st, 448.0, 0x3000, 0x3008, 0x4002,
                                s) == kv.KVStatus.ERR_INVALID_ARG


def test_absmax_workspace_back_to_back_calls():
    """Calls sharing one workspace on a stream, back to back and from a CUDA
    graph: each call's result is its own tensors' (no maximum carried over from
    the previous call, whose values are larger), and the workspace ends zero."""
    import torch
    import fp8_quant_gb300 as kv
    dev = torch.device("cuda")
    T, H, D = 3000, 8, 128
    xs = [torch.randn(T, H, D, device=dev).to(torch.bfloat16) * (8.0 / (i + 1)) for i in range(4)]
    work = torch.zeros(2, dtype=torch.int32, device=dev)
    outs = [torch.zeros(4, dtype=torch.float32, device=dev) for _ in range(4)]
    R = H * D * 2
    strides = (R, D * 2, 2, R, D * 2, 2) + (0,) * 6
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(4):
            assert kv.raw.kv_absmax_inv(xs[i].data_ptr(), xs[3 - i].data_ptr(), 1, T, H, D,
                                        strides, 448.0, outs[i].data_ptr(),
                                        outs[i].data_ptr() + 8, work.data_ptr(),
                                        s.cuda_stream) == 0
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        for i in range(4):
            a = np.array([xs[i].float().abs().max().item(), xs[3 - i].float().abs().max().item()],
                         np.float32)
            got = outs[i].cpu().numpy()
            assert np.array_equal(got[:2], a) and np.array_equal(got[2:], np.float32(448.0) / a)
        assert work.cpu().tolist() == [0, 0]

