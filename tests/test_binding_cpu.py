"""CPU checks of the tensor-level binding: the byte strides, shapes and flags
it passes to the C ABI for each supported tensor layout (the raw calls are
intercepted, so no GPU is needed)."""

import pytest
import torch

import fp8_quant_gb300 as kv


class Capture:
    def __init__(self, monkeypatch):
        self.calls = []
        monkeypatch.setattr(kv.raw, "kv_store", self._store)
        monkeypatch.setattr(kv.raw, "kv_store_fp8", self._store8)
        monkeypatch.setattr(kv, "_stream_handle", lambda stream, device: 1234)
        monkeypatch.setattr(kv, "_default_record", lambda device: torch.zeros(2, dtype=torch.int64))

    def _store(self, *a):
        self.calls.append(("kv_store", a))
        return 0

    def _store8(self, *a):
        self.calls.append(("kv_store_fp8", a))
        return 0


def test_contiguous_3d(monkeypatch):
    cap = Capture(monkeypatch)
    T, H, D, n = 4, 8, 128, 64
    k = torch.zeros(T, H, D, dtype=torch.bfloat16)
    kc = torch.zeros(n, H, D, dtype=torch.bfloat16)
    idx = torch.arange(T, dtype=torch.int64)
    kv.kv_store(k, k, kc, kc, idx)
    name, a = cap.calls[0]
    assert name == "kv_store"
    (_, _, _, _, _, idt, istride, ntok, h, d, e, strides, limit, split, _, stream) = a
    assert (idt, istride, ntok, h, d, e, limit, split, stream) == (1, 1, 4, 8, 128, 2, 64, 0, 1234)
    assert strides == (2048, 256, 2, 2048, 256, 2, 2048, 256, 2, 2048, 256, 2)


def test_qkv_views_and_padded_2d_cache(monkeypatch):
    cap = Capture(monkeypatch)
    T, HQ, H, D, n = 3, 32, 8, 128, 10
    qkv = torch.zeros(T, (HQ + 2 * H) * D, dtype=torch.float16)
    k = qkv[:, HQ * D:(HQ + H) * D]
    v = qkv[:, (HQ + H) * D:]
    store = torch.zeros(n, H * D + 64, dtype=torch.float16)
    kc = store[:, :H * D]
    idx = torch.arange(6, dtype=torch.int32)[::2]
    kv.kv_store(k, v, kc, kc, idx, num_heads=H, head_dim=D, size_limit=7, num_split=2)
    _, a = cap.calls[0]
    assert a[0] == k.data_ptr() and a[1] == v.data_ptr()
    assert a[0] - qkv.data_ptr() == HQ * D * 2
    assert (a[5], a[6], a[7]) == (0, 2, 3)          # int32, stride 2, 3 tokens
    assert a[11] == (12288, 256, 2, 12288, 256, 2, 2176, 256, 2, 2176, 256, 2)
    assert (a[12], a[13]) == (7, 2)


def test_fp8_3d_and_4d_caches(monkeypatch):
    cap = Capture(monkeypatch)
    T, H, D, ps, pages = 5, 4, 64, 16, 8
    k = torch.zeros(T, H * D, dtype=torch.bfloat16)
    idx = torch.arange(T, dtype=torch.int64)
    ik = torch.ones((), dtype=torch.float32)
    c3 = torch.zeros(ps * pages, H, D, dtype=torch.uint8)
    with pytest.raises(TypeError):       # scales must live on the device
        kv.kv_store_fp8(k, k, c3, c3, idx, page_size=ps, inv_k_scale=ik, inv_v_scale=ik)
    kv.kv_store_fp8(k, k, c3, c3, idx, page_size=ps)
    _, a = cap.calls[-1]
    assert a[10] == 1                                       # bf16
    assert a[11] == (512, 128, 2, 512, 128, 2, 256, 64, 1, 256, 64, 1)
    assert (a[12], a[13], a[14], a[15]) == (ps, ps * 256, ps * 256, ps * pages)
    assert (a[16], a[17], a[18]) == (None, None, 0)          # no scale
    big = torch.zeros(pages, ps * H * D + 128, dtype=torch.uint8)
    c4 = big[:, :ps * H * D].view(pages, ps, H, D)
    kv.kv_store_fp8(k.to(torch.float16), k.to(torch.float16), c4, c4, idx, page_size=ps)
    _, a = cap.calls[-1]
    assert a[10] == 0                                       # fp16
    assert a[11][6:] == (256, 64, 1, 256, 64, 1)
    assert (a[13], a[14], a[15]) == (ps * H * D + 128, ps * H * D + 128, ps * pages)
    with pytest.raises(ValueError):
        kv.kv_store_fp8(k, k, c4, c4, idx, page_size=8)


def test_binding_rejects_mismatches(monkeypatch):
    Capture(monkeypatch)
    k = torch.zeros(4, 2, 8, dtype=torch.bfloat16)
    kc = torch.zeros(16, 2, 8, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        kv.kv_store(k, k, kc.float(), kc, torch.arange(4))
    with pytest.raises(TypeError):
        kv.kv_store(k, k, kc, kc, torch.arange(4, dtype=torch.int16))
    with pytest.raises(ValueError):
        kv.kv_store(k, k, kc, kc, torch.arange(5))
    with pytest.raises(ValueError):
        kv.kv_store(torch.zeros(4, 3, 8, dtype=torch.bfloat16), k, kc, kc, torch.arange(4))


class CaptureAll(Capture):
    def __init__(self, monkeypatch):
        super().__init__(monkeypatch)
        for name in ("kv_store_paged", "kv_store_fp8_ex", "kv_gather_paged", "kv_gather_fp8_ex",
                     "kv_inv_scale", "kv_absmax_inv"):
            monkeypatch.setattr(kv.raw, name, self._make(name))

    def _make(self, name):
        def f(*a):
            self.calls.append((name, a))
            return 0
        return f


def test_paged_and_gather_wrappers(monkeypatch):
    cap = CaptureAll(monkeypatch)
    T, H, D, ps, pages = 6, 4, 32, 8, 16
    k = torch.zeros(T, H, D, dtype=torch.bfloat16)
    big = torch.zeros(pages, ps * H * D + 64, dtype=torch.bfloat16)
    cache = big[:, :ps * H * D].view(pages, ps, H, D)
    idx = torch.arange(T, dtype=torch.int32)
    kv.kv_store_paged(k, k, cache, cache, idx, page_size=ps)
    name, a = cap.calls[-1]
    assert name == "kv_store_paged"
    assert a[11] == (256, 64, 2, 256, 64, 2, 256, 64, 2, 256, 64, 2)
    assert (a[12], a[13], a[14], a[15]) == (ps, (ps * H * D + 64) * 2, (ps * H * D + 64) * 2,
                                            ps * pages)
    out = torch.zeros(T, H * D, dtype=torch.bfloat16)
    kv.kv_gather(cache, cache, out, out, idx, page_size=ps)
    name, a = cap.calls[-1]
    assert name == "kv_gather_paged" and a[10] == 2
    assert a[11][:6] == (256, 64, 2, 256, 64, 2)


def test_fp8_ex_wrappers(monkeypatch):
    cap = CaptureAll(monkeypatch)
    T, H, D, n = 5, 2, 64, 32
    k = torch.zeros(T, H, D, dtype=torch.float16)
    c = torch.zeros(n, H, D, dtype=torch.uint8)
    sc = torch.zeros(n, H + 2, dtype=torch.float32)
    idx = torch.arange(T, dtype=torch.int64)
    kv.kv_store_fp8_ex(k, k, c, c, idx, page_size=4, fmt="e5m2", scale_mode="token_head",
                       k_scales=sc, v_scales=sc)
    name, a = cap.calls[-1]
    assert name == "kv_store_fp8_ex"
    assert a[10] == 0 and (a[16], a[17]) == (1, 3)               # fp16, e5m2, token_head
    assert a[22] == H + 2 and a[20] == sc.data_ptr()
    assert (a[12], a[13]) == (4, 4 * H * D)
    out = torch.zeros(T, H, D, dtype=torch.bfloat16)
    kv.kv_gather_fp8(c, c, out, out, idx, page_size=4, scale_mode="token_head", k_scales=sc,
                     v_scales=sc)
    name, a = cap.calls[-1]
    assert name == "kv_gather_fp8_ex" and a[10] == 1 and a[22] == H + 2


def test_scale_wrappers(monkeypatch):
    cap = CaptureAll(monkeypatch)
    s = torch.ones(3, dtype=torch.float32)
    out = kv.kv_inv_scale(s)
    assert cap.calls[-1][0] == "kv_inv_scale" and cap.calls[-1][1][2] == 3 and out.shape == (3,)
    k = torch.zeros(7, 2, 16, dtype=torch.bfloat16)
    kv.kv_absmax_inv(k, k)
    name, a = cap.calls[-1]
    assert name == "kv_absmax_inv" and a[2:6] == (1, 7, 2, 16) and a[7] == 448.0
    assert a[10] is None
    w = torch.zeros(2, dtype=torch.int32)
    kv.kv_absmax_inv(k, k, work=w)
    assert cap.calls[-1][1][10] == w.data_ptr()


def test_fused_fp8_set_kv_buffer_argument_list(monkeypatch):
    """The wrapper with the argument list of the fused FP8 write's page: the
    unscaled call passes use_scale 0 and the page layout on; a 3-D cache whose
    slot count is not a multiple of page_size, or a page_size that differs
    from a 4-D cache's, is rejected; given both scales, their reciprocals are
    formed by kv_inv_scale (two values) before the write."""
    cap = CaptureAll(monkeypatch)
    T, H, D, ps, pages = 5, 4, 64, 16, 8
    k = torch.zeros(T, H * D, dtype=torch.bfloat16)
    idx = torch.arange(T, dtype=torch.int32)
    c3 = torch.zeros(ps * pages, H, D, dtype=torch.uint8)
    kv.fused_fp8_set_kv_buffer(k, k, c3, c3, idx)              # page_size defaults to 16
    name, a = cap.calls[-1]
    assert name == "kv_store_fp8"
    assert (a[12], a[13], a[14], a[15]) == (ps, ps * 256, ps * 256, ps * pages)
    assert (a[16], a[17], a[18]) == (None, None, 0)
    with pytest.raises(ValueError):
        kv.fused_fp8_set_kv_buffer(k, k, c3[:ps * pages - 1], c3[:ps * pages - 1], idx)
    c4 = torch.zeros(pages, ps, H, D, dtype=torch.uint8)
    with pytest.raises(ValueError):
        kv.fused_fp8_set_kv_buffer(k, k, c4, c4, idx, page_size=8)
    n = len(cap.calls)
    with pytest.raises(TypeError):          # host-side scales reach kv_store_fp8's device check
        kv.fused_fp8_set_kv_buffer(k, k, c4, c4, idx, 2.0, torch.tensor(0.5))
    assert cap.calls[n][0] == "kv_inv_scale" and cap.calls[n][1][2] == 2
    kv.fused_fp8_set_kv_buffer(k, k, c4, c4, idx, 2.0, None)   # one scale alone: unscaled
    assert cap.calls[-1][0] == "kv_store_fp8" and cap.calls[-1][1][18] == 0
    with pytest.raises(ValueError):
        kv.fused_fp8_set_kv_buffer(k, k, c4, c4, idx, torch.ones(2), 1.0)
