"""Pins for the CPU oracle, each against something other than the oracle.

* The e4m3fn encoder against a brute-force nearest-finite-code search over a
  decode table taken from a library (torch's float8_e4m3fn), on every bf16 and
  fp16 bit pattern and on a million random float32 patterns, plus the closed
  forms in ``golden/e4m3fn_points.txt``.
* The decoder against the same library table and against closed forms.
* The bf16/fp16 widening and the fp32 scale multiply against numpy / torch.
* The copy scatter against the worked example in ``golden/worked_copy.txt``,
  the untouched-slot invariant, a round-trip gather, and index-dtype,
  stride and page-layout equivalences.
* The FP8 scatter element by element against the brute-force encoder of the
  numpy fp32 product, the +-half-step error bound, and the use_scale=0 / inv=1
  and page-layout equivalences.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# Independent e4m3fn references
# ---------------------------------------------------------------------------

def _library_table() -> np.ndarray:
    """Values of all 256 e4m3fn codes according to torch (float64)."""
    return (torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn)
            .to(torch.float64).numpy())


LIB = _library_table()
POS_FINITE = np.arange(0x7F)          # 0x00 .. 0x7E


def brute_encode(x32: np.ndarray) -> np.ndarray:
    """Nearest finite e4m3fn value by exhaustive search; ties to the even code.

    Saturation needs no rule here: above 448 the nearest finite value is 448.
    """
    x = np.asarray(x32, dtype=np.float32).ravel()
    out = np.empty(x.size, dtype=np.uint8)
    vals = LIB[POS_FINITE]
    for c0 in range(0, x.size, 1 << 15):
        with np.errstate(invalid="ignore"):       # signalling NaN patterns
            xs = x[c0:c0 + (1 << 15)].astype(np.float64)
        a = np.abs(xs)
        # beyond 448 every magnitude has the same nearest finite value (448); cap
        # it so that the float64 distances stay distinguishable
        a = np.minimum(a, 1024.0)
        d = np.abs(a[:, None] - vals[None, :])
        best = d.min(axis=1, keepdims=True)
        tied = d == best
        # among the (at most two) nearest codes prefer the even one
        even = tied & ((POS_FINITE[None, :] & 1) == 0)
        code = np.where(even.any(axis=1), np.argmax(even, axis=1), np.argmax(tied, axis=1))
        code = code.astype(np.uint8) | np.where(np.signbit(xs), 0x80, 0).astype(np.uint8)
        code = np.where(np.isnan(xs), 0x7F, code)
        out[c0:c0 + xs.size] = code
    return out


def all_bf16_as_f32() -> np.ndarray:
    return (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)


def all_f16_as_f32() -> np.ndarray:
    return np.arange(1 << 16, dtype=np.uint16).view(np.float16).astype(np.float32)


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def test_decode_matches_library_table():
    got = oracle.e4m3fn_decode(np.arange(256))
    nan = np.isnan(LIB)
    assert np.array_equal(np.isnan(got), nan)
    assert list(np.flatnonzero(nan)) == [0x7F, 0xFF]
    assert np.array_equal(got[~nan], LIB[~nan])


def test_decode_closed_forms():
    d = oracle.e4m3fn_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x7E, 0xFE, 0x80]))
    assert list(d[:6]) == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 448.0]
    assert d[6] == -448.0 and d[7] == 0.0 and math.copysign(1, d[7]) == -1
    # strictly increasing over the non-negative finite codes; sign is the top bit
    pos = oracle.e4m3fn_decode(POS_FINITE)
    assert np.all(np.diff(pos) > 0)
    neg = oracle.e4m3fn_decode(POS_FINITE | 0x80)
    assert np.array_equal(neg[1:], -pos[1:])


def _golden_points():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3fn_points.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            x, code, why = [s.strip() for s in line.split(";")]
            rows.append((float(x), int(code, 16), why))
    return rows


def test_encode_golden_points():
    rows = _golden_points()
    assert len(rows) >= 25
    x = np.array([r[0] for r in rows], dtype=np.float32)
    # every listed input in the finite range is exactly representable in float32
    assert all(not abs(r[0]) <= 448 or float(np.float32(r[0])) == r[0] for r in rows)
    got = oracle.e4m3fn_encode(x)
    want = np.array([r[1] for r in rows], dtype=np.uint8)
    bad = [(rows[i][0], hex(got[i]), hex(want[i]), rows[i][2])
           for i in np.flatnonzero(got != want)]
    assert not bad, bad
    # and the brute-force search agrees with every hand-derived point
    assert np.array_equal(brute_encode(x), want)


def test_encode_exhaustive_bf16_and_f16():
    for x in (all_bf16_as_f32(), all_f16_as_f32()):
        got = oracle.e4m3fn_encode(x)
        want = brute_encode(x)
        assert np.array_equal(got, want), np.flatnonzero(got != want)[:10]


def test_encode_random_f32_patterns():
    # random bit patterns (all magnitudes, NaN, Inf, subnormals) ...
    bits = (wl.splitmix64(0xE4E3, 0, 1 << 19) >> np.uint64(32)).astype(np.uint32)
    x1 = bits.view(np.float32)
    # ... and random values concentrated where e4m3fn codes are (products)
    u = wl.uniform01(0xE4E4, 1 << 19)
    x2 = (np.sign(u - 0.5) * np.exp2(-12 + 22 * np.abs(2 * u - 1))).astype(np.float32)
    for x in (x1, x2):
        assert np.array_equal(oracle.e4m3fn_encode(x), brute_encode(x))


def test_encode_library_crosscheck_below_448():
    # torch's cast rounds to nearest-even too but does not saturate; below 448
    # the two must agree.
    x = all_bf16_as_f32()
    keep = np.isfinite(x) & (np.abs(x) < 448)
    lib = torch.from_numpy(x[keep]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3fn_encode(x[keep]), lib)


def test_encode_error_bound():
    # |decode(enc(y)) - clamp(y)| <= half the spacing of e4m3fn around y
    x = wl.normal(77, 1 << 16) * np.float32(60.0)
    q = oracle.e4m3fn_decode(oracle.e4m3fn_encode(x))
    y = np.clip(x.astype(np.float64), -448, 448)
    a = np.abs(y)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    half_step = 2.0 ** (e - 3) / 2
    assert np.all(np.abs(q - y) <= half_step)


def test_widening_and_scale():
    bits = np.arange(1 << 16, dtype=np.uint16)
    lib_bf = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    lib_f16 = bits.view(np.float16).astype(np.float32)
    for i in range(0, 1 << 16, 97):
        a, b = oracle.bf16_to_f32(int(bits[i])), lib_bf[i]
        assert (np.isnan(a) and np.isnan(b)) or a == b
        c, d = oracle.f16_to_f32(int(bits[i])), lib_f16[i]
        assert (np.isnan(c) and np.isnan(d)) or c == d
    # the fp32 multiply equals numpy's IEEE float32 multiply (subnormals kept)
    x = wl.normal(5, 4096) * np.float32(3)
    inv = np.float32(448.0) / np.float32(np.abs(x).max())
    tiny = np.float32(1e-38)
    for xi in list(x[:512]) + [tiny, -tiny, np.float32(3e-39)]:
        got = oracle.scale_f32(float(xi), float(inv))
        assert np.float32(got) == np.float32(xi) * inv
    assert oracle.scale_f32(1e-38, 0.25) == float(np.float32(1e-38) * np.float32(0.25)) != 0.0


# ---------------------------------------------------------------------------
# Plain copy scatter
# ---------------------------------------------------------------------------

def _contig_strides(H, D, e, slot_stride=None):
    R = H * D * e
    ss = R if slot_stride is None else slot_stride
    return oracle.Strides(k_token=R, k_head=D * e, k_dim=e, v_token=R, v_head=D * e, v_dim=e,
                          kc_slot=ss, kc_head=D * e, kc_dim=e, vc_slot=ss, vc_head=D * e,
                          vc_dim=e)


def _read_worked():
    spec = {}
    with open(os.path.join(GOLDEN, "worked_copy.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, *vals = line.split()
                spec[key] = vals
    return spec


def test_copy_worked_example():
    s = _read_worked()
    T, H, D = int(s["T"][0]), int(s["H"][0]), int(s["D"][0])
    hexa = lambda key: np.array([int(x, 16) for x in s[key]], dtype=np.uint16)
    k, v = hexa("k"), hexa("v")
    idx = np.array([int(x) for x in s["indices"]], dtype=np.int32)
    limit = int(s["size_limit"][0])
    kc = np.full(limit * H * D, int(s["sentinel"][0], 16), dtype=np.uint16)
    vc = kc.copy()
    bad, first = oracle.store_copy(k, v, kc, vc, idx, _contig_strides(H, D, 2), H, D, 2, limit)
    assert np.array_equal(kc, hexa("k_cache"))
    assert np.array_equal(vc, hexa("v_cache"))
    assert (bad, first) == (int(s["bad_count"][0]), int(s["first_bad"][0]))
    assert T == k.size // (H * D)


def _copy_problem(T, H, D, n_slots, seed, slot_stride=None, idx_dtype=np.int64):
    R = H * D * 2
    ss = R if slot_stride is None else slot_stride
    k = wl._normal_rows(seed, T, H, D, "bf16")
    v = wl._normal_rows(seed + 1, T, H, D, "bf16")
    idx = wl.distinct_slots(seed + 2, n_slots, T).astype(idx_dtype)
    kc = np.full(n_slots * ss // 2, wl.BF16_SENTINEL, dtype=np.uint16)
    vc = kc.copy()
    return k, v, idx, kc, vc, ss


@pytest.mark.parametrize("slot_stride", [None, 2 * 8 * 64 + 128])
def test_copy_roundtrip_and_untouched(slot_stride):
    T, H, D, n = 200, 8, 64, 1000
    k, v, idx, kc, vc, ss = _copy_problem(T, H, D, n, 11, slot_stride)
    bad, _ = oracle.store_copy(k, v, kc, vc, idx, _contig_strides(H, D, 2, ss), H, D, 2, n)
    assert bad == 0
    R16 = H * D
    kc2, vc2 = kc.reshape(n, ss // 2), vc.reshape(n, ss // 2)
    # round trip: gathering the named rows gives back K and V exactly
    assert np.array_equal(kc2[idx, :R16], k.reshape(T, R16))
    assert np.array_equal(vc2[idx, :R16], v.reshape(T, R16))
    # untouched: every other slot, and the padding of named slots, is pre-fill
    other = np.setdiff1d(np.arange(n), idx)
    assert np.all(kc2[other] == wl.BF16_SENTINEL) and np.all(vc2[other] == wl.BF16_SENTINEL)
    assert np.all(kc2[idx, R16:] == wl.BF16_SENTINEL)


def test_copy_index_dtype_and_oob():
    T, H, D, n = 64, 2, 32, 128
    k, v, idx, kc, vc, ss = _copy_problem(T, H, D, n, 21)
    idx = idx.copy()
    idx[5], idx[9], idx[40] = -1, n, np.iinfo(np.int64).max
    st = _contig_strides(H, D, 2)
    kc64, vc64 = kc.copy(), vc.copy()
    b64 = oracle.store_copy(k, v, kc64, vc64, idx, st, H, D, 2, n)
    assert b64 == (3, 5)
    idx32 = idx.copy()
    idx32[40] = np.iinfo(np.int32).min
    kc32, vc32 = kc.copy(), vc.copy()
    b32 = oracle.store_copy(k, v, kc32, vc32, idx32.astype(np.int32), st, H, D, 2, n)
    assert b32 == (3, 5)
    assert np.array_equal(kc64, kc32) and np.array_equal(vc64, vc32)
    # the skipped tokens wrote nothing: only 61 slots differ from the pre-fill
    changed = np.any(kc64.reshape(n, -1) != wl.BF16_SENTINEL, axis=1)
    assert changed.sum() == T - 3


def test_copy_strided_source_and_head_strides():
    # K/V as column views of a fused QKV row; caches with a head-major padding
    T, H, D, n, HQ = 50, 4, 16, 80, 6
    width = (HQ + 2 * H) * D
    qkv = wl._normal_rows(31, T, HQ + 2 * H, D, "f16").reshape(T, width)
    idx = wl.distinct_slots(32, n, T)
    e = 2
    cache_head = D * e + 32                       # padded head stride in the cache
    ss = H * cache_head
    st = oracle.Strides(k_token=width * e, k_head=D * e, k_dim=e, v_token=width * e,
                        v_head=D * e, v_dim=e, kc_slot=ss, kc_head=cache_head, kc_dim=e,
                        vc_slot=ss, vc_head=cache_head, vc_dim=e)
    kc = np.full(n * ss // 2, wl.BF16_SENTINEL, dtype=np.uint16)
    vc = kc.copy()
    oracle.store_copy(qkv, qkv, kc, vc, idx, st, H, D, 2, n,
                      k_off=HQ * D * e, v_off=(HQ + H) * D * e)
    kc4 = kc.reshape(n, H, cache_head // 2)
    kq = qkv.reshape(T, HQ + 2 * H, D)
    assert np.array_equal(kc4[idx, :, :D], kq[:, HQ:HQ + H])
    assert np.all(kc4[idx, :, D:] == wl.BF16_SENTINEL)
    vc4 = vc.reshape(n, H, cache_head // 2)
    assert np.array_equal(vc4[idx, :, :D], kq[:, HQ + H:])


def test_copy_duplicate_slots_take_one_candidate():
    T, H, D, n = 16, 1, 8, 8
    k, v, _, kc, vc, _ = _copy_problem(T, H, D, 64, 41)
    kc, vc = kc[:n * H * D].copy(), vc[:n * H * D].copy()
    idx = (np.array([3, 3, 5, 3] + list(range(12)), dtype=np.int32) % n)[:T]
    oracle.store_copy(k, v, kc, vc, idx, _contig_strides(H, D, 2), H, D, 2, n)
    rows = kc.reshape(n, H * D)
    for s in np.unique(idx):
        cands = k.reshape(T, -1)[idx == s]
        assert any(np.array_equal(rows[s], c) for c in cands)


# ---------------------------------------------------------------------------
# FP8 scatter
# ---------------------------------------------------------------------------

def _widen(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32)
    return bits.view(np.float16).astype(np.float32)


def _fp8_strides(H, D, e_src, slot_stride):
    R = H * D * e_src
    return oracle.Strides(k_token=R, k_head=D * e_src, k_dim=e_src, v_token=R,
                          v_head=D * e_src, v_dim=e_src, kc_slot=slot_stride, kc_head=D,
                          kc_dim=1, vc_slot=slot_stride, vc_head=D, vc_dim=1)


@pytest.mark.parametrize("src", ["bf16", "f16"])
@pytest.mark.parametrize("use_scale", [0, 1])
def test_fp8_elementwise_against_brute_force(src, use_scale):
    T, H, D, n, ps = 96, 4, 32, 256, 16
    w = wl.make_fp8("t", T, H, D, n, seed=91, dtype=src, page_size=ps)
    kc = np.full(n * H * D, wl.FP8_SENTINEL, dtype=np.uint8)
    vc = kc.copy()
    bad, _ = oracle.store_fp8(w.k, w.v, kc, vc, w.indices, _fp8_strides(H, D, 2, H * D), H, D,
                              src, ps, ps * H * D, ps * H * D, n, w.inv_k, w.inv_v, use_scale)
    assert bad == 0
    for bits, cache, inv in ((w.k, kc, w.inv_k), (w.v, vc, w.inv_v)):
        x = _widen(bits.reshape(T, -1), src)
        y = x * np.float32(inv) if use_scale else x
        want = brute_encode(y).reshape(T, -1)
        got = cache.reshape(n, -1)[w.indices]
        assert np.array_equal(got, want)
        other = np.setdiff1d(np.arange(n), w.indices)
        assert np.all(cache.reshape(n, -1)[other] == wl.FP8_SENTINEL)
    if not use_scale:
        # the outliers saturate: some codes are +-448
        assert np.any((kc & 0x7F) == 0x7E)


def test_fp8_use_scale_off_equals_inv_one():
    T, H, D, n, ps = 64, 2, 64, 128, 8
    w = wl.make_fp8("t", T, H, D, n, seed=92, page_size=ps)
    st = _fp8_strides(H, D, 2, H * D)
    outs = []
    for use, inv in ((0, 123.0), (1, 1.0)):
        kc = np.full(n * H * D, wl.FP8_SENTINEL, dtype=np.uint8)
        vc = kc.copy()
        oracle.store_fp8(w.k, w.v, kc, vc, w.indices, st, H, D, "bf16", ps, ps * H * D,
                         ps * H * D, n, inv, inv, use)
        outs.append((kc, vc))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


def test_fp8_page_layouts():
    # A 3-D cache: page decomposition equals direct slot addressing for any page size.
    T, H, D, n = 40, 2, 16, 96
    w = wl.make_fp8("t", T, H, D, n, seed=93, page_size=8)
    st = _fp8_strides(H, D, 2, H * D)
    ref = None
    for ps in (1, 8, 32, 96):
        kc = np.full(n * H * D, wl.FP8_SENTINEL, dtype=np.uint8)
        vc = kc.copy()
        oracle.store_fp8(w.k, w.v, kc, vc, w.indices, st, H, D, "bf16", ps, ps * H * D,
                         ps * H * D, n, w.inv_k, w.inv_v, 1)
        ref = (kc, vc) if ref is None else ref
        assert np.array_equal(kc, ref[0]) and np.array_equal(vc, ref[1])
    # A 4-D cache [pages, page_size, H, D] with a padded page stride: row of slot
    # s lands at (s // ps) * page_stride + (s % ps) * slot_stride.
    ps, pad = 8, 64
    page_stride = ps * H * D + pad
    n_pages = n // ps
    kc = np.full(n_pages * page_stride, wl.FP8_SENTINEL, dtype=np.uint8)
    vc = kc.copy()
    oracle.store_fp8(w.k, w.v, kc, vc, w.indices, st, H, D, "bf16", ps, page_stride,
                     page_stride, n, w.inv_k, w.inv_v, 1)
    pages = kc.reshape(n_pages, page_stride)
    rows = pages[:, :ps * H * D].reshape(n, H * D)
    assert np.array_equal(rows, ref[0].reshape(n, H * D))
    assert np.all(pages[:, ps * H * D:] == wl.FP8_SENTINEL)


def test_fp8_oob_skipped():
    T, H, D, n, ps = 32, 2, 16, 64, 4
    w = wl.make_fp8("t", T, H, D, n, seed=94, page_size=ps)
    idx = w.indices.copy()
    idx[[3, 17]] = [n, -5]
    kc = np.full(n * H * D, wl.FP8_SENTINEL, dtype=np.uint8)
    vc = kc.copy()
    bad = oracle.store_fp8(w.k, w.v, kc, vc, idx, _fp8_strides(H, D, 2, H * D), H, D, "bf16",
                           ps, ps * H * D, ps * H * D, n, w.inv_k, w.inv_v, 1)
    assert bad == (2, 3)
    changed = np.any(kc.reshape(n, -1) != wl.FP8_SENTINEL, axis=1)
    assert changed.sum() == T - 2


# ---------------------------------------------------------------------------
# bf16 / fp16 encoders and the inverse path (gather with dequantisation)
# ---------------------------------------------------------------------------

def _random_f32(seed, n):
    bits = (wl.splitmix64(seed, 0, n) >> np.uint64(32)).astype(np.uint32)
    return bits.view(np.float32)


def _ties_f32(keep_bits):
    """float32 values exactly halfway between two representable narrow values
    (and one ulp either side), for every narrow bit pattern."""
    drop = 23 - keep_bits
    base = np.arange(1 << 16, dtype=np.uint32) << 16 if keep_bits == 7 else \
        (np.arange(1 << 16, dtype=np.uint32) << np.uint32(drop)) & np.uint32(0x7FFFFFFF)
    half = np.uint32(1 << (drop - 1))
    out = np.concatenate([base + half, base + half - 1, base + half + 1])
    return out.view(np.float32)


def test_bf16_encoder_against_library():
    for x in (_random_f32(0xBF16, 1 << 20), _ties_f32(7)):
        keep = ~np.isnan(x)
        lib = torch.from_numpy(x[keep].copy()).to(torch.bfloat16).view(torch.int16).numpy()
        assert np.array_equal(oracle.f32_to_bf16(x[keep]), lib.view(np.uint16))
    assert np.all(oracle.f32_to_bf16(np.array([np.nan, -np.nan], np.float32)) == 0x7FFF)


def test_f16_encoder_against_library():
    # fp16 halfway points: widen every fp16 pattern and add half an fp16 ulp
    h = np.arange(1 << 15, dtype=np.uint16).view(np.float16).astype(np.float64)
    h = h[np.isfinite(h)]
    with np.errstate(over="ignore"):
        ulp = np.spacing(h.astype(np.float16)).astype(np.float64)
    mids = (h + ulp / 2).astype(np.float32)
    for x in (_random_f32(0xF16, 1 << 20), mids, -mids, np.nextafter(mids, np.float32(0))):
        keep = ~np.isnan(x)
        with np.errstate(over="ignore"):
            lib = x[keep].astype(np.float16).view(np.uint16)
        assert np.array_equal(oracle.f32_to_f16(x[keep]), lib)
    assert np.all(oracle.f32_to_f16(np.array([np.nan], np.float32)) == 0x7FFF)
    assert oracle.f32_to_f16(np.array([65520.0], np.float32))[0] == 0x7C00   # rounds to Inf
    assert oracle.f32_to_f16(np.array([2.0 ** -25], np.float32))[0] == 0      # tie to even 0


def test_gather_copy_round_trip_and_oob():
    T, H, D, n = 150, 4, 32, 400
    k, v, idx, kc, vc, ss = _copy_problem(T, H, D, n, 61)
    st = _contig_strides(H, D, 2)
    oracle.store_copy(k, v, kc, vc, idx, st, H, D, 2, n)
    ko = np.zeros_like(k)
    vo = np.zeros_like(v)
    assert oracle.gather_copy(kc, vc, ko, vo, idx, st, H, D, 2, n) == (0, -1)
    assert np.array_equal(ko, k) and np.array_equal(vo, v)
    bad = idx.copy()
    bad[[7, 100]] = [n, -3]
    ko[:] = 0x1234
    assert oracle.gather_copy(kc, vc, ko, vo, bad, st, H, D, 2, n) == (2, 7)
    assert np.all(ko[7] == 0x1234) and np.all(ko[100] == 0x1234)
    assert np.array_equal(ko[8], k[8])


def _lib_dequant(codes, scale, out):
    """Library restatement: torch's e4m3fn decode, float32 multiply, torch/numpy rounding."""
    x = LIB[codes].astype(np.float32)
    y = x * np.float32(scale)
    if out == "bf16":
        r = torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    else:
        with np.errstate(over="ignore", invalid="ignore"):
            r = y.astype(np.float16).view(np.uint16)
    return np.where(np.isnan(y), np.uint16(0x7FFF), r)


@pytest.mark.parametrize("out", ["bf16", "f16"])
@pytest.mark.parametrize("scale", [None, 1.0, 0.0078125, 3.3, 1e4])
def test_gather_fp8_every_code(out, scale):
    # one slot per token, each cache row holding all 256 codes in some order
    T, H, D, n = 8, 2, 128, 16
    codes = np.concatenate([np.arange(256, dtype=np.uint8)] * (T * H * D // 256))
    codes = codes.reshape(T, H * D)
    rng = wl.splitmix64(71, 0, T * H * D) % np.uint64(256)
    codes = (codes + rng.reshape(T, H * D).astype(np.uint8)).astype(np.uint8)
    kc = np.full(n * H * D, 0x7F, np.uint8)
    idx = wl.distinct_slots(72, n, T)
    kc.reshape(n, H * D)[idx] = codes
    vc = kc.copy()
    R = H * D * 2
    st = oracle.Strides(k_token=R, k_head=D * 2, k_dim=2, v_token=R, v_head=D * 2, v_dim=2,
                        kc_slot=H * D, kc_head=D, kc_dim=1, vc_slot=H * D, vc_head=D, vc_dim=1)
    ko = np.zeros(T * H * D, np.uint16)
    vo = np.zeros_like(ko)
    use = scale is not None
    s = 1.0 if scale is None else scale
    oracle.gather_fp8(kc, vc, ko, vo, idx, st, H, D, out, 4, 4 * H * D, 4 * H * D, n,
                      s, s, int(use))
    want = _lib_dequant(codes.ravel(), s, out)
    assert np.array_equal(ko, want) and np.array_equal(vo, want)


def test_fp8_store_then_gather_within_half_step():
    T, H, D, n, ps = 64, 4, 64, 256, 16
    w = wl.make_fp8("t", T, H, D, n, seed=73, page_size=ps)
    st = _fp8_strides(H, D, 2, H * D)
    kc = np.full(n * H * D, wl.FP8_SENTINEL, np.uint8)
    vc = kc.copy()
    oracle.store_fp8(w.k, w.v, kc, vc, w.indices, st, H, D, "bf16", ps, ps * H * D, ps * H * D,
                     n, w.inv_k, w.inv_v, 1)
    ko = np.zeros(T * H * D, np.uint16)
    vo = np.zeros_like(ko)
    sk = float(np.float32(1.0) / np.float32(w.inv_k))
    oracle.gather_fp8(kc, vc, ko, vo, w.indices, st, H, D, "bf16", ps, ps * H * D, ps * H * D,
                      n, sk, sk, 1)
    x = _widen(w.k.reshape(-1), "bf16").astype(np.float64)
    back = (ko.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    # scaled value y = x*inv is within half an e4m3 step of the code; dequantising
    # multiplies that by 1/inv and rounds to bf16 (relative 2^-9)
    y = x * w.inv_k
    a = np.abs(np.clip(y, -448, 448))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    bound = (2.0 ** (e - 4)) * sk * (1 + 2 ** -7) + np.abs(back) * 2.0 ** -8
    assert np.all(np.abs(back - np.clip(y, -448, 448) * sk) <= bound + 1e-30)


def test_paged_copy_layouts():
    """Paged copy: a dense page stride equals the flat copy for any page size,
    and a padded 4-D layout lands rows at page*page_stride + offset*slot_stride
    (numpy fancy indexing k_cache[page_ids, page_offsets] = k as the check)."""
    T, H, D, n = 120, 4, 16, 512
    k, v, idx, kc0, vc0, ss = _copy_problem(T, H, D, n, 81)
    st = _contig_strides(H, D, 2)
    flat_k, flat_v = kc0.copy(), vc0.copy()
    oracle.store_copy(k, v, flat_k, flat_v, idx, st, H, D, 2, n)
    for ps in (1, 16, 64, 512):
        pk, pv = kc0.copy(), vc0.copy()
        assert oracle.store_copy_paged(k, v, pk, pv, idx, st, H, D, 2, ps, ps * ss, ps * ss,
                                       n) == (0, -1)
        assert np.array_equal(pk, flat_k) and np.array_equal(pv, flat_v)
    ps, pad = 16, 96
    page = ps * ss + pad
    n_pages = n // ps
    pk = np.full(n_pages * page // 2, wl.BF16_SENTINEL, np.uint16)
    pv = pk.copy()
    oracle.store_copy_paged(k, v, pk, pv, idx, st, H, D, 2, ps, page, page, n)
    pages = pk.view(np.uint8).reshape(n_pages, page)
    view4 = pages[:, :ps * ss].reshape(n_pages, ps, ss)
    want = np.full((n_pages, ps, ss), 0, np.uint8)
    want.view(np.uint16)[:] = wl.BF16_SENTINEL
    want[idx // ps, idx % ps] = k.view(np.uint8).reshape(T, ss)
    assert np.array_equal(view4, want)
    assert np.all(pages[:, ps * ss:].view(np.uint16) == wl.BF16_SENTINEL)


def test_inv_scale_is_ieee_fp32_division():
    x = np.concatenate([wl.normal(91, 4096) * np.float32(100),
                        np.array([1.0, 3.0, 448.0, 1e-38, 3e-39, 1e38, -7.5], np.float32),
                        np.abs(_random_f32(92, 4096))])
    x = x[np.isfinite(x) & (x != 0)]
    with np.errstate(over="ignore", divide="ignore"):
        want = np.float32(1.0) / x.astype(np.float32)
    got = oracle.inv_scale(x)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("src", ["bf16", "f16"])
def test_absmax_inv_against_numpy(src):
    T, H, D = 300, 4, 32
    w = wl.make_fp8("t", T, H, D, 1024, seed=93, dtype=src)
    kb, vb = w.k.copy(), w.v.copy()
    # a NaN and an outlier of each sign must not / must count
    kb.reshape(-1)[17] = 0x7FC0 if src == "bf16" else 0x7E00
    st = _fp8_strides(H, D, 2, H * D)
    amax, inv = oracle.absmax_inv(kb, vb, st, T, H, D, src)
    for bits, a, i in ((kb, amax[0], inv[0]), (vb, amax[1], inv[1])):
        x = _widen(bits.reshape(-1), src)
        want = np.float32(np.nanmax(np.abs(x)))
        assert a == want
        assert i == np.float32(448.0) / want
    # all-zero tensors give inv = 1
    z = np.zeros_like(kb)
    amax, inv = oracle.absmax_inv(z, z, st, T, H, D, src)
    assert list(amax) == [0.0, 0.0] and list(inv) == [1.0, 1.0]
    # the fp8 workload's recipe (host numpy) is exactly this
    amax, inv = oracle.absmax_inv(w.k, w.v, st, T, H, D, src)
    assert inv[0] == np.float32(w.inv_k) and inv[1] == np.float32(w.inv_v)


# ---------------------------------------------------------------------------
# e5m2 and the extended FP8 write (formats, dynamic per-token / per-head scales)
# ---------------------------------------------------------------------------

LIB52 = (torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).to(torch.float64).numpy())
POS52 = np.arange(0x7C)          # 0x00 .. 0x7B finite non-negative


def brute_encode_e5m2(x32):
    x = np.asarray(x32, dtype=np.float32).ravel()
    out = np.empty(x.size, dtype=np.uint8)
    vals = LIB52[POS52]
    for c0 in range(0, x.size, 1 << 14):
        with np.errstate(invalid="ignore"):
            xs = x[c0:c0 + (1 << 14)].astype(np.float64)
        a = np.minimum(np.abs(xs), 1e6)
        d = np.abs(a[:, None] - vals[None, :])
        tied = d == d.min(axis=1, keepdims=True)
        even = tied & ((POS52[None, :] & 1) == 0)
        code = np.where(even.any(axis=1), np.argmax(even, axis=1), np.argmax(tied, axis=1))
        code = code.astype(np.uint8) | np.where(np.signbit(xs), 0x80, 0).astype(np.uint8)
        out[c0:c0 + xs.size] = np.where(np.isnan(xs), 0x7F, code)
    return out


def test_e5m2_decode_and_encode():
    d = oracle.e5m2_decode(np.arange(256))
    nan = np.isnan(LIB52)
    assert np.array_equal(np.isnan(d), nan) and np.array_equal(d[~nan], LIB52[~nan])
    assert d[0x7B] == 57344.0 and d[0x7C] == np.inf and d[0x04] == 2.0 ** -14
    for x in (all_bf16_as_f32(), all_f16_as_f32(), _random_f32(0xE5, 1 << 18)):
        assert np.array_equal(oracle.e5m2_encode(x), brute_encode_e5m2(x))
    pts = np.array([57344, 61439, 61440, 1e20, np.inf, -np.inf, 2 ** -17, 1.125, 1.375],
                   np.float32)
    assert list(oracle.e5m2_encode(pts)) == [0x7B, 0x7B, 0x7B, 0x7B, 0x7B, 0xFB, 0x00, 0x3C,
                                             0x3E]


def _ex_problem(T, H, D, n, seed, src="bf16", ps=8):
    w = wl.make_fp8("x", T, H, D, n, seed=seed, dtype=src, page_size=ps, scale=3.0)
    st = _fp8_strides(H, D, 2, H * D)
    return w, st


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("mode", ["token", "token_head"])
def test_store_fp8_ex_dynamic_groups(fmt, mode):
    T, H, D, n, ps = 40, 4, 32, 128, 8
    w, st = _ex_problem(T, H, D, n, seed=101)
    kb = w.k.copy()
    kb.reshape(T, -1)[3] = 0                    # an all-zero row: scale 1
    kb.reshape(-1)[200] = 0x7FC0                # a NaN element: ignored by amax
    kc = np.full(n * H * D, 0x7F, np.uint8)
    vc = kc.copy()
    G = H if mode == "token_head" else 1
    ks = np.full(n * G, -1.0, np.float32)
    vs = ks.copy()
    oracle.store_fp8_ex(kb, w.v, kc, vc, w.indices, st, H, D, "bf16", ps, ps * H * D, ps * H * D,
                        n, fmt=fmt, scale_mode=mode, k_scales=ks, v_scales=vs,
                        scales_slot_stride=G)
    fmax = np.float32(448.0 if fmt == "e4m3fn" else 57344.0)
    enc = brute_encode if fmt == "e4m3fn" else brute_encode_e5m2
    for bits, cache, sc in ((kb, kc, ks), (w.v, vc, vs)):
        x = _widen(bits.reshape(T, H, D), "bf16")
        groups = x.reshape(T, G, -1)
        amax = np.nanmax(np.abs(groups), axis=2).astype(np.float32)
        with np.errstate(divide="ignore"):
            inv = np.where(amax > 0, fmax / amax, np.float32(1)).astype(np.float32)
            scale = np.where(amax > 0, amax / fmax, np.float32(1)).astype(np.float32)
        y = (groups * inv[:, :, None]).astype(np.float32)
        want = enc(y).reshape(T, -1)
        assert np.array_equal(cache.reshape(n, -1)[w.indices], want)
        assert np.array_equal(sc.reshape(n, G)[w.indices], scale)
        untouched = np.setdiff1d(np.arange(n), w.indices)
        assert np.all(sc.reshape(n, G)[untouched] == -1.0)
    assert ks.reshape(n, G)[w.indices[3]][0] == 1.0


def test_store_fp8_ex_static_modes_match_store_fp8():
    T, H, D, n, ps = 64, 2, 64, 256, 16
    w, st = _ex_problem(T, H, D, n, seed=102, ps=ps)
    for mode, use in (("none", 0), ("tensor", 1)):
        a = [np.full(n * H * D, 0x7F, np.uint8) for _ in range(4)]
        oracle.store_fp8(w.k, w.v, a[0], a[1], w.indices, st, H, D, "bf16", ps, ps * H * D,
                         ps * H * D, n, w.inv_k, w.inv_v, use)
        oracle.store_fp8_ex(w.k, w.v, a[2], a[3], w.indices, st, H, D, "bf16", ps, ps * H * D,
                            ps * H * D, n, fmt="e4m3fn", scale_mode=mode, inv_k=w.inv_k,
                            inv_v=w.inv_v)
        assert np.array_equal(a[0], a[2]) and np.array_equal(a[1], a[3])


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_gather_fp8_ex_per_slot_scales(fmt):
    T, H, D, n, ps = 48, 4, 32, 128, 8
    w, st = _ex_problem(T, H, D, n, seed=103, ps=ps)
    kc = np.full(n * H * D, 0x7F, np.uint8)
    vc = kc.copy()
    ks = np.zeros(n * H, np.float32)
    vs = ks.copy()
    oracle.store_fp8_ex(w.k, w.v, kc, vc, w.indices, st, H, D, "bf16", ps, ps * H * D,
                        ps * H * D, n, fmt=fmt, scale_mode="token_head", k_scales=ks, v_scales=vs,
                        scales_slot_stride=H)
    ko = np.zeros(T * H * D, np.uint16)
    vo = ko.copy()
    R = H * D * 2
    ost = oracle.Strides(k_token=R, k_head=D * 2, k_dim=2, v_token=R, v_head=D * 2, v_dim=2,
                         kc_slot=H * D, kc_head=D, kc_dim=1, vc_slot=H * D, vc_head=D, vc_dim=1)
    oracle.gather_fp8_ex(kc, vc, ko, vo, w.indices, ost, H, D, "bf16", ps, ps * H * D, ps * H * D,
                         n, fmt=fmt, scale_mode="token_head", k_scales=ks, v_scales=vs,
                         scales_slot_stride=H)
    table = LIB if fmt == "e4m3fn" else LIB52
    codes = kc.reshape(n, H, D)[w.indices]
    sc = ks.reshape(n, H)[w.indices]
    y = (table[codes].astype(np.float32) * sc[:, :, None]).astype(np.float32)
    want = torch.from_numpy(y.reshape(-1)).to(torch.bfloat16).view(torch.int16).numpy()
    want = np.where(np.isnan(y.reshape(-1)), 0x7FFF, want.view(np.uint16))
    assert np.array_equal(ko, want)
    # and the round trip is close: within one fp8 step of the group scale
    x = _widen(w.k.reshape(-1), "bf16").reshape(T, H, D)
    back = (ko.astype(np.uint32) << 16).view(np.float32).reshape(T, H, D)
    step = 2.0 ** -3 if fmt == "e4m3fn" else 2.0 ** -2
    assert np.all(np.abs(back - x) <= np.abs(x) * step + sc[:, :, None] * 2.0 ** -9 * 16)


def test_paged_gather_round_trip():
    T, H, D, n, ps, pad = 100, 4, 16, 512, 16, 96
    k, v, idx, _, _, ss = _copy_problem(T, H, D, n, 85)
    st = _contig_strides(H, D, 2)
    page = ps * ss + pad
    pk = np.full(n // ps * page // 2, wl.BF16_SENTINEL, np.uint16)
    pv = pk.copy()
    oracle.store_copy_paged(k, v, pk, pv, idx, st, H, D, 2, ps, page, page, n)
    ko, vo = np.zeros_like(k), np.zeros_like(v)
    bad = idx.copy()
    bad[5] = -1
    assert oracle.gather_copy_paged(pk, pv, ko, vo, bad, st, H, D, 2, ps, page, page, n) == (1, 5)
    keep = np.arange(T) != 5
    assert np.array_equal(ko[keep], k[keep]) and np.array_equal(vo[keep], v[keep])
    assert np.all(ko[5] == 0)


# ---------------------------------------------------------------------------
# Per-page scales (one fp32 scale per cache page, page = slot // page_size)
# ---------------------------------------------------------------------------

def _page_scales(n_pages, seed):
    """Positive fp32 inverse scales of assorted magnitudes, one per page: some
    pages scale into saturation, some far down, one is exactly 1."""
    u = wl.uniform01(seed, n_pages)
    inv = (2.0 ** (np.floor(u * 24) - 12) * (1.0 + wl.uniform01(seed + 1, n_pages)))
    inv = inv.astype(np.float32)
    inv[0] = 1.0
    return inv


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("src", ["bf16", "f16"])
def test_store_fp8_ex_per_page_scales(fmt, src):
    """Every code is the brute-force code of numpy's fp32 product x * inv[page]
    of its slot's page; rows land at page * page_stride + offset * slot_stride
    of padded 4-D pages; every other byte keeps the pre-fill."""
    T, H, D, ps, n_pages = 96, 4, 32, 8, 32
    n = ps * n_pages
    w = wl.make_fp8("t", T, H, D, n, seed=121, dtype=src, page_size=ps)
    R8 = H * D
    page_stride = ps * R8 + 64                      # 64 bytes of pad per page
    st = _fp8_strides(H, D, 2, R8)
    inv_k = _page_scales(n_pages, 122)
    inv_v = _page_scales(n_pages, 124)
    kc = np.full(n_pages * page_stride, 0x7F, np.uint8)
    vc = kc.copy()
    assert oracle.store_fp8_ex(w.k, w.v, kc, vc, w.indices, st, H, D, src, ps, page_stride,
                               page_stride, n, fmt=fmt, scale_mode="page", k_scales=inv_k,
                               v_scales=inv_v) == (0, -1)
    enc = brute_encode if fmt == "e4m3fn" else brute_encode_e5m2
    page, off = w.indices // ps, w.indices % ps
    for bits, cache, inv in ((w.k, kc, inv_k), (w.v, vc, inv_v)):
        x = _widen(bits.reshape(T, H * D), src)
        y = (x * inv[page][:, None]).astype(np.float32)
        want = enc(y).reshape(T, R8)
        rows = cache.reshape(n_pages, page_stride)[:, :ps * R8].reshape(n_pages, ps, R8)
        assert np.array_equal(rows[page, off], want)
        touched = np.zeros((n_pages, ps), bool)
        touched[page, off] = True
        assert np.all(rows[~touched] == 0x7F)
        assert np.all(cache.reshape(n_pages, page_stride)[:, ps * R8:] == 0x7F)


def test_store_fp8_ex_page_constant_equals_tensor_mode():
    """With the same inverse scale on every page, the per-page write equals the
    per-tensor write byte for byte (flat and padded pages)."""
    T, H, D, ps, n_pages = 64, 2, 64, 16, 16
    n = ps * n_pages
    w, st = _ex_problem(T, H, D, n, seed=126, ps=ps)
    for page_stride in (ps * H * D, ps * H * D + 128):
        a = [np.full(n_pages * page_stride, 0x7F, np.uint8) for _ in range(4)]
        oracle.store_fp8_ex(w.k, w.v, a[0], a[1], w.indices, st, H, D, "bf16", ps, page_stride,
                            page_stride, n, scale_mode="tensor", inv_k=w.inv_k, inv_v=w.inv_v)
        oracle.store_fp8_ex(w.k, w.v, a[2], a[3], w.indices, st, H, D, "bf16", ps, page_stride,
                            page_stride, n, scale_mode="page",
                            k_scales=np.full(n_pages, w.inv_k, np.float32),
                            v_scales=np.full(n_pages, w.inv_v, np.float32))
        assert np.array_equal(a[0], a[2]) and np.array_equal(a[1], a[3])


@pytest.mark.parametrize("out", ["bf16", "f16"])
def test_gather_fp8_ex_per_page_scales(out):
    """Each output element is torch's e4m3fn decode of its code times the
    scale of its slot's page in fp32, rounded by torch (bf16) / numpy (fp16);
    an out-of-range slot leaves its row alone."""
    T, H, D, ps, n_pages = 40, 2, 64, 4, 64
    n = ps * n_pages
    R8 = H * D
    idx = wl.distinct_slots(127, n, T)
    codes = (wl.splitmix64(128, 0, T * R8) % np.uint64(256)).astype(np.uint8).reshape(T, R8)
    kc = np.full(n * R8, 0x7F, np.uint8)
    kc.reshape(n, R8)[idx] = codes
    vc = kc.copy()
    sk = _page_scales(n_pages, 129)
    sv = (sk * np.float32(0.5)).astype(np.float32)
    st = oracle.Strides(k_token=R8 * 2, k_head=D * 2, k_dim=2, v_token=R8 * 2, v_head=D * 2,
                        v_dim=2, kc_slot=R8, kc_head=D, kc_dim=1, vc_slot=R8, vc_head=D,
                        vc_dim=1)
    ko = np.full(T * R8, 0x1234, np.uint16)
    vo = ko.copy()
    bad = idx.copy()
    bad[9] = n
    assert oracle.gather_fp8_ex(kc, vc, ko, vo, bad, st, H, D, out, ps, ps * R8, ps * R8, n,
                                scale_mode="page", k_scales=sk, v_scales=sv) == (1, 9)
    keep = np.arange(T) != 9
    for o, s in ((ko, sk), (vo, sv)):
        rows = o.reshape(T, R8)
        for t in np.nonzero(keep)[0]:
            assert np.array_equal(rows[t], _lib_dequant(codes[t], s[idx[t] // ps], out))
        assert np.all(rows[9] == 0x1234)


def test_per_page_store_then_gather_within_half_step():
    """Writing with inv[page] and reading back with 1/inv[page] lands within
    half an e4m3 step of the scaled value, mapped back by the page's scale."""
    T, H, D, ps, n_pages = 64, 4, 32, 8, 64
    n = ps * n_pages
    w, st = _ex_problem(T, H, D, n, seed=131, ps=ps)
    amax = np.float32(np.max(np.abs(_widen(w.k.reshape(-1), "bf16"))))
    inv = (np.float32(448.0) / amax * _page_scales(n_pages, 132) /
           np.float32(2.0)).astype(np.float32)
    inv = np.minimum(inv, np.float32(448.0) / amax).astype(np.float32)  # no saturation
    scale = (np.float32(1.0) / inv).astype(np.float32)
    kc = np.full(n * H * D, 0x7F, np.uint8)
    vc = kc.copy()
    oracle.store_fp8_ex(w.k, w.v, kc, vc, w.indices, st, H, D, "bf16", ps, ps * H * D,
                        ps * H * D, n, scale_mode="page", k_scales=inv, v_scales=inv)
    ko = np.zeros(T * H * D, np.uint16)
    vo = ko.copy()
    ost = oracle.Strides(k_token=H * D * 2, k_head=D * 2, k_dim=2, v_token=H * D * 2,
                         v_head=D * 2, v_dim=2, kc_slot=H * D, kc_head=D, kc_dim=1,
                         vc_slot=H * D, vc_head=D, vc_dim=1)
    oracle.gather_fp8_ex(kc, vc, ko, vo, w.indices, ost, H, D, "bf16", ps, ps * H * D,
                         ps * H * D, n, scale_mode="page", k_scales=scale, v_scales=scale)
    x = _widen(w.k.reshape(T, -1), "bf16").astype(np.float64)
    back = (ko.astype(np.uint32) << 16).view(np.float32).reshape(T, -1).astype(np.float64)
    pinv = inv[w.indices // ps].astype(np.float64)[:, None]
    psc = scale[w.indices // ps].astype(np.float64)[:, None]
    y = x * pinv
    e = np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6)))
    bound = 2.0 ** (e - 4) * psc * (1 + 2 ** -7) + np.abs(back) * 2.0 ** -8 + np.abs(y) * psc * 2 ** -22
    assert np.all(np.abs(back - y * psc) <= bound + 1e-30)
