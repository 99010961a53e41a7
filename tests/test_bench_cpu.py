"""Host-side pieces of bench.py that need no GPU: the CPU-oracle timing
(one thread, and split over host threads by token range) and the reference
arm's JSON line."""

import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_threaded_oracle_run_writes_the_same_caches():
    """Token ranges on several POSIX threads write exactly what one
    whole-batch oracle call writes (copy and FP8 kinds)."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as wl
    for name in ("tiny", "fp8_small"):
        w = (bench.load_workload(name) if name == "tiny" else
             wl.make_fp8(name, T=512, H=8, D=128, n_slots=4096, seed=3, page_size=32))
        bench._ORACLE_CACHE.pop(name, None)
        job = bench.oracle_job(name, w)
        kc, vc = bench._ORACLE_CACHE[name][:2]
        kc[:] = 0
        vc[:] = 0
        bench.oracle_step(name, w, w.T)
        want = kc.copy(), vc.copy()
        kc[:] = 0
        vc[:] = 0
        done, el, bad = job.run(4)
        assert done == w.T and bad == 0 and el >= 0
        assert np.array_equal(kc, want[0]) and np.array_equal(vc, want[1])
        assert np.count_nonzero(want[0]) > 0
        bench._ORACLE_CACHE.pop(name, None)


def test_threaded_runner_counts_tokens_and_bad_slots():
    """The runner's bookkeeping: every thread's passes are counted, and
    out-of-range slots met by the oracle are summed over threads."""
    sys.path.insert(0, ROOT)
    import oracle
    T, H, D = 40, 1, 8
    k = np.arange(T * H * D, dtype=np.uint16)
    v = k[::-1].copy()
    kc = np.zeros(64 * H * D, np.uint16)
    vc = kc.copy()
    idx = np.arange(T, dtype=np.int32)
    idx[[3, 17, 39]] = [-1, 64, 1000]
    R = H * D * 2
    st = oracle.Strides(k_token=R, k_head=D * 2, k_dim=2, v_token=R, v_head=D * 2, v_dim=2,
                        kc_slot=R, kc_head=D * 2, kc_dim=2, vc_slot=R, vc_head=D * 2, vc_dim=2)
    job = oracle.ThreadedJob("copy", k, v, kc, vc, idx, st, H, D, 64, elem_bytes=2)
    done, el, bad = job.run(3, 0.0, 2)
    assert done % T == 0 and done >= 2 * T and bad == 3 * (done // T)
    assert np.array_equal(kc.reshape(64, D)[:T][idx >= 0][: 3], k.reshape(T, D)[:3])


def test_oracle_rates_are_positive():
    sys.path.insert(0, ROOT)
    import bench
    r1, s1, c1 = bench.oracle_tokens_per_s("tiny", 0.2)
    r4, s4, c4 = bench.oracle_tokens_per_s("tiny", 0.2, threads=4)
    assert r1 > 0 and r4 > 0 and c1 == 1 and c4 == 4
    assert "1 POSIX thread," in s1 and "4 POSIX threads" in s4


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    # the same config object as the GPU arm's line
    sys.path.insert(0, ROOT)
    import bench
    w = bench.load_workload("tiny")
    assert line["config"] == bench.line_config("tiny", w, 1, 512 << 20)
    assert line["steps"] == 3 and line["warmup"] == 3


def test_workload_sizes():
    """Cache sizes and algorithmic bytes of the bench workloads, from their
    definitions: rows read, rows (and scales) written, slot ids read."""
    sys.path.insert(0, ROOT)
    import workloads as wl
    d = wl.decode()
    assert d.algorithmic_bytes() == 256 * (2 * 2048 + 2 * 2048 + 8)
    assert d.cache_bytes == (1 << 20) * 2048 and not d.paged
    f = wl.fp8()
    assert f.algorithmic_bytes() == 8192 * (2 * 2048 + 2 * 1024 + 8)
    fd = wl.fp8_dynamic()
    assert fd.kind == "fp8_dyn" and fd.algorithmic_bytes() == f.algorithmic_bytes() + 8192 * 2 * 8 * 4
    pg = wl.paged()
    assert pg.paged and pg.page_stride == 64 * 2048 + 2048
    assert pg.cache_bytes == (1 << 22) // 64 * pg.page_stride
    # whole pages: every page named holds 64 consecutive slots
    pages, counts = np.unique(pg.indices // 64, return_counts=True)
    assert len(pages) == 512 and (counts == 64).all()
    gp = wl.gather_prefill()
    assert gp.kind == "gather" and gp.algorithmic_bytes() == 32768 * (4 * 2048 + 4)
    o = wl.odd()
    assert o.slot_stride == 1280 and o.algorithmic_bytes() == 65536 * (4 * 1152 + 4)


def test_fused_dynamic_workload_and_oracle_step():
    """The fused per-tensor dynamic write's workload counts K and V once plus
    the two scales, and the reference arm's oracle step for it equals the
    oracle's absmax followed by the per-tensor write on the same tokens."""
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    import workloads as wl
    w = wl.fp8_tensor_dynamic(n_slots=1 << 14)
    assert w.algorithmic_bytes() == wl.fp8(n_slots=1 << 14).algorithmic_bytes() + 8
    name = "fp8_tensor_dynamic_cpu_test"
    bench._ORACLE_CACHE.pop(name, None)
    tokens = 48
    kc, vc, k, v, st = bench.oracle_buffers(name, w)
    kc[:] = 0x7F
    vc[:] = 0x7F
    bench.oracle_step(name, w, tokens)
    amax, inv = oracle.absmax_inv(k, v, st, tokens, w.H, w.D, w.src_dtype, 448.0)
    okc = np.full_like(kc, 0x7F)
    ovc = okc.copy()
    oracle.store_fp8_ex(k, v, okc, ovc, w.indices, st, w.H, w.D, w.src_dtype, w.page_size,
                        w.page_stride, w.page_stride, w.n_slots, fmt="e4m3fn",
                        scale_mode="tensor", inv_k=float(inv[0]), inv_v=float(inv[1]),
                        t_end=tokens)
    assert np.array_equal(kc, okc) and np.array_equal(vc, ovc)
    assert (kc != 0x7F).sum() > 0
    bench._ORACLE_CACHE.pop(name, None)
