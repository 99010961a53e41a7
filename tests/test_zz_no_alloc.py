"""kv_store_noalloc: the entry point for callers that cannot allocate device
memory (code inside allocator hooks, plugins without a memory pool, processes
whose device memory is all reserved by a pool they do not own).

It must write exactly what kv_store writes, and report out-of-range slots
through its own static record, which every call clears first. Two calls in a
row are checked against kv_store through the C ABI: the first call has bad
slots, so the record is dirty; the second call is clean and must report zero.
The copy is byte-exact, so the comparison is too.

This file is collected last on purpose, and it must also pass alone in a
fresh process: its first call is also the first use of the static record on
the device.
"""

import numpy as np
import pytest

import workloads as wl
from kvcheck import DeviceRun, copy_problem, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    yield


def _noalloc_call(g):
    import fp8_quant_gb300 as kv
    p = g.p
    return kv.raw.kv_store_noalloc(
        g.k_src.data_ptr() + p.k_view.offset, g.v_src.data_ptr() + p.v_view.offset,
        g.kc.data_ptr() + p.kc_view.offset, g.vc.data_ptr() + p.vc_view.offset,
        g.idx.data_ptr(), 1 if p.indices.dtype == np.int64 else 0, p.index_stride, p.T, p.H,
        p.D, p.elem, p.strides(), p.size_limit, p.num_split,
        g.torch.cuda.current_stream(g.dev).cuda_stream)


def test_noalloc_matches_kv_store_on_two_calls_in_a_row():
    T, n = 700, 4096
    bad_slots = wl.distinct_slots(501, n, T)
    bad_slots[[4, 9, 650]] = [-1, n, 2 ** 40]
    problems = [
        copy_problem(T=T, H=8, D=128, n_slots=n, seed=502, slots=bad_slots),
        copy_problem(T=T, H=8, D=128, n_slots=n, seed=503, idx_dtype=np.int32),
    ]
    expect = [(4, 3, 4), (0, 0, -1)]          # (status, oob_count, first_bad_token)
    for p, (want_rc, want_n, want_first) in zip(problems, expect):
        ref = DeviceRun(p)                       # existing entry point, caller's record
        assert ref.call() == 0
        ref_rc, ref_n, ref_first = ref.poll()
        new = DeviceRun(p)                       # same inputs, fresh sentinel caches
        rc, nbad, first = _noalloc_call(new)
        assert (ref_rc, ref_n, ref_first) == (want_rc, want_n, want_first)
        assert (rc, nbad, first) == (want_rc, want_n, want_first)
        rk, rv = ref.caches()
        nk, nv = new.caches()
        assert np.array_equal(nk, rk) and np.array_equal(nv, rv)
        # and both equal the oracle
        ok, ov, _ = run_oracle(p)
        assert np.array_equal(nk, ok) and np.array_equal(nv, ov)


def test_noalloc_argument_errors_and_empty_batch():
    import fp8_quant_gb300 as kv
    zeros = (0,) * 12
    assert kv.raw.kv_store_noalloc(None, None, None, None, None, 0, 1, 0, 8, 128, 2, zeros, 0, 0,
                                   None) == (0, 0, -1)
    p = copy_problem(T=16, H=2, D=64, n_slots=64, seed=504, num_split=4)   # 256 B rows
    g = DeviceRun(p)
    rc, _, _ = _noalloc_call(g)
    assert rc == kv.KVStatus.ERR_INVALID_ARG                               # split rule
