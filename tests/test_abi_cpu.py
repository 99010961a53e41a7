"""CPU checks of the C ABI: the library builds, loads and exports every symbol
``include/kvstore.h`` declares; host-side argument validation answers without
touching a GPU; and, with no GPU, a valid call reports a CUDA error rather
than doing the work anywhere else (there is no CPU fallback)."""

import ctypes
import os
import re
import subprocess

import pytest

import fp8_quant_gb300 as kv
from fp8_quant_gb300 import build as kvbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvstore.h")

# fake, never dereferenced device addresses (validation happens before any CUDA call)
A = 0x10000
S = (4096, 256, 2, 4096, 256, 2, 4096, 256, 2, 4096, 256, 2)
S8 = (4096, 256, 2, 4096, 256, 2, 2048, 128, 1, 2048, 128, 1)


@pytest.fixture(scope="module")
def lib():
    kvbuild.build()
    return kv.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \t\*]*?\b(kv_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_api():
    names = declared_functions()
    for n in ("kv_store", "kv_store_fp8", "kv_error_poll", "kv_error_reset", "kv_status_str",
              "kv_last_cuda_error", "kv_abi_version"):
        assert n in names
    assert len(names) >= 7


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in kvstore.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", kv.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported
    # nothing else of ours leaks out with C linkage
    assert {n for n in exported if n.startswith("kv_")} == set(declared_functions())


def test_abi_version_and_status_strings(lib):
    m = re.search(r"#define\s+KV_ABI_VERSION\s+(\d+)", open(HEADER).read())
    assert lib.kv_abi_version() == int(m.group(1))
    for code, name in [(0, "KV_OK"), (1, "KV_ERR_INVALID_ARG"), (2, "KV_ERR_UNSUPPORTED"),
                       (3, "KV_ERR_CUDA"), (4, "KV_ERR_INDEX_OOB")]:
        assert kv.kv_status_str(code) == name
        assert kv.KVStatus(code).value == code
    assert kv.kv_status_str(99) == "KV_STATUS_UNKNOWN"


def store(**over):
    a = dict(k=A, v=A, k_cache=A, v_cache=A, indices=A, index_dtype=0, index_stride=1,
             num_tokens=16, num_heads=8, head_dim=128, elem_bytes=2, strides=S,
             size_limit=100, num_split=0, d_err=A, stream=None)
    a.update(over)
    return kv.raw.kv_store(**a)


def store8(**over):
    a = dict(k=A, v=A, k_cache=A, v_cache=A, indices=A, index_dtype=1, index_stride=1,
             num_tokens=16, num_heads=8, head_dim=128, src_dtype=1, strides=S8, page_size=16,
             kc_page_stride=16 * 2048, vc_page_stride=16 * 2048, size_limit=100,
             inv_k_scale=A, inv_v_scale=A, use_scale=1, d_err=A, stream=None)
    a.update(over)
    return kv.raw.kv_store_fp8(**a)


INVALID, CUDA = kv.KVStatus.ERR_INVALID_ARG, kv.KVStatus.ERR_CUDA


@pytest.mark.parametrize("over", [
    dict(num_tokens=-1), dict(k=None), dict(v=None), dict(k_cache=None), dict(v_cache=None),
    dict(indices=None), dict(d_err=None), dict(d_err=A + 4), dict(index_dtype=2),
    dict(index_stride=0), dict(num_heads=0), dict(head_dim=0), dict(elem_bytes=3),
    dict(elem_bytes=16), dict(size_limit=-1), dict(num_split=3), dict(num_split=8),
    dict(num_split=4, head_dim=120),     # 8*120*2 = 1920 B is not a multiple of 512
    dict(num_split=2, num_heads=1, head_dim=64),   # 128 B is not a multiple of 256
])
def test_kv_store_rejects_bad_arguments(lib, over):
    assert store(**over) == INVALID


@pytest.mark.parametrize("over", [
    dict(num_tokens=-5), dict(src_dtype=2), dict(page_size=0), dict(inv_k_scale=None),
    dict(inv_v_scale=None), dict(inv_k_scale=A + 2), dict(k=A + 1), dict(v=A + 3),
    dict(strides=(4095,) + S8[1:]), dict(d_err=None), dict(index_stride=-1),
    dict(num_heads=-2),
])
def test_kv_store_fp8_rejects_bad_arguments(lib, over):
    assert store8(**over) == INVALID


def test_empty_batch_is_ok_without_pointers(lib):
    z = (0,) * 12
    assert kv.raw.kv_store(None, None, None, None, None, 0, 1, 0, 1, 1, 2, z, 0, 0, None,
                           None) == 0
    assert kv.raw.kv_store_fp8(None, None, None, None, None, 0, 1, 0, 1, 1, 1, z, 1, 0, 0, 0,
                               None, None, 0, None, None) == 0


def test_unscaled_fp8_ignores_scale_pointers(lib):
    # use_scale = 0: NULL scales are legal, so validation passes and the call
    # proceeds to CUDA, which has no device here.
    assert store8(use_scale=0, inv_k_scale=None, inv_v_scale=None) == CUDA


def test_valid_calls_need_a_gpu(lib):
    # Arguments are fine, so the library goes to the CUDA runtime, which has
    # no device in this container: the call fails instead of running elsewhere.
    assert store() == CUDA
    assert lib.kv_last_cuda_error() != 0
    assert store(num_split=4) == CUDA
    assert store8() == CUDA
    assert kv.raw.kv_error_reset(A, None) == CUDA
    assert kv.raw.kv_error_poll(A, None)[0] == CUDA
    assert kv.raw.kv_error_poll(None, None)[0] == INVALID
    assert kv.raw.kv_error_reset(A + 1, None) == INVALID
    assert kv.raw.kv_launch_floor(1024, None) == CUDA
    assert kv.raw.kv_launch_floor(0, None) == INVALID
    assert kv.raw.kv_launch_floor(-3, None) == INVALID


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        kv.load_library(str(tmp_path / "nope.so"))


def store8ex(**over):
    a = dict(k=A, v=A, k_cache=A, v_cache=A, indices=A, index_dtype=1, index_stride=1,
             num_tokens=16, num_heads=8, head_dim=128, src_dtype=1, strides=S8, page_size=16,
             kc_page_stride=16 * 2048, vc_page_stride=16 * 2048, size_limit=100, fmt=0,
             scale_mode=4, inv_k_scale=A, inv_v_scale=A, k_scales=None, v_scales=None,
             scales_slot_stride=0, d_err=A, stream=None)
    a.update(over)
    return kv.raw.kv_store_fp8_ex(**a)


def gather8ex(**over):
    a = dict(k_cache=A, v_cache=A, k_out=A, v_out=A, indices=A, index_dtype=1, index_stride=1,
             num_tokens=16, num_heads=8, head_dim=128, out_dtype=1, strides=S8, page_size=16,
             kc_page_stride=16 * 2048, vc_page_stride=16 * 2048, size_limit=100, fmt=0,
             scale_mode=4, k_scale=A, v_scale=A, k_scales=None, v_scales=None,
             scales_slot_stride=0, d_err=A, stream=None)
    a.update(over)
    return kv.raw.kv_gather_fp8_ex(**a)


@pytest.mark.parametrize("over", [
    dict(inv_k_scale=None), dict(inv_v_scale=None), dict(inv_k_scale=A + 2), dict(page_size=0),
    dict(scale_mode=5), dict(scale_mode=-1), dict(fmt=2),
])
def test_per_page_scale_mode_rejects_bad_arguments(lib, over):
    assert store8ex(**over) == INVALID
    g = {("k_scale" if k == "inv_k_scale" else "v_scale" if k == "inv_v_scale" else k): x
         for k, x in over.items()}
    assert gather8ex(**g) == INVALID


def test_per_page_scale_mode_valid_calls_need_a_gpu(lib):
    assert store8ex() == CUDA
    assert gather8ex() == CUDA


def store8dyn(**over):
    a = dict(k=A, v=A, k_cache=A, v_cache=A, indices=A, index_dtype=1, index_stride=1,
             num_tokens=16, num_heads=8, head_dim=128, src_dtype=1, strides=S8, page_size=16,
             kc_page_stride=16 * 2048, vc_page_stride=16 * 2048, size_limit=100, fmt=0,
             k_scale=A, v_scale=A + 4, work=A, d_err=A, stream=None)
    a.update(over)
    return kv.raw.kv_store_fp8_dynamic_tensor(**a)


@pytest.mark.parametrize("over", [
    dict(k_scale=None), dict(v_scale=None), dict(work=None), dict(work=A + 4),
    dict(k_scale=A + 2), dict(fmt=2), dict(num_tokens=-1), dict(d_err=None), dict(page_size=0),
    dict(src_dtype=2), dict(k=A + 1), dict(strides=(4097,) + S8[1:]),
])
def test_dynamic_tensor_write_rejects_bad_arguments(lib, over):
    """Every argument error is found before anything is launched (a reduction
    that ran without its write would leave the workspace mid-call)."""
    assert store8dyn(**over) == INVALID


def test_dynamic_tensor_write_dims_and_empty_batch(lib):
    assert store8dyn(strides=(4096, 256, 4) + S8[3:]) == kv.KVStatus.ERR_UNSUPPORTED
    assert store8dyn(num_tokens=0, k=None, v=None, k_cache=None, v_cache=None, indices=None,
                     d_err=None) == 0
    assert store8dyn() == CUDA          # valid arguments: the device checks need a GPU
