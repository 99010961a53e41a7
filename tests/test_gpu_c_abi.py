"""The library used from plain C: tests/c/abi_example.c and
tests/c/noalloc_reset.c are compiled with gcc against include/kvstore.h only,
linked with libkvstore.so and the CUDA runtime, and run; each checks its own
results and exits 0."""

import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _build_and_run(tmp_path, name):
    import __graft_entry__
    __graft_entry__.build()
    import fp8_quant_gb300 as kv
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    libdir = os.path.dirname(kv.LIB_PATH)
    exe = tmp_path / name
    subprocess.check_call(["gcc", "-std=c11", "-O1", "-o", str(exe),
                           os.path.join(HERE, "c", name + ".c"),
                           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                           "-L", libdir, "-lkvstore", "-L", os.path.join(cuda, "lib64"),
                           "-lcudart", f"-Wl,-rpath,{libdir}",
                           f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr + out.stdout
    assert f"{name}: ok" in out.stdout


def test_plain_c_caller(tmp_path):
    _build_and_run(tmp_path, "abi_example")


def test_noalloc_record_after_a_device_reset(tmp_path):
    """kv_store_noalloc keeps its record's device address per CUDA context:
    after cudaDeviceReset (a new context) the next call looks it up again and
    still writes the rows and reports the bad slot (tests/c/noalloc_reset.c,
    its own process)."""
    _build_and_run(tmp_path, "noalloc_reset")
