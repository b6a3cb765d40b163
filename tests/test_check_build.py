"""The MHC_CHECK build: device index checks that record a failure (site,
offset, extent) and skip the access, instead of faulting.

`python gemm_rms_sinkhorn_gb300/build.py --check` builds
libmhc_gb300_check.so beside the default library; MHC_GB300_CHECK=1 makes the
package load it, and conftest then asserts after every GPU test that no check
failed.  The self-test asks for one element past the end of a 16-element
buffer, which the check refuses before any access.
"""
import ctypes
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "gemm_rms_sinkhorn_gb300")


def test_default_library_has_no_checks():
    lib = ctypes.CDLL(os.path.join(PKG, "libmhc_gb300.so"))
    assert lib.mhc_testing_check_build() == 0


def test_check_library_reports_itself():
    path = os.path.join(PKG, "libmhc_gb300_check.so")
    if not os.path.exists(path):
        pytest.skip("the MHC_CHECK build is not built here")
    assert ctypes.CDLL(path).mhc_testing_check_build() == 1


def test_check_sources_compile_with_the_flag(tmp_path):
    """Source files compile with -DMHC_CHECK, the flag of the check library
    (the lighter translation units, unoptimised, so the CPU suite stays quick;
    the full check library is built on the GPU machine)."""
    import shutil
    from concurrent.futures import ThreadPoolExecutor

    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("no nvcc")

    def compile_one(name):
        cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O0", "-Xptxas", "-O0",
               "-std=c++17", "-DMHC_CHECK", "-I" + os.path.join(ROOT, "include"),
               "-I" + os.path.join(PKG, "csrc"), "-Xcompiler", "-fPIC", "-c",
               os.path.join(PKG, "csrc", name), "-o", str(tmp_path / (name + ".o"))]
        return name, subprocess.run(cmd, capture_output=True, text=True)

    names = ("apply.cu", "apply_e4m3.cu", "coeffs.cu", "rmsnorm_gemm.cu")
    with ThreadPoolExecutor(len(names)) as ex:
        for name, res in ex.map(compile_one, names):
            assert res.returncode == 0, (name, res.stderr[-2000:])


@pytest.mark.gpu
def test_check_selftest_records_the_refused_index():
    import gemm_rms_sinkhorn_gb300 as mhc

    st = mhc._lib.mhc_testing_check_selftest()
    if not mhc.CHECK_BUILD:
        assert st == mhc.MHC_ERR_UNSUPPORTED
        assert mhc.mhc_testing_check_record() == (0, 0, 0)
        return
    assert st == mhc.MHC_OK
    assert mhc.mhc_device_status() == mhc.MHC_ERR_BOUNDS
    assert mhc.mhc_testing_check_record() == (900, 16, 16)
    assert mhc.mhc_device_status() == mhc.MHC_OK
    assert mhc.mhc_testing_check_record() == (0, 0, 0)
