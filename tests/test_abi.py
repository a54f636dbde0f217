"""The C-ABI library loads, exports what include/fp8w8a8.h declares, and
rejects bad arguments on the host before any CUDA work (no GPU needed)."""
import ctypes
import re

import pytest

from fp8_w8a8_quantized_group_gb300 import _lib, build

FAKE = 0x10000  # 16-byte aligned non-null address; never dereferenced on the error paths
ODD = FAKE + 8  # 8-byte aligned only


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


@pytest.fixture
def host_only(lib):
    """The library for calls with fake device addresses, which only the
    host-side checks keep from reaching a kernel: not used where a GPU is
    visible, so that a regression of those checks cannot launch on them."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-side argument checks are tested where no GPU is visible")
    return lib


def test_header_declares_the_entry_points():
    names = _lib.header_functions()
    for n in ["fp8_quant_act_group", "fp8_quant_weight_block", "fp8_quant_per_tensor", "fp8_block_gemm",
              "fp8_tensor_gemm", "fp8_block_linear"]:
        assert n in names
    assert set(names) == set(_lib.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in _lib.header_functions():
        assert hasattr(lib, name), name


def test_status_codes_match_header(lib):
    text = open(_lib.HEADER).read()
    codes = dict((k, int(v)) for k, v in re.findall(r"(FP8_\w+)\s*=\s*(\d+)", text))
    assert {v: k for k, v in codes.items()} == _lib.STATUS
    for code in range(9):
        assert lib.fp8_status_string(code)
    assert lib.fp8_status_string(99) == b"unknown status"


@pytest.mark.usefixtures("host_only")
def test_quant_act_group_validation(lib):
    f = lib.fp8_quant_act_group
    assert f(FAKE, FAKE, FAKE, -1, 128, 128, None) == 2
    assert f(FAKE, FAKE, FAKE, 4, 100, 128, None) == 2      # K not a multiple of 128
    assert f(FAKE, FAKE, FAKE, 4, 0, 128, None) == 2        # K == 0
    assert f(FAKE, FAKE, FAKE, 4, 256, 64, None) == 4       # group size
    assert f(None, FAKE, FAKE, 4, 256, 128, None) == 1
    assert f(FAKE, None, FAKE, 4, 256, 128, None) == 1
    assert f(FAKE, FAKE, None, 4, 256, 128, None) == 1
    assert f(ODD, FAKE, FAKE, 4, 256, 128, None) == 3
    assert f(FAKE, FAKE, FAKE + 2, 4, 256, 128, None) == 3  # scales need 4 bytes
    assert f(None, None, None, 0, 256, 128, None) == 0      # M == 0 is a no-op


@pytest.mark.usefixtures("host_only")
def test_quant_weight_block_validation(lib):
    f = lib.fp8_quant_weight_block
    assert f(FAKE, FAKE, FAKE, 256, 256, 64, 128, None) == 4
    assert f(FAKE, FAKE, FAKE, 256, 256, 128, 256, None) == 4
    assert f(FAKE, FAKE, FAKE, 256, 200, 128, 128, None) == 2
    assert f(FAKE, FAKE, FAKE, -5, 256, 128, 128, None) == 2
    assert f(FAKE, ODD, FAKE, 256, 256, 128, 128, None) == 3
    assert f(None, None, None, 0, 256, 128, 128, None) == 0


@pytest.mark.usefixtures("host_only")
def test_quant_per_tensor_validation(lib):
    f = lib.fp8_quant_per_tensor
    assert f(FAKE, FAKE, FAKE, 4, 24, 0, None) == 2          # cols % 16
    assert f(FAKE, FAKE, None, 4, 32, 0, None) == 1          # scale slot required
    assert f(None, FAKE, FAKE, 4, 32, 0, None) == 1
    assert f(FAKE, FAKE, FAKE + 1, 4, 32, 0, None) == 3
    assert f(None, None, FAKE, 0, 32, 1, None) == 0          # empty static: no-op


@pytest.mark.usefixtures("host_only")
def test_block_gemm_validation(lib):
    f = lib.fp8_block_gemm
    ok = (FAKE, FAKE, FAKE, FAKE, FAKE)
    assert f(*ok, 16, 256, 256, 64, 128, 128, 1, None, None) == 4
    assert f(*ok, 16, 256, 256, 128, 128, 128, 0, None, None) == 5   # num_groups
    assert f(*ok, 16, 256, 256, 128, 128, 128, 257, FAKE, None) == 4
    assert f(*ok, 16, 256, 256, 128, 128, 128, 4, None, None) == 5   # offsets required
    assert f(*ok, 16, 250, 256, 128, 128, 128, 1, None, None) == 2   # N % 16
    assert f(*ok, 16, 256, 192, 128, 128, 128, 1, None, None) == 2   # K % 128
    assert f(*ok, -1, 256, 256, 128, 128, 128, 1, None, None) == 2
    assert f(FAKE, None, FAKE, FAKE, FAKE, 16, 256, 256, 128, 128, 128, 1, None, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, ODD, 16, 256, 256, 128, 128, 128, 1, None, None) == 3
    assert f(*ok, 16, 256, 256, 128, 128, 128, 2, FAKE + 2, None) == 3
    assert f(None, None, None, None, None, 0, 256, 256, 128, 128, 128, 1, None, None) == 0


@pytest.mark.usefixtures("host_only")
def test_tensor_gemm_validation(lib):
    f = lib.fp8_tensor_gemm
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 24, None) == 2
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 24, 256, None) == 2
    assert f(FAKE, FAKE, None, FAKE, FAKE, 4, 256, 256, None) == 1
    assert f(ODD, FAKE, FAKE, FAKE, FAKE, 4, 256, 256, None) == 3
    assert f(None, None, None, None, None, 0, 256, 256, None) == 0


@pytest.mark.usefixtures("host_only")
def test_block_linear_validation(lib):
    f = lib.fp8_block_linear
    ok6 = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
    assert f(*ok6, 4, 256, 200, None) == 2            # K % 128
    assert f(*ok6, 4, 250, 256, None) == 2            # N % 16
    assert f(FAKE, None, FAKE, FAKE, FAKE, FAKE, 4, 256, 256, None) == 1
    assert f(FAKE, FAKE, FAKE + 2, FAKE, FAKE, FAKE, 4, 256, 256, None) == 3
    assert f(None, None, None, None, None, None, 0, 256, 256, None) == 0


def test_valid_call_without_gpu_fails_loudly(lib):
    """On a machine without a usable sm_103 GPU a well-formed call reports an
    error status instead of computing anything (there is no CPU fallback)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = lib.fp8_quant_act_group(FAKE, FAKE, FAKE, 4, 256, 128, None)
    assert st in (6, 7)
    code = ctypes.c_int(0)
    assert lib.fp8_device_error(None, ctypes.byref(code), None) in (6, 7)


def test_python_binding_names_match_header():
    import fp8_w8a8_quantized_group_gb300 as pkg
    for name in _lib.header_functions():
        assert callable(getattr(pkg, name)), name


def test_header_compiles_as_c_and_links(lib, tmp_path):
    """A C11 client (tests/abi_client.c) compiles against include/fp8w8a8.h
    with gcc in pedantic mode, with no C++ or CUDA header, links the library
    and gets the expected statuses for calls that are refused on the host."""
    import os
    import subprocess

    here = os.path.dirname(os.path.abspath(__file__))
    exe = str(tmp_path / "abi_client")
    libdir = os.path.dirname(_lib.LIB_PATH)
    subprocess.run(["gcc", "-std=c11", "-pedantic", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.dirname(_lib.HEADER), os.path.join(here, "abi_client.c"), "-o", exe,
                    "-L", libdir, "-lfp8w8a8", f"-Wl,-rpath,{libdir}"], check=True)
    import torch
    if torch.cuda.is_available():
        # The client passes fake device addresses that only the host checks
        # keep from being used; it is not run where a regression of those
        # checks could launch a kernel on them.
        pytest.skip("compiled and linked; run only where no GPU is visible")
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip().endswith("checks passed")
