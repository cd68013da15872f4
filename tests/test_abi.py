"""CPU checks of the C ABI: the library loads without a GPU, exports every
function include/fp8lin.h declares, and rejects bad arguments on the host
before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8lin.h")


@pytest.fixture(scope="module")
def lib():
    from fp8_mixed_precision_history_gb300 import build

    if not build.up_to_date():
        build.build()
    import fp8_mixed_precision_history_gb300 as fp8

    return fp8.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(fp8_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_path_calls():
    names = declared_functions()
    for must in ("fp8_recipe_create", "fp8_amax_quantize", "fp8_gemm", "fp8_update_scales"):
        assert must in names
    assert len(names) >= 10


def test_every_declared_symbol_is_exported(lib):
    import fp8_mixed_precision_history_gb300 as fp8

    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(fp8.EXPORTS)


def test_library_does_not_link_the_driver(lib):
    import shutil
    import subprocess

    from fp8_mixed_precision_history_gb300 import build

    if shutil.which("readelf") is None:
        pytest.skip("readelf not available")
    dyn = subprocess.run(["readelf", "-d", build.LIB], capture_output=True, text=True).stdout
    needed = re.findall(r"\(NEEDED\).*\[(.+?)\]", dyn)
    assert needed and not any(n.startswith("libcuda") for n in needed), needed


def test_status_strings(lib):
    import fp8_mixed_precision_history_gb300 as fp8

    assert fp8.fp8_status_string(0) == "ok"
    assert "invalid" in fp8.fp8_status_string(1)
    assert fp8.fp8_status_string(99) == "unknown status"


def test_create_rejects_bad_arguments_before_cuda(lib):
    h = ctypes.c_void_p()
    assert lib.fp8_recipe_create(None, 0, 16, 0, 1, None) == 1
    assert lib.fp8_recipe_create(ctypes.byref(h), 7, 16, 0, 1, None) == 1
    assert lib.fp8_recipe_create(ctypes.byref(h), 0, 0, 0, 1, None) == 1
    assert lib.fp8_recipe_create(ctypes.byref(h), 0, 16, 9, 1, None) == 1
    assert lib.fp8_recipe_create(ctypes.byref(h), 0, 16, 0, 0, None) == 1
    assert b"num_tensors" in lib.fp8_last_error_message()


def test_calls_on_null_recipe_are_invalid(lib):
    assert lib.fp8_amax_quantize(None, 0, 16, 1, 16, 0, 0, 0, 16, None, None) == 1
    assert lib.fp8_gemm(None, 0, 16, 0, 16, 0, 16, 0, 16, 16, 16, 16, 16, 0, 16, -1, None) == 1
    assert lib.fp8_gemm_layout(None, 0, 16, 0, 1, 16, 0, 16, 0, 1, 16, 16, 16, 16, 16, 0, 16, -1, None) == 1
    assert lib.fp8_update_scales(None, None) == 1
    assert lib.fp8_check_device_error(None, None) == 1
    assert lib.fp8_recipe_destroy(None) == 0


def test_create_without_a_gpu_reports_cuda_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    assert lib.fp8_recipe_create(ctypes.byref(h), 0, 16, 0, 4, None) == 3
    assert h.value is None


def test_binding_raises_with_message(lib):
    import fp8_mixed_precision_history_gb300 as fp8

    with pytest.raises(fp8.Fp8Error) as e:
        fp8.fp8_recipe_create(num_tensors=0, stream=0)
    assert e.value.status == 1 and "num_tensors" in str(e.value)


def test_mx_calls_check_arguments_before_cuda(lib):
    import fp8_mixed_precision_history_gb300 as fp8

    assert lib.fp8_mx_quantize(None, None, 16, 16, 0, None, None, None, None, None) == 1
    assert lib.fp8_mx_gemm(None, None, 0, 16, None, None, 0, 16, None, 16, 16, 16, None, 0, 16, None) == 1
    assert fp8.fp8_mx_scale_bytes(1, 1) == 512
    assert fp8.fp8_mx_scale_bytes(129, 128) == 1024
    assert fp8.fp8_mx_scale_bytes(300, 1000) == 3 * 8 * 512
    assert fp8.fp8_mx_scale_bytes(0, 16) == -1


def test_grad_allreduce_calls_check_arguments_before_cuda(lib):
    assert lib.fp8_grad_amax(None, 16, None, None) == 1
    assert lib.fp8_grad_quantize(None, 16, None, 2, None, 16, None, None) == 1
    assert lib.fp8_grad_reduce(None, 2, 16, None, None) == 1
    assert lib.fp8_grad_dequantize(None, 16, None, 2, 0, None, None) == 1
