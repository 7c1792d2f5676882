"""CPU tests of the C-ABI library: it loads, exports every symbol the header
declares, and the calls that need no GPU behave (no compute without a GPU)."""
import ctypes
import os
import re

import pytest

import mla_decode_attention_09_gb300 as mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla_decode.h")


@pytest.fixture(scope="module")
def lib():
    from mla_decode_attention_09_gb300 import build
    build.build()
    return mla.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(mla_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_header_declares_the_binding_exports():
    assert _declared_functions() == sorted(mla.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    # exported as plain C symbols from the shared object itself
    dl = ctypes.CDLL(mla.LIB_PATH)
    for name in _declared_functions():
        assert ctypes.cast(getattr(dl, name), ctypes.c_void_p).value


def test_strerror_and_version(lib):
    for code, name in mla.STATUS.items():
        s = lib.mla_strerror(code).decode()
        assert s and s != "unknown status", (code, name)
    assert lib.mla_strerror(12345).decode() == "unknown status"
    assert lib.mla_version() >= 100


def test_null_arguments_are_rejected_without_a_gpu(lib):
    # argument checks run before any CUDA call
    assert lib.mla_decode_plan(1, None, 0, None) == -1
    assert lib.mla_plan_release(None) == -1
    assert lib.mla_plan_get_info(None, None) == -1
    assert lib.mla_plan_destroy(None) == -1
    assert lib.mla_plan_workspace_bytes(None) == 0
    assert lib.mla_decode_reduce(None, None, None) == -1
    assert lib.mla_plan_check_error(None, None) == -1
    args = [None] * 6 + [ctypes.c_float(0.1), 0, None, None]
    assert lib.mla_decode(*args) == -1
    assert lib.mla_decode_stage1(*args) == -1
    assert lib.mla_plan_compute_host(1, None, 4, None, None, None, 0, None, 0, None, 0) == -1


def test_sources_have_no_cpu_fallback():
    # the product path is the CUDA library only: nothing in the package imports the oracle
    pkg = os.path.dirname(mla.__file__)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cpp", ".h", ".cuh")):
                text = open(os.path.join(dirpath, f), errors="ignore").read()
                assert "import oracle" not in text and "from oracle" not in text and "liboracle" not in text, f


def test_missing_library_fails_loudly(tmp_path):
    # without the compiled library every entry raises; nothing falls back to a CPU path
    with pytest.raises(OSError):
        mla.load_library(str(tmp_path / "libmla_decode.so"))
