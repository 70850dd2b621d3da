"""The C-ABI library loads and exports every function include/zc.h declares
(CPU only: no call here touches a GPU)."""
import ctypes
import os
import re

import pytest

from lossless_bit_level_bf16_gb300 import abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "zc.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(zc_\w+|ibp_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(abi.LIB_PATH):
        import __graft_entry__ as g
        g.build()
    return abi.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 19, names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in zc.h but not exported"
    assert set(names) == set(abi.SIGNATURES), set(names) ^ set(abi.SIGNATURES)


def test_host_only_calls(lib):
    assert lib.zc_version() >= 100
    assert lib.zc_strerror(0) == b"ok"
    assert b"corrupt" in lib.zc_strerror(abi.ZC_ERR_FORMAT)
    assert lib.ibp_meta_bytes(512) == 64 + 1024
    assert lib.zc_decompress_workspace_bytes() == 256
    assert lib.ibp_workspace_bytes(512, 1 << 20, 0) >= 256
    assert lib.ibp_workspace_bytes(12, 1 << 20, 0) >= 256  # any multiple of 4 bytes
    assert lib.ibp_workspace_bytes(14, 1 << 20, 0) == 0  # not a multiple of 4
    assert lib.ibp_workspace_bytes(4100, 1 << 20, 0) == 0  # above 4096
    assert lib.ibp_max_compressed_bytes(512, 4096) > 4096


def test_argument_checks_need_no_gpu(lib):
    h = ctypes.c_void_p()
    # chunk size not a multiple of 1024 / too large / zero segments
    assert lib.zc_plan_create(100, None, 1, 1000, ctypes.byref(h)) == abi.ZC_ERR_ARG
    assert lib.zc_plan_create(100, None, 1, 1 << 17, ctypes.byref(h)) == abi.ZC_ERR_ARG
    assert lib.zc_plan_create(100, None, 0, 4096, ctypes.byref(h)) == abi.ZC_ERR_ARG
    # any multiple of 1024 up to 65536, powers of two or not, passes the
    # argument checks (without a GPU the plan's device table then fails)
    for C in (1024, 3072, 5120, 9216, 64512, 65536):
        rc = lib.zc_plan_create(100, None, 1, C, ctypes.byref(h))
        assert rc in (abi.ZC_OK, abi.ZC_ERR_CUDA, abi.ZC_ERR_NOMEM), (C, rc)
        if rc == abi.ZC_OK:
            lib.zc_plan_destroy(h)
    # bad segment offsets
    so = (ctypes.c_uint64 * 3)(0, 60, 50)
    assert lib.zc_plan_create(50, so, 2, 4096, ctypes.byref(h)) == abi.ZC_ERR_ARG
    assert lib.zc_compress(None, None, None, 0, None, None, 0, None) == abi.ZC_ERR_ARG
    assert lib.zc_decompress(None, 0, None, 0, None, 0, None) == abi.ZC_ERR_ARG
    assert lib.ibp_build_meta(None, 0, 512, 0.9, 0, None, None, 0, None) == abi.ZC_ERR_ARG
    assert lib.ibp_compress(None, 512, None, 0, None, 0, None, None, 0, None) == abi.ZC_ERR_ARG
    assert lib.ibp_decompress(None, 512, None, 0, None, 0, None, 0, None) == abi.ZC_ERR_ARG


def test_product_path_fails_loudly_without_library(tmp_path):
    with pytest.raises(abi.LibraryMissing):
        abi._lib_saved = abi._lib
        try:
            abi._lib = None
            abi.load(str(tmp_path / "missing.so"))
        finally:
            abi._lib = abi._lib_saved
