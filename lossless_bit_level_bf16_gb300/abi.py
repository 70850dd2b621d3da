"""ctypes binding of liblbb16.so (declared in include/zc.h).

Argument marshalling only: pointers, sizes and the CUDA stream handle go
through unchanged; every step of both codecs runs in the library's kernels.
Loading fails loudly (``LibraryMissing``) when the library has not been built:
there is no CPU fallback.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liblbb16.so")

ZC_OK = 0
ZC_ERR_ARG = -1
ZC_ERR_CAPACITY = -2
ZC_ERR_FORMAT = -3
ZC_ERR_META_MISMATCH = -4
ZC_ERR_TIMEOUT = -5
ZC_ERR_CUDA = -6
ZC_ERR_UNSUPPORTED = -7
ZC_ERR_NOMEM = -8

# every exported symbol of include/zc.h with (restype, argtypes)
_vp, _u8p, _u64p, _dp = C.c_void_p, C.POINTER(C.c_uint8), C.POINTER(C.c_uint64), C.POINTER(C.c_double)
SIGNATURES = {
    "zc_strerror": (C.c_char_p, [C.c_int]),
    "zc_version": (C.c_int, []),
    "zc_test_wait_fault": (C.c_int, [C.c_uint64, C.c_uint32]),
    "zc_test_ibp_single_pass": (C.c_int, [C.c_int]),
    "zc_status": (C.c_int, [_vp, _vp, C.POINTER(C.c_int)]),
    "zc_plan_create": (C.c_int, [C.c_uint64, _u64p, C.c_uint32, C.c_uint32, C.POINTER(_vp)]),
    "zc_plan_destroy": (None, [_vp]),
    "zc_workspace_bytes": (C.c_size_t, [_vp]),
    "zc_max_compressed_bytes": (C.c_uint64, [_vp]),
    "zc_plan": (C.c_int, [_vp, _vp, _vp, C.c_size_t, _vp]),
    "zc_plan_set_books": (C.c_int, [_vp, _u8p]),
    "zc_plan_info": (C.c_int, [_vp, _vp, _u8p, _dp]),
    "zc_compress": (C.c_int, [_vp, _vp, _vp, C.c_uint64, _vp, _vp, C.c_size_t, _vp]),
    "zc_compress_static": (C.c_int, [_vp, _vp, _vp, C.c_uint64, _vp, _vp, _vp]),
    "zc_compress_fit": (C.c_int, [_vp, _vp, _vp, C.c_uint64, _vp, _vp, C.c_size_t, _vp]),
    "zc_decompress_workspace_bytes": (C.c_size_t, []),
    "zc_decompress": (C.c_int, [_vp, C.c_uint64, _vp, C.c_uint64, _vp, C.c_size_t, _vp]),
    "ibp_meta_bytes": (C.c_uint64, [C.c_uint32]),
    "ibp_workspace_bytes": (C.c_size_t, [C.c_uint32, C.c_uint64, C.c_uint64]),
    "ibp_max_compressed_bytes": (C.c_uint64, [C.c_uint32, C.c_uint64]),
    "ibp_build_meta": (C.c_int, [_vp, C.c_uint64, C.c_uint32, C.c_double, C.c_int, _vp, _vp,
                                 C.c_size_t, _vp]),
    "ibp_compress": (C.c_int, [_vp, C.c_uint32, _vp, C.c_uint64, _vp, C.c_uint64, _vp, _vp,
                               C.c_size_t, _vp]),
    "ibp_decompress": (C.c_int, [_vp, C.c_uint32, _vp, C.c_uint64, _vp, C.c_uint64, _vp,
                                 C.c_size_t, _vp]),
    "ibp_slots_compress": (C.c_int, [_vp, C.c_uint32, _vp, C.c_uint64, _vp, _vp, _vp, C.c_size_t,
                                     _vp]),
    "ibp_slots_gather": (C.c_int, [_vp, C.c_uint32, _vp, C.c_uint64, _vp, _vp, C.c_uint64, _vp,
                                   _vp, _vp, C.c_size_t, _vp]),
}


class LibraryMissing(RuntimeError):
    pass


class CodecError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


_lib = None


def load(path: str = LIB_PATH):
    """Load the library (once) and attach the signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise LibraryMissing(
            f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    L = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return _lib


def strerror(code: int) -> str:
    try:
        return load().zc_strerror(code).decode()
    except LibraryMissing:
        return f"error {code}"


def check(rc: int, what: str):
    if rc != ZC_OK:
        raise CodecError(rc, what)


def stream_handle(stream=None):
    """The raw cudaStream_t of a torch stream (current stream if None)."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else C.c_void_p(0)


def status(ws, stream=None) -> int:
    v = C.c_int(0)
    check(load().zc_status(ptr(ws), stream_handle(stream), C.byref(v)), "zc_status")
    return v.value
