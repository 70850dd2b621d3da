"""ZipCCL exponent coding of bf16 tensors (Python side of zc_plan /
zc_compress / zc_decompress).

Page: "ZipCCL: Efficient Lossless Data Compression of Communication
Collectives for Accelerating LLM Training", 2. Metodologia A-D.  The Python
code only allocates buffers with torch and passes pointers; the statistics,
the codebook prediction, the encoding and the decoding run in the CUDA
kernels of liblbb16.so.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import abi


def _bits(x: torch.Tensor) -> torch.Tensor:
    if x.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"expected bf16 (or its 16-bit pattern), got {x.dtype}")
    if not x.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not x.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return x


class Plan:
    """Layout (segments, chunk size) plus the per-segment codebooks.

    ``seg_off``: element offsets [0, ..., n] of the segments (None: one
    segment).  Each segment gets its own codebook from its own statistics.
    """

    def __init__(self, n: int, seg_off=None, chunk_elems: int = 4096, device=None):
        self.lib = abi.load()
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.n = int(n)
        if seg_off is None:
            self.nseg = 1
            so = None
        else:
            arr = np.ascontiguousarray(np.asarray(seg_off, dtype=np.uint64))
            self.nseg = arr.size - 1
            so = arr.ctypes.data_as(C.POINTER(C.c_uint64))
            self._seg_off = arr
        self.chunk_elems = int(chunk_elems)
        h = C.c_void_p()
        with torch.cuda.device(self.device):
            abi.check(self.lib.zc_plan_create(self.n, so, self.nseg, self.chunk_elems, C.byref(h)),
                      "zc_plan_create")
        self._h = h
        self.workspace_bytes = int(self.lib.zc_workspace_bytes(h))
        self.max_compressed_bytes = int(self.lib.zc_max_compressed_bytes(h))
        # zeroed once: the status word reads 0 until an op reports an error
        self.ws = torch.zeros(self.workspace_bytes, dtype=torch.uint8, device=self.device)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            try:
                torch.cuda.synchronize(self.device)
            except Exception:
                pass
            self.lib.zc_plan_destroy(h)
            self._h = None

    def fit(self, x: torch.Tensor, stream=None, ws: torch.Tensor | None = None):
        """zc_plan: statistics and codebooks from x (asynchronous)."""
        x = _bits(x)
        if x.numel() != self.n:
            raise ValueError(f"plan is for {self.n} elements, tensor has {x.numel()}")
        w = self.ws if ws is None else ws
        abi.check(self.lib.zc_plan(self._h, abi.ptr(x), abi.ptr(w), w.numel(),
                                   abi.stream_handle(stream)), "zc_plan")
        return self

    def set_books(self, books):
        b = np.ascontiguousarray(np.asarray(books, dtype=np.uint8).reshape(-1))
        if b.size != 7 * self.nseg:
            raise ValueError("need 7 fields per segment")
        abi.check(self.lib.zc_plan_set_books(self._h, b.ctypes.data_as(C.POINTER(C.c_uint8))),
                  "zc_plan_set_books")

    def info(self, stream=None):
        """(books [nseg, 7] uint8, mu [nseg], sigma [nseg]); synchronises."""
        b = np.zeros(7 * self.nseg, np.uint8)
        ms = np.zeros(2 * self.nseg, np.float64)
        abi.check(self.lib.zc_plan_info(self._h, abi.stream_handle(stream),
                                        b.ctypes.data_as(C.POINTER(C.c_uint8)),
                                        ms.ctypes.data_as(C.POINTER(C.c_double))), "zc_plan_info")
        return b.reshape(self.nseg, 7), ms[0::2].copy(), ms[1::2].copy()

    def compress(self, x: torch.Tensor, out: torch.Tensor | None = None,
                 out_bytes: torch.Tensor | None = None, stream=None,
                 ws: torch.Tensor | None = None):
        """zc_compress: returns (out uint8 tensor, out_bytes int64[1] tensor),
        both on the device; nothing is synchronised."""
        x = _bits(x)
        if x.numel() != self.n:
            raise ValueError(f"plan is for {self.n} elements, tensor has {x.numel()}")
        if out is None:
            out = torch.empty(self.max_compressed_bytes, dtype=torch.uint8, device=self.device)
        if out_bytes is None:
            out_bytes = torch.zeros(1, dtype=torch.int64, device=self.device)
        w = self.ws if ws is None else ws
        abi.check(self.lib.zc_compress(self._h, abi.ptr(x), abi.ptr(out), out.numel(),
                                       abi.ptr(out_bytes), abi.ptr(w), w.numel(),
                                       abi.stream_handle(stream)), "zc_compress")
        return out, out_bytes

    def compress_fit(self, x: torch.Tensor, out: torch.Tensor | None = None,
                     out_bytes: torch.Tensor | None = None, stream=None,
                     ws: torch.Tensor | None = None):
        """zc_compress_fit: encode with the current codebooks and, from the
        same read, refit the plan's statistics and codebooks to ``x`` for the
        next call.  Returns (out, out_bytes) like compress."""
        x = _bits(x)
        if x.numel() != self.n:
            raise ValueError(f"plan is for {self.n} elements, tensor has {x.numel()}")
        if out is None:
            out = torch.empty(self.max_compressed_bytes, dtype=torch.uint8, device=self.device)
        if out_bytes is None:
            out_bytes = torch.zeros(1, dtype=torch.int64, device=self.device)
        w = self.ws if ws is None else ws
        abi.check(self.lib.zc_compress_fit(self._h, abi.ptr(x), abi.ptr(out), out.numel(),
                                           abi.ptr(out_bytes), abi.ptr(w), w.numel(),
                                           abi.stream_handle(stream)), "zc_compress_fit")
        return out, out_bytes

    def compress_static(self, x: torch.Tensor, out: torch.Tensor, out_bytes: torch.Tensor,
                        status: torch.Tensor | None = None, stream=None):
        """zc_compress_static: the caller passes every buffer (out, out_bytes
        int64[1], status int32[1] or None); nothing is allocated or synchronised."""
        x = _bits(x)
        if x.numel() != self.n:
            raise ValueError(f"plan is for {self.n} elements, tensor has {x.numel()}")
        abi.check(self.lib.zc_compress_static(self._h, abi.ptr(x), abi.ptr(out), out.numel(),
                                              abi.ptr(out_bytes), abi.ptr(status),
                                              abi.stream_handle(stream)), "zc_compress_static")
        return out, out_bytes

    def status(self, stream=None) -> int:
        return abi.status(self.ws, stream)


_dec_ws = {}


def decompress_workspace(device) -> torch.Tensor:
    d = torch.device(device)
    if d not in _dec_ws:
        n = int(abi.load().zc_decompress_workspace_bytes())
        _dec_ws[d] = torch.empty(max(n, 256), dtype=torch.uint8, device=d)
    return _dec_ws[d]


def decompress(stream_bytes: torch.Tensor, n: int | None = None, out: torch.Tensor | None = None,
               in_bytes: int | None = None, stream=None, ws: torch.Tensor | None = None):
    """zc_decompress: decode a ZCC1 stream (uint8 CUDA tensor) into bf16.

    ``n`` (element count) sizes the output when ``out`` is not given; if both
    are None the header is read from the device (a synchronising copy)."""
    lib = abi.load()
    if in_bytes is None:
        in_bytes = stream_bytes.numel()
    if out is None:
        if n is None:
            n = int(stream_bytes[16:24].cpu().numpy().view(np.uint64)[0])
        out = torch.empty(n, dtype=torch.bfloat16, device=stream_bytes.device)
    w = decompress_workspace(stream_bytes.device) if ws is None else ws
    abi.check(lib.zc_decompress(abi.ptr(stream_bytes), in_bytes, abi.ptr(out), out.numel(),
                                abi.ptr(w), w.numel(), abi.stream_handle(stream)), "zc_decompress")
    return out
