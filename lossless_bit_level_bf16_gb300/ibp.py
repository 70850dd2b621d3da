"""IBP invariant bit packing (Python side of ibp_build_meta / ibp_compress /
ibp_decompress).

Page: "Riepilogo Tecnico: Riduzione del Collo di Bottiglia della Memoria GPU
con la Compressione Lossless per il ML", Metodologia: Invariant Bit Packing
(IBP), Algoritmo Core steps 1-3.  This module allocates buffers with torch and
passes pointers; the metadata reduction, the packing and the unpacking run in
the CUDA kernels of liblbb16.so.
"""
from __future__ import annotations

import torch

from . import abi


def _dev_tensor(x: torch.Tensor, name: str):
    if not x.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return x


def workspace_bytes(chunk_bytes: int, n_bytes: int = 0, n_samples: int = 0) -> int:
    return int(abi.load().ibp_workspace_bytes(chunk_bytes, n_bytes, n_samples))


def max_compressed_bytes(chunk_bytes: int, n_bytes: int) -> int:
    return int(abi.load().ibp_max_compressed_bytes(chunk_bytes, n_bytes))


def build_meta(samples: torch.Tensor, chunk_bytes: int, T: float = 0.9, mode: int = 0,
               meta: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None):
    """ibp_build_meta: the IBPM blob (uint8 CUDA tensor) from the sample
    chunks laid end to end in ``samples`` (any dtype; its bytes are used)."""
    lib = abi.load()
    samples = _dev_tensor(samples, "samples")
    nbytes = samples.numel() * samples.element_size()
    if nbytes % chunk_bytes:
        raise ValueError("samples must hold a whole number of chunks")
    n_samples = nbytes // chunk_bytes
    if meta is None:
        meta = torch.empty(int(lib.ibp_meta_bytes(chunk_bytes)), dtype=torch.uint8,
                           device=samples.device)
    if ws is None:
        ws = torch.empty(max(workspace_bytes(chunk_bytes, 0, n_samples), 256), dtype=torch.uint8,
                         device=samples.device)
    abi.check(lib.ibp_build_meta(abi.ptr(samples), n_samples, chunk_bytes, float(T), int(mode),
                                 abi.ptr(meta), abi.ptr(ws), ws.numel(), abi.stream_handle(stream)),
              "ibp_build_meta")
    meta._lbb_ws = ws  # keep the workspace alive until the kernels ran
    return meta


def _reachable(x: torch.Tensor, name: str):
    """A CUDA tensor, or a pinned host tensor the GPU reads in place."""
    if not (x.is_cuda or x.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return x


def compress(meta: torch.Tensor, x: torch.Tensor, chunk_bytes: int, out: torch.Tensor | None = None,
             out_bytes: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None):
    """ibp_compress: returns (stream uint8 tensor, out_bytes int64[1] tensor)
    on the device; nothing is synchronised.  ``x`` and ``out`` may be pinned
    host tensors (read and written in place over the host link)."""
    lib = abi.load()
    x = _reachable(x, "x")
    if out is not None:
        _reachable(out, "out")
    dev = meta.device  # workspace and size word live on the metadata's GPU
    n_bytes = x.numel() * x.element_size()
    if out is None:
        out = torch.empty(max_compressed_bytes(chunk_bytes, n_bytes), dtype=torch.uint8,
                          device=dev)
    if out_bytes is None:
        out_bytes = torch.zeros(1, dtype=torch.int64, device=dev)
    if ws is None:
        ws = torch.empty(max(workspace_bytes(chunk_bytes, n_bytes, 0), 256), dtype=torch.uint8,
                         device=dev)
    abi.check(lib.ibp_compress(abi.ptr(meta), chunk_bytes, abi.ptr(x), n_bytes, abi.ptr(out),
                               out.numel(), abi.ptr(out_bytes), abi.ptr(ws), ws.numel(),
                               abi.stream_handle(stream)), "ibp_compress")
    out._lbb_ws = ws
    return out, out_bytes


def decompress(meta: torch.Tensor, stream_bytes: torch.Tensor, n_bytes: int, chunk_bytes: int,
               out: torch.Tensor | None = None, in_bytes: int | None = None,
               ws: torch.Tensor | None = None, stream=None, dtype=torch.float32):
    """ibp_decompress: decode into a new tensor of ``n_bytes`` bytes viewed as
    ``dtype`` (or into ``out``).  ``stream_bytes`` may be a pinned host tensor:
    the kernel then reads the stream in place over the host link."""
    lib = abi.load()
    _reachable(stream_bytes, "stream_bytes")
    if out is not None:
        _reachable(out, "out")
    # a pinned host stream is decoded in place; by default the output lives
    # on the metadata's GPU
    dev = meta.device
    if out is None:
        esize = torch.empty(0, dtype=dtype).element_size()
        out = torch.empty(n_bytes // esize, dtype=dtype, device=dev)
    if ws is None:
        ws = torch.empty(256, dtype=torch.uint8, device=dev)
    if in_bytes is None:
        in_bytes = stream_bytes.numel()
    abi.check(lib.ibp_decompress(abi.ptr(meta), chunk_bytes, abi.ptr(stream_bytes), in_bytes,
                                 abi.ptr(out), out.numel() * out.element_size(), abi.ptr(ws),
                                 ws.numel(), abi.stream_handle(stream)), "ibp_decompress")
    out._lbb_ws = ws
    return out


def slots_compress(meta: torch.Tensor, x: torch.Tensor, chunk_bytes: int,
                   slots: torch.Tensor | None = None, bitmask: torch.Tensor | None = None,
                   ws: torch.Tensor | None = None, stream=None):
    """ibp_slots_compress: the in-place slot form of ``x`` and the bitmask of
    compressed slots.  ``slots`` defaults to ``x`` itself (compression in
    place); either may be pinned host memory.  Returns (slots, bitmask int32
    CUDA tensor)."""
    lib = abi.load()
    x = _reachable(x, "x")
    slots = x if slots is None else _reachable(slots, "slots")
    dev = meta.device
    n_bytes = x.numel() * x.element_size()
    nch = (n_bytes + chunk_bytes - 1) // chunk_bytes
    if bitmask is None:
        bitmask = torch.zeros(max(1, (nch + 31) // 32), dtype=torch.int32, device=dev)
    if ws is None:
        ws = torch.empty(256, dtype=torch.uint8, device=dev)
    abi.check(lib.ibp_slots_compress(abi.ptr(meta), chunk_bytes, abi.ptr(x), n_bytes,
                                     abi.ptr(slots), abi.ptr(bitmask), abi.ptr(ws), ws.numel(),
                                     abi.stream_handle(stream)), "ibp_slots_compress")
    bitmask._lbb_ws = ws
    return slots, bitmask


def slots_gather(meta: torch.Tensor, slots: torch.Tensor, n_bytes: int, chunk_bytes: int,
                 bitmask: torch.Tensor, idx: torch.Tensor, out: torch.Tensor | None = None,
                 read_bytes: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                 stream=None, dtype=torch.float32):
    """ibp_slots_gather: chunks ``idx`` (int64 CUDA tensor) decoded from their
    slots into rows [len(idx), chunk_bytes] viewed as ``dtype`` (or into
    ``out``).  Returns (rows, read_bytes int64[1])."""
    lib = abi.load()
    _reachable(slots, "slots")
    idx = _dev_tensor(idx, "idx")
    if idx.dtype != torch.int64:
        raise ValueError("idx must be int64")
    dev = meta.device
    if out is None:
        esize = torch.empty(0, dtype=dtype).element_size()
        out = torch.zeros(idx.numel(), chunk_bytes // esize, dtype=dtype, device=dev)
    if read_bytes is None:
        read_bytes = torch.zeros(1, dtype=torch.int64, device=dev)
    if ws is None:
        ws = torch.empty(256, dtype=torch.uint8, device=dev)
    abi.check(lib.ibp_slots_gather(abi.ptr(meta), chunk_bytes, abi.ptr(slots), n_bytes,
                                   abi.ptr(bitmask), abi.ptr(idx), idx.numel(), abi.ptr(out),
                                   abi.ptr(read_bytes), abi.ptr(ws), ws.numel(),
                                   abi.stream_handle(stream)), "ibp_slots_gather")
    out._lbb_ws = ws
    return out, read_bytes


def status(ws: torch.Tensor, stream=None) -> int:
    return abi.status(ws, stream)
