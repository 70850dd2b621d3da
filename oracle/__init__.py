"""Bit-serial CPU oracle for the ZipCCL exponent codec and IBP bit packing.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the product package never imports it.
It shares no code with the CUDA library: the C source here restates every
format constant on its own.

This module compiles ``oracle.c`` with gcc (``build()``) and wraps it with
ctypes + numpy.  Every wrapper returns numpy arrays / Python ints.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

OK, E_ARG, E_CAPACITY, E_FORMAT, E_META = 0, -1, -2, -3, -4


class OracleError(RuntimeError):
    def __init__(self, rc, what):
        super().__init__(f"oracle {what} failed with code {rc}")
        self.rc = rc


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (portable C11, no
    target-specific flags, floating-point contraction off)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))
    ):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(
        ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
         "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = C.CDLL(build())
        u8p, u16p, u64p = C.POINTER(C.c_uint8), C.POINTER(C.c_uint16), C.POINTER(C.c_uint64)
        dp = C.POINTER(C.c_double)
        sig = {
            "ora_zc_stats": (None, [u16p, C.c_uint64, u64p, dp, dp]),
            "ora_zc_moments": (None, [C.c_uint64, C.c_double, C.c_double, dp, dp]),
            "ora_zc_mass": (C.c_double, [C.c_double, C.c_double, C.c_int]),
            "ora_zc_predict": (None, [C.c_double, C.c_double, u8p]),
            "ora_zc_stream_bytes": (C.c_uint64, [C.c_uint64, C.c_uint32, u64p, C.c_uint32, C.c_uint64]),
            "ora_zc_encode": (C.c_int, [u16p, C.c_uint64, u64p, C.c_uint32, C.c_uint32, u8p,
                                        u8p, C.c_uint64, u64p, u8p, dp, dp]),
            "ora_zc_decode": (C.c_int, [u8p, C.c_uint64, u16p, C.c_uint64, u64p]),
            "ora_zc_encode_chunk": (C.c_int, [u16p, C.c_uint32, C.c_uint32, u8p, u8p, u8p,
                                              C.POINTER(C.c_uint32), C.POINTER(C.c_int)]),
            "ora_ibp_meta_bytes": (C.c_uint64, [C.c_uint32]),
            "ora_fnv1a64": (C.c_uint64, [u8p, C.c_size_t]),
            "ora_ibp_build_meta": (C.c_int, [u8p, C.c_uint64, C.c_uint32, C.c_double, C.c_int, u8p]),
            "ora_ibp_make_meta": (C.c_int, [C.c_uint32, u8p, u8p, u8p]),
            "ora_ibp_chunk_p": (C.c_int, [u8p, u8p]),
            "ora_ibp_stream_bytes_bound": (C.c_uint64, [C.c_uint32, C.c_uint64]),
            "ora_ibp_encode": (C.c_int, [u8p, u8p, C.c_uint64, u8p, C.c_uint64, u64p]),
            "ora_ibp_decode": (C.c_int, [u8p, u8p, C.c_uint64, u8p, C.c_uint64, u64p]),
            "ora_ibp_encode_group": (C.c_int, [u8p, u8p, C.c_uint32, C.c_uint32, u8p,
                                               C.c_uint64, u64p]),
            "ora_ibp_slot_read_bytes": (C.c_uint32, [u8p, C.c_int, C.c_uint32]),
            "ora_ibp_slot_encode": (C.c_int, [u8p, u8p, C.c_uint32, u8p, C.POINTER(C.c_int)]),
            "ora_ibp_slot_decode": (C.c_int, [u8p, u8p, C.c_uint32, C.c_int, u8p]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _p(a, ct):
    return a.ctypes.data_as(C.POINTER(ct))


def _u8(a):
    a = np.ascontiguousarray(a)
    return a.view(np.uint8).reshape(-1)


def _chk(rc, what):
    if rc != OK:
        raise OracleError(rc, what)


# ------------------------------------------------------------------ ZipCCL

def zc_stats(x):
    x = np.ascontiguousarray(x, dtype=np.uint16)
    cnt, s1, s2 = C.c_uint64(), C.c_double(), C.c_double()
    lib().ora_zc_stats(_p(x, C.c_uint16), x.size, C.byref(cnt), C.byref(s1), C.byref(s2))
    return cnt.value, s1.value, s2.value


def zc_moments(cnt, s1, s2):
    mu, sg = C.c_double(), C.c_double()
    lib().ora_zc_moments(cnt, s1, s2, C.byref(mu), C.byref(sg))
    return mu.value, sg.value


def zc_mass(mu, sigma, f):
    return lib().ora_zc_mass(mu, sigma, f)


def zc_predict(mu, sigma):
    b = np.zeros(7, np.uint8)
    lib().ora_zc_predict(mu, sigma, _p(b, C.c_uint8))
    return b


def _segs(n, seg_off):
    if seg_off is None:
        return None, 1
    s = np.ascontiguousarray(seg_off, dtype=np.uint64)
    return s, s.size - 1


def zc_stream_bytes(n, seg_off, chunk_elems, n_esc):
    s, nseg = _segs(n, seg_off)
    return lib().ora_zc_stream_bytes(n, nseg, None if s is None else _p(s, C.c_uint64),
                                     chunk_elems, n_esc)


def zc_encode(x, seg_off=None, chunk_elems=4096, books=None):
    """Returns (stream uint8 array, books (nseg,7), mus, sigmas)."""
    x = np.ascontiguousarray(x, dtype=np.uint16).reshape(-1)
    n = x.size
    s, nseg = _segs(n, seg_off)
    cap = zc_stream_bytes(n, seg_off, chunk_elems, n) + 128
    out = np.zeros(cap, np.uint8)
    used = np.zeros(7 * nseg, np.uint8)
    mus = np.zeros(nseg, np.float64)
    sig = np.zeros(nseg, np.float64)
    ob = C.c_uint64()
    bk = None
    if books is not None:
        bk = np.ascontiguousarray(books, dtype=np.uint8).reshape(-1)
        assert bk.size == 7 * nseg
    rc = lib().ora_zc_encode(
        _p(x, C.c_uint16), n, None if s is None else _p(s, C.c_uint64), nseg, chunk_elems,
        None if bk is None else _p(bk, C.c_uint8), _p(out, C.c_uint8), cap, C.byref(ob),
        _p(used, C.c_uint8), _p(mus, C.c_double), _p(sig, C.c_double))
    _chk(rc, "zc_encode")
    return out[: ob.value].copy(), used.reshape(nseg, 7), mus, sig


def zc_decode(stream, y_cap=None):
    st = _u8(stream)
    if y_cap is None:
        y_cap = int(st[16:24].view(np.uint64)[0]) if st.size >= 24 else 0
    y = np.zeros(max(y_cap, 1), np.uint16)
    n = C.c_uint64()
    rc = lib().ora_zc_decode(_p(st, C.c_uint8), st.size, _p(y, C.c_uint16), y_cap, C.byref(n))
    return rc, y[: n.value] if rc == OK else None


def zc_encode_chunk(x, chunk_elems, book):
    """Returns (slot, dynamic bytes, raw flag) of one chunk."""
    x = np.ascontiguousarray(x, dtype=np.uint16).reshape(-1)
    book = np.ascontiguousarray(book, dtype=np.uint8)
    slot = np.zeros(chunk_elems * 11 // 8, np.uint8)
    esc = np.zeros(chunk_elems, np.uint8)
    ne = C.c_uint32()
    raw = C.c_int()
    rc = lib().ora_zc_encode_chunk(_p(x, C.c_uint16), x.size, chunk_elems, _p(book, C.c_uint8),
                                   _p(slot, C.c_uint8), _p(esc, C.c_uint8), C.byref(ne),
                                   C.byref(raw))
    _chk(rc, "zc_encode_chunk")
    return slot, esc[: ne.value].copy(), bool(raw.value)


# ------------------------------------------------------------------ IBP

def ibp_meta_bytes(chunk_bytes):
    return lib().ora_ibp_meta_bytes(chunk_bytes)


def fnv1a64(b):
    b = _u8(b)
    return lib().ora_fnv1a64(_p(b, C.c_uint8), b.size)


def ibp_build_meta(samples, chunk_bytes, T=0.9, mode=0):
    sm = _u8(samples)
    assert sm.size % chunk_bytes == 0
    N = sm.size // chunk_bytes
    meta = np.zeros(ibp_meta_bytes(chunk_bytes), np.uint8)
    rc = lib().ora_ibp_build_meta(_p(sm, C.c_uint8), N, chunk_bytes, T, mode, _p(meta, C.c_uint8))
    _chk(rc, "ibp_build_meta")
    return meta


def ibp_make_meta(chunk_bytes, mask, bitval):
    mask, bitval = _u8(mask), _u8(bitval)
    meta = np.zeros(ibp_meta_bytes(chunk_bytes), np.uint8)
    rc = lib().ora_ibp_make_meta(chunk_bytes, _p(mask, C.c_uint8), _p(bitval, C.c_uint8),
                                 _p(meta, C.c_uint8))
    _chk(rc, "ibp_make_meta")
    return meta


def ibp_chunk_p(meta, chunk):
    meta, chunk = _u8(meta), _u8(chunk)
    return lib().ora_ibp_chunk_p(_p(meta, C.c_uint8), _p(chunk, C.c_uint8))


def ibp_encode(meta, x):
    meta, xb = _u8(meta), _u8(x)
    cb = int(meta[8:12].view(np.uint32)[0])
    cap = lib().ora_ibp_stream_bytes_bound(cb, xb.size)
    out = np.zeros(cap, np.uint8)
    ob = C.c_uint64()
    rc = lib().ora_ibp_encode(_p(meta, C.c_uint8), _p(xb, C.c_uint8), xb.size,
                              _p(out, C.c_uint8), cap, C.byref(ob))
    _chk(rc, "ibp_encode")
    return out[: ob.value].copy()


def ibp_decode(meta, stream, y_cap=None):
    meta, st = _u8(meta), _u8(stream)
    if y_cap is None:
        y_cap = int(st[16:24].view(np.uint64)[0]) if st.size >= 24 else 0
    y = np.zeros(max(y_cap, 1), np.uint8)
    n = C.c_uint64()
    rc = lib().ora_ibp_decode(_p(meta, C.c_uint8), _p(st, C.c_uint8), st.size,
                              _p(y, C.c_uint8), y_cap, C.byref(n))
    return rc, y[: n.value] if rc == OK else None


def ibp_encode_group(meta, x_chunks, nch, last_bytes=0):
    meta, xb = _u8(meta), _u8(x_chunks)
    cb = int(meta[8:12].view(np.uint32)[0])
    cap = 4 + 32 * cb + 16
    out = np.zeros(cap, np.uint8)
    bits = C.c_uint64()
    rc = lib().ora_ibp_encode_group(_p(meta, C.c_uint8), _p(xb, C.c_uint8), nch, last_bytes,
                                    _p(out, C.c_uint8), cap, C.byref(bits))
    _chk(rc, "ibp_encode_group")
    return out[: bits.value // 8].copy()


# ------------------------------------------------------------------ IBP slots

def ibp_slot_read_bytes(meta, p, length):
    meta = _u8(meta)
    return lib().ora_ibp_slot_read_bytes(_p(meta, C.c_uint8), int(p), int(length))


def _slot_ranges(nch, pieces):
    pieces = max(1, min(pieces, nch))
    e = [nch * i // pieces for i in range(pieces + 1)]
    return [(e[i], e[i + 1]) for i in range(pieces) if e[i + 1] > e[i]]


def ibp_slots_encode(meta, x, slots=None, threads=None):
    """In-place slot form of the bytes x (a multiple of 4): returns (slots,
    bitmask).  `slots` starts as a copy of x unless given (its bytes past a
    compressed slot's body are left as they are); bitmask is uint32 words, bit
    s % 32 of word s / 32 set when slot s is compressed.  Chunk ranges are
    encoded in threads (one C call per chunk)."""
    from concurrent.futures import ThreadPoolExecutor
    meta, xb = _u8(meta), _u8(x)
    cb = int(meta[8:12].view(np.uint32)[0])
    n = xb.size
    nch = (n + cb - 1) // cb
    out = xb.copy() if slots is None else slots
    bits = np.zeros(nch, np.uint8)
    L = lib()
    mp = _p(meta, C.c_uint8)

    def run(r):
        pv = C.c_int()
        for s in range(*r):
            ln = min(cb, n - s * cb)
            ch = np.ascontiguousarray(xb[s * cb: s * cb + ln])
            rc = L.ora_ibp_slot_encode(mp, _p(ch, C.c_uint8), ln,
                                       _p(out[s * cb:], C.c_uint8), C.byref(pv))
            _chk(rc, "ibp_slot_encode")
            bits[s] = pv.value
    with ThreadPoolExecutor(threads or min(32, os.cpu_count() or 1)) as ex:
        list(ex.map(run, _slot_ranges(nch, 4 * (threads or min(32, os.cpu_count() or 1)))))
    words = np.zeros((nch + 31) // 32, np.uint32)
    for w in range(words.size):
        b = bits[32 * w: 32 * w + 32]
        words[w] = int(sum(int(v) << i for i, v in enumerate(b)))
    return out, words


def ibp_slots_gather(meta, slots, n_bytes, bitmask, idx):
    """Chunks idx[0], idx[1], ... decoded from their slots: returns
    (rows uint8 [len(idx), chunk_bytes] (a short last chunk's row is zero past
    its length), bytes read from the slots)."""
    meta, sl = _u8(meta), _u8(slots)
    bitmask = np.ascontiguousarray(bitmask, np.uint32)
    cb = int(meta[8:12].view(np.uint32)[0])
    idx = np.asarray(idx, np.int64).reshape(-1)
    rows = np.zeros((idx.size, cb), np.uint8)
    L = lib()
    mp = _p(meta, C.c_uint8)
    read = 0
    for i, s in enumerate(idx):
        s = int(s)
        ln = min(cb, n_bytes - s * cb)
        p = int((int(bitmask[s // 32]) >> (s % 32)) & 1)
        rb = L.ora_ibp_slot_read_bytes(mp, p, ln)
        src = np.ascontiguousarray(sl[s * cb: s * cb + rb])  # only the part that is read
        buf = np.zeros(cb, np.uint8)
        buf[:rb] = src
        row = np.zeros(cb, np.uint8)
        _chk(L.ora_ibp_slot_decode(mp, _p(buf, C.c_uint8), ln, p, _p(row, C.c_uint8)),
             "ibp_slot_decode")
        rows[i, :ln] = row[:ln]
        read += rb
    return rows, read
