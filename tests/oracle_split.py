"""Whole-stream comparison with the oracle for inputs too large to encode in
one oracle call within a test's time.

Both stream formats are made of independent parts: a ZipCCL segment's chunks
(fixed-size slot + that chunk's escape bytes) and an IBP stream's groups of 32
chunks (each group's payload starts 128-bit aligned).  The input is cut at
chunk (ZipCCL) or group (IBP) boundaries into pieces; each piece is encoded by
one ordinary oracle call (``oracle.zc_encode`` / ``oracle.ibp_encode``, not a
per-element shortcut) in a thread of its own -- ctypes releases the GIL, so
the calls run on all host cores -- and the GPU stream's regions for that piece
are compared byte for byte with the piece's stream:

* ZipCCL: the piece's slots, its escape bytes and its escape-offset table
  (shifted by the GPU's offset of the piece's first chunk);
* IBP: the piece's group payloads and its group-offset table (shifted by the
  GPU's offset of the piece's first group).

The shifts themselves are checked (each piece starts where the pieces before
it end), the header fields are checked against the pieces' headers and the
oracle's size formula, and every padding byte of the GPU stream must be zero.
Together this covers every byte of the GPU stream.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle as O


def _workers():
    return max(1, min(32, os.cpu_count() or 1))


def _u64(b, off, k=1):
    return b[off:off + 8 * k].view(np.uint64)


def _ranges(total, pieces):
    pieces = max(1, min(pieces, total))
    edges = [total * i // pieces for i in range(pieces + 1)]
    return [(edges[i], edges[i + 1]) for i in range(pieces) if edges[i + 1] > edges[i]]


def _zero(b, lo, hi, what):
    if hi > lo:
        nz = np.flatnonzero(b[lo:hi])
        assert nz.size == 0, f"{what}: nonzero padding byte at {lo + int(nz[0])}"


def zc_stream_equal(stream, x_bits, chunk, book, pieces=None):
    """Asserts that `stream` (uint8, one segment) is the oracle's ZCC1 stream
    of the bf16 bit patterns `x_bits` with chunk size `chunk` and codebook
    `book` (7 ascending fields).  Returns the number of escapes."""
    st = np.ascontiguousarray(stream, np.uint8).reshape(-1)
    x = np.ascontiguousarray(x_bits, np.uint16).reshape(-1)
    book = np.ascontiguousarray(book, np.uint8).reshape(7)
    n, C = x.size, int(chunk)
    S = C * 11 // 8
    nchunks = (n + C - 1) // C
    h = _u64(st, 16, 8)  # n, nchunks, escapes, off_seg, off_escoff, off_static, off_esc, total
    assert int(h[0]) == n and int(h[1]) == nchunks, (h[0], h[1])
    off_seg, off_escoff, off_static, off_esc = (int(v) for v in h[3:7])
    assert off_esc == off_static + nchunks * S
    # bit 63 of an entry marks a chunk stored raw; bits 62..0 are the offset
    eo_all = _u64(st, off_escoff, nchunks + 1)
    eo_raw = (eo_all >> np.uint64(63)).astype(np.int64)
    eo = (eo_all & np.uint64((1 << 63) - 1)).astype(np.int64)
    if nchunks == 0:
        ref, _, _, _ = O.zc_encode(x, None, C, books=book)
        assert np.array_equal(st, ref)
        return 0

    def one(rng):
        c0, c1 = rng
        piece = x[c0 * C: min(n, c1 * C)]
        ps, _, _, _ = O.zc_encode(piece, None, C, books=book)
        ph = _u64(ps, 16, 8)
        p_escoff, p_static, p_esc = int(ph[4]), int(ph[5]), int(ph[6])
        p_n_esc = int(ph[2])
        k = c1 - c0
        bad = []
        if not np.array_equal(st[off_static + c0 * S: off_static + c1 * S],
                              ps[p_static: p_static + k * S]):
            bad.append("slots")
        p_all = _u64(ps, p_escoff, k + 1)
        p_eo = (p_all & np.uint64((1 << 63) - 1)).astype(np.int64)
        if not np.array_equal(eo[c0:c1 + 1] - eo[c0], p_eo):
            bad.append("escape offsets")
        if not np.array_equal(eo_raw[c0:c1], (p_all[:k] >> np.uint64(63)).astype(np.int64)):
            bad.append("raw-chunk flags")
        base = int(eo[c0])
        if not np.array_equal(st[off_esc + base: off_esc + base + p_n_esc],
                              ps[p_esc: p_esc + p_n_esc]):
            bad.append("escape bytes")
        return c0, c1, p_n_esc, bytes(ps[:16]), bytes(ps[off_seg + 48: off_seg + 55]), bad

    parts = _ranges(nchunks, pieces or 4 * _workers())
    with ThreadPoolExecutor(_workers()) as ex:
        res = sorted(ex.map(one, parts))
    esc = 0
    for c0, c1, ne, head, pbook, bad in res:
        assert not bad, f"chunks {c0}..{c1}: {', '.join(bad)} differ from the oracle"
        assert int(eo[c0]) == esc, (c0, int(eo[c0]), esc)
        assert head == bytes(st[:16]), "magic, version, header size, chunk, segments"
        assert pbook == bytes(st[off_seg + 48: off_seg + 55]) == bytes(book)
        esc += ne
    assert int(eo[nchunks]) == esc and int(h[2]) == esc and eo_raw[nchunks] == 0
    total = O.zc_stream_bytes(n, None, C, esc)
    assert st.size == total and int(h[7]) == total, (st.size, total)
    rec = _u64(st, off_seg, 6)
    assert [int(v) for v in rec] == [0, n, 0, nchunks, 0, esc], rec
    _zero(st, 80, off_seg, "header")
    _zero(st, off_seg + 55, off_escoff, "segment record")
    _zero(st, off_escoff + 8 * (nchunks + 1), off_static, "escape-offset table")
    _zero(st, off_esc + esc, total, "escape region")
    return esc


def ibp_stream_equal(stream, meta, x_bytes, pieces=None):
    """Asserts that `stream` (uint8) is the oracle's IBP1 stream of the bytes
    `x_bytes` under the IBPM blob `meta`.  Returns the payload bits."""
    st = np.ascontiguousarray(stream, np.uint8).reshape(-1)
    meta = np.ascontiguousarray(meta, np.uint8).reshape(-1)
    xb = np.ascontiguousarray(x_bytes, np.uint8).reshape(-1)
    n = xb.size
    cb = int(meta[8:12].view(np.uint32)[0])
    nch = (n + cb - 1) // cb
    ng = (nch + 31) // 32
    h = _u64(st, 16, 8)  # n_bytes, nchunks, ngroups, meta hash, off_grp, off_pay, bits, total
    assert int(h[0]) == n and int(h[1]) == nch and int(h[2]) == ng, h[:3]
    off_grp, off_pay = int(h[4]), int(h[5])
    if ng == 0:
        assert np.array_equal(st, O.ibp_encode(meta, xb))
        return 0
    grp = _u64(st, off_grp, ng + 1).astype(np.int64)
    gb = 32 * cb  # input bytes of a full group

    def one(rng):
        g0, g1 = rng
        ps = O.ibp_encode(meta, xb[g0 * gb: min(n, g1 * gb)])
        ph = _u64(ps, 16, 8)
        p_grp, p_pay, p_bits = int(ph[4]), int(ph[5]), int(ph[6])
        k = g1 - g0
        bad = []
        pg = _u64(ps, p_grp, k + 1).astype(np.int64)
        if not np.array_equal(grp[g0:g1 + 1] - grp[g0], pg):
            bad.append("group offsets")
        base = off_pay + int(grp[g0]) // 8
        if not np.array_equal(st[base: base + p_bits // 8], ps[p_pay: p_pay + p_bits // 8]):
            bad.append("payload")
        return g0, g1, p_bits, bytes(ps[:16]), bytes(ps[40:48]), bad

    parts = _ranges(ng, pieces or 4 * _workers())
    with ThreadPoolExecutor(_workers()) as ex:
        res = sorted(ex.map(one, parts))
    bits = 0
    for g0, g1, pb, head, mhash, bad in res:
        assert not bad, f"groups {g0}..{g1}: {', '.join(bad)} differ from the oracle"
        assert int(grp[g0]) == bits, (g0, int(grp[g0]), bits)
        assert head == bytes(st[:16]), "magic, version, header size, chunk bytes, m"
        assert mhash == bytes(st[40:48]), "metadata hash"
        bits += pb
    assert int(grp[ng]) == bits and int(h[6]) == bits
    assert bits % 128 == 0
    total = off_pay + bits // 8
    assert st.size == total and int(h[7]) == total, (st.size, total)
    # the header size and the table's padding: the oracle's own layout for a
    # one-group input of the same chunk size has the table at the same offset
    one_group = O.ibp_encode(meta, xb[:min(n, cb)])
    assert int(_u64(one_group, 48)[0]) == off_grp
    assert off_pay == off_grp + (8 * (ng + 1) + 127) // 128 * 128
    _zero(st, 80, off_grp, "header")
    _zero(st, off_grp + 8 * (ng + 1), off_pay, "group-offset table")
    return bits
