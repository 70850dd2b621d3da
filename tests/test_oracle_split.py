"""The piecewise whole-stream comparison (tests/oracle_split.py) accepts
exactly the oracle's own stream: on inputs small enough for one oracle call,
the full stream passes and a stream with any one byte changed -- in a slot,
an escape, a table entry, a payload, a header field or a padding byte -- is
rejected.  CPU only."""
import numpy as np
import pytest

import oracle as O
from oracle_split import ibp_stream_equal, zc_stream_equal


def _bf16(f32):
    u = np.ascontiguousarray(f32, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("pieces", [1, 3, 7])
def test_zc_split_accepts_oracle_stream(pieces):
    rng = np.random.default_rng(pieces)
    C = 1024
    x = _bf16(rng.normal(0, 0.01, size=23 * C + 301))
    x[::53] = 0x7FC1  # escapes in every chunk
    book = np.arange(115, 122, dtype=np.uint8)
    ref, _, _, _ = O.zc_encode(x, None, C, books=book)
    esc = zc_stream_equal(ref, x, C, book, pieces=pieces)
    assert esc == int(ref[32:40].view(np.uint64)[0]) > 0


def test_zc_split_with_raw_chunks():
    rng = np.random.default_rng(8)
    C = 1024
    x = _bf16(rng.normal(0, 0.01, size=12 * C + 5))
    x[3 * C:4 * C] = rng.integers(0, 65536, size=C).astype(np.uint16)  # stored raw
    x[7 * C:8 * C] = 0x7FC0
    book = np.arange(115, 122, dtype=np.uint8)
    ref, _, _, _ = O.zc_encode(x, None, C, books=book)
    zc_stream_equal(ref, x, C, book, pieces=5)
    off_escoff = int(ref[48:56].view(np.uint64)[0])
    bad = ref.copy()
    bad[off_escoff + 8 * 3 + 7] ^= 0x80  # the raw flag of chunk 3
    with pytest.raises(AssertionError):
        zc_stream_equal(bad, x, C, book, pieces=5)


def test_zc_split_rejects_any_changed_byte():
    rng = np.random.default_rng(5)
    C = 1024
    x = _bf16(rng.normal(0, 0.01, size=9 * C + 77))
    x[::41] = 0xFF80
    book = np.arange(115, 122, dtype=np.uint8)
    ref, _, _, _ = O.zc_encode(x, None, C, books=book)
    h = ref[16:80].view(np.uint64)
    off_seg, off_escoff, off_static, off_esc, total = (int(v) for v in h[3:8])
    places = [0, 9, 20, 100, off_seg + 3, off_seg + 40, off_seg + 50, off_seg + 60,
              off_escoff + 8 * 4, off_escoff + 8 * 10 + 1, off_static - 1, off_static + 5,
              off_static + 3 * 1408 + 1100, off_esc - 1, off_esc + 7, total - 1]
    for p in places:
        bad = ref.copy()
        bad[p] ^= 0x10
        with pytest.raises(AssertionError):
            zc_stream_equal(bad, x, C, book, pieces=4)
    with pytest.raises(AssertionError):
        zc_stream_equal(ref[:-128], x, C, book, pieces=4)
    with pytest.raises(AssertionError):
        zc_stream_equal(ref, x, C, np.arange(116, 123, dtype=np.uint8), pieces=4)


def _ibp_case(cb, nch, seed):
    rng = np.random.default_rng(seed)
    B = 8 * cb
    mask = (rng.uniform(size=B) < 0.3).astype(np.uint8)
    bitval = rng.integers(0, 2, size=B).astype(np.uint8) & mask
    meta = O.ibp_make_meta(cb, np.packbits(mask, bitorder="little"),
                           np.packbits(bitval, bitorder="little"))
    bits = rng.integers(0, 2, size=(nch, B)).astype(np.uint8)
    force = rng.uniform(size=nch) < 0.5
    bits[force] = np.where(mask.astype(bool), bitval, bits[force])
    x = np.packbits(bits, axis=1, bitorder="little").reshape(-1)
    return meta, x


@pytest.mark.parametrize("pieces", [1, 2, 5])
@pytest.mark.parametrize("cb,tail", [(64, 0), (512, 20), (48, 4)])
def test_ibp_split_accepts_oracle_stream(pieces, cb, tail):
    meta, x = _ibp_case(cb, 32 * 9 + 5, cb + pieces)
    x = x[: x.size - tail]
    ref = O.ibp_encode(meta, x)
    bits = ibp_stream_equal(ref, meta, x, pieces=pieces)
    assert bits == int(ref[64:72].view(np.uint64)[0])


def test_ibp_split_rejects_any_changed_byte():
    cb = 64
    meta, x = _ibp_case(cb, 32 * 7 + 3, 9)
    ref = O.ibp_encode(meta, x)
    h = ref[16:80].view(np.uint64)
    off_grp, off_pay, total = int(h[4]), int(h[5]), int(h[7])
    places = [0, 5, 10, 13, 17, 30, 42, 60, 70, 100, off_grp + 8 * 3, off_grp + 8 * 8 + 2,
              off_pay - 1, off_pay, off_pay + 200, total - 1]
    for p in places:
        bad = ref.copy()
        bad[p] ^= 0x04
        with pytest.raises(AssertionError):
            ibp_stream_equal(bad, meta, x, pieces=3)
    other = meta.copy()
    other[64] ^= 1  # another Mask
    with pytest.raises(AssertionError):
        ibp_stream_equal(ref, O.ibp_make_meta(cb, other[64:64 + cb], other[64 + cb:64 + 2 * cb]),
                         x, pieces=3)
