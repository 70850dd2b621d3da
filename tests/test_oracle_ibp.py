"""Pins for the IBP oracle (CPU only).

Ties the oracle to: a stream derived by hand from the layout, published FNV-1a
test vectors, the T = 1 closed form of the metadata (Mask = positions constant
over all samples), brute-force bit counts, the defining predicate of the
participation bit, the closed-form stream size, and the round trip.

Page cited: "Riepilogo Tecnico: Riduzione del Collo di Bottiglia della Memoria
GPU con la Compressione Lossless per il ML", Metodologia: Invariant Bit Packing
(IBP), Algoritmo Core steps 1-3.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_fnv1a64_vectors():
    g = json.load(open(os.path.join(GOLD, "fnv1a64_vectors.json")))
    for s, hx in g["vectors"]:
        b = np.frombuffer(s.encode(), np.uint8) if s else np.zeros(0, np.uint8)
        assert O.fnv1a64(b) == int(hx, 16)


def test_golden_tiny_stream():
    g = json.load(open(os.path.join(GOLD, "ibp_tiny_stream.json")))
    cb = g["chunk_bytes"]
    mask = np.frombuffer(bytes.fromhex(g["mask_hex"]), np.uint8)
    bitval = np.frombuffer(bytes.fromhex(g["bitval_hex"]), np.uint8)
    meta = O.ibp_make_meta(cb, mask, bitval)
    x = np.frombuffer(bytes.fromhex(g["input_hex"]), np.uint8)
    st = O.ibp_encode(meta, x)
    assert st.size == g["total_bytes"]
    want = np.zeros(g["total_bytes"], np.uint8)
    for off, hx in g["spans"]:
        b = bytes.fromhex(hx)
        want[off:off + len(b)] = np.frombuffer(b, np.uint8)
    h = O.fnv1a64(np.concatenate([np.frombuffer(np.uint32(cb).tobytes(), np.uint8), mask, bitval]))
    want[g["hash_span_offset"]:g["hash_span_offset"] + 8] = np.frombuffer(np.uint64(h).tobytes(), np.uint8)
    bad = np.nonzero(st != want)[0]
    assert bad.size == 0, f"first differing bytes at {bad[:8]}"
    rc, y = O.ibp_decode(meta, st)
    assert rc == 0 and np.array_equal(y, x)


def _bits(chunks):
    """[N, chunk_bytes] uint8 -> [N, B] bits (bit j = bit j%8 of byte j/8)."""
    return np.unpackbits(chunks, axis=1, bitorder="little")


def _meta_parts(meta, cb):
    m = int(meta[16:20].view(np.uint32)[0])
    mask = meta[64:64 + cb]
    bitval = meta[64 + cb:64 + 2 * cb]
    return m, mask, bitval


@pytest.mark.parametrize("cb", [4, 8, 16])
def test_meta_T1_is_constant_positions(cb):
    rng = np.random.default_rng(cb)
    N = 17
    base = rng.integers(0, 256, size=cb, dtype=np.uint8)
    noise = rng.integers(0, 256, size=(N, cb), dtype=np.uint8)
    keep = rng.integers(0, 256, size=cb, dtype=np.uint8)  # bits forced constant
    s = (noise & ~keep) | (base & keep)
    meta = O.ibp_build_meta(s, cb, T=1.0, mode=0)
    m, mask, bitval = _meta_parts(meta, cb)
    OR = np.bitwise_or.reduce(s, axis=0)
    AND = np.bitwise_and.reduce(s, axis=0)
    want_mask = ~(OR ^ AND) & 0xFF
    assert np.array_equal(mask, want_mask)
    assert np.array_equal(bitval, AND & want_mask)
    assert m == int(np.unpackbits(want_mask).sum())
    # at T = 1 the joint reading keeps exactly the same positions
    meta1 = O.ibp_build_meta(s, cb, T=1.0, mode=1)
    assert np.array_equal(meta1[64:64 + 2 * cb], meta[64:64 + 2 * cb])


@pytest.mark.parametrize("T", [0.6, 0.75, 0.9, 0.95])
def test_meta_per_position_counts(T):
    rng = np.random.default_rng(int(T * 100))
    cb, N = 8, 20
    p1 = rng.uniform(0, 1, size=cb * 8)  # per-position probability of a 1
    bits = (rng.uniform(size=(N, cb * 8)) < p1).astype(np.uint8)
    s = np.packbits(bits, axis=1, bitorder="little")
    meta = O.ibp_build_meta(s, cb, T=T, mode=0)
    m, mask, bitval = _meta_parts(meta, cb)
    ones = bits.sum(axis=0)
    k = math.ceil(T * N)
    agree = np.maximum(ones, N - ones)
    want = agree >= k
    got = np.unpackbits(mask, bitorder="little").astype(bool)
    assert np.array_equal(got, want)
    gotv = np.unpackbits(bitval, bitorder="little").astype(bool)
    assert np.array_equal(gotv, want & (ones >= k))
    assert int(meta[32:40].view(np.uint64)[0]) == k


@pytest.mark.parametrize("seed", range(6))
def test_meta_joint_is_feasible_and_maximal(seed):
    rng = np.random.default_rng(100 + seed)
    cb, N, T = 4, 40, 0.8
    p1 = rng.choice([0.02, 0.05, 0.1, 0.5, 0.9, 0.97], size=cb * 8)
    bits = (rng.uniform(size=(N, cb * 8)) < p1).astype(np.uint8)
    s = np.packbits(bits, axis=1, bitorder="little")
    k = math.ceil(T * N)
    meta0 = O.ibp_build_meta(s, cb, T=T, mode=0)
    meta1 = O.ibp_build_meta(s, cb, T=T, mode=1)
    m0 = np.unpackbits(meta0[64:64 + cb], bitorder="little").astype(bool)
    m1 = np.unpackbits(meta1[64:64 + cb], bitorder="little").astype(bool)
    v1 = np.unpackbits(meta1[64 + cb:64 + 2 * cb], bitorder="little").astype(np.uint8)
    assert not np.any(m1 & ~m0), "joint positions are per-position invariant too"

    def matches(sel, vals):
        return np.all(bits[:, sel] == vals[sel], axis=1)

    # feasible: at least k samples match every kept position
    assert matches(m1, v1).sum() >= k
    # maximal: no other candidate position can be added
    ones = bits.sum(axis=0)
    for j in np.nonzero(m0 & ~m1)[0]:
        sel = m1.copy()
        sel[j] = True
        vals = v1.copy()
        vals[j] = 1 if ones[j] >= k else 0
        assert matches(sel, vals).sum() < k
    # the position agreeing most (lowest index on ties) is always kept
    if m0.any():
        agree = np.maximum(ones, N - ones)
        cand = np.nonzero(m0)[0]
        first = cand[np.lexsort((cand, -agree[cand]))[0]]
        assert m1[first]


def _rand_meta(rng, cb, frac):
    mask = (rng.uniform(size=cb * 8) < frac).astype(np.uint8)
    bitval = rng.integers(0, 2, size=cb * 8).astype(np.uint8) & mask
    return (O.ibp_make_meta(cb, np.packbits(mask, bitorder="little"),
                            np.packbits(bitval, bitorder="little")), mask, bitval)


@pytest.mark.parametrize("cb,frac", [(16, 0.3), (64, 0.1), (512, 0.15), (2048, 0.05),
                                     (512, 0.0), (16, 1.0)])
def test_participation_bit_and_size(cb, frac):
    rng = np.random.default_rng(cb + int(frac * 1000))
    meta, mask, bitval = _rand_meta(rng, cb, frac)
    m = int(mask.sum())
    nch = 70
    tail = (cb // 2) // 4 * 4
    n_bytes = (nch - 1) * cb + (tail if tail else cb)
    bits = rng.integers(0, 2, size=(nch, cb * 8)).astype(np.uint8)
    # force about half of the chunks to carry the invariant bits
    force = rng.uniform(size=nch) < 0.5
    bits[force] = np.where(mask.astype(bool), bitval, bits[force])
    x = np.packbits(bits, axis=1, bitorder="little").reshape(-1)[:n_bytes]
    st = O.ibp_encode(meta, x)
    ng = (nch + 31) // 32
    grp = st[128:128 + 8 * (ng + 1)].view(np.uint64)
    off_pay = int(st[56:64].view(np.uint64)[0])
    pay = st[off_pay:]
    total_bits = 0
    for g in range(ng):
        word = int(pay[grp[g] // 8: grp[g] // 8 + 4].view(np.uint32)[0])
        used = 32
        for t in range(32):
            c = 32 * g + t
            p = (word >> t) & 1
            if c >= nch:
                assert p == 0
                continue
            full = (c + 1) * cb <= n_bytes
            match = bool(np.all(bits[c][mask.astype(bool)] == bitval[mask.astype(bool)]))
            # set exactly when the chunk is full, matches and so saves space
            assert p == int(full and m > 0 and match)
            assert O.ibp_chunk_p(meta, x[c * cb:(c + 1) * cb]) == int(m > 0 and match) or not full
            used += (cb * 8 - m) if p else (cb * 8 if full else (n_bytes - c * cb) * 8)
        padded = -(-used // 128) * 128
        assert int(grp[g + 1] - grp[g]) == padded
        total_bits += padded
    assert int(st[64:72].view(np.uint64)[0]) == total_bits
    rc, y = O.ibp_decode(meta, st)
    assert rc == 0 and np.array_equal(y, x)


def test_roundtrip_fp32_rows_and_group_entry():
    rng = np.random.default_rng(42)
    rows = rng.normal(0, 0.1, size=(300, 128)).clip(-1, 1).astype(np.float32)
    x = rows.view(np.uint8).reshape(-1)
    for mode in (0, 1):
        meta = O.ibp_build_meta(x[: 100 * 512], 512, T=0.9, mode=mode)
        st = O.ibp_encode(meta, x)
        rc, y = O.ibp_decode(meta, st)
        assert rc == 0 and np.array_equal(y, x)
        off_pay = int(st[56:64].view(np.uint64)[0])
        grp = st[128:128 + 8 * 11].view(np.uint64)
        for g in range(10):
            nch = min(32, 300 - 32 * g)
            gb = O.ibp_encode_group(meta, x[32 * g * 512:(32 * g + nch) * 512], nch)
            assert np.array_equal(gb, st[off_pay + grp[g] // 8: off_pay + grp[g + 1] // 8])


def test_degenerate_and_mismatch():
    rng = np.random.default_rng(0)
    x = rng.integers(0, 256, size=4096, dtype=np.uint8)
    meta_none, _, _ = _rand_meta(rng, 64, 0.0)   # m = 0: nothing invariant
    st = O.ibp_encode(meta_none, x)
    assert O.ibp_decode(meta_none, st)[1].tobytes() == x.tobytes()
    # empty input
    st0 = O.ibp_encode(meta_none, np.zeros(0, np.uint8))
    assert st0.size == 256 and O.ibp_decode(meta_none, st0)[0] == 0
    # a stream decoded with other metadata is refused
    meta_other, _, _ = _rand_meta(rng, 64, 0.2)
    assert O.ibp_decode(meta_other, st)[0] == O.E_META
    # corrupt group offsets / header
    bad = st.copy()
    bad[136] ^= 0x80
    assert O.ibp_decode(meta_none, bad)[0] == O.E_FORMAT
    bad = st.copy()
    bad[0] ^= 1
    assert O.ibp_decode(meta_none, bad)[0] == O.E_FORMAT
    assert O.ibp_decode(meta_none, st[:-16])[0] == O.E_FORMAT


# ---------------------------------------------------------------- in-place slots
# ([IBP] Integrazione del Sistema: tensors compressed in place in fixed-size
# buffers, only the compressed part read, a GPU bitmask of compressed tensors)

def _slot_case(cb, frac, nch, seed, tail=0):
    rng = np.random.default_rng(seed)
    B = 8 * cb
    mask = (rng.uniform(size=B) < frac).astype(np.uint8)
    bitval = rng.integers(0, 2, size=B).astype(np.uint8) & mask
    meta = O.ibp_make_meta(cb, np.packbits(mask, bitorder="little"),
                           np.packbits(bitval, bitorder="little"))
    bits = rng.integers(0, 2, size=(nch, B)).astype(np.uint8)
    force = rng.uniform(size=nch) < 0.6
    bits[force] = np.where(mask.astype(bool), bitval, bits[force])
    x = np.packbits(bits, axis=1, bitorder="little").reshape(-1)
    return meta, x[: x.size - tail]


@pytest.mark.parametrize("cb,frac,tail", [(64, 0.3, 0), (512, 0.12, 20), (20, 0.5, 0),
                                          (48, 0.0, 8), (32, 1.0, 0), (2048, 0.02, 1024)])
def test_slots_are_the_stream_bodies(cb, frac, tail):
    """A slot's first bits are exactly the chunk's body in the IBP1 stream
    (the layout pinned by the hand-derived golden stream): kept bits when the
    participation bit is set, the raw chunk otherwise; the bitmask words are
    the groups' participation words; a compressed slot is read for
    4*ceil((B-m)/32) bytes and its bytes past that are left as they were."""
    meta, x = _slot_case(cb, frac, 32 * 3 + 7, cb + int(frac * 100), tail)
    n = x.size
    nch = (n + cb - 1) // cb
    m = int(meta[16:20].view(np.uint32)[0])
    B = 8 * cb
    slots, bm = O.ibp_slots_encode(meta, x, threads=3)
    assert bm.size == (nch + 31) // 32
    for g in range((nch + 31) // 32):
        nin = min(32, nch - 32 * g)
        last = n - (32 * g + nin - 1) * cb
        pay = O.ibp_encode_group(meta, x[32 * g * cb: 32 * g * cb + (nin - 1) * cb + min(cb, last)],
                                 nin, min(cb, last) if last < cb else 0)
        pbits = np.unpackbits(pay, bitorder="little")
        assert int(pay[:4].view(np.uint32)[0]) == int(bm[g])
        q = 32
        for t in range(nin):
            s = 32 * g + t
            ln = min(cb, n - s * cb)
            p = (int(bm[g]) >> t) & 1
            blen = (B - m) if p else 8 * ln
            sb = np.unpackbits(slots[s * cb: s * cb + ln], bitorder="little")
            assert np.array_equal(sb[:blen], pbits[q:q + blen]), (s, p)
            rb = O.ibp_slot_read_bytes(meta, p, ln)
            assert rb == (4 * ((B - m + 31) // 32) if p else ln)
            if p:
                assert not sb[blen:8 * rb].any()  # zero bits up to the word
                assert np.array_equal(slots[s * cb + rb: s * cb + ln], x[s * cb + rb: s * cb + ln])
            q += blen


@pytest.mark.parametrize("cb,frac", [(64, 0.3), (512, 0.12), (20, 0.5), (32, 1.0), (16, 0.0)])
def test_slots_gather_round_trip(cb, frac):
    meta, x = _slot_case(cb, frac, 150, 7 + cb, tail=4 if cb > 4 else 0)
    n = x.size
    nch = (n + cb - 1) // cb
    slots, bm = O.ibp_slots_encode(meta, x)
    rng = np.random.default_rng(cb)
    idx = np.concatenate([rng.integers(0, nch, 200), [nch - 1, 0, nch - 1]])
    rows, read = O.ibp_slots_gather(meta, slots, n, bm, idx)
    want_read = 0
    for i, s in enumerate(idx):
        ln = min(cb, n - s * cb)
        assert np.array_equal(rows[i, :ln], x[s * cb: s * cb + ln]), s
        p = (int(bm[s // 32]) >> (s % 32)) & 1
        want_read += O.ibp_slot_read_bytes(meta, p, ln)
    assert read == want_read
    # reading a compressed slot reads less than the raw chunk exactly when
    # m >= 32 (whole words dropped)
    m = int(meta[16:20].view(np.uint32)[0])
    if m >= 32 and bm.any():
        assert read < sum(min(cb, n - s * cb) for s in idx)
