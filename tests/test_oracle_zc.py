"""Pins for the ZipCCL oracle (CPU only).

Each test ties the oracle to something other than itself: a stream derived by
hand from the layout, the exact round trip over every bf16 bit pattern, the
closed-form size, numpy's statistics, the closed-form codebook window for
zero-mean Gaussians (with its switch point solved independently with scipy),
and the empirical top-7 exponents of large Gaussian samples.

Page cited: "ZipCCL: Efficient Lossless Data Compression of Communication
Collectives for Accelerating LLM Training", 2. Metodologia A-C.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _fields(u16):
    return (np.asarray(u16, np.uint16) >> 7) & 0xFF


def _bf16_round(f32):
    """Round float32 values to bf16 bit patterns with torch's cast (RNE)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(f32, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- format pins

def _dynamic_bytes(x, C, book):
    """Dynamic-region bytes of a one-segment stream, chunk by chunk: the
    escape count, or for a full chunk the raw form's remainder 5C/8 when that
    is smaller (the raw fallback)."""
    tot = 0
    for c0 in range(0, x.size, C):
        xc = x[c0:c0 + C]
        ne = int(np.count_nonzero(~np.isin(_fields(xc), book)))
        tot += min(ne, 5 * C // 8) if xc.size == C else ne
    return tot


def test_golden_tiny_stream():
    g = json.load(open(os.path.join(GOLD, "zc_tiny_stream.json")))
    x = np.array([int(h, 16) for h in g["input_u16_hex"]], np.uint16)
    st, books, _, _ = O.zc_encode(x, chunk_elems=g["chunk_elems"],
                                  books=np.array(g["book"], np.uint8))
    assert st.size == g["total_bytes"]
    want = np.zeros(g["total_bytes"], np.uint8)
    for off, hx in g["spans"]:
        b = bytes.fromhex(hx)
        want[off:off + len(b)] = np.frombuffer(b, np.uint8)
    bad = np.nonzero(st != want)[0]
    assert bad.size == 0, f"first differing byte at {bad[:8]}"
    rc, y = O.zc_decode(st)
    assert rc == 0 and np.array_equal(y, x)


BOOKS = [
    np.arange(116, 123, dtype=np.uint8),               # N(0, 0.02)
    np.arange(0, 7, dtype=np.uint8),                   # zero / subnormal field
    np.arange(249, 256, dtype=np.uint8),               # inf / NaN field 255
    np.array([0, 50, 100, 127, 128, 200, 255], np.uint8),
]


@pytest.mark.parametrize("C", [1024, 4096])
@pytest.mark.parametrize("bi", range(len(BOOKS)))
def test_bruteforce_every_bf16_pattern(C, bi):
    rng = np.random.default_rng(1234 + bi)
    allv = rng.permutation(np.arange(65536, dtype=np.uint32)).astype(np.uint16)
    book = BOOKS[bi]
    for n in (1, 1023, C - 1, C + 1, 65536):
        x = allv[:n]
        st, _, _, _ = O.zc_encode(x, chunk_elems=C, books=book)
        rc, y = O.zc_decode(st)
        assert rc == 0
        assert np.array_equal(y, x), "round trip must be bit-exact"
        assert int(st[32:40].view(np.uint64)[0]) == _dynamic_bytes(x, C, book)
        assert st.size == O.zc_stream_bytes(n, None, C, _dynamic_bytes(x, C, book))


@pytest.mark.parametrize("C", [1024, 4096, 8192])
def test_size_is_sum_of_code_lengths(C):
    # 11 bits per in-book element, 19 (11 + 8 escaped exponent bits) otherwise
    rng = np.random.default_rng(7)
    x = _bf16_round(rng.normal(0, 0.02, size=8 * C).astype(np.float32))
    x[::97] = 0x7FC1  # NaNs: always escape
    book = np.arange(116, 123, dtype=np.uint8)
    st, _, _, _ = O.zc_encode(x, chunk_elems=C, books=book)
    hdr = st[:80].view(np.uint64)
    off_static, off_esc, esc_total = int(hdr[7]), int(hdr[8]), int(hdr[4])
    n_in = int(np.count_nonzero(np.isin(_fields(x), book)))
    n_out = x.size - n_in
    payload_bits = 8 * ((off_esc - off_static) + esc_total)
    assert payload_bits == 11 * n_in + 19 * n_out
    assert esc_total == n_out


def test_chunk_entry_matches_stream():
    rng = np.random.default_rng(3)
    C = 4096
    x = _bf16_round(rng.normal(0, 1.0, size=3 * C + 77).astype(np.float32))
    book = np.arange(122, 129, dtype=np.uint8)
    st, _, _, _ = O.zc_encode(x, chunk_elems=C, books=book)
    hdr = st[:80].view(np.uint64)
    off_escoff, off_static, off_esc = int(hdr[6]), int(hdr[7]), int(hdr[8])
    S = C * 11 // 8
    eo = st[off_escoff:off_escoff + 8 * 5].view(np.uint64)
    for c in range(4):
        slot, esc, raw = O.zc_encode_chunk(x[c * C:(c + 1) * C], C, book)
        assert not raw
        assert np.array_equal(slot, st[off_static + c * S: off_static + (c + 1) * S])
        assert np.array_equal(esc, st[off_esc + int(eo[c]): off_esc + int(eo[c + 1])])


def test_multisegment_layout_and_books():
    rng = np.random.default_rng(11)
    sig = [0.02, 1e-3, 5.0, 0.3]
    lens = [10000, 0, 4096, 12345, 1]
    parts, seg = [], [0]
    for i, L in enumerate(lens):
        s = sig[i % len(sig)]
        parts.append(_bf16_round(rng.normal(0, s, size=L).astype(np.float32)))
        seg.append(seg[-1] + L)
    x = np.concatenate(parts)
    st, books, mus, sgs = O.zc_encode(x, seg_off=seg, chunk_elems=2048)
    rc, y = O.zc_decode(st)
    assert rc == 0 and np.array_equal(y, x)
    nseg = len(lens)
    recs = st[128:128 + 64 * nseg].reshape(nseg, 64)
    esc_start = 0
    chunk_start = 0
    for s in range(nseg):
        r = recs[s, :48].view(np.uint64)
        assert int(r[0]) == seg[s] and int(r[1]) == lens[s]
        # each segment is chunked on its own: ceil(len / C) chunks, numbered
        # after the chunks of the segments before it
        assert int(r[2]) == chunk_start
        assert int(r[3]) == -(-lens[s] // 2048)
        chunk_start += -(-lens[s] // 2048)
        assert int(r[4]) == esc_start
        xs = x[seg[s]:seg[s + 1]]
        # the book of each segment comes from that segment's own values
        fin = _fields(xs) != 255
        vals = xs[fin].astype(np.uint32) << 16
        v = vals.view(np.float32).astype(np.float64)
        if v.size:
            assert mus[s] == pytest.approx(v.mean(), rel=1e-12, abs=1e-300)
            assert sgs[s] == pytest.approx(v.std(), rel=1e-9, abs=1e-300)
        assert np.array_equal(books[s], O.zc_predict(mus[s], sgs[s]))
        assert np.array_equal(recs[s, 48:55], books[s])
        n_esc = int(np.count_nonzero(~np.isin(_fields(xs), books[s])))
        assert int(r[5]) == n_esc
        esc_start += n_esc
    assert st.size == O.zc_stream_bytes(x.size, seg, 2048, esc_start)
    assert int(st[24:32].view(np.uint64)[0]) == chunk_start == 5 + 0 + 2 + 7 + 1


def test_empty_input():
    x = np.zeros(0, np.uint16)
    st, books, _, _ = O.zc_encode(x, chunk_elems=4096)
    assert st.size == 128 + 128 + 128
    assert np.array_equal(books[0], np.arange(7))
    rc, y = O.zc_decode(st)
    assert rc == 0 and y.size == 0


def test_decode_rejects_corruption():
    rng = np.random.default_rng(5)
    x = _bf16_round(rng.normal(0, 0.02, size=5000).astype(np.float32))
    st, _, _, _ = O.zc_encode(x, chunk_elems=1024)
    for off, val in [(0, 0x00), (8, 0x01), (24, 0x09), (72, 0x00), (64, 0x05)]:
        bad = st.copy()
        bad[off] ^= 0xFF if val == 0 else val
        rc, _ = O.zc_decode(bad)
        assert rc == O.E_FORMAT, off
    rc, _ = O.zc_decode(st[: st.size - 128])
    assert rc == O.E_FORMAT
    # escape-offset table made non-monotone
    hdr = st[:80].view(np.uint64)
    bad = st.copy()
    bad[int(hdr[6]) + 8: int(hdr[6]) + 16] = np.frombuffer(
        np.uint64(10 ** 9).tobytes(), np.uint8)
    assert O.zc_decode(bad)[0] == O.E_FORMAT


# ---------------------------------------------------------------- statistics

def test_stats_match_numpy():
    rng = np.random.default_rng(9)
    x = _bf16_round(rng.normal(0.001, 0.02, size=200001).astype(np.float32))
    x[::1000] = 0x7F80   # +inf
    x[1::1000] = 0xFFC0  # NaN
    cnt, s1, s2 = O.zc_stats(x)
    fin = _fields(x) != 255
    v = (x[fin].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert cnt == v.size
    assert s1 == pytest.approx(v.sum(), rel=1e-12)
    assert s2 == pytest.approx((v * v).sum(), rel=1e-12)
    mu, sg = O.zc_moments(cnt, s1, s2)
    assert mu == pytest.approx(v.mean(), rel=1e-11)
    assert sg == pytest.approx(v.std(ddof=0), rel=1e-10)


# ---------------------------------------------------------------- predictor

def _switch_point():
    """m* such that, for sigma = m * 2^E, the zero-mean window moves up one
    field: the binade [2^(E-5), 2^(E-4)) and [2^(E+2), 2^(E+3)) then hold
    equal Gaussian mass.  Solved with scipy's normal CDF."""
    from scipy.optimize import brentq
    from scipy.stats import norm

    def diff(m):
        z = 1.0 / m  # 2^E / sigma
        lo = norm.cdf(z / 16) - norm.cdf(z / 32)
        hi = norm.cdf(8 * z) - norm.cdf(4 * z)
        return lo - hi
    return brentq(diff, 1.0, 2.0 - 1e-12, xtol=1e-15)


def test_switch_point_value():
    assert _switch_point() == pytest.approx(1.6467032064597, abs=1e-9)


def test_zero_mean_window_closed_form():
    ms = _switch_point()
    sig = np.concatenate([np.logspace(-30, 30, 1501), [0.02, 0.01, 0.1, 1.0, 2.0]])
    checked = 0
    for s in sig:
        m, E = math.frexp(float(s))  # s = m * 2^E, m in [0.5, 1)
        m, E = 2 * m, E - 1
        if abs(m - ms) < 1e-6:
            continue
        lo = E - 5 + (1 if m >= ms else 0) + 127
        if lo < 1 or lo + 6 > 254:
            continue
        assert np.array_equal(O.zc_predict(0.0, float(s)), np.arange(lo, lo + 7)), s
        checked += 1
    assert checked > 1400


@pytest.mark.parametrize("sigma", [0.02, 0.01, 0.1, 1.0, 3e-4, 7.5, 1e-2 * 1.9])
def test_predicted_book_is_empirical_top7(sigma):
    rng = np.random.default_rng(int(sigma * 1e6) % 2**31)
    x = _bf16_round(rng.normal(0.0, sigma, size=1 << 22).astype(np.float32))
    cnt = np.bincount(_fields(x), minlength=256)
    top = np.sort(np.argsort(-cnt, kind="stable")[:7])
    book = O.zc_predict(0.0, sigma)
    assert np.array_equal(book, top)
    cover = cnt[book].sum() / x.size
    # the page reports the top 7 exponents covering more than 97 % of values;
    # for an exact Gaussian the coverage of the best 7 binades is >= 96.97 %
    assert cover >= 0.9690


@pytest.mark.parametrize("mu_over_sigma", [0.25, 1.0, 3.0])
def test_predicted_book_nonzero_mean(mu_over_sigma):
    sigma = 0.013
    mu = mu_over_sigma * sigma
    rng = np.random.default_rng(99)
    x = _bf16_round(rng.normal(mu, sigma, size=1 << 22).astype(np.float32))
    cnt = np.bincount(_fields(x), minlength=256)
    book = O.zc_predict(mu, sigma)
    top = np.sort(np.argsort(-cnt, kind="stable")[:7])
    # compare as sets of the 6 surest fields plus the mass of the 7th
    assert len(set(book) & set(top)) >= 6
    emp_cover = cnt[top].sum() / x.size
    pred_cover = cnt[book].sum() / x.size
    assert pred_cover >= emp_cover - 0.002


def test_predictor_degenerate_cases():
    assert np.array_equal(O.zc_predict(0.0, 0.0), np.arange(7))
    assert np.array_equal(O.zc_predict(1.0, 0.0), np.arange(124, 131))
    assert np.array_equal(O.zc_predict(-3e38, 0.0), np.arange(248, 255))
    assert np.array_equal(O.zc_predict(1e-40, 0.0), np.arange(7))
    # all values non-finite: no statistics -> mu = sigma = 0
    x = np.full(100, 0x7FC0, np.uint16)
    st, books, mus, sgs = O.zc_encode(x, chunk_elems=1024)
    assert mus[0] == 0 and sgs[0] == 0 and np.array_equal(books[0], np.arange(7))
    # constant data: sigma exactly 0, window centred on the value's field
    x = np.full(5000, 0x3F80, np.uint16)  # 1.0, field 127
    st, books, mus, sgs = O.zc_encode(x, chunk_elems=1024)
    assert sgs[0] == 0.0 and np.array_equal(books[0], np.arange(124, 131))
    assert int(st[32:40].view(np.uint64)[0]) == 0


def test_mass_sums_to_one():
    for mu, s in [(0.0, 0.02), (0.5, 0.1), (-2.0, 3.0)]:
        tot = sum(O.zc_mass(mu, s, f) for f in range(1, 255))
        assert tot == pytest.approx(1.0, abs=1e-12)


def _norm_mass(mu, sigma, f):
    """P(2^(f-127) <= |X| < 2^(f-126)) for X ~ N(mu, sigma), from scipy's
    normal distribution: the positive interval [a, 2a) plus the negative one
    (-2a, -a], each as a difference of upper tails (or of lower tails when
    the interval lies below the mean), which keeps the difference accurate."""
    from scipy.stats import norm
    a = 2.0 ** (f - 127)

    def interval(lo, hi):  # P(lo <= X < hi)
        if lo >= mu:
            return norm.sf(lo, mu, sigma) - norm.sf(hi, mu, sigma)
        if hi <= mu:
            return norm.cdf(hi, mu, sigma) - norm.cdf(lo, mu, sigma)
        return 1.0 - norm.cdf(lo, mu, sigma) - norm.sf(hi, mu, sigma)
    return interval(a, 2 * a) + interval(-2 * a, -a)


@pytest.mark.parametrize("mu,sigma", [(0.0, 0.02), (0.013, 0.013), (-0.05, 0.02), (3.0, 1.0),
                                      (-7.5e-4, 1e-3), (1e5, 2e3), (-0.2, 0.9)])
def test_mass_matches_scipy_normal(mu, sigma):
    """Every field mass for a nonzero mean against scipy: a wrong sign of mu in
    either the positive or the negative interval, or a swapped edge, moves the
    masses by far more than the tolerance."""
    checked = 0
    for f in range(1, 255):
        want = _norm_mass(mu, sigma, f)
        got = O.zc_mass(mu, sigma, f)
        if want < 1e-250:
            assert got < 1e-15  # rounding noise of CDF differences at most
            continue
        # absolute 1e-15: both sides take differences of normal CDF values
        # near 1/2 for bins far inside the bulk, each rounded to ~1e-16
        assert got == pytest.approx(want, rel=2e-9, abs=1e-15), (f, got, want)
        checked += want > 1e-6
    assert checked >= 1


@pytest.mark.parametrize("mu,sigma", [(0.013, 0.013), (-0.05, 0.02), (3.0, 1.0), (-0.2, 0.9),
                                      (0.02, 0.004), (-1e-3, 0.02)])
def test_nonzero_mean_book_is_top7_of_scipy_masses(mu, sigma):
    m = np.array([_norm_mass(mu, sigma, f) for f in range(1, 255)])
    order = np.argsort(-m, kind="stable")  # ties toward the smaller field
    gap = (m[order[6]] - m[order[7]]) / m[order[6]]
    assert gap > 1e-6, "case chosen away from a tie"
    want = np.sort(order[:7] + 1).astype(np.uint8)
    assert np.array_equal(O.zc_predict(mu, sigma), want)


# ---------------------------------------------------------------- raw fallback

@pytest.mark.parametrize("C", [1024, 3072, 4096])
def test_raw_fallback_chunks(C):
    """Full chunks whose escapes outnumber the raw form's remainder (5C/8
    bytes) are stored raw: the bf16 values' bytes fill the slot, their last
    5C/8 bytes are the chunk's dynamic part, bit 63 of its table entry is set;
    such a chunk takes exactly 2C bytes.  A chunk with exactly 5C/8 escapes
    stays coded, and so does the short last chunk, however many escapes it
    has.  Mixed, the round trip stays exact."""
    rng = np.random.default_rng(C)
    book = np.arange(116, 123, dtype=np.uint8)
    coded = _bf16_round(rng.normal(0, 0.01, size=C).astype(np.float32))
    noise = rng.integers(0, 65536, size=C, dtype=np.uint32).astype(np.uint16)
    edge = coded.copy()
    S = 11 * C // 8
    k = 5 * C // 8  # exactly as many escapes as the raw remainder: stays coded
    edge[:k] = 0x7FC0
    edge[k:] = np.where(np.isin(_fields(edge[k:]), book), edge[k:], 0x3C00 | (edge[k:] & 0x807F))
    tail = noise[:300]  # short last chunk: coded whatever its escapes
    x = np.concatenate([coded, noise, edge, noise[::-1], tail])
    st, _, _, _ = O.zc_encode(x, chunk_elems=C, books=book)
    rc, y = O.zc_decode(st)
    assert rc == 0 and np.array_equal(y, x)
    h = st[16:80].view(np.uint64)
    off_escoff, off_static, off_esc = int(h[4]), int(h[5]), int(h[6])
    eo = st[off_escoff:off_escoff + 8 * 6].view(np.uint64)
    raw = [int(v) >> 63 for v in eo[:5]]
    assert raw == [0, 1, 0, 1, 0] and int(eo[5]) >> 63 == 0
    dyn = [int(eo[c + 1] & ~np.uint64(1 << 63)) - int(eo[c] & ~np.uint64(1 << 63)) for c in range(5)]
    assert dyn[1] == dyn[3] == 5 * C // 8 and dyn[2] == k
    assert dyn[4] == int(np.count_nonzero(~np.isin(_fields(tail), book))) > 0
    for c in (1, 3):
        xb = x[c * C:(c + 1) * C].view(np.uint8)
        slot = st[off_static + c * S: off_static + (c + 1) * S]
        assert np.array_equal(slot, xb[:S])
        o = int(eo[c] & ~np.uint64(1 << 63))
        assert np.array_equal(st[off_esc + o: off_esc + o + dyn[c]], xb[S:])
    assert st.size == O.zc_stream_bytes(x.size, None, C, sum(dyn))
    s2, d2, r2 = O.zc_encode_chunk(x[C:2 * C], C, book)
    assert r2 and np.array_equal(s2, st[off_static + S: off_static + 2 * S]) and d2.size == 5 * C // 8


def test_raw_fallback_bounds_expansion():
    """Every value escaping (random bit patterns, a book none of them uses):
    the stream is the raw bytes plus headers, tables and padding -- at most
    19/16 of the input without the fallback, at most the input plus a few
    hundred bytes with it."""
    rng = np.random.default_rng(1)
    C = 4096
    x = rng.integers(0, 65536, size=40 * C + 17, dtype=np.uint32).astype(np.uint16)
    x = np.where(np.isin(_fields(x), [0, 1, 2, 3, 4, 5, 6]), x | 0x0400, x).astype(np.uint16)
    st, _, _, _ = O.zc_encode(x, chunk_elems=C, books=np.arange(7, dtype=np.uint8))
    rc, y = O.zc_decode(st)
    assert rc == 0 and np.array_equal(y, x)
    fixed = O.zc_stream_bytes(x.size, None, C, 0)
    assert st.size - fixed <= 40 * (5 * C // 8) + 17 + 128  # the 17-value tail is coded
    assert st.size <= 2 * x.size + 11 * C // 8 + 1024


def test_decode_rejects_bad_raw_flags():
    rng = np.random.default_rng(4)
    C = 1024
    book = np.arange(116, 123, dtype=np.uint8)
    x = np.concatenate([_bf16_round(rng.normal(0, 0.01, size=C).astype(np.float32)),
                        rng.integers(0, 65536, size=C, dtype=np.uint32).astype(np.uint16)])
    st, _, _, _ = O.zc_encode(x, chunk_elems=C, books=book)
    off_escoff = int(st[48:56].view(np.uint64)[0])
    for c in (0, 1, 2):  # flag a coded chunk, clear a raw one, flag the end entry
        bad = st.copy()
        bad[off_escoff + 8 * c + 7] ^= 0x80
        assert O.zc_decode(bad)[0] == O.E_FORMAT, c
