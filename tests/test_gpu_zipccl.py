"""GPU parity of the ZipCCL codec against the bit-serial oracle.

Every test runs the CUDA path through the C ABI (liblbb16.so via ctypes) on
seeded inputs and compares, byte for byte, with the oracle on the same input
bytes: the compressed stream (header, tables, slots, escapes, padding) and the
decoded tensor.  The codebooks follow the parity protocol of zc_parity.py.
"""
import numpy as np
import pytest
import torch

import oracle as O
from lossless_bit_level_bf16_gb300 import abi, workloads as W, zipccl as Z
from oracle_split import zc_stream_equal
from zc_parity import check_plan, check_stream_equal, fields

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _bits_np(t):
    return W.bf16_bits(t)


def _roundtrip(x, seg=None, chunk=4096, books=None, fit=True):
    """Returns (stream bytes on host, plan, decoded tensor)."""
    plan = Z.Plan(x.numel(), seg, chunk)
    if books is not None:
        plan.set_books(books)
    elif fit:
        plan.fit(x)
    out, nb = plan.compress(x)
    torch.cuda.synchronize()
    assert plan.status() == 0
    total = int(nb.item())
    y = Z.decompress(out, n=x.numel(), in_bytes=total)
    torch.cuda.synchronize()
    assert abi.status(Z.decompress_workspace(out.device)) == 0
    return out[:total].cpu().numpy(), plan, y


def _check_full(x, seg=None, chunk=4096, books=None, near_ties=False):
    xb = _bits_np(x)
    st, plan, y = _roundtrip(x, seg, chunk, books)
    bk, mu, sg = plan.info()
    if books is None:
        check_plan(xb, seg, bk, mu, sg, allow_near_ties=near_ties)
    else:
        assert np.array_equal(bk.reshape(-1), np.asarray(books, np.uint8).reshape(-1))
    check_stream_equal(st, xb, seg, chunk, bk)
    assert torch.equal(y.view(torch.int16), x.view(torch.int16)), "decode must be bit-exact"
    rc, yo = O.zc_decode(st)
    assert rc == 0 and np.array_equal(yo, xb)
    return st, plan


def test_gaussian_1m():
    x = W.zc_gaussian(1 << 20, sigma=0.02, seed=0, device=DEV)
    st, plan = _check_full(x)
    bk, mu, sg = plan.info()
    assert list(bk[0]) == list(range(116, 123))
    ratio = x.numel() * 2 / st.size
    assert ratio > 1.40


@pytest.mark.parametrize("chunk", [1024, 2048, 4096, 8192, 65536])
def test_every_bf16_pattern(chunk):
    g = torch.Generator().manual_seed(chunk)
    allv = torch.randperm(65536, generator=g).to(torch.int32)
    allv = (allv - (allv >= 32768).to(torch.int32) * 65536).to(torch.int16)
    for books in ([116, 117, 118, 119, 120, 121, 122], [0, 1, 2, 3, 4, 5, 6],
                  [249, 250, 251, 252, 253, 254, 255], [0, 50, 100, 127, 128, 200, 255]):
        for n in (1, 15, 1023, chunk + 17, 65536):
            x = allv[:n].to(DEV).view(torch.bfloat16)
            _check_full(x, None, chunk, books)


@pytest.mark.parametrize("ntiles", [127, 128, 129, 257])
def test_escape_overflow_across_lookback_blocks(ntiles):
    """The encoder groups its 8192-slot tickets in blocks of 128 for the
    look-back.  Every third ticket here holds random bit patterns (almost
    every value an escape, more than a ticket stages, so the ticket resolves
    its offset at once); the others N(0, 0.01) (about 2 % escapes, resolved a
    ticket later); across block boundaries, with a ragged last ticket."""
    n = ntiles * 8192 - 5
    x = W.zc_gaussian(n, sigma=0.01, seed=ntiles)
    xb = x.view(torch.int16)
    g = torch.Generator().manual_seed(1000 + ntiles)
    for t in range(0, ntiles, 3):
        lo, hi = t * 8192, min(n, (t + 1) * 8192)
        xb[lo:hi] = torch.randint(-32768, 32768, (hi - lo,), generator=g, dtype=torch.int32).to(torch.int16)
    _check_full(x.to(DEV), None, 4096, [116, 117, 118, 119, 120, 121, 122])


def test_gradient_blocks_64m():
    x, seg = W.zc_gradient(device=DEV)
    st, plan = _check_full(x, seg)
    assert x.numel() * 2 / st.size > 1.3


def test_moe_experts():
    x, seg, counts = W.zc_moe(device=DEV)
    assert sum(counts) == 8192 and len(seg) == 65
    st, plan = _check_full(x, seg)


def test_predictor_scales_and_near_ties():
    """Codebooks of many tiny segments with chosen statistics.

    {+a, -a} has mean 0 and sigma a exactly; {+a, -a, +b, -b} has mean 0 and
    sigma sqrt((a^2 + b^2)/2), which lands within 4e-5 (relative) of the
    mantissa 1.6467... where the 7th and 8th field masses of a zero-mean
    Gaussian swap places, so close that the predictor must fall back from its
    fp32 ranking to exact fp64 masses; {a, b} gives mean (a + b)/2.  Every
    book must equal the oracle's for the GPU's own mean and sigma.
    """
    segs = []
    for E in range(-40, 20, 3):
        for m in (1.0, 1.25, 1.5, 1.6328125, 1.640625, 1.6484375, 1.65625, 1.75, 1.9921875):
            a = m * 2.0 ** E
            segs.append([a, -a])
    for E in range(-30, 20, 5):
        for a, b in ((1.1171875, 0.328125), (1.21875, 1.984375), (1.1015625, 9.25),
                     (1.15625, 0.1376953125), (1.078125, 4.53125)):
            segs.append([x * 2.0 ** E for x in (a, -a, b, -b)])
    rng = np.random.default_rng(0)
    for _ in range(150):
        a = float(rng.standard_normal()) * 2.0 ** int(rng.integers(-30, 10))
        b = float(rng.standard_normal()) * 2.0 ** int(rng.integers(-30, 10))
        segs.append([a, b])
    seg = [0]
    for v in segs:
        seg.append(seg[-1] + len(v))
    x = torch.tensor([v for vs in segs for v in vs], dtype=torch.float32).to(torch.bfloat16).to(DEV)
    _check_full(x, seg, 1024, near_ties=True)


@pytest.mark.parametrize("chunk", [1024, 4096, 16384])
def test_ragged_segments_and_alignment(chunk):
    # empty segments, odd starts (no 16-byte alignment), tiny and large ones
    lens = [0, 1, 7, 4095, 0, 4097, 12345, 3, 65536 + 5, 0]
    seg = [0]
    for L in lens:
        seg.append(seg[-1] + L)
    parts = []
    for i, L in enumerate(lens):
        parts.append(W.zc_gaussian(L, sigma=[0.02, 1e-3, 3.0, 1e-5][i % 4], seed=i, device=DEV))
    x = torch.cat(parts)
    _check_full(x, seg, chunk)
    # a view at an odd element offset (input pointer not 16-byte aligned)
    big = W.zc_gaussian(50001, sigma=0.5, seed=5, device=DEV)
    _check_full(big[1:], None, chunk)


@pytest.mark.parametrize("chunk", [3072, 5120, 7168, 9216, 15360, 64512])
def test_chunk_not_power_of_two(chunk):
    """Chunk sizes that are multiples of 1024 but not powers of two: the
    encoder's 8192-slot tickets then start inside chunks and touch up to two
    partial chunks.  Segments of mixed scales and ragged lengths, one with
    every value escaping, against the oracle; then every bf16 pattern."""
    lens = [5, 8192 * 3 + 1000, 0, chunk * 2 + 1, 100_000, chunk - 1, 70_001]
    seg = [0]
    for L in lens:
        seg.append(seg[-1] + L)
    parts = [W.zc_gaussian(L, sigma=[0.02, 1.0, 1e-3, 3e-5][i % 4], seed=40 + i, device=DEV)
             for i, L in enumerate(lens)]
    parts[3] = torch.full((lens[3],), float("nan"), dtype=torch.bfloat16, device=DEV)
    x = torch.cat(parts)
    _check_full(x, seg, chunk)
    g = torch.Generator().manual_seed(chunk)
    allv = torch.randperm(65536, generator=g).to(torch.int32)
    allv = (allv - (allv >= 32768).to(torch.int32) * 65536).to(torch.int16)
    _check_full(allv.to(DEV).view(torch.bfloat16), None, chunk, [116, 117, 118, 119, 120, 121, 122])


@pytest.mark.parametrize("chunk", [1024, 3072, 4096, 9216, 65536])
def test_raw_fallback(chunk):
    """Incompressible full chunks (random bit patterns, all-NaN runs) are
    stored raw -- 2C bytes, bit 63 of the table entry -- next to coded chunks,
    in several segments with ragged ends, in tickets that take the direct
    path (raw chunks) and the staged one; with the plan's own books and with
    a given book; stream equal to the oracle's, decode exact."""
    g = torch.Generator().manual_seed(chunk)
    lens = [chunk * 3 + 5, 7, chunk * 9, 2 * chunk - 3, 40_000]
    parts = []
    for i, L in enumerate(lens):
        v = W.zc_gaussian(L, sigma=0.01, seed=60 + i)
        bits = v.view(torch.int16)
        for c0 in range(0, L, chunk):
            if (c0 // chunk + i) % 3 == 1:  # every third chunk incompressible
                n = min(chunk, L - c0)
                bits[c0:c0 + n] = torch.randint(-32768, 32768, (n,), generator=g,
                                                dtype=torch.int32).to(torch.int16)
        if i == 3:
            v[: min(L, chunk)] = float("nan")
        parts.append(v)
    x = torch.cat(parts).to(DEV)
    seg = [0]
    for L in lens:
        seg.append(seg[-1] + L)
    st, plan = _check_full(x, seg, chunk)
    off_escoff = int(st[48:56].view(np.uint64)[0])
    nch = int(st[24:32].view(np.uint64)[0])
    flags = st[off_escoff:off_escoff + 8 * nch].view(np.uint64) >> np.uint64(63)
    assert flags.sum() >= 5
    _check_full(x, seg, chunk, [[116, 117, 118, 119, 120, 121, 122]] * len(lens))


def _fit_cases():
    x1 = W.zc_gaussian(1 << 20, sigma=0.02, seed=0, device=DEV)
    yield "gaussian", x1, None, W.zc_gaussian(1 << 20, sigma=0.05, seed=1, device=DEV)
    x, seg = W.zc_gradient(n_blocks=64, device=DEV)
    y, _ = W.zc_gradient(n_blocks=64, seed=1, device=DEV)
    yield "gradient", x, seg, y
    lens = [0, 1, 7, 4095, 0, 4097, 12345, 3, 65536 + 5, 20000, 20000, 20000]
    seg = [0]
    for L in lens:
        seg.append(seg[-1] + L)
    parts = [W.zc_gaussian(L, sigma=[0.02, 1e-3, 3.0, 1e-5, 1e-30, 1e30][i % 6], seed=i, device=DEV)
             for i, L in enumerate(lens)]
    parts[9][::13] = float("inf")
    parts[10][::17] = float("nan")
    x = torch.cat(parts)
    yield "ragged", x, seg, x.flip(0).contiguous()


def test_compress_fit():
    """zc_compress_fit: the stream is the oracle's for the codebooks in force
    when the call starts; afterwards the plan's mean, sigma and codebooks are
    those of the data (the oracle's fp64 statistics, within the fused sums'
    rounding; the codebook equal to the oracle's own); the next call encodes
    with them.  Includes empty, tiny, ragged segments, inf/NaN values and
    values whose squares leave the fp32 range (summed in fp64)."""
    for name, x, seg, y in _fit_cases():
        nseg = 1 if seg is None else len(seg) - 1
        plan = Z.Plan(x.numel(), seg, 4096)
        first = [[116, 117, 118, 119, 120, 121, 122]] * nseg
        plan.set_books(first)
        xb, yb = _bits_np(x), _bits_np(y)
        out, nb = plan.compress_fit(x)
        torch.cuda.synchronize()
        assert plan.status() == 0, name
        check_stream_equal(out[: int(nb.item())].cpu().numpy(), xb, seg, 4096, first)
        bk, mu, sg = plan.info()
        check_plan(xb, seg, bk, mu, sg, rel=12)
        out2, nb2 = plan.compress_fit(y)  # encodes with x's codebooks, refits to y
        torch.cuda.synchronize()
        assert plan.status() == 0, name
        check_stream_equal(out2[: int(nb2.item())].cpu().numpy(), yb, seg, 4096, bk)
        bk2, mu2, sg2 = plan.info()
        check_plan(yb, seg, bk2, mu2, sg2, rel=12)
        # the same books as the separate statistics pass, except at a near-tie
        ref = Z.Plan(y.numel(), seg, 4096)
        ref.fit(y)
        assert np.array_equal(ref.info()[0], bk2), name


def test_degenerate_values():
    n = 10000
    # constant data (sigma = 0), all zeros, NaN / inf mixes, huge and tiny values
    cases = [
        torch.full((n,), 1.0, device=DEV, dtype=torch.bfloat16),
        torch.zeros(n, device=DEV, dtype=torch.bfloat16),
        torch.full((n,), float("nan"), device=DEV, dtype=torch.bfloat16),
        W.zc_gaussian(n, sigma=1e30, seed=1, device=DEV),
        W.zc_gaussian(n, sigma=1e-30, seed=2, device=DEV),
    ]
    mix = W.zc_gaussian(n, sigma=0.02, seed=3, device=DEV)
    mix[::17] = float("inf")
    mix[1::17] = float("-inf")
    mix[2::19] = float("nan")
    mix[3::23] = 3e38
    cases.append(mix)
    for x in cases:
        _check_full(x)


def test_empty_input():
    x = torch.empty(0, device=DEV, dtype=torch.bfloat16)
    st, plan, y = _roundtrip(x)
    assert st.size == 384 and y.numel() == 0
    check_stream_equal(st, np.zeros(0, np.uint16), None, 4096, plan.info()[0])


@pytest.mark.parametrize("mb", [1, 4, 16, 64, 256])
def test_sweep_sizes_full(mb):
    n = mb * (1 << 20) // 2
    x = W.zc_gaussian(n, sigma=0.01, seed=0, device=DEV)
    _check_full(x)


@pytest.mark.slow
@pytest.mark.parametrize("gib", [1, 4])
def test_sweep_sizes_full_large(gib):
    """The sweep's 1 and 4 GiB points (bf16 N(0, 0.01), one segment, chunk
    4096): codebook checked as for every other size, the whole stream equal to
    the oracle's (encoded in pieces of whole chunks on all host cores), exact
    decode on the device."""
    n = gib * (1 << 30) // 2
    C = 4096
    x = W.zc_gaussian(n, sigma=0.01, seed=0, device=DEV)
    plan = Z.Plan(n, None, C)
    plan.fit(x)
    out, nb = plan.compress(x)
    y = Z.decompress(out, n=n)
    torch.cuda.synchronize()
    assert plan.status() == 0 and abi.status(Z.decompress_workspace(out.device)) == 0
    assert torch.equal(y.view(torch.int16), x.view(torch.int16))
    del y
    total = int(nb.item())
    st = out[:total].cpu().numpy()
    del out
    xb = _bits_np(x)
    del x
    bk, mu, sg = plan.info()
    check_plan(xb, None, bk, mu, sg)
    zc_stream_equal(st, xb, C, bk[0])
    assert int(st[:4].view(np.uint32)[0]) == 0x3143435A


def test_decode_rejects_corrupt_streams():
    x = W.zc_gaussian(100000, sigma=0.02, seed=9, device=DEV)
    plan = Z.Plan(x.numel(), None, 4096)
    plan.fit(x)
    out, nb = plan.compress(x)
    torch.cuda.synchronize()
    total = int(nb.item())
    good = out[:total].clone()
    ws = Z.decompress_workspace(out.device)

    def run(buf, in_bytes=None, n=x.numel()):
        y = torch.zeros(n, dtype=torch.bfloat16, device=DEV)
        Z.decompress(buf, out=y, in_bytes=in_bytes if in_bytes is not None else buf.numel())
        torch.cuda.synchronize()
        return abi.status(ws)

    assert run(good) == 0
    hdr = good[:128].cpu().numpy().view(np.uint64)
    for off in (0, 8, 16, 24, 32, 48, 56, 64, 72):
        bad = good.clone()
        bad[off] ^= 0x5A
        assert run(bad) in (abi.ZC_ERR_FORMAT, abi.ZC_ERR_CAPACITY), off
    assert run(good, in_bytes=total - 128) == abi.ZC_ERR_FORMAT
    assert run(good, n=x.numel() - 1) == abi.ZC_ERR_CAPACITY
    # escape-offset table entries out of range / inconsistent with the planes
    off_escoff = int(hdr[6])
    bad = good.clone()
    bad[off_escoff + 8 * 5: off_escoff + 8 * 6] = torch.tensor(
        list(np.uint64(1 << 40).tobytes()), dtype=torch.uint8, device=DEV)
    assert run(bad) == abi.ZC_ERR_FORMAT
    bad = good.clone()
    bad[off_escoff + 8 * 5] ^= 1
    assert run(bad) == abi.ZC_ERR_FORMAT
    # eight codes of chunk 0 zeroed in all three planes: they read as escapes,
    # so the chunk's escape count no longer matches the table
    off_static = int(hdr[7])
    bad = good.clone()
    for k in range(3):
        bad[off_static + 4096 + 512 * k + 3] = 0
    assert run(bad) == abi.ZC_ERR_FORMAT


def test_output_capacity_reported():
    x = torch.full((50000,), float("nan"), dtype=torch.bfloat16, device=DEV)  # all escapes
    plan = Z.Plan(x.numel(), None, 4096)
    plan.fit(x)
    fixed = O.zc_stream_bytes(x.numel(), None, 4096, 0)  # everything but the dynamic bytes
    out = torch.zeros(fixed + 1000, dtype=torch.uint8, device=DEV)
    plan.compress(x, out=out)
    torch.cuda.synchronize()
    assert plan.status() == abi.ZC_ERR_CAPACITY


def test_plan_is_deterministic_and_reusable():
    x = W.zc_gaussian(3 << 20, sigma=0.07, seed=4, device=DEV)
    plan = Z.Plan(x.numel(), None, 4096)
    plan.fit(x)
    a, na = plan.compress(x)
    a = a[: int(na.item())].clone()
    plan.fit(x)
    b, nb = plan.compress(x)
    assert torch.equal(a, b[: int(nb.item())])
    # reuse the plan's codebook on another tensor of the same layout
    x2 = W.zc_gaussian(3 << 20, sigma=0.07, seed=5, device=DEV)
    c, nc = plan.compress(x2)
    torch.cuda.synchronize()
    st = c[: int(nc.item())].cpu().numpy()
    check_stream_equal(st, _bits_np(x2), None, 4096, plan.info()[0])
