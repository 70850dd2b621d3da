"""GPU parity of the IBP codec against the bit-serial oracle.

The CUDA path runs through the C ABI on seeded inputs; the metadata blob, the
compressed stream and the decoded bytes are compared byte for byte with the
oracle on the same input bytes.  At full size (the 512 MB table, the sweep's
points up to 4 GiB) the whole stream is compared too: the oracle encodes the
input in pieces of whole groups, one oracle call per piece on all host cores,
and every byte of the GPU stream is checked against them (oracle_split.py).
"""
import numpy as np
import pytest
import torch

import oracle as O
from lossless_bit_level_bf16_gb300 import abi, ibp as I, workloads as W
from oracle_split import ibp_stream_equal

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ws(cb, n_bytes=0, n_samples=0):
    return torch.empty(max(I.workspace_bytes(cb, n_bytes, n_samples), 256), dtype=torch.uint8,
                       device=DEV)


def _u8(t):
    return t.detach().contiguous().view(torch.uint8).cpu().numpy().reshape(-1)


def _gpu_roundtrip(meta_dev, x, cb):
    n_bytes = x.numel() * x.element_size()
    ws = _ws(cb, n_bytes)
    st, nb = I.compress(meta_dev, x, cb, ws=ws)
    torch.cuda.synchronize()
    assert I.status(ws) == 0, abi.strerror(I.status(ws))
    total = int(nb.item())
    dws = _ws(cb)
    y = I.decompress(meta_dev, st, n_bytes, cb, in_bytes=total, ws=dws, dtype=torch.uint8)
    torch.cuda.synchronize()
    assert I.status(dws) == 0, abi.strerror(I.status(dws))
    return st[:total], y


@pytest.mark.parametrize("mode", [0, 1])
def test_meta_table_rows(mode):
    rows, idx = W.ibp_table(rows=200_000, cols=128, std=0.1, seed=0, device=DEV)
    samples = rows[idx].contiguous()
    ws = _ws(512, 0, samples.shape[0])
    meta = I.build_meta(samples, 512, T=0.9, mode=mode, ws=ws)
    torch.cuda.synchronize()
    assert I.status(ws) == 0
    ref = O.ibp_build_meta(_u8(samples), 512, T=0.9, mode=mode)
    got = _u8(meta)
    assert np.array_equal(got, ref), np.nonzero(got != ref)[0][:10]
    m = int(got[16:20].view(np.uint32)[0])
    assert (mode == 0 and m >= 512) or (mode == 1 and 400 <= m <= 640)


@pytest.mark.parametrize("cb", [16, 48, 64, 512, 1024, 1040, 2048, 4096])
@pytest.mark.parametrize("frac", [0.0, 0.12, 0.5, 1.0])
def test_random_masks(cb, frac):
    rng = np.random.default_rng(cb * 10 + int(frac * 100))
    B = cb * 8
    mask = (rng.uniform(size=B) < frac).astype(np.uint8)
    bitval = rng.integers(0, 2, size=B).astype(np.uint8) & mask
    meta = O.ibp_make_meta(cb, np.packbits(mask, bitorder="little"),
                           np.packbits(bitval, bitorder="little"))
    nch = 97
    bits = rng.integers(0, 2, size=(nch, B)).astype(np.uint8)
    force = rng.uniform(size=nch) < 0.6
    bits[force] = np.where(mask.astype(bool), bitval, bits[force])
    x = np.packbits(bits, axis=1, bitorder="little").reshape(-1)
    for n_bytes in (x.size, x.size - cb // 2 // 4 * 4 if cb >= 8 else x.size, 4, 0):
        xs = np.ascontiguousarray(x[:n_bytes])
        xd = torch.from_numpy(xs.copy()).to(DEV)
        md = torch.from_numpy(meta).to(DEV)
        st, y = _gpu_roundtrip(md, xd, cb)
        ref = O.ibp_encode(meta, xs)
        got = st.cpu().numpy()
        assert got.size == ref.size and np.array_equal(got, ref), (n_bytes, np.nonzero(got != ref)[0][:8])
        assert np.array_equal(y.cpu().numpy(), xs)


@pytest.mark.parametrize("mode", [0, 1])
def test_table_full_size(mode):
    """The 1,000,000 x 128 fp32 table (512 MB): metadata from its own 10,000
    seeded sample rows equal to the oracle's, the whole stream equal to the
    oracle's, exact decode."""
    rows, idx = W.ibp_table(device=DEV)
    samples = rows[idx].contiguous()
    assert samples.shape[0] == 10_000
    cb = 512
    ws = _ws(cb, 0, samples.shape[0])
    meta = I.build_meta(samples, cb, T=0.9, mode=mode, ws=ws)
    torch.cuda.synchronize()
    assert I.status(ws) == 0
    mh = _u8(meta)
    mref = O.ibp_build_meta(_u8(samples), cb, T=0.9, mode=mode)
    assert np.array_equal(mh, mref), np.nonzero(mh != mref)[0][:10]
    st, y = _gpu_roundtrip(meta, rows, cb)
    assert torch.equal(y.view(torch.int32), rows.view(-1).view(torch.int32))
    del y
    ibp_stream_equal(st.cpu().numpy(), mref, _u8(rows))
    m = int(mh[16:20].view(np.uint32)[0])
    print(f"mode {mode}: m={m} ratio={rows.numel() * 4 / st.numel():.4f}")


@pytest.mark.parametrize("mb", [1, 4, 16])
def test_sweep_full(mb):
    cb = 2048
    x = W.ibp_gaussian(mb * (1 << 20) // 4, std=0.02, seed=0, device=DEV)
    nch = x.numel() * 4 // cb
    idx = W.sample_rows(nch, 10_000, seed=1, device=DEV)
    samples = x.view(nch, cb // 4)[idx].contiguous()
    for mode in (0, 1):
        ws = _ws(cb, 0, samples.shape[0])
        meta = I.build_meta(samples, cb, T=0.9, mode=mode, ws=ws)
        mref = O.ibp_build_meta(_u8(samples), cb, T=0.9, mode=mode)
        assert np.array_equal(_u8(meta), mref)
        st, y = _gpu_roundtrip(meta, x, cb)
        ref = O.ibp_encode(mref, _u8(x))
        assert np.array_equal(st.cpu().numpy(), ref)
        assert torch.equal(y.view(torch.int32), x.view(torch.int32))


@pytest.mark.slow
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("mb", [64, 256, 1024, 4096])
def test_sweep_full_large(mb, mode):
    """The sweep's fp32 N(0, 0.02) weights at 64 MiB .. 4 GiB, 2048-byte
    chunks, metadata from 10,000 seeded sample chunks: metadata and the whole
    stream equal to the oracle's, exact decode."""
    cb = 2048
    x = W.ibp_gaussian(mb * (1 << 20) // 4, std=0.02, seed=0, device=DEV)
    nch = x.numel() * 4 // cb
    idx = W.sample_rows(nch, 10_000, seed=1, device=DEV)
    samples = x.view(nch, cb // 4)[idx].contiguous()
    meta = I.build_meta(samples, cb, T=0.9, mode=mode, ws=_ws(cb, 0, samples.shape[0]))
    mref = O.ibp_build_meta(_u8(samples), cb, T=0.9, mode=mode)
    assert np.array_equal(_u8(meta), mref)
    del samples
    st, y = _gpu_roundtrip(meta, x, cb)
    assert torch.equal(y.view(torch.int32), x.view(torch.int32))
    del y
    st_h = st.cpu().numpy()
    del st
    ibp_stream_equal(st_h, mref, _u8(x))


@pytest.mark.parametrize("cb", [4, 20, 52, 300, 2060, 4092])
@pytest.mark.parametrize("mode", [0, 1])
def test_chunk_sizes_not_multiple_of_16(cb, mode):
    """Chunk sizes that are multiples of 4 bytes but not of 16 (the format
    allows any multiple of 4): metadata from seeded sample chunks, the whole
    stream with a ragged last chunk, and the decode, against the oracle."""
    if mode == 1 and cb > 2048:
        pytest.skip("the joint reading is built for chunks of up to 2048 bytes")
    nch = 32 * 7 + 9
    x = W.ibp_gaussian(nch * cb // 4 - 1, std=0.02, seed=cb, device=DEV)  # ragged last chunk
    full = x.numel() * 4 // cb
    idx = W.sample_rows(full, 150, seed=2, device=DEV)
    samples = x[: full * (cb // 4)].view(full, cb // 4)[idx].contiguous()
    ws = _ws(cb, 0, samples.shape[0])
    meta = I.build_meta(samples, cb, T=0.9, mode=mode, ws=ws)
    torch.cuda.synchronize()
    assert I.status(ws) == 0
    mref = O.ibp_build_meta(_u8(samples), cb, T=0.9, mode=mode)
    assert np.array_equal(_u8(meta), mref)
    st, y = _gpu_roundtrip(meta, x, cb)
    ref = O.ibp_encode(mref, _u8(x))
    assert np.array_equal(st.cpu().numpy(), ref)
    assert torch.equal(y.view(torch.int32), x.view(torch.int32))
    # chunks participate: smaller than the stream with every chunk raw
    assert ref.size < O.lib().ora_ibp_stream_bytes_bound(cb, x.numel() * 4)


def test_errors_reported():
    rng = np.random.default_rng(3)
    cb = 512
    meta = O.ibp_make_meta(cb, np.packbits((rng.uniform(size=cb * 8) < 0.2).astype(np.uint8),
                                           bitorder="little"), np.zeros(cb, np.uint8))
    md = torch.from_numpy(meta).to(DEV)
    x = torch.from_numpy(rng.integers(0, 256, size=cb * 40, dtype=np.uint8)).to(DEV)
    st, y = _gpu_roundtrip(md, x, cb)
    n = x.numel()

    def dec(meta_dev, buf, y_bytes=n, in_bytes=None):
        ws = _ws(cb)
        out = torch.zeros(y_bytes, dtype=torch.uint8, device=DEV)
        I.decompress(meta_dev, buf, y_bytes, cb, out=out, ws=ws,
                     in_bytes=buf.numel() if in_bytes is None else in_bytes)
        torch.cuda.synchronize()
        return I.status(ws)

    other = O.ibp_make_meta(cb, np.packbits((rng.uniform(size=cb * 8) < 0.2).astype(np.uint8),
                                            bitorder="little"), np.zeros(cb, np.uint8))
    assert dec(torch.from_numpy(other).to(DEV), st) == abi.ZC_ERR_META_MISMATCH
    assert dec(md, st, y_bytes=n - 4) == abi.ZC_ERR_CAPACITY
    assert dec(md, st, in_bytes=st.numel() - 16) == abi.ZC_ERR_FORMAT
    bad = st.clone()
    bad[136] ^= 0x80  # second group offset
    assert dec(md, bad) == abi.ZC_ERR_FORMAT
    bad = st.clone()
    bad[0] ^= 1
    assert dec(md, bad) == abi.ZC_ERR_FORMAT
    # participation bit set on a chunk that does not match: lengths disagree
    bad = st.clone()
    off_pay = int(st[56:64].cpu().numpy().view(np.uint64)[0])
    bad[off_pay] ^= 0xFF
    assert dec(md, bad) in (abi.ZC_ERR_FORMAT,)
    # compress into a buffer that is too small
    ws = _ws(cb, n)
    small = torch.zeros(300, dtype=torch.uint8, device=DEV)
    I.compress(md, x, cb, out=small, ws=ws)
    torch.cuda.synchronize()
    assert I.status(ws) == abi.ZC_ERR_CAPACITY
    # metadata made for another chunk size
    ws = _ws(1024, n)
    I.compress(md, x, 1024, ws=ws)
    torch.cuda.synchronize()
    assert I.status(ws) == abi.ZC_ERR_META_MISMATCH


@pytest.mark.parametrize("cb", [512, 2048])
def test_host_resident_input_and_streams(cb):
    """Pinned host tensors as encode input, encode output, decode input and
    decode output (read and written in place by the kernels) give the
    oracle's stream and the exact input back; pageable host memory is
    refused."""
    import ctypes as C

    rows = 3000 if cb == 512 else 1500
    x, idx = W.ibp_table(rows=rows, cols=cb // 4, std=0.1, seed=5, device=DEV, n_samples=400)
    x = x.reshape(-1)
    meta = I.build_meta(x.view(-1, cb // 4)[idx].contiguous(), cb, T=0.9, mode=1)
    n = x.numel() * 4
    ref, nb = I.compress(meta, x, cb)
    torch.cuda.synchronize()
    total = int(nb.item())
    ref = ref[:total].clone()
    # the stream every placement must give is the oracle's
    assert np.array_equal(ref.cpu().numpy(), O.ibp_encode(_u8(meta), _u8(x)))
    # host input
    xh = x.cpu().pin_memory()
    st, nb2 = I.compress(meta, xh, cb)
    torch.cuda.synchronize()
    assert int(nb2.item()) == total and torch.equal(st[:total], ref)
    # host output
    oh = torch.full((I.max_compressed_bytes(cb, n),), 0xA5, dtype=torch.uint8, pin_memory=True)
    nb3 = torch.zeros(1, dtype=torch.int64, device=DEV)
    I.compress(meta, x, cb, out=oh, out_bytes=nb3)
    torch.cuda.synchronize()
    assert int(nb3.item()) == total and torch.equal(oh[:total], ref.cpu())
    # host stream in, device out; device stream in, host out
    sh = ref.cpu().pin_memory()
    y = I.decompress(meta, sh, n, cb, in_bytes=total)
    yh = torch.empty(x.numel(), dtype=torch.float32, pin_memory=True)
    I.decompress(meta, ref, n, cb, out=yh, in_bytes=total)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), x.view(torch.int32))
    assert torch.equal(yh.view(torch.int32), x.cpu().view(torch.int32))
    # pageable host memory: refused by the host checks, nothing reaches the GPU
    page = ref.cpu()
    assert not page.is_pinned()
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)
    out = torch.empty(x.numel(), dtype=torch.float32, device=DEV)
    rc = abi.load().ibp_decompress(abi.ptr(meta), cb, C.c_void_p(page.data_ptr()), total,
                                   abi.ptr(out), n, abi.ptr(ws), 256, abi.stream_handle(None))
    assert rc == abi.ZC_ERR_ARG


@pytest.mark.parametrize("cb", [512, 2048])
@pytest.mark.parametrize("mode", [0, 1])
def test_bf16_weights(mode, cb):
    """IBP on 16-bit data: bf16 N(0, 0.02) weights in 512- and 2048-byte
    chunks (256 and 1024 values; keep masks of three runs per word).  The
    codec sees bytes; metadata and stream must equal the oracle's, the round
    trip must be exact, and the sign/exponent bits that the weights share
    make the stream smaller than the input."""
    x16 = W.zc_gaussian((cb // 2) * 1000 + 128, sigma=0.02, seed=21, device=DEV)  # ragged last chunk
    xb = W.bf16_bits(x16).view("uint8")
    x32 = x16.view(torch.int32).view(torch.float32)
    idx = W.sample_rows(x32.numel() * 4 // cb, 600, seed=2, device=DEV)
    samples = x32[: (x32.numel() * 4 // cb) * (cb // 4)].view(-1, cb // 4)[idx].contiguous()
    meta = I.build_meta(samples, cb, T=0.9, mode=mode)
    st, nb = I.compress(meta, x32, cb)
    torch.cuda.synchronize()
    total = int(nb.item())
    m_ref = O.ibp_build_meta(W.f32_bytes(samples), cb, T=0.9, mode=mode)
    assert np.array_equal(meta.cpu().numpy(), m_ref)
    s_ref = O.ibp_encode(m_ref, xb)
    assert np.array_equal(st[:total].cpu().numpy(), s_ref)
    y = I.decompress(meta, st, x32.numel() * 4, cb, in_bytes=total)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), x32.view(torch.int32))
    assert total < xb.size


@pytest.mark.parametrize("mode", [0, 1])
def test_three_launch_encode(mode):
    """The path the single-pass encoders fall back to when their grid cannot
    be resident at once (three launches: match, offsets, pack) gives the
    oracle's stream for the chunk sizes the single-pass encoders take."""
    lib = abi.load()
    rows, idx = W.ibp_table(rows=150_000, cols=128, std=0.1, seed=4, device=DEV, n_samples=3000)
    try:
        lib.zc_test_ibp_single_pass(0)
        for cb, x in ((512, rows.reshape(-1)), (256, rows.reshape(-1)[: 150_000 * 64 - 8]),
                      (64, rows.reshape(-1)[:1_000_000]), (1024, rows.reshape(-1)[:-40]),
                      (2048, rows.reshape(-1)[: 100_000 * 128 + 12])):
            nch = x.numel() * 4 // cb
            sidx = W.sample_rows(nch, 3000, seed=5, device=DEV)
            meta = I.build_meta(x[: nch * (cb // 4)].view(nch, cb // 4)[sidx].contiguous(), cb,
                                T=0.9, mode=mode)
            st, y = _gpu_roundtrip(meta, x, cb)
            assert np.array_equal(st.cpu().numpy(), O.ibp_encode(_u8(meta), _u8(x))), cb
            assert torch.equal(y.view(torch.int32), x.view(torch.int32))
    finally:
        lib.zc_test_ibp_single_pass(1)


def test_encode_next_to_another_stream():
    """The single-pass encoder's blocks wait for lengths that other blocks of
    the same launch publish.  Here its launches share the GPU with ZipCCL
    kernels on a second stream, so some of its blocks start only when those
    finish; every stream must still equal the one encoded alone."""
    from lossless_bit_level_bf16_gb300 import zipccl as Z
    cb = 512
    rows, idx = W.ibp_table(rows=200_000, cols=128, std=0.1, seed=3, device=DEV, n_samples=2000)
    meta = I.build_meta(rows[idx].contiguous(), cb, T=0.9, mode=1, ws=_ws(cb, 0, 2000))
    n_bytes = rows.numel() * 4
    ws0 = _ws(cb, n_bytes)
    ref, nb = I.compress(meta, rows, cb, ws=ws0)
    torch.cuda.synchronize()
    assert I.status(ws0) == 0
    ref = ref[:int(nb.item())].clone()
    x, seg = W.zc_gradient(n_blocks=64, device=DEV)
    plan = Z.Plan(x.numel(), seg, 4096)
    plan.fit(x)
    zref, znb = plan.compress(x)
    torch.cuda.synchronize()
    zref = zref[:int(znb.item())].clone()
    s_ibp, s_zc = torch.cuda.Stream(), torch.cuda.Stream()
    for order in range(4):
        ws = _ws(cb, n_bytes)
        with torch.cuda.stream(s_zc):
            zs = [plan.compress(x) for _ in range(1 + order)]
        with torch.cuda.stream(s_ibp):
            st, nb = I.compress(meta, rows, cb, ws=ws)
        with torch.cuda.stream(s_zc):
            zs.append(plan.compress(x))
        torch.cuda.synchronize()
        assert I.status(ws) == 0, abi.strerror(I.status(ws))
        assert plan.status() == 0
        assert int(nb.item()) == ref.numel() and torch.equal(st[:ref.numel()], ref), order
        for zo, zn in zs:
            assert int(zn.item()) == zref.numel() and torch.equal(zo[:zref.numel()], zref), order
