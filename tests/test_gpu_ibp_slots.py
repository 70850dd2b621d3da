"""GPU parity of the IBP in-place slots (compression into fixed-size host
slots, a device bitmask of compressed slots, a gather that reads only the
stored part of each slot) against the oracle's slot functions.

Page: "Riepilogo Tecnico: Riduzione del Collo di Bottiglia della Memoria GPU
con la Compressione Lossless per il ML", Integrazione del Sistema (PCIe
transfer compression) and Algoritmo Core steps 2-3.
"""
import numpy as np
import pytest
import torch

import oracle as O
from lossless_bit_level_bf16_gb300 import abi, ibp as I, workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _u8(t):
    return t.detach().contiguous().view(torch.uint8).cpu().numpy().reshape(-1)


def _case(cb, rows, mode, seed, tail_words=0):
    x = W.ibp_gaussian(rows * cb // 4 - tail_words, std=0.02, seed=seed, device=DEV)
    nch = x.numel() * 4 // cb
    idx = W.sample_rows(nch, 2000, seed=seed + 1, device=DEV)
    meta = I.build_meta(x[: nch * (cb // 4)].view(nch, cb // 4)[idx].contiguous(), cb, T=0.9,
                        mode=mode)
    return x, meta


def _check_slots(meta, x_h, slots_h, bm_gpu, initial):
    """GPU slots and bitmask against the oracle's, starting from the same
    initial slot bytes (the bytes a compressed slot does not write)."""
    ref_slots, ref_bm = O.ibp_slots_encode(_u8(meta), x_h, slots=initial.copy())
    assert np.array_equal(bm_gpu, ref_bm.view(np.int32))
    assert np.array_equal(slots_h, ref_slots), np.nonzero(slots_h != ref_slots)[0][:8]
    return ref_bm


@pytest.mark.parametrize("cb,mode,tail", [(512, 0, 0), (512, 1, 7), (2048, 0, 0), (2048, 1, 100),
                                          (20, 1, 1), (4096, 0, 3), (64, 1, 0)])
@pytest.mark.parametrize("where", ["host", "in_place_host", "device"])
def test_slots_compress_and_gather(cb, mode, tail, where):
    rows = 3000 if cb <= 512 else 600
    x, meta = _case(cb, rows, mode, seed=cb + mode, tail_words=tail)
    n = x.numel() * 4
    x_h = _u8(x)
    if where == "host":
        src = x
        slots = torch.full((x.numel(),), 7.0, dtype=torch.float32).pin_memory()
        initial = _u8(slots)
    elif where == "in_place_host":
        slots = x.cpu().pin_memory()
        src = slots
        initial = x_h.copy()
    else:
        src = x
        slots = torch.full((x.numel(),), 3.0, dtype=torch.float32, device=DEV)
        initial = _u8(slots)
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)
    slots, bm = I.slots_compress(meta, src, cb, slots=slots, ws=ws)
    torch.cuda.synchronize()
    assert I.status(ws) == 0
    ref_bm = _check_slots(meta, x_h, _u8(slots), bm.cpu().numpy(), initial)
    assert ref_bm.any()  # some chunks are stored compressed
    nch = (n + cb - 1) // cb
    rng = np.random.default_rng(cb + mode)
    idx_h = np.concatenate([rng.integers(0, nch, 777), [nch - 1, 0, nch - 1, 5]]).astype(np.int64)
    idx = torch.from_numpy(idx_h).to(DEV)
    gws = torch.empty(256, dtype=torch.uint8, device=DEV)
    rows_g, rb = I.slots_gather(meta, slots, n, cb, bm, idx, ws=gws, dtype=torch.uint8)
    torch.cuda.synchronize()
    assert I.status(gws) == 0
    ref_rows, ref_read = O.ibp_slots_gather(_u8(meta), _u8(slots), n, ref_bm, idx_h)
    got = rows_g.cpu().numpy().reshape(idx_h.size, cb)
    for i, s in enumerate(idx_h):
        ln = min(cb, n - int(s) * cb)
        assert np.array_equal(got[i, :ln], x_h[int(s) * cb: int(s) * cb + ln]), (i, s)
        assert np.array_equal(got[i, :ln], ref_rows[i, :ln])
    assert int(rb.item()) == ref_read


def test_slots_full_table():
    """The 1,000,000 x 128 fp32 table (joint metadata from its 10,000 sample
    rows) compressed into pinned host slots: every slot and the bitmask equal
    the oracle's; a gather of 100,000 random rows equals the table rows and
    reads fewer bytes than the rows hold."""
    rows, idx = W.ibp_table(device=DEV)
    cb = 512
    meta = I.build_meta(rows[idx].contiguous(), cb, T=0.9, mode=1)
    slots = torch.zeros(rows.numel(), dtype=torch.float32).pin_memory()
    slots, bm = I.slots_compress(meta, rows, cb, slots=slots)
    torch.cuda.synchronize()
    x_h = _u8(rows)
    ref_bm = _check_slots(meta, x_h, _u8(slots), bm.cpu().numpy(), np.zeros(x_h.size, np.uint8))
    g = torch.Generator(device=DEV).manual_seed(5)
    pick = torch.randint(0, rows.shape[0], (100_000,), generator=g, device=DEV)
    got, rb = I.slots_gather(meta, slots, x_h.size, cb, bm, pick)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int32), rows[pick].view(torch.int32))
    comp = np.unpackbits(ref_bm.view(np.uint8), bitorder="little")[pick.cpu().numpy()]
    m = int(_u8(meta)[16:20].view(np.uint32)[0])
    want = int(comp.sum()) * 4 * ((cb * 8 - m + 31) // 32) + int((1 - comp).sum()) * cb
    assert int(rb.item()) == want < 100_000 * cb


def test_slots_errors():
    cb = 512
    x, meta = _case(cb, 200, 1, seed=9)
    n = x.numel() * 4
    slots, bm = I.slots_compress(meta, x, cb, slots=torch.empty_like(x))
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)
    # an index past the last chunk: status ARG, the others still gathered
    idx = torch.tensor([3, n // cb, 1], dtype=torch.int64, device=DEV)
    out, _ = I.slots_gather(meta, slots, n, cb, bm, idx, ws=ws)
    torch.cuda.synchronize()
    assert I.status(ws) == abi.ZC_ERR_ARG
    assert torch.equal(out[0].view(torch.int32), x.view(-1, cb // 4)[3].view(torch.int32))
    # metadata for another chunk size
    ws2 = torch.empty(256, dtype=torch.uint8, device=DEV)
    I.slots_gather(meta, slots, n, 1024, bm, idx[:1], ws=ws2)
    torch.cuda.synchronize()
    assert I.status(ws2) == abi.ZC_ERR_META_MISMATCH
    # input overlapping the slots without being them; pageable host slots
    lib = abi.load()
    rc = lib.ibp_slots_compress(abi.ptr(meta), cb, abi.ptr(x), n - 512, abi.ptr(x[128:]),
                                abi.ptr(bm), abi.ptr(ws), 256, abi.stream_handle(None))
    assert rc == abi.ZC_ERR_ARG
    page = torch.zeros(x.numel(), dtype=torch.float32)
    rc = lib.ibp_slots_compress(abi.ptr(meta), cb, abi.ptr(x), n, abi.ptr(page), abi.ptr(bm),
                                abi.ptr(ws), 256, abi.stream_handle(None))
    assert rc == abi.ZC_ERR_ARG
