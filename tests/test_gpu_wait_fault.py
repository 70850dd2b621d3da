"""The encoders' waits between thread blocks end, and say so, when a state
they wait for never comes.

zc_test_wait_fault (a test-only switch of the C ABI, off by default) makes
one tile of an encode leave out its scan state -- the escape count (ZipCCL)
or stream length (IBP) that later tiles wait for -- and limits each wait to a
few thousand polls.  The call must end with ZC_ERR_TIMEOUT in its status word
(no fault, no hang: the waits give up, every write stays inside the output
buffer), and the next call on the same GPU, with the switch off, must give
the oracle's stream again.  Nothing here makes the GPU fault: the missing
state is a store the kernel leaves out.
"""
import numpy as np
import pytest
import torch

import oracle as O
from lossless_bit_level_bf16_gb300 import abi, ibp as I, workloads as W, zipccl as Z

pytestmark = pytest.mark.gpu
DEV = "cuda"
OFF = 2 ** 64 - 1


@pytest.fixture
def lib():
    L = abi.load()
    L.zc_test_wait_fault(OFF, 0)
    yield L
    L.zc_test_wait_fault(OFF, 0)


def _u8(t):
    return t.detach().contiguous().view(torch.uint8).cpu().numpy().reshape(-1)


@pytest.mark.parametrize("tile", [0, 5, 130])
def test_zipccl_wait_runs_out(lib, tile):
    # 300 tickets of 8192 slots: three look-back blocks of 128 tickets
    x = W.zc_gaussian(300 * 8192 - 11, sigma=0.01, seed=7, device=DEV)
    plan = Z.Plan(x.numel(), None, 4096)
    plan.fit(x)
    lib.zc_test_wait_fault(tile, 2000)
    out, nb = plan.compress(x)
    torch.cuda.synchronize()
    assert plan.status() == abi.ZC_ERR_TIMEOUT
    lib.zc_test_wait_fault(OFF, 0)
    out, nb = plan.compress(x)
    torch.cuda.synchronize()
    assert plan.status() == 0
    st = out[: int(nb.item())].cpu().numpy()
    bk = plan.info()[0]
    ref, _, _, _ = O.zc_encode(W.bf16_bits(x), None, 4096, books=bk.reshape(-1))
    assert np.array_equal(st, ref)


@pytest.mark.parametrize("cb,mb,tile,single", [(512, 3, 7, 1), (512, 3, 0, 1), (2048, 9, 5, 1),
                                               (1024, 130, 0, 0), (4096, 3, 3, 1)])
def test_ibp_wait_runs_out(lib, cb, mb, tile, single):
    """512-byte chunks: the single-pass encoder (tiles of 16 KB); 2048: the
    single-pass encoder in pieces (a group per tile); 1024 with the single
    pass switched off: the offsets pass of the three-launch encode (tiles of
    4096 groups, so 130 MiB gives two); 4096: the group-by-group encoder."""
    x = W.ibp_gaussian(mb * (1 << 20) // 4, std=0.02, seed=3, device=DEV)
    nch = x.numel() * 4 // cb
    idx = W.sample_rows(nch, 2000, seed=1, device=DEV)
    # joint metadata (chunks participate) where it is built, else per-position
    meta = I.build_meta(x.view(nch, cb // 4)[idx].contiguous(), cb, T=0.9,
                        mode=1 if cb <= 2048 else 0)
    n_bytes = x.numel() * 4
    ws = torch.empty(I.workspace_bytes(cb, n_bytes, 0), dtype=torch.uint8, device=DEV)
    lib.zc_test_ibp_single_pass(single)
    try:
        lib.zc_test_wait_fault(tile, 2000)
        I.compress(meta, x, cb, ws=ws)
        torch.cuda.synchronize()
        assert I.status(ws) == abi.ZC_ERR_TIMEOUT
        lib.zc_test_wait_fault(OFF, 0)
    finally:
        lib.zc_test_ibp_single_pass(1)
    st, nb = I.compress(meta, x, cb, ws=ws)
    torch.cuda.synchronize()
    assert I.status(ws) == 0
    got = st[: int(nb.item())].cpu().numpy()
    assert np.array_equal(got, O.ibp_encode(_u8(meta), _u8(x)))
