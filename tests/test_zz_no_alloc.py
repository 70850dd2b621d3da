"""zc_compress_static (the workspace-free ZipCCL encode) against zc_compress.

Collected last on purpose: the entry point's scratch is one array per device
shared by every call, so it is checked after whatever the other tests left
running on the device, and (test_static_in_a_fresh_process) on its own in a
new Python process whose first library call it is.  Each case calls the new
entry point twice in a row, on two different inputs, through the C ABI, and
compares each stream byte for byte (the codec is exact, so the tolerance is
zero) with zc_compress on the same input.
"""
import ctypes as C
import os
import subprocess
import sys

import pytest
import torch

import oracle as O
from lossless_bit_level_bf16_gb300 import abi, workloads as W, zipccl as Z

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _static_call(lib, plan, x, out, out_bytes, status):
    return lib.zc_compress_static(plan._h, abi.ptr(x), abi.ptr(out), out.numel(),
                                  abi.ptr(out_bytes), abi.ptr(status),
                                  abi.stream_handle(None))


@pytest.mark.parametrize("chunk", [1024, 4096])
def test_static_matches_workspace_entry_point_twice(chunk):
    lib = abi.load()
    # two segments with a ragged end, several look-back tiles
    n = 3 * 65536 + 777
    seg = [0, 70001, n]
    xs = [W.zc_gaussian(n, sigma=0.02, seed=11, device=DEV),
          W.zc_gaussian(n, sigma=0.5, seed=12, device=DEV)]
    plan = Z.Plan(n, seg, chunk)
    plan.fit(xs[0])
    cap = plan.max_compressed_bytes
    out = torch.full((cap,), 0xA5, dtype=torch.uint8, device=DEV)
    out_bytes = torch.zeros(1, dtype=torch.int64, device=DEV)
    status = torch.full((1,), 12345, dtype=torch.int32, device=DEV)
    for x in xs:  # two calls in a row share the one scratch array
        ref, ref_nb = plan.compress(x)
        torch.cuda.synchronize()
        assert plan.status() == 0
        rc = _static_call(lib, plan, x, out, out_bytes, status)
        assert rc == abi.ZC_OK, abi.strerror(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        total = int(ref_nb.item())
        assert int(out_bytes.item()) == total
        assert torch.equal(out[:total], ref[:total])
        y = Z.decompress(out, n=n, in_bytes=total)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), x.view(torch.int16))


def test_static_status_reports_capacity():
    lib = abi.load()
    n = 1 << 16
    x = W.zc_gaussian(n, sigma=0.01, seed=3, device=DEV)
    x[::7] = float("inf")  # every 7th element escapes
    plan = Z.Plan(n, None, 4096)
    plan.fit(x)
    # room for the fixed part only (header, tables, slots): the escapes do not fit
    plan_fixed = O.zc_stream_bytes(n, None, 4096, 0)
    out = torch.zeros(plan_fixed, dtype=torch.uint8, device=DEV)
    out_bytes = torch.zeros(1, dtype=torch.int64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert _static_call(lib, plan, x, out, out_bytes, status) == abi.ZC_OK
    torch.cuda.synchronize()
    assert int(status.item()) == abi.ZC_ERR_CAPACITY


def test_static_rejects_plans_beyond_its_scratch():
    lib = abi.load()
    n = 130024 * 8192 + 1  # one slot more than the fixed scratch covers
    x = torch.zeros(16, dtype=torch.bfloat16, device=DEV)  # never read: the call refuses
    out = torch.zeros(1 << 10, dtype=torch.uint8, device=DEV)
    nb = torch.zeros(1, dtype=torch.int64, device=DEV)
    h = C.c_void_p()
    assert lib.zc_plan_create(n, None, 1, 4096, C.byref(h)) == abi.ZC_OK
    try:
        rc = lib.zc_compress_static(h, abi.ptr(x), abi.ptr(out), out.numel(), abi.ptr(nb),
                                    None, abi.stream_handle(None))
        assert rc == abi.ZC_ERR_CAPACITY
    finally:
        lib.zc_plan_destroy(h)


def test_static_in_a_fresh_process():
    """The two-input comparison again, in a new process where the first call
    into the library is zc_compress_static (so its address lookup is the
    process's first use of the array)."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = """
import torch
from lossless_bit_level_bf16_gb300 import abi, workloads as W, zipccl as Z
lib = abi.load()
n = 2 * 65536 + 333
xs = [W.zc_gaussian(n, sigma=0.02, seed=21, device="cuda"),
      W.zc_gaussian(n, sigma=0.3, seed=22, device="cuda")]
plan = Z.Plan(n, None, 4096)
plan.set_books([116, 117, 118, 119, 120, 121, 122])
out = torch.zeros(plan.max_compressed_bytes, dtype=torch.uint8, device="cuda")
nb = torch.zeros(1, dtype=torch.int64, device="cuda")
status = torch.full((1,), 777, dtype=torch.int32, device="cuda")
for x in xs:
    rc = lib.zc_compress_static(plan._h, abi.ptr(x), abi.ptr(out), out.numel(), abi.ptr(nb),
                                abi.ptr(status), abi.stream_handle(None))
    assert rc == abi.ZC_OK, rc
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out[: int(nb.item())].clone()
    ref, ref_nb = plan.compress(x)
    torch.cuda.synchronize()
    assert plan.status() == 0 and int(ref_nb.item()) == got.numel()
    assert torch.equal(got, ref[: got.numel()])
print("fresh-process-ok")
"""
    env = dict(os.environ)
    env["PYTHONPATH"] = root + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "fresh-process-ok" in r.stdout, r.stdout + r.stderr
