"""Benchmark of the codec hot path on GB300: one JSON line on stdout.

A step is one pass of every row of the hot path over one batch of synthetic
input:
  ZipCCL on the gradient-like bf16 buffer (64M elements, 256 layer blocks,
  chunk 4096): zc_plan (statistics + codebooks) -> zc_compress -> zc_decompress;
  IBP on the fp32 embedding table (1,000,000 x 128, one row per chunk, T = 0.9,
  metadata from 10,000 seeded rows): ibp_build_meta -> ibp_compress ->
  ibp_decompress.
value = uncompressed bytes of both inputs / device time of the step (GB/s).
Every op is bracketed by CUDA events on the stream it is launched on; L2 is
flushed (a 512 MB buffer written) before every step, outside the timed
events.  `e2e` repeats the step through host memory: pinned host inputs are
copied in and the compressed streams copied out inside the timed region, the
ZipCCL and IBP chains on two streams so that copies overlap kernels.

--impl reference times the bit-serial CPU oracle (the checker) on all host
cores (independent oracle calls on disjoint pieces) over a bounded sample of
the same workload; the GPU line's cpu_baseline carries that figure and the
single-thread one.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "encode/decode GB/s (uncompressed) and % of HBM roofline; compression ratio"
WORKLOAD = ("zipccl gradient-like bf16 64M (256 blocks, chunk 4096) + "
            "ibp fp32 table 1,000,000x128 (chunk 512 B, T=0.9, 10,000 samples)")

# Algorithmic bytes per launch are computed from the actual stream sizes.


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def csrc_hash():
    """sha1 (12 hex digits) over every file of the CUDA sources: a committed
    traffic figure is used only while the kernels are the ones it measured."""
    import glob
    import hashlib
    h = hashlib.sha1()
    for path in sorted(glob.glob(os.path.join(ROOT, "lossless_bit_level_bf16_gb300", "csrc", "*"))):
        h.update(os.path.basename(path).encode())
        h.update(open(path, "rb").read())
    return h.hexdigest()[:12]


def kernel_hash(kernel):
    """sha1 (12 hex digits) over the CUDA source file that defines `kernel`
    and every header the sources share (csrc/*.cuh, csrc/*.h, include/zc.h):
    a committed traffic figure is used only while the kernel's own sources
    are the ones it measured (an edit to another kernel's file leaves it
    valid)."""
    import glob
    import hashlib
    import re
    csrc = os.path.join(ROOT, "lossless_bit_level_bf16_gb300", "csrc")
    pat = re.compile(r"__global__[^;{]*?\b" + re.escape(kernel) + r"\s*\(", re.S)
    tus = [p for p in sorted(glob.glob(os.path.join(csrc, "*.cu"))) if pat.search(open(p).read())]
    if len(tus) != 1:
        raise KeyError(f"{kernel}: defined in {len(tus)} source files")
    heads = sorted(glob.glob(os.path.join(csrc, "*.cuh")) + glob.glob(os.path.join(csrc, "*.h")))
    heads.append(os.path.join(ROOT, "include", "zc.h"))
    h = hashlib.sha1()
    for path in tus + heads:
        h.update(os.path.basename(path).encode())
        h.update(open(path, "rb").read())
    return h.hexdigest()[:12]


def _traffic_table():
    """Measured DRAM traffic per launch from the committed ncu summaries, as
    {kernel: {sha1: [(bytes per launch, uncompressed bytes, case), ...]}}.
    Lines in profiles/*.md read 'traffic <kernel> <kernel_hash> <bytes>
    <uncompressed bytes of the captured launch> <case>', the case naming the
    data and chunking the capture ran on (a kernel may have lines from several
    captures)."""
    import glob
    out = {}
    for f in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for line in open(f):
            parts = line.strip().strip("`").split()
            if len(parts) == 6 and parts[0] == "traffic" and parts[3].isdigit() \
                    and parts[4].isdigit():
                out.setdefault(parts[1], {}).setdefault(parts[2], []).append(
                    (int(parts[3]), int(parts[4]), parts[5]))
    return out


def measured_traffic(kernel, case, unc, table=None, sha=None):
    """The kernel's DRAM bytes for a launch over `unc` uncompressed bytes of
    `case`, from a capture on the current sources: the captured figure, scaled
    by unc / captured bytes when the sizes differ (traffic grows in proportion
    with the input for these streaming kernels at a fixed data distribution
    and chunking).  Returns (bytes, captured uncompressed bytes), or
    (None, None) when no capture of that case matches the sources."""
    table = _traffic_table() if table is None else table
    sha = kernel_hash(kernel) if sha is None else sha
    for nbytes, cap, c in table.get(kernel, {}).get(sha, []):
        if c == case:
            return (nbytes if cap == unc else round(nbytes * unc / cap)), cap
    return None, None


class ClockSampler:
    """nvidia-smi samples (every 20 ms) while the timed region runs.  The GPU is
    named by its UUID (CUDA ordinals and nvidia-smi indices can differ); the
    sampler's first line, taken before the timed region, is dropped."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.gid = str(device_index)
        try:
            import torch
            u = getattr(torch.cuda.get_device_properties(device_index), "uuid", None)
            if u is not None:
                u = str(u)
                self.gid = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
        self.p = None

    def __enter__(self):
        import select
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gid}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            # wait (at most 5 s) for the first sample, so sampling covers the
            # whole timed region; that sample is taken before it and dropped
            r, _, _ = select.select([self.p.stdout], [], [], 5.0)
            if r:
                self.p.stdout.readline()
        except (OSError, ValueError):
            self.p = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.p is not None:
            self.p.terminate()
            try:
                out, _ = self.p.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
                out, _ = self.p.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


class NvmlSampler:
    """Clock and throttle-reason samples taken through NVML (the driver's
    libnvidia-ml, read-only queries) every millisecond by a background
    thread, so that even a timed region of a few milliseconds has samples.
    Falls back to ClockSampler (nvidia-smi, 20 ms) when NVML is missing."""

    HW_SLOWDOWN, SW_POWER_CAP, SW_THERMAL, HW_THERMAL = 0x8, 0x4, 0x20, 0x40

    def __init__(self, device_index, period_s=0.001):
        self.index = device_index
        self.period = period_s
        self.fallback = None
        self.samples = []
        self.max_mhz = None

    def _open(self):
        import ctypes as C
        import torch
        lib = C.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        u = str(getattr(torch.cuda.get_device_properties(self.index), "uuid", ""))
        u = u if u.startswith("GPU-") else "GPU-" + u
        h = C.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(u.encode(), C.byref(h)) != 0:
            raise OSError("no NVML handle for " + u)
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = C.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, C.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        return lib, h, reasons

    def __enter__(self):
        import threading
        try:
            lib, h, reasons = self._open()
        except (OSError, AttributeError):
            self.fallback = ClockSampler(self.index).__enter__()
            return self
        import ctypes as C
        self._stop = threading.Event()

        def run():
            clk, r = C.c_uint(), C.c_ulonglong()
            while not self._stop.is_set():
                if lib.nvmlDeviceGetClockInfo(h, 1, C.byref(clk)) == 0 and \
                        reasons(h, C.byref(r)) == 0:
                    self.samples.append((float(clk.value), int(r.value)))
                time.sleep(self.period)
        self._lib = lib
        self._t = threading.Thread(target=run, daemon=True)
        self._t.start()
        time.sleep(0.005)  # the thread is sampling before the region starts
        self.samples.clear()
        return self

    def __exit__(self, *a):
        if self.fallback is not None:
            return self.fallback.__exit__(*a)
        self._stop.set()
        self._t.join()

    def summary(self):
        if self.fallback is not None:
            d = self.fallback.summary()
            d["source"] = "nvidia-smi"
            return d
        mhz = [c for c, _ in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        names = [(self.HW_SLOWDOWN, "hw_slowdown"), (self.HW_THERMAL, "hw_thermal_slowdown"),
                 (self.SW_THERMAL, "sw_thermal_slowdown"), (self.SW_POWER_CAP, "sw_power_cap")]
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in names if bits & b), "samples": len(mhz),
                "source": "nvml, 1 ms"}


def reduce_max(x: float) -> float:
    """Maximum of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(ms_local: float, bytes_per_rank: int, world: int):
    """Replicas: every rank runs the whole workload on its own GPU; the job's
    time is the slowest rank's, its throughput all ranks' bytes over that
    time.  Returns (ms_max, GB/s)."""
    ms = reduce_max(ms_local)
    return ms, bytes_per_rank * world / (ms * 1e-3) / 1e9


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------- GPU arm

class Workload:
    def __init__(self, device, scale=1.0):
        import torch

        from lossless_bit_level_bf16_gb300 import ibp as I, workloads as W, zipccl as Z
        self.torch, self.I, self.Z = torch, I, Z
        self.dev = device
        nblk = max(1, int(256 * scale))
        self.x, self.seg = W.zc_gradient(n_blocks=nblk, device=device)
        self.n = self.x.numel()
        self.plan = Z.Plan(self.n, self.seg, 4096, device=device)
        self.zout = torch.empty(self.plan.max_compressed_bytes, dtype=torch.uint8, device=device)
        self.znb = torch.zeros(1, dtype=torch.int64, device=device)
        self.zy = torch.empty_like(self.x)
        self.zdws = torch.empty(256, dtype=torch.uint8, device=device)
        rows = max(1000, int(1_000_000 * scale))
        self.table, idx = W.ibp_table(rows=rows, device=device)
        self.samples = self.table[idx].contiguous()
        self.cb = 512
        self.tbytes = self.table.numel() * 4
        self.meta = torch.empty(64 + 2 * self.cb,
                                dtype=torch.uint8, device=device)
        self.mws = torch.empty(I.workspace_bytes(self.cb, 0, self.samples.shape[0]),
                               dtype=torch.uint8, device=device)
        self.iws = torch.empty(I.workspace_bytes(self.cb, self.tbytes, 0), dtype=torch.uint8,
                               device=device)
        self.iout = torch.empty(I.max_compressed_bytes(self.cb, self.tbytes), dtype=torch.uint8,
                                device=device)
        self.inb = torch.zeros(1, dtype=torch.int64, device=device)
        self.iy = torch.empty_like(self.table)
        self.idws = torch.empty(256, dtype=torch.uint8, device=device)
        self.mode = 0
        self.unc_bytes = 2 * self.n + self.tbytes
        # kernels each op launches (cudaMemsetAsync of a control block aside)
        self.kernels = {op: kernels_of(op, self.cb) for op in
                        ("zc_plan", "zc_compress", "zc_decompress", "ibp_build_meta",
                         "ibp_compress", "ibp_decompress")}
        self.launches_per_step = sum(len(v) for v in self.kernels.values())
        # the data each op runs on, as named in the traffic lines of the profiles
        self.case = {op: ("zc_gradient_c4096" if op.startswith("zc") else
                          f"ibp_table_{self.cb}B_mode{self.mode}")
                     for op in self.kernels}

    def ops(self):
        I, Z = self.I, self.Z
        return [
            ("zc_plan", lambda: self.plan.fit(self.x)),
            ("zc_compress", lambda: self.plan.compress(self.x, out=self.zout, out_bytes=self.znb)),
            ("zc_decompress", lambda: Z.decompress(self.zout, out=self.zy, in_bytes=self.zout.numel(),
                                                   ws=self.zdws)),
            ("ibp_build_meta", lambda: I.build_meta(self.samples, self.cb, T=0.9, mode=self.mode,
                                                    meta=self.meta, ws=self.mws)),
            ("ibp_compress", lambda: I.compress(self.meta, self.table, self.cb, out=self.iout,
                                                out_bytes=self.inb, ws=self.iws)),
            ("ibp_decompress", lambda: I.decompress(self.meta, self.iout, self.tbytes, self.cb,
                                                    out=self.iy, in_bytes=self.iout.numel(),
                                                    ws=self.idws)),
        ]

    def check(self):
        from lossless_bit_level_bf16_gb300 import abi
        torch = self.torch
        torch.cuda.synchronize()
        for ws in (self.plan.ws, self.zdws, self.mws, self.iws, self.idws):
            s = abi.status(ws)
            if s != 0:
                raise RuntimeError(f"device status {s}: {abi.strerror(s)}")
        assert torch.equal(self.zy.view(torch.int16), self.x.view(torch.int16))
        assert torch.equal(self.iy.view(torch.int32), self.table.view(torch.int32))

    def sizes(self):
        return int(self.znb.item()), int(self.inb.item())


def gpu_arm(args, rank, world, local_rank):
    import torch
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = Workload(dev, args.scale)
    ops = wl.ops()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(timed):
        flush.add_(1)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)]
        evs[0].record(stream)
        for i, (_, fn) in enumerate(ops):
            fn()
            evs[i + 1].record(stream)
        return evs

    for _ in range(args.warmup):
        step(False)
    wl.check()
    zsz, isz = wl.sizes()
    barrier()
    torch.cuda.synchronize()
    all_evs = []
    with NvmlSampler(local_rank) as clk:
        t0 = time.perf_counter()
        for _ in range(args.steps):
            all_evs.append(step(True))
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    barrier()
    # the same step repeated for at least a second, with its own clock record
    # (reported beside the K-step figure, which it does not replace)
    sus_evs = []
    with NvmlSampler(local_rank) as sclk:
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < args.sustain_s or len(sus_evs) < 3:
            sus_evs.append(step(True))
            if len(sus_evs) % 64 == 0:
                sus_evs[-1][-1].synchronize()
        torch.cuda.synchronize()
        sus_wall = time.perf_counter() - t0
    sus_ms = statistics.mean(e[0].elapsed_time(e[-1]) for e in sus_evs)
    sustained = {"steps": len(sus_evs), "wall_s": round(sus_wall, 3), "ms_per_step": round(sus_ms, 4),
                 "clocks": sclk.summary()}
    if sustained["clocks"].get("sm_mhz"):
        sustained["ms_x_mhz"] = round(sus_ms * sustained["clocks"]["sm_mhz"], 1)
    per_op = {name: [] for name, _ in ops}
    steps_ms = []
    for evs in all_evs:
        steps_ms.append(evs[0].elapsed_time(evs[-1]))
        for i, (name, _) in enumerate(ops):
            per_op[name].append(evs[i].elapsed_time(evs[i + 1]))
    ms = statistics.mean(steps_ms)
    ms_max, _ = aggregate(ms, wl.unc_bytes, world)
    wl.check()

    # ---- end to end through host memory (pinned inputs in, streams out)
    hx = torch.empty(wl.x.shape, dtype=wl.x.dtype, pin_memory=True)
    hx.copy_(wl.x)
    ht = torch.empty(wl.table.shape, dtype=wl.table.dtype, pin_memory=True)
    ht.copy_(wl.table)
    hs = torch.empty(wl.samples.shape, dtype=wl.samples.dtype, pin_memory=True)
    hs.copy_(wl.samples)
    hz = torch.empty(zsz, dtype=torch.uint8, pin_memory=True)
    hi = torch.empty(isz, dtype=torch.uint8, pin_memory=True)
    h_status = torch.empty(5 * 4, dtype=torch.uint8, pin_memory=True)
    # The two codecs' chains (copy in, plan/meta, encode, decode, copy out)
    # run on two streams, so one codec's copies overlap the other's kernels.
    # The table goes over the host-to-device link first (the IBP chain is the
    # longer one), the ZipCCL input after it; each codec's stream goes back
    # on a stream of its own as soon as it is encoded, while it is decoded.
    zs, ist, zos, ios = (torch.cuda.Stream() for _ in range(4))
    zops, iops = dict(ops[:3]), dict(ops[3:])
    e2e_ms = []
    for it in range(args.warmup + args.steps):
        flush.add_(1)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        t_in, z_enc, i_enc = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
        a.record(stream)
        ist.wait_event(a)
        with torch.cuda.stream(ist):
            wl.table.copy_(ht, non_blocking=True)
            wl.samples.copy_(hs, non_blocking=True)
            t_in.record(ist)
            iops["ibp_build_meta"]()
            iops["ibp_compress"]()
            i_enc.record(ist)
            iops["ibp_decompress"]()
            for j, ws in enumerate((wl.mws, wl.iws, wl.idws)):
                h_status[8 + 4 * j:12 + 4 * j].copy_(ws[:4], non_blocking=True)
        ios.wait_event(i_enc)
        with torch.cuda.stream(ios):
            hi.copy_(wl.iout[:isz], non_blocking=True)
        zs.wait_event(t_in)
        with torch.cuda.stream(zs):
            wl.x.copy_(hx, non_blocking=True)
            zops["zc_plan"]()
            zops["zc_compress"]()
            z_enc.record(zs)
            zops["zc_decompress"]()
            for j, ws in enumerate((wl.plan.ws, wl.zdws)):
                h_status[4 * j:4 * j + 4].copy_(ws[:4], non_blocking=True)
        zos.wait_event(z_enc)
        with torch.cuda.stream(zos):
            hz.copy_(wl.zout[:zsz], non_blocking=True)
        for st_ in (zs, ist, zos, ios):
            stream.wait_stream(st_)
        b.record(stream)
        b.synchronize()
        if it >= args.warmup:
            e2e_ms.append(a.elapsed_time(b))
    torch.cuda.synchronize()
    wl.check()
    e2e = statistics.mean(e2e_ms)
    e2e_max = reduce_max(e2e)
    h2d = hx.numel() * 2 + ht.numel() * 4 + hs.numel() * 4
    d2h = zsz + isz + 20
    targets = target_ops(args, dev, flush, stream) if args.targets else {}
    return dict(wl=wl, per_op=per_op, ms=ms_max, ms_local=ms, wall=wall, clocks=clk.summary(),
                e2e_ms=e2e_max, h2d=h2d, d2h=d2h, zsz=zsz, isz=isz, sustained=sustained,
                targets=targets)


def case_of(kind, cb, mode):
    """The traffic lines' name for a size-sweep workload: ZipCCL on bf16
    N(0, 0.01), chunk 4096; IBP on fp32 N(0, 0.02) in cb-byte chunks and
    metadata mode `mode`."""
    return "zc_gauss0.01_c4096" if kind == "zipccl" else f"ibp_gauss0.02_{cb}B_mode{mode}"


# kernels each op launches, by codec and IBP chunk size
def kernels_of(op, cb=512):
    return {"zc_plan": ["zc_stats_kernel", "zc_predict_kernel"],
            "zc_compress": ["zc_encode_kernel"],
            "zc_compress_fit": ["zc_encode_kernel", "zc_predict_kernel"],
            "zc_decompress": ["zc_decode_kernel"],
            "ibp_build_meta": ["ibp_columns_kernel", "ibp_meta_kernel"],
            "ibp_compress": (["ibp_encode_ws_kernel"] if cb <= 512 else
                             ["ibp_encode_wsp_kernel"] if cb in (1024, 2048) else
                             ["ibp_match_kernel", "ibp_offsets_kernel", "ibp_pack_kernel"]),
            "ibp_decompress": ["ibp_decode_pipe_kernel"]}[op]


TARGETS = [("zipccl", 1 << 30, 0, "zipccl bf16 N(0,0.01) 1 GiB, chunk 4096"),
           ("ibp", 1 << 30, 0, "ibp fp32 N(0,0.02) 1 GiB, 2048-B chunks, per-position"),
           ("ibp", 1 << 30, 1, "ibp fp32 N(0,0.02) 1 GiB, 2048-B chunks, joint")]


def target_ops(args, dev, flush, stream):
    """The workload list's >= 256 MB points where the roofline target applies,
    timed op by op after the step (median of CUDA-event times, L2 flushed
    before every launch): ZipCCL on the 1 GiB bf16 sweep point and IBP on the
    1 GiB fp32 sweep point (2048-byte chunks, where chunks participate), in
    both metadata modes.  Returns ops entries, each with its roofline."""
    import torch

    from lossless_bit_level_bf16_gb300 import abi
    peak, peak_kind = _peaks()
    out = {}
    steps = max(5, min(args.steps, 20))
    for kind, nbytes, mode, label in TARGETS:
        ops, wss, unc, sbytes, check, nb, cb = _case(kind, nbytes, dev, mode)
        ms = _time_ops(ops, flush, stream, 3, steps)
        for ws in wss:
            st = abi.status(ws)
            if st != 0:
                raise RuntimeError(f"{label}: device status {st}: {abi.strerror(st)}")
        if not check():
            raise RuntimeError(f"{label}: round trip differs")
        comp = int(nb.item())
        for name, t in ms.items():
            if name == "ibp_build_meta":
                continue  # 20 MB of samples: not a >= 256 MB op
            alg = unc if name == "zc_plan" else unc + comp
            ach = alg / (t * 1e-3) / 1e9
            ks = kernels_of(name, cb)
            traffic, cap = measured_traffic(ks[0], case_of(kind, cb, mode), unc) \
                if len(ks) == 1 else (None, None)
            out[f"{name} [{label}]"] = {
                "ms": round(t, 4), "GBps_uncompressed": round(unc / (t * 1e-3) / 1e9, 1),
                "ratio": round(unc / comp, 4), "kernels": ks, "launches_timed": steps,
                "roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": peak,
                             "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s",
                             "frac": round(ach / peak, 4), "algorithmic_bytes_per_launch": alg,
                             "traffic": traffic, "traffic_capture_bytes": cap}}
        del ops, wss, check, nb
        torch.cuda.empty_cache()
    return out


def report_gpu(args, r, world):
    wl = r["wl"]
    peak, peak_kind = _peaks()
    n = wl.n
    unc_total = wl.unc_bytes * world
    value = unc_total / (r["ms"] * 1e-3) / 1e9
    zsz, isz = r["zsz"], r["isz"]
    # algorithmic bytes per launch (read + written)
    nsamp = wl.samples.numel() * 4
    alg = {
        "zc_plan": 2 * n,
        "zc_compress": 2 * n + zsz,
        "zc_decompress": zsz + 2 * n,
        "ibp_build_meta": nsamp,
        "ibp_compress": wl.tbytes + isz,
        "ibp_decompress": isz + wl.tbytes,
    }
    unc = {"zc_plan": 2 * n, "zc_compress": 2 * n, "zc_decompress": 2 * n,
           "ibp_build_meta": nsamp, "ibp_compress": wl.tbytes, "ibp_decompress": wl.tbytes}
    ops = {}
    for name, ts in r["per_op"].items():
        t = statistics.mean(ts)
        ach = alg[name] / (t * 1e-3) / 1e9
        ops[name] = {"ms": round(t, 4), "GBps_uncompressed": round(unc[name] / (t * 1e-3) / 1e9, 1),
                     "GBps_traffic": round(ach, 1), "frac_hbm": round(ach / peak, 4),
                     "kernels": wl.kernels[name]}
    # the dominant kernel: the longest op that is a single kernel (ops of
    # several kernels are timed as a whole and listed under "ops")
    single = [k for k in r["per_op"] if len(wl.kernels[k]) == 1]
    dom = max(single, key=lambda k: statistics.mean(r["per_op"][k]))
    t_dom = statistics.mean(r["per_op"][dom])
    kname = wl.kernels[dom][0]
    traffic, cap = measured_traffic(kname, wl.case[dom], unc[dom])
    achieved = alg[dom] / (t_dom * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(r["ms"], 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u8",
        "data": "synthetic (seeded generators: gradient-like bf16 blocks, N(0,0.1) fp32 table)",
        "config": {"workload": WORKLOAD, "zc_elements": n, "zc_segments": len(wl.seg) - 1,
                   "zc_chunk": 4096, "ibp_rows": wl.table.shape[0], "ibp_chunk_bytes": wl.cb,
                   "ibp_T": 0.9, "ibp_mode": "per-position", "ibp_samples": wl.samples.shape[0],
                   "l2": "flushed before every step (512 MB write)",
                   "parallelism": f"replicas x{world}"},
        "ratio": {"zipccl": round(2 * n / zsz, 4), "ibp": round(wl.tbytes / isz, 4)},
        "ops": ops,
        "roofline": {"bound": "hbm", "kernel": kname, "op": dom, "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "algorithmic_bytes_per_launch": alg[dom], "traffic": traffic,
                     "traffic_capture_bytes": cap},
        "e2e": {"value": round(unc_total / (r["e2e_ms"] * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": wl.launches_per_step * args.steps,
        "clocks": r["clocks"],
        "sustained": r["sustained"],
    }
    if r["clocks"].get("sm_mhz"):
        line["clocks"]["ms_x_mhz"] = round(r["ms"] * r["clocks"]["sm_mhz"], 1)
    for name, d in r["targets"].items():
        ops[name] = d
    if args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return line


# ---------------------------------------------------------------- size sweep

SWEEP_OPS = {"zipccl": ("zc_plan", "zc_compress", "zc_decompress"),
             "ibp": ("ibp_build_meta", "ibp_compress", "ibp_decompress")}


def _time_ops(ops, flush, stream, warmup, steps):
    """Median CUDA-event time (ms) of each op over `steps` launches after
    `warmup` untimed ones; L2 is flushed before every launch."""
    import torch
    per = {name: [] for name, _ in ops}
    for it in range(warmup + steps):
        for name, fn in ops:
            flush.add_(1)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            if it >= warmup:
                per[name].append((a, b))
    torch.cuda.synchronize()
    return {name: statistics.median(a.elapsed_time(b) for a, b in v) for name, v in per.items()}


def _case(kind, nbytes, dev, ibp_mode):
    """One codec workload on the device: (ops, workspaces, uncompressed bytes,
    bytes of the metadata samples, round-trip check, output-size tensor, chunk)."""
    import torch

    from lossless_bit_level_bf16_gb300 import ibp as I, workloads as W, zipccl as Z
    if kind in ("zipccl", "gradient", "moe"):
        if kind == "zipccl":
            n = nbytes // 2
            x, seg = W.zc_gaussian(n, sigma=0.01, seed=0, device=dev), None
        elif kind == "gradient":
            x, seg = W.zc_gradient(device=dev)
        else:
            x, seg, _ = W.zc_moe(device=dev)
        n = x.numel()
        plan = Z.Plan(n, seg, 4096, device=dev)
        out = torch.empty(plan.max_compressed_bytes, dtype=torch.uint8, device=dev)
        nb = torch.zeros(1, dtype=torch.int64, device=dev)
        y = torch.empty_like(x)
        dws = torch.zeros(256, dtype=torch.uint8, device=dev)
        ops = [("zc_plan", lambda: plan.fit(x)),
               ("zc_compress", lambda: plan.compress(x, out=out, out_bytes=nb)),
               ("zc_decompress", lambda: Z.decompress(out, out=y, in_bytes=out.numel(), ws=dws)),
               # plan and encode from one read (the codebooks refit for the next call)
               ("zc_compress_fit", lambda: plan.compress_fit(x, out=out, out_bytes=nb))]
        check = lambda: torch.equal(y.view(torch.int16), x.view(torch.int16))  # noqa: E731
        return ops, (plan.ws, dws), 2 * n, 0, check, nb, 4096
    if kind == "ibp16":
        # 16-bit weights: bf16 N(0, 0.02), 512-byte chunks (256 values); the
        # codec sees bytes, so the tensor is handled as 32-bit words
        cb = 512
        x16 = W.zc_gaussian(nbytes // 2, sigma=0.02, seed=0, device=dev)
        x = x16.view(torch.int32).view(torch.float32)
        n = x.numel()
        idx = W.sample_rows(4 * n // cb, 10_000, seed=1, device=dev)
        samples = x.view(-1, cb // 4)[idx].contiguous()
    elif kind == "ibp":
        cb = 2048
        n = nbytes // 4
        x = W.ibp_gaussian(n, std=0.02, seed=0, device=dev)
        idx = W.sample_rows(4 * n // cb, 10_000, seed=1, device=dev)
        samples = x.view(-1, cb // 4)[idx].contiguous()
    else:  # the embedding table, one 128-value row per chunk
        cb = 512
        x, idx = W.ibp_table(device=dev)
        samples = x[idx].contiguous()
        x = x.view(-1)
        n = x.numel()
    if kind == "table_host":
        # the table and its stream stay in pinned host memory: the kernels read
        # them in place over the host link (the output of each op is on the GPU)
        xd = x
        xh = xd.cpu().pin_memory()
        meta = I.build_meta(samples, cb, T=0.9, mode=ibp_mode)
        st, stn = I.compress(meta, xd, cb)
        torch.cuda.synchronize()
        sh = st[: int(stn.item())].cpu().pin_memory()
        mws = torch.zeros(I.workspace_bytes(cb, 0, samples.shape[0]), dtype=torch.uint8, device=dev)
        iws = torch.zeros(I.workspace_bytes(cb, 4 * n, 0), dtype=torch.uint8, device=dev)
        out = torch.empty(I.max_compressed_bytes(cb, 4 * n), dtype=torch.uint8, device=dev)
        nb = torch.zeros(1, dtype=torch.int64, device=dev)
        y = torch.empty_like(xd)
        dws = torch.zeros(256, dtype=torch.uint8, device=dev)
        ops = [("ibp_build_meta", lambda: I.build_meta(samples, cb, T=0.9, mode=ibp_mode,
                                                       meta=meta, ws=mws)),
               ("ibp_compress", lambda: I.compress(meta, xh, cb, out=out, out_bytes=nb, ws=iws)),
               ("ibp_decompress", lambda: I.decompress(meta, sh, 4 * n, cb, out=y,
                                                       in_bytes=sh.numel(), ws=dws))]
        check = lambda: torch.equal(y.view(torch.int32), xd.view(torch.int32)) and torch.equal(  # noqa: E731
            out[: sh.numel()].cpu(), sh)
        return ops, (mws, iws, dws), 4 * n, samples.shape[0] * cb, check, nb, cb
    ns = samples.shape[0]
    meta = torch.empty(64 + 2 * cb, dtype=torch.uint8, device=dev)
    mws = torch.zeros(I.workspace_bytes(cb, 0, ns), dtype=torch.uint8, device=dev)
    iws = torch.zeros(I.workspace_bytes(cb, 4 * n, 0), dtype=torch.uint8, device=dev)
    out = torch.empty(I.max_compressed_bytes(cb, 4 * n), dtype=torch.uint8, device=dev)
    nb = torch.zeros(1, dtype=torch.int64, device=dev)
    y = torch.empty_like(x)
    dws = torch.zeros(256, dtype=torch.uint8, device=dev)
    ops = [("ibp_build_meta", lambda: I.build_meta(samples, cb, T=0.9, mode=ibp_mode, meta=meta,
                                                   ws=mws)),
           ("ibp_compress", lambda: I.compress(meta, x, cb, out=out, out_bytes=nb, ws=iws)),
           ("ibp_decompress", lambda: I.decompress(meta, out, 4 * n, cb, out=y, in_bytes=out.numel(),
                                                   ws=dws))]
    check = lambda: torch.equal(y.view(torch.int32), x.view(torch.int32))  # noqa: E731
    return ops, (mws, iws, dws), 4 * n, ns * cb, check, nb, cb


def slots_arm(args):
    """IBP in-place slots on the 1,000,000 x 128 table (joint metadata, where
    most rows are stored compressed): ibp_slots_compress from the device
    table into pinned host slots, and ibp_slots_gather of 100,000 random rows
    from them.  Beside it, the host link measured in the same run: the copy
    engine (a pinned -> device copy of the whole table) and the same gather
    kernel on raw slots (metadata without invariant bits: every slot a plain
    row copy over the link).  GB/s of uncompressed bytes delivered; link GB/s
    = bytes read from host memory / time."""
    import torch

    from lossless_bit_level_bf16_gb300 import abi, ibp as I, workloads as W
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    cb = 512
    rows, idx = W.ibp_table(device=dev)
    n = rows.numel() * 4
    meta = I.build_meta(rows[idx].contiguous(), cb, T=0.9, mode=args.ibp_mode)
    rnd = torch.randint(-2**31, 2**31 - 1, (10_000, cb // 4), dtype=torch.int32, device=dev)
    meta_raw = I.build_meta(rnd, cb, T=1.0, mode=0)  # no position is invariant: m = 0
    slots = torch.empty(rows.numel(), dtype=torch.float32).pin_memory()
    slots_raw = torch.empty(rows.numel(), dtype=torch.float32).pin_memory()
    bm = torch.zeros((n // cb + 31) // 32, dtype=torch.int32, device=dev)
    bm_raw = torch.zeros_like(bm)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    gws = torch.zeros(256, dtype=torch.uint8, device=dev)
    K = 100_000
    g = torch.Generator(device=dev).manual_seed(7)
    pick = torch.randint(0, rows.shape[0], (K,), generator=g, device=dev)
    out = torch.empty(K, cb // 4, dtype=torch.float32, device=dev)
    rb = torch.zeros(1, dtype=torch.int64, device=dev)
    rb_raw = torch.zeros(1, dtype=torch.int64, device=dev)
    I.slots_compress(meta_raw, rows, cb, slots=slots_raw, bitmask=bm_raw, ws=ws)
    dtab = torch.empty(rows.numel(), dtype=torch.float32, device=dev)
    ops = [("ibp_slots_compress", lambda: I.slots_compress(meta, rows, cb, slots=slots, bitmask=bm,
                                                           ws=ws)),
           ("ibp_slots_gather", lambda: I.slots_gather(meta, slots, n, cb, bm, pick, out=out,
                                                       read_bytes=rb, ws=gws)),
           ("gather_raw_slots", lambda: I.slots_gather(meta_raw, slots_raw, n, cb, bm_raw, pick,
                                                       out=out, read_bytes=rb_raw, ws=gws)),
           ("dma_copy_table", lambda: dtab.copy_(slots_raw, non_blocking=True))]
    ms = _time_ops(ops, flush, stream, max(3, args.warmup), args.steps)
    for w in (ws, gws):
        st = abi.status(w)
        if st != 0:
            raise RuntimeError(f"device status {st}: {abi.strerror(st)}")
    I.slots_gather(meta, slots, n, cb, bm, pick, out=out, read_bytes=rb, ws=gws)
    torch.cuda.synchronize()
    if not torch.equal(out.view(torch.int32), rows[pick].view(torch.int32)):
        raise RuntimeError("gathered rows differ from the table")
    import numpy as np
    compressed = int(np.unpackbits(bm.cpu().numpy().view(np.uint8)).sum())
    link = {"dma_pinned_to_device_GBps": round(n / (ms["dma_copy_table"] * 1e-3) / 1e9, 1),
            "gather_raw_slots_link_GBps": round(int(rb_raw.item()) / (ms["gather_raw_slots"] * 1e-3)
                                                / 1e9, 1)}
    res = {}
    for name in ("ibp_slots_compress", "ibp_slots_gather", "gather_raw_slots"):
        t = ms[name]
        if name == "ibp_slots_compress":
            unc, host = n, None  # reads the device table, writes the host slots
        else:
            unc = K * cb
            host = int((rb if name == "ibp_slots_gather" else rb_raw).item())
        res[name] = {"ms": round(t, 4), "GBps_uncompressed": round(unc / (t * 1e-3) / 1e9, 1)}
        if host is not None:
            res[name]["host_bytes_read"] = host
            res[name]["link_GBps"] = round(host / (t * 1e-3) / 1e9, 1)
            res[name]["frac_of_raw_gather_link"] = round(
                host / (t * 1e-3) / 1e9 / link["gather_raw_slots_link_GBps"], 4)
    line = {"sweep": "table_slots", "bytes": n, "rows_gathered": K,
            "ibp_mode": args.ibp_mode, "slots_compressed": compressed, "ops": res,
            "host_link": link,
            "speedup_vs_raw_gather": round(ms["gather_raw_slots"] / ms["ibp_slots_gather"], 4),
            "config": {"chunk": cb, "warmup": args.warmup, "steps": args.steps,
                       "slots": "pinned host memory", "l2": "flushed before every launch"}}
    print(json.dumps(line), flush=True)


def sweep_arm(args):
    """Per-op throughput, one JSON line per workload and size.

    --codec zipccl / ibp: the size sweep (1 MiB .. 4 GiB in x4 steps, or
    --sizes in MiB): ZipCCL on bf16 N(0, 0.01), one segment, chunk 4096; IBP on
    fp32 N(0, 0.02) weights, 2048-byte chunks (512 values), T = 0.9, metadata
    from 10,000 seeded sample chunks.  --codec table / gradient / moe: the
    full-size embedding table, gradient-like buffer and MoE activations;
    table_host: the table and its stream in pinned host memory, read in place;
    ibp16: IBP on bf16 N(0, 0.02) weights in 512-byte chunks (size sweep).
    --only limits the timed ops (the ops before them run once, untimed)."""
    import torch

    from lossless_bit_level_bf16_gb300 import abi, workloads as W
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    peak, peak_kind = _peaks()
    sizes = [int(float(v) * (1 << 20)) for v in args.sizes.split(",")] if args.sizes \
        else list(W.SWEEP_BYTES)
    if args.codec == "table_slots":
        return slots_arm(args)
    kinds = {"both": ["zipccl", "ibp"]}.get(args.codec, [args.codec])
    for kind in kinds:
        for nbytes in (sizes if kind in ("zipccl", "ibp", "ibp16") else [0]):
            ops, wss, unc, sbytes, check, nb, cb = _case(kind, nbytes, dev, args.ibp_mode)
            if args.only:
                names = args.only.split(",")
                first = min(i for i, o in enumerate(ops) if o[0] in names)
                for _, fn in ops[:first]:
                    fn()
                ops = [o for o in ops if o[0] in names]
            ms = _time_ops(ops, flush, stream, args.warmup, args.steps)
            for ws in wss:
                st = abi.status(ws)
                if st != 0:
                    raise RuntimeError(f"device status {st}: {abi.strerror(st)}")
            comp = int(nb.item())
            if not args.only and not check():
                raise RuntimeError(f"{kind} round trip differs at {unc} bytes")
            res = {}
            for name, t in ms.items():
                if name == "ibp_build_meta":
                    alg = unc_op = sbytes
                elif name == "zc_plan":
                    alg = unc_op = unc
                else:
                    alg, unc_op = unc + comp, unc
                gbs = alg / (t * 1e-3) / 1e9
                res[name] = {"ms": round(t, 4),
                             "GBps_uncompressed": round(unc_op / (t * 1e-3) / 1e9, 1),
                             "GBps_traffic": round(gbs, 1), "frac_hbm": round(gbs / peak, 4)}
            line = {"sweep": kind, "bytes": unc, "ratio": round(unc / comp, 4) if comp else None,
                    "l2_resident": unc <= 128 << 20, "peak_GBps": peak, "peak_kind": peak_kind,
                    "ops": res,
                    "config": {"chunk": cb, "ibp_mode": args.ibp_mode if cb != 4096 else None,
                               "warmup": args.warmup, "steps": args.steps,
                               "l2": "flushed before every launch"}}
            print(json.dumps(line), flush=True)
            del ops, wss, check
            torch.cuda.empty_cache()


# ---------------------------------------------------------------- oracle arm

def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            k = line.split(":")[0].strip().lower()
            if k in ("model name", "cpu model"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


class OracleSample:
    """The step's data on the host (the gradient-like buffer's 256 blocks and
    the 1,000,000-row table with its 10,000 sample rows), and one pass of the
    bit-serial oracle over part of it: ZipCCL encode + decode of `nblk`
    blocks, IBP metadata + encode + decode of `rows` rows.  With threads > 1
    the blocks and rows are cut into that many pieces (whole blocks; whole
    groups of 32 rows) and each piece is an ordinary oracle call in a thread
    of its own (ctypes releases the GIL), all pieces at once."""

    def __init__(self):
        import oracle as O
        from lossless_bit_level_bf16_gb300 import workloads as W
        O.build()
        self.O = O
        x, self.seg = W.zc_gradient(device="cpu")
        self.xb = W.bf16_bits(x)
        tab, idx = W.ibp_table(device="cpu")
        self.tb = W.f32_bytes(tab)
        self.sbytes = W.f32_bytes(tab[idx].contiguous())

    def run(self, nblk, rows, threads=1):
        import numpy as np
        from concurrent.futures import ThreadPoolExecutor
        O, B = self.O, 262144
        nblk, rows = max(1, min(256, nblk)), max(32, min(1_000_000, rows))

        def zc_piece(b0, b1):
            st, _, _, _ = O.zc_encode(self.xb[b0 * B:b1 * B],
                                      seg_off=[B * i for i in range(b1 - b0 + 1)], chunk_elems=4096)
            rc, y = O.zc_decode(st)
            assert rc == 0 and np.array_equal(y, self.xb[b0 * B:b1 * B])

        def ibp_piece(meta, r0, r1):
            xb = self.tb[r0 * 512:r1 * 512]
            st = O.ibp_encode(meta, xb)
            rc, y = O.ibp_decode(meta, st)
            assert rc == 0 and np.array_equal(y, xb)

        def cuts(n, k, unit=1):
            k = max(1, min(k, n // unit))
            e = [n * i // k // unit * unit for i in range(k)] + [n]
            return [(e[i], e[i + 1]) for i in range(k) if e[i + 1] > e[i]]

        with ThreadPoolExecutor(threads) as ex:
            t0 = time.perf_counter()
            list(ex.map(lambda c: zc_piece(*c), cuts(nblk, threads)))
            tz = time.perf_counter() - t0
            t0 = time.perf_counter()
            meta = O.ibp_build_meta(self.sbytes, 512, T=0.9, mode=0)
            tm = time.perf_counter() - t0
            t0 = time.perf_counter()
            list(ex.map(lambda c: ibp_piece(meta, *c), cuts(rows, threads, 32)))
            ti = time.perf_counter() - t0
        return nblk * B, tz, tm, rows, ti

    def rate(self, seconds, threads):
        """GB/s of the whole step's bytes (128 MiB ZipCCL + 512 MB IBP) at the
        rates a pass sized to take about `seconds` measures."""
        n_z, tz, tm, rows, ti = self.run(8, 25_000, threads)
        scale = max(0.5, seconds) / max(tz + tm + ti, 1e-3)
        if scale > 1.5:
            n_z, tz, tm, rows, ti = self.run(int(8 * scale), int(25_000 * scale), threads)
        zc_bytes, ibp_bytes = 2 * 256 * 262144, 1_000_000 * 512
        step_s = zc_bytes / (n_z * 2 / tz) + ibp_bytes / (rows * 512 / ti) + tm
        sample = (f"ZipCCL encode+decode of {n_z // 262144} of the 256 gradient blocks; IBP metadata "
                  f"from the 10,000 sample rows + encode+decode of {rows} of the 1,000,000 table "
                  f"rows; scaled to the step's 128 MiB + 512 MB")
        return (zc_bytes + ibp_bytes) / step_s / 1e9, sample, tz + tm + ti


def cpu_baseline(seconds=15.0):
    """The bit-serial oracle on the host cores: all cores (chunk-parallel:
    independent oracle calls on disjoint whole blocks / groups of rows) and a
    single thread, each on a bounded sample scaled to the step's byte mix."""
    smp = OracleSample()
    nproc = os.cpu_count() or 1
    v1, sample1, s1 = smp.rate(seconds, 1)
    vn, samplen, sn = smp.rate(seconds / 3, nproc)
    return {"value": round(vn, 4), "unit": "GB/s", "cores": nproc, "kind": "oracle",
            "sample": samplen + f"; {nproc} threads, one oracle call per piece",
            "sample_seconds": round(sn, 2), "cpu_model": cpu_model(), "nproc": nproc,
            "single_thread": {"value": round(v1, 4), "cores": 1, "sample": sample1,
                              "sample_seconds": round(s1, 2)}}


def reference_arm(args):
    """The oracle, as it stands, on all host cores: each step is one
    chunk-parallel pass over a bounded sample of the workload, sized so the
    whole --steps/--warmup run ends within a few minutes."""
    smp = OracleSample()
    nproc = os.cpu_count() or 1
    per_step = min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup))
    steps_s, vals = [], []
    last = None
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        v, last, _ = smp.rate(per_step, nproc)
        if i >= args.warmup:
            steps_s.append(time.perf_counter() - t0)
            vals.append(v)
    v = round(statistics.mean(vals), 4)
    return {
        "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1000 * statistics.mean(steps_s), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded generators; a bounded sample per step)",
        "config": {"workload": WORKLOAD, "zc_chunk": 4096, "ibp_chunk_bytes": 512, "ibp_T": 0.9,
                   "parallelism": f"host cores x{nproc}"},
        "impl": "reference",
        "cpu_baseline": {"kind": "oracle", "cores": nproc, "sample": last, "value": v,
                         "cpu_model": cpu_model()},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--scale", type=float, default=1.0, help="workload scale (1 = full size)")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--sweep", action="store_true",
                    help="size sweep of both codecs instead of the step (one line per size)")
    ap.add_argument("--codec", default="both",
                    choices=["both", "zipccl", "ibp", "ibp16", "table", "table_host", "gradient",
                             "moe", "table_slots"])
    ap.add_argument("--sizes", default="", help="sweep sizes in MiB, comma separated")
    ap.add_argument("--ibp-mode", type=int, default=0, choices=[0, 1])
    ap.add_argument("--only", default="", help="sweep: time only these ops (comma separated)")
    ap.add_argument("--no-targets", dest="targets", action="store_false",
                    help="skip the 1 GiB target cases after the step")
    ap.add_argument("--sustain-s", type=float, default=1.0,
                    help="seconds of repeated steps for the sustained clock record")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.sweep:
        args.warmup = max(args.warmup, 3)
        sweep_arm(args)
        return
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    args.warmup = max(args.warmup, 3)
    r = gpu_arm(args, rank, world, local_rank)
    if rank == 0:
        args.cpu_baseline = args.cpu_baseline and world >= 1
        line = report_gpu(args, r, world)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
