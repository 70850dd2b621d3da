"""Host logic of the benchmark: the roofline's measured-traffic lookup and
peaks.  A committed ncu figure may be used only for the kernel sources it was
measured on; these tests need no GPU."""
import glob
import os
import re

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_traffic_lookup_takes_the_capture_of_the_current_sources():
    table = {"k_kernel": {"aaaaaaaaaaaa": [(100, 1000, "c1")],
                          "bbbbbbbbbbbb": [(200, 1000, "c1"), (50, 500, "c2")]}}
    assert bench.measured_traffic("k_kernel", "c1", 1000, table, "bbbbbbbbbbbb") == (200, 1000)
    assert bench.measured_traffic("k_kernel", "c2", 500, table, "bbbbbbbbbbbb") == (50, 500)
    assert bench.measured_traffic("k_kernel", "c1", 1000, table, "aaaaaaaaaaaa") == (100, 1000)
    assert bench.measured_traffic("k_kernel", "c2", 500, table, "aaaaaaaaaaaa") == (None, None)
    assert bench.measured_traffic("k_kernel", "c1", 1000, table, "cccccccccccc") == (None, None)
    assert bench.measured_traffic("other_kernel", "c1", 1000, table, "aaaaaaaaaaaa") == \
        (None, None)


def test_traffic_scales_with_the_launch_size():
    """A capture of a smaller launch of the same case stands for a larger one
    in proportion to the uncompressed bytes."""
    table = {"k_kernel": {"aaaaaaaaaaaa": [(1_700_000_000, 1 << 30, "c1")]}}
    got, cap = bench.measured_traffic("k_kernel", "c1", 1 << 31, table, "aaaaaaaaaaaa")
    assert (got, cap) == (3_400_000_000, 1 << 30)
    got, _ = bench.measured_traffic("k_kernel", "c1", 1 << 29, table, "aaaaaaaaaaaa")
    assert got == 850_000_000


def test_traffic_lines_are_well_formed():
    """Every 'traffic' line of the profile summaries names a kernel, a 12-digit
    source hash, a byte count, the captured launch's uncompressed bytes and
    its case; a kernel never has two figures for the same sources and case."""
    seen = {}
    n = 0
    for f in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for line in open(f):
            parts = line.strip().strip("`").split()
            if not parts or parts[0] != "traffic":
                continue
            n += 1
            assert len(parts) == 6, (f, line)
            _, kernel, sha, nbytes, unc, case = parts
            assert re.fullmatch(r"[a-z0-9_]+_kernel", kernel), (f, line)
            assert re.fullmatch(r"[0-9a-f]{12}", sha), (f, line)
            assert nbytes.isdigit() and int(nbytes) > 0, (f, line)
            assert unc.isdigit() and int(unc) > 0, (f, line)
            assert re.fullmatch(r"[A-Za-z0-9_.]+", case), (f, line)
            key = (kernel, sha, case)
            assert key not in seen or seen[key] == (int(nbytes), int(unc)), (f, line, seen[key])
            seen[key] = (int(nbytes), int(unc))
    assert n > 0
    # the parser reads the same lines
    table = bench._traffic_table()
    for (kernel, sha, case), (nbytes, unc) in seen.items():
        assert bench.measured_traffic(kernel, case, unc, table, sha) == (nbytes, unc)


def test_bench_cases_name_the_captured_workloads():
    """The case names the bench looks up are the ones the captures use."""
    assert bench.case_of("zipccl", 2048, 0) == "zc_gauss0.01_c4096"
    assert bench.case_of("ibp", 2048, 1) == "ibp_gauss0.02_2048B_mode1"
    cases = {c for per in bench._traffic_table().values() for lines in per.values()
             for _, _, c in lines}
    assert "ibp_table_512B_mode0" in cases and "zc_gauss0.01_c4096" in cases


def test_roofline_kernel_has_a_capture():
    """The bench's roofline kernel (the single-pass IBP encoder) has a committed
    DRAM-traffic figure on its workload, within a few percent of its
    algorithmic bytes (table read once, stream written once)."""
    figures = bench._traffic_table().get("ibp_encode_ws_kernel", {})
    assert figures
    alg = 1_024_728_640  # 512,000,000 bytes read + 512,728,640 bytes of stream written
    lines = [t for per in figures.values() for t in per if t[2] == "ibp_table_512B_mode0"]
    assert lines
    for nbytes, unc, _ in lines:
        assert unc == 512_000_000 and 0.9 * alg < nbytes < 1.1 * alg


def test_source_hash_covers_every_cuda_source():
    srcs = sorted(glob.glob(os.path.join(ROOT, "lossless_bit_level_bf16_gb300", "csrc", "*")))
    assert any(s.endswith(".cu") for s in srcs) and any(s.endswith(".cuh") for s in srcs)
    h = bench.csrc_hash()
    assert re.fullmatch(r"[0-9a-f]{12}", h) and h == bench.csrc_hash()


def test_kernel_hash_follows_the_kernels_own_sources():
    """A kernel's hash covers its own source file and the shared headers:
    kernels of one file share it, kernels of different files differ, and a
    name no source defines is refused."""
    ws, dec = bench.kernel_hash("ibp_encode_ws_kernel"), bench.kernel_hash("ibp_decode_pipe_kernel")
    zenc, zdec = bench.kernel_hash("zc_encode_kernel"), bench.kernel_hash("zc_decode_kernel")
    stats = bench.kernel_hash("zc_stats_kernel")
    assert all(re.fullmatch(r"[0-9a-f]{12}", h) for h in (ws, dec, zenc, zdec, stats))
    assert ws == dec and zenc == zdec
    assert len({ws, zenc, stats}) == 3
    with pytest.raises(KeyError):
        bench.kernel_hash("no_such_kernel")


def test_every_bench_kernel_has_one_defining_source():
    """Each kernel the bench names for an op is defined in exactly one CUDA
    source file, so its traffic figures are keyed by that file's hash; and
    every committed traffic line names such a kernel."""
    names = set()
    for op in ("zc_plan", "zc_compress", "zc_compress_fit", "zc_decompress", "ibp_build_meta",
               "ibp_decompress"):
        names.update(bench.kernels_of(op))
    for cb in (512, 1024, 2048, 1536):
        names.update(bench.kernels_of("ibp_compress", cb))
    for k in sorted(names):
        assert re.fullmatch(r"[0-9a-f]{12}", bench.kernel_hash(k)), k
    for k in bench._traffic_table():
        assert k in names, k


def test_peaks_come_from_the_measured_file():
    peak, kind = bench._peaks()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        assert kind == "measured" and peak > 1000.0
    else:
        assert (peak, kind) == (6800.0, "fallback")
