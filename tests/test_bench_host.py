"""Host logic of the benchmark: the roofline's measured-traffic lookup and
peaks.  A committed ncu figure may be used only for the kernel sources it was
measured on; these tests need no GPU."""
import glob
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_traffic_lookup_takes_the_capture_of_the_current_sources():
    table = {"k_kernel": {"aaaaaaaaaaaa": 100, "bbbbbbbbbbbb": 200}}
    assert bench.measured_traffic("k_kernel", table, "bbbbbbbbbbbb") == 200
    assert bench.measured_traffic("k_kernel", table, "aaaaaaaaaaaa") == 100
    assert bench.measured_traffic("k_kernel", table, "cccccccccccc") is None
    assert bench.measured_traffic("other_kernel", table, "aaaaaaaaaaaa") is None


def test_traffic_lines_are_well_formed():
    """Every 'traffic' line of the profile summaries names a kernel, a 12-digit
    source hash and a byte count; a kernel never has two figures for the same
    sources."""
    seen = {}
    n = 0
    for f in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for line in open(f):
            parts = line.strip().strip("`").split()
            if not parts or parts[0] != "traffic":
                continue
            n += 1
            assert len(parts) == 4, (f, line)
            _, kernel, sha, nbytes = parts
            assert re.fullmatch(r"[a-z0-9_]+_kernel", kernel), (f, line)
            assert re.fullmatch(r"[0-9a-f]{12}", sha), (f, line)
            assert nbytes.isdigit() and int(nbytes) > 0, (f, line)
            key = (kernel, sha)
            assert key not in seen or seen[key] == int(nbytes), (f, line, seen[key])
            seen[key] = int(nbytes)
    assert n > 0
    # the parser reads the same lines
    table = bench._traffic_table()
    for (kernel, sha), nbytes in seen.items():
        assert table[kernel][sha] == nbytes


def test_roofline_kernel_has_a_capture():
    """The bench's roofline kernel (the single-pass IBP encoder) has a committed
    DRAM-traffic figure, within a few percent of its algorithmic bytes (table
    read once, stream written once)."""
    figures = bench._traffic_table().get("ibp_encode_ws_kernel", {})
    assert figures
    alg = 1_024_728_640  # 512,000,000 bytes read + 512,728,640 bytes of stream written
    for nbytes in figures.values():
        assert 0.9 * alg < nbytes < 1.1 * alg


def test_source_hash_covers_every_cuda_source():
    srcs = sorted(glob.glob(os.path.join(ROOT, "lossless_bit_level_bf16_gb300", "csrc", "*")))
    assert any(s.endswith(".cu") for s in srcs) and any(s.endswith(".cuh") for s in srcs)
    h = bench.csrc_hash()
    assert re.fullmatch(r"[0-9a-f]{12}", h) and h == bench.csrc_hash()


def test_peaks_come_from_the_measured_file():
    peak, kind = bench._peaks()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        assert kind == "measured" and peak > 1000.0
    else:
        assert (peak, kind) == (6800.0, "fallback")
