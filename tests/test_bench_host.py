"""Host logic of bench.py that needs no GPU: the roofline bound and
fraction, the measured-peak file, and the DRAM traffic records, which are
reported only while the kernel sources they were captured on are unchanged."""
import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_roofline_compute_bound_square():
    """8192^3 fp16: 2731 FLOP per byte, far above the ridge, so the bound is
    the tensor peak and the fraction is the peak time over the measured one."""
    flops = 2.0 * 8192 ** 3
    alg = 3 * 8192 * 8192 * 2
    peak, hbm = 1886.1, 6777.3
    t_peak = flops / (peak * 1e12)
    bound, frac = bench.roofline_of(flops, alg, t_peak / 0.98, peak, hbm)
    assert bound == "tensor"
    assert frac == pytest.approx(0.98)


def test_roofline_memory_bound_skinny():
    """16 x 4096 x 4096: 15.9 FLOP per byte, below the ridge, so the bound
    is HBM and the fraction is the copy time of the bytes over the measured
    time."""
    M, N, K = 16, 4096, 4096
    flops = 2.0 * M * N * K
    alg = (M * K + K * N + M * N) * 2
    bound, frac = bench.roofline_of(flops, alg, 10e-6, 1886.1, 6777.3)
    assert bound == "hbm"
    assert frac == pytest.approx(alg / 6777.3e9 / 10e-6)


def test_roofline_alu_bound():
    """The SIMT fp32 path reports against its own FMA peak when given one."""
    flops, alg = 2.0 * 128 ** 3, 3 * 128 * 128 * 4
    bound, frac = bench.roofline_of(flops, alg, 1e-3, 1886.1, 6777.3, alu_tflops=80.0)
    assert bound == "alu"
    assert frac == pytest.approx(flops / 80e12 / 1e-3)


def test_measured_peaks_are_read_when_present():
    peaks, source = bench.load_peaks()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            want = json.load(f)
        assert source == "measured" and peaks == want
    else:
        assert source == "fallback" and peaks == bench.FALLBACK_PEAKS


def test_traffic_records_match_the_committed_sources():
    """Every committed traffic record was captured on the sources as they
    are now; a record whose hash no longer matches is reported as null."""
    for table in (bench.NCU_TRAFFIC, bench.ATTN_NCU_TRAFFIC):
        for name, rec in table.items():
            assert bench.traffic_of(table, name) == rec["bytes"], name
    stale = {"x": {"bytes": 1, "kernel_hash": "0" * 16, "sources": bench.PAIR_SOURCES}}
    assert bench.traffic_of(stale, "x") is None
    assert bench.traffic_of(stale, "missing") is None


def test_kernel_hash_covers_every_listed_source(tmp_path):
    """The hash changes with any byte of any listed source (checked on
    copies: absolute paths to them stand in for the listed ones)."""
    copies = []
    for i, src in enumerate(bench.MAIN_SOURCES):
        dst = tmp_path / f"{i}_{os.path.basename(src)}"
        with open(os.path.join(ROOT, src), "rb") as f:
            dst.write_bytes(f.read())
        copies.append(str(dst))
    base = bench.kernel_hash(copies)
    assert len(base) == 16 and base == bench.kernel_hash(bench.MAIN_SOURCES)
    assert bench.kernel_hash(bench.PAIR_SOURCES) != base
    for c in copies:
        data = open(c, "rb").read()
        with open(c, "wb") as f:
            f.write(data + b" ")
        assert bench.kernel_hash(copies) != base, c
        with open(c, "wb") as f:
            f.write(data)
    assert bench.kernel_hash(copies) == base
