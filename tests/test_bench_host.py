"""Host-side pieces of bench.py, on the CPU: the visible-pair count behind every
throughput figure (4 * pairs * H * d real-token flops; with a window, pairs
inside each query's band), the lookup of the committed DRAM-traffic records,
and the summary of the nvidia-smi samples taken during the timed region."""

import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _brute_pairs(lengths, first_token, window):
    """Counts (query, key) pairs one by one: query r of a sequence of length L
    sees key c when 0 <= c < L and, with a window (left, right), r - left <= c
    <= r + right (a negative bound is unbounded); a first-token call has only
    the query at position 0."""
    total = 0
    for length in lengths:
        for r in ([0] if first_token else range(length)):
            for c in range(length):
                if window is not None:
                    left, right = window
                    if left >= 0 and c < r - left:
                        continue
                    if right >= 0 and c > r + right:
                        continue
                total += 1
    return total


@pytest.mark.parametrize("window", [None, (0, 0), (3, 5), (-1, 2), (4, -1), (64, 64)])
@pytest.mark.parametrize("first_token", [False, True])
def test_visible_pairs_match_brute_force(window, first_token):
    lengths = np.random.default_rng(7).integers(1, 40, size=25)
    want = _brute_pairs(lengths, first_token, window)
    assert bench.visible_pairs(lengths, first_token, window) == want
    assert bench.real_flops(lengths, 3, 16, first_token, window) == 4.0 * want * 3 * 16


def test_full_attention_flops_closed_form():
    """Full attention: 4 * sum L^2 * H * d (the metric's definition)."""
    lengths = [1, 7, 128, 300]
    assert bench.real_flops(lengths, 16, 64) == 4.0 * sum(x * x for x in lengths) * 16 * 64
    assert bench.real_flops(lengths, 16, 64, first_token=True) == 4.0 * sum(lengths) * 16 * 64


def _record_files():
    prof = os.path.join(ROOT, "profiles")
    return sorted(f for f in os.listdir(prof) if f.endswith("_traffic.txt"))


def _fields(name):
    out = {}
    with open(os.path.join(ROOT, "profiles", name)) as fh:
        for line in fh:
            if line.startswith("#"):
                continue
            key, _, value = line.partition(":")
            out[key.strip()] = value.strip()
    return out


@pytest.mark.parametrize("name", _record_files())
def test_traffic_records_are_well_formed(name):
    """Every committed record names a kernel family bench.py knows, its source
    list is that family's, and its figures are positive bytes."""
    kernel = name[: -len("_traffic.txt")]
    assert kernel in bench.KERNEL_SOURCES
    f = _fields(name)
    srcs = [s.strip().split("/")[-1] for s in f["source_file"].split(",")] \
        if "source_file" in f else bench.KERNEL_SOURCES[kernel]
    assert srcs == bench.KERNEL_SOURCES[kernel]
    assert len(f["source_sha1"]) == 40
    assert float(f["dram_bytes_per_launch"]) > 0
    assert float(f["algorithmic_bytes_per_launch"]) > 0


@pytest.mark.parametrize("name", _record_files())
def test_traffic_lookup_needs_matching_sources_and_workload(name):
    """The figure is reported only for the recorded workload and only while the
    sources hash to the recorded sha1; anything else reads as no figure."""
    kernel = name[: -len("_traffic.txt")]
    f = _fields(name)
    srcs = bench.KERNEL_SOURCES[kernel]
    got = bench.committed_traffic(kernel, srcs, f["config"])
    if bench.source_sha1(srcs) == f["source_sha1"]:
        assert got == float(f["dram_bytes_per_launch"])
    else:
        assert got is None
    assert bench.committed_traffic(kernel, srcs, f["config"] + " other") is None
    assert bench.committed_traffic(kernel, srcs[:1], f["config"]) is None or len(srcs) == 1
    assert bench.committed_traffic(kernel, None, f["config"]) is None


def _sampler_with(tmp_path, lines):
    path = tmp_path / "clocks.csv"
    path.write_text("".join(line + "\n" for line in lines))
    s = bench.ClockSampler(0, str(path))
    s.proc = object()       # as if nvidia-smi had run
    return s


def test_clock_summary_median_max_and_reasons(tmp_path):
    row = "0, {sm}, 2070, 900.1, 0x{bits}, {hw}, Not Active, Not Active, {cap}"
    lines = [row.format(sm=sm, bits="0", hw="Not Active", cap="Not Active") for sm in
             (2070, 2070, 1980)]
    lines.append(row.format(sm=2040, bits="4", hw="Not Active", cap="Active"))
    lines.append("garbage line")
    s = _sampler_with(tmp_path, lines)
    out = s.summary()
    assert out["sm_mhz"] == 2055.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 4
    lines.append(row.format(sm=1500, bits="8", hw="Active", cap="Not Active"))
    assert _sampler_with(tmp_path, lines).summary()["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_clock_summary_without_samples(tmp_path):
    assert _sampler_with(tmp_path, ["no samples here"]).summary()["reasons"] == ["no samples"]
    s = bench.ClockSampler(0, str(tmp_path / "absent.csv"))
    assert s.summary()["reasons"] == ["unavailable"]
