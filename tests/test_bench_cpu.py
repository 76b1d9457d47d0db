"""CPU tests of bench.py's host logic: the roofline arithmetic, the whole-job
rate, and the rule that a stored ncu traffic figure is used only for the
device code it was measured on."""

import json
import os
import shutil

import pytest

import bench


def test_roofline_fraction_and_units():
    rf = bench.roofline(1200.0, 1600.0, "TFLOP/s", "tensor", 5.0e8, 2.7e11, "FLOP")
    assert rf["frac"] == pytest.approx(0.75)
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s" and rf["traffic"] == 5.0e8


def test_whole_job_rate_counts_every_rank():
    # 2 ranks, 1e12 flops each, slowest rank 1 ms -> 2e15 flop/s = 2000 TFLOP/s
    assert bench.whole_job_rate(1e12, 2, 1.0, 1e12) == pytest.approx(2000.0)


def test_kernel_source_sha_is_per_kernel():
    shas = {k: bench.kernel_source_sha(k) for k in bench.KERNEL_SOURCES}
    assert len(set(shas.values())) == len(shas), "each kernel hashes its own sources"
    for files in bench.KERNEL_SOURCES.values():
        for f in files:
            assert os.path.exists(os.path.join(bench.ROOT, bench.PKG, "csrc", f)), f


def test_prefill_kernel_name_follows_the_library_dispatch():
    """bench.py names the kernel a prefill workload runs with the same rule as
    attn_fwd: the band kernel for a non-causal window of at most the library's
    kBandMaxWindow keys per side at d = 64."""
    import re
    src = open(os.path.join(bench.ROOT, bench.PKG, "csrc", "b300attn.cu")).read()
    m = re.search(r"constexpr int kBandMaxWindow = (\d+);", src)
    assert m and int(m.group(1)) == bench.BAND_MAX_WINDOW
    name = bench.prefill_kernel_name
    assert name(64, False, 128) == "prefill_band_kernel"
    assert name(64, False, 0) == "prefill_band_kernel"
    assert name(64, False, bench.BAND_MAX_WINDOW + 1) == "prefill_kernel"
    assert name(64, False, -1) == "prefill_kernel"
    assert name(64, True, 128) == "prefill_kernel"
    assert name(128, False, 128) == "prefill_kernel"


def test_stored_traffic_needs_matching_device_code(tmp_path, monkeypatch):
    """A traffic row is returned only when kernel, workload and source hash
    all match; a changed kernel (different hash) yields None."""
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    csrc = root / bench.PKG / "csrc"
    csrc.mkdir(parents=True)
    src = os.path.join(bench.ROOT, bench.PKG, "csrc")
    for f in ("prefill.cuh", "ptx.cuh"):
        shutil.copy(os.path.join(src, f), csrc / f)
    monkeypatch.setattr(bench, "ROOT", str(root))
    sha = bench.kernel_source_sha("prefill_kernel")
    rows = [{"kernel": "prefill_kernel", "workload": "w", "source_sha": sha,
             "dram_bytes_per_launch": 123.0}]
    (root / "profiles" / "traffic.json").write_text(json.dumps(rows))
    assert bench.stored_traffic("prefill_kernel", "w") == 123.0
    assert bench.stored_traffic("prefill_kernel", "other") is None
    with open(csrc / "prefill.cuh", "a") as fh:  # the kernel changes
        fh.write("\n// edited\n")
    assert bench.stored_traffic("prefill_kernel", "w") is None
