"""The committed ncu summaries are readable by bench.py: every per-kernel
summary names its DRAM bytes per launch, the hash of the sources it was taken
on and the command that produced it (which runs committed files only)."""
import glob
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _summaries():
    return sorted(p for p in glob.glob(os.path.join(ROOT, "profiles", "*.md"))
                  if not os.path.basename(p).startswith("launches_"))


def test_per_kernel_summaries_carry_bytes_hash_and_command():
    files = _summaries()
    assert files, "no per-kernel summaries"
    for p in files:
        txt = open(p).read()
        m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
        h = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", txt)
        assert m and float(m.group(1)) > 0, p
        assert h, p
        assert "ncu " in txt and "--clock-control none" in txt, p
        assert "_work" not in txt, p


def test_summary_names_map_to_kernels_bench_reports():
    known = {pre for pre, _ in bench.KERNEL_SOURCE}
    for p in _summaries():
        kernel = os.path.basename(p).rsplit("_", 1)[0]
        assert any(kernel.startswith(pre) for pre in known), p
        assert bench.src_hash(kernel) is not None, p


def test_launch_lists_give_their_command():
    files = glob.glob(os.path.join(ROOT, "profiles", "launches_*.md"))
    assert files
    for p in files:
        txt = open(p).read()
        assert "gpu__time_duration.sum" in txt and "--clock-control none" in txt, p
