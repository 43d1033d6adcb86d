"""bench.py reports the profiled DRAM traffic (roofline.traffic) only for the
kernel sources the counters were taken on: the sha256 of the class-column
kernel, the small-N kernel and the device header they include must all
match the ones recorded in profiles/tq2_matvec_mma_stack_m1.md; any other
source gives None (no GPU needed)."""
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

FILES = ("tq2_matvec_mma.cu", "tq2_matvec_smalln.cu", "tq2_device.cuh")


@pytest.fixture
def tree(tmp_path, monkeypatch):
    csrc = tmp_path / "quantized_gemv_tq2_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in FILES:
        shutil.copy(os.path.join(ROOT, "quantized_gemv_tq2_gb300", "csrc", f), csrc / f)
    (tmp_path / "profiles").mkdir()
    shutil.copy(os.path.join(ROOT, "profiles", "tq2_matvec_mma_stack_m1.md"), tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def test_traffic_read_for_the_profiled_sources(tree):
    v = bench.read_profile_traffic()
    assert v is not None and 8.7e6 < v < 8.9e6  # ~1.003 x the 8,765,733 algorithmic bytes per launch


@pytest.mark.parametrize("f", FILES)
def test_traffic_dropped_once_a_source_changes(tree, f):
    p = tree / "quantized_gemv_tq2_gb300" / "csrc" / f
    p.write_bytes(p.read_bytes() + b"\n// changed\n")
    assert bench.read_profile_traffic() is None


def test_traffic_dropped_without_the_profile(tree):
    os.remove(tree / "profiles" / "tq2_matvec_mma_stack_m1.md")
    assert bench.read_profile_traffic() is None
