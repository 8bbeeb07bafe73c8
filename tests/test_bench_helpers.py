"""bench.py's host-side helpers: the DRAM traffic figure is taken from the
committed ncu summary only while the decode kernel's source is the one the
counters were taken on, and the algorithmic bytes of a step follow from the
lengths and shapes alone."""
import importlib
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    return importlib.import_module("bench")


def test_traffic_only_for_the_profiled_kernel_source(tmp_path, monkeypatch):
    bench = _bench()
    good = tmp_path / "good.md"
    good.write_text(f"# x\n\n- kernel_source_hash: `{bench.kernel_hash()}`\n- dram_bytes_per_launch: `123456`\n")
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(good))
    assert bench.profiled_traffic() == 123456.0
    stale = tmp_path / "stale.md"
    stale.write_text("- kernel_source_hash: `0000000000000000`\n- dram_bytes_per_launch: `123456`\n")
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(stale))
    assert bench.profiled_traffic() is None
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(tmp_path / "missing.md"))
    assert bench.profiled_traffic() is None


def test_step_bytes_from_lengths_and_shapes():
    bench = _bench()
    lens = np.array([5, 16, 17, 40])
    B, H, Hkv, D, e = 4, 8, 2, 128, 2
    decode_b, append_b = bench.step_bytes(lens, B, H, Hkv, D, e, 2)
    assert decode_b == int(lens.sum()) * Hkv * D * e * 2 + 2 * B * H * D * e
    # new K and V read and written, plus the int64 slot of each token
    assert append_b == B * Hkv * D * e * 2 * 2 + 8 * B
