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


def test_workloads_without_values_keep_lengths_and_free_lists():
    """The bench's MHA and long-context extras draw their values on the
    device; their lengths, pool and free-list order must be the parity
    workloads' own."""
    from paged_kv_cache_142_gb300 import workloads as W
    # small instances: the draw order does not depend on the sizes
    for make in (lambda v: W.mha_bf16(num_seqs=6, values=v),
                 lambda v: W.long_bf16(block_size=32, num_seqs=2, context_len=512, values=v)):
        full, bare = make(True), make(False)
        assert np.array_equal(full.context_lens, bare.context_lens)
        assert np.array_equal(full.free_order, bare.free_order)
        assert full.num_blocks == bare.num_blocks and bare.key_hist is None and bare.q is None
