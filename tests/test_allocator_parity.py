"""C++ BlockAllocator (through the C ABI) against the oracle allocator:
identical free-list order, reference counts, tables, slots and copy pairs."""
import numpy as np
import pytest

import oracle
from oracle import OracleAllocator, AllocatorOOM
from paged_kv_cache_142_gb300 import workloads as W


@pytest.fixture(scope="module")
def ops(lib):
    import importlib
    return importlib.import_module("paged_kv_cache_142_gb300.ops")


def test_workload_prefill_bit_exact(ops):
    for wl in (W.tiny_fp32(), W.mha_bf16(), W.gqa_bf16()):
        a = ops.BlockAllocator(wl.num_blocks, wl.block_size, wl.free_order)
        o = OracleAllocator(wl.num_blocks, wl.block_size, wl.free_order)
        for i in range(wl.num_seqs):
            s1, s2 = a.seq_create(), o.seq_create()
            assert s1 == s2 == i
            n = int(wl.context_lens[i])
            assert a.append_tokens(s1, n).tolist() == o.append_tokens(s2, n)
        assert a.snapshot() == o.snapshot()
        tables, lens = a.export_tables(list(range(wl.num_seqs)), wl.max_blocks_per_seq, pad_value=0)
        for i in range(wl.num_seqs):
            t = o.block_table(i)
            assert tables[i, :len(t)].tolist() == t and (tables[i, len(t):] == 0).all()
        assert lens.tolist() == wl.context_lens.tolist()


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_beam_workload_bit_exact(ops, bs):
    """The shared-prefix + beam workload's allocator trace: fork, free, append
    with copy-on-write; same pairs, slots and state on both sides."""
    wl = W.prefix_bf16(block_size=bs, steps=8)
    a = ops.BlockAllocator(wl.num_blocks, bs, wl.free_order)
    o = OracleAllocator(wl.num_blocks, bs, wl.free_order)
    ra, ro = a.seq_create(), o.seq_create()
    assert a.append_tokens(ra, wl.prefix_len).tolist() == o.append_tokens(ro, wl.prefix_len)
    beams_a = [a.fork(ra) for _ in range(wl.num_seqs)]
    beams_o = [o.fork(ro) for _ in range(wl.num_seqs)]
    a.free_seq(ra)
    o.free_seq(ro)
    total_cow = 0
    for step in range(wl.steps):
        if step > 0:
            new_a, new_o = [], []
            for g in range(wl.groups):
                for j in range(wl.beam):
                    par = g * wl.beam + int(wl.parents[step, g, j])
                    new_a.append(a.fork(beams_a[par]))
                    new_o.append(o.fork(beams_o[par]))
            for s in beams_a:
                a.free_seq(s)
            for s in beams_o:
                o.free_seq(s)
            beams_a, beams_o = new_a, new_o
        slots, pairs = a.append_slots(beams_a)
        ref = [o.append_slot(s) for s in beams_o]
        assert slots.tolist() == [r[0] for r in ref]
        assert pairs.tolist() == [[r[1], r[2]] for r in ref if r[1] >= 0]
        total_cow += len(pairs)
        assert a.snapshot() == o.snapshot()
    assert total_cow > 0 or bs == 8


def test_random_ops_fuzz_bit_exact(ops):
    rng = np.random.default_rng(142)
    NB, bs = 48, 4
    order = rng.permutation(NB)
    a = ops.BlockAllocator(NB, bs, order)
    o = OracleAllocator(NB, bs, order)
    for step in range(3000):
        live = o.live_seqs()
        op = int(rng.integers(0, 5))
        if op == 0 or not live:
            assert a.seq_create() == o.seq_create()
        elif op in (1, 2):
            s = int(rng.choice(live))
            try:
                r = o.append_slot(s)
            except AllocatorOOM:
                before = a.snapshot()
                with pytest.raises(ops.AllocatorOOM):
                    a.append_slot(s)
                assert a.snapshot() == before
            else:
                assert a.append_slot(s) == r
        elif op == 3:
            s = int(rng.choice(live))
            assert a.fork(s) == o.fork(s)
        else:
            s = int(rng.choice(live))
            a.free_seq(s)
            o.free_seq(s)
        if step % 50 == 0:
            assert a.snapshot() == o.snapshot()
    assert a.snapshot() == o.snapshot()


def test_errors(ops):
    a = ops.BlockAllocator(4, 2)
    with pytest.raises(ops.PAError):
        a.free_seq(0)  # no such sequence
    with pytest.raises(ops.PAError):
        a.decref(1)    # already free
    with pytest.raises(ops.PAError):
        ops.BlockAllocator(4, 2, [0, 1, 1, 2])  # not a permutation
    s = a.seq_create()
    before = a.snapshot()
    with pytest.raises(ops.AllocatorOOM):
        a.append_tokens(s, 9)  # needs 5 blocks of 4
    assert a.snapshot() == before
    a.append_tokens(s, 3)
    c = a.fork(s)
    with pytest.raises(ops.PAError):
        a.append_tokens(c, 1)  # would need a copy: not a bulk append


def test_outputs_written_into_caller_arrays(ops):
    """append_slots / export_tables with caller-provided arrays (e.g. views of
    a pinned staging buffer) write exactly what they would return."""
    wl = W.tiny_fp32()
    a = ops.BlockAllocator(wl.num_blocks, wl.block_size, wl.free_order)
    b = ops.BlockAllocator(wl.num_blocks, wl.block_size, wl.free_order)
    seqs = [a.seq_create() for _ in range(wl.num_seqs)]
    assert [b.seq_create() for _ in range(wl.num_seqs)] == seqs
    for s, n in zip(seqs, wl.context_lens):
        a.append_tokens(s, int(n))
        b.append_tokens(s, int(n))
    stage = np.zeros(64, dtype=np.int64)
    for _ in range(20):
        want_slots, want_pairs = a.append_slots(seqs)
        got_slots, got_pairs = b.append_slots(seqs, out=stage[8:8 + len(seqs)])
        assert np.array_equal(stage[8:8 + len(seqs)], want_slots) and np.array_equal(got_slots, want_slots)
        assert np.array_equal(got_pairs, want_pairs)
    mb = wl.max_blocks_per_seq + 2
    want_t, want_l = a.export_tables(seqs, mb)
    buf = np.full(len(seqs) * mb + len(seqs), -7, dtype=np.int32)
    t_view, l_view = buf[:len(seqs) * mb].reshape(len(seqs), mb), buf[len(seqs) * mb:]
    b.export_tables(seqs, mb, out=(t_view, l_view))
    assert np.array_equal(t_view, want_t) and np.array_equal(l_view, want_l)
    with pytest.raises(ValueError):
        b.export_tables(seqs, mb, out=(t_view[:, :-1], l_view))
    with pytest.raises(ValueError):
        b.append_slots(seqs, out=np.zeros(len(seqs), dtype=np.int32))
