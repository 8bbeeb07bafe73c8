"""Shared-prefix decode (each group's shared blocks read once for all its
members) against the oracle's decode and against pa_decode.

The oracle's cache is a host copy that the oracle's own reshape_and_cache and
copy_blocks fill from the same inputs, slots and copy pairs as the device's."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_142_gb300 import workloads as W
from paged_case import TOL, to_device, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops(lib):
    import importlib
    return importlib.import_module("paged_kv_cache_142_gb300.ops")


class _Mirror:
    """The device cache's host twin, written only by the oracle."""

    def __init__(self, shape):
        self.k = np.zeros(shape, dtype=np.float32)
        self.v = np.zeros(shape, dtype=np.float32)

    def append(self, key, value, slots):
        oracle.reshape_and_cache(key.f32, value.f32, self.k, self.v, np.asarray(slots))

    def copy(self, pairs):
        oracle.copy_blocks(self.k, self.v, np.asarray(pairs))


def _common_prefix_blocks(tables, lens, members, bs):
    """Leading table entries shared by every member, whole blocks only."""
    n = min(int(lens[m]) for m in members) // bs
    k = 0
    while k < n and all(tables[m, k] == tables[members[0], k] for m in members):
        k += 1
    return k


def _shared_decode(ops, q, kc, vc, tables, lens, scale, Hkv, groups, bs):
    """groups: list of member index lists, consecutive and covering the batch."""
    starts, prefix = [0], []
    for g in groups:
        prefix.append(_common_prefix_blocks(tables, lens, g, bs) * bs)
        starts.append(starts[-1] + len(g))
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.pa_decode_shared_prefix(out, q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                                scale, Hkv, int(lens.max()), torch.tensor(starts, dtype=torch.int32, device="cuda"),
                                torch.tensor(prefix, dtype=torch.int32, device="cuda"),
                                max(len(g) for g in groups), max(prefix), status=status)
    torch.cuda.synchronize()
    return out, int(status.item()), prefix


@pytest.mark.parametrize("bs", [16, 8, 32])
def test_beam_search_shared_prefix_decode(ops, bs):
    wl = W.prefix_bf16(block_size=bs)
    S, H, Hkv, D = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    ga = ops.BlockAllocator(wl.num_blocks, bs, wl.free_order)
    kc = torch.zeros((wl.num_blocks, Hkv, bs, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    mirror = _Mirror(tuple(kc.shape))
    root = ga.seq_create()
    slots = ga.append_tokens(root, wl.prefix_len)
    ops.pa_reshape_and_cache(to_device(wl.prefix_key), to_device(wl.prefix_value),
                             torch.from_numpy(slots).cuda(), kc, vc)
    mirror.append(wl.prefix_key, wl.prefix_value, slots)
    beams = [ga.fork(root) for _ in range(S)]
    ga.free_seq(root)
    maxb = -(-(wl.prefix_len + wl.steps) // bs)
    max_len = wl.prefix_len + wl.steps
    ws = ops.make_workspace(S, H, Hkv, D, bs, "bf16", max_len)
    for step in range(wl.steps):
        if step > 0:
            nb = [ga.fork(beams[grp * wl.beam + int(wl.parents[step, grp, j])])
                  for grp in range(wl.groups) for j in range(wl.beam)]
            for s in beams:
                ga.free_seq(s)
            beams = nb
        slots, pairs = ga.append_slots(beams)
        if len(pairs):
            ops.pa_copy_blocks(kc, vc, torch.from_numpy(pairs).cuda())
            mirror.copy(pairs)
        ops.pa_reshape_and_cache(to_device(wl.step_key[step]), to_device(wl.step_value[step]),
                                 torch.from_numpy(slots).cuda(), kc, vc)
        mirror.append(wl.step_key[step], wl.step_value[step], slots)
        if step not in (0, wl.steps // 2, wl.steps - 1):
            continue
        tables, lens = ga.export_tables(beams, maxb)
        q = to_device(wl.step_q[step])
        plain = torch.empty((S, H, D), dtype=torch.float32, device="cuda")
        ops.pa_decode(plain, q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                      wl.scale, Hkv, max_len, ws)
        ref = oracle.paged_decode(wl.step_q[step].f32, mirror.k, mirror.v, tables, lens, wl.scale, Hkv)
        # one group of all sequences (the prompt's full blocks), then the 16 beam groups
        for groups in ([list(range(S))], [list(range(g * wl.beam, (g + 1) * wl.beam)) for g in range(wl.groups)]):
            out, st, prefix = _shared_decode(ops, q, kc, vc, tables, lens, wl.scale, Hkv, groups, bs)
            assert st == 0
            assert min(prefix) >= (wl.prefix_len // bs) * bs
            assert float(np.abs(to_f64(out) - ref).max()) <= TOL["bf16"]
            assert float(np.abs(to_f64(out) - to_f64(plain)).max()) <= 2 * TOL["bf16"]


@pytest.mark.parametrize("G,Hkv", [(1, 2), (4, 2), (8, 2), (1, 1)])
def test_random_groups(ops, G, Hkv):
    """Groups of several sizes and prefix lengths, singletons without a
    prefix, members whose length equals the prefix.  With one query head
    and an odd number of sequences the partial-result rows are odd in
    number, which the workspace layout must still keep 16-byte aligned."""
    _random_groups(ops, G, Hkv, 16)


@pytest.mark.parametrize("bs", [8, 64, 128])
def test_random_groups_block_sizes(ops, bs):
    """The same groups at other block sizes: up to 64 the own-token items hold
    two members each (one block per box in a 64-key half, one box at 64), at
    128 one member each."""
    _random_groups(ops, 4, 2, bs)


def _random_groups(ops, G, Hkv, bs):
    D = 128
    H = G * Hkv
    rng = np.random.default_rng(70 + G)
    NB = 900
    ga = ops.BlockAllocator(NB, bs, rng.permutation(NB).astype(np.int32))
    kc = torch.zeros((NB, Hkv, bs, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    mirror = _Mirror(tuple(kc.shape))
    # (members, prefix tokens), the prompts cut to whole blocks (members then
    # append past an unshared block)
    spec = [(m, P // bs * bs) for m, P in [(5, 480), (1, 0), (3, 32), (40, 160), (1, 0), (2, 1024), (3, 0)]]
    seqs, groups = [], []
    for members, P in spec:
        root = ga.seq_create()
        if P:
            sl = ga.append_tokens(root, P)
            kv = W.Values.from_f32((rng.standard_normal((2, P, Hkv, D)) * 0.5).astype(np.float32), "bf16")
            ops.pa_reshape_and_cache(to_device(kv[0]), to_device(kv[1]), torch.from_numpy(sl).cuda(), kc, vc)
            mirror.append(kv[0], kv[1], sl)
        g = []
        for m in range(members):
            s = ga.fork(root)
            extra = 0 if (m == 0 and P) else int(rng.integers(1, 70))
            if extra:
                sl = ga.append_tokens(s, extra)
                kv = W.Values.from_f32((rng.standard_normal((2, extra, Hkv, D)) * 0.5).astype(np.float32), "bf16")
                ops.pa_reshape_and_cache(to_device(kv[0]), to_device(kv[1]), torch.from_numpy(sl).cuda(), kc, vc)
                mirror.append(kv[0], kv[1], sl)
            g.append(len(seqs))
            seqs.append(s)
        ga.free_seq(root)
        groups.append(g)
    tables, lens = ga.export_tables(seqs, -(-1100 // bs) + 2)
    qv = W.Values.from_f32(rng.standard_normal((len(seqs), H, D)).astype(np.float32), "bf16")
    q = to_device(qv)
    scale = float(np.float32(1 / np.sqrt(D)))
    out, st, prefix = _shared_decode(ops, q, kc, vc, tables, lens, scale, Hkv, groups, bs)
    assert st == 0
    # the members share the prompt's whole blocks; a one-member group may use
    # all its whole blocks as its "prefix"
    assert [pf for pf, (m, _) in zip(prefix, spec) if m > 1] == [P for m, P in spec if m > 1]
    ref = oracle.paged_decode(qv.f32, mirror.k, mirror.v, tables, lens, scale, Hkv)
    assert float(np.abs(to_f64(out) - ref).max()) <= TOL["bf16"]
