"""Shared 3000-token prefix + beam search with copy-on-write, end to end:
C++ allocator + GPU copy/append/decode against the oracle allocator + oracle
ops.  Allocator state and caches bit-exact at every step, decode outputs
within tolerance."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_142_gb300 import workloads as W
from paged_case import TOL, cache_bits, to_device, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops(lib):
    import importlib
    return importlib.import_module("paged_kv_cache_142_gb300.ops")


def _f64(bits):
    return W.bf16_bits_to_f32(bits).reshape(bits.shape).astype(np.float64)


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_prefix_beam_cow(ops, bs):
    wl = W.prefix_bf16(block_size=bs)
    S, H, Hkv, D = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    shape = (wl.num_blocks, Hkv, bs, D)
    # ---- GPU side ----
    ga = ops.BlockAllocator(wl.num_blocks, bs, wl.free_order)
    kc = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    root = ga.seq_create()
    slots = ga.append_tokens(root, wl.prefix_len)
    ops.pa_reshape_and_cache(to_device(wl.prefix_key), to_device(wl.prefix_value),
                             torch.from_numpy(slots).cuda(), kc, vc)
    gbeams = [ga.fork(root) for _ in range(S)]
    ga.free_seq(root)
    # ---- oracle side ----
    oa = oracle.OracleAllocator(wl.num_blocks, bs, wl.free_order)
    ok = np.zeros(shape, dtype=np.uint16)
    ov = np.zeros_like(ok)
    oroot = oa.seq_create()
    oracle.reshape_and_cache(wl.prefix_key.bits, wl.prefix_value.bits, ok, ov,
                             oa.append_tokens(oroot, wl.prefix_len))
    obeams = [oa.fork(oroot) for _ in range(S)]
    oa.free_seq(oroot)
    assert ga.snapshot() == oa.snapshot()

    maxb = -(-(wl.prefix_len + wl.steps) // bs)
    max_len = wl.prefix_len + wl.steps
    ws = ops.make_workspace(S, H, Hkv, D, bs, "bf16", max_len)
    n_cow = 0
    for step in range(wl.steps):
        if step > 0:
            ng, no = [], []
            for grp in range(wl.groups):
                for j in range(wl.beam):
                    par = grp * wl.beam + int(wl.parents[step, grp, j])
                    ng.append(ga.fork(gbeams[par]))
                    no.append(oa.fork(obeams[par]))
            for s in gbeams:
                ga.free_seq(s)
            for s in obeams:
                oa.free_seq(s)
            gbeams, obeams = ng, no
        # GPU step: COW copies, then the new token's K/V, then decode
        slots, pairs = ga.append_slots(gbeams)
        if len(pairs):
            ops.pa_copy_blocks(kc, vc, torch.from_numpy(pairs).cuda())
        n_cow += len(pairs)
        ops.pa_reshape_and_cache(to_device(wl.step_key[step]), to_device(wl.step_value[step]),
                                 torch.from_numpy(slots).cuda(), kc, vc)
        tables, lens = ga.export_tables(gbeams, maxb)
        out = torch.empty((S, H, D), dtype=torch.float32, device="cuda")
        ops.pa_decode(out, to_device(wl.step_q[step]), kc, vc, torch.from_numpy(tables).cuda(),
                      torch.from_numpy(lens).cuda(), wl.scale, Hkv, max_len, ws)
        # oracle step
        oref = [oa.append_slot(s) for s in obeams]
        opairs = [(a, b) for _, a, b in oref if a >= 0]
        assert slots.tolist() == [r[0] for r in oref]
        assert pairs.tolist() == [list(p) for p in opairs]
        oracle.copy_blocks(ok, ov, opairs)
        oracle.reshape_and_cache(wl.step_key[step].bits, wl.step_value[step].bits, ok, ov,
                                 [r[0] for r in oref])
        torch.cuda.synchronize()
        assert ops.pa_workspace_error(ws) == 0
        assert ga.snapshot() == oa.snapshot()
        assert np.array_equal(cache_bits(kc), ok) and np.array_equal(cache_bits(vc), ov)
        if step in (0, 1, wl.steps // 2, wl.steps - 1):
            otab = np.zeros((S, maxb), dtype=np.int64)
            for j, s in enumerate(obeams):
                t = oa.block_table(s)
                otab[j, :len(t)] = t
            ref = oracle.paged_decode(wl.step_q[step].f32, _f64(ok), _f64(ov), otab,
                                      [oa.seq_len(s) for s in obeams], wl.scale, Hkv)
            assert float(np.abs(to_f64(out) - ref).max()) <= TOL["bf16"]
    assert n_cow > 0


def test_shared_prefix_equals_private_copies_on_gpu(ops):
    """Invariant (c) on the GPU: a forked prefix decodes to the same bits as
    private copies of it."""
    wl = W.prefix_bf16(block_size=16, groups=4, beam=4, steps=4)
    S, H, Hkv, D, bs = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, 16
    L = wl.prefix_len + 1
    maxb = -(-L // bs)
    outs = []
    for shared in (True, False):
        NB = (S + 1) * (maxb + 1)
        a = ops.BlockAllocator(NB, bs, np.random.default_rng(4).permutation(NB))
        kc = torch.zeros((NB, Hkv, bs, D), dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        pk, pv = to_device(wl.prefix_key), to_device(wl.prefix_value)
        if shared:
            root = a.seq_create()
            ops.pa_reshape_and_cache(pk, pv, torch.from_numpy(a.append_tokens(root, wl.prefix_len)).cuda(), kc, vc)
            beams = [a.fork(root) for _ in range(S)]
            a.free_seq(root)
        else:
            beams = []
            for _ in range(S):
                s = a.seq_create()
                ops.pa_reshape_and_cache(pk, pv, torch.from_numpy(a.append_tokens(s, wl.prefix_len)).cuda(), kc, vc)
                beams.append(s)
        slots, pairs = a.append_slots(beams)
        if len(pairs):
            ops.pa_copy_blocks(kc, vc, torch.from_numpy(pairs).cuda())
        ops.pa_reshape_and_cache(to_device(wl.step_key[0]), to_device(wl.step_value[0]),
                                 torch.from_numpy(slots).cuda(), kc, vc)
        tables, lens = a.export_tables(beams, maxb)
        ws = ops.make_workspace(S, H, Hkv, D, bs, "bf16", L)
        out = torch.empty((S, H, D), dtype=torch.float32, device="cuda")
        ops.pa_decode(out, to_device(wl.step_q[0]), kc, vc, torch.from_numpy(tables).cuda(),
                      torch.from_numpy(lens).cuda(), wl.scale, Hkv, L, ws)
        torch.cuda.synchronize()
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
