"""Pins for the fp64 oracle: printed examples, closed forms, brute force,
invariants.  CPU only; independent of the CUDA path."""
import math

import numpy as np
import pytest

import oracle
from oracle import OracleAllocator, AllocatorOOM
from paged_kv_cache_142_gb300 import workloads as W
from conftest import read_golden


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------
def build_cache_with_allocator(wl, alloc=None):
    """Oracle-side paged state for a decode workload: allocator tables, slots,
    caches filled by the oracle slot write."""
    NB, Hkv, bs, D = wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim
    alloc = alloc or OracleAllocator(NB, bs, wl.free_order)
    slots = []
    for i in range(wl.num_seqs):
        s = alloc.seq_create()
        slots += alloc.append_tokens(s, int(wl.context_lens[i]))
    maxb = wl.max_blocks_per_seq
    tables = np.zeros((wl.num_seqs, maxb), dtype=np.int32)
    for i in range(wl.num_seqs):
        t = alloc.block_table(i)
        tables[i, :len(t)] = t
    kc = np.zeros((NB, Hkv, bs, D), dtype=np.float64)
    vc = np.zeros_like(kc)
    oracle.reshape_and_cache(wl.key_hist.f32, wl.value_hist.f32, kc, vc, slots)
    return alloc, tables, np.asarray(slots, dtype=np.int64), kc, vc


# --------------------------------------------------------------------------
# block counts: printed example + self-check question
# --------------------------------------------------------------------------
@pytest.mark.parametrize("row", read_golden("block_counts.txt"))
def test_block_counts_golden(row):
    n, bs, blocks, slots = map(int, row)
    assert oracle.blocks_for(n, bs) == blocks
    assert blocks * bs == slots
    assert oracle.slack_for(n, bs) == slots - n
    a = OracleAllocator(blocks + 3, bs)
    s = a.seq_create()
    a.append_tokens(s, n)
    assert len(a.block_table(s)) == blocks
    assert a.num_free() == 3


def test_waste_below_one_block_random():
    rng = np.random.default_rng(1)
    for bs in (1, 8, 16, 32):
        lens = rng.integers(1, 3000, size=40)
        a = OracleAllocator(int(sum(-(-int(n) // bs) for n in lens)), bs,
                            rng.permutation(sum(-(-int(n) // bs) for n in lens)))
        for n in lens:
            s = a.seq_create()
            a.append_tokens(s, int(n))
            held = len(a.block_table(s)) * bs
            assert 0 <= held - n < bs
        assert a.num_free() == 0


# --------------------------------------------------------------------------
# block table walk: the pages' printed tables
# --------------------------------------------------------------------------
def _golden_tables():
    out = {}
    for row in read_golden("block_table_examples.txt"):
        name, bs = row[0], int(row[1])
        pairs = sorted((int(a), int(b)) for a, b in (p.split(":") for p in row[2:]))
        out[name] = (bs, [b for _, b in pairs])
    return out


@pytest.mark.parametrize("name", ["vllm2", "pa"])
def test_table_walk_golden(name):
    bs, table = _golden_tables()[name]
    NB, Hkv, D = 24, 2, 4
    # each slot holds a value naming its physical block and offset
    cache = np.zeros((NB, Hkv, bs, D))
    for b in range(NB):
        for off in range(bs):
            cache[b, :, off, :] = 1000 * b + off
    n = len(table) * bs
    g = oracle.gather_sequence(cache, table, n)
    for t in range(n):
        assert g[t, 0, 0] == 1000 * table[t // bs] + t % bs
    # logical block 2 offset 5 -> physical table[2]
    assert oracle.slot_of(table, 2 * bs + 5, bs) == table[2] * bs + 5


def test_allocator_reproduces_golden_table():
    """A free list starting 7,2,9,4 yields the page's table for a 4-block request."""
    bs, table = _golden_tables()["pa"]
    order = table + [b for b in range(12) if b not in table]
    a = OracleAllocator(12, bs, order)
    s = a.seq_create()
    slots = a.append_tokens(s, 4 * bs)
    assert a.block_table(s) == table
    assert slots[37] == 9 * 16 + 5
    assert slots[0] == 7 * 16 and slots[16] == 2 * 16


# --------------------------------------------------------------------------
# attention: closed forms
# --------------------------------------------------------------------------
def _single_seq_cache(K, V, bs, NB=None, table=None):
    """Place contiguous K/V [T, Hkv, D] into a paged cache (table given)."""
    T, Hkv, D = K.shape
    nblk = -(-T // bs)
    NB = NB or nblk
    table = list(range(nblk)) if table is None else table
    kc = np.zeros((NB, Hkv, bs, D))
    vc = np.zeros_like(kc)
    for t in range(T):
        kc[table[t // bs], :, t % bs] = K[t]
        vc[table[t // bs], :, t % bs] = V[t]
    return kc, vc, np.asarray([table]), np.asarray([T])


def test_single_token_returns_its_value():
    rng = np.random.default_rng(2)
    K = rng.standard_normal((1, 2, 8))
    V = rng.standard_normal((1, 2, 8))
    q = rng.standard_normal((1, 4, 8))
    kc, vc, tab, lens = _single_seq_cache(K, V, 16)
    out = oracle.paged_decode(q, kc, vc, tab, lens, 0.3, 2)
    for h in range(4):
        assert np.array_equal(out[0, h], V[0, h // 2])


def test_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(3)
    T = 37
    K = np.tile(rng.standard_normal((1, 1, 16)), (T, 1, 1))
    V = rng.standard_normal((T, 1, 16))
    q = rng.standard_normal((1, 1, 16))
    kc, vc, tab, lens = _single_seq_cache(K, V, 8, NB=6, table=[5, 0, 3, 1, 4])
    out = oracle.paged_decode(q, kc, vc, tab, lens, 0.125, 1)
    np.testing.assert_allclose(out[0, 0], V[:, 0].mean(axis=0), rtol=0, atol=1e-13)


def test_two_token_softmax_weights():
    """Logits 0 and ln 3 -> weights 1/4, 3/4; pins scale, sign of exp, V order."""
    scale = 0.5
    K = np.zeros((2, 1, 2))
    K[1, 0, 0] = math.log(3.0) / scale
    V = np.array([[[4.0, -8.0]], [[12.0, 16.0]]])
    q = np.array([[[1.0, 7.0]]])
    kc, vc, tab, lens = _single_seq_cache(K, V, 1, NB=3, table=[2, 0])
    out = oracle.paged_decode(q, kc, vc, tab, lens, scale, 1)
    np.testing.assert_allclose(out[0, 0], [0.25 * 4 + 0.75 * 12, 0.25 * -8 + 0.75 * 16], atol=1e-13)


def test_dominant_logit_selects_its_value():
    rng = np.random.default_rng(4)
    T, D = 20, 8
    K = rng.standard_normal((T, 1, D)) * 0.1
    K[13, 0] = 50.0 * np.ones(D)
    V = rng.standard_normal((T, 1, D))
    q = np.ones((1, 1, D))
    kc, vc, tab, lens = _single_seq_cache(K, V, 4)
    out = oracle.paged_decode(q, kc, vc, tab, lens, 1.0, 1)
    np.testing.assert_allclose(out[0, 0], V[13, 0], atol=1e-12)


def test_gqa_groups_are_contiguous():
    """q heads 0,1 read kv head 0 and heads 2,3 read kv head 1 (H=4, Hkv=2)."""
    T = 9
    rng = np.random.default_rng(5)
    K = rng.standard_normal((T, 2, 4))
    V = np.zeros((T, 2, 4))
    V[:, 0] = 1.0
    V[:, 1] = 2.0
    q = rng.standard_normal((1, 4, 4))
    kc, vc, tab, lens = _single_seq_cache(K, V, 4)
    out = oracle.paged_decode(q, kc, vc, tab, lens, 0.7, 2)
    np.testing.assert_allclose(out[0, :, 0], [1.0, 1.0, 2.0, 2.0], atol=1e-14)


def test_zero_length_gives_zeros():
    kc = np.ones((2, 1, 4, 8))
    out = oracle.paged_decode(np.ones((1, 2, 8)), kc, kc, np.zeros((1, 1), int), [0], 1.0, 1)
    assert not out.any()


def test_high_precision_reference():
    """fp64 oracle agrees with 50-digit arithmetic on a small case."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    rng = np.random.default_rng(6)
    T, D = 23, 16
    K = rng.standard_normal((T, 1, D))
    V = rng.standard_normal((T, 1, D))
    q = rng.standard_normal((1, 1, D))
    scale = 0.25
    kc, vc, tab, lens = _single_seq_cache(K, V, 8, NB=5, table=[4, 1, 3])
    out = oracle.paged_decode(q, kc, vc, tab, lens, scale, 1)[0, 0]
    s = [mp.mpf(scale) * mp.fsum(mp.mpf(float(q[0, 0, d])) * mp.mpf(float(K[t, 0, d])) for d in range(D))
         for t in range(T)]
    m = max(s)
    w = [mp.e ** (x - m) for x in s]
    tot = mp.fsum(w)
    ref = [mp.fsum(w[t] * mp.mpf(float(V[t, 0, d])) for t in range(T)) / tot for d in range(D)]
    np.testing.assert_allclose(out, [float(r) for r in ref], rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# brute force and invariants on the seeded tiny workload
# --------------------------------------------------------------------------
def test_bruteforce_agrees_on_tiny():
    wl = W.tiny_fp32()
    _, tables, _, kc, vc = build_cache_with_allocator(wl)
    ref = oracle.paged_decode(wl.q.f32, kc, vc, tables, wl.context_lens, wl.scale, wl.num_kv_heads)
    bf = np.array(oracle.decode_bruteforce(wl.q.f32.tolist(), kc.tolist(), vc.tolist(),
                                           tables.tolist(), wl.context_lens.tolist(), wl.scale,
                                           wl.num_kv_heads))
    np.testing.assert_allclose(ref, bf, rtol=0, atol=1e-12)


def test_matches_contiguous_attention_on_unpaged_arrays():
    """Invariant (a): the table walk reproduces token order exactly."""
    wl = W.tiny_fp32()
    _, tables, _, kc, vc = build_cache_with_allocator(wl)
    ref = oracle.paged_decode(wl.q.f32, kc, vc, tables, wl.context_lens, wl.scale, wl.num_kv_heads)
    st = wl.seq_starts
    for i in range(wl.num_seqs):
        K = wl.key_hist.f32[st[i]:st[i + 1]]
        V = wl.value_hist.f32[st[i]:st[i + 1]]
        c = oracle.contiguous_attention(wl.q.f32[i], K, V, wl.scale)
        assert np.array_equal(ref[i], c)


def test_block_permutation_invariance():
    """Invariant (a): moving physical blocks and remapping tables changes nothing."""
    wl = W.tiny_fp32()
    _, tables, _, kc, vc = build_cache_with_allocator(wl)
    ref = oracle.paged_decode(wl.q.f32, kc, vc, tables, wl.context_lens, wl.scale, wl.num_kv_heads)
    rng = np.random.default_rng(7)
    for _ in range(3):
        perm = rng.permutation(wl.num_blocks)
        kc2 = np.empty_like(kc)
        vc2 = np.empty_like(vc)
        kc2[perm] = kc
        vc2[perm] = vc
        out = oracle.paged_decode(wl.q.f32, kc2, vc2, perm[tables], wl.context_lens, wl.scale,
                                  wl.num_kv_heads)
        assert np.array_equal(out, ref)


def test_shared_prefix_equals_private_copies():
    """Invariant (c): sequences sharing prefix blocks give the results of
    sequences holding private copies of the prefix."""
    rng = np.random.default_rng(8)
    bs, Hkv, H, D, P, tail, S = 16, 2, 4, 8, 45, 5, 3
    Kp = rng.standard_normal((P, Hkv, D))
    Vp = rng.standard_normal((P, Hkv, D))
    Kt = rng.standard_normal((S, tail, Hkv, D))
    Vt = rng.standard_normal((S, tail, Hkv, D))
    q = rng.standard_normal((S, H, D))
    outs = []
    for shared in (True, False):
        NB = 40
        a = OracleAllocator(NB, bs, rng.permutation(NB))
        kc = np.zeros((NB, Hkv, bs, D))
        vc = np.zeros_like(kc)
        seqs = []
        if shared:
            root = a.seq_create()
            oracle.reshape_and_cache(Kp, Vp, kc, vc, a.append_tokens(root, P))
            seqs = [a.fork(root) for _ in range(S)]
            a.free_seq(root)
        else:
            for _ in range(S):
                s = a.seq_create()
                oracle.reshape_and_cache(Kp, Vp, kc, vc, a.append_tokens(s, P))
                seqs.append(s)
        for j, s in enumerate(seqs):
            for t in range(tail):
                slot, src, dst = a.append_slot(s)
                if src >= 0:
                    oracle.copy_blocks(kc, vc, [(src, dst)])
                oracle.reshape_and_cache(Kt[j, t:t + 1], Vt[j, t:t + 1], kc, vc, [slot])
        tables = np.zeros((S, 4), dtype=np.int64)
        for j, s in enumerate(seqs):
            tb = a.block_table(s)
            tables[j, :len(tb)] = tb
        outs.append(oracle.paged_decode(q, kc, vc, tables, [P + tail] * S, 0.3, Hkv))
    assert np.array_equal(outs[0], outs[1])


# --------------------------------------------------------------------------
# prefill (causal): [PA] "KV Cache 为什么难管理" -- prefill runs the prompt's
# tokens together, each attending to its own position and earlier ones
# --------------------------------------------------------------------------
def _prefill_case(rng, lens, starts, H=4, Hkv=2, D=8, bs=4, NB=40):
    kc = rng.standard_normal((NB, Hkv, bs, D))
    vc = rng.standard_normal((NB, Hkv, bs, D))
    perm = rng.permutation(NB)
    maxb = max(-(-(s + n) // bs) for s, n in zip(starts, lens))
    tables = np.zeros((len(lens), maxb), dtype=np.int64)
    k = 0
    for i, (s, n) in enumerate(zip(starts, lens)):
        nb = -(-(s + n) // bs)
        tables[i, :nb] = perm[k:k + nb]
        k += nb
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    q = rng.standard_normal((int(cu[-1]), H, D))
    return q, kc, vc, tables, cu, np.asarray(starts), Hkv


def test_prefill_first_token_returns_its_value():
    rng = np.random.default_rng(31)
    q, kc, vc, tables, cu, st, Hkv = _prefill_case(rng, [5], [0])
    out = oracle.paged_prefill(q, kc, vc, tables, cu, st, 0.7, Hkv)
    v0 = vc[tables[0, 0], :, 0, :]
    G = q.shape[1] // Hkv
    for h in range(q.shape[1]):
        assert np.allclose(out[0, h], v0[h // G], atol=1e-15)


def test_prefill_is_causal_and_last_row_is_decode():
    rng = np.random.default_rng(32)
    q, kc, vc, tables, cu, st, Hkv = _prefill_case(rng, [9], [0])
    out = oracle.paged_prefill(q, kc, vc, tables, cu, st, 0.5, Hkv)
    # later keys do not change earlier rows: overwrite positions 5.. and recompute
    kc2, vc2 = kc.copy(), vc.copy()
    bs = kc.shape[2]
    for t in range(5, 9):
        kc2[tables[0, t // bs], :, t % bs] += 3.0
        vc2[tables[0, t // bs], :, t % bs] -= 2.0
    out2 = oracle.paged_prefill(q, kc2, vc2, tables, cu, st, 0.5, Hkv)
    assert np.array_equal(out[:5], out2[:5]) and not np.allclose(out[5:], out2[5:])
    # the last token of the prompt is a decode step over the whole prompt
    dec = oracle.paged_decode(q[8:9], kc, vc, tables, [9], 0.5, Hkv)
    assert np.allclose(out[8], dec[0], atol=1e-13)


def test_chunked_prefill_equals_whole_prompt():
    """A prompt split into chunks (later starts) gives the rows of one call."""
    rng = np.random.default_rng(33)
    q, kc, vc, tables, cu, st, Hkv = _prefill_case(rng, [13], [0])
    whole = oracle.paged_prefill(q, kc, vc, tables, cu, st, 0.6, Hkv)
    parts = oracle.paged_prefill(q, kc, vc, np.repeat(tables, 3, axis=0), [0, 4, 9, 13], [0, 4, 9], 0.6, Hkv)
    assert np.allclose(whole, parts, atol=1e-14)


def test_prefill_bruteforce_on_tiny():
    rng = np.random.default_rng(34)
    q, kc, vc, tables, cu, st, Hkv = _prefill_case(rng, [3, 2], [0, 5], H=2, Hkv=1, D=3, bs=2, NB=12)
    out = oracle.paged_prefill(q, kc, vc, tables, cu, st, 0.9, Hkv)
    import math
    for i in range(2):
        for j in range(int(cu[i + 1] - cu[i])):
            p = int(st[i]) + j
            for h in range(2):
                s = [0.9 * sum(q[cu[i] + j, h, d] * kc[tables[i, t // 2], 0, t % 2, d] for d in range(3))
                     for t in range(p + 1)]
                m = max(s)
                w = [math.exp(x - m) for x in s]
                for d in range(3):
                    ref = sum(w[t] * vc[tables[i, t // 2], 0, t % 2, d] for t in range(p + 1)) / sum(w)
                    assert abs(out[cu[i] + j, h, d] - ref) < 1e-12


# --------------------------------------------------------------------------
# slot write and block copy
# --------------------------------------------------------------------------
def test_reshape_and_cache_positions_and_skip():
    NB, Hkv, bs, D = 6, 2, 4, 3
    kc = np.zeros((NB, Hkv, bs, D))
    vc = np.zeros_like(kc)
    key = np.arange(1, 4)[:, None, None] * np.ones((3, Hkv, D))
    val = -key
    oracle.reshape_and_cache(key, val, kc, vc, [4 * 5 + 2, -1, 1 * 4 + 3])
    assert (kc[5, :, 2] == 1).all() and (vc[5, :, 2] == -1).all()
    assert (kc[1, :, 3] == 3).all()
    assert np.count_nonzero(kc) == 2 * Hkv * D  # token 1 skipped
    with pytest.raises(ValueError):
        oracle.reshape_and_cache(key[:1], val[:1], kc, vc, [NB * bs])


def test_copy_blocks_uses_pre_call_state():
    rng = np.random.default_rng(9)
    kc = rng.standard_normal((6, 2, 4, 3))
    vc = rng.standard_normal((6, 2, 4, 3))
    k0, v0 = kc.copy(), vc.copy()
    oracle.copy_blocks(kc, vc, [(1, 4), (3, 0)])
    assert np.array_equal(kc[4], k0[1]) and np.array_equal(vc[0], v0[3])
    for b in (1, 2, 3, 5):
        assert np.array_equal(kc[b], k0[b]) and np.array_equal(vc[b], v0[b])
    with pytest.raises(ValueError):
        oracle.copy_blocks(kc, vc, [(1, 2), (2, 3)])  # 2 is both a destination and a source
    with pytest.raises(ValueError):
        oracle.copy_blocks(kc, vc, [(1, 2), (3, 2)])  # repeated destination


def test_layered_append_writes_m_token_elements_per_token():
    """[PA] "KV Cache 为什么难管理": one token's cache is M_token = 2*L*H_kv*d
    elements; every layer receives its own K/V at the same slot."""
    Lyr, NB, Hkv, bs, D = 3, 5, 2, 4, 3
    kc = np.zeros((Lyr, NB, Hkv, bs, D))
    vc = np.zeros_like(kc)
    T = 3
    # key[l, t] = 100*(l+1) + (t+1), value = its negative
    key = (100 * np.arange(1, Lyr + 1)[:, None, None, None] + np.arange(1, T + 1)[None, :, None, None]
           ) * np.ones((Lyr, T, Hkv, D))
    val = -key
    slots = [2 * bs + 1, -1, 4 * bs + 3]
    oracle.reshape_and_cache_layers(key, val, kc, vc, slots)
    written = 2  # token 1 is padding
    assert np.count_nonzero(kc) + np.count_nonzero(vc) == written * 2 * Lyr * Hkv * D
    for layer in range(Lyr):
        assert (kc[layer, 2, :, 1] == 100 * (layer + 1) + 1).all()
        assert (vc[layer, 4, :, 3] == -(100 * (layer + 1) + 3)).all()
    with pytest.raises(ValueError):
        oracle.reshape_and_cache_layers(key[:2], val[:2], kc, vc, slots)  # layer count mismatch


def test_layered_copy_copies_each_layer_from_its_own_source():
    rng = np.random.default_rng(11)
    kc = rng.standard_normal((4, 6, 2, 4, 3))
    vc = rng.standard_normal((4, 6, 2, 4, 3))
    k0, v0 = kc.copy(), vc.copy()
    oracle.copy_blocks_layers(kc, vc, [(1, 4), (3, 0)])
    for layer in range(4):
        assert np.array_equal(kc[layer, 4], k0[layer, 1]) and np.array_equal(vc[layer, 0], v0[layer, 3])
        for b in (1, 2, 3, 5):
            assert np.array_equal(kc[layer, b], k0[layer, b]) and np.array_equal(vc[layer, b], v0[layer, b])
    assert not np.array_equal(kc[0, 4], kc[1, 4])  # layers stay distinct


# --------------------------------------------------------------------------
# allocator: refcounts, fork, copy-on-write, shared-prefix scenario
# --------------------------------------------------------------------------
def _conservation(a: OracleAllocator):
    held = {}
    for s in a.live_seqs():
        for b in a.block_table(s):
            held[b] = held.get(b, 0) + 1
    for b in range(a.num_blocks):
        assert a.refcount(b) == held.get(b, 0)
    assert a.num_free() + len(held) == a.num_blocks
    assert sorted(a.free) == sorted(set(range(a.num_blocks)) - set(held))


@pytest.mark.parametrize("bs,blocks,last_fill,cows", [(16, 188, 8, 63), (8, 375, 8, 0), (32, 94, 24, 63)])
def test_shared_prefix_cow_scenario(bs, blocks, last_fill, cows):
    """3000-token prompt forked to 64 beams: the first append of each beam
    copies a shared, partly filled last block except for the last holder."""
    NB = blocks + 64 * 3
    a = OracleAllocator(NB, bs)
    root = a.seq_create()
    a.append_tokens(root, 3000)
    assert len(a.block_table(root)) == blocks
    assert 3000 - (blocks - 1) * bs == last_fill
    beams = [a.fork(root) for _ in range(64)]
    a.free_seq(root)
    assert all(a.refcount(b) == 64 for b in a.block_table(beams[0]))
    pairs = []
    for s in beams:
        _, src, dst = a.append_slot(s)
        if src >= 0:
            pairs.append((src, dst))
    assert len(pairs) == cows
    if cows:
        last = a.block_table(beams[-1])[-1]
        assert all(p[0] == last for p in pairs)  # every copy is of the shared tail
        assert a.refcount(last) == 1
    _conservation(a)


def test_fork_cow_keeps_parent_tables():
    a = OracleAllocator(10, 4, [3, 1, 4, 0, 5, 9, 2, 6, 8, 7])
    p = a.seq_create()
    a.append_tokens(p, 6)           # blocks 3, 1 ; block 1 half full
    c = a.fork(p)
    slot, src, dst = a.append_slot(c)
    assert (src, dst) == (1, 4) and slot == 4 * 4 + 2
    assert a.block_table(p) == [3, 1] and a.block_table(c) == [3, 4]
    slot, src, dst = a.append_slot(p)   # parent is now sole holder of block 1
    assert (src, dst) == (-1, -1) and slot == 1 * 4 + 2
    _conservation(a)
    a.free_seq(c)
    assert list(a.free)[-1] == 4 and a.refcount(3) == 1
    _conservation(a)


def test_oom_leaves_state_unchanged():
    a = OracleAllocator(2, 4)
    s = a.seq_create()
    a.append_tokens(s, 8)
    before = a.snapshot()
    with pytest.raises(AllocatorOOM):
        a.append_slot(s)
    assert a.snapshot() == before
    c = a.fork(s)
    a.free_seq(s)
    before = a.snapshot()
    # c's last block is full, so its next token needs a fresh block: OOM again
    with pytest.raises(AllocatorOOM):
        a.append_slot(c)
    assert a.snapshot() == before


def test_free_returns_blocks_fifo_in_table_order():
    a = OracleAllocator(6, 2, [5, 4, 3, 2, 1, 0])
    s1 = a.seq_create()
    a.append_tokens(s1, 5)          # 5, 4, 3
    s2 = a.seq_create()
    a.append_tokens(s2, 2)          # 2
    a.free_seq(s1)
    assert list(a.free) == [1, 0, 5, 4, 3]
    assert a.allocate() == 1
    a.decref(1)                     # a raw allocation released goes to the back
    assert list(a.free) == [0, 5, 4, 3, 1]
    _conservation(a)


def test_random_ops_keep_invariants():
    rng = np.random.default_rng(10)
    a = OracleAllocator(64, 4, rng.permutation(64))
    for _ in range(2000):
        live = a.live_seqs()
        op = rng.integers(0, 4)
        try:
            if op == 0 or not live:
                a.seq_create()
            elif op == 1:
                a.append_slot(int(rng.choice(live)))
            elif op == 2:
                a.fork(int(rng.choice(live)))
            else:
                a.free_seq(int(rng.choice(live)))
        except AllocatorOOM:
            pass
        _conservation(a)
        for s in a.live_seqs():
            assert len(a.block_table(s)) == oracle.blocks_for(a.seq_len(s), 4)
