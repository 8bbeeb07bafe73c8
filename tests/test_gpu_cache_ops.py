"""GPU slot write and block copy against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_142_gb300 import workloads as W
from paged_case import GpuState, OracleState, cache_bits, raw_bits, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops(lib):
    import importlib
    return importlib.import_module("paged_kv_cache_142_gb300.ops")


@pytest.mark.parametrize("make", [W.tiny_fp32, W.mha_bf16, W.gqa_bf16])
def test_prefill_slot_write_bit_exact(ops, make):
    wl = make()
    g = GpuState(wl, ops)
    o = OracleState(wl, bits=True)
    assert np.array_equal(g.slots, o.slots)
    assert np.array_equal(cache_bits(g.k_cache), o.k_cache)
    assert np.array_equal(cache_bits(g.v_cache), o.v_cache)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_slot_write_skips_padding_and_out_of_range(ops, dtype):
    NB, Hkv, bs, D, T = 6, 2, 8, 64, 7
    rng = np.random.default_rng(3)
    key = W.Values.from_f32(rng.standard_normal((T, Hkv, D)).astype(np.float32), dtype)
    val = W.Values.from_f32(rng.standard_normal((T, Hkv, D)).astype(np.float32), dtype)
    slots = np.array([5, -1, NB * bs, 17, -7, NB * bs + 3, 40], dtype=np.int64)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    kc = torch.zeros((NB, Hkv, bs, D), dtype=dt, device="cuda")
    vc = torch.zeros_like(kc)
    ops.pa_reshape_and_cache(to_device(key), to_device(val), torch.from_numpy(slots).cuda(), kc, vc)
    kb, vb = raw_bits(key.bits), raw_bits(val.bits)
    ek = np.zeros((NB, Hkv, bs, D), dtype=kb.dtype)
    ev = np.zeros_like(ek)
    keep = (slots >= 0) & (slots < NB * bs)
    oracle.reshape_and_cache(kb[keep], vb[keep], ek, ev, slots[keep])
    assert np.array_equal(cache_bits(kc), ek)
    assert np.array_equal(cache_bits(vc), ev)


@pytest.mark.parametrize("dtype,bs,Hkv,D", [("bf16", 16, 8, 128), ("bf16", 8, 8, 128),
                                            ("bf16", 32, 8, 128), ("f32", 16, 4, 64)])
def test_copy_blocks_bit_exact(ops, dtype, bs, Hkv, D):
    NB = 40
    rng = np.random.default_rng(11)
    k = W.Values.from_f32(rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32), dtype)
    v = W.Values.from_f32(rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32), dtype)
    perm = rng.permutation(NB)
    pairs = np.stack([perm[:9], perm[9:18]], axis=1).astype(np.int64)  # disjoint src/dst
    kc = to_device(k).contiguous()
    vc = to_device(v).contiguous()
    ops.pa_copy_blocks(kc, vc, torch.from_numpy(pairs).cuda())
    ek, ev = raw_bits(k.bits).copy(), raw_bits(v.bits).copy()
    oracle.copy_blocks(ek, ev, pairs)
    assert np.array_equal(cache_bits(kc), ek)
    assert np.array_equal(cache_bits(vc), ev)


def test_copy_blocks_skips_out_of_range_and_empty(ops):
    NB, Hkv, bs, D = 8, 2, 16, 64
    kc = torch.arange(NB * Hkv * bs * D, dtype=torch.float32, device="cuda").reshape(NB, Hkv, bs, D)
    vc = -kc
    k0, v0 = kc.clone(), vc.clone()
    ops.pa_copy_blocks(kc, vc, torch.empty((0, 2), dtype=torch.int64, device="cuda"))
    pairs = torch.tensor([[1, NB], [-1, 2], [3, 4]], dtype=torch.int64, device="cuda")
    ops.pa_copy_blocks(kc, vc, pairs)
    torch.cuda.synchronize()
    k0[4] = k0[3]
    v0[4] = v0[3]
    assert torch.equal(kc, k0) and torch.equal(vc, v0)


@pytest.mark.parametrize("dtype,Lyr,bs,Hkv,D", [("bf16", 4, 16, 8, 128), ("bf16", 3, 8, 2, 64),
                                                ("f32", 2, 16, 4, 64), ("bf16", 1, 16, 8, 128)])
def test_layered_append_and_copy_bit_exact(ops, dtype, Lyr, bs, Hkv, D):
    """All layers in one launch, against the oracle applied layer by layer;
    the caches live in one pool with a padded layer stride."""
    NB, T = 24, 13
    rng = np.random.default_rng(100 + Lyr * bs + D)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    cache0 = W.Values.from_f32(rng.standard_normal((Lyr, NB, Hkv, bs, D)).astype(np.float32), dtype)
    key = W.Values.from_f32(rng.standard_normal((Lyr, T, Hkv, D)).astype(np.float32), dtype)
    val = W.Values.from_f32(rng.standard_normal((Lyr, T, Hkv, D)).astype(np.float32), dtype)
    # pool with one spare block of padding per layer: layer stride > one layer's elements
    pool_k = torch.zeros((Lyr, NB + 1, Hkv, bs, D), dtype=dt, device="cuda")
    pool_v = torch.zeros_like(pool_k)
    kc, vc = pool_k[:, :NB], pool_v[:, :NB]
    kc.copy_(to_device(cache0))
    vc.copy_(-to_device(cache0))
    perm = rng.permutation(NB * bs)
    slots = np.concatenate([perm[:T - 2], [-1, NB * bs + 5]]).astype(np.int64)
    ops.pa_reshape_and_cache_layers(to_device(key), to_device(val), torch.from_numpy(slots).cuda(), kc, vc)
    bperm = rng.permutation(NB)
    pairs = np.stack([bperm[:5], bperm[5:10]], axis=1).astype(np.int64)
    ops.pa_copy_blocks_layers(kc, vc, torch.from_numpy(pairs).cuda())
    ek = raw_bits(cache0.bits).copy()
    ev = raw_bits(cache_bits(-to_device(cache0)))
    keep = (slots >= 0) & (slots < NB * bs)
    oracle.reshape_and_cache_layers(raw_bits(key.bits)[:, keep], raw_bits(val.bits)[:, keep], ek, ev,
                                    slots[keep])
    oracle.copy_blocks_layers(ek, ev, pairs)
    torch.cuda.synchronize()
    assert np.array_equal(cache_bits(kc.contiguous()), ek)
    assert np.array_equal(cache_bits(vc.contiguous()), ev)
    assert not pool_k[:, NB].any() and not pool_v[:, NB].any()  # padding untouched


def test_layered_calls_equal_per_layer_calls(ops):
    Lyr, NB, Hkv, bs, D, T = 5, 16, 8, 16, 128, 32
    g = torch.Generator(device="cuda").manual_seed(5)
    key = torch.randn((Lyr, T, Hkv, D), device="cuda", generator=g).to(torch.bfloat16)
    val = torch.randn((Lyr, T, Hkv, D), device="cuda", generator=g).to(torch.bfloat16)
    slots = torch.randperm(NB * bs, device="cuda", generator=g)[:T].to(torch.int64)
    a_k = torch.zeros((Lyr, NB, Hkv, bs, D), dtype=torch.bfloat16, device="cuda")
    a_v = torch.zeros_like(a_k)
    b_k, b_v = a_k.clone(), a_v.clone()
    ops.pa_reshape_and_cache_layers(key, val, slots, a_k, a_v)
    for layer in range(Lyr):
        ops.pa_reshape_and_cache(key[layer], val[layer], slots, b_k[layer], b_v[layer])
    torch.cuda.synchronize()
    assert torch.equal(a_k, b_k) and torch.equal(a_v, b_v)


def test_layered_argument_errors(ops):
    from paged_kv_cache_142_gb300 import _lib as L
    lib = L.load()
    # layer stride shorter than a layer, or not a multiple of 16 bytes
    assert lib.pa_reshape_and_cache_layers(1, 1, 10, 2, 4, 1, 16, 16, 16 * 2 * 16 * 64, 16, 16, 2, 64, 1,
                                           None) == L.PA_ERR_INVALID_ARG
    assert lib.pa_copy_blocks_layers(16, 16, 16 * 2 * 16 * 64 + 1, 2, 16, 16, 2, 64, 1, 16, 1,
                                     None) == L.PA_ERR_INVALID_ARG
    assert lib.pa_copy_blocks_layers(16, 16, 0, 0, 16, 16, 2, 64, 1, 16, 1, None) == L.PA_ERR_INVALID_ARG


# ---------------------------------------------------------------------------
# checked mode: a device status word instead of silent skips
# ---------------------------------------------------------------------------
def _oracle_raises(fn, *args) -> bool:
    try:
        fn(*args)
    except ValueError:
        return True
    return False


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("bad", [False, True])
def test_checked_append_reports_slots_past_the_pool(ops, dtype, bad):
    """The oracle raises on a slot past the pool; the checked append reports
    it in the status word, writes no such slot, and writes every other token
    bit-exactly (padding skipped)."""
    NB, Hkv, bs, D, T = 6, 2, 8, 64, 9
    rng = np.random.default_rng(5 + bad)
    key = W.Values.from_f32(rng.standard_normal((T, Hkv, D)).astype(np.float32), dtype)
    val = W.Values.from_f32(rng.standard_normal((T, Hkv, D)).astype(np.float32), dtype)
    slots = np.array([5, -1, 17, 47, 0, -3, 40, 9, 33], dtype=np.int64)
    if bad:
        slots[[2, 6]] = [NB * bs, NB * bs + 11]
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    kc = torch.zeros((NB, Hkv, bs, D), dtype=dt, device="cuda")
    vc = torch.zeros_like(kc)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.pa_reshape_and_cache(to_device(key), to_device(val), torch.from_numpy(slots).cuda(), kc, vc,
                             status=status)
    kb, vb = raw_bits(key.bits), raw_bits(val.bits)
    ek = np.zeros((NB, Hkv, bs, D), dtype=kb.dtype)
    ev = np.zeros_like(ek)
    raised = _oracle_raises(oracle.reshape_and_cache, kb, vb, ek.copy(), ev.copy(), slots)
    assert int(status.item()) == (1 if raised else 0)
    assert raised == bad
    keep = slots < NB * bs
    oracle.reshape_and_cache(kb[keep], vb[keep], ek, ev, slots[keep])
    assert np.array_equal(cache_bits(kc), ek)
    assert np.array_equal(cache_bits(vc), ev)


def _invalid_pair_sets(NB, rng):
    perm = rng.permutation(NB)
    good = np.stack([perm[:12], perm[12:24]], axis=1).astype(np.int64)
    out = {}
    dup = good.copy()
    dup[7, 1] = dup[2, 1]                 # one destination named twice
    out["duplicate destination"] = dup
    src = good.copy()
    src[4, 1] = src[9, 0]                 # a destination that is another pair's source
    out["destination is a source"] = src
    self_ = good.copy()
    self_[0, 1] = self_[0, 0]             # a block copied onto itself
    out["self copy"] = self_
    rng_ = good.copy()
    rng_[11, 0] = NB                      # a source outside the pool
    out["source outside the pool"] = rng_
    neg = good.copy()
    neg[3, 1] = -1                        # a destination outside the pool
    out["negative destination"] = neg
    return good, out


@pytest.mark.parametrize("dtype,bs,Hkv,D", [("bf16", 16, 8, 128), ("f32", 8, 2, 64)])
def test_checked_copy_validates_before_copying(ops, dtype, bs, Hkv, D):
    """Valid pairs: status stays 0 and the copy is bit-exact.  Each invalid
    set (the oracle raises ValueError before copying anything): status 1 and
    no block changes."""
    NB = 48
    rng = np.random.default_rng(21)
    k = W.Values.from_f32(rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32), dtype)
    v = W.Values.from_f32(rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32), dtype)
    good, bad_sets = _invalid_pair_sets(NB, rng)
    for name, pairs in [("valid", good)] + list(bad_sets.items()):
        kc = to_device(k).contiguous()
        vc = to_device(v).contiguous()
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        ops.pa_copy_blocks(kc, vc, torch.from_numpy(pairs).cuda(), status=status)
        ek, ev = raw_bits(k.bits).copy(), raw_bits(v.bits).copy()
        raised = _oracle_raises(oracle.copy_blocks, ek, ev, pairs)
        assert raised == (name != "valid"), name
        assert int(status.item()) == (1 if raised else 0), name
        assert np.array_equal(cache_bits(kc), ek), name   # unchanged when the oracle raised
        assert np.array_equal(cache_bits(vc), ev), name


def test_checked_copy_many_pairs_and_sticky_status(ops):
    """Several hundred pairs (the validation spans several tiles of pairs):
    a duplicate between the first and the last tile is found; a status left
    non-zero suppresses a later checked copy; empty pair lists do nothing."""
    NB, Hkv, bs, D = 1400, 2, 8, 64
    rng = np.random.default_rng(8)
    kc = torch.randn((NB, Hkv, bs, D), device="cuda")
    vc = torch.randn((NB, Hkv, bs, D), device="cuda")
    perm = rng.permutation(NB)
    n = 650
    pairs = np.stack([perm[:n], perm[n:2 * n]], axis=1).astype(np.int64)
    k0, v0 = kc.clone(), vc.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.pa_copy_blocks(kc, vc, torch.from_numpy(pairs).cuda(), status=status)
    assert int(status.item()) == 0
    ek, ev = k0.cpu().numpy(), v0.cpu().numpy()
    oracle.copy_blocks(ek, ev, pairs)
    assert np.array_equal(kc.cpu().numpy(), ek) and np.array_equal(vc.cpu().numpy(), ev)
    bad = pairs.copy()
    bad[n - 1, 1] = bad[1, 1]
    k1, v1 = kc.clone(), vc.clone()
    ops.pa_copy_blocks(kc, vc, torch.from_numpy(bad).cuda(), status=status)
    assert int(status.item()) == 1
    assert torch.equal(kc, k1) and torch.equal(vc, v1)
    # the status is still 1: a valid checked copy is suppressed too
    ops.pa_copy_blocks(kc, vc, torch.from_numpy(pairs[:5].copy()).cuda(), status=status)
    assert int(status.item()) == 1 and torch.equal(kc, k1)
    status.zero_()
    ops.pa_copy_blocks(kc, vc, torch.empty((0, 2), dtype=torch.int64, device="cuda"), status=status)
    assert int(status.item()) == 0 and torch.equal(kc, k1)
