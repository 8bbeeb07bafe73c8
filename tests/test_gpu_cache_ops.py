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
