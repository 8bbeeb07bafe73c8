"""GPU paged decode attention against the fp64 oracle."""
import numpy as np
import pytest
import torch

from paged_kv_cache_142_gb300 import workloads as W
from paged_case import (GpuState, OracleState, TOL, bf16_half_ulp, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops(lib):
    import importlib
    return importlib.import_module("paged_kv_cache_142_gb300.ops")


def max_err(out: torch.Tensor, ref: np.ndarray, rows=None) -> float:
    got = to_f64(out)
    if rows is not None:
        got = got[rows]
    return float(np.abs(got - ref).max())


@pytest.mark.parametrize("partition_tokens", [0, 32])
def test_tiny_fp32(ops, partition_tokens):
    wl = W.tiny_fp32()
    g = GpuState(wl, ops)
    ref = OracleState(wl).decode()
    out = g.decode(partition_tokens=partition_tokens)
    assert max_err(out, ref) <= TOL["f32"]


def test_mha_bf16_all_sequences(ops):
    wl = W.mha_bf16()
    g = GpuState(wl, ops)
    ref = OracleState(wl).decode()
    assert max_err(g.decode(), ref) <= TOL["bf16"]


@pytest.fixture(scope="module")
def gqa_full():
    """The batch-256 workload and the oracle's output for all of its sequences."""
    wl = W.gqa_bf16()
    return wl, OracleState(wl).decode()


def test_gqa_bf16_batch256_all_sequences(ops, gqa_full):
    """Every row of the benchmark batch (256 sequences x 32 heads x 128) in
    the bench's launch configuration (automatic partitions)."""
    wl, ref = gqa_full
    g = GpuState(wl, ops)
    out = g.decode()
    assert torch.isfinite(out).all()
    assert max_err(out, ref) <= TOL["bf16"]
    # bf16 output: the kernel's error plus the final rounding
    got = to_f64(g.decode(out_dtype=torch.bfloat16))
    assert (np.abs(got - ref) <= TOL["bf16"] + bf16_half_ulp(ref)).all()


@pytest.mark.parametrize("bs", [16, 32])
def test_long_context_split_k_all_sequences(ops, bs):
    """All 8 sequences of 32768 tokens, automatic and 1024-token partitions."""
    wl = W.long_bf16(block_size=bs)
    g = GpuState(wl, ops)
    ref = OracleState(wl).decode()
    for pt in (0, 1024):
        out = g.decode(partition_tokens=pt)
        assert torch.isfinite(out).all()
        assert max_err(out, ref) <= TOL["bf16"]


@pytest.fixture
def kv_per_item(ops, request):
    """Plans under the given work-item shape, automatic again afterwards."""
    ops.pa_set_decode_kv_per_item(request.param)
    yield request.param
    ops.pa_set_decode_kv_per_item(0)


EDGE_LENS = [0, 1, 7, 8, 15, 16, 17, 31, 32, 33, 63, 64, 65, 255, 256, 257, 511, 600, 1000]


@pytest.mark.parametrize("dtype,D,G,bs", [
    ("f32", 64, 1, 16), ("f32", 64, 4, 8), ("f32", 128, 2, 32), ("f32", 128, 8, 16),
    ("bf16", 64, 8, 16), ("bf16", 64, 1, 1), ("bf16", 128, 1, 16), ("bf16", 128, 2, 8),
    ("bf16", 128, 4, 16), ("bf16", 128, 8, 32), ("bf16", 256, 4, 16), ("bf16", 256, 8, 64),
    ("bf16", 128, 16, 16), ("bf16", 128, 4, 256),
    # two kv heads per item with blocks of 32 and 64 tokens (a warp's rows all
    # belong to one kv head there)
    ("bf16", 128, 4, 32), ("bf16", 128, 2, 64), ("bf16", 128, 1, 64),
])
@pytest.mark.parametrize("partition_tokens", [0, 64])
@pytest.mark.parametrize("kv_per_item", [0, 1, 2], indirect=True)
def test_shape_sweep_edge_lengths(ops, dtype, D, G, bs, partition_tokens, kv_per_item):
    """Edge lengths over dtype x head_dim x G x block size; each case with the
    automatic work-item shape and with one and two kv heads per item forced
    (two only where the shape allows it)."""
    Hkv = 2
    wl = W.custom(f"sweep_{dtype}_{D}_{G}_{bs}", dtype, EDGE_LENS, G * Hkv, Hkv, D, bs,
                  pool_factor=1.3, seed=D * 10 + G + bs)
    g = GpuState(wl, ops)
    ref = OracleState(wl).decode()
    out = g.decode(partition_tokens=partition_tokens)
    assert max_err(out, ref) <= TOL[dtype]
    assert not to_f64(out)[0].any()  # the empty sequence gives zeros


@pytest.mark.parametrize("kv_per_item", [1, 2], indirect=True)
def test_block_permutation_invariance_bit_identical(ops, kv_per_item):
    """Other physical placement, same logical content: identical bits."""
    base = W.gqa_bf16(num_seqs=32)
    outs = []
    for seed in (1, 2, 3):
        wl = W.gqa_bf16(num_seqs=32)
        wl.free_order = np.random.default_rng(seed).permutation(wl.num_blocks).astype(np.int32)
        outs.append(GpuState(wl, ops).decode(partition_tokens=128))
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    del base


def test_repeatable_and_workspace_reuse(ops):
    wl = W.long_bf16(num_seqs=2, context_len=5000)
    g = GpuState(wl, ops)
    ws = ops.make_workspace(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                            wl.block_size, wl.dtype, g.max_len, 256)
    first = g.decode(partition_tokens=256, workspace=ws)
    for _ in range(3):
        assert torch.equal(g.decode(partition_tokens=256, workspace=ws), first)
    # the bookkeeping words are back to zero after every call
    pt, _ = ops.pa_decode_plan(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                               wl.block_size, wl.dtype, g.max_len, 256)
    assert pt == 256
    assert int(ws[:256 + 4 * wl.num_seqs * wl.num_kv_heads].sum()) == 0


def test_device_checks_report_bad_lengths_and_tables(ops):
    wl = W.custom("bad", "bf16", [40, 20], 8, 2, 128, 16, seed=5)
    g = GpuState(wl, ops)
    ws = ops.make_workspace(2, 8, 2, 128, 16, "bf16", 40)
    out = torch.empty_like(g.q, dtype=torch.float32)
    # a context length above max_context_len is clamped and reported
    lens = torch.tensor([40, 30], dtype=torch.int32, device="cuda")
    ops.pa_decode(out, g.q, g.k_cache, g.v_cache, g.tables, lens, wl.scale, 2, 25, ws)
    assert ops.pa_workspace_error(ws) == 1
    # a block id outside the pool is never read and is reported
    tables = g.tables.clone()
    tables[1, 0] = wl.num_blocks + 5
    ops.pa_decode(out, g.q, g.k_cache, g.v_cache, tables, g.lens, wl.scale, 2, 40, ws)
    assert ops.pa_workspace_error(ws) == 1
    # and a clean call reports nothing
    ops.pa_decode(out, g.q, g.k_cache, g.v_cache, g.tables, g.lens, wl.scale, 2, 40, ws)
    assert ops.pa_workspace_error(ws) == 0


def test_workspace_too_small_is_rejected(ops):
    wl = W.custom("ws", "bf16", [600, 20], 8, 2, 128, 16, seed=6)
    g = GpuState(wl, ops)
    need = ops.pa_decode_workspace_size(2, 8, 2, 128, 16, "bf16", 600, 64)
    ws = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(g.q, dtype=torch.float32)
    with pytest.raises(ops.PAError) as e:
        ops.pa_decode(out, g.q, g.k_cache, g.v_cache, g.tables, g.lens, wl.scale, 2, 600, ws,
                      partition_tokens=64)
    assert e.value.status == 5


@pytest.mark.parametrize("partition_tokens", [0, 512, 2048])
def test_batch256_repeated_calls_bit_identical(ops, gqa_full, partition_tokens):
    """Repeated decodes of the batch-256 workload on one reused workspace give
    identical bits (the split-K merge order and every tile's arithmetic are
    fixed by logical position), and agree with the oracle on every row."""
    wl, ref = gqa_full
    g = GpuState(wl, ops)
    ws = ops.make_workspace(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                            wl.block_size, wl.dtype, g.max_len, partition_tokens)
    first = g.decode(partition_tokens=partition_tokens, workspace=ws)
    for _ in range(12):
        assert torch.equal(g.decode(partition_tokens=partition_tokens, workspace=ws), first)
    assert max_err(first, ref) <= TOL["bf16"]


def test_odd_kv_head_count_keeps_one_head_per_item(ops):
    """Three kv heads cannot pair up: the tensor-core kernel runs one kv head
    per item, and the result still matches the oracle."""
    wl = W.custom("odd_kv", "bf16", [0, 1, 17, 200, 777, 1500], 6, 3, 128, 16, seed=31)
    g = GpuState(wl, ops)
    ref = OracleState(wl).decode()
    for pt in (0, 64):
        assert max_err(g.decode(partition_tokens=pt), ref) <= TOL["bf16"]
