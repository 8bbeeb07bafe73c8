"""pa_decode_no_alloc: the decode entry point for callers that cannot
allocate device memory (it uses the library's fixed device scratch array
instead of a caller workspace).  Its output must match pa_decode's, on two
calls in a row, since the shared scratch keeps the previous call's contents.
Collected last on purpose."""
import pytest
import torch

from paged_kv_cache_142_gb300 import workloads as W
from paged_case import GpuState, TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops(lib):
    import importlib
    return importlib.import_module("paged_kv_cache_142_gb300.ops")


def _no_alloc(ops, g, partition_tokens=0):
    wl = g.wl
    out = torch.empty(g.q.shape, dtype=torch.float32, device=g.q.device)
    ops.pa_decode_no_alloc(out, g.q, g.k_cache, g.v_cache, g.tables, g.lens, wl.scale,
                           wl.num_kv_heads, g.max_len, partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("make", [
    lambda: W.long_bf16(num_seqs=3, context_len=7000),   # split, fits directly
    lambda: W.gqa_bf16(),                                 # needs larger partitions to fit
    W.tiny_fp32,
])
def test_no_alloc_matches_workspace_decode_twice(ops, make):
    wl = make()
    g = GpuState(wl, ops)
    ref = g.decode()
    tol = TOL[wl.dtype]
    for _ in range(2):
        out = _no_alloc(ops, g)
        assert float((out.double() - ref.double()).abs().max()) <= tol


def test_no_alloc_rejects_a_fixed_partition_that_does_not_fit(ops):
    wl = W.gqa_bf16()
    g = GpuState(wl, ops)
    need = ops.pa_decode_workspace_size(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                        wl.block_size, wl.dtype, g.max_len, 32)
    assert need > 32 << 20
    with pytest.raises(ops.PAError) as e:
        _no_alloc(ops, g, partition_tokens=32)
    assert e.value.status == 5  # PA_ERR_WORKSPACE


def test_no_alloc_reports_device_status(ops):
    """A table entry outside the pool is never read and is reported through
    pa_decode_no_alloc_error; the next clean call reports nothing."""
    wl = W.custom("na_bad", "bf16", [300, 40], 8, 2, 128, 16, seed=9)
    g = GpuState(wl, ops)
    out = torch.empty(g.q.shape, dtype=torch.float32, device="cuda")
    tables = g.tables.clone()
    tables[0, 3] = wl.num_blocks + 7
    ops.pa_decode_no_alloc(out, g.q, g.k_cache, g.v_cache, tables, g.lens, wl.scale,
                           wl.num_kv_heads, g.max_len)
    assert ops.pa_decode_no_alloc_error() == 1   # PA_ERR_INVALID_ARG
    ref = g.decode()
    for _ in range(2):
        got = _no_alloc(ops, g)
        assert ops.pa_decode_no_alloc_error() == 0
        assert float((got.double() - ref.double()).abs().max()) <= TOL["bf16"]


def test_no_alloc_split_cuda_core_matches_workspace_decode(ops):
    """fp32 K/V run on the CUDA-core kernel: a split history of several
    thousand tokens gives pa_decode's result, on two calls in a row."""
    wl = W.custom("na_f32_split", "f32", [6000, 2500, 17, 4097], 8, 2, 128, 16, seed=12)
    g = GpuState(wl, ops)
    ref = g.decode()
    for _ in range(2):
        got = _no_alloc(ops, g)
        assert ops.pa_decode_no_alloc_error() == 0
        assert float((got.double() - ref.double()).abs().max()) <= TOL["f32"]


def test_no_alloc_enlarges_cuda_core_partitions(ops):
    """64 fp32 sequences of 8200 tokens need 35 MB of split-K scratch at the
    CUDA-core kernel's 256-token partitions, more than the 32 MiB array: the
    call enlarges the partitions until it fits and matches pa_decode."""
    B, H, Hkv, D, bs, n = 64, 32, 8, 128, 16, 8200
    need = ops.pa_decode_workspace_size(B, H, Hkv, D, bs, "f32", n, 0)
    assert need > 32 << 20
    nb = -(-n // bs)
    gen = torch.Generator(device="cuda").manual_seed(4)
    kc = torch.randn((B * nb, Hkv, bs, D), generator=gen, device="cuda")
    vc = torch.randn((B * nb, Hkv, bs, D), generator=gen, device="cuda")
    q = torch.randn((B, H, D), generator=gen, device="cuda")
    tables = torch.randperm(B * nb, generator=gen, device="cuda").to(torch.int32).reshape(B, nb).contiguous()
    lens = torch.full((B,), n, dtype=torch.int32, device="cuda")
    scale = D ** -0.5
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ref = torch.empty_like(q)
    ops.pa_decode(ref, q, kc, vc, tables, lens, scale, Hkv, n, ws)
    assert ops.pa_workspace_error(ws) == 0
    for _ in range(2):
        got = torch.empty_like(q)
        ops.pa_decode_no_alloc(got, q, kc, vc, tables, lens, scale, Hkv, n)
        assert ops.pa_decode_no_alloc_error() == 0
        assert float((got - ref).abs().max()) <= TOL["f32"]
