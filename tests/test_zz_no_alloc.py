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
