"""Failure detection on the device: a bounded wait that runs out.

Every wait of the tensor-core decode is bounded.  When one gives up, the CTA
raises its stop word, every role stops, copies and tensor-core work already
issued are waited for, tensor memory is freed, and PA_ERR_DEVICE_TIMEOUT
reaches the host through the workspace.  The test makes a wait run out
without any fault: the library's test hook has the compute warps first wait,
with a 100 us limit, for an event that never comes (a barrier no role
arrives at).  Nothing traps, and the context stays usable: after the
workspace is zeroed again the next decode matches the oracle."""
import time

import numpy as np
import pytest
import torch

from paged_kv_cache_142_gb300 import workloads as W
from paged_case import GpuState, OracleState, TOL, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops(lib):
    import importlib
    return importlib.import_module("paged_kv_cache_142_gb300.ops")


@pytest.mark.parametrize("partition_tokens", [0, 256])
def test_expired_wait_is_reported_and_the_next_decode_is_correct(ops, lib, partition_tokens):
    wl = W.gqa_bf16(num_seqs=48)
    g = GpuState(wl, ops)
    ref = OracleState(wl).decode()
    ws = ops.make_workspace(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
                            wl.dtype, g.max_len, partition_tokens)
    assert float(np.abs(to_f64(g.decode(partition_tokens=partition_tokens, workspace=ws)) - ref).max()) <= TOL["bf16"]
    out = torch.empty(g.q.shape, dtype=torch.float32, device="cuda")
    lib.pa_test_stall_decode(100_000)
    try:
        t0 = time.perf_counter()
        ops.pa_decode(out, g.q, g.k_cache, g.v_cache, g.tables, g.lens, wl.scale, wl.num_kv_heads,
                      g.max_len, ws, partition_tokens=partition_tokens)
        status = ops.pa_workspace_error(ws)   # synchronises the stream
        elapsed = time.perf_counter() - t0
    finally:
        lib.pa_test_stall_decode(0)
    assert status == 6  # PA_ERR_DEVICE_TIMEOUT
    # the stop word ends every role at once, far inside the 2 s default limit
    # that the other roles' waits keep
    assert elapsed < 1.0, elapsed
    # the merge counters may be left set: zero the workspace, then decode again
    ops.pa_workspace_init(ws)
    again = g.decode(partition_tokens=partition_tokens, workspace=ws)   # asserts status 0
    assert float(np.abs(to_f64(again) - ref).max()) <= TOL["bf16"]
    assert ops.pa_workspace_error(ws) == 0
