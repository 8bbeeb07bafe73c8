"""Prefix caching end to end on the GPU: requests that share a prompt prefix
reuse its cached blocks, only the uncached tokens' K/V are written, and the
decode through the shared tables equals the oracle's attention over each
request's whole history ([KV02] section 4 "프리픽스 캐시": a hit skips the
prefill of the cached part)."""
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


def test_prefix_hits_skip_prefill_and_decode_matches(ops):
    bs, H, Hkv, D = 16, 32, 8, 128
    rng = np.random.default_rng(1421)
    prefix = rng.integers(0, 32000, size=3000).tolist()
    prompts = [prefix + rng.integers(0, 32000, size=32).tolist() for _ in range(6)]
    prompts.append(prefix[:1000] + rng.integers(0, 32000, size=200).tolist())  # diverges at 1000
    prompts.append(rng.integers(0, 32000, size=500).tolist())                   # shares nothing
    # K/V of position p: the prefix's values while the tokens so far equal the
    # prefix's (same tokens, same K/V), values of the request's own otherwise
    kv_prefix = W.Values.from_f32((rng.standard_normal((2, 3000, Hkv, D)) * 0.5).astype(np.float32), "bf16")
    seq_kv = []
    for i, p in enumerate(prompts):
        own = W.Values.from_f32((rng.standard_normal((2, len(p), Hkv, D)) * 0.5).astype(np.float32), "bf16")
        bits = own.bits.copy()
        same = 0
        while same < min(len(p), 3000) and p[same] == prefix[same]:
            same += 1
        bits[:, :same] = kv_prefix.bits[:, :same]
        seq_kv.append(bits)
    NB = 4096
    alloc = ops.BlockAllocator(NB, bs, rng.permutation(NB).astype(np.int32))
    alloc.enable_prefix_cache()
    kc = torch.zeros((NB, Hkv, bs, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    seqs, cached_all, written = [], [], 0
    for i, p in enumerate(prompts):
        s, cached, slots = alloc.seq_create_prefix(p)
        seqs.append(s)
        cached_all.append(cached)
        new = slice(cached, len(p))                 # prefill only what the cache lacks
        k = torch.from_numpy(np.ascontiguousarray(seq_kv[i][0, new])).view(torch.bfloat16).cuda()
        v = torch.from_numpy(np.ascontiguousarray(seq_kv[i][1, new])).view(torch.bfloat16).cuda()
        ops.pa_reshape_and_cache(k, v, torch.from_numpy(np.ascontiguousarray(slots[new])).cuda(), kc, vc)
        written += len(p) - cached
    assert cached_all == [0] + [2992] * 5 + [992, 0]
    assert written == sum(len(p) for p in prompts) - 5 * 2992 - 992
    maxb = max(len(p) for p in prompts) // bs + 1
    tables, lens = alloc.export_tables(seqs, maxb)
    q = W.Values.from_f32(rng.standard_normal((len(prompts), H, D)).astype(np.float32), "bf16")
    out = torch.empty((len(prompts), H, D), dtype=torch.float32, device="cuda")
    ws = ops.make_workspace(len(prompts), H, Hkv, D, bs, "bf16", int(lens.max()))
    scale = float(np.float32(1.0 / np.sqrt(D)))
    ops.pa_decode(out, to_device(q), kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                  scale, Hkv, int(lens.max()), ws)
    torch.cuda.synchronize()
    assert ops.pa_workspace_error(ws) == 0
    ref = np.stack([oracle.contiguous_attention(_f64(q.bits[i]), _f64(seq_kv[i][0]), _f64(seq_kv[i][1]), scale)
                    for i in range(len(prompts))])
    assert float(np.abs(to_f64(out) - ref).max()) <= TOL["bf16"]


def _f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 values."""
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
