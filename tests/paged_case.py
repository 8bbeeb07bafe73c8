"""Test helpers: build a paged decode state on the GPU (C++ allocator +
CUDA kernels, through the C ABI) and, independently, on the CPU (oracle
allocator + oracle ops) from the same seeded workload."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_cache_142_gb300 import workloads as W

TOL = {"f32": 1e-5, "bf16": 2e-3}


def torch_dtype(dtype: str):
    return torch.float32 if dtype == W.DTYPE_F32 else torch.bfloat16


def to_device(vals: W.Values, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(vals.bits))
    if vals.dtype == W.DTYPE_BF16:
        t = t.view(torch.bfloat16)
    return t.to(device)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def raw_bits(a: np.ndarray) -> np.ndarray:
    """Element bit patterns of a host array of bf16 bits or float32 values."""
    a = np.ascontiguousarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a


def cache_bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy().view(np.uint32)


class GpuState:
    """C++ allocator tables/slots + caches filled by pa_reshape_and_cache."""

    def __init__(self, wl: W.DecodeWorkload, ops, device="cuda"):
        self.wl = wl
        self.ops = ops
        dt = torch_dtype(wl.dtype)
        self.alloc = ops.BlockAllocator(wl.num_blocks, wl.block_size, wl.free_order)
        slots = []
        for i in range(wl.num_seqs):
            s = self.alloc.seq_create()
            slots.append(self.alloc.append_tokens(s, int(wl.context_lens[i])))
        self.slots = np.concatenate(slots) if slots else np.zeros(0, np.int64)
        self.max_blocks = wl.max_blocks_per_seq
        tables, lens = self.alloc.export_tables(list(range(wl.num_seqs)), self.max_blocks, pad_value=0)
        self.tables_np = tables
        self.lens_np = lens
        shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
        self.k_cache = torch.zeros(shape, dtype=dt, device=device)
        self.v_cache = torch.zeros(shape, dtype=dt, device=device)
        self.tables = torch.from_numpy(tables).to(device)
        self.lens = torch.from_numpy(lens).to(device)
        self.q = to_device(wl.q, device)
        key = to_device(wl.key_hist, device)
        value = to_device(wl.value_hist, device)
        ops.pa_reshape_and_cache(key, value, torch.from_numpy(self.slots).to(device), self.k_cache,
                                 self.v_cache)
        del key, value
        self.max_len = int(lens.max()) if len(lens) else 0

    def decode(self, out_dtype=torch.float32, partition_tokens=0, workspace=None, q=None):
        wl = self.wl
        q = self.q if q is None else q
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
        ws = workspace if workspace is not None else self.ops.make_workspace(
            wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, wl.dtype,
            self.max_len, partition_tokens)
        self.ops.pa_decode(out, q, self.k_cache, self.v_cache, self.tables, self.lens, wl.scale,
                           wl.num_kv_heads, self.max_len, ws, partition_tokens=partition_tokens)
        torch.cuda.synchronize()
        assert self.ops.pa_workspace_error(ws) == 0
        return out


class OracleState:
    """Oracle allocator tables/slots and an oracle cache holding the given
    sequences' tokens (all sequences by default)."""

    def __init__(self, wl: W.DecodeWorkload, seqs=None, bits=False):
        self.wl = wl
        self.alloc = oracle.OracleAllocator(wl.num_blocks, wl.block_size, wl.free_order)
        per_seq = []
        for i in range(wl.num_seqs):
            s = self.alloc.seq_create()
            per_seq.append(self.alloc.append_tokens(s, int(wl.context_lens[i])))
        self.slots = np.array([x for sl in per_seq for x in sl], dtype=np.int64)
        self.tables = np.zeros((wl.num_seqs, wl.max_blocks_per_seq), dtype=np.int64)
        for i in range(wl.num_seqs):
            t = self.alloc.block_table(i)
            self.tables[i, :len(t)] = t
        shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
        src_k = raw_bits(wl.key_hist.bits) if bits else wl.key_hist.f32
        src_v = raw_bits(wl.value_hist.bits) if bits else wl.value_hist.f32
        dt = src_k.dtype if bits else np.float64
        self.k_cache = np.zeros(shape, dtype=dt)
        self.v_cache = np.zeros(shape, dtype=dt)
        starts = wl.seq_starts
        sel = range(wl.num_seqs) if seqs is None else seqs
        for i in sel:
            a, b = int(starts[i]), int(starts[i + 1])
            oracle.reshape_and_cache(src_k[a:b], src_v[a:b], self.k_cache, self.v_cache, per_seq[i])

    def decode(self, seqs=None):
        wl = self.wl
        return oracle.paged_decode(wl.q.f32, self.k_cache, self.v_cache, self.tables,
                                   wl.context_lens, wl.scale, wl.num_kv_heads, seqs=seqs)


def sample_seqs(lens: np.ndarray, k: int, seed: int = 0) -> list:
    """Shortest, longest, and a seeded random sample of the rest."""
    order = np.argsort(lens, kind="stable")
    pick = {int(order[0]), int(order[-1])}
    rng = np.random.default_rng(seed)
    rest = [i for i in range(len(lens)) if i not in pick]
    pick.update(int(x) for x in rng.choice(rest, size=min(k - len(pick), len(rest)), replace=False))
    return sorted(pick)


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half a bf16 unit in the last place at |x| (rounding error of a bf16 store)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    e = np.floor(np.log2(ax))
    return np.exp2(e - 8)
