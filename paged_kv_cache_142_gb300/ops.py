"""Thin Python binding over the C ABI (include/pa.h), same names.

Argument marshalling only: tensors are passed by data pointer with their
sizes, on torch's current CUDA stream unless one is given.  Every step of the
paged decode path runs in libpa_gb300.so; PyTorch provides device memory and
streams.  Importing this module loads the library and fails loudly if it is
missing.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import _lib as L

_LIB = L.load()

PA_DTYPE_F32 = L.PA_DTYPE_F32
PA_DTYPE_BF16 = L.PA_DTYPE_BF16
PAError = L.PAError


def dtype_code(dt) -> int:
    if dt in (torch.float32, "f32", PA_DTYPE_F32):
        return PA_DTYPE_F32
    if dt in (torch.bfloat16, "bf16", PA_DTYPE_BF16):
        return PA_DTYPE_BF16
    raise ValueError(f"unsupported dtype {dt}")


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _need(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _on_current_device(*tensors) -> None:
    """The library launches on the current device (and its default stream),
    so every tensor handed to it must live there."""
    dev = torch.cuda.current_device()
    for t in tensors:
        if t is not None and t.is_cuda:
            _need(t.device.index == dev, f"tensor on cuda:{t.device.index} but the current device is "
                  f"cuda:{dev}: call inside torch.cuda.device(...) of the tensors' device")


def _cache_dims(k_cache: torch.Tensor, v_cache: torch.Tensor):
    _need(k_cache.dim() == 4 and v_cache.shape == k_cache.shape, "caches must be [NB, Hkv, bs, D]")
    _need(k_cache.dtype == v_cache.dtype, "K and V caches must share a dtype")
    _need(k_cache.is_contiguous() and v_cache.is_contiguous(), "caches must be contiguous")
    _need(k_cache.is_cuda and v_cache.is_cuda, "caches must be CUDA tensors")
    _on_current_device(k_cache, v_cache)
    return k_cache.shape


# --------------------------------------------------------------------------
# device calls
# --------------------------------------------------------------------------
def pa_reshape_and_cache(key, value, slot_mapping, k_cache, v_cache, stream=None, status=None) -> None:
    """Write key/value ``[T, Hkv, D]`` into the cache slots ``slot_mapping[T]``.
    ``status`` (a zeroed CUDA int32 tensor): the checked call, which reports
    slots past the pool there (pa_reshape_and_cache_checked)."""
    NB, Hkv, bs, D = _cache_dims(k_cache, v_cache)
    _on_current_device(key, value, slot_mapping, status)
    T = key.shape[0]
    _need(key.shape == (T, Hkv, D) and value.shape == key.shape, "key/value must be [T, Hkv, D]")
    _need(key.dtype == k_cache.dtype and value.dtype == k_cache.dtype, "key/value dtype != cache dtype")
    _need(key.is_contiguous() and value.is_contiguous(), "key/value must be contiguous")
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.numel() == T and slot_mapping.is_cuda,
          "slot_mapping must be a CUDA int64 tensor of num_tokens entries")
    if status is not None:
        _need(status.dtype == torch.int32 and status.is_cuda and status.numel() >= 1,
              "status must be a CUDA int32 tensor")
        L.check(_LIB.pa_reshape_and_cache_checked(
            key.data_ptr(), value.data_ptr(), T, slot_mapping.data_ptr(), k_cache.data_ptr(),
            v_cache.data_ptr(), NB, bs, Hkv, D, dtype_code(k_cache.dtype), status.data_ptr(),
            _stream(stream)), "pa_reshape_and_cache_checked")
        return
    L.check(_LIB.pa_reshape_and_cache(key.data_ptr(), value.data_ptr(), T, slot_mapping.data_ptr(),
                                      k_cache.data_ptr(), v_cache.data_ptr(), NB, bs, Hkv, D,
                                      dtype_code(k_cache.dtype), _stream(stream)),
            "pa_reshape_and_cache")


def pa_copy_blocks(k_cache, v_cache, block_pairs, stream=None, status=None) -> None:
    """cache[dst] = cache[src] for every row (src, dst) of ``block_pairs``.
    ``status`` (a zeroed CUDA int32 tensor): the checked call, which validates
    the pairs first and copies nothing if any is invalid
    (pa_copy_blocks_checked)."""
    NB, Hkv, bs, D = _cache_dims(k_cache, v_cache)
    _on_current_device(block_pairs, status)
    n = block_pairs.shape[0] if block_pairs.numel() else 0
    if n:
        _need(block_pairs.dtype == torch.int64 and block_pairs.is_cuda and block_pairs.is_contiguous()
              and block_pairs.shape == (n, 2), "block_pairs must be a contiguous CUDA int64 [n, 2]")
    if status is not None:
        _need(status.dtype == torch.int32 and status.is_cuda and status.numel() >= 1,
              "status must be a CUDA int32 tensor")
        L.check(_LIB.pa_copy_blocks_checked(k_cache.data_ptr(), v_cache.data_ptr(), NB, bs, Hkv, D,
                                            dtype_code(k_cache.dtype), block_pairs.data_ptr() if n else None,
                                            n, status.data_ptr(), _stream(stream)),
                "pa_copy_blocks_checked")
        return
    L.check(_LIB.pa_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), NB, bs, Hkv, D,
                                dtype_code(k_cache.dtype), block_pairs.data_ptr() if n else None, n,
                                _stream(stream)),
            "pa_copy_blocks")


def _layer_cache_dims(k_cache, v_cache):
    _need(k_cache.dim() == 5 and v_cache.shape == k_cache.shape, "caches must be [L, NB, Hkv, bs, D]")
    _need(k_cache.dtype == v_cache.dtype and k_cache.is_cuda and v_cache.is_cuda,
          "caches must be CUDA tensors of one dtype")
    _need(k_cache[0].is_contiguous() and v_cache[0].is_contiguous()
          and k_cache.stride(0) == v_cache.stride(0), "each cache layer must be contiguous, "
          "with the same layer stride for K and V")
    return tuple(k_cache.shape)


def pa_reshape_and_cache_layers(key, value, slot_mapping, k_cache, v_cache, stream=None) -> None:
    """Every layer at once: key/value ``[L, T, Hkv, D]`` into the caches
    ``[L, NB, Hkv, bs, D]`` at ``slot_mapping[T]`` (the same slots in every layer)."""
    Lyr, NB, Hkv, bs, D = _layer_cache_dims(k_cache, v_cache)
    _on_current_device(k_cache, v_cache, key, value, slot_mapping)
    T = key.shape[1]
    _need(key.shape == (Lyr, T, Hkv, D) and value.shape == key.shape, "key/value must be [L, T, Hkv, D]")
    _need(key.dtype == k_cache.dtype and value.dtype == k_cache.dtype, "key/value dtype != cache dtype")
    _need(key[0].is_contiguous() and value[0].is_contiguous() and key.stride(0) == value.stride(0),
          "each key/value layer must be contiguous, with the same layer stride")
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.numel() == T and slot_mapping.is_cuda,
          "slot_mapping must be a CUDA int64 tensor of num_tokens entries")
    L.check(_LIB.pa_reshape_and_cache_layers(
        key.data_ptr(), value.data_ptr(), key.stride(0), Lyr, T, slot_mapping.data_ptr(),
        k_cache.data_ptr(), v_cache.data_ptr(), k_cache.stride(0), NB, bs, Hkv, D,
        dtype_code(k_cache.dtype), _stream(stream)), "pa_reshape_and_cache_layers")


def pa_copy_blocks_layers(k_cache, v_cache, block_pairs, stream=None) -> None:
    """cache[l, dst] = cache[l, src] for every layer l and row (src, dst) of ``block_pairs``."""
    Lyr, NB, Hkv, bs, D = _layer_cache_dims(k_cache, v_cache)
    _on_current_device(k_cache, v_cache, block_pairs)
    n = block_pairs.shape[0] if block_pairs.numel() else 0
    if n:
        _need(block_pairs.dtype == torch.int64 and block_pairs.is_cuda and block_pairs.is_contiguous()
              and block_pairs.shape == (n, 2), "block_pairs must be a contiguous CUDA int64 [n, 2]")
    L.check(_LIB.pa_copy_blocks_layers(k_cache.data_ptr(), v_cache.data_ptr(), k_cache.stride(0), Lyr,
                                       NB, bs, Hkv, D, dtype_code(k_cache.dtype),
                                       block_pairs.data_ptr() if n else None, n, _stream(stream)),
            "pa_copy_blocks_layers")


def pa_prefill(out, q, k_cache, v_cache, cu_q, q_start, block_tables, scale, num_kv_heads,
               max_q_len, status=None, stream=None) -> None:
    """Causal paged attention of each sequence's chunk ``q[cu_q[i]:cu_q[i+1]]``
    (positions from ``q_start[i]``) over its K/V through ``block_tables``."""
    NB, Hkv, bs, D = _cache_dims(k_cache, v_cache)
    _need(Hkv == num_kv_heads, "num_kv_heads does not match the cache")
    T, H, Dq = q.shape
    _need(Dq == D and out.shape == q.shape, "q / out must be [T, H, D]")
    _need(q.is_contiguous() and out.is_contiguous() and q.dtype == k_cache.dtype, "q must be contiguous, cache dtype")
    S = cu_q.numel() - 1
    _need(cu_q.dtype == torch.int32 and q_start.dtype == torch.int32 and q_start.numel() == S
          and block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] >= S,
          "cu_q [S+1], q_start [S], block_tables [S, M] must be int32")
    _need(block_tables.is_contiguous(), "block_tables must be contiguous")
    _on_current_device(out, q, cu_q, q_start, block_tables, status)
    L.check(_LIB.pa_prefill(out.data_ptr(), dtype_code(out.dtype), q.data_ptr(), T, cu_q.data_ptr(),
                            q_start.data_ptr(), S, int(max_q_len), H, k_cache.data_ptr(), v_cache.data_ptr(),
                            NB, bs, Hkv, D, dtype_code(k_cache.dtype), block_tables.data_ptr(),
                            block_tables.shape[1], float(scale),
                            status.data_ptr() if status is not None else None, _stream(stream)),
            "pa_prefill")


def pa_decode_shared_prefix(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                            max_context_len, group_start, prefix_len, max_group_size, max_prefix_len,
                            workspace=None, status=None, stream=None):
    """Decode with each group's shared prefix read once for all its members
    (groups of consecutive sequences; see pa_decode_shared_prefix).  Returns
    the workspace it used (allocated here when not given)."""
    NB, Hkv, bs, D = _cache_dims(k_cache, v_cache)
    _need(Hkv == num_kv_heads, "num_kv_heads does not match the cache")
    B, H, Dq = q.shape
    _need(Dq == D and out.shape == q.shape and q.is_contiguous() and out.is_contiguous(), "q/out [B, H, D]")
    Gn = prefix_len.numel()
    _need(group_start.dtype == torch.int32 and prefix_len.dtype == torch.int32 and group_start.numel() == Gn + 1,
          "group_start [G+1] and prefix_len [G] must be int32")
    _on_current_device(out, q, block_tables, context_lens, group_start, prefix_len, workspace, status)
    need = _LIB.pa_decode_shared_prefix_workspace_size(B, H, Hkv, Gn, int(max_group_size), int(max_prefix_len))
    if need == 0:
        raise PAError(L.PA_ERR_UNSUPPORTED, "pa_decode_shared_prefix_workspace_size")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    L.check(_LIB.pa_decode_shared_prefix(
        out.data_ptr(), dtype_code(out.dtype), q.data_ptr(), B, H, k_cache.data_ptr(), v_cache.data_ptr(),
        NB, bs, Hkv, D, dtype_code(k_cache.dtype), block_tables.data_ptr(), block_tables.shape[1],
        context_lens.data_ptr(), int(max_context_len), group_start.data_ptr(), prefix_len.data_ptr(), Gn,
        int(max_group_size), int(max_prefix_len), float(scale),
        status.data_ptr() if status is not None else None, workspace.data_ptr(), workspace.numel(),
        _stream(stream)), "pa_decode_shared_prefix")
    return workspace


def pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, dtype,
                             max_context_len, partition_tokens=0) -> int:
    n = _LIB.pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                      dtype_code(dtype), max_context_len, partition_tokens)
    if n == 0:
        raise PAError(L.PA_ERR_UNSUPPORTED, "pa_decode_workspace_size")
    return int(n)


def pa_set_decode_kv_per_item(kv_per_item: int) -> None:
    """Work-item shape of the tensor-core decode: 0 automatic, 1 or 2 kv heads
    per item (process-wide; size the workspace under the same setting)."""
    L.check(_LIB.pa_set_decode_kv_per_item(int(kv_per_item)), "pa_set_decode_kv_per_item")


def pa_decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, dtype,
                   max_context_len, partition_tokens=0):
    """(partition tokens, CTAs) pa_decode would use on the current device."""
    pt = C.c_int32(0)
    ctas = C.c_int32(0)
    L.check(_LIB.pa_decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                dtype_code(dtype), max_context_len, partition_tokens,
                                C.byref(pt), C.byref(ctas)), "pa_decode_plan")
    return pt.value, ctas.value


def make_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, dtype,
                   max_context_len, partition_tokens=0, device="cuda") -> torch.Tensor:
    """A zero-filled decode workspace of the required size."""
    n = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, dtype,
                                 max_context_len, partition_tokens)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
              max_context_len, workspace, partition_tokens=0, stream=None) -> None:
    """out[B, H, D] = paged decode attention of q[B, H, D] over the cache."""
    NB, Hkv, bs, D = _cache_dims(k_cache, v_cache)
    _need(Hkv == num_kv_heads, "num_kv_heads does not match the cache")
    B, H, Dq = q.shape
    _need(Dq == D and q.dtype == k_cache.dtype and q.is_contiguous(), "q must be [B, H, D] in the cache dtype")
    _need(out.shape == q.shape and out.is_contiguous() and out.dtype in (torch.float32, torch.bfloat16),
          "out must be a contiguous [B, H, D] fp32 or bf16 tensor")
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == B
          and block_tables.is_contiguous(), "block_tables must be contiguous int32 [B, max_blocks]")
    _need(context_lens.dtype == torch.int32 and context_lens.numel() == B, "context_lens must be int32 [B]")
    _need(workspace.dtype == torch.uint8 and workspace.is_cuda, "workspace must be a CUDA uint8 tensor")
    _on_current_device(out, q, block_tables, context_lens, workspace)
    L.check(_LIB.pa_decode(out.data_ptr(), dtype_code(out.dtype), q.data_ptr(), B, H,
                           k_cache.data_ptr(), v_cache.data_ptr(), NB, bs, Hkv, D,
                           dtype_code(k_cache.dtype), block_tables.data_ptr(), block_tables.shape[1],
                           context_lens.data_ptr(), int(max_context_len), float(scale),
                           int(partition_tokens), workspace.data_ptr(), workspace.numel(),
                           _stream(stream)),
            "pa_decode")


def pa_decode_no_alloc(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                       max_context_len, partition_tokens=0, stream=None) -> None:
    """pa_decode with the library's fixed device scratch instead of a workspace,
    for callers that cannot allocate device memory (see include/pa.h)."""
    NB, Hkv, bs, D = _cache_dims(k_cache, v_cache)
    _need(Hkv == num_kv_heads, "num_kv_heads does not match the cache")
    B, H, Dq = q.shape
    _need(Dq == D and q.dtype == k_cache.dtype and q.is_contiguous(), "q must be [B, H, D] in the cache dtype")
    _need(out.shape == q.shape and out.is_contiguous() and out.dtype in (torch.float32, torch.bfloat16),
          "out must be a contiguous [B, H, D] fp32 or bf16 tensor")
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == B
          and block_tables.is_contiguous(), "block_tables must be contiguous int32 [B, max_blocks]")
    _need(context_lens.dtype == torch.int32 and context_lens.numel() == B, "context_lens must be int32 [B]")
    _on_current_device(out, q, block_tables, context_lens)
    L.check(_LIB.pa_decode_no_alloc(out.data_ptr(), dtype_code(out.dtype), q.data_ptr(), B, H,
                                    k_cache.data_ptr(), v_cache.data_ptr(), NB, bs, Hkv, D,
                                    dtype_code(k_cache.dtype), block_tables.data_ptr(),
                                    block_tables.shape[1], context_lens.data_ptr(),
                                    int(max_context_len), float(scale), int(partition_tokens),
                                    _stream(stream)),
            "pa_decode_no_alloc")


def pa_decode_no_alloc_error(stream=None) -> int:
    """Synchronise, return and clear the device status word of the last
    pa_decode_no_alloc call on the current device."""
    st = C.c_int32(0)
    L.check(_LIB.pa_decode_no_alloc_error(_stream(stream), C.byref(st)), "pa_decode_no_alloc_error")
    return st.value


def pa_workspace_init(workspace, stream=None) -> None:
    L.check(_LIB.pa_workspace_init(workspace.data_ptr(), workspace.numel(), _stream(stream)),
            "pa_workspace_init")


def pa_workspace_error(workspace, stream=None) -> int:
    """Synchronise, return and clear the workspace's device status word."""
    st = C.c_int32(0)
    L.check(_LIB.pa_workspace_error(workspace.data_ptr(), _stream(stream), C.byref(st)),
            "pa_workspace_error")
    return st.value


# --------------------------------------------------------------------------
# host allocator
# --------------------------------------------------------------------------
def _p32(a: np.ndarray):
    return a.ctypes.data_as(L.P_i32)


def _p64(a: np.ndarray):
    return a.ctypes.data_as(L.P_i64)


class AllocatorOOM(PAError):
    pass


def _acheck(status, what):
    if status == L.PA_ERR_OOM:
        raise AllocatorOOM(status, what)
    L.check(status, what)


class BlockAllocator:
    """Host block pool (free list, reference counts, fork, copy-on-write):
    the pa_alloc_* calls of include/pa.h."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        h = C.c_void_p()
        order = None
        if free_order is not None:
            self._order = np.ascontiguousarray(free_order, dtype=np.int32)
            order = _p32(self._order)
        _acheck(_LIB.pa_alloc_create(num_blocks, block_size, order, C.byref(h)), "pa_alloc_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            _LIB.pa_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def num_blocks(self) -> int:
        return _LIB.pa_alloc_num_blocks(self._h)

    @property
    def block_size(self) -> int:
        return _LIB.pa_alloc_block_size(self._h)

    def num_free(self) -> int:
        return _LIB.pa_alloc_num_free(self._h)

    def refcount(self, block: int) -> int:
        return _LIB.pa_alloc_refcount(self._h, block)

    def allocate(self) -> int:
        b = C.c_int32(-1)
        st = _LIB.pa_alloc_allocate(self._h, C.byref(b))
        if st == L.PA_ERR_OOM:
            return -1
        L.check(st, "pa_alloc_allocate")
        return b.value

    def incref(self, block: int) -> None:
        L.check(_LIB.pa_alloc_incref(self._h, block), "pa_alloc_incref")

    def decref(self, block: int) -> None:
        L.check(_LIB.pa_alloc_decref(self._h, block), "pa_alloc_decref")

    def seq_create(self) -> int:
        s = C.c_int32()
        L.check(_LIB.pa_alloc_seq_create(self._h, C.byref(s)), "pa_alloc_seq_create")
        return s.value

    def fork(self, parent: int) -> int:
        c = C.c_int32()
        L.check(_LIB.pa_alloc_fork(self._h, parent, C.byref(c)), "pa_alloc_fork")
        return c.value

    def append_slot(self, seq: int):
        slot = C.c_int64()
        a = C.c_int32()
        b = C.c_int32()
        _acheck(_LIB.pa_alloc_append_slot(self._h, seq, C.byref(slot), C.byref(a), C.byref(b)),
                "pa_alloc_append_slot")
        return slot.value, a.value, b.value

    def append_slots(self, seqs, out=None):
        """One append per sequence; returns (slots int64 [n], cow pairs int64
        [k, 2]); ``out`` = a contiguous int64 array [n] to write the slots into."""
        seqs = np.ascontiguousarray(seqs, dtype=np.int32)
        n = len(seqs)
        if out is not None:
            _need(isinstance(out, np.ndarray) and out.dtype == np.int64 and out.shape == (n,)
                  and out.flags.c_contiguous, "out must be a contiguous int64 array [n]")
            slots = out
        else:
            slots = np.empty(n, dtype=np.int64)
        pairs = np.empty((max(n, 1), 2), dtype=np.int64)
        ncow = C.c_int32(0)
        done = C.c_int32(0)
        _acheck(_LIB.pa_alloc_append_slots(self._h, _p32(seqs), n, _p64(slots), _p64(pairs),
                                           C.byref(ncow), C.byref(done)), "pa_alloc_append_slots")
        return slots, pairs[:ncow.value].copy()

    def append_tokens(self, seq: int, n: int) -> np.ndarray:
        slots = np.empty(max(n, 1), dtype=np.int64)
        _acheck(_LIB.pa_alloc_append_tokens(self._h, seq, n, _p64(slots)), "pa_alloc_append_tokens")
        return slots[:n]

    def free_seq(self, seq: int) -> None:
        L.check(_LIB.pa_alloc_free_seq(self._h, seq), "pa_alloc_free_seq")

    def seq_len(self, seq: int) -> int:
        return _LIB.pa_alloc_seq_len(self._h, seq)

    def num_seqs(self) -> int:
        return _LIB.pa_alloc_num_seqs(self._h)

    def block_table(self, seq: int) -> list:
        n = C.c_int32(0)
        cap = self.seq_len(seq) // max(1, self.block_size) + 2
        buf = np.empty(max(cap, 1), dtype=np.int32)
        L.check(_LIB.pa_alloc_block_table(self._h, seq, _p32(buf), cap, C.byref(n)), "pa_alloc_block_table")
        return buf[:n.value].tolist()

    def export_tables(self, seqs, max_blocks: int, pad_value: int = 0, out=None):
        """(tables int32 [n, max_blocks], lens int32 [n]) for a batch; ``out``
        = (tables, lens) contiguous int32 arrays of those shapes to write into
        (e.g. views of a pinned staging buffer)."""
        seqs = np.ascontiguousarray(seqs, dtype=np.int32)
        n = len(seqs)
        if out is not None:
            tables, lens = out
            _need(isinstance(tables, np.ndarray) and tables.dtype == np.int32 and tables.shape == (n, max_blocks)
                  and tables.flags.c_contiguous and isinstance(lens, np.ndarray) and lens.dtype == np.int32
                  and lens.shape == (n,) and lens.flags.c_contiguous and n > 0,
                  "out must be contiguous int32 arrays [n, max_blocks] and [n]")
        else:
            tables = np.empty((max(n, 1), max_blocks), dtype=np.int32)
            lens = np.empty(max(n, 1), dtype=np.int32)
        L.check(_LIB.pa_alloc_export_tables(self._h, _p32(seqs), n, _p32(tables), max_blocks,
                                            _p32(lens), pad_value), "pa_alloc_export_tables")
        return tables[:n], lens[:n]

    def free_list(self) -> list:
        n = C.c_int32(0)
        cap = self.num_blocks
        buf = np.empty(max(cap, 1), dtype=np.int32)
        L.check(_LIB.pa_alloc_free_list(self._h, _p32(buf), cap, C.byref(n)), "pa_alloc_free_list")
        return buf[:n.value].tolist()

    def live_seqs(self) -> list:
        n = C.c_int32(0)
        cap = max(self.num_seqs(), 1)
        buf = np.empty(cap, dtype=np.int32)
        L.check(_LIB.pa_alloc_live_seqs(self._h, _p32(buf), cap, C.byref(n)), "pa_alloc_live_seqs")
        return buf[:n.value].tolist()

    def snapshot(self):
        """(free list in order, reference counts, {seq: (table, len)})."""
        refs = [self.refcount(b) for b in range(self.num_blocks)]
        seqs = {s: (self.block_table(s), self.seq_len(s)) for s in self.live_seqs()}
        return self.free_list(), refs, seqs

    # ---- prefix caching (pa_alloc_enable_prefix_cache and friends) ----
    def enable_prefix_cache(self) -> None:
        L.check(_LIB.pa_alloc_enable_prefix_cache(self._h), "pa_alloc_enable_prefix_cache")

    def seq_create_prefix(self, token_ids, extra: bytes = b""):
        """(seq, cached_tokens, slots[n]) for a new tracked sequence of these tokens."""
        ids = np.ascontiguousarray(token_ids, dtype=np.int32)
        n = len(ids)
        slots = np.empty(max(n, 1), dtype=np.int64)
        s, cached = C.c_int32(-1), C.c_int32(0)
        ex = C.create_string_buffer(bytes(extra), max(len(extra), 1))
        _acheck(_LIB.pa_alloc_seq_create_prefix(self._h, _p32(ids) if n else None, n,
                                                C.cast(ex, C.c_void_p) if extra else None, len(extra),
                                                C.byref(s), C.byref(cached), _p64(slots)),
                "pa_alloc_seq_create_prefix")
        return s.value, cached.value, slots[:n]

    def append_token_ids(self, seq: int, token_ids) -> np.ndarray:
        ids = np.ascontiguousarray(token_ids, dtype=np.int32)
        n = len(ids)
        slots = np.empty(max(n, 1), dtype=np.int64)
        _acheck(_LIB.pa_alloc_append_token_ids(self._h, seq, _p32(ids) if n else None, n, _p64(slots)),
                "pa_alloc_append_token_ids")
        return slots[:n]

    def num_cached(self) -> int:
        return _LIB.pa_alloc_num_cached(self._h)

    def block_key(self, block: int):
        """The block's 32-byte key, or None if it holds none."""
        buf = C.create_string_buffer(32)
        if _LIB.pa_alloc_block_key(self._h, block, buf) != L.PA_OK:
            return None
        return buf.raw


def sha256(data: bytes) -> bytes:
    """pa_sha256 (FIPS 180-4) of ``data``."""
    buf = C.create_string_buffer(32)
    src = C.create_string_buffer(bytes(data), max(len(data), 1))
    L.check(_LIB.pa_sha256(C.cast(src, C.c_void_p), len(data), buf), "pa_sha256")
    return buf.raw
