"""KV slot write and copy-on-write block copy.  Test infrastructure only.

Slot write ([PA] "Block Table 如何工作"; [KV02] section 2): while a sequence
keeps generating, only the current block receives the new token's K/V.  A
token's slot is ``physical_block * block_size + offset``; its K lands at
``k_cache[slot // bs, :, slot % bs, :]`` (layout ``[NB, Hkv, bs, D]``), V the
same in ``v_cache``.  A negative slot marks a padding token and is skipped.

Block copy ([PA] "支持块级共享"; [KV02] section 2 "블록을 함께 쓰기"): when a
branch has to write into a block it shares, the block is copied to a fresh
one first (copy-on-write).  ``copy_blocks`` copies every (src, dst) pair's
K and V tiles, all kv heads, from the state before the call.
"""
from __future__ import annotations

import numpy as np


def slot_of(block_table_row, position: int, block_size: int) -> int:
    """Slot of logical token ``position``: physical block * block_size + offset."""
    return int(block_table_row[position // block_size]) * block_size + position % block_size


def reshape_and_cache(key, value, k_cache: np.ndarray, v_cache: np.ndarray, slot_mapping) -> None:
    """Write token t's K/V ([T, Hkv, D]) into slot ``slot_mapping[t]``, in place."""
    NB, _, bs, _ = k_cache.shape
    for t in range(len(slot_mapping)):
        s = int(slot_mapping[t])
        if s < 0:
            continue
        if s >= NB * bs:
            raise ValueError(f"slot {s} outside the pool of {NB} blocks x {bs}")
        blk, off = divmod(s, bs)
        k_cache[blk, :, off, :] = key[t]
        v_cache[blk, :, off, :] = value[t]


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, pairs) -> None:
    """For each (src, dst): cache[dst] = cache[src] (pre-call state), in place.

    Destinations must be distinct and must not appear among the sources of the
    same call (copy-on-write pairs always satisfy this).
    """
    pairs = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
    if len(pairs) == 0:
        return
    src = [int(s) for s in pairs[:, 0]]
    dst = [int(d) for d in pairs[:, 1]]
    NB = k_cache.shape[0]
    if len(set(dst)) != len(dst) or set(dst) & set(src):
        raise ValueError("copy destinations must be distinct and not also sources")
    for b in src + dst:
        if not 0 <= b < NB:
            raise ValueError(f"block {b} outside the pool of {NB}")
    k_src = [k_cache[s].copy() for s in src]
    v_src = [v_cache[s].copy() for s in src]
    for j, d in enumerate(dst):
        k_cache[d] = k_src[j]
        v_cache[d] = v_src[j]


# Every layer of a model ([PA] "KV Cache 为什么难管理": a token costs
# M_token = 2 * L * H_kv * d cache elements, K and V in each of the L layers):
# a step appends its tokens in every layer, and a copy-on-write copies the
# block in every layer.  The pool holds the layers as ``[L, NB, Hkv, bs, D]``
# and the step's keys/values as ``[L, T, Hkv, D]``; each layer is written
# exactly as the single-layer operation writes it, with the same slots or
# pairs for every layer.

def reshape_and_cache_layers(key, value, k_cache: np.ndarray, v_cache: np.ndarray,
                             slot_mapping) -> None:
    """Layer l of key/value into layer l of the caches, for every l, in place."""
    if k_cache.ndim != 5 or key.ndim != 4 or key.shape[0] != k_cache.shape[0]:
        raise ValueError("expected caches [L, NB, Hkv, bs, D] and key/value [L, T, Hkv, D]")
    for layer in range(k_cache.shape[0]):
        reshape_and_cache(key[layer], value[layer], k_cache[layer], v_cache[layer], slot_mapping)


def copy_blocks_layers(k_cache: np.ndarray, v_cache: np.ndarray, pairs) -> None:
    """Every (src, dst) pair copied in every layer (pre-call state), in place."""
    if k_cache.ndim != 5:
        raise ValueError("expected caches [L, NB, Hkv, bs, D]")
    for layer in range(k_cache.shape[0]):
        copy_blocks(k_cache[layer], v_cache[layer], pairs)
