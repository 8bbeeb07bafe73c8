"""Paged decode attention, float64.  Test infrastructure only (see package doc).

What it computes ([PA] "Block Table 如何工作"; [vLLM2] block-table section;
[KV02] section 2 "블록과 블록 표"): the attention kernel reads the block table
to turn each logical block number into a physical block id, so the request
still sees its KV cache contiguous in token order while the physical blocks
are scattered.  Paging changes only where K/V live, not the arithmetic
([PA] "不改变模型精度"; [KV02] section 2: the computation is the same as over a
contiguous array).  So for sequence i, query head h and kv head
kvh = h // (H / Hkv):

  1. walk the table:  for t < len_i,  phys = table[i][t // bs],  off = t % bs,
     Kc[t] = k_cache[phys, kvh, off, :],  Vc[t] = v_cache[phys, kvh, off, :]
  2. s_t   = scale * sum_d q[i, h, d] * Kc[t, d]
  3. p_t   = exp(s_t - max_t s) / sum_t exp(s_t - max_t s)
  4. out[i, h, :] = sum_t p_t * Vc[t, :]

A decode query attends to every visible history token ([PA] "不会降低单请求的
理论读取量"), the one appended this step included.  A sequence with no tokens
gets a zero output.  Cache layout: ``[num_blocks, num_kv_heads, block_size,
head_dim]``.  Query heads map to kv heads in contiguous groups of H / Hkv.
"""
from __future__ import annotations

import math

import numpy as np


def gather_sequence(cache: np.ndarray, table_row, length: int) -> np.ndarray:
    """Step 1: walk one sequence's block table; return [length, Hkv, D] float64."""
    bs = cache.shape[2]
    out = np.empty((length, cache.shape[1], cache.shape[3]), dtype=np.float64)
    for t in range(length):
        phys = int(table_row[t // bs])
        off = t % bs
        out[t] = cache[phys, :, off, :]
    return out


def contiguous_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Steps 2-4 over contiguous arrays.

    q: [H, D]; K, V: [T, Hkv, D].  Returns [H, D] float64.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    H, D = q.shape
    T, Hkv, _ = K.shape
    out = np.zeros((H, D), dtype=np.float64)
    if T == 0:
        return out
    G = H // Hkv
    for h in range(H):
        kvh = h // G
        s = float(scale) * (K[:, kvh, :] @ q[h])
        s = s - s.max()
        w = np.exp(s)
        p = w / w.sum()
        out[h] = p @ V[:, kvh, :]
    return out


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                 num_kv_heads: int, seqs=None) -> np.ndarray:
    """Decode-step attention through the block tables.

    q: [B, H, D]; k_cache, v_cache: [NB, Hkv, bs, D]; block_tables: [B, maxb];
    context_lens: [B].  ``seqs`` selects a subset of sequences (rows of the
    result follow its order).  Returns float64 [len(seqs), H, D].
    """
    q = np.asarray(q)
    if k_cache.shape[1] != num_kv_heads or v_cache.shape != k_cache.shape:
        raise ValueError("cache shape does not match num_kv_heads")
    H = q.shape[1]
    if H % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    if seqs is None:
        seqs = range(q.shape[0])
    seqs = list(seqs)
    out = np.zeros((len(seqs), H, q.shape[2]), dtype=np.float64)
    for r, i in enumerate(seqs):
        n = int(context_lens[i])
        K = gather_sequence(k_cache, block_tables[i], n)
        V = gather_sequence(v_cache, block_tables[i], n)
        out[r] = contiguous_attention(q[i], K, V, scale)
    return out


def decode_bruteforce(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                      num_kv_heads: int) -> list:
    """The same definition as scalar Python loops (tiny inputs only).

    Independent of NumPy linear algebra: returns nested lists [B][H][D].
    """
    B = len(q)
    H = len(q[0])
    D = len(q[0][0])
    bs = len(k_cache[0][0])
    G = H // num_kv_heads
    res = []
    for i in range(B):
        n = int(context_lens[i])
        rows = []
        for h in range(H):
            kvh = h // G
            if n == 0:
                rows.append([0.0] * D)
                continue
            scores = []
            for t in range(n):
                blk = int(block_tables[i][t // bs])
                off = t % bs
                acc = 0.0
                for d in range(D):
                    acc += float(q[i][h][d]) * float(k_cache[blk][kvh][off][d])
                scores.append(float(scale) * acc)
            mx = max(scores)
            ws = [math.exp(s - mx) for s in scores]
            tot = math.fsum(ws)
            o = [0.0] * D
            for t in range(n):
                blk = int(block_tables[i][t // bs])
                off = t % bs
                pt = ws[t] / tot
                for d in range(D):
                    o[d] += pt * float(v_cache[blk][kvh][off][d])
            rows.append(o)
        res.append(rows)
    return res


def paged_prefill(q, k_cache, v_cache, block_tables, cu_q, q_start, scale: float,
                  num_kv_heads: int) -> np.ndarray:
    """Prefill attention through the block tables, causal.

    [PA] "KV Cache 为什么难管理": the prefill phase runs the prompt's tokens
    together; each token's query attends to the keys of its own position and
    every earlier one.  Sequence i's chunk is q[cu_q[i]:cu_q[i+1]] and its
    token j sits at position q_start[i] + j (a later start is the next piece
    of a chunked prefill).  Returns float64 [T, H, D]; rows outside every
    chunk stay zero.
    """
    q = np.asarray(q)
    T, H, D = q.shape
    G = H // num_kv_heads
    out = np.zeros((T, H, D), dtype=np.float64)
    for i in range(len(cu_q) - 1):
        b, e = int(cu_q[i]), int(cu_q[i + 1])
        start = int(q_start[i])
        last = start + (e - b)
        K = gather_sequence(k_cache, block_tables[i], last)
        V = gather_sequence(v_cache, block_tables[i], last)
        for j in range(e - b):
            p = start + j
            out[b + j] = contiguous_attention(q[b + j], K[:p + 1], V[:p + 1], scale)
    assert G * num_kv_heads == H
    return out
