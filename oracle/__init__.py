"""Plain, slow CPU oracle for the paged decode step.  TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it, and it
shares no code with the CUDA path: it reads the same seeded inputs and
computes everything else on its own, in float64 NumPy (or plain Python loops
for tiny inputs).

Sources (the three pages on PagedAttention; cited by title and section):
  [vLLM2]  "vLLM internals (2) - why PagedAttention splits the KV cache into
           pages" (youngju.dev), sections on the block table, block size and
           sharing.
  [PA]     "PagedAttention" (icarus.shaojiemike.top), sections "Block Table
           如何工作", "KV Cache 为什么难管理", "先看直观解释", "支持块级共享",
           "不改变模型精度", "自检问题".
  [KV02]   "LLM KV cache 02 - serving engine KV" (ttlab.hopto.org), section 2
           "PagedAttention: KV 를 블록으로 나누기" (blocks, block table, sharing,
           copy-on-write) and section 4 "프리픽스 캐시" (prefix caching).

Modules:
  attention   paged decode attention (table walk + softmax(q K^T scale) V)
  cache_ops   slot write of new K/V, copy-on-write block copy
  allocator   block pool with a free list, reference counts, fork and COW
  prefix_cache  automatic prefix caching on the pool (chained SHA-256 block
              keys over full blocks, LRU eviction of freed cached blocks)

Every function here is pinned by ``tests/test_oracle_pins.py`` against values
the pages print, closed forms and brute force; none is "parity unpinned".
"""
from .attention import (paged_decode, contiguous_attention, decode_bruteforce, gather_sequence,
                        paged_prefill)
from .cache_ops import (reshape_and_cache, copy_blocks, slot_of, reshape_and_cache_layers,
                        copy_blocks_layers)
from .allocator import OracleAllocator, AllocatorOOM, blocks_for, slack_for
from .prefix_cache import OraclePrefixCacheAllocator, block_key

__all__ = [
    "paged_decode", "contiguous_attention", "decode_bruteforce", "gather_sequence",
    "reshape_and_cache", "copy_blocks", "slot_of",
    "OracleAllocator", "AllocatorOOM", "blocks_for", "slack_for",
]
