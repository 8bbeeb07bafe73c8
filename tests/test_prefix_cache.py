"""Automatic prefix caching: the oracle pinned by what [KV02] section 4
("프리픽스 캐시") states, and the C++ allocator (through the C ABI, on the CPU)
against the oracle, state for state.

[KV02] = "llm-kv-cache-02-serving-engine-kv" (ttlab.hopto.org).
"""
import numpy as np
import pytest

import oracle
from oracle import OraclePrefixCacheAllocator, block_key


def _ops():
    from paged_kv_cache_142_gb300 import build, ops
    build.build(quiet=True)
    return ops


# --------------------------------------------------------------------------
# SHA-256 of the C ABI against the FIPS 180 published test vectors
# --------------------------------------------------------------------------
@pytest.mark.parametrize("msg,digest", [
    (b"abc", "ba7816bf8f01cfea414140de5dae2223b00361a396177a9cb410ff61f20015ad"),
    (b"", "e3b0c44298fc1c149afbf4c8996fb92427ae41e4649b934ca495991b7852b855"),
    (b"abcdbcdecdefdefgefghfghighijhijkijkljklmklmnlmnomnopnopq",
     "248d6a61d20638b8e5c026930c3e6039a33ce45964ff2167f6ecedd419db06c1"),
])
def test_sha256_fips_vectors(msg, digest):
    assert _ops().sha256(msg).hex() == digest


def test_sha256_padding_boundaries_match_hashlib():
    import hashlib
    ops = _ops()
    rng = np.random.default_rng(4)
    for n in (1, 55, 56, 57, 63, 64, 65, 119, 120, 128, 1000, 65536):
        m = rng.integers(0, 256, size=n, dtype=np.uint8).tobytes()
        assert ops.sha256(m) == hashlib.sha256(m).digest(), n


# --------------------------------------------------------------------------
# oracle pins: the page's statements
# --------------------------------------------------------------------------
def test_key_stands_for_the_whole_prefix():
    """"같은 토큰 16개라도 앞부분이 다르면 열쇠가 다릅니다": the same 16 tokens
    after a different prefix give a different key."""
    block = list(range(500, 516))
    k_a = block_key(block_key(None, list(range(16))), block)
    k_b = block_key(block_key(None, list(range(1, 17))), block)
    k_a2 = block_key(block_key(None, list(range(16))), block)
    assert k_a != k_b and k_a == k_a2
    # the documented byte layout: previous key, <i4 token ids, extra bytes
    import hashlib
    raw = bytes(32) + np.arange(16, dtype="<i4").tobytes() + b"salt"
    assert block_key(None, list(range(16)), b"salt") == hashlib.sha256(raw).digest()


def test_only_full_blocks_are_cached():
    """"꽉 찬 블록만 캐시합니다"."""
    a = OraclePrefixCacheAllocator(32, 16)
    s, cached, _ = a.seq_create_prefix(range(40))
    assert cached == 0 and len(a.block_table(s)) == 3
    assert set(a.key_of_block) == set(a.block_table(s)[:2])  # the 8-token tail block has no key
    a.append_token_ids(s, range(40, 48))                     # completes the third block
    assert set(a.key_of_block) == set(a.block_table(s))


@pytest.mark.parametrize("bs,hit", [(16, 2992), (8, 3000), (32, 2976)])
def test_page_scenario_3000_token_prefix_with_32_token_tails(bs, hit):
    """The page's measurement: a 3000-token common prefix and a different
    32-token tail per request; every later request skips the prefill of the
    prefix's full blocks (3000 = 187*16 + 8 = 375*8 = 93*32 + 24)."""
    rng = np.random.default_rng(bs)
    prefix = rng.integers(0, 32000, size=3000).tolist()
    a = OraclePrefixCacheAllocator(4096, bs)
    first = a.seq_create_prefix(prefix + rng.integers(0, 32000, size=32).tolist())
    assert first[1] == 0
    for _ in range(3):
        s, cached, _ = a.seq_create_prefix(prefix + rng.integers(0, 32000, size=32).tolist())
        assert cached == hit
        shared = a.block_table(s)[:hit // bs]
        assert shared == a.block_table(first[0])[:hit // bs]
    assert all(a.refcount(b) == 4 for b in shared)


def test_freed_blocks_evicted_lru_tail_first():
    """Blocks of a finished request wait in the queue with their contents;
    allocation evicts the least recently freed first, and a finished
    request's tail enters the queue before its head."""
    bs = 4
    a = OraclePrefixCacheAllocator(8, bs)
    prompt = list(range(100, 116))               # 4 full blocks
    s, _, _ = a.seq_create_prefix(prompt)
    blocks = a.block_table(s)
    a.free_seq(s)
    assert list(a.free)[-4:] == blocks[::-1]     # tail first
    held = [a.allocate() for _ in range(4)]      # the never-used blocks go first
    assert len(a.cache) == 4
    held.append(a.allocate())                    # evicts the old tail block
    assert held[-1] == blocks[3]
    assert blocks[3] not in a.key_of_block and len(a.cache) == 3
    a.decref(held.pop())                         # one free block for the request's tail
    s2, cached, _ = a.seq_create_prefix(prompt)  # the first three blocks still hit
    assert cached == 3 * bs and a.block_table(s2) == blocks


def test_extra_bytes_separate_requests():
    """The extra information (e.g. a per-user cache salt) is part of every key."""
    a = OraclePrefixCacheAllocator(32, 16)
    a.seq_create_prefix(range(64), extra=b"user-a")
    assert a.seq_create_prefix(range(64), extra=b"user-b")[1] == 0
    assert a.seq_create_prefix(range(64), extra=b"user-a")[1] == 64


def test_hit_stops_at_first_miss_and_takes_blocks_off_the_queue():
    a = OraclePrefixCacheAllocator(32, 4)
    s, _, _ = a.seq_create_prefix(range(16))
    a.free_seq(s)
    free_before = a.num_free()
    ids = list(range(8)) + [99, 99, 99, 99] + list(range(12, 16))  # block 2 differs
    s2, cached, _ = a.seq_create_prefix(ids)
    assert cached == 8                            # blocks 0,1 hit; block 3 is after the miss
    assert a.num_free() == free_before - 4        # 2 hits taken off the queue + 2 fresh blocks
    assert all(a.refcount(b) == 1 for b in a.block_table(s2))


# --------------------------------------------------------------------------
# C++ allocator against the oracle, operation by operation
# --------------------------------------------------------------------------
def _state(cpp, num_blocks):
    free, refs, seqs = cpp.snapshot()
    keys = {b: cpp.block_key(b) for b in range(num_blocks) if cpp.block_key(b) is not None}
    return free, refs, seqs, keys


@pytest.mark.parametrize("seed", range(6))
def test_cpp_matches_oracle_on_random_operations(seed):
    ops = _ops()
    rng = np.random.default_rng(seed)
    NB, bs = 96, 4
    order = rng.permutation(NB).astype(np.int32)
    cpp = ops.BlockAllocator(NB, bs, order)
    cpp.enable_prefix_cache()
    ora = OraclePrefixCacheAllocator(NB, bs, order)
    prompts = [rng.integers(0, 50, size=rng.integers(4, 30)).tolist() for _ in range(5)]
    live = []

    def both(f_cpp, f_ora):
        """Run one operation on both; both run out of blocks or neither does."""
        try:
            want, want_oom = f_ora(), False
        except oracle.AllocatorOOM:
            want, want_oom = None, True
        try:
            got, got_oom = f_cpp(), False
        except ops.AllocatorOOM:
            got, got_oom = None, True
        assert got_oom == want_oom
        return got, want

    ooms = 0
    for step in range(300):
        op = rng.integers(0, 6)
        if ora.num_free() < 12 and live:
            op = 5
        if op <= 1 or not live:
            base = prompts[rng.integers(0, len(prompts))]
            ids = base[:rng.integers(0, len(base) + 1)] + rng.integers(0, 50, size=rng.integers(0, 9)).tolist()
            extra = b"" if rng.random() < 0.8 else b"x"
            got, want = both(lambda: cpp.seq_create_prefix(ids, extra), lambda: ora.seq_create_prefix(ids, extra))
            if want is None:
                ooms += 1
            else:
                assert got[0] == want[0] and got[1] == want[1] and list(got[2]) == want[2]
                live.append(got[0])
        elif op == 2:
            s = live[rng.integers(0, len(live))]
            ids = rng.integers(0, 50, size=rng.integers(1, 7)).tolist()
            pos = ora.seq_len(s)
            if pos % bs and ora.refcount(ora.block_table(s)[pos // bs]) > 1:
                continue  # a shared last block needs the copy-on-write path (op 4)
            got, want = both(lambda: list(cpp.append_token_ids(s, ids)), lambda: ora.append_token_ids(s, ids))
            assert got == want
        elif op == 3:
            s = live[rng.integers(0, len(live))]
            c = cpp.fork(s)
            assert c == ora.fork(s)
            live.append(c)
        elif op == 4:
            s = live[rng.integers(0, len(live))]
            got, want = both(lambda: tuple(cpp.append_slot(s)), lambda: tuple(ora.append_slot(s)))
            assert got == want
        else:
            s = live.pop(rng.integers(0, len(live)))
            cpp.free_seq(s)
            ora.free_seq(s)
        assert _state(cpp, NB) == ora.snapshot(), f"step {step} op {op}"
    assert len(ora.cache) > 0
