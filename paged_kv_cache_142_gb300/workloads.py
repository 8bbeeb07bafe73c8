"""Seeded synthetic inputs for the paged decode step.

This module only draws inputs: context lengths, the initial free-list order
of the physical block pool, query / key / value values, and the beam-parent
choices of the shared-prefix workload.  It holds none of the method's
arithmetic (no slot mapping, no block-table walk, no attention): both the
CUDA path and the fp64 oracle consume what it returns, each computing the
rest on its own.

Workloads follow the shapes of the paged decode configurations described on
the pages (block size 16 tokens, "vLLM internals (2)", section on the block
table; "LLM KV cache 02", section 2):

  tiny_fp32    4 seqs, lens {5,16,17,40}, 4 q = 4 kv heads, D 64, bs 16,
               32-block pool with a shuffled free list, N(0,1) fp32 values.
  mha_bf16     64 seqs, 32 = 32 heads, D 128, bs 16, lens U[128,2048],
               shuffled free list, pool 1.2x the blocks needed, N(0,1).
  gqa_bf16     256 seqs, 32 q / 8 kv heads, D 128, bs 16,
               lens = clip(round(exp(ln 800 + 0.5 z)), 16, 4096),
               pool 1.2x the blocks needed, N(0,1)*0.5.
  long_bf16    8 seqs x 32768 tokens, 64 q / 8 kv heads, D 128, bs 16 or 32,
               pool exactly the blocks needed, shuffled, N(0,1).
  prefix_bf16  16 groups x beam width 4 sharing a 3000-token prefix, 32
               decode steps with seeded beam-parent choices, 32 q / 8 kv
               heads, D 128, bs 8/16/32, N(0,1)*0.5.

Values are drawn as float32 from numpy's PCG64 generator and, for bf16
workloads, rounded to bfloat16 (round to nearest even).  The same bytes go to
the GPU and to the oracle.
"""
from __future__ import annotations

from dataclasses import dataclass, field
import math

import numpy as np

DTYPE_F32 = "f32"
DTYPE_BF16 = "bf16"

SEEDS = {
    "tiny_fp32": 14201,
    "mha_bf16": 14202,
    "gqa_bf16": 14203,
    "long_bf16": 14204,
    "prefix_bf16": 14205,
}


# --------------------------------------------------------------------------
# bfloat16 encoding helpers (input preparation only)
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Values:
    """A tensor of input values in the workload's element type.

    ``bits`` holds the raw element bytes that go to the device (uint16 for
    bf16, float32 for f32); ``f32`` holds the exact same values widened to
    float32 (for the oracle, which widens again to float64).
    """

    dtype: str
    bits: np.ndarray
    f32: np.ndarray

    @staticmethod
    def from_f32(x: np.ndarray, dtype: str) -> "Values":
        x = np.ascontiguousarray(x, dtype=np.float32)
        if dtype == DTYPE_F32:
            return Values(dtype, x, x)
        if dtype == DTYPE_BF16:
            b = f32_to_bf16_bits(x)
            return Values(dtype, b, bf16_bits_to_f32(b).reshape(x.shape))
        raise ValueError(dtype)

    @property
    def shape(self):
        return self.f32.shape

    def __getitem__(self, idx) -> "Values":
        return Values(self.dtype, self.bits[idx], self.f32[idx])


def _normal(rng: np.random.Generator, shape, sigma: float, chunk: int = 1 << 24) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        rng.standard_normal(e - s, dtype=np.float32, out=out[s:e])
    if sigma != 1.0:
        out *= np.float32(sigma)
    return out.reshape(shape)


def elem_bytes(dtype: str) -> int:
    return 4 if dtype == DTYPE_F32 else 2


# --------------------------------------------------------------------------
# decode-step workload
# --------------------------------------------------------------------------
@dataclass
class DecodeWorkload:
    """One decode step over a batch of sequences held in a paged KV pool.

    ``context_lens[i]`` counts every token sequence ``i`` attends to in this
    step, the newly appended one included.  ``key_hist``/``value_hist`` hold
    the K/V of all those tokens, token-major in logical order
    (``[sum(context_lens), Hkv, D]``; sequence ``i`` starts at
    ``seq_starts[i]``).  The last token of each sequence is the one the step
    appends; the ones before it are the history already in the pool.
    ``free_order`` is the initial order of the allocator's free list.
    """

    name: str
    dtype: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    context_lens: np.ndarray          # int32 [B]
    free_order: np.ndarray            # int32 [NB], a permutation of 0..NB-1
    q: Values                         # [B, H, D] (None when drawn without values)
    key_hist: Values                  # [sum(len), Hkv, D]
    value_hist: Values                # [sum(len), Hkv, D]
    scale: float
    seed: int
    sigma: float
    extra: dict = field(default_factory=dict)

    @property
    def seq_starts(self) -> np.ndarray:
        s = np.zeros(self.num_seqs + 1, dtype=np.int64)
        np.cumsum(self.context_lens, out=s[1:])
        return s

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_blocks_per_seq(self) -> int:
        return max(1, -(-int(self.context_lens.max()) // self.block_size))

    @property
    def total_tokens(self) -> int:
        return int(self.context_lens.sum())


def _pool_for(lens: np.ndarray, bs: int, factor: float) -> int:
    need = int(sum(-(-int(n) // bs) for n in lens))
    return int(math.ceil(factor * need)) if factor != 1.0 else need


def _make(name, dtype, lens, H, Hkv, D, bs, NB, sigma, seed, rng, extra=None,
          values: bool = True) -> DecodeWorkload:
    """values=False skips drawing Q/K/V (q, key_hist and value_hist are None);
    lengths and the free-list order are drawn first, so they are the same."""
    lens = np.asarray(lens, dtype=np.int32)
    B = len(lens)
    free_order = rng.permutation(NB).astype(np.int32)
    T = int(lens.sum())
    q = k = v = None
    if values:
        q = Values.from_f32(_normal(rng, (B, H, D), sigma), dtype)
        k = Values.from_f32(_normal(rng, (T, Hkv, D), sigma), dtype)
        v = Values.from_f32(_normal(rng, (T, Hkv, D), sigma), dtype)
    return DecodeWorkload(
        name=name, dtype=dtype, num_seqs=B, num_q_heads=H, num_kv_heads=Hkv,
        head_dim=D, block_size=bs, num_blocks=NB, context_lens=lens,
        free_order=free_order, q=q, key_hist=k, value_hist=v,
        scale=float(np.float32(1.0 / math.sqrt(D))), seed=seed, sigma=sigma,
        extra=dict(extra or {}))


def tiny_fp32(seed: int = SEEDS["tiny_fp32"]) -> DecodeWorkload:
    rng = np.random.Generator(np.random.PCG64(seed))
    return _make("tiny_fp32", DTYPE_F32, [5, 16, 17, 40], 4, 4, 64, 16, 32, 1.0, seed, rng)


def mha_bf16(seed: int = SEEDS["mha_bf16"], num_seqs: int = 64,
             len_range=(128, 2048), values: bool = True) -> DecodeWorkload:
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = rng.integers(len_range[0], len_range[1], size=num_seqs, endpoint=True)
    NB = _pool_for(lens, 16, 1.2)
    return _make("mha_bf16", DTYPE_BF16, lens, 32, 32, 128, 16, NB, 1.0, seed, rng, values=values)


def gqa_lens(rng: np.random.Generator, num_seqs: int, median: float = 800.0,
             sigma_log: float = 0.5, lo: int = 16, hi: int = 4096) -> np.ndarray:
    z = rng.standard_normal(num_seqs)
    return np.clip(np.rint(np.exp(math.log(median) + sigma_log * z)), lo, hi).astype(np.int32)


def gqa_bf16(seed: int = SEEDS["gqa_bf16"], num_seqs: int = 256,
             block_size: int = 16, values: bool = True) -> DecodeWorkload:
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = gqa_lens(rng, num_seqs)
    NB = _pool_for(lens, block_size, 1.2)
    return _make("gqa_bf16", DTYPE_BF16, lens, 32, 8, 128, block_size, NB, 0.5, seed, rng,
                 extra={"len_dist": "lognormal(median 800, sigma 0.5) clipped [16,4096]"}, values=values)


def long_bf16(seed: int = SEEDS["long_bf16"], block_size: int = 16, num_seqs: int = 8,
              context_len: int = 32768, values: bool = True) -> DecodeWorkload:
    rng = np.random.Generator(np.random.PCG64(seed + block_size))
    lens = np.full(num_seqs, context_len, dtype=np.int32)
    NB = _pool_for(lens, block_size, 1.0)
    return _make("long_bf16", DTYPE_BF16, lens, 64, 8, 128, block_size, NB, 1.0, seed, rng, values=values)


def custom(name: str, dtype: str, lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
           block_size: int, pool_factor: float = 1.5, sigma: float = 1.0, seed: int = 7,
           extra_blocks: int = 0) -> DecodeWorkload:
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = np.asarray(lens, dtype=np.int32)
    NB = max(1, _pool_for(lens, block_size, pool_factor) + extra_blocks)
    return _make(name, dtype, lens, num_q_heads, num_kv_heads, head_dim, block_size, NB,
                 sigma, seed, rng)


# --------------------------------------------------------------------------
# shared prefix + beam search workload
# --------------------------------------------------------------------------
@dataclass
class PrefixBeamWorkload:
    """A 3000-token prompt shared by ``groups * beam`` sequences, then
    ``steps`` decode steps.  At every step each group picks the parents of its
    ``beam`` new beams among its current beams (``parents[step, group, j]``),
    the chosen beams are forked, the old beams freed, and every new beam
    appends one token.  Values of the prompt tokens, of each step's appended
    token and of each step's queries are drawn here."""

    name: str
    dtype: str
    groups: int
    beam: int
    prefix_len: int
    steps: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    free_order: np.ndarray            # int32 [NB]
    parents: np.ndarray               # int32 [steps, groups, beam]
    prefix_key: Values                # [prefix_len, Hkv, D]
    prefix_value: Values              # [prefix_len, Hkv, D]
    step_key: Values                  # [steps, groups*beam, Hkv, D]
    step_value: Values                # [steps, groups*beam, Hkv, D]
    step_q: Values                    # [steps, groups*beam, H, D]
    scale: float
    seed: int
    sigma: float

    @property
    def num_seqs(self) -> int:
        return self.groups * self.beam


def prefix_bf16(block_size: int = 16, seed: int = SEEDS["prefix_bf16"], groups: int = 16,
                beam: int = 4, prefix_len: int = 3000, steps: int = 32,
                num_q_heads: int = 32, num_kv_heads: int = 8, head_dim: int = 128,
                dtype: str = DTYPE_BF16) -> PrefixBeamWorkload:
    rng = np.random.Generator(np.random.PCG64(seed + block_size))
    S = groups * beam
    prefix_blocks = -(-prefix_len // block_size)
    tail_blocks = -(-steps // block_size) + 2
    NB = prefix_blocks + S * tail_blocks + 8
    free_order = rng.permutation(NB).astype(np.int32)
    parents = rng.integers(0, beam, size=(steps, groups, beam)).astype(np.int32)
    sig = 0.5
    pk = Values.from_f32(_normal(rng, (prefix_len, num_kv_heads, head_dim), sig), dtype)
    pv = Values.from_f32(_normal(rng, (prefix_len, num_kv_heads, head_dim), sig), dtype)
    sk = Values.from_f32(_normal(rng, (steps, S, num_kv_heads, head_dim), sig), dtype)
    sv = Values.from_f32(_normal(rng, (steps, S, num_kv_heads, head_dim), sig), dtype)
    sq = Values.from_f32(_normal(rng, (steps, S, num_q_heads, head_dim), sig), dtype)
    return PrefixBeamWorkload(
        name="prefix_bf16", dtype=dtype, groups=groups, beam=beam, prefix_len=prefix_len,
        steps=steps, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
        block_size=block_size, num_blocks=NB, free_order=free_order, parents=parents,
        prefix_key=pk, prefix_value=pv, step_key=sk, step_value=sv, step_q=sq,
        scale=float(np.float32(1.0 / math.sqrt(head_dim))), seed=seed, sigma=sig)


CONFIGS = {
    "tiny_fp32": tiny_fp32,
    "mha_bf16": mha_bf16,
    "gqa_bf16": gqa_bf16,
    "long_bf16": long_bf16,
    "prefix_bf16": prefix_bf16,
}
