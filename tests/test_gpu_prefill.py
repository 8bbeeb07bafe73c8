"""Paged prefill on the tensor cores against the oracle's causal attention.

Chunks of several sequences (whole prompts and later pieces of chunked
prefills, lengths around the tile sizes) read their K/V through shuffled
block tables; outputs must match the fp64 oracle within the bf16 tolerance.
"""
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


def _bf16_f64(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _case(G, bs, chunks, seed, Hkv=2, D=128):
    """chunks: [(start, n)]; K/V exist for positions [0, start + n) of each sequence."""
    rng = np.random.default_rng(seed)
    H = G * Hkv
    need = [-(-(s + n) // bs) for s, n in chunks]
    NB = sum(need) + 7
    perm = rng.permutation(NB)
    maxb = max(need)
    tables = np.zeros((len(chunks), maxb), dtype=np.int32)
    k = 0
    for i, nb in enumerate(need):
        tables[i, :nb] = perm[k:k + nb]
        k += nb
    kv = W.Values.from_f32((rng.standard_normal((2, NB, Hkv, bs, D)) * 0.5).astype(np.float32), "bf16")
    lens = [n for _, n in chunks]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = W.Values.from_f32(rng.standard_normal((int(cu[-1]), H, D)).astype(np.float32), "bf16")
    starts = np.array([s for s, _ in chunks], dtype=np.int32)
    return dict(H=H, Hkv=Hkv, D=D, bs=bs, NB=NB, tables=tables, kv=kv, cu=cu, q=q, starts=starts,
                max_q=max(lens))


def _run(ops, c, out_dtype=torch.float32, scale=None):
    kc = to_device(c["kv"][0]).contiguous()
    vc = to_device(c["kv"][1]).contiguous()
    q = to_device(c["q"]).contiguous()
    out = torch.full(q.shape, float("nan"), dtype=out_dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = scale or float(np.float32(1.0 / np.sqrt(c["D"])))
    ops.pa_prefill(out, q, kc, vc, torch.from_numpy(c["cu"]).cuda(), torch.from_numpy(c["starts"]).cuda(),
                   torch.from_numpy(c["tables"]).cuda(), scale, c["Hkv"], c["max_q"], status=status)
    torch.cuda.synchronize()
    ref = oracle.paged_prefill(_bf16_f64(c["q"].bits), _bf16_f64(c["kv"].bits[0]), _bf16_f64(c["kv"].bits[1]),
                               c["tables"], c["cu"], c["starts"], scale, c["Hkv"])
    return out, ref, int(status.item())


CHUNKS = [(0, 1), (0, 7), (0, 33), (0, 130), (100, 20), (250, 64), (17, 200), (0, 300)]


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("bs", [16, 32, 8])
def test_prefill_matches_oracle(ops, G, bs):
    c = _case(G, bs, CHUNKS, seed=100 * G + bs)
    out, ref, st = _run(ops, c)
    assert st == 0
    assert float(np.abs(to_f64(out) - ref).max()) <= TOL["bf16"]


@pytest.mark.parametrize("G", [1, 4])
@pytest.mark.parametrize("bs", [64, 128, 256])
def test_prefill_large_blocks(ops, G, bs):
    """Blocks of 64 to 256 tokens: one TMA box per block up to 128 rows, two
    boxes of 128 rows for a 256-token block; bf16 and fp32 output."""
    c = _case(G, bs, CHUNKS, seed=500 + 10 * G + bs)
    out, ref, st = _run(ops, c)
    assert st == 0
    assert float(np.abs(to_f64(out) - ref).max()) <= TOL["bf16"]
    out_b, ref_b, st = _run(ops, c, out_dtype=torch.bfloat16)
    assert st == 0
    from paged_case import bf16_half_ulp
    assert (np.abs(to_f64(out_b) - ref_b) <= np.maximum(TOL["bf16"], TOL["bf16"] + bf16_half_ulp(ref_b))).all()


def test_prefill_bf16_output_and_long_prompt(ops):
    c = _case(4, 16, [(0, 1000), (1000, 77)], seed=7)
    out, ref, st = _run(ops, c, out_dtype=torch.bfloat16)
    assert st == 0
    got = to_f64(out)
    from paged_case import bf16_half_ulp
    assert (np.abs(got - ref) <= np.maximum(TOL["bf16"], TOL["bf16"] + bf16_half_ulp(ref))).all()


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_prefill_bf16_output_every_group(ops, G):
    """bf16 output for every GQA group size: a tile's rows leave in boxes of
    one warp's 32 rows (32 tokens of one head for 128 / G >= 32, else 128 / G
    tokens of 32 G / 128 heads) when all of them are valid, row by row
    otherwise; the chunks mix whole tiles and ragged ends."""
    c = _case(G, 16, [(0, 300), (40, 256), (0, 129), (5, 3)], seed=31 + G)
    out, ref, st = _run(ops, c, out_dtype=torch.bfloat16)
    assert st == 0
    got = to_f64(out)
    from paged_case import bf16_half_ulp
    assert np.isfinite(got).all()
    assert (np.abs(got - ref) <= np.maximum(TOL["bf16"], TOL["bf16"] + bf16_half_ulp(ref))).all()


def test_chunked_prefill_equals_whole(ops):
    """The same prompt in one call and in three pieces (later starts)."""
    whole = _case(4, 16, [(0, 257)], seed=9)
    out_w, ref_w, st = _run(ops, whole)
    assert st == 0 and float(np.abs(to_f64(out_w) - ref_w).max()) <= TOL["bf16"]
    parts = dict(whole)
    parts["tables"] = np.repeat(whole["tables"], 3, axis=0)
    parts["cu"] = np.array([0, 100, 200, 257], dtype=np.int32)
    parts["starts"] = np.array([0, 100, 200], dtype=np.int32)
    parts["max_q"] = 100
    out_p, ref_p, st = _run(ops, parts)
    assert st == 0 and np.allclose(ref_p, ref_w, atol=1e-12)
    assert float(np.abs(to_f64(out_p) - ref_w).max()) <= TOL["bf16"]


def test_chunk_outside_the_table_is_reported_and_skipped(ops):
    c = _case(4, 16, [(0, 40), (0, 10)], seed=11)
    c["starts"] = np.array([0, c["tables"].shape[1] * 16], dtype=np.int32)  # past the table
    kc = to_device(c["kv"][0]).contiguous()
    vc = to_device(c["kv"][1]).contiguous()
    q = to_device(c["q"]).contiguous()
    out = torch.zeros(q.shape, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.pa_prefill(out, q, kc, vc, torch.from_numpy(c["cu"]).cuda(), torch.from_numpy(c["starts"]).cuda(),
                   torch.from_numpy(c["tables"]).cuda(), 0.1, c["Hkv"], c["max_q"], status=status)
    torch.cuda.synchronize()
    from paged_kv_cache_142_gb300 import _lib as L
    assert int(status.item()) == L.PA_ERR_INVALID_ARG
    assert not to_f64(out)[40:].any()          # the bad chunk's rows were not written
    ref = oracle.paged_prefill(_bf16_f64(c["q"].bits[:40]), _bf16_f64(c["kv"].bits[0]),
                               _bf16_f64(c["kv"].bits[1]), c["tables"][:1], c["cu"][:2], c["starts"][:1],
                               0.1, c["Hkv"])
    assert float(np.abs(to_f64(out)[:40] - ref).max()) <= TOL["bf16"]


def test_scores_rising_along_the_keys(ops):
    """Key magnitudes stepped up along the positions so the running max of
    later rows grows by far more than 2^8 at several points: inside the first
    tile, in the first and second halves of the second tile, and in later
    tiles.  Every growth forces the reference max up, rescaling the partial
    output (and the tile's probabilities already formed) by the factor
    2^(m_old - m_new)."""
    G, bs, Hkv, D = 4, 16, 2, 128
    n = 520
    rng = np.random.default_rng(31)
    H = G * Hkv
    nb = -(-n // bs)
    NB = nb + 3
    tables = rng.permutation(NB)[:nb].astype(np.int32)[None, :]
    step = np.zeros(n)
    for pos, mag in ((40, 1.0), (150, 2.5), (230, 4.0), (300, 5.5), (450, 7.0)):
        step[pos:] = mag
    # key rows of position t: step(t) * ones + noise, queries ~ ones: score ~ 11.3 * step(t)
    k_tok = step[:, None, None] + 0.1 * rng.standard_normal((n, Hkv, D))
    v_tok = rng.standard_normal((n, Hkv, D)) * 0.5
    kv = np.zeros((2, NB, Hkv, bs, D), dtype=np.float32)
    for t in range(n):
        kv[0, tables[0, t // bs], :, t % bs] = k_tok[t]
        kv[1, tables[0, t // bs], :, t % bs] = v_tok[t]
    q = 1.0 + 0.05 * rng.standard_normal((n, H, D))
    c = dict(H=H, Hkv=Hkv, D=D, bs=bs, NB=NB, tables=tables, kv=W.Values.from_f32(kv, "bf16"),
             cu=np.array([0, n], dtype=np.int32), q=W.Values.from_f32(q.astype(np.float32), "bf16"),
             starts=np.array([0], dtype=np.int32), max_q=n)
    out, ref, st = _run(ops, c)
    assert st == 0
    assert float(np.abs(to_f64(out) - ref).max()) <= TOL["bf16"]


def test_empty_chunks_among_others_and_no_tokens(ops):
    """Sequences whose chunk is empty (one with K/V history, one without)
    between non-empty ones, and a call with no tokens at all."""
    c = _case(4, 16, [(0, 50), (30, 0), (0, 0), (10, 90)], seed=13)
    out, ref, st = _run(ops, c)
    assert st == 0
    assert float(np.abs(to_f64(out) - ref).max()) <= TOL["bf16"]
    empty = dict(c)
    empty["q"] = W.Values.from_f32(np.zeros((0, c["H"], c["D"]), dtype=np.float32), "bf16")
    empty["cu"] = np.zeros(5, dtype=np.int32)
    empty["max_q"] = 0
    out0, ref0, st = _run(ops, empty)
    assert st == 0 and out0.shape == (0, c["H"], c["D"]) and ref0.shape == (0, c["H"], c["D"])


def test_bench_size_sampled_rows(ops):
    """The bench's prefill launch (16 causal prompts of 2048 tokens, 32 q /
    8 kv heads, block 16, shuffled blocks): sampled rows against the oracle's
    attention over each row's visible keys, gathered through the table."""
    n, S = 2048, 16
    c = _case(4, 16, [(0, n)] * S, seed=17, Hkv=8)
    kc = to_device(c["kv"][0]).contiguous()
    vc = to_device(c["kv"][1]).contiguous()
    q = to_device(c["q"]).contiguous()
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = float(np.float32(1.0 / np.sqrt(c["D"])))
    ops.pa_prefill(out, q, kc, vc, torch.from_numpy(c["cu"]).cuda(), torch.from_numpy(c["starts"]).cuda(),
                   torch.from_numpy(c["tables"]).cuda(), scale, c["Hkv"], n, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().numpy()
    assert not np.isnan(got).any()
    kf = _bf16_f64(c["kv"].bits[0])
    vf = _bf16_f64(c["kv"].bits[1])
    rng = np.random.default_rng(18)
    rows = np.concatenate([[0, n - 1, n, S * n - 1], rng.integers(0, S * n, size=60)])
    for tok in rows:
        i, pos = int(tok) // n, int(tok) % n
        K = oracle.gather_sequence(kf, c["tables"][i], pos + 1)
        V = oracle.gather_sequence(vf, c["tables"][i], pos + 1)
        ref = oracle.contiguous_attention(_bf16_f64(c["q"].bits[tok]), K, V, scale)
        assert float(np.abs(got[tok].astype(np.float64) - ref).max()) <= TOL["bf16"], (i, pos)
