"""bench.py's multi-rank host logic on the CPU: two gloo ranks.

Each rank decodes an independent batch (its own seed; rank 0 the benchmark
batch) and the ranks meet only to take the max of their times and the sum of
their work.  No GPU is involved: the data path has no collective to test.
"""
import os
import socket
import sys


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, queue) -> None:
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = bench.W.gqa_bf16(seed=bench.rank_seed(rank), num_seqs=32)
        tokens = float(wl.context_lens.sum())
        step_ms = 1.0 + rank          # rank 1 is the slower one
        times, counts = bench.reduce_over_ranks([step_ms, 3.0 - rank], [tokens, 32], world)
        queue.put((rank, times, counts, tokens, wl.context_lens.tolist()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_shard_and_reduce():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = {}
        for _ in range(2):
            r = queue.get(timeout=180)
            got[r[0]] = r
    finally:
        for p in procs:
            p.join(60)
    assert all(p.exitcode == 0 for p in procs)
    tok0, tok1 = got[0][3], got[1][3]
    for rank in (0, 1):
        _, times, counts, _, _ = got[rank]
        assert times == [2.0, 3.0]                  # max over ranks, per entry
        assert counts == [tok0 + tok1, 64.0]         # work summed over ranks
    # independent shards of one distribution; rank 0 holds the benchmark batch
    import bench
    assert got[0][4] != got[1][4]
    assert got[0][4] == bench.W.gqa_bf16(num_seqs=32).context_lens.tolist()
    assert 16 <= min(got[1][4]) and max(got[1][4]) <= 4096


def test_single_rank_reduce_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks([1.5, 2], [3, 4], 1) == ([1.5, 2.0], [3.0, 4.0])
    assert bench.rank_seed(0) == bench.W.SEEDS["gqa_bf16"]
    assert len({bench.rank_seed(r) for r in range(8)}) == 8
