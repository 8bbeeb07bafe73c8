"""Benchmark of the paged decode step on GB300.

One step = the whole hot path over one batch: the KV append of each
sequence's new token (pa_reshape_and_cache) and paged decode attention over
every sequence's history (pa_decode).  Workload: batch 256, 32 q / 8 kv heads,
head_dim 128, bf16, block size 16, context lengths lognormal (median 800,
sigma 0.5) clipped to [16, 4096], pool 1.2x the blocks needed.

Prints one JSON line (rank 0):
  value      algorithmic GB/s of a step with inputs resident in HBM
             (KV read + Q read + O write of decode, plus the append's
             read + write), timed with CUDA events over exactly K steps
  e2e        the same metric through the C ABI from pinned host buffers: per
             step the host allocator reserves the slots, tables/lens/q/new
             K,V go host->device in one copy, the kernels run (a CUDA graph
             per buffer set), the output comes back; the upload of the next
             step and the download of the last overlap the kernels
  roofline   pa_decode's algorithmic bytes / its mean duration (CUDA events
             around back-to-back launches on the launching stream), against
             the measured HBM copy bandwidth; DRAM traffic from the committed
             ncu summary of the full-size launch while the kernel source is
             unchanged
  cpu_baseline  the fp64 oracle on a bounded sample, on the host
  extras     the other rows' kernels on their own workloads: multi-layer
             append and copy, paged prefill, shared-prefix decode, the MHA
             and long-context decode configurations, prefix caching

``--impl reference`` times the oracle instead (the reference arm).
Multi-GPU: data-parallel shards, one per rank.  Sequences are independent,
so each rank decodes its own batch of the same distribution (rank 0 the
benchmark batch) with its own pool and allocator, and no collective runs on
the data path; ranks meet only to time (barriers, max over ranks) and to sum
the bytes they processed.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_142_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak); seq-steps/s at batch 256"
UNIT = "GB/s"
WORKLOAD = ("paged decode step (KV append + decode), batch 256, 32 q / 8 kv heads, head_dim 128, "
            "bf16, block 16, lens lognormal(median 800, sigma 0.5) clipped [16,4096], "
            "pool 1.2x needed, values N(0,1)*0.5")
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_gqa_bf16_b256.md")
KERNEL_SOURCES = [os.path.join(ROOT, "paged_kv_cache_142_gb300", "csrc", f)
                  for f in ("decode_umma.cuh", "decode_common.cuh", "decode.cuh", "ptx.cuh")]


def kernel_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def profiled_traffic():
    """dram bytes per pa_decode launch from the committed ncu summary, if it
    was taken on the current kernel source."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None
    kv = {}
    with open(PROFILE_SUMMARY) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                kv[k.strip()] = v.strip().strip("`")
    if kv.get("kernel_source_hash") != kernel_hash():
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [r for t, r in self.rows if any(a - 0.05 <= t <= b + 0.05 for a, b in self.windows)]
        used = inside or [min(self.rows, key=lambda tr: min(abs(tr[0] - a) for a, _ in self.windows))[1]]
        sm = [float(r[1]) for r in used if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in used if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in used for k in range(4) if len(r) > 5 + k and r[5 + k] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside)}


# --------------------------------------------------------------------------
# byte accounting (algorithmic, per step)
# --------------------------------------------------------------------------
def step_bytes(lens: np.ndarray, B, H, Hkv, D, e, e_out):
    kv = int(lens.sum()) * 2 * Hkv * D * e       # every visible token's K and V, each kv head
    qo = B * H * D * e + B * H * D * e_out        # queries in, outputs out
    append = 2 * (2 * B * Hkv * D * e) + 8 * B    # new K,V read + written, slot ids
    return kv + qo, append


# --------------------------------------------------------------------------
# reference arm / CPU baseline: the fp64 oracle on a bounded sample
# --------------------------------------------------------------------------
def _oracle_sample_setup(wl, nseq):
    import oracle
    st = wl.seq_starts
    a = oracle.OracleAllocator(wl.num_blocks, wl.block_size, wl.free_order)
    per = [a.append_tokens(a.seq_create(), int(n)) for n in wl.context_lens]
    tables = np.zeros((wl.num_seqs, wl.max_blocks_per_seq), dtype=np.int64)
    for i in range(wl.num_seqs):
        t = a.block_table(i)
        tables[i, :len(t)] = t
    shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    kc = np.zeros(shape, dtype=np.float64)
    vc = np.zeros(shape, dtype=np.float64)
    for i in range(nseq):
        oracle.reshape_and_cache(wl.key_hist.f32[st[i]:st[i + 1]], wl.value_hist.f32[st[i]:st[i + 1]],
                                 kc, vc, per[i])
    return tables, kc, vc


_POOL_STATE = None


def _decode_share(args):
    """Worker of the oracle pool: decode the given sequences in turn."""
    import oracle
    seqs = args
    wl, tables, kc, vc, per_seq = _POOL_STATE
    t0 = time.perf_counter()
    for i in seqs:
        oracle.paged_decode(wl.q.f32, kc, vc, tables, wl.context_lens, wl.scale, wl.num_kv_heads, seqs=[i])
    return time.perf_counter() - t0, sum(per_seq[i] for i in seqs)


def _oracle_child(argv):
    """Runs in a child process with no CUDA in it, one BLAS thread per
    process.  Phase "seq": one process decodes the first 64 sequences in turn,
    for ``budget`` s.  Phase "batch": ``procs`` forked processes decode all
    nseq sequences per step, each a disjoint share, for ``steps`` steps or
    until ``budget`` s have passed (per-step wall times).  Mode "both" runs
    the two phases on one set-up."""
    mode, budget, nseq, steps, procs = argv[0], float(argv[1]), int(argv[2]), int(argv[3]), int(argv[4])
    import oracle
    wl = W.gqa_bf16()
    tables, kc, vc = _oracle_sample_setup(wl, nseq)
    e = W.elem_bytes(wl.dtype)
    per_seq = [step_bytes(wl.context_lens[i:i + 1], 1, wl.num_q_heads, wl.num_kv_heads,
                          wl.head_dim, e, e)[0] for i in range(nseq)]
    out = {}
    if mode in ("seq", "both"):
        times, nbytes = [], []
        t_start = time.perf_counter()
        k = 0
        while True:
            i = k % min(nseq, 64)
            t0 = time.perf_counter()
            oracle.paged_decode(wl.q.f32, kc, vc, tables, wl.context_lens, wl.scale, wl.num_kv_heads,
                                seqs=[i])
            times.append(time.perf_counter() - t0)
            nbytes.append(per_seq[i])
            k += 1
            if time.perf_counter() - t_start >= budget:
                break
        out.update(times=times, bytes=nbytes)
    if mode in ("batch", "both"):
        import multiprocessing as mp
        global _POOL_STATE
        _POOL_STATE = (wl, tables, kc, vc, per_seq)    # shared with the workers by fork
        # longest first over the shares, so every process gets a similar load
        order = sorted(range(nseq), key=lambda i: -int(wl.context_lens[i]))
        shares = [order[r::procs] for r in range(procs)]
        step_times, step_bytes_ = [], []
        with mp.get_context("fork").Pool(procs) as pool:   # this process never touches CUDA
            pool.map(_decode_share, [[0]] * procs)          # workers up
            t_start = time.perf_counter()
            while True:
                t0 = time.perf_counter()
                res = pool.map(_decode_share, shares)
                step_times.append(time.perf_counter() - t0)
                step_bytes_.append(sum(r[1] for r in res))
                if (steps and len(step_times) >= steps) or (not steps and time.perf_counter() - t_start >= budget):
                    break
        out.update(procs=procs, step_times=step_times, step_bytes=step_bytes_, seqs_per_step=nseq)
    print(json.dumps(out))


def run_oracle(mode: str, budget_s: float, nseq: int, steps: int = 0, procs: int = 1):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--_oracle_child", mode,
                        str(budget_s), str(nseq), str(steps), str(procs)],
                       capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError(f"oracle baseline failed:\n{r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(budget_s: float) -> dict:
    """The fp64 oracle on the host: all cores (one process per core, one BLAS
    thread each, decoding the whole 256-sequence batch per step) and a single
    core (the first 64 sequences in turn), each for about ``budget_s`` s."""
    cores = os.cpu_count() or 1
    res = run_oracle("both" if cores > 1 else "seq", budget_s, 256, procs=cores)
    t1 = sum(res["times"])
    single = {"value": round(sum(res["bytes"]) / t1 / 1e9, 4), "unit": UNIT, "cores": 1,
              "seq_steps_per_s": round(len(res["times"]) / t1, 2),
              "sample": (f"fp64 oracle decode of the first 64 of the 256 sequences in turn for {t1:.1f} s "
                         f"({len(res['times'])} sequence decodes), 1 process, 1 BLAS thread")}
    if cores == 1:
        return dict(single, kind="oracle", single_core=dict(single))
    wall = sum(res["step_times"])
    n = len(res["step_times"])
    return {"value": round(sum(res["step_bytes"]) / wall / 1e9, 4), "unit": UNIT, "cores": cores,
            "kind": "oracle", "seq_steps_per_s": round(256 * n / wall, 2),
            "sample": (f"fp64 oracle decode of all 256 sequences per step, {n} steps in {wall:.1f} s, "
                       f"{cores} processes (one per host core, 1 BLAS thread each) on disjoint shares"),
            "single_core": single}


def reference_arm(args):
    """The oracle as the reference arm, on all the host's cores: each step
    decodes the whole 256-sequence batch, split over one process per core;
    W warm-up steps, then K timed steps."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    res = run_oracle("batch", 0, 256, steps=args.steps + args.warmup, procs=cores)
    times = res["step_times"][args.warmup:]
    nbytes = res["step_bytes"][args.warmup:]
    t = sum(times)
    value = sum(nbytes) / t / 1e9
    sample = (f"fp64 oracle decode of all 256 sequences per step, {cores} processes (one per host core, "
              f"1 BLAS thread each) on disjoint shares")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000 * t / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "num_seqs": 256},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "seq_steps_per_s": round(256 * args.steps / t, 3),
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# multi-rank helpers (host only; covered by a gloo test on the CPU)
# --------------------------------------------------------------------------
def rank_seed(rank: int) -> int:
    """Workload seed of a rank's shard: rank 0 holds the benchmark batch, every
    other rank an independent batch of the same distribution."""
    return W.SEEDS["gqa_bf16"] + 7919 * rank


def reduce_over_ranks(times, counts, world: int, device=None):
    """Max over ranks of each time and sum over ranks of each count."""
    times, counts = [float(x) for x in times], [float(x) for x in counts]
    if world == 1:
        return times, counts
    import torch
    import torch.distributed as dist
    t = torch.tensor(times, dtype=torch.float64, device=device)
    c = torch.tensor(counts, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(c, op=dist.ReduceOp.SUM)
    return t.tolist(), c.tolist()


# --------------------------------------------------------------------------
# secondary kernels (reported under "extras"; not part of the step)
# --------------------------------------------------------------------------
def _event_time_us(fn, iters: int, stream) -> float:
    import torch
    for _ in range(3):
        fn()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(iters):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1000.0 / iters


def _graph_time_us(fn, n: int = 20, reps: int = 10) -> float:
    """Device time per call of fn, replayed from a CUDA graph of n calls (no
    host dispatch between the kernels)."""
    import torch
    fn()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(n):
            fn()
    graph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        graph.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1000.0 / (n * reps)


def measure_extras(ops, dev, seed: int = 1420) -> dict:
    """Multi-layer append and copy-on-write copy of a decode step, one launch
    for all layers, against one launch per layer (algorithmic bytes: read +
    write of every moved K/V element)."""
    import torch
    Lyr, T, Hkv, D, bs, NB, pairs_n = 32, 256, 8, 128, 16, 512, 64
    g = torch.Generator(device=dev).manual_seed(seed)
    stream = torch.cuda.current_stream(dev)
    kc = torch.zeros((Lyr, NB, Hkv, bs, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    key = torch.randn((Lyr, T, Hkv, D), generator=g, device=dev).to(torch.bfloat16)
    val = torch.randn((Lyr, T, Hkv, D), generator=g, device=dev).to(torch.bfloat16)
    slots = torch.randperm(NB * bs, generator=g, device=dev)[:T].to(torch.int64)
    perm = torch.randperm(NB, generator=g, device=dev)
    pairs = torch.stack([perm[:pairs_n], perm[pairs_n:2 * pairs_n]], dim=1).to(torch.int64).contiguous()
    append_b = Lyr * T * Hkv * D * 2 * 2 * 2
    copy_b = Lyr * pairs_n * 2 * Hkv * bs * D * 2 * 2
    t_app = _graph_time_us(lambda: ops.pa_reshape_and_cache_layers(key, val, slots, kc, vc))
    t_app_e = _event_time_us(lambda: ops.pa_reshape_and_cache_layers(key, val, slots, kc, vc), 50, stream)
    t_app1 = _event_time_us(lambda: [ops.pa_reshape_and_cache(key[i], val[i], slots, kc[i], vc[i])
                                     for i in range(Lyr)], 20, stream)
    t_cp = _graph_time_us(lambda: ops.pa_copy_blocks_layers(kc, vc, pairs))
    t_cp_e = _event_time_us(lambda: ops.pa_copy_blocks_layers(kc, vc, pairs), 50, stream)
    t_cp1 = _event_time_us(lambda: [ops.pa_copy_blocks(kc[i], vc[i], pairs) for i in range(Lyr)], 20, stream)
    gbs = lambda b, us: round(b / (us * 1e-6) / 1e9, 1)
    del kc, vc
    # paged prefill (tensor cores): 16 prompts of 2048 tokens, causal
    S_, n_, Hq_ = 16, 2048, 32
    pf_launch, flops, stat = _prefill_case(ops, dev, g, S_, n_, Hq_, Hkv, D, bs)
    t_pf = _event_time_us(pf_launch, 10, stream)
    pf_tflops = flops / (t_pf * 1e-6) / 1e12
    pf_ok = int(stat.item()) == 0
    del pf_launch
    # shared-prefix decode: the beam-search workload's last step, 64 sequences
    # = one 3000-token prompt + 32 tokens of their own (the prompt's 187 full
    # blocks shared by all), plain decode against one group of 64
    sp = _shared_prefix_case(ops, dev, g, Hq_, Hkv, D, bs)
    Sb, pref, own, shared = sp["Sb"], sp["pref"], sp["own"], sp["shared"]
    osp, qs, ksp, vsp, t_tb, t_ln, mlen = sp["out"], sp["q"], sp["k"], sp["v"], sp["tables"], sp["lens"], sp["mlen"]
    gs, pl_, st_sp, tb, ln = sp["group_start"], sp["prefix_len"], sp["status"], sp["tables_np"], sp["lens_np"]
    wsd = ops.make_workspace(Sb, Hq_, Hkv, D, bs, "bf16", mlen, device=dev)
    wss = sp["launch"]()
    t_plain = _event_time_us(lambda: ops.pa_decode(osp, qs, ksp, vsp, t_tb, t_ln, 1.0 / math.sqrt(D), Hkv, mlen,
                                                   wsd), 50, stream)
    t_shared = _graph_time_us(lambda: sp["launch"](wss))
    t_shared_e = _event_time_us(lambda: sp["launch"](wss), 50, stream)
    logical = int(ln.sum()) * Hkv * D * 2 * 2 + 2 * Sb * Hq_ * D * 2
    unique_blocks = len(set(tb[:, :int(ln.max()) // bs + 1].ravel().tolist()))
    sp_ok = int(st_sp.item()) == 0
    del ksp, vsp, sp, osp, qs
    # decode on the other decode configurations: MHA (G = 1) and long-context
    # split-K (G = 8, block 16 and 32).  Lengths, pool and free list are the
    # workloads'; the values are drawn on the device (throughput only; parity
    # is covered by the tests).  Every launch reads > 1 GB, larger than L2.
    hbm_peak, _ = measured_peaks()
    other = {}
    for label, wl_o in (("mha_bf16: 64 seqs, 32 q = 32 kv heads, lens U[128,2048], block 16",
                         W.mha_bf16(values=False)),
                        ("long_bf16: 8 seqs, 64 q / 8 kv heads, len 32768, block 16",
                         W.long_bf16(block_size=16, values=False)),
                        ("long_bf16: 8 seqs, 64 q / 8 kv heads, len 32768, block 32",
                         W.long_bf16(block_size=32, values=False))):
        Bo, Ho, Hko, Do, bso = wl_o.num_seqs, wl_o.num_q_heads, wl_o.num_kv_heads, wl_o.head_dim, wl_o.block_size
        ao = ops.BlockAllocator(wl_o.num_blocks, bso, wl_o.free_order)
        so = [ao.seq_create() for _ in range(Bo)]
        for s_, n_o in zip(so, wl_o.context_lens):
            ao.append_tokens(s_, int(n_o))
        tbo, lno = ao.export_tables(so, wl_o.max_blocks_per_seq)
        ao.close()
        kco = (torch.randn((wl_o.num_blocks, Hko, bso, Do), generator=g, device=dev, dtype=torch.bfloat16)
               * wl_o.sigma)
        vco = (torch.randn((wl_o.num_blocks, Hko, bso, Do), generator=g, device=dev, dtype=torch.bfloat16)
               * wl_o.sigma)
        qo = torch.randn((Bo, Ho, Do), generator=g, device=dev, dtype=torch.bfloat16) * wl_o.sigma
        oo = torch.empty_like(qo)
        mlo = int(lno.max())
        wso = ops.make_workspace(Bo, Ho, Hko, Do, bso, "bf16", mlo, device=dev)
        d_tbo, d_lno = torch.from_numpy(tbo).to(dev), torch.from_numpy(lno).to(dev)
        t_o = _event_time_us(lambda: ops.pa_decode(oo, qo, kco, vco, d_tbo, d_lno, wl_o.scale, Hko, mlo, wso),
                             20, stream)
        ok_o = ops.pa_workspace_error(wso) == 0
        by_o = int(lno.sum()) * Hko * Do * 2 * 2 + 2 * Bo * Ho * Do * 2
        pt_o, ctas_o = ops.pa_decode_plan(Bo, Ho, Hko, Do, bso, "bf16", mlo, 0)
        other[label] = {"us": round(t_o, 2), "bytes": by_o, "GB/s": gbs(by_o, t_o),
                        "frac_of_measured_hbm": round(by_o / (t_o * 1e-6) / 1e9 / hbm_peak, 4),
                        "partition_tokens": pt_o, "status_ok": ok_o}
        del kco, vco, qo, oo, wso
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    bf16_peak = float(peaks.get("bf16_tflops", 1900.0))
    # prefix caching (host): 64 requests of one 3000-token prefix + their own
    # 32-token tails, keys hashed with SHA-256 in the allocator
    rng = np.random.default_rng(seed)
    prefix = rng.integers(0, 32000, size=3000)
    reqs = [np.concatenate([prefix, rng.integers(0, 32000, size=32)]).astype(np.int32) for _ in range(64)]
    pc = ops.BlockAllocator(8192, bs)
    pc.enable_prefix_cache()
    t0 = time.perf_counter()
    hits = [pc.seq_create_prefix(r)[1] for r in reqs]
    t_pc = (time.perf_counter() - t0) / len(reqs) * 1e6
    used = pc.num_blocks - pc.num_free()
    pc.close()
    return {
        "append_layers": {"layers": Lyr, "tokens": T, "bytes": append_b, "us": round(t_app, 2),
                          "GB/s": gbs(append_b, t_app), "us_called_from_python": round(t_app_e, 2),
                          "us_one_launch_per_layer": round(t_app1, 2)},
        "copy_blocks_layers": {"layers": Lyr, "pairs": pairs_n, "bytes": copy_b, "us": round(t_cp, 2),
                               "GB/s": gbs(copy_b, t_cp), "us_called_from_python": round(t_cp_e, 2),
                               "us_one_launch_per_layer": round(t_cp1, 2)},
        "note": "bf16, 8 kv heads, head_dim 128, block 16; bytes = read + write of the moved K/V; "
                "us = device time per launch, replayed from a CUDA graph; us_called_from_python = "
                "back-to-back calls through the binding (host dispatch bound); "
                "us_one_launch_per_layer = the same work as one call per layer, from Python; "
                "the append's 67 MB stay in L2 across launches, the copy's 268 MB straddle it",
        "prefill": {"prompts": S_, "tokens_per_prompt": n_, "q_heads": Hq_, "kv_heads": Hkv, "head_dim": D,
                    "us": round(t_pf, 1), "TFLOP/s": round(pf_tflops, 1),
                    "frac_of_bf16_peak": round(pf_tflops / bf16_peak, 4), "bf16_peak_tflops": bf16_peak,
                    "status_ok": pf_ok,
                    "flops": "causal algorithmic: 2*D*H*n*(n+1) per prompt (Q.K^T and P.V)"},
        "shared_prefix_decode": {"sequences": Sb, "shared_tokens": shared, "own_tokens": pref + own - shared,
                                 "logical_bytes": logical, "unique_kv_bytes": unique_blocks * Hkv * bs * D * 2 * 2,
                                 "us_pa_decode": round(t_plain, 2), "us_shared_prefix": round(t_shared, 2),
                                 "us_shared_prefix_called_from_python": round(t_shared_e, 2),
                                 "logical_GB/s_pa_decode": gbs(logical, t_plain),
                                 "logical_GB/s_shared_prefix": gbs(logical, t_shared), "status_ok": sp_ok,
                                 "note": "the unique K/V fits in L2: logical bytes are what the tables name"},
        "decode_other_configs": other,
        "prefix_cache": {"requests": len(reqs), "tokens_per_request": 3032,
                         "cached_tokens_per_hit": int(hits[1]), "hits": int(sum(h > 0 for h in hits)),
                         "blocks_used": int(used), "blocks_without_cache": 64 * 190,
                         "us_per_request": round(t_pc, 1),
                         "note": "host allocator, SHA-256 block keys; K/V prefill skipped for the "
                                 "cached tokens"},
    }


def _prefill_case(ops, dev, g, S_, n_=2048, Hq_=32, Hkv=8, D=128, bs=16):
    """Causal prefill of S_ prompts of n_ tokens through shuffled blocks:
    returns a no-argument launcher and the causal algorithmic flops."""
    import torch
    nb_seq = n_ // bs
    NBp = S_ * nb_seq
    kpp = torch.randn((NBp, Hkv, bs, D), generator=g, device=dev).to(torch.bfloat16)
    vpp = torch.randn((NBp, Hkv, bs, D), generator=g, device=dev).to(torch.bfloat16)
    tab = torch.randperm(NBp, generator=g, device=dev).to(torch.int32).reshape(S_, nb_seq).contiguous()
    qp = torch.randn((S_ * n_, Hq_, D), generator=g, device=dev).to(torch.bfloat16)
    op = torch.empty_like(qp)
    cu = torch.arange(0, (S_ + 1) * n_, n_, dtype=torch.int32, device=dev)
    st0 = torch.zeros(S_, dtype=torch.int32, device=dev)
    stat = torch.zeros(1, dtype=torch.int32, device=dev)

    def launch():
        ops.pa_prefill(op, qp, kpp, vpp, cu, st0, tab, 1.0 / math.sqrt(D), Hkv, n_, status=stat)

    return launch, S_ * 2.0 * D * Hq_ * n_ * (n_ + 1), stat


def _shared_prefix_case(ops, dev, g, Hq_=32, Hkv=8, D=128, bs=16):
    """The beam-search workload's last step for the shared-prefix decode: 64
    sequences = one 3000-token prompt + 32 tokens of their own, built with the
    allocator (fork, then one append per step), values drawn on the device.
    ``launch(workspace=None)`` runs pa_decode_shared_prefix on one group of 64
    and returns its workspace."""
    import torch
    Sb, pref, own = 64, 3000, 32
    NBs = pref // bs + 1 + Sb * (own // bs + 2)
    al = ops.BlockAllocator(NBs, bs)
    root = al.seq_create()
    al.append_tokens(root, pref)
    beams = [al.fork(root) for _ in range(Sb)]
    al.free_seq(root)
    for _ in range(own):
        al.append_slots(beams)
    tb, ln = al.export_tables(beams, (pref + own) // bs + 2)
    al.close()
    c = {"Sb": Sb, "pref": pref, "own": own, "shared": (pref // bs) * bs, "tables_np": tb, "lens_np": ln}
    c["k"] = torch.randn((NBs, Hkv, bs, D), generator=g, device=dev).to(torch.bfloat16)
    c["v"] = torch.randn((NBs, Hkv, bs, D), generator=g, device=dev).to(torch.bfloat16)
    c["q"] = torch.randn((Sb, Hq_, D), generator=g, device=dev).to(torch.bfloat16)
    c["out"] = torch.empty((Sb, Hq_, D), dtype=torch.bfloat16, device=dev)
    c["tables"], c["lens"] = torch.from_numpy(tb).to(dev), torch.from_numpy(ln).to(dev)
    c["mlen"] = int(ln.max())
    c["group_start"] = torch.tensor([0, Sb], dtype=torch.int32, device=dev)
    c["prefix_len"] = torch.tensor([c["shared"]], dtype=torch.int32, device=dev)
    c["status"] = torch.zeros(1, dtype=torch.int32, device=dev)

    def launch(workspace=None):
        return ops.pa_decode_shared_prefix(c["out"], c["q"], c["k"], c["v"], c["tables"], c["lens"],
                                           1.0 / math.sqrt(D), Hkv, c["mlen"], c["group_start"],
                                           c["prefix_len"], Sb, c["shared"], workspace=workspace,
                                           status=c["status"])

    c["launch"] = launch
    return c


def kernel_profile(args):
    """Profiling case for the per-kernel DRAM captures: --warmup untimed, then
    --steps launches of each of, in this order, the step's append (256
    tokens into the batch-256 pool), the 32-layer append, the 64-pair copy
    (one layer and 32 layers), the shared-prefix decode (its pass and its
    merge) and the 16 x 2048 causal prefill."""
    import torch
    dev = torch.device("cuda", 0)
    from paged_kv_cache_142_gb300 import build as B_
    B_.build(quiet=True)
    from paged_kv_cache_142_gb300 import ops
    g = torch.Generator(device=dev).manual_seed(7)
    wl = W.gqa_bf16(values=False)
    Hkv, D, bs, T = wl.num_kv_heads, wl.head_dim, wl.block_size, wl.num_seqs
    kc = torch.zeros((wl.num_blocks, Hkv, bs, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    key = torch.randn((T, Hkv, D), generator=g, device=dev).to(torch.bfloat16)
    val = torch.randn((T, Hkv, D), generator=g, device=dev).to(torch.bfloat16)
    slots = torch.randperm(wl.num_blocks * bs, generator=g, device=dev)[:T].to(torch.int64)
    Lyr, NBl, npairs = 32, 512, 64
    kl = torch.zeros((Lyr, NBl, Hkv, bs, D), dtype=torch.bfloat16, device=dev)
    vl = torch.zeros_like(kl)
    keyl = torch.randn((Lyr, T, Hkv, D), generator=g, device=dev).to(torch.bfloat16)
    vall = torch.randn((Lyr, T, Hkv, D), generator=g, device=dev).to(torch.bfloat16)
    slotsl = torch.randperm(NBl * bs, generator=g, device=dev)[:T].to(torch.int64)
    perm = torch.randperm(NBl, generator=g, device=dev)
    pairs = torch.stack([perm[:npairs], perm[npairs:2 * npairs]], dim=1).to(torch.int64).contiguous()
    sp = _shared_prefix_case(ops, dev, g, 32, Hkv, D, bs)
    wss = sp["launch"]()
    pf_launch, _, pf_stat = _prefill_case(ops, dev, g, 16)
    cases = [
        ("append", lambda: ops.pa_reshape_and_cache(key, val, slots, kc, vc)),
        ("append_layers", lambda: ops.pa_reshape_and_cache_layers(keyl, vall, slotsl, kl, vl)),
        ("copy", lambda: ops.pa_copy_blocks(kl[0], vl[0], pairs)),
        ("copy_layers", lambda: ops.pa_copy_blocks_layers(kl, vl, pairs)),
        ("shared_prefix", lambda: sp["launch"](wss)),
        ("prefill", pf_launch),
    ]
    times = {}
    for name, fn in cases:
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        times[name] = round(a.elapsed_time(b) * 1000.0 / args.steps, 2)
    if int(sp["status"].item()) != 0 or int(pf_stat.item()) != 0:
        raise RuntimeError("a profiled kernel reported an error")
    print(json.dumps({"profile_kernels": True, "us_per_call": times,
                      "shared_prefix_unique_blocks": int(len(set(sp["tables_np"].ravel().tolist())))}), flush=True)


def prefill_profile(args):
    """Small prefill case for ncu: --warmup + --steps launches of pa_prefill."""
    import torch
    dev = torch.device("cuda", 0)
    from paged_kv_cache_142_gb300 import build as B_
    B_.build(quiet=True)
    from paged_kv_cache_142_gb300 import ops
    g = torch.Generator(device=dev).manual_seed(1)
    launch, flops, stat = _prefill_case(ops, dev, g, args.profile_prefill)
    for _ in range(args.warmup):
        launch()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        launch()
    b.record()
    torch.cuda.synchronize()
    if int(stat.item()) != 0:
        raise RuntimeError("pa_prefill reported an error")
    us = a.elapsed_time(b) * 1000.0 / args.steps
    print(json.dumps({"profile_prefill": True, "prompts": args.profile_prefill, "tokens_per_prompt": 2048,
                      "us": round(us, 2), "TFLOP/s": round(flops / (us * 1e-6) / 1e12, 1)}), flush=True)


def cuda_core_profile(args):
    """The CUDA-core decode kernel (fp32 K/V) on the batch-256 workload's
    lengths, tables and pool: --warmup + --steps back-to-back launches of
    pa_decode, values drawn on the device."""
    import torch
    dev = torch.device("cuda", 0)
    from paged_kv_cache_142_gb300 import build as B_
    B_.build(quiet=True)
    from paged_kv_cache_142_gb300 import ops
    g = torch.Generator(device=dev).manual_seed(9)
    wl = W.gqa_bf16(num_seqs=args.num_seqs, block_size=args.block_size, values=False)
    B, H, Hkv, D, bs = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size
    a = ops.BlockAllocator(wl.num_blocks, bs, wl.free_order)
    seqs = [a.seq_create() for _ in range(B)]
    for s_, n in zip(seqs, wl.context_lens):
        a.append_tokens(s_, int(n))
    tb, ln = a.export_tables(seqs, wl.max_blocks_per_seq)
    a.close()
    kc = torch.randn((wl.num_blocks, Hkv, bs, D), generator=g, device=dev) * wl.sigma
    vc = torch.randn((wl.num_blocks, Hkv, bs, D), generator=g, device=dev) * wl.sigma
    q = torch.randn((B, H, D), generator=g, device=dev) * wl.sigma
    out = torch.empty_like(q)
    ml = int(ln.max())
    ws = ops.make_workspace(B, H, Hkv, D, bs, "f32", ml, args.partition_tokens, device=dev)
    d_tb, d_ln = torch.from_numpy(tb).to(dev), torch.from_numpy(ln).to(dev)
    run = lambda: ops.pa_decode(out, q, kc, vc, d_tb, d_ln, wl.scale, Hkv, ml, ws,
                                partition_tokens=args.partition_tokens)
    for _ in range(args.warmup):
        run()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        run()
    t1.record()
    torch.cuda.synchronize()
    if ops.pa_workspace_error(ws) != 0:
        raise RuntimeError("pa_decode reported an error")
    us = t0.elapsed_time(t1) * 1000.0 / args.steps
    by = int(ln.sum()) * Hkv * D * 4 * 2 + 2 * B * H * D * 4
    pt, ctas = ops.pa_decode_plan(B, H, Hkv, D, bs, "f32", ml, args.partition_tokens)
    print(json.dumps({"profile_cuda_core": True, "num_seqs": B, "dtype": "f32", "us": round(us, 2),
                      "bytes": by, "GB/s": round(by / (us * 1e-6) / 1e9, 1),
                      "partition_tokens": pt, "ctas": ctas}), flush=True)


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------
def gpu_arm(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from paged_kv_cache_142_gb300 import build as B_
    B_.build(quiet=True)
    from paged_kv_cache_142_gb300 import ops

    wl = W.gqa_bf16(seed=rank_seed(rank), num_seqs=args.num_seqs, block_size=args.block_size)
    B, H, Hkv, D, bs = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size
    e = W.elem_bytes(wl.dtype)
    K, Wm = args.steps, args.warmup
    # pool: the workload's 1.2x plus room for the e2e leg's growth
    grow = K + Wm + 1
    NB = wl.num_blocks + B * (grow // bs + 2)
    free_order = np.concatenate([wl.free_order, np.arange(wl.num_blocks, NB, dtype=np.int32)])
    alloc = ops.BlockAllocator(NB, bs, free_order)
    seqs = [alloc.seq_create() for _ in range(B)]
    hist = [alloc.append_tokens(s, int(n)) for s, n in zip(seqs, wl.context_lens)]
    slots_all = np.concatenate(hist)
    new_slots = np.array([h[-1] for h in hist], dtype=np.int64)  # this step's token
    max_len = int(wl.context_lens.max())
    e2e_max_len = max_len + grow
    maxb = -(-e2e_max_len // bs)
    tables, lens = alloc.export_tables(seqs, maxb)

    kc = torch.zeros((NB, Hkv, bs, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)

    def dev_vals(v):
        return torch.from_numpy(np.ascontiguousarray(v.bits)).view(torch.bfloat16).to(dev)

    key_all, val_all = dev_vals(wl.key_hist), dev_vals(wl.value_hist)
    ops.pa_reshape_and_cache(key_all, val_all, torch.from_numpy(slots_all).to(dev), kc, vc)
    st = wl.seq_starts
    last = torch.from_numpy(st[1:] - 1).to(dev)
    new_k = key_all.index_select(0, last).contiguous()
    new_v = val_all.index_select(0, last).contiguous()
    del key_all, val_all
    q = dev_vals(wl.q)
    t_tables = torch.from_numpy(tables).to(dev)
    t_lens = torch.from_numpy(lens).to(dev)
    t_slots = torch.from_numpy(new_slots).to(dev)
    out = torch.empty((B, H, D), dtype=torch.bfloat16, device=dev)
    ws = ops.make_workspace(B, H, Hkv, D, bs, "bf16", e2e_max_len, args.partition_tokens, device=dev)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)

    decode_bytes, append_bytes = step_bytes(lens, B, H, Hkv, D, e, 2)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)

    def step():
        ops.pa_reshape_and_cache(new_k, new_v, t_slots, kc, vc)
        ops.pa_decode(out, q, kc, vc, t_tables, t_lens, wl.scale, Hkv, e2e_max_len, ws,
                      partition_tokens=args.partition_tokens)

    # ---------------- device-resident steps ----------------
    # The K timed steps record no event between the two kernels, so the
    # decode's set-up can overlap the append as in a serving loop; the decode
    # kernel's own duration (for the roofline) is timed afterwards with an
    # event pair around each decode launch.
    for _ in range(Wm):
        step()
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    w0 = time.time()
    t0e.record(stream)
    for k in range(K):
        step()
    t1e.record(stream)
    torch.cuda.synchronize(dev)
    w1 = time.time()
    sampler.mark(w0, w1)
    if world > 1:
        dist.barrier()
    total_ms = t0e.elapsed_time(t1e)
    # The decode kernel's own average duration: K2 back-to-back launches on
    # the launching stream between one event pair (the kernel's launches
    # follow one another as they do inside the steps).  For comparison, the
    # same decode with an event pair around each launch after an append,
    # which also counts each launch's start-up gap.
    K2 = min(K, 500)
    w0b = time.time()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for k in range(K2):
        ops.pa_decode(out, q, kc, vc, t_tables, t_lens, wl.scale, Hkv, e2e_max_len, ws,
                      partition_tokens=args.partition_tokens)
    d1.record(stream)
    torch.cuda.synchronize(dev)
    dec_ms = [d0.elapsed_time(d1) / K2]
    K3 = min(K, 100)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K3)]
    for k in range(K3):
        ops.pa_reshape_and_cache(new_k, new_v, t_slots, kc, vc)
        ev[k][0].record(stream)
        ops.pa_decode(out, q, kc, vc, t_tables, t_lens, wl.scale, Hkv, e2e_max_len, ws,
                      partition_tokens=args.partition_tokens)
        ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    sampler.mark(w0b, time.time())
    dec_pair_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    dev_status = ops.pa_workspace_error(ws)
    if dev_status != 0:
        raise RuntimeError(f"device status {dev_status} after the timed steps")
    if args.profile:
        # profiling case: device-resident steps only
        sampler.stop()
        print(json.dumps({"profile": True, "num_seqs": B, "steps": K, "ms_per_step": total_ms / K,
                          "partition_tokens": ops.pa_decode_plan(B, H, Hkv, D, bs, "bf16", e2e_max_len,
                                                                 args.partition_tokens)[0],
                          "decode_ms": statistics.mean(dec_ms),
                          "decode_gbs": decode_bytes / (statistics.mean(dec_ms) * 1e-3) / 1e9,
                          "decode_bytes": decode_bytes}), flush=True)
        return

    # ---------------- end to end through the C ABI, host buffers ----------------
    # The e2e leg replays the last R decode steps of every sequence: a fresh
    # allocator state holds max(1, len - R) history tokens per sequence, and
    # each timed step reserves one more slot per sequence on the host,
    # copies that step's inputs from pinned host memory, runs the kernels and
    # reads the output back.  Steps alternate between two sets of pinned and
    # device buffers, so the host prepares step k + 1 while step k runs; an
    # event per set orders each reuse.
    R = min(K, 128)
    e2e_warm = min(Wm, 3)
    alloc2 = ops.BlockAllocator(NB, bs, free_order)
    seqs2 = [alloc2.seq_create() for _ in range(B)]
    start_len = np.maximum(1, wl.context_lens.astype(np.int64) - R)
    hist2 = np.concatenate([alloc2.append_tokens(s, int(n)) for s, n in zip(seqs2, start_len)])
    sel = np.concatenate([np.arange(st[i], st[i] + start_len[i]) for i in range(B)])
    ops.pa_reshape_and_cache(
        torch.from_numpy(np.ascontiguousarray(wl.key_hist.bits[sel])).view(torch.bfloat16).to(dev),
        torch.from_numpy(np.ascontiguousarray(wl.value_hist.bits[sel])).view(torch.bfloat16).to(dev),
        torch.from_numpy(hist2).to(dev), kc, vc)
    torch.cuda.synchronize(dev)
    # one staging area per buffer set holds all of a step's inputs, so a step
    # uploads them with one copy: q | k | v | slots | tables | lens, each
    # section 256-byte aligned (views of one pinned / one device byte buffer)
    sections = [("q", (B, H, D), torch.bfloat16), ("k", (B, Hkv, D), torch.bfloat16),
                ("v", (B, Hkv, D), torch.bfloat16), ("slots", (B,), torch.int64),
                ("tables", (B, maxb), torch.int32), ("lens", (B,), torch.int32)]
    offs, total = {}, 0
    for name, shape, dt in sections:
        offs[name] = total
        total += -(-int(np.prod(shape)) * torch.empty((), dtype=dt).element_size() // 256) * 256

    def views(buf):
        out_v = {}
        for name, shape, dt in sections:
            n = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
            out_v[name] = buf[offs[name]:offs[name] + n].view(dt).view(shape)
        return out_v

    h_stage = [torch.zeros(total, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    d_stage = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    hb = [views(x) for x in h_stage]
    db = [views(x) for x in d_stage]
    for x in hb:   # the synthetic q / new K / new V are the same every step
        x["q"].copy_(torch.from_numpy(np.ascontiguousarray(wl.q.bits)).view(torch.bfloat16))
        x["k"].copy_(new_k.cpu())
        x["v"].copy_(new_v.cpu())
    b_np = [{k_: x[k_].numpy() for k_ in ("slots", "tables", "lens")} for x in hb]
    seqs_np = np.asarray(seqs2, dtype=np.int32)
    h_out = [torch.empty((B, H, D), dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    d_out = [torch.empty_like(out) for _ in range(2)]
    h_pairs = torch.empty((B, 2), dtype=torch.int64, pin_memory=True)
    d_pairs = torch.empty((B, 2), dtype=torch.int64, device=dev)
    # Each step is one upload of its staging area (stream `up`), the append
    # and the decode, captured once per buffer set as a CUDA graph and
    # replayed (stream `cs`), and one download of its output (stream
    # `down`); per-set events order the three, so the upload of step k + 1
    # and the download of step k - 1 overlap the kernels of step k, and the
    # host only runs the allocator and fills the pinned staging area.
    up, cs, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    graphs = [None, None]
    ev_up = [torch.cuda.Event() for _ in range(2)]     # set j's inputs are on the device
    ev_comp = [torch.cuda.Event() for _ in range(2)]   # set j's kernels are done
    ev_down = [torch.cuda.Event() for _ in range(2)]   # set j's output is on the host
    used = [False, False]
    e2e_bytes = []
    counter = [0]
    waited = [0.0]   # host time spent waiting for the GPU inside the steps

    def kernels(j):
        d = db[j]
        ops.pa_reshape_and_cache(d["k"], d["v"], d["slots"], kc, vc)
        ops.pa_decode(d_out[j], d["q"], kc, vc, d["tables"], d["lens"], wl.scale, Hkv, e2e_max_len, ws,
                      partition_tokens=args.partition_tokens)

    def e2e_step():
        j = counter[0] % 2
        counter[0] += 1
        if used[j]:
            w0_ = time.perf_counter()
            ev_down[j].synchronize()                   # set j's last step is complete
            waited[0] += time.perf_counter() - w0_
        # host allocator: reserve the slots and export the tables, straight
        # into the pinned staging area
        _, pairs = alloc2.append_slots(seqs_np, out=b_np[j]["slots"])
        _, ln = alloc2.export_tables(seqs_np, maxb, out=(b_np[j]["tables"], b_np[j]["lens"]))
        with torch.cuda.stream(up):
            d_stage[j].copy_(h_stage[j], non_blocking=True)   # all of the step's inputs
            ev_up[j].record(up)
        with torch.cuda.stream(cs):
            cs.wait_event(ev_up[j])
            if len(pairs):                             # copy-on-write (none in this workload)
                h_pairs.numpy()[:len(pairs)] = pairs
                d_pairs[:len(pairs)].copy_(h_pairs[:len(pairs)], non_blocking=True)
                ops.pa_copy_blocks(kc, vc, d_pairs[:len(pairs)])
                cs.synchronize()                       # h_pairs is reused next step
            if graphs[j] is not None:
                graphs[j].replay()
            else:
                kernels(j)
            ev_comp[j].record(cs)
        with torch.cuda.stream(down):
            down.wait_event(ev_comp[j])
            h_out[j].copy_(d_out[j], non_blocking=True)    # the step's result back to the host
            ev_down[j].record(down)
        used[j] = True
        return ln

    for _ in range(e2e_warm):
        e2e_step()
    torch.cuda.synchronize(dev)
    for j in range(2):                                 # capture after the eager warm-up steps
        graphs[j] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graphs[j], stream=cs):
            kernels(j)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w2 = time.time()
    e0.record(up)
    host_s = 0.0
    waited[0] = 0.0
    for _ in range(R):
        h0 = time.perf_counter()
        ln = e2e_step()
        host_s += time.perf_counter() - h0
        e2e_bytes.append(sum(step_bytes(ln, B, H, Hkv, D, e, 2)))
    e1.record(down)
    torch.cuda.synchronize(dev)
    w3 = time.time()
    sampler.mark(w2, w3)
    e2e_ms = e0.elapsed_time(e1)
    sampler.stop()
    if ops.pa_workspace_error(ws) != 0:
        raise RuntimeError("device status after the e2e steps")

    h2d = total                                        # the staging area, copied whole every step
    d2h = B * H * D * 2

    # max over ranks of the times, sum over ranks of the work
    (t_step, t_dec, t_e2e), (sum_step_b, sum_dec_b, sum_e2e_b, sum_seqs) = reduce_over_ranks(
        [total_ms / K, statistics.mean(dec_ms), e2e_ms / R],
        [decode_bytes + append_bytes, decode_bytes, statistics.mean(e2e_bytes), B], world, dev)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peaks()
    value = sum_step_b / (t_step * 1e-3) / 1e9
    achieved = sum_dec_b / world / (t_dec * 1e-3) / 1e9   # per GPU, at the slowest rank's time
    e2e_val = sum_e2e_b / (t_e2e * 1e-3) / 1e9
    pt, ctas = ops.pa_decode_plan(B, H, Hkv, D, bs, "bf16", e2e_max_len, args.partition_tokens)
    clocks = sampler.summary()
    extras = measure_extras(ops, dev) if world == 1 else None

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_seconds)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": round(t_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "num_seqs": B, "num_q_heads": H, "num_kv_heads": Hkv,
                   "head_dim": D, "block_size": bs, "total_tokens": int(lens.sum()),
                   "max_context_len": max_len, "partition_tokens": pt, "ctas": ctas,
                   "l2": "inputs larger than L2: %.2f GB of KV read per step vs 129 MB L2"
                         % (decode_bytes / 1e9),
                   "parallelism": (f"data-parallel: {world} independent batches of {B} sequences, "
                                   "one per GPU, no collective on the data path")
                                  if world > 1 else "single GPU"},
        "seq_steps_per_s": round(sum_seqs / (t_step * 1e-3), 1),
        "decode_ms": round(t_dec, 5),
        "decode_ms_event_pair_per_launch": round(dec_pair_ms, 5),
        "decode_bytes_per_step": decode_bytes,
        "append_bytes_per_step": append_bytes,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic(), "kernel": "pa_decode",
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "pct_of_nominal_8tbs": round(100 * achieved / 8000.0, 2),
        "e2e": {"value": round(e2e_val, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "seq_steps_per_s": round(sum_seqs / (t_e2e * 1e-3), 1),
                "ms_per_step": round(t_e2e, 5), "steps": R,
                "host_ms_per_step": round((host_s - waited[0]) * 1e3 / R, 5),
                "note": "last R decode steps of each sequence, host allocator in the loop; each step "
                        "uploads its inputs in one copy, replays a CUDA graph of the append and the "
                        "decode, and downloads its output, on three streams over two buffer sets"},
        "gpu_launches": 2 * K,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "extras": extras,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    if len(sys.argv) > 1 and sys.argv[1] == "--_oracle_child":
        _oracle_child(sys.argv[2:])
        return
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--num-seqs", type=int, default=256,
                    help="batch size (the benchmark workload is 256; smaller for profiling)")
    ap.add_argument("--block-size", type=int, default=16,
                    help="KV block size in tokens (the benchmark workload uses 16)")
    ap.add_argument("--partition-tokens", type=int, default=0,
                    help="split-K partition size passed to pa_decode (0 = automatic)")
    ap.add_argument("--profile", action="store_true",
                    help="device-resident steps only (no e2e leg, no CPU baseline)")
    ap.add_argument("--profile-kernels", action="store_true",
                    help="profiling case: --warmup + --steps launches of each secondary kernel "
                         "(append, copy, shared-prefix decode, prefill) at its bench size")
    ap.add_argument("--profile-cuda-core", action="store_true",
                    help="profiling case: only the CUDA-core decode kernel (fp32 K/V) on the batch's "
                         "lengths, --warmup + --steps back-to-back launches")
    ap.add_argument("--profile-prefill", type=int, default=0, metavar="PROMPTS",
                    help="profiling case: only pa_prefill on PROMPTS causal prompts of 2048 tokens "
                         "(32 q / 8 kv heads), --warmup + --steps launches")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.profile_kernels:
        kernel_profile(args)
    elif args.profile_cuda_core:
        cuda_core_profile(args)
    elif args.profile_prefill:
        prefill_profile(args)
    elif args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
