// Paged decode attention on the 5th-generation tensor cores (sm_103a),
// bf16 K/V, head_dim 128, block size 8..256, GQA group G in {1,2,4,8,16}.
//
// Same result as the CUDA-core kernel ("PagedAttention", section "Block
// Table 如何工作": K/V of token t come from the physical block the block table
// names for logical block t / block_size; softmax(scale q.K) V over the
// history).  The GQA group turns both products into dense tiles:
//   S^T[128 tokens x 16] = K_tile[128 x 128 dims] . Q^T[128 dims x 16 heads]
//   O^T[128 dims x N]   += V_tile^T[128 dims x 128 tokens] . P^T[128 tokens x N]
// (heads padded to 16), each a handful of tcgen05.mma instructions with fp32
// accumulators in tensor memory.  P enters the second product as two bf16
// terms, hi = bf16(p) and lo = bf16(p - hi), side by side in the B tile
// (N = 16: columns 0..7 and 8..15 for G <= 8; N = 32 for G = 16), so the
// result keeps about 16 bits of each probability instead of bf16's 8.
//
// One CTA per SM, persistent over (sequence, kv head, partition) work items.
// Items are enumerated from context_lens in shared memory, full partitions
// first and the shorter last partitions after them, longest first, and claimed
// dynamically: the K-stream warp takes the next item index from a global
// counter in the workspace when one of the CTA's two compute groups reaches
// the last tile of its item, and publishes it to that group's queue in shared memory,
// which every other role reads in order.  The two groups' 128-token tiles
// are interleaved into one stream (group 0 tile, group 1 tile, ...) that
// every stream-walking warp derives identically.  The K path and the V path run decoupled,
// each with its own ring of 32 KB stages, streaming warp and MMA warp:
//  * warp 0 streams K: per item it copies the partition's block-table slice
//    into shared memory and loads the query rows (TMA tensor copy); per tile
//    it issues, from one lane per block, one 4-D TMA tensor copy (128-byte
//    swizzle, L2 evict-first) of that block's K rows into the K ring, laid
//    out as [8-row group][64-dim half][8 rows][128 B] so that each 8-row
//    half is one swizzle atom of the K-major (Q.K^T) and MN-major (P.V)
//    operands;
//  * warp 10 streams V the same way into the V ring;
//  * warps 1 and 12 issue Q.K^T (one lane each) of group 0's and group 1's
//    tiles as soon as the tile's K has landed; warp 1 owns the tensor memory
//    (per group: S and O, double-buffered);
//  * warps 11 and 13 issue P.V of group 0's and group 1's tiles once the
//    tile's V has landed and its P is ready (zeroing first the V rows past
//    the end of a sequence inside the tile's last 16-token step).  One
//    issuing thread per group and product keeps a group's tile from waiting
//    behind the other group's in one in-order issuer (an MMA takes a thread
//    about a hundred cycles to issue whatever its size; separate warps
//    issue in parallel);
//  * warps 2-5 and 6-9 are the two compute groups (one thread per token row,
//    then per head-dim row): online softmax in fp32 on the score tile (block
//    max via shuffles + shared memory, exp2 in the log2 domain), P written to
//    shared memory as bf16 hi/lo, rescale-and-accumulate of each tile's P.V
//    in registers, and the item's epilogue: store, or write (max, sum,
//    unnormalised O) and, in the last CTA to finish a (sequence, kv head),
//    merge the partitions by log-sum-exp.
// Rows past the end of a sequence: their scores are masked, their P is 0,
// V rows inside the last 16-token MMA step are zeroed in shared memory, and
// later steps are not issued, so stale or uninitialised memory never enters
// the sums.  Every mbarrier wait is made by a role that consumed the
// previous phase of the same barrier itself, so no parity wait can alias a
// phase two ahead.  All mbarrier waits are bounded; on expiry every role stops,
// the MMA lanes drain their work, tensor memory is freed and
// PA_ERR_DEVICE_TIMEOUT is written to the workspace.
#pragma once

#include <cuda.h>

#include "decode_common.cuh"

namespace pa {

// warps: 0 K stream, 1 / 12 Q.K^T MMA of group 0 / 1, 2-9 compute, 10 V
// stream, 11 / 13 P.V MMA of group 0 / 1
constexpr int kUmmaThreads = 448;
constexpr int kUmmaTile = 128;           // tokens per tile (MMA M)
constexpr int kUmmaTileBytes = 32768;    // one K or V tile: 16 row groups x 2 halves x 8 rows x 128 B
constexpr int kUmmaMaxStages = 8;
constexpr int kUmmaQBytes = 4096;        // query tile: 2 halves x 16 rows x 128 B (one per group)
// per compute group: maxima and rescale factors [2][4][16] + [2][16] floats,
// then the row-sum scratch: [4][16] while an item's totals stay in registers
// (one kv head per item, G <= 4), or [2][4][16] + the final maxima [2][16]
// when they go through shared memory (HG = KH * G query heads per item)
__host__ __device__ constexpr int umma_small_bytes(int HG, int KH) {
  return (HG >= 8 || KH == 2) ? 1280 : 1024;
}
constexpr int kUmmaGroupBars = 16;
constexpr int kUmmaQueue = 8;            // per-group item queue depth
constexpr int kUmmaQueueReaders = 9;     // V stream, 2 Q.K and 2 P.V warps, a group's 4 compute warps
constexpr int kUmmaBarriers = 6 * kUmmaMaxStages + 2 * kUmmaGroupBars + 4 + 4 * kUmmaQueue + 1;

__host__ __device__ constexpr int umma_p_bytes(int G) { return G <= 8 ? 4096 : 8192; }

namespace umma_detail {

// barrier indices: K ring, V ring, per-group blocks, drains.  A ring slot
// has two "full" barriers that its successive fills use in turn: the two
// groups' MMA warps consume the shared rings independently, and a consumer
// waiting for fill k of a slot may find fill k - 1 not yet landed but never
// fill k - 2 (its own previous tile was at most two tiles back, which forced
// fill k - 1 to be issued, which needs fill k - 2 released), so a parity
// wait on the copy used by fills k - 2, k, k + 2 cannot alias.
constexpr int kKFull = 0;                          // [fill parity][stage]
constexpr int kKEmpty = 2 * kUmmaMaxStages;
constexpr int kVFull = 3 * kUmmaMaxStages;         // [fill parity][stage]
constexpr int kVEmpty = 5 * kUmmaMaxStages;
constexpr int kGroup0 = 6 * kUmmaMaxStages;
// within a group's block of kUmmaGroupBars
constexpr int kQFull = 0, kQEmpty = 2, kSFull = 4, kSEmpty = 6, kPFull = 8, kPEmpty = 10,
              kOFull = 12, kOEmpty = 14;
constexpr int kDrainQK = 6 * kUmmaMaxStages + 2 * kUmmaGroupBars;   // [group]
constexpr int kDrainPV = kDrainQK + 2;                               // [group]
constexpr int kItemFull = kDrainPV + 2;                   // [group][kUmmaQueue]
constexpr int kItemEmpty = kItemFull + 2 * kUmmaQueue;    // [group][kUmmaQueue]
constexpr int kNever = kItemEmpty + 2 * kUmmaQueue;       // no role ever arrives (timeout-path test)

// An item: partition `part` of sequence `seq` for kv-head group `kvg` (kv
// heads kvg * KH .. kvg * KH + KH - 1, KH = 1 or 2 per item).
struct Item {
  int seq, kvg, part, len, t0, ntok, nparts;
};

// Item enumeration: first every full partition (part_tokens tokens) of
// every sequence, sequence-major, kv head fastest; then the sequences' last,
// shorter partitions (a sequence of length 0: one empty item per kv head),
// longest first: by 128-token tile count (counts of kTailBuckets - 1 and
// more share one class), sequence order within a count, empty ones last; kv
// head fastest.  Every CTA derives the same order from context_lens, so an
// item index names the same work in every CTA; handing out the long work
// first leaves short items for the end of the launch, where they even out
// the CTAs' finishing times.
constexpr int kTailBuckets = 64;

struct Ctx {
  const DecodeParams* p;
  const int32_t* prefix_full;  // exclusive prefix of the full-partition item counts
  const int32_t* tail_seq;     // sequences with a last partition, in item order
  const int32_t* lens;
  int n_full, total;
  int nkg;                     // kv-head groups per sequence (num_kv_heads / KH)
  int tile_tokens;             // tokens per 128-row tile (128 / KH)
};

// First s with prefix[s + 1] > w (prefix non-decreasing, prefix[0] = 0).
__device__ __forceinline__ int seq_of(int w, const int32_t* prefix, int nseq) {
  int lo = 0, hi = nseq - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid + 1] > w) hi = mid;
    else lo = mid + 1;
  }
  return lo;
}

__device__ __forceinline__ Item item_at(const Ctx& c, int w) {
  Item it;
  const int nkg = c.nkg;
  const int pt = c.p->part_tokens;
  if (w < c.n_full) {
    it.seq = seq_of(w, c.prefix_full, c.p->num_seqs);
    const int u = w - c.prefix_full[it.seq];
    it.part = u / nkg;
    it.kvg = u - it.part * nkg;
  } else {
    const int v = w - c.n_full;
    const int sp = v / nkg;
    it.seq = c.tail_seq[sp];
    it.kvg = v - sp * nkg;
    it.part = c.lens[it.seq] / pt;
  }
  it.len = c.lens[it.seq];
  it.t0 = it.part * pt;
  it.ntok = min(it.len - it.t0, pt);
  it.nparts = it.len > 0 ? (it.len + pt - 1) / pt : 1;
  return it;
}

// Class of a sequence's last partition: -1 none (length a positive multiple
// of the partition), 0 empty sequence, else its 128-token tile count capped.
__device__ __forceinline__ int tail_class(int len, int pt) {
  if (len == 0) return 0;
  const int r = len % pt;
  if (r == 0) return -1;
  return min((r + kUmmaTile - 1) / kUmmaTile, kTailBuckets - 1);
}

// Builds lens, prefix_full and tail_seq and returns the number of sequences
// with a last partition; every thread calls it; the CTA is synchronised on
// return.  scratch: (nthreads / 32 + 1) * kTailBuckets + 1 ints of shared
// memory that no role touches before the set-up ends.  CTA 0 reports lengths
// outside [0, max_context_len] in the workspace error word.
//
// The tail order is a stable counting sort spread over every warp: thread t
// takes a run of `per` consecutive sequences, so warp w covers a contiguous
// range; each warp counts its range's sequences per class, one warp turns the
// counts into each (warp, class) pair's first position (classes longest
// first, warps in sequence order within a class), and each warp then places
// its own range, 32 sequences per round.
__device__ __forceinline__ int build_item_order(const DecodeParams& p, int32_t* lens,
                                                int32_t* prefix_full, int32_t* tail_seq,
                                                int* warp_sums, int* scratch, int tid, int nthreads,
                                                int nkg) {
  const int nseq = p.num_seqs, pt = p.part_tokens;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
  int* cnt = scratch;                              // [warp][class]: counts, then first positions
  int* n_tail_word = scratch + nwarps * kTailBuckets;
  const int per = (nseq + nthreads - 1) / nthreads;
  const int beg = min(nseq, tid * per);
  const int end = min(nseq, beg + per);
  for (int i = tid; i < nwarps * kTailBuckets; i += nthreads) cnt[i] = 0;
  __syncthreads();
  int lf = 0;
  for (int i = beg; i < end; ++i) {
    const int raw = p.context_lens[i];
    if (blockIdx.x == 0 && (raw < 0 || raw > p.max_context_len)) atomicExch(p.ws_err, kDevErrInvalidArg);
    const int len = decode_detail::clamp_len(raw, p.max_context_len);
    lens[i] = len;
    lf += (len / pt) * nkg;
    const int c = tail_class(len, pt);
    if (c >= 0) atomicAdd(&cnt[warp * kTailBuckets + c], 1);
  }
  int xf = lf;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int yf = __shfl_up_sync(0xffffffffu, xf, off);
    if (lane >= off) xf += yf;
  }
  if (lane == 31) warp_sums[warp] = xf;
  __syncthreads();
  int rf = xf - lf;
  for (int w = 0; w < warp; ++w) rf += warp_sums[w];
  for (int i = beg; i < end; ++i) {
    prefix_full[i] = rf;
    rf += (lens[i] / pt) * nkg;
  }
  if (tid == nthreads - 1) prefix_full[nseq] = rf;
  if (warp == 0) {
    // class totals and bases, longest class first: lane l owns classes
    // 63 - 2l and 62 - 2l; then each warp's first position per class
    static_assert(kTailBuckets == 64, "two classes per lane");
    const int ca = kTailBuckets - 1 - 2 * lane, cb = ca - 1;
    int ta = 0, tb = 0;
    for (int w = 0; w < nwarps; ++w) {
      ta += cnt[w * kTailBuckets + ca];
      tb += cnt[w * kTailBuckets + cb];
    }
    int x = ta + tb;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    const int total = __shfl_sync(0xffffffffu, x, 31);
    int ra = x - ta - tb, rb = ra + ta;
    for (int w = 0; w < nwarps; ++w) {
      const int na = cnt[w * kTailBuckets + ca], nb = cnt[w * kTailBuckets + cb];
      cnt[w * kTailBuckets + ca] = ra;
      cnt[w * kTailBuckets + cb] = rb;
      ra += na;
      rb += nb;
    }
    if (lane == 0) *n_tail_word = total;
  }
  __syncthreads();
  // stable placement of this warp's range, 32 sequences per round
  const int wbeg = min(nseq, warp * 32 * per), wend = min(nseq, (warp + 1) * 32 * per);
  int* wcnt = cnt + warp * kTailBuckets;
  for (int c = wbeg; c < wend; c += 32) {
    const int s = c + lane;
    const int k = s < wend ? tail_class(lens[s], pt) : -1;
    const unsigned m = __match_any_sync(0xffffffffu, k);
    const int rank = __popc(m & ((1u << lane) - 1u));
    const int pos = k >= 0 ? wcnt[k] + rank : 0;
    __syncwarp();
    if (k >= 0) {
      tail_seq[pos] = s;
      if (rank == 0) wcnt[k] += __popc(m);
    }
    __syncwarp();
  }
  __syncthreads();
  const int n_tail = *n_tail_word;
  // the scratch is later overwritten by tensor copies (the async proxy)
  ptx::fence_proxy_async_smem();
  __syncthreads();  // the scratch belongs to later roles from here on
  return n_tail;
}

// One compute group's item sequence, as published in its queue.
struct GroupIter {
  int j, nt;
  uint32_t k;      // queue entries consumed so far
  uint32_t items;  // non-empty items started so far (query slot phase)
  bool valid;
  Item it;
};

// One tile of the merged stream.
struct Rec {
  int g;          // compute group
  Item it;
  int j, nt, nv;  // tile index in the item, tiles of the item, valid tokens
  uint32_t u;     // tile index in the CTA's stream (stage u % depth of each ring)
  uint32_t ug;    // tile index within the group (S/P/O buffers)
  uint32_t qi;    // item index within the group (query slot phase)
};

// Next item of group g from `next_w(g, k)` (the publisher claims and
// publishes, readers read the queue); empty items go to on_empty.
template <typename NextW, typename OnEmpty>
__device__ __forceinline__ void seek(const Ctx& c, GroupIter& s, int g, NextW&& next_w,
                                     OnEmpty&& on_empty) {
  while (true) {
    const int w = next_w(g, s.k++);
    if (w < 0) break;
    s.it = item_at(c, w);
    if (s.it.ntok > 0) {
      s.nt = (s.it.ntok + c.tile_tokens - 1) / c.tile_tokens;
      s.j = 0;
      s.valid = true;
      return;
    }
    on_empty(g, s.it);
  }
  s.valid = false;
}

struct Stream {
  GroupIter a, b;  // the two groups' item iterators (named: no dynamic indexing)
  int turn;
  uint32_t u, ua, ub;

  template <typename NextW, typename OnEmpty>
  __device__ __forceinline__ void init(const Ctx& c, NextW&& next_w, OnEmpty&& on_empty) {
    a.k = a.items = 0;
    b.k = b.items = 0;
    seek(c, a, 0, next_w, on_empty);
    seek(c, b, 1, next_w, on_empty);
    turn = 0;
    u = ua = ub = 0;
  }

  template <typename NextW, typename OnEmpty>
  __device__ __forceinline__ void take(const Ctx& c, GroupIter& s, int g, uint32_t& ug, Rec& r,
                                       NextW&& next_w, OnEmpty&& on_empty) {
    r.g = g;
    r.it = s.it;
    r.j = s.j;
    r.nt = s.nt;
    r.nv = min(c.tile_tokens, s.it.ntok - s.j * c.tile_tokens);
    r.u = u++;
    r.ug = ug++;
    r.qi = s.items;
    if (++s.j == s.nt) {
      ++s.items;
      seek(c, s, g, next_w, on_empty);
    }
    turn = g ^ 1;
  }

  template <typename NextW, typename OnEmpty>
  __device__ __forceinline__ bool next(const Ctx& c, Rec& r, NextW&& next_w, OnEmpty&& on_empty) {
    // alternate groups; when one group has no work left, take from the other
    const bool use_b = turn ? b.valid : !a.valid;
    if (use_b) {
      if (!b.valid) return false;
      take(c, b, 1, ub, r, next_w, on_empty);
    } else {
      if (!a.valid) return false;
      take(c, a, 0, ua, r, next_w, on_empty);
    }
    return true;
  }
};

struct NoOp {
  __device__ __forceinline__ void operator()(int, const Item&) const {}
};

// Bounded wait; once a role has given up, its later waits are skipped.
// `stop` is the CTA's shared stop word: a role that gives up raises it, and
// every role still spinning gives up at once rather than after its own limit.
__device__ __forceinline__ void wait(uint64_t* bar, uint32_t parity, bool& aborted,
                                     volatile int* stop, uint64_t limit_ns = kWaitLimitNs) {
  if (aborted || ptx::mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = ptx::global_ns();
  while (!ptx::mbar_try_wait_sleep(bar, parity, ptx::kSleepHintNs)) {
    if (*stop || ptx::global_ns() - t0 > limit_ns) {
      aborted = true;
      *stop = 1;
      return;
    }
  }
}

// Wait for work already issued (copies, MMAs) to finish before the CTA
// exits: bounded by the default limit and not cut short by the stop word.
__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  return ptx::mbar_wait(bar, parity, kWaitLimitNs);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 2^x by the ex2.approx.ftz instruction (relative error about 2^-22; -inf
// and very negative x give 0)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace umma_detail

// KH kv heads per item (1, or 2 for G <= 4 and blocks of 8..64 tokens): a
// tile then holds 128 / KH tokens of each of the item's kv heads, its rows
// block by block and, within a block, kv head by kv head, as one block's K
// (or V) of consecutive kv heads lies in the pool; one TMA box per block
// covers both heads.  Q.K^T puts all KH x G heads against every row (row r
// keeps the G columns of its own kv head); P is block-diagonal (row r has
// non-zero columns only for its kv head's G heads), so P.V gives every head
// its own output.  Both products keep their shapes (N = 16).
template <int G, int KH>
__global__ void __launch_bounds__(kUmmaThreads, 1)
    paged_decode_umma_kernel(const __grid_constant__ DecodeParams p,
                             const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v,
                             const __grid_constant__ CUtensorMap tm_q) {
  using namespace umma_detail;
  static_assert(G == 1 || G == 2 || G == 4 || G == 8 || G == 16, "GQA group");
  static_assert(KH == 1 || (KH == 2 && G <= 4), "kv heads per item");
  constexpr int HD = 128;
  constexpr int HG = KH * G;               // query heads of an item
  constexpr int TT = kUmmaTile / KH;       // tokens per tile
  constexpr int NP = HG <= 8 ? 16 : 32;    // P.V columns: hi heads, then lo heads
  constexpr int LO = NP / 2;               // column of the lo half
  constexpr int PGRP = NP / 8;             // 8-column core matrices per P row group
  constexpr int PB = umma_p_bytes(HG);     // one P buffer
  constexpr uint32_t TMEM_COLS = HG <= 8 ? 128 : 256;  // S[2][2] x 16, then O[2][2] x NP

  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int NSK = p.stages;                 // K ring stages
  const int NSV = p.stages_v;               // V ring stages
  unsigned char* kring = smem;
  unsigned char* vring = smem + NSK * kUmmaTileBytes;
  unsigned char* qbuf = smem + p.off_q;    // [group] x 4 KB
  unsigned char* pbuf = smem + p.off_p;    // [group][buffer] x PB
  unsigned char* small = smem + p.off_small;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kUmmaBarriers);
  // [0] a streaming or MMA role gave up, [1..2] group merges its item,
  // [3..4] group gave up, [5] the stop word (some role gave up)
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* stop = flags + 5;
  int* warp_sums = const_cast<int*>(flags) + 6;   // one int per warp
  int32_t* tbl = reinterpret_cast<int32_t*>(smem + p.off_tbl);  // [K/V stream][group][tbl_stride]
  int32_t* lens = reinterpret_cast<int32_t*>(smem + p.off_lens);
  int32_t* prefix_full = reinterpret_cast<int32_t*>(smem + p.off_prefix);
  int32_t* tail_seq = prefix_full + ((p.num_seqs + 4) & ~3);
  constexpr int kSmall = umma_small_bytes(HG, KH);
  volatile int* queue = reinterpret_cast<volatile int*>(small + 2 * kSmall);  // [group][kUmmaQueue]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int hkv = p.num_kv_heads;
  const int bs = p.block_size;
  const int bs_log_c = __ffs(bs) - 1;  // block size is a power of two

  // barriers: one per thread, each initialiser fencing its own inits
  if (tid < kUmmaBarriers) {
    uint32_t count = 1;
    if (tid >= kGroup0 && tid < kGroup0 + 2 * kUmmaGroupBars) {
      const int gi = (tid - kGroup0) % kUmmaGroupBars;
      if ((gi >= kSEmpty && gi < kSEmpty + 2) || (gi >= kPFull && gi < kPFull + 2) ||
          (gi >= kOEmpty && gi < kOEmpty + 2))
        count = 4;  // one arrival per compute warp
    } else if (tid >= kItemEmpty && tid < kItemEmpty + 2 * kUmmaQueue) {
      count = kUmmaQueueReaders;
    }
    ptx::mbar_init(&bars[tid], count);
    ptx::mbar_init_fence();
  }
  if (tid < 6) flags[tid] = 0;
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, TMEM_COLS);
    ptx::tc_fence_before();
  }
  // launched behind the step's append with programmatic serialisation, the
  // set-up above overlaps it; every input is read after this point
  ptx::griddep_wait();
  // the K ring is idle until the set-up ends: it holds the sort's scratch
  const int nkg = hkv / KH;
  const int n_tail = build_item_order(p, lens, prefix_full, tail_seq, warp_sums,
                                      reinterpret_cast<int*>(kring), tid, kUmmaThreads, nkg);  // syncs
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_full = prefix_full[p.num_seqs];
  const Ctx ctx{&p, prefix_full, tail_seq, lens, n_full, n_full + n_tail * nkg, nkg, TT};
  bool aborted = false;
  int* item_counter = p.ws_err + 1;   // next unclaimed item (all CTAs)
  int* done_counter = p.ws_err + 2;   // CTAs finished

  // Readers of group g's queue: lane 0 waits for entry k, reads it and
  // frees it; the warp gets it by shuffle.  -1 ends the group.
  auto read_item = [&](int g, uint32_t k) -> int {
    int w = -1;
    if (lane == 0) {
      const int slot = g * kUmmaQueue + static_cast<int>(k % kUmmaQueue);
      wait(&bars[kItemFull + slot], (k / kUmmaQueue) & 1u, aborted, stop);
      if (!aborted) w = queue[slot];
      ptx::mbar_arrive(&bars[kItemEmpty + slot]);
    }
    return __shfl_sync(0xffffffffu, w, 0);
  };

  if (warp == 0 || warp == 10) {
    // ============================ TMA streaming ============================
    // warp 0: query rows and K tiles; warp 10: V tiles
    const bool is_v = warp == 10;
    if (lane == 0) {
      ptx::prefetch_tensormap(is_v ? &tm_v : &tm_k);
      if (!is_v) ptx::prefetch_tensormap(&tm_q);
    }
    const uint64_t pol_kv = ptx::policy_evict_first();
    const uint64_t pol_q = ptx::policy_evict_normal();
    const CUtensorMap* tm = is_v ? &tm_v : &tm_k;
    unsigned char* ring = is_v ? vring : kring;
    uint64_t* full = bars + (is_v ? kVFull : kKFull);
    uint64_t* empty = bars + (is_v ? kVEmpty : kKEmpty);
    const int NS = is_v ? NSV : NSK;
    // a box: box_tok tokens of each of the item's KH kv heads (KH = 2: one
    // whole block of both heads)
    const int box_tok = KH == 1 ? min(bs, kUmmaTile) : bs;
    const int box_rows = KH * box_tok;
    const int bs_log = __ffs(bs) - 1;  // block size is a power of two
    // warp 0 claims items for both groups and publishes them; warp 10 reads.
    // Each group's first item is fixed by the CTA index (items blockIdx.x and
    // gridDim.x + blockIdx.x: the first 2 * gridDim.x items, the longest, need
    // no claim at the start of the launch); later ones are claimed from the
    // shared counter, only when the stream takes a group's last tile of its
    // current item, so no CTA holds work another could start sooner.
    auto publish_item = [&](int g, uint32_t k) -> int {
      int w = -1;
      if (lane == 0) {
        const int slot = g * kUmmaQueue + static_cast<int>(k % kUmmaQueue);
        wait(&bars[kItemEmpty + slot], ((k / kUmmaQueue) & 1u) ^ 1u, aborted, stop);
        if (!aborted) {
          w = k == 0 ? g * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x)
                     : atomicAdd(item_counter, 1) + 2 * static_cast<int>(gridDim.x);
          if (w >= ctx.total) w = -1;
        }
        queue[slot] = w;
        ptx::mbar_arrive(&bars[kItemFull + slot]);
      }
      return __shfl_sync(0xffffffffu, w, 0);
    };
    auto next_w = [&](int g, uint32_t k) -> int { return is_v ? read_item(g, k) : publish_item(g, k); };
    // block-table slice of the group's current item, [stream][group] in shared memory
    auto slice = [&](int g) -> int32_t* { return tbl + ((is_v ? 2 : 0) + g) * p.tbl_stride; };
    Stream st;
    st.init(ctx, next_w, NoOp{});
    int slot = 0;
    uint32_t wrap = 0;   // fills of each slot so far: full copy wrap & 1, empty parity
    uint32_t nfill = 0;  // ring fills whose copies were issued (fill n: slot n % NS)
    uint32_t qfill0 = 0, qfill1 = 0;  // query fills issued per group (K stream)
    Rec r;
    while (!aborted && st.next(ctx, r, next_w, NoOp{})) {
      int32_t* gtbl = slice(r.g);
      const int b0 = r.it.t0 >> bs_log;
      if (r.j == 0) {
        const int nb = ((r.it.t0 + r.it.ntok + bs - 1) >> bs_log) - b0;
        const int32_t* trow = p.block_tables + static_cast<int64_t>(r.it.seq) * p.max_blocks_per_seq + b0;
        for (int j0 = 0; j0 < nb; j0 += 128) {  // four loads in flight per lane, then the stores
          int v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = j0 + 32 * u + lane;
            v[u] = j < nb ? __ldg(trow + j) : 0;
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = j0 + 32 * u + lane;
            if (j < nb) gtbl[j] = v[u];
          }
        }
        __syncwarp();
        if (!is_v && lane == 0) {
          uint64_t* gb = bars + kGroup0 + r.g * kUmmaGroupBars;
          wait(&gb[kQEmpty], (r.qi & 1u) ^ 1u, aborted, stop);
          if (!aborted) {
            ptx::mbar_arrive_expect_tx(&gb[kQFull], 2u * HG * 128u);
            unsigned char* qd = qbuf + r.g * kUmmaQBytes;
            for (int h = 0; h < 2; ++h)
              ptx::tma_load_2d(qd + h * 2048, &tm_q, 64 * h, r.it.seq * p.num_q_heads + r.it.kvg * HG,
                               &gb[kQFull], pol_q);
            if (r.g) qfill1 = r.qi + 1;
            else qfill0 = r.qi + 1;
          }
        }
      }
      // this lane's block of the tile (lanes < nbox)
      const int tok0 = r.it.t0 + r.j * TT;
      const int nbox = (r.nv + box_tok - 1) / box_tok;
      int row = 0;
      if (lane < nbox) {
        const int tok = tok0 + lane * box_tok;
        const int lb = tok >> bs_log;
        int phys = gtbl[lb - b0];
        if (phys < 0 || phys >= p.num_blocks) {  // never read outside the pool
          atomicExch(p.ws_err, kDevErrInvalidArg);
          phys = 0;
        }
        row = ((phys * hkv + r.it.kvg * KH) << bs_log) + (tok - (lb << bs_log));
      }
      uint64_t* fb = &full[(wrap & 1u) * kUmmaMaxStages + slot];
      if (lane == 0) {
        wait(&empty[slot], (wrap & 1u) ^ 1u, aborted, stop);
        if (!aborted) ptx::mbar_arrive_expect_tx(fb, static_cast<uint32_t>(nbox * box_rows * 256));
      }
      aborted = __shfl_sync(0xffffffffu, aborted, 0);
      if (aborted) break;
      if (lane < nbox) {
        unsigned char* dst = ring + slot * kUmmaTileBytes + lane * box_rows * 256;
        ptx::tma_load_4d(dst, tm, 0, 0, 0, row >> 3, fb, pol_kv);
      }
      ++nfill;
      __syncwarp();
      if (++slot == NS) {
        slot = 0;
        ++wrap;
      }
    }
    if (lane == 0 && (aborted || *stop)) {
      // The copies this warp issued must land before the CTA exits: wait for
      // the last fill of every slot (earlier fills of a slot completed before
      // its next fill was issued) and, on the K stream, each group's last
      // query fill.
      const uint32_t first = nfill > static_cast<uint32_t>(NS) ? nfill - NS : 0u;
      for (uint32_t n = first; n < nfill; ++n) {
        const uint32_t s = n % NS, w = n / NS;
        drain_wait(&full[(w & 1u) * kUmmaMaxStages + s], (w >> 1) & 1u);
      }
      if (!is_v && qfill0 > 0) drain_wait(&bars[kGroup0 + kQFull], (qfill0 - 1u) & 1u);
      if (!is_v && qfill1 > 0) drain_wait(&bars[kGroup0 + kUmmaGroupBars + kQFull], (qfill1 - 1u) & 1u);
    }
  } else if (warp == 1 || warp == 12) {
    // ============================ Q.K^T issue ============================
    // warp 1: group 0's tiles (and the tensor memory), warp 12: group 1's
    const int my_g = warp == 12 ? 1 : 0;
    if (lane == 0) {
      constexpr uint32_t kIdQK = ptx::idesc_bf16_f32(128, 16, 0, 0);
      auto read_one = [&](int g, uint32_t k) -> int {
        const int slot = g * kUmmaQueue + static_cast<int>(k % kUmmaQueue);
        wait(&bars[kItemFull + slot], (k / kUmmaQueue) & 1u, aborted, stop);
        const int w = aborted ? -1 : queue[slot];
        ptx::mbar_arrive(&bars[kItemEmpty + slot]);
        return w;
      };
      Stream st;
      st.init(ctx, read_one, NoOp{});
      Rec r;
      int kslot = 0;
      uint32_t kwrap = 0;
      while (!aborted && st.next(ctx, r, read_one, NoOp{})) {
        if (r.g != my_g) {  // the other group's tile: only the ring position advances
          if (++kslot == NSK) {
            kslot = 0;
            ++kwrap;
          }
          continue;
        }
        uint64_t* gb = bars + kGroup0 + r.g * kUmmaGroupBars;
        const uint32_t b = r.ug & 1u, ph = (r.ug >> 1) & 1u;
        if (r.j == 0) wait(&gb[kQFull], r.qi & 1u, aborted, stop);
        wait(&bars[kKFull + (kwrap & 1u) * kUmmaMaxStages + kslot], (kwrap >> 1) & 1u, aborted, stop);
        wait(&gb[kSEmpty + b], ph ^ 1u, aborted, stop);
        if (aborted) break;  // nothing is issued or released past a wait that gave up
        ptx::tc_fence_after();
        const unsigned char* kt = kring + kslot * kUmmaTileBytes;
        const unsigned char* qt = qbuf + r.g * kUmmaQBytes;
        const uint32_t sd = tmem + (r.g * 2 + b) * 16;
        // a rolled loop: smaller code for the SM's warps to share, measured
        // faster than eight unrolled issues
#pragma unroll 1
        for (int kk = 0; kk < 8; ++kk) {
          const int h = kk >> 2, k4 = kk & 3;
          ptx::umma_bf16(sd, ptx::smem_desc(kt + h * 1024 + k4 * 32, 16, 2048, ptx::kLayoutSw128),
                         ptx::smem_desc(qt + h * 2048 + k4 * 32, 16, 1024, ptx::kLayoutSw128), kIdQK,
                         kk > 0);
        }
        ptx::umma_commit(&gb[kSFull + b]);
        ptx::umma_commit(&bars[kKEmpty + kslot]);
        if (r.j == r.nt - 1) ptx::umma_commit(&gb[kQEmpty]);
        if (++kslot == NSK) {
          kslot = 0;
          ++kwrap;
        }
      }
      // nothing may be in flight when tensor memory is freed
      ptx::umma_commit(&bars[kDrainQK + my_g]);
      const bool drained = drain_wait(&bars[kDrainQK + my_g], 0);
      if (aborted || !drained) flags[0] = 1;
    }
    __syncwarp();
  } else if (warp == 11 || warp == 13) {
    // ============================ P.V issue ============================
    // warp 11: group 0's tiles, warp 13: group 1's
    // Lane 0 waits and issues; the whole warp zeroes, in a tile whose last
    // 16-token step is partly past the end of the sequence, the V rows past
    // the end (they may hold stale or uninitialised data and P is 0 there).
    // V tiles are consumed strictly in order, so the wait on the V ring is
    // always for the phase after the one this warp consumed last.
    constexpr uint32_t kIdPV = ptx::idesc_bf16_f32(128, NP, 1, 1);
    Stream st;
    st.init(ctx, read_item, NoOp{});
    const int my_g = warp == 13 ? 1 : 0;
    Rec r;
    int vslot = 0;
    uint32_t vwrap = 0;
    while (!aborted && st.next(ctx, r, read_item, NoOp{})) {
      if (r.g != my_g) {  // the other group's tile: only the ring position advances
        if (++vslot == NSV) {
          vslot = 0;
          ++vwrap;
        }
        continue;
      }
      uint64_t* gb = bars + kGroup0 + r.g * kUmmaGroupBars;
      const uint32_t b = r.ug & 1u, ph = (r.ug >> 1) & 1u;
      unsigned char* vt = vring + vslot * kUmmaTileBytes;
      if (lane == 0) {
        wait(&bars[kVFull + (vwrap & 1u) * kUmmaMaxStages + vslot], (vwrap >> 1) & 1u, aborted, stop);
        wait(&gb[kPFull + b], ph, aborted, stop);
        wait(&gb[kOEmpty + b], ph ^ 1u, aborted, stop);
      }
      aborted = __shfl_sync(0xffffffffu, aborted, 0);
      if (aborted) break;
      int nks;
      if (KH == 1) {
        // the valid rows are a prefix; zero the rest of its last 16-row step
        nks = (r.nv + 15) / 16;
        if (r.nv & 15) {
          const int row0 = r.nv, nrows = nks * 16 - r.nv;   // 1..15 rows, both halves
          for (int c = lane; c < nrows * 16; c += 32) {
            const int rr = row0 + (c >> 4), half = (c >> 3) & 1, ch = c & 7;
            *reinterpret_cast<uint4*>(vt + (rr >> 3) * 2048 + half * 1024 + (rr & 7) * 128 + ch * 16) =
                make_uint4(0, 0, 0, 0);
          }
          ptx::fence_proxy_async_smem();
        }
      } else {
        // the valid rows are the blocks holding a valid token (2 * bs rows
        // each, 16-row steps); in the last one, both heads' rows past the end
        const int nbv = (r.nv + bs - 1) >> bs_log_c;
        nks = (nbv * 2 * bs) / 16;
        const int pv = r.nv - ((nbv - 1) << bs_log_c);      // valid tokens of the last block
        if (pv < bs) {
          const int gap = bs - pv, base = (nbv - 1) * 2 * bs + pv;
          for (int c = lane; c < 2 * gap * 16; c += 32) {
            const int idx = c >> 4, half = (c >> 3) & 1, ch = c & 7;
            const int rr = base + (idx >= gap ? bs + idx - gap : idx);
            *reinterpret_cast<uint4*>(vt + (rr >> 3) * 2048 + half * 1024 + (rr & 7) * 128 + ch * 16) =
                make_uint4(0, 0, 0, 0);
          }
          ptx::fence_proxy_async_smem();
        }
      }
      __syncwarp();
      if (lane == 0) {
        ptx::tc_fence_after();
        const unsigned char* pt = pbuf + (r.g * 2 + b) * PB;
        const uint32_t od = tmem + 64 + (r.g * 2 + b) * NP;
        for (int ks = 0; ks < nks; ++ks)
          ptx::umma_bf16(od, ptx::smem_desc(vt + ks * 4096, 1024, 2048, ptx::kLayoutSw128),
                         ptx::smem_desc(pt + ks * 2 * PGRP * 128, PGRP * 128, 128, ptx::kLayoutNone),
                         kIdPV, ks > 0);
        ptx::umma_commit(&gb[kOFull + b]);
        ptx::umma_commit(&bars[kVEmpty + vslot]);
        ptx::umma_commit(&gb[kPEmpty + b]);
      }
      __syncwarp();
      if (++vslot == NSV) {
        vslot = 0;
        ++vwrap;
      }
    }
    if (lane == 0) {
      ptx::umma_commit(&bars[kDrainPV + my_g]);
      const bool drained = drain_wait(&bars[kDrainPV + my_g], 0);
      if (aborted || !drained) flags[0] = 1;
    }
    __syncwarp();
  } else {
    // ===================== compute groups: softmax, accumulate, epilogue =====================
    const int cg = (warp - 2) >> 2;          // compute group 0 / 1
    const int cw = (warp - 2) & 3;           // warp within the group
    const int ctid = tid - 64 - 128 * cg;    // 0..127 within the group
    const int quarter = warp & 3;            // tensor-memory lanes 32*quarter .. +31
    const int r = 32 * quarter + lane;       // token row of S, head-dim row of O
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const uint32_t bar_id = 1 + cg;
    const float sl2 = p.scale_log2;
    uint64_t* gb = bars + kGroup0 + cg * kUmmaGroupBars;
    unsigned char* gp = pbuf + cg * 2 * PB;
    // Row r's kv head within the item (KH = 2: rows go block by block, and
    // within a block bs rows of the first head, then bs of the second) and
    // its token within the tile.
    const int kl = KH == 1 ? 0 : (r >> bs_log_c) & 1;
    const int rtok = KH == 1 ? r : ((r >> (bs_log_c + 1)) << bs_log_c) + (r & (bs - 1));
    // the two rows that publish each kv head's per-head values: row 0 (the
    // first head) and row bs (the second)
    const bool publisher = r == 0 || (KH == 2 && r == bs);
    // An item's totals (final max, row sums) are needed by its epilogue,
    // which runs after the next tile's softmax.  G <= 4 with one kv head per
    // item keeps them in registers, one copy per tile parity; otherwise each
    // thread holds only its kv head's values or is short of registers (128
    // per thread at 448 threads), and they go through shared memory.
    constexpr bool kTotalsInSmem = HG >= 8 || KH == 2;
    constexpr int NF = kTotalsInSmem ? 1 : G;
    float* red_m = reinterpret_cast<float*>(small + cg * kSmall);  // [2][4][16]
    float* alpha_s = red_m + 2 * 4 * 16;  // [2][16]
    float* red_l = alpha_s + 2 * 16;      // registers: [4][16]; shared: [2][4][16] by tile parity
    float* red_mf = red_l + 2 * 4 * 16;   // shared: [2][16] an item's final max by tile parity
    volatile int* merge_flag = flags + 1 + cg;
    volatile int* gabort = flags + 3 + cg;

    float m_run[G], l_thr[G], o_acc[HG];
    float m_fin0[NF], l_fin0[NF], m_fin1[NF], l_fin1[NF];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m_run[g] = -CUDART_INF_F;
      l_thr[g] = 0.f;
    }
#pragma unroll
    for (int h = 0; h < HG; ++h) o_acc[h] = 0.f;
#pragma unroll
    for (int g = 0; g < NF; ++g) {
      m_fin0[g] = m_fin1[g] = -CUDART_INF_F;
      l_fin0[g] = l_fin1[g] = 0.f;
    }

    auto write_zeros = [&](int g_owner, const Item& it) {
      if (g_owner != cg) return;  // the owning group writes the zero output
      const int64_t ob = (static_cast<int64_t>(it.seq) * p.num_q_heads + it.kvg * HG) * HD + r;
#pragma unroll
      for (int h = 0; h < HG; ++h) decode_detail::store_out(p.out, p.out_bf16, ob + h * HD, 0.f);
    };

    auto softmax = [&](const Rec& t) {
      const uint32_t b = t.ug & 1u, ph = (t.ug >> 1) & 1u;
      const bool first = t.j == 0, last = t.j == t.nt - 1;
      if (first) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          m_run[g] = -CUDART_INF_F;
          l_thr[g] = 0.f;
        }
      }
      wait(&gb[kSFull + b], ph, aborted, stop);
      ptx::tc_fence_after();
      uint32_t sr[HG];
      ptx::TmemLd<HG>::run(tmem + lane_base + (cg * 2 + b) * 16, sr);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&gb[kSEmpty + b]);
      const bool valid = rtok < t.nv;
      float s[G], mx[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const uint32_t v = KH == 1 ? sr[g] : (kl ? sr[(KH - 1) * G + g] : sr[g]);  // this row's head g
        s[g] = valid ? __uint_as_float(v) * sl2 : -CUDART_INF_F;
        mx[g] = s[g];
      }
      // max over the warp's rows of the same kv head (KH = 2, bs < 32: lane
      // bit bs tells the two heads apart, so that step is skipped)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        if (KH == 2 && off == bs) continue;
#pragma unroll
        for (int g = 0; g < G; ++g) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xffffffffu, mx[g], off));
      }
      if (KH == 1) {
        if (lane == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g) red_m[(b * 4 + cw) * 16 + g] = mx[g];
        }
      } else if (bs < 32) {
        // lanes 0 and bs hold the warp's maxima of the two kv heads
        if (lane == 0 || lane == bs) {
#pragma unroll
          for (int g = 0; g < G; ++g) red_m[(b * 4 + cw) * 16 + kl * G + g] = mx[g];
        }
      } else if (lane == 0) {
        // the whole warp is one kv head's rows: the other head gets -inf
#pragma unroll
        for (int g = 0; g < G; ++g) {
          red_m[(b * 4 + cw) * 16 + kl * G + g] = mx[g];
          red_m[(b * 4 + cw) * 16 + (kl ^ 1) * G + g] = -CUDART_INF_F;
        }
      }
      ptx::bar_sync(bar_id, 128);
      float pr[G], al[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const int hh = kl * G + g;
        float mt = red_m[(b * 4) * 16 + hh];
#pragma unroll
        for (int k = 1; k < 4; ++k) mt = fmaxf(mt, red_m[(b * 4 + k) * 16 + hh]);
        const float mn = fmaxf(m_run[g], mt);
        al[g] = fast_exp2(m_run[g] - mn);
        pr[g] = valid ? fast_exp2(s[g] - mn) : 0.f;
        l_thr[g] = l_thr[g] * al[g] + pr[g];
        m_run[g] = mn;
      }
      if (publisher) {
#pragma unroll
        for (int g = 0; g < G; ++g) alpha_s[b * 16 + kl * G + g] = al[g];
      }
      if constexpr (!kTotalsInSmem) {
        if (last) {
#pragma unroll
          for (int g = 0; g < NF; ++g) {
            if (b) {
              m_fin1[g] = m_run[g];
              l_fin1[g] = l_thr[g];
            } else {
              m_fin0[g] = m_run[g];
              l_fin0[g] = l_thr[g];
            }
          }
        }
      }
      // P row r: columns [0, LO) hold hi = p with its low 16 bits cleared
      // (a bf16 value, exact) for heads 0..G-1, columns [LO, NP) the exact
      // fp32 remainder p - hi cut the same way (|p - hi - lo| < 2^-16 p),
      // as bf16 bit patterns; unused heads are zero
      uint32_t pc[NP];
#pragma unroll
      for (int c = 0; c < NP; ++c) pc[c] = 0u;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const uint32_t hb = __float_as_uint(pr[g]) & 0xffff0000u;
        const uint32_t lb = __float_as_uint(pr[g] - __uint_as_float(hb)) >> 16;
        if (KH == 1) {
          pc[g] = hb >> 16;
          pc[LO + g] = lb;
        } else {
          // block-diagonal: this row's kv head's columns only
          pc[g] = kl ? 0u : hb >> 16;
          pc[LO + g] = kl ? 0u : lb;
          pc[(KH - 1) * G + g] = kl ? hb >> 16 : 0u;
          pc[LO + (KH - 1) * G + g] = kl ? lb : 0u;
        }
      }
      uint32_t wp[NP / 2];
#pragma unroll
      for (int k = 0; k < NP / 2; ++k) wp[k] = pc[2 * k] | (pc[2 * k + 1] << 16);
      wait(&gb[kPEmpty + b], ph ^ 1u, aborted, stop);
      unsigned char* prow = gp + b * PB + (r >> 3) * (PGRP * 128) + (r & 7) * 16;
#pragma unroll
      for (int c = 0; c < PGRP; ++c)
        *reinterpret_cast<uint4*>(prow + c * 128) =
            make_uint4(wp[4 * c], wp[4 * c + 1], wp[4 * c + 2], wp[4 * c + 3]);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&gb[kPFull + b]);
      if constexpr (kTotalsInSmem) {
        if (last) {
          // row sums reduced per warp and the final max (the same in every
          // thread), taken after P is handed over.  Slot b is next written
          // two tiles on, past that tile's group barrier, which every warp
          // reaches only after this item's epilogue.
          float lw[G];
#pragma unroll
          for (int g = 0; g < G; ++g) lw[g] = l_thr[g];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
            if (KH == 2 && off == bs) continue;  // sums over rows of the same kv head
#pragma unroll
            for (int g = 0; g < G; ++g) lw[g] += __shfl_xor_sync(0xffffffffu, lw[g], off);
          }
          if (KH == 1 || bs < 32) {
            if (lane == 0 || (KH == 2 && lane == bs)) {
#pragma unroll
              for (int g = 0; g < G; ++g) red_l[(b * 4 + cw) * 16 + kl * G + g] = lw[g];
            }
          } else if (lane == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
              red_l[(b * 4 + cw) * 16 + kl * G + g] = lw[g];
              red_l[(b * 4 + cw) * 16 + (kl ^ 1) * G + g] = 0.f;
            }
          }
          if (publisher) {
#pragma unroll
            for (int g = 0; g < G; ++g) red_mf[b * 16 + kl * G + g] = m_run[g];
          }
        }
      }
    };

    auto epilogue = [&](const Rec& t) {
      float mf[HG], L[HG];
      if constexpr (kTotalsInSmem) {
        // every warp's totals of this item, written in its last tile's softmax
        const int pb = static_cast<int>(t.ug & 1u);
        ptx::bar_sync(bar_id, 128);
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          mf[h] = red_mf[pb * 16 + h];
          L[h] = red_l[(pb * 4) * 16 + h] + red_l[(pb * 4 + 1) * 16 + h] + red_l[(pb * 4 + 2) * 16 + h] +
                 red_l[(pb * 4 + 3) * 16 + h];
        }
      } else {
        float lf[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          mf[g] = (t.ug & 1u) ? m_fin1[g] : m_fin0[g];
          lf[g] = (t.ug & 1u) ? l_fin1[g] : l_fin0[g];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
          for (int g = 0; g < G; ++g) lf[g] += __shfl_xor_sync(0xffffffffu, lf[g], off);
        if (lane == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g) red_l[cw * 16 + g] = lf[g];
        }
        ptx::bar_sync(bar_id, 128);
#pragma unroll
        for (int g = 0; g < G; ++g) L[g] = red_l[g] + red_l[16 + g] + red_l[32 + g] + red_l[48 + g];
      }
      const int64_t obase = (static_cast<int64_t>(t.it.seq) * p.num_q_heads + t.it.kvg * HG) * HD + r;
      if (t.it.nparts == 1) {
#pragma unroll
        for (int h = 0; h < HG; ++h)
          decode_detail::store_out(p.out, p.out_bf16, obase + h * HD, o_acc[h] / L[h]);
        return;
      }
      const int row = t.it.seq * nkg + t.it.kvg;
      const int64_t rec = static_cast<int64_t>(row) * p.max_parts + t.it.part;
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        p.ws_o[(rec * HG + h) * HD + r] = o_acc[h];
        if (ctid == h) {
          p.ws_ml[rec * HG * 2 + 2 * h] = mf[h];
          p.ws_ml[rec * HG * 2 + 2 * h + 1] = L[h];
        }
      }
      // release: every writer orders its partial stores before the barrier;
      // the counting thread acquires right after the atomic and only then
      // publishes the result to the group
      __threadfence();
      ptx::bar_sync(bar_id, 128);
      if (ctid == 0) {
        const int arrived = atomicAdd(&p.ws_counters[row], 1);
        __threadfence();
        *merge_flag = (arrived == t.it.nparts - 1) ? 1 : 0;
      }
      ptx::bar_sync(bar_id, 128);
      if (*merge_flag) {
        // last partition of this (sequence, kv-head group) to finish: merge
        // all heads at once so the partial loads are independent
        const float* ml = p.ws_ml + static_cast<int64_t>(row) * p.max_parts * HG * 2;
        const float* os = p.ws_o + static_cast<int64_t>(row) * p.max_parts * HG * HD + r;
        const int np = t.it.nparts;
        float M[HG], Ls[HG], Os[HG];
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          M[h] = -CUDART_INF_F;
          Ls[h] = 0.f;
          Os[h] = 0.f;
        }
#pragma unroll 4
        for (int q = 0; q < np; ++q)
#pragma unroll
          for (int h = 0; h < HG; ++h) M[h] = fmaxf(M[h], __ldcg(ml + q * HG * 2 + 2 * h));
#pragma unroll 2
        for (int q = 0; q < np; ++q) {
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            const float2 mlq = __ldcg(reinterpret_cast<const float2*>(ml + q * HG * 2 + 2 * h));
            const float wq = exp2f(mlq.x - M[h]);
            Ls[h] = fmaf(wq, mlq.y, Ls[h]);
            Os[h] = fmaf(wq, __ldcg(os + (static_cast<int64_t>(q) * HG + h) * HD), Os[h]);
          }
        }
#pragma unroll
        for (int h = 0; h < HG; ++h) decode_detail::store_out(p.out, p.out_bf16, obase + h * HD, Os[h] / Ls[h]);
        if (ctid == 0) p.ws_counters[row] = 0;
      }
    };

    auto accumulate = [&](const Rec& t) {
      const uint32_t b = t.ug & 1u, ph = (t.ug >> 1) & 1u;
      wait(&gb[kOFull + b], ph, aborted, stop);
      ptx::tc_fence_after();
      uint32_t orr[NP];
      ptx::TmemLd<NP>::run(tmem + lane_base + 64 + (cg * 2 + b) * NP, orr);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&gb[kOEmpty + b]);
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const float o = __uint_as_float(orr[h]) + __uint_as_float(orr[LO + h]);
        o_acc[h] = t.j == 0 ? o : fmaf(o_acc[h], alpha_s[b * 16 + h], o);
      }
      if (t.j == t.nt - 1) epilogue(t);
    };

    // timeout-path test hook: wait, with a short limit, for an event that
    // never comes, so the group gives up and the CTA takes its stop path
    if (p.test_stall_ns) wait(&bars[kNever], 0, aborted, stop, p.test_stall_ns);
    // this group's items only, in queue order
    GroupIter gi;
    gi.k = gi.items = 0;
    seek(ctx, gi, cg, read_item, write_zeros);
    uint32_t ug = 0;
    Rec t, prev;
    bool have_prev = false;
    while (gi.valid) {
      t.g = cg;
      t.it = gi.it;
      t.j = gi.j;
      t.nt = gi.nt;
      t.nv = min(TT, gi.it.ntok - gi.j * TT);
      t.u = 0;
      t.ug = ug++;
      t.qi = gi.items;
      if (++gi.j == gi.nt) {
        ++gi.items;
        seek(ctx, gi, cg, read_item, write_zeros);
      }
      softmax(t);
      if (have_prev) accumulate(prev);
      prev = t;
      have_prev = true;
      if (t.j == t.nt - 1) {
        // item boundary: the group leaves together if any thread gave up
        if (aborted) *gabort = 1;
        ptx::bar_sync(bar_id, 128);
        if (*gabort) break;  // uniform: read after the barrier, written only before one
      }
    }
    ptx::bar_sync(bar_id, 128);
    if (have_prev && !*gabort) accumulate(prev);
  }

  // ============================ teardown ============================
  if (aborted) flags[0] = 1;
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, TMEM_COLS);
  if (tid == 0) {
    if (flags[0] || flags[3] || flags[4] || *stop) atomicExch(p.ws_err, kDevErrTimeout);
    // the last CTA to finish returns the item counter to zero for the next call
    __threadfence();
    if (atomicAdd(done_counter, 1) == static_cast<int>(gridDim.x) - 1) {
      atomicExch(item_counter, 0);
      atomicExch(done_counter, 0);
    }
  }
}

}  // namespace pa
