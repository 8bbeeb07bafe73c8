// Paged prefill attention on the 5th-generation tensor cores (sm_103a):
// bf16 K/V and queries, head_dim 128, block size >= 8, GQA group G in
// {1, 2, 4, 8, 16}.
//
// The other phase of a step ("PagedAttention", section "KV Cache
// 为什么难管理": prefill processes the prompt's tokens together, decode one
// token at a time).  A chunk of a sequence's tokens -- its whole prompt, or
// the next piece of a chunked prefill -- attends causally to its sequence's
// history through the block table ("Block Table 如何工作"): the token at
// position p sees keys 0 .. p, including the chunk's own, whose K/V are
// appended before the call.
//
// Unlike decode, the contraction here is dense: a tile puts 128 query rows
// (TQ = 128 / G tokens x the G query heads of one kv head) against 128 keys,
//   S[128 rows x 128 keys]   = Q[128 x 128 dims] . K_tile^T
//   O[128 rows x 128 dims]  += P[128 x 128 keys] . V_tile
// each eight tcgen05.mma (M = N = 128, K = 16) with fp32 accumulators in
// tensor memory (three S buffers, then O).  P enters the second product as
// bf16 hi = bf16(p) and lo = bf16(p - hi), sixteen MMAs into the one O, so
// each probability keeps about 16 bits.  P is written back into tensor
// memory over the S tile it came from and read from there as the A operand
// of P.V, so the S buffers hold P as well.  With three of them, Q.K^T of
// tile t + 1 waits only for P.V of tile t - 2: the next S is usually ready
// when the softmax of tile t ends, while P.V of t and t - 1 are in flight.
//
// One CTA per SM, 256 threads, persistent over (tile of TQ tokens, sequence,
// kv head) items, in blocks of a few (sequence, kv head) pairs so that the
// CTAs at work share those pairs' keys and values in L2, later (longer) tiles
// first within a block:
//  * warp 0 loads the item's query rows (2-D TMA boxes, one per head and
//    64-dim half; two buffers, so the next item's rows load during this
//    item) and its K tiles (one 4-D TMA box per block, as in decode)
//    into a ring of kRingStages; warp 2 loads the V tiles likewise;
//  * warp 1 issues Q.K^T of every tile as soon as its K tile has landed and
//    an S buffer is free (so the softmax of tile t overlaps Q.K^T of t + 1);
//  * warp 3 issues P.V, per 16-key step the hi then the lo half of P, in a
//    fixed order so the fp32 sums are reproducible, zeroing first the V rows
//    past the end inside the last 16-key step of the item's last tile;
//  * warps 4-7 own tensor-memory lanes 0-127, one query row per thread: per
//    tile they read the row of S from tensor memory (max, then the
//    exponentials), mask keys past the row's position, run the online
//    softmax in fp32 (log2 domain) and store the row's P hi/lo over its S
//    (per 16-key MMA step: 8 columns of hi, then 8 of lo, bf16 pairs).  The
//    running max is the reference of P and O and is raised only when a row's
//    max grows by more than 2^8 (then the warp rescales its O rows in tensor
//    memory), so most tiles leave O alone.  At the item's end each thread
//    divides its O row by the row sum (the shared-prefix passes keep it
//    unnormalised, with the row's max and sum); a warp whose 32 rows are all
//    valid writes them to its 8 KB of shared memory and stores them with TMA
//    stores (bf16 or fp32 rows, one instantiation each), other rows are
//    stored one by one.
// Every mbarrier wait is bounded; on expiry the roles stop, the issuer
// drains, tensor memory is freed and PA_ERR_DEVICE_TIMEOUT is written to the
// caller's status word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include "decode.cuh"
#include "ptx.cuh"

namespace pa {

namespace prefill_detail {

constexpr int kThreads = 256;  // 8 warps
constexpr int kTileBytes = 32768;
constexpr int kRingStages = 2;               // K ring and V ring depth
constexpr int kOffQ = 0;                     // 2 query buffers (consecutive items)
constexpr int kOffK = 65536;
constexpr int kOffV = kOffK + kRingStages * kTileBytes;
constexpr int kOffBar = kOffV + kRingStages * kTileBytes;
constexpr int kOffStage = kOffBar + 1024;        // 4 x 8 KB: a softmax warp's output rows
constexpr int kSmemBytes = kOffStage + 4 * 8192 + 1024;  // then slack to align the base
constexpr float kRescaleLog2 = 8.0f;          // raise the reference max only past 2^8

constexpr int kNumS = 3;                     // S buffers in tensor memory

// barriers
// [S buffer]: kSFull (Q.K^T done), kPFull (P stored over S), kSFree (P.V of
// the tile done: S, P and every earlier O update are free)
constexpr int kQFull = 0, kQEmpty = 2, kKFull = 4, kKEmpty = kKFull + kRingStages,
              kVFull = kKEmpty + kRingStages, kVEmpty = kVFull + kRingStages, kSFull = kVEmpty + kRingStages,
              kSFree = kSFull + kNumS, kPFull = kSFree + kNumS, kOEmpty = kPFull + kNumS, kDrain = kOEmpty + 1,
              kNumBars = kDrain + 2;  // drains: Q.K^T, P.V
static_assert(kNumBars * 8 + 8 + 4 <= 256, "barrier area");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
constexpr uint32_t kColO = kNumS * 128;  // O after the S buffers
static_assert(kColO + 128 <= 512, "tensor memory columns");

struct Item {
  int seq, kvh, qb, tok0, ntq, pos0, k_start, kend, ntiles, trow_seq, causal, part;
  // a packed own-token item: members qb and qb + 1, each in its own 64-key
  // half of every tile, own tokens [k_start, k_start + own0) and
  // [k_start1, k_start1 + own1) of their tables (rows trow_seq, trow_seq1)
  int packed, own0, own1, k_start1, trow_seq1;
};

// The group of batch sequence i (group_start is non-decreasing).
__device__ __forceinline__ int group_of(const PrefillParams& p, int i) {
  int lo = 0, hi = p.num_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.group_start[mid] <= i) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void bad_input(const PrefillParams& p) {
  if (p.status) atomicExch(p.status, kDevErrInvalidArg);
}

// Work item w.  Mode 0 (prefill): (tile of TQ tokens, sequence, kv head) in
// blocks of pairs, later tiles first within a block, causal keys [0, position].  Mode 1 (shared prefix):
// (prefix partition, tile of TQ members, group, kv head) over the group's
// prefix keys, read through its first member's table.  Mode 2 (own tokens):
// (member, kv head) over keys [prefix, len) of the member's table.  Mode 3:
// every mode-1 item, then every mode-2 item, in one launch.
__device__ __forceinline__ int prefix_items(const PrefillParams& p) {
  return p.num_parts * p.num_groups * p.num_kv_heads * p.tiles_per_seq;
}
__device__ __forceinline__ int own_items(const PrefillParams& p) {
  return (p.pack2 ? (p.num_seqs + 1) / 2 : p.num_seqs) * p.num_kv_heads;
}
// Member m's own tokens [k_start, kend) past its group's prefix; false (and
// the error reported) for inconsistent lengths or prefixes.
__device__ __forceinline__ bool own_range(const PrefillParams& p, int m, int64_t table_tokens, int& k_start,
                                          int& kend);
__device__ __forceinline__ bool own_range(const PrefillParams& p, int m, int64_t table_tokens, int& k_start,
                                          int& kend) {
  const int grp = group_of(p, m);
  const int P = p.prefix_len[grp];
  const int len = p.context_lens[m];
  if (len < 0 || len > p.max_context_len || static_cast<int64_t>(len) > table_tokens || P < 0 ||
      P % p.block_size != 0 || P > len) {
    bad_input(p);
    return false;
  }
  k_start = P;
  kend = len;
  return true;
}
__device__ __forceinline__ bool item_at(const PrefillParams& p, int w, int G, Item& it) {
  it.packed = 0;
  const int hkv = p.num_kv_heads;
  const int TQ = 128 / G;
  const int64_t table_tokens = static_cast<int64_t>(p.max_blocks_per_seq) * p.block_size;
  int mode = p.mode;
  if (mode == 3) {
    const int n1 = prefix_items(p);
    mode = w < n1 ? 1 : 2;
    if (mode == 2) w -= n1;
  }
  if (mode == 0) {
    // blocks of pair_block (sequence, kv head) pairs, one block after the
    // other; within a block later tiles first, pairs fastest.  The CTAs
    // working at the same time then share a few pairs' keys and values, which
    // stay in L2 between their tiles.
    const int T = p.tiles_per_seq;
    const int npairs = p.num_seqs * hkv;
    const int per_block = p.pair_block * T;
    const int blk = w / per_block;
    const int r = w - blk * per_block;
    const int nb = min(p.pair_block, npairs - blk * p.pair_block);  // pairs in this block
    const int tile = T - 1 - r / nb;
    const int pair = blk * p.pair_block + (r - (r / nb) * nb);
    it.seq = pair / hkv;
    it.kvh = pair - it.seq * hkv;
    it.qb = p.cu_q[it.seq];
    const int n = p.cu_q[it.seq + 1] - it.qb;
    it.tok0 = tile * TQ;
    if (n <= 0 || it.tok0 >= n) return false;  // no tokens in this tile
    const int q0 = p.q_start[it.seq];
    if (it.qb < 0 || it.qb + n > p.num_tokens || q0 < 0 || static_cast<int64_t>(q0) + n > table_tokens) {
      bad_input(p);  // offsets outside q or the table
      return false;
    }
    it.ntq = min(TQ, n - it.tok0);
    it.pos0 = q0 + it.tok0;
    it.k_start = 0;
    it.kend = it.pos0 + it.ntq;
    it.trow_seq = it.seq;
    it.causal = 1;
    it.part = 0;
  } else if (mode == 1) {
    const int per_part = p.num_groups * hkv * p.tiles_per_seq;
    it.part = w / per_part;
    const int rem = w - it.part * per_part;
    const int tile = rem / (p.num_groups * hkv);
    const int r2 = rem - tile * (p.num_groups * hkv);
    const int grp = r2 / hkv;
    it.kvh = r2 - grp * hkv;
    it.seq = grp;
    it.qb = p.group_start[grp];
    const int n = p.group_start[grp + 1] - it.qb;
    it.tok0 = tile * TQ;
    if (n <= 0 || it.tok0 >= n) return false;
    const int P = p.prefix_len[grp];
    if (it.qb < 0 || it.qb + n > p.num_seqs || P < 0 || P % p.block_size != 0 || P > table_tokens) {
      bad_input(p);
      return false;
    }
    it.k_start = it.part * p.part_tokens;
    it.kend = min(P, it.k_start + p.part_tokens);
    if (it.k_start >= it.kend) return false;  // the group's prefix has fewer partitions
    it.ntq = min(TQ, n - it.tok0);
    it.pos0 = 0;
    it.trow_seq = it.qb;  // the prefix blocks are the same in every member's table
    it.causal = 0;
  } else if (p.pack2) {
    // two members per item, each in a 64-key half of every tile
    const int i = w / hkv;
    it.kvh = w - i * hkv;
    const int m0 = 2 * i, m1 = m0 + 1;
    const bool has1 = m1 < p.num_seqs;
    int e0 = 0, ks1 = 0, e1 = 0;
    if (!own_range(p, m0, table_tokens, it.k_start, e0)) return false;
    if (has1 && !own_range(p, m1, table_tokens, ks1, e1)) return false;
    it.seq = m0;
    it.qb = m0;
    it.tok0 = 0;
    it.ntq = has1 ? 2 : 1;
    it.pos0 = 0;
    it.kend = e0;
    it.own0 = e0 - it.k_start;
    it.own1 = has1 ? e1 - ks1 : 0;
    it.k_start1 = ks1;
    it.trow_seq = m0;
    it.trow_seq1 = has1 ? m1 : m0;
    it.causal = 0;
    it.part = p.num_parts;
    it.packed = 1;
    if (it.own0 <= 0 && it.own1 <= 0) return false;  // no own tokens: the merge skips this part
    it.ntiles = (max(it.own0, it.own1) + 63) / 64;
    return true;
  } else {
    const int i = w / hkv;
    it.kvh = w - i * hkv;
    it.seq = i;
    it.qb = i;
    it.tok0 = 0;
    it.ntq = 1;
    it.pos0 = 0;
    const int grp = group_of(p, i);
    const int P = p.prefix_len[grp];
    const int len = p.context_lens[i];
    if (len < 0 || len > p.max_context_len || static_cast<int64_t>(len) > table_tokens || P < 0 ||
        P % p.block_size != 0 || P > len) {
      bad_input(p);
      return false;
    }
    it.k_start = P;
    it.kend = len;
    if (it.kend <= it.k_start) return false;  // no own tokens: the merge skips this part
    it.trow_seq = i;
    it.causal = 0;
    it.part = p.num_parts;
  }
  it.ntiles = (it.kend - it.k_start + 127) / 128;
  return true;
}

__device__ __forceinline__ void wait(uint64_t* bar, uint32_t parity, bool& aborted) {
  if (!aborted && !ptx::mbar_wait(bar, parity, kWaitLimitNs)) aborted = true;
}

// 2^x by the ex2.approx.ftz instruction (relative error about 2^-22; very
// negative x gives 0)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// D[tmem] (+)= A[tmem] * B[smem]: A (M x 16, K-major) read from tensor
// memory, lane m holding row m as 8 columns of bf16 pairs; issued by one thread.
__device__ __forceinline__ void umma_ts_bf16(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

}  // namespace prefill_detail

// F32: full tiles' rows leave as fp32 (the output, or the shared-prefix
// partial O) by TMA stores; else as bf16 (the causal prefill's output).  Two
// instantiations keep each epilogue's code out of the other's kernel.
template <int G, bool F32>
__global__ void __launch_bounds__(prefill_detail::kThreads, 1)
    paged_prefill_umma_kernel(const __grid_constant__ PrefillParams p,
                              const __grid_constant__ CUtensorMap tm_q,
                              const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v,
                              const __grid_constant__ CUtensorMap tm_o) {
  using namespace prefill_detail;
  static_assert(G == 1 || G == 2 || G == 4 || G == 8 || G == 16, "GQA group");
  constexpr int TQ = 128 / G;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* qbuf = smem + kOffQ;
  unsigned char* kring = smem + kOffK;
  unsigned char* vring = smem + kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [0] a role gave up

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hkv = p.num_kv_heads, bs = p.block_size;
  const int bs_log = __ffs(bs) - 1;
  const int items = p.mode == 0   ? p.num_seqs * hkv * p.tiles_per_seq
                    : p.mode == 1 ? prefix_items(p)
                    : p.mode == 2 ? own_items(p)
                                  : prefix_items(p) + own_items(p);

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bars[kQFull + s], 1);
      ptx::mbar_init(&bars[kQEmpty + s], 1);
    }
    for (int s = 0; s < kRingStages; ++s) {
      ptx::mbar_init(&bars[kKFull + s], 1);
      ptx::mbar_init(&bars[kKEmpty + s], 1);
      ptx::mbar_init(&bars[kVFull + s], 1);
      ptx::mbar_init(&bars[kVEmpty + s], 1);
    }
    for (int s = 0; s < kNumS; ++s) {
      ptx::mbar_init(&bars[kSFull + s], 1);
      ptx::mbar_init(&bars[kSFree + s], 1);
      ptx::mbar_init(&bars[kPFull + s], 4);
    }
    ptx::mbar_init(&bars[kOEmpty], 4);
    for (int d = 0; d < 2; ++d) ptx::mbar_init(&bars[kDrain + d], 1);
    flags[0] = 0;
    ptx::mbar_init_fence();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, 512);  // S[3] x 128 columns, then O x 128
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool aborted = false;

  if (warp == 0 || warp == 2) {
    // ============ loaders: warp 0 queries + K tiles, warp 2 V tiles ============
    const bool is_v = warp == 2;
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
    const int box_rows = min(bs, 128);
    uint32_t ic = 0, fc = 0;  // items, tile fills
    for (int w = blockIdx.x; w < items && !aborted; w += gridDim.x) {
      Item it;
      if (!item_at(p, w, G, it)) continue;
      if (!is_v && lane == 0) {
        const uint32_t qs = ic & 1u;
        wait(&bars[kQEmpty + qs], ((ic >> 1) & 1u) ^ 1u, aborted);
        ptx::mbar_arrive_expect_tx(&bars[kQFull + qs], 2u * 128u * 128u);
        for (int g = 0; g < G; ++g)
          for (int h = 0; h < 2; ++h)
            ptx::tma_load_2d(qbuf + qs * 32768 + h * 16384 + g * TQ * 128, &tm_q,
                             (it.kvh * G + g) * 128 + h * 64, it.qb + it.tok0, &bars[kQFull + qs], pol_q);
      }
      const int32_t* trow = p.block_tables + static_cast<int64_t>(it.trow_seq) * p.max_blocks_per_seq;
      for (int t = 0; t < it.ntiles && !aborted; ++t, ++fc) {
        const int slot = static_cast<int>(fc % kRingStages);
        const uint32_t ph = (fc / kRingStages) & 1u;
        // this lane's box: of the tile (rows lane * box_rows ..), or in a
        // packed item of member lane / 8's 64-key half (box lane % 8)
        int nbox_total, tok = 0, dst_row = 0;
        bool mine;
        const int32_t* brow_tbl = trow;
        if (F32 && it.packed) {
          const int j = lane >> 3, bi = lane & 7;
          const int n0 = min(64, max(0, it.own0 - t * 64)), n1 = min(64, max(0, it.own1 - t * 64));
          const int nb0 = (n0 + box_rows - 1) / box_rows, nb1 = (n1 + box_rows - 1) / box_rows;
          nbox_total = nb0 + nb1;
          mine = lane < 16 && bi < (j ? nb1 : nb0);
          tok = (j ? it.k_start1 : it.k_start) + t * 64 + bi * box_rows;
          dst_row = j * 64 + bi * box_rows;
          if (j) brow_tbl = p.block_tables + static_cast<int64_t>(it.trow_seq1) * p.max_blocks_per_seq;
        } else {
          const int nv = min(128, it.kend - it.k_start - t * 128);
          nbox_total = (nv + box_rows - 1) / box_rows;
          mine = lane < nbox_total;
          tok = it.k_start + t * 128 + lane * box_rows;
          dst_row = lane * box_rows;
        }
        int row = 0;
        if (mine) {
          const int lb = tok >> bs_log;
          int phys = brow_tbl[lb];
          if (phys < 0 || phys >= p.num_blocks) {  // never read outside the pool
            if (p.status) atomicExch(p.status, kDevErrInvalidArg);
            phys = 0;
          }
          row = ((phys * hkv + it.kvh) << bs_log) + (tok - (lb << bs_log));
        }
        if (lane == 0) {
          wait(&empty[slot], ph ^ 1u, aborted);
          ptx::mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(nbox_total * box_rows * 256));
        }
        aborted = __shfl_sync(0xffffffffu, aborted, 0);
        if (!aborted && mine)
          ptx::tma_load_4d(ring + slot * kTileBytes + dst_row * 256, tm, 0, 0, 0, row >> 3, &full[slot], pol_kv);
        __syncwarp();
      }
      ++ic;
    }
  } else if (warp == 1) {
    // ============================ Q.K^T issue ============================
    constexpr uint32_t kIdQK = ptx::idesc_bf16_f32(128, 128, 0, 0);
    uint32_t ic = 0, kc = 0, sc = 0;
    for (int w = blockIdx.x; w < items && !aborted; w += gridDim.x) {
      Item it;
      if (!item_at(p, w, G, it)) continue;
      if (lane == 0) {
        const uint32_t qs = ic & 1u;
        const unsigned char* qt = qbuf + qs * 32768;
        wait(&bars[kQFull + qs], (ic >> 1) & 1u, aborted);
        for (int t = 0; t < it.ntiles && !aborted; ++t, ++kc, ++sc) {
          const int b = static_cast<int>(sc % kNumS);
          const int kslot = static_cast<int>(kc % kRingStages);
          wait(&bars[kKFull + kslot], (kc / kRingStages) & 1u, aborted);
          wait(&bars[kSFree + b], ((sc / kNumS) & 1u) ^ 1u, aborted);
          if (aborted) break;
          ptx::tc_fence_after();
          const unsigned char* kt = kring + kslot * kTileBytes;
          const uint32_t sd = tmem + b * 128;
          // a rolled loop: smaller code than eight unrolled issues, which
          // measured faster with the other roles' code sharing the SM
#pragma unroll 1
          for (int kk = 0; kk < 8; ++kk) {
            const int h = kk >> 2, k4 = kk & 3;
            ptx::umma_bf16(sd, ptx::smem_desc(qt + h * 16384 + k4 * 32, 16, 1024, ptx::kLayoutSw128),
                           ptx::smem_desc(kt + h * 1024 + k4 * 32, 16, 2048, ptx::kLayoutSw128), kIdQK,
                           kk > 0);
          }
          ptx::umma_commit(&bars[kSFull + b]);
          ptx::umma_commit(&bars[kKEmpty + kslot]);
          if (t == it.ntiles - 1) ptx::umma_commit(&bars[kQEmpty + qs]);
        }
      }
      aborted = __shfl_sync(0xffffffffu, aborted, 0);
      ++ic;
    }
    if (lane == 0) {  // nothing may be in flight when tensor memory is freed
      ptx::umma_commit(&bars[kDrain]);
      bool drain_aborted = false;
      wait(&bars[kDrain], 0, drain_aborted);
      if (aborted || drain_aborted) flags[0] = 1;
    }
    __syncwarp();
  } else if (warp == 3) {
    // ============================ P.V issue ============================
    // Per 16-key step, the hi half of P then the lo half into the one O
    // accumulator, in a fixed order, so the sums are reproducible.  P is
    // the A operand, read from the tile's S buffer in tensor memory.
    constexpr uint32_t kIdPV = ptx::idesc_bf16_f32(128, 128, 0, 1);
    const uint32_t od = tmem + kColO;
    uint32_t ic = 0, vc = 0, tc = 0;
    for (int w = blockIdx.x; w < items && !aborted; w += gridDim.x) {
      Item it;
      if (!item_at(p, w, G, it)) continue;
      for (int t = 0; t < it.ntiles; ++t, ++vc, ++tc) {
        const int vslot = static_cast<int>(vc % kRingStages);
        const int b = static_cast<int>(tc % kNumS);
        unsigned char* vt = vring + vslot * kTileBytes;
        if (lane == 0) {
          wait(&bars[kVFull + vslot], (vc / kRingStages) & 1u, aborted);
          wait(&bars[kPFull + b], (tc / kNumS) & 1u, aborted);
          if (t == 0) wait(&bars[kOEmpty], (ic & 1u) ^ 1u, aborted);
        }
        aborted = __shfl_sync(0xffffffffu, aborted, 0);
        if (aborted) break;
        int nks;
        if (F32 && it.packed) {
          // both 64-key halves take part: the rows past each member's own
          // tokens in this tile are zeroed (P is 0 there; the rows may hold
          // anything, even non-finite values)
          nks = 8;
#pragma unroll 1
          for (int j = 0; j < 2; ++j) {
            const int nvj = min(64, max(0, (j ? it.own1 : it.own0) - t * 64));
            for (int c = lane; c < (64 - nvj) * 16; c += 32) {
              const int rr = j * 64 + nvj + (c >> 4), half = (c >> 3) & 1, ch = c & 7;
              *reinterpret_cast<uint4*>(vt + (rr >> 3) * 2048 + half * 1024 + (rr & 7) * 128 + ch * 16) =
                  make_uint4(0, 0, 0, 0);
            }
          }
          ptx::fence_proxy_async_smem();
        } else {
          const int nv = min(128, it.kend - it.k_start - t * 128);
          nks = (nv + 15) / 16;
          if (nv & 15) {  // V rows past the end inside the last 16-key step: zeroed
            const int nrows = nks * 16 - nv;
            for (int c = lane; c < nrows * 16; c += 32) {
              const int rr = nv + (c >> 4), half = (c >> 3) & 1, ch = c & 7;
              *reinterpret_cast<uint4*>(vt + (rr >> 3) * 2048 + half * 1024 + (rr & 7) * 128 + ch * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            ptx::fence_proxy_async_smem();
          }
        }
        __syncwarp();
        if (lane == 0) {
          ptx::tc_fence_after();
          const uint32_t pa = tmem + static_cast<uint32_t>(b * 128);
          for (int ks = 0; ks < nks; ++ks) {
            const uint64_t vd = ptx::smem_desc(vt + ks * 4096, 1024, 2048, ptx::kLayoutSw128);
            umma_ts_bf16(od, pa + ks * 16, vd, kIdPV, t > 0 || ks > 0);
            umma_ts_bf16(od, pa + ks * 16 + 8, vd, kIdPV, 1u);
          }
          ptx::umma_commit(&bars[kSFree + b]);
          ptx::umma_commit(&bars[kVEmpty + vslot]);
        }
        __syncwarp();
      }
      ++ic;
    }
    if (lane == 0) {
      ptx::umma_commit(&bars[kDrain + 1]);
      bool drain_aborted = false;
      wait(&bars[kDrain + 1], 0, drain_aborted);
      if (aborted || drain_aborted) flags[0] = 1;
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // ============ softmax / epilogue: one query row per thread ============
    const int quarter = warp & 3;
    const int r = 32 * quarter + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const int g = r / TQ, trow = r - (r / TQ) * TQ;
    const float sl2 = p.scale_log2;
    uint32_t sc = 0;
    // max of the first n (<= 32, may be <= 0) raw scores of a 32-column chunk
    auto chunk_max = [](const uint32_t (&v)[32], int n) -> float {
      float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, m2 = -CUDART_INF_F, m3 = -CUDART_INF_F;
      if (n >= 32) {  // the common case: no mask
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          m0 = fmaxf(m0, __uint_as_float(v[j]));
          m1 = fmaxf(m1, __uint_as_float(v[j + 1]));
          m2 = fmaxf(m2, __uint_as_float(v[j + 2]));
          m3 = fmaxf(m3, __uint_as_float(v[j + 3]));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          m0 = j < n ? fmaxf(m0, __uint_as_float(v[j])) : m0;
      }
      return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
    };
    // p for the chunk's 32 columns (0 past the first n), added to the four
    // partial sums, and the chunk's P hi/lo stored over the same 32 columns
    // of S: for each of its two 16-key MMA steps, 8 columns of hi pairs, then
    // 8 of lo pairs (the even key in the low half).  hi = p with its low 16
    // bits cleared (a bf16 value, exact), lo = the exact fp32 remainder cut
    // the same way: |p - hi - lo| < 2^-16 p, both packed by bit moves
    auto write_p = [&](const uint32_t (&v)[32], uint32_t dst, int n, float neg_m, float (&ls)[4]) {
      uint32_t w[32];
      auto put = [&](int j, float p0, float p1) {
        const uint32_t h0 = __float_as_uint(p0) & 0xffff0000u, h1 = __float_as_uint(p1) & 0xffff0000u;
        const int step = j >> 4, pair = (j & 15) >> 1;  // MMA step in the chunk, pair in the step
        w[step * 16 + pair] = __byte_perm(h0, h1, 0x7632);  // high halves
        w[step * 16 + 8 + pair] = __byte_perm(__float_as_uint(p0 - __uint_as_float(h0)),
                                              __float_as_uint(p1 - __uint_as_float(h1)), 0x7632);
      };
      if (n >= 32) {  // the common case: every key visible
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float p0 = fast_exp2(fmaf(__uint_as_float(v[j]), sl2, neg_m));
          const float p1 = fast_exp2(fmaf(__uint_as_float(v[j + 1]), sl2, neg_m));
          ls[j & 3] += p0;
          ls[(j + 1) & 3] += p1;
          put(j, p0, p1);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float p0 = j < n ? fast_exp2(fmaf(__uint_as_float(v[j]), sl2, neg_m)) : 0.f;
          const float p1 = j + 1 < n ? fast_exp2(fmaf(__uint_as_float(v[j + 1]), sl2, neg_m)) : 0.f;
          ls[j & 3] += p0;
          ls[(j + 1) & 3] += p1;
          put(j, p0, p1);
        }
      }
      ptx::tmem_st32(dst, w);
    };
    // An item's epilogue: its O row divided by the row sum and stored, once
    // its last P.V (tile last_sc) has landed.  O is handed to the next item
    // as soon as its last chunk is read, before that chunk's stores.  It runs after the next item's first softmax tile, so that P.V
    // is usually done by then and the wait costs nothing.
    auto epilogue = [&](const Item& eit, bool evalid, float em, float el, uint32_t last_sc) -> bool {
      wait(&bars[kSFree + last_sc % kNumS], (last_sc / kNumS) & 1u, aborted);
      aborted = __any_sync(0xffffffffu, aborted);
      if (aborted) return false;
      ptx::tc_fence_after();
      const bool partial = p.mode != 0;  // shared-prefix decode: (max, sum, unnormalised O)
      const float inv = partial ? 1.f : (evalid && el > 0.f ? 1.f / el : 0.f);
      const int64_t prow = static_cast<int64_t>(eit.qb + eit.tok0 + trow) * p.num_q_heads + eit.kvh * G + g;
      const int64_t orow = prow * 128;
      const int64_t slot_rows = static_cast<int64_t>(eit.part) * p.num_seqs * p.num_q_heads;
      if (partial && evalid) {
        p.part_ml[(slot_rows + prow) * 2] = em;
        p.part_ml[(slot_rows + prow) * 2 + 1] = el;
      }
      if (F32 && p.o_tma == 2 && __all_sync(0xffffffffu, evalid)) {
        // fp32 rows (the output, or the shared-prefix partial O): per 64-dim
        // half, the warp's 32 rows into its 8 KB of shared memory as two
        // boxes of 32 floats (128-byte swizzled), then two TMA stores
        constexpr int HB = TQ >= 32 ? 1 : 32 / TQ;
        const int brow = TQ >= 32 ? lane : (lane % TQ) * HB + lane / TQ;
        unsigned char* stg = smem + kOffStage + quarter * 8192;
        const int r0 = 32 * quarter;
        const int y = eit.kvh * G + r0 / TQ;
        const int z = (partial ? eit.part * p.num_seqs : 0) + eit.qb + eit.tok0 + r0 % TQ;
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t v[64];
          ptx::TmemLd<32>::run(tmem + lane_base + kColO + hh * 64, *reinterpret_cast<uint32_t(*)[32]>(v));
          ptx::TmemLd<32>::run(tmem + lane_base + kColO + hh * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
          ptx::tmem_wait_ld();
          if (hh == 1) {  // O is read: the next item's P.V may start
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bars[kOEmpty]);
          }
          if (lane == 0) ptx::bulk_wait_read();  // earlier stores have read the staging
          __syncwarp();
#pragma unroll
          for (int bx = 0; bx < 2; ++bx) {
            unsigned char* line = stg + bx * 4096 + brow * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float* f = reinterpret_cast<const float*>(v + 32 * bx + 4 * q);
              *reinterpret_cast<float4*>(line + (q ^ (brow & 7)) * 16) =
                  make_float4(f[0] * inv, f[1] * inv, f[2] * inv, f[3] * inv);
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_3d(&tm_o, stg, hh * 64, y, z);
            ptx::tma_store_3d(&tm_o, stg + 4096, hh * 64 + 32, y, z);
            ptx::bulk_commit();
          }
        }
        return true;
      }
      if (!F32 && p.o_tma == 1 && __all_sync(0xffffffffu, evalid)) {
        // The warp's 32 rows, scaled and rounded to bf16, into its 8 KB of
        // shared memory in the output map's box order (token-major, then
        // head; two 64-dim halves, 128-byte swizzled), then two TMA stores.
        constexpr int HB = TQ >= 32 ? 1 : 32 / TQ;  // heads in the warp's box
        const int brow = TQ >= 32 ? lane : (lane % TQ) * HB + lane / TQ;
        unsigned char* stg = smem + kOffStage + quarter * 8192;
        if (lane == 0) ptx::bulk_wait_read();  // the previous item's stores have read it
        __syncwarp();
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {  // one 64-dim half per tensor-memory wait
          uint32_t v[64];
          ptx::TmemLd<32>::run(tmem + lane_base + kColO + hh * 64, *reinterpret_cast<uint32_t(*)[32]>(v));
          ptx::TmemLd<32>::run(tmem + lane_base + kColO + hh * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
          ptx::tmem_wait_ld();
          if (hh == 1) {  // O is read: the next item's P.V may start
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bars[kOEmpty]);
          }
          unsigned char* line = stg + hh * 4096 + brow * 128;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w4[e] = pack_bf16(__uint_as_float(v[8 * q + 2 * e]) * inv, __uint_as_float(v[8 * q + 2 * e + 1]) * inv);
            const int chunk = q ^ (brow & 7);
            *reinterpret_cast<uint4*>(line + chunk * 16) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int r0 = 32 * quarter;
          const int y = eit.kvh * G + r0 / TQ, z = eit.qb + eit.tok0 + r0 % TQ;
          ptx::tma_store_3d(&tm_o, stg, 0, y, z);
          ptx::tma_store_3d(&tm_o, stg + 4096, 64, y, z);
          ptx::bulk_commit();
        }
        return true;
      }
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        ptx::TmemLd<32>::run(tmem + lane_base + kColO + c * 32, v);
        ptx::tmem_wait_ld();
        if (c == 3) {  // O is read: the next item's P.V may start
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&bars[kOEmpty]);
        }
        if (evalid && partial) {
          float4* dst = reinterpret_cast<float4*>(p.part_o + (slot_rows + prow) * 128 + c * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                 __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        } else if (evalid) {
          if (p.out_bf16) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + orow + c * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w4[e] = pack_bf16(__uint_as_float(v[8 * q + 2 * e]) * inv, __uint_as_float(v[8 * q + 2 * e + 1]) * inv);
              dst[q] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow + c * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(__uint_as_float(v[4 * q]) * inv, __uint_as_float(v[4 * q + 1]) * inv,
                                   __uint_as_float(v[4 * q + 2]) * inv, __uint_as_float(v[4 * q + 3]) * inv);
          }
        }
      }
      return true;
    };
    bool pending = false;  // an item whose epilogue is still to run
    Item pit{};
    bool pvalid = false;
    float pm = 0.f, pl = 0.f;
    uint32_t psc = 0;
    for (int w = blockIdx.x; w < items && !aborted; w += gridDim.x) {
      Item it;
      if (!item_at(p, w, G, it)) continue;
      const bool valid = trow < it.ntq;
      // keys visible to this row: its causal position, or the whole range
      const int limit = !valid ? 0 : (it.causal ? it.pos0 + trow + 1 : it.kend);
      float m_ref = -CUDART_INF_F, l = 0.f;
      for (int t = 0; t < it.ntiles; ++t) {
        const int b = static_cast<int>(sc % kNumS);
        wait(&bars[kSFull + b], (sc / kNumS) & 1u, aborted);
        aborted = __any_sync(0xffffffffu, aborted);
        if (aborted) break;
        ptx::tc_fence_after();
        const uint32_t sbase = tmem + lane_base + b * 128;
        const int key0 = it.k_start + t * 128;
        // keys of this tile visible to the row: a prefix of nvis columns; in a
        // packed item, a prefix of the row's member's 64-key half
        int nvis = min(128, max(0, limit - key0));
        int half_own = -1;  // packed: the row's member's half (0, 1), else -1
        if (F32 && it.packed) {
          half_own = trow;
          nvis = valid ? min(64, max(0, (trow ? it.own1 : it.own0) - t * 64)) : 0;
        }
        // visible columns of the 32-column chunk c, counted from its start
        auto ncol = [&](int c) -> int {
          if (F32 && half_own >= 0) return (c >> 1) == half_own ? nvis - (c & 1) * 32 : 0;
          return nvis - c * 32;
        };
        // pass 1: the row's max over its visible raw scores (scale > 0 keeps
        // the order), two 32-column chunks per tensor-memory wait
        float mraw = -CUDART_INF_F;
#pragma unroll 1
        for (int c = 0; c < 4; c += 2) {
          uint32_t va[32], vb[32];
          ptx::TmemLd<32>::run(sbase + c * 32, va);
          ptx::TmemLd<32>::run(sbase + c * 32 + 32, vb);
          ptx::tmem_wait_ld();
          mraw = fmaxf(mraw, chunk_max(va, ncol(c)));
          mraw = fmaxf(mraw, chunk_max(vb, ncol(c + 1)));
        }
        const float mt = mraw * sl2;
        const float mn = fmaxf(m_ref, mt);
        bool rescale = t > 0 && mn > m_ref + kRescaleLog2;
        float alpha = 1.f;
        if (t == 0) {
          m_ref = mn;
        } else if (rescale) {
          alpha = exp2f(m_ref - mn);
          m_ref = mn;
          l *= alpha;
        }
        if (__any_sync(0xffffffffu, rescale)) {
          // warp-collective rescale of both O in tensor memory, once P.V of
          // the previous tile (and so every earlier one) has landed in O
          const uint32_t pb = (sc - 1u) % kNumS;
          wait(&bars[kSFree + pb], ((sc - 1u) / kNumS) & 1u, aborted);
          ptx::tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            ptx::TmemLd<32>::run(tmem + lane_base + kColO + c * 32, v);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
            ptx::tmem_st32(tmem + lane_base + kColO + c * 32, v);
          }
          ptx::tmem_wait_st();
        }
        // pass 2: p = 2^(s * scale_log2 - m_ref) (0 for masked keys), row sum,
        // P hi/lo stored over the columns of S just read; one chunk per
        // tensor-memory wait (one call site of write_p: the smaller loop body
        // measured faster than two chunks per wait)
        const float neg_m = -m_ref;
        float lsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t va[32];
          ptx::TmemLd<32>::run(sbase + c * 32, va);
          ptx::tmem_wait_ld();
          write_p(va, sbase + c * 32, ncol(c), neg_m, lsum);
        }
        l += (lsum[0] + lsum[1]) + (lsum[2] + lsum[3]);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars[kPFull + b]);
        ++sc;
        if (t == 0 && pending) {  // the previous item's epilogue, its P.V likely done
          pending = false;
          if (!epilogue(pit, pvalid, pm, pl, psc)) break;
        }
      }
      if (aborted) break;
      pending = true;
      pit = it;
      pvalid = valid;
      pm = m_ref;
      pl = l;
      psc = sc - 1u;
    }
    if (pending && !aborted) epilogue(pit, pvalid, pm, pl, psc);
    if (lane == 0) ptx::bulk_wait_all();  // this warp's output stores are complete
  }

  // ============================ teardown ============================
  // a merge launched behind this kernel with programmatic serialisation may
  // start; it waits for this grid's completion before reading its results
  ptx::griddep_launch_dependents();
  if (aborted) flags[0] = 1;
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, 512);
  if (tid == 0 && flags[0] && p.status) atomicExch(p.status, kDevErrTimeout);
}

// Shared-prefix decode, last step: for each (member, q head), the prefix
// partitions' and the own tokens' (max, sum, O) merged by log-sum-exp.
__global__ void __launch_bounds__(128) cascade_merge_kernel(const __grid_constant__ PrefillParams p) {
  const int rows = p.num_seqs * p.num_q_heads;
  const int row = blockIdx.x;  // member * H + head
  if (row >= rows) return;
  ptx::griddep_wait();  // launched behind the passes: their partial results are complete past here
  const int i = row / p.num_q_heads;
  const int d = threadIdx.x;
  const int grp = prefill_detail::group_of(p, i);
  const int P = max(0, p.prefix_len[grp]);
  const int len = p.context_lens[i];
  if (len < P && d == 0) prefill_detail::bad_input(p);  // a member shorter than its group's prefix
  const int nparts = (P + p.part_tokens - 1) / p.part_tokens;
  float M = -CUDART_INF_F;
  for (int k = 0; k < nparts; ++k) M = fmaxf(M, p.part_ml[(static_cast<int64_t>(k) * rows + row) * 2]);
  const bool own = len > P;
  const int64_t srow = static_cast<int64_t>(p.num_parts) * rows + row;
  if (own) M = fmaxf(M, p.part_ml[srow * 2]);
  float L = 0.f, O = 0.f;
  for (int k = 0; k < nparts; ++k) {
    const int64_t r = static_cast<int64_t>(k) * rows + row;
    const float wk = exp2f(p.part_ml[r * 2] - M);
    L = fmaf(wk, p.part_ml[r * 2 + 1], L);
    O = fmaf(wk, p.part_o[r * 128 + d], O);
  }
  if (own) {
    const float ws = exp2f(p.part_ml[srow * 2] - M);
    L = fmaf(ws, p.part_ml[srow * 2 + 1], L);
    O = fmaf(ws, p.part_o[srow * 128 + d], O);
  }
  const float v = L > 0.f ? O / L : 0.f;  // a sequence with no tokens gives zeros
  const int64_t idx = static_cast<int64_t>(row) * 128 + d;
  if (p.out_bf16) static_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
  else static_cast<float*>(p.out)[idx] = v;
}

cudaError_t launch_cascade_merge(const PrefillParams& p, cudaStream_t stream) {
  const int rows = p.num_seqs * p.num_q_heads;
  if (rows == 0) return cudaSuccess;
  // programmatic serialisation: the launch overlaps the passes' tail
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(rows));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, cascade_merge_kernel, p);
}

const void* prefill_umma_fn(int group, bool fp32_rows) {
  switch (group) {
    case 1: return fp32_rows ? reinterpret_cast<const void*>(&paged_prefill_umma_kernel<1, true>)
                             : reinterpret_cast<const void*>(&paged_prefill_umma_kernel<1, false>);
    case 2: return fp32_rows ? reinterpret_cast<const void*>(&paged_prefill_umma_kernel<2, true>)
                             : reinterpret_cast<const void*>(&paged_prefill_umma_kernel<2, false>);
    case 4: return fp32_rows ? reinterpret_cast<const void*>(&paged_prefill_umma_kernel<4, true>)
                             : reinterpret_cast<const void*>(&paged_prefill_umma_kernel<4, false>);
    case 8: return fp32_rows ? reinterpret_cast<const void*>(&paged_prefill_umma_kernel<8, true>)
                             : reinterpret_cast<const void*>(&paged_prefill_umma_kernel<8, false>);
    case 16: return fp32_rows ? reinterpret_cast<const void*>(&paged_prefill_umma_kernel<16, true>)
                              : reinterpret_cast<const void*>(&paged_prefill_umma_kernel<16, false>);
    default: return nullptr;
  }
}

int prefill_umma_smem_bytes() { return prefill_detail::kSmemBytes; }

}  // namespace pa
