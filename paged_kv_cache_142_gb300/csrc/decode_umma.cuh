// Paged decode attention on the 5th-generation tensor cores (sm_103a),
// bf16 K/V, head_dim 128, block size 8..256, GQA group G in {1,2,4,8,16}.
//
// Same result as the CUDA-core kernel ("PagedAttention", section "Block
// Table 如何工作": K/V of token t come from the physical block the block table
// names for logical block t / block_size; softmax(scale q.K) V over the
// history).  The GQA group turns both products into dense tiles:
//   S^T[128 tokens x 16] = K_tile[128 x 128 dims] . Q^T[128 dims x 16 heads]
//   O^T[128 dims x 16]  += V_tile^T[128 dims x 128 tokens] . P^T[128 tokens x 16]
// (heads padded to N = 16), each a handful of tcgen05.mma instructions with
// fp32 accumulators in tensor memory.  P enters the second product as two
// bf16 terms, hi = bf16(p) and lo = bf16(p - hi), side by side in the B tile
// (columns 0..7 and 8..15 for G <= 8, N = 32 for G = 16), so the result
// keeps about 16 bits of each probability instead of bf16's 8.
//
// Warp roles (one CTA per SM, persistent over (sequence, kv head, partition)
// work items enumerated from context_lens in shared memory):
//  * warp 0 streams: per item it hoists the partition's block-table slice
//    into shared memory, loads the query rows with a TMA tensor copy, and for
//    every 128-token tile issues TMA tensor copies (128-byte swizzle, L2
//    evict-first) of each block's K rows, then V rows, into a ring of 32 KB
//    stages;
//  * warp 1 owns 64 tensor-memory columns (S and O, double-buffered) and one
//    lane issues the MMAs: Q.K of tile u+1 goes out before P.V of tile u so
//    the score tile of the next tile is ready while softmax runs;
//  * warps 2-5 (one thread per token row, then per head-dim row): online
//    softmax in fp32 on the score tile (block max via shuffles + shared
//    memory, exp2 in the log2 domain), P written to shared memory as bf16,
//    rescale-and-accumulate of each tile's P.V in registers, and the item's
//    epilogue: store, or write (max, sum, unnormalised O) and, in the last
//    CTA to finish a (sequence, kv head), merge the partitions by
//    log-sum-exp.
// Rows past the end of a sequence: their scores are masked, their P is 0,
// V rows inside the last 16-token MMA step are zeroed in shared memory, and
// later steps are not issued, so stale or uninitialised memory never enters
// the sums.  All mbarrier waits are bounded; on expiry every role stops,
// the MMA lane drains its work, tensor memory is freed and
// PA_ERR_DEVICE_TIMEOUT is written to the workspace.
#pragma once

#include <cuda.h>

#include "decode_common.cuh"

namespace pa {

constexpr int kUmmaThreads = 192;
constexpr int kUmmaTile = 128;          // tokens per tile (MMA M)
constexpr int kUmmaTileBytes = 32768;   // one K or V tile: 2 halves x 128 rows x 128 B
constexpr int kUmmaMaxStages = 8;
constexpr int kUmmaQBytes = 4096;       // query tile: 2 halves x 16 rows x 128 B
constexpr int kUmmaPBytes = 8192;       // P tile: 128 tokens x (hi, lo) x up to 16 heads x bf16
constexpr int kUmmaSmallBytes = 1024;   // reductions and rescale factors
constexpr int kUmmaBarriers = 2 * kUmmaMaxStages + 13;
// tensor memory: S[2] at columns 0 and 16; O[2] (hi and lo halves) from column 32

namespace umma_detail {

enum Bar : int {
  kFull = 0,
  kEmpty = kUmmaMaxStages,
  kQFull = 2 * kUmmaMaxStages,
  kQEmpty = kQFull + 2,
  kSFull = kQEmpty + 2,
  kSEmpty = kSFull + 2,
  kPFull = kSEmpty + 2,
  kPEmpty = kPFull + 2,
  kOFull = kPEmpty + 2,
  kOEmpty = kOFull + 2,
  kDrain = kOEmpty + 2,
};

struct Item {
  int seq, kvh, part, len, t0, ntok, nparts;
};

__device__ __forceinline__ Item item_at(const DecodeParams& p, const int32_t* prefix, int w) {
  Item it;
  decode_detail::find_item(w, prefix, p.num_seqs, p.num_kv_heads, it.seq, it.kvh, it.part);
  it.len = decode_detail::clamp_len(p.context_lens[it.seq], p.max_context_len);
  it.t0 = it.part * p.part_tokens;
  it.ntok = min(it.len - it.t0, p.part_tokens);
  it.nparts = it.len > 0 ? (it.len + p.part_tokens - 1) / p.part_tokens : 1;
  return it;
}

// bounded wait; once a CTA has given up, later waits are skipped
__device__ __forceinline__ void wait(uint64_t* bar, uint32_t parity, bool& aborted) {
  if (!aborted && !ptx::mbar_wait(bar, parity, kWaitLimitNs)) aborted = true;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

}  // namespace umma_detail

template <int G>
__global__ void __launch_bounds__(kUmmaThreads, 1)
    paged_decode_umma_kernel(const __grid_constant__ DecodeParams p,
                             const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v,
                             const __grid_constant__ CUtensorMap tm_q) {
  using namespace umma_detail;
  static_assert(G == 1 || G == 2 || G == 4 || G == 8 || G == 16, "GQA group");
  constexpr int HD = 128;
  constexpr int NP = G <= 8 ? 16 : 32;        // P.V columns: hi heads, then lo heads
  constexpr int LO = NP / 2;                  // column of the lo half
  constexpr int PGRP = NP / 8;                // 8-column core matrices per P row group
  constexpr uint32_t TMEM_COLS = G <= 8 ? 64 : 128;

  extern __shared__ unsigned char smem_raw[];
  __shared__ int warp_sums[kUmmaThreads / 32];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* ring = smem;
  unsigned char* qbuf = smem + p.off_q;
  unsigned char* pbuf = smem + p.off_p;
  float* red_m = reinterpret_cast<float*>(smem + p.off_small);  // [2][4][16]
  float* red_l = red_m + 2 * 4 * 16;                            // [4][16]
  float* alpha_s = red_l + 4 * 16;                              // [2][16]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kUmmaBarriers);
  // [0] stream/MMA gave up, [1] merge this item, [2] compute warps gave up
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* tbl = reinterpret_cast<int32_t*>(smem + p.off_tbl);
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + p.off_prefix);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int NS = p.stages;
  const int hkv = p.num_kv_heads;
  const int bs = p.block_size;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(&bars[kFull + s], 1);
      ptx::mbar_init(&bars[kEmpty + s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&bars[kQFull + b], 1);
      ptx::mbar_init(&bars[kQEmpty + b], 1);
      ptx::mbar_init(&bars[kSFull + b], 1);
      ptx::mbar_init(&bars[kSEmpty + b], 4);
      ptx::mbar_init(&bars[kPFull + b], 4);
      ptx::mbar_init(&bars[kPEmpty + b], 1);
      ptx::mbar_init(&bars[kOFull + b], 1);
      ptx::mbar_init(&bars[kOEmpty + b], 4);
    }
    ptx::mbar_init(&bars[kDrain], 1);
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
    ptx::mbar_init_fence();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, TMEM_COLS);
    ptx::tc_fence_before();
  }
  decode_detail::build_item_prefix(p, prefix, warp_sums, tid, kUmmaThreads);  // syncs the CTA
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = prefix[p.num_seqs];
  bool aborted = false;

  if (warp == 0) {
    // ============================ TMA streaming ============================
    if (lane == 0) {
      ptx::prefetch_tensormap(&tm_k);
      ptx::prefetch_tensormap(&tm_v);
      ptx::prefetch_tensormap(&tm_q);
    }
    const uint64_t pol_kv = ptx::policy_evict_first();
    const uint64_t pol_q = ptx::policy_evict_normal();
    const int box_rows = min(bs, kUmmaTile);
    uint32_t u = 0, qi = 0;
    for (int w = blockIdx.x; w < total && !aborted; w += gridDim.x) {
      const Item it = item_at(p, prefix, w);
      if (it.ntok <= 0) continue;
      const int b0 = it.t0 / bs;
      const int nb = (it.t0 + it.ntok + bs - 1) / bs - b0;
      const int32_t* trow = p.block_tables + static_cast<int64_t>(it.seq) * p.max_blocks_per_seq + b0;
      for (int j = lane; j < nb; j += 32) {
        int phys = trow[j];
        if (phys < 0 || phys >= p.num_blocks) {  // never read outside the pool
          atomicExch(p.ws_err, kDevErrInvalidArg);
          phys = 0;
        }
        tbl[j] = phys;
      }
      __syncwarp();
      const int nt = (it.ntok + kUmmaTile - 1) / kUmmaTile;
      if (lane == 0) {
        const uint32_t qs = qi & 1u;
        wait(&bars[kQEmpty + qs], ((qi >> 1) & 1u) ^ 1u, aborted);
        ptx::mbar_arrive_expect_tx(&bars[kQFull + qs], 2u * G * 128u);
        for (int h = 0; h < 2; ++h)
          ptx::tma_load_2d(qbuf + qs * kUmmaQBytes + h * 2048, &tm_q, 64 * h,
                           it.seq * p.num_q_heads + it.kvh * G, &bars[kQFull + qs], pol_q);
        for (int j = 0; j < nt && !aborted; ++j) {
          const int tok0 = it.t0 + j * kUmmaTile;
          const int nv = min(kUmmaTile, it.ntok - j * kUmmaTile);
          const int nbox = (nv + box_rows - 1) / box_rows;
          for (int kv = 0; kv < 2; ++kv) {
            const uint32_t e = 2u * (u + j) + kv;
            const int slot = static_cast<int>(e % NS);
            wait(&bars[kEmpty + slot], ((e / NS) & 1u) ^ 1u, aborted);
            ptx::mbar_arrive_expect_tx(&bars[kFull + slot], static_cast<uint32_t>(nbox * box_rows * 256));
            unsigned char* dst = ring + slot * kUmmaTileBytes;
            const CUtensorMap* tm = kv ? &tm_v : &tm_k;
            for (int bi = 0; bi < nbox; ++bi) {
              const int tok = tok0 + bi * box_rows;
              const int lb = tok / bs;
              const int row = (tbl[lb - b0] * hkv + it.kvh) * bs + (tok - lb * bs);
              for (int h = 0; h < 2; ++h)
                ptx::tma_load_2d(dst + h * 16384 + bi * box_rows * 128, tm, 64 * h, row,
                                 &bars[kFull + slot], pol_kv);
            }
          }
        }
      }
      u += nt;
      ++qi;
      aborted = __shfl_sync(0xffffffffu, aborted, 0);
      __syncwarp();  // the table slice is rewritten by the next item
    }
  } else if (warp == 1) {
    // ============================ MMA issue ============================
    if (lane == 0) {
      constexpr uint32_t kIdQK = ptx::idesc_bf16_f32(128, 16, 0, 0);
      constexpr uint32_t kIdPV = ptx::idesc_bf16_f32(128, NP, 1, 1);
      bool have_prev = false;
      uint32_t prev_u = 0;
      int prev_nv = 0;
      auto issue_pv = [&](uint32_t pu, int pnv) {
        const uint32_t e = 2u * pu + 1u;
        const int vslot = static_cast<int>(e % NS);
        const uint32_t b = pu & 1u;
        wait(&bars[kFull + vslot], (e / NS) & 1u, aborted);
        wait(&bars[kPFull + b], (pu >> 1) & 1u, aborted);
        wait(&bars[kOEmpty + b], ((pu >> 1) & 1u) ^ 1u, aborted);
        ptx::tc_fence_after();
        const unsigned char* vt = ring + vslot * kUmmaTileBytes;
        const unsigned char* pt = pbuf + b * kUmmaPBytes;
        const int nks = (pnv + 15) / 16;
        for (int ks = 0; ks < nks; ++ks)
          ptx::umma_bf16(tmem + 32 + b * NP,
                         ptx::smem_desc(vt + ks * 2048, 16384, 1024, ptx::kLayoutSw128),
                         ptx::smem_desc(pt + ks * 2 * PGRP * 128, PGRP * 128, 128, ptx::kLayoutNone),
                         kIdPV, ks > 0);
        ptx::umma_commit(&bars[kOFull + b]);
        ptx::umma_commit(&bars[kEmpty + vslot]);
        ptx::umma_commit(&bars[kPEmpty + b]);
      };
      uint32_t u = 0, qi = 0;
      for (int w = blockIdx.x; w < total && !aborted; w += gridDim.x) {
        const Item it = item_at(p, prefix, w);
        if (it.ntok <= 0) continue;
        const int nt = (it.ntok + kUmmaTile - 1) / kUmmaTile;
        const uint32_t qs = qi & 1u;
        wait(&bars[kQFull + qs], (qi >> 1) & 1u, aborted);
        const unsigned char* qt = qbuf + qs * kUmmaQBytes;
        for (int j = 0; j < nt && !aborted; ++j, ++u) {
          const uint32_t e = 2u * u;
          const int kslot = static_cast<int>(e % NS);
          const uint32_t b = u & 1u;
          wait(&bars[kFull + kslot], (e / NS) & 1u, aborted);
          wait(&bars[kSEmpty + b], ((u >> 1) & 1u) ^ 1u, aborted);
          ptx::tc_fence_after();
          const unsigned char* kt = ring + kslot * kUmmaTileBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const int h = kk >> 2, k4 = kk & 3;
            ptx::umma_bf16(tmem + b * 16,
                           ptx::smem_desc(kt + h * 16384 + k4 * 32, 16, 1024, ptx::kLayoutSw128),
                           ptx::smem_desc(qt + h * 2048 + k4 * 32, 16, 1024, ptx::kLayoutSw128), kIdQK,
                           kk > 0);
          }
          ptx::umma_commit(&bars[kSFull + b]);
          ptx::umma_commit(&bars[kEmpty + kslot]);
          if (j == nt - 1) ptx::umma_commit(&bars[kQEmpty + qs]);
          if (have_prev) issue_pv(prev_u, prev_nv);
          have_prev = true;
          prev_u = u;
          prev_nv = min(kUmmaTile, it.ntok - j * kUmmaTile);
        }
        ++qi;
      }
      if (have_prev && !aborted) issue_pv(prev_u, prev_nv);
      // nothing may be in flight when tensor memory is freed
      ptx::umma_commit(&bars[kDrain]);
      bool drain_aborted = false;
      wait(&bars[kDrain], 0, drain_aborted);
      if (aborted || drain_aborted) flags[0] = 1;
    }
    __syncwarp();
  } else {
    // ===================== softmax, accumulation, epilogue =====================
    const int ctid = tid - 64;
    const int cw = warp - 2;                // compute warp 0..3
    const int quarter = warp & 3;           // tensor-memory lanes 32*quarter .. +31
    const int r = 32 * quarter + lane;      // token row of S, head-dim row of O
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const float sl2 = p.scale_log2;

    float m_run[G], l_thr[G], o_acc[G];
    float m_fin0[G], l_fin0[G], m_fin1[G], l_fin1[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m_run[g] = -CUDART_INF_F;
      l_thr[g] = 0.f;
      o_acc[g] = 0.f;
      m_fin0[g] = m_fin1[g] = -CUDART_INF_F;
      l_fin0[g] = l_fin1[g] = 0.f;
    }
    struct Prev {
      uint32_t u;
      int first, last, seq, kvh, part, nparts;
    } prev = {0, 0, 0, 0, 0, 0, 0};
    bool have_prev = false;

    auto softmax = [&](uint32_t u, int nv, bool first, bool last) {
      const uint32_t b = u & 1u, ph = (u >> 1) & 1u;
      if (first) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          m_run[g] = -CUDART_INF_F;
          l_thr[g] = 0.f;
        }
      }
      wait(&bars[kSFull + b], ph, aborted);
      ptx::tc_fence_after();
      uint32_t sr[G];
      ptx::TmemLd<G>::run(tmem + lane_base + b * 16, sr);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars[kSEmpty + b]);
      const bool valid = r < nv;
      float s[G], mx[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        s[g] = valid ? __uint_as_float(sr[g]) * sl2 : -CUDART_INF_F;
        mx[g] = s[g];
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int g = 0; g < G; ++g) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xffffffffu, mx[g], off));
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) red_m[(b * 4 + cw) * 16 + g] = mx[g];
      }
      ptx::bar_sync(1, 128);
      float pr[G], al[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float mt = red_m[(b * 4) * 16 + g];
#pragma unroll
        for (int k = 1; k < 4; ++k) mt = fmaxf(mt, red_m[(b * 4 + k) * 16 + g]);
        const float mn = fmaxf(m_run[g], mt);
        al[g] = exp2f(m_run[g] - mn);
        pr[g] = valid ? exp2f(s[g] - mn) : 0.f;
        l_thr[g] = l_thr[g] * al[g] + pr[g];
        m_run[g] = mn;
      }
      if (ctid == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) alpha_s[b * 16 + g] = al[g];
      }
      if (last) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          if (b) {
            m_fin1[g] = m_run[g];
            l_fin1[g] = l_thr[g];
          } else {
            m_fin0[g] = m_run[g];
            l_fin0[g] = l_thr[g];
          }
        }
      }
      // P row r: columns [0, LO) hold bf16(p) of heads 0..G-1, columns
      // [LO, NP) the bf16 remainder p - bf16(p); unused heads are zero
      float ph_[NP];
#pragma unroll
      for (int c = 0; c < NP; ++c) ph_[c] = 0.f;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float hi = __bfloat162float(__float2bfloat16_rn(pr[g]));
        ph_[g] = hi;
        ph_[LO + g] = pr[g] - hi;
      }
      uint32_t wp[NP / 2];
#pragma unroll
      for (int k = 0; k < NP / 2; ++k) wp[k] = pack_bf16(ph_[2 * k], ph_[2 * k + 1]);
      wait(&bars[kPEmpty + b], ph ^ 1u, aborted);
      unsigned char* prow = pbuf + b * kUmmaPBytes + (r >> 3) * (PGRP * 128) + (r & 7) * 16;
#pragma unroll
      for (int c = 0; c < PGRP; ++c)
        *reinterpret_cast<uint4*>(prow + c * 128) =
            make_uint4(wp[4 * c], wp[4 * c + 1], wp[4 * c + 2], wp[4 * c + 3]);
      if ((nv & 15) && r >= nv && r < ((nv + 15) & ~15)) {
        // V rows past the end inside the last MMA step: zero them
        const uint32_t e = 2u * u + 1u;
        const int vslot = static_cast<int>(e % NS);
        wait(&bars[kFull + vslot], (e / NS) & 1u, aborted);
        unsigned char* vrow = ring + vslot * kUmmaTileBytes + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(vrow + 16384 + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars[kPFull + b]);
    };

    auto epilogue = [&](const Prev& t) {
      float mf[G], lf[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        mf[g] = (t.u & 1u) ? m_fin1[g] : m_fin0[g];
        lf[g] = (t.u & 1u) ? l_fin1[g] : l_fin0[g];
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int g = 0; g < G; ++g) lf[g] += __shfl_xor_sync(0xffffffffu, lf[g], off);
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) red_l[cw * 16 + g] = lf[g];
      }
      ptx::bar_sync(1, 128);
      float L[G];
#pragma unroll
      for (int g = 0; g < G; ++g) L[g] = red_l[g] + red_l[16 + g] + red_l[32 + g] + red_l[48 + g];
      const int64_t obase = (static_cast<int64_t>(t.seq) * p.num_q_heads + t.kvh * G) * HD + r;
      if (t.nparts == 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) decode_detail::store_out(p.out, p.out_bf16, obase + g * HD, o_acc[g] / L[g]);
        return;
      }
      const int row = t.seq * hkv + t.kvh;
      const int64_t rec = static_cast<int64_t>(row) * p.max_parts + t.part;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        p.ws_o[(rec * G + g) * HD + r] = o_acc[g];
        if (ctid == g) {
          p.ws_ml[rec * G * 2 + 2 * g] = mf[g];
          p.ws_ml[rec * G * 2 + 2 * g + 1] = L[g];
        }
      }
      ptx::bar_sync(1, 128);
      if (ctid == 0) {
        __threadfence();
        flags[1] = (atomicAdd(&p.ws_counters[row], 1) == t.nparts - 1) ? 1 : 0;
      }
      ptx::bar_sync(1, 128);
      if (flags[1]) {
        // last partition of this (sequence, kv head) to finish: merge
        __threadfence();
        const float* ml = p.ws_ml + static_cast<int64_t>(row) * p.max_parts * G * 2;
        const float* os = p.ws_o + static_cast<int64_t>(row) * p.max_parts * G * HD + r;
#pragma unroll 1
        for (int g = 0; g < G; ++g) {
          float M = -CUDART_INF_F;
          for (int q = 0; q < t.nparts; ++q) M = fmaxf(M, __ldcg(ml + q * G * 2 + 2 * g));
          float Ls = 0.f, Os = 0.f;
          for (int q = 0; q < t.nparts; ++q) {
            const float wq = exp2f(__ldcg(ml + q * G * 2 + 2 * g) - M);
            Ls += wq * __ldcg(ml + q * G * 2 + 2 * g + 1);
            Os += wq * __ldcg(os + (static_cast<int64_t>(q) * G + g) * HD);
          }
          decode_detail::store_out(p.out, p.out_bf16, obase + g * HD, Os / Ls);
        }
        if (ctid == 0) p.ws_counters[row] = 0;
      }
    };

    auto accumulate = [&](const Prev& t) {
      const uint32_t b = t.u & 1u, ph = (t.u >> 1) & 1u;
      wait(&bars[kOFull + b], ph, aborted);
      ptx::tc_fence_after();
      uint32_t orr[NP];
      ptx::TmemLd<NP>::run(tmem + lane_base + 32 + b * NP, orr);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars[kOEmpty + b]);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float o = __uint_as_float(orr[g]) + __uint_as_float(orr[LO + g]);
        o_acc[g] = t.first ? o : fmaf(o_acc[g], alpha_s[b * 16 + g], o);
      }
      if (t.last) epilogue(t);
    };

    uint32_t u = 0;
    for (int w = blockIdx.x; w < total; w += gridDim.x) {
      const Item it = item_at(p, prefix, w);
      if (it.ntok <= 0) {  // empty sequence: zero output
        const int64_t obase = (static_cast<int64_t>(it.seq) * p.num_q_heads + it.kvh * G) * HD + r;
#pragma unroll
        for (int g = 0; g < G; ++g) decode_detail::store_out(p.out, p.out_bf16, obase + g * HD, 0.f);
        continue;
      }
      const int nt = (it.ntok + kUmmaTile - 1) / kUmmaTile;
      for (int j = 0; j < nt; ++j, ++u) {
        const int nv = min(kUmmaTile, it.ntok - j * kUmmaTile);
        softmax(u, nv, j == 0, j == nt - 1);
        if (have_prev) accumulate(prev);
        prev = Prev{u, j == 0, j == nt - 1, it.seq, it.kvh, it.part, it.nparts};
        have_prev = true;
      }
      if (aborted) flags[2] = 1;
      ptx::bar_sync(1, 128);
      if (flags[2]) break;  // uniform: read after the barrier, written only before one
    }
    if (have_prev && !flags[2]) accumulate(prev);
  }

  // ============================ teardown ============================
  if (aborted) flags[0] = 1;
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, TMEM_COLS);
  if (tid == 0 && (flags[0] || flags[2])) atomicExch(p.ws_err, kDevErrTimeout);
}

}  // namespace pa
