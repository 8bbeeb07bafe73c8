// Paged decode attention for sm_103a.
//
// What it computes ("PagedAttention", section "Block Table 如何工作"; same
// page, "不改变模型精度"): for every sequence and query head, softmax(scale *
// q . K_t) V over the sequence's tokens t, where token t's K/V live in the
// physical block the sequence's block table names for logical block
// t / block_size, at row t % block_size.  The result equals attention over
// the contiguous history.
//
// Design (one GPU, HBM-bound: every history byte is read once):
//  * Work items are (sequence, kv head, partition) with partitions of
//    `part_tokens` consecutive tokens.  A persistent grid walks the items
//    round-robin; each CTA derives the item list from context_lens with a
//    prefix sum in shared memory, so no planning kernel runs.
//  * Warp 0 streams.  Per item it hoists the partition's slice of the block
//    table into shared memory, then issues 1-D bulk async copies (TMA bulk
//    engine, L2 evict-first) of whole (block, kv head) K tiles, then V tiles,
//    into a ring of kStages shared-memory stages tracked by mbarriers.  The
//    item's query rows ride in the first K stage.  It runs ahead across item
//    boundaries, bounded only by the ring.
//  * Warps 1-4 compute in fp32.  Scores: each token is shared by kLpt lanes,
//    every lane holding a slice of the GQA group's G query rows in registers,
//    so one read of a K row serves all G heads; paired fp32 FMAs; partial
//    dots combined by xor shuffles.  The partition's scores sit in shared
//    memory; max and sum are block reductions (shuffles + shared memory) and
//    the probabilities are exp2 of log2-domain scores.  Then V: each lane owns
//    a 16-byte slice of head_dim for all G heads over a subset of tokens.
//  * One partition: normalise and store.  Several: store (max, sum,
//    unnormalised output) to the workspace; the last CTA to finish a
//    (sequence, kv head) -- found with a device-scope atomic counter, no
//    waiting -- merges the partials by log-sum-exp and resets the counter.
//  * Every mbarrier wait is bounded; on expiry the CTA records
//    PA_ERR_DEVICE_TIMEOUT in the workspace and all its warps leave together.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include "decode_common.cuh"

namespace pa {
namespace decode_detail {

constexpr int ceil_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}
constexpr int cmax(int a, int b) { return a > b ? a : b; }
constexpr int cmin(int a, int b) { return a < b ? a : b; }

template <int E, int D, int G>
struct Shape {
  static constexpr int kRow = D * E;                    // bytes: one token, one kv head
  static constexpr int kVec = 16 / E;                   // elements per 16-byte chunk
  static constexpr int kChunks = kRow / 16;             // chunks per row
  static constexpr int kTokStage = kStageBytes / kRow;  // tokens per ring stage
  static constexpr int kQBytes = G * kRow;              // query rows of one GQA group
  static constexpr int kStageAlloc = (kStageBytes + kQBytes + 127) / 128 * 128;
  // scores: kLpt lanes per token, so that a lane holds <= 64 query values
  static constexpr int kLpt = cmin(cmax(ceil_pow2((G * D) / 64), 4), cmin(kChunks, 32));
  static constexpr int kCpl = kChunks / kLpt;             // chunks per lane
  static constexpr int kTokPass = kConsumerThreads / kLpt;  // tokens per pass
  static constexpr int kPasses = (kTokStage + kTokPass - 1) / kTokPass;
  // tokens of one quarter-warp; lanes rotate their chunk order by token so a
  // quarter-warp's 16-byte loads hit 8 distinct bank groups
  static constexpr int kSwz = (kLpt < 8) ? 8 / kLpt : 1;
  // P.V: kDg lanes per token, one 16-byte chunk each; kTg token groups
  static constexpr int kDg = kChunks;
  static constexpr int kTg = kConsumerThreads / kDg;
  static_assert(kRow % 128 == 0, "row bytes must be a multiple of 128");
  static_assert(kTokStage >= 1 && kTokStage * kRow == kStageBytes, "stage holds whole rows");
  static_assert(kCpl >= 1 && (kCpl & (kCpl - 1)) == 0, "chunks per lane: power of two");
  static_assert(kLpt >= 8 || kCpl >= kSwz, "bank swizzle needs enough chunks per lane");
  static_assert(kDg <= 32 && 32 % kDg == 0, "a P.V token group fits in a warp");
  static_assert(32 % G == 0, "softmax reduction pattern");
};

}  // namespace decode_detail

template <typename T, int D, int G>
__global__ void __launch_bounds__(kDecodeThreads, 3)
    paged_decode_kernel(const __grid_constant__ DecodeParams p) {
  using namespace decode_detail;
  using S = Shape<Elem<T>::kBytes, D, G>;
  constexpr int kV2 = S::kVec / 2;

  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int warp_sums[kDecodeThreads / 32];
  __shared__ int flags[2];  // [0] abort, [1] this CTA merges the current item

  unsigned char* ring = smem;
  float* sc = reinterpret_cast<float*>(smem + p.off_sc);
  float* red = reinterpret_cast<float*>(smem + p.off_red);
  float* red_m = red + kConsumerWarps * G * D;
  float* red_l = red_m + kConsumerWarps * G;
  float* mrg = red_l + kConsumerWarps * G;
  int32_t* tbl = reinterpret_cast<int32_t*>(smem + p.off_tbl);
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + p.off_prefix);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* empty = full + kStages;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int nseq = p.num_seqs;
  const int hkv = p.num_kv_heads;
  const int bs = p.block_size;
  const int pt = p.part_tokens;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], kConsumerWarps);
    }
    flags[0] = 0;
    flags[1] = 0;
    ptx::mbar_init_fence();
  }

  // ---- work items per sequence: max(1, ceil(len / pt)) * hkv; prefix sum ----
  build_item_prefix(p, prefix, warp_sums, tid, kDecodeThreads);
  const int total = prefix[nseq];

  // =========================== streaming warp ===========================
  if (warp == 0) {
    const uint64_t pol = ptx::policy_evict_first();
    uint32_t stage = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      int seq, kvh, part;
      find_item(w, prefix, nseq, hkv, seq, kvh, part);
      const int len = clamp_len(p.context_lens[seq], p.max_context_len);
      const int t0 = part * pt;
      const int ntok = min(len - t0, pt);
      if (ntok <= 0) continue;
      // hoist this partition's slice of the block table into shared memory
      const int b0 = t0 / bs;
      const int nb = (t0 + ntok + bs - 1) / bs - b0;
      const int32_t* trow = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks_per_seq + b0;
      for (int j = lane; j < nb; j += 32) {
        int phys = trow[j];
        if (phys < 0 || phys >= p.num_blocks) {  // never read outside the pool
          atomicExch(p.ws_err, kDevErrInvalidArg);
          phys = 0;
        }
        tbl[j] = phys;
      }
      __syncwarp();
      if (lane == 0) {
        const int nst = (ntok + S::kTokStage - 1) / S::kTokStage;
        const int prow = min(bs, S::kTokStage);
        for (int kv = 0; kv < 2 && ok; ++kv) {
          const unsigned char* base = static_cast<const unsigned char*>(kv ? p.v_cache : p.k_cache);
          for (int s = 0; s < nst; ++s) {
            const int slot = stage % kStages;
            const uint32_t par = ((stage / kStages) & 1u) ^ 1u;
            if (!ptx::mbar_wait(&empty[slot], par, kWaitLimitNs)) {
              ok = false;
              break;
            }
            const int ts = s * S::kTokStage;
            const int nv = min(S::kTokStage, ntok - ts);
            const int npc = (nv + prow - 1) / prow;
            const bool with_q = (kv == 0 && s == 0);
            const uint32_t bytes =
                static_cast<uint32_t>(npc * prow * S::kRow + (with_q ? S::kQBytes : 0));
            unsigned char* dst = ring + slot * S::kStageAlloc;
            ptx::mbar_arrive_expect_tx(&full[slot], bytes);
            for (int pc = 0; pc < npc; ++pc) {
              const int tok = t0 + ts + pc * prow;
              const int lb = tok / bs;
              const int64_t row =
                  (static_cast<int64_t>(tbl[lb - b0]) * hkv + kvh) * bs + (tok - lb * bs);
              ptx::bulk_g2s(dst + pc * prow * S::kRow, base + row * S::kRow,
                            static_cast<uint32_t>(prow * S::kRow), &full[slot], pol);
            }
            if (with_q) {
              const unsigned char* qsrc =
                  static_cast<const unsigned char*>(p.q) +
                  (static_cast<int64_t>(seq) * p.num_q_heads + kvh * G) * S::kRow;
              ptx::bulk_g2s(dst + kStageBytes, qsrc, S::kQBytes, &full[slot], pol);
            }
            ++stage;
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      __syncwarp();  // the table slice is rewritten by the next item
    }
    if (!ok && lane == 0) atomicExch(p.ws_err, kDevErrTimeout);
    return;
  }

  // ============================ compute warps ============================
  const int ctid = tid - 32;
  const int cw = warp - 1;
  uint32_t stage = 0;
  bool aborted = false;

  for (int w = blockIdx.x; w < total; w += gridDim.x) {
    int seq, kvh, part;
    find_item(w, prefix, nseq, hkv, seq, kvh, part);
    const int len = clamp_len(p.context_lens[seq], p.max_context_len);
    const int t0 = part * pt;
    const int ntok = min(len - t0, pt);
    const int nparts = len > 0 ? (len + pt - 1) / pt : 1;
    const int64_t obase = (static_cast<int64_t>(seq) * p.num_q_heads + kvh * G) * D;

    if (ntok <= 0) {  // empty sequence: zero output
      for (int i = ctid; i < G * D; i += kConsumerThreads) store_out(p.out, p.out_bf16, obase + i, 0.f);
      continue;
    }
    const int nst = (ntok + S::kTokStage - 1) / S::kTokStage;

    // ---------------- scores: s = (q * scale * log2 e) . K ----------------
    {
      const int c = ctid % S::kLpt;
      const int tq = (ctid / S::kLpt) % S::kSwz;
      const int tslot = ctid / S::kLpt;
      float2 qr[G][S::kCpl][kV2];
      for (int s = 0; s < nst; ++s) {
        const int slot = stage % kStages;
        const uint32_t par = (stage / kStages) & 1u;
        if (!aborted && !ptx::mbar_wait(&full[slot], par, kWaitLimitNs)) aborted = true;
        const unsigned char* st = ring + slot * S::kStageAlloc;
        if (s == 0) {
          const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int j = 0; j < S::kCpl; ++j) {
              const int ch = c + S::kLpt * (j ^ tq);
              const uint4 raw =
                  *reinterpret_cast<const uint4*>(st + kStageBytes + g * S::kRow + ch * 16);
              Elem<T>::unpack(raw, qr[g][j]);
#pragma unroll
              for (int e = 0; e < kV2; ++e) qr[g][j][e] = __fmul2_rn(qr[g][j][e], sc2);
            }
        }
        const int nv = min(S::kTokStage, ntok - s * S::kTokStage);
        float* sc_stage = sc + s * S::kTokStage * G;
#pragma unroll
        for (int ps = 0; ps < S::kPasses; ++ps) {
          const int tl = ps * S::kTokPass + tslot;
          const unsigned char* krow = st + (tl < S::kTokStage ? tl : 0) * S::kRow;
          float2 acc[G];
#pragma unroll
          for (int g = 0; g < G; ++g) acc[g] = make_float2(0.f, 0.f);
#pragma unroll
          for (int j = 0; j < S::kCpl; ++j) {
            const int ch = c + S::kLpt * (j ^ tq);
            const uint4 raw = *reinterpret_cast<const uint4*>(krow + ch * 16);
            float2 k2[kV2];
            Elem<T>::unpack(raw, k2);
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
              for (int e = 0; e < kV2; ++e) acc[g] = __ffma2_rn(qr[g][j][e], k2[e], acc[g]);
          }
          float sg[G];
#pragma unroll
          for (int g = 0; g < G; ++g) sg[g] = acc[g].x + acc[g].y;
#pragma unroll
          for (int off = 1; off < S::kLpt; off <<= 1)
#pragma unroll
            for (int g = 0; g < G; ++g) sg[g] += __shfl_xor_sync(0xffffffffu, sg[g], off);
          if (c == 0 && tl < nv) {
            float* dstp = sc_stage + tl * G;
            if constexpr (G % 4 == 0) {
#pragma unroll
              for (int g = 0; g < G; g += 4)
                *reinterpret_cast<float4*>(dstp + g) = make_float4(sg[g], sg[g + 1], sg[g + 2], sg[g + 3]);
            } else if constexpr (G == 2) {
              *reinterpret_cast<float2*>(dstp) = make_float2(sg[0], sg[1]);
            } else {
              dstp[0] = sg[0];
            }
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&empty[slot]);
        ++stage;
      }
    }
    ptx::bar_sync(1, kConsumerThreads);

    // ---------------- softmax over the partition (log2 domain) ----------------
    {
      const int n = ntok * G;
      const int gq = ctid % G;
      float mx = -CUDART_INF_F;
      for (int i = ctid; i < n; i += kConsumerThreads) mx = fmaxf(mx, sc[i]);
#pragma unroll
      for (int off = G; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      if (lane < G) red_m[cw * G + lane] = mx;
      ptx::bar_sync(1, kConsumerThreads);
      float m = red_m[gq];
#pragma unroll
      for (int k = 1; k < kConsumerWarps; ++k) m = fmaxf(m, red_m[k * G + gq]);
      float sum = 0.f;
      for (int i = ctid; i < n; i += kConsumerThreads) {
        const float e = exp2f(sc[i] - m);
        sc[i] = e;
        sum += e;
      }
#pragma unroll
      for (int off = G; off < 32; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      if (lane < G) red_l[cw * G + lane] = sum;
      ptx::bar_sync(1, kConsumerThreads);
    }

    // ---------------- o = P . V ----------------
    float2 o[G][kV2];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < kV2; ++e) o[g][e] = make_float2(0.f, 0.f);
    {
      const int dg = ctid % S::kDg;
      const int tg = ctid / S::kDg;
      for (int s = 0; s < nst; ++s) {
        const int slot = stage % kStages;
        const uint32_t par = (stage / kStages) & 1u;
        if (!aborted && !ptx::mbar_wait(&full[slot], par, kWaitLimitNs)) aborted = true;
        const unsigned char* st = ring + slot * S::kStageAlloc;
        const int nv = min(S::kTokStage, ntok - s * S::kTokStage);
        const float* psc = sc + s * S::kTokStage * G;
        for (int tl = tg; tl < nv; tl += S::kTg) {
          const uint4 raw = *reinterpret_cast<const uint4*>(st + tl * S::kRow + dg * 16);
          float2 v2[kV2];
          Elem<T>::unpack(raw, v2);
          float pg[G];
          if constexpr (G % 4 == 0) {
#pragma unroll
            for (int g = 0; g < G; g += 4) {
              const float4 t4 = *reinterpret_cast<const float4*>(psc + tl * G + g);
              pg[g] = t4.x; pg[g + 1] = t4.y; pg[g + 2] = t4.z; pg[g + 3] = t4.w;
            }
          } else if constexpr (G == 2) {
            const float2 t2 = *reinterpret_cast<const float2*>(psc + tl * G);
            pg[0] = t2.x; pg[1] = t2.y;
          } else {
            pg[0] = psc[tl];
          }
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float2 pp = make_float2(pg[g], pg[g]);
#pragma unroll
            for (int e = 0; e < kV2; ++e) o[g][e] = __ffma2_rn(pp, v2[e], o[g][e]);
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&empty[slot]);
        ++stage;
      }
    }

    // ---------------- epilogue ----------------
#pragma unroll
    for (int off = S::kDg; off < 32; off <<= 1)
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < kV2; ++e) {
          o[g][e].x += __shfl_xor_sync(0xffffffffu, o[g][e].x, off);
          o[g][e].y += __shfl_xor_sync(0xffffffffu, o[g][e].y, off);
        }
    if (lane < S::kDg) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < kV2; ++e)
          *reinterpret_cast<float2*>(red + (cw * G + g) * D + lane * S::kVec + 2 * e) = o[g][e];
    }
    ptx::bar_sync(1, kConsumerThreads);

    if (nparts == 1) {
      for (int i = ctid; i < G * D; i += kConsumerThreads) {
        const int g = i / D;
        float l = 0.f, a = 0.f;
#pragma unroll
        for (int k = 0; k < kConsumerWarps; ++k) {
          l += red_l[k * G + g];
          a += red[k * G * D + i];
        }
        store_out(p.out, p.out_bf16, obase + i, a / l);
      }
    } else {
      const int row = seq * hkv + kvh;
      const int64_t rec = static_cast<int64_t>(row) * p.max_parts + part;
      float* po = p.ws_o + rec * G * D;
      for (int i = ctid; i < G * D; i += kConsumerThreads) {
        float a = 0.f;
#pragma unroll
        for (int k = 0; k < kConsumerWarps; ++k) a += red[k * G * D + i];
        po[i] = a;
      }
      if (ctid < G) {
        float m = red_m[ctid], l = red_l[ctid];
#pragma unroll
        for (int k = 1; k < kConsumerWarps; ++k) {
          m = fmaxf(m, red_m[k * G + ctid]);
          l += red_l[k * G + ctid];
        }
        p.ws_ml[rec * G * 2 + 2 * ctid] = m;
        p.ws_ml[rec * G * 2 + 2 * ctid + 1] = l;
      }
      // release: every writer orders its partial stores before the barrier;
      // the counting thread acquires right after the atomic and only then
      // publishes the result
      __threadfence();
      ptx::bar_sync(1, kConsumerThreads);
      if (ctid == 0) {
        const int arrived = atomicAdd(&p.ws_counters[row], 1);
        __threadfence();
        flags[1] = (arrived == nparts - 1) ? 1 : 0;
      }
      ptx::bar_sync(1, kConsumerThreads);
      if (flags[1]) {
        // last partition of this (sequence, kv head) to finish: merge
        const float* mlrow = p.ws_ml + static_cast<int64_t>(row) * p.max_parts * G * 2;
        const float* orow = p.ws_o + static_cast<int64_t>(row) * p.max_parts * G * D;
        float* wm = sc;                // [nparts * G]: max, then merge weights
        float* wl = sc + nparts * G;   // [nparts * G]: sums
        for (int idx = ctid; idx < nparts * G; idx += kConsumerThreads) {
          wm[idx] = __ldcg(mlrow + 2 * idx);
          wl[idx] = __ldcg(mlrow + 2 * idx + 1);
        }
        ptx::bar_sync(1, kConsumerThreads);
        if (ctid < G) {
          float M = -CUDART_INF_F;
          for (int q = 0; q < nparts; ++q) M = fmaxf(M, wm[q * G + ctid]);
          float L = 0.f;
          for (int q = 0; q < nparts; ++q) L += exp2f(wm[q * G + ctid] - M) * wl[q * G + ctid];
          mrg[ctid] = M;
          mrg[G + ctid] = 1.f / L;
        }
        ptx::bar_sync(1, kConsumerThreads);
        for (int idx = ctid; idx < nparts * G; idx += kConsumerThreads) {
          const int g = idx % G;
          wm[idx] = exp2f(wm[idx] - mrg[g]) * mrg[G + g];
        }
        ptx::bar_sync(1, kConsumerThreads);
        for (int i = ctid; i < G * D; i += kConsumerThreads) {
          const int g = i / D;
          float a = 0.f;
          for (int q = 0; q < nparts; ++q) a += wm[q * G + g] * __ldcg(orow + static_cast<int64_t>(q) * G * D + i);
          store_out(p.out, p.out_bf16, obase + i, a);
        }
        if (ctid == 0) p.ws_counters[row] = 0;
      }
    }
    if (aborted) flags[0] = 1;
    ptx::bar_sync(1, kConsumerThreads);  // shared buffers are reused by the next item
    if (flags[0]) break;
  }
  if (flags[0] && ctid == 0) atomicExch(p.ws_err, kDevErrTimeout);
}

// Registration helper used by the per-dtype instantiation units.
template <typename T, int D, int G>
inline void fill_info(DecodeKernelInfo* info) {
  using S = decode_detail::Shape<decode_detail::Elem<T>::kBytes, D, G>;
  info->fn = reinterpret_cast<const void*>(&paged_decode_kernel<T, D, G>);
  info->ring_bytes = kStages * S::kStageAlloc;
  info->tokens_per_stage = S::kTokStage;
  info->q_bytes = S::kQBytes;
}

}  // namespace pa
