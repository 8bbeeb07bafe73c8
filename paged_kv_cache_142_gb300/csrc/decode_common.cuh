// Device helpers shared by the paged decode kernels.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include "decode.cuh"
#include "ptx.cuh"

namespace pa {
namespace decode_detail {

template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kBytes = 4;
  __device__ __forceinline__ static void unpack(const uint4& r, float2 (&o)[2]) {
    o[0] = make_float2(__uint_as_float(r.x), __uint_as_float(r.y));
    o[1] = make_float2(__uint_as_float(r.z), __uint_as_float(r.w));
  }
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  __device__ __forceinline__ static float2 pair(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  __device__ __forceinline__ static void unpack(const uint4& r, float2 (&o)[4]) {
    o[0] = pair(r.x);
    o[1] = pair(r.y);
    o[2] = pair(r.z);
    o[3] = pair(r.w);
  }
};

// Context lengths outside [0, max_len] are clamped (the workspace is sized
// for max_len); the caller reports them.
__device__ __forceinline__ int clamp_len(int len, int max_len) {
  return len < 0 ? 0 : (len > max_len ? max_len : len);
}

// Largest s with prefix[s] <= w (prefix strictly increasing, prefix[0] = 0).
__device__ __forceinline__ void find_item(int w, const int32_t* prefix, int nseq, int hkv,
                                          int& seq, int& kvh, int& part) {
  int lo = 0, hi = nseq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= w) lo = mid;
    else hi = mid - 1;
  }
  seq = lo;
  const int u = w - prefix[lo];
  part = u / hkv;
  kvh = u - part * hkv;
}

__device__ __forceinline__ void store_out(void* out, int bf16, int64_t i, float v) {
  if (bf16) static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
  else static_cast<float*>(out)[i] = v;
}


// Work items are (sequence, kv head, partition); sequence i owns
// max(1, ceil(len_i / part_tokens)) * num_kv_heads of them, enumerated
// sequence-major, partition-major, kv head fastest.  Every thread of the CTA
// calls this; prefix[0..num_seqs] receives the exclusive prefix sum (and
// lens_out, if given, the clamped lengths) and the CTA is synchronised on
// return.  CTA 0 reports lengths outside
// [0, max_context_len] in the workspace error word.
__device__ __forceinline__ void build_item_prefix(const DecodeParams& p, int32_t* prefix,
                                                  int* warp_sums, int tid, int nthreads,
                                                  int32_t* lens_out = nullptr) {
  const int nseq = p.num_seqs;
  const int pt = p.part_tokens;
  const int hkv = p.num_kv_heads;
  const int lane = tid & 31, warp = tid >> 5;
  const int per = (nseq + nthreads - 1) / nthreads;
  const int beg = min(nseq, tid * per);
  const int end = min(nseq, beg + per);
  int local = 0;
  for (int i = beg; i < end; ++i) {
    const int raw = p.context_lens[i];
    if (blockIdx.x == 0 && (raw < 0 || raw > p.max_context_len)) atomicExch(p.ws_err, kDevErrInvalidArg);
    const int len = clamp_len(raw, p.max_context_len);
    if (lens_out) lens_out[i] = len;
    local += max(1, (len + pt - 1) / pt) * hkv;
  }
  int x = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  int run = x - local;
  for (int w = 0; w < warp; ++w) run += warp_sums[w];
  for (int i = beg; i < end; ++i) {
    prefix[i] = run;
    const int len = clamp_len(p.context_lens[i], p.max_context_len);
    run += max(1, (len + pt - 1) / pt) * hkv;
  }
  if (tid == nthreads - 1) prefix[nseq] = run;
  __syncthreads();
}

}  // namespace decode_detail
}  // namespace pa
