// KV slot write and copy-on-write block copy.
//
// Slot write ("PagedAttention", section "Block Table 如何工作"; "LLM KV cache
// 02 - serving engine KV", section 2): a generating sequence writes each new
// token's K/V into its slot, physical_block * block_size + offset.
// Block copy ("PagedAttention", section "支持块级共享"): a shared block is
// copied to a fresh one before a branch writes different content into it.
//
// Both also run over the L layers of a pool that holds every layer's cache
// at a fixed stride, in one launch: a step's append writes a token's K/V in
// every layer ("PagedAttention", section "KV Cache 为什么难管理": a token
// costs 2 * L * H_kv * d elements of cache), and a copy-on-write copies the
// block in every layer.
//
// Both are pure data movement in 16-byte vectors: consecutive threads move
// consecutive 16-byte chunks of a token row (slot write) or of a whole block
// (copy), so every global access is coalesced.  Out-of-range slots / blocks
// are skipped, never written.
//
// Checked mode (a device status word): the slot write reports a slot past
// the pool instead of skipping it silently, and the copy first validates its
// pairs (every block in the pool, destinations distinct and none also a
// source, the condition under which copying pair by pair equals copying from
// the state before the call) and copies nothing if any pair fails.
#include "decode.cuh"
#include "ptx.cuh"

namespace pa {
namespace {

// Layer l of every buffer starts l * stride 16-byte chunks after layer 0
// (one pool holding all layers); blockIdx.y is the layer.
__global__ void __launch_bounds__(256)
    reshape_and_cache_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                             int64_t kv_layer_chunks, int32_t num_tokens,
                             const int64_t* __restrict__ slots, uint4* __restrict__ k_cache,
                             uint4* __restrict__ v_cache, int64_t cache_layer_chunks,
                             int64_t num_slots, int32_t bs, int32_t hkv, int32_t chunks,
                             int32_t* __restrict__ status) {
  // a decode launched behind this append may begin its set-up now; it waits
  // for this grid's writes before reading the cache
  ptx::griddep_launch_dependents();
  const int32_t per_token = hkv * chunks;  // 16-byte chunks of one token's K (all kv heads)
  const int64_t total = static_cast<int64_t>(num_tokens) * per_token;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t layer = blockIdx.y;
  key += layer * kv_layer_chunks;
  value += layer * kv_layer_chunks;
  k_cache += layer * cache_layer_chunks;
  v_cache += layer * cache_layer_chunks;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t t = i / per_token;
    const int32_t r = static_cast<int32_t>(i - t * per_token);
    const int64_t slot = slots[t];
    if (slot < 0) continue;  // padding
    if (slot >= num_slots) {  // past the pool: never written; reported in checked mode
      if (status && r == 0 && blockIdx.y == 0) atomicExch(status, kDevErrInvalidArg);
      continue;
    }
    const int64_t blk = slot / bs;
    const int32_t off = static_cast<int32_t>(slot - blk * bs);
    const int32_t h = r / chunks;
    const int32_t c = r - h * chunks;
    const int64_t dst = ((blk * hkv + h) * bs + off) * chunks + c;
    k_cache[dst] = key[i];
    v_cache[dst] = value[i];
  }
}

// blockIdx.x: pair; blockIdx.y: layer * 2 + (0 K, 1 V); blockIdx.z: slice of
// the block.  gate (checked mode): nothing is copied while *gate != 0.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                       int64_t cache_layer_chunks, int32_t num_blocks, int64_t chunks_per_block,
                       const int64_t* __restrict__ pairs, const int32_t* gate) {
  if (gate && *reinterpret_cast<const volatile int32_t*>(gate) != 0) return;
  const int64_t src = pairs[2 * static_cast<int64_t>(blockIdx.x)];
  const int64_t dst = pairs[2 * static_cast<int64_t>(blockIdx.x) + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return;
  uint4* base = ((blockIdx.y & 1u) ? v_cache : k_cache) + (blockIdx.y >> 1) * cache_layer_chunks;
  const uint4* s = base + src * chunks_per_block;
  uint4* d = base + dst * chunks_per_block;
  const int64_t step = static_cast<int64_t>(blockDim.x) * gridDim.z;
  for (int64_t i = static_cast<int64_t>(blockIdx.z) * blockDim.x + threadIdx.x; i < chunks_per_block;
       i += step)
    d[i] = s[i];
}

// Checked copy: thread i owns pair i and compares it with every pair j,
// staged through shared memory a tile at a time (num_pairs^2 comparisons in
// all: a debugging aid, not a hot-path step).  Any block outside
// [0, num_blocks), a destination named twice, or a destination that is also
// a source (itself included) sets *status.
constexpr int kPairTile = 256;
__global__ void __launch_bounds__(kPairTile)
    validate_pairs_kernel(const int64_t* __restrict__ pairs, int32_t num_pairs, int32_t num_blocks,
                          int32_t* __restrict__ status) {
  __shared__ int64_t tsrc[kPairTile], tdst[kPairTile];
  const int i = blockIdx.x * kPairTile + threadIdx.x;
  const bool mine = i < num_pairs;
  const int64_t si = mine ? pairs[2 * static_cast<int64_t>(i)] : 0;
  const int64_t di = mine ? pairs[2 * static_cast<int64_t>(i) + 1] : 0;
  bool bad = mine && (si < 0 || si >= num_blocks || di < 0 || di >= num_blocks);
  for (int j0 = 0; j0 < num_pairs; j0 += kPairTile) {
    const int j = j0 + threadIdx.x;
    if (j < num_pairs) {
      tsrc[threadIdx.x] = pairs[2 * static_cast<int64_t>(j)];
      tdst[threadIdx.x] = pairs[2 * static_cast<int64_t>(j) + 1];
    }
    __syncthreads();
    const int n = min(kPairTile, num_pairs - j0);
    if (mine && !bad) {
      for (int k = 0; k < n; ++k) {
        if (tsrc[k] == di || (tdst[k] == di && j0 + k != i)) {
          bad = true;
          break;
        }
      }
    }
    __syncthreads();
  }
  if (bad) atomicExch(status, kDevErrInvalidArg);
}

}  // namespace

cudaError_t launch_reshape_and_cache(const void* key, const void* value, int64_t kv_layer_bytes,
                                     int32_t num_layers, int32_t num_tokens,
                                     const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                     int64_t cache_layer_bytes, int32_t num_blocks,
                                     int32_t block_size, int32_t num_kv_heads, int32_t row_bytes,
                                     int32_t* status, cudaStream_t stream) {
  const int32_t chunks = row_bytes / 16;
  const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * chunks;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  // about 16 CTAs per SM in all, grid-striding beyond that
  int64_t cap = device_sm_count() * 16 / num_layers;
  if (cap < 1) cap = 1;
  if (blocks > cap) blocks = cap;
  reshape_and_cache_kernel<<<dim3(static_cast<unsigned>(blocks), static_cast<unsigned>(num_layers)),
                             threads, 0, stream>>>(
      static_cast<const uint4*>(key), static_cast<const uint4*>(value), kv_layer_bytes / 16,
      num_tokens, slot_mapping, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
      cache_layer_bytes / 16, static_cast<int64_t>(num_blocks) * block_size, block_size,
      num_kv_heads, chunks, status);
  return cudaGetLastError();
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, int64_t cache_layer_bytes,
                               int32_t num_layers, int32_t num_blocks, int64_t block_bytes,
                               const int64_t* pairs, int32_t num_pairs, int32_t* status,
                               cudaStream_t stream) {
  if (status) {
    validate_pairs_kernel<<<static_cast<unsigned>((num_pairs + kPairTile - 1) / kPairTile), kPairTile, 0,
                            stream>>>(pairs, num_pairs, num_blocks, status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int64_t chunks = block_bytes / 16;
  const int threads = 256;
  // about 8 chunks (128 bytes) per thread per CTA
  int64_t split = (chunks + threads * 8 - 1) / (threads * 8);
  if (split < 1) split = 1;
  if (split > 64) split = 64;
  dim3 grid(static_cast<unsigned>(num_pairs), static_cast<unsigned>(2 * num_layers),
            static_cast<unsigned>(split));
  copy_blocks_kernel<<<grid, threads, 0, stream>>>(static_cast<uint4*>(k_cache),
                                                   static_cast<uint4*>(v_cache),
                                                   cache_layer_bytes / 16, num_blocks, chunks,
                                                   pairs, status);
  return cudaGetLastError();
}

}  // namespace pa
