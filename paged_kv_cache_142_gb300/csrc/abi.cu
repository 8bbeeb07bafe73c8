// C ABI shim: argument validation, split-K planning, workspace carve-up and
// launches on the caller's stream.  Declarations and contracts: include/pa.h.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>

#include "decode.cuh"
#include "pa.h"

namespace pa {
bool decode_info_bf16(int head_dim, int group, DecodeKernelInfo* info);
bool decode_info_f32(int head_dim, int group, DecodeKernelInfo* info);

bool decode_kernel_info(int dtype_bf16, int head_dim, int group, DecodeKernelInfo* info) {
  return dtype_bf16 ? decode_info_bf16(head_dim, group, info)
                    : decode_info_f32(head_dim, group, info);
}

constexpr int64_t kSmCountDefault = 152;  // GB300; used only when no device can be queried

// SMs of the current device, which shape the default partition sizes (host
// planning calls also work without a GPU, with the GB300's count).
int64_t device_sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();  // clear the query's error
    return kSmCountDefault;
  }
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      return kSmCountDefault;
    }
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}
}  // namespace pa

namespace {

using pa::DecodeKernelInfo;
using pa::DecodeParams;

// Timeout-path test hook (pa_test_stall_decode): 0 = off.
std::atomic<uint64_t> g_test_stall_ns{0};
// kv heads per decode work item (pa_set_decode_kv_per_item): 0 = automatic.
std::atomic<int> g_kv_per_item{0};

constexpr int kMaxSmem = 227 * 1024;
constexpr int kDefaultPartTokens = 256;
constexpr int32_t kMaxLayers = 32767;  // grid y of the copy kernel holds 2 * layers
int dtype_bytes(pa_dtype d) {
  return d == PA_DTYPE_F32 ? 4 : (d == PA_DTYPE_BF16 ? 2 : 0);
}
bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

pa_status check_cache_shape(int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                            int32_t head_dim, pa_dtype dtype) {
  if (num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0) return PA_ERR_INVALID_ARG;
  if (dtype_bytes(dtype) == 0) return PA_ERR_INVALID_ARG;
  if (!is_pow2(block_size) || block_size > 256) return PA_ERR_UNSUPPORTED;
  const int64_t row = static_cast<int64_t>(head_dim) * dtype_bytes(dtype);
  if (row % 16 != 0) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

// Tensor-core kernel layout constants (must match decode_umma.cuh).
constexpr int kUmmaThreadsHost = 448;
constexpr int kUmmaTileBytesHost = 32768;
// per compute group scratch of the tensor-core decode (with an item's totals for G >= 8)
// (must match umma_small_bytes in decode_umma.cuh)
constexpr int umma_small_bytes_host(int HG, int kh) { return (HG >= 8 || kh == 2) ? 1280 : 1024; }
constexpr int kPrefillThreads = 256;  // must match the prefill kernel

struct Plan {
  DecodeKernelInfo info;
  bool umma;       // tensor-core kernel (bf16, head_dim 128, block >= 8)
  int kh;          // kv heads per work item (tensor cores: 2 for G <= 4, blocks of 8..64)
  int stages, stages_v;
  int tbl_stride;
  int off_q, off_p, off_small, off_lens;
  int group;
  int part_tokens;
  int max_parts;
  int smem;
  int off_sc, off_red, off_tbl, off_prefix, off_bar;
  size_t ws_counters, ws_ml, ws_o, ws_total;
};

pa_status make_plan(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                    int32_t head_dim, int32_t block_size, pa_dtype dtype,
                    int32_t max_context_len, int32_t partition_tokens, Plan* pl) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_context_len < 0 ||
      partition_tokens < 0)
    return PA_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  if (dtype_bytes(dtype) == 0) return PA_ERR_INVALID_ARG;
  if (!is_pow2(block_size) || block_size > 256) return PA_ERR_UNSUPPORTED;
  const int G = num_q_heads / num_kv_heads;
  std::memset(pl, 0, sizeof(*pl));
  pl->group = G;
  // bf16 K/V with head_dim 128 and blocks of >= 8 tokens run on the tensor
  // cores; everything else on the CUDA-core kernel
  pl->umma = dtype == PA_DTYPE_BF16 && head_dim == 128 && block_size >= 8 &&
             pa::decode_umma_fn(G, 1) != nullptr;
  // two kv heads per item: one TMA box per block covers both heads (twice the
  // bytes per copy) and half as many items, with the same MMA shapes.  Taken
  // only with about five such items per SM or more: with fewer, the longer
  // items leave SMs idle at the end of the launch (GQA G = 4 sweep: one head
  // per item wins up to 1024 sequence x kv-head pairs, two heads from 1536).
  const int64_t pair_items = static_cast<int64_t>(num_seqs) * (num_kv_heads / 2);
  const bool pairs_ok = pl->umma && G <= 4 && num_kv_heads % 2 == 0 && block_size <= 64 &&
                        pa::decode_umma_fn(G, 2) != nullptr;
  const int want_kh = g_kv_per_item.load(std::memory_order_relaxed);
  pl->kh = pairs_ok && (want_kh == 2 || (want_kh == 0 && pair_items >= 5 * pa::device_sm_count())) ? 2 : 1;
  if (!pl->umma && !pa::decode_kernel_info(dtype == PA_DTYPE_BF16, head_dim, G, &pl->info))
    return PA_ERR_UNSUPPORTED;
  // partition size: a multiple of the block size and of the stage (tensor
  // cores: of the 128-token tile); at most part/2 partitions per sequence
  const int64_t unit = pl->umma ? 128 / pl->kh : pl->info.tokens_per_stage;
  const int64_t gran = block_size > unit ? block_size : unit;
  // tensor cores: long partitions (each item costs a block-table load, a
  // query load and an epilogue; fewer items mean fewer merges), 4096 tokens
  // for contexts past 4096 and 2048 otherwise, halved while the (sequence, kv
  // head, partition) items would not give every SM two; CUDA cores: 256
  int64_t def_pt = kDefaultPartTokens;
  if (pl->umma) {
    def_pt = max_context_len > 4096 ? 4096 : 2048;
    const int64_t units = static_cast<int64_t>(num_seqs) * (num_kv_heads / pl->kh);
    const int64_t sms = pa::device_sm_count();
    while (def_pt > 256 && units * ceil_div(max_context_len, def_pt) < 2 * sms) def_pt /= 2;
  }
  int64_t pt = round_up(partition_tokens > 0 ? partition_tokens : def_pt, gran);
  while (ceil_div(max_context_len, pt) > pt / 2) pt *= 2;
  if (pt > (1 << 20)) return PA_ERR_UNSUPPORTED;
  pl->part_tokens = static_cast<int>(pt);
  pl->max_parts = static_cast<int>(ceil_div(max_context_len, pt) > 1 ? ceil_div(max_context_len, pt) : 1);
  // shared memory
  if (pl->umma) {
    // K ring | V ring | queries [2 groups] | P [2 groups][2] | per-group
    // scratch | barriers, flags | table slices [2 streams][2 groups] |
    // lengths | prefix | align slack
    const int HG = G * pl->kh;  // query heads per item
    const int64_t pbytes = HG <= 8 ? 4096 : 8192;
    const int64_t tbl_stride = round_up(pt / block_size + 1, 4);
    const int64_t fixed = 2 * 4096 + 2 * 2 * pbytes + 2 * umma_small_bytes_host(HG, pl->kh) + 256 + 1024 + 4 * tbl_stride * 4 +
                          round_up(static_cast<int64_t>(num_seqs) * 4, 16) +
                          2 * round_up((static_cast<int64_t>(num_seqs) + 4) / 4 * 4 * 4, 16) + 1024;
    int sk = 3, sv = 3;
    while (sk + sv > 4 && (sk + sv) * kUmmaTileBytesHost + fixed > kMaxSmem) {
      if (sv > sk) --sv; else --sk;
    }
    if ((sk + sv) * kUmmaTileBytesHost + fixed > kMaxSmem) {
      pl->umma = false;  // too many sequences for one CTA's shared memory: CUDA cores
    } else {
      pl->stages = sk;
      pl->stages_v = sv;
      pl->tbl_stride = static_cast<int>(tbl_stride);
      int64_t off = static_cast<int64_t>(sk + sv) * kUmmaTileBytesHost;
      pl->off_q = static_cast<int>(off);
      off += 2 * 4096;
      pl->off_p = static_cast<int>(off);
      off += 2 * 2 * pbytes;
      pl->off_small = static_cast<int>(off);
      off += 2 * umma_small_bytes_host(HG, pl->kh) + 256;  // per-group scratch, then the two item queues
      pl->off_bar = static_cast<int>(off);
      off += 1024;
      pl->off_tbl = static_cast<int>(off);  // [K/V stream][group]
      off += 4 * tbl_stride * 4;
      pl->off_lens = static_cast<int>(off);
      off += round_up(static_cast<int64_t>(num_seqs) * 4, 16);
      pl->off_prefix = static_cast<int>(off);  // prefix and tail-order arrays of (num_seqs + 4) & ~3 ints
      off += 2 * round_up((static_cast<int64_t>(num_seqs) + 4) / 4 * 4 * 4, 16);
      pl->smem = static_cast<int>(off + 1024);  // slack to align the base to 1024 bytes
    }
  }
  if (!pl->umma) pl->kh = 1;
  if (!pl->umma && !pl->info.fn &&
      !pa::decode_kernel_info(dtype == PA_DTYPE_BF16, head_dim, G, &pl->info))
    return PA_ERR_UNSUPPORTED;
  if (!pl->umma) {
    int64_t off = pl->info.ring_bytes;
    pl->off_sc = static_cast<int>(off);
    off += round_up(pt * G * 4, 16);
    pl->off_red = static_cast<int>(off);
    off += round_up((static_cast<int64_t>(pa::kConsumerWarps) * G * head_dim + 2 * pa::kConsumerWarps * G + 2 * G) * 4, 16);
    pl->off_tbl = static_cast<int>(off);
    off += round_up((pt / block_size + 1) * 4, 16);
    pl->off_prefix = static_cast<int>(off);
    off += round_up((static_cast<int64_t>(num_seqs) + 1) * 4, 16);
    pl->off_bar = static_cast<int>(off);
    off += 2 * pa::kStages * 8;
    if (off + 64 > kMaxSmem) return PA_ERR_UNSUPPORTED;  // + static shared memory
    pl->smem = static_cast<int>(off);
  }
  // workspace: header | counters | (max, sum) partials | output partials, by
  // (sequence, kv-head group) row and the group's kh * G query heads
  const int64_t rows = static_cast<int64_t>(num_seqs) * (num_kv_heads / pl->kh);
  const int64_t heads = static_cast<int64_t>(G) * pl->kh;
  pl->ws_counters = 256;
  int64_t w = 256 + round_up(rows * 4, 256);
  pl->ws_ml = static_cast<size_t>(w);
  if (pl->max_parts > 1) {
    w += round_up(rows * pl->max_parts * heads * 2 * 4, 256);
    pl->ws_o = static_cast<size_t>(w);
    w += round_up(rows * pl->max_parts * heads * static_cast<int64_t>(head_dim) * 4, 256);
  } else {
    pl->ws_o = static_cast<size_t>(w);
  }
  pl->ws_total = static_cast<size_t>(w);
  return PA_OK;
}

const void* plan_kernel(const Plan& pl) { return pl.umma ? pa::decode_umma_fn(pl.group, pl.kh) : pl.info.fn; }
int plan_threads(const Plan& pl) { return pl.umma ? kUmmaThreadsHost : pa::kDecodeThreads; }

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D map over rows of 128 bf16 (256 bytes): boxes of 64 elements (one
// 128-byte swizzle span) by box_rows rows.
bool encode_rows_128(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map over the K or V pool viewed as 8-row groups: (64 dims of a
// 128-byte swizzle span, 8 rows 256 bytes apart, 2 halves of the row 128
// bytes apart, row groups 2048 bytes apart).  One box of box_rows rows lands
// in shared memory as [row group][half][8 rows][128 B]: every 8-row atom of
// a half is a 1024-byte swizzle atom, atoms of one half 2048 bytes apart.
bool encode_kv_groups(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[4] = {64, 8, 2, static_cast<cuuint64_t>(rows / 8)};
  cuuint64_t strides[3] = {256, 128, 2048};
  cuuint32_t box[4] = {64, 8, 2, box_rows / 8};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-kernel dynamic shared memory attribute and occupancy, cached.
struct KernelCache {
  const void* fn;
  int device;
  int smem_set;
  int smem_occ;
  int occ;
};
std::mutex g_mu;
KernelCache g_cache[64];
int g_ncache = 0;

pa_status prepare_kernel(const void* fn, int threads, int smem, int* ctas) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  KernelCache* kc = nullptr;
  for (int i = 0; i < g_ncache; ++i)
    if (g_cache[i].fn == fn && g_cache[i].device == dev) kc = &g_cache[i];
  if (!kc) {
    if (g_ncache == 64) return PA_ERR_UNSUPPORTED;
    kc = &g_cache[g_ncache++];
    *kc = KernelCache{fn, dev, 0, -1, 0};
  }
  if (smem > kc->smem_set) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return PA_ERR_CUDA;
    kc->smem_set = smem;
  }
  if (kc->smem_occ != smem) {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, threads, smem) !=
        cudaSuccess)
      return PA_ERR_CUDA;
    kc->occ = occ;
    kc->smem_occ = smem;
  }
  if (kc->occ <= 0) return PA_ERR_UNSUPPORTED;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PA_ERR_CUDA;
  *ctas = sms * kc->occ;
  return PA_OK;
}

}  // namespace

extern "C" {

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_OOM: return "PA_ERR_OOM";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_DEVICE_TIMEOUT: return "PA_ERR_DEVICE_TIMEOUT";
  }
  return "PA_ERR_UNKNOWN";
}

const char* pa_version(void) { return "pa_gb300 1.0 sm_103a"; }

}  // extern "C"

namespace {
pa_status reshape_and_cache_impl(const void* key, const void* value, int64_t kv_layer_stride,
                                      int32_t num_layers, int32_t num_tokens,
                                      const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                      int64_t cache_layer_stride, int32_t num_blocks,
                                      int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                      pa_dtype dtype, int32_t* status, void* stream) {
  pa_status st = check_cache_shape(num_blocks, block_size, num_kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (num_tokens < 0 || num_layers < 1 || num_layers > kMaxLayers) return PA_ERR_INVALID_ARG;
  const int64_t e = dtype_bytes(dtype);
  const int64_t kv_layer = static_cast<int64_t>(num_tokens) * num_kv_heads * head_dim;
  const int64_t cache_layer = static_cast<int64_t>(num_blocks) * num_kv_heads * block_size * head_dim;
  if (num_layers > 1 && (kv_layer_stride < kv_layer || cache_layer_stride < cache_layer ||
                         (kv_layer_stride * e) % 16 != 0 || (cache_layer_stride * e) % 16 != 0))
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
  if (status && !aligned4(status)) return PA_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const int32_t row = head_dim * static_cast<int32_t>(e);
  cudaError_t err = pa::launch_reshape_and_cache(
      key, value, num_layers > 1 ? kv_layer_stride * e : 0, num_layers, num_tokens, slot_mapping,
      k_cache, v_cache, num_layers > 1 ? cache_layer_stride * e : 0, num_blocks, block_size,
      num_kv_heads, row, status, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
}  // namespace

extern "C" {

pa_status pa_reshape_and_cache_layers(const void* key, const void* value, int64_t kv_layer_stride,
                                      int32_t num_layers, int32_t num_tokens,
                                      const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                      int64_t cache_layer_stride, int32_t num_blocks,
                                      int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                      pa_dtype dtype, void* stream) {
  return reshape_and_cache_impl(key, value, kv_layer_stride, num_layers, num_tokens, slot_mapping,
                                k_cache, v_cache, cache_layer_stride, num_blocks, block_size,
                                num_kv_heads, head_dim, dtype, nullptr, stream);
}

pa_status pa_reshape_and_cache(const void* key, const void* value, int32_t num_tokens,
                               const int64_t* slot_mapping, void* k_cache, void* v_cache,
                               int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                               int32_t head_dim, pa_dtype dtype, void* stream) {
  return pa_reshape_and_cache_layers(key, value, 0, 1, num_tokens, slot_mapping, k_cache, v_cache,
                                     0, num_blocks, block_size, num_kv_heads, head_dim, dtype,
                                     stream);
}

pa_status pa_reshape_and_cache_checked(const void* key, const void* value, int32_t num_tokens,
                                       const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                       int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                       int32_t head_dim, pa_dtype dtype, int32_t* status,
                                       void* stream) {
  if (!status) return PA_ERR_INVALID_ARG;
  return reshape_and_cache_impl(key, value, 0, 1, num_tokens, slot_mapping, k_cache, v_cache, 0,
                                num_blocks, block_size, num_kv_heads, head_dim, dtype, status,
                                stream);
}

}  // extern "C"

namespace {
pa_status copy_blocks_impl(void* k_cache, void* v_cache, int64_t cache_layer_stride,
                                int32_t num_layers, int32_t num_blocks, int32_t block_size,
                                int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype,
                                const int64_t* block_pairs, int32_t num_pairs, int32_t* status,
                                void* stream) {
  pa_status st = check_cache_shape(num_blocks, block_size, num_kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (num_pairs < 0 || num_layers < 1 || num_layers > kMaxLayers) return PA_ERR_INVALID_ARG;
  const int64_t e = dtype_bytes(dtype);
  const int64_t cache_layer = static_cast<int64_t>(num_blocks) * num_kv_heads * block_size * head_dim;
  if (num_layers > 1 && (cache_layer_stride < cache_layer || (cache_layer_stride * e) % 16 != 0))
    return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !block_pairs) return PA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
  if (status && !aligned4(status)) return PA_ERR_INVALID_ARG;
  const int64_t block_bytes = static_cast<int64_t>(num_kv_heads) * block_size * head_dim * e;
  cudaError_t err = pa::launch_copy_blocks(k_cache, v_cache,
                                           num_layers > 1 ? cache_layer_stride * e : 0, num_layers,
                                           num_blocks, block_bytes, block_pairs, num_pairs, status,
                                           static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
}  // namespace

extern "C" {

pa_status pa_copy_blocks_layers(void* k_cache, void* v_cache, int64_t cache_layer_stride,
                                int32_t num_layers, int32_t num_blocks, int32_t block_size,
                                int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype,
                                const int64_t* block_pairs, int32_t num_pairs, void* stream) {
  return copy_blocks_impl(k_cache, v_cache, cache_layer_stride, num_layers, num_blocks, block_size,
                          num_kv_heads, head_dim, dtype, block_pairs, num_pairs, nullptr, stream);
}

pa_status pa_copy_blocks_checked(void* k_cache, void* v_cache, int32_t num_blocks,
                                 int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                 pa_dtype dtype, const int64_t* block_pairs, int32_t num_pairs,
                                 int32_t* status, void* stream) {
  if (!status) return PA_ERR_INVALID_ARG;
  return copy_blocks_impl(k_cache, v_cache, 0, 1, num_blocks, block_size, num_kv_heads, head_dim,
                          dtype, block_pairs, num_pairs, status, stream);
}

pa_status pa_copy_blocks(void* k_cache, void* v_cache, int32_t num_blocks, int32_t block_size,
                         int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype,
                         const int64_t* block_pairs, int32_t num_pairs, void* stream) {
  return pa_copy_blocks_layers(k_cache, v_cache, 0, 1, num_blocks, block_size, num_kv_heads,
                               head_dim, dtype, block_pairs, num_pairs, stream);
}

// 2-D map over the queries [num_tokens, num_q_heads * 128] (bf16): boxes of
// 64 elements (one 128-byte swizzle span) by box_rows tokens.
bool encode_q_tokens(CUtensorMap* m, const void* base, uint64_t tokens, uint64_t row_elems,
                     uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {row_elems, tokens};
  cuuint64_t strides[1] = {row_elems * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over output rows [tokens][num_heads][128] of bf16 or fp32: boxes
// of one 128-byte swizzle span (64 bf16 or 32 fp32 elements) x hb heads x tb
// tokens, the rows of one softmax warp of the prefill kernel (hb * tb = 32).
bool encode_out_rows(CUtensorMap* m, void* base, bool fp32, uint64_t tokens, uint64_t heads, uint32_t hb,
                     uint32_t tb) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const uint64_t row = fp32 ? 512 : 256;
  cuuint64_t dims[3] = {128, heads, tokens};
  cuuint64_t strides[2] = {row, heads * row};
  cuuint32_t box[3] = {fp32 ? 32u : 64u, hb, tb};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides,
             box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor-core prefill kernel over `items` work items (any mode).
pa_status launch_prefill(pa::PrefillParams& p, int G, int64_t items, const void* q,
                         const void* k_cache, const void* v_cache, int64_t cache_rows,
                         void* stream) {
  if (items >= (int64_t(1) << 31)) return PA_ERR_UNSUPPORTED;
  if (items == 0) return PA_OK;
  // fp32 rows: the output of an fp32 prefill, or the shared-prefix partials
  const bool fp32_rows = p.mode != 0 || !p.out_bf16;
  const void* fn = pa::prefill_umma_fn(G, fp32_rows);
  const int smem = pa::prefill_umma_smem_bytes();
  int ctas = 0;
  pa_status st = prepare_kernel(fn, kPrefillThreads, smem, &ctas);
  if (st != PA_OK) return st;
  if (ctas > items) ctas = static_cast<int>(items);
  if (p.mode == 0) {
    // While every (sequence, kv head) pair's keys and values fit in half of L2
    // (the other half for the query and output streams), one block holds all
    // pairs: the tile-major order, whose round-robin waves have the most even
    // costs.  Past that, blocks of about two waves of the launch's items, so
    // that the CTAs at work share a few pairs' keys in L2.
    const int64_t pairs = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads;
    const int64_t tokens = static_cast<int64_t>(p.tiles_per_seq) * (128 / G);  // longest chunk, rounded up
    const int64_t kv_bytes = pairs * tokens * 2 * 128 * 2;                       // K and V, bf16, head_dim 128
    int64_t pb = (2 * static_cast<int64_t>(ctas) + p.tiles_per_seq - 1) / (p.tiles_per_seq > 0 ? p.tiles_per_seq : 1);
    if (kv_bytes <= (int64_t(64) << 20)) pb = pairs;
    p.pair_block = static_cast<int32_t>(pb < 1 ? 1 : (pb > pairs ? pairs : pb));
  }
  CUtensorMap tmq, tmk, tmv;
  const uint32_t box_rows = static_cast<uint32_t>(p.block_size < 128 ? p.block_size : 128);
  if (!encode_q_tokens(&tmq, q, static_cast<uint64_t>(p.num_tokens),
                       static_cast<uint64_t>(p.num_q_heads) * 128, static_cast<uint32_t>(128 / G)) ||
      !encode_kv_groups(&tmk, k_cache, static_cast<uint64_t>(cache_rows), box_rows) ||
      !encode_kv_groups(&tmv, v_cache, static_cast<uint64_t>(cache_rows), box_rows))
    return PA_ERR_CUDA;
  // full tiles' rows leave through shared memory and TMA stores: the bf16 or
  // fp32 output of a causal prefill, or the shared-prefix passes' fp32
  // partial O [parts + 1][num_seqs][num_q_heads][128] (else plain stores)
  CUtensorMap tmo = tmq;
  const uint32_t tq = static_cast<uint32_t>(128 / G);
  void* obase = p.mode == 0 ? p.out : static_cast<void*>(p.part_o);
  const uint64_t orows = p.mode == 0 ? static_cast<uint64_t>(p.num_tokens)
                                     : static_cast<uint64_t>(p.num_parts + 1) * static_cast<uint64_t>(p.num_seqs);
  p.o_tma = 0;
  if ((reinterpret_cast<uintptr_t>(obase) & 15u) == 0 &&
      encode_out_rows(&tmo, obase, fp32_rows, orows, static_cast<uint64_t>(p.num_q_heads),
                      tq >= 32 ? 1u : 32u / tq, tq >= 32 ? 32u : tq))
    p.o_tma = fp32_rows ? 2 : 1;
  else
    tmo = tmq;
  void* args[] = {&p, &tmq, &tmk, &tmv, &tmo};
  cudaError_t e = cudaLaunchKernel(fn, dim3(static_cast<unsigned>(ctas)), dim3(kPrefillThreads), args,
                                   static_cast<size_t>(smem), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_prefill(void* out, pa_dtype out_dtype, const void* q, int32_t num_tokens,
                     const int32_t* cu_q, const int32_t* q_start, int32_t num_seqs,
                     int32_t max_q_len, int32_t num_q_heads, const void* k_cache,
                     const void* v_cache, int32_t num_blocks, int32_t block_size,
                     int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype,
                     const int32_t* block_tables, int32_t max_blocks_per_seq, float scale,
                     int32_t* status, void* stream) {
  pa_status st = check_cache_shape(num_blocks, block_size, num_kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (num_tokens < 0 || num_seqs < 0 || max_q_len < 0 || num_q_heads <= 0 ||
      max_blocks_per_seq <= 0 || !(scale > 0.f) || dtype_bytes(out_dtype) == 0)
    return PA_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  const int G = num_q_heads / num_kv_heads;
  if (dtype != PA_DTYPE_BF16 || head_dim != 128 || block_size < 8 || !pa::prefill_umma_fn(G))
    return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0 || num_seqs == 0 || max_q_len == 0) return PA_OK;
  if (!out || !q || !cu_q || !q_start || !k_cache || !v_cache || !block_tables)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const int64_t cache_rows = static_cast<int64_t>(num_blocks) * num_kv_heads * block_size;
  if (cache_rows >= (int64_t(1) << 31)) return PA_ERR_UNSUPPORTED;
  const int TQ = 128 / G;
  pa::PrefillParams p{};
  p.out = out;
  p.out_bf16 = out_dtype == PA_DTYPE_BF16 ? 1 : 0;
  p.cu_q = cu_q;
  p.q_start = q_start;
  p.block_tables = block_tables;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.num_blocks = num_blocks;
  p.block_size = block_size;
  p.num_tokens = num_tokens;
  p.tiles_per_seq = (max_q_len + TQ - 1) / TQ;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status;
  const int64_t items = static_cast<int64_t>(num_seqs) * num_kv_heads * p.tiles_per_seq;
  return launch_prefill(p, G, items, q, k_cache, v_cache, cache_rows, stream);
}

// Shared-prefix decode: partition size of the groups' prefixes and the
// partial-result scratch [partitions + 1][num_seqs * num_q_heads][2 + 128].
namespace {
int64_t cascade_part_tokens(int64_t max_prefix, int64_t items_per_part) {
  // enough (prefix partition, tile, group, kv head) items for every SM twice,
  // partitions of at least 256 keys, in 128-key multiples
  int64_t parts = (2 * pa::device_sm_count() + items_per_part - 1) / (items_per_part > 0 ? items_per_part : 1);
  if (parts < 1) parts = 1;
  int64_t pt = (max_prefix + parts - 1) / parts;
  pt = round_up(pt < 256 ? 256 : pt, 128);
  return pt;
}
}  // namespace

// The partial-result scratch holds (max, sum) per (part, row), then the
// unnormalised O rows; the O part starts 256 bytes in, so that its 512-byte
// rows stay 16-byte aligned (vector and TMA stores) for any row count.
static int64_t cascade_ml_floats(int64_t parts, int64_t rows) { return round_up((parts + 1) * rows * 2, 64); }

size_t pa_decode_shared_prefix_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                              int32_t num_kv_heads, int32_t num_groups,
                                              int32_t max_group_size, int32_t max_prefix_len) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_groups < 0 ||
      max_group_size < 0 || max_prefix_len < 0 || num_q_heads % num_kv_heads)
    return 0;
  const int G = num_q_heads / num_kv_heads;
  if (!pa::prefill_umma_fn(G)) return 0;
  const int64_t tiles = (static_cast<int64_t>(max_group_size) + 128 / G - 1) / (128 / G);
  const int64_t pt = cascade_part_tokens(max_prefix_len, static_cast<int64_t>(num_groups) * num_kv_heads * tiles);
  const int64_t parts = (max_prefix_len + pt - 1) / pt;
  const int64_t rows = static_cast<int64_t>(num_seqs) * num_q_heads;
  return static_cast<size_t>((cascade_ml_floats(parts, rows) + (parts + 1) * rows * 128) * 4 + 256);
}

pa_status pa_decode_shared_prefix(void* out, pa_dtype out_dtype, const void* q, int32_t num_seqs,
                                  int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                  int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                  int32_t head_dim, pa_dtype dtype, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* context_lens,
                                  int32_t max_context_len, const int32_t* group_start,
                                  const int32_t* prefix_len, int32_t num_groups,
                                  int32_t max_group_size, int32_t max_prefix_len, float scale,
                                  int32_t* status, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  pa_status st = check_cache_shape(num_blocks, block_size, num_kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (num_seqs < 0 || num_q_heads <= 0 || num_groups < 0 || max_group_size < 0 ||
      max_prefix_len < 0 || max_context_len < 0 || max_blocks_per_seq <= 0 || !(scale > 0.f) ||
      dtype_bytes(out_dtype) == 0 || num_q_heads % num_kv_heads)
    return PA_ERR_INVALID_ARG;
  const int G = num_q_heads / num_kv_heads;
  if (dtype != PA_DTYPE_BF16 || head_dim != 128 || block_size < 8 || !pa::prefill_umma_fn(G))
    return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (num_groups <= 0 || !out || !q || !k_cache || !v_cache || !block_tables || !context_lens ||
      !group_start || !prefix_len || !workspace)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(workspace))
    return PA_ERR_INVALID_ARG;
  const size_t need = pa_decode_shared_prefix_workspace_size(num_seqs, num_q_heads, num_kv_heads,
                                                             num_groups, max_group_size, max_prefix_len);
  if (need == 0) return PA_ERR_UNSUPPORTED;
  if (workspace_bytes < need) return PA_ERR_WORKSPACE;
  const int64_t cache_rows = static_cast<int64_t>(num_blocks) * num_kv_heads * block_size;
  if (cache_rows >= (int64_t(1) << 31)) return PA_ERR_UNSUPPORTED;
  const int TQ = 128 / G;
  const int64_t tiles = (static_cast<int64_t>(max_group_size) + TQ - 1) / TQ;
  const int64_t pt = cascade_part_tokens(max_prefix_len, static_cast<int64_t>(num_groups) * num_kv_heads * tiles);
  const int64_t parts = (max_prefix_len + pt - 1) / pt;
  const int64_t rows = static_cast<int64_t>(num_seqs) * num_q_heads;
  pa::PrefillParams p{};
  p.out = out;
  p.out_bf16 = out_dtype == PA_DTYPE_BF16 ? 1 : 0;
  p.block_tables = block_tables;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.num_blocks = num_blocks;
  p.block_size = block_size;
  p.num_tokens = num_seqs;  // the queries are one row per sequence: q [num_seqs][H][128]
  p.tiles_per_seq = static_cast<int32_t>(tiles);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status;
  p.group_start = group_start;
  p.prefix_len = prefix_len;
  p.context_lens = context_lens;
  p.num_groups = num_groups;
  p.max_context_len = max_context_len;
  p.part_tokens = static_cast<int32_t>(pt);
  p.num_parts = static_cast<int32_t>(parts);
  p.part_ml = static_cast<float*>(workspace);
  p.part_o = p.part_ml + cascade_ml_floats(parts, rows);
  // one launch: the groups' prefixes (every member's queries against each
  // prefix block once), then every member's own tokens past its group's prefix
  p.mode = 3;
  // own-token items hold two members each (64-key halves of a tile) while a
  // block's TMA box fits in a half
  p.pack2 = block_size <= 64 ? 1 : 0;
  const int64_t own_items = (p.pack2 ? (static_cast<int64_t>(num_seqs) + 1) / 2 : num_seqs) * num_kv_heads;
  st = launch_prefill(p, G, parts * num_groups * num_kv_heads * tiles + own_items, q, k_cache, v_cache, cache_rows,
                      stream);
  if (st != PA_OK) return st;
  // then the log-sum-exp merge into out
  cudaError_t e = pa::launch_cascade_merge(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t block_size, pa_dtype dtype,
                                int32_t max_context_len, int32_t partition_tokens) {
  Plan pl;
  if (make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, dtype, max_context_len,
                partition_tokens, &pl) != PA_OK)
    return 0;
  return pl.ws_total;
}

pa_status pa_decode_plan(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, pa_dtype dtype,
                         int32_t max_context_len, int32_t partition_tokens,
                         int32_t* partition_tokens_out, int32_t* num_ctas_out) {
  Plan pl;
  pa_status st = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, dtype,
                           max_context_len, partition_tokens, &pl);
  if (st != PA_OK) return st;
  if (partition_tokens_out) *partition_tokens_out = pl.part_tokens;
  if (num_ctas_out) {
    int ctas = 0;
    st = prepare_kernel(plan_kernel(pl), plan_threads(pl), pl.smem, &ctas);
    if (st != PA_OK) return st;
    *num_ctas_out = ctas;
  }
  return PA_OK;
}

pa_status pa_decode(void* out, pa_dtype out_dtype, const void* q, int32_t num_seqs,
                    int32_t num_q_heads, const void* k_cache, const void* v_cache,
                    int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                    int32_t head_dim, pa_dtype dtype, const int32_t* block_tables,
                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                    int32_t max_context_len, float scale, int32_t partition_tokens,
                    void* workspace, size_t workspace_bytes, void* stream) {
  pa_status st = check_cache_shape(num_blocks, block_size, num_kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (dtype_bytes(out_dtype) == 0 || !std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (num_seqs < 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size < max_context_len)
    return PA_ERR_INVALID_ARG;
  Plan pl;
  st = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, dtype, max_context_len,
                 partition_tokens, &pl);
  if (st != PA_OK) return st;
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < pl.ws_total || !aligned16(workspace))
    return PA_ERR_WORKSPACE;
  int ctas = 0;
  st = prepare_kernel(plan_kernel(pl), plan_threads(pl), pl.smem, &ctas);
  if (st != PA_OK) return st;
  const int64_t max_items = static_cast<int64_t>(num_seqs) * (num_kv_heads / pl.kh) * pl.max_parts;
  if (ctas > max_items) ctas = static_cast<int>(max_items);

  DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.num_blocks = num_blocks;
  p.block_size = block_size;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.max_context_len = max_context_len;
  p.part_tokens = pl.part_tokens;
  p.max_parts = pl.max_parts;
  p.out_bf16 = out_dtype == PA_DTYPE_BF16 ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.stages = pl.stages;
  p.stages_v = pl.stages_v;
  p.tbl_stride = pl.tbl_stride;
  p.off_lens = pl.off_lens;
  p.off_q = pl.off_q;
  p.off_p = pl.off_p;
  p.off_small = pl.off_small;
  p.off_sc = pl.off_sc;
  p.off_red = pl.off_red;
  p.off_tbl = pl.off_tbl;
  p.off_prefix = pl.off_prefix;
  p.off_bar = pl.off_bar;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  p.ws_err = reinterpret_cast<int32_t*>(ws);
  p.ws_counters = reinterpret_cast<int32_t*>(ws + pl.ws_counters);
  p.ws_ml = reinterpret_cast<float*>(ws + pl.ws_ml);
  p.ws_o = reinterpret_cast<float*>(ws + pl.ws_o);
  p.test_stall_ns = g_test_stall_ns.load(std::memory_order_relaxed);

  cudaError_t e;
  if (pl.umma) {
    // TMA tensor maps over the K and V pools (one box per block, at most 128
    // rows, in 8-row groups) and over the queries (one box per GQA group and
    // 64-dim half)
    const int64_t cache_rows = static_cast<int64_t>(num_blocks) * num_kv_heads * block_size;
    const int64_t q_rows = static_cast<int64_t>(num_seqs) * num_q_heads;
    if (cache_rows >= (int64_t(1) << 31) || q_rows >= (int64_t(1) << 31)) return PA_ERR_UNSUPPORTED;
    CUtensorMap tmk, tmv, tmq;
    // a box: one block's tokens of the item's kv heads (two heads: a whole
    // block of both, contiguous in the pool), at most 128 rows
    const uint32_t box_rows = static_cast<uint32_t>(
        pl.kh == 2 ? 2 * block_size : (block_size < 128 ? block_size : 128));
    if (!encode_kv_groups(&tmk, k_cache, static_cast<uint64_t>(cache_rows), box_rows) ||
        !encode_kv_groups(&tmv, v_cache, static_cast<uint64_t>(cache_rows), box_rows) ||
        !encode_rows_128(&tmq, q, static_cast<uint64_t>(q_rows), static_cast<uint32_t>(pl.group * pl.kh)))
      return PA_ERR_CUDA;
    void* args[] = {&p, &tmk, &tmv, &tmq};
    // programmatic serialisation: the kernel's set-up may overlap the tail of
    // the previous kernel on the stream (the append signals it early); the
    // kernel waits for that kernel's completion before reading any input
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(kUmmaThreadsHost);
    cfg.dynamicSmemBytes = static_cast<size_t>(pl.smem);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelExC(&cfg, plan_kernel(pl), args);
  } else {
    void* args[] = {&p};
    e = cudaLaunchKernel(pl.info.fn, dim3(static_cast<unsigned>(ctas)), dim3(pa::kDecodeThreads),
                         args, static_cast<size_t>(pl.smem), static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_set_decode_kv_per_item(int32_t kv_per_item) {
  if (kv_per_item < 0 || kv_per_item > 2) return PA_ERR_INVALID_ARG;
  g_kv_per_item.store(kv_per_item, std::memory_order_relaxed);
  return PA_OK;
}

void pa_test_stall_decode(uint64_t ns) {
  g_test_stall_ns.store(ns < pa::kWaitLimitNs ? ns : pa::kWaitLimitNs, std::memory_order_relaxed);
}

pa_status pa_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace) return PA_ERR_INVALID_ARG;
  if (workspace_bytes == 0) return PA_OK;
  return cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

pa_status pa_workspace_error(void* workspace, void* stream, int32_t* device_status) {
  if (!workspace || !device_status) return PA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(v), s) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  *device_status = v;
  return PA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Paged decode for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: code that runs inside
// another runtime whose memory pool already owns the device memory (a stray
// allocation would fail or fragment that pool), plugin hooks that may only
// use the buffers they are handed, and latency-critical loops where the
// implicit device synchronisation of cudaMalloc/cudaFree is not acceptable.
// For them pa_decode_no_alloc runs the same decode kernel with its scratch in
// the file-scope device array below instead of a caller workspace.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};

}  // namespace

namespace {

// Device address of the scratch array on the current device, looked up once
// per device with that device current (the host-side symbol is only a
// stand-in, not a device address).
pa_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_no_alloc(void* out, pa_dtype out_dtype, const void* q,
                                        int32_t num_seqs, int32_t num_q_heads,
                                        const void* k_cache, const void* v_cache,
                                        int32_t num_blocks, int32_t block_size,
                                        int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* context_lens, int32_t max_context_len,
                                        float scale, int32_t partition_tokens, void* stream) {
  void* scratch = nullptr;
  pa_status st = noalloc_scratch(&scratch);
  if (st != PA_OK) return st;
  // Plan; with automatic partitions, enlarge them until the scratch fits.  A
  // plan that fails while partitions are being enlarged (partitions past the
  // planner's limit, or shared memory for them) means the scratch is too small
  // for this batch.
  Plan pl;
  int32_t pt = partition_tokens;
  st = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, dtype,
                 max_context_len, pt, &pl);
  if (st != PA_OK) return st;
  while (pl.ws_total > kNoAllocScratchBytes) {
    if (partition_tokens > 0 || pl.max_parts == 1 || pl.part_tokens > (1 << 29))
      return PA_ERR_WORKSPACE;
    pt = pl.part_tokens * 2;
    if (make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, dtype,
                  max_context_len, pt, &pl) != PA_OK)
      return PA_ERR_WORKSPACE;
  }
  if (num_seqs == 0) return PA_OK;
  // The array keeps the previous call's contents: zero the error word and the
  // per-(sequence, kv head) counters, which must start at zero.
  if (cudaMemsetAsync(scratch, 0, pl.ws_ml, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  return pa_decode(out, out_dtype, q, num_seqs, num_q_heads, k_cache, v_cache, num_blocks,
                   block_size, num_kv_heads, head_dim, dtype, block_tables, max_blocks_per_seq,
                   context_lens, max_context_len, scale, pt, scratch, kNoAllocScratchBytes, stream);
}

extern "C" pa_status pa_decode_no_alloc_error(void* stream, int32_t* device_status) {
  if (!device_status) return PA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const pa_status st = noalloc_scratch(&scratch);
  if (st != PA_OK) return st;
  return pa_workspace_error(scratch, stream, device_status);
}
