// Internal interface between the C ABI shim and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace pa {

constexpr int kConsumerWarps = 4;
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kDecodeThreads = 32 + kConsumerThreads;  // warp 0 streams, warps 1-4 compute
constexpr int kStageBytes = 8192;                      // K or V rows per ring stage
constexpr int kStages = 6;                             // ring depth
constexpr uint64_t kWaitLimitNs = 2000000000ull;       // bounded device waits: 2 s

// Device error codes written to the workspace header (match pa_status).
constexpr int kDevErrInvalidArg = 1;
constexpr int kDevErrTimeout = 6;

struct DecodeParams {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t num_blocks;
  int32_t block_size;
  int32_t max_blocks_per_seq;
  int32_t max_context_len;
  int32_t part_tokens;  // tokens per split-K partition
  int32_t max_parts;    // partial slots per (sequence, kv head) in the workspace
  int32_t out_bf16;     // 1: bf16 output, 0: fp32
  float scale_log2;     // softmax scale * log2(e)
  // dynamic shared memory carve-up (byte offsets)
  int32_t stages;      // K ring depth of the tensor-core kernel
  int32_t stages_v;    // V ring depth of the tensor-core kernel
  int32_t tbl_stride;  // table-slice entries per compute group (tensor-core kernel)
  int32_t off_lens;
  int32_t off_q;
  int32_t off_p;
  int32_t off_small;
  int32_t off_sc;
  int32_t off_red;
  int32_t off_tbl;
  int32_t off_prefix;
  int32_t off_bar;
  // workspace carve-up
  int32_t* ws_err;
  int32_t* ws_counters;
  float* ws_ml;
  float* ws_o;
  // timeout-path test hook of the tensor-core kernel (0 = off): its compute
  // warps first wait this long for an event that never comes, then give up
  uint64_t test_stall_ns;
};

// SMs of the current device (152, the GB300's, when none can be queried).
int64_t device_sm_count();

// Per (dtype, head_dim, group) kernel entry: shared memory need and launch.
struct DecodeKernelInfo {
  const void* fn;
  int ring_bytes;   // kStages * stage allocation
  int tokens_per_stage;
  int q_bytes;
};

// Returns false if the combination is not compiled.
bool decode_kernel_info(int dtype_bf16, int head_dim, int group, DecodeKernelInfo* info);

// Tensor-core kernel (bf16, head_dim 128) for a GQA group with 1 or 2 kv
// heads per work item, or nullptr.
const void* decode_umma_fn(int group, int kv_per_item);

// Paged prefill (tensor cores, bf16, head_dim 128, block size >= 8).
struct PrefillParams {
  void* out;
  int32_t out_bf16;
  const int32_t* cu_q;     // [num_seqs + 1] chunk offsets into q / out (tokens)
  const int32_t* q_start;  // [num_seqs] position of each chunk's first token
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_tokens;
  int32_t tiles_per_seq;   // ceil(max chunk length / tokens per tile)
  int32_t pair_block;      // mode 0: (sequence, kv head) pairs per block of the item order
  int32_t o_tma;           // a warp's rows of a full tile leave by TMA stores: 1 bf16, 2 fp32 rows
  int32_t pack2;           // modes 2-3: two members per own-token item (block size <= 64)
  float scale_log2;
  int32_t* status;         // device error word (may be null)
  // shared-prefix decode (mode 1: the groups' prefixes, mode 2: the members'
  // own tokens past them, mode 3: both in one launch); mode 0 is causal prefill
  int32_t mode;
  const int32_t* group_start;   // [num_groups + 1] member ranges of the batch
  const int32_t* prefix_len;    // [num_groups] shared tokens (whole blocks)
  const int32_t* context_lens;  // [num_seqs]
  int32_t num_groups;
  int32_t max_context_len;
  int32_t part_tokens;          // keys per prefix partition (multiple of 128)
  int32_t num_parts;            // prefix partitions per group (max); the suffix is slot num_parts
  float* part_ml;               // [num_parts + 1][num_seqs * num_q_heads][2]: max (log2), sum
  float* part_o;                // [num_parts + 1][num_seqs * num_q_heads][128]: unnormalised O
};
const void* prefill_umma_fn(int group, bool fp32_rows = false);
int prefill_umma_smem_bytes();
cudaError_t launch_cascade_merge(const PrefillParams& p, cudaStream_t stream);

// Cache ops over num_layers layers of one pool (layer strides in bytes,
// multiples of 16); one layer is num_layers == 1.  status == nullptr: the
// unchecked calls; else the checked mode (see cache_ops.cu).
cudaError_t launch_reshape_and_cache(const void* key, const void* value, int64_t kv_layer_bytes,
                                     int32_t num_layers, int32_t num_tokens,
                                     const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                     int64_t cache_layer_bytes, int32_t num_blocks,
                                     int32_t block_size, int32_t num_kv_heads, int32_t row_bytes,
                                     int32_t* status, cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, int64_t cache_layer_bytes,
                               int32_t num_layers, int32_t num_blocks, int64_t block_bytes,
                               const int64_t* pairs, int32_t num_pairs, int32_t* status,
                               cudaStream_t stream);

}  // namespace pa
