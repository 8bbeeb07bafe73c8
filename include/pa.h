/*
 * pa.h -- C ABI of the GB300 paged KV cache library (libpa_gb300.so).
 *
 * The operations follow the three pages on PagedAttention, cited by title
 * and section:
 *   [vLLM2] "vLLM internals (2) - why PagedAttention splits the KV cache into
 *           pages" (youngju.dev): block table, block size, sharing.
 *   [PA]    "PagedAttention" (icarus.shaojiemike.top): "Block Table 如何工作",
 *           "KV Cache 为什么难管理", "支持块级共享", "不改变模型精度".
 *   [KV02]  "LLM KV cache 02 - serving engine KV" (ttlab.hopto.org), section 2:
 *           blocks, block table, sharing, copy-on-write.
 *
 * Conventions shared by every call:
 *   - KV cache layout (the pages name none; this library fixes it): k_cache
 *     and v_cache are each a row-major array [num_blocks][num_kv_heads]
 *     [block_size][head_dim] of `dtype`.  One (block, kv head) tile of K is
 *     block_size*head_dim contiguous elements; one whole block across kv heads
 *     is contiguous too.  Both base pointers must be 16-byte aligned.
 *   - Every pointer named "device" is a CUDA device pointer owned by the
 *     caller; the library never allocates, frees or keeps device memory,
 *     except the fixed scratch array of pa_decode_no_alloc.
 *     "host" pointers are read or written before the call returns.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Device
 *     work is enqueued asynchronously on it; the call does not synchronise.
 *   - Argument errors are detected on the host and returned before anything is
 *     enqueued.  A launch failure returns PA_ERR_CUDA.  No call throws,
 *     prints, exits or traps.
 *   - Supported: dtype F32 or BF16; head_dim 64, 128 or 256; block_size a
 *     power of two from 1 to 256; num_q_heads / num_kv_heads in {1,2,4,8}.
 */
#ifndef PA_GB300_H
#define PA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,   /* a size, pointer or precondition is wrong       */
  PA_ERR_UNSUPPORTED = 2,   /* valid but outside the supported shapes          */
  PA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed            */
  PA_ERR_OOM = 4,           /* allocator: no free block (state unchanged)      */
  PA_ERR_WORKSPACE = 5,     /* workspace missing or smaller than required      */
  PA_ERR_DEVICE_TIMEOUT = 6 /* a bounded device wait gave up (see pa_decode)   */
} pa_status;

typedef enum pa_dtype {
  PA_DTYPE_F32 = 0,
  PA_DTYPE_BF16 = 1
} pa_dtype;

/* Human-readable name of a status code (static string). */
const char* pa_status_string(pa_status status);

/* Library version string, e.g. "pa_gb300 1.0 sm_103a". */
const char* pa_version(void);

/* ------------------------------------------------------------------------
 * KV append -- [PA] "Block Table 如何工作": a generating sequence writes the new
 * token's K/V into the current block; [KV02] section 2: a new block is taken
 * when the current one is full.  Slot = physical_block * block_size + offset.
 *
 * For t < num_tokens with s = slot_mapping[t] >= 0, writes
 *   k_cache[s / block_size][h][s % block_size][:] = key[t][h][:]
 *   v_cache[...same...]                             = value[t][h][:]
 * for every kv head h.  Negative slots (padding) are skipped; slots >=
 * num_blocks*block_size are skipped too (never written; the slots are in
 * device memory, so they are not checked on the host, and
 * pa_reshape_and_cache_checked below reports them).
 *
 *   key, value    device, [num_tokens][num_kv_heads][head_dim] of dtype
 *   slot_mapping  device, int64 [num_tokens]
 *   k_cache/v_cache device, layout above
 * Two tokens mapped to the same slot in one call race (last writer wins).
 * num_tokens == 0 is a no-op.
 * ---------------------------------------------------------------------- */
pa_status pa_reshape_and_cache(const void* key, const void* value, int32_t num_tokens,
                               const int64_t* slot_mapping,
                               void* k_cache, void* v_cache,
                               int32_t num_blocks, int32_t block_size,
                               int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype,
                               void* stream);

/* ------------------------------------------------------------------------
 * Copy-on-write block copy -- [PA] "支持块级共享"; [KV02] section 2: a
 * shared block is copied to a fresh one only when a branch has to write
 * different content into it.
 *
 * For each pair j: k_cache[dst_j] = k_cache[src_j] and v_cache[dst_j] =
 * v_cache[src_j] (all kv heads, all block_size tokens), where
 * block_pairs[2j] = src_j and block_pairs[2j+1] = dst_j.
 *   block_pairs   device, int64 [num_pairs][2]
 * Pairs are valid when every block is in [0, num_blocks), the destinations
 * are distinct and none is also a source in the same call (copy-on-write
 * pairs always are); then the result equals copying from the state before
 * the call.  The pairs live in device memory, so this call does not read or
 * check them on the host: a pair naming a block outside the pool is skipped,
 * and overlapping pairs give an undefined result for the blocks involved.
 * pa_copy_blocks_checked reports invalid pairs instead.  num_pairs == 0 is
 * a no-op.
 * ---------------------------------------------------------------------- */
pa_status pa_copy_blocks(void* k_cache, void* v_cache,
                         int32_t num_blocks, int32_t block_size,
                         int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype,
                         const int64_t* block_pairs, int32_t num_pairs,
                         void* stream);

/* ------------------------------------------------------------------------
 * Checked append and copy (an opt-in validation mode for debugging) --
 * [PA] "Block Table 如何工作": a slot is physical_block * block_size +
 * offset, so a slot at or past num_blocks * block_size names no block of the
 * pool; [PA] "支持块级共享": a copy-on-write copies a shared block to a fresh
 * one, so its destinations are new blocks, distinct and never sources.
 *
 * Same arguments and result as pa_reshape_and_cache / pa_copy_blocks, plus
 *   status   device int32, caller-zeroed (required, 4-byte aligned).  After
 *            the call's work completes (stream order) it holds
 *            PA_ERR_INVALID_ARG if anything was invalid, else it is unchanged.
 * pa_reshape_and_cache_checked: a token whose slot is >= num_blocks *
 *   block_size sets *status and is not written; every other token is
 *   written as by pa_reshape_and_cache (negative slots are padding, skipped).
 * pa_copy_blocks_checked: first validates every pair (a block outside
 *   [0, num_blocks), a destination named twice, or a destination that is
 *   also a source, itself included, sets *status), then copies only if
 *   *status is still zero: on an invalid pair set no block is copied.  A
 *   status left non-zero by an earlier call suppresses the copy too.  Two
 *   launches on stream; the validation makes num_pairs^2 comparisons.
 * ---------------------------------------------------------------------- */
pa_status pa_reshape_and_cache_checked(const void* key, const void* value, int32_t num_tokens,
                                       const int64_t* slot_mapping,
                                       void* k_cache, void* v_cache,
                                       int32_t num_blocks, int32_t block_size,
                                       int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype,
                                       int32_t* status, void* stream);

pa_status pa_copy_blocks_checked(void* k_cache, void* v_cache,
                                 int32_t num_blocks, int32_t block_size,
                                 int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype,
                                 const int64_t* block_pairs, int32_t num_pairs,
                                 int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * Multi-layer KV append and block copy -- [PA] "KV Cache 为什么难管理": a
 * token's cache costs M_token = 2 * L * H_kv * d elements, K and V of every
 * one of the model's L layers, so a step appends a token in every layer and
 * a copy-on-write copies the block in every layer ([PA] "支持块级共享").
 *
 * One pool holds all layers: layer l of the K cache starts at
 * k_cache + l * cache_layer_stride elements (likewise V), and layer l of the
 * step's key/value input at key + l * kv_layer_stride elements.  Per layer
 * the operation and layouts are those of pa_reshape_and_cache /
 * pa_copy_blocks, applied to layers 0 .. num_layers-1 in one launch.
 *   kv_layer_stride     elements between layers of key/value, >=
 *                       num_tokens*num_kv_heads*head_dim
 *   cache_layer_stride  elements between cache layers, >=
 *                       num_blocks*num_kv_heads*block_size*head_dim
 * Both strides times the element size must be multiples of 16 bytes (the
 * strides are ignored when num_layers == 1).  1 <= num_layers <= 32767,
 * else PA_ERR_INVALID_ARG.  The single-layer calls above are these calls
 * with num_layers == 1.
 * ---------------------------------------------------------------------- */
pa_status pa_reshape_and_cache_layers(const void* key, const void* value,
                                      int64_t kv_layer_stride, int32_t num_layers,
                                      int32_t num_tokens, const int64_t* slot_mapping,
                                      void* k_cache, void* v_cache,
                                      int64_t cache_layer_stride,
                                      int32_t num_blocks, int32_t block_size,
                                      int32_t num_kv_heads, int32_t head_dim,
                                      pa_dtype dtype, void* stream);

pa_status pa_copy_blocks_layers(void* k_cache, void* v_cache,
                                int64_t cache_layer_stride, int32_t num_layers,
                                int32_t num_blocks, int32_t block_size,
                                int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype,
                                const int64_t* block_pairs, int32_t num_pairs,
                                void* stream);

/* ------------------------------------------------------------------------
 * Paged decode attention -- [PA] "Block Table 如何工作": the kernel reads the
 * block table to turn logical block numbers into physical block ids, so each
 * sequence sees its K/V in token order; [PA] "不改变模型精度": the result is
 * the attention over the contiguous history.
 *
 * For sequence i < num_seqs, query head h, kv head g = h / (num_q_heads /
 * num_kv_heads) and len = context_lens[i] (the token appended this step
 * included):
 *   K_t = k_cache[block_tables[i*max_blocks_per_seq + t/block_size]][g][t%block_size]
 *   out[i][h][:] = sum_t softmax_t(scale * q[i][h]·K_t) * V_t ,  t < len
 * and out[i][h][:] = 0 when len == 0.  Accumulation is fp32.
 *
 *   out           device, [num_seqs][num_q_heads][head_dim] of out_dtype
 *   q             device, [num_seqs][num_q_heads][head_dim] of dtype
 *   block_tables  device, int32 [num_seqs][max_blocks_per_seq]; entries past
 *                 ceil(len/block_size) are never read; every entry read must
 *                 be in [0, num_blocks)
 *   context_lens  device, int32 [num_seqs]; each in [0, max_context_len]
 *   max_context_len  host bound used for planning (no device sync)
 *   partition_tokens 0 = automatic; else the number of tokens each split-K
 *                 partition covers (rounded up to the plan's granularity)
 *   workspace     device scratch of at least pa_decode_workspace_size(...)
 *                 bytes, 256-byte aligned, ZERO-FILLED before its first use
 *                 (e.g. pa_workspace_init).  Every call leaves its
 *                 bookkeeping words zero again, so one workspace serves any
 *                 number of calls issued in stream order; calls that overlap
 *                 on the GPU must use different workspaces.
 * A long history is split into partitions processed by different CTAs; each
 * writes (max, sum, unnormalised output) to the workspace and the last CTA
 * to finish a (sequence, kv head) merges them by log-sum-exp.
 * If a bounded device wait ever expires, the kernel stops early, the output
 * is undefined, and pa_workspace_error() reports PA_ERR_DEVICE_TIMEOUT.
 * The tensor-core kernel is launched with programmatic stream serialisation:
 * its set-up may overlap the tail of the kernel before it on the stream (the
 * append signals this at its start), and it reads no input before that
 * kernel has completed, so stream order holds as for any launch.
 * ---------------------------------------------------------------------- */
size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t block_size, pa_dtype dtype,
                                int32_t max_context_len, int32_t partition_tokens);

pa_status pa_decode(void* out, pa_dtype out_dtype,
                    const void* q, int32_t num_seqs, int32_t num_q_heads,
                    const void* k_cache, const void* v_cache,
                    int32_t num_blocks, int32_t block_size,
                    int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype,
                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* context_lens, int32_t max_context_len,
                    float scale, int32_t partition_tokens,
                    void* workspace, size_t workspace_bytes,
                    void* stream);

/* pa_decode without a caller workspace, for callers that cannot allocate
 * device memory: code running inside another runtime whose memory pool owns
 * the device memory, plugin hooks that may only use the buffers they are
 * handed, and latency-critical loops that cannot afford the device
 * synchronisation cudaMalloc/cudaFree may imply.  The pages have no
 * counterpart for this call; it exists only for such callers.
 *
 * Arguments and result as pa_decode, minus the workspace.  The scratch is a
 * fixed 32 MiB array in the library's device memory, held by every GPU that
 * loads the library until the process exits.  With partition_tokens == 0 the
 * partitions are enlarged until the scratch suffices; PA_ERR_WORKSPACE if it
 * cannot (a fixed partition_tokens whose workspace exceeds 32 MiB, or more
 * than about 8 million (sequence, kv head) pairs).  The call allocates
 * nothing.  Its first call on a device looks up the array's device address
 * (once per device, with that device current); make that first call before
 * any stream capture.  Every call shares the one array and zeroes its
 * bookkeeping words first, so calls that overlap on the GPU (other streams,
 * other host threads) race and corrupt each other: issue them in one stream
 * order.  Device-side status (a table entry outside the pool, a length above
 * max_context_len, a wait that timed out) goes to the array's error word,
 * which pa_decode_no_alloc_error reads. */
pa_status pa_decode_no_alloc(void* out, pa_dtype out_dtype,
                             const void* q, int32_t num_seqs, int32_t num_q_heads,
                             const void* k_cache, const void* v_cache,
                             int32_t num_blocks, int32_t block_size,
                             int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* context_lens, int32_t max_context_len,
                             float scale, int32_t partition_tokens, void* stream);

/* Device status of the pa_decode_no_alloc calls on the current device since
 * the last call (each call clears the word first, so this reports the last
 * one): synchronises `stream` (the stream the decode ran on), reads the
 * scratch array's error word into *device_status (PA_OK,
 * PA_ERR_INVALID_ARG or PA_ERR_DEVICE_TIMEOUT, as pa_workspace_error) and
 * clears it.  Like pa_decode_no_alloc, it allocates nothing. */
pa_status pa_decode_no_alloc_error(void* stream, int32_t* device_status);

/* Work-item shape of the tensor-core decode (bf16, head_dim 128), a
 * process-wide planning setting: 0 = automatic (the default), 1 = one kv head
 * per work item, 2 = two kv heads per item where the shape allows it (GQA
 * group <= 4, an even kv-head count, blocks of 8..64 tokens; otherwise one).
 * Two heads per item read each block of both heads with one tensor copy and
 * halve the item count; the automatic choice takes them with about five
 * two-head items per SM or more.  The result is the same either way up to
 * fp32 rounding order.  The workspace size depends on the setting: size and
 * decode under the same setting.  PA_ERR_INVALID_ARG for other values. */
pa_status pa_set_decode_kv_per_item(int32_t kv_per_item);

/* Partition size and CTA count pa_decode would use (host only; either out
 * pointer may be NULL). */
pa_status pa_decode_plan(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, pa_dtype dtype,
                         int32_t max_context_len, int32_t partition_tokens,
                         int32_t* partition_tokens_out, int32_t* num_ctas_out);

/* Testing hook for the timeout path, not for production use.  With ns > 0,
 * every pa_decode launch of the tensor-core kernel (bf16, head_dim 128) made
 * after this call in this process has its compute warps first wait for an
 * event that never comes, giving up after ns nanoseconds (at most 2 s); 0
 * turns the hook off.  A CTA whose wait gives up raises its stop word: every
 * role stops, copies and tensor-core work already issued are waited for,
 * tensor memory is freed, the output is left undefined, and
 * PA_ERR_DEVICE_TIMEOUT reaches the host through pa_workspace_error.  The
 * workspace must be zeroed again (pa_workspace_init) before its next use.
 * The same stop path serves any real wait that runs out its 2 s limit. */
void pa_test_stall_decode(uint64_t ns);

/* Zero a decode workspace (enqueued on `stream`). */
pa_status pa_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Synchronises `stream`, then reads the workspace's device error word into
 * *device_status (PA_OK; PA_ERR_INVALID_ARG for a table entry outside the
 * pool or a context length outside [0, max_context_len]; or
 * PA_ERR_DEVICE_TIMEOUT) and clears it. */
pa_status pa_workspace_error(void* workspace, void* stream, int32_t* device_status);

/* ------------------------------------------------------------------------
 * Shared-prefix decode -- [PA] "支持块级共享", [KV02] section 2: sequences
 * that share a prefix (a common prompt, parallel samples, beams) point at the
 * same physical blocks; this decode reads each shared block once per group
 * instead of once per sequence.  The result is that of pa_decode.
 *
 * The batch's sequences form groups of consecutive indices:
 * group j is [group_start[j], group_start[j+1]).  The first prefix_len[j]
 * tokens of every member are the same blocks: the first prefix_len[j] /
 * block_size entries of every member's table are equal.  A sequence that
 * shares nothing is a group of its own with prefix 0.  The call runs, in one
 * launch,
 *  (1) every group's queries (members x heads of a kv head, as the rows of
 *      dense 128-row tiles) against its prefix, split into partitions, and
 *  (2) every member's own tokens [prefix_len, context_len);
 * then, in a second launch that may start as the first drains,
 *  (3) a log-sum-exp merge of the partial results into out.
 *   q, out           device, [num_seqs][num_q_heads][128]; q bf16
 *   group_start      device, int32 [num_groups + 1], group_start[0] == 0,
 *                    non-decreasing, group_start[num_groups] == num_seqs
 *   prefix_len       device, int32 [num_groups], multiples of block_size,
 *                    <= every member's context length
 *   max_group_size   host, >= every group's size
 *   max_prefix_len   host, >= every prefix_len
 *   workspace        device scratch of
 *                    pa_decode_shared_prefix_workspace_size(...) bytes
 *                    (no zeroing needed)
 *   status           device int32, caller-zeroed, or NULL: PA_ERR_INVALID_ARG
 *                    for inconsistent groups, prefixes or lengths,
 *                    PA_ERR_DEVICE_TIMEOUT if a bounded wait expired
 * Supported: bf16 K/V and q, head_dim 128, block_size 8..256, num_q_heads /
 * num_kv_heads in {1, 2, 4, 8, 16}; PA_ERR_UNSUPPORTED otherwise;
 * PA_ERR_WORKSPACE if the workspace is too small.  Two launches on stream.
 * ---------------------------------------------------------------------- */
size_t    pa_decode_shared_prefix_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                                 int32_t num_kv_heads, int32_t num_groups,
                                                 int32_t max_group_size, int32_t max_prefix_len);
pa_status pa_decode_shared_prefix(void* out, pa_dtype out_dtype, const void* q,
                                  int32_t num_seqs, int32_t num_q_heads,
                                  const void* k_cache, const void* v_cache, int32_t num_blocks,
                                  int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                  pa_dtype dtype, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* context_lens,
                                  int32_t max_context_len, const int32_t* group_start,
                                  const int32_t* prefix_len, int32_t num_groups,
                                  int32_t max_group_size, int32_t max_prefix_len, float scale,
                                  int32_t* status, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* ------------------------------------------------------------------------
 * Paged prefill attention -- [PA] "KV Cache 为什么难管理": the prefill phase
 * processes a prompt's tokens together; [PA] "Block Table 如何工作": every
 * token reads its sequence's K/V through the block table.  Chunked prefill
 * (a prompt split over several calls) is the same call with a later start.
 *
 * Sequence i's chunk is q[cu_q[i] .. cu_q[i+1]) (tokens); its token j sits
 * at position p = q_start[i] + j of the sequence and attends causally:
 *   K_t = k_cache[block_tables[i*max_blocks_per_seq + t/block_size]][g][t%block_size]
 *   out[cu_q[i]+j][h][:] = sum_{t <= p} softmax_t(scale * q[cu_q[i]+j][h]·K_t) * V_t
 * with g = h / (num_q_heads / num_kv_heads).  The chunk's own K/V must be in
 * the cache already (pa_reshape_and_cache first).  Accumulation is fp32.
 *
 *   out          device, [num_tokens][num_q_heads][128] of out_dtype
 *   q            device, [num_tokens][num_q_heads][128] bf16
 *   cu_q         device, int32 [num_seqs + 1], non-decreasing, cu_q[0] >= 0,
 *                cu_q[num_seqs] <= num_tokens
 *   q_start      device, int32 [num_seqs]
 *   max_q_len    host, >= every chunk length (sizes the launch)
 *   status       device int32, caller-zeroed, or NULL: receives
 *                PA_ERR_INVALID_ARG for a chunk outside q or beyond the table,
 *                or for a table entry outside the pool (never read: block 0
 *                is read instead), and PA_ERR_DEVICE_TIMEOUT if a bounded wait
 *                expired.
 * Supported: bf16 K/V and q, head_dim 128, block_size 8..256 (power of two),
 * num_q_heads / num_kv_heads in {1, 2, 4, 8, 16}; PA_ERR_UNSUPPORTED
 * otherwise.  num_tokens, num_seqs or max_q_len == 0 is a no-op.
 * ---------------------------------------------------------------------- */
pa_status pa_prefill(void* out, pa_dtype out_dtype, const void* q, int32_t num_tokens,
                     const int32_t* cu_q, const int32_t* q_start, int32_t num_seqs,
                     int32_t max_q_len, int32_t num_q_heads,
                     const void* k_cache, const void* v_cache, int32_t num_blocks,
                     int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                     pa_dtype dtype, const int32_t* block_tables, int32_t max_blocks_per_seq,
                     float scale, int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * Host block allocator -- [vLLM2] block-table section and [KV02] section 2:
 * fixed-size blocks handed out on demand from anywhere in the pool; [PA]
 * "Block Table 如何工作": full blocks trigger a new allocation, freed blocks
 * nobody references return to the pool; [PA] "支持块级共享": reference
 * counts, fork and copy-on-write.  Host memory only; not thread-safe (one
 * caller at a time per handle).
 *
 * Policy: the free list starts in `free_order` (a permutation of
 * 0..num_blocks-1; NULL = identity); allocation takes the front; a block
 * whose count drops to 0 goes to the back.  Sequence ids count up from 0
 * and are never reused.
 * ---------------------------------------------------------------------- */
typedef struct pa_allocator pa_allocator;

pa_status pa_alloc_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order,
                          pa_allocator** out);
void      pa_alloc_destroy(pa_allocator* a);
int32_t   pa_alloc_num_blocks(const pa_allocator* a);
int32_t   pa_alloc_block_size(const pa_allocator* a);
int32_t   pa_alloc_num_free(const pa_allocator* a);
/* Reference count of `block` (-1 if out of range). */
int32_t   pa_alloc_refcount(const pa_allocator* a, int32_t block);
/* Take one block (count 1) -> *block; PA_ERR_OOM if none is free. */
pa_status pa_alloc_allocate(pa_allocator* a, int32_t* block);
pa_status pa_alloc_incref(pa_allocator* a, int32_t block);
/* Drop one reference; at zero the block goes to the back of the free list.
 * PA_ERR_INVALID_ARG if the block is already free. */
pa_status pa_alloc_decref(pa_allocator* a, int32_t block);

/* New empty sequence -> *seq. */
pa_status pa_alloc_seq_create(pa_allocator* a, int32_t* seq);
/* New sequence sharing every block of `parent` (each count + 1). */
pa_status pa_alloc_fork(pa_allocator* a, int32_t parent, int32_t* child);
/* Reserve the slot of the next token of `seq`.  With pos = current length:
 * pos % block_size == 0 -> a fresh block is appended to the table; else if
 * the last block is shared (count > 1) it is replaced by a new block and
 * (old, new) is reported in *cow_src, *cow_dst (both -1 otherwise).
 * *slot = table[pos/bs]*bs + pos%bs.  PA_ERR_OOM leaves the state unchanged. */
pa_status pa_alloc_append_slot(pa_allocator* a, int32_t seq, int64_t* slot,
                               int32_t* cow_src, int32_t* cow_dst);
/* One append_slot per entry of seqs[0..n), in order.  slots[j] receives
 * sequence seqs[j]'s slot; copy pairs are appended to cow_pairs ([n][2],
 * int64) and counted in *num_cow.  Stops at the first failure; *num_done
 * tells how many appends took effect. */
pa_status pa_alloc_append_slots(pa_allocator* a, const int32_t* seqs, int32_t n,
                                int64_t* slots, int64_t* cow_pairs, int32_t* num_cow,
                                int32_t* num_done);
/* n successive append_slot calls on an unshared sequence (bulk prompt
 * fill); slots[0..n) receive the slots.  PA_ERR_INVALID_ARG if a copy would
 * be needed.  On PA_ERR_OOM nothing changes. */
pa_status pa_alloc_append_tokens(pa_allocator* a, int32_t seq, int32_t n, int64_t* slots);
/* Release every block of `seq` in table order (last block first when
 * prefix caching is on); the id becomes invalid. */
pa_status pa_alloc_free_seq(pa_allocator* a, int32_t seq);
/* Length of `seq` (-1 if it is not live). */
int32_t   pa_alloc_seq_len(const pa_allocator* a, int32_t seq);
/* Number of sequences currently live. */
int32_t   pa_alloc_num_seqs(const pa_allocator* a);
/* Copy the block table of `seq` into out[0..cap); *n = its length. */
pa_status pa_alloc_block_table(const pa_allocator* a, int32_t seq, int32_t* out, int32_t cap,
                               int32_t* n);
/* Dense tables for a batch: tables[j*max_blocks + k] = block k of seqs[j]
 * (pad_value past its end), lens[j] = its length.  PA_ERR_INVALID_ARG if a
 * table does not fit in max_blocks. */
pa_status pa_alloc_export_tables(const pa_allocator* a, const int32_t* seqs, int32_t n,
                                 int32_t* tables, int32_t max_blocks, int32_t* lens,
                                 int32_t pad_value);
/* Copy the free list, front first, into out[0..cap); *n = its length. */
pa_status pa_alloc_free_list(const pa_allocator* a, int32_t* out, int32_t cap, int32_t* n);
/* Copy the live sequence ids, ascending, into out[0..cap); *n = count. */
pa_status pa_alloc_live_seqs(const pa_allocator* a, int32_t* out, int32_t cap, int32_t* n);

/* ------------------------------------------------------------------------
 * Automatic prefix caching -- [KV02] section 4 "프리픽스 캐시": requests that
 * share a leading part of their prompt share its K/V blocks, so that part
 * needs no prefill.
 *  - A full block's key is SHA-256(previous block's key, or 32 zero bytes for
 *    the first block || the block's block_size token ids as little-endian
 *    int32 || the request's extra bytes).  The extra bytes are the caller's
 *    composition of what else separates requests (cache salt, adapter, input
 *    hashes).  A key therefore stands for the whole prefix up to its block.
 *  - Only full blocks are keyed; a key maps to the first block that held it.
 *  - A block whose count drops to zero keeps its key and contents on the
 *    free list.  Allocation takes the front of the list and drops that
 *    block's key: least recently freed cached blocks go first, and a
 *    released sequence queues its last block first, so tails are evicted
 *    before the prefixes they extend.
 *  - A cache hit takes its block off the free list.
 * The decode, append and copy calls are unchanged: a hit is a block shared
 * through the tables, like a fork.
 * ---------------------------------------------------------------------- */
/* Turn prefix caching on; only while no sequence exists and every block is
 * free (PA_ERR_INVALID_ARG otherwise).  No effect if already on. */
pa_status pa_alloc_enable_prefix_cache(pa_allocator* a);
/* New tracked sequence holding token_ids[0..num_tokens).  Its leading full
 * blocks are taken from the cache while their keys hit (up to the first
 * miss).  The rest get fresh blocks, and every full block is keyed.
 * slots[t] receives every token's slot; *cached_tokens receives the number
 * of leading tokens whose K/V are already in the cache (a multiple of
 * block_size), so the caller writes K/V only for tokens >= *cached_tokens.
 * extra: extra_bytes bytes (may be NULL when 0).  On PA_ERR_OOM nothing
 * changes; PA_ERR_INVALID_ARG if prefix caching is off. */
pa_status pa_alloc_seq_create_prefix(pa_allocator* a, const int32_t* token_ids,
                                     int32_t num_tokens, const void* extra, int32_t extra_bytes,
                                     int32_t* seq, int32_t* cached_tokens, int64_t* slots);
/* pa_alloc_append_tokens with the tokens' ids: a tracked sequence keys the
 * blocks they complete.  (Appends without ids, pa_alloc_append_slot(s) and
 * pa_alloc_append_tokens, end the keying of that sequence.) */
pa_status pa_alloc_append_token_ids(pa_allocator* a, int32_t seq, const int32_t* token_ids,
                                    int32_t n, int64_t* slots);
/* Number of keyed blocks (in use or on the free list); -1 for NULL. */
int32_t   pa_alloc_num_cached(const pa_allocator* a);
/* Key of `block` -> key[32]; PA_ERR_INVALID_ARG if it holds none. */
pa_status pa_alloc_block_key(const pa_allocator* a, int32_t block, uint8_t key[32]);

/* SHA-256 (FIPS 180-4) of data[0..num_bytes) -> digest[32]; the block-key
 * hash above, exported for checking. */
pa_status pa_sha256(const void* data, size_t num_bytes, uint8_t digest[32]);

#ifdef __cplusplus
}
#endif
#endif /* PA_GB300_H */
