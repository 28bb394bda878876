/*
 * pkv.h -- C ABI of the GB300 (sm_103a) paged KV-cache decode library, libpkv.so.
 *
 * What it computes.  A KV cache kept as a pool of fixed-size physical blocks of
 * 16 tokens; each sequence owns a block table mapping its logical block i to a
 * physical block ("Series 03: why the KV cache eats memory, and how
 * PagedAttention pages it", sections 3.1-3.3).  A decode step appends the new
 * token's K and V rows to the cache and then lets the token's query attend over
 * every cached row of its sequence ("KV Cache, the memory notepad of LLM
 * inference", sections 二 and 三):
 *      out[b, h] = sum_j softmax_j(scale * <q[b, h], K_j>) V_j,   j < context_lens[b]
 * where K_j / V_j of KV head g = h / G (G = num_q_heads / num_kv_heads, the GQA
 * group of the same page's section 六) are found through the block table.  An
 * E4M3 (8-bit float) cache stores code = E4M3(fl32(x / scale[g])) with one fp32
 * scale per KV head and dequantises before the arithmetic ("KV cache capacity
 * planning, from the budget to task-level regression", sections 4 and 5).
 *
 * Data layout (all row-major, C order):
 *   k_cache, v_cache   [num_blocks, num_kv_heads, block_size, head_dim]; K and V
 *                      are separate buffers ("What a KV cache is and why it is
 *                      the crux of LLM inference", section 3.1); one
 *                      (block, head) slab of 16 rows is contiguous.
 *   slot               physical row index = block_id * block_size + offset.
 *   block_tables       int32 [batch, max_blocks_per_seq]; entries past
 *                      ceil(context_len / block_size) are never read.
 *   q, out             [batch, num_q_heads, head_dim] in the 16-bit dtype.
 *   k_new, v_new       [num_tokens, num_kv_heads, head_dim].
 *
 * Conventions.
 *   - Ownership: every buffer is allocated and owned by the caller.  Device
 *     pointers must stay valid until the stream work they feed completes.  The
 *     library allocates no device memory and keeps no device state.
 *   - Execution: launches are asynchronous on `stream` (a cudaStream_t passed
 *     as void*; NULL = the legacy default stream).  The returned status only
 *     reports argument validation and launch errors.
 *   - Alignment: every device pointer is 16-byte aligned; head_dim is 64 or 128
 *     and block_size is 16 (anything else returns PKV_ERR_UNSUPPORTED).
 *   - Device-detected errors (a block id outside [0, num_blocks), a slot past
 *     the pool, a context longer than its table or than max_context_len, an
 *     internal wait that timed out) make the kernel skip the access and, when
 *     `err_flag` (a device int32, nullable) is given, store the first error
 *     code there.  No kernel traps.  The caller synchronises and reads it.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,  /* bad pointer, size or shape                      */
  PKV_ERR_UNSUPPORTED = 2,  /* valid but not built: head_dim, group, block size */
  PKV_ERR_NO_BLOCKS = 3,    /* the host block pool has no free block            */
  PKV_ERR_OOB = 4,          /* (device) block id / slot / length out of range   */
  PKV_ERR_CUDA = 5,         /* a CUDA runtime call failed                        */
  PKV_ERR_WORKSPACE = 6,    /* workspace missing or smaller than required        */
  PKV_ERR_TIMEOUT = 7       /* (device) a bounded internal wait expired          */
} pkv_status;

typedef enum { PKV_F16 = 0, PKV_BF16 = 1 } pkv_dtype;

/* Library version (major * 10000 + minor * 100 + patch). */
int pkv_version(void);

/* Static text for a status code. */
const char* pkv_status_string(int status);

/* The CUDA runtime call that made the calling thread's last PKV_ERR_CUDA
 * (name, error name and text); "" when none has failed.  Thread-local. */
const char* pkv_last_error(void);

/* ---------------------------------------------------------------------------
 * Slot mapping.  For token t of sequence b = seq_idx[t] (or b = t when seq_idx
 * is NULL) at logical position p = positions[t] + position_offset:
 *     slot_mapping[t] = block_tables[b][p / block_size] * block_size + p % block_size
 * (the block-table lookup of "Series 03 ...", section 3.1).  p < 0 gives -1 (a
 * padding token).  A table entry outside [0, num_blocks) or p past the table
 * gives -1 and PKV_ERR_OOB in err_flag.  Decode: positions = context_lens with
 * position_offset = -1 (the last position).  All pointers are device memory.
 * ------------------------------------------------------------------------- */
pkv_status pkv_slot_mapping(const int32_t* block_tables, int max_blocks_per_seq, int64_t num_blocks,
                            const int32_t* seq_idx, const int32_t* positions, int32_t position_offset,
                            int64_t num_tokens, int block_size, int64_t* slot_mapping, int32_t* err_flag,
                            void* stream);

/* ---------------------------------------------------------------------------
 * Append ("KV Cache, the memory notepad ...", section 三: each step appends the
 * new token's K/V to the cache).  Copies k_new[t, h, :] to
 * k_cache[s / block_size, h, s % block_size, :] with s = slot_mapping[t], and
 * the same for V; a bit-exact copy.  s < 0 skips the token; s >= num_blocks *
 * block_size is skipped and reported as PKV_ERR_OOB.  dtype is the element type
 * of k_new, v_new and the caches.
 * ------------------------------------------------------------------------- */
pkv_status pkv_kv_append(const void* k_new, const void* v_new, const int64_t* slot_mapping, int64_t num_tokens,
                         void* k_cache, void* v_cache, int64_t num_blocks, int num_kv_heads, int head_dim,
                         int block_size, pkv_dtype dtype, int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * E4M3 append ("KV cache capacity planning ...", section 4: FP8 E4M3 storage
 * with a per-attention-head scale).  Stores
 *     code = E4M3_RN_satfinite(fl32(x) / k_scale[h])
 * (IEEE fp32 division, round to nearest even, magnitudes above 448 clamp to
 * 448) for every element x of k_new (in_dtype) into the uint8 cache, and the
 * same for V with v_scale.  k_scale, v_scale: device float32 [num_kv_heads].
 * Slots as in pkv_kv_append.
 * ------------------------------------------------------------------------- */
pkv_status pkv_kv_append_fp8(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                             int64_t num_tokens, uint8_t* k_cache, uint8_t* v_cache, int64_t num_blocks,
                             const float* k_scale, const float* v_scale, int num_kv_heads, int head_dim,
                             int block_size, pkv_dtype in_dtype, int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * E5M2 append ("KV cache capacity planning ...", section 4: the second FP8
 * format it names, with the wider exponent range and the lower precision; the
 * OCP 8-bit floating point specification of its reference list: bias 15, two
 * mantissa bits, largest finite value 57344).  Stores
 *     code = E5M2_RN_satfinite(fl32(x) / k_scale[h])
 * (IEEE fp32 division, round to nearest even, magnitudes above 57344 --
 * infinities included -- clamp to 57344, NaN stores a NaN code) for every
 * element x of k_new (in_dtype) into the uint8 cache, and the same for V with
 * v_scale.  Arguments, layout and errors as in pkv_kv_append_fp8.
 * ------------------------------------------------------------------------- */
pkv_status pkv_kv_append_e5m2(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                              int64_t num_tokens, uint8_t* k_cache, uint8_t* v_cache, int64_t num_blocks,
                              const float* k_scale, const float* v_scale, int num_kv_heads, int head_dim,
                              int block_size, pkv_dtype in_dtype, int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * Workspace for decode attention, in bytes, on the current CUDA device.  The
 * decode splits the work over the flattened (sequence, KV head, block) space;
 * pieces of a sequence handled by different thread blocks leave fp32 partial
 * results (running max, sum, unnormalised output) that a combine kernel merges
 * by log-sum-exp.  partition_tokens = 0 sizes the balanced split (one equal
 * share per resident thread block); > 0 (a multiple of block_size) sizes a
 * split into fixed partitions of that many tokens of the flattened space, an
 * equal number of consecutive partitions per resident thread block (the
 * partitions of one sequence and KV head that one thread block holds are
 * merged as it streams them, so each pair leaves one partial per thread block
 * it meets).  Returns 0 on invalid arguments or when the device cannot be
 * queried.
 * ------------------------------------------------------------------------- */
size_t pkv_decode_workspace_bytes(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                  int max_blocks_per_seq, int max_context_len, int partition_tokens);

/* ---------------------------------------------------------------------------
 * Paged decode attention, 16-bit cache.  For every sequence b and query head h:
 *     out[b, h] = sum_{j < n} softmax_j(scale * <q[b, h], K_j>) V_j
 * with n = context_lens[b] and K_j = k_cache[block_tables[b][j / 16], h / G,
 * j % 16, :] (V likewise).  Softmax arithmetic is fp32 with the running
 * maximum subtracted; out is rounded to dtype (nearest even).  n = 0 gives
 * out[b, :, :] = 0.  One thread block serves all G query heads of a KV head,
 * so each KV byte is read from HBM once.
 *   q, k_cache, v_cache, out      dtype (F16 / BF16), layouts above.
 *   block_tables, context_lens    device int32.
 *   max_context_len               an upper bound of context_lens (sizes the
 *                                 partition split; longer contexts are clamped
 *                                 and reported as PKV_ERR_OOB).
 *   partition_tokens              0 = balanced split; > 0 see the workspace query.
 *   workspace, workspace_bytes    caller-owned device scratch of at least
 *                                 pkv_decode_workspace_bytes(...); its contents
 *                                 need no initialisation and are overwritten.
 *                                 Two calls running at the same time on the GPU
 *                                 must not share a workspace.
 * Requirements: num_q_heads % num_kv_heads == 0 with G in {1, 2, 4, 8};
 * head_dim in {64, 128}; block_size == 16.
 * ------------------------------------------------------------------------- */
pkv_status pkv_paged_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, const int32_t* context_lens, int batch,
                                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                      int max_blocks_per_seq, int64_t num_blocks, int max_context_len,
                                      float scale, void* out, pkv_dtype dtype, int partition_tokens,
                                      void* workspace, size_t workspace_bytes, int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * Paged decode attention without a workspace argument, for callers that
 * cannot allocate device memory: a plugin or C host program whose host
 * application owns every device allocation and exposes no allocator, or a
 * latency-critical loop where cudaMalloc / cudaFree (which synchronise the
 * device) are not allowed.  The pages have no counterpart: this is a calling
 * convention, not part of the method.
 *
 * Computes exactly what pkv_paged_decode_attention computes (same arguments,
 * minus workspace / workspace_bytes).  The scratch is one file-scope device
 * array of PKV_NOALLOC_SCRATCH_BYTES bytes that every GPU loading the library
 * holds until the process exits.  This function allocates nothing.
 *   - Limit: a call whose pkv_decode_workspace_bytes(...) exceeds
 *     PKV_NOALLOC_SCRATCH_BYTES (16 MiB) is refused with PKV_ERR_WORKSPACE.
 *     Either split needs about 5 MB at most on a 152-SM GPU (head_dim 128,
 *     group 8) plus 8 bytes per sequence, so calls of up to about a million
 *     sequences fit.
 *   - Set-up: every call looks up the array's device address on the current
 *     device (cudaGetSymbolAddress, which allocates nothing), so the address
 *     is right after a cudaDeviceReset too.  The first call on a device also
 *     loads the library's device code there: make that first call before any
 *     stream capture.
 *   - Argument errors are reported as pkv_paged_decode_attention reports
 *     them (batch 0 included); only a size check comes first.
 *   - Sharing: every call on a device uses the same array and it keeps the
 *     last call's contents; the kernel writes each scratch word before reading
 *     it, so nothing needs clearing.  Calls that overlap on the GPU (other
 *     streams, or other host threads) race on the scratch: serialise them.
 * ------------------------------------------------------------------------- */
#define PKV_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

pkv_status pkv_paged_decode_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                              const int32_t* block_tables, const int32_t* context_lens, int batch,
                                              int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                              int max_blocks_per_seq, int64_t num_blocks, int max_context_len,
                                              float scale, void* out, pkv_dtype dtype, int partition_tokens,
                                              int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * Paged decode attention over an E4M3 cache (uint8 codes) with per-KV-head
 * scales: K_j and V_j above are replaced by E4M3(code) * k_scale[g] and
 * E4M3(code) * v_scale[g], dequantised in registers before the arithmetic
 * ("KV cache capacity planning ...", section 5).  q and out use q_dtype.  All
 * other arguments as in pkv_paged_decode_attention.
 * ------------------------------------------------------------------------- */
pkv_status pkv_paged_decode_attention_fp8(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                          const float* k_scale, const float* v_scale,
                                          const int32_t* block_tables, const int32_t* context_lens, int batch,
                                          int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                          int max_blocks_per_seq, int64_t num_blocks, int max_context_len,
                                          float scale, void* out, pkv_dtype q_dtype, int partition_tokens,
                                          void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                          void* stream);

/* ---------------------------------------------------------------------------
 * Paged decode attention over an E5M2 cache (uint8 codes, as stored by
 * pkv_kv_append_e5m2) with per-KV-head scales: K_j and V_j are
 * E5M2(code) * k_scale[g] and E5M2(code) * v_scale[g], dequantised in
 * registers before the arithmetic ("KV cache capacity planning ...", sections
 * 4 and 5).  Arguments as in pkv_paged_decode_attention_fp8.
 * ------------------------------------------------------------------------- */
pkv_status pkv_paged_decode_attention_e5m2(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                           const float* k_scale, const float* v_scale,
                                           const int32_t* block_tables, const int32_t* context_lens, int batch,
                                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                           int max_blocks_per_seq, int64_t num_blocks, int max_context_len,
                                           float scale, void* out, pkv_dtype q_dtype, int partition_tokens,
                                           void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                           void* stream);

/* ---------------------------------------------------------------------------
 * One whole decode step in a single decode launch (plus the partial merge):
 * for every sequence b, append k_new[b] / v_new[b] at position
 * p = context_lens[b] - 1 (slot = block_tables[b][p / 16] * 16 + p % 16,
 * written to slot_mapping_out[b] when that pointer is not NULL; -1 for an
 * empty context or an out-of-range table entry), then attend
 * over the context_lens[b] tokens.  Same results as pkv_slot_mapping +
 * pkv_kv_append + pkv_paged_decode_attention, bit for bit.
 *   k_new, v_new    device [batch, num_kv_heads, head_dim] in dtype.
 *   k_cache, v_cache written (the new rows) and read.
 * The new row's slot must belong to sequence b alone (not a block shared with
 * another table), as for any append.  Other arguments as in
 * pkv_paged_decode_attention.
 * ------------------------------------------------------------------------- */
pkv_status pkv_paged_decode_step(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                                 const int32_t* block_tables, const int32_t* context_lens, int batch,
                                 int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                 int max_blocks_per_seq, int64_t num_blocks, int max_context_len, float scale,
                                 void* out, pkv_dtype dtype, int partition_tokens, int64_t* slot_mapping_out,
                                 void* workspace, size_t workspace_bytes, int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * The same fused step over an E4M3 cache: the new rows (q_dtype) are stored as
 * E4M3_RN_satfinite(fl32(x) / scale[h]) exactly as pkv_kv_append_fp8 stores
 * them, and attention uses those codes, as pkv_paged_decode_attention_fp8.
 * ------------------------------------------------------------------------- */
pkv_status pkv_paged_decode_step_fp8(const void* q, const void* k_new, const void* v_new, uint8_t* k_cache,
                                     uint8_t* v_cache, const float* k_scale, const float* v_scale,
                                     const int32_t* block_tables, const int32_t* context_lens, int batch,
                                     int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                     int max_blocks_per_seq, int64_t num_blocks, int max_context_len, float scale,
                                     void* out, pkv_dtype q_dtype, int partition_tokens, int64_t* slot_mapping_out,
                                     void* workspace, size_t workspace_bytes, int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * The same fused step over an E5M2 cache: the new rows (q_dtype) are stored as
 * pkv_kv_append_e5m2 stores them, and attention uses those codes, as
 * pkv_paged_decode_attention_e5m2.  Arguments as in pkv_paged_decode_step_fp8.
 * ------------------------------------------------------------------------- */
pkv_status pkv_paged_decode_step_e5m2(const void* q, const void* k_new, const void* v_new, uint8_t* k_cache,
                                      uint8_t* v_cache, const float* k_scale, const float* v_scale,
                                      const int32_t* block_tables, const int32_t* context_lens, int batch,
                                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                      int max_blocks_per_seq, int64_t num_blocks, int max_context_len, float scale,
                                      void* out, pkv_dtype q_dtype, int partition_tokens, int64_t* slot_mapping_out,
                                      void* workspace, size_t workspace_bytes, int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * One whole decode step from HOST buffers: copies q, k_new, v_new,
 * block_tables and context_lens from (preferably pinned) host memory into the
 * caller's device staging buffers, runs pkv_paged_decode_step (slots of the
 * new tokens into d_slots, append, attention) and copies out back to host
 * memory, all enqueued on `stream`.  The caller synchronises the stream before reading h_out.
 *   h_*        host pointers; shapes as above with num_tokens = batch.
 *   d_*        device staging buffers of the same sizes; d_slots is int64 [batch].
 *   caches     device, persistent across steps.
 * ------------------------------------------------------------------------- */
pkv_status pkv_decode_step_host(const void* h_q, const void* h_k_new, const void* h_v_new,
                                const int32_t* h_block_tables, const int32_t* h_context_lens, void* h_out,
                                void* d_q, void* d_k_new, void* d_v_new, int32_t* d_block_tables,
                                int32_t* d_context_lens, int64_t* d_slots, void* d_out, void* k_cache,
                                void* v_cache, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_blocks_per_seq, int64_t num_blocks, int max_context_len,
                                float scale, pkv_dtype dtype, int partition_tokens, void* workspace,
                                size_t workspace_bytes, int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * INT8 KV cache with per-block min-max scaling ("What a KV cache is ...",
 * section 3.3: q = round((k - k_min) / (k_max - k_min) * 255), two scalars
 * per block).  Codes are uint8, num_blocks x num_kv_heads slabs of 16 x
 * head_dim bytes.  A K slab holds the 16 rows in order, [16][head_dim].  A V
 * slab is the same with head_dim 64; with head_dim 128 it is stored
 * transposed, [128][16], and the 16 columns of a row hold tokens 0 1 8 9 2 3
 * 10 11 4 5 12 13 6 7 14 15 (column c: token 2 (c / 4) + c % 2 +
 * 8 ((c / 2) % 2)), the order in which the decode kernel's tensor-core
 * consumer multiplies them (so it needs no transpose).  The
 * scalars are per (block, KV head) for K and for V, stored as float
 * [num_blocks, num_kv_heads, 4] = (k_min, k_max, v_min, v_max) (16-byte
 * aligned).  Encoding: float32 in the formula's order with IEEE rounding,
 * round half to even, clamped to [0, 255]; max == min gives 0; rows of a
 * block that hold no token have code 0 and do not enter min / max.
 * Decoding: x = min + q (max - min) / 255.
 *
 * pkv_kv_quantize_int8: quantise 16-bit pools k_src / v_src [num_blocks,
 * num_kv_heads, 16, head_dim] of src_dtype; rows_used (device int32
 * [num_blocks], nullable = 16 each) gives the rows of each block that hold
 * tokens.
 * pkv_kv_append_int8: write token t's rows k_new / v_new [T, num_kv_heads,
 * head_dim] (in_dtype) at slot_mapping[t] (< 0 skips; past the pool:
 * PKV_ERR_OOB) and re-quantise rows 0..slot % 16 of that block: the old codes
 * are decoded in float32 as min + ((q * (max - min)) / 255), min / max are
 * taken again over those rows and the new one, and all of them are encoded
 * again.  The tokens of one call must lie in distinct blocks; k_cache, v_cache
 * and slab_params must be 16-byte aligned (PKV_ERR_INVALID_ARG otherwise).
 * pkv_paged_decode_attention_int8: pkv_paged_decode_attention over such a
 * cache; dequantisation happens in registers as k_min sum(q) + dk (q . codes)
 * per score and v_min sum(p) + dv (p . codes) per output.  q_dtype is the type
 * of q and out.
 * ------------------------------------------------------------------------- */
pkv_status pkv_kv_quantize_int8(const void* k_src, const void* v_src, uint8_t* k_cache, uint8_t* v_cache,
                                float* slab_params, const int32_t* rows_used, int64_t num_blocks, int num_kv_heads,
                                int head_dim, int block_size, pkv_dtype src_dtype, int32_t* err_flag, void* stream);
pkv_status pkv_kv_append_int8(const void* k_new, const void* v_new, const int64_t* slot_mapping, int64_t num_tokens,
                              uint8_t* k_cache, uint8_t* v_cache, float* slab_params, int64_t num_blocks,
                              int num_kv_heads, int head_dim, int block_size, pkv_dtype in_dtype, int32_t* err_flag,
                              void* stream);
pkv_status pkv_paged_decode_attention_int8(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                           const float* slab_params, const int32_t* block_tables,
                                           const int32_t* context_lens, int batch, int num_q_heads, int num_kv_heads,
                                           int head_dim, int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                           int max_context_len, float scale, void* out, pkv_dtype q_dtype,
                                           int partition_tokens, void* workspace, size_t workspace_bytes,
                                           int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * Multi-layer cache and whole-step launch ("What a KV cache is ...", section
 * 2.2: one preallocated cache of shape (num_blocks, num_layers, H_kv,
 * block_size, head_dim) for the whole model, so one block id addresses a token
 * range in every layer).  k_cache / v_cache are [num_blocks, num_layers,
 * num_kv_heads, 16, head_dim] (16-bit, 16-byte aligned); block tables and
 * lengths are shared by all layers.
 *
 * pkv_paged_decode_step_layer: pkv_paged_decode_step on layer `layer` of such a
 * cache (0 <= layer < num_layers; PKV_ERR_INVALID_ARG otherwise).
 *
 * pkv_step_graph_create: capture one decode step over all num_layers layers --
 * for each layer l the fused step with q + l * batch * num_q_heads * head_dim,
 * k_new / v_new + l * batch * num_kv_heads * head_dim and out + l * batch *
 * num_q_heads * head_dim elements (q, out [num_layers, batch, Hq, D]; k_new,
 * v_new [num_layers, batch, Hkv, D]), one workspace reused layer after layer --
 * into a CUDA graph.  The graph holds these pointers: later launches read
 * whatever the buffers hold then.  pkv_step_graph_launch replays it on
 * `stream` (one host call per model step); pkv_step_graph_destroy frees it.
 * Errors: PKV_ERR_INVALID_ARG for a null handle or bad sizes, PKV_ERR_CUDA if
 * capture or instantiation fails (pkv_last_error names the call).
 * ------------------------------------------------------------------------- */
pkv_status pkv_paged_decode_step_layer(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                       void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
                                       int batch, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                       int max_blocks_per_seq, int64_t num_blocks, int num_layers, int layer,
                                       int max_context_len, float scale, void* out, pkv_dtype dtype,
                                       int partition_tokens, int64_t* slot_mapping_out, void* workspace,
                                       size_t workspace_bytes, int32_t* err_flag, void* stream);

typedef struct pkv_step_graph pkv_step_graph;

pkv_status pkv_step_graph_create(pkv_step_graph** graph, const void* q, const void* k_new, const void* v_new,
                                 void* k_cache, void* v_cache, const int32_t* block_tables,
                                 const int32_t* context_lens, int batch, int num_q_heads, int num_kv_heads,
                                 int head_dim, int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                 int num_layers, int max_context_len, float scale, void* out, pkv_dtype dtype,
                                 int partition_tokens, int64_t* slot_mapping_out, void* workspace,
                                 size_t workspace_bytes, int32_t* err_flag);
pkv_status pkv_step_graph_launch(pkv_step_graph* graph, void* stream);
void pkv_step_graph_destroy(pkv_step_graph* graph);

/* ---------------------------------------------------------------------------
 * The INT8 decode step: for every sequence b, the new rows k_new[b] /
 * v_new[b] (q_dtype, [batch, num_kv_heads, head_dim]) go to position
 * p = context_lens[b] - 1 (slot written to slot_mapping_out[b] when not NULL;
 * -1 for an empty context or an out-of-range table entry, which also records
 * PKV_ERR_OOB) and rows 0..p % 16 of that block are re-quantised as
 * pkv_kv_append_int8 does; then the attention of
 * pkv_paged_decode_attention_int8 runs over the context_lens[b] tokens.  The
 * same codes, scalars, slots and outputs as pkv_slot_mapping +
 * pkv_kv_append_int8 + pkv_paged_decode_attention_int8, bit for bit, in three
 * launches (append with the slots from the table, decode, combine) that
 * overlap: the decode kernel starts while the append runs and waits for it
 * before reading the cache.  The new row's block must belong to sequence b
 * alone.  Other arguments as in pkv_paged_decode_attention_int8.
 * ------------------------------------------------------------------------- */
pkv_status pkv_paged_decode_step_int8(const void* q, const void* k_new, const void* v_new, uint8_t* k_cache,
                                      uint8_t* v_cache, float* slab_params, const int32_t* block_tables,
                                      const int32_t* context_lens, int batch, int num_q_heads, int num_kv_heads,
                                      int head_dim, int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                      int max_context_len, float scale, void* out, pkv_dtype q_dtype,
                                      int partition_tokens, int64_t* slot_mapping_out, void* workspace,
                                      size_t workspace_bytes, int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * Host-side block pool ("Series 03 ...", sections 3.2-3.3; "What a KV cache
 * is ...", section 3.2): a preallocated set of block ids handed out on demand,
 * with reference counts for blocks shared by several block tables.  Policy: a
 * LIFO free list whose first allocations return 0, 1, 2, ...; a block freed by
 * its last decref is the next one handed out.  Not thread-safe.
 * ------------------------------------------------------------------------- */
typedef struct pkv_pool pkv_pool;

/* NULL on invalid arguments or host allocation failure. */
pkv_pool* pkv_pool_create(int64_t num_blocks, int block_size);
void pkv_pool_destroy(pkv_pool* pool);
/* PKV_ERR_NO_BLOCKS when the pool is empty ("What a KV cache is ...", 4.2). */
pkv_status pkv_pool_alloc(pkv_pool* pool, int32_t* block_id);
/* PKV_ERR_INVALID_ARG for an id that is not allocated. */
pkv_status pkv_pool_incref(pkv_pool* pool, int32_t block_id);
pkv_status pkv_pool_decref(pkv_pool* pool, int32_t block_id);
int64_t pkv_pool_num_free(const pkv_pool* pool);
int32_t pkv_pool_refcount(const pkv_pool* pool, int32_t block_id);   /* -1 for a bad id */
/* Blocks needed for n tokens: ceil(n / block_size) ("Series 03 ...", 3.2). */
int64_t pkv_blocks_needed(int64_t num_tokens, int block_size);

/* ---------------------------------------------------------------------------
 * Copy-on-write ("Series 03 ...", section 3.3: the branches of a beam search,
 * or parallel samples, share the prefix blocks without copying; when a branch
 * writes its first token of its own into a shared block, a new block is taken,
 * the old contents are copied into it and the token is written there, while
 * the other branches keep the old block).
 *
 * pkv_pool_cow: make block_id private before a write.  Reference count 1:
 * *out_id = block_id, nothing changes.  Otherwise a fresh block is taken
 * (reference count 1), block_id loses one reference and *out_id is the new
 * id; the caller points its table at it and copies block_id into it
 * (pkv_copy_blocks) before writing.  PKV_ERR_NO_BLOCKS (nothing changed) when
 * the pool is empty, PKV_ERR_INVALID_ARG for an id that is not allocated.
 * ------------------------------------------------------------------------- */
pkv_status pkv_pool_cow(pkv_pool* pool, int32_t block_id, int32_t* out_id);

/* Host side of one decode step over tables that may share blocks.  For each
 * sequence b the step's token sits at position p = context_lens[b] - 1 (the
 * length after the append; 0 means no token for b).  Entry i = p / block_size
 * of row b of block_tables ([batch, max_blocks_per_seq], host memory):
 *   - negative: the sequence grows into a new block; a fresh block is taken
 *     and stored there;
 *   - a shared block: pkv_pool_cow, the new id is stored and the pair
 *     (old, new) is appended to src_blocks / dst_blocks (host arrays of
 *     capacity batch);
 *   - a private block: nothing.
 * Sequences are taken in order b = 0, 1, ..., so when several rows share one
 * block, all but the last of them copy and the last writes in place.
 * *num_pairs receives the number of copies.  All-or-nothing: when the pool
 * cannot supply every block the step needs, PKV_ERR_NO_BLOCKS and nothing
 * changes.  PKV_ERR_INVALID_ARG for p past the row or an entry that is not an
 * allocated block.
 * ------------------------------------------------------------------------- */
pkv_status pkv_prepare_append(pkv_pool* pool, int32_t* block_tables, int batch, int max_blocks_per_seq,
                              const int32_t* context_lens, int32_t* src_blocks, int32_t* dst_blocks,
                              int32_t* num_pairs);

/* Block copy on the device (the data movement of copy-on-write): for each
 * i < num_pairs, physical block dst_blocks[i] of k_cache and of v_cache takes
 * the contents of block src_blocks[i], all heads and all rows; a bit-exact
 * copy of num_kv_heads * block_size * head_dim elements of elt_bytes bytes
 * (2 for fp16/bf16 caches, 1 for E4M3) per block and cache.  src_blocks and
 * dst_blocks are device int32 arrays.  A pair with an id outside
 * [0, num_blocks) is skipped and reported as PKV_ERR_OOB in err_flag.  The
 * destinations must be distinct and none may be a source (the pairs
 * pkv_prepare_append returns are); otherwise the result is undefined.
 * ------------------------------------------------------------------------- */
pkv_status pkv_copy_blocks(const int32_t* src_blocks, const int32_t* dst_blocks, int64_t num_pairs, void* k_cache,
                           void* v_cache, int64_t num_blocks, int num_kv_heads, int head_dim, int block_size,
                           int elt_bytes, int32_t* err_flag, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
