/*
 * pkv_prefill.h -- C ABI of the paged prefill library, libpkv_prefill.so.
 *
 * The prefill kernel is a separate shared library so that a process that only
 * decodes never loads it.  Its thread blocks run in clusters of two that share
 * each K/V tile through TMA loads multicast to both blocks of the pair; those
 * loads read this GPU's own cache only, and the library is meant for
 * single-GPU processes.  libpkv_prefill.so depends on libpkv.so (found next to
 * it) for error reporting: a PKV_ERR_CUDA status is described by
 * pkv_last_error() of pkv.h.  Types, status codes and conventions are those of
 * pkv.h.
 */
#ifndef PKV_PREFILL_H_
#define PKV_PREFILL_H_

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------------------
 * Paged prefill / extend attention ("KV Cache, the memory notepad ...",
 * sections 二-四: prefill attends over the prompt; "Series 03 ...", section 3.1:
 * K/V through the block table, section 5.1: chunked prefill).  The new tokens
 * of sequence b are its last n_b = cu_seqlens[b+1] - cu_seqlens[b] positions
 * (context_lens[b] counts them; the cache must already hold their K/V, e.g.
 * written by pkv_kv_append).  Token i of sequence b, at position
 * p = context_lens[b] - n_b + i, attends causally to positions 0..p:
 *     out[cu_seqlens[b] + i, h] = sum_{j <= p} softmax_j(scale <q, K_j>) V_j
 * with K_j, V_j of KV head h / G (G = num_q_heads / num_kv_heads in {1, 2, 4,
 * 8}).  q and out are [T, num_q_heads, 128] of dtype (T = cu_seqlens[batch]);
 * the caches [num_blocks, num_kv_heads, 16, 128] of the same dtype;
 * block_tables int32 [batch, max_blocks_per_seq]; context_lens, cu_seqlens
 * int32 device arrays; max_query_len >= every n_b.  Runs on the tensor cores
 * (tcgen05, scores, P and accumulators in tensor memory) with fp32 softmax;
 * fp16 P is rounded to fp16 before P.V, bf16 P is multiplied as a pair of
 * bf16 parts (hi = p truncated, lo = p - hi rounded), exact to ~2^-16.  The
 * kernel launches in clusters of two thread blocks that share each K/V tile
 * load; a launch the device cannot schedule returns PKV_ERR_CUDA.  head_dim
 * 128 and block_size 16 only (else PKV_ERR_UNSUPPORTED).  Device errors in err_flag: PKV_ERR_OOB for a block id
 * outside [0, num_blocks), more new tokens than context or a context past the
 * table (that sequence's tile is skipped); PKV_ERR_TIMEOUT if a pipeline wait
 * exceeds its limit.
 * ------------------------------------------------------------------------- */
pkv_status pkv_paged_prefill_attention(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, const int32_t* context_lens,
                                       const int32_t* cu_seqlens, int batch, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                       int max_query_len, float scale, void* out, pkv_dtype dtype,
                                       int32_t* err_flag, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_PREFILL_H_ */
