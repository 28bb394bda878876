// Paged decode attention for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: a plugin or C host program
// whose host application owns every device allocation and exposes no
// allocator, or a latency-critical loop in which cudaMalloc / cudaFree (which
// synchronise the device) are not allowed.  This entry point gives them decode
// attention without a workspace argument: the scratch lives in one file-scope
// device array of fixed size, which every GPU that loads the library keeps
// until the process exits.  Nothing here allocates.
#include <cuda_runtime.h>

#include "../../include/pkv.h"
#include "host_util.h"

namespace pkv {
namespace {

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch in the current device's context.  It is
// looked up on every call (cudaGetSymbolAddress allocates nothing and, once
// the module is loaded, is a host-side table lookup), so the address stays
// right after a cudaDeviceReset or in another context of the same device.
// The first call on a device loads the library's device code there.
pkv_status scratch_on_current_device(void** out) {
  void* p = nullptr;
  if (cuda_failed(cudaGetSymbolAddress(&p, g_noalloc_scratch), "cudaGetSymbolAddress")) return PKV_ERR_CUDA;
  *out = p;
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_paged_decode_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                         const int32_t* block_tables, const int32_t* context_lens,
                                                         int batch, int num_q_heads, int num_kv_heads,
                                                         int head_dim, int block_size, int max_blocks_per_seq,
                                                         int64_t num_blocks, int max_context_len, float scale,
                                                         void* out, pkv_dtype dtype, int partition_tokens,
                                                         int32_t* err_flag, void* stream) {
  // Sizes beyond the scratch are refused before anything else.  A size of 0
  // (arguments the query rejects, or a failed device query) falls through:
  // the workspace entry point below validates in its own order and returns
  // the same status it would return to a caller with a workspace.
  const size_t need = pkv_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                                 max_context_len, partition_tokens);
  if (need > PKV_NOALLOC_SCRATCH_BYTES) {
    // too large for the fixed scratch: refuse rather than overrun it
    pkv::cuda_failed(cudaErrorMemoryAllocation, "pkv_paged_decode_attention_noalloc: scratch too small");
    return PKV_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const pkv_status st = pkv::scratch_on_current_device(&scratch);
  if (st != PKV_OK) return st;
  // The decode kernel writes every scratch word before it reads it, so the
  // previous call's contents need no clearing.
  return pkv_paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, batch, num_q_heads,
                                    num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
                                    max_context_len, scale, out, dtype, partition_tokens, scratch,
                                    PKV_NOALLOC_SCRATCH_BYTES, err_flag, stream);
}
