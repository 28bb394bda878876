// Host-side helpers shared by the C-ABI translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/pkv.h"

namespace pkv {

// Record a failed CUDA runtime call (name + error) for pkv_last_error() and
// clear the runtime's last-error state so it cannot leak into a later call.
// Returns true when `e` is an error.
bool cuda_failed(cudaError_t e, const char* what);

// Tiled TMA view of a KV cache [rows, head_dim] (rows = num_blocks * H_kv * 16)
// with a [16 rows x 128 bytes] box and the 128-byte swizzle.  Returns false
// (with the reason kept for pkv_last_error) on failure.
// Launch with programmatic stream serialisation allowed (the kernel must call
// pdl_wait_and_release() before it touches global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

bool encode_cache_tmap(CUtensorMap* map, const void* base, int64_t rows, int head_dim, int elt_bytes);

// The append of the INT8 decode step (append_int8.cu): slots from the block
// table, re-quantising append, early release of the decode launch that
// follows (which waits for it before reading the cache).
pkv_status launch_append_int8_step(const void* k_new, const void* v_new, uint8_t* k_cache, uint8_t* v_cache,
                                   float* slab_params, const int32_t* block_tables, const int32_t* context_lens,
                                   int batch, int max_blocks_per_seq, int64_t num_blocks, int num_kv_heads,
                                   int head_dim, pkv_dtype in_dtype, int64_t* slots_out, int32_t* err_flag,
                                   cudaStream_t stream);

}  // namespace pkv
