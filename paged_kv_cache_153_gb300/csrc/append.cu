// Slot mapping and KV append kernels (sm_103a) and their C-ABI entry points.
//
// Slot of token t: table[b][p / 16] * 16 + p % 16 (the block-table lookup of
// "Series 03: why the KV cache eats memory, and how PagedAttention pages it",
// section 3.1).  Append writes the token's K/V rows into that slot ("KV Cache,
// the memory notepad of LLM inference", section 三), as a bit copy or, for the
// E4M3 cache of "KV cache capacity planning ..." section 4, as
// E4M3_RN_satfinite(fl32(x) / scale[h]).
#include <cuda_runtime.h>

#include "host_util.h"
#include "pkv_common.cuh"

namespace pkv {

__global__ void slot_mapping_kernel(const int32_t* __restrict__ tables, int max_blocks, int64_t num_blocks,
                                    const int32_t* __restrict__ seq_idx, const int32_t* __restrict__ positions,
                                    int32_t offset, int64_t n_tokens, int64_t* __restrict__ slots,
                                    int32_t* err) {
  pdl_wait_and_release();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n_tokens) return;
  const int64_t b = seq_idx ? seq_idx[t] : t;
  const int64_t p = static_cast<int64_t>(positions[t]) + offset;
  if (p < 0) {
    slots[t] = -1;
    return;
  }
  const int64_t logical = p / kBlockSize;
  if (b < 0 || logical >= max_blocks) {
    slots[t] = -1;
    record_error(err, PKV_ERR_OOB);
    return;
  }
  const int32_t phys = tables[b * max_blocks + logical];
  if (phys < 0 || phys >= num_blocks) {
    slots[t] = -1;
    record_error(err, PKV_ERR_OOB);
    return;
  }
  slots[t] = static_cast<int64_t>(phys) * kBlockSize + (p % kBlockSize);
}

// One thread moves 16 bytes (8 elements) of one row of K or V.
__global__ void kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                 const int64_t* __restrict__ slots, int64_t n_tokens, uint4* __restrict__ k_cache,
                                 uint4* __restrict__ v_cache, int64_t num_slots, int n_heads, int chunks_per_row,
                                 int32_t* err) {
  pdl_wait_and_release();
  const int64_t per_kv = n_tokens * n_heads * chunks_per_row;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= 2 * per_kv) return;
  const bool is_v = i >= per_kv;
  if (is_v) i -= per_kv;
  const int c = static_cast<int>(i % chunks_per_row);
  const int64_t row = i / chunks_per_row;          // t * H + h
  const int h = static_cast<int>(row % n_heads);
  const int64_t t = row / n_heads;
  const int64_t s = slots[t];
  if (s < 0) return;
  if (s >= num_slots) {
    record_error(err, PKV_ERR_OOB);
    return;
  }
  const int64_t blk = s / kBlockSize, off = s % kBlockSize;
  const int64_t dst = ((blk * n_heads + h) * kBlockSize + off) * chunks_per_row + c;
  if (is_v)
    v_cache[dst] = v_new[i];
  else
    k_cache[dst] = k_new[i];
}

// One thread quantises 8 elements (16 input bytes -> 8 code bytes).
template <typename IN>
__global__ void kv_append_fp8_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                     const int64_t* __restrict__ slots, int64_t n_tokens,
                                     uint2* __restrict__ k_cache, uint2* __restrict__ v_cache,
                                     const float* __restrict__ k_scale, const float* __restrict__ v_scale,
                                     int64_t num_slots, int n_heads, int chunks_per_row, int32_t* err) {
  pdl_wait_and_release();
  const int64_t per_kv = n_tokens * n_heads * chunks_per_row;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= 2 * per_kv) return;
  const bool is_v = i >= per_kv;
  if (is_v) i -= per_kv;
  const int c = static_cast<int>(i % chunks_per_row);
  const int64_t row = i / chunks_per_row;
  const int h = static_cast<int>(row % n_heads);
  const int64_t t = row / n_heads;
  const int64_t s = slots[t];
  if (s < 0) return;
  if (s >= num_slots) {
    record_error(err, PKV_ERR_OOB);
    return;
  }
  const float scale = is_v ? v_scale[h] : k_scale[h];
  const uint2 packed = quant8_e4m3(is_v ? &v_new[i] : &k_new[i], scale, IN{});
  const int64_t blk = s / kBlockSize, off = s % kBlockSize;
  const int64_t dst = ((blk * n_heads + h) * kBlockSize + off) * chunks_per_row + c;
  if (is_v)
    v_cache[dst] = packed;
  else
    k_cache[dst] = packed;
}

}  // namespace pkv

using namespace pkv;

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

extern "C" pkv_status pkv_slot_mapping(const int32_t* block_tables, int max_blocks_per_seq, int64_t num_blocks,
                                       const int32_t* seq_idx, const int32_t* positions, int32_t position_offset,
                                       int64_t num_tokens, int block_size, int64_t* slot_mapping,
                                       int32_t* err_flag, void* stream) {
  if (num_tokens < 0 || max_blocks_per_seq <= 0 || num_blocks < 0) return PKV_ERR_INVALID_ARG;
  if (block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!block_tables || !positions || !slot_mapping) return PKV_ERR_INVALID_ARG;
  const int threads = 128;
  const int64_t grid = (num_tokens + threads - 1) / threads;
  const cudaError_t e = launch_pdl(slot_mapping_kernel, dim3(static_cast<unsigned>(grid)), dim3(threads), 0,
                                   static_cast<cudaStream_t>(stream), block_tables, max_blocks_per_seq,
                                   num_blocks, seq_idx, positions, position_offset, num_tokens, slot_mapping,
                                   err_flag);
  return cuda_failed(e, "slot_mapping_kernel launch") ? PKV_ERR_CUDA : PKV_OK;
}

extern "C" pkv_status pkv_kv_append(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                    int64_t num_tokens, void* k_cache, void* v_cache, int64_t num_blocks,
                                    int num_kv_heads, int head_dim, int block_size, pkv_dtype dtype,
                                    int32_t* err_flag, void* stream) {
  if (num_tokens < 0 || num_blocks < 0 || num_kv_heads <= 0) return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (block_size != kBlockSize || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  const int chunks = head_dim * 2 / 16;
  const int64_t total = 2 * num_tokens * num_kv_heads * chunks;
  const int threads = 256;
  const int64_t grid = (total + threads - 1) / threads;
  const cudaError_t e = launch_pdl(
      kv_append_kernel, dim3(static_cast<unsigned>(grid)), dim3(threads), 0, static_cast<cudaStream_t>(stream),
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping, num_tokens,
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_blocks * kBlockSize, num_kv_heads, chunks,
      err_flag);
  return cuda_failed(e, "kv_append_kernel launch") ? PKV_ERR_CUDA : PKV_OK;
}

extern "C" pkv_status pkv_kv_append_fp8(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                        int64_t num_tokens, uint8_t* k_cache, uint8_t* v_cache,
                                        int64_t num_blocks, const float* k_scale, const float* v_scale,
                                        int num_kv_heads, int head_dim, int block_size, pkv_dtype in_dtype,
                                        int32_t* err_flag, void* stream) {
  if (num_tokens < 0 || num_blocks < 0 || num_kv_heads <= 0) return PKV_ERR_INVALID_ARG;
  if (in_dtype != PKV_F16 && in_dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (block_size != kBlockSize || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  const int chunks = head_dim / 8;
  const int64_t total = 2 * num_tokens * num_kv_heads * chunks;
  const int threads = 256;
  const unsigned grid = static_cast<unsigned>((total + threads - 1) / threads);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto kern = (in_dtype == PKV_F16) ? kv_append_fp8_kernel<F16> : kv_append_fp8_kernel<BF16>;
  const cudaError_t e = launch_pdl(kern, dim3(grid), dim3(threads), 0, s, static_cast<const uint4*>(k_new),
                                   static_cast<const uint4*>(v_new), slot_mapping, num_tokens,
                                   reinterpret_cast<uint2*>(k_cache), reinterpret_cast<uint2*>(v_cache), k_scale,
                                   v_scale, num_blocks * kBlockSize, num_kv_heads, chunks, err_flag);
  return cuda_failed(e, "kv_append_fp8_kernel launch") ? PKV_ERR_CUDA : PKV_OK;
}
