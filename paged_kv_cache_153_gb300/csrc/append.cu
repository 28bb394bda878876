// Slot mapping, KV append and copy-on-write block copy kernels (sm_103a) and
// their C-ABI entry points.
//
// Slot of token t: table[b][p / 16] * 16 + p % 16 (the block-table lookup of
// "Series 03: why the KV cache eats memory, and how PagedAttention pages it",
// section 3.1).  Append writes the token's K/V rows into that slot ("KV Cache,
// the memory notepad of LLM inference", section 三), as a bit copy or, for the
// FP8 caches of "KV cache capacity planning ..." section 4 (E4M3 or E5M2), as
// FP8_RN_satfinite(fl32(x) / scale[h]).
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "host_util.h"
#include "pkv_common.cuh"

namespace pkv {

__global__ void slot_mapping_kernel(const int32_t* __restrict__ tables, int max_blocks, int64_t num_blocks,
                                    const int32_t* __restrict__ seq_idx, const int32_t* __restrict__ positions,
                                    int32_t offset, int64_t n_tokens, int64_t* __restrict__ slots,
                                    int32_t* err) {
  pdl_wait_and_release();   // (writes only the slots, which no kernel reads before its wait)
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
  pdl_wait();   // (writes the cache: no early release of the next launch)
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

// One thread quantises 8 elements (16 input bytes -> 8 code bytes) to the
// FP8 format FMT.
template <typename FMT, typename IN>
__global__ void kv_append_fp8_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                     const int64_t* __restrict__ slots, int64_t n_tokens,
                                     uint2* __restrict__ k_cache, uint2* __restrict__ v_cache,
                                     const float* __restrict__ k_scale, const float* __restrict__ v_scale,
                                     int64_t num_slots, int n_heads, int chunks_per_row, int32_t* err) {
  pdl_wait();   // (writes the cache: no early release of the next launch)
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
  const uint2 packed = quant8_fp8<FMT>(is_v ? &v_new[i] : &k_new[i], scale, IN{});
  const int64_t blk = s / kBlockSize, off = s % kBlockSize;
  const int64_t dst = ((blk * n_heads + h) * kBlockSize + off) * chunks_per_row + c;
  if (is_v)
    v_cache[dst] = packed;
  else
    k_cache[dst] = packed;
}

// Copy-on-write data movement: block dst[i] of both caches takes block
// src[i].  The copy is staged through shared memory by TMA: the work is cut
// into (pair, cache, chunk) items of `chunk` bytes, thread block c takes items
// c, c + grid, ..., and one thread keeps kCopyStages 1-D bulk loads (global ->
// shared, completion on an mbarrier per stage) and bulk stores (shared ->
// global, bulk groups) in flight.  A stage is reloaded only after the store
// that read it has finished reading (bulk wait_group.read).
constexpr int kCopyStages = 6;
constexpr int kCopyChunkMax = 16384;

__global__ void __launch_bounds__(32) copy_blocks_kernel(const int32_t* __restrict__ src,
                                                         const int32_t* __restrict__ dst, int64_t n_pairs,
                                                         char* k_cache, char* v_cache, int64_t num_blocks,
                                                         int64_t block_bytes, int chunk, int chunks_per_block,
                                                         int32_t* err) {
  extern __shared__ __align__(128) unsigned char cp_smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(cp_smem + static_cast<size_t>(kCopyStages) * chunk);
  pdl_wait();   // (writes the cache: no early release of the next launch)
  if (threadIdx.x != 0) return;
  for (int s = 0; s < kCopyStages; ++s) mbar_init(&full[s], 1);
  fence_mbar_init();
  const int64_t per_pair = 2ll * chunks_per_block;
  const int64_t items = n_pairs * per_pair;
  const int64_t mine = items > blockIdx.x ? (items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const uint64_t pol = policy_evict_first();
  // item k of this block: source and destination addresses; false for a pair out of range
  auto locate = [&](int64_t k, const char*& from, char*& to) -> bool {
    const int64_t item = blockIdx.x + k * gridDim.x;
    const int64_t pair = item / per_pair;
    const int64_t rem = item - pair * per_pair;
    const int32_t s = src[pair], d = dst[pair];
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
      if (rem == 0) record_error(err, PKV_ERR_OOB);
      return false;
    }
    char* base = rem >= chunks_per_block ? v_cache : k_cache;
    const int64_t off = (rem % chunks_per_block) * chunk;
    from = base + s * block_bytes + off;
    to = base + d * block_bytes + off;
    return true;
  };
  uint32_t live = 0;   // bit s: stage s holds a real load
  auto load = [&](int64_t k) {
    const int s = static_cast<int>(k % kCopyStages);
    const char* from;
    char* to;
    if (locate(k, from, to)) {
      mbar_arrive_expect_tx(&full[s], chunk);
      bulk_g2s(cp_smem + static_cast<size_t>(s) * chunk, from, chunk, &full[s], pol);
      live |= 1u << s;
    } else {
      mbar_arrive(&full[s]);   // completes the phase with no bytes, so parities stay in step
      live &= ~(1u << s);
    }
  };
  for (int64_t k = 0; k < mine && k < kCopyStages; ++k) load(k);
  int64_t k = 0;
  for (; k < mine; ++k) {
    const int s = static_cast<int>(k % kCopyStages);
    if (!mbar_wait(&full[s], static_cast<uint32_t>((k / kCopyStages) & 1), err)) break;
    const char* from;
    char* to;
    if (((live >> s) & 1u) && locate(k, from, to)) bulk_s2g(to, cp_smem + static_cast<size_t>(s) * chunk, chunk);
    bulk_commit_group();
    // reload the previous item's stage once its store has read it
    if (k >= 1 && k - 1 + kCopyStages < mine) {
      bulk_wait_group_read<1>();
      load(k - 1 + kCopyStages);
    }
  }
  if (k < mine) {
    // a load never completed: wait (bounded) for the loads still in flight
    // before the block's shared memory goes away
    const unsigned long long deadline = global_ns() + kWaitLimitNs;
    for (int64_t j = k; j < mine && j < k + kCopyStages; ++j) {
      const int s = static_cast<int>(j % kCopyStages);
      mbar_wait_until(&full[s], static_cast<uint32_t>((j / kCopyStages) & 1), deadline);
    }
  }
  bulk_wait_group<0>();
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

namespace pkv {
namespace {

template <typename FMT>
pkv_status append_fp8(const void* k_new, const void* v_new, const int64_t* slot_mapping, int64_t num_tokens,
                      uint8_t* k_cache, uint8_t* v_cache, int64_t num_blocks, const float* k_scale,
                      const float* v_scale, int num_kv_heads, int head_dim, int block_size, pkv_dtype in_dtype,
                      int32_t* err_flag, void* stream, const char* what) {
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
  auto kern = (in_dtype == PKV_F16) ? kv_append_fp8_kernel<FMT, F16> : kv_append_fp8_kernel<FMT, BF16>;
  const cudaError_t e = launch_pdl(kern, dim3(grid), dim3(threads), 0, s, static_cast<const uint4*>(k_new),
                                   static_cast<const uint4*>(v_new), slot_mapping, num_tokens,
                                   reinterpret_cast<uint2*>(k_cache), reinterpret_cast<uint2*>(v_cache), k_scale,
                                   v_scale, num_blocks * kBlockSize, num_kv_heads, chunks, err_flag);
  return cuda_failed(e, what) ? PKV_ERR_CUDA : PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_kv_append_fp8(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                        int64_t num_tokens, uint8_t* k_cache, uint8_t* v_cache,
                                        int64_t num_blocks, const float* k_scale, const float* v_scale,
                                        int num_kv_heads, int head_dim, int block_size, pkv_dtype in_dtype,
                                        int32_t* err_flag, void* stream) {
  return pkv::append_fp8<E4M3>(k_new, v_new, slot_mapping, num_tokens, k_cache, v_cache, num_blocks, k_scale,
                               v_scale, num_kv_heads, head_dim, block_size, in_dtype, err_flag, stream,
                               "kv_append_fp8_kernel launch");
}

extern "C" pkv_status pkv_kv_append_e5m2(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                         int64_t num_tokens, uint8_t* k_cache, uint8_t* v_cache,
                                         int64_t num_blocks, const float* k_scale, const float* v_scale,
                                         int num_kv_heads, int head_dim, int block_size, pkv_dtype in_dtype,
                                         int32_t* err_flag, void* stream) {
  return pkv::append_fp8<E5M2>(k_new, v_new, slot_mapping, num_tokens, k_cache, v_cache, num_blocks, k_scale,
                               v_scale, num_kv_heads, head_dim, block_size, in_dtype, err_flag, stream,
                               "kv_append_fp8_kernel launch (E5M2)");
}

extern "C" pkv_status pkv_copy_blocks(const int32_t* src_blocks, const int32_t* dst_blocks, int64_t num_pairs,
                                      void* k_cache, void* v_cache, int64_t num_blocks, int num_kv_heads,
                                      int head_dim, int block_size, int elt_bytes, int32_t* err_flag, void* stream) {
  if (num_pairs < 0 || num_blocks < 0 || num_kv_heads <= 0 || head_dim <= 0) return PKV_ERR_INVALID_ARG;
  if (elt_bytes != 1 && elt_bytes != 2) return PKV_ERR_INVALID_ARG;
  if (block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PKV_OK;
  if (!src_blocks || !dst_blocks || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID_ARG;
  const int64_t block_bytes = static_cast<int64_t>(num_kv_heads) * kBlockSize * head_dim * elt_bytes;
  if (block_bytes % 16) return PKV_ERR_UNSUPPORTED;
  // chunk: the largest piece of at most kCopyChunkMax bytes that cuts a block evenly in multiples of 16
  int64_t pieces = (block_bytes + kCopyChunkMax - 1) / kCopyChunkMax;
  while (block_bytes % pieces || (block_bytes / pieces) % 16) ++pieces;
  const int chunk = static_cast<int>(block_bytes / pieces);
  const size_t smem = static_cast<size_t>(kCopyStages) * chunk + 8 * kCopyStages;
  int dev = 0, sms = 0;
  if (cuda_failed(cudaGetDevice(&dev), "cudaGetDevice") ||
      cuda_failed(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute"))
    return PKV_ERR_CUDA;
  static std::mutex mu;
  static bool attr_done[64] = {};
  if (dev < 0 || dev >= 64) return PKV_ERR_UNSUPPORTED;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_done[dev]) {
      if (cuda_failed(cudaFuncSetAttribute(copy_blocks_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kCopyStages) * kCopyChunkMax + 8 * kCopyStages),
                      "cudaFuncSetAttribute"))
        return PKV_ERR_CUDA;
      attr_done[dev] = true;
    }
  }
  // two blocks per SM (each ~96 KiB of stages in flight)
  const int64_t items = num_pairs * 2 * pieces;
  const int64_t grid = std::min<int64_t>(items, 2ll * sms);
  const cudaError_t e =
      launch_pdl(copy_blocks_kernel, dim3(static_cast<unsigned>(grid)), dim3(32), smem,
                 static_cast<cudaStream_t>(stream), src_blocks, dst_blocks, num_pairs, static_cast<char*>(k_cache),
                 static_cast<char*>(v_cache), num_blocks, block_bytes, chunk, static_cast<int>(pieces), err_flag);
  return cuda_failed(e, "copy_blocks_kernel launch") ? PKV_ERR_CUDA : PKV_OK;
}
