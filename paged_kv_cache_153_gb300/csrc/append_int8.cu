// INT8 KV cache with per-block min-max scaling ("What a KV cache is and why it
// is the crux of LLM inference", section 3.3):
//   q = round((x - min) / (max - min) * 255)
// with (min, max) per (block, KV head) for K and for V, kept as float4
// (k_min, k_max, v_min, v_max) per slab.  Arithmetic is float32 in the
// formula's order with IEEE rounding (no contraction), round half to even,
// clamped to [0, 255]; max == min gives 0.  Rows past the ones holding tokens
// have code 0.  Appending a token re-quantises its block's rows so far: the
// old codes are decoded as min + ((q * (max - min)) / 255), the new row added,
// min / max taken again and every row encoded again.
//
// Layout.  K codes of a (block, head) slab are stored as the rows: [16][d].
// With d = 128, V codes are stored transposed, [d][16], and the 16 columns of
// a row hold the tokens in the order 0 1 8 9 2 3 10 11 4 5 12 13 6 7 14 15
// (column c holds token 2 (c / 4) + c % 2 + 8 ((c / 2) % 2)): an 8 x 16-byte
// ldmatrix of that slab hands each lane of the decode kernel's p . V tensor
// core MMA exactly the four tokens of its A fragment, so no transpose is
// needed there.  With d = 64, V is stored as the rows, like K.
#include <cuda_runtime.h>

#include "host_util.h"
#include "pkv_common.cuh"

namespace pkv {

// byte offset, inside a V slab, of row r (token), column c (head_dim index),
// i = r * d + c in the row layout (see the layout note above)
__device__ __forceinline__ int v_code_index(int i, int d) {
  if (d != 128) return i;
  const int r = i >> 7, c = i & 127;
  return c * kBlockSize + int8_vt_column(r);
}

constexpr int kQThreads = 256;
constexpr int kQPer = 8;   // values per thread: 16 rows x 128 / 256

// block-wide min and max of one value per thread (NaN-free inputs)
__device__ __forceinline__ float2 block_minmax(float lo, float hi, float2* scratch) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, m));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, m));
  }
  const int warp = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) scratch[warp] = make_float2(lo, hi);
  __syncthreads();
  float2 r = scratch[0];
  for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) {
    r.x = fminf(r.x, scratch[w].x);
    r.y = fmaxf(r.y, scratch[w].y);
  }
  return r;
}

template <typename IN>
__device__ __forceinline__ float in_f32(const void* base, int64_t i, IN);
template <>
__device__ __forceinline__ float in_f32(const void* base, int64_t i, F16) {
  return __half2float(static_cast<const __half*>(base)[i]);
}
template <>
__device__ __forceinline__ float in_f32(const void* base, int64_t i, BF16) {
  return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
}

// one thread block per (block, KV head): quantise rows [0, n) of the K and V slabs
template <typename IN>
__global__ void __launch_bounds__(kQThreads) quantize_int8_kernel(const void* k_src, const void* v_src,
                                                                  uint8_t* k_codes, uint8_t* v_codes,
                                                                  float4* params, const int32_t* rows_used,
                                                                  int n_heads, int d) {
  __shared__ float2 scratch[kQThreads / 32];
  pdl_wait();   // (writes the cache: no early release of the next launch)
  const int64_t slab = blockIdx.x;             // block * n_heads + head
  const int blk = static_cast<int>(slab / n_heads);
  const int n = rows_used ? min(max(rows_used[blk], 0), kBlockSize) : kBlockSize;
  const int count = n * d;
  float lohi[4];
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {
    const void* src = which ? v_src : k_src;
    uint8_t* dst = (which ? v_codes : k_codes) + slab * kBlockSize * d;
    float x[kQPer];
    float lo = INFINITY, hi = -INFINITY;
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int i = threadIdx.x + k * kQThreads;
      x[k] = (i < count) ? in_f32(src, slab * kBlockSize * d + i, IN{}) : 0.f;
      if (i < count) {
        lo = fminf(lo, x[k]);
        hi = fmaxf(hi, x[k]);
      }
    }
    const float2 mm = block_minmax(lo, hi, scratch);
    const float span = (count > 0) ? __fsub_rn(mm.y, mm.x) : 0.f;
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int i = threadIdx.x + k * kQThreads;
      if (i < kBlockSize * d) dst[which ? v_code_index(i, d) : i] = (i < count) ? int8_code(x[k], mm.x, span) : 0;
    }
    lohi[2 * which] = count > 0 ? mm.x : 0.f;
    lohi[2 * which + 1] = count > 0 ? mm.y : 0.f;
  }
  if (threadIdx.x == 0) params[slab] = make_float4(lohi[0], lohi[1], lohi[2], lohi[3]);
}

// min and max over one half of the block (128 threads, 4 warps, named barrier
// 1 + half); NaN-free inputs
__device__ __forceinline__ float2 half_minmax(float lo, float hi, float2* scratch, int half) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, m));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, m));
  }
  const int w = (threadIdx.x >> 5) & 3;
  if ((threadIdx.x & 31) == 0) scratch[4 * half + w] = make_float2(lo, hi);
  asm volatile("bar.sync %0, 128;" ::"r"(1 + half) : "memory");
  float2 r = scratch[4 * half];
#pragma unroll
  for (int k = 1; k < 4; ++k) {
    r.x = fminf(r.x, scratch[4 * half + k].x);
    r.y = fmaxf(r.y, scratch[4 * half + k].y);
  }
  return r;
}

// Where the decode step's new rows go when the slots come from the block
// table: token b is sequence b's new token at position context_lens[b] - 1.
struct TableSlots {
  const int32_t* block_tables;   // [B, max_blocks_per_seq]
  const int32_t* context_lens;   // [B]
  int max_blocks_per_seq;
  int64_t* slots_out;            // [B] slots written (nullable); -1 for none
};

// one thread block per (token, KV head): write the token's row and re-quantise
// rows [0, row] of its block's K slab (threads 0-127) and V slab (128-255)
// side by side.  FROM_TABLE (the append of the INT8 decode step): the slot of
// token b is found from the block table (position context_lens[b] - 1) and
// reported; the slab is read at once and written after the wait for the
// previous kernel -- the previous step's combine, which may have released
// this launch early and completes after the previous decode kernel, the last
// reader of these slabs.  (The slabs were last written by the previous step's append,
// which had completed before that decode kernel released its combine.)  The
// next launch, the step's decode kernel, may start at once: it waits for this
// grid before it reads a block this grid writes, and this grid completes only
// after the previous kernel has.
template <typename IN, bool FROM_TABLE>
__global__ void __launch_bounds__(kQThreads) append_int8_kernel(const void* k_new, const void* v_new,
                                                                const int64_t* slots, uint8_t* k_codes,
                                                                uint8_t* v_codes, float4* params,
                                                                int64_t num_slots, int n_heads, int d,
                                                                int32_t* err, TableSlots ts) {
  constexpr int kPer = 2 * kQPer;   // values per thread: 16 rows x 128 / 128
  __shared__ float2 scratch[8];
  __shared__ float2 lohi_out[2];
  if constexpr (FROM_TABLE)
    pdl_release();
  else
    pdl_wait();   // (writes the cache: no early release of the next launch)
  const int64_t t = blockIdx.x / n_heads;
  const int h = static_cast<int>(blockIdx.x % n_heads);
  int64_t s;
  if constexpr (FROM_TABLE) {
    // the slot-mapping rule: table[b][p / 16] * 16 + p % 16 for p = ctx - 1
    const int p = ts.context_lens[t] - 1;
    s = -1;
    bool oob = false;
    if (p >= 0) {
      if (p / kBlockSize >= ts.max_blocks_per_seq) {
        oob = true;
      } else {
        const int32_t phys = ts.block_tables[t * ts.max_blocks_per_seq + p / kBlockSize];
        if (phys < 0 || static_cast<int64_t>(phys) * kBlockSize >= num_slots) oob = true;
        else s = static_cast<int64_t>(phys) * kBlockSize + p % kBlockSize;
      }
    }
    if (h == 0 && threadIdx.x == 0) {
      if (ts.slots_out != nullptr) ts.slots_out[t] = s;
      if (oob) record_error(err, PKV_ERR_OOB);
    }
    if (s < 0) {
      pdl_wait();   // (every thread block waits: this grid completes after the previous one)
      return;
    }
  } else {
    s = slots[t];
    if (s < 0) return;
    if (s >= num_slots) {
      if (threadIdx.x == 0) record_error(err, PKV_ERR_OOB);
      return;
    }
  }
  const int which = threadIdx.x >> 7;   // 0: K, 1: V
  const int ht = threadIdx.x & 127;
  const int64_t slab = (s / kBlockSize) * n_heads + h;
  const int row = static_cast<int>(s % kBlockSize);
  const int count = (row + 1) * d;
  const float4 prm = params[slab];
  uint8_t* codes = (which ? v_codes : k_codes) + slab * kBlockSize * d;
  const float lo_old = which ? prm.z : prm.x, hi_old = which ? prm.w : prm.y;
  const void* src = which ? v_new : k_new;
  uint8_t q[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int i = ht + k * 128;
    q[k] = (i < row * d) ? codes[which ? v_code_index(i, d) : i] : 0;
  }
  float x[kPer];
  float lo = INFINITY, hi = -INFINITY;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int i = ht + k * 128;
    x[k] = 0.f;
    if (i < count) {
      x[k] = (i >= row * d) ? in_f32(src, (t * n_heads + h) * d + (i - row * d), IN{})
                            : int8_decode_f32(q[k], lo_old, hi_old);
      lo = fminf(lo, x[k]);
      hi = fmaxf(hi, x[k]);
    }
  }
  // (each thread rewrites only the codes it read, so no barrier is needed
  // between the reads and the writes)
  const float2 mm = half_minmax(lo, hi, scratch, which);
  if constexpr (FROM_TABLE) pdl_wait();   // (the previous decode may still read this slab)
  const float span = __fsub_rn(mm.y, mm.x);
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int i = ht + k * 128;
    if (i < count) codes[which ? v_code_index(i, d) : i] = int8_code(x[k], mm.x, span);
  }
  if (ht == 0) lohi_out[which] = mm;
  __syncthreads();
  if (threadIdx.x == 0)
    params[slab] = make_float4(lohi_out[0].x, lohi_out[0].y, lohi_out[1].x, lohi_out[1].y);
}

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_kv_quantize_int8(const void* k_src, const void* v_src, uint8_t* k_cache, uint8_t* v_cache,
                                           float* slab_params, const int32_t* rows_used, int64_t num_blocks,
                                           int num_kv_heads, int head_dim, int block_size, pkv_dtype src_dtype,
                                           int32_t* err_flag, void* stream) {
  (void)err_flag;
  if (num_blocks < 0 || num_kv_heads <= 0) return PKV_ERR_INVALID_ARG;
  if (src_dtype != PKV_F16 && src_dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (block_size != kBlockSize || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
  if (num_blocks == 0) return PKV_OK;
  if (!k_src || !v_src || !k_cache || !v_cache || !slab_params || (reinterpret_cast<uintptr_t>(slab_params) & 15u))
    return PKV_ERR_INVALID_ARG;
  const int64_t slabs = num_blocks * num_kv_heads;
  if (slabs > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  auto kern = src_dtype == PKV_F16 ? quantize_int8_kernel<F16> : quantize_int8_kernel<BF16>;
  const cudaError_t e = launch_pdl(kern, dim3(static_cast<unsigned>(slabs)), dim3(kQThreads), 0,
                                   static_cast<cudaStream_t>(stream), k_src, v_src, k_cache, v_cache,
                                   reinterpret_cast<float4*>(slab_params), rows_used, num_kv_heads, head_dim);
  return cuda_failed(e, "quantize_int8_kernel launch") ? PKV_ERR_CUDA : PKV_OK;
}

extern "C" pkv_status pkv_kv_append_int8(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                         int64_t num_tokens, uint8_t* k_cache, uint8_t* v_cache, float* slab_params,
                                         int64_t num_blocks, int num_kv_heads, int head_dim, int block_size,
                                         pkv_dtype in_dtype, int32_t* err_flag, void* stream) {
  if (num_tokens < 0 || num_blocks < 0 || num_kv_heads <= 0) return PKV_ERR_INVALID_ARG;
  if (in_dtype != PKV_F16 && in_dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (block_size != kBlockSize || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache || !slab_params ||
      ((reinterpret_cast<uintptr_t>(slab_params) | reinterpret_cast<uintptr_t>(k_cache) |
        reinterpret_cast<uintptr_t>(v_cache)) & 15u))
    return PKV_ERR_INVALID_ARG;
  if (num_tokens * num_kv_heads > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  auto kern = in_dtype == PKV_F16 ? append_int8_kernel<F16, false> : append_int8_kernel<BF16, false>;
  const cudaError_t e = launch_pdl(kern, dim3(static_cast<unsigned>(num_tokens * num_kv_heads)), dim3(kQThreads), 0,
                                   static_cast<cudaStream_t>(stream), k_new, v_new, slot_mapping, k_cache, v_cache,
                                   reinterpret_cast<float4*>(slab_params), num_blocks * kBlockSize, num_kv_heads,
                                   head_dim, err_flag, TableSlots{});
  return cuda_failed(e, "append_int8_kernel launch") ? PKV_ERR_CUDA : PKV_OK;
}

namespace pkv {

// the append of the INT8 decode step: one new token per sequence at
// position context_lens[b] - 1, slots from the block table (arguments checked
// by the caller)
pkv_status launch_append_int8_step(const void* k_new, const void* v_new, uint8_t* k_cache, uint8_t* v_cache,
                                   float* slab_params, const int32_t* block_tables, const int32_t* context_lens,
                                   int batch, int max_blocks_per_seq, int64_t num_blocks, int num_kv_heads,
                                   int head_dim, pkv_dtype in_dtype, int64_t* slots_out, int32_t* err_flag,
                                   cudaStream_t stream) {
  if (static_cast<int64_t>(batch) * num_kv_heads > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  auto kern = in_dtype == PKV_F16 ? append_int8_kernel<F16, true> : append_int8_kernel<BF16, true>;
  const TableSlots ts{block_tables, context_lens, max_blocks_per_seq, slots_out};
  const cudaError_t e = launch_pdl(kern, dim3(static_cast<unsigned>(batch * num_kv_heads)), dim3(kQThreads), 0,
                                   stream, k_new, v_new, static_cast<const int64_t*>(nullptr), k_cache, v_cache,
                                   reinterpret_cast<float4*>(slab_params), num_blocks * kBlockSize, num_kv_heads,
                                   head_dim, err_flag, ts);
  return cuda_failed(e, "append_int8_kernel launch") ? PKV_ERR_CUDA : PKV_OK;
}

}  // namespace pkv
