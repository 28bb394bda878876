// Device-side helpers shared by the paged KV-cache kernels (sm_103a).
//
// * mbarrier / 1-D bulk-copy (TMA) wrappers in inline PTX.  Every wait is
//   bounded by the global timer: a wait that runs past kWaitLimitNs records
//   PKV_ERR_TIMEOUT in the caller's error word and returns false, so no kernel
//   here can spin forever.
// * 16-bit / E4M3 / E5M2 -> fp32 conversions, the fp32 -> FP8 encoders and
//   the fp32 -> 16-bit output rounding.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

constexpr int kBlockSize = 16;                       // tokens per physical block
constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // 1 s per wait
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// error word: the first error code wins; later ones are dropped
// ---------------------------------------------------------------------------
__device__ __forceinline__ void record_error(int32_t* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// shared-memory addresses and mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// make the initialised barriers visible to the async (TMA) proxy
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and
// records PKV_ERR_TIMEOUT) if it has not completed within limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* err,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > limit_ns) {
      record_error(err, PKV_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// L2 policy for data read exactly once (private KV blocks)
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes must be a
// multiple of 16 and both addresses 16-byte aligned)
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 1-D bulk copy shared -> global, tracked by bulk groups of the issuing thread
__device__ __forceinline__ void bulk_s2g(void* dst_gmem, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst_gmem),
               "r"(smem_u32(src_smem)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most N of this thread's bulk groups still read shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// wait until at most N of this thread's bulk groups are still in flight
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// 2-D tiled TMA load of a [16 x 128 B] box at (x elements, y rows)
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// named barrier among a subset of warps (id 0 is __syncthreads)
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// named barrier that also ORs a predicate over the participating threads, so
// every participant takes the same decision
__device__ __forceinline__ bool named_bar_red_or(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, "
      "q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}

// Wait for a phase until an absolute global-timer deadline (used when draining
// copies before exit); returns false on expiry without recording an error.
__device__ __forceinline__ bool mbar_wait_until(uint64_t* bar, uint32_t parity, unsigned long long deadline) {
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() > deadline) return false;
  }
  return true;
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: kernels of one decode step are launched so
// that the next kernel's launch overlaps this one's tail.  A kernel waits for
// its predecessor's completion (and memory) before it touches global data the
// predecessor may read or write, and lets its own successor start launching
// once that is safe (pdl_release).  A kernel that writes the KV cache, the
// block tables or the lengths releases its successor only after those writes
// are fenced (or not at all: then at its completion), so a decode kernel may
// read those inputs before its own wait.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_and_release() {
  pdl_wait();
  pdl_release();
}

// ---------------------------------------------------------------------------
// element conversions
// ---------------------------------------------------------------------------
struct F16 {
  using storage = __half;
  static constexpr int kBytes = 2;
};
struct BF16 {
  using storage = __nv_bfloat16;
  static constexpr int kBytes = 2;
};
struct E4M3 {
  using storage = uint8_t;
  static constexpr int kBytes = 1;
};
// OCP E5M2: bias 15, two mantissa bits -- the upper byte of an IEEE half
struct E5M2 {
  using storage = uint8_t;
  static constexpr int kBytes = 1;
};
// INT8 codes with per-(block, head) min-max scaling: x = min + q (max - min) / 255
struct U8 {
  using storage = uint8_t;
  static constexpr int kBytes = 1;
};

// two packed 16-bit values -> two floats
__device__ __forceinline__ float2 unpack2(uint32_t w, F16) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}
__device__ __forceinline__ float2 unpack2(uint32_t w, BF16) {
  // bf16 is the upper half of an fp32: shifting is an exact conversion
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// two packed E4M3 codes (low byte first) -> two floats, exactly
__device__ __forceinline__ float2 unpack2_e4m3(uint16_t w) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(w));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// two packed E5M2 codes (low byte first) -> packed f16x2, exactly: each code
// is the upper byte of the half with the same value
__device__ __forceinline__ uint32_t e5m2x2_to_f16x2(uint32_t w) { return __byte_perm(w, 0u, 0x1404u); }
__device__ __forceinline__ float2 unpack2_e5m2(uint32_t w) {
  const uint32_t h2 = e5m2x2_to_f16x2(w);
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// 8 consecutive elements of a row -> 8 floats
__device__ __forceinline__ void load8(const void* p, float* f, F16) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  float2 a = unpack2(v.x, F16{}), b = unpack2(v.y, F16{}), c = unpack2(v.z, F16{}), d = unpack2(v.w, F16{});
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}
__device__ __forceinline__ void load8(const void* p, float* f, BF16) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  float2 a = unpack2(v.x, BF16{}), b = unpack2(v.y, BF16{}), c = unpack2(v.z, BF16{}), d = unpack2(v.w, BF16{});
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}
__device__ __forceinline__ void load8(const void* p, float* f, E4M3) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  float2 a = unpack2_e4m3(static_cast<uint16_t>(v.x & 0xffffu));
  float2 b = unpack2_e4m3(static_cast<uint16_t>(v.x >> 16));
  float2 c = unpack2_e4m3(static_cast<uint16_t>(v.y & 0xffffu));
  float2 d = unpack2_e4m3(static_cast<uint16_t>(v.y >> 16));
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

__device__ __forceinline__ void load8(const void* p, float* f, E5M2) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  float2 a = unpack2_e5m2(v.x & 0xffffu), b = unpack2_e5m2(v.x >> 16);
  float2 c = unpack2_e5m2(v.y & 0xffffu), d = unpack2_e5m2(v.y >> 16);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

// eight INT8 codes -> their integer values as floats (exact: 2^23 + q has q
// in the low mantissa bits)
__device__ __forceinline__ void load8(const void* p, float* f, U8) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w = i < 4 ? v.x : v.y;
    f[i] = __uint_as_float(0x4B000000u | ((w >> (8 * (i & 3))) & 0xffu)) - 8388608.0f;
  }
}

// two floats -> two FP8 codes (lo in the low byte), round to nearest even,
// magnitudes above the largest finite value (448 for E4M3, 57344 for E5M2)
// clamp to it
__device__ __forceinline__ uint32_t fp8x2_from_f32(float lo, float hi, E4M3) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t fp8x2_from_f32(float lo, float hi, E5M2) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// 8 consecutive 16-bit elements -> 8 FP8 codes (format FMT) of fl32(x) /
// scale (IEEE division, not a reciprocal multiply), packed low byte first
template <typename FMT, typename IN>
__device__ __forceinline__ uint2 quant8_fp8(const void* src, float scale, IN) {
  float x[8];
  load8(src, x, IN{});
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    w[e] = fp8x2_from_f32(__fdiv_rn(x[2 * e], scale), __fdiv_rn(x[2 * e + 1], scale), FMT{});
  return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// two floats -> packed 16-bit pair (lo in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack2(float lo, float hi, BF16) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi, F16) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// INT8 per-block min-max codes: q = round((x - lo) / (hi - lo) * 255) in
// float32 in that order (IEEE rounding, no contraction), half to even,
// clamped to [0, 255]; hi == lo gives 0.  Decoding before a re-quantisation:
// lo + ((q * (hi - lo)) / 255).
__device__ __forceinline__ uint8_t int8_code(float x, float lo, float span) {
  if (span == 0.f) return 0;
  const float t = __fmul_rn(__fdiv_rn(__fsub_rn(x, lo), span), 255.f);
  return static_cast<uint8_t>(fminf(fmaxf(rintf(t), 0.f), 255.f));
}
__device__ __forceinline__ float int8_decode_f32(uint32_t q, float lo, float hi) {
  const float span = __fsub_rn(hi, lo);
  return __fadd_rn(lo, __fdiv_rn(__fmul_rn(static_cast<float>(q), span), 255.f));
}
// column of token r (0..15) in a transposed INT8 V slab row (head_dim 128)
__host__ __device__ __forceinline__ constexpr int int8_vt_column(int r) {
  return 4 * ((r & 7) >> 1) + 2 * (r >> 3) + (r & 1);
}

// fp32 -> output element, round to nearest even
__device__ __forceinline__ __half to_out(float x, F16) { return __float2half_rn(x); }
__device__ __forceinline__ __nv_bfloat16 to_out(float x, BF16) { return __float2bfloat16_rn(x); }

}  // namespace pkv
