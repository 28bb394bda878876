// Paged prefill / extend attention on the 5th-generation tensor cores (sm_103a).
//
// What is computed ("KV Cache, the memory notepad of LLM inference", sections
// 二-四: prefill attention over the prompt; "Series 03: why the KV cache eats
// memory, and how PagedAttention pages it", section 3.1: K/V through the block
// table, section 5.1: chunked prefill).  The new tokens of sequence b are its
// last n_b = cu_seqlens[b+1] - cu_seqlens[b] positions; token i sits at
// position p = context_lens[b] - n_b + i and attends causally:
//   out[cu_seqlens[b] + i, h] = sum_{j <= p} softmax_j(scale <q, K_j>) V_j
// with K_j, V_j of KV head h / G read from the paged cache, which already holds
// the new tokens' rows.
//
// Tiling.  A thread block owns one (sequence, KV head, query tile): 128 rows,
// each a (token, query head of the group) pair, token-major (row r = token
// r / G, head r % G), so one K/V tile serves the whole GQA group.  Key tiles
// are 128 keys = 8 cache blocks, gathered through the block table by tiled TMA
// loads of [16 rows x 128 B] boxes into the 128-byte swizzled K-major layout
// the tensor cores read.  Per key tile j:
//   S = Q K^T     tcgen05.mma kind::f16, M = N = 128, 8 k-steps of 16, fp32
//                 into TMEM buffer j % 3
//   softmax       8 warps, two threads per row (warps w and w + 4 share TMEM
//                 lane quarter w % 4, each owns 64 of the 128 columns): one
//                 tcgen05.ld of its columns, mask, partial row maximum, which
//                 the two threads of a row exchange through shared memory;
//                 P = 2^(s scale log2 e - m) is written back into the same
//                 TMEM columns in the input type (tcgen05.st)
//   O += P V      tcgen05.mma with A = P read from TMEM and B = V as an
//                 MN-major shared-memory operand (keys x head_dim as staged),
//                 fp32 in TMEM.  bf16 keeps only 8 significant bits, so for
//                 bf16 P is split into P_hi (p truncated to bf16) and
//                 P_lo = bf16(p - P_hi) and both are multiplied (two MMA
//                 passes): P is then exact to ~2^-16 relative, where a single
//                 bf16 rounding (2^-9) could exceed the 2e-3 tolerance on
//                 outputs of a few keys.  fp16 P (2^-12) needs one pass.
//                 The softmax arithmetic runs on packed fp32 pairs.
// P overwrites its own S in TMEM: the 32 columns of each 32-key chunk hold its
// P_hi pairs in the first 16 and its P_lo pairs in the next 16, so a thread
// only ever writes columns it has already read.  With three S / P buffers the
// scores of tile j + 2 are computed while the softmax of tile j + 1 and the
// P V of tile j run.  The row reference m moves only when a tile's maximum
// exceeds it by more than 2^8 (P stays <= 256, exact in fp32 accumulation):
// only then is the O row rescaled, after the previous P V has completed, so
// in the steady state the softmax never waits for the tensor cores.
// Loads.  A TMA load of one 16-row block moves only about 25 B per clock per
// SM on GB300 (small boxes are request-bound), short of the ~42 B/clk the
// tensor cores consume here, so CTAs run in clusters of two that hold
// adjacent query tiles of the same (sequence, KV head): each loads half of the
// blocks of every K / V tile with multicast into both, and a ring stage is
// released by both CTAs' MMA commits (multicast to both).  Both run the key
// tiles of the longer query tile; the other's rows see the extra keys masked.
// Warp roles: warps 0-7 softmax and epilogue; warp 8 TMA producer (K in a
// 2-stage ring, V in a 3-stage one, issued in the order the MMAs consume
// them: V of tile j, then K of tile j + 2, with block-table entries read a
// tile ahead); warp 9 TMEM owner and Q K^T issuer, warp 10 P V issuer (one
// elected lane each: a commit holds its thread until the MMA queue has
// drained to a few entries, so two issuers keep the queue fed).  Every wait
// is bounded; on expiry the block records PKV_ERR_TIMEOUT, drains what it
// has in flight and frees its TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "../../include/pkv_prefill.h"
#include "host_util.h"
#include "pkv_common.cuh"

namespace pkv {

struct PrefillParams {
  CUtensorMap tmap_k;            // [NB * Hkv * 16 rows, D] 16-bit, [16 x 64] boxes, 128B swizzle
  CUtensorMap tmap_v;
  const void* q;                 // [T, Hq, D]
  void* out;                     // [T, Hq, D]
  const int32_t* block_tables;   // [B, max_blocks_per_seq]
  const int32_t* context_lens;   // [B] lengths after the new tokens
  const int32_t* cu_seqlens;     // [B + 1] new-token offsets
  int32_t* err;
  int64_t num_blocks;
  int batch;
  int n_q_heads;
  int n_kv_heads;
  int max_blocks_per_seq;
  float qk_scale_log2;           // softmax scale * log2(e)
};

constexpr int kPM = 128;                  // query rows per tile
constexpr int kPN = 128;                  // keys per tile
constexpr int kPD = 128;                  // head_dim
constexpr int kTile = kPM * kPD * 2;      // bytes of a 128 x 128 16-bit tile (Q, K or V)
constexpr int kPThreads = 352;           // 8 softmax warps, 1 TMA warp, 2 MMA warps
constexpr int kSoftmax = 256;            // softmax threads: 2 per query row
constexpr int kSBufs = 3;                 // S / P buffers in TMEM
constexpr int kCluster = 2;               // CTAs (adjacent query tiles) sharing each K / V tile load
constexpr int kKStages = 2, kVStages = 3; // K and V rings in shared memory
constexpr int kTmemCols = 512;            // S / P buffers at columns 0, 128, 256; O at 384
constexpr int kOCol = kSBufs * kPN;
constexpr float kRescaleLog2 = 8.f;      // the row reference moves when the max outgrows it by > 2^8

// offsets in the 1024-aligned shared block: Q | K ring | V ring | barriers | row exchange
constexpr int kOffQ = 0;
constexpr int kOffK = kTile;                          // stage s at kOffK + s kTile
constexpr int kOffV = kOffK + kKStages * kTile;       // stage s at kOffV + s kTile
constexpr int kOffBar = kOffV + kVStages * kTile;
constexpr int kBarWords = 2 * (kKStages + kVStages) + 3 * kSBufs + 3 + 2;   // barriers, TMEM slot, abort flag
static_assert(kBarWords * 8 <= 256, "barrier block overflows its 256 bytes");
constexpr int kOffRed = kOffBar + 256;                // float [3][2][128]: row maxima (2 slots), row sums
constexpr size_t kPrefillSmem = static_cast<size_t>(kOffRed) + 3 * 2 * kPM * 4 + 1024;

// ---------------------------------------------------------------------------
// tcgen05 helpers
// ---------------------------------------------------------------------------
// shared-memory matrix descriptor: start, leading / stride byte offsets, the
// fixed version field of this architecture, 128-byte swizzle
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFF) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// instruction descriptor of kind::f16: fp32 accumulate, A/B of one 16-bit type,
// A K-major, B K-major or MN-major, M = N = 128
template <typename QT>
__host__ __device__ constexpr uint32_t umma_idesc(bool b_mn_major) {
  return (1u << 4) | ((std::is_same<QT, BF16>::value ? 1u : 0u) << 7) |
         ((std::is_same<QT, BF16>::value ? 1u : 0u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(kPN >> 3) << 17) | (static_cast<uint32_t>(kPM >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(static_cast<uint32_t>(acc))
      : "memory");
}

// the same with A read from TMEM (lane m = row m, column c holding the 16-bit
// pair of k = 2c, 2c + 1 of the 16-wide k-step, low half first)
__device__ __forceinline__ void umma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(static_cast<uint32_t>(acc))
      : "memory");
}

// arrive on `bar` once every tcgen05 operation issued so far by this thread has completed
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// arrive on `bar` in both CTAs of the cluster (same shared offset) once every
// tcgen05 operation issued so far by this thread has completed
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(static_cast<uint16_t>((1u << kCluster) - 1))
      : "memory");
}

// tiled TMA load written to the same shared offset of every CTA of the cluster,
// completing on the barrier at `bar`'s offset in each
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5, %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)),
      "h"(static_cast<uint16_t>((1u << kCluster) - 1)),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ int cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return static_cast<int>(r);
}

// every thread of both CTAs of the cluster
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 2^x by the hardware approximation (relative error about 2^-22; 2^-inf = 0)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 16 / 32 consecutive 32-bit columns of this thread's TMEM lane (no wait)
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// 64 consecutive 32-bit columns of this thread's TMEM lane in one store (no wait)
__device__ __forceinline__ void tmem_st64u(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]), "r"(v[32]), "r"(v[33]), "r"(v[34]), "r"(v[35]), "r"(v[36]), "r"(v[37]), "r"(v[38]), "r"(v[39]), "r"(v[40]), "r"(v[41]), "r"(v[42]), "r"(v[43]), "r"(v[44]), "r"(v[45]), "r"(v[46]), "r"(v[47]), "r"(v[48]), "r"(v[49]), "r"(v[50]), "r"(v[51]), "r"(v[52]), "r"(v[53]), "r"(v[54]), "r"(v[55]), "r"(v[56]), "r"(v[57]), "r"(v[58]), "r"(v[59]), "r"(v[60]), "r"(v[61]), "r"(v[62]), "r"(v[63])
               : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 64 consecutive fp32 columns of this thread's TMEM lane: one load, one wait.
// The wait names the loaded registers as operands so that no use of them is
// scheduled before it.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
  asm volatile(""
               : "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]), "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63])
               :
               : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// packed fp32 pairs (the f32x2 instructions of this architecture)
__device__ __forceinline__ uint64_t f32x2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f32x2_split(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// maximum of 64 values: eight independent chains, then a short tree
__device__ __forceinline__ float max64(const float* v) {
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float* x = v + 8 * k;
    m[k] = fmaxf(fmax3(fmax3(x[0], x[1], x[2]), x[3], x[4]), fmax3(x[5], x[6], x[7]));
  }
  return fmax3(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

// byte offset of 16-byte chunk c (elements 8c..8c+7) of row r in a 128 x 128
// 16-bit tile stored K-major with the 128-byte swizzle: two 64-column halves of
// 16 KiB, 8-row atoms of 1 KiB, chunk index XOR row within the atom
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return (c >> 3) * (kTile / 2) + (r >> 3) * 1024 + (r & 7) * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <typename QT, int G>
__global__ void __launch_bounds__(kPThreads, 1) paged_prefill_kernel(const __grid_constant__ PrefillParams p) {
  constexpr int TPT = kPM / G;                       // tokens per query tile
  constexpr bool kSplit = std::is_same<QT, BF16>::value;
  extern __shared__ unsigned char psm_raw[];
  unsigned char* sm = psm_raw + ((1024 - (smem_u32(psm_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  // barrier array offsets follow the ring sizes (kBarWords words in all)
  uint64_t* k_full = bars;                    // [kKStages] K of the stage's tile landed
  uint64_t* k_empty = k_full + kKStages;      // [kKStages] Q K^T of the stage's tile done in both CTAs
  uint64_t* v_full = k_empty + kKStages;      // [kVStages] V landed
  uint64_t* v_empty = v_full + kVStages;      // [kVStages] P V done in both CTAs
  uint64_t* s_full = v_empty + kVStages;      // [3] per S / P buffer: scores ready
  uint64_t* p_full = s_full + kSBufs;         // [3] per buffer, kSoftmax arrivals: P written, O rescaled
  uint64_t* pv_done = p_full + kSBufs;        // [3] per buffer: P V of its tile done
  uint64_t* q_ready = pv_done + kSBufs;       // kSoftmax arrivals
  uint64_t* mma_idle = q_ready + 1;           // Q K^T issuer drained
  uint64_t* pv_idle = mma_idle + 1;           // P V issuer drained
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pv_idle + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(pv_idle + 2);
  float* red = reinterpret_cast<float*>(sm + kOffRed);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);   // longest tiles first
  const int g = blockIdx.y, b = blockIdx.z;
  pdl_wait_and_release();

  const int cu0 = p.cu_seqlens[b];
  const int n_new = p.cu_seqlens[b + 1] - cu0;
  const int ctx = p.context_lens[b];
  const int q_start = ctx - n_new;                    // position of new token 0
  // (the same decision in both CTAs of the cluster: they share the sequence)
  if (q_start < 0 || ctx > p.max_blocks_per_seq * kBlockSize) {
    if (tid == 0) record_error(p.err, PKV_ERR_OOB);
    return;
  }
  // The two CTAs of a cluster hold adjacent query tiles of one (sequence, KV
  // head): rank 0 the later one.  Each loads half of every K / V tile into
  // both, so both run the key tiles of the longer one (the shorter one's rows
  // see the extra keys masked).
  const int rank = cluster_rank();
  auto tiles_of = [&](int qtile) -> int {
    const int a = qtile * TPT;
    return (qtile < 0 || a >= n_new) ? 0 : (q_start + min(n_new, a + TPT) - 1) / kPN + 1;
  };
  int n_tiles = 0;   // the longest query tile of the cluster: rank r holds qt = qt_of_rank_0 - r
  for (int r = 0; r < kCluster; ++r) n_tiles = max(n_tiles, tiles_of(qt + rank - r));
  if (n_tiles == 0) return;                           // neither CTA holds a token
  const int i0 = qt * TPT;
  const int i1 = max(i0, min(n_new, i0 + TPT));       // i1 == i0: no rows of this CTA
  const int nblk = (ctx + kBlockSize - 1) / kBlockSize;

  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], kCluster);   // released by every CTA's MMAs
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], kCluster);
    }
    for (int s = 0; s < kSBufs; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], kSoftmax);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(q_ready, kSoftmax);
    mbar_init(mma_idle, 1);
    mbar_init(pv_idle, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers exist before any multicast write or remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_o = tmem + kOCol;
  auto t_s = [&](int j) -> uint32_t { return tmem + (j % kSBufs) * kPN; };

  if (warp < 8) {
    // ============================ softmax / epilogue ============================
    const int r = tid & (kPM - 1);                     // row = TMEM lane
    const int half = tid >> 7;                         // columns [64 half, 64 half + 64) of S and O
    const int pair_bar = 2 + (warp & 3);               // named barrier of warps w and w + 4 (one row each)
    const int tok = i0 + r / G, head = g * G + r % G;
    const bool row_live = tok < i1;
    const int pos = row_live ? q_start + tok : -1;
    // stage this row of Q (zeros for rows past the tile's tokens)
    {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(p.q) +
                                                        ((static_cast<int64_t>(cu0) + tok) * p.n_q_heads + head) *
                                                            kPD * 2);
#pragma unroll
      for (int c = 8 * half; c < 8 * half + 8; ++c) {
        const uint4 v = row_live ? src[c] : make_uint4(0, 0, 0, 0);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(sm + kOffQ) + tile_off(r, c)),
                     "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                     : "memory");
      }
      fence_proxy_async_smem();
      mbar_arrive(q_ready);
    }
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int col0 = 64 * half;
    float m_ref = -INFINITY, l_run = 0.f;
    bool ok = true;
    // A failed wait is published at the next row exchange, where both warps of
    // the pair see it and leave together (a warp must never leave its partner
    // waiting at the named barrier).
    for (int j = 0; j < n_tiles; ++j) {
      const int buf = j % kSBufs, ph = (j / kSBufs) & 1;
      const uint32_t ts = t_s(j) + lane_base + col0;
      if (ok) {
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[buf], ph, p.err));
        tc_fence_after();
      }
      float v[64];
      float mx = -INFINITY;
      if (ok) {
        tmem_ld64(ts, v);
        // only tiles reaching past a row's position need the causal mask
        if (__any_sync(0xffffffffu, j * kPN + kPN - 1 > pos)) {
#pragma unroll
          for (int i = 0; i < 64; ++i) v[i] = (j * kPN + col0 + i <= pos) ? v[i] : -INFINITY;
        }
        mx = max64(v);
        red[((j & 1) * 2 + half) * kPM + r] = mx;
      }
      if (named_bar_red_or(pair_bar, 64, !ok)) {
        ok = false;
        break;
      }
      mx = fmaxf(mx, red[((j & 1) * 2 + (1 - half)) * kPM + r]);
      // scores in the log2 domain: s * scale * log2(e) (the scale is positive,
      // so the maximum commutes with it).  The reference moves only when the
      // tile's maximum outgrows it by more than 2^8 (always on a row's first
      // unmasked tile, where m_ref = -inf and alpha = 0).
      const float m_tile = mx * p.qk_scale_log2;
      float alpha = 1.f;
      if (m_tile > m_ref + kRescaleLog2) {
        alpha = ex2_approx(m_ref - m_tile);
        m_ref = m_tile;
      }
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O may be touched once the previous tile's P V has completed
        const int pb = (j - 1) % kSBufs;
        if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[pb], ((j - 1) / kSBufs) & 1, p.err))) {
          ok = false;
          continue;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c0 = col0; c0 < col0 + 64; c0 += 32) {
          float o[32];
          tmem_ld32(t_o + lane_base + c0, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(t_o + lane_base + c0, o);
        }
      }
      // P over this thread's two 32-key chunks, written over the chunk's own
      // columns: 16 pairs of P_hi, then (bf16) 16 pairs of P_lo.  Masked scores
      // are -inf and give 2^-inf = 0.  For bf16, P_hi is p truncated to bf16
      // (its top 16 bits) and P_lo = bf16(p - P_hi), where p - P_hi is exact.
      const float nref = (m_ref == -INFINITY) ? 0.f : -m_ref;
      const uint64_t scale2 = f32x2(p.qk_scale_log2, p.qk_scale_log2), nref2 = f32x2(nref, nref);
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};   // (+0, +0) pairs
      uint32_t pk2[64];   // bf16: both chunks' columns, stored at once
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t* pk = pk2 + 32 * c;
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 x = f32x2_split(fma_f32x2(f32x2(v[32 * c + i], v[32 * c + i + 1]), scale2, nref2));
          const float e0 = ex2_approx(x.x), e1 = ex2_approx(x.y);
          const uint64_t e01 = f32x2(e0, e1);
          acc[(i / 2) & 3] = add_f32x2(acc[(i / 2) & 3], e01);
          if constexpr (kSplit) {
            const uint32_t b0 = __float_as_uint(e0), b1 = __float_as_uint(e1);
            pk[i / 2] = __byte_perm(b0, b1, 0x7632);
            const float2 lo = f32x2_split(
                sub_f32x2(e01, f32x2(__uint_as_float(b0 & 0xffff0000u), __uint_as_float(b1 & 0xffff0000u))));
            pk[16 + i / 2] = pack2(lo.x, lo.y, QT{});
          } else {
            pk[i / 2] = pack2(e0, e1, QT{});
          }
        }
        if constexpr (!kSplit) tmem_st16u(ts + 32 * c, pk);
      }
      if constexpr (kSplit) tmem_st64u(ts, pk2);
      const float2 s0 = f32x2_split(add_f32x2(add_f32x2(acc[0], acc[1]), add_f32x2(acc[2], acc[3])));
      const float psum = s0.x + s0.y;
      tmem_wait_st();
      // l sums the fp32 weights (the multiplied hi + lo, or fp16, parts match
      // them to ~2^-16 / 2^-12 relative)
      l_run = l_run * alpha + psum;
      tc_fence_before();
      mbar_arrive(&p_full[buf]);
    }
    if (!ok) *abort_flag = 1;
    // epilogue: out = O / l.  The two threads of a row add their halves' sums.
    ok = __all_sync(0xffffffffu, ok);
    const bool fin = ok && __all_sync(0xffffffffu, mbar_wait(&pv_done[(n_tiles - 1) % kSBufs],
                                                             ((n_tiles - 1) / kSBufs) & 1, p.err));
    float* lx = red + 4 * kPM;
    lx[half * kPM + r] = l_run;
    named_bar_sync(1, kSoftmax);
    const float l_tot = l_run + lx[(1 - half) * kPM + r];
    if (fin) {
      tc_fence_after();
      const float inv = (l_tot > 0.f) ? 1.f / l_tot : 0.f;
      auto* dst = reinterpret_cast<uint4*>(static_cast<typename QT::storage*>(p.out) +
                                           ((static_cast<int64_t>(cu0) + tok) * p.n_q_heads + head) * kPD);
#pragma unroll 1
      for (int c0 = col0; c0 < col0 + 64; c0 += 32) {
        float o[32];
        tmem_ld32(t_o + lane_base + c0, o);
        if (row_live) {
#pragma unroll
          for (int i = 0; i < 32; i += 8)
            dst[(c0 + i) / 8] = make_uint4(pack2(o[i] * inv, o[i + 1] * inv, QT{}),
                                           pack2(o[i + 2] * inv, o[i + 3] * inv, QT{}),
                                           pack2(o[i + 4] * inv, o[i + 5] * inv, QT{}),
                                           pack2(o[i + 6] * inv, o[i + 7] * inv, QT{}));
        }
      }
    } else {
      *abort_flag = 1;
    }
  } else if (warp == 8) {
    // ============================ TMA producer ============================
    const uint64_t pol = policy_evict_last();   // K/V tiles are re-read by the other query tiles
    const int32_t* row = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq;
    // block id of this lane's block of key tile j (-1 past the context), and
    // its cache row: a block past the context, or a bad id, is read from rows
    // outside the tensor, which TMA fills with zeros
    auto fetch_id = [&](int j) -> int {
      const int blk = j * (kPN / kBlockSize) + lane;
      return (lane < kPN / kBlockSize && blk < nblk) ? row[blk] : -1;
    };
    auto to_row = [&](int j, int id) -> int {
      const int blk = j * (kPN / kBlockSize) + lane;
      if (lane < kPN / kBlockSize && blk < nblk && (id < 0 || id >= p.num_blocks)) {
        record_error(p.err, PKV_ERR_OOB);
        id = -1;
      }
      return (id >= 0) ? (id * p.n_kv_heads + g) * kBlockSize : -2 * kBlockSize;
    };
    // load K (is_v = 0) or V of key tile j into its ring stage from cache row
    // y, after the stage's previous tile has been consumed
    int issued_k = 0, issued_v = 0;
    auto load = [&](int j, bool is_v, int y) -> bool {
      const int stages = is_v ? kVStages : kKStages;
      const int s = j % stages;
      uint64_t* full = is_v ? &v_full[s] : &k_full[s];
      uint64_t* empty = is_v ? &v_empty[s] : &k_empty[s];
      if (j >= stages && !__all_sync(0xffffffffu, mbar_wait(empty, ((j / stages) - 1) & 1, p.err))) return false;
      // the whole tile lands in this CTA: its own half and the peer's
      if (lane == 0) mbar_arrive_expect_tx(full, kTile);
      __syncwarp();
      if (lane < kPN / kBlockSize && lane / (kPN / kBlockSize / kCluster) == rank) {
        unsigned char* dst = sm + (is_v ? kOffV : kOffK) + s * kTile + lane * 2048;
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tma_load_2d_pair(dst + h * (kTile / 2), is_v ? &p.tmap_v : &p.tmap_k, h * 64, y, full, pol);
      }
      __syncwarp();
      (is_v ? issued_v : issued_k) = j + 1;
      return true;
    };
    // the order the MMAs consume them in: K0, K1, then V of tile j and K of
    // tile j + 2.  Block ids are fetched a tile ahead of their first use (r0,
    // r1 rows of tiles j, j + 1; id2 the raw id of tile j + 2), so the table's
    // latency is spent while the ring waits.
    int r0 = to_row(0, fetch_id(0)), r1 = (n_tiles > 1) ? to_row(1, fetch_id(1)) : 0;
    int id2 = (n_tiles > 2) ? fetch_id(2) : -1;
    bool good = load(0, false, r0) && (n_tiles < 2 || load(1, false, r1));
    for (int j = 0; good && j < n_tiles && !*abort_flag; ++j) {
      const int r2 = (j + 2 < n_tiles) ? to_row(j + 2, id2) : 0;
      if (j + 3 < n_tiles) id2 = fetch_id(j + 3);
      good = load(j, true, r0) && (j + 2 >= n_tiles || load(j + 2, false, r2));
      r0 = r1;
      r1 = r2;
    }
    if (!good) *abort_flag = 1;
    if (*abort_flag && lane == 0) {
      // loads this warp issued that nobody consumed: wait for them (bounded)
      const unsigned long long deadline = global_ns() + kWaitLimitNs;
      for (int jj = max(0, issued_k - kKStages); jj < issued_k; ++jj)
        mbar_wait_until(&k_full[jj % kKStages], (jj / kKStages) & 1, deadline);
      for (int jj = max(0, issued_v - kVStages); jj < issued_v; ++jj)
        mbar_wait_until(&v_full[jj % kVStages], (jj / kVStages) & 1, deadline);
    }
  } else {
    // ============================ MMA issuers (warps 9, 10) ============================
    // Warp 9 issues Q K^T, warp 10 P V, one elected lane each.  A commit holds
    // its thread until the MMA queue ahead of the tensor cores has drained to a
    // few MMAs; with two issuing threads one of them can feed the queue while
    // the other is held, and neither waits for the other's batches.
    constexpr int kPasses = kSplit ? 2 : 1;   // P_hi, then P_lo
    constexpr uint32_t kIdQK = umma_idesc<QT>(false), kIdPV = umma_idesc<QT>(true);
    const bool qk_warp = (warp == 9);
    uint64_t* idle = qk_warp ? mma_idle : pv_idle;
    bool ok = true;
    if (qk_warp) {
      const uint32_t sq = smem_u32(sm + kOffQ);
      if (lane == 0) ok = mbar_wait(q_ready, 0, p.err);
      // S = Q K^T of tile t into S buffer t % 3, once the P V of tile t - 3
      // (which read P from that buffer) has completed
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int s = t % kKStages;
        if (lane == 0) {
          ok = (t < kSBufs || mbar_wait(&pv_done[(t - kSBufs) % kSBufs], ((t - kSBufs) / kSBufs) & 1, p.err)) &&
               mbar_wait(&k_full[s], (t / kKStages) & 1, p.err) && !*abort_flag;
          if (ok) {
            // descriptors built once per tile; each k-step adds a compile-time
            // offset to the address field (addr >> 4, no carry out of its 14
            // bits for shared addresses below 256 KiB)
            const uint64_t a0 = umma_desc(sq, 16, 1024), b0 = umma_desc(smem_u32(sm + kOffK + s * kTile), 16, 1024);
            const uint32_t d = t_s(t);
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < kPD / 16; ++ks) {
              const uint64_t koff = static_cast<uint64_t>(((ks >> 2) * (kTile / 2) + (ks & 3) * 32) >> 4);
              umma_f16(d, a0 + koff, b0 + koff, kIdQK, ks > 0);
            }
            umma_commit(&s_full[t % kSBufs]);
            umma_commit_pair(&k_empty[s]);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
    } else {
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int buf = j % kSBufs, vs = j % kVStages;
        const uint32_t sv = smem_u32(sm + kOffV + vs * kTile);
        if (lane == 0)
          ok = mbar_wait(&p_full[buf], (j / kSBufs) & 1, p.err) && mbar_wait(&v_full[vs], (j / kVStages) & 1, p.err) &&
               !*abort_flag;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        // the tile holding the context's last, partial block: its rows past the
        // context have zero probability but may hold any bits; clear them in V
        const int tail = ctx % kBlockSize;
        if (tail != 0 && (nblk - 1) / (kPN / kBlockSize) == j) {
          const int slot = (nblk - 1) % (kPN / kBlockSize);
          for (int x = lane; x < (kBlockSize - tail) * 16; x += 32) {
            const int rr = slot * kBlockSize + tail + x / 16, c = x % 16;
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(sv + tile_off(rr, c)), "r"(0u) : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          tc_fence_after();
          // k-step ks takes keys 16 ks .. 16 ks + 15: chunk ks / 2, columns
          // 8 (ks % 2) of its P_hi half (pass 0) or P_lo half (pass 1)
          const uint64_t b0 = umma_desc(sv, kTile / 2, 1024);
          const uint32_t a0 = t_s(j);
#pragma unroll
          for (int pass = 0; pass < kPasses; ++pass)
#pragma unroll
            for (int ks = 0; ks < kPN / 16; ++ks)
              umma_f16_tmem_a(t_o, a0 + 32 * (ks >> 1) + 16 * pass + 8 * (ks & 1),
                              b0 + static_cast<uint64_t>((ks * 2048) >> 4), kIdPV, j > 0 || ks > 0 || pass > 0);
          umma_commit(&pv_done[buf]);
          umma_commit_pair(&v_empty[vs]);
        }
        __syncwarp();
      }
    }
    if (!ok) *abort_flag = 1;
    // every MMA this lane issued has completed before TMEM is released
    if (lane == 0) {
      umma_commit(idle);
      mbar_wait(idle, 0, p.err);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  // no multicast write or remote arrive of the peer is still in flight to this CTA
  cluster_sync();
  tc_fence_after();
  if (warp == 9)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

template <typename QT, int G>
pkv_status launch_prefill(PrefillParams& p, int q_tiles, cudaStream_t stream) {
  auto kern = paged_prefill_kernel<QT, G>;
  int dev = 0;
  if (cuda_failed(cudaGetDevice(&dev), "cudaGetDevice")) return PKV_ERR_CUDA;
  static std::mutex mu;
  static bool done[64] = {};
  if (dev < 0 || dev >= 64) return PKV_ERR_UNSUPPORTED;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
      if (cuda_failed(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kPrefillSmem)),
                      "cudaFuncSetAttribute"))
        return PKV_ERR_CUDA;
      done[dev] = true;
    }
  }
  // clusters of two CTAs along the query tiles (an even count), launched
  // with programmatic dependent launch like the other kernels
  const dim3 grid(static_cast<unsigned>((q_tiles + kCluster - 1) / kCluster * kCluster), static_cast<unsigned>(p.n_kv_heads),
                  static_cast<unsigned>(p.batch));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kPrefillSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cuda_failed(cudaLaunchKernelEx(&cfg, kern, p), "paged_prefill_kernel launch") ? PKV_ERR_CUDA : PKV_OK;
}

template <typename QT>
pkv_status launch_prefill_group(PrefillParams& p, int group, int max_query_len, cudaStream_t stream) {
  const int tpt = kPM / group;
  const int q_tiles = (max_query_len + tpt - 1) / tpt;
  switch (group) {
    case 1: return launch_prefill<QT, 1>(p, q_tiles, stream);
    case 2: return launch_prefill<QT, 2>(p, q_tiles, stream);
    case 4: return launch_prefill<QT, 4>(p, q_tiles, stream);
    case 8: return launch_prefill<QT, 8>(p, q_tiles, stream);
    default: return PKV_ERR_UNSUPPORTED;
  }
}

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_paged_prefill_attention(const void* q, const void* k_cache, const void* v_cache,
                                                  const int32_t* block_tables, const int32_t* context_lens,
                                                  const int32_t* cu_seqlens, int batch, int num_q_heads,
                                                  int num_kv_heads, int head_dim, int block_size,
                                                  int max_blocks_per_seq, int64_t num_blocks, int max_query_len,
                                                  float scale, void* out, pkv_dtype dtype, int32_t* err_flag,
                                                  void* stream) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0 || num_blocks < 0 ||
      max_query_len < 0 || !(scale == scale))
    return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads) return PKV_ERR_INVALID_ARG;
  if (block_size != kBlockSize || head_dim != kPD) return PKV_ERR_UNSUPPORTED;
  const int group = num_q_heads / num_kv_heads;
  if (group != 1 && group != 2 && group != 4 && group != 8) return PKV_ERR_UNSUPPORTED;
  if (batch == 0 || max_query_len == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !cu_seqlens || !out)
    return PKV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache)) & 15u)
    return PKV_ERR_INVALID_ARG;
  const int64_t rows = num_blocks * num_kv_heads * kBlockSize;
  if (rows > INT32_MAX || num_kv_heads > 65535 || batch > 65535) return PKV_ERR_UNSUPPORTED;
  PrefillParams p{};
  if (!encode_cache_tmap(&p.tmap_k, k_cache, rows, head_dim, 2) ||
      !encode_cache_tmap(&p.tmap_v, v_cache, rows, head_dim, 2))
    return PKV_ERR_CUDA;
  p.q = q;
  p.out = out;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.cu_seqlens = cu_seqlens;
  p.err = err_flag;
  p.num_blocks = num_blocks;
  p.batch = batch;
  p.n_q_heads = num_q_heads;
  p.n_kv_heads = num_kv_heads;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.qk_scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return dtype == PKV_F16 ? launch_prefill_group<F16>(p, group, max_query_len, s)
                          : launch_prefill_group<BF16>(p, group, max_query_len, s);
}
