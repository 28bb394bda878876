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
// the tensor cores read.  Per key tile:
//   S = Q K^T     tcgen05.mma kind::f16, M = N = 128, 8 k-steps of 16, fp32 in TMEM
//   softmax       8 warps, two threads per row (warps w and w + 4 share TMEM
//                 lane quarter w % 4; each takes 64 of the 128 columns and both
//                 take the row maximum over all of them): tcgen05.ld of S, mask,
//                 online max / sum in the log2 domain, P stored to shared
//                 memory in the input type (K-major, swizzled); when a row's
//                 max grows its O row in TMEM is rescaled (ld, scale, st)
//   O += P V      tcgen05.mma with V as an MN-major operand (keys x head_dim as
//                 staged), fp32 in TMEM.  bf16 keeps only 8 significant bits,
//                 so for bf16 P is split into P_hi = bf16(p) and
//                 P_lo = bf16(p - P_hi) and both are multiplied (two MMA
//                 passes): P is then exact to ~2^-17 relative, where a single
//                 bf16 rounding (2^-9) could exceed the 2e-3 tolerance on
//                 outputs of a few keys.  fp16 P (2^-12) needs one pass.
// Warp roles: warps 0-7 softmax and epilogue, warp 8 TMA producer (a 2-stage
// ring with separate K and V barriers: K of tile j + 2 is loaded as soon as
// Q K^T of tile j is done, V once P V of tile j is), warp 9 TMEM owner and
// MMA issuer (one elected lane).  S has two
// TMEM buffers: the MMA warp issues Q K^T of tile j+1 before it waits for the
// softmax of tile j, so the tensor cores compute the next scores while the
// softmax warps work.  Every wait
// is bounded; on expiry the block records PKV_ERR_TIMEOUT, drains what it has
// in flight and frees its TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

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
constexpr int kTile = kPM * kPD * 2;      // bytes of a 128 x 128 16-bit tile (Q, P, K or V)
constexpr int kPThreads = 320;           // 8 softmax warps, 1 TMA warp, 1 MMA warp
constexpr int kSoftmax = 256;            // softmax threads: 2 per query row
constexpr int kTmemCols = 512;            // S of even tiles: 0-127, O: 128-255, S of odd tiles: 256-383
constexpr size_t kPrefillSmem = 7 * static_cast<size_t>(kTile) + 256 + 1024;

// offsets in the 1024-aligned shared block: Q | P (hi part) | P (lo part) | K0 V0 | K1 V1 | barriers
constexpr int kOffQ = 0, kOffP = kTile, kOffPlo = 2 * kTile;
constexpr int kOffKV = 3 * kTile;   // stage s: K at kOffKV + 2 s kTile, V after it
constexpr int kOffBar = 7 * kTile;

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

// arrive on `bar` once every tcgen05 operation issued so far by this thread has completed
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
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
  extern __shared__ unsigned char psm_raw[];
  unsigned char* sm = psm_raw + ((1024 - (smem_u32(psm_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint64_t* k_full = bars;           // [2] per stage: K of the stage's tile landed
  uint64_t* v_full = bars + 2;       // [2] V landed
  uint64_t* k_empty = bars + 4;      // [2] Q K^T of the stage's tile done: K may be reloaded
  uint64_t* v_empty = bars + 6;      // [2] P V done: V may be reloaded
  uint64_t* s_full = bars + 8;       // [2], one per S buffer
  uint64_t* p_full = bars + 10;      // kSoftmax arrivals
  uint64_t* pv_done = bars + 11;
  uint64_t* q_ready = bars + 12;     // kSoftmax arrivals
  uint64_t* mma_idle = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 15);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);   // longest tiles first
  const int g = blockIdx.y, b = blockIdx.z;
  pdl_wait_and_release();

  const int cu0 = p.cu_seqlens[b];
  const int n_new = p.cu_seqlens[b + 1] - cu0;
  const int ctx = p.context_lens[b];
  const int i0 = qt * TPT;
  if (i0 >= n_new) return;                            // whole block: no tile here
  const int i1 = min(n_new, i0 + TPT);
  const int q_start = ctx - n_new;                    // position of new token 0
  if (q_start < 0 || ctx > p.max_blocks_per_seq * kBlockSize) {
    if (tid == 0) record_error(p.err, PKV_ERR_OOB);
    return;
  }
  const int last_pos = q_start + i1 - 1;
  const int n_tiles = last_pos / kPN + 1;
  const int nblk = (ctx + kBlockSize - 1) / kBlockSize;

  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, kSoftmax);
    mbar_init(pv_done, 1);
    mbar_init(q_ready, kSoftmax);
    mbar_init(mma_idle, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_o = tmem + kPN;
  auto t_s = [&](int j) -> uint32_t { return tmem + ((j & 1) ? 2 * kPN : 0); };

  if (warp < 8) {
    // ============================ softmax / epilogue ============================
    const int r = tid & (kPM - 1);                     // row = TMEM lane
    const int half = tid >> 7;                         // columns [64 half, 64 half + 64) of S, P and O
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
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
      // waits are made warp-uniform: the tcgen05.ld / st below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[j & 1], (j >> 1) & 1, p.err))) { ok = false; break; }
      tc_fence_after();
      // Two passes over the S row in chunks of 32 columns, re-read from TMEM
      // (a compact loop: the fully unrolled row did not fit the instruction
      // cache).  Only tiles that reach past a row's position need the mask.
      const bool masked = __any_sync(0xffffffffu, j * kPN + kPN - 1 > pos);   // (for pass 1; pass 2 re-tests)
      float mx = -INFINITY;
#pragma unroll 1
      for (int c0 = 0; c0 < kPN; c0 += 32) {
        float v[32];
        tmem_ld32(t_s(j) + lane_base + c0, v);
        if (masked) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = (j * kPN + c0 + i <= pos) ? v[i] : -INFINITY;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) mx = fmaxf(mx, v[i]);
      }
      // scores in the log2 domain: s * scale * log2(e) (the scale is positive,
      // so the maximum commutes with it)
      const float m_new = fmaxf(m_run, mx * p.qk_scale_log2);
      const float ref = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2_approx(m_run - ref);
      // O and the P buffer are free once the previous p.V has completed
      if (j > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(pv_done, (j - 1) & 1, p.err))) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 32) {
            float o[32];
            tmem_ld32(t_o + lane_base + c0, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(t_o + lane_base + c0, o);
          }
        }
      }
      constexpr bool kSplit = std::is_same<QT, BF16>::value;
      float psum = 0.f;
      const float nref = -ref;
#pragma unroll 1
      for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 32) {
        float v[32];
        tmem_ld32(t_s(j) + lane_base + c0, v);
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float e0 = ex2_approx(fmaf(v[i], p.qk_scale_log2, nref));
          float e1 = ex2_approx(fmaf(v[i + 1], p.qk_scale_log2, nref));
          if (masked) {
            e0 = (j * kPN + c0 + i <= pos) ? e0 : 0.f;
            e1 = (j * kPN + c0 + i + 1 <= pos) ? e1 : 0.f;
          }
          psum += e0 + e1;
          hi[i / 2] = pack2(e0, e1, QT{});
          if constexpr (kSplit) {
            const float2 b = unpack2(hi[i / 2], QT{});
            lo[i / 2] = pack2(e0 - b.x, e1 - b.y, QT{});
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t off = tile_off(r, c0 / 8 + c);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(sm + kOffP) + off),
                       "r"(hi[4 * c]), "r"(hi[4 * c + 1]), "r"(hi[4 * c + 2]), "r"(hi[4 * c + 3])
                       : "memory");
          if constexpr (kSplit)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(sm + kOffPlo) + off),
                         "r"(lo[4 * c]), "r"(lo[4 * c + 1]), "r"(lo[4 * c + 2]), "r"(lo[4 * c + 3])
                         : "memory");
        }
      }
      // l sums the fp32 weights (the multiplied hi + lo, or fp16, parts match
      // them to ~2^-17 / 2^-12 relative)
      l_run = l_run * alpha + psum;
      m_run = m_new;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (!ok) *abort_flag = 1;
    // epilogue: out = O / l.  The two threads of a row hold the sums of their
    // halves; they meet in the P buffer, free once the last p.V is done.
    ok = __all_sync(0xffffffffu, ok);
    const bool fin = ok && __all_sync(0xffffffffu, mbar_wait(pv_done, (n_tiles - 1) & 1, p.err));
    float* lx = reinterpret_cast<float*>(sm + kOffP);
    lx[half * kPM + r] = l_run;
    named_bar_sync(1, kSoftmax);
    const float l_tot = l_run + lx[(1 - half) * kPM + r];
    if (fin) {
      tc_fence_after();
      const float inv = (l_tot > 0.f) ? 1.f / l_tot : 0.f;
      auto* dst = reinterpret_cast<uint4*>(static_cast<typename QT::storage*>(p.out) +
                                           ((static_cast<int64_t>(cu0) + tok) * p.n_q_heads + head) * kPD);
#pragma unroll 1
      for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 32) {
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
    int j = 0, issued_k = 0, issued_v = 0;
    for (; j < n_tiles && !*abort_flag; ++j) {
      const int s = j & 1;
      int id = -1;
      if (lane < kPN / kBlockSize) {
        const int blk = j * (kPN / kBlockSize) + lane;
        id = (blk < nblk) ? row[blk] : -1;
        if (blk < nblk && (id < 0 || id >= p.num_blocks)) {
          record_error(p.err, PKV_ERR_OOB);
          id = -1;
        }
      }
      // a block past the context (or a bad id) is read from rows outside the
      // tensor, which TMA fills with zeros
      const int y = (id >= 0) ? (id * p.n_kv_heads + g) * kBlockSize : -2 * kBlockSize;
      unsigned char* kd = sm + kOffKV + 2 * s * kTile + lane * 2048;
      unsigned char* vd = kd + kTile;
      // K, then V, each after its previous use in this stage is done
      if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(&k_empty[s], ((j >> 1) - 1) & 1, p.err))) {
        *abort_flag = 1;
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&k_full[s], kTile);
      __syncwarp();
      if (lane < kPN / kBlockSize) {
#pragma unroll
        for (int h = 0; h < 2; ++h) tma_load_2d(kd + h * (kTile / 2), &p.tmap_k, h * 64, y, &k_full[s], pol);
      }
      __syncwarp();
      issued_k = j + 1;
      if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(&v_empty[s], ((j >> 1) - 1) & 1, p.err))) {
        *abort_flag = 1;
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&v_full[s], kTile);
      __syncwarp();
      if (lane < kPN / kBlockSize) {
#pragma unroll
        for (int h = 0; h < 2; ++h) tma_load_2d(vd + h * (kTile / 2), &p.tmap_v, h * 64, y, &v_full[s], pol);
      }
      __syncwarp();
      issued_v = j + 1;
    }
    if (*abort_flag && lane == 0) {
      // loads this warp issued that nobody consumed: wait for them (bounded)
      const unsigned long long deadline = global_ns() + kWaitLimitNs;
      for (int jj = max(0, issued_k - 2); jj < issued_k; ++jj)
        mbar_wait_until(&k_full[jj & 1], (jj >> 1) & 1, deadline);
      for (int jj = max(0, issued_v - 2); jj < issued_v; ++jj)
        mbar_wait_until(&v_full[jj & 1], (jj >> 1) & 1, deadline);
    }
  } else {
    // ============================ MMA issuer (warp 5) ============================
    const uint32_t sq = smem_u32(sm + kOffQ), sp = smem_u32(sm + kOffP), splo = smem_u32(sm + kOffPlo);
    constexpr int kPasses = std::is_same<QT, BF16>::value ? 2 : 1;   // P_hi, then P_lo
    constexpr uint32_t kIdQK = umma_idesc<QT>(false), kIdPV = umma_idesc<QT>(true);
    bool ok = true;
    if (lane == 0) ok = mbar_wait(q_ready, 0, p.err);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    // S = Q K^T of tile j into S buffer j & 1 (its previous tile's softmax has
    // finished reading it: the p_full wait of that tile came before)
    auto issue_qk = [&](int j) -> bool {
      const int s = j & 1;
      bool good = true;
      if (lane == 0) good = mbar_wait(&k_full[s], (j >> 1) & 1, p.err);
      good = __shfl_sync(0xffffffffu, good, 0);
      if (good && lane == 0) {
        const uint32_t sk = smem_u32(sm + kOffKV + 2 * s * kTile);
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kPD / 16; ++ks) {
          const uint32_t koff = (ks >> 2) * (kTile / 2) + (ks & 3) * 32;
          umma_f16(t_s(j), umma_desc(sq + koff, 16, 1024), umma_desc(sk + koff, 16, 1024), kIdQK, ks > 0);
        }
        umma_commit(&s_full[s]);
        umma_commit(&k_empty[s]);
      }
      __syncwarp();
      return good;
    };
    if (ok && n_tiles > 0) ok = issue_qk(0);
    for (int j = 0; j < n_tiles && ok && !*abort_flag; ++j) {
      const int s = j & 1;
      const uint32_t sv = smem_u32(sm + kOffKV + 2 * s * kTile) + kTile;
      if (j + 1 < n_tiles && !issue_qk(j + 1)) {
        ok = false;
        break;
      }
      if (lane == 0) ok = mbar_wait(p_full, j & 1, p.err) && mbar_wait(&v_full[s], (j >> 1) & 1, p.err);
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
#pragma unroll
        for (int pass = 0; pass < kPasses; ++pass)
#pragma unroll
          for (int ks = 0; ks < kPN / 16; ++ks) {
            const uint32_t poff = (ks >> 2) * (kTile / 2) + (ks & 3) * 32;
            umma_f16(t_o, umma_desc((pass ? splo : sp) + poff, 16, 1024),
                     umma_desc(sv + ks * 2048, kTile / 2, 1024), kIdPV, j > 0 || ks > 0 || pass > 0);
          }
        umma_commit(pv_done);
        umma_commit(&v_empty[s]);
      }
      __syncwarp();
    }
    if (!ok) *abort_flag = 1;
    // every MMA this thread issued has completed before TMEM is released
    if (lane == 0) {
      umma_commit(mma_idle);
      mbar_wait(mma_idle, 0, p.err);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
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
  const dim3 grid(static_cast<unsigned>(q_tiles), static_cast<unsigned>(p.n_kv_heads),
                  static_cast<unsigned>(p.batch));
  return cuda_failed(launch_pdl(kern, grid, dim3(kPThreads), kPrefillSmem, stream, p), "paged_prefill_kernel launch")
             ? PKV_ERR_CUDA
             : PKV_OK;
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
