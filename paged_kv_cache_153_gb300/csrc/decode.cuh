// Paged decode attention kernels (sm_103a).
//
// What is computed (per sequence b, query head h, KV head g = h / G):
//   out[b, h] = sum_{j < n_b} softmax_j(scale * <q[b, h], K_j>) V_j
// with K_j, V_j read through the block table ("Series 03: why the KV cache eats
// memory, and how PagedAttention pages it", section 3.1; the attention formula
// of "KV Cache, the memory notepad of LLM inference", section 二; GQA groups of
// its section 六).
//
// Work decomposition.  The (sequence, KV head, logical block) triples are laid
// out flat, sequence-major; thread block c owns range c of R = grid size: an
// equal share of a cost axis (balanced mode) or an equal share of the flat
// space's fixed partitions of `part_blocks` blocks (partition mode).  A range
// is cut into segments at (sequence, KV head) boundaries.  A segment holding a
// whole (sequence, KV head) writes its G outputs directly; any other segment
// writes a fp32 partial (running max m, sum l, unnormalised o) into slot 2r
// (the range's first segment) or 2r + 1 (its last), and the combine kernel
// merges the partials of each (sequence, KV head) by log-sum-exp.
//
// Thread block.  NW consumer warps + 1 producer warp.  The producer walks the
// segments, reads block ids from the table (32 at a time, one per lane; each
// lane then issues the copies of its own block, many lanes at once) and
// stages each (block, KV head) slab of K and of V -- [16, head_dim], contiguous
// in the (num_blocks, H_kv, 16, head_dim) layout -- into shared memory with
// TMA: one 1-D bulk copy per slab (linear layout), or, for the tensor-core
// consumer, tiled tensor copies of [16 rows x 128 bytes] with the 128-byte
// swizzle so that ldmatrix reads are free of bank conflicts.  The CTA's
// blocks are dealt round-robin to the consumer warps (block k -> warp k % NW)
// and every warp owns a private ring of S / NW stages, so a warp only ever
// waits on a stage whose previous phase it consumed itself.  The query rows of
// the next segment travel through a 2-deep ring with the segment descriptor.
//
// Consumers.  Scores are kept in the log2 domain (scale * log2(e) applied in
// fp32), so exponentials are exp2.
//  * CUDA-core consumer (G = 1 on 16-bit and FP8 caches; one-byte caches with
//    64-byte rows): a token row is split over
//    LPT = D / 8 lanes; partial dot products are reduced by a butterfly
//    reduce-scatter; p is shared through a per-warp scratch row; p.V
//    accumulates in fp32 registers, each lane owning 8 output elements.
//  * Tensor-core consumer (G >= 2 on a 16-bit cache or an FP8 cache with
//    128-byte rows, converted to f16 in registers; an INT8 cache with 128-byte
//    rows at every G, its codes entering the MMAs as 1024 + code with the
//    affine terms applied per block): q.K^T of a block is one
//    mma.m16n8k16 per 16 head_dim elements with the 16 tokens as M and the G
//    query heads (zero-padded to 8) as N; the fp32 scores of the C fragment
//    go through the online softmax in registers; p is rounded to the cache's
//    16-bit type, transposed in registers (movmatrix) into the B operand of
//    p.V, which accumulates O^T[head_dim x heads] in fp32 with V^T read by
//    ldmatrix.trans.  For bf16, p is multiplied as hi + lo bf16 parts (one
//    rounding of p to bf16 can exceed the tolerance on short contexts).  The
//    normaliser l sums exactly the p that is multiplied.
//
// Fused step (k_new != null).  The same launch also appends each sequence's
// new K/V row at position ctx - 1: the consumer warps of all thread blocks
// share these global writes (slots from the block table) after their wait for
// the previous kernel, and the consumer of the last block of every (sequence,
// KV head) overwrites that row of its staged block with the new row, so no
// block of the grid depends on another's write.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "pkv_common.cuh"

namespace pkv {

struct DecodeParams {
  CUtensorMap tmap_k;            // tiled views of the caches (tensor-core variant only)
  CUtensorMap tmap_v;
  const void* q;                 // [B, Hq, D] 16-bit
  const void* k_cache;           // [NB, Hkv, 16, D] KV element type
  const void* v_cache;
  const float* k_scale;          // [Hkv] (FP8 cache only)
  const float* v_scale;
  const float4* slab_params;     // INT8 cache: [NB * block_heads] (k_min, k_max, v_min, v_max)
  const int32_t* block_tables;   // [B, max_blocks_per_seq]
  const int32_t* context_lens;   // [B]
  void* out;                     // [B, Hq, D] 16-bit
  const void* k_new;             // fused step: [B, Hkv, D] rows appended at position ctx - 1 (else null)
  const void* v_new;
  int64_t* slots_out;            // fused step: [B] slots of the appended rows (nullable)
  float* ws_ml;                  // [slots, G, 2]
  float* ws_o;                   // [slots, G, D]
  int32_t* ws_cum;               // [2 (B + 1)]: block-count prefix, then non-empty-sequence prefix (for the combine)
  int32_t* err;
  int64_t num_blocks;
  int batch;
  int n_q_heads;
  int n_kv_heads;
  int block_heads;               // (block, head) slabs per cache block: n_kv_heads, or
                                 // num_layers * n_kv_heads for a layer-major cache whose
                                 // base points at this layer
  int max_blocks_per_seq;
  int max_nblk;                  // ceil(max_context_len / 16)
  int part_blocks;               // 0 = balanced ranges
  int unit_cost;                 // balanced ranges: cost of a (sequence, KV head), in quarter blocks
  int slot_capacity;             // number of partial slots in the workspace
  int stages;                    // multiple of the consumer warp count
  float qk_scale_log2;           // softmax scale * log2(e)
  unsigned long long wait_limit_ns;   // limit of each pipeline wait (kWaitLimitNs unless overridden)
  int combine_early;             // 1: the combine releases the next launch at its start (else after its wait)
  int wait_first;                // 1: the previous kernel (the INT8 step's append) writes the last block of
                                 // every (sequence, KV head): the producer waits for it before it loads such a
                                 // block, the consumers before their first global write
};

struct SegDesc {
  int b, g, i0, i1;              // logical blocks [i0, i1) of (b, g)
  int n_tokens;                  // valid tokens of (b, g)
  int nblk;                      // blocks of (b, g)
  int slot;                      // -1 = write out directly, -2 = dropped, else partial slot
  int end;                       // 1 = no more segments
};

// producer-side view of a segment
struct ProdSeg {
  int b, g, i0, i1, nb;
  int slot;                      // as SegDesc::slot
  int64_t r;                     // its range
  int64_t f_end, f_hi;           // flat end of the segment and of its range
};

// number of blocks of sequence b after clamping to the table and the bound
__device__ __forceinline__ int seq_blocks(const DecodeParams& p, int ctx, int32_t* err) {
  if (ctx < 0) {
    record_error(err, PKV_ERR_OOB);
    return 0;
  }
  int nb = (ctx + kBlockSize - 1) / kBlockSize;
  const int cap = min(p.max_blocks_per_seq, p.max_nblk);
  if (nb > cap) {
    record_error(err, PKV_ERR_OOB);
    nb = cap;
  }
  return nb;
}

// Partition mode: the flat space of W blocks is cut into NP = ceil(W / P)
// partitions of P = part_blocks blocks (the last may be shorter), and range r
// of R owns the consecutive partitions [floor(r NP / R), floor((r + 1) NP / R)).
// Consecutive partitions of one (sequence, KV head) that fall in one range
// are streamed by the same thread block as one segment: the online softmax
// merges them in registers, so a pair leaves one partial per range it meets.
__device__ __forceinline__ int64_t part_range_start(int64_t r, int64_t W, int64_t R, int part_blocks) {
  const int64_t np = (W + part_blocks - 1) / part_blocks;
  return min(((r * np) / R) * part_blocks, W);
}

// the range of partition mode that holds flat block f < W (largest r with
// part_range_start(r) <= f)
__device__ __forceinline__ int64_t part_range_of(int64_t f, int64_t W, int64_t R, int part_blocks) {
  const int64_t np = (W + part_blocks - 1) / part_blocks;
  const int64_t q = f / part_blocks;
  return min(((q + 1) * R + np - 1) / np - 1, R - 1);
}

// Balanced ranges split a cost axis, not the block axis: every block costs
// kBlockCost and every non-empty (sequence, KV head) adds unit_cost ahead of
// its first block (the per-segment work: query load, merge, output), so
// ranges that hold many short sequences get fewer blocks.  Block i of
// (b, g) sits at cost
//   pos = C(b) + g (kBlockCost nb + A) + A + kBlockCost i,
//   C(b) = Hkv (kBlockCost cum[b] + A ne[b])
// (cum: block prefix, ne: non-empty-sequence prefix, A = unit_cost), and
// range r of R owns the blocks with floor(r V / R) <= pos < floor((r+1) V / R).
constexpr int kBlockCost = 4;

// batches up to this size: the narrow combine sums the block counts itself
// (each of its warps reads every context length once)
constexpr int kCombineLocalPrefix = 256;

__device__ __forceinline__ int64_t seq_cost(const int* cum, const int* ne, int b, int Hkv, int A) {
  return static_cast<int64_t>(Hkv) * (static_cast<int64_t>(kBlockCost) * cum[b] + static_cast<int64_t>(A) * ne[b]);
}

// number of blocks whose cost position is below v (0 <= v <= V)
__device__ __forceinline__ int64_t blocks_before_cost(int64_t v, const int* cum, const int* ne, int batch, int Hkv,
                                                      int A) {
  if (v >= seq_cost(cum, ne, batch, Hkv, A)) return static_cast<int64_t>(Hkv) * cum[batch];
  int lo = 0, hi = batch - 1;   // largest b with C(b) <= v: a non-empty sequence
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (seq_cost(cum, ne, mid, Hkv, A) <= v) lo = mid; else hi = mid - 1;
  }
  const int nb = cum[lo + 1] - cum[lo];
  const int64_t unit = static_cast<int64_t>(kBlockCost) * nb + A;
  const int64_t rem = v - seq_cost(cum, ne, lo, Hkv, A);
  const int64_t g = rem / unit, w = rem % unit;
  const int64_t cnt = (w <= A) ? 0 : min(static_cast<int64_t>(nb), (w - A + kBlockCost - 1) / kBlockCost);
  return static_cast<int64_t>(Hkv) * cum[lo] + g * nb + cnt;
}

template <int D, int G, int NW, typename KV, bool MMA>
struct DecodeTraits {
  static constexpr int kEsz = KV::kBytes;
  static constexpr int kSlab = kBlockSize * D * kEsz;          // bytes of one (block, head) slab
  static constexpr int kStage = 2 * kSlab;                     // K + V
  // INT8 caches also stage each block's 16-byte (k_min, k_max, v_min, v_max),
  // into a per-stage slot of its own (the K/V tiles stay 1024-byte aligned)
  static constexpr int kParam = std::is_same<KV, U8>::value ? 16 : 0;
  static constexpr int kTx = 2 * kSlab;                          // bytes a stage receives by TMA
  // (an INT8 stage's scalars are stored into it by the issuing producer lane)
  static constexpr int kSubTiles = (D * kEsz) / 128;           // swizzled [16 x 128 B] tiles per slab
  static constexpr int kQBytes = G * D * 2;
  static constexpr int kThreads = (NW + 1) * 32;
  // CUDA-core consumer geometry
  static constexpr int kLPT = D / 8;                           // lanes per token row
  static constexpr int kNTG = 32 / kLPT;                       // token groups per warp
  static constexpr int kTPG = kBlockSize / kNTG;               // tokens per group per block
  static constexpr int kNV = kTPG * G;                         // partial scores per lane
  static constexpr int kNF = (kNV >= kLPT) ? kNV / kLPT : 1;   // held scores after reduce-scatter
  static_assert(kNF == (G >= 2 ? G / 2 : 1), "lane/head mapping");
  static_assert(!MMA || ((G >= 2 || std::is_same<KV, U8>::value) && G <= 8 && (D * kEsz) % 128 == 0 &&
                          (kEsz == 2 || D * kEsz == 128)),
                "tensor-core variant");
  // INT8 through the tensor cores: V slabs are stored transposed ([d][16]
  // token columns, see append_int8.cu) and staged by a plain 1-D copy
  static constexpr bool kVT = MMA && std::is_same<KV, U8>::value;

  // shared memory layout (byte offsets from a 1024-byte aligned base)
  static __host__ __device__ size_t q_off(int stages) { return static_cast<size_t>(stages) * kStage; }
  static __host__ __device__ size_t prm_off(int stages) { return q_off(stages) + 2 * kQBytes; }
  static __host__ __device__ size_t p_off(int stages) { return prm_off(stages) + static_cast<size_t>(stages) * kParam; }
  static __host__ __device__ size_t merge_off(int stages) {
    return p_off(stages) + sizeof(float) * NW * kBlockSize * G;
  }
  static __host__ __device__ size_t bar_off(int stages) {
    return merge_off(stages) + sizeof(float) * NW * G * (D + 2);
  }
  static __host__ __device__ size_t misc_off(int stages) { return bar_off(stages) + 8 * (2 * stages + 4); }
  // misc: stage_ok[stages], issued[stages + 2], seg[2], abort (16 B), warp totals (32 ints), scales[2 * Hkv]
  static __host__ __device__ size_t seg_off(int stages) { return misc_off(stages) + 4 * stages + 4 * (stages + 2); }
  static __host__ __device__ size_t scales_off(int stages) { return seg_off(stages) + sizeof(SegDesc) * 2 + 16 + 4 * 32; }
  static __host__ __device__ size_t cum_off(int stages, int n_kv_heads) {
    return (scales_off(stages) + 4 * 2 * n_kv_heads + 15) & ~static_cast<size_t>(15);
  }
  // + 1024 bytes so that the base can be rounded up to a 1024-byte boundary
  static __host__ __device__ size_t smem_bytes(int stages, int batch, int n_kv_heads) {
    return 1024 + cum_off(stages, n_kv_heads) + 4 * (3 * static_cast<size_t>(batch) + 3);
  }
};

// ---------------------------------------------------------------------------
// warp-level helpers
// ---------------------------------------------------------------------------
// butterfly reduce-scatter step over lanes xor MASK on N values
template <int N, int MASK>
__device__ __forceinline__ void rs_step(float* v, int lane) {
  if constexpr (N >= 2) {
    const bool upper = (lane & MASK) != 0;
#pragma unroll
    for (int k = 0; k < N / 2; ++k) {
      const float a = v[k], b = v[k + N / 2];
      const float send = upper ? a : b;
      const float keep = upper ? b : a;
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, MASK);
    }
  } else {
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], MASK);
  }
}

template <int N, int MASK>
__device__ __forceinline__ void reduce_scatter(float* v, int lane) {
  if constexpr (MASK >= 1) {
    rs_step<N, MASK>(v, lane);
    reduce_scatter<(N >= 2 ? N / 2 : 1), MASK / 2>(v, lane);
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1, BF16) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1, F16) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// two E4M3 codes (bits 0-15 of w: low byte first) -> packed f16x2, exactly
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<uint16_t>(w & 0xffffu)));
  return r;
}
// two one-byte codes (bits 0-15 of w) -> packed f16x2, exactly: E4M3 or E5M2
// values (every one is a half), or INT8 codes offset by 1024 (0x64cc is 1024 + cc in f16, one byte permute;
// the consumer folds the offset into its per-block affine terms)
__device__ __forceinline__ uint32_t byte2_to_f16x2(uint32_t w, E4M3) { return e4m3x2_to_f16x2(w); }
__device__ __forceinline__ uint32_t byte2_to_f16x2(uint32_t w, E5M2) { return e5m2x2_to_f16x2(w); }
__device__ __forceinline__ uint32_t byte2_to_f16x2(uint32_t w, U8) { return __byte_perm(w, 0x64u, 0x4140u); }
// the same for the two codes in bits 16-31 of w (no shift: the permute
// selects bytes 2 and 3; the E4M3 conversion reads the upper half register)
__device__ __forceinline__ uint32_t byte2_hi_to_f16x2(uint32_t w, E4M3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, hi;\n\t}" : "=r"(r) : "r"(w));
  return r;
}
__device__ __forceinline__ uint32_t byte2_hi_to_f16x2(uint32_t w, E5M2) { return __byte_perm(w, 0u, 0x3424u); }
__device__ __forceinline__ uint32_t byte2_hi_to_f16x2(uint32_t w, U8) { return __byte_perm(w, 0x64u, 0x4342u); }


// address of 16-byte chunk `chunk` of row `row` in a slab staged as 128B-swizzled
// [16 x 128 B] sub-tiles (each 2 KiB, 1024-byte aligned)
__device__ __forceinline__ uint32_t swz_addr(uint32_t slab, int row, int chunk) {
  return slab + (chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

// ---------------------------------------------------------------------------
// fused step: write the new token's K and V rows over row r of a staged block
// (swizzled [16 x 128 B] sub-tiles for the tensor-core layout, linear rows
// otherwise).  One lane per 16-byte chunk of a cache row; FP8 (E4M3 or E5M2)
// rows are quantised exactly as the append kernel does.
// ---------------------------------------------------------------------------
// (out of line: it runs once per (sequence, KV head) and must not raise the
// register allocation of the consumer loop)
template <typename NT, typename KV, int D, int ESZ, bool SWZ>
__device__ __noinline__ void patch_new_row(uint32_t kslab, uint32_t vslab, int r, const void* k_row,
                                              const void* v_row, float kscale, float vscale, int lane) {
  constexpr int kChunks = D * ESZ / 16;    // 16-byte chunks per cache row
  if (lane < 2 * kChunks) {
    const bool is_v = lane >= kChunks;
    const int c = is_v ? lane - kChunks : lane;
    const uint32_t slab = is_v ? vslab : kslab;
    const uint32_t addr = SWZ ? swz_addr(slab, r, c) : slab + r * D * ESZ + c * 16;
    const unsigned char* src = static_cast<const unsigned char*>(is_v ? v_row : k_row);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (ESZ == 2) {
      v = *reinterpret_cast<const uint4*>(src + c * 16);
    } else if constexpr (!std::is_same<KV, U8>::value) {   // (an INT8 cache has no fused append)
      const uint2 lo = quant8_fp8<KV>(src + c * 32, is_v ? vscale : kscale, NT{});
      const uint2 hi = quant8_fp8<KV>(src + c * 32 + 16, is_v ? vscale : kscale, NT{});
      v = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
    // order these generic-proxy writes before the stage's next TMA refill
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Rows r0..15 of a staged V block lie past the context: their probabilities
// are zero, but the rows may hold any bit pattern (a NaN would survive the
// 0 * x of p . V), so they are cleared before p . V.  Whole rows are cleared,
// which is the same in the swizzled and the linear layout.
// ---------------------------------------------------------------------------
template <int D, int ESZ, bool SWZ>
__device__ __noinline__ void clear_rows(uint32_t vslab, int r0, int lane) {
  constexpr int kChunks = D * ESZ / 16;    // 16-byte chunks per cache row
  for (int x = lane; x < (kBlockSize - r0) * kChunks; x += 32) {
    const int r = r0 + x / kChunks, c = x % kChunks;
    const uint32_t addr = SWZ ? vslab + (c >> 3) * 2048 + r * 128 + (c & 7) * 16 : vslab + r * D * ESZ + c * 16;
    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
}

// ---------------------------------------------------------------------------
// the decode kernel
// ---------------------------------------------------------------------------
template <typename QT, typename KV, int D, int G, int NW, bool MMA>
__global__ void __launch_bounds__((NW + 1) * 32, MMA ? 3 : 1) paged_decode_kernel(const __grid_constant__ DecodeParams p) {
  using T = DecodeTraits<D, G, NW, KV, MMA>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);   // 1024-byte aligned base
  const int S = p.stages;
  const int SPW = S / NW;                                         // private stages per consumer warp
  unsigned char* ring = smem;
  unsigned char* q_ring = smem + T::q_off(S);
  float* p_scr = reinterpret_cast<float*>(smem + T::p_off(S));
  float* merge = reinterpret_cast<float*>(smem + T::merge_off(S));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + T::bar_off(S));
  uint64_t* empty_bar = full_bar + S;
  uint64_t* qfull_bar = empty_bar + S;
  uint64_t* qempty_bar = qfull_bar + 2;
  int* stage_ok = reinterpret_cast<int*>(smem + T::misc_off(S));
  // issued[s]: the last use of stage s (s < S) or of query slot s - S whose
  // phase was armed (a copy issued, or an arrival made); -1 = none
  int* issued = stage_ok + S;
  SegDesc* seg = reinterpret_cast<SegDesc*>(smem + T::seg_off(S));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::seg_off(S) + 2 * sizeof(SegDesc));
  int* warp_tot = reinterpret_cast<int*>(smem + T::seg_off(S) + 2 * sizeof(SegDesc) + 16);
  float* scales = reinterpret_cast<float*>(smem + T::scales_off(S));
  int* cum = reinterpret_cast<int*>(smem + T::cum_off(S, p.n_kv_heads));   // [B + 1] block prefix
  int* ntok = cum + p.batch + 1;                                             // [B]
  int* ne = ntok + p.batch;                                                  // [B + 1] non-empty prefix

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = p.n_kv_heads;
  // Early start.  This launch may begin while the previous kernel on the
  // stream still runs (when that kernel released it early).  Everything up to
  // the consumers' wait below, and all of the producer warp's work, only READS
  // inputs -- lengths, scales, tables, q and the cache -- which no kernel of
  // this library that releases early writes (the append, copy and quantise
  // kernels never release early, except the INT8 step's own append, which
  // writes only the last block of each pair: the producer waits for it before
  // it loads such a block, and the consumers before their first write --
  // wait_first).  Every global write (the new rows, slots,
  // outputs, partials, prefixes) is made by the consumer warps after their
  // wait for the previous kernel.
  //   When the combine is released.  With combine_early = 0 the combine
  // releases its own successor only after its wait, and this kernel releases
  // the combine at once.  With combine_early = 1 the combine releases the
  // next step's kernel at once: the next decode, whose producer reads the
  // cache before its wait, or the next INT8 append, which reads before its
  // wait the slabs that this step's append wrote.  So this kernel then
  // releases at once only if it neither appends the step's new rows (fused
  // step: it releases once those cache writes are fenced) nor waits for such
  // an append (wait_first: it releases at the first return from that wait).
  if (!p.combine_early || (p.k_new == nullptr && !p.wait_first)) pdl_release();

  // ---- 1. per-sequence block counts and their prefix (all threads) -------
  if (tid == 0) *abort_flag = 0;
  for (int x = tid; x < S + 2; x += blockDim.x) issued[x] = -1;
  for (int h = tid; h < Hkv; h += blockDim.x) {
    scales[h] = p.k_scale ? p.k_scale[h] : 1.0f;
    scales[Hkv + h] = p.v_scale ? p.v_scale[h] : 1.0f;
  }
  static_assert(NW + 1 <= 16, "warp totals: 16 slots per scanned quantity");
  int carry = 0, carry_ne = 0;
  for (int base = 0; base < p.batch; base += blockDim.x) {
    const int b = base + tid;
    int nb = 0;
    if (b < p.batch) {
      const int ctx = p.context_lens[b];
      nb = seq_blocks(p, ctx, p.err);
      ntok[b] = min(max(ctx, 0), nb * kBlockSize);
    }
    int x = nb, y = nb > 0 ? 1 : 0;   // inclusive block-wide scans: blocks, non-empty sequences
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int xu = __shfl_up_sync(0xffffffffu, x, o);
      const int yu = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) {
        x += xu;
        y += yu;
      }
    }
    if (lane == 31) {
      warp_tot[warp] = x;
      warp_tot[16 + warp] = y;
    }
    __syncthreads();
    int before = 0, before_ne = 0;
    for (int w2 = 0; w2 < warp; ++w2) {
      before += warp_tot[w2];
      before_ne += warp_tot[16 + w2];
    }
    if (b < p.batch) {
      cum[b + 1] = carry + before + x;
      ne[b + 1] = carry_ne + before_ne + y;
    }
    for (int w2 = 0; w2 < static_cast<int>(blockDim.x >> 5); ++w2) {
      carry += warp_tot[w2];
      carry_ne += warp_tot[16 + w2];
    }
    __syncthreads();
  }
  if (tid == 0) {
    cum[0] = 0;
    ne[0] = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&qfull_bar[s], 1);
      mbar_init(&qempty_bar[s], NW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int64_t W = static_cast<int64_t>(Hkv) * cum[p.batch];

  const int64_t R = gridDim.x;
  const int A = p.unit_cost;
  const int64_t V = seq_cost(cum, ne, p.batch, Hkv, A);   // balanced mode: total cost

  // ---- 2. the consumers' first global writes ------------------------------
  // They follow the wait for the previous kernel (whose completion makes its
  // writes visible) and come just before a consumer group's first output or
  // partial, or at its end: until then the consumers only compute from the
  // staged blocks, while the previous kernel finishes.  They are the
  // prefixes for the combine (thread block 0) and, in the fused step, the
  // new rows (position ctx - 1).  The slot is computed from the block table
  // here.  No thread block of this grid reads that slot from the cache: the
  // consumer that processes the last block of (b, g) patches the row in
  // shared memory instead (below).  Chunks of the new rows are dealt to
  // thread blocks first (chunk c to block c mod grid), so every block carries
  // an equal share.  Called by all consumer threads together (a named
  // barrier inside).
  using NT = std::conditional_t<T::kEsz == 1, QT, KV>;   // element type of the new rows
  bool writes_done = false;
  auto first_writes = [&]() {
    if (writes_done) return;
    writes_done = true;
    pdl_wait();
    if (blockIdx.x == 0 && p.ws_cum != nullptr)
      for (int b = tid; b <= p.batch; b += NW * 32) {
        p.ws_cum[b] = cum[b];
        p.ws_cum[p.batch + 1 + b] = ne[b];
      }
    if (p.k_new != nullptr) {
      constexpr int kChunks = D / 8;                           // 8 input elements per chunk
      const int64_t total = 2ll * p.batch * Hkv * kChunks;
      for (int64_t idx = static_cast<int64_t>(tid) * gridDim.x + blockIdx.x; idx < total;
           idx += static_cast<int64_t>(gridDim.x) * (NW * 32)) {
        int64_t x = idx;
        const int c = static_cast<int>(x % kChunks);
        x /= kChunks;
        const int g = static_cast<int>(x % Hkv);
        x /= Hkv;
        const int b = static_cast<int>(x % p.batch);
        const bool is_v = x >= p.batch;
        const bool reports = !is_v && g == 0 && c == 0 && p.slots_out != nullptr;   // one thread per sequence
        // the new row's chunk is loaded before the table entry, so both loads are in flight together
        const unsigned char* src = static_cast<const unsigned char*>(is_v ? p.v_new : p.k_new) +
                                   ((static_cast<int64_t>(b) * Hkv + g) * D + 8 * c) * 2;
        const uint4 raw = *reinterpret_cast<const uint4*>(src);
        const int n = ntok[b];
        if (n == 0) {
          if (reports) p.slots_out[b] = -1;   // nothing appended (as the slot mapping reports padding)
          continue;
        }
        const int pos = n - 1;
        const int32_t blk = p.block_tables[static_cast<int64_t>(b) * p.max_blocks_per_seq + pos / kBlockSize];
        if (blk < 0 || blk >= p.num_blocks) {
          record_error(p.err, PKV_ERR_OOB);
          if (reports) p.slots_out[b] = -1;
          continue;
        }
        const int64_t row = (static_cast<int64_t>(blk) * p.block_heads + g) * kBlockSize + pos % kBlockSize;
        if (reports) p.slots_out[b] = static_cast<int64_t>(blk) * kBlockSize + pos % kBlockSize;
        unsigned char* dst =
            static_cast<unsigned char*>(const_cast<void*>(is_v ? p.v_cache : p.k_cache)) + (row * D + 8 * c) * T::kEsz;
        if constexpr (T::kEsz == 2)
          *reinterpret_cast<uint4*>(dst) = raw;
        else if constexpr (!std::is_same<KV, U8>::value)   // (an INT8 cache has no fused append)
          *reinterpret_cast<uint2*>(dst) = quant8_fp8<KV>(&raw, is_v ? scales[Hkv + g] : scales[g], NT{});
      }
      // every consumer's rows are in memory before any thread releases the
      // combine (the first release of a thread block counts for all of it;
      // the producer warp never releases)
      __threadfence();
      named_bar_sync(1, NW * 32);
      pdl_release();
    } else if (p.wait_first) {
      pdl_release();
    }
  };
  // The CUDA-core consumer defers these writes as described (on the 16-way
  // MHA batch: 151.3 against 156.5 us per step on GB300).  The tensor-core
  // consumer makes them at once: its first segment is often most of its
  // range, and deferring the combine's release that long measured slower
  // (64-sequence GQA 76.1 against 74.4 us, shared prefix 24.7 against 20.9).
  if constexpr (MMA) {
    if (warp < NW) first_writes();
  }

  if (warp == NW) {
    // ======================= producer warp ===============================
    const uint64_t pol_stream = policy_evict_first();
    const char* kbase = static_cast<const char*>(p.k_cache);
    const char* vbase = static_cast<const char*>(p.v_cache);
    const char* qbase = static_cast<const char*>(p.q);
    if (MMA && lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_k)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_v)) : "memory");
    }
    uint32_t k = 0, j = 0;
    // Segments in order: the range of this thread block, cut at (sequence,
    // KV head) boundaries.
    const int64_t r_step = R;
    auto bounds = [&](int64_t r, int64_t& lo, int64_t& hi) {
      if (p.part_blocks) {
        lo = part_range_start(r, W, R, p.part_blocks);
        hi = part_range_start(r + 1, W, R, p.part_blocks);
      } else {
        lo = blocks_before_cost((r * V) / R, cum, ne, p.batch, Hkv, A);
        hi = blocks_before_cost(((r + 1) * V) / R, cum, ne, p.batch, Hkv, A);
      }
    };
    // the segment that starts at block f of range r = [f_lo, f_hi)
    auto locate = [&](int64_t r, int64_t f, int64_t f_lo, int64_t f_hi, ProdSeg& sg) {
      int lo = 0, hi = p.batch - 1;   // largest b with Hkv * cum[b] <= f
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<int64_t>(Hkv) * cum[mid] <= f) lo = mid; else hi = mid - 1;
      }
      sg.b = lo;
      sg.nb = cum[lo + 1] - cum[lo];
      const int64_t rem = f - static_cast<int64_t>(Hkv) * cum[lo];
      sg.g = static_cast<int>(rem / sg.nb);
      sg.i0 = static_cast<int>(rem % sg.nb);
      sg.f_end = min(f_hi, f + (sg.nb - sg.i0));
      sg.i1 = sg.i0 + static_cast<int>(sg.f_end - f);
      sg.r = r;
      sg.f_hi = f_hi;
      sg.slot = -1;
      if (!(sg.i0 == 0 && sg.i1 == sg.nb)) {
        const int64_t sl = (f == f_lo) ? 2 * r : 2 * r + 1;
        sg.slot = (sl < p.slot_capacity) ? static_cast<int>(sl) : -2;   // -2: computed but not stored
      }
    };
    // the first segment of the first non-empty range from r on
    auto first_from = [&](int64_t r, ProdSeg& sg) -> bool {
      for (; r < R; r += r_step) {
        int64_t lo, hi;
        bounds(r, lo, hi);
        if (lo < hi) {
          locate(r, lo, lo, hi, sg);
          return true;
        }
      }
      return false;
    };
    auto next_of = [&](const ProdSeg& cur, ProdSeg& sg) -> bool {
      if (cur.f_end < cur.f_hi) {
        locate(cur.r, cur.f_end, -1, cur.f_hi, sg);
        return true;
      }
      return first_from(cur.r + r_step, sg);
    };
    // table entry i0 + w + lane of a segment (0 past its end)
    auto table_at = [&](const ProdSeg& sg, int w) -> int {
      return (sg.i0 + w + lane < sg.i1)
                 ? p.block_tables[static_cast<int64_t>(sg.b) * p.max_blocks_per_seq + sg.i0 + w + lane]
                 : 0;
    };
    ProdSeg cur;
    bool have = first_from(blockIdx.x, cur);
    int ids = have ? table_at(cur, 0) : 0;
    // Stopping.  A wait that runs out, or an abort raised by a consumer, stops
    // the producer: every decision to stop is a vote of the whole warp, and
    // after it no barrier receives another arrival (a stage or query slot
    // whose previous copy may still be in flight is never completed by hand).
    // Consumers stop through their own bounded waits.  Before the warp
    // exits, lane 0 waits for the last armed phase of every stage and query
    // slot (issued[]), so no copy is left in flight into shared memory.
    const uint32_t full = 0xffffffffu;
    while (have && !__any_sync(full, *abort_flag != 0)) {
      if (cur.slot == -2 && lane == 0) record_error(p.err, PKV_ERR_WORKSPACE);
      // publish the segment descriptor and its query rows
      const int qs = j & 1;
      if (lane == 0) {
        const bool slot_free =
            j < 2 || mbar_wait(&qempty_bar[qs], ((j >> 1) - 1) & 1, p.err, p.wait_limit_ns);
        if (!slot_free || *abort_flag) {
          *abort_flag = 1;
        } else {
          SegDesc d;
          d.b = cur.b; d.g = cur.g; d.i0 = cur.i0; d.i1 = cur.i1; d.n_tokens = ntok[cur.b]; d.nblk = cur.nb;
          d.slot = cur.slot;
          d.end = 0;
          seg[qs] = d;
          issued[S + qs] = static_cast<int>(j >> 1);
          mbar_arrive_expect_tx(&qfull_bar[qs], T::kQBytes);
          bulk_g2s(q_ring + qs * T::kQBytes,
                   qbase + (static_cast<int64_t>(cur.b) * p.n_q_heads + static_cast<int64_t>(cur.g) * G) * D * 2,
                   T::kQBytes, &qfull_bar[qs], pol_stream);
        }
      }
      if (__any_sync(full, *abort_flag != 0)) break;
      ++j;
      ProdSeg nxt;
      const bool have_nxt = next_of(cur, nxt);
      // Stream the segment's K/V slabs.  Lane j of the producer warp owns
      // block j of each 32-block window of the table (its table entry is
      // loaded by that lane one window ahead; the last window of a segment
      // loads the first window of the next segment).  The window is issued
      // in sub-batches of min(S, 32) blocks: the blocks of a sub-batch
      // occupy distinct stages, so their lanes wait and issue in parallel;
      // the __syncwarp between sub-batches keeps each stage's uses in order.
      const int g = cur.g;
      const int sub = S < 32 ? S : 32;
      const int nseg = cur.i1 - cur.i0;
      bool stop = false;
      for (int w0 = 0; w0 < nseg && !stop; w0 += 32) {
        const int nxt_ids = (w0 + 32 < nseg) ? table_at(cur, w0 + 32) : (have_nxt ? table_at(nxt, 0) : 0);
        const int cnt = min(32, nseg - w0);
        // INT8: each lane loads its block's (k_min, k_max, v_min, v_max) now,
        // while the window is issued, and stores them into the stage itself
        // (one TMA request fewer per block).  A last block written by the INT8
        // step's append is read after the wait for it, below.
        float4 prm_v = make_float4(0.f, 0.f, 0.f, 0.f);
        const bool last_blk = p.wait_first && cur.i0 + w0 + lane == cur.nb - 1;
        if constexpr (T::kParam > 0)
          if (lane < cnt && !last_blk && ids >= 0 && ids < p.num_blocks)
            prm_v = __ldcg(p.slab_params + static_cast<int64_t>(ids) * p.block_heads + g);
        for (int sb = 0; sb < cnt; sb += sub) {
          if (lane >= sb && lane < min(sb + sub, cnt) && !*abort_flag) {
            const uint32_t kk = k + lane;                        // CTA-local block counter
            const uint32_t jw = kk / NW;                         // index in its warp's ring
            const int s = static_cast<int>(kk % NW) + NW * static_cast<int>(jw % SPW);
            const uint32_t use = jw / SPW;
            // (the INT8 step's append writes the last block of each pair: wait for it first)
            if (last_blk) {
              pdl_wait_and_release();
              if constexpr (T::kParam > 0)
                if (ids >= 0 && ids < p.num_blocks)
                  prm_v = __ldcg(p.slab_params + static_cast<int64_t>(ids) * p.block_heads + g);
            }
            const bool stage_free = use == 0 || mbar_wait(&empty_bar[s], (use - 1) & 1, p.err, p.wait_limit_ns);
            if (!stage_free) {
              *abort_flag = 1;                                   // the stage is left as it is
            } else {
              const bool ok = ids >= 0 && ids < p.num_blocks;
              stage_ok[s] = ok ? 1 : 0;
              issued[s] = static_cast<int>(use);
              unsigned char* dst = ring + static_cast<size_t>(s) * T::kStage;
              if (ok) {
                // (the scalars' store is ordered before the consumer's read by
                // this arrive, which releases; the stage was free)
                if constexpr (T::kParam > 0)
                  *reinterpret_cast<float4*>(smem + T::prm_off(S) + s * T::kParam) = prm_v;
                mbar_arrive_expect_tx(&full_bar[s], T::kTx);
                if constexpr (MMA) {
                  const int y = (ids * p.block_heads + g) * kBlockSize;
#pragma unroll
                  for (int t = 0; t < T::kSubTiles; ++t) {
                    tma_load_2d(dst + t * 2048, &p.tmap_k, t * (128 / T::kEsz), y, &full_bar[s], pol_stream);
                    if constexpr (!T::kVT)
                      tma_load_2d(dst + T::kSlab + t * 2048, &p.tmap_v, t * (128 / T::kEsz), y, &full_bar[s],
                                  pol_stream);
                  }
                  if constexpr (T::kVT)
                    bulk_g2s(dst + T::kSlab, vbase + (static_cast<int64_t>(ids) * p.block_heads + g) * T::kSlab,
                             T::kSlab, &full_bar[s], pol_stream);
                } else {
                  const int64_t slab = (static_cast<int64_t>(ids) * p.block_heads + g) * T::kSlab;
                  bulk_g2s(dst, kbase + slab, T::kSlab, &full_bar[s], pol_stream);
                  bulk_g2s(dst + T::kSlab, vbase + slab, T::kSlab, &full_bar[s], pol_stream);
                }
              } else {
                // an id outside the pool: the stage's phase completes with no data
                record_error(p.err, PKV_ERR_OOB);
                mbar_arrive(&full_bar[s]);
              }
            }
          }
          __syncwarp();
          stop = __any_sync(full, *abort_flag != 0);
          if (stop) break;
        }
        k += cnt;
        ids = nxt_ids;
      }
      cur = nxt;
      have = have_nxt;
    }
    __syncwarp();
    if (lane == 0) {
      // end marker (only on a normal finish)
      const int qs = j & 1;
      if (!*abort_flag) {
        const bool slot_free =
            j < 2 || mbar_wait(&qempty_bar[qs], ((j >> 1) - 1) & 1, p.err, p.wait_limit_ns);
        if (slot_free) {
          seg[qs].end = 1;
          issued[S + qs] = static_cast<int>(j >> 1);
          mbar_arrive(&qfull_bar[qs]);
        } else {
          *abort_flag = 1;
        }
      }
      // Drain: the last armed phase of each stage and query slot completes
      // before the warp exits (earlier phases of a slot completed before it
      // was re-armed); one overall time limit for the drain.
      const unsigned long long deadline = global_ns() + kWaitLimitNs;
      for (int x = 0; x < S + 2; ++x) {
        const int u = issued[x];
        if (u >= 0) mbar_wait_until(x < S ? &full_bar[x] : &qfull_bar[x - S], static_cast<uint32_t>(u) & 1, deadline);
      }
    }
    __syncwarp();
    return;
  }

  // ========================== consumer warps ===============================
  constexpr int LPT = T::kLPT, TPG = T::kTPG, NF = T::kNF;
  const int li = lane & (LPT - 1);       // CUDA-core: owns elements [8 li, 8 li + 8) of a row
  const int tg = lane / LPT;             // CUDA-core: token group
  const int hsel = lane & 1;             // CUDA-core: which half of the heads this lane holds
  const int t_held = tg * TPG + (li >> 1);
  float* pw = p_scr + warp * kBlockSize * G;
  // tensor-core lane geometry (C fragment: tokens lane/4 and lane/4 + 8, heads 2 (lane%4) + {0, 1})
  const int q4 = lane & 3, r4 = lane >> 2;
  const int h0 = 2 * q4;
  const int mrow = lane & 7, mi = lane >> 3;      // ldmatrix: row within matrix, matrix index
  uint32_t j = 0;
  uint32_t k_base = 0;                   // CTA-local counter of the segment's first block
  // This warp consumes CTA-local blocks warp, warp + NW, ... in turn, the
  // j-th of them from stage warp + NW (j % SPW) at phase (j / SPW) & 1:
  // js = j % SPW and ph are kept as running counters.
  int js = 0;
  uint32_t ph = 0;
  while (true) {
    const int qs = j & 1;
    const bool got = !*abort_flag && mbar_wait(&qfull_bar[qs], (j >> 1) & 1, p.err, p.wait_limit_ns);
    if (!got) *abort_flag = 1;
    // every consumer warp must take the same exit decision (named barriers follow)
    if (named_bar_red_or(2, NW * 32, !got || seg[qs].end)) break;
    const SegDesc d = seg[qs];
    const unsigned char* qrow = q_ring + qs * T::kQBytes;
    const float sc = p.qk_scale_log2 * scales[d.g];
    const int nseg = d.i1 - d.i0;
    const int first = static_cast<int>((warp + NW - (k_base % NW)) % NW);   // first local index for this warp
    // fused step: local index of the block holding the new token (-1: none here)
    const int patch_ii = (p.k_new != nullptr && d.i1 == d.nblk && d.n_tokens > 0) ? d.nblk - 1 - d.i0 : -1;
    float* mw = merge + warp * G * (D + 2);        // [G][D] o, then [G] m, [G] l

    if constexpr (MMA) {
      // ------------------------- tensor-core consumer -------------------------
      // MT: operand type of the MMAs.  A 16-bit cache multiplies in its own
      // type.  An FP8 cache is converted to f16 in registers (every E4M3 or E5M2
      // value is exact in f16) and q is converted to f16 (exact in f16's
      // normal range); fp8 rows are 128 bytes, one swizzled sub-tile.
      constexpr bool kFp8 = (T::kEsz == 1);
      using MT = std::conditional_t<kFp8, F16, QT>;
      constexpr int KS = D / 16;
      uint32_t bq[KS][2];
      {
        const bool live = r4 < G;
        const int hq = live ? r4 : 0;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          if constexpr (kFp8) {
            // k-step ks covers head_dim [16 ks, 16 ks + 16) in the order the
            // converted fp8 A fragments use: k = 2 q4 + {0,1} <-> d = 16 ks + 4 q4 + {0,1},
            // k = 2 q4 + 8 + {0,1} <-> d = 16 ks + 4 q4 + {2,3}
            const uint2 raw = *reinterpret_cast<const uint2*>(qrow + (hq * D + 16 * ks + 4 * q4) * 2);
            const float2 lo = unpack2(raw.x, QT{}), hi = unpack2(raw.y, QT{});
            bq[ks][0] = live ? pack2(lo.x, lo.y, F16{}) : 0u;
            bq[ks][1] = live ? pack2(hi.x, hi.y, F16{}) : 0u;
          } else {
            const unsigned char* qh = qrow + (hq * D + 16 * ks + 2 * q4) * 2;
            bq[ks][0] = live ? *reinterpret_cast<const uint32_t*>(qh) : 0u;
            bq[ks][1] = live ? *reinterpret_cast<const uint32_t*>(qh + 16) : 0u;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&qempty_bar[qs]);
      // INT8 cache: the MMAs see the codes as integers offset by 1024; a
      // score is dk (q . codes) + k_min sum(q) and p . V is
      // dv (p . codes) + v_min sum(p), the offset taken out of both sums
      // (for p . V through a third MMA, of all-ones rows with the same p:
      // its accumulator cz holds sum(f16(p dv)) per head, rescaled with o)
      constexpr bool kInt8 = T::kParam > 0;
      float qs0 = 0.f, qs1 = 0.f, b0r = 0.f, b1r = 0.f;   // sc sum(q) of heads h0, h0 + 1; v_min sum(p)
      float cz[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (kInt8) {
        float a = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const float2 u = unpack2(bq[ks][0], F16{}), v = unpack2(bq[ks][1], F16{});
          a += (u.x + u.y) + (v.x + v.y);
        }
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        a += __shfl_xor_sync(0xffffffffu, a, 2);        // sum(q) of head r4
        qs0 = sc * __shfl_sync(0xffffffffu, a, 4 * h0);
        qs1 = sc * __shfl_sync(0xffffffffu, a, 4 * (h0 + 1) < 32 ? 4 * (h0 + 1) : 0);
      }
      float o[KS][4];
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
      const int krow = mrow + 8 * (mi & 1), kchunk = mi >> 1;   // A of q.K^T (and fp8 V)
      const int vrow = mrow + 8 * (mi >> 1), vchunk = mi & 1;   // A of p.V (16-bit transposed load)
      for (int ii = first; ii < nseg; ii += NW) {
        const int s = warp + NW * js;
        // (a warp vote: every lane of the warp takes the same decision)
        const bool ready = !*abort_flag && mbar_wait(&full_bar[s], ph, p.err, p.wait_limit_ns);
        if (++js == SPW) {
          js = 0;
          ph ^= 1u;
        }
        if (!__all_sync(0xffffffffu, ready)) {
          *abort_flag = 1;
          break;
        }
        const int i = d.i0 + ii;
        const int n_valid = stage_ok[s] ? min(kBlockSize, d.n_tokens - i * kBlockSize) : 0;
        const uint32_t kslab = smem_u32(ring + static_cast<size_t>(s) * T::kStage);
        const uint32_t vslab = kslab + T::kSlab;
        if (ii == patch_ii && n_valid > 0) {
          const int64_t nr = (static_cast<int64_t>(d.b) * Hkv + d.g) * D * 2;
          patch_new_row<NT, KV, D, T::kEsz, true>(kslab, vslab, (d.n_tokens - 1) % kBlockSize,
                                              static_cast<const unsigned char*>(p.k_new) + nr,
                                              static_cast<const unsigned char*>(p.v_new) + nr, scales[d.g],
                                              scales[Hkv + d.g], lane);
        }
        // (INT8 codes are finite: a zero p needs no cleared row)
        if constexpr (!kInt8)
          if (n_valid > 0 && n_valid < kBlockSize) clear_rows<D, T::kEsz, true>(vslab, n_valid, lane);
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (kFp8) {
#pragma unroll
          for (int cp = 0; cp < KS / 2; ++cp) {
            uint32_t r[4];   // (tokens 0-7, chunk 2cp), (8-15, 2cp), (0-7, 2cp+1), (8-15, 2cp+1)
            ldsm_x4(swz_addr(kslab, krow, 2 * cp + kchunk), r);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const uint32_t a[4] = {byte2_to_f16x2(r[2 * h2], KV{}), byte2_to_f16x2(r[2 * h2 + 1], KV{}),
                                     byte2_hi_to_f16x2(r[2 * h2], KV{}),
                                     byte2_hi_to_f16x2(r[2 * h2 + 1], KV{})};
              mma16816(c, a, bq[2 * cp + h2][0], bq[2 * cp + h2][1], F16{});
            }
          }
        } else {
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            uint32_t a[4];
            ldsm_x4(swz_addr(kslab, krow, 2 * ks + kchunk), a);
            mma16816(c, a, bq[ks][0], bq[ks][1], MT{});
          }
        }
        float dv = 0.f, vmin = 0.f;
        if constexpr (kInt8) {
          const float4 prm = n_valid > 0 ? *reinterpret_cast<const float4*>(smem + T::prm_off(S) + s * T::kParam)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
          // the MMAs saw 1024 + code: dk (q . (1024 + codes)) + (k_min - 1024 dk) sum(q),
          // times the score scale (folded into dk and into qs0, qs1)
          const float dk = (prm.y - prm.x) * (1.f / 255.f);
          dv = (prm.w - prm.z) * (1.f / 255.f);
          vmin = prm.z;
          const float kmin = prm.x - 1024.f * dk, dks = dk * sc;
          const float k0 = kmin * qs0, k1 = kmin * qs1;
          c[0] = fmaf(c[0], dks, k0);
          c[1] = fmaf(c[1], dks, k1);
          c[2] = fmaf(c[2], dks, k0);
          c[3] = fmaf(c[3], dks, k1);
        } else {
          c[0] *= sc;
          c[1] *= sc;
          c[2] *= sc;
          c[3] *= sc;
        }
        const bool v0 = r4 < n_valid, v1 = r4 + 8 < n_valid;
        const float s00 = v0 ? c[0] : -INFINITY, s01 = v0 ? c[1] : -INFINITY;
        const float s10 = v1 ? c[2] : -INFINITY, s11 = v1 ? c[3] : -INFINITY;
        float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
        for (int msk = 4; msk < 32; msk <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, msk));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, msk));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float ref0 = (mn0 == -INFINITY) ? 0.f : mn0, ref1 = (mn1 == -INFINITY) ? 0.f : mn1;
        const float a0 = exp2f(m0 - ref0), a1 = exp2f(m1 - ref1);
        // p in the MMA type.  bf16 keeps 8 significant bits, and one rounding
        // of p (2^-9 relative) can exceed the 2e-3 tolerance on outputs of a
        // few keys, so bf16 p is multiplied as hi = bf16(p) plus
        // lo = bf16(p - hi) (exact to ~2^-17); fp16 p (2^-12) is used as is.
        constexpr bool kSplitP = std::is_same<MT, BF16>::value;
        const float e00 = exp2f(s00 - ref0), e01 = exp2f(s01 - ref1);
        const float e10 = exp2f(s10 - ref0), e11 = exp2f(s11 - ref1);
        // (INT8: the MMA multiplies the codes by p dv; the v_min sum(p) part is kept apart)
        const float ps = kInt8 ? dv : 1.f;
        const uint32_t x0 = pack2(e00 * ps, e01 * ps, MT{});   // tokens 0..7
        const uint32_t x1 = pack2(e10 * ps, e11 * ps, MT{});   // tokens 8..15
        const float2 p0 = kInt8 ? make_float2(e00, e01) : unpack2(x0, MT{});
        const float2 p1 = kInt8 ? make_float2(e10, e11) : unpack2(x1, MT{});
        uint32_t x0l = 0u, x1l = 0u;
        float2 r0 = make_float2(0.f, 0.f), r1 = make_float2(0.f, 0.f);
        if constexpr (kSplitP) {
          x0l = pack2(e00 - p0.x, e01 - p0.y, MT{});
          x1l = pack2(e10 - p1.x, e11 - p1.y, MT{});
          r0 = unpack2(x0l, MT{});
          r1 = unpack2(x1l, MT{});
        }
        // l sums exactly what is multiplied
        l0 = l0 * a0 + ((p0.x + r0.x) + (p1.x + r1.x));
        l1 = l1 * a1 + ((p0.y + r0.y) + (p1.y + r1.y));
        if constexpr (kInt8) {
          // v_min sum(p) (the MMA's 1024 f16(p dv) per key is taken out through cz)
          b0r = b0r * a0 + (p0.x + p1.x) * vmin;
          b1r = b1r * a1 + (p0.y + p1.y) * vmin;
        }
        const bool resc = __any_sync(0xffffffffu, (mn0 != m0) | (mn1 != m1));
        m0 = mn0;
        m1 = mn1;
        const uint32_t b0 = movmatrix_trans(x0), b1 = movmatrix_trans(x1);
        uint32_t b0l = 0u, b1l = 0u;
        if constexpr (kSplitP) {
          b0l = movmatrix_trans(x0l);
          b1l = movmatrix_trans(x1l);
        }
        if (resc) {
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            o[mt][0] *= a0; o[mt][1] *= a1; o[mt][2] *= a0; o[mt][3] *= a1;
          }
          if constexpr (kInt8) {
            cz[0] *= a0; cz[1] *= a1; cz[2] *= a0; cz[3] *= a1;
          }
        }
        if constexpr (kInt8) {
          constexpr uint32_t kOnes = 0x3C003C00u;   // f16 1.0 pairs
          const uint32_t ones[4] = {kOnes, kOnes, kOnes, kOnes};
          mma16816(cz, ones, b0, b1, F16{});
        }
        if constexpr (T::kVT) {
          // INT8 V stored transposed: rows d = 32 cp + lane of the slab are
          // the four 8-row matrices of two m-tiles; lane (r4, q4) gets the
          // codes of columns 4 q4 .. 4 q4 + 3 of its row, which hold tokens
          // 2 q4, 2 q4 + 1 (the A fragment's k, k + 1, paired with b0) and
          // 2 q4 + 8, 2 q4 + 9 (paired with b1); rows in natural d order
#pragma unroll
          for (int cp = 0; cp < KS / 2; ++cp) {
            uint32_t r[4];
            ldsm_x4(vslab + (32 * cp + lane) * 16, r);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const uint32_t a[4] = {byte2_to_f16x2(r[2 * h2], KV{}), byte2_to_f16x2(r[2 * h2 + 1], KV{}),
                                     byte2_hi_to_f16x2(r[2 * h2], KV{}),
                                     byte2_hi_to_f16x2(r[2 * h2 + 1], KV{})};
              mma16816(o[2 * cp + h2], a, b0, b1, F16{});
            }
          }
        } else if constexpr (kFp8) {
          // V rows converted to f16 and transposed in registers: m-tile c's row
          // r < 8 is d = 16c + 4(r/2) + r%2, row r + 8 is that d + 2
#pragma unroll
          for (int cp = 0; cp < KS / 2; ++cp) {
            uint32_t r[4];
            ldsm_x4(swz_addr(vslab, krow, 2 * cp + kchunk), r);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const uint32_t a[4] = {movmatrix_trans(byte2_to_f16x2(r[2 * h2], KV{})),
                                     movmatrix_trans(byte2_hi_to_f16x2(r[2 * h2], KV{})),
                                     movmatrix_trans(byte2_to_f16x2(r[2 * h2 + 1], KV{})),
                                     movmatrix_trans(byte2_hi_to_f16x2(r[2 * h2 + 1], KV{}))};
              mma16816(o[2 * cp + h2], a, b0, b1, F16{});
            }
          }
        } else {
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            uint32_t a[4];
            ldsm_x4_trans(swz_addr(vslab, vrow, 2 * mt + vchunk), a);
            mma16816(o[mt], a, b0, b1, MT{});
            if constexpr (kSplitP) mma16816(o[mt], a, b0l, b1l, MT{});
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
      }
      k_base += nseg;
      // sum l over the lanes of a head column; write o, m, l to the merge area
#pragma unroll
      for (int msk = 4; msk < 32; msk <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, msk);
        l1 += __shfl_xor_sync(0xffffffffu, l1, msk);
        if constexpr (kInt8) {
          b0r += __shfl_xor_sync(0xffffffffu, b0r, msk);
          b1r += __shfl_xor_sync(0xffffffffu, b1r, msk);
        }
      }
      if constexpr (kInt8) {
        // (cz is the same in every row: all-ones A)
        const float t0 = fmaf(-1024.f, cz[0], b0r), t1 = fmaf(-1024.f, cz[1], b1r);
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          o[mt][0] += t0; o[mt][1] += t1; o[mt][2] += t0; o[mt][3] += t1;
        }
      }
      if (h0 < G) {
        constexpr bool kPermD = kFp8 && !T::kVT;   // E4M3 / E5M2 V rows come out permuted
        const bool two = h0 + 1 < G;                // (G = 1: the second column holds no head)
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int d_lo = kPermD ? 16 * mt + 4 * (r4 >> 1) + (r4 & 1) : 16 * mt + r4;
          const int d_hi = kPermD ? d_lo + 2 : d_lo + 8;
          mw[h0 * D + d_lo] = o[mt][0];
          mw[h0 * D + d_hi] = o[mt][2];
          if (two) {
            mw[(h0 + 1) * D + d_lo] = o[mt][1];
            mw[(h0 + 1) * D + d_hi] = o[mt][3];
          }
        }
        if (r4 == 0) {
          mw[G * D + h0] = m0;
          mw[G * D + G + h0] = l0;
          if (two) {
            mw[G * D + h0 + 1] = m1;
            mw[G * D + G + h0 + 1] = l1;
          }
        }
      }
    } else {
      // -------------------------- CUDA-core consumer --------------------------
      float qf[G][8];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        load8(qrow + (h * D + li * 8) * 2, qf[h], QT{});
#pragma unroll
        for (int e = 0; e < 8; ++e) qf[h][e] *= sc;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&qempty_bar[qs]);
      // INT8 cache: x = min + q (max - min) / 255 per (block, head), so a score
      // is dk (q . codes) + k_min sum(q) and p . V is dv (p . codes) + v_min sum(p):
      // the codes are used as integers and the affine terms added per block
      constexpr bool kInt8 = T::kParam > 0;
      float qsum[G], b_run[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        b_run[h] = 0.f;
        qsum[h] = 0.f;
        if constexpr (kInt8) {
          float a = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) a += qf[h][e];
#pragma unroll
          for (int msk = 1; msk < LPT; msk <<= 1) a += __shfl_xor_sync(0xffffffffu, a, msk);
          qsum[h] = a;
        }
      }

      float m_run[G], l_part[NF], acc[G][8];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        m_run[h] = -INFINITY;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;
      }
#pragma unroll
      for (int x = 0; x < NF; ++x) l_part[x] = 0.f;

      for (int ii = first; ii < nseg; ii += NW) {
        const int s = warp + NW * js;
        // (a warp vote: every lane of the warp takes the same decision)
        const bool ready = !*abort_flag && mbar_wait(&full_bar[s], ph, p.err, p.wait_limit_ns);
        if (++js == SPW) {
          js = 0;
          ph ^= 1u;
        }
        if (!__all_sync(0xffffffffu, ready)) {
          *abort_flag = 1;
          break;
        }
        const int i = d.i0 + ii;
        const int n_valid = stage_ok[s] ? min(kBlockSize, d.n_tokens - i * kBlockSize) : 0;
        const unsigned char* kslab = ring + static_cast<size_t>(s) * T::kStage;
        const unsigned char* vslab = kslab + T::kSlab;
        if (ii == patch_ii && n_valid > 0) {
          const int64_t nr = (static_cast<int64_t>(d.b) * Hkv + d.g) * D * 2;
          patch_new_row<NT, KV, D, T::kEsz, false>(smem_u32(kslab), smem_u32(vslab), (d.n_tokens - 1) % kBlockSize,
                                               static_cast<const unsigned char*>(p.k_new) + nr,
                                               static_cast<const unsigned char*>(p.v_new) + nr, scales[d.g],
                                               scales[Hkv + d.g], lane);
        }
        if constexpr (!kInt8)   // (INT8 codes are finite: a zero p needs no cleared row)
          if (n_valid > 0 && n_valid < kBlockSize) clear_rows<D, T::kEsz, false>(smem_u32(vslab), n_valid, lane);

        // ---- scores: partial dot products over this lane's 8 elements ----
        float part[T::kNV];
#pragma unroll
        for (int i2 = 0; i2 < TPG; ++i2) {
          float kf[8];
          load8(kslab + ((tg * TPG + i2) * D + li * 8) * T::kEsz, kf, KV{});
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float a0 = qf[h][0] * kf[0], a1 = qf[h][1] * kf[1];
#pragma unroll
            for (int e = 2; e < 8; e += 2) {
              a0 = fmaf(qf[h][e], kf[e], a0);
              a1 = fmaf(qf[h][e + 1], kf[e + 1], a1);
            }
            part[i2 * G + h] = a0 + a1;
          }
        }
        reduce_scatter<T::kNV, LPT / 2>(part, lane);
        float4 prm = make_float4(0.f, 0.f, 0.f, 0.f);
        float dv = 0.f;
        if constexpr (kInt8) {
          if (n_valid > 0) prm = *reinterpret_cast<const float4*>(smem + T::prm_off(S) + s * T::kParam);
          const float dk = (prm.y - prm.x) * (1.f / 255.f);
          dv = (prm.w - prm.z) * (1.f / 255.f);
#pragma unroll
          for (int x = 0; x < NF; ++x) {
            const int h = (G == 1) ? 0 : (hsel ? NF + x : x);
            float qs = qsum[0];
#pragma unroll
            for (int hh = 1; hh < G; ++hh)
              if (hh == h) qs = qsum[hh];
            part[x] = fmaf(part[x], dk, prm.x * qs);
          }
        }

        // ---- online softmax over the block --------------------------------
        float scv[NF], bm[NF];
#pragma unroll
        for (int x = 0; x < NF; ++x) {
          scv[x] = (t_held < n_valid) ? part[x] : -INFINITY;
          bm[x] = scv[x];
        }
#pragma unroll
        for (int msk = 2; msk < 32; msk <<= 1)
#pragma unroll
          for (int x = 0; x < NF; ++x) bm[x] = fmaxf(bm[x], __shfl_xor_sync(0xffffffffu, bm[x], msk));
        float bmax[G];
        if constexpr (G == 1) {
          bmax[0] = bm[0];
        } else {
#pragma unroll
          for (int x = 0; x < NF; ++x) {
            const float other = __shfl_xor_sync(0xffffffffu, bm[x], 1);
            bmax[x] = hsel ? other : bm[x];
            bmax[NF + x] = hsel ? bm[x] : other;
          }
        }
        float m_new[G], alpha[G];
        bool rescale = false;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          m_new[h] = fmaxf(m_run[h], bmax[h]);
          const float ref = (m_new[h] == -INFINITY) ? 0.f : m_new[h];
          alpha[h] = exp2f(m_run[h] - ref);
          rescale |= (m_new[h] != m_run[h]);
          m_run[h] = m_new[h];
        }
#pragma unroll
        for (int x = 0; x < NF; ++x) {
          const int h = (G == 1) ? 0 : (hsel ? NF + x : x);
          float mh = m_new[0], ah = alpha[0];
#pragma unroll
          for (int hh = 1; hh < G; ++hh)
            if (hh == h) { mh = m_new[hh]; ah = alpha[hh]; }
          const float ref = (mh == -INFINITY) ? 0.f : mh;
          const float pr = exp2f(scv[x] - ref);
          l_part[x] = l_part[x] * ah + pr;
          pw[t_held * G + h] = pr;
        }
        __syncwarp();
        if (rescale) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[h][e] *= alpha[h];
            b_run[h] *= alpha[h];
          }
        }
        // ---- p . V --------------------------------------------------------
#pragma unroll
        for (int i2 = 0; i2 < TPG; ++i2) {
          const int t = tg * TPG + i2;
          float vf[8];
          load8(vslab + (t * D + li * 8) * T::kEsz, vf, KV{});
          float pv[G];
#pragma unroll
          for (int h = 0; h < G; ++h) pv[h] = pw[t * G + h];
          if constexpr (kInt8) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
              b_run[h] = fmaf(pv[h], prm.z, b_run[h]);
              pv[h] *= dv;
            }
          }
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[h][e] = fmaf(pv[h], vf[e], acc[h][e]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
      }
      k_base += nseg;

      // ---- merge the warp's state ------------------------------------------
#pragma unroll
      for (int msk = LPT; msk < 32; msk <<= 1)
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], msk);
          if constexpr (kInt8) b_run[h] += __shfl_xor_sync(0xffffffffu, b_run[h], msk);
        }
      if constexpr (kInt8) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[h][e] += b_run[h];
      }
#pragma unroll
      for (int msk = 2; msk < 32; msk <<= 1)
#pragma unroll
        for (int x = 0; x < NF; ++x) l_part[x] += __shfl_xor_sync(0xffffffffu, l_part[x], msk);
      if (lane < LPT) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < 8; ++e) mw[h * D + li * 8 + e] = acc[h][e];
      }
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) mw[G * D + h] = m_run[h];
      }
      if (lane < 2) {
#pragma unroll
        for (int x = 0; x < NF; ++x) mw[G * D + G + ((G == 1) ? 0 : (hsel ? NF + x : x))] = l_part[x];
      }
    }

    // ---- merge the NW warps' states and write the result ---------------------
    first_writes();
    named_bar_sync(1, NW * 32);
    const float vscale = scales[Hkv + d.g];
    for (int idx = tid; idx < G * D; idx += NW * 32) {
      const int h = idx / D, e = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w2 = 0; w2 < NW; ++w2) M = fmaxf(M, merge[w2 * G * (D + 2) + G * D + h]);
      const float ref = (M == -INFINITY) ? 0.f : M;
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < NW; ++w2) {
        const float* m2 = merge + w2 * G * (D + 2);
        const float wgt = exp2f(m2[G * D + h] - ref);
        L += wgt * m2[G * D + G + h];
        O += wgt * m2[h * D + e];
      }
      O *= vscale;
      if (d.slot == -1) {
        const float r = (L > 0.f) ? O / L : 0.f;
        auto* o = static_cast<typename QT::storage*>(p.out);
        o[(static_cast<int64_t>(d.b) * p.n_q_heads + d.g * G + h) * D + e] = to_out(r, QT{});
      } else if (d.slot >= 0) {
        p.ws_o[(static_cast<int64_t>(d.slot) * G + h) * D + e] = O;
        if (e == 0) {
          p.ws_ml[(static_cast<int64_t>(d.slot) * G + h) * 2 + 0] = M;
          p.ws_ml[(static_cast<int64_t>(d.slot) * G + h) * 2 + 1] = L;
        }
      }
    }
    named_bar_sync(1, NW * 32);
    ++j;
  }
  first_writes();   // (a consumer group that wrote nothing: the wait, prefixes and new rows)
}

// ---------------------------------------------------------------------------
// Where the partials of a (sequence, KV head) pair lie, from the pair's
// geometry: c0 / ne_b blocks and non-empty sequences before sequence b, tot /
// tot_ne in all, nb blocks of b.  Ranges r0..r1 hold its blocks; its first
// piece is in slot 2 r0 when its first block opens range r0, else 2 r0 + 1;
// every later piece is in slot 2 r of its range r (the range's first segment).
// ---------------------------------------------------------------------------
struct CombineSpan {
  int64_t r0, r1;
  bool first_is_head;
  int64_t pos0, V, W;            // balanced: cost of the first block, total cost; partition: flat blocks
};

__device__ __forceinline__ CombineSpan combine_span(const DecodeParams& p, int g, int64_t c0, int nb, int64_t tot,
                                                    int64_t ne_b, int64_t tot_ne, int64_t R) {
  const int Hkv = p.n_kv_heads;
  CombineSpan s;
  s.W = static_cast<int64_t>(Hkv) * tot;
  const int64_t S0 = static_cast<int64_t>(Hkv) * c0 + static_cast<int64_t>(g) * nb;
  // Balanced mode works on the cost axis (see blocks_before_cost): u0 is the
  // cost where (b, g) starts, pos0 that of its first block; the block before
  // S0, if any, is the last of the previous non-empty pair, at u0 - kBlockCost.
  const int A = p.unit_cost;
  s.V = static_cast<int64_t>(Hkv) * (static_cast<int64_t>(kBlockCost) * tot + static_cast<int64_t>(A) * tot_ne);
  const int64_t u0 = static_cast<int64_t>(Hkv) * (static_cast<int64_t>(kBlockCost) * c0 + static_cast<int64_t>(A) * ne_b) +
                     static_cast<int64_t>(g) * (static_cast<int64_t>(kBlockCost) * nb + A);
  s.pos0 = u0 + A;
  if (p.part_blocks) {
    s.r0 = part_range_of(S0, s.W, R, p.part_blocks);
    s.r1 = part_range_of(S0 + nb - 1, s.W, R, p.part_blocks);
    s.first_is_head = (S0 == part_range_start(s.r0, s.W, R, p.part_blocks));
  } else {
    s.r0 = ((s.pos0 + 1) * R + s.V - 1) / s.V - 1;   // largest r with floor(r V / R) <= pos0
    const int64_t posl = s.pos0 + static_cast<int64_t>(kBlockCost) * (nb - 1);
    s.r1 = ((posl + 1) * R + s.V - 1) / s.V - 1;
    s.first_is_head = (S0 == 0) || ((s.r0 * s.V) / R > u0 - kBlockCost);
  }
  return s;
}

// range r of [r0, r1] holds a block of the pair unless it is narrower than a
// block (fewer blocks than ranges)
__device__ __forceinline__ bool combine_has_piece(const CombineSpan& s, const DecodeParams& p, int64_t r, int64_t R) {
  if (p.part_blocks)
    return part_range_start(r + 1, s.W, R, p.part_blocks) > part_range_start(r, s.W, R, p.part_blocks);
  if (r == s.r0) return true;
  const int64_t i = ((r * s.V) / R - s.pos0 + kBlockCost - 1) / kBlockCost;
  return s.pos0 + static_cast<int64_t>(kBlockCost) * i < ((r + 1) * s.V) / R;
}

__device__ __forceinline__ int64_t combine_slot(const CombineSpan& s, int64_t r) {
  return (r == s.r0 && !s.first_is_head) ? 2 * r + 1 : 2 * r;
}

// ---------------------------------------------------------------------------
// The wide combine, for pairs split into many pieces (the partition split of
// long contexts): out[b, g*G + h] = sum_r 2^(m_r - M) o_r / sum_r 2^(m_r - M)
// l_r over the partial slots of (b, g); zeros for an empty context.  One
// thread block per (b, g).  Each group of kSplit adjacent lanes owns 4
// consecutive outputs; lane s of the group merges pieces s, s + kSplit, ...
// (loads issued 4 at a time), then the group combines its states with xor
// shuffles.  (b, g) pairs written directly by the decode kernel are skipped.
// Up to 8 lanes per output quad and at most 512 threads: a thread block of
// 1024 threads at 64 registers holds a whole SM's register file, and the
// 256 pairs of a 32-sequence batch then ran in two waves (the combine took
// 10.6 us of a 90.7 us long-context FP8 step on GB300).
// ---------------------------------------------------------------------------
template <int D, int G>
__host__ __device__ constexpr int combine_split() {
  return 512 / (G * D / 4) >= 8 ? 8 : 512 / (G * D / 4) >= 1 ? 512 / (G * D / 4) : 1;
}
template <int D, int G>
__host__ __device__ constexpr int combine_threads() {
  return (G * D / 4) * combine_split<D, G>() < 32 ? 32 : (G * D / 4) * combine_split<D, G>();
}

template <typename QT, int D, int G>
__global__ void __launch_bounds__(combine_threads<D, G>())
    paged_decode_combine_wide_kernel(const __grid_constant__ DecodeParams p, int grid_ranges) {
  constexpr int kSplit = combine_split<D, G>();
  const int u = blockIdx.x;
  const int b = u / p.n_kv_heads, g = u % p.n_kv_heads;
  const int t = threadIdx.x / kSplit, sub = threadIdx.x % kSplit;
  const bool live_t = t < G * D / 4;
  auto* out = static_cast<typename QT::storage*>(p.out);
  // The next launch is released at once (combine_early), or after the wait
  // below: it is the next step's decode kernel (or INT8 append), which reads
  // only inputs before its own wait and writes -- the cache, the workspace,
  // the outputs -- only after it, that is after this grid (and so the decode
  // grid before it) has completed.  The geometry (blocks and non-empty
  // sequences before b and in all, the blocks of b) is read after the wait
  // from the prefixes the decode kernel leaves in the workspace.
  if (p.combine_early) pdl_release();
  pdl_wait_and_release();
  const int64_t c0 = p.ws_cum[b];
  const int nb = p.ws_cum[b + 1] - p.ws_cum[b];
  const int64_t tot = p.ws_cum[p.batch];
  const int64_t ne_b = p.ws_cum[p.batch + 1 + b];
  const int64_t tot_ne = p.ws_cum[2 * p.batch + 1];
  const int64_t base_out = (static_cast<int64_t>(b) * p.n_q_heads + g * G) * D + 4 * t;
  auto store4 = [&](float a, float b2, float c, float d) {
    const uint32_t lo = pack2(a, b2, QT{}), hi = pack2(c, d, QT{});
    *reinterpret_cast<uint2*>(out + base_out) = make_uint2(lo, hi);
  };
  if (nb == 0) {
    if (live_t && sub == 0) store4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int64_t R = grid_ranges;
  const CombineSpan sp = combine_span(p, g, c0, nb, tot, ne_b, tot_ne, R);
  if (sp.r0 == sp.r1) return;   // one segment: written by the decode kernel
  const int h = live_t ? (4 * t) / D : 0, e = live_t ? (4 * t) % D : 0;
  float M = -INFINITY, L = 0.f, O0 = 0.f, O1 = 0.f, O2 = 0.f, O3 = 0.f;
  constexpr int kBatch = 4;   // partials whose loads are issued together, per lane
  for (int64_t rb = sp.r0 + sub; rb <= sp.r1; rb += kBatch * kSplit) {
    float2 ml[kBatch];
    float4 ov[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int64_t r = rb + static_cast<int64_t>(q) * kSplit;
      // ranges between r0 and r1 may be empty (fewer blocks than ranges):
      // they wrote nothing for this (b, g)
      const bool live = live_t && r <= sp.r1 && combine_has_piece(sp, p, r, R);
      const int64_t sl = combine_slot(sp, r);
      ml[q] = live ? *reinterpret_cast<const float2*>(p.ws_ml + (sl * G + h) * 2) : make_float2(-INFINITY, 0.f);
      ov[q] = live ? *reinterpret_cast<const float4*>(p.ws_o + (sl * G + h) * D + e) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const float mn = fmaxf(M, ml[q].x);
      const float ref = (mn == -INFINITY) ? 0.f : mn;
      const float a = exp2f(M - ref), w = exp2f(ml[q].x - ref);
      L = L * a + w * ml[q].y;
      O0 = O0 * a + w * ov[q].x;
      O1 = O1 * a + w * ov[q].y;
      O2 = O2 * a + w * ov[q].z;
      O3 = O3 * a + w * ov[q].w;
      M = mn;
    }
  }
  // combine the kSplit lane states of each output quad
#pragma unroll
  for (int msk = 1; msk < kSplit; msk <<= 1) {
    // (kSplit = 1: no exchange)
    const float Mo = __shfl_xor_sync(0xffffffffu, M, msk), Lo = __shfl_xor_sync(0xffffffffu, L, msk);
    const float A0 = __shfl_xor_sync(0xffffffffu, O0, msk), A1 = __shfl_xor_sync(0xffffffffu, O1, msk);
    const float A2 = __shfl_xor_sync(0xffffffffu, O2, msk), A3 = __shfl_xor_sync(0xffffffffu, O3, msk);
    const float mn = fmaxf(M, Mo);
    const float ref = (mn == -INFINITY) ? 0.f : mn;
    const float a = exp2f(M - ref), w = exp2f(Mo - ref);
    // combine in a lane-order independent way: the lower lane's state first
    const bool low = (sub & msk) == 0;
    const float as = low ? a : w, ws = low ? w : a;
    L = (low ? L : Lo) * as + (low ? Lo : L) * ws;
    const float n0 = (low ? O0 : A0) * as + (low ? A0 : O0) * ws;
    const float n1 = (low ? O1 : A1) * as + (low ? A1 : O1) * ws;
    const float n2 = (low ? O2 : A2) * as + (low ? A2 : O2) * ws;
    const float n3 = (low ? O3 : A3) * as + (low ? A3 : O3) * ws;
    O0 = n0; O1 = n1; O2 = n2; O3 = n3;
    M = mn;
  }
  if (live_t && sub == 0) {
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    store4(O0 * inv, O1 * inv, O2 * inv, O3 * inv);
  }
}

// ---------------------------------------------------------------------------
// The narrow combine: one warp per (sequence, KV head) pair, kCombineWarps
// pairs per thread block.  Lane l owns output quads l, l + 32, ... and merges
// the pair's pieces into each in range order (the loads of kBatch pieces are
// issued together).  The thread blocks are small and hold no shared memory,
// so they become resident beside the decode grid as soon as they launch:
// they sum the block counts from the context lengths (small batches) while
// the decode grid runs and start on the partials the moment it completes.
// ---------------------------------------------------------------------------
constexpr int kCombineWarps = 4;

template <typename QT, int D, int G>
__global__ void __launch_bounds__(kCombineWarps * 32)
    paged_decode_combine_warps_kernel(const __grid_constant__ DecodeParams p, int grid_ranges) {
  constexpr int kQuads = G * D / 4;
  constexpr int kQPL = (kQuads + 31) / 32;          // output quads per lane
  constexpr int kBatch = kQPL >= 8 ? 1 : kQPL >= 4 ? 2 : 4;   // pieces loaded together
  const int lane = threadIdx.x & 31;
  const int u = blockIdx.x * kCombineWarps + static_cast<int>(threadIdx.x >> 5);
  // (release: as in paged_decode_combine_wide_kernel)
  if (p.combine_early) pdl_release();
  if (u >= p.batch * p.n_kv_heads) {
    pdl_wait();   // (every warp waits: this grid completes after the decode grid)
    return;
  }
  const int b = u / p.n_kv_heads, g = u % p.n_kv_heads;
  int64_t c0, ne_b, tot, tot_ne;
  int nb;
  if (p.batch <= kCombineLocalPrefix) {
    // the prefixes from the context lengths, clamped as the decode kernel
    // clamps them, before the wait
    long long v0 = 0, v1 = 0, v2 = 0, v3 = 0, v4 = 0;
    for (int i = lane; i < p.batch; i += 32) {
      const int ctx = p.context_lens[i];
      const int n = ctx < 0 ? 0 : min((ctx + kBlockSize - 1) / kBlockSize, min(p.max_blocks_per_seq, p.max_nblk));
      v2 += n;
      v3 += n > 0;
      if (i < b) {
        v0 += n;
        v1 += n > 0;
      }
      if (i == b) v4 = n;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      v0 += __shfl_xor_sync(0xffffffffu, v0, o);
      v1 += __shfl_xor_sync(0xffffffffu, v1, o);
      v2 += __shfl_xor_sync(0xffffffffu, v2, o);
      v3 += __shfl_xor_sync(0xffffffffu, v3, o);
      v4 += __shfl_xor_sync(0xffffffffu, v4, o);
    }
    c0 = v0, ne_b = v1, tot = v2, tot_ne = v3;
    nb = static_cast<int>(v4);
    pdl_wait_and_release();
  } else {
    pdl_wait_and_release();
    c0 = p.ws_cum[b];
    nb = p.ws_cum[b + 1] - p.ws_cum[b];
    tot = p.ws_cum[p.batch];
    ne_b = p.ws_cum[p.batch + 1 + b];
    tot_ne = p.ws_cum[2 * p.batch + 1];
  }
  auto* out = static_cast<typename QT::storage*>(p.out) + (static_cast<int64_t>(b) * p.n_q_heads + g * G) * D;
  auto store4 = [&](int quad, float a, float b2, float c, float d) {
    const uint32_t lo = pack2(a, b2, QT{}), hi = pack2(c, d, QT{});
    *reinterpret_cast<uint2*>(out + 4 * quad) = make_uint2(lo, hi);
  };
  if (nb == 0) {
#pragma unroll
    for (int k = 0; k < kQPL; ++k)
      if (lane + 32 * k < kQuads) store4(lane + 32 * k, 0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int64_t R = grid_ranges;
  const CombineSpan sp = combine_span(p, g, c0, nb, tot, ne_b, tot_ne, R);
  if (sp.r0 == sp.r1) return;   // one segment: written by the decode kernel
  float M[kQPL], L[kQPL], O[kQPL][4];
#pragma unroll
  for (int k = 0; k < kQPL; ++k) {
    M[k] = -INFINITY;
    L[k] = 0.f;
    O[k][0] = O[k][1] = O[k][2] = O[k][3] = 0.f;
  }
  for (int64_t rb = sp.r0; rb <= sp.r1; rb += kBatch) {
    float2 ml[kBatch][kQPL];
    float4 ov[kBatch][kQPL];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int64_t r = rb + q;
      const bool live = r <= sp.r1 && combine_has_piece(sp, p, r, R);
      const int64_t sl = combine_slot(sp, r);
#pragma unroll
      for (int k = 0; k < kQPL; ++k) {
        const int quad = lane + 32 * k;
        const bool lq = live && quad < kQuads;
        const int h = lq ? (4 * quad) / D : 0, e = lq ? (4 * quad) % D : 0;
        ml[q][k] = lq ? *reinterpret_cast<const float2*>(p.ws_ml + (sl * G + h) * 2) : make_float2(-INFINITY, 0.f);
        ov[q][k] = lq ? *reinterpret_cast<const float4*>(p.ws_o + (sl * G + h) * D + e)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q)
#pragma unroll
      for (int k = 0; k < kQPL; ++k) {
        const float mn = fmaxf(M[k], ml[q][k].x);
        const float ref = (mn == -INFINITY) ? 0.f : mn;
        const float a = exp2f(M[k] - ref), w = exp2f(ml[q][k].x - ref);
        L[k] = L[k] * a + w * ml[q][k].y;
        O[k][0] = O[k][0] * a + w * ov[q][k].x;
        O[k][1] = O[k][1] * a + w * ov[q][k].y;
        O[k][2] = O[k][2] * a + w * ov[q][k].z;
        O[k][3] = O[k][3] * a + w * ov[q][k].w;
        M[k] = mn;
      }
  }
#pragma unroll
  for (int k = 0; k < kQPL; ++k)
    if (lane + 32 * k < kQuads) {
      const float inv = (L[k] > 0.f) ? 1.f / L[k] : 0.f;
      store4(lane + 32 * k, O[k][0] * inv, O[k][1] * inv, O[k][2] * inv, O[k][3] * inv);
    }
}

}  // namespace pkv
