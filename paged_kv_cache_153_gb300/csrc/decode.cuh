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
// out flat, sequence-major; thread block c owns the flat range
// [c * W / R, (c + 1) * W / R) (balanced mode, R = grid size) or the ranges
// c, c + grid, ... of `part_blocks` blocks each (partition mode).  A range is
// cut into segments at (sequence, KV head) boundaries.  A segment holding a
// whole (sequence, KV head) writes its G outputs directly; any other segment
// writes a fp32 partial (running max m, sum l, unnormalised o) into slot 2r
// (the range's first segment) or 2r + 1 (its last), and the combine kernel
// merges the partials of each (sequence, KV head) by log-sum-exp.
//
// Thread block.  NW consumer warps + 1 producer warp.  The producer walks the
// segments, reads block ids from the table (32 at a time, one per lane) and
// issues one 1-D bulk copy (TMA) per K slab and per V slab -- each
// [16, head_dim] slab of a (block, KV head) is contiguous in the
// (num_blocks, H_kv, 16, head_dim) layout -- into a ring of `stages` shared
// memory stages guarded by full/empty mbarriers.  The query rows of the next
// segment travel the same way through a 2-deep ring together with the
// segment's descriptor.  Consumer warp w takes every NW-th block of the range.
//
// Consumer arithmetic (fp32).  A token row is split over LPT = D / 8 lanes
// (8 elements, 16 bytes per lane); a warp covers 32 / LPT token rows at once.
// Partial dot products for the G heads are reduced across the LPT lanes by a
// butterfly reduce-scatter, the block maximum by shuffles, the probabilities
// are shared through a per-warp scratch row, and p.V accumulates in registers
// with each lane owning 8 output elements of every head.  Scores are kept in
// the log2 domain (scale * log2(e) folded into q), so exponentials are exp2.
#pragma once

#include <cuda_runtime.h>

#include "pkv_common.cuh"

namespace pkv {

struct DecodeParams {
  const void* q;                 // [B, Hq, D] 16-bit
  const void* k_cache;           // [NB, Hkv, 16, D] KV element type
  const void* v_cache;
  const float* k_scale;          // [Hkv] (E4M3 cache only)
  const float* v_scale;
  const int32_t* block_tables;   // [B, max_blocks_per_seq]
  const int32_t* context_lens;   // [B]
  void* out;                     // [B, Hq, D] 16-bit
  int32_t* ws_cum;               // [B + 1] block-count prefix written for the combine
  float* ws_ml;                  // [slots, G, 2]
  float* ws_o;                   // [slots, G, D]
  int32_t* err;
  int64_t num_blocks;
  int batch;
  int n_q_heads;
  int n_kv_heads;
  int max_blocks_per_seq;
  int max_nblk;                  // ceil(max_context_len / 16)
  int part_blocks;               // 0 = balanced ranges
  int slot_capacity;             // number of partial slots in the workspace
  int stages;
  float qk_scale_log2;           // softmax scale * log2(e)
};

struct SegDesc {
  int b, g, i0, i1;              // logical blocks [i0, i1) of (b, g)
  int n_tokens;                  // valid tokens of (b, g)
  int nblk;                      // blocks of (b, g)
  int slot;                      // -1 = write out directly, else partial slot
  int end;                       // 1 = no more segments
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

// flat index of range boundary r
__device__ __forceinline__ int64_t range_start(int64_t r, int64_t W, int64_t R, int part_blocks) {
  return part_blocks ? min(r * part_blocks, W) : (r * W) / R;
}

template <int D, int G, int NW, typename KV>
struct DecodeTraits {
  static constexpr int kEsz = KV::kBytes;
  static constexpr int kSlab = kBlockSize * D * kEsz;          // bytes of one (block, head) slab
  static constexpr int kStage = 2 * kSlab;                     // K + V
  static constexpr int kLPT = D / 8;                           // lanes per token row
  static constexpr int kNTG = 32 / kLPT;                       // token groups per warp
  static constexpr int kTPG = kBlockSize / kNTG;               // tokens per group per block
  static constexpr int kNV = kTPG * G;                         // partial scores per lane
  static constexpr int kNF = (kNV >= kLPT) ? kNV / kLPT : 1;   // held scores after reduce-scatter
  static constexpr int kQBytes = G * D * 2;
  static constexpr int kThreads = (NW + 1) * 32;
  static_assert(kNF == (G >= 2 ? G / 2 : 1), "lane/head mapping");

  // shared memory layout (byte offsets); the ring comes first (128-B aligned)
  static __host__ __device__ size_t ring_off() { return 0; }
  static __host__ __device__ size_t q_off(int stages) { return static_cast<size_t>(stages) * kStage; }
  static __host__ __device__ size_t p_off(int stages) { return q_off(stages) + 2 * kQBytes; }
  static __host__ __device__ size_t merge_off(int stages) {
    return p_off(stages) + sizeof(float) * NW * kBlockSize * G;
  }
  static __host__ __device__ size_t bar_off(int stages) {
    return merge_off(stages) + sizeof(float) * NW * G * (D + 2);
  }
  static __host__ __device__ size_t misc_off(int stages) { return bar_off(stages) + 8 * (2 * stages + 4); }
  static __host__ __device__ size_t cum_off(int stages, int n_kv_heads) {
    // stage_ok[stages], seg[2], abort, scales[2 * Hkv]
    size_t o = misc_off(stages) + 4 * stages + sizeof(SegDesc) * 2 + 16 + 4 * 2 * n_kv_heads;
    return (o + 15) & ~static_cast<size_t>(15);
  }
  static __host__ __device__ size_t smem_bytes(int stages, int batch, int n_kv_heads) {
    return cum_off(stages, n_kv_heads) + 4 * (2 * static_cast<size_t>(batch) + 2);
  }
};

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

template <typename QT, typename KV, int D, int G, int NW>
__global__ void __launch_bounds__((NW + 1) * 32, 1) paged_decode_kernel(const DecodeParams p) {
  using T = DecodeTraits<D, G, NW, KV>;
  constexpr int LPT = T::kLPT, TPG = T::kTPG, NF = T::kNF;
  extern __shared__ __align__(128) unsigned char smem[];
  const int S = p.stages;
  unsigned char* ring = smem + T::ring_off();
  unsigned char* q_ring = smem + T::q_off(S);
  float* p_scr = reinterpret_cast<float*>(smem + T::p_off(S));
  float* merge = reinterpret_cast<float*>(smem + T::merge_off(S));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + T::bar_off(S));
  uint64_t* empty_bar = full_bar + S;
  uint64_t* qfull_bar = empty_bar + S;
  uint64_t* qempty_bar = qfull_bar + 2;
  int* stage_ok = reinterpret_cast<int*>(smem + T::misc_off(S));
  SegDesc* seg = reinterpret_cast<SegDesc*>(smem + T::misc_off(S) + 4 * S);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::misc_off(S) + 4 * S + 2 * sizeof(SegDesc));
  float* scales = reinterpret_cast<float*>(smem + T::misc_off(S) + 4 * S + 2 * sizeof(SegDesc) + 16);
  int* cum = reinterpret_cast<int*>(smem + T::cum_off(S, p.n_kv_heads));   // [B + 1]
  int* ntok = cum + p.batch + 1;                                             // [B]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = p.n_kv_heads;

  // ---- 1. per-sequence block counts and their prefix (all threads) -------
  if (tid == 0) *abort_flag = 0;
  for (int h = tid; h < Hkv; h += blockDim.x) {
    scales[h] = p.k_scale ? p.k_scale[h] : 1.0f;
    scales[Hkv + h] = p.v_scale ? p.v_scale[h] : 1.0f;
  }
  int carry = 0;
  for (int base = 0; base < p.batch; base += blockDim.x) {
    const int b = base + tid;
    int nb = 0;
    if (b < p.batch) {
      const int ctx = p.context_lens[b];
      nb = seq_blocks(p, ctx, p.err);
      ntok[b] = min(max(ctx, 0), nb * kBlockSize);
    }
    // inclusive block-wide scan of nb
    int x = nb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    __shared__ int warp_tot[32];
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    int before = 0;
    for (int w2 = 0; w2 < warp; ++w2) before += warp_tot[w2];
    if (b < p.batch) cum[b + 1] = carry + before + x;
    int tot = 0;
    for (int w2 = 0; w2 < (int)(blockDim.x >> 5); ++w2) tot += warp_tot[w2];
    carry += tot;
    __syncthreads();
  }
  if (tid == 0) cum[0] = 0;
  if (tid == 0) {
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
  if (blockIdx.x == 0 && p.ws_cum != nullptr)
    for (int b = tid; b <= p.batch; b += blockDim.x) p.ws_cum[b] = cum[b];

  const int64_t R = p.part_blocks ? (W + p.part_blocks - 1) / p.part_blocks : gridDim.x;

  if (warp == NW) {
    // ======================= producer warp ===============================
    const uint64_t pol_stream = policy_evict_first();
    const char* kbase = static_cast<const char*>(p.k_cache);
    const char* vbase = static_cast<const char*>(p.v_cache);
    const char* qbase = static_cast<const char*>(p.q);
    uint32_t k = 0, j = 0;
    for (int64_t r = blockIdx.x; r < R && !*abort_flag; r += (p.part_blocks ? gridDim.x : R)) {
      const int64_t f_lo = range_start(r, W, R, p.part_blocks);
      const int64_t f_hi = range_start(r + 1, W, R, p.part_blocks);
      int64_t f = f_lo;
      while (f < f_hi && !*abort_flag) {
        // locate the sequence: largest b with Hkv * cum[b] <= f
        int lo = 0, hi = p.batch - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (static_cast<int64_t>(Hkv) * cum[mid] <= f) lo = mid; else hi = mid - 1;
        }
        const int b = lo;
        const int nb = cum[b + 1] - cum[b];
        const int64_t rem = f - static_cast<int64_t>(Hkv) * cum[b];
        const int g = static_cast<int>(rem / nb);
        const int i0 = static_cast<int>(rem % nb);
        const int64_t f_end = min(f_hi, f + (nb - i0));
        const int i1 = i0 + static_cast<int>(f_end - f);
        int slot = -1;
        if (!(i0 == 0 && i1 == nb)) {
          const int64_t sl = (f == f_lo) ? 2 * r : 2 * r + 1;
          if (sl >= p.slot_capacity) {
            record_error(p.err, PKV_ERR_WORKSPACE);
            slot = -2;                       // computed but not stored
          } else {
            slot = static_cast<int>(sl);
          }
        }
        // publish the segment descriptor and its query rows
        const int qs = j & 1;
        if (lane == 0) {
          if (j >= 2 && !*abort_flag && !mbar_wait(&qempty_bar[qs], ((j >> 1) - 1) & 1, p.err)) *abort_flag = 1;
          SegDesc d;
          d.b = b; d.g = g; d.i0 = i0; d.i1 = i1; d.n_tokens = ntok[b]; d.nblk = nb; d.slot = slot;
          d.end = *abort_flag ? 1 : 0;
          seg[qs] = d;
          if (!*abort_flag) {
            mbar_arrive_expect_tx(&qfull_bar[qs], T::kQBytes);
            bulk_g2s(q_ring + qs * T::kQBytes,
                     qbase + (static_cast<int64_t>(b) * p.n_q_heads + static_cast<int64_t>(g) * G) * D * 2,
                     T::kQBytes, &qfull_bar[qs], pol_stream);
          } else {
            mbar_arrive(&qfull_bar[qs]);
          }
        }
        __syncwarp();
        ++j;
        // stream the segment's K/V slabs
        const int32_t* row = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq;
        int ids = (i0 + lane < i1) ? row[i0 + lane] : 0;
        for (int ib = i0; ib < i1; ib += 32) {
          const int nxt = (ib + 32 + lane < i1) ? row[ib + 32 + lane] : 0;   // prefetch the next 32
          const int cnt = min(32, i1 - ib);
          for (int jj = 0; jj < cnt; ++jj) {
            const int pid = __shfl_sync(0xffffffffu, ids, jj);
            if (lane == 0) {
              const int s = k % S;
              if (k >= static_cast<uint32_t>(S) && !*abort_flag &&
                  !mbar_wait(&empty_bar[s], ((k / S) - 1) & 1, p.err))
                *abort_flag = 1;
              const bool ok = pid >= 0 && pid < p.num_blocks && !*abort_flag;
              stage_ok[s] = ok ? 1 : 0;
              if (ok) {
                const int64_t slab = (static_cast<int64_t>(pid) * Hkv + g) * T::kSlab;
                mbar_arrive_expect_tx(&full_bar[s], T::kStage);
                bulk_g2s(ring + static_cast<size_t>(s) * T::kStage, kbase + slab, T::kSlab, &full_bar[s],
                         pol_stream);
                bulk_g2s(ring + static_cast<size_t>(s) * T::kStage + T::kSlab, vbase + slab, T::kSlab,
                         &full_bar[s], pol_stream);
              } else {
                if (!*abort_flag) record_error(p.err, PKV_ERR_OOB);
                mbar_arrive(&full_bar[s]);
              }
            }
            ++k;
          }
          ids = nxt;
          __syncwarp();
        }
        f = f_end;
      }
    }
    // end marker
    const int qs = j & 1;
    if (lane == 0) {
      if (j >= 2 && !*abort_flag && !mbar_wait(&qempty_bar[qs], ((j >> 1) - 1) & 1, p.err)) *abort_flag = 1;
      seg[qs].end = 1;
      mbar_arrive(&qfull_bar[qs]);
      // Before exiting, make sure no copy issued by this warp is still in
      // flight into shared memory (one overall time limit for the drain).
      const unsigned long long deadline = global_ns() + kWaitLimitNs;
      const uint32_t first = k > static_cast<uint32_t>(S) ? k - S : 0;
      for (uint32_t kk = first; kk < k; ++kk)
        if (stage_ok[kk % S]) mbar_wait_until(&full_bar[kk % S], (kk / S) & 1, deadline);
      // Only the last segment's query copy can still be in flight: the one
      // before it shares its slot with the end marker, whose publication
      // waited until the consumers had read that copy (and re-armed the slot).
      if (j >= 1) mbar_wait_until(&qfull_bar[(j - 1) & 1], ((j - 1) >> 1) & 1, deadline);
    }
    __syncwarp();
    return;
  }

  // ========================== consumer warps ===============================
  const int li = lane & (LPT - 1);       // owns elements [8 li, 8 li + 8) of a row
  const int tg = lane / LPT;             // token group
  const int hsel = lane & 1;             // which half of the heads this lane holds
  const int t_held = tg * TPG + (li >> 1);
  float* pw = p_scr + warp * kBlockSize * G;
  uint32_t j = 0;
  uint32_t k_base = 0;                   // flat counter of the segment's first block in this CTA
  while (true) {
    const int qs = j & 1;
    const bool got = !*abort_flag && mbar_wait(&qfull_bar[qs], (j >> 1) & 1, p.err);
    if (!got) *abort_flag = 1;
    // every consumer warp must take the same exit decision (named barriers follow)
    if (named_bar_red_or(2, NW * 32, !got || seg[qs].end)) break;
    const SegDesc d = seg[qs];
    float qf[G][8];
    {
      const float qscale = p.qk_scale_log2 * scales[d.g];
      const unsigned char* qrow = q_ring + qs * T::kQBytes;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        load8(qrow + (h * D + li * 8) * 2, qf[h], QT{});
#pragma unroll
        for (int e = 0; e < 8; ++e) qf[h][e] *= qscale;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&qempty_bar[qs]);

    float m_run[G], l_part[NF], acc[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m_run[h] = -INFINITY;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;
    }
#pragma unroll
    for (int x = 0; x < NF; ++x) l_part[x] = 0.f;

    const int nseg = d.i1 - d.i0;
    int first = static_cast<int>((warp + NW - (k_base % NW)) % NW);   // first local index for this warp
    for (int ii = first; ii < nseg; ii += NW) {
      const uint32_t k = k_base + ii;
      const int s = k % S;
      if (*abort_flag || !mbar_wait(&full_bar[s], (k / S) & 1, p.err)) {
        *abort_flag = 1;
        break;
      }
      const int i = d.i0 + ii;
      const int n_valid = stage_ok[s] ? min(kBlockSize, d.n_tokens - i * kBlockSize) : 0;
      const unsigned char* kslab = ring + static_cast<size_t>(s) * T::kStage;
      const unsigned char* vslab = kslab + T::kSlab;

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

      // ---- online softmax over the block --------------------------------
      float sc[NF], bm[NF];
#pragma unroll
      for (int x = 0; x < NF; ++x) {
        sc[x] = (t_held < n_valid) ? part[x] : -INFINITY;
        bm[x] = sc[x];
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
        const float pr = exp2f(sc[x] - ref);
        l_part[x] = l_part[x] * ah + pr;
        pw[t_held * G + h] = pr;
      }
      __syncwarp();
      if (rescale) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[h][e] *= alpha[h];
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
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[h][e] = fmaf(pv[h], vf[e], acc[h][e]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
    k_base += nseg;

    // ---- merge the warp's state, then the NW warps' states ---------------
#pragma unroll
    for (int msk = LPT; msk < 32; msk <<= 1)
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], msk);
#pragma unroll
    for (int msk = 2; msk < 32; msk <<= 1)
#pragma unroll
      for (int x = 0; x < NF; ++x) l_part[x] += __shfl_xor_sync(0xffffffffu, l_part[x], msk);
    float* mw = merge + warp * G * (D + 2);        // [G][D] o, then [G] m, [G] l
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
}

// ---------------------------------------------------------------------------
// combine: out[b, g*G + h] = sum_r 2^(m_r - M) o_r / sum_r 2^(m_r - M) l_r over
// the partial slots of (b, g); zeros for an empty context.  One thread block
// per (b, g); (b, g) pairs written directly by the decode kernel are skipped.
// ---------------------------------------------------------------------------
template <typename QT, int D, int G>
__global__ void __launch_bounds__(128) paged_decode_combine_kernel(const DecodeParams p, int grid_ranges) {
  const int u = blockIdx.x;
  const int b = u / p.n_kv_heads, g = u % p.n_kv_heads;
  auto* out = static_cast<typename QT::storage*>(p.out);
  const int c0 = p.ws_cum[b], c1 = p.ws_cum[b + 1];
  const int nb = c1 - c0;
  const int64_t base_out = (static_cast<int64_t>(b) * p.n_q_heads + g * G) * D;
  if (nb == 0) {
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) out[base_out + idx] = to_out(0.f, QT{});
    return;
  }
  const int64_t W = static_cast<int64_t>(p.n_kv_heads) * p.ws_cum[p.batch];
  const int64_t S0 = static_cast<int64_t>(p.n_kv_heads) * c0 + static_cast<int64_t>(g) * nb;
  const int64_t E0 = S0 + nb;
  const int64_t R = p.part_blocks ? (W + p.part_blocks - 1) / p.part_blocks : grid_ranges;
  auto range_of = [&](int64_t f) -> int64_t {
    if (p.part_blocks) return f / p.part_blocks;
    return ((f + 1) * R + W - 1) / W - 1;
  };
  const int64_t r0 = range_of(S0), r1 = range_of(E0 - 1);
  if (r0 == r1) return;   // one segment: written by the decode kernel
  const bool first_is_head = (S0 == range_start(r0, W, R, p.part_blocks));
  // ranges between r0 and r1 may be empty (fewer blocks than ranges): they
  // wrote nothing for this (b, g) and are skipped
  auto touches = [&](int64_t r) {
    return range_start(r + 1, W, R, p.part_blocks) > range_start(r, W, R, p.part_blocks);
  };
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int h = idx / D, e = idx % D;
    float M = -INFINITY;
    for (int64_t r = r0; r <= r1; ++r) {
      if (!touches(r)) continue;
      const int64_t sl = (r == r0 && !first_is_head) ? 2 * r + 1 : 2 * r;
      M = fmaxf(M, p.ws_ml[(sl * G + h) * 2]);
    }
    const float ref = (M == -INFINITY) ? 0.f : M;
    float L = 0.f, O = 0.f;
    for (int64_t r = r0; r <= r1; ++r) {
      if (!touches(r)) continue;
      const int64_t sl = (r == r0 && !first_is_head) ? 2 * r + 1 : 2 * r;
      const float wgt = exp2f(p.ws_ml[(sl * G + h) * 2] - ref);
      L += wgt * p.ws_ml[(sl * G + h) * 2 + 1];
      O += wgt * p.ws_o[(sl * G + h) * D + e];
    }
    out[base_out + idx] = to_out(L > 0.f ? O / L : 0.f, QT{});
  }
}

}  // namespace pkv
