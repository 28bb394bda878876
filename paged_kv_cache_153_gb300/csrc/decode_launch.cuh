// Host-side launch of one decode-kernel variant plus its combine kernel.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "decode.cuh"
#include "host_util.h"

namespace pkv {

struct LaunchInfo {
  int num_sms;
  int max_ctas_per_sm;     // resident decode blocks per SM (0 = the variant's default)
  int stages;              // 0 = fill the SM's shared memory; else a request (rounded to the warp count)
  int grid;                // out: decode grid used
  int64_t part_ranges_cap; // partition mode: max ranges the workspace holds
};

using DecodeLauncher = pkv_status (*)(DecodeParams&, LaunchInfo&, cudaStream_t);

constexpr int kMaxDevices = 64;
constexpr int kSmemPerSm = 233472;        // shared memory per SM on sm_100-class parts (228 KiB)
constexpr int kSmemReservedPerCta = 1024; // system-reserved shared memory per resident block
constexpr int kMaxStagesPerWarp = 8;

template <typename QT, typename KV, int D, int G, int NW, bool MMA>
pkv_status launch_decode_variant(DecodeParams& p, LaunchInfo& li, cudaStream_t stream) {
  using Tr = DecodeTraits<D, G, NW, KV, MMA>;
  auto kern = paged_decode_kernel<QT, KV, D, G, NW, MMA>;
  int max_optin = 0, dev = 0;
  if (cuda_failed(cudaGetDevice(&dev), "cudaGetDevice")) return PKV_ERR_CUDA;
  if (cuda_failed(cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev),
                  "cudaDeviceGetAttribute"))
    return PKV_ERR_CUDA;
  cudaFuncAttributes fattr;
  if (cuda_failed(cudaFuncGetAttributes(&fattr, kern), "cudaFuncGetAttributes")) return PKV_ERR_CUDA;
  // dynamic shared memory may use what the static part leaves of the opt-in limit
  const size_t dyn_max = static_cast<size_t>(max_optin) - fattr.sharedSizeBytes;
  // the opt-in is a per-device function attribute: set it once per device
  static std::mutex attr_mu;
  static bool attr_done[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
  {
    std::lock_guard<std::mutex> lock(attr_mu);
    if (!attr_done[dev]) {
      if (cuda_failed(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(dyn_max)),
                      "cudaFuncSetAttribute"))
        return PKV_ERR_CUDA;
      attr_done[dev] = true;
    }
  }
  // Stages come in multiples of NW (each consumer warp owns stages/NW of them).
  // By default, the ring fills the SM's shared memory across as many resident
  // blocks as the registers allow (capped by max_ctas_per_sm).
  int occ = 0;
  size_t smem = Tr::smem_bytes(NW, p.batch, p.n_kv_heads);
  if (smem > dyn_max) return PKV_ERR_UNSUPPORTED;   // batch too large for one block's shared memory
  if (cuda_failed(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, Tr::kThreads, smem),
                  "cudaOccupancyMaxActiveBlocksPerMultiprocessor"))
    return PKV_ERR_CUDA;
  if (occ < 1) return PKV_ERR_UNSUPPORTED;
  // Upper bound on the (sequence, KV head, block) work items, from max_context_len.
  const int64_t w_max = static_cast<int64_t>(p.batch) * p.n_kv_heads *
                        std::min<int64_t>(p.max_blocks_per_seq, p.max_nblk);
  // Resident blocks per SM (li.max_ctas_per_sm overrides), measured best on
  // GB300: 3 for one-byte caches through the tensor cores, whose per-block
  // conversions want more consumer warps; 2 for 16-bit caches, where a deeper
  // stage ring per block beats more consumer warps (with the combine released
  // early, below: the mixed-length 64-sequence GQA batch 76.1 us at 2 against
  // 77.4 at 3).
  const int want = li.max_ctas_per_sm > 0 ? li.max_ctas_per_sm : (MMA && Tr::kEsz == 1) ? 3 : 2;
  // Cost of one (sequence, KV head) in the balanced split, in quarter blocks:
  // the per-segment work (query load, cross-warp merge, output or partial
  // write) and the consumer warps left idle by short segments.  Measured on
  // GB300 with mixed context lengths: 24 (6 blocks' worth of streaming) for
  // the CUDA-core consumer; 48 for the tensor-core one over one-byte caches,
  // whose per-segment set-up is larger (INT8 60.9 -> 59.0 us against 24); 32
  // for the tensor-core one over 16-bit caches (sweeps of 8..48 on the GQA
  // batch above and on a 16-sequence shared-prefix batch).
  if (p.unit_cost < 0) p.unit_cost = !MMA ? 24 : Tr::kEsz == 1 ? 48 : 32;
  occ = std::min(occ, want);
  int spw = 1;
  if (li.stages > 0) {
    spw = std::max(1, li.stages / NW);
  } else {
    for (int cand = kMaxStagesPerWarp; cand >= 1; --cand) {
      const size_t s = Tr::smem_bytes(NW * cand, p.batch, p.n_kv_heads);
      if (s <= dyn_max && static_cast<size_t>(occ) * (s + kSmemReservedPerCta) <= kSmemPerSm) {
        spw = cand;
        break;
      }
    }
  }
  spw = std::min(spw, kMaxStagesPerWarp);
  while (spw > 1 && Tr::smem_bytes(NW * spw, p.batch, p.n_kv_heads) > dyn_max) --spw;
  const int stages = NW * spw;
  smem = Tr::smem_bytes(stages, p.batch, p.n_kv_heads);
  if (cuda_failed(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, Tr::kThreads, smem),
                  "cudaOccupancyMaxActiveBlocksPerMultiprocessor"))
    return PKV_ERR_CUDA;
  if (occ < 1) return PKV_ERR_UNSUPPORTED;
  occ = std::min(occ, want);
  int grid = li.num_sms * occ;
  if (p.part_blocks > 0 && li.part_ranges_cap < grid) grid = static_cast<int>(li.part_ranges_cap);
  // a small workload (upper bound on blocks known from max_context_len) needs
  // no more than one thread block per few blocks of work
  if (p.part_blocks == 0) {
    const int64_t w_max = static_cast<int64_t>(p.batch) * p.n_kv_heads *
                          std::min<int64_t>(p.max_blocks_per_seq, p.max_nblk);
    grid = static_cast<int>(std::min<int64_t>(grid, std::max<int64_t>(1, (w_max + 3) / 4)));
  }
  if (grid < 1) grid = 1;
  p.stages = stages;
  // The combine releases the next launch before its own wait when at most
  // two decode blocks share each SM of a full grid (its small thread blocks
  // then become resident beside them at once): the next step's decode kernel
  // starts streaming during this one's tail.  With three per SM the
  // combine's blocks get an SM only as decode blocks leave, and an early
  // release measured far slower on GB300 (the 64-sequence GQA batch 111 us
  // against 77); a grid smaller than the GPU has no tail to overlap (4 short
  // sequences: 9.65 us against 9.28).  There the combine releases after its
  // wait.
  p.combine_early = (occ <= 2 && grid == li.num_sms * occ) ? 1 : 0;
  li.grid = grid;
  li.stages = stages;
  if constexpr (MMA) {
    // rows from this layer's base to the end of its last block's slabs
    const int64_t rows = ((p.num_blocks - 1) * p.block_heads + p.n_kv_heads) * kBlockSize;
    if (rows > INT32_MAX) return PKV_ERR_UNSUPPORTED;    // TMA row coordinates are 32-bit
    if (!encode_cache_tmap(&p.tmap_k, p.k_cache, rows, D, Tr::kEsz) ||
        !encode_cache_tmap(&p.tmap_v, p.v_cache, rows, D, Tr::kEsz))
      return PKV_ERR_CUDA;
  }
  if (cuda_failed(launch_pdl(kern, dim3(grid), dim3(Tr::kThreads), smem, stream, p), "paged_decode_kernel launch"))
    return PKV_ERR_CUDA;
  const int units = p.batch * p.n_kv_heads;
  if (units > 0) {
    // a partition split of long contexts can leave many pieces per (sequence,
    // KV head) (one per range it meets): merge those with several lanes per output
    const bool wide = p.part_blocks > 0 && (p.max_nblk + p.part_blocks - 1) / p.part_blocks >= 16;
    const cudaError_t e =
        wide ? launch_pdl(paged_decode_combine_wide_kernel<QT, D, G>, dim3(units),
                          dim3(combine_threads<D, G>()), 0, stream, p, grid)
             : launch_pdl(paged_decode_combine_warps_kernel<QT, D, G>,
                          dim3((units + kCombineWarps - 1) / kCombineWarps), dim3(kCombineWarps * 32), 0, stream,
                          p, grid);
    if (cuda_failed(e, "combine kernel launch")) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

// Variants compiled in each translation unit (by KV element type).
DecodeLauncher decode_launcher_f16(int head_dim, int group);
DecodeLauncher decode_launcher_bf16(int head_dim, int group);
DecodeLauncher decode_launcher_e4m3(int q_dtype, int head_dim, int group);
DecodeLauncher decode_launcher_e5m2(int q_dtype, int head_dim, int group);
DecodeLauncher decode_launcher_int8(int q_dtype, int head_dim, int group);

constexpr int kCoreWarps = 8;   // consumer warps of the CUDA-core variant
constexpr int kMmaWarps = 4;    // consumer warps of the tensor-core variant

// G = 1 uses the CUDA-core consumer; G >= 2 over a 16-bit cache, or over a
// one-byte (E4M3, E5M2 or INT8) cache with 128-byte rows, uses the tensor-core
// consumer (the q-group times a 16-token block is an MMA tile), and so does
// an INT8 cache with 128-byte rows at G = 1.
template <typename QT, typename KV, int D, int G>
DecodeLauncher pick_variant() {
  // (an INT8 cache with 128-byte rows takes the tensor-core consumer for every
  // group size: its V slabs are stored transposed for that consumer)
  if constexpr ((G >= 2 || std::is_same<KV, U8>::value) && (KV::kBytes == 2 || D * KV::kBytes == 128))
    return launch_decode_variant<QT, KV, D, G, kMmaWarps, true>;
  else
    return launch_decode_variant<QT, KV, D, G, kCoreWarps, false>;
}

template <typename QT, typename KV, int D>
DecodeLauncher pick_group(int group) {
  switch (group) {
    case 1: return pick_variant<QT, KV, D, 1>();
    case 2: return pick_variant<QT, KV, D, 2>();
    case 4: return pick_variant<QT, KV, D, 4>();
    case 8: return pick_variant<QT, KV, D, 8>();
    default: return nullptr;
  }
}

template <typename QT, typename KV>
DecodeLauncher pick_dim_group(int head_dim, int group) {
  if (head_dim == 64) return pick_group<QT, KV, 64>(group);
  if (head_dim == 128) return pick_group<QT, KV, 128>(group);
  return nullptr;
}

}  // namespace pkv
