// Host-side launch of one decode-kernel variant plus its combine kernel.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

#include "decode.cuh"
#include "host_util.h"

namespace pkv {

struct LaunchInfo {
  int num_sms;
  int max_ctas_per_sm;     // cap on resident decode blocks per SM
  int stages;              // 0 = default for the variant
  int grid;                // out: decode grid used
  int64_t part_ranges_cap; // partition mode: max ranges the workspace holds
};

using DecodeLauncher = pkv_status (*)(DecodeParams&, LaunchInfo&, cudaStream_t);

constexpr int kDefaultRingBytes = 64 * 1024;
constexpr int kMaxDevices = 64;

template <typename QT, typename KV, int D, int G, int NW>
pkv_status launch_decode_variant(DecodeParams& p, LaunchInfo& li, cudaStream_t stream) {
  using Tr = DecodeTraits<D, G, NW, KV>;
  auto kern = paged_decode_kernel<QT, KV, D, G, NW>;
  int stages = li.stages > 0 ? li.stages : kDefaultRingBytes / Tr::kStage;
  if (stages < 2) stages = 2;
  if (stages > 32) stages = 32;
  size_t smem = Tr::smem_bytes(stages, p.batch, p.n_kv_heads);
  int max_optin = 0, dev = 0;
  if (cuda_failed(cudaGetDevice(&dev), "cudaGetDevice")) return PKV_ERR_CUDA;
  if (cuda_failed(cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev),
                  "cudaDeviceGetAttribute"))
    return PKV_ERR_CUDA;
  cudaFuncAttributes fattr;
  if (cuda_failed(cudaFuncGetAttributes(&fattr, kern), "cudaFuncGetAttributes")) return PKV_ERR_CUDA;
  // dynamic shared memory may use what the static part leaves of the opt-in limit
  const size_t dyn_max = static_cast<size_t>(max_optin) - fattr.sharedSizeBytes;
  while (smem > dyn_max && stages > 2) {
    --stages;
    smem = Tr::smem_bytes(stages, p.batch, p.n_kv_heads);
  }
  if (smem > dyn_max) return PKV_ERR_UNSUPPORTED;   // batch too large for one block's shared memory
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
  int occ = 0;
  if (cuda_failed(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, Tr::kThreads, smem),
                  "cudaOccupancyMaxActiveBlocksPerMultiprocessor"))
    return PKV_ERR_CUDA;
  if (occ < 1) return PKV_ERR_UNSUPPORTED;
  if (occ > li.max_ctas_per_sm) occ = li.max_ctas_per_sm;
  int grid = li.num_sms * occ;
  if (p.part_blocks > 0 && li.part_ranges_cap < grid) grid = static_cast<int>(li.part_ranges_cap);
  if (grid < 1) grid = 1;
  p.stages = stages;
  li.grid = grid;
  li.stages = stages;
  kern<<<grid, Tr::kThreads, smem, stream>>>(p);
  if (cuda_failed(cudaGetLastError(), "paged_decode_kernel launch")) return PKV_ERR_CUDA;
  const int units = p.batch * p.n_kv_heads;
  if (units > 0) {
    paged_decode_combine_kernel<QT, D, G><<<units, 128, 0, stream>>>(p, grid);
    if (cuda_failed(cudaGetLastError(), "paged_decode_combine_kernel launch")) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

// Variants compiled in each translation unit (by KV element type).
DecodeLauncher decode_launcher_f16(int head_dim, int group);
DecodeLauncher decode_launcher_bf16(int head_dim, int group);
DecodeLauncher decode_launcher_e4m3(int q_dtype, int head_dim, int group);

template <typename QT, typename KV, int D>
DecodeLauncher pick_group(int group) {
  switch (group) {
    case 1: return launch_decode_variant<QT, KV, D, 1, 8>;
    case 2: return launch_decode_variant<QT, KV, D, 2, 8>;
    case 4: return launch_decode_variant<QT, KV, D, 4, 8>;
    case 8: return launch_decode_variant<QT, KV, D, 8, 8>;
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
