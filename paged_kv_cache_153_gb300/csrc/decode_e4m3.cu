// E4M3 cache decode variants (q and out in fp16 or bf16).
#include "decode_launch.cuh"

namespace pkv {
DecodeLauncher decode_launcher_e4m3(int q_dtype, int head_dim, int group) {
  if (q_dtype == PKV_F16) return pick_dim_group<F16, E4M3>(head_dim, group);
  if (q_dtype == PKV_BF16) return pick_dim_group<BF16, E4M3>(head_dim, group);
  return nullptr;
}
}  // namespace pkv
