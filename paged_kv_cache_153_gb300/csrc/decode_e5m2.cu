// E5M2 cache decode variants (q and out in fp16 or bf16).
#include "decode_launch.cuh"

namespace pkv {
DecodeLauncher decode_launcher_e5m2(int q_dtype, int head_dim, int group) {
  if (q_dtype == PKV_F16) return pick_dim_group<F16, E5M2>(head_dim, group);
  if (q_dtype == PKV_BF16) return pick_dim_group<BF16, E5M2>(head_dim, group);
  return nullptr;
}
}  // namespace pkv
