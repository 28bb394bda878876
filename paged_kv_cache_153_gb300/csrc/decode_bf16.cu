// bf16 q / bf16 cache decode variants.
#include "decode_launch.cuh"

namespace pkv {
DecodeLauncher decode_launcher_bf16(int head_dim, int group) { return pick_dim_group<BF16, BF16>(head_dim, group); }
}  // namespace pkv
