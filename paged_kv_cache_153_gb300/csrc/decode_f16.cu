// fp16 q / fp16 cache decode variants.
#include "decode_launch.cuh"

namespace pkv {
DecodeLauncher decode_launcher_f16(int head_dim, int group) { return pick_dim_group<F16, F16>(head_dim, group); }
}  // namespace pkv
