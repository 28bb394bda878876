// Host-side helpers shared by the C-ABI translation units.
#pragma once

#include <cuda_runtime.h>

namespace pkv {

// Record a failed CUDA runtime call (name + error) for pkv_last_error() and
// clear the runtime's last-error state so it cannot leak into a later call.
// Returns true when `e` is an error.
bool cuda_failed(cudaError_t e, const char* what);

}  // namespace pkv
