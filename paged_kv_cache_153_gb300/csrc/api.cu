// C-ABI entry points for decode attention: argument checks, workspace
// planning and dispatch to the compiled kernel variants.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdlib>
#include <mutex>
#include <new>

#include "decode_launch.cuh"
#include "host_util.h"

#include <cudaTypedefs.h>

#include <cstdio>
#include <cstring>

namespace pkv {

namespace {
thread_local char g_last_error[256] = "";
}

bool cuda_failed(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return false;
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", what, cudaGetErrorName(e),
                cudaGetErrorString(e));
  cudaGetLastError();   // clear the non-sticky error state
  return true;
}

bool encode_cache_tmap(CUtensorMap* map, const void* base, int64_t rows, int head_dim, int elt_bytes) {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static cudaError_t lookup_err = cudaSuccess;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    lookup_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (lookup_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (encode == nullptr) {
    cuda_failed(lookup_err == cudaSuccess ? cudaErrorSymbolNotFound : lookup_err,
                "cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)");
    return false;
  }
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * elt_bytes};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elt_bytes), 16};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, elt_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled: CUresult %d", static_cast<int>(r));
    return false;
  }
  return true;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int env_int(const char* name, int fallback) {
  const char* v = std::getenv(name);
  if (v == nullptr || *v == '\0') return fallback;
  return std::atoi(v);
}

constexpr int kMaxCtasPerSm = 4;   // partial slots are sized for this many blocks per SM

int sm_count() {
  int dev = 0, n = 0;
  if (cuda_failed(cudaGetDevice(&dev), "cudaGetDevice")) return 0;
  if (cuda_failed(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute"))
    return 0;
  return n;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
  size_t cum_off, ml_off, o_off, total;
  int64_t slots, ranges_cap;
};

// Workspace: [2 (B + 1)] int32 block-count and non-empty-sequence prefixes |
// [slots, G, 2] fp32 (m, l) | [slots, G, D] fp32 o.  Two partial slots per
// range of the split.
bool ws_layout(int batch, int n_kv_heads, int group, int head_dim, int max_blocks_per_seq, int max_context_len,
               int partition_tokens, int num_sms, WsLayout* w) {
  if (batch < 0 || n_kv_heads <= 0 || group <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 ||
      max_context_len < 0 || partition_tokens < 0 || num_sms <= 0)
    return false;
  if (partition_tokens % kBlockSize) return false;
  // one range per resident decode block; a partition split never has more
  // ranges than partitions
  int64_t ranges = static_cast<int64_t>(num_sms) * kMaxCtasPerSm;
  if (partition_tokens > 0) {
    const int64_t nblk = std::min<int64_t>(max_blocks_per_seq, (max_context_len + kBlockSize - 1) / kBlockSize);
    const int64_t w_max = static_cast<int64_t>(batch) * n_kv_heads * nblk;
    const int64_t pb = partition_tokens / kBlockSize;
    ranges = std::min(ranges, std::max<int64_t>((w_max + pb - 1) / pb, 1));
  }
  w->ranges_cap = ranges;
  w->slots = 2 * ranges;
  w->cum_off = 0;
  w->ml_off = round256(sizeof(int32_t) * 2 * (static_cast<size_t>(batch) + 1));
  w->o_off = w->ml_off + round256(sizeof(float) * 2 * group * static_cast<size_t>(w->slots));
  w->total = w->o_off + round256(sizeof(float) * static_cast<size_t>(head_dim) * group * w->slots);
  return true;
}

pkv_status decode_common(int kv_kind, const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                         const float* v_scale, const int32_t* block_tables, const int32_t* context_lens,
                         int batch, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                         int max_blocks_per_seq, int64_t num_blocks, int max_context_len, float scale, void* out,
                         pkv_dtype dtype, int partition_tokens, void* workspace, size_t workspace_bytes,
                         int32_t* err_flag, void* stream, const void* k_new = nullptr, const void* v_new = nullptr,
                         int64_t* slots_out = nullptr, int num_layers = 1, int layer = 0,
                         const void* slab_params = nullptr, bool wait_first = false) {
  // kv_kind: 0 = 16-bit cache, 1 = E4M3 with per-head scales, 2 = INT8 with
  // per-(block, head) min-max parameters, 3 = E5M2 with per-head scales
  const bool fp8 = kv_kind == 1 || kv_kind == 3, int8 = kv_kind == 2;
  if (batch < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || max_blocks_per_seq <= 0 || num_blocks < 0 ||
      max_context_len < 0 || partition_tokens < 0 || !std::isfinite(scale))
    return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (n_q_heads % n_kv_heads) return PKV_ERR_INVALID_ARG;
  if (partition_tokens % kBlockSize) return PKV_ERR_INVALID_ARG;
  const int group = n_q_heads / n_kv_heads;
  if (block_size != kBlockSize || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
  if (group != 1 && group != 2 && group != 4 && group != 8) return PKV_ERR_UNSUPPORTED;
  if (num_layers < 1 || layer < 0 || layer >= num_layers) return PKV_ERR_INVALID_ARG;
  if (batch == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !workspace)
    return PKV_ERR_INVALID_ARG;
  if (fp8 && (!k_scale || !v_scale)) return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(workspace))
    return PKV_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_INVALID_ARG;
  if (k_new != nullptr && (!aligned16(k_new) || !aligned16(v_new))) return PKV_ERR_INVALID_ARG;
  const int num_sms = sm_count();
  if (num_sms <= 0) return PKV_ERR_CUDA;
  WsLayout w;
  if (!ws_layout(batch, n_kv_heads, group, head_dim, max_blocks_per_seq, max_context_len, partition_tokens,
                 num_sms, &w))
    return PKV_ERR_INVALID_ARG;
  if (workspace_bytes < w.total) return PKV_ERR_WORKSPACE;
  if (w.slots > INT32_MAX) return PKV_ERR_UNSUPPORTED;

  if (int8 && (!slab_params || (reinterpret_cast<uintptr_t>(slab_params) & 15u) || k_new != nullptr))
    return PKV_ERR_INVALID_ARG;
  DecodeLauncher launch = int8 ? decode_launcher_int8(dtype, head_dim, group)
                        : kv_kind == 3 ? decode_launcher_e5m2(dtype, head_dim, group)
                        : fp8 ? decode_launcher_e4m3(dtype, head_dim, group)
                              : (dtype == PKV_F16 ? decode_launcher_f16(head_dim, group)
                                                  : decode_launcher_bf16(head_dim, group));
  if (launch == nullptr) return PKV_ERR_UNSUPPORTED;

  char* ws = static_cast<char*>(workspace);
  DecodeParams p{};
  p.q = q;
  // A layer-major cache [num_blocks, num_layers, H_kv, 16, d]: this layer's
  // view starts layer * H_kv slabs into block 0, and blocks are num_layers *
  // H_kv slabs apart (per-layer scales [num_layers, H_kv]).
  const int64_t slab_bytes = static_cast<int64_t>(kBlockSize) * head_dim * (kv_kind ? 1 : 2);
  const int64_t layer_off = static_cast<int64_t>(layer) * n_kv_heads * slab_bytes;
  p.k_cache = k_cache ? static_cast<const char*>(k_cache) + layer_off : nullptr;
  p.v_cache = v_cache ? static_cast<const char*>(v_cache) + layer_off : nullptr;
  p.k_scale = fp8 ? k_scale + static_cast<int64_t>(layer) * n_kv_heads : nullptr;
  p.v_scale = fp8 ? v_scale + static_cast<int64_t>(layer) * n_kv_heads : nullptr;
  p.block_heads = num_layers * n_kv_heads;
  p.slab_params = int8 ? static_cast<const float4*>(slab_params) + static_cast<int64_t>(layer) * n_kv_heads
                       : nullptr;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = out;
  p.k_new = k_new;
  p.v_new = v_new;
  p.slots_out = slots_out;
  p.ws_cum = reinterpret_cast<int32_t*>(ws + w.cum_off);
  p.ws_ml = reinterpret_cast<float*>(ws + w.ml_off);
  p.ws_o = reinterpret_cast<float*>(ws + w.o_off);
  p.err = err_flag;
  p.num_blocks = num_blocks;
  p.batch = batch;
  p.n_q_heads = n_q_heads;
  p.n_kv_heads = n_kv_heads;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.max_nblk = (max_context_len + kBlockSize - 1) / kBlockSize;
  p.part_blocks = partition_tokens / kBlockSize;
  // (-1: the launched variant's default cost per (sequence, KV head))
  p.unit_cost = std::max(-1, std::min(1 << 16, env_int("PKV_UNIT_COST", -1)));
  p.slot_capacity = static_cast<int>(w.slots);
  p.wait_first = wait_first ? 1 : 0;
  p.qk_scale_log2 = scale * kLog2e;
  // limit of each pipeline wait of the decode kernel: 1 s, or (for tests of
  // the timeout path) PKV_WAIT_LIMIT_NS nanoseconds
  {
    const char* v = std::getenv("PKV_WAIT_LIMIT_NS");
    const long long lim = (v != nullptr && *v != '\0') ? std::atoll(v) : 0;
    p.wait_limit_ns = lim > 0 ? static_cast<unsigned long long>(lim) : kWaitLimitNs;
  }

  LaunchInfo li{};
  li.num_sms = num_sms;
  li.max_ctas_per_sm = std::max(0, std::min(kMaxCtasPerSm, env_int("PKV_CTAS_PER_SM", 0)));
  li.stages = env_int("PKV_STAGES", 0);
  li.part_ranges_cap = w.ranges_cap;
  return launch(p, li, static_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int pkv_version(void) { return 100; }

extern "C" const char* pkv_last_error(void) { return g_last_error; }

extern "C" const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_NO_BLOCKS: return "no free block in the pool";
    case PKV_ERR_OOB: return "block id, slot or context length out of range";
    case PKV_ERR_CUDA: return "CUDA runtime error";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_TIMEOUT: return "an internal device wait timed out";
    default: return "unknown status";
  }
}

extern "C" size_t pkv_decode_workspace_bytes(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                             int max_blocks_per_seq, int max_context_len, int partition_tokens) {
  if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads) return 0;
  const int num_sms = sm_count();
  if (num_sms <= 0) return 0;
  WsLayout w;
  if (!ws_layout(batch, num_kv_heads, num_q_heads / num_kv_heads, head_dim, max_blocks_per_seq, max_context_len,
                 partition_tokens, num_sms, &w))
    return 0;
  return w.total;
}

extern "C" pkv_status pkv_paged_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                                 const int32_t* block_tables, const int32_t* context_lens,
                                                 int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                                 int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                                 int max_context_len, float scale, void* out, pkv_dtype dtype,
                                                 int partition_tokens, void* workspace, size_t workspace_bytes,
                                                 int32_t* err_flag, void* stream) {
  return decode_common(false, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens, batch,
                       num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
                       max_context_len, scale, out, dtype, partition_tokens, workspace, workspace_bytes, err_flag,
                       stream);
}

extern "C" pkv_status pkv_paged_decode_attention_fp8(const void* q, const uint8_t* k_cache,
                                                     const uint8_t* v_cache, const float* k_scale,
                                                     const float* v_scale, const int32_t* block_tables,
                                                     const int32_t* context_lens, int batch, int num_q_heads,
                                                     int num_kv_heads, int head_dim, int block_size,
                                                     int max_blocks_per_seq, int64_t num_blocks,
                                                     int max_context_len, float scale, void* out,
                                                     pkv_dtype q_dtype, int partition_tokens, void* workspace,
                                                     size_t workspace_bytes, int32_t* err_flag, void* stream) {
  return decode_common(true, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, batch,
                       num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
                       max_context_len, scale, out, q_dtype, partition_tokens, workspace, workspace_bytes,
                       err_flag, stream);
}

extern "C" pkv_status pkv_paged_decode_attention_e5m2(const void* q, const uint8_t* k_cache,
                                                      const uint8_t* v_cache, const float* k_scale,
                                                      const float* v_scale, const int32_t* block_tables,
                                                      const int32_t* context_lens, int batch, int num_q_heads,
                                                      int num_kv_heads, int head_dim, int block_size,
                                                      int max_blocks_per_seq, int64_t num_blocks,
                                                      int max_context_len, float scale, void* out,
                                                      pkv_dtype q_dtype, int partition_tokens, void* workspace,
                                                      size_t workspace_bytes, int32_t* err_flag, void* stream) {
  return decode_common(3, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, batch, num_q_heads,
                       num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, max_context_len, scale,
                       out, q_dtype, partition_tokens, workspace, workspace_bytes, err_flag, stream);
}

extern "C" pkv_status pkv_paged_decode_step_e5m2(const void* q, const void* k_new, const void* v_new,
                                                 uint8_t* k_cache, uint8_t* v_cache, const float* k_scale,
                                                 const float* v_scale, const int32_t* block_tables,
                                                 const int32_t* context_lens, int batch, int num_q_heads,
                                                 int num_kv_heads, int head_dim, int block_size,
                                                 int max_blocks_per_seq, int64_t num_blocks, int max_context_len,
                                                 float scale, void* out, pkv_dtype q_dtype, int partition_tokens,
                                                 int64_t* slot_mapping_out, void* workspace, size_t workspace_bytes,
                                                 int32_t* err_flag, void* stream) {
  if (batch > 0 && (k_new == nullptr || v_new == nullptr)) return PKV_ERR_INVALID_ARG;
  return decode_common(3, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, batch, num_q_heads,
                       num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, max_context_len, scale,
                       out, q_dtype, partition_tokens, workspace, workspace_bytes, err_flag, stream, k_new, v_new,
                       slot_mapping_out);
}

extern "C" pkv_status pkv_paged_decode_step(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                            void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
                                            int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                            int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                            int max_context_len, float scale, void* out, pkv_dtype dtype,
                                            int partition_tokens, int64_t* slot_mapping_out, void* workspace,
                                            size_t workspace_bytes, int32_t* err_flag, void* stream) {
  if (batch > 0 && (k_new == nullptr || v_new == nullptr)) return PKV_ERR_INVALID_ARG;
  return decode_common(false, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens, batch,
                       num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
                       max_context_len, scale, out, dtype, partition_tokens, workspace, workspace_bytes, err_flag,
                       stream, k_new, v_new, slot_mapping_out);
}

extern "C" pkv_status pkv_paged_decode_attention_int8(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                                      const float* slab_params, const int32_t* block_tables,
                                                      const int32_t* context_lens, int batch, int num_q_heads,
                                                      int num_kv_heads, int head_dim, int block_size,
                                                      int max_blocks_per_seq, int64_t num_blocks, int max_context_len,
                                                      float scale, void* out, pkv_dtype q_dtype, int partition_tokens,
                                                      void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                                      void* stream) {
  return decode_common(2, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens, batch, num_q_heads,
                       num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, max_context_len, scale,
                       out, q_dtype, partition_tokens, workspace, workspace_bytes, err_flag, stream, nullptr, nullptr,
                       nullptr, 1, 0, slab_params);
}

extern "C" pkv_status pkv_paged_decode_step_int8(const void* q, const void* k_new, const void* v_new,
                                                 uint8_t* k_cache, uint8_t* v_cache, float* slab_params,
                                                 const int32_t* block_tables, const int32_t* context_lens, int batch,
                                                 int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                                 int max_blocks_per_seq, int64_t num_blocks, int max_context_len,
                                                 float scale, void* out, pkv_dtype q_dtype, int partition_tokens,
                                                 int64_t* slot_mapping_out, void* workspace, size_t workspace_bytes,
                                                 int32_t* err_flag, void* stream) {
  // checks of pkv_kv_append_int8 and of the decode, before any launch
  if (batch < 0 || num_kv_heads <= 0 || num_blocks < 0 || max_blocks_per_seq <= 0) return PKV_ERR_INVALID_ARG;
  if (q_dtype != PKV_F16 && q_dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (block_size != kBlockSize || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
  if (batch == 0) return PKV_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slab_params || !block_tables || !context_lens || !q || !out ||
      !workspace ||
      ((reinterpret_cast<uintptr_t>(slab_params) | reinterpret_cast<uintptr_t>(k_cache) |
        reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out) |
        reinterpret_cast<uintptr_t>(workspace)) & 15u))
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_q_heads % num_kv_heads || max_context_len < 0 || partition_tokens < 0 ||
      partition_tokens % kBlockSize || !std::isfinite(scale))
    return PKV_ERR_INVALID_ARG;
  {
    const int group = num_q_heads / num_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8) return PKV_ERR_UNSUPPORTED;
    const size_t need = pkv_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                                   max_context_len, partition_tokens);
    if (need == 0) return PKV_ERR_CUDA;
    if (workspace_bytes < need) return PKV_ERR_WORKSPACE;
  }
  const pkv_status st = launch_append_int8_step(k_new, v_new, k_cache, v_cache, slab_params, block_tables,
                                                context_lens, batch, max_blocks_per_seq, num_blocks, num_kv_heads,
                                                head_dim, q_dtype, slot_mapping_out, err_flag,
                                                static_cast<cudaStream_t>(stream));
  if (st != PKV_OK) return st;
  return decode_common(2, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens, batch, num_q_heads,
                       num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, max_context_len, scale,
                       out, q_dtype, partition_tokens, workspace, workspace_bytes, err_flag, stream, nullptr, nullptr,
                       nullptr, 1, 0, slab_params, true);
}

extern "C" pkv_status pkv_paged_decode_step_layer(const void* q, const void* k_new, const void* v_new,
                                                  void* k_cache, void* v_cache, const int32_t* block_tables,
                                                  const int32_t* context_lens, int batch, int num_q_heads,
                                                  int num_kv_heads, int head_dim, int block_size,
                                                  int max_blocks_per_seq, int64_t num_blocks, int num_layers,
                                                  int layer, int max_context_len, float scale, void* out,
                                                  pkv_dtype dtype, int partition_tokens, int64_t* slot_mapping_out,
                                                  void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                                  void* stream) {
  if (batch > 0 && (k_new == nullptr || v_new == nullptr)) return PKV_ERR_INVALID_ARG;
  return decode_common(false, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens, batch,
                       num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
                       max_context_len, scale, out, dtype, partition_tokens, workspace, workspace_bytes, err_flag,
                       stream, k_new, v_new, slot_mapping_out, num_layers, layer);
}

// One decode step over every layer of a layer-major cache, captured once into
// a CUDA graph and replayed with one launch.
struct pkv_step_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

extern "C" void pkv_step_graph_destroy(pkv_step_graph* g) {
  if (g == nullptr) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  delete g;
}

extern "C" pkv_status pkv_step_graph_create(pkv_step_graph** out_graph, const void* q, const void* k_new,
                                            const void* v_new, void* k_cache, void* v_cache,
                                            const int32_t* block_tables, const int32_t* context_lens, int batch,
                                            int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                            int max_blocks_per_seq, int64_t num_blocks, int num_layers,
                                            int max_context_len, float scale, void* out, pkv_dtype dtype,
                                            int partition_tokens, int64_t* slot_mapping_out, void* workspace,
                                            size_t workspace_bytes, int32_t* err_flag) {
  if (out_graph == nullptr || num_layers < 1 || batch <= 0 || !q || !k_new || !v_new || !out)
    return PKV_ERR_INVALID_ARG;
  *out_graph = nullptr;
  const int64_t q_layer = static_cast<int64_t>(batch) * num_q_heads * head_dim * 2;
  const int64_t kv_layer = static_cast<int64_t>(batch) * num_kv_heads * head_dim * 2;
  cudaStream_t cs = nullptr;
  if (cuda_failed(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking), "cudaStreamCreateWithFlags"))
    return PKV_ERR_CUDA;
  pkv_step_graph* g = new (std::nothrow) pkv_step_graph;
  if (g == nullptr) {
    cudaStreamDestroy(cs);
    return PKV_ERR_CUDA;
  }
  pkv_status st = PKV_OK;
  if (cuda_failed(cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed), "cudaStreamBeginCapture")) {
    st = PKV_ERR_CUDA;
  } else {
    for (int l = 0; l < num_layers && st == PKV_OK; ++l)
      st = decode_common(false, static_cast<const char*>(q) + l * q_layer, k_cache, v_cache, nullptr, nullptr,
                         block_tables, context_lens, batch, num_q_heads, num_kv_heads, head_dim, block_size,
                         max_blocks_per_seq, num_blocks, max_context_len, scale, static_cast<char*>(out) + l * q_layer,
                         dtype, partition_tokens, workspace, workspace_bytes, err_flag, cs,
                         static_cast<const char*>(k_new) + l * kv_layer, static_cast<const char*>(v_new) + l * kv_layer,
                         slot_mapping_out, num_layers, l);
    const cudaError_t e = cudaStreamEndCapture(cs, &g->graph);
    if (st == PKV_OK && cuda_failed(e, "cudaStreamEndCapture")) st = PKV_ERR_CUDA;
  }
  if (st == PKV_OK && cuda_failed(cudaGraphInstantiate(&g->exec, g->graph, 0), "cudaGraphInstantiate"))
    st = PKV_ERR_CUDA;
  cudaStreamDestroy(cs);
  if (st != PKV_OK) {
    pkv_step_graph_destroy(g);
    return st;
  }
  *out_graph = g;
  return PKV_OK;
}

extern "C" pkv_status pkv_step_graph_launch(pkv_step_graph* g, void* stream) {
  if (g == nullptr || g->exec == nullptr) return PKV_ERR_INVALID_ARG;
  return cuda_failed(cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream)), "cudaGraphLaunch") ? PKV_ERR_CUDA
                                                                                                     : PKV_OK;
}

extern "C" pkv_status pkv_paged_decode_step_fp8(const void* q, const void* k_new, const void* v_new,
                                                uint8_t* k_cache, uint8_t* v_cache, const float* k_scale,
                                                const float* v_scale, const int32_t* block_tables,
                                                const int32_t* context_lens, int batch, int num_q_heads,
                                                int num_kv_heads, int head_dim, int block_size,
                                                int max_blocks_per_seq, int64_t num_blocks, int max_context_len,
                                                float scale, void* out, pkv_dtype q_dtype, int partition_tokens,
                                                int64_t* slot_mapping_out, void* workspace, size_t workspace_bytes,
                                                int32_t* err_flag, void* stream) {
  if (batch > 0 && (k_new == nullptr || v_new == nullptr)) return PKV_ERR_INVALID_ARG;
  return decode_common(true, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, batch,
                       num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
                       max_context_len, scale, out, q_dtype, partition_tokens, workspace, workspace_bytes, err_flag,
                       stream, k_new, v_new, slot_mapping_out);
}

extern "C" pkv_status pkv_decode_step_host(const void* h_q, const void* h_k_new, const void* h_v_new,
                                           const int32_t* h_block_tables, const int32_t* h_context_lens,
                                           void* h_out, void* d_q, void* d_k_new, void* d_v_new,
                                           int32_t* d_block_tables, int32_t* d_context_lens, int64_t* d_slots,
                                           void* d_out, void* k_cache, void* v_cache, int batch,
                                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                           int max_blocks_per_seq, int64_t num_blocks, int max_context_len,
                                           float scale, pkv_dtype dtype, int partition_tokens, void* workspace,
                                           size_t workspace_bytes, int32_t* err_flag, void* stream) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0)
    return PKV_ERR_INVALID_ARG;
  if (batch == 0) return PKV_OK;
  if (!h_q || !h_k_new || !h_v_new || !h_block_tables || !h_context_lens || !h_out || !d_q || !d_k_new ||
      !d_v_new || !d_block_tables || !d_context_lens || !d_slots || !d_out)
    return PKV_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t qo_bytes = static_cast<size_t>(batch) * num_q_heads * head_dim * 2;
  const size_t kv_bytes = static_cast<size_t>(batch) * num_kv_heads * head_dim * 2;
  const size_t tab_bytes = static_cast<size_t>(batch) * max_blocks_per_seq * sizeof(int32_t);
  if (cuda_failed(cudaMemcpyAsync(d_q, h_q, qo_bytes, cudaMemcpyHostToDevice, s), "cudaMemcpyAsync q") ||
      cuda_failed(cudaMemcpyAsync(d_k_new, h_k_new, kv_bytes, cudaMemcpyHostToDevice, s), "cudaMemcpyAsync k") ||
      cuda_failed(cudaMemcpyAsync(d_v_new, h_v_new, kv_bytes, cudaMemcpyHostToDevice, s), "cudaMemcpyAsync v") ||
      cuda_failed(cudaMemcpyAsync(d_block_tables, h_block_tables, tab_bytes, cudaMemcpyHostToDevice, s),
                  "cudaMemcpyAsync tables") ||
      cuda_failed(cudaMemcpyAsync(d_context_lens, h_context_lens, sizeof(int32_t) * batch,
                                  cudaMemcpyHostToDevice, s),
                  "cudaMemcpyAsync lens"))
    return PKV_ERR_CUDA;
  const pkv_status st = pkv_paged_decode_step(d_q, d_k_new, d_v_new, k_cache, v_cache, d_block_tables,
                                              d_context_lens, batch, num_q_heads, num_kv_heads, head_dim, block_size,
                                              max_blocks_per_seq, num_blocks, max_context_len, scale, d_out, dtype,
                                              partition_tokens, d_slots, workspace, workspace_bytes, err_flag,
                                              stream);
  if (st != PKV_OK) return st;
  if (cuda_failed(cudaMemcpyAsync(h_out, d_out, qo_bytes, cudaMemcpyDeviceToHost, s), "cudaMemcpyAsync out"))
    return PKV_ERR_CUDA;
  return PKV_OK;
}
