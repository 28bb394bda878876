// Host-side block pool: preallocated block ids handed out on demand, with
// reference counts for blocks shared by several block tables ("Series 03: why
// the KV cache eats memory, and how PagedAttention pages it", sections 3.2 and
// 3.3).  LIFO free list; the first allocations return 0, 1, 2, ...
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pkv.h"

struct pkv_pool {
  int64_t num_blocks;
  int block_size;
  std::vector<int32_t> free_stack;   // back() is the next id handed out
  std::vector<int32_t> refs;
};

extern "C" pkv_pool* pkv_pool_create(int64_t num_blocks, int block_size) {
  if (num_blocks < 0 || num_blocks > INT32_MAX || block_size <= 0) return nullptr;
  pkv_pool* p = new (std::nothrow) pkv_pool;
  if (p == nullptr) return nullptr;
  try {
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->refs.assign(static_cast<size_t>(num_blocks), 0);
    p->free_stack.reserve(static_cast<size_t>(num_blocks));
    for (int64_t i = num_blocks - 1; i >= 0; --i) p->free_stack.push_back(static_cast<int32_t>(i));
  } catch (...) {
    delete p;
    return nullptr;
  }
  return p;
}

extern "C" void pkv_pool_destroy(pkv_pool* pool) { delete pool; }

extern "C" pkv_status pkv_pool_alloc(pkv_pool* pool, int32_t* block_id) {
  if (pool == nullptr || block_id == nullptr) return PKV_ERR_INVALID_ARG;
  if (pool->free_stack.empty()) return PKV_ERR_NO_BLOCKS;
  const int32_t id = pool->free_stack.back();
  pool->free_stack.pop_back();
  pool->refs[id] = 1;
  *block_id = id;
  return PKV_OK;
}

static bool allocated(const pkv_pool* pool, int32_t id) {
  return pool != nullptr && id >= 0 && id < pool->num_blocks && pool->refs[id] > 0;
}

extern "C" pkv_status pkv_pool_incref(pkv_pool* pool, int32_t block_id) {
  if (!allocated(pool, block_id)) return PKV_ERR_INVALID_ARG;
  ++pool->refs[block_id];
  return PKV_OK;
}

extern "C" pkv_status pkv_pool_decref(pkv_pool* pool, int32_t block_id) {
  if (!allocated(pool, block_id)) return PKV_ERR_INVALID_ARG;
  if (--pool->refs[block_id] == 0) pool->free_stack.push_back(block_id);
  return PKV_OK;
}

extern "C" int64_t pkv_pool_num_free(const pkv_pool* pool) {
  return pool == nullptr ? -1 : static_cast<int64_t>(pool->free_stack.size());
}

extern "C" int32_t pkv_pool_refcount(const pkv_pool* pool, int32_t block_id) {
  if (pool == nullptr || block_id < 0 || block_id >= pool->num_blocks) return -1;
  return pool->refs[block_id];
}

extern "C" int64_t pkv_blocks_needed(int64_t num_tokens, int block_size) {
  if (num_tokens < 0 || block_size <= 0) return -1;
  return (num_tokens + block_size - 1) / block_size;
}

extern "C" pkv_status pkv_pool_cow(pkv_pool* pool, int32_t block_id, int32_t* out_id) {
  if (!allocated(pool, block_id) || out_id == nullptr) return PKV_ERR_INVALID_ARG;
  if (pool->refs[block_id] == 1) {
    *out_id = block_id;
    return PKV_OK;
  }
  int32_t fresh = -1;
  const pkv_status st = pkv_pool_alloc(pool, &fresh);
  if (st != PKV_OK) return st;
  --pool->refs[block_id];   // still >= 1: the other sharers keep it
  *out_id = fresh;
  return PKV_OK;
}

extern "C" pkv_status pkv_prepare_append(pkv_pool* pool, int32_t* block_tables, int batch, int max_blocks_per_seq,
                                         const int32_t* context_lens, int32_t* src_blocks, int32_t* dst_blocks,
                                         int32_t* num_pairs) {
  if (pool == nullptr || batch < 0 || max_blocks_per_seq <= 0 || num_pairs == nullptr) return PKV_ERR_INVALID_ARG;
  if (batch > 0 && (block_tables == nullptr || context_lens == nullptr || src_blocks == nullptr ||
                    dst_blocks == nullptr))
    return PKV_ERR_INVALID_ARG;
  const int bs = pool->block_size;
  // Pass 1: validate and count the blocks the step takes, following the
  // reference counts as the copies of earlier rows lower them.
  std::unordered_map<int32_t, int32_t> dropped;   // block -> references given up so far
  int64_t need = 0;
  for (int b = 0; b < batch; ++b) {
    const int32_t ctx = context_lens[b];
    if (ctx < 0) return PKV_ERR_INVALID_ARG;
    if (ctx == 0) continue;
    const int64_t i = (static_cast<int64_t>(ctx) - 1) / bs;
    if (i >= max_blocks_per_seq) return PKV_ERR_INVALID_ARG;
    const int32_t id = block_tables[static_cast<int64_t>(b) * max_blocks_per_seq + i];
    if (id < 0) {
      ++need;
      continue;
    }
    if (!allocated(pool, id)) return PKV_ERR_INVALID_ARG;
    auto it = dropped.find(id);
    const int32_t left = pool->refs[id] - (it == dropped.end() ? 0 : it->second);
    if (left > 1) {
      ++need;
      ++dropped[id];
    }
  }
  if (need > static_cast<int64_t>(pool->free_stack.size())) return PKV_ERR_NO_BLOCKS;
  // Pass 2: apply (cannot fail now).
  int32_t n = 0;
  for (int b = 0; b < batch; ++b) {
    const int32_t ctx = context_lens[b];
    if (ctx == 0) continue;
    const int64_t i = (static_cast<int64_t>(ctx) - 1) / bs;
    int32_t& entry = block_tables[static_cast<int64_t>(b) * max_blocks_per_seq + i];
    int32_t id = -1;
    if (entry < 0) {
      pkv_pool_alloc(pool, &id);
      entry = id;
      continue;
    }
    pkv_pool_cow(pool, entry, &id);
    if (id != entry) {
      src_blocks[n] = entry;
      dst_blocks[n] = id;
      ++n;
      entry = id;
    }
  }
  *num_pairs = n;
  return PKV_OK;
}
