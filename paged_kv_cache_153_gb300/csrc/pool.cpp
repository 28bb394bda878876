// Host-side block pool: preallocated block ids handed out on demand, with
// reference counts for blocks shared by several block tables ("Series 03: why
// the KV cache eats memory, and how PagedAttention pages it", sections 3.2 and
// 3.3).  LIFO free list; the first allocations return 0, 1, 2, ...
#include <cstdint>
#include <new>
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
