// Internal declarations shared by the translation units of libpagedkv.so.
#pragma once
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

struct PoolGeometry {
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    pkv_dtype dtype;
};

// Geometry of a pool ledger; false on NULL.
bool pool_geometry(const pkv_pool *p, PoolGeometry *g);

inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace pkv
