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

// Some block of the pool is referenced by two or more sequences right now.
bool pool_has_shared_blocks(const pkv_pool *p);

inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Element type of the pool is fp16 or bf16 (not an 8-bit cache).
inline bool is_16bit(const PoolGeometry &g) { return g.dtype == PKV_F16 || g.dtype == PKV_BF16; }

// Pool holds 8-bit codes with fp16 scales.
inline bool is_8bit(const PoolGeometry &g) { return g.dtype == PKV_Q8_BF16 || g.dtype == PKV_Q8_F16; }

}  // namespace pkv
