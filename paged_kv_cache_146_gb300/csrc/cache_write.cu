// Cache-write kernel: store this step's K/V rows into their slots.
//
// "vLLM-and-PagedAttention-KR", section "가장 기본적인 decoding", steps 3-4:
// a generated token's KV goes after the tokens already in its logical block.
// Layout R1 ([block][kv_head][slot_in_block][head_dim]) and slot reading R2
// (slot = block * block_size + offset, negative = skip).
//
// HBM-bound byte copy: one thread moves one 16-byte chunk of one row of K and
// the same chunk of V, so a warp covers two 256-byte rows (head_dim 128) with
// fully coalesced 128-bit loads and stores.  Bit-exact by construction.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pagedkv.h"
#include "pkv_internal.h"

namespace {

__global__ void __launch_bounds__(256)
cache_write_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                   const int64_t *__restrict__ slot_mapping, int64_t num_chunks,
                   int32_t chunks_per_token, int32_t chunks_per_row, int32_t num_kv_heads,
                   int32_t block_size, int64_t num_slots, uint4 *__restrict__ k_pool,
                   uint4 *__restrict__ v_pool, int32_t *__restrict__ status)
{
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < num_chunks;
         e += (int64_t)gridDim.x * blockDim.x) {
        int64_t t = e / chunks_per_token;
        int32_t within = (int32_t)(e - t * chunks_per_token);
        int32_t h = within / chunks_per_row;
        int32_t c = within - h * chunks_per_row;
        int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (within == 0) atomicOr(status, PKV_DEV_BAD_SLOT);
            continue;
        }
        int64_t block = slot / block_size;
        int64_t offset = slot - block * block_size;
        int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * chunks_per_row + c;
        uint4 kv = __ldcs(k_new + e);   // streamed once
        uint4 vv = __ldcs(v_new + e);
        k_pool[dst] = kv;
        v_pool[dst] = vv;
    }
}

// Copy-on-write: block dst[i] receives block src[i] (K and V, all kv heads),
// 16 bytes per thread; pairs naming a block outside the pool are skipped and
// flagged.  The destinations are fresh blocks, so pairs never overlap.
__global__ void __launch_bounds__(256)
block_copy_kernel(const int32_t *__restrict__ src, const int32_t *__restrict__ dst, int32_t n,
                  int64_t chunks_per_block, int32_t num_blocks, uint4 *__restrict__ k_pool,
                  uint4 *__restrict__ v_pool, int32_t *__restrict__ status)
{
    const int64_t total = (int64_t)n * chunks_per_block;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = e / chunks_per_block;
        const int64_t c = e - i * chunks_per_block;
        const int32_t a = __ldg(src + i), b = __ldg(dst + i);
        if (a < 0 || a >= num_blocks || b < 0 || b >= num_blocks) {
            if (c == 0) atomicOr(status, PKV_DEV_BAD_BLOCK);
            continue;
        }
        k_pool[(int64_t)b * chunks_per_block + c] = k_pool[(int64_t)a * chunks_per_block + c];
        if (v_pool)     // 8-bit pools: one pool of records
            v_pool[(int64_t)b * chunks_per_block + c] = v_pool[(int64_t)a * chunks_per_block + c];
    }
}

// Swap staging: gather blocks ids[0..n) into staging [n][K|V][Hkv][16][D]
// (to_staging = true) or scatter staging back into blocks ids (false); an 8-bit
// pool (v_pool NULL) stages [n][Hkv][record].  One thread per 16-byte chunk;
// out-of-pool ids are skipped and flagged.
__global__ void __launch_bounds__(256)
swap_kernel(const int32_t *__restrict__ ids, int32_t n, int64_t chunks_per_block, int32_t num_blocks,
            uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool, uint4 *__restrict__ staging,
            bool to_staging, int32_t *__restrict__ status)
{
    const int64_t total = (int64_t)n * chunks_per_block;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = e / chunks_per_block;
        const int64_t c = e - i * chunks_per_block;
        const int32_t b = __ldg(ids + i);
        if (b < 0 || b >= num_blocks) {
            if (c == 0) atomicOr(status, PKV_DEV_BAD_BLOCK);
            continue;
        }
        const int parts = v_pool ? 2 : 1;
        uint4 *sk = staging + (parts * i) * chunks_per_block + c;
        uint4 *pk = k_pool + (int64_t)b * chunks_per_block + c;
        if (to_staging) *sk = __ldcs(pk);
        else *pk = __ldcs(sk);
        if (v_pool) {
            uint4 *sv = sk + chunks_per_block;
            uint4 *pv = v_pool + (int64_t)b * chunks_per_block + c;
            if (to_staging) *sv = __ldcs(pv);
            else *pv = __ldcs(sv);
        }
    }
}

// 8-bit cache write: quantise 4 values per lane of a 128-value row in groups
// of 32 (8 lanes): scale = fp16(min(amax / 127, 65504)), code = clamp(rn(x /
// scale), -127, 127), all decisions in fp32 with IEEE-rounded division.
template <bool BF16>
__device__ __forceinline__ void q8_quantise4(const uint16_t *src, int lane, uint32_t &codes,
                                             uint16_t &scale_bits)
{
    const uint2 raw = *reinterpret_cast<const uint2 *>(src + 4 * lane);
    const uint16_t e[4] = {(uint16_t)(raw.x & 0xffffu), (uint16_t)(raw.x >> 16),
                           (uint16_t)(raw.y & 0xffffu), (uint16_t)(raw.y >> 16)};
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        v[i] = BF16 ? __uint_as_float((uint32_t)e[i] << 16)
                    : __half2float(__ushort_as_half(e[i]));
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    const float d32 = fminf(__fdiv_rn(amax, 127.0f), 65504.0f);
    const __half dh = __float2half_rn(d32);
    const float dq = __half2float(dh);
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int c = 0;
        if (dq != 0.0f) c = max(-127, min(127, __float2int_rn(__fdiv_rn(v[i], dq))));
        w |= (uint32_t)(c & 0xff) << (8 * i);
    }
    codes = w;
    scale_bits = __half_as_ushort(dh);
}

// One warp per (token, kv head) row, head_dim 128, into the slab's record
// (layout in pagedkv.h): lane l quantises dimensions 4l .. 4l + 3 (group l / 8).
template <bool BF16>
__global__ void __launch_bounds__(256)
cache_write_q8_kernel(const uint16_t *__restrict__ k_new, const uint16_t *__restrict__ v_new,
                      const int64_t *__restrict__ slot_mapping, int64_t rows, int32_t num_kv_heads,
                      int64_t num_slots, uint8_t *__restrict__ kv, int32_t *__restrict__ status)
{
    constexpr int D = 128, BS = 16, SLAB = PKV_Q8_SLAB_BYTES;
    const int lane = threadIdx.x & 31;
    const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
        const int64_t t = r / num_kv_heads;
        const int h = (int)(r - t * num_kv_heads);
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (lane == 0) atomicOr(status, PKV_DEV_BAD_SLOT);
            continue;
        }
        const int64_t block = slot / BS;
        const int off = (int)(slot - block * BS);
        uint8_t *rec = kv + (block * num_kv_heads + h) * SLAB;
        uint32_t kc, vc;
        uint16_t ks, vs;
        q8_quantise4<BF16>(k_new + r * D, lane, kc, ks);
        q8_quantise4<BF16>(v_new + r * D, lane, vc, vs);
        // K: token off = 4a + 2b + c -> row 8b + 2a + c, chunk (lane / 4) rotated by the row
        const int row = 8 * ((off >> 1) & 1) + 2 * (off >> 2) + (off & 1);
        // codes are stored biased: byte = code + 128 (code XOR 0x80)
        *reinterpret_cast<uint32_t *>(rec + row * 128 + (((lane >> 2) ^ (row & 7)) << 4) +
                                      4 * (lane & 3)) = kc ^ 0x80808080u;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            rec[2048 + (4 * lane + i) * BS + off] = (uint8_t)(((vc >> (8 * i)) & 0xff) ^ 0x80u);
        if ((lane & 7) == 0) {
            *reinterpret_cast<uint16_t *>(rec + 4096 + off * 8 + 2 * (lane >> 3)) = ks;
            *reinterpret_cast<uint16_t *>(rec + 4224 + (lane >> 3) * 32 + off * 2) = vs;
        }
    }
}

}  // namespace

extern "C" int kv_cache_write_q8(const pkv_pool *pool, const void *k_new, const void *v_new,
                                 const int64_t *slot_mapping, int32_t num_tokens, void *kv_q8,
                                 int32_t *d_status, void *stream)
{
    pkv::PoolGeometry g;
    if (!pkv::pool_geometry(pool, &g) || num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (!pkv::is_8bit(g)) return PKV_ERR_INVALID_ARG;
    if (g.head_dim != 128 || g.block_size != 16) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !kv_q8 || !d_status) return PKV_ERR_INVALID_ARG;
    if (((uintptr_t)k_new & 7u) || ((uintptr_t)v_new & 7u) || ((uintptr_t)kv_q8 & 15u) ||
        ((uintptr_t)slot_mapping & 7u) || ((uintptr_t)d_status & 3u))
        return PKV_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)num_tokens * g.num_kv_heads;
    const int threads = 256;
    int64_t blocks = (rows * 32 + threads - 1) / threads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t slots = (int64_t)g.num_blocks * g.block_size;
    if (g.dtype == PKV_Q8_BF16)
        cache_write_q8_kernel<true><<<(unsigned)blocks, threads, 0, st>>>(
            (const uint16_t *)k_new, (const uint16_t *)v_new, slot_mapping, rows, g.num_kv_heads,
            slots, (uint8_t *)kv_q8, d_status);
    else
        cache_write_q8_kernel<false><<<(unsigned)blocks, threads, 0, st>>>(
            (const uint16_t *)k_new, (const uint16_t *)v_new, slot_mapping, rows, g.num_kv_heads,
            slots, (uint8_t *)kv_q8, d_status);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

static int launch_swap(const pkv_pool *pool, const int32_t *ids, int32_t n, void *k_pool,
                       void *v_pool, void *staging, bool to_staging, int32_t *d_status,
                       void *stream)
{
    pkv::PoolGeometry g;
    if (!pkv::pool_geometry(pool, &g) || n < 0) return PKV_ERR_INVALID_ARG;
    const bool q8 = pkv::is_8bit(g);
    if (q8) v_pool = nullptr;
    if (n == 0) return PKV_OK;
    if (!ids || !k_pool || (!q8 && !v_pool) || !staging || !d_status) return PKV_ERR_INVALID_ARG;
    if (!pkv::aligned16(k_pool) || (!q8 && !pkv::aligned16(v_pool)) || !pkv::aligned16(staging) ||
        ((uintptr_t)ids & 3u) || ((uintptr_t)d_status & 3u))
        return PKV_ERR_INVALID_ARG;
    if (q8 && (g.head_dim != 128 || g.block_size != 16)) return PKV_ERR_UNSUPPORTED;
    const int64_t block_bytes = q8 ? (int64_t)g.num_kv_heads * PKV_Q8_SLAB_BYTES
                                   : (int64_t)g.num_kv_heads * g.block_size * g.head_dim * 2;
    if (block_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
    const int64_t chunks = block_bytes / 16;
    const int threads = 256;
    int64_t blocks = ((int64_t)n * chunks + threads - 1) / threads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    swap_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
        ids, n, chunks, g.num_blocks, (uint4 *)k_pool, (uint4 *)v_pool, (uint4 *)staging,
        to_staging, d_status);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int kv_gather_blocks(const pkv_pool *pool, const int32_t *ids, int32_t n,
                                const void *k_pool, const void *v_pool, void *staging,
                                int32_t *d_status, void *stream)
{
    return launch_swap(pool, ids, n, const_cast<void *>(k_pool), const_cast<void *>(v_pool),
                       staging, true, d_status, stream);
}

extern "C" int kv_scatter_blocks(const pkv_pool *pool, const int32_t *ids, int32_t n,
                                 const void *staging, void *k_pool, void *v_pool,
                                 int32_t *d_status, void *stream)
{
    return launch_swap(pool, ids, n, k_pool, v_pool, const_cast<void *>(staging), false,
                       d_status, stream);
}

extern "C" int kv_block_copy(const pkv_pool *pool, const int32_t *src_ids, const int32_t *dst_ids,
                             int32_t n, void *k_pool, void *v_pool, int32_t *d_status,
                             void *stream)
{
    pkv::PoolGeometry g;
    if (!pkv::pool_geometry(pool, &g) || n < 0) return PKV_ERR_INVALID_ARG;
    const bool q8 = pkv::is_8bit(g);
    if (q8) v_pool = nullptr;
    if (n == 0) return PKV_OK;
    if (!src_ids || !dst_ids || !k_pool || (!q8 && !v_pool) || !d_status) return PKV_ERR_INVALID_ARG;
    if (!pkv::aligned16(k_pool) || (!q8 && !pkv::aligned16(v_pool)) || ((uintptr_t)src_ids & 3u) ||
        ((uintptr_t)dst_ids & 3u) || ((uintptr_t)d_status & 3u))
        return PKV_ERR_INVALID_ARG;
    if (q8 && (g.head_dim != 128 || g.block_size != 16)) return PKV_ERR_UNSUPPORTED;
    const int64_t block_bytes = q8 ? (int64_t)g.num_kv_heads * PKV_Q8_SLAB_BYTES
                                   : (int64_t)g.num_kv_heads * g.block_size * g.head_dim * 2;
    if (block_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
    const int64_t chunks = block_bytes / 16;
    const int threads = 256;
    int64_t blocks = ((int64_t)n * chunks + threads - 1) / threads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    block_copy_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
        src_ids, dst_ids, n, chunks, g.num_blocks, (uint4 *)k_pool, (uint4 *)v_pool, d_status);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int kv_cache_write(const pkv_pool *pool, const void *k_new, const void *v_new,
                              const int64_t *slot_mapping, int32_t num_tokens, void *k_pool,
                              void *v_pool, int32_t *d_status, void *stream)
{
    pkv::PoolGeometry g;
    if (!pkv::pool_geometry(pool, &g) || num_tokens < 0 || !pkv::is_16bit(g)) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_pool || !v_pool || !d_status)
        return PKV_ERR_INVALID_ARG;
    const int row_bytes = g.head_dim * 2;
    if (row_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
    if (!pkv::aligned16(k_new) || !pkv::aligned16(v_new) || !pkv::aligned16(k_pool) ||
        !pkv::aligned16(v_pool) || ((uintptr_t)slot_mapping & 7u) || ((uintptr_t)d_status & 3u))
        return PKV_ERR_INVALID_ARG;
    const int32_t chunks_per_row = row_bytes / 16;
    const int32_t chunks_per_token = chunks_per_row * g.num_kv_heads;
    const int64_t num_chunks = (int64_t)num_tokens * chunks_per_token;
    const int threads = 256;
    int64_t blocks = (num_chunks + threads - 1) / threads;
    if (blocks > 152 * 16) blocks = 152 * 16;   // grid-stride beyond a few waves
    cache_write_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
        (const uint4 *)k_new, (const uint4 *)v_new, slot_mapping, num_chunks, chunks_per_token,
        chunks_per_row, g.num_kv_heads, g.block_size, (int64_t)g.num_blocks * g.block_size,
        (uint4 *)k_pool, (uint4 *)v_pool, d_status);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int kv_status_check(int32_t *d_status, void *stream, int32_t *out_word)
{
    if (!d_status) return PKV_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    int32_t word = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaMemcpy(&word, d_status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (word != 0 && cudaMemset(d_status, 0, sizeof(word)) != cudaSuccess) return PKV_ERR_CUDA;
    if (out_word) *out_word = word;
    if (word & PKV_DEV_TIMEOUT) return PKV_ERR_DEVICE_TIMEOUT;
    if (word) return PKV_ERR_DEVICE_BOUNDS;
    return PKV_OK;
}
