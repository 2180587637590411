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
#include <algorithm>
#include <mutex>

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

// Correctly rounded x / d from y = rn(1 / d): q0 = rn(x y) is within one ulp
// of x / d, the residual x - q0 d is exact in one fma, and rn(q0 + residual y)
// is the IEEE quotient (Markstein's theorem, "IA-64 and Elementary Functions",
// ch. 8).  It holds while the residual stays a normal number; on the values a
// group can reach (|x| <= amax, d the group's scale) it was checked against IEEE
// division for every finite bf16 and fp16 x and every positive fp16 d: the
// quotient's integer rounding agrees everywhere, and the quotient itself
// differs only below 2e-31, where the code is 0 either way.  Infinite x gives
// NaN here, so groups holding an infinity divide the IEEE way.
__device__ __forceinline__ float q8_div(float x, float d, float y)
{
    const float q0 = __fmul_rn(x, y);
    return __fmaf_rn(__fmaf_rn(-q0, d, x), y, q0);
}

// 8-bit quantisation of one group of 32 values held by one lane (raw: the
// group's 64 bytes of bf16 or fp16): scale = fp16(min(amax / 127, 65504)),
// code = clamp(rn(x / scale), -127, 127), codes 0 when the scale is 0; every
// quotient is rounded as IEEE fp32 division rounds it (q8_div).  codes[w]
// holds the stored bytes (code + 128) of values 4w .. 4w + 3, low byte first.
// Rounding to an integer adds 1.5 * 2^23: the sum of a value in [-127, 127]
// and that constant lies where the fp32 spacing is 1, so the addition rounds
// to the nearest integer, ties to even, and the sum's low byte is the code.
template <bool BF16>
__device__ __forceinline__ void q8_group32(const uint4 (&raw)[4], uint32_t (&codes)[8],
                                           uint16_t &scale_bits)
{
    float v[32];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (BF16) {
                v[8 * k + 2 * i] = __uint_as_float(w[i] << 16);
                v[8 * k + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            } else {
                v[8 * k + 2 * i] = __half2float(__ushort_as_half((uint16_t)(w[i] & 0xffffu)));
                v[8 * k + 2 * i + 1] = __half2float(__ushort_as_half((uint16_t)(w[i] >> 16)));
            }
        }
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    constexpr float kRcp127 = 0x1.020408p-7f;            // rn(1 / 127)
    const float d32 = fminf(q8_div(amax, 127.0f, kRcp127), 65504.0f);
    const __half dh = __float2half_rn(d32);
    const float dq = __half2float(dh);
    scale_bits = __half_as_ushort(dh);
    if (isinf(amax)) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __fdiv_rn(v[i], dq);
    } else {
        const float y = dq != 0.0f ? __frcp_rn(dq) : 0.0f;   // y = 0 makes every quotient 0
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = q8_div(v[i], dq, y);
    }
    constexpr float kRound = 12582912.0f;                 // 1.5 * 2^23
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        uint32_t b[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            b[k] = __float_as_uint(__fadd_rn(fminf(fmaxf(v[4 * w + k], -127.0f), 127.0f), kRound));
        codes[w] = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040),
                               0x5410) ^ 0x80808080u;
    }
}

// The 64 bytes of group g of a 128-value row.
__device__ __forceinline__ void q8_load_group(const uint16_t *row, int g, uint4 (&raw)[4])
{
    const uint4 *p = reinterpret_cast<const uint4 *>(row) + 4 * g;
#pragma unroll
    for (int k = 0; k < 4; ++k) raw[k] = __ldg(p + k);
}

// K codes of token o (0..15), group g (dimensions 32g .. 32g + 31 = 16-byte
// chunks 2g, 2g + 1): token o = 4a + 2b + c is stored as row 8b + 2a + c,
// chunk j of a row at chunk position j ^ (row % 8).  Scales: K token-major at
// 4096, V group-major at 4224.
__device__ __forceinline__ void q8_store_k(uint8_t *rec, int o, int g, const uint32_t (&c)[8],
                                           uint16_t ks, uint16_t vs)
{
    const int row = 8 * ((o >> 1) & 1) + 2 * (o >> 2) + (o & 1);
    uint8_t *base = rec + row * 128;
    *reinterpret_cast<uint4 *>(base + (((2 * g) ^ (row & 7)) << 4)) = make_uint4(c[0], c[1], c[2], c[3]);
    *reinterpret_cast<uint4 *>(base + (((2 * g + 1) ^ (row & 7)) << 4)) =
        make_uint4(c[4], c[5], c[6], c[7]);
    *reinterpret_cast<uint16_t *>(rec + 4096 + o * 8 + 2 * g) = ks;
    *reinterpret_cast<uint16_t *>(rec + 4224 + g * 32 + o * 2) = vs;
}

// V codes of one token at offset off: dimension d's byte at 2048 + 16 d + off.
__device__ __forceinline__ void q8_store_v_token(uint8_t *rec, int off, int g, const uint32_t (&c)[8])
{
#pragma unroll
    for (int w = 0; w < 8; ++w)
#pragma unroll
        for (int k = 0; k < 4; ++k)
            rec[2048 + (32 * g + 4 * w + k) * 16 + off] = (uint8_t)(c[w] >> (8 * k));
}

// 4 x 4 byte transpose: word k of the result holds byte k of a, b, c, d (in
// that order, low byte first).
__device__ __forceinline__ void transpose4x4(uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                             uint32_t (&out)[4])
{
    const uint32_t ab_lo = __byte_perm(a, b, 0x5140), ab_hi = __byte_perm(a, b, 0x7362);
    const uint32_t cd_lo = __byte_perm(c, d, 0x5140), cd_hi = __byte_perm(c, d, 0x7362);
    out[0] = __byte_perm(ab_lo, cd_lo, 0x5410);
    out[1] = __byte_perm(ab_lo, cd_lo, 0x7632);
    out[2] = __byte_perm(ab_hi, cd_hi, 0x5410);
    out[3] = __byte_perm(ab_hi, cd_hi, 0x7632);
}

// 8-bit cache write, head_dim 128, into the records laid out in pagedkv.h.
// A lane quantises one group of 32 values: lane l takes group l % 4 of row
// l / 4, so a warp works on 8 rows at a time.
//
// V codes are stored dimension-major (16 tokens to a 16-byte row), so a lone
// token writes its 128 V codes as single bytes 16 bytes apart.  A block that
// the call fills whole with 16 consecutive tokens in slot order (a prompt) is
// written in one go instead: its V codes pass through a per-warp tile in
// shared memory ([token][dimension], chunks rotated), from which lane l reads dimensions
// 4l .. 4l + 3 of all 16 tokens and stores them as four whole 16-byte rows.
// Both ways store the same bytes.
//
// whole_blocks: one warp per window of 16 consecutive tokens of the call and
// one kv head.  The window holding a whole block's first token writes that
// block; every other token of the window is written on its own.  The warp
// finds both sets from one load of the slots of tokens tb - 16 .. tb + 47
// (tb = the window's first token): bit i of the masks below is token tb - 16 + i.
// A call of fewer than kQ8WindowsForBlocks windows (a decode step's one token
// per sequence; too few windows to give every resident warp several) runs with
// whole_blocks = false: 8 (token, kv head) rows per warp, each on its own.
constexpr int64_t kQ8WindowsForBlocks = 8192;

template <bool BF16>
__global__ void __launch_bounds__(128, 4)
cache_write_q8_kernel(const uint16_t *__restrict__ k_new, const uint16_t *__restrict__ v_new,
                      const int64_t *__restrict__ slot_mapping, int64_t num_tokens,
                      int32_t num_kv_heads, int64_t num_slots, bool whole_blocks,
                      uint8_t *__restrict__ kv, int32_t *__restrict__ status)
{
    constexpr int D = 128, BS = 16, SLAB = PKV_Q8_SLAB_BYTES;
    constexpr unsigned kAll = 0xffffffffu;
    __shared__ __align__(16) uint8_t vstage[4][BS * D];   // per warp: [token][dimension]
    const int lane = threadIdx.x & 31, r8 = lane >> 2, g = lane & 3;
    uint8_t *vt = vstage[threadIdx.x >> 5];
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t rows = num_tokens * num_kv_heads;
    if (!whole_blocks) {
        for (int64_t base = warp * 8; base < rows; base += warps * 8) {
            const int64_t r = base + r8;
            if (r >= rows) continue;
            const int64_t t = r / num_kv_heads;
            const int h = (int)(r - t * num_kv_heads);
            const int64_t slot = __ldg(slot_mapping + t);
            if (slot < 0) continue;
            if (slot >= num_slots) {
                if (g == 0) atomicOr(status, PKV_DEV_BAD_SLOT);
                continue;
            }
            const int64_t block = slot / BS;
            const int off = (int)(slot - block * BS);
            uint8_t *rec = kv + (block * num_kv_heads + h) * SLAB;
            uint4 kr[4], vr[4];
            q8_load_group(k_new + r * D, g, kr);
            q8_load_group(v_new + r * D, g, vr);
            uint32_t kc[8], vc[8];
            uint16_t ks, vs;
            q8_group32<BF16>(kr, kc, ks);
            q8_group32<BF16>(vr, vc, vs);
            q8_store_k(rec, off, g, kc, ks, vs);
            q8_store_v_token(rec, off, g, vc);
        }
        return;
    }
    const int64_t windows = (num_tokens + BS - 1) / BS * num_kv_heads;
    // slots of window w's span: lane l holds tokens tb - 16 + l and tb + 16 + l
    auto span_slots = [&](int64_t w, int64_t &a, int64_t &b) {
        const int64_t tb = w / num_kv_heads * BS;
        const int64_t p0 = tb - BS + lane, p1 = tb + BS + lane;
        a = w < windows && p0 >= 0 && p0 < num_tokens ? __ldg(slot_mapping + p0) : -1;
        b = w < windows && p1 < num_tokens ? __ldg(slot_mapping + p1) : -1;
    };
    int64_t s0_next, s1_next;
    span_slots(warp, s0_next, s1_next);
    for (int64_t w = warp; w < windows; w += warps) {
        const int64_t c = w / num_kv_heads;
        const int h = (int)(w - c * num_kv_heads);
        const int64_t tb = c * BS;
        const int64_t s0 = s0_next, s1 = s1_next;
        span_slots(w + warps, s0_next, s1_next);             // in flight while this one runs
        // the slot of the next token (none past the loaded span)
        const int64_t s1_first = __shfl_sync(kAll, s1, 0);
        int64_t n0 = __shfl_down_sync(kAll, s0, 1), n1 = __shfl_down_sync(kAll, s1, 1);
        if (lane == 31) n0 = s1_first, n1 = -1;
        const bool ok0 = s0 >= 0 && s0 < num_slots, ok1 = s1 >= 0 && s1 < num_slots;
        const uint64_t link = (uint64_t)__ballot_sync(kAll, ok0 && n0 == s0 + 1) |
                              (uint64_t)__ballot_sync(kAll, ok1 && n1 == s1 + 1) << 32;
        const uint64_t start = (uint64_t)__ballot_sync(kAll, ok0 && s0 % BS == 0) |
                               (uint64_t)__ballot_sync(kAll, ok1 && s1 % BS == 0) << 32;
        // whole blocks: a block start followed by 15 links (bits i .. i + 14)
        uint64_t run = link & (link >> 1);      // links i, i + 1
        run &= run >> 2;                        // i .. i + 3
        run &= run >> 4;                        // i .. i + 7
        const uint64_t full = start & run & (run >> 7);
        uint64_t covered = full | (full << 1);  // a whole block's 16 tokens
        covered |= covered << 2;
        covered |= covered << 4;
        covered |= covered << 8;
        const uint32_t mine = 0xffff0000u;      // tokens tb .. tb + 15 (bits 16 .. 31)
        if (__ballot_sync(kAll, s0 >= num_slots) & mine) {
            if (lane == 0) atomicOr(status, PKV_DEV_BAD_SLOT);
        }
        const uint32_t lead = (uint32_t)full & mine;                 // at most one bit
        const uint32_t single = __ballot_sync(kAll, ok0) & ~(uint32_t)covered & mine;
        if (lead) {
            const int i0 = __ffs(lead) - 1;
            const int64_t t0 = tb - BS + i0;
            const int64_t block = __shfl_sync(kAll, s0, i0) / BS;
            uint8_t *rec = kv + (block * num_kv_heads + h) * SLAB;
            uint4 kr[2][4], vr[2][4];
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int64_t r = (t0 + 8 * b + r8) * num_kv_heads + h;
                q8_load_group(k_new + r * D, g, kr[b]);
                q8_load_group(v_new + r * D, g, vr[b]);
            }
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int o = 8 * b + r8;
                uint32_t kc[8], vc[8];
                uint16_t ks, vs;
                q8_group32<BF16>(kr[b], kc, ks);
                q8_group32<BF16>(vr[b], vc, vs);
                q8_store_k(rec, o, g, kc, ks, vs);
                // tile row o, 16-byte chunk c at position c ^ (o % 8): the
                // stores of one instruction then spread over all 32 banks
                *reinterpret_cast<uint4 *>(vt + o * D + (((2 * g) ^ (o & 7)) << 4)) =
                    make_uint4(vc[0], vc[1], vc[2], vc[3]);
                *reinterpret_cast<uint4 *>(vt + o * D + (((2 * g + 1) ^ (o & 7)) << 4)) =
                    make_uint4(vc[4], vc[5], vc[6], vc[7]);
            }
            __syncwarp();
            uint32_t vw[BS];                         // token j: dimensions 4l .. 4l + 3
#pragma unroll
            for (int j = 0; j < BS; ++j)
                vw[j] = *reinterpret_cast<const uint32_t *>(vt + j * D + (((lane >> 2) ^ (j & 7)) << 4) +
                                                            4 * (lane & 3));
            __syncwarp();                            // the tile is free for the next window
            uint32_t vrow[4][4];                     // [dimension 4l + i][tokens 4q .. 4q + 3]
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t tr[4];
                transpose4x4(vw[4 * q], vw[4 * q + 1], vw[4 * q + 2], vw[4 * q + 3], tr);
#pragma unroll
                for (int i = 0; i < 4; ++i) vrow[i][q] = tr[i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<uint4 *>(rec + 2048 + (4 * lane + i) * BS) =
                    make_uint4(vrow[i][0], vrow[i][1], vrow[i][2], vrow[i][3]);
        }
        if (single) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int j = 8 * b + r8;                           // token tb + j
                const int64_t slot = __shfl_sync(kAll, s0, BS + j);
                if (!((single >> (BS + j)) & 1u)) continue;
                const int64_t block = slot / BS;
                const int off = (int)(slot - block * BS);
                uint8_t *rec = kv + (block * num_kv_heads + h) * SLAB;
                const int64_t r = (tb + j) * num_kv_heads + h;
                uint4 kr[4], vr[4];
                q8_load_group(k_new + r * D, g, kr);
                q8_load_group(v_new + r * D, g, vr);
                uint32_t kc[8], vc[8];
                uint16_t ks, vs;
                q8_group32<BF16>(kr, kc, ks);
                q8_group32<BF16>(vr, vc, vs);
                q8_store_k(rec, off, g, kc, ks, vs);
                q8_store_v_token(rec, off, g, vc);
            }
        }
    }
}

// CTAs of the 8-bit write that fit on the device at once, cached per device.
static int q8_write_grid_cap(const void *fn)
{
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    static int cap[kMaxDev][2];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return -1;
    const int which = fn == reinterpret_cast<const void *>(cache_write_q8_kernel<true>) ? 1 : 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cap[dev][which] == 0) {
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, 128, 0) != cudaSuccess ||
            per_sm < 1)
            return -1;
        cap[dev][which] = sms * per_sm;
    }
    return cap[dev][which];
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
    if (((uintptr_t)k_new & 15u) || ((uintptr_t)v_new & 15u) || ((uintptr_t)kv_q8 & 15u) ||
        ((uintptr_t)slot_mapping & 7u) || ((uintptr_t)d_status & 3u))
        return PKV_ERR_INVALID_ARG;
    const void *fn = g.dtype == PKV_Q8_BF16
                         ? reinterpret_cast<const void *>(cache_write_q8_kernel<true>)
                         : reinterpret_cast<const void *>(cache_write_q8_kernel<false>);
    const int cap = q8_write_grid_cap(fn);
    if (cap < 1) return PKV_ERR_CUDA;
    const int64_t rows = (int64_t)num_tokens * g.num_kv_heads;
    const int64_t windows = ((int64_t)num_tokens + 15) / 16 * g.num_kv_heads;
    const bool whole_blocks = windows >= kQ8WindowsForBlocks;
    const int64_t units = whole_blocks ? windows : (rows + 7) / 8;    // warps of work
    const int64_t blocks = std::min<int64_t>((units + 3) / 4, cap);
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t slots = (int64_t)g.num_blocks * g.block_size;
    if (g.dtype == PKV_Q8_BF16)
        cache_write_q8_kernel<true><<<(unsigned)blocks, 128, 0, st>>>(
            (const uint16_t *)k_new, (const uint16_t *)v_new, slot_mapping, (int64_t)num_tokens,
            g.num_kv_heads, slots, whole_blocks, (uint8_t *)kv_q8, d_status);
    else
        cache_write_q8_kernel<false><<<(unsigned)blocks, 128, 0, st>>>(
            (const uint16_t *)k_new, (const uint16_t *)v_new, slot_mapping, (int64_t)num_tokens,
            g.num_kv_heads, slots, whole_blocks, (uint8_t *)kv_q8, d_status);
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
