// Chunked-prefill attention over the paged KV cache for sm_103a.
//
// "vLLM과 Ollama의 차이" (chunked prefill: long prompts are cut into chunks
// that run in the same batch as the decoding sequences) and "LLM 추론 배칭
// 전략 정리", section 0 (a prefill step processes a prompt's tokens together):
// the chunk's K/V has been written into the cache (kv_cache_write); each of
// its queries, at position p, attends causally over the sequence's tokens 0..p,
// gathered through the block table exactly like decode.
//
// Design (GB300): two tcgen05 kernels (sections "tcgen05 prefill kernel" and
// "..., 128-key tiles"): per item, two query tiles of 128 rows of one kv group
// against the sequence's cache in tiles of 64 or 128 keys, S and O accumulated
// in tensor memory by tcgen05.mma from TMA-filled, 128-byte-swizzled shared
// memory, softmax by warpgroups whose threads each own one tensor-memory lane.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "pagedkv.h"
#include "decode_params.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "tc_device.cuh"

namespace pkv {
namespace prefill {

struct Params {
    void *out;
    const void *q;
    const int32_t *block_tables;
    const int32_t *query_start;     // [S + 1]
    const int32_t *context_lens;    // [S]
    int32_t num_seqs, num_tokens, num_q_heads, num_kv_heads, group, max_blocks_per_seq;
    int32_t num_blocks, tile_tokens;
    float scale_log2;
    int32_t *header;                // [0] = number of (sequence, tile) pairs
    int2 *items;                    // (sequence, tile)
    int64_t max_items;
    int32_t *status;
    // fp16 copy of V (bf16 pools with a workspace that holds it; else null):
    // [num_seqs * max_blocks_per_seq][Hkv][16][D] by logical block, and per
    // (sequence, kv head) the largest bf16 exponent field of its V
    uint16_t *v16;
    int32_t *v_emax;                // [num_seqs][Hkv]
    // Shared-prefix mode (a decode call whose neighbouring sequences share
    // their leading blocks): an item is (first member, members | chunk << 16,
    // first block, end block) of a run; the member sequences' queries (rows of
    // q [num_seqs][Hq][D]) attend over those blocks of the first member's table,
    // without a causal limit, and each row leaves its unnormalised output,
    // maximum and sum as piece piece_info[member].x + chunk of the decode call.
    const int4 *prefix_items;
    const int32_t *prefix_count;
    const int2 *piece_info;
    float2 *part_ml;                // [pieces * Hkv * G]
    float *part_o;                  // [pieces * Hkv * G * D]
};

// Scale of a (sequence, kv head)'s fp16 copy of V: v16 = v * 2^-k with
// k = E - 142, E the largest bf16 exponent field of its V, so the largest |v|
// (below 2^(E - 126)) lands in [2^15, 2^16), under fp16's largest value; k is
// clamped to [-100, 113] so both 2^k and 2^-k are normal fp32 numbers.
__device__ __forceinline__ int v16_shift(int emax)
{
    return min(113, max(-100, emax - 142));
}

// (sequence, tile) pairs and zero rows for chunks of invalid sequences.
__global__ void __launch_bounds__(1024) prefill_prep_kernel(Params p, int32_t head_dim)
{
    __shared__ int warp_tot[32];
    __shared__ int carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    griddep_launch_dependents();
    if (tid == 0) carry = 0;
    if (p.v_emax)       // the staging kernels that follow take maxima into these
        for (int i = tid; i < p.num_seqs * p.num_kv_heads; i += 1024) p.v_emax[i] = 0;
    __syncthreads();
    const int64_t max_tokens = (int64_t)p.max_blocks_per_seq * kBlock;
    for (int base = 0; base < p.num_seqs; base += 1024) {
        const int s = base + tid;
        int ntiles = 0;
        int r0 = 0, r1 = 0;
        bool zero = false;
        if (s < p.num_seqs) {
            r0 = p.query_start[s];
            r1 = p.query_start[s + 1];
            const int L = p.context_lens[s];
            const bool rows_ok = 0 <= r0 && r0 <= r1 && r1 <= p.num_tokens;
            if (!rows_ok || L < r1 - r0 || (int64_t)L > max_tokens) {
                atomicOr(p.status, PKV_DEV_BAD_LEN);
                zero = rows_ok;
            } else {
                ntiles = (r1 - r0 + p.tile_tokens - 1) / p.tile_tokens;
            }
        }
        int x = ntiles;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int t = warp_tot[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, t, o);
                if (lane >= o) t += y;
            }
            warp_tot[lane] = t;
        }
        __syncthreads();
        const int excl = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + x - ntiles;
        if (s < p.num_seqs) {
            if ((int64_t)excl + ntiles <= p.max_items)
                for (int k = 0; k < ntiles; ++k) p.items[excl + k] = make_int2(s, k);
            if (zero) {
                const int n16 = p.num_q_heads * head_dim * 2 / 16;
                for (int r = r0; r < r1; ++r) {
                    uint4 *o = reinterpret_cast<uint4 *>(static_cast<char *>(p.out) +
                                                         (size_t)r * p.num_q_heads * head_dim * 2);
                    for (int i = 0; i < n16; ++i) o[i] = make_uint4(0, 0, 0, 0);
                }
            }
        }
        __syncthreads();
        if (tid == 0) carry += warp_tot[31];
        __syncthreads();
    }
    if (tid == 0) {
        const bool fits = (int64_t)carry <= p.max_items;   // overlapping row ranges overflow it
        if (!fits) atomicOr(p.status, PKV_DEV_BAD_LEN);
        p.header[0] = fits ? carry : 0;
    }
}

// ======================================= fp16 copy of V (bf16 pools)
// With bf16 K/V, P V needs P as two bf16 parts (one bf16 part is too coarse
// for the tolerance); with V in fp16, one fp16 part of P will do and the P V
// products halve.  So, when the caller's workspace holds it, V of every
// attended token is copied once per call as fp16, scaled per (sequence, kv
// head) by a power of two (v16_shift): a bf16 significand (8 bits) fits in
// fp16's 11, so every value within 2^30 of the largest converts exactly (for a
// largest |v| of at least 2^-85, where the shift is not clamped); only values
// below that (fp16 subnormals) round, by at most 2^(k-25).  The
// attention kernel multiplies its result by 2^k.  Two passes over 256-token
// chunks: the largest exponent field (atomicMax into v_emax, zeroed by the
// prep kernel), then the conversion.  Tokens past a sequence's length are not
// written (the attention kernel zeroes those V rows in shared memory), nor
// are blocks with a bad table entry (flagged by the attention kernel).
constexpr int kStageTokens = 256;

__device__ __forceinline__ int stage_len(const Params &p, int s)
{
    const int L = __ldg(p.context_lens + s);
    return (L < 0 || (int64_t)L > (int64_t)p.max_blocks_per_seq * kBlock) ? 0 : L;
}

template <int D, bool CONVERT>
__global__ void __launch_bounds__(256) prefill_v16_kernel(const uint16_t *__restrict__ v_pool,
                                                          const Params p)
{
    // a CTA takes 256 tokens (16 blocks) of one (sequence, kv head); a block's
    // slab is 16 rows of D values, one 16-byte piece per thread (D = 128) or
    // per half of the threads (D = 64)
    constexpr int kBlocks = kStageTokens / kBlock;
    constexpr int kPieces = kBlock * D / 8;             // 16-byte pieces per slab
    constexpr int kPerThread = (kPieces + 255) / 256;
    const int Hkv = p.num_kv_heads;
    const int chunks = (p.max_blocks_per_seq * kBlock + kStageTokens - 1) / kStageTokens;
    const int64_t units = (int64_t)p.num_seqs * Hkv * chunks;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int64_t sg = u / chunks;
        const int c = (int)(u - sg * chunks);
        const int s = (int)(sg / Hkv), g = (int)(sg - (int64_t)s * Hkv);
        const int L = stage_len(p, s), t0 = c * kStageTokens;
        if (t0 >= L) continue;                      // the same for the whole CTA
        const int j0 = t0 / kBlock, nblk = min(kBlocks, (L - t0 + kBlock - 1) / kBlock);
        const int32_t *row = p.block_tables + (int64_t)s * p.max_blocks_per_seq + j0;
        float scale = 1.f;
        if constexpr (CONVERT) scale = __int_as_float((127 - v16_shift(p.v_emax[sg])) << 23);
        unsigned emax2 = 0;                         // two exponent fields per word
#pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            const int piece = threadIdx.x + 256 * k;
            if (piece >= kPieces) break;
            const int r = piece / (D / 8), q = piece % (D / 8);   // row (token) in the block
            uint4 w[kBlocks];
            bool ok[kBlocks];
#pragma unroll
            for (int b = 0; b < kBlocks; ++b) {     // every load of the thread in flight at once
                const int id = b < nblk ? __ldg(row + b) : -1;
                // the largest exponent counts visible tokens only
                ok[b] = id >= 0 && id < p.num_blocks && (CONVERT || t0 + b * kBlock + r < L);
                w[b] = ok[b] ? __ldg(reinterpret_cast<const uint4 *>(
                                       v_pool + (((int64_t)id * Hkv + g) * kBlock + r) * D) + q)
                             : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int b = 0; b < kBlocks; ++b) {
                if (!ok[b]) continue;
                if constexpr (CONVERT) {
                    const uint32_t in[4] = {w[b].x, w[b].y, w[b].z, w[b].w};
                    uint32_t o[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const __half2 h = __floats2half2_rn(__uint_as_float(in[i] << 16) * scale,
                                                            __uint_as_float(in[i] & 0xffff0000u) * scale);
                        o[i] = *reinterpret_cast<const uint32_t *>(&h);
                    }
                    *(reinterpret_cast<uint4 *>(
                          p.v16 + ((((int64_t)s * p.max_blocks_per_seq + j0 + b) * Hkv + g) * kBlock + r) * D) +
                      q) = make_uint4(o[0], o[1], o[2], o[3]);
                } else {
                    emax2 = __vmaxu2(emax2, __vmaxu2(__vmaxu2(w[b].x & 0x7f807f80u, w[b].y & 0x7f807f80u),
                                                     __vmaxu2(w[b].z & 0x7f807f80u, w[b].w & 0x7f807f80u)));
                }
            }
        }
        if constexpr (!CONVERT) {
            unsigned e = max((emax2 >> 7) & 0xffu, (emax2 >> 23) & 0xffu);
            e = __reduce_max_sync(kFull, e);
            if ((threadIdx.x & 31) == 0 && e > 0) atomicMax(p.v_emax + sg, (int)e);
        }
    }
}

// ================================================== tcgen05 prefill kernel
// Items are (sequence, kv head, two query tiles of 128 / G tokens): per tile
// 128 query rows (token-major: row r = token r / G, head r % G), both tiles
// against the same KV tiles of 64 keys (4 blocks) up to the second tile's last
// position, so each K/V tile is loaded once for 256 rows.
//   warp 8 (producer): TMA of the item's Q rows (one 4-D box per 64 columns)
//     and of each KV tile's 4 K and 4 V blocks into the stage ring.
//   warps 9 and 10, lane 0 (MMA issuers, one per query tile): S = Q K^T into
//     one of two tensor-memory buffers (M 128, N 64), then O += P V for the
//     previous tile (M 128, N D, V as an MN-major operand), P as a high and a
//     low bf16 part (bf16 pools) or one fp16 part (fp16 pools, and bf16 pools
//     whose V was copied to fp16 for the call).  One issuer
//     per query tile lets each group's S and P V go out as soon as that
//     group's inputs are ready, without waiting behind the other group's.
//   warps 0-3 and 4-7 (softmax, one warpgroup per query tile, ping-pong on the
//     tensor pipe): thread r of a group owns row r = tensor-memory lane r.  Running
//     maximum with lazy rescaling: the reference maximum moves only when a
//     tile's maximum exceeds it by more than 8 (log2 units), so weights stay
//     <= 2^8 and O in tensor memory is rescaled rarely.  V rows past the last
//     visible key are zeroed in shared memory before the P V product (stale
//     pool rows may hold anything, and 0 * NaN is NaN).
// Every wait is bounded; on expiry the kernel flags PKV_DEV_TIMEOUT and stops.
namespace tcp {

constexpr int kRows = 128;             // M: query rows per query tile
constexpr int kGroups = 2;             // query tiles per item, sharing every K/V tile
constexpr int kKeys = 64;              // keys per KV tile
// softmax warps 0-7, producer 8, MMA issuers 9 (query tile 0) and 10 (query tile 1)
constexpr int kThreads = (5 * kGroups + 1) * 32;
constexpr int kProducer = 4 * kGroups, kIssuer = 4 * kGroups + 1;
constexpr float kLazy = 8.f;           // rescale threshold (log2 units)

// ---- softmax arithmetic helpers: three-input max/min, packed fp32 pairs
__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float min3f(float a, float b, float c)
{
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ uint64_t pack2f(float a, float b)
{
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ float2 unpack2f(uint64_t v)
{
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t fma2f(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2f(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t mul2f(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t sub2f(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// bf16 weights (p0, p1) (pp = the same pair packed) as a high and a low part,
// the even index in the low half of each word: the high part is the weight
// truncated to bf16 (its upper 16 bits, exact), the low part the remainder
// rounded to bf16, so high + low carries the weight to ~2^-16.  (fp16 pools
// keep a single fp16 part: its relative error, <= 2^-11, is inside the
// tolerance, where a single bf16 part's 2^-9 is not.)
template <bool BF16>
__device__ __forceinline__ void split_hi_lo(float p0, float p1, uint64_t pp, uint32_t &hi,
                                            uint32_t &lo)
{
    static_assert(BF16, "fp16 weights take one part");
    const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
    hi = __byte_perm(b0, b1, 0x7632);
    const float2 d = unpack2f(sub2f(pp, pack2f(__uint_as_float(b0 & 0xffff0000u),
                                               __uint_as_float(b1 & 0xffff0000u))));
    lo = Elem<true>::pack(d.x, d.y);
}

template <int D>
struct Layout {
    static constexpr int kRegions = D / 64;
    static constexpr int kStages = D == 128 ? 5 : 8;           // K/V tiles in flight
    static constexpr int kQBytes = kRegions * kRows * 128;     // one query tile: [region][row][128 B]
    static constexpr int kKVBytes = kRegions * kKeys * 128;    // one K (or V) tile
    static constexpr int kStageBytes = 2 * kKVBytes;           // K tile, then V tile
    static constexpr int kStage0 = kGroups * kQBytes;
    static constexpr int kMisc = kStage0 + kStages * kStageBytes;   // barriers and flags
    static constexpr int kTotal = 1024 + kMisc + 512;
    // S of group g, buffer b at 64 (2g + b), overwritten by that tile's P (high
    // part in its first 32 columns, low part in the next 32); O of group g at
    // 256 + 128 g
    static constexpr uint32_t kTmemCols = 512;
};

// An item: the query tiles [t0, t0 + QT) (group 0) and [t0 + QT, t0 + 2 QT)
// (group 1) of one sequence's chunk and one kv head; keys 0 .. nkeys - 1.
struct Item {
    int s, g, r0, C, L, t0, t1, nkeys, ntiles;
    int kb0, chunk;      // shared-prefix mode: first block of the keys, piece of the chunk
};

template <bool PREFIX, int KEYS = kKeys>
__device__ __forceinline__ Item load_item(const Params &p, int i, int total, int QT)
{
    Item it;
    const int id = total - 1 - i;          // longest tiles first
    const int Hkv = p.num_kv_heads;
    const int sj = id / Hkv;
    it.g = id - sj * Hkv;
    if constexpr (PREFIX) {
        const int4 e = __ldg(p.prefix_items + sj);
        it.s = e.x;                         // every member's table begins with these blocks
        it.r0 = e.x;
        it.C = e.y & 0xffff;
        it.chunk = e.y >> 16;
        it.kb0 = e.z;
        it.L = (e.w - e.z) * kBlock;
        it.t0 = 0;
        it.t1 = it.C;
        it.nkeys = it.L;
        it.ntiles = (it.nkeys + KEYS - 1) / KEYS;
        return it;
    }
    it.kb0 = 0;
    it.chunk = 0;
    const int2 e = p.items[sj];
    it.s = e.x;
    it.r0 = __ldg(p.query_start + e.x);
    it.C = __ldg(p.query_start + e.x + 1) - it.r0;
    it.L = __ldg(p.context_lens + e.x);
    it.t0 = e.y * kGroups * QT;
    it.t1 = min(it.t0 + kGroups * QT, it.C);
    it.nkeys = it.L - it.C + it.t1;
    it.ntiles = (it.nkeys + KEYS - 1) / KEYS;
    return it;
}

// VS: V comes from the fp16 copy (tmV maps it; bf16 pools only), so P V takes
// one fp16 part of P and the result is scaled by 2^k.
// PREFIX: shared-prefix mode of a decode call (see Params): items from
// prefix_items, no causal limit, pieces instead of output rows.
template <int D, bool BF16, bool VS, bool PREFIX>
__global__ void __launch_bounds__(kThreads)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmQ, const Params p)
{
    static_assert(BF16 || !VS, "fp16 pools take V as it is");
    static_assert(!(VS && PREFIX), "the shared-prefix mode reads V from the pool");
    constexpr bool kTwoParts = BF16 && !VS;    // P as bf16 high + low parts
    using E = Elem<BF16>;
    using T = typename E::T;
    using LY = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *q_s = base;
    uint8_t *stage_s = base + LY::kStage0;
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + LY::kMisc);
    uint64_t *q_full = bars + 0, *q_empty = bars + 1;
    uint64_t *kv_full = bars + 2, *kv_empty = kv_full + LY::kStages;   // [LY::kStages] each
    uint64_t *s_full = kv_empty + LY::kStages;                 // [group][buffer]
    // P of a group out / P V of a group done, for even and odd tiles: a parity
    // wait is exact only while its barrier runs at most one phase ahead of the
    // waiter, and alternating barriers keep them so (P of tile t + 2 needs
    // S(t + 2), issued after P V of tile t; P V of tile t + 1 needs P(t + 1),
    // published after the wait for P V of tile t - 1)
    uint64_t *p_full = s_full + 2 * kGroups;                   // [group][tile & 1]
    uint64_t *o_full = p_full + 2 * kGroups;                   // [group][tile & 1]
    uint64_t *done = o_full + 2 * kGroups;                     // [group]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + kGroups);
    int *stage_bad = reinterpret_cast<int *>(tslot + 1);            // [LY::kStages]
    volatile int *abort_flag = stage_bad + LY::kStages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(q_full), 1);
        mbar_init(smem_addr(q_empty), kGroups);     // one commit per issuer
        for (int i = 0; i < LY::kStages; ++i) {
            mbar_init(smem_addr(&kv_full[i]), 1);
            mbar_init(smem_addr(&kv_empty[i]), kGroups);
        }
        for (int i = 0; i < 2 * kGroups; ++i) mbar_init(smem_addr(&s_full[i]), 1);
        for (int i = 0; i < 2 * kGroups; ++i) {
            mbar_init(smem_addr(&p_full[i]), 4);
            mbar_init(smem_addr(&o_full[i]), 1);
        }
        for (int i = 0; i < kGroups; ++i) mbar_init(smem_addr(&done[i]), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tc::tmem_alloc(tslot, LY::kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;
    griddep_wait();

    const int Hkv = p.num_kv_heads, G = p.group, QT = p.tile_tokens / kGroups;   // one query tile
    const int total = (PREFIX ? *p.prefix_count : p.header[0]) * Hkv;

    if (warp == kProducer) {
        if (lane == 0) {
            uint32_t kv_cnt = 0, it_cnt = 0;
            int last_par[LY::kStages], last_q = -1;          // phases of the last copies issued
            for (int k = 0; k < LY::kStages; ++k) last_par[k] = -1;
            for (int i = blockIdx.x; i < total && !*abort_flag; i += gridDim.x, ++it_cnt) {
                const Item it = load_item<PREFIX>(p, i, total, QT);
                if (it_cnt > 0 &&
                    !mbar_wait(smem_addr(q_empty), (it_cnt - 1) & 1u, abort_flag, p.status))
                    break;
                const uint32_t qb = smem_addr(q_full);
                last_q = (int)(it_cnt & 1u);
                mbar_arrive_expect_tx(qb, (uint32_t)(kGroups * LY::kRegions * QT * G * 128));
                for (int gr = 0; gr < kGroups; ++gr)
                    for (int rg = 0; rg < LY::kRegions; ++rg)
                        tc::tma_load_4d(smem_addr(q_s + gr * LY::kQBytes + rg * kRows * 128), &tmQ,
                                        rg * 64, 0, it.g, it.r0 + it.t0 + gr * QT, qb);
                const int32_t *row = p.block_tables + (int64_t)it.s * p.max_blocks_per_seq + it.kb0;
                const int nb = (it.nkeys + kBlock - 1) / kBlock;
                for (int t = 0; t < it.ntiles; ++t, ++kv_cnt) {
                    const int st = (int)(kv_cnt % LY::kStages);
                    const uint32_t fill = kv_cnt / LY::kStages;
                    if (fill >= 1 && !mbar_wait(smem_addr(&kv_empty[st]), (fill - 1) & 1u,
                                                abort_flag, p.status))
                        break;
                    int ids[4];
                    int bad = 0;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const int id = __ldg(row + min(4 * t + b, nb - 1));
                        const bool ok = id >= 0 && id < p.num_blocks;
                        bad |= !ok;
                        ids[b] = ok ? id : 0;
                    }
                    if (bad) atomicOr(p.status, PKV_DEV_BAD_BLOCK);
                    stage_bad[st] = bad;
                    last_par[st] = (int)(fill & 1u);
                    const uint32_t fb = smem_addr(&kv_full[st]);
                    mbar_arrive_expect_tx(fb, (uint32_t)(2 * LY::kKVBytes));
                    const uint32_t ks = smem_addr(stage_s + st * LY::kStageBytes);
                    const uint32_t vs = ks + LY::kKVBytes;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const int y = (ids[b] * Hkv + it.g) * kBlock;
                        // the fp16 copy is by logical block
                        const int yv = VS ? ((it.s * p.max_blocks_per_seq + min(4 * t + b, nb - 1)) * Hkv +
                                             it.g) * kBlock
                                          : y;
#pragma unroll
                        for (int rg = 0; rg < LY::kRegions; ++rg) {
                            const uint32_t off = rg * kKeys * 128 + b * kBlock * 128;
                            tma_load_2d(ks + off, &tmK, rg * 64, y, fb);
                            tma_load_2d(vs + off, &tmV, rg * 64, yv, fb);
                        }
                    }
                }
            }
            // after a timed-out wait: let the copies still in flight land first
            if (*abort_flag) {
                for (int k = 0; k <= LY::kStages; ++k) {
                    const int par = k < LY::kStages ? last_par[k] : last_q;
                    if (par < 0) continue;
                    const uint32_t fb = smem_addr(k < LY::kStages ? &kv_full[k] : q_full);
                    const unsigned long long t0 = globaltimer();
                    while (!mbar_try_wait(fb, (uint32_t)par)) {
                        if (globaltimer() - t0 > kTimeoutNs) break;
                    }
                }
            }
        }
    } else if (warp == kIssuer || warp == kIssuer + 1) {
        // one issuer per query tile
        if (lane == 0) {
            const int gr = warp - kIssuer;
            const uint32_t id_qk = tc::idesc_f16(BF16, kRows, kKeys, 0, 0);
            const uint32_t id_pv = tc::idesc_f16(kTwoParts, kRows, D, 0, 1);   // P and V: same type
            const uint32_t q_a = smem_addr(q_s) + gr * LY::kQBytes, st_a = smem_addr(stage_s);
            const uint32_t o_t = tmem + 256 + 128 * gr;
            // Descriptors are built once per operand base; each MMA adds its
            // constant offset to the address field (offset >> 4: no carry
            // leaves the field, shared memory is below 256 KB), which keeps the
            // issuing thread's instruction stream short -- it shares its
            // scheduler with two softmax warps.
            const uint64_t qa_d = tc::desc_sw128(q_a, 16, 1024);
            uint32_t tg = 0, it_cnt = 0;
            bool ok = true;
            // P V of tile t for this group, then its share of freeing the stage
            auto issue_pv = [&](uint32_t t, bool first) {
                const uint32_t vs = st_a + (t % LY::kStages) * LY::kStageBytes + LY::kKVBytes;
                if (!mbar_wait(smem_addr(&p_full[2 * gr + (t & 1u)]), (t >> 1) & 1u, abort_flag,
                               p.status)) {
                    ok = false;
                    return;
                }
                tc::fence_after_sync();
                const uint32_t pt = tmem + 64 * (2 * gr + (t & 1u));   // P of tile t
                const uint64_t vb_d = tc::desc_sw128(vs, kKeys * 128, 1024);
#pragma unroll
                for (int part = 0; part < (kTwoParts ? 2 : 1); ++part)
#pragma unroll
                    for (int kk = 0; kk < kKeys / 16; ++kk) {
                        const uint64_t b = vb_d + (uint64_t)((kk * 16 * 128) >> 4);
                        tc::mma_f16_ts(o_t, pt + part * 32 + kk * 8, b, id_pv,
                                       !(first && part == 0 && kk == 0));
                    }
                tc::mma_commit(smem_addr(&o_full[2 * gr + (t & 1u)]));
                tc::mma_commit(smem_addr(&kv_empty[t % LY::kStages]));
            };
            for (int i = blockIdx.x; i < total && ok; i += gridDim.x, ++it_cnt) {
                const Item it = load_item<PREFIX>(p, i, total, QT);
                if (!mbar_wait(smem_addr(q_full), it_cnt & 1u, abort_flag, p.status)) break;
                for (int t = 0; t < it.ntiles && ok; ++t, ++tg) {
                    const uint32_t st = tg % LY::kStages, sb = tg & 1u;
                    if (!mbar_wait(smem_addr(&kv_full[st]), (tg / LY::kStages) & 1u, abort_flag,
                                   p.status)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint64_t kb_d = tc::desc_sw128(st_a + st * LY::kStageBytes, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk & 3) * 32;     // 16 values inside the row
                        const uint64_t a = qa_d + (uint64_t)(((kk >> 2) * kRows * 128 + off) >> 4);
                        const uint64_t b = kb_d + (uint64_t)(((kk >> 2) * kKeys * 128 + off) >> 4);
                        tc::mma_f16(tmem + 64 * (2 * gr + sb), a, b, id_qk, kk > 0);
                    }
                    tc::mma_commit(smem_addr(&s_full[2 * gr + sb]));
                    if (t == it.ntiles - 1) tc::mma_commit(smem_addr(q_empty));
                    if (t >= 1) issue_pv(tg - 1, t == 1);
                }
                if (ok) issue_pv(tg - 1, it.ntiles == 1);
            }
            // every MMA this thread issued has completed before the columns are freed
            tc::mma_commit(smem_addr(&done[gr]));
            const unsigned long long t0 = globaltimer();
            while (!mbar_try_wait(smem_addr(&done[gr]), 0)) {
                if (globaltimer() - t0 > kTimeoutNs) {
                    atomicOr(p.status, PKV_DEV_TIMEOUT);
                    break;
                }
            }
        }
    } else {
        // ---------------------------------------------------------- softmax
        const int gr = warp >> 2;                   // query tile of this warpgroup
        const int r = threadIdx.x - kRows * gr;     // row = tensor-memory lane
        const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const uint32_t s_col = 64 * 2 * gr, o_col = 256 + 128 * gr;
        uint32_t tg = 0, it_cnt = 0;
        bool alive = true;
        for (int i = blockIdx.x; i < total && alive; i += gridDim.x, ++it_cnt) {
            const Item it = load_item<PREFIX>(p, i, total, QT);
            const int jj = r / G, h = r - (r / G) * G;
            const int tg0 = it.t0 + gr * QT;            // this group's first token
            const bool valid = r < QT * G && tg0 + jj < it.t1;
            const int pos = valid && !PREFIX ? it.L - it.C + tg0 + jj : it.nkeys - 1;
            float m_ref = -INFINITY, l = 0.f;
            int bad = 0;
            for (int t = 0; t < it.ntiles; ++t, ++tg) {
                const uint32_t st = tg % LY::kStages, sb = tg & 1u;
                const bool ok1 = mbar_wait(smem_addr(&kv_full[st]), (tg / LY::kStages) & 1u, abort_flag,
                                           p.status);
                const bool ok2 = ok1 && mbar_wait(smem_addr(&s_full[2 * gr + sb]), (tg >> 1) & 1u,
                                                  abort_flag, p.status);
                if (!__all_sync(kFull, ok2)) { alive = false; break; }
                tc::fence_after_sync();
                bad |= stage_bad[st];
                float x[kKeys];
                {
                    uint32_t v[2][32];
                    tc::tmem_ld32(lane_base + s_col + 64 * sb, v[0]);
                    tc::tmem_ld32(lane_base + s_col + 64 * sb + 32, v[1]);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        x[c] = __uint_as_float(v[0][c]);
                        x[32 + c] = __uint_as_float(v[1][c]);
                    }
                }
                // raw scores; the scale enters inside the exponent (one FFMA each).
                // Hidden keys are kept out of the maximum here and get weight 0 below.
                const int k0 = t * kKeys;
                const bool cross = k0 + kKeys - 1 > pos;   // the tile crosses this row's position
                if (cross) {
                    const float hide = p.scale_log2 < 0.f ? INFINITY : -INFINITY;
#pragma unroll
                    for (int c = 0; c < kKeys; ++c)
                        if (k0 + c > pos) x[c] = hide;
                }
                float mx;
                if (p.scale_log2 >= 0.f) {
                    mx = fmaxf(x[0], x[1]);
#pragma unroll
                    for (int c = 2; c < kKeys; c += 2) mx = max3f(mx, x[c], x[c + 1]);
                } else {                           // the largest scaled score is the smallest raw one
                    mx = fminf(x[0], x[1]);
#pragma unroll
                    for (int c = 2; c < kKeys; c += 2) mx = min3f(mx, x[c], x[c + 1]);
                }
                mx *= p.scale_log2;
                float f = 1.f;
                bool resc = false;
                if (mx > m_ref + kLazy) {          // also the first tile: m_ref = -inf
                    if (m_ref != -INFINITY) {
                        f = fast_exp2(m_ref - mx);
                        resc = true;
                    }
                    m_ref = mx;
                }
                // weights in pairs: packed fp32 arithmetic (f32x2), then a high and a
                // low 16-bit part per weight
                uint32_t hi[kKeys / 2], lo[kKeys / 2];
                const uint64_t sc2 = pack2f(p.scale_log2, p.scale_log2), nm2 = pack2f(-m_ref, -m_ref);
                uint64_t lsum2 = pack2f(0.f, 0.f);
                // two copies of the loop: only a tile that crosses the row's
                // position pays for the per-key causal test
                auto weights = [&](auto masked) {
#pragma unroll
                    for (int c = 0; c < kKeys; c += 2) {
                        const float2 e = unpack2f(fma2f(pack2f(x[c], x[c + 1]), sc2, nm2));
                        float p0 = fast_exp2(e.x), p1 = fast_exp2(e.y);
                        if constexpr (decltype(masked)::value) {
                            if (k0 + c > pos) p0 = 0.f;
                            if (k0 + c + 1 > pos) p1 = 0.f;
                        }
                        const uint64_t pp = pack2f(p0, p1);
                        lsum2 = add2f(lsum2, pp);
                        if constexpr (kTwoParts)
                            split_hi_lo<true>(p0, p1, pp, hi[c / 2], lo[c / 2]);
                        else                   // fp16 (relative error <= 2^-11): one part
                            hi[c / 2] = Elem<false>::pack(p0, p1);
                    }
                };
                if (cross) weights(std::true_type{});
                else weights(std::false_type{});
                const float2 ls = unpack2f(lsum2);
                l = l * f + (ls.x + ls.y);
                // O is rescaled before P V of this tile, once P V of the previous
                // tile has finished writing it; the wait for that P V consumes the
                // o_full phase of the previous tile either here or after P is out
                const bool any_resc = __any_sync(kFull, resc);
                if (t >= 1 && any_resc) {
                    const bool okp = mbar_wait(smem_addr(&o_full[2 * gr + ((tg - 1) & 1u)]),
                                               ((tg - 1) >> 1) & 1u, abort_flag, p.status);
                    if (!__all_sync(kFull, okp)) { alive = false; break; }
                    tc::fence_after_sync();
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t v[32];
                        tc::tmem_ld32(lane_base + o_col + c0, v);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * f);
                        tc::tmem_st32(lane_base + o_col + c0, v);
                    }
                }
                // P of this tile over its own S columns (already read): high part
                // in the first 32, low part in the next 32
                tc::tmem_st32(lane_base + s_col + 64 * sb, hi);
                if constexpr (kTwoParts) tc::tmem_st32(lane_base + s_col + 64 * sb + 32, lo);
                // zero the V rows of keys past the last visible one (last tile only)
                const int nvis = it.nkeys - k0;
                if (nvis < kKeys) {      // both groups write the same zeros, each before its P
                    uint8_t *vs = stage_s + st * LY::kStageBytes + LY::kKVBytes;
                    const int nrows = kKeys - nvis;
                    for (int e = r; e < nrows * LY::kRegions * 8; e += kRows) {
                        const int row = nvis + e / (LY::kRegions * 8);
                        const int rem = e % (LY::kRegions * 8);
                        *reinterpret_cast<uint4 *>(vs + (rem >> 3) * kKeys * 128 + row * 128 +
                                                   (rem & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&p_full[2 * gr + (tg & 1u)]));
                if (t >= 1 && !any_resc) {
                    const bool okp = mbar_wait(smem_addr(&o_full[2 * gr + ((tg - 1) & 1u)]),
                                               ((tg - 1) >> 1) & 1u, abort_flag, p.status);
                    if (!__all_sync(kFull, okp)) { alive = false; break; }
                }
            }
            if (!alive) break;
            // ---- the item's result: O / l once the last P V is done
            const bool oko = mbar_wait(smem_addr(&o_full[2 * gr + ((tg - 1) & 1u)]),
                                       ((tg - 1) >> 1) & 1u, abort_flag, p.status);
            if (!__all_sync(kFull, oko)) break;
            tc::fence_after_sync();
            if constexpr (PREFIX) {
                // the row's piece: O as it stands (weights taken against m_ref), m_ref, l
                size_t piece = 0;
                if (valid) {
                    const int member = it.r0 + tg0 + jj;
                    piece = ((size_t)(__ldg(p.piece_info + member).x + it.chunk) * Hkv + it.g) * G + h;
                    p.part_ml[piece] = make_float2(m_ref, bad ? -1.f : l);
                }
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t v[32];
                    tc::tmem_ld32(lane_base + o_col + c0, v);
                    tc::tmem_wait_ld();
                    if (valid) {
                        float4 *dst = reinterpret_cast<float4 *>(p.part_o + piece * D + c0);
#pragma unroll
                        for (int c = 0; c < 32; c += 4)
                            dst[c / 4] = make_float4(__uint_as_float(v[c]), __uint_as_float(v[c + 1]),
                                                     __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
                    }
                }
                tc::fence_before_sync();
                continue;
            }
            const float inv = 1.f / l;
            T *out = static_cast<T *>(p.out) +
                     ((size_t)(it.r0 + tg0 + jj) * p.num_q_heads + (size_t)it.g * G + h) * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t v[32];
                tc::tmem_ld32(lane_base + o_col + c0, v);
                tc::tmem_wait_ld();
                if constexpr (VS) {     // O / l in the fp16 copy's units, then times 2^k
                    const float p2k = __int_as_float(
                        (127 + v16_shift(p.v_emax[(size_t)it.s * Hkv + it.g])) << 23);
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        v[c] = __float_as_uint(__uint_as_float(v[c]) * inv * p2k);
                }
                const float vin = VS ? 1.f : inv;
                if (valid) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint4 w;
                        w.x = bad ? 0u : E::pack(__uint_as_float(v[c]) * vin, __uint_as_float(v[c + 1]) * vin);
                        w.y = bad ? 0u : E::pack(__uint_as_float(v[c + 2]) * vin, __uint_as_float(v[c + 3]) * vin);
                        w.z = bad ? 0u : E::pack(__uint_as_float(v[c + 4]) * vin, __uint_as_float(v[c + 5]) * vin);
                        w.w = bad ? 0u : E::pack(__uint_as_float(v[c + 6]) * vin, __uint_as_float(v[c + 7]) * vin);
                        *reinterpret_cast<uint4 *>(out + c0 + c) = w;
                    }
                }
            }
            tc::fence_before_sync();
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, LY::kTmemCols);
}

}  // namespace tcp

// ======================================= tcgen05 prefill kernel, 128-key tiles
// For P in one fp16 part (fp16 pools; bf16 pools whose V was copied to fp16 for
// the call).  The same items as the 64-key kernel, but each K/V tile holds 128
// keys (8 blocks), so S = Q K^T runs at N 128 (the full MMA rate) and a row's
// softmax takes twice the keys per turn.  Tensor memory (512 columns) then
// holds one S buffer per query tile (128 columns each) and the two O (128
// each):
//   warp 8 (producer): TMA of the item's Q rows and of each tile's K and V
//     into two rings that fill and drain separately (K is free once both query
//     tiles' S is done, V once both P V are); blocks past the keys are copied
//     from past the end of the tensor, which fills them with zeros.  It also
//     brings the next item's query rows into L2.
//   warps 9 and 10, lane 0 (MMA issuers, one per query tile): for each tile t,
//     O += P V of tile t - 1, then S = Q K^T of tile t into the query tile's S
//     buffer.  P of tile t - 1 lives in that buffer's columns; the tensor core
//     runs one thread's MMAs in the order issued, so S(t) overwrites them only
//     after P V(t - 1) has read them, and the commit that signals S(t) also
//     signals P V(t - 1).
//   warps 0-3 and 4-7 (softmax, one warpgroup per query tile): thread r owns
//     row r = tensor-memory lane r and holds the row's 128 scores of a tile in
//     registers; the two warpgroups take turns at the weights, warp by warp
//     (warps w and w + 4 share a scheduler and its SFU, and while one
//     computes, the tensor core runs the other's P V and next S).  Weights
//     are taken against a lazy reference maximum in one pass; the tile's
//     maximum is computed only for an item's first tile and when a score
//     exceeds the reference by more than 8 (log2 units), which moves the
//     reference, rescales O and the sum and takes the weights again.  The
//     output of an item goes through shared memory, so that its stores write
//     whole lines.
//   warp 11 holds no role: the copy/issue warpgroup gives its registers to the
//     softmax warpgroups (setmaxnreg).
// Every wait is bounded; on expiry the kernel flags PKV_DEV_TIMEOUT and stops.
namespace tcw {

using tcp::add2f;
using tcp::fma2f;
using tcp::Item;
using tcp::kGroups;
using tcp::kRows;
using tcp::max3f;
using tcp::min3f;
using tcp::mul2f;
using tcp::pack2f;
using tcp::unpack2f;

constexpr int kKeys = 128;             // keys per KV tile (N of S = Q K^T)
constexpr int kTileBlocks = kKeys / kBlock;
constexpr int kThreads = 12 * 32;      // softmax 0-7, producer 8, issuers 9 and 10, warp 11
constexpr int kProducer = 4 * kGroups, kIssuer = 4 * kGroups + 1;
// registers per thread: the launch gives kLaunchRegs = 65536 / 384 rounded
// down to 8; the copy/issue warpgroup keeps kRegsIo and hands the rest to the
// two softmax warpgroups, 2 * 128 * kRegsSoftmax + 128 * kRegsIo = 384 *
// kLaunchRegs.  A launch with fewer registers would leave setmaxnreg.inc
// waiting for ever, so the host launches only a build whose kernels use
// exactly kLaunchRegs (launch_regs_ok).
constexpr int kLaunchRegs = 168;
constexpr int kRegsIo = 72, kRegsSoftmax = 216;
static_assert(2 * kRegsSoftmax + kRegsIo == 3 * kLaunchRegs, "register split of the launch");
constexpr float kLazy = 8.f;           // rescale threshold (log2 units)

template <int D>
struct Layout {
    static constexpr int kRegions = D / 64;
    static constexpr int kStages = D == 128 ? 2 : 5;           // K/V tiles in flight
    static constexpr int kQBytes = kRegions * kRows * 128;     // one query tile: [region][row][128 B]
    static constexpr int kKVBytes = kRegions * kKeys * 128;    // one K (or V) tile
    static constexpr int kStageBytes = 2 * kKVBytes;           // K tile, then V tile
    static constexpr int kStage0 = kGroups * kQBytes;
    static constexpr int kMisc = kStage0 + kStages * kStageBytes;   // barriers and flags
    // output staging of the softmax warps: 32 rows x 128 bytes each
    static constexpr int kEpi = kMisc + 512;
    static constexpr int kEpiWarpBytes = 32 * 128;
    static constexpr int kTotal = 1024 + kEpi + 4 * kGroups * kEpiWarpBytes;
    // S of group g at kKeys g, overwritten by that tile's P (its first
    // kKeys / 2 columns); O of group g at 256 + 128 g
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kTotal <= 227 * 1024, "shared memory of one CTA");
    static_assert(kKeys == 128, "the softmax takes a tile as four 32-key chunks");
};

// VS: V comes from the fp16 copy (tmV maps it; bf16 pools), so P V takes one
// fp16 part of P and the result is scaled by 2^k.  The host sends this kernel
// the staged bf16 calls only; calls that need P in two parts (bf16 V as it
// is), fp16 pools and the shared-prefix mode take the 64-key kernel.
template <int D, bool BF16, bool VS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmQ, const Params p)
{
    static_assert(BF16 || !VS, "fp16 pools take V as it is");
    static_assert(!BF16 || VS, "P takes one fp16 part: fp16 pools, or bf16 pools with V in fp16");
    using E = Elem<BF16>;
    using T = typename E::T;
    using LY = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *q_s = base;
    uint8_t *stage_s = base + LY::kStage0;
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + LY::kMisc);
    uint64_t *q_full = bars + 0, *q_empty = bars + 1;
    // K and V of a stage fill and drain separately: K is free once both query
    // tiles' S is done, V once both P V are, so the next K tile can come in
    // while the softmax still runs on this one
    uint64_t *k_full = bars + 2, *k_empty = k_full + LY::kStages;      // [LY::kStages] each
    uint64_t *v_full = k_empty + LY::kStages, *v_empty = v_full + LY::kStages;
    // per group: S of the tile (and, with it, P V of the one before) done;
    // P of the tile out; the item's last P V done.  Each waiter is at most one
    // phase behind its barrier: S(t + 1) is issued after P(t), which the
    // softmax publishes after its wait for S(t); P(t + 1) follows S(t + 1).
    uint64_t *s_full = v_empty + LY::kStages;                  // [group]
    uint64_t *p_full = s_full + kGroups;                       // [group]
    uint64_t *o_full = p_full + kGroups;                       // [group], one phase per item
    uint64_t *done = o_full + kGroups;                         // [group]
    // the two query tiles take turns at the weights, warp by warp: softmax
    // warps w and w + 4 share a scheduler (and its SFU, which their
    // exponentials keep busy), and while one computes, the tensor core runs
    // the other's P V and next S.  Warp w's weights of a tile done:
    uint64_t *w_done = done + kGroups;                         // [softmax warp]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(w_done + 4 * kGroups);
    int *stage_bad = reinterpret_cast<int *>(tslot + 1);            // [LY::kStages]
    volatile int *abort_flag = stage_bad + LY::kStages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(q_full), 1);
        mbar_init(smem_addr(q_empty), kGroups);     // one commit per issuer
        for (int i = 0; i < LY::kStages; ++i) {
            mbar_init(smem_addr(&k_full[i]), 1);
            mbar_init(smem_addr(&k_empty[i]), kGroups);
            mbar_init(smem_addr(&v_full[i]), 1);
            mbar_init(smem_addr(&v_empty[i]), kGroups);
        }
        for (int i = 0; i < 4 * kGroups; ++i) mbar_init(smem_addr(&w_done[i]), 1);
        for (int i = 0; i < kGroups; ++i) {
            mbar_init(smem_addr(&s_full[i]), 1);
            mbar_init(smem_addr(&p_full[i]), 4);
            mbar_init(smem_addr(&o_full[i]), 1);
            mbar_init(smem_addr(&done[i]), 1);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tc::tmem_alloc(tslot, LY::kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;
    griddep_wait();

    const int Hkv = p.num_kv_heads, G = p.group, QT = p.tile_tokens / kGroups;   // one query tile
    const int total = p.header[0] * Hkv;

    // the register split is taken inside each role's branch, so that every
    // block of a role's code lies under one limit
    if (warp >= kProducer) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsIo));
        if (warp == kProducer) {
            if (lane == 0) {
                uint32_t kv_cnt = 0, it_cnt = 0;
                const int k_rows = p.num_blocks * Hkv * kBlock;
                const int v_rows = VS ? p.num_seqs * p.max_blocks_per_seq * Hkv * kBlock : k_rows;
                // phases of the last copies issued: K of each stage, V of each stage, Q
                int last_par[2 * LY::kStages + 1];
                for (int k = 0; k <= 2 * LY::kStages; ++k) last_par[k] = -1;
                // every role reads an item's description one item ahead, so the
                // dependent loads behind it are off the path between items
                Item nxt = {};
                if ((int)blockIdx.x < total) nxt = tcp::load_item<false, kKeys>(p, blockIdx.x, total, QT);
                for (int i = blockIdx.x; i < total && !*abort_flag; i += gridDim.x, ++it_cnt) {
                    const Item it = nxt;
                    if (i + (int)gridDim.x < total) nxt = tcp::load_item<false, kKeys>(p, i + gridDim.x, total, QT);
                    if (it_cnt > 0 &&
                        !mbar_wait(smem_addr(q_empty), (it_cnt - 1) & 1u, abort_flag, p.status))
                        break;
                    const uint32_t qb = smem_addr(q_full);
                    last_par[2 * LY::kStages] = (int)(it_cnt & 1u);
                    mbar_arrive_expect_tx(qb, (uint32_t)(kGroups * LY::kRegions * QT * G * 128));
                    for (int gr = 0; gr < kGroups; ++gr)
                        for (int rg = 0; rg < LY::kRegions; ++rg)
                            tc::tma_load_4d(smem_addr(q_s + gr * LY::kQBytes + rg * kRows * 128), &tmQ,
                                            rg * 64, 0, it.g, it.r0 + it.t0 + gr * QT, qb);
                    // the next item's query rows into L2 now: its load above comes
                    // only once this item's last S is done, about one softmax
                    // before its first S
                    if (i + (int)gridDim.x < total) {
                        for (int gr = 0; gr < kGroups; ++gr)
                            for (int rg = 0; rg < LY::kRegions; ++rg)
                                tc::tma_prefetch_4d(&tmQ, rg * 64, 0, nxt.g, nxt.r0 + nxt.t0 + gr * QT);
                    }
                    const int32_t *row = p.block_tables + (int64_t)it.s * p.max_blocks_per_seq + it.kb0;
                    const int nb = (it.nkeys + kBlock - 1) / kBlock;
                    for (int t = 0; t < it.ntiles; ++t, ++kv_cnt) {
                        const int st = (int)(kv_cnt % LY::kStages);
                        const uint32_t fill = kv_cnt / LY::kStages;
                        // rows of K/V for every block of the tile; blocks past the
                        // keys' last are copied from past the end of the tensor,
                        // which the copy fills with zeros
                        int yk[kTileBlocks], yv[kTileBlocks];
                        int bad = 0;
#pragma unroll
                        for (int b = 0; b < kTileBlocks; ++b) {
                            const int lb = kTileBlocks * t + b;
                            const int id = lb < nb ? __ldg(row + lb) : 0;
                            const bool ok = id >= 0 && id < p.num_blocks;
                            bad |= !ok;
                            yk[b] = lb < nb ? (ok ? id : 0) * Hkv * kBlock + it.g * kBlock : k_rows;
                            if constexpr (VS)   // the fp16 copy is by logical block
                                yv[b] = lb < nb ? ((it.s * p.max_blocks_per_seq + lb) * Hkv + it.g) * kBlock
                                                : v_rows;
                            else
                                yv[b] = yk[b];
                        }
                        if (bad) atomicOr(p.status, PKV_DEV_BAD_BLOCK);
                        const uint32_t ks = smem_addr(stage_s + st * LY::kStageBytes);
                        const uint32_t vs = ks + LY::kKVBytes;
                        // K of the tile, once both S of the tile two back are done
                        if (fill >= 1 && !mbar_wait(smem_addr(&k_empty[st]), (fill - 1) & 1u,
                                                    abort_flag, p.status))
                            break;
                        last_par[st] = (int)(fill & 1u);
                        const uint32_t kfb = smem_addr(&k_full[st]);
                        mbar_arrive_expect_tx(kfb, (uint32_t)LY::kKVBytes);
#pragma unroll
                        for (int b = 0; b < kTileBlocks; ++b) {
#pragma unroll
                            for (int rg = 0; rg < LY::kRegions; ++rg)
                                tma_load_2d(ks + rg * kKeys * 128 + b * kBlock * 128, &tmK, rg * 64, yk[b], kfb);
                        }
                        // V, once both P V of the tile two back are done (issued
                        // before the S above, so this rarely waits); the bad-block
                        // flag goes with V, which the softmax waits for
                        if (fill >= 1 && !mbar_wait(smem_addr(&v_empty[st]), (fill - 1) & 1u,
                                                    abort_flag, p.status))
                            break;
                        stage_bad[st] = bad;
                        last_par[LY::kStages + st] = (int)(fill & 1u);
                        const uint32_t vfb = smem_addr(&v_full[st]);
                        mbar_arrive_expect_tx(vfb, (uint32_t)LY::kKVBytes);
#pragma unroll
                        for (int b = 0; b < kTileBlocks; ++b) {
#pragma unroll
                            for (int rg = 0; rg < LY::kRegions; ++rg)
                                tma_load_2d(vs + rg * kKeys * 128 + b * kBlock * 128, &tmV, rg * 64, yv[b], vfb);
                        }
                    }
                }
                // after a timed-out wait: let the copies still in flight land first
                if (*abort_flag) {
                    for (int k = 0; k <= 2 * LY::kStages; ++k) {
                        const int par = last_par[k];
                        if (par < 0) continue;
                        const uint32_t fb = smem_addr(k < LY::kStages       ? &k_full[k]
                                                      : k < 2 * LY::kStages ? &v_full[k - LY::kStages]
                                                                            : q_full);
                        const unsigned long long t0 = globaltimer();
                        while (!mbar_try_wait(fb, (uint32_t)par)) {
                            if (globaltimer() - t0 > kTimeoutNs) break;
                        }
                    }
                }
            }
        } else if (warp == kIssuer || warp == kIssuer + 1) {
            // one issuer per query tile
            if (lane == 0) {
                const int gr = warp - kIssuer;
                const uint32_t id_qk = tc::idesc_f16(BF16, kRows, kKeys, 0, 0);
                const uint32_t id_pv = tc::idesc_f16(false, kRows, D, 0, 1);       // P and V: fp16
                const uint32_t q_a = smem_addr(q_s) + gr * LY::kQBytes, st_a = smem_addr(stage_s);
                const uint32_t s_t = tmem + kKeys * gr, o_t = tmem + 256 + 128 * gr;
                // Descriptors are built once per operand base; each MMA adds its
                // constant offset to the address field (offset >> 4: no carry
                // leaves the field, shared memory is below 256 KB), which keeps the
                // issuing thread's instruction stream short.
                const uint64_t qa_d = tc::desc_sw128(q_a, 16, 1024);
                uint32_t tg = 0, it_cnt = 0;
                bool ok = true;
                // P V of tile t for this group, then its share of freeing the stage
                auto issue_pv = [&](uint32_t t, bool first) {
                    const uint32_t vs = st_a + (t % LY::kStages) * LY::kStageBytes + LY::kKVBytes;
                    if (!mbar_wait(smem_addr(&p_full[gr]), t & 1u, abort_flag, p.status) ||
                        !mbar_wait(smem_addr(&v_full[t % LY::kStages]), (t / LY::kStages) & 1u, abort_flag,
                                   p.status)) {
                        ok = false;
                        return;
                    }
                    tc::fence_after_sync();
                    const uint64_t vb_d = tc::desc_sw128(vs, kKeys * 128, 1024);
#pragma unroll
                    for (int kk = 0; kk < kKeys / 16; ++kk) {
                        const uint64_t b = vb_d + (uint64_t)((kk * 16 * 128) >> 4);
                        tc::mma_f16_ts(o_t, s_t + kk * 8, b, id_pv, !(first && kk == 0));
                    }
                    tc::mma_commit(smem_addr(&v_empty[t % LY::kStages]));
                };
                Item nxt = {};
                if ((int)blockIdx.x < total) nxt = tcp::load_item<false, kKeys>(p, blockIdx.x, total, QT);
                for (int i = blockIdx.x; i < total && ok; i += gridDim.x, ++it_cnt) {
                    const Item it = nxt;
                    if (i + (int)gridDim.x < total) nxt = tcp::load_item<false, kKeys>(p, i + gridDim.x, total, QT);
                    if (!mbar_wait(smem_addr(q_full), it_cnt & 1u, abort_flag, p.status)) break;
                    for (int t = 0; t < it.ntiles && ok; ++t, ++tg) {
                        if (t >= 1) {
                            issue_pv(tg - 1, t == 1);
                            if (!ok) break;
                        }
                        const uint32_t st = tg % LY::kStages;
                        if (!mbar_wait(smem_addr(&k_full[st]), (tg / LY::kStages) & 1u, abort_flag,
                                       p.status)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
                        const uint64_t kb_d = tc::desc_sw128(st_a + st * LY::kStageBytes, 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = (kk & 3) * 32;     // 16 values inside the row
                            const uint64_t a = qa_d + (uint64_t)(((kk >> 2) * kRows * 128 + off) >> 4);
                            const uint64_t b = kb_d + (uint64_t)(((kk >> 2) * kKeys * 128 + off) >> 4);
                            tc::mma_f16(s_t, a, b, id_qk, kk > 0);
                        }
                        tc::mma_commit(smem_addr(&s_full[gr]));
                        tc::mma_commit(smem_addr(&k_empty[st]));
                        if (t == it.ntiles - 1) tc::mma_commit(smem_addr(q_empty));
                    }
                    if (!ok) break;
                    issue_pv(tg - 1, it.ntiles == 1);
                    if (ok) tc::mma_commit(smem_addr(&o_full[gr]));
                }
                // every MMA this thread issued has completed before the columns are freed
                tc::mma_commit(smem_addr(&done[gr]));
                const unsigned long long t0 = globaltimer();
                while (!mbar_try_wait(smem_addr(&done[gr]), 0)) {
                    if (globaltimer() - t0 > kTimeoutNs) {
                        atomicOr(p.status, PKV_DEV_TIMEOUT);
                        break;
                    }
                }
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // ---------------------------------------------------------- softmax
        const int gr = warp >> 2;                   // query tile of this warpgroup
        const int r = threadIdx.x - kRows * gr;     // row = tensor-memory lane
        const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const uint32_t s_col = kKeys * gr, o_col = 256 + 128 * gr;
        uint32_t tg = 0, it_cnt = 0;
        bool alive = true;
        Item nxt = {};
        if ((int)blockIdx.x < total) nxt = tcp::load_item<false, kKeys>(p, blockIdx.x, total, QT);
        for (int i = blockIdx.x; i < total && alive; i += gridDim.x, ++it_cnt) {
            const Item it = nxt;
            if (i + (int)gridDim.x < total) nxt = tcp::load_item<false, kKeys>(p, i + gridDim.x, total, QT);
            const int jj = r / G, h = r - (r / G) * G;
            const int tg0 = it.t0 + gr * QT;            // this group's first token
            const bool valid = r < QT * G && tg0 + jj < it.t1;
            const int pos = valid ? it.L - it.C + tg0 + jj : it.nkeys - 1;
            // the fp16 copy's scale 2^k, loaded now so its latency is hidden
            float p2k = 1.f;
            if constexpr (VS)
                p2k = __int_as_float((127 + v16_shift(__ldg(p.v_emax + (size_t)it.s * Hkv + it.g))) << 23);
            float m_ref = -INFINITY, l = 0.f;
            int bad = 0;
            for (int t = 0; t < it.ntiles; ++t, ++tg) {
                const uint32_t st = tg % LY::kStages;
                const bool okS = mbar_wait(smem_addr(&s_full[gr]), tg & 1u, abort_flag, p.status);
                if (!__all_sync(kFull, okS)) { alive = false; break; }
                tc::fence_after_sync();
                float x[kKeys];
#pragma unroll
                for (int q = 0; q < kKeys / 32; ++q) {
                    uint32_t v[32];
                    tc::tmem_ld32(lane_base + s_col + 32 * q, v);
#pragma unroll
                    for (int c = 0; c < 32; ++c) x[32 * q + c] = __uint_as_float(v[c]);
                }
                tc::tmem_wait_ld();
                // raw scores; the scale enters inside the exponent (one FFMA each).
                // Per 32-key chunk, warp-wide: every row of the warp sees all of it,
                // none of it (no maximum, weights 0, no exponentials), or some of
                // it (hidden keys kept out of the maximum and given weight 0).  A
                // warp's rows are consecutive tokens, so at most a chunk or two
                // of the tile is mixed.
                const int k0 = t * kKeys;
                const int nv = pos - k0 + 1;          // keys of the tile this row sees
                uint32_t vis = 0, hid = 0;
#pragma unroll
                for (int q = 0; q < kKeys / 32; ++q) {
                    vis |= (uint32_t)__all_sync(kFull, nv >= 32 * (q + 1)) << q;
                    hid |= (uint32_t)__all_sync(kFull, nv <= 32 * q) << q;
                }
                const bool neg = p.scale_log2 < 0.f;   // the largest scaled score is the smallest raw one
                const float hide = neg ? INFINITY : -INFINITY;
                constexpr uint32_t kAll = (1u << (kKeys / 32)) - 1;
                // the largest scaled score of the keys the row sees (hidden keys'
                // scores are overwritten with `hide`)
                auto tile_max = [&]() -> float {
                    float mx = hide;
                    if (vis == kAll) {          // the usual tile: two chains, no branches
                        if (!neg) {
                            float ma = fmaxf(x[0], x[1]), mb = fmaxf(x[64], x[65]);
#pragma unroll
                            for (int c = 2; c < 64; c += 2) {
                                ma = max3f(ma, x[c], x[c + 1]);
                                mb = max3f(mb, x[64 + c], x[64 + c + 1]);
                            }
                            mx = fmaxf(ma, mb);
                        } else {
                            float ma = fminf(x[0], x[1]), mb = fminf(x[64], x[65]);
#pragma unroll
                            for (int c = 2; c < 64; c += 2) {
                                ma = min3f(ma, x[c], x[c + 1]);
                                mb = min3f(mb, x[64 + c], x[64 + c + 1]);
                            }
                            mx = fminf(ma, mb);
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < kKeys / 32; ++q) {
                            if ((hid >> q) & 1u) continue;
                            float *xq = x + 32 * q;
                            if (!((vis >> q) & 1u)) {
#pragma unroll
                                for (int c = 0; c < 32; ++c)
                                    if (32 * q + c >= nv) xq[c] = hide;
                            }
                            float m;
                            if (!neg) {
                                m = fmaxf(xq[0], xq[1]);
#pragma unroll
                                for (int c = 2; c < 32; c += 2) m = max3f(m, xq[c], xq[c + 1]);
                                mx = fmaxf(mx, m);
                            } else {
                                m = fminf(xq[0], xq[1]);
#pragma unroll
                                for (int c = 2; c < 32; c += 2) m = min3f(m, xq[c], xq[c + 1]);
                                mx = fminf(mx, m);
                            }
                        }
                    }
                    return mx * p.scale_log2;
                };
                // weights 2^(scale x - m_ref) in pairs (packed fp32 arithmetic,
                // f32x2), stored as fp16 P over the tile's S columns (all read
                // above), columns [0, kKeys / 2), 16 per chunk of 32 keys.
                // Hidden keys get exponent -inf (weight 0).  emax is the largest
                // exponent of a key the row sees.
                const uint64_t sc2 = pack2f(p.scale_log2, p.scale_log2);
                uint64_t lsum2 = pack2f(0.f, 0.f);
                float emax = -INFINITY;
                auto weights = [&](auto masked, const int q, const uint64_t nm2) {
                    uint32_t hi[16];
#pragma unroll
                    for (int cc = 0; cc < 32; cc += 2) {
                        const int c = 32 * q + cc;
                        float2 e = unpack2f(fma2f(pack2f(x[c], x[c + 1]), sc2, nm2));
                        if constexpr (decltype(masked)::value) {
                            if (c >= nv) e.x = -INFINITY;
                            if (c + 1 >= nv) e.y = -INFINITY;
                        }
                        emax = max3f(emax, e.x, e.y);
                        const float p0 = fast_exp2(e.x), p1 = fast_exp2(e.y);
                        const uint64_t pp = pack2f(p0, p1);
                        lsum2 = add2f(lsum2, pp);
                        hi[cc / 2] = Elem<false>::pack(p0, p1);   // fp16: relative error <= 2^-11
                    }
                    tc::tmem_st16(lane_base + s_col + 16 * q, hi);
                };
                // the chunk choice is warp-uniform, as the warp-wide tcgen05.st in
                // each branch needs
                auto weights_pass = [&]() {
                    const uint64_t nm2 = pack2f(-m_ref, -m_ref);
                    lsum2 = pack2f(0.f, 0.f);
                    emax = -INFINITY;
                    if (vis == kAll) {
#pragma unroll
                        for (int q = 0; q < kKeys / 32; ++q) weights(std::false_type{}, q, nm2);
                    } else {
#pragma unroll
                        for (int q = 0; q < kKeys / 32; ++q) {
                            if ((hid >> q) & 1u) {
                                uint32_t z[16];
#pragma unroll
                                for (int k = 0; k < 16; ++k) z[k] = 0u;
                                tc::tmem_st16(lane_base + s_col + 16 * q, z);
                            } else if ((vis >> q) & 1u) {
                                weights(std::false_type{}, q, nm2);
                            } else {
                                weights(std::true_type{}, q, nm2);
                            }
                        }
                    }
                };
                // Lazy reference maximum: weights are taken against m_ref as it
                // stands; only when a score the row sees exceeds it by more than
                // kLazy (log2 units) does m_ref move to the tile's maximum, with O
                // and the sum rescaled and the weights taken again (over the P
                // just stored).  Weights thus stay <= 2^kLazy.  The first tile of
                // an item sets m_ref from its maximum.
                float f = 1.f;
                if (t == 0) m_ref = tile_max();
                // turns: warp w (group 0) takes tile tg after warp w + 4's tile
                // tg - 1, warp w + 4 (group 1) after warp w's tile tg (each waiter
                // is at most one phase behind: the other warp's next turn needs
                // this one's)
                if (gr == 1 || tg > 0) {
                    const uint32_t ph = gr == 0 ? tg - 1 : tg;
                    const bool okw = mbar_wait(smem_addr(&w_done[warp ^ 4]), ph & 1u, abort_flag, p.status);
                    if (!__all_sync(kFull, okw)) { alive = false; break; }
                }
                weights_pass();
                // rows past the query tile's tokens (stale query rows) do not vote:
                // their weights never reach an output
                if (__any_sync(kFull, valid && emax > kLazy)) {
                    const float mx = tile_max();
                    bool resc = false;
                    if (mx > m_ref + kLazy) {
                        f = fast_exp2(m_ref - mx);
                        resc = true;
                        m_ref = mx;
                    }
                    // O is rescaled before P V of this tile: S of this tile being
                    // done means P V of the previous one is too (issued before it)
                    if (__any_sync(kFull, resc)) {
#pragma unroll
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t v[32];
                            tc::tmem_ld32(lane_base + o_col + c0, v);
                            tc::tmem_wait_ld();
#pragma unroll
                            for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * f);
                            tc::tmem_st32(lane_base + o_col + c0, v);
                        }
                    }
                    weights_pass();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&w_done[warp]));
                const float2 ls = unpack2f(lsum2);
                l = l * f + (ls.x + ls.y);
                // V of the tile has landed (its bad-block flag comes with it; the
                // next V into this stage waits for this tile's P V)
                const bool okV = mbar_wait(smem_addr(&v_full[st]), (tg / LY::kStages) & 1u, abort_flag,
                                           p.status);
                if (!__all_sync(kFull, okV)) { alive = false; break; }
                bad |= stage_bad[st];
                // zero the V rows of keys past the last one inside its block (the
                // rest of the last block: stale pool rows; blocks after it came in
                // as zeros)
                const int nvis = it.nkeys - k0;
                const int nstale = min(kKeys, ((it.nkeys + kBlock - 1) / kBlock) * kBlock - k0) - nvis;
                if (nstale > 0) {      // both groups write the same zeros, each before its P
                    uint8_t *vs = stage_s + st * LY::kStageBytes + LY::kKVBytes;
                    const int nrows = nstale;
                    for (int e = r; e < nrows * LY::kRegions * 8; e += kRows) {
                        const int row = nvis + e / (LY::kRegions * 8);
                        const int rem = e % (LY::kRegions * 8);
                        *reinterpret_cast<uint4 *>(vs + (rem >> 3) * kKeys * 128 + row * 128 +
                                                   (rem & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&p_full[gr]));
            }
            if (!alive) break;
            // ---- the item's result: O / l once the last P V is done
            const bool oko = mbar_wait(smem_addr(&o_full[gr]), it_cnt & 1u, abort_flag, p.status);
            if (!__all_sync(kFull, oko)) break;
            tc::fence_after_sync();
            // O / l (VS: in the fp16 copy's units, times 2^k), 64 columns at a
            // time through this warp's staging rows, so that every store
            // instruction writes whole 128-byte lines: lane l writes its row
            // (16-byte chunk j at position j ^ (l & 7), free of bank conflicts),
            // then the warp stores 4 rows x 128 bytes per instruction.
            const float scl = (1.f / l) * p2k;
            const uint64_t scl2 = pack2f(scl, scl);
            T *out = static_cast<T *>(p.out) +
                     ((size_t)(it.r0 + tg0 + jj) * p.num_q_heads + (size_t)it.g * G + h) * D;
            uint8_t *ep = base + LY::kEpi + warp * LY::kEpiWarpBytes;
#pragma unroll
            for (int half = 0; half < D / 64; ++half) {
                uint32_t v[2][32];
                tc::tmem_ld32(lane_base + o_col + 64 * half, v[0]);
                tc::tmem_ld32(lane_base + o_col + 64 * half + 32, v[1]);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t *x = &v[j >> 2][8 * (j & 3)];
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 y = unpack2f(
                            mul2f(pack2f(__uint_as_float(x[2 * e]), __uint_as_float(x[2 * e + 1])), scl2));
                        w[e] = bad ? 0u : E::pack(y.x, y.y);
                    }
                    *reinterpret_cast<uint4 *>(ep + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = 4 * i + (lane >> 3), j = lane & 7;
                    const uint4 w = *reinterpret_cast<const uint4 *>(ep + row * 128 + ((j ^ (row & 7)) << 4));
                    const unsigned long long dst =
                        __shfl_sync(kFull, (unsigned long long)reinterpret_cast<uintptr_t>(out), row);
                    if (__shfl_sync(kFull, (int)valid, row))
                        *reinterpret_cast<uint4 *>(reinterpret_cast<T *>(dst) + 64 * half + 8 * j) = w;
                }
                __syncwarp();
            }
            tc::fence_before_sync();
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, LY::kTmemCols);
}

}  // namespace tcw

// --------------------------------------------------------------------- host side
static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

static int64_t max_items(int64_t S, int64_t T, int64_t QT) { return T / QT + S + 1; }

// tokens of one item: kGroups query tiles of kRows / G tokens each
static int tile_tokens(int G) { return tcp::kGroups * (tcp::kRows / G); }

static size_t ws_bytes(int64_t S, int64_t T, int64_t G)
{
    return 256 + align256((size_t)max_items(S, T, tile_tokens((int)G)) * 8);
}

// The workspace with room for the fp16 copy of V after the work list: the
// per-(sequence, kv head) exponent maxima, then [S * maxb][Hkv][16][D] fp16.
struct StagedLayout {
    size_t emax, v16, total;
};
static StagedLayout staged_layout(int64_t S, int64_t T, int64_t G, int64_t Hkv, int64_t D,
                                  int64_t maxb)
{
    StagedLayout l;
    l.emax = ws_bytes(S, T, G);
    l.v16 = l.emax + align256((size_t)(S * Hkv) * 4);
    l.total = l.v16 + align256((size_t)(S * maxb) * Hkv * kBlock * D * 2);
    return l;
}

using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

static EncodeFn encode_fn()
{
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(ptr);
    });
    return fn;
}

// Rows of head_dim values (a pool viewed as [blocks * Hkv * 16][D], or the fp16
// copy of V as [S * maxb * Hkv * 16][D]); a box is 16 rows of 64 values.
static bool make_rows_map(CUtensorMap *map, const void *base, int64_t rows, int head_dim, bool bf16)
{
    EncodeFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBoxCols, (cuuint32_t)kBlock};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
               2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool make_pool_map(CUtensorMap *map, const void *pool, const PoolGeometry &g)
{
    return make_rows_map(map, pool, (int64_t)g.num_blocks * g.num_kv_heads * g.block_size,
                         g.head_dim, g.dtype == PKV_BF16);
}

// Query rows [T][Hq][D] as a 4-D view (D, G, Hkv, T): a box (64, G, 1, QT)
// brings the QT x G rows of one kv group's query tile, token-major, into one
// 128-byte-swizzled region.
static bool make_q_map(CUtensorMap *map, const void *q, int64_t T, int Hkv, int G, int D, int QT,
                       bool bf16)
{
    EncodeFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)G, (cuuint64_t)Hkv, (cuuint64_t)T};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)G * D * 2, (cuuint64_t)Hkv * G * D * 2};
    cuuint32_t box[4] = {64u, (cuuint32_t)G, 1u, (cuuint32_t)QT};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
               const_cast<void *>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

using TcKernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, Params);

// The kernel for a call: bf16 pools whose V is copied to fp16 take the 128-key
// kernel; P in two bf16 parts takes the 64-key one (whose two S buffers per
// query tile hide the doubled P V), and so do fp16 pools, where it measured
// 1 % faster (0.574 against 0.580 ms on 16 x 2,048-token prompts).
struct TcPick {
    TcKernelFn fn;
    int smem, threads;
    bool reg_split;     // setmaxnreg kernel: the launch must give tcw::kLaunchRegs
};

static bool pick_tc(int D, bool bf16, bool staged, TcPick *k)
{
    if (D != 128 && D != 64) return false;
    if (!bf16 || !staged) {
        k->fn = D == 128 ? (bf16 ? &tcp::prefill_tc_kernel<128, true, false, false>
                                 : &tcp::prefill_tc_kernel<128, false, false, false>)
                         : (bf16 ? &tcp::prefill_tc_kernel<64, true, false, false>
                                 : &tcp::prefill_tc_kernel<64, false, false, false>);
        k->smem = D == 128 ? tcp::Layout<128>::kTotal : tcp::Layout<64>::kTotal;
        k->threads = tcp::kThreads;
        k->reg_split = false;
        return true;
    }
    k->fn = D == 128 ? &tcw::prefill_tc_kernel<128, true, true> : &tcw::prefill_tc_kernel<64, true, true>;
    k->smem = D == 128 ? tcw::Layout<128>::kTotal : tcw::Layout<64>::kTotal;
    k->threads = tcw::kThreads;
    k->reg_split = true;
    return true;
}

// The 128-key kernel's register split assumes the launch gives every thread
// exactly tcw::kLaunchRegs registers (see tcw::kRegsIo).
static bool launch_regs_ok(TcKernelFn fn)
{
    cudaFuncAttributes a;
    return cudaFuncGetAttributes(&a, reinterpret_cast<const void *>(fn)) == cudaSuccess &&
           a.numRegs == tcw::kLaunchRegs;
}

// Resident CTAs per SM of a kernel on the current device, cached per device
// (every kernel of this file fits the table; one that did not would be
// measured again on each call rather than fail).
static int resident(const void *fn, int smem, int threads, int *sms_out)
{
    constexpr int kMaxDev = 64, kMaxVar = 16;
    static std::mutex mu;
    static const void *fns[kMaxDev][kMaxVar];
    static int ctas[kMaxDev][kMaxVar];
    static int sms[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return -1;
    std::lock_guard<std::mutex> lock(mu);
    if (sms[dev] == 0 &&
        cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
    *sms_out = sms[dev];
    for (int i = 0; i < kMaxVar; ++i) {
        if (fns[dev][i] == fn) return ctas[dev][i];
        if (fns[dev][i] == nullptr) {
            if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess)
                return -1;
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess ||
                n < 1)
                return -1;
            fns[dev][i] = fn;
            ctas[dev][i] = n;
            return n;
        }
    }
    int n = 0;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess)
        return -1;
    return n;
}

}  // namespace prefill
}  // namespace pkv

extern "C" size_t paged_prefill_workspace_bytes(int32_t num_seqs, int32_t num_tokens,
                                                int32_t num_q_heads, int32_t num_kv_heads)
{
    if (num_seqs < 0 || num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_q_heads % num_kv_heads || num_q_heads / num_kv_heads > 16)
        return 0;
    return pkv::prefill::ws_bytes(num_seqs, num_tokens, num_q_heads / num_kv_heads);
}

extern "C" size_t paged_prefill_workspace_bytes_staged(int32_t num_seqs, int32_t num_tokens,
                                                       int32_t num_q_heads, int32_t num_kv_heads,
                                                       int32_t head_dim, int32_t max_blocks_per_seq)
{
    if (num_seqs < 0 || num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_q_heads % num_kv_heads || num_q_heads / num_kv_heads > 16 ||
        (head_dim != 64 && head_dim != 128) || max_blocks_per_seq <= 0)
        return 0;
    return pkv::prefill::staged_layout(num_seqs, num_tokens, num_q_heads / num_kv_heads,
                                       num_kv_heads, head_dim, max_blocks_per_seq)
        .total;
}

extern "C" int paged_prefill_attention(const pkv_pool *pool, void *out, const void *q,
                                       const void *k_pool, const void *v_pool,
                                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                                       const int32_t *query_start, const int32_t *context_lens,
                                       int32_t num_seqs, int32_t num_tokens, int32_t num_q_heads,
                                       float scale, void *workspace, size_t workspace_bytes,
                                       int32_t *d_status, void *stream)
{
    using namespace pkv::prefill;
    pkv::PoolGeometry g;
    if (!pkv::pool_geometry(pool, &g) || !pkv::is_16bit(g)) return PKV_ERR_INVALID_ARG;
    if (num_seqs < 0 || num_tokens < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0)
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % g.num_kv_heads) return PKV_ERR_INVALID_ARG;
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return PKV_ERR_INVALID_ARG;
    const int G = num_q_heads / g.num_kv_heads;
    if (g.block_size != pkv::kBlock || G > 16) return PKV_ERR_UNSUPPORTED;
    // a bf16 pool whose caller gave room for the fp16 copy of V takes it
    const StagedLayout sl = staged_layout(num_seqs, num_tokens, G, g.num_kv_heads, g.head_dim,
                                          max_blocks_per_seq);
    const bool staged = g.dtype == PKV_BF16 && workspace_bytes >= sl.total &&
                        (int64_t)num_seqs * max_blocks_per_seq * g.num_kv_heads * pkv::kBlock <
                            ((int64_t)1 << 31);
    TcPick kp;
    if (!pick_tc(g.head_dim, g.dtype == PKV_BF16, staged, &kp)) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0 || num_tokens == 0) return PKV_OK;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !query_start || !context_lens ||
        !workspace || !d_status)
        return PKV_ERR_INVALID_ARG;
    if (!pkv::aligned16(out) || !pkv::aligned16(q) || !pkv::aligned16(k_pool) ||
        !pkv::aligned16(v_pool) || ((uintptr_t)workspace & 255u) ||
        ((uintptr_t)block_tables & 3u) || ((uintptr_t)query_start & 3u) ||
        ((uintptr_t)context_lens & 3u) || ((uintptr_t)d_status & 3u))
        return PKV_ERR_INVALID_ARG;
    if (workspace_bytes < ws_bytes(num_seqs, num_tokens, G)) return PKV_ERR_INVALID_ARG;
    if ((int64_t)g.num_blocks * g.num_kv_heads * g.block_size > (int64_t)1 << 31)
        return PKV_ERR_UNSUPPORTED;
    char *ws = static_cast<char *>(workspace);
    CUtensorMap tk, tv, tq;
    const bool vmap = staged ? make_rows_map(&tv, ws + sl.v16,
                                             (int64_t)num_seqs * max_blocks_per_seq * g.num_kv_heads *
                                                 pkv::kBlock,
                                             g.head_dim, false)
                             : make_pool_map(&tv, v_pool, g);
    if (!make_pool_map(&tk, k_pool, g) || !vmap ||
        !make_q_map(&tq, q, num_tokens, g.num_kv_heads, G, g.head_dim, tcp::kRows / G,
                    g.dtype == PKV_BF16))
        return PKV_ERR_CUDA;

    Params prm;
    prm.out = out;
    prm.q = q;
    prm.block_tables = block_tables;
    prm.query_start = query_start;
    prm.context_lens = context_lens;
    prm.num_seqs = num_seqs;
    prm.num_tokens = num_tokens;
    prm.num_q_heads = num_q_heads;
    prm.num_kv_heads = g.num_kv_heads;
    prm.group = G;
    prm.max_blocks_per_seq = max_blocks_per_seq;
    prm.num_blocks = g.num_blocks;
    prm.tile_tokens = tile_tokens(G);
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.header = static_cast<int32_t *>(workspace);
    prm.items = reinterpret_cast<int2 *>(static_cast<char *>(workspace) + 256);
    prm.max_items = max_items(num_seqs, num_tokens, prm.tile_tokens);
    prm.status = d_status;
    prm.v16 = staged ? reinterpret_cast<uint16_t *>(ws + sl.v16) : nullptr;
    prm.v_emax = staged ? reinterpret_cast<int32_t *>(ws + sl.emax) : nullptr;

    int sms = 0;
    const int per_sm = resident(reinterpret_cast<const void *>(kp.fn), kp.smem, kp.threads, &sms);
    if (per_sm < 1 || (kp.reg_split && !launch_regs_ok(kp.fn))) return PKV_ERR_CUDA;
    int64_t grid = (int64_t)per_sm * sms;
    const int64_t upper = prm.max_items * g.num_kv_heads;
    if (grid > upper) grid = upper;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    prefill_prep_kernel<<<1, 1024, 0, st>>>(prm, g.head_dim);
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    if (staged) {       // exponent maxima, then the fp16 copy of V
        const int64_t units = (int64_t)num_seqs * g.num_kv_heads *
                              ((max_blocks_per_seq * pkv::kBlock + kStageTokens - 1) / kStageTokens);
        const unsigned sgrid = (unsigned)std::min<int64_t>(units, (int64_t)sms * 8);
        const uint16_t *vp = static_cast<const uint16_t *>(v_pool);
        if (g.head_dim == 128) {
            prefill_v16_kernel<128, false><<<sgrid, 256, 0, st>>>(vp, prm);
            prefill_v16_kernel<128, true><<<sgrid, 256, 0, st>>>(vp, prm);
        } else {
            prefill_v16_kernel<64, false><<<sgrid, 256, 0, st>>>(vp, prm);
            prefill_v16_kernel<64, true><<<sgrid, 256, 0, st>>>(vp, prm);
        }
        if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    }
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kp.threads);
    cfg.dynamicSmemBytes = (size_t)kp.smem;
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kp.fn, tk, tv, tq, prm) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// ------------------------------------------------- shared-prefix launcher
// Called by the decode launcher (paged_decode.cu) between its prep kernel,
// which lists the work, and its main kernel; see prefill_tc_kernel's PREFIX mode.
namespace pkv {
namespace prefill {

int shared_prefix_tile_seqs(int G) { return tile_tokens(G); }

bool shared_prefix_supported(const PoolGeometry &g, int G)
{
    return is_16bit(g) && g.block_size == kBlock && (g.head_dim == 64 || g.head_dim == 128) &&
           G >= 1 && G <= 16;
}

int launch_shared_prefix(const SharedPrefixLaunch &a)
{
    const PoolGeometry &g = a.geometry;
    const int G = a.num_q_heads / g.num_kv_heads;
    if (!shared_prefix_supported(g, G)) return PKV_ERR_UNSUPPORTED;
    const bool bf16 = g.dtype == PKV_BF16;
    TcKernelFn fn;
    int smem;
    if (g.head_dim == 128) {
        fn = bf16 ? &tcp::prefill_tc_kernel<128, true, false, true>
                  : &tcp::prefill_tc_kernel<128, false, false, true>;
        smem = tcp::Layout<128>::kTotal;
    } else {
        fn = bf16 ? &tcp::prefill_tc_kernel<64, true, false, true>
                  : &tcp::prefill_tc_kernel<64, false, false, true>;
        smem = tcp::Layout<64>::kTotal;
    }
    CUtensorMap tk, tv, tq;
    if (!make_pool_map(&tk, a.k_pool, g) || !make_pool_map(&tv, a.v_pool, g) ||
        !make_q_map(&tq, a.q, a.num_seqs, g.num_kv_heads, G, g.head_dim, tcp::kRows / G, bf16))
        return PKV_ERR_CUDA;
    Params prm = {};
    prm.q = a.q;
    prm.block_tables = a.block_tables;
    prm.num_seqs = a.num_seqs;
    prm.num_tokens = a.num_seqs;
    prm.num_q_heads = a.num_q_heads;
    prm.num_kv_heads = g.num_kv_heads;
    prm.group = G;
    prm.max_blocks_per_seq = a.max_blocks_per_seq;
    prm.num_blocks = g.num_blocks;
    prm.tile_tokens = tile_tokens(G);
    prm.scale_log2 = a.scale_log2;
    prm.status = a.status;
    prm.prefix_items = a.items;
    prm.prefix_count = a.count;
    prm.piece_info = a.piece_info;
    prm.part_ml = a.part_ml;
    prm.part_o = a.part_o;
    int sms = 0;
    const int per_sm = resident(reinterpret_cast<const void *>(fn), smem, tcp::kThreads, &sms);
    if (per_sm < 1) return PKV_ERR_CUDA;
    // persistent: the number of items is known on the device only
    int64_t grid = (int64_t)per_sm * sms;
    if (grid > (int64_t)a.max_items * g.num_kv_heads) grid = (int64_t)a.max_items * g.num_kv_heads;
    if (grid < 1) grid = 1;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(tcp::kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = a.stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, tk, tv, tq, prm) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace prefill
}  // namespace pkv
