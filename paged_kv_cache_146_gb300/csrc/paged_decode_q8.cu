// PagedAttention decode over an 8-bit KV cache for sm_103a: the kernel behind
// paged_decode_attention_q8 (launched, with the shared prep and merge kernels,
// from paged_decode.cu).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "decode_params.h"
#include "pagedkv.h"
#include "pkv_device.cuh"

namespace pkv {
namespace decode {

// Four stored bytes (byte i = code i + 128) -> fp16 pairs lo = (code0, code1),
// hi = (code2, code3), each value carrying an offset of 1152: the byte u is
// the low mantissa of 1024 (fp16 bits 0x6400 | u = 1024 + u = 1152 + code),
// exact.
__device__ __forceinline__ void offset_pairs(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    lo = __byte_perm(w, 0x64646464u, 0x4140);     // (0x64, u0), (0x64, u1)
    hi = __byte_perm(w, 0x64646464u, 0x4342);     // (0x64, u2), (0x64, u3)
}

// The same pairs without the offset: one packed subtraction of 1152, exact.
__device__ __forceinline__ void code_pairs(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    offset_pairs(w, lo, hi);
    const uint32_t bias = 0x64806480u;                    // (1152, 1152)
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(bias));
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(bias));
}

// (-1152, -1152) as an fp16 pair.  The score products take K codes with their
// offset and start their accumulators from -1152 x (the query row's sum over
// the group), which a product with an all -1152 operand gives:
//   sum_d q_d (-1152) + sum_d q_d (1152 + c_d) = sum_d q_d c_d.
// Every product of an fp16 value and 1152 + c (11 significant bits each) is
// exact in fp32; the offset only makes the terms of the fp32 sums larger
// (up to 1279 |q| instead of 127 |q|), and with them their rounding.
constexpr uint32_t kNegOffset = 0xE480E480u;

// An 8-bit pool ("kv-cache-by-model", section 1: one-byte codes with one fp16
// scale per 32 values) keeps each (block, kv head) slab as one record of
// q8::kSlab = 4,352 bytes, so a block costs one bulk copy:
// Codes are stored biased (byte = code + 128), which saves the decode kernel a
// bias step per code word.
//   [0, 2048)     K codes, 16 rows of 128 bytes: token t = 4a + 2b + c sits in
//                 row 8b + 2a + c, its 16-byte chunk j at position j ^ (row & 7)
//   [2048, 4096)  V codes, 128 dimension rows of 16 bytes (byte = token)
//   [4096, 4224)  K scales, fp16 [16 tokens][4 groups of 32 dimensions]
//   [4224, 4352)  V scales, fp16 [4 groups][16 tokens]
// The row order puts the tokens of each 8-column MMA tile in rows 0-7 and 8-15,
// and the chunk rotation lets ldmatrix read them without bank conflicts.
//
// Work division: every warp is its own producer.  A warp takes whole items
// (sequence, kv head, partition of up to 32 blocks) in a fixed stride over the
// grid, keeps a private ring of kSlots stages and issues the bulk copy of block
// i + kSlots -- across item boundaries, with the next item's metadata and block
// ids prefetched into registers -- right after it has consumed block i.  The
// next item's query rows are copied into the warp's query buffer as soon as the
// current item's rows have been read out of it.  Each copy also prefetches the
// record kPrefetch blocks further on into L2, which raises the bytes in flight
// without taking shared memory.  No producer warp, no cross-warp barriers, no shared-memory merge:
// the warp writes its rows (or its partition's piece) itself.
namespace q8 {
#ifndef PKV_Q8_WARPS
#define PKV_Q8_WARPS 4
#endif
#ifndef PKV_Q8_SLOTS
#define PKV_Q8_SLOTS 3
#endif
#ifndef PKV_Q8_CTAS
#define PKV_Q8_CTAS 3
#endif
constexpr int kSlab = 4352;
constexpr int kWarps = PKV_Q8_WARPS;             // independent warps per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kSlots = PKV_Q8_SLOTS;             // ring stages per warp
constexpr int kMinBlocks = PKV_Q8_CTAS;          // CTAs per SM
#ifndef PKV_Q8_PREFETCH
#define PKV_Q8_PREFETCH 2
#endif
constexpr int kPrefetch = PKV_Q8_PREFETCH;       // L2 prefetch this many blocks past the copy
constexpr int kQBytes = 8 * 128 * 2;              // one item's query rows (G <= 8), fp16/bf16
constexpr int kQOffBytes = 8 * 4 * 4;             // -1152 x query sums, [8 rows][4 groups] fp32
constexpr int kWarpBytes = kSlots * kSlab + kQBytes + kQOffBytes + 128;   // + barriers
constexpr int kSmemBytes = 128 + kWarps * kWarpBytes;
static_assert(kSlab % 128 == 0 && kWarpBytes % 128 == 0, "stages stay 128-byte aligned");
}  // namespace q8

// ------------------------------------------------------------ 8-bit block step
// One 16-token block of an 8-bit slab for the G <= 8 query rows of a warp, all
// products on fp16 tensor cores (codes are exact in fp16; bf16 queries enter as
// fp16 after a power-of-two prescale of their row, exact in the fp16 normal range).
//
// S = Q K^T: Q rows as A (rows 8-15 zero), K codes as B.  Column c of tile b is
// token 4 (c >> 1) + 2b + (c & 1), so lane (hrow, q4) holds the scores of tokens
// 4q4 .. 4q4 + 3 of query row hrow; the K scales multiply the partial score of
// each 32-dimension group.
//   S[t] = sum_i ks[t][i] * (q . codes[t]) over group i
// (the code values enter with an offset of 1152 that the accumulators' start
// value, -1152 x the row's query sum over the group, cancels)
// O^T = V^T P^T: V codes as A (16 dimensions per MMA, k = the 16 tokens), the
// softmax weights times the V scale of the group as B -- exactly the four weights
// the lane holds -- so o[t] covers dimensions 16t + r and 16t + r + 8 (r = lane/4)
// of query rows 2q4 and 2q4 + 1.
//   O[d][h] += sum_t vcode[d][t] * (p[h][t] * vs[t][d / 32])
// (the V codes enter without the offset: cancelling it there cost a product
// per tile, more than the subtraction)
__device__ __forceinline__ void consume_q8_block(uint32_t kb, const uint8_t *scales,
                                                 const uint32_t (&qa)[8][4],
                                                 const float *qoff_row, float (&o)[8][4],
                                                 float &m0, float &l0, int valid,
                                                 float scale_row, int lane)
{
    using H = Elem<false>;
    const int q4 = lane & 3, r8 = lane & 7;
    // ldmatrix rows: matrix (lane >> 3) = (tile (lane >> 3) & 1, step 2i + (lane >> 4))
    const uint32_t krow = kb + ((lane >> 3) & 1) * 1024 + r8 * 128;
    const int kstep_hi = lane >> 4;
    const uint32_t vb = kb + 2048;

    float sc[4] = {0.f, 0.f, 0.f, 0.f};
    {
        const float4 qo = *reinterpret_cast<const float4 *>(qoff_row);
        const float qoff[4] = {qo.x, qo.y, qo.z, qo.w};
        float ks[4][4];        // [token j][group i]
        const uint4 a = *reinterpret_cast<const uint4 *>(scales + 32 * q4);
        const uint4 b = *reinterpret_cast<const uint4 *>(scales + 32 * q4 + 16);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[k]));
            ks[k >> 1][2 * (k & 1)] = f.x;
            ks[k >> 1][2 * (k & 1) + 1] = f.y;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t kr[4];
            ldsm_x4(kr, krow + (((2 * i + kstep_hi) ^ r8) << 4));
            // start from -1152 x (the row's query sum over group i)
            float c0[4] = {qoff[i], qoff[i], 0.f, 0.f}, c1[4] = {qoff[i], qoff[i], 0.f, 0.f};
            uint32_t lo, hi;
            offset_pairs(kr[0], lo, hi);
            H::mma(c0, qa[2 * i], lo, hi);
            offset_pairs(kr[1], lo, hi);
            H::mma(c1, qa[2 * i], lo, hi);
            offset_pairs(kr[2], lo, hi);
            H::mma(c0, qa[2 * i + 1], lo, hi);
            offset_pairs(kr[3], lo, hi);
            H::mma(c1, qa[2 * i + 1], lo, hi);
            sc[0] = fmaf(ks[0][i], c0[0], sc[0]);
            sc[1] = fmaf(ks[1][i], c0[1], sc[1]);
            sc[2] = fmaf(ks[2][i], c1[0], sc[2]);
            sc[3] = fmaf(ks[3][i], c1[1], sc[3]);
        }
    }
    float x[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = sc[j] * scale_row;
    // V scales of this lane's tokens as fp16 pairs: group i -> (4q4, 4q4 + 1),
    // (4q4 + 2, 4q4 + 3)
    uint2 vs[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        vs[i] = *reinterpret_cast<const uint2 *>(scales + 128 + 32 * i + 8 * q4);
    if (valid < kBlock) {
        // tokens past the context: no score, and no scale (a stale one may be NaN)
        const int n = valid - 4 * q4;       // tokens of this lane inside the context
        const uint32_t m01 = n <= 0 ? 0u : (n == 1 ? 0x0000ffffu : 0xffffffffu);
        const uint32_t m23 = n <= 2 ? 0u : (n == 3 ? 0x0000ffffu : 0xffffffffu);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            vs[i].x &= m01;
            vs[i].y &= m23;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (4 * q4 + j >= valid) x[j] = -INFINITY;
    }
    // Lazy reference maximum: m0 moves (exactly to the row maximum, with the
    // accumulators rescaled) only when a score exceeds it by more than
    // kQ8Lazy, so most blocks skip the cross-lane maximum.  Weights then reach
    // 2^kQ8Lazy = 64, and the fp16 product p * vs below stays finite while
    // every V scale of the block is at most 1023 (64 * 1023 < 65504); a block
    // with a larger scale (V values beyond ~1.3e5) takes the exact path, where
    // weights stay <= 1 as they always did.
    constexpr float kQ8Lazy = 6.f;
    bool raise = x[0] > m0 + kQ8Lazy || x[1] > m0 + kQ8Lazy ||
                 x[2] > m0 + kQ8Lazy || x[3] > m0 + kQ8Lazy;
    {
        __half2 m = __hmax2(*reinterpret_cast<const __half2 *>(&vs[0].x),
                            *reinterpret_cast<const __half2 *>(&vs[0].y));
#pragma unroll
        for (int i = 1; i < 4; ++i) {
            m = __hmax2(m, *reinterpret_cast<const __half2 *>(&vs[i].x));
            m = __hmax2(m, *reinterpret_cast<const __half2 *>(&vs[i].y));
        }
        const float2 mf = __half22float2(m);
        raise |= !(mf.x <= 1023.f && mf.y <= 1023.f);
    }
    if (__any_sync(kFull, raise)) {
        float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
        const float mn = fmaxf(m0, mx);
        const float a0 = fast_exp2(m0 - mn);
        l0 *= a0;
        m0 = mn;
        if (__any_sync(kFull, a0 != 1.f)) {
            // this lane's accumulators belong to query rows 2q4 and 2q4 + 1
            const float f0 = __shfl_sync(kFull, a0, 8 * q4);
            const float f1 = __shfl_sync(kFull, a0, 8 * q4 + 4);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                o[t][0] *= f0; o[t][1] *= f1; o[t][2] *= f0; o[t][3] *= f1;
            }
        }
    }
    float pj[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) pj[j] = fast_exp2(x[j] - m0);
    l0 += (pj[0] + pj[1]) + (pj[2] + pj[3]);
    const uint32_t p01 = H::pack(pj[0], pj[1]), p23 = H::pack(pj[2], pj[3]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // weights of group i: p * vs, one fp16 product per pair
        uint32_t b0, b1;
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(b0) : "r"(p01), "r"(vs[i].x));
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(b1) : "r"(p23), "r"(vs[i].y));
        // matrix m: dimensions 32i + 8m .. 32i + 8m + 7 (lane row r = dimension)
        uint32_t vr[4];
        ldsm_x4(vr, vb + (32 * i + lane) * 16);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            uint32_t a[4];
            code_pairs(vr[2 * t], a[0], a[2]);
            code_pairs(vr[2 * t + 1], a[1], a[3]);
            H::mma(o[2 * i + t], a, b0, b1);
        }
    }
}

// An item as one warp sees it; lane l holds the id of the item's block l.
struct Q8Item {
    int item;        // global item index; >= the item count: none
    int s, g, L, b0, nb, nsplit, pair;
    int id;
};

__device__ __forceinline__ void q8_load_item(const Params &p, int it, int total, int lane,
                                             Q8Item &c)
{
    c.item = it;
    c.nb = 0;
    if (it >= total) return;
    const int Hkv = p.num_kv_heads;
    const int pi = it / Hkv;
    c.g = it - pi * Hkv;
    const int2 sp = p.items[pi];
    c.s = sp.x;
    c.L = __ldg(p.context_lens + sp.x);
    const int2 info = __ldg(p.seq_info + sp.x);
    c.nsplit = info.y;
    c.pair = info.x + sp.y;
    c.b0 = sp.y * p.blocks_per_split;
    c.nb = min(p.blocks_per_split, (c.L + kBlock - 1) / kBlock - c.b0);
    c.id = lane < c.nb
               ? __ldg(p.block_tables + (int64_t)c.s * p.max_blocks_per_seq + c.b0 + lane)
               : 0;
}

template <bool BF16>
__global__ void __launch_bounds__(q8::kThreads, q8::kMinBlocks)
    decode_q8_kernel(const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap,
                     const Params p)
{
    using namespace q8;
    using E = Elem<BF16>;
    using T = typename E::T;
    constexpr int D = 128;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    __shared__ int cta_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hrow = lane >> 2, q4 = lane & 3;
    uint8_t *ring = base + warp * kWarpBytes;
    uint8_t *qbuf = ring + kSlots * kSlab;                       // [8 rows][128]
    float *qoff_buf = reinterpret_cast<float *>(qbuf + kQBytes);  // [8 rows][4 groups]
    uint64_t *full = reinterpret_cast<uint64_t *>(qbuf + kQBytes + kQOffBytes);
    uint64_t *qfull = full + kSlots;
    volatile int *abort_flag = &cta_abort;
    if (threadIdx.x == 0) cta_abort = 0;
    // query rows >= G stay zero: the copies write G rows only
    for (int i = lane; i < kQBytes / 16; i += 32)
        reinterpret_cast<uint4 *>(qbuf)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (lane == 0) {
        for (int i = 0; i <= kSlots; ++i) mbar_init(smem_addr(&full[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    zero_idle_rows(p.out, p.context_lens, p.num_seqs, p.num_q_heads * D * 2,
                   (int64_t)p.max_blocks_per_seq * kBlock);
    griddep_wait();                // the work list comes from the prep kernel

    const int Hkv = p.num_kv_heads, G = p.group;
    const int total = p.header[0] * Hkv;
    const int wstride = gridDim.x * kWarps;
    Q8Item cur, nxt;
    q8_load_item(p, blockIdx.x * kWarps + warp, total, lane, cur);
    q8_load_item(p, cur.item + wstride, total, lane, nxt);

    // copy cursor: block cj of the current item, or of the next one (cnext)
    int cj = 0;
    bool cnext = false;
    uint32_t issued = 0, used = 0, bad_mask = 0;
    auto issue = [&]() {
        if (!cnext && cj >= cur.nb) {
            cnext = true;
            cj = 0;
        }
        const int c_item = cnext ? nxt.item : cur.item;
        const int c_nb = cnext ? nxt.nb : cur.nb;
        if (c_item >= total || cj >= c_nb) return;
        const int c_id = cnext ? nxt.id : cur.id;
        const int id = __shfl_sync(kFull, c_id, cj);
        const int c_g = cnext ? nxt.g : cur.g;
        const int slot = (int)(issued % kSlots);
        const bool ok = id >= 0 && id < p.num_blocks;
        // the block kPrefetch further on: in this item, or in the next one
        const int pj = cj + kPrefetch;
        const bool in_c = pj < c_nb;
        const bool in_n = !cnext && !in_c && nxt.item < total && pj - c_nb < nxt.nb;
        const int pf_id = __shfl_sync(kFull, in_c ? c_id : nxt.id, in_c ? pj : (pj - c_nb) & 31);
        const int pf_g = in_c ? c_g : nxt.g;
        if (lane == 0) {
            const uint32_t fb = smem_addr(&full[slot]);
            if (ok) {
                mbar_arrive_expect_tx(fb, kSlab);
                bulk_load(smem_addr(ring + slot * kSlab),
                          p.kv_q8 + ((int64_t)id * Hkv + c_g) * kSlab, kSlab, fb);
            } else {
                atomicOr(p.status, PKV_DEV_BAD_BLOCK);
                mbar_arrive(fb);
            }
            if ((in_c || in_n) && pf_id >= 0 && pf_id < p.num_blocks)
                bulk_prefetch_l2(p.kv_q8 + ((int64_t)pf_id * Hkv + pf_g) * kSlab, kSlab);
        }
        bad_mask = ok ? bad_mask & ~(1u << slot) : bad_mask | (1u << slot);
        ++issued;
        ++cj;
    };
    // query rows of an item: one bulk copy of G rows into the warp's buffer
    const uint32_t q_bytes = (uint32_t)(G * D * 2);
    uint32_t q_issued = 0, q_used = 0;
    auto issue_q = [&](int s, int g) {
        if (lane == 0) {
            const uint32_t qb = smem_addr(qfull);
            mbar_arrive_expect_tx(qb, q_bytes);
            bulk_load(smem_addr(qbuf),
                      static_cast<const T *>(p.q) + ((size_t)s * p.num_q_heads + (size_t)g * G) * D,
                      q_bytes, qb);
        }
        ++q_issued;
    };
    if (cur.item < total) issue_q(cur.s, cur.g);
    for (int k = 0; k < kSlots; ++k) issue();

    bool alive = true;
    while (alive && cur.item < total) {
        // this lane's query words: row hrow, dimensions 16kk + 4q4 .. + 3, as
        // fp16 A fragments (rows 8-15 zero), dimensions permuted inside each
        // 16-wide step to match the K-code words: k slots 2q4 + e <- 16kk + 4q4 + e,
        // 8 + 2q4 + e <- 16kk + 4q4 + 2 + e
        const bool q_landed = mbar_wait(smem_addr(qfull), q_used & 1u, abort_flag, p.status);
        if (!__all_sync(kFull, q_landed)) break;
        ++q_used;
        const uint2 *qrow = reinterpret_cast<const uint2 *>(qbuf + hrow * (D * 2)) + q4;
        uint32_t qa[8][4];
        float scale_row = p.scale_log2;
        if constexpr (BF16) {
            // bf16 row -> fp16 after scaling by 2^-e, e >= 0 the smallest that
            // brings the row's largest magnitude below 2^15; exact for every
            // element in the fp16 normal range.  2^e goes into the row's scale.
            float amax = 0.f;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint2 w = qrow[4 * kk];
                const float2 f0 = E::unpack(w.x), f1 = E::unpack(w.y);
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)),
                                         fmaxf(fabsf(f1.x), fabsf(f1.y))));
            }
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
            const int e = max(0, ((__float_as_int(amax) >> 23) & 0xff) - 127 - 14);
            const float down = __int_as_float((127 - e) << 23);
            scale_row = p.scale_log2 * __int_as_float((127 + e) << 23);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint2 w = qrow[4 * kk];
                const float2 f0 = E::unpack(w.x), f1 = E::unpack(w.y);
                qa[kk][0] = Elem<false>::pack(f0.x * down, f0.y * down);
                qa[kk][2] = Elem<false>::pack(f1.x * down, f1.y * down);
                qa[kk][1] = qa[kk][3] = 0u;
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint2 w = qrow[4 * kk];
                qa[kk][0] = w.x; qa[kk][1] = 0u; qa[kk][2] = w.y; qa[kk][3] = 0u;
            }
        }
        // -1152 x the row's query sum over each 32-dimension group, taken by
        // the tensor cores from the same fp16 operands the scores use
        // (kept in shared memory, [row][group], to spare registers)
        {
            const uint32_t neg = kNegOffset;
            float qoff[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float c[4];
                Elem<false>::mma0(c, qa[2 * i], neg, neg);
                Elem<false>::mma(c, qa[2 * i + 1], neg, neg);
                qoff[i] = c[0];
            }
            if (q4 == 0)
                *reinterpret_cast<float4 *>(qoff_buf + 4 * hrow) =
                    make_float4(qoff[0], qoff[1], qoff[2], qoff[3]);
        }
        // the buffer is free: the next item's rows may come in (async proxy)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (nxt.item < total) issue_q(nxt.s, nxt.g);

        float o[8][4];
#pragma unroll
        for (int t = 0; t < 8; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
        float m0 = -INFINITY, l0 = 0.f;
        uint32_t bad = 0;
        for (int j = 0; j < cur.nb; ++j) {
            const int slot = (int)(used % kSlots);
            const bool landed = mbar_wait(smem_addr(&full[slot]), (used / kSlots) & 1u,
                                          abort_flag, p.status);
            if (!__all_sync(kFull, landed)) {
                alive = false;
                break;
            }
            const uint32_t b = (bad_mask >> slot) & 1u;
            bad |= b;
            if (!b) {
                const int valid = min(kBlock, cur.L - (cur.b0 + j) * kBlock);
                uint8_t *st = ring + slot * kSlab;
                consume_q8_block(smem_addr(st), st + 4096, qa, qoff_buf + 4 * hrow, o, m0, l0,
                                 valid, scale_row, lane);
            }
            // the next copy into this stage goes through the async proxy: order
            // this warp's reads of it first
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            ++used;
            issue();
        }
        if (!alive) break;

        // ---- the item's result.  Lane (hrow, q4) holds dimensions 16t + hrow
        // (+ 8) of query rows 2q4 and 2q4 + 1; row sums come from that row's lanes.
        float lsum = l0 + __shfl_xor_sync(kFull, l0, 1);
        lsum += __shfl_xor_sync(kFull, lsum, 2);
        const float mA = __shfl_sync(kFull, m0, 8 * q4), lA = __shfl_sync(kFull, lsum, 8 * q4);
        const float mB = __shfl_sync(kFull, m0, 8 * q4 + 4);
        const float lB = __shfl_sync(kFull, lsum, 8 * q4 + 4);
        (void)mA; (void)mB;
        const int hA = 2 * q4, hB = 2 * q4 + 1;
        if (cur.nsplit == 1) {
            T *out = static_cast<T *>(p.out) + ((size_t)cur.s * p.num_q_heads + (size_t)cur.g * G) * D;
            const float iA = 1.f / lA, iB = 1.f / lB;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int d = 16 * t + hrow;
                if (hA < G) {
                    out[hA * D + d] = E::from_float(bad ? 0.f : o[t][0] * iA);
                    out[hA * D + d + 8] = E::from_float(bad ? 0.f : o[t][2] * iA);
                }
                if (hB < G) {
                    out[hB * D + d] = E::from_float(bad ? 0.f : o[t][1] * iB);
                    out[hB * D + d + 8] = E::from_float(bad ? 0.f : o[t][3] * iB);
                }
            }
        } else {
            const size_t piece = (size_t)cur.pair * Hkv + cur.g;
            float *po = p.part_o + piece * G * D;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int d = 16 * t + hrow;
                if (hA < G) {
                    po[hA * D + d] = o[t][0];
                    po[hA * D + d + 8] = o[t][2];
                }
                if (hB < G) {
                    po[hB * D + d] = o[t][1];
                    po[hB * D + d + 8] = o[t][3];
                }
            }
            if (q4 == 0 && hrow < G)
                p.part_ml[piece * G + hrow] = make_float2(m0, bad ? -1.f : lsum);
        }

        // ---- move on: the copy cursor, if already in the next item, stays there
        cur = nxt;
        cnext = false;
        q8_load_item(p, cur.item + wstride, total, lane, nxt);
    }

    // after a timed-out wait: let the copies still in flight land before exit
    if (lane == 0) {
        for (uint32_t k = used; k < issued + (q_issued - q_used); ++k) {
            const bool is_q = k >= issued;     // the query copy, if one is pending
            const uint32_t fb = smem_addr(is_q ? qfull : &full[k % kSlots]);
            const uint32_t par = is_q ? (q_used & 1u) : (k / kSlots) & 1u;
            const unsigned long long t0 = globaltimer();
            while (!mbar_try_wait(fb, par)) {
                if (globaltimer() - t0 > kTimeoutNs) {
                    atomicOr(p.status, PKV_DEV_TIMEOUT);
                    break;
                }
            }
        }
    }
}

Q8KernelInfo q8_kernel_info(bool bf16_queries)
{
    const KernelFn fn = bf16_queries ? reinterpret_cast<KernelFn>(&decode_q8_kernel<true>)
                                     : reinterpret_cast<KernelFn>(&decode_q8_kernel<false>);
    return Q8KernelInfo{fn, q8::kSmemBytes, q8::kThreads, q8::kWarps};
}

}  // namespace decode
}  // namespace pkv
