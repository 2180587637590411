// Chunked-prefill attention over the paged KV cache for sm_103a.
//
// "vLLM과 Ollama의 차이" (chunked prefill: long prompts are cut into chunks
// that run in the same batch as the decoding sequences) and "LLM 추론 배칭
// 전략 정리", section 0 (a prefill step processes a prompt's tokens together):
// the chunk's K/V has been written into the cache (kv_cache_write); each of
// its queries, at position p, attends causally over the sequence's tokens 0..p,
// gathered through the block table exactly like decode.
//
// Design (GB300):
//   * Work items are (sequence, kv head, query tile).  A tile holds 64 / G
//     query tokens x the G heads of the GQA group = up to 64 rows, 16 per
//     consumer warp; a persistent grid walks the items in a fixed stride.
//   * Warp 4 streams every K/V block the tile can see (positions up to the
//     tile's last query) with 2-D TMA into an mbarrier ring; all four consumer
//     warps read every stage, each for its own 16 rows, so a stage is released
//     after four arrivals and no warp ever waits more than one phase ahead.
//   * Per block and warp: S = Q K^T on tensor cores (mma.sync m16n8k16),
//     causal mask per row, fp32 online softmax, O += P V with P split into a
//     high and a low bf16/fp16 part (two MMAs) for fp32-grade weights.  Each
//     warp owns complete rows: no split-K, no cross-warp merge.
//   * Waits are bounded (1 s) and report PKV_DEV_TIMEOUT; a slot is released
//     only after its data is consumed, behind fence.proxy.async.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace prefill {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kRows = 16 * kConsumerWarps;      // query rows (token x head) per item

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
};

// (sequence, tile) pairs and zero rows for chunks of invalid sequences.
__global__ void __launch_bounds__(1024) prefill_prep_kernel(Params p, int32_t head_dim)
{
    __shared__ int warp_tot[32];
    __shared__ int carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    griddep_launch_dependents();
    if (tid == 0) carry = 0;
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

template <int D, int NST>
struct Smem {
    static constexpr int kStageBytes = 2 * (D / kBoxCols) * kBoxBytes;
    static constexpr int kTotal = 1024 + NST * kStageBytes + 2 * NST * 8 + 16;
};

template <int D, bool BF16, int NST, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
    prefill_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const Params p)
{
    using E = Elem<BF16>;
    using T = typename E::T;
    using SM = Smem<D, NST>;
    constexpr int kBoxes = D / kBoxCols;
    constexpr int kSlabBytes = kBoxes * kBoxBytes;
    constexpr int KSTEPS = D / 16;
    constexpr int NTILES = D / 8;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *stages = base;
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(base + NST * SM::kStageBytes);
    uint64_t *empty_bar = full_bar + NST;
    volatile int *sm_abort = reinterpret_cast<int *>(empty_bar + NST);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(smem_addr(&full_bar[i]), 1);
            mbar_init(smem_addr(&empty_bar[i]), kConsumerWarps);
        }
        *sm_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    griddep_wait();

    const int Hkv = p.num_kv_heads, G = p.group, QT = p.tile_tokens;
    const int total_items = p.header[0] * Hkv;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        uint32_t cnt = 0, issued = 0, issued_par = 0;
        for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
            const int sj = item / Hkv, g = item - sj * Hkv;
            const int2 it = p.items[sj];
            const int s = it.x;
            const int r0 = __ldg(p.query_start + s), C = __ldg(p.query_start + s + 1) - r0;
            const int L = __ldg(p.context_lens + s);
            const int t1 = min((it.y + 1) * QT, C);
            const int nb = (L - C + t1 - 1) / kBlock + 1;        // blocks up to the last query
            const int32_t *row = p.block_tables + (int64_t)s * p.max_blocks_per_seq;
            for (int cb = 0; cb < nb; cb += 32) {
                const int n = min(32, nb - cb);
                const int my_id = lane < n ? __ldg(row + cb + lane) : 0;
                for (int j = 0; j < n; ++j) {
                    const int pid = __shfl_sync(kFull, my_id, j);
                    if (lane == 0) {
                        const int slot = (int)(cnt % NST);
                        const uint32_t par = (cnt / NST) & 1u;
                        const uint32_t fb = smem_addr(&full_bar[slot]);
                        if (mbar_wait(smem_addr(&empty_bar[slot]), par ^ 1u, sm_abort, p.status)) {
                            if (pid >= 0 && pid < p.num_blocks) {
                                mbar_arrive_expect_tx(fb, 2 * kSlabBytes);
                                const uint32_t dk = smem_addr(stages + slot * SM::kStageBytes);
                                const int y = (pid * Hkv + g) * kBlock;
#pragma unroll
                                for (int bx = 0; bx < kBoxes; ++bx) {
                                    tma_load_2d(dk + bx * kBoxBytes, &tmK, bx * kBoxCols, y, fb);
                                    tma_load_2d(dk + kSlabBytes + bx * kBoxBytes, &tmV,
                                                bx * kBoxCols, y, fb);
                                }
                                issued |= 1u << slot;
                                issued_par = (issued_par & ~(1u << slot)) | (par << slot);
                            } else {
                                atomicOr(p.status, PKV_DEV_BAD_BLOCK);
                                mbar_arrive(fb);
                            }
                        }
                    }
                    ++cnt;
                }
            }
        }
        if (lane == 0) {
            for (int slot = 0; slot < NST; ++slot) {
                if (!(issued & (1u << slot))) continue;
                const uint32_t fb = smem_addr(&full_bar[slot]);
                const uint32_t par = (issued_par >> slot) & 1u;
                const unsigned long long t0 = globaltimer();
                while (!mbar_try_wait(fb, par)) {
                    if (globaltimer() - t0 > kTimeoutNs) {
                        atomicOr(p.status, PKV_DEV_TIMEOUT);
                        break;
                    }
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int hrow = lane >> 2, q4 = lane & 3;
    const int mi = lane >> 3, r8 = lane & 7;
    const int k_tok = ((mi >> 1) << 3) + r8, k_chunk = mi & 1;
    const int v_tok = ((mi & 1) << 3) + r8, v_chunk = mi >> 1;
    uint32_t cnt = 0;

    for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
        const int sj = item / Hkv, g = item - sj * Hkv;
        const int2 it = p.items[sj];
        const int s = it.x;
        const int r0 = __ldg(p.query_start + s), C = __ldg(p.query_start + s + 1) - r0;
        const int L = __ldg(p.context_lens + s);
        const int t0 = it.y * QT, t1 = min(t0 + QT, C);
        const int max_pos = L - C + t1 - 1;
        const int nb = max_pos / kBlock + 1;
        // this thread's two rows: a = warp*16 + hrow, b = a + 8
        const int ra = warp * 16 + hrow, rb = ra + 8;
        const int ta = ra / G, tb = rb / G;
        const bool va = t0 + ta < t1, vb = t0 + tb < t1;
        // positions: invalid rows see the tile's last position (finite, never written)
        const int pa_pos = va ? L - C + t0 + ta : max_pos;
        const int pb_pos = vb ? L - C + t0 + tb : max_pos;
        const size_t qrow_a = ((size_t)(r0 + t0 + ta) * p.num_q_heads + (size_t)g * G + ra % G);
        const size_t qrow_b = ((size_t)(r0 + t0 + tb) * p.num_q_heads + (size_t)g * G + rb % G);
        uint32_t qa[KSTEPS][4];
        {
            const uint32_t *qw = static_cast<const uint32_t *>(p.q);
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                const int c = (kk * 16 + 2 * q4) >> 1;
                qa[kk][0] = va ? __ldg(qw + qrow_a * (D / 2) + c) : 0u;
                qa[kk][2] = va ? __ldg(qw + qrow_a * (D / 2) + c + 4) : 0u;
                qa[kk][1] = vb ? __ldg(qw + qrow_b * (D / 2) + c) : 0u;
                qa[kk][3] = vb ? __ldg(qw + qrow_b * (D / 2) + c + 4) : 0u;
            }
        }
        float o[NTILES][4];
#pragma unroll
        for (int j = 0; j < NTILES; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

        for (int b = 0; b < nb; ++b, ++cnt) {
            const int slot = (int)(cnt % NST);
            const uint32_t par = (cnt / NST) & 1u;
            const bool landed = mbar_wait(smem_addr(&full_bar[slot]), par, sm_abort, p.status);
            if (!__all_sync(kFull, landed)) continue;
            const uint32_t kb = smem_addr(stages + slot * SM::kStageBytes);
            const uint32_t vbase = kb + kSlabBytes;
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
            float u0[4] = {0.f, 0.f, 0.f, 0.f}, u1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                const int chunk = 2 * kk + k_chunk;
                const uint32_t addr = kb + (chunk >> 3) * kBoxBytes + k_tok * 128 +
                                      (((chunk & 7) ^ r8) << 4);
                uint32_t kr[4];
                ldsm_x4(kr, addr);
                if (kk & 1) {
                    E::mma(u0, qa[kk], kr[0], kr[1]);
                    E::mma(u1, qa[kk], kr[2], kr[3]);
                } else {
                    E::mma(s0, qa[kk], kr[0], kr[1]);
                    E::mma(s1, qa[kk], kr[2], kr[3]);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) { s0[i] += u0[i]; s1[i] += u1[i]; }
            // causal mask: key position k is visible to a row at position p iff k <= p
            const int kbase = b * kBlock + 2 * q4;
            float x0 = s0[0] * p.scale_log2, x1 = s0[1] * p.scale_log2;
            float x2 = s1[0] * p.scale_log2, x3 = s1[1] * p.scale_log2;
            float y0 = s0[2] * p.scale_log2, y1 = s0[3] * p.scale_log2;
            float y2 = s1[2] * p.scale_log2, y3 = s1[3] * p.scale_log2;
            if (kbase > pa_pos) x0 = -INFINITY;
            if (kbase + 1 > pa_pos) x1 = -INFINITY;
            if (kbase + 8 > pa_pos) x2 = -INFINITY;
            if (kbase + 9 > pa_pos) x3 = -INFINITY;
            if (kbase > pb_pos) y0 = -INFINITY;
            if (kbase + 1 > pb_pos) y1 = -INFINITY;
            if (kbase + 8 > pb_pos) y2 = -INFINITY;
            if (kbase + 9 > pb_pos) y3 = -INFINITY;
            float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
            float my = fmaxf(fmaxf(y0, y1), fmaxf(y2, y3));
            my = fmaxf(my, __shfl_xor_sync(kFull, my, 1));
            my = fmaxf(my, __shfl_xor_sync(kFull, my, 2));
            // a row whose keys of this block are all hidden keeps its state
            const float mn0 = fmaxf(m0, mx), mn1 = fmaxf(m1, my);
            const float a0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0);
            const float a1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
            const float p0 = exp2f(x0 - mn0), p1 = exp2f(x1 - mn0);
            const float p2 = exp2f(x2 - mn0), p3 = exp2f(x3 - mn0);
            const float e0 = exp2f(y0 - mn1), e1 = exp2f(y1 - mn1);
            const float e2 = exp2f(y2 - mn1), e3 = exp2f(y3 - mn1);
            l0 = l0 * a0 + ((p0 + p1) + (p2 + p3));
            l1 = l1 * a1 + ((e0 + e1) + (e2 + e3));
            m0 = mn0;
            m1 = mn1;
            if (__any_sync(kFull, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                for (int j = 0; j < NTILES; ++j) {
                    o[j][0] *= a0; o[j][1] *= a0; o[j][2] *= a1; o[j][3] *= a1;
                }
            }
            uint32_t ph[4], pl[4];
            ph[0] = E::pack(p0, p1);
            ph[1] = E::pack(e0, e1);
            ph[2] = E::pack(p2, p3);
            ph[3] = E::pack(e2, e3);
            {
                const float2 h0 = E::unpack(ph[0]), h1 = E::unpack(ph[1]);
                const float2 h2 = E::unpack(ph[2]), h3 = E::unpack(ph[3]);
                pl[0] = E::pack(p0 - h0.x, p1 - h0.y);
                pl[1] = E::pack(e0 - h1.x, e1 - h1.y);
                pl[2] = E::pack(p2 - h2.x, p3 - h2.y);
                pl[3] = E::pack(e2 - h3.x, e3 - h3.y);
            }
            // V rows past the tile's last position may hold stale data: zero them
            const int valid = min(kBlock, max_pos + 1 - b * kBlock);
            uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
            if (valid < kBlock) {
                const int t0r = 2 * q4;
                mlo = (t0r < valid ? 0x0000ffffu : 0u) | (t0r + 1 < valid ? 0xffff0000u : 0u);
                mhi = (t0r + 8 < valid ? 0x0000ffffu : 0u) | (t0r + 9 < valid ? 0xffff0000u : 0u);
            }
#pragma unroll
            for (int jj = 0; jj < NTILES / 2; ++jj) {
                const int chunk = 2 * jj + v_chunk;
                const uint32_t addr = vbase + (chunk >> 3) * kBoxBytes + v_tok * 128 +
                                      (((chunk & 7) ^ r8) << 4);
                uint32_t vr[4];
                ldsm_x4_trans(vr, addr);
                vr[0] &= mlo; vr[2] &= mlo;
                vr[1] &= mhi; vr[3] &= mhi;
                E::mma(o[2 * jj], ph, vr[0], vr[1]);
                E::mma(o[2 * jj + 1], ph, vr[2], vr[3]);
                E::mma(o[2 * jj], pl, vr[0], vr[1]);
                E::mma(o[2 * jj + 1], pl, vr[2], vr[3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&empty_bar[slot]));
        }
        // rows are complete: normalise and store
        l0 += __shfl_xor_sync(kFull, l0, 1);
        l0 += __shfl_xor_sync(kFull, l0, 2);
        l1 += __shfl_xor_sync(kFull, l1, 1);
        l1 += __shfl_xor_sync(kFull, l1, 2);
        if (*sm_abort) continue;
        T *out = static_cast<T *>(p.out);
        const float ia = 1.f / l0, ib = 1.f / l1;
#pragma unroll
        for (int j = 0; j < NTILES; ++j) {
            const int d0 = 8 * j + 2 * q4;
            if (va)
                *reinterpret_cast<uint32_t *>(out + qrow_a * D + d0) =
                    E::pack(o[j][0] * ia, o[j][1] * ia);
            if (vb)
                *reinterpret_cast<uint32_t *>(out + qrow_b * D + d0) =
                    E::pack(o[j][2] * ib, o[j][3] * ib);
        }
    }
}

// --------------------------------------------------------------------- host side
static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

static int64_t max_items(int64_t S, int64_t T, int64_t QT) { return T / QT + S + 1; }

static int tile_tokens(int G) { return kRows / G; }

static size_t ws_bytes(int64_t S, int64_t T, int64_t G)
{
    return 256 + align256((size_t)max_items(S, T, tile_tokens((int)G)) * 8);
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

static bool make_pool_map(CUtensorMap *map, const void *pool, const PoolGeometry &g)
{
    EncodeFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)g.head_dim,
                          (cuuint64_t)g.num_blocks * g.num_kv_heads * g.block_size};
    cuuint64_t strides[1] = {(cuuint64_t)g.head_dim * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBoxCols, (cuuint32_t)kBlock};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, g.dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
               2, const_cast<void *>(pool), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

using KernelFn = void (*)(CUtensorMap, CUtensorMap, Params);

template <int D, bool BF16, int NST, int MINB>
static KernelFn kernel_of() { return &prefill_kernel<D, BF16, NST, MINB>; }

static bool pick(int D, bool bf16, KernelFn *fn, int *smem)
{
    if (D == 128) {
        *fn = bf16 ? kernel_of<128, true, 8, 2>() : kernel_of<128, false, 8, 2>();
        *smem = Smem<128, 8>::kTotal;
        return true;
    }
    if (D == 64) {
        *fn = bf16 ? kernel_of<64, true, 16, 2>() : kernel_of<64, false, 16, 2>();
        *smem = Smem<64, 16>::kTotal;
        return true;
    }
    return false;
}

static int resident(KernelFn fn, int smem, int *sms_out)
{
    constexpr int kMaxDev = 64, kMaxVar = 8;
    static std::mutex mu;
    static KernelFn fns[kMaxDev][kMaxVar];
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
            if (cudaFuncSetAttribute(reinterpret_cast<const void *>(fn),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess)
                return -1;
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                    &n, reinterpret_cast<const void *>(fn), kThreads, smem) != cudaSuccess ||
                n < 1)
                return -1;
            fns[dev][i] = fn;
            ctas[dev][i] = n;
            return n;
        }
    }
    return -1;
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
    KernelFn fn;
    int smem = 0;
    if (!pick(g.head_dim, g.dtype == PKV_BF16, &fn, &smem)) return PKV_ERR_UNSUPPORTED;
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
    CUtensorMap tk, tv;
    if (!make_pool_map(&tk, k_pool, g) || !make_pool_map(&tv, v_pool, g)) return PKV_ERR_CUDA;

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

    int sms = 0;
    const int per_sm = resident(fn, smem, &sms);
    if (per_sm < 1) return PKV_ERR_CUDA;
    int64_t grid = (int64_t)per_sm * sms;
    const int64_t upper = prm.max_items * g.num_kv_heads;
    if (grid > upper) grid = upper;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    prefill_prep_kernel<<<1, 1024, 0, st>>>(prm, g.head_dim);
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, tk, tv, prm) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
