// PagedAttention decode for sm_103a.
//
// The operation ("vLLM의 핵심 원리 PagedAttention 파헤치기", section "KV Cache를
// 블록으로 쪼개다"): for each sequence, follow its block table to the 16-token
// blocks that hold its K and V anywhere in the pool, and compute single-query
// softmax attention for every query head.  Decode attention is bound by the
// bytes of KV it reads, which grow with the batch and are never reused
// ("LLM 추론 배칭 전략 정리", section 2.3), so the kernel is built to keep HBM
// busy:
//
//   * Work items are (sequence, kv head, partition of up to P blocks); a
//     persistent grid walks them in rounds of one item per CTA, alternate
//     rounds from the other end of the list.  A prep kernel turns the
//     device-side context lengths into the item list (no host round trip).
//   * Per CTA: one producer warp issues 2-D TMA copies (cp.async.bulk.tensor,
//     128-byte swizzle) of each block's K and V slab for the item's kv head
//     into a ring of NST shared-memory stages, completed through mbarriers;
//     it streams across item boundaries.  Four consumer warps take the blocks
//     round-robin by their position in the CTA's stream, so every ring slot has
//     a single consumer warp (NST is a multiple of 4).
//   * Consumer, per 16-token block: S = Q K^T on tensor cores (mma.sync
//     m16n8k16, the G query heads of the GQA group as rows, 16 tokens as
//     columns, head_dim as the reduction), fp32 online softmax in registers,
//     then O += P V on tensor cores with P split into a bf16/fp16 high part
//     and a low part (rows 0-7 carry the high part, rows 8-15 the low part when
//     G <= 8), which keeps the weights accurate to ~2^-17.
//   * The producer also copies each item's Q rows (one 1-D bulk copy) and the
//     item's metadata into a double-buffered slot, prefetching the next item's
//     table entries while the current one streams, so consumers never wait on
//     global memory at an item boundary.
//   * The four warps' (o, max, sum) are merged in shared memory; items of a
//     multi-partition sequence write their pieces to the workspace and a small
//     merge kernel combines them by log-sum-exp in partition order --
//     deterministic, and independent of where the blocks physically sit.
//   * Every wait is bounded (1 s); on expiry the kernel flags PKV_DEV_TIMEOUT,
//     stops issuing copies, drains the ones in flight and finishes without
//     trapping.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "pagedkv.h"
#include "decode_params.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace decode {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

// Checked builds (-DPKV_DEBUG_CHECKS) test every data-dependent index before it
// is used, record the first failure in the debug word and skip the access.
// Normal builds compile the checks away.
__device__ __forceinline__ bool dbg_fail(bool ok, int32_t *dbg, int site, long long val)
{
#ifdef PKV_DEBUG_CHECKS
    if (!ok) {
        atomicCAS(dbg, 0, (site << 24) | (int)(val & 0xffffff));
        return true;
    }
#endif
    (void)ok; (void)dbg; (void)site; (void)val;
    return false;
}

// Shared-memory footprint of one kernel variant (without the 1 KiB alignment slack).
template <int D, int GROWS, int NST>
struct Smem {
    static constexpr int kStageBytes = 2 * (D / kBoxCols) * kBoxBytes;  // K slab + V slab
    static constexpr int kStagesBytes = NST * kStageBytes;
    static constexpr int kQSlotBytes = 16 * D * 2;                      // 16 query rows
    static constexpr int kQBytes = 2 * kQSlotBytes;                     // double buffered
    static constexpr int kBarBytes = (2 * NST + 4) * 8;
    static constexpr int kMetaBytes = 2 * 8 * 4;
    static constexpr int kScratchBytes =
        kConsumerWarps * GROWS * (D + 2) * 4 + NST * 4 + kConsumerWarps * 4 + 16;
    static constexpr int kTotal =
        1024 + kStagesBytes + kQBytes + kBarBytes + kMetaBytes + kScratchBytes;
};

// Item metadata the producer hands to the consumers with each item's Q rows:
// sequence, kv head, context length, blocks [b0, b1), the sequence's pieces
// and this partition's piece.
struct ItemMeta {
    int s, g, L, b0, b1, nsplit, pair, pad;
};

// ----------------------------------------------------------------- prep kernel
// One CTA: partitions per sequence, their prefix sum, the item list, and zero
// rows for empty or invalid sequences.
//
// Item order: the persistent grid takes items in rounds of one per CTA, so the
// list ends with the smallest ones and every CTA's last item is short.  Full
// partitions (P blocks) come first, in sequence order; then each sequence's
// partial last partition, by size from large to small (kOrderBins size bins,
// sequence order inside a bin).  The list must not vary between launches with
// equal inputs: a CTA hands its blocks to its consumer warps by their position
// in its own stream, so which CTA takes an item decides how the item's sum is
// split between warps, and with it the last bits of the result.
constexpr int kOrderBins = 64;

// Automatic partition size: the candidates are P0, 2 P0 and 4 P0 blocks (P0 =
// the size the workspace was laid out for, so every candidate fits it).  Larger
// partitions mean fewer pieces to merge and less per-item work; the size stops
// growing once it would leave fewer than kAutoItemsPerCta items per resident
// CTA, below which the grid runs out of parallel work.
constexpr int kAutoSizes = 3;
constexpr int kAutoItemsPerCta = 5;

// Inclusive scan of two counters over the 1024 threads of the prep CTA.
__device__ __forceinline__ int2 prep_scan2(int2 x, int2 (&warp_tot)[32], int lane, int warp)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(kFull, x.x, o), b = __shfl_up_sync(kFull, x.y, o);
        if (lane >= o) { x.x += a; x.y += b; }
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int2 t = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(kFull, t.x, o), b = __shfl_up_sync(kFull, t.y, o);
            if (lane >= o) { t.x += a; t.y += b; }
        }
        warp_tot[lane] = t;
    }
    __syncthreads();
    if (warp > 0) { x.x += warp_tot[warp - 1].x; x.y += warp_tot[warp - 1].y; }
    return x;
}

// Shared prefixes, found from the tables (first part of the prep kernel when
// the call looks for them).  The link from sequence s to s + 1 is the number
// of leading table entries they share, up to the blocks that lie before the
// last token of both (so each keeps at least one token of its own), counting
// valid block ids only.  Links of at least kPrefixMinBlocks join sequences
// into runs; a run of two or more members shares its shortest link: those
// blocks are read once, split into at most kPrefixMaxPieces key chunks, each
// chunk one piece per member (written by the shared-prefix kernel), and each
// member's decode partitions start after them.  Writes seq_skip for every
// sequence, the shared-prefix work list and its count (header[4]).
__device__ void prep_prefix_runs(const Params &p, int2 (&warp_tot)[32], int tid, int lane,
                                 int warp)
{
    const int S = p.num_seqs;
    int32_t *lcp = p.prefix_scratch, *run_start = lcp + S, *run_min = run_start + S,
            *run_n = run_min + S;
    __shared__ int carry_start, n_items;
    const int64_t max_tokens = (int64_t)p.max_blocks_per_seq * kBlock;
    // links: one warp per neighbouring pair, 128 table entries per round
    for (int s = warp; s < S; s += 32) {
        int link = 0;
        if (s + 1 < S) {
            const int La = p.context_lens[s], Lb = p.context_lens[s + 1];
            int f = 0;
            if (La > 0 && (int64_t)La <= max_tokens && Lb > 0 && (int64_t)Lb <= max_tokens)
                f = min((La - 1) / kBlock, (Lb - 1) / kBlock);
            const int32_t *ra = p.block_tables + (int64_t)s * p.max_blocks_per_seq;
            const int32_t *rb = ra + p.max_blocks_per_seq;
            for (int base = 0; base < f; base += 128) {
                int a[4], b[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int i = base + 32 * j + lane;
                    a[j] = i < f ? __ldg(ra + i) : 0;
                    b[j] = i < f ? __ldg(rb + i) : 0;
                }
                int first = 128;
#pragma unroll
                for (int j = 3; j >= 0; --j) {
                    const int i = base + 32 * j + lane;
                    const bool eq = i >= f || (a[j] == b[j] && a[j] >= 0 && a[j] < p.num_blocks);
                    const unsigned ne = __ballot_sync(kFull, !eq);
                    if (ne) first = 32 * j + __ffs(ne) - 1;
                }
                if (first < 128) {
                    link = base + first;
                    break;
                }
                link = min(f, base + 128);
            }
        }
        if (lane == 0) {
            lcp[s] = link;
            run_min[s] = 0x7fffffff;
            run_n[s] = 0;
        }
    }
    if (tid == 0) {
        carry_start = 0;
        n_items = 0;
    }
    __syncthreads();
    // runs: the start of s's run is the last t <= s not linked from t - 1 (a
    // prefix maximum); every member counts itself into its run, every link
    // takes part in the run's minimum
    for (int base = 0; base < S; base += 1024) {
        const int s = base + tid;
        const bool in = s < S;
        const bool from_prev = in && s > 0 && lcp[s - 1] >= kPrefixMinBlocks;
        const bool to_next = in && lcp[s] >= kPrefixMinBlocks;
        int x = in && !from_prev ? s : -1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x = max(x, y);
        }
        if (lane == 31) warp_tot[warp].x = x;
        __syncthreads();
        if (warp == 0) {
            int t = warp_tot[lane].x;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, t, o);
                if (lane >= o) t = max(t, y);
            }
            warp_tot[lane].x = t;
        }
        __syncthreads();
        const int rs = max(max(x, warp > 0 ? warp_tot[warp - 1].x : -1), carry_start);
        if (in) {
            run_start[s] = rs;
            if (to_next) atomicMin(&run_min[rs], lcp[s]);
            if (to_next || from_prev) atomicAdd(&run_n[rs], 1);
        }
        __syncthreads();
        if (tid == 0) carry_start = max(carry_start, warp_tot[31].x);
        __syncthreads();
    }
    // members: skip and pieces; the first member of a run lists its work
    for (int s = tid; s < S; s += 1024) {
        const int rs = run_start[s];
        const int n = run_n[rs];
        int2 sk = make_int2(0, 0);
        if (n >= 2) {
            const int pb = run_min[rs];
            const int pieces = min(kPrefixMaxPieces, (pb + kPrefixMinBlocks - 1) / kPrefixMinBlocks);
            sk = make_int2(pb, pieces);
            if (s == rs) {
                const int cb = (pb + pieces - 1) / pieces;
                const int tt = p.prefix_tile_seqs;
                const int tiles = (n + tt - 1) / tt;
                const int at = atomicAdd(&n_items, tiles * pieces);
                for (int t = 0; t < tiles; ++t)
                    for (int j = 0; j < pieces; ++j) {
                        const int k = at + t * pieces + j;
                        if (dbg_fail(k < p.max_prefix_items, p.debug, 14, k)) continue;
                        p.prefix_items[k] = make_int4(rs + t * tt, min(tt, n - t * tt) | (j << 16),
                                                      j * cb, min(pb, (j + 1) * cb));
                    }
            }
        }
        p.seq_skip[s] = sk;
    }
    __syncthreads();
    if (tid == 0) p.header[4] = min(n_items, p.max_prefix_items);
}

__global__ void __launch_bounds__(1024) decode_prep_kernel(Params p, int32_t head_dim)
{
    __shared__ int2 warp_tot[32];
    __shared__ int2 carry;               // (pairs, full partitions) of earlier chunks
    __shared__ int bin_next[kOrderBins];
    __shared__ int warp_bin[32][kOrderBins];   // pass 2: per-warp counts, then offsets
    __shared__ long long auto_tot[32][kAutoSizes];
    __shared__ int chosen_split;
    __shared__ int multi_count, n_partial;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    griddep_launch_dependents();   // the main kernel may set up its CTAs meanwhile
    if (tid == 0) {
        carry = make_int2(0, 0);
        multi_count = 0;
        n_partial = 0;
    }
    for (int i = tid; i < kOrderBins; i += 1024) bin_next[i] = 0;
    for (int i = tid; i < 32 * kOrderBins; i += 1024) (&warp_bin[0][0])[i] = 0;
    const int64_t max_tokens = (int64_t)p.max_blocks_per_seq * kBlock;
    const bool prefix = p.seq_skip != nullptr;
    if (prefix) prep_prefix_runs(p, warp_tot, tid, lane, warp);
    // blocks of sequence s its decode partitions cover, and its shared-prefix pieces
    auto own = [&](int s, int nb) {
        if (!prefix) return make_int2(nb, 0);
        const int2 sk = p.seq_skip[s];
        return make_int2(nb - sk.x, sk.y);
    };
    // pass 0 (automatic partition size): pairs at P0, 2 P0, 4 P0 blocks per
    // partition; the largest size that still gives auto_split_pairs pairs wins
    if (p.auto_split_pairs > 0) {
        long long n[kAutoSizes] = {};
        for (int s = tid; s < p.num_seqs; s += 1024) {
            const int L = p.context_lens[s];
            if (L <= 0 || (int64_t)L > max_tokens) continue;
            const int nb = own(s, (L + kBlock - 1) / kBlock).x;
#pragma unroll
            for (int k = 0; k < kAutoSizes; ++k) {
                const int Pk = p.blocks_per_split << k;
                n[k] += (nb + Pk - 1) / Pk;
            }
        }
#pragma unroll
        for (int k = 0; k < kAutoSizes; ++k) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) n[k] += __shfl_xor_sync(kFull, n[k], o);
            if (lane == 0) auto_tot[warp][k] = n[k];
        }
        __syncthreads();
        if (tid == 0) {
            int pick = 0;
            for (int k = 1; k < kAutoSizes; ++k) {
                long long t = 0;
                for (int w = 0; w < 32; ++w) t += auto_tot[w][k];
                if (t >= p.auto_split_pairs) pick = k;
            }
            chosen_split = p.blocks_per_split << pick;
        }
    } else if (tid == 0) {
        chosen_split = p.blocks_per_split;
    }
    __syncthreads();
    const int P = chosen_split;
    // bin of a partial last partition of r blocks, 0 < r < P: larger r, lower bin
    auto bin_of = [P](int r) { return (int)((int64_t)(P - 1 - r) * kOrderBins / P); };
    // pass 1: partitions, pair offsets, full partitions, size histogram (a
    // sequence with no context or a bad length gets no partition)
    // (pieces of a sequence: its shared-prefix pieces, then its partitions;
    // carry.x counts pieces, carry.y full partitions, n_partial the rest)
    for (int base = 0; base < p.num_seqs; base += 1024) {
        const int s = base + tid;
        int nsplit = 0, partial = 0, r = 0, npre = 0;
        if (s < p.num_seqs) {
            const int L = p.context_lens[s];
            if (L < 0 || (int64_t)L > max_tokens) {
                atomicOr(p.status, PKV_DEV_BAD_LEN);
            } else if (L > 0) {
                const int2 o = own(s, (L + kBlock - 1) / kBlock);
                npre = o.y;
                nsplit = (o.x + P - 1) / P;
                r = o.x - (nsplit - 1) * P;
                partial = r < P;
            }
        }
        const int npieces = npre + nsplit;
        const int2 inc = prep_scan2(make_int2(npieces, nsplit - partial), warp_tot, lane, warp);
        const int2 c0 = carry;
        const int excl = c0.x + inc.x - npieces;
        const int excl_full = c0.y + inc.y - (nsplit - partial);
        if (s < p.num_seqs &&
            dbg_fail((int64_t)excl + npieces <= p.max_pairs, p.debug, 12, excl)) {
            nsplit = 0;
            partial = 0;
            npre = 0;
        }
        if (s < p.num_seqs) {
            p.seq_info[s] = make_int2(excl, npre + nsplit);
            for (int k = 0; k < nsplit - partial; ++k) p.items[excl_full + k] = make_int2(s, k);
            if (partial) {
                atomicAdd(&bin_next[bin_of(r)], 1);
                atomicAdd(&n_partial, 1);
            }
            if (npre + nsplit > 1) p.multi[atomicAdd(&multi_count, 1)] = s;   // for the merge kernel
            // (a zero row's output is written by the main kernel: zero_idle_rows)
        }
        __syncthreads();
        if (tid == 0) carry = make_int2(c0.x + warp_tot[31].x, c0.y + warp_tot[31].y);
        __syncthreads();
    }
    // bin counts -> first item index of each bin (after the full partitions)
    if (warp == 0) {
        constexpr int kPer = kOrderBins / 32;
        int c[kPer], sum = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) { c[i] = bin_next[lane * kPer + i]; sum += c[i]; }
        int x = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += y;
        }
        int at = carry.y + x - sum;
#pragma unroll
        for (int i = 0; i < kPer; ++i) { bin_next[lane * kPer + i] = at; at += c[i]; }
    }
    __syncthreads();
    // pass 2: partial last partitions into their bins, a stable counting sort:
    // within a chunk, rank among the warp's lanes of the same bin, then the
    // counts of lower warps, then the earlier chunks (bin_next)
    for (int base = 0; base < p.num_seqs; base += 1024) {
        const int s = base + tid;
        int bin = -1, nsplit = 0;
        if (s < p.num_seqs) {
            const int L = p.context_lens[s];
            if (L > 0 && (int64_t)L <= max_tokens && p.seq_info[s].y > 0) {
                const int nb = own(s, (L + kBlock - 1) / kBlock).x;
                nsplit = (nb + P - 1) / P;
                const int r = nb - (nsplit - 1) * P;
                if (r < P) bin = bin_of(r);
            }
        }
        const unsigned peers = __match_any_sync(kFull, bin);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (bin >= 0 && rank == 0) warp_bin[warp][bin] = __popc(peers);
        __syncthreads();
        if (tid < kOrderBins) {
            int at = bin_next[tid];
            for (int w = 0; w < 32; ++w) {
                const int c = warp_bin[w][tid];
                warp_bin[w][tid] = at;
                at += c;
            }
            bin_next[tid] = at;
        }
        __syncthreads();
        if (bin >= 0) {
            const int at = warp_bin[warp][bin] + rank;
            if (!dbg_fail(at < p.max_pairs, p.debug, 13, at)) p.items[at] = make_int2(s, nsplit - 1);
        }
        __syncthreads();
        for (int i = tid; i < 32 * kOrderBins; i += 1024) (&warp_bin[0][0])[i] = 0;
        __syncthreads();
    }
    if (tid == 0) {
        p.header[0] = carry.y + n_partial;      // decode items: full and partial partitions
        p.header[2] = P;
        p.header[3] = multi_count;
        p.header[5] = carry.x;                  // pieces
    }
}

// ----------------------------------------------------------------- main kernel
template <int D, bool BF16, int GROWS, int NST, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const Params p)
{
    using E = Elem<BF16>;
    using T = typename E::T;
    using SM = Smem<D, GROWS, NST>;
    static_assert(NST % kConsumerWarps == 0, "each slot must keep one consumer warp");
    constexpr int kBoxes = D / kBoxCols;          // TMA boxes per slab
    constexpr int kSlabBytes = kBoxes * kBoxBytes;
    constexpr int KSTEPS = D / 16;                // QK reduction steps
    constexpr int NTILES = D / 8;                 // PV output tiles of 8 dims
    constexpr int OSTRIDE = D + 2;                // padded scratch row

    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *stages = base;
    uint8_t *qbuf = base + SM::kStagesBytes;                               // [2][16][D]
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(qbuf + SM::kQBytes);
    uint64_t *empty_bar = full_bar + NST;
    uint64_t *qfull_bar = empty_bar + NST;
    uint64_t *qempty_bar = qfull_bar + 2;
    ItemMeta *sm_meta = reinterpret_cast<ItemMeta *>(qempty_bar + 2);     // [2]
    // per consumer warp, per row: D output sums, then the row's max and sum
    float *sm_o = reinterpret_cast<float *>(sm_meta + 2);                  // [4][GROWS][D + 2]
    int *stage_bad = reinterpret_cast<int *>(sm_o + kConsumerWarps * GROWS * OSTRIDE);
    int *sm_bad = stage_bad + NST;
    volatile int *sm_abort = sm_bad + kConsumerWarps;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // query rows >= G stay zero for the whole kernel: the copies write G rows only
    for (int i = threadIdx.x; i < SM::kQBytes / 16; i += kThreads)
        reinterpret_cast<uint4 *>(qbuf)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(smem_addr(&full_bar[i]), 1);
            mbar_init(smem_addr(&empty_bar[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&qfull_bar[i]), 1);
            mbar_init(smem_addr(&qempty_bar[i]), kConsumerWarps);
        }
        *sm_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    zero_idle_rows(p.out, p.context_lens, p.num_seqs, p.num_q_heads * D * 2,
                   (int64_t)p.max_blocks_per_seq * kBlock);
    griddep_wait();                // the work list comes from the prep kernel

    const int Hkv = p.num_kv_heads, G = p.group, P = p.header[2];   // chosen by the prep kernel
    const int total_items = p.header[0] * Hkv;
    const int stride = gridDim.x;
    // The CTA's k-th item.  The list runs from the largest items to the
    // smallest, so the CTAs take each round of `stride` items in turn from
    // opposite ends (CTA b takes the b-th of even rounds and the b-th from the
    // end of odd ones): every CTA's total stays close to the mean, where a
    // plain stride would give CTA 0 the largest item of every round.  Still a
    // fixed function of the list, so equal inputs give equal bits.
    auto item_of = [&](int k) {
        return k * stride + ((k & 1) ? stride - 1 - (int)blockIdx.x : (int)blockIdx.x);
    };

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        // Metadata of item k+1 is fetched while item k is issued: the item's
        // (sequence, partition) one item ahead, its length, partition info and
        // first 32 block ids one item ahead of that.
        uint32_t cnt = 0, issued = 0, issued_par = 0, q_issued = 0, q_par = 0;
        const uint32_t q_bytes = (uint32_t)(G * D * 2);
        int item = item_of(0);
        int2 it_cur = item < total_items ? p.items[item / Hkv] : make_int2(0, 0);
        int2 it_nxt = item_of(1) < total_items ? p.items[item_of(1) / Hkv] : make_int2(0, 0);
        // info = (first piece of this partition, pieces of the sequence);
        // b0 = first block of the partition (after a shared prefix, if any)
        auto fetch = [&](int2 it, int valid, int &L, int2 &info, int &b0, int &id) {
            L = 0; info = make_int2(0, 0); b0 = 0; id = 0;
            if (!valid) return;
            L = __ldg(p.context_lens + it.x);
            info = __ldg(p.seq_info + it.x);
            b0 = it.y * P;
            info.x += it.y;
            if (p.seq_skip) {
                const int2 sk = __ldg(p.seq_skip + it.x);
                b0 += sk.x;
                info.x += sk.y;
            }
            const int b = b0 + lane;
            if (b < p.max_blocks_per_seq)
                id = __ldg(p.block_tables + (int64_t)it.x * p.max_blocks_per_seq + b);
        };
        int L_cur, id_cur, b0_cur;
        int2 info_cur;
        fetch(it_cur, item < total_items, L_cur, info_cur, b0_cur, id_cur);
        for (int k = 0; item < total_items; ++k, item = item_of(k)) {
            // prefetch
            const int item2 = item_of(k + 2);
            const int2 it_fut = item2 < total_items ? p.items[item2 / Hkv] : make_int2(0, 0);
            int L_nxt, id_nxt, b0_nxt;
            int2 info_nxt;
            fetch(it_nxt, item_of(k + 1) < total_items, L_nxt, info_nxt, b0_nxt, id_nxt);

            const int g = item - (item / Hkv) * Hkv;
            const int s = it_cur.x;
            const int nb = (L_cur + kBlock - 1) / kBlock;
            const int b0 = b0_cur, b1 = min(b0 + P, nb);
            // Q rows + metadata for the consumers
            if (lane == 0) {
                const int qs = k & 1;
                const uint32_t qpar = (k >> 1) & 1;
                if (mbar_wait(smem_addr(&qempty_bar[qs]), qpar ^ 1u, sm_abort, p.status)) {
                    sm_meta[qs] = ItemMeta{s, g, L_cur, b0, b1, info_cur.y, info_cur.x, 0};
                    const uint32_t qb = smem_addr(&qfull_bar[qs]);
                    mbar_arrive_expect_tx(qb, q_bytes);
                    bulk_load(smem_addr(qbuf + qs * SM::kQSlotBytes),
                              static_cast<const T *>(p.q) +
                                  ((size_t)s * p.num_q_heads + (size_t)g * G) * D,
                              q_bytes, qb);
                    q_issued |= 1u << qs;
                    q_par = (q_par & ~(1u << qs)) | (qpar << qs);
                }
            }
            // K/V blocks
            for (int cb = b0; cb < b1; cb += 32) {
                const int n = min(32, b1 - cb);
                int my_id = id_cur;
                if (cb != b0)
                    my_id = lane < n ? __ldg(p.block_tables + (int64_t)s * p.max_blocks_per_seq +
                                             cb + lane)
                                     : 0;
                for (int j = 0; j < n; ++j) {
                    const int pid = __shfl_sync(kFull, my_id, j);
                    if (lane == 0) {
                        const int slot = (int)(cnt % NST);
                        const uint32_t par = (cnt / NST) & 1u;
                        const uint32_t fb = smem_addr(&full_bar[slot]);
                        if (mbar_wait(smem_addr(&empty_bar[slot]), par ^ 1u, sm_abort, p.status)) {
                            if (pid >= 0 && pid < p.num_blocks) {
                                stage_bad[slot] = 0;
                                mbar_arrive_expect_tx(fb, 2 * kSlabBytes);
                                const uint32_t dk = smem_addr(stages + slot * SM::kStageBytes);
                                const uint32_t dv = dk + kSlabBytes;
                                const int y = (pid * Hkv + g) * kBlock;
#pragma unroll
                                for (int bx = 0; bx < kBoxes; ++bx) {
                                    tma_load_2d(dk + bx * kBoxBytes, &tmK, bx * kBoxCols, y, fb);
                                    tma_load_2d(dv + bx * kBoxBytes, &tmV, bx * kBoxCols, y, fb);
                                }
                                issued |= 1u << slot;
                                issued_par = (issued_par & ~(1u << slot)) | (par << slot);
                            } else {
                                stage_bad[slot] = 1;
                                atomicOr(p.status, PKV_DEV_BAD_BLOCK);
                                mbar_arrive(fb);
                            }
                        }
                    }
                    ++cnt;
                }
            }
            it_cur = it_nxt; it_nxt = it_fut;
            L_cur = L_nxt; id_cur = id_nxt; info_cur = info_nxt; b0_cur = b0_nxt;
        }
        // drain: every copy this warp issued must land before the CTA exits
        if (lane == 0) {
            for (int slot = 0; slot < NST + 2; ++slot) {
                const bool is_q = slot >= NST;
                const int sl = is_q ? slot - NST : slot;
                if (!((is_q ? q_issued : issued) & (1u << sl))) continue;
                const uint32_t fb = smem_addr(is_q ? &qfull_bar[sl] : &full_bar[sl]);
                const uint32_t par = ((is_q ? q_par : issued_par) >> sl) & 1u;
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
    const int ctid = threadIdx.x;          // 0..127
    uint32_t cnt_base = 0;
    // ldmatrix lane offsets inside a slab (128-byte swizzle: chunk ^= row % 8)
    const int mi = lane >> 3, r8 = lane & 7;
    const int k_tok = ((mi >> 1) << 3) + r8, k_chunk = mi & 1;   // K: tokens x (chunk, chunk+1)
    const int v_tok = ((mi & 1) << 3) + r8, v_chunk = mi >> 1;   // V^T pairs of 8-dim tiles
    const int q_row = ((mi & 1) << 3) + r8, q_chunk = mi >> 1;   // Q: rows x (chunk, chunk+1)

    for (int k = 0; item_of(k) < total_items; ++k) {
        const int qs = k & 1;
        const bool q_landed = mbar_wait(smem_addr(&qfull_bar[qs]), (k >> 1) & 1, sm_abort, p.status);
        const bool q_ok = __all_sync(kFull, q_landed);
        // after a timed-out wait the slot may be stale: run the item empty
        const ItemMeta mt = q_ok ? sm_meta[qs] : ItemMeta{0, 0, 0, 0, 0, 1, 0, 0};
        // Q rows of the group as the A operand (rows >= G are zero in shared memory)
        uint32_t qa[KSTEPS][4];
        {
            const uint32_t qb = smem_addr(qbuf + qs * SM::kQSlotBytes);
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                if (q_ok)
                    ldsm_x4(qa[kk], qb + q_row * (D * 2) + ((2 * kk + q_chunk) << 4));
                else
                    qa[kk][0] = qa[kk][1] = qa[kk][2] = qa[kk][3] = 0u;
            }
        }
        const int s = mt.s, g = mt.g, L = mt.L, b0 = mt.b0, b1 = mt.b1;

        float o[NTILES][4];
#pragma unroll
        for (int j = 0; j < NTILES; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        int bad = 0;

        // Block c of this CTA's stream (c = cnt_base + b - b0) goes to warp c % 4 and
        // slot c % NST; NST is a multiple of 4, so the previous user of a slot is this
        // same warp, which has seen that phase complete.  A parity wait is only exact
        // when the waiter is at most one phase ahead of the barrier.
        const int first = (warp - (int)(cnt_base % kConsumerWarps) + kConsumerWarps) % kConsumerWarps;
        for (int b = b0 + first; b < b1; b += kConsumerWarps) {
            const uint32_t c = cnt_base + (uint32_t)(b - b0);
            const int slot = (int)(c % NST);
            const uint32_t par = (c / NST) & 1u;
            // warp-uniform: the ldmatrix/mma below need the whole warp
            const bool landed = mbar_wait(smem_addr(&full_bar[slot]), par, sm_abort, p.status);
            if (!__all_sync(kFull, landed)) continue;
            bad |= stage_bad[slot];
            const int valid = min(kBlock, L - b * kBlock);
            const uint32_t kb = smem_addr(stages + slot * SM::kStageBytes);
            const uint32_t vb = kb + kSlabBytes;
            if (dbg_fail(slot < NST && (kb & 1023u) == 0u, p.debug, 7, slot)) continue;

            // ---- S = Q K^T : two 8-token tiles, two accumulation chains each
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
            // ---- online softmax (row hrow: s0[0..1], s1[0..1]; row hrow+8: [2..3])
            const int t0 = 2 * q4;
            float x0 = s0[0] * p.scale_log2, x1 = s0[1] * p.scale_log2;
            float x2 = s1[0] * p.scale_log2, x3 = s1[1] * p.scale_log2;
            float y0 = s0[2] * p.scale_log2, y1 = s0[3] * p.scale_log2;
            float y2 = s1[2] * p.scale_log2, y3 = s1[3] * p.scale_log2;
            if (valid < kBlock) {
                if (t0 >= valid) x0 = y0 = -INFINITY;
                if (t0 + 1 >= valid) x1 = y1 = -INFINITY;
                if (t0 + 8 >= valid) x2 = y2 = -INFINITY;
                if (t0 + 9 >= valid) x3 = y3 = -INFINITY;
            }
            float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
            const float mn0 = fmaxf(m0, mx);
            const float a0 = exp2f(m0 - mn0);
            const float p0 = exp2f(x0 - mn0), p1 = exp2f(x1 - mn0);
            const float p2 = exp2f(x2 - mn0), p3 = exp2f(x3 - mn0);
            l0 = l0 * a0 + ((p0 + p1) + (p2 + p3));
            m0 = mn0;
            uint32_t pa[4], pb[4];
            if constexpr (GROWS == 8) {
                if (__any_sync(kFull, a0 != 1.f)) {
#pragma unroll
                    for (int j = 0; j < NTILES; ++j) {
                        o[j][0] *= a0; o[j][1] *= a0; o[j][2] *= a0; o[j][3] *= a0;
                    }
                }
                // rows 0-7: high part of P, rows 8-15: low part
                pa[0] = E::pack(p0, p1);
                pa[2] = E::pack(p2, p3);
                const float2 h01 = E::unpack(pa[0]), h23 = E::unpack(pa[2]);
                pa[1] = E::pack(p0 - h01.x, p1 - h01.y);
                pa[3] = E::pack(p2 - h23.x, p3 - h23.y);
                (void)pb;
            } else {
                float my = fmaxf(fmaxf(y0, y1), fmaxf(y2, y3));
                my = fmaxf(my, __shfl_xor_sync(kFull, my, 1));
                my = fmaxf(my, __shfl_xor_sync(kFull, my, 2));
                const float mn1 = fmaxf(m1, my);
                const float a1 = exp2f(m1 - mn1);
                const float e0 = exp2f(y0 - mn1), e1 = exp2f(y1 - mn1);
                const float e2 = exp2f(y2 - mn1), e3 = exp2f(y3 - mn1);
                l1 = l1 * a1 + ((e0 + e1) + (e2 + e3));
                m1 = mn1;
                if (__any_sync(kFull, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                    for (int j = 0; j < NTILES; ++j) {
                        o[j][0] *= a0; o[j][1] *= a0; o[j][2] *= a1; o[j][3] *= a1;
                    }
                }
                pa[0] = E::pack(p0, p1);
                pa[1] = E::pack(e0, e1);
                pa[2] = E::pack(p2, p3);
                pa[3] = E::pack(e2, e3);
                const float2 h0 = E::unpack(pa[0]), h1 = E::unpack(pa[1]);
                const float2 h2 = E::unpack(pa[2]), h3 = E::unpack(pa[3]);
                pb[0] = E::pack(p0 - h0.x, p1 - h0.y);
                pb[1] = E::pack(e0 - h1.x, e1 - h1.y);
                pb[2] = E::pack(p2 - h2.x, p3 - h2.y);
                pb[3] = E::pack(e2 - h3.x, e3 - h3.y);
            }
            // ---- O += P V
            uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;   // zero V rows past the context
            if (valid < kBlock) {
                mlo = (t0 < valid ? 0x0000ffffu : 0u) | (t0 + 1 < valid ? 0xffff0000u : 0u);
                mhi = (t0 + 8 < valid ? 0x0000ffffu : 0u) | (t0 + 9 < valid ? 0xffff0000u : 0u);
            }
#pragma unroll
            for (int jj = 0; jj < NTILES / 2; ++jj) {
                const int chunk = 2 * jj + v_chunk;
                const uint32_t addr = vb + (chunk >> 3) * kBoxBytes + v_tok * 128 +
                                      (((chunk & 7) ^ r8) << 4);
                uint32_t vr[4];
                ldsm_x4_trans(vr, addr);
                vr[0] &= mlo; vr[2] &= mlo;
                vr[1] &= mhi; vr[3] &= mhi;
                E::mma(o[2 * jj], pa, vr[0], vr[1]);
                E::mma(o[2 * jj + 1], pa, vr[2], vr[3]);
                if constexpr (GROWS == 16) {
                    E::mma(o[2 * jj], pb, vr[0], vr[1]);
                    E::mma(o[2 * jj + 1], pb, vr[2], vr[3]);
                }
            }
            // The stage's next contents arrive through the async proxy (TMA):
            // order this warp's generic-proxy reads of it before the release.
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&empty_bar[slot]));
        }
        cnt_base += (uint32_t)(b1 - b0);
        // Release the Q slot only now, after the QK products have consumed the
        // fragments read from it (the next copy into it may land at once).
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0 && q_ok) mbar_arrive(smem_addr(&qempty_bar[qs]));

        // ---- per-warp state into shared memory
        l0 += __shfl_xor_sync(kFull, l0, 1);
        l0 += __shfl_xor_sync(kFull, l0, 2);
        if constexpr (GROWS == 16) {
            l1 += __shfl_xor_sync(kFull, l1, 1);
            l1 += __shfl_xor_sync(kFull, l1, 2);
        }
        float *wo = sm_o + warp * GROWS * OSTRIDE;
        if (q4 == 0) {
            wo[hrow * OSTRIDE + D] = m0;
            wo[hrow * OSTRIDE + D + 1] = l0;
            if constexpr (GROWS == 16) {
                wo[(hrow + 8) * OSTRIDE + D] = m1;
                wo[(hrow + 8) * OSTRIDE + D + 1] = l1;
            }
        }
#pragma unroll
        for (int j = 0; j < NTILES; ++j) {
            const int d0 = 8 * j + 2 * q4;
            if constexpr (GROWS == 8) {
                *reinterpret_cast<float2 *>(&wo[hrow * OSTRIDE + d0]) =
                    make_float2(o[j][0] + o[j][2], o[j][1] + o[j][3]);
            } else {
                *reinterpret_cast<float2 *>(&wo[hrow * OSTRIDE + d0]) = make_float2(o[j][0], o[j][1]);
                *reinterpret_cast<float2 *>(&wo[(hrow + 8) * OSTRIDE + d0]) =
                    make_float2(o[j][2], o[j][3]);
            }
        }
        if (lane == 0) sm_bad[warp] = bad;
        named_barrier_sync<kConsumerWarps * 32>();

        // ---- merge the four warps; write the output or this partition's piece
        if (q_ok && !*sm_abort) {
            const int bad_any = sm_bad[0] | sm_bad[1] | sm_bad[2] | sm_bad[3];
            const size_t piece = (size_t)mt.pair * Hkv + g;
            T *out = static_cast<T *>(p.out) + ((size_t)s * p.num_q_heads + (size_t)g * G) * D;
            for (int e = ctid; e < G * D; e += kConsumerWarps * 32) {
                const int h = e / D, d = e - h * D;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w)
                    M = fmaxf(M, sm_o[(w * GROWS + h) * OSTRIDE + D]);
                float acc = 0.f, lsum = 0.f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const float *r = sm_o + (w * GROWS + h) * OSTRIDE;
                    const float f = exp2f(r[D] - M);
                    acc += r[d] * f;
                    lsum += r[D + 1] * f;
                }
                if (mt.nsplit == 1) {
                    out[h * D + d] = bad_any ? E::from_float(0.f) : E::from_float(acc / lsum);
                } else {
                    p.part_o[(piece * G + h) * D + d] = acc;
                    if (d == 0) p.part_ml[piece * G + h] = make_float2(M, bad_any ? -1.f : lsum);
                }
            }
        }
        named_barrier_sync<kConsumerWarps * 32>();
    }
}

// ---------------------------------------------------------------- merge kernel
// Sequences cut into several pieces get their pieces combined by log-sum-exp:
//   M = max_p m_p,  out = sum_p o_p 2^(m_p - M) / sum_p l_p 2^(m_p - M)
// (maxima in the log2 domain).  The kernel walks the (sequence, kv head) units
// of the split sequences grid-stride, one warp per query head of the group:
// lanes reduce M and the denominator over the pieces with a fixed shuffle tree,
// then each lane sums its D/32 dimensions over the pieces in partition order,
// with the piece loads independent of the sums so many are in flight.
// Deterministic.  A poisoned piece (sum < 0) zeroes the row.
//
// One (sequence, kv head, query head h): the sequence's partition pieces
// combined by log-sum-exp, in partition order.
template <bool BF16, int D>
__device__ __forceinline__ void merge_one(const Params &p, int s, int g, int h, int lane)
{
    using E = Elem<BF16>;
    using T = typename E::T;
    constexpr int PER_LANE = D / 32;
    const int Hkv = p.num_kv_heads, G = p.group;
    const int2 info = p.seq_info[s];
    const int n = info.y;
    const float2 *ml = p.part_ml + ((size_t)info.x * Hkv + g) * G + h;   // stride Hkv * G
    const size_t mstride = (size_t)Hkv * G;
    // one pass: each lane keeps (max, sum) of its pieces, then a fixed butterfly
    // combines the lanes' pairs with rescaling
    float M = -INFINITY, lsum = 0.f;
    int poisoned = 0;
    for (int k = lane; k < n; k += 32) {
        const float2 v = __ldg(ml + k * mstride);
        poisoned |= v.y < 0.f;
        const float Mn = fmaxf(M, v.x);
        lsum = lsum * exp2f(M - Mn) + v.y * exp2f(v.x - Mn);
        M = Mn;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float M2 = __shfl_xor_sync(kFull, M, o);
        const float l2 = __shfl_xor_sync(kFull, lsum, o);
        poisoned |= __shfl_xor_sync(kFull, poisoned, o);
        const float Mn = fmaxf(M, M2);
        const float a = M == -INFINITY ? 0.f : exp2f(M - Mn);
        const float b = M2 == -INFINITY ? 0.f : exp2f(M2 - Mn);
        lsum = lsum * a + l2 * b;
        M = Mn;
    }

    const float *po = p.part_o + (((size_t)info.x * Hkv + g) * G + h) * D + PER_LANE * lane;
    const size_t ostride = mstride * D;
    float acc[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) acc[i] = 0.f;
#pragma unroll 16
    for (int k = 0; k < n; ++k) {
        const float w = exp2f(__ldg(&ml[k * mstride].x) - M);
        if constexpr (PER_LANE == 4) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(po + k * ostride));
            acc[0] += v.x * w; acc[1] += v.y * w; acc[2] += v.z * w; acc[3] += v.w * w;
        } else {
            const float2 v = __ldg(reinterpret_cast<const float2 *>(po + k * ostride));
            acc[0] += v.x * w; acc[1] += v.y * w;
        }
    }
    T *out = static_cast<T *>(p.out) + ((size_t)s * p.num_q_heads + (size_t)g * G + h) * D +
             PER_LANE * lane;
    const float inv = 1.f / lsum;
    if constexpr (PER_LANE == 4) {
        uint2 w2;
        w2.x = poisoned ? 0u : E::pack(acc[0] * inv, acc[1] * inv);
        w2.y = poisoned ? 0u : E::pack(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2 *>(out) = w2;
    } else {
        *reinterpret_cast<uint32_t *>(out) = poisoned ? 0u : E::pack(acc[0] * inv, acc[1] * inv);
    }
}

// The sequences the prep kernel listed as split, grid-stride over (sequence,
// kv head); one warp per query head of the group.
template <bool BF16, int D>
__global__ void __launch_bounds__(512, 2) decode_merge_kernel(const Params p)
{
    const int Hkv = p.num_kv_heads, G = p.group;
    const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
    griddep_wait();                // pieces and the list come from the prep and main kernels
    if (h >= G) return;
    const int units = p.header[3] * Hkv;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int s = p.multi[u / Hkv], g = u - (u / Hkv) * Hkv;
        merge_one<BF16, D>(p, s, g, h, lane);
    }
}

// --------------------------------------------------------------------- host side
// The work plan comes first (header, per-sequence info, items, the split
// sequences and, with shared prefixes, the skips, the shared-prefix items and
// the run scratch), then the pieces.
struct WsLayout {
    size_t header, seq_info, items, multi, part_ml, part_o, total;
    size_t seq_skip, prefix_items, prefix_scratch;   // shared-prefix layouts only
    size_t plan;                                      // bytes of the plan
    int64_t max_pairs, max_prefix_items;
};

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// With `prefix`, room for shared prefixes: kPrefixMaxPieces more pieces per
// sequence, the per-sequence skips, the run scratch and the shared-prefix work
// list (at most 2.25 S items: a run has two members or more, and its items are
// ceil(members / tile) <= members / 16 + 1 tiles times at most 4 chunks).
static bool ws_layout(int64_t S, int32_t Hq, int32_t Hkv, int32_t D, int32_t maxb, int32_t P,
                      bool prefix, WsLayout *w)
{
    if (S < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || maxb <= 0 || P <= 0 || Hq % Hkv) return false;
    const int64_t G = Hq / Hkv;
    w->max_pairs = S * ((maxb + P - 1) / P + (prefix ? kPrefixMaxPieces : 0));
    w->max_prefix_items = prefix ? 3 * S : 0;
    size_t off = 0;
    w->header = off; off += 256;
    w->seq_info = off; off += align256((size_t)S * 8);
    w->items = off; off += align256((size_t)w->max_pairs * 8);
    w->multi = off; off += align256((size_t)S * 4);
    w->seq_skip = w->prefix_scratch = w->prefix_items = 0;
    if (prefix) {
        w->seq_skip = off; off += align256((size_t)S * 8);
        w->prefix_items = off; off += align256((size_t)w->max_prefix_items * 16);
        w->prefix_scratch = off; off += align256((size_t)S * 16);
    }
    w->plan = off;
    w->part_ml = off; off += align256((size_t)w->max_pairs * Hkv * G * 8);
    w->part_o = off; off += align256((size_t)w->max_pairs * Hkv * G * D * 4);
    w->total = off;
    return true;
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

// 2-D view of a pool: rows = num_blocks * Hkv * 16 of head_dim elements; box of
// 64 columns x 16 rows with the 128-byte swizzle.
static bool make_pool_map(CUtensorMap *map, const void *pool, const PoolGeometry &g)
{
    EncodeFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)g.head_dim,
                          (cuuint64_t)g.num_blocks * g.num_kv_heads * g.block_size};
    cuuint64_t strides[1] = {(cuuint64_t)g.head_dim * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBoxCols, (cuuint32_t)kBlock};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, g.dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                     2, const_cast<void *>(pool), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}


struct Variant {
    KernelFn fn;
    int smem;
    int threads;
    int items_per_cta;      // items a CTA works on at once (consumer groups)
};

template <int D, bool BF16, int GROWS, int NST, int MINB>
static Variant variant()
{
    return Variant{reinterpret_cast<KernelFn>(&decode_kernel<D, BF16, GROWS, NST, MINB>),
                   Smem<D, GROWS, NST>::kTotal, kThreads, 1};
}

static Variant q8_variant(bool bf16)
{
    const Q8KernelInfo k = q8_kernel_info(bf16);
    return Variant{k.fn, k.smem, k.threads, k.warps};
}

static bool pick_variant(int D, bool bf16, int G, Variant *v)
{
    const bool wide = G > 8;
#define PKV_PICK(DD, NST, MINB)                                                         \
    if (D == DD) {                                                                      \
        if (bf16) *v = wide ? variant<DD, true, 16, NST, MINB>() : variant<DD, true, 8, NST, MINB>(); \
        else *v = wide ? variant<DD, false, 16, NST, MINB>() : variant<DD, false, 8, NST, MINB>();   \
        return true;                                                                    \
    }
    PKV_PICK(128, 8, 2)
    PKV_PICK(64, 16, 3)
#undef PKV_PICK
    return false;
}

// Resident CTAs per SM for a variant on the current device, cached per device.
static int persistent_ctas(const Variant &v, int *num_sms_out)
{
    constexpr int kMaxDev = 64, kMaxVar = 16;
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
    *num_sms_out = sms[dev];
    for (int i = 0; i < kMaxVar; ++i) {
        if (fns[dev][i] == v.fn) return ctas[dev][i];
        if (fns[dev][i] == nullptr) {
            if (cudaFuncSetAttribute(reinterpret_cast<const void *>(v.fn),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     v.smem) != cudaSuccess)
                return -1;
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                    &n, reinterpret_cast<const void *>(v.fn), v.threads, v.smem) != cudaSuccess ||
                n < 1)
                return -1;
            fns[dev][i] = v.fn;
            ctas[dev][i] = n;
            return n;
        }
    }
    int n = 0;    // the table is full: measure without caching
    if (cudaFuncSetAttribute(reinterpret_cast<const void *>(v.fn),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, v.smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, reinterpret_cast<const void *>(v.fn),
                                                      v.threads, v.smem) != cudaSuccess)
        return -1;
    return n;
}

// 8-bit pool (k_pool = the record pool, v_pool unused) or 16-bit K and V pools.
// planned >= 0: the work plan is already at the start of the workspace (built
// by paged_decode_plan on the host), no prep kernel; `planned` is its number
// of shared-prefix items.
static int launch(const pkv_pool *pool, void *out, const void *q, const void *k_pool,
                  const void *v_pool, bool want_8bit, const int32_t *block_tables, int32_t maxb,
                  const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads, float scale,
                  int32_t P, bool auto_split, void *workspace, size_t workspace_bytes,
                  int32_t *d_status, void *stream, int32_t planned = -1)
{
    PoolGeometry g;
    if (!pool_geometry(pool, &g)) return PKV_ERR_INVALID_ARG;
    if (want_8bit ? !is_8bit(g) : !is_16bit(g)) return PKV_ERR_INVALID_ARG;
    if (num_seqs < 0 || num_q_heads <= 0 || maxb <= 0 || P <= 0) return PKV_ERR_INVALID_ARG;
    if (num_q_heads % g.num_kv_heads) return PKV_ERR_INVALID_ARG;
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return PKV_ERR_INVALID_ARG;
    const int G = num_q_heads / g.num_kv_heads;
    const bool bf = g.dtype == PKV_BF16 || g.dtype == PKV_Q8_BF16;
    if (g.block_size != kBlock || G > (want_8bit ? 8 : 16)) return PKV_ERR_UNSUPPORTED;
    Variant v;
    if (want_8bit) {
        if (g.head_dim != 128 || P > 32) return PKV_ERR_UNSUPPORTED;
        v = q8_variant(bf);
    } else if (!pick_variant(g.head_dim, bf, G, &v)) {
        return PKV_ERR_UNSUPPORTED;
    }
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_pool || (!want_8bit && !v_pool) || !block_tables || !context_lens ||
        !workspace || !d_status)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) ||
        (!want_8bit && !aligned16(v_pool)) || ((uintptr_t)workspace & 255u) ||
        ((uintptr_t)block_tables & 3u) || ((uintptr_t)context_lens & 3u) ||
        ((uintptr_t)d_status & 3u))
        return PKV_ERR_INVALID_ARG;
    // the automatic 16-bit call lays its workspace out for shared prefixes; it
    // looks for them when the ledger says some block is shared right now
    const bool prefix_layout = auto_split && !want_8bit;
    const bool prefix = planned >= 0 ? planned > 0
                                     : prefix_layout && pool_has_shared_blocks(pool) &&
                                           maxb > kPrefixMinBlocks &&
                                           prefill::shared_prefix_supported(g, G);
    WsLayout w;
    if (!ws_layout(num_seqs, num_q_heads, g.num_kv_heads, g.head_dim, maxb, P, prefix_layout, &w) ||
        workspace_bytes < w.total || planned > w.max_prefix_items)
        return PKV_ERR_INVALID_ARG;
    if ((int64_t)g.num_blocks * g.num_kv_heads * g.block_size > (int64_t)1 << 31)
        return PKV_ERR_UNSUPPORTED;   // TMA row coordinate is a signed 32-bit value

    CUtensorMap tk = {}, tv = {};     // the 8-bit kernel copies whole records, without maps
    if (!want_8bit && (!make_pool_map(&tk, k_pool, g) || !make_pool_map(&tv, v_pool, g)))
        return PKV_ERR_CUDA;

    char *ws = static_cast<char *>(workspace);
    Params prm;
    prm.out = out;
    prm.q = q;
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.num_seqs = num_seqs;
    prm.num_q_heads = num_q_heads;
    prm.num_kv_heads = g.num_kv_heads;
    prm.group = G;
    prm.max_blocks_per_seq = maxb;
    prm.blocks_per_split = P;
    prm.num_blocks = g.num_blocks;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.header = reinterpret_cast<int32_t *>(ws + w.header);
    prm.seq_info = reinterpret_cast<int2 *>(ws + w.seq_info);
    prm.items = reinterpret_cast<int2 *>(ws + w.items);
    prm.part_ml = reinterpret_cast<float2 *>(ws + w.part_ml);
    prm.part_o = reinterpret_cast<float *>(ws + w.part_o);
    prm.multi = reinterpret_cast<int32_t *>(ws + w.multi);
    prm.status = d_status;
    prm.kv_q8 = want_8bit ? static_cast<const uint8_t *>(k_pool) : nullptr;
    prm.max_pairs = w.max_pairs;
    prm.debug = prm.header + 1;
    // (a plan without shared-prefix items has zero skips: the kernels need not read them)
    prm.seq_skip = prefix ? reinterpret_cast<int2 *>(ws + w.seq_skip) : nullptr;
    prm.prefix_scratch = prefix ? reinterpret_cast<int32_t *>(ws + w.prefix_scratch) : nullptr;
    prm.prefix_items = prefix ? reinterpret_cast<int4 *>(ws + w.prefix_items) : nullptr;
    prm.max_prefix_items = (int32_t)w.max_prefix_items;
    prm.prefix_tile_seqs = prefix ? prefill::shared_prefix_tile_seqs(G) : 0;


    int num_sms = 0;
    const int per_sm = persistent_ctas(v, &num_sms);
    if (per_sm < 1) return PKV_ERR_CUDA;
    int64_t grid = (int64_t)per_sm * num_sms;
    prm.auto_split_pairs =
        auto_split ? (int32_t)((kAutoItemsPerCta * grid + g.num_kv_heads - 1) / g.num_kv_heads) : 0;
    const int64_t upper = (w.max_pairs * g.num_kv_heads + v.items_per_cta - 1) / v.items_per_cta;
    if (grid > upper) grid = upper;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
#ifdef PKV_DEBUG_CHECKS
    if (cudaMemsetAsync(prm.header + 1, 0, 4, st) != cudaSuccess) return PKV_ERR_CUDA;
#endif
    if (planned < 0) {
        decode_prep_kernel<<<1, 1024, 0, st>>>(prm, g.head_dim);
        if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    }
    if (prefix) {     // shared prefixes: their pieces, before the partitions after them
        prefill::SharedPrefixLaunch a;
        a.geometry = g;
        a.k_pool = k_pool;
        a.v_pool = v_pool;
        a.q = q;
        a.block_tables = block_tables;
        a.max_blocks_per_seq = maxb;
        a.num_seqs = num_seqs;
        a.num_q_heads = num_q_heads;
        a.scale_log2 = prm.scale_log2;
        a.items = prm.prefix_items;
        a.count = prm.header + 4;
        a.max_items = prm.max_prefix_items;
        a.piece_info = prm.seq_info;
        a.part_ml = prm.part_ml;
        a.part_o = prm.part_o;
        a.status = d_status;
        a.stream = st;
        const int rc = prefill::launch_shared_prefix(a);
        if (rc != PKV_OK) return rc;
    }
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(v.threads);
    cfg.dynamicSmemBytes = (size_t)v.smem;
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, v.fn, tk, tv, prm) != cudaSuccess) return PKV_ERR_CUDA;
    if (maxb > P || prefix) {   // some sequence may have several pieces
        // a grid-stride grid over the (sequence, kv head) units the prep kernel
        // lists: a few waves when many sequences are split, and little to
        // launch when none is
        int64_t pairs = (int64_t)num_seqs * g.num_kv_heads;
        if (pairs > (int64_t)num_sms * 8) pairs = (int64_t)num_sms * 8;
        void (*merge)(Params) =
            g.head_dim == 128 ? (bf ? decode_merge_kernel<true, 128> : decode_merge_kernel<false, 128>)
                              : (bf ? decode_merge_kernel<true, 64> : decode_merge_kernel<false, 64>);
        cudaLaunchConfig_t mcfg = {};
        mcfg.gridDim = dim3((unsigned)pairs);
        mcfg.blockDim = dim3(32u * (unsigned)G);
        mcfg.stream = st;
        mcfg.attrs = pdl;
        mcfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&mcfg, merge, prm) != cudaSuccess) return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

// ------------------------------------------------------------ host planner
// The prep kernel's work plan, built on the host from host copies of the
// context lengths and (for shared prefixes) the block tables, in the same
// layout and order: a caller that already holds them (the ledger wrote them)
// copies the plan to the workspace with its other per-step copies, and the
// call then starts with the main kernel.
static int plan_on_host(const pkv_pool *pool, const int32_t *lens, const int32_t *tables,
                        int32_t maxb, int32_t S, int32_t Hq, void *plan, size_t plan_bytes,
                        int32_t *prefix_items_out)
{
    PoolGeometry g;
    if (!pool_geometry(pool, &g) || !is_16bit(g) || !lens || !plan || S < 0 || Hq <= 0 ||
        maxb <= 0 || Hq % g.num_kv_heads)
        return PKV_ERR_INVALID_ARG;
    const int G = Hq / g.num_kv_heads, Hkv = g.num_kv_heads;
    const bool bf = g.dtype == PKV_BF16;
    Variant v;
    if (g.block_size != kBlock || G > 16 || !pick_variant(g.head_dim, bf, G, &v))
        return PKV_ERR_UNSUPPORTED;
    WsLayout w;
    if (!ws_layout(S, Hq, Hkv, g.head_dim, maxb, kDefaultSplit, true, &w) || plan_bytes < w.plan)
        return PKV_ERR_INVALID_ARG;
    const int64_t max_tokens = (int64_t)maxb * kBlock;
    for (int32_t s = 0; s < S; ++s)
        if (lens[s] < 0 || lens[s] > max_tokens) return PKV_ERR_INVALID_ARG;
    char *base = static_cast<char *>(plan);
    std::memset(base + w.header, 0, 256);                  // every other word is written below
    std::memset(base + w.seq_skip, 0, (size_t)S * 8);     // zero outside shared-prefix runs
    int32_t *header = reinterpret_cast<int32_t *>(base + w.header);
    int2 *seq_info = reinterpret_cast<int2 *>(base + w.seq_info);
    int2 *items = reinterpret_cast<int2 *>(base + w.items);
    int32_t *multi = reinterpret_cast<int32_t *>(base + w.multi);
    int2 *seq_skip = reinterpret_cast<int2 *>(base + w.seq_skip);
    int4 *pitems = reinterpret_cast<int4 *>(base + w.prefix_items);
    auto nblocks = [](int32_t L) { return (L + kBlock - 1) / kBlock; };

    // shared prefixes: links between neighbours, runs, the shortest link of each
    int32_t n_pitems = 0;
    if (tables && pool_has_shared_blocks(pool) && maxb > kPrefixMinBlocks &&
        prefill::shared_prefix_supported(g, G)) {
        std::vector<int32_t> link((size_t)S, 0);
        for (int32_t s = 0; s + 1 < S; ++s) {
            const int32_t La = lens[s], Lb = lens[s + 1];
            if (La <= 0 || Lb <= 0) continue;
            const int32_t f = std::min((La - 1) / kBlock, (Lb - 1) / kBlock);
            const int32_t *ra = tables + (int64_t)s * maxb, *rb = ra + maxb;
            int32_t k = 0;
            while (k < f && ra[k] == rb[k] && ra[k] >= 0 && ra[k] < g.num_blocks) ++k;
            link[(size_t)s] = k;
        }
        const int tt = prefill::shared_prefix_tile_seqs(G);
        for (int32_t s = 0; s < S;) {
            int32_t e = s;   // run [s, e]
            int32_t pb = 0x7fffffff;
            while (e + 1 < S && link[(size_t)e] >= kPrefixMinBlocks) pb = std::min(pb, link[(size_t)e++]);
            const int32_t n = e - s + 1;
            if (n >= 2) {
                const int pieces = std::min(kPrefixMaxPieces, (pb + kPrefixMinBlocks - 1) / kPrefixMinBlocks);
                const int cb = (pb + pieces - 1) / pieces;
                for (int32_t m = s; m <= e; ++m) seq_skip[m] = make_int2(pb, pieces);
                for (int t = 0; t * tt < n; ++t)
                    for (int j = 0; j < pieces; ++j) {
                        if (n_pitems >= w.max_prefix_items) return PKV_ERR_INVALID_ARG;
                        pitems[n_pitems++] = make_int4(s + t * tt, std::min(tt, n - t * tt) | (j << 16),
                                                       j * cb, std::min(pb, (j + 1) * cb));
                    }
            }
            s = e + 1;
        }
    }
    auto own = [&](int32_t s) {
        return make_int2(nblocks(lens[s]) - seq_skip[s].x, seq_skip[s].y);
    };
    // partition size: as the prep kernel chooses it
    int num_sms = 0;
    const int per_sm = persistent_ctas(v, &num_sms);
    if (per_sm < 1) return PKV_ERR_CUDA;
    const int64_t grid = (int64_t)per_sm * num_sms;
    const int64_t want = (kAutoItemsPerCta * grid + Hkv - 1) / Hkv;
    int P = kDefaultSplit;
    for (int k = 1; k < kAutoSizes; ++k) {
        const int Pk = kDefaultSplit << k;
        int64_t pairs = 0;
        for (int32_t s = 0; s < S; ++s)
            if (lens[s] > 0) pairs += (own(s).x + Pk - 1) / Pk;
        if (pairs >= want) P = Pk;
    }
    // pieces, full partitions in sequence order, partial ones by size bin
    int32_t piece = 0, n_items = 0, n_multi = 0;
    std::vector<int32_t> bin_count(kOrderBins, 0);
    auto bin_of = [P](int r) { return (int)((int64_t)(P - 1 - r) * kOrderBins / P); };
    for (int32_t s = 0; s < S; ++s) {
        int nsplit = 0, npre = 0;
        if (lens[s] > 0) {
            const int2 o = own(s);
            npre = o.y;
            nsplit = (o.x + P - 1) / P;
            const int r = o.x - (nsplit - 1) * P;
            const int full = r < P ? nsplit - 1 : nsplit;
            for (int k = 0; k < full; ++k) items[n_items++] = make_int2(s, k);
            if (r < P) ++bin_count[(size_t)bin_of(r)];
        }
        seq_info[s] = make_int2(piece, npre + nsplit);
        piece += npre + nsplit;
        if (npre + nsplit > 1) multi[n_multi++] = s;
    }
    std::vector<int32_t> bin_at(kOrderBins, 0);
    for (int b = 0, at = n_items; b < kOrderBins; ++b) {
        bin_at[(size_t)b] = at;
        at += bin_count[(size_t)b];
    }
    for (int32_t s = 0; s < S; ++s) {
        if (lens[s] <= 0) continue;
        const int2 o = own(s);
        const int nsplit = (o.x + P - 1) / P;
        const int r = o.x - (nsplit - 1) * P;
        if (r < P) {
            items[bin_at[(size_t)bin_of(r)]++] = make_int2(s, nsplit - 1);
            ++n_items;
        }
    }
    if (piece > w.max_pairs) return PKV_ERR_INVALID_ARG;
    header[0] = n_items;
    header[2] = P;
    header[3] = n_multi;
    header[4] = n_pitems;
    header[5] = piece;
    if (prefix_items_out) *prefix_items_out = n_pitems;
    return PKV_OK;
}

}  // namespace decode
}  // namespace pkv

extern "C" {

int32_t paged_decode_default_split(void) { return pkv::decode::kDefaultSplit; }

size_t paged_decode_plan_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_dim, int32_t max_blocks_per_seq)
{
    pkv::decode::WsLayout w;
    if (!pkv::decode::ws_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                pkv::decode::kDefaultSplit, true, &w))
        return 0;
    return w.plan;
}

int paged_decode_plan(const pkv_pool *pool, const int32_t *context_lens,
                      const int32_t *block_tables, int32_t max_blocks_per_seq, int32_t num_seqs,
                      int32_t num_q_heads, void *plan, size_t plan_bytes,
                      int32_t *shared_prefix_items)
{
    return pkv::decode::plan_on_host(pool, context_lens, block_tables, max_blocks_per_seq,
                                     num_seqs, num_q_heads, plan, plan_bytes, shared_prefix_items);
}

int paged_decode_attention_planned(const pkv_pool *pool, void *out, const void *q,
                                   const void *k_pool, const void *v_pool,
                                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *context_lens, int32_t num_seqs,
                                   int32_t num_q_heads, float scale, int32_t shared_prefix_items,
                                   void *workspace, size_t workspace_bytes, int32_t *d_status,
                                   void *stream)
{
    if (shared_prefix_items < 0) return PKV_ERR_INVALID_ARG;
    return pkv::decode::launch(pool, out, q, k_pool, v_pool, false, block_tables,
                               max_blocks_per_seq, context_lens, num_seqs, num_q_heads, scale,
                               pkv::decode::kDefaultSplit, true, workspace, workspace_bytes,
                               d_status, stream, shared_prefix_items);
}

size_t paged_decode_workspace_bytes_split(int32_t num_seqs, int32_t num_q_heads,
                                          int32_t num_kv_heads, int32_t head_dim,
                                          int32_t max_blocks_per_seq, int32_t blocks_per_split)
{
    pkv::decode::WsLayout w;
    if (!pkv::decode::ws_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                blocks_per_split, false, &w))
        return 0;
    return w.total;
}

size_t paged_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t max_blocks_per_seq)
{
    pkv::decode::WsLayout w;
    if (!pkv::decode::ws_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                pkv::decode::kDefaultSplit, true, &w))
        return 0;
    return w.total;
}

int paged_decode_attention_split(const pkv_pool *pool, void *out, const void *q,
                                 const void *k_pool, const void *v_pool,
                                 const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 const int32_t *context_lens, int32_t num_seqs,
                                 int32_t num_q_heads, float scale, int32_t blocks_per_split,
                                 void *workspace, size_t workspace_bytes, int32_t *d_status,
                                 void *stream)
{
    return pkv::decode::launch(pool, out, q, k_pool, v_pool, false, block_tables,
                               max_blocks_per_seq, context_lens, num_seqs, num_q_heads, scale,
                               blocks_per_split, false, workspace, workspace_bytes, d_status,
                               stream);
}

int paged_decode_attention(const pkv_pool *pool, void *out, const void *q, const void *k_pool,
                           const void *v_pool, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *context_lens,
                           int32_t num_seqs, int32_t num_q_heads, float scale, void *workspace,
                           size_t workspace_bytes, int32_t *d_status, void *stream)
{
    return pkv::decode::launch(pool, out, q, k_pool, v_pool, false, block_tables,
                               max_blocks_per_seq, context_lens, num_seqs, num_q_heads, scale,
                               pkv::decode::kDefaultSplit, true, workspace, workspace_bytes,
                               d_status, stream);
}

int paged_decode_attention_q8(const pkv_pool *pool, void *out, const void *q, const void *kv_q8,
                              const int32_t *block_tables, int32_t max_blocks_per_seq,
                              const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                              float scale, void *workspace, size_t workspace_bytes,
                              int32_t *d_status, void *stream)
{
    return pkv::decode::launch(pool, out, q, kv_q8, nullptr, true, block_tables,
                               max_blocks_per_seq, context_lens, num_seqs, num_q_heads, scale,
                               pkv::decode::kDefaultSplit, false, workspace, workspace_bytes,
                               d_status, stream);
}

}  // extern "C"

// ------------------------------------------------------- fixed-scratch variant
// paged_decode_attention_noalloc runs the same kernels as paged_decode_attention
// but keeps their scratch (work list and split-K pieces) in a fixed array that
// belongs to this library, so the caller passes no workspace and nothing is
// allocated at call time.  The array lives in global memory of every device
// that loads the library, from module load until the process exits.
namespace pkv {
namespace decode {

constexpr size_t kNoallocScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch on the current device.  In host code the
// symbol only names a host-side stand-in, so the address is looked up once per
// device (with that device current) and cached; NULL if the lookup fails.
static void *noalloc_scratch_address()
{
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    static void *addr[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace decode
}  // namespace pkv

extern "C" int paged_decode_attention_noalloc(const pkv_pool *pool, void *out, const void *q,
                                              const void *k_pool, const void *v_pool,
                                              const int32_t *block_tables,
                                              int32_t max_blocks_per_seq,
                                              const int32_t *context_lens, int32_t num_seqs,
                                              int32_t num_q_heads, float scale,
                                              int32_t *d_status, void *stream)
{
    using namespace pkv::decode;
    pkv::PoolGeometry g;
    if (!pkv::pool_geometry(pool, &g) || num_seqs < 0 || num_q_heads <= 0 ||
        max_blocks_per_seq <= 0)
        return PKV_ERR_INVALID_ARG;
    // The default partition size if its scratch fits; otherwise the smallest
    // partition count per sequence that fits, down to one partition.
    const int32_t maxb = max_blocks_per_seq;
    int32_t P = 0;
    for (int32_t k = (maxb + kDefaultSplit - 1) / kDefaultSplit; k >= 1; --k) {
        const int32_t cand = (maxb + k - 1) / k;
        WsLayout w;
        if (!ws_layout(num_seqs, num_q_heads, g.num_kv_heads, g.head_dim, maxb, cand, false, &w))
            return PKV_ERR_INVALID_ARG;
        if (w.total <= kNoallocScratchBytes) {
            P = cand;
            break;
        }
    }
    if (P == 0) return PKV_ERR_INVALID_ARG;   // scratch would exceed PKV_NOALLOC_SCRATCH_BYTES
    void *scratch = noalloc_scratch_address();
    if (!scratch) return PKV_ERR_CUDA;
    return launch(pool, out, q, k_pool, v_pool, false, block_tables, maxb, context_lens,
                  num_seqs, num_q_heads, scale, P, false, scratch, kNoallocScratchBytes, d_status,
                  stream);
}
