// Parameters shared by the decode kernels of libpagedkv.so (16-bit kernel,
// 8-bit kernel, their prep and merge kernels).  Internal to the library.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <vector_types.h>

#include "pkv_internal.h"

namespace pkv {
namespace decode {

constexpr int kDefaultSplit = 32;        // blocks per partition (512 tokens)

// Shared prefixes: two neighbouring sequences are linked when their tables
// agree on at least kPrefixMinBlocks leading blocks; a run of linked sequences
// reads the shortest link of the run once.  Its blocks go out in
// min(kPrefixMaxPieces, ceil(blocks / kPrefixMinBlocks)) key chunks of equal
// size (to a block), one piece per member and chunk.
constexpr int kPrefixMinBlocks = 16;
constexpr int kPrefixMaxPieces = 4;

struct Params {
    void *out;
    const void *q;
    const int32_t *block_tables;
    const int32_t *context_lens;
    int32_t num_seqs, num_q_heads, num_kv_heads, group, max_blocks_per_seq;
    int32_t blocks_per_split;   // fixed size, or the smallest candidate (automatic)
    int32_t num_blocks;
    int32_t auto_split_pairs;   // > 0: the prep kernel picks the size (header[2])
    float scale_log2;           // softmax scale * log2(e): scores live in the exp2 domain
    int32_t *header;            // [0] decode items, [1] debug word, [2] blocks per partition,
                                // [3] sequences with more than one piece,
                                // [4] shared-prefix items, [5] pieces
    int32_t *multi;             // [S]: those sequences (any order)
    int2 *seq_info;             // [S]: first piece index, number of pieces
    int2 *items;                // [S * ceil(maxb / P)]: (sequence, partition)
    // Shared prefixes (null when the call does not look for them): runs of
    // consecutive sequences whose tables begin with the same blocks read those
    // blocks once, in the shared-prefix kernel; their decode partitions cover
    // the blocks after the prefix.
    int2 *seq_skip;             // [S]: (prefix blocks, prefix pieces), (0, 0) outside a run
    int32_t *prefix_scratch;    // [4][S]: link lengths, run starts, run minima, member counts
    int4 *prefix_items;         // (first member, members | chunk << 16, first block, end block)
    int32_t max_prefix_items;
    int32_t prefix_tile_seqs;   // members per shared-prefix item
    float2 *part_ml;            // [pairs * Hkv * G]: (max, sum) of a partition; sum < 0 = poisoned
    float *part_o;              // [pairs * Hkv * G * D]: unnormalised partition output
    int32_t *status;
    const uint8_t *kv_q8;       // 8-bit pool: one record of kQ8Slab bytes per (block, kv head)
    int64_t max_pairs;          // capacity of items / partial arrays (checked builds)
    int32_t *debug;             // first failed check: site << 24 | value (checked builds)
};

using KernelFn = void (*)(CUtensorMap, CUtensorMap, Params);

}  // namespace decode

namespace prefill {
// The shared-prefix kernel (the tcgen05 kernel of paged_prefill.cu in its
// shared-prefix mode) as the decode launcher sees it.
struct SharedPrefixLaunch {
    PoolGeometry geometry;
    const void *k_pool, *v_pool, *q;
    const int32_t *block_tables;
    int32_t max_blocks_per_seq, num_seqs, num_q_heads;
    float scale_log2;
    const int4 *items;           // written by the decode prep kernel
    const int32_t *count;        // number of items (decode header[4])
    int32_t max_items;
    const int2 *piece_info;      // decode seq_info
    float2 *part_ml;
    float *part_o;
    int32_t *status;
    cudaStream_t stream;
};
int shared_prefix_tile_seqs(int G);
bool shared_prefix_supported(const PoolGeometry &g, int G);
int launch_shared_prefix(const SharedPrefixLaunch &a);
}  // namespace prefill

namespace decode {

// The 8-bit decode kernel (paged_decode_q8.cu) as the launcher sees it.
struct Q8KernelInfo {
    KernelFn fn;
    int smem;          // dynamic shared memory per CTA
    int threads;       // threads per CTA
    int warps;         // items a CTA works on at once (one per warp)
};
Q8KernelInfo q8_kernel_info(bool bf16_queries);

#ifdef __CUDACC__
// Output rows of sequences with no context, or with a length the table cannot
// hold, are zeros.  context_lens is an input of the call, not something the
// prep kernel writes, so each main kernel's CTAs store these rows before they
// wait for the prep kernel's work list, while it still runs (grid-stride over
// sequences, the CTA's threads over the row's 16-byte pieces).  Not inlined,
// so it leaves the main loop's register allocation alone; its arguments are
// values, so no copy of the kernel's parameters is taken.
static __device__ __noinline__ void zero_idle_rows(void *out, const int32_t *context_lens,
                                                   int num_seqs, int row_bytes, int64_t max_tokens)
{
    const int n16 = row_bytes / 16;
    for (int s = blockIdx.x; s < num_seqs; s += gridDim.x) {
        const int L = __ldg(context_lens + s);
        if (L > 0 && (int64_t)L <= max_tokens) continue;
        uint4 *o = reinterpret_cast<uint4 *>(static_cast<char *>(out) + (size_t)s * row_bytes);
        for (int i = threadIdx.x; i < n16; i += blockDim.x) o[i] = make_uint4(0u, 0u, 0u, 0u);
    }
}
#endif

}  // namespace decode
}  // namespace pkv
