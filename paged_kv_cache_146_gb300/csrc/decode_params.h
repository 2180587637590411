// Parameters shared by the decode kernels of libpagedkv.so (16-bit kernel,
// 8-bit kernel, their prep and merge kernels).  Internal to the library.
#pragma once
#include <cuda.h>
#include <stdint.h>
#include <vector_types.h>

namespace pkv {
namespace decode {

constexpr int kDefaultSplit = 32;        // blocks per partition (512 tokens)

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
    int32_t *header;            // [0] pairs, [1] debug word, [2] blocks per partition,
                                // [3] sequences with more than one partition
    int32_t *multi;             // [S]: those sequences (any order)
    int2 *seq_info;             // [S]: first pair index, number of partitions
    int2 *items;                // [S * ceil(maxb / P)]: (sequence, partition)
    float2 *part_ml;            // [pairs * Hkv * G]: (max, sum) of a partition; sum < 0 = poisoned
    float *part_o;              // [pairs * Hkv * G * D]: unnormalised partition output
    int32_t *status;
    const uint8_t *kv_q8;       // 8-bit pool: one record of kQ8Slab bytes per (block, kv head)
    int64_t max_pairs;          // capacity of items / partial arrays (checked builds)
    int32_t *debug;             // first failed check: site << 24 | value (checked builds)
};

using KernelFn = void (*)(CUtensorMap, CUtensorMap, Params);

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
