/*
 * pagedkv.h -- C ABI of libpagedkv.so: a paged KV cache and its decode step
 * (host block ledger, cache-write kernel, paged decode attention) for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation, as the source pages state it:
 *   - "vLLM의 핵심 원리 PagedAttention 파헤치기" (donmain.dev), section
 *     "KV Cache를 블록으로 쪼개다": the KV cache is cut into fixed blocks of 16
 *     tokens; each sequence owns a block table mapping its logical blocks to
 *     physical blocks anywhere in a pool; blocks are taken one at a time as the
 *     sequence grows; attention gathers a sequence's blocks through its table.
 *   - "LLM 추론 배칭 전략 정리" (velog.io), section 5 ("누가 배치를 다시
 *     짜는가", "한 스텝의 전체 흐름", "왜 이게 가능한가"): the ledger of who
 *     owns which block lives on the CPU and reaches the GPU each step as a
 *     block table; the pool is one region reserved up front, a physical block
 *     is a block number inside it.
 *   - "vLLM-and-PagedAttention-KR" (ghkdgus29.github.io), sections
 *     "가장 기본적인 decoding" and "Parallel Sampling decoding": a new token's
 *     K/V goes after the tokens already in its logical block; blocks shared by
 *     several sequences carry a reference count; a finished request releases
 *     its blocks.
 *
 * Conventions the pages leave open (the library's readings):
 *   R1  K and V pools are separate arrays laid out
 *       [num_blocks][num_kv_heads][block_size][head_dim], fp16 or bf16;
 *       one (block, kv head) slab is contiguous.
 *   R2  slot = physical_block * block_size + offset_in_block (int64);
 *       a negative slot means "no token here" and is skipped.
 *   R3  query head h reads kv head h / (num_q_heads / num_kv_heads).
 *   R4  a decode step writes this step's K/V first, then attends;
 *       context_lens include the token just written.
 *   R6  q and out are [num_seqs][num_q_heads][head_dim] in the pool's dtype;
 *       block_tables is int32 [num_seqs][max_blocks_per_seq] (row-major);
 *       context_lens is int32 [num_seqs].
 *   R7  context_len == 0 yields an all-zero output row.
 *
 * Ownership: the caller owns every device buffer (pools, q, out, tables,
 * slot mapping, workspace, status word).  The library never allocates device
 * memory.  A pkv_pool owns host memory only (free stack and refcounts).
 *
 * Errors: every call returns a pkv_status.  Kernel launches are asynchronous
 * on the given stream (a cudaStream_t passed as void*, NULL = legacy default
 * stream); their arguments are validated on the host before launch, and
 * nothing is launched when validation fails.  Range errors inside device
 * data (a slot or block id outside the pool, a context length longer than its
 * table row) are recorded with atomicOr in the caller's device status word;
 * the offending token is skipped or the offending sequence's output row is
 * written as zeros, and no kernel ever traps.  kv_status_check() reads and
 * clears that word.  A pkv_pool is not thread-safe.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of a pool.  PKV_F16 / PKV_BF16: K and V stored as is.
 * PKV_Q8_BF16 / PKV_Q8_F16: 8-bit cache (one fp16 scale per 32 values; q and
 * out in bf16 / fp16), see kv_cache_write_q8. */
typedef enum pkv_dtype { PKV_F16 = 0, PKV_BF16 = 1, PKV_Q8_BF16 = 2, PKV_Q8_F16 = 3 } pkv_dtype;

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = -1,    /* bad pointer, size, shape or alignment          */
    PKV_ERR_OUT_OF_BLOCKS = -2,  /* the free pool cannot cover the request         */
    PKV_ERR_BAD_BLOCK = -3,      /* unknown id, double free, refcount underflow    */
    PKV_ERR_CUDA = -4,           /* a CUDA runtime call failed                     */
    PKV_ERR_DEVICE_BOUNDS = -5,  /* device status word reports a range error       */
    PKV_ERR_DEVICE_TIMEOUT = -6, /* a kernel gave up waiting (status word bit)     */
    PKV_ERR_SHARED_BLOCK = -7,   /* append would write into a block shared by others */
    PKV_ERR_UNSUPPORTED = -8     /* shape the kernels do not implement             */
} pkv_status;

/* Bits of the device status word (int32, caller-allocated, zero before use). */
#define PKV_DEV_BAD_SLOT  0x1   /* cache write: slot >= num_blocks * block_size     */
#define PKV_DEV_BAD_BLOCK 0x2   /* attention: table entry outside [0, num_blocks)   */
#define PKV_DEV_BAD_LEN   0x4   /* attention: context_len < 0 or longer than table  */
#define PKV_DEV_TIMEOUT   0x8   /* a bounded wait inside a kernel ran out           */

typedef struct pkv_pool pkv_pool;

/* Library version (major * 10000 + minor * 100 + patch). */
int pkv_version(void);

/* Static, human-readable name of a pkv_status value. */
const char *pkv_status_string(int status);

/* ------------------------------------------------------------------ sizing */

/* Bytes of KV cache per token: 2 (K and V) x kv_heads x head_dim x elem_bytes
 * per layer, times layers.  "vLLM-and-PagedAttention-KR", section
 * "KV Cache Size 계산 방법" (2 x H x L x B = 819,200 bytes for OPT-13B);
 * "kv-cache-by-model" (sotaaz.com), section 1.  Returns -1 on a negative
 * argument. */
int64_t kv_bytes_per_token(int32_t layers, int32_t kv_heads, int32_t head_dim,
                           int32_t elem_bytes);

/* Blocks a sequence of num_tokens tokens owns: ceil(num_tokens / block_size)
 * ("PagedAttention 파헤치기", section "낭비가 4% 밑으로": 100 tokens -> 7
 * blocks).  Returns -1 on a bad argument. */
int64_t kv_blocks_for_tokens(int64_t num_tokens, int32_t block_size);

/* Bytes of ONE of the K or V pools under layout R1. 0 on a bad argument. */
size_t kv_pool_bytes(int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                     int32_t head_dim, pkv_dtype dtype);

/* --------------------------------------------------------- host block ledger */

/* Create the ledger of a pool of num_blocks blocks.  initial_free_order, if not
 * NULL, is a permutation of 0..num_blocks-1 giving the order in which free
 * blocks are handed out (NULL = 0, 1, 2, ...).  Free blocks form a LIFO stack:
 * the pages allow any free block ("KV Cache를 블록으로 쪼개다"); this policy
 * makes ids reproducible.  A released block is the next one handed out.
 * num_kv_heads, head_dim and dtype describe the device pools the caller pairs
 * with this ledger; the kernels take the geometry from here.
 * Errors: PKV_ERR_INVALID_ARG (non-positive sizes, unknown dtype, order not a
 * permutation, out == NULL). */
int kv_pool_create(int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                   int32_t head_dim, pkv_dtype dtype, const int32_t *initial_free_order,
                   pkv_pool **out);

/* Free the ledger (host memory only).  NULL is accepted. */
int kv_pool_destroy(pkv_pool *pool);

/* Geometry of a pool; any output pointer may be NULL. */
int kv_pool_info(const pkv_pool *pool, int32_t *num_blocks, int32_t *block_size,
                 int32_t *num_kv_heads, int32_t *head_dim, int32_t *dtype);

/* Take n free blocks (all or nothing), each with refcount 1, into out_ids[n].
 * Errors: PKV_ERR_OUT_OF_BLOCKS (nothing taken), PKV_ERR_INVALID_ARG. */
int kv_block_alloc(pkv_pool *pool, int32_t n, int32_t *out_ids);

/* Add one reference to each listed block (a sequence starts sharing it:
 * "Parallel Sampling decoding").  All or nothing.
 * Errors: PKV_ERR_BAD_BLOCK if any id is not currently allocated. */
int kv_block_ref(pkv_pool *pool, int32_t n, const int32_t *ids);

/* Drop one reference from each listed block, in order; a block whose count
 * reaches 0 returns to the top of the free stack ("가장 기본적인 decoding",
 * step 5).  An id may appear several times.  All or nothing.
 * Errors: PKV_ERR_BAD_BLOCK if any id would be released more often than it is
 * referenced (double free, unknown id); nothing changes then. */
int kv_block_free(pkv_pool *pool, int32_t n, const int32_t *ids);

/* Current reference count of one block (0 = free). */
int kv_block_refcount(const pkv_pool *pool, int32_t id, int32_t *out);

/* Number of free blocks. */
int kv_pool_num_free(const pkv_pool *pool, int32_t *out);

/* Number of blocks currently referenced by two or more sequences ("vLLM의 핵심
 * 원리 PagedAttention 파헤치기", section "같은 블록을 여러 요청이 나눠 쓴다":
 * requests with a common prompt point their tables at the same physical
 * blocks).  paged_decode_attention reads it to decide whether to look for
 * shared table prefixes in the batch. */
int kv_pool_num_shared(const pkv_pool *pool, int64_t *out);

/* ------------------------------------------- on-demand allocation + slots */

/* Grow num_seqs sequences: sequence s holds seq_lens[s] tokens and gains
 * num_new[s] more.  The token at position n needs logical block n / block_size;
 * when n is a multiple of block_size that block does not exist yet and one
 * free block is taken into block_tables[s][n / block_size] ("KV Cache를 블록으로
 * 쪼개다": first token -> first block, token 17 -> a second block).  For every
 * new token, in sequence order, slot_mapping receives
 * block_tables[s][n / block_size] * block_size + n % block_size  (R2).
 *   seq_lens, num_new   host int32 [num_seqs]
 *   block_tables        host int32 [num_seqs][max_blocks_per_seq], updated
 *   slot_mapping        host int64 [sum(num_new)], written
 * All or nothing: on any error nothing changes.
 * Errors: PKV_ERR_INVALID_ARG (negative length, row too short),
 * PKV_ERR_OUT_OF_BLOCKS, PKV_ERR_BAD_BLOCK (a partly filled tail block that is
 * not allocated), PKV_ERR_SHARED_BLOCK (a partly filled tail block with
 * refcount > 1: the write needs a copy first). */
int kv_append_slots(pkv_pool *pool, int32_t num_seqs, const int32_t *seq_lens,
                    const int32_t *num_new, int32_t *block_tables,
                    int32_t max_blocks_per_seq, int64_t *slot_mapping);

/* --------------------------------------------- sharing and copy-on-write */

/* A child sequence starts sharing every block of its parent ("vLLM-and-
 * PagedAttention-KR", "Parallel Sampling decoding": the samples of one prompt
 * share its blocks, each block's reference count equals its sharers).  The
 * first ceil(parent_len / block_size) entries of parent_row are copied into
 * child_row and gain one reference each; the rest of child_row (up to
 * max_blocks_per_seq entries) is set to -1.  Host arrays.  All or nothing.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_BAD_BLOCK (an entry is not allocated). */
int kv_seq_fork(pkv_pool *pool, const int32_t *parent_row, int32_t parent_len,
                int32_t *child_row, int32_t max_blocks_per_seq);

/* kv_append_slots with copy-on-write ("Parallel Sampling decoding": when the
 * samples write different tokens into a shared block, that block is copied and
 * its reference count drops; "PagedAttention 파헤치기", "같은 블록을 여러 요청이
 * 나눠 쓴다").  Sequences are handled in order; a sequence whose partly filled
 * tail block is still referenced by others takes a fresh block for it, records
 * the pair (copy_src[i] = shared, copy_dst[i] = fresh), points its table at the
 * fresh block and drops one reference from the shared one; the last remaining
 * user of a block writes in place.  Then blocks are taken and slots written as
 * in kv_append_slots.  copy_src / copy_dst: host int32 [num_seqs] capacity;
 * *num_copies receives the count.  The caller runs kv_block_copy on the pairs
 * before writing the new tokens' K/V.  All or nothing.
 * Errors: as kv_append_slots (no PKV_ERR_SHARED_BLOCK). */
int kv_append_slots_cow(pkv_pool *pool, int32_t num_seqs, const int32_t *seq_lens,
                        const int32_t *num_new, int32_t *block_tables,
                        int32_t max_blocks_per_seq, int64_t *slot_mapping, int32_t *copy_src,
                        int32_t *copy_dst, int32_t *num_copies);

/* Device copy of n whole blocks: K and V of block dst_ids[i] become those of
 * block src_ids[i] (all kv heads and slots, bit for bit).  src_ids / dst_ids:
 * device int32 [n]; destinations must differ from each other and from every
 * source (kv_append_slots_cow guarantees it: they are fresh blocks).  A pair
 * naming a block outside the pool is skipped and sets PKV_DEV_BAD_BLOCK.
 * 8-bit pools: k_pool is the record pool, v_pool is ignored (may be NULL); a
 * block is its num_kv_heads records.
 * Asynchronous on stream.  Errors: PKV_ERR_INVALID_ARG, PKV_ERR_CUDA. */
int kv_block_copy(const pkv_pool *pool, const int32_t *src_ids, const int32_t *dst_ids,
                  int32_t n, void *k_pool, void *v_pool, int32_t *d_status, void *stream);

/* --------------------------------------------------------------- 8-bit cache */

/* An 8-bit cache stores each token's K and V as one-byte codes with one fp16
 * scale per group of 32 values: 34 bytes per 32 values, 53.1 % of fp16
 * ("kv-cache-by-model", section 1: Qwen3-8B at 32K, 4,608 -> 2,448 MiB).
 * Quantisation (a reading; the pages give only the group size and the size):
 * scale = fp16(min(max|x| / 127, 65504)); code = clamp(round-half-even(x /
 * scale), -127, 127) computed in fp32 (codes 0 when the scale is 0); the
 * cached value is code * scale.
 *
 * Pool layout (head_dim 128, block_size 16): one record of
 * PKV_Q8_SLAB_BYTES bytes per (block, kv head), records in the order
 * [num_blocks][num_kv_heads], so a block's slab is one contiguous copy.  A
 * code c is stored as the byte c + 128 (c XOR 0x80):
 *   bytes [0, 2048)     K codes: 16 rows of 128 bytes.  Token t = 4a + 2b + c
 *                       (a in 0..3, b and c in 0..1) is row r = 8b + 2a + c; its
 *                       16-byte chunk j (dimensions 16j .. 16j + 15) is stored
 *                       at byte 128 r + 16 (j XOR (r mod 8)).
 *   bytes [2048, 4096)  V codes: dimension d's 16 tokens at 2048 + 16 d + t.
 *   bytes [4096, 4224)  K scales: fp16, token t's group i at 4096 + 8 t + 2 i.
 *   bytes [4224, 4352)  V scales: fp16, token t's group i at 4224 + 32 i + 2 t.
 * kv_pool_bytes with PKV_Q8_BF16 / PKV_Q8_F16 gives the size of the pool. */
#define PKV_Q8_SLAB_BYTES 4352

/* Quantising cache write: k_new / v_new are bf16 (PKV_Q8_BF16) or fp16
 * (PKV_Q8_F16) rows [num_tokens][Hkv][128], 16-byte aligned; slots as in
 * kv_cache_write; kv_q8 is the pool (16-byte aligned).  Codes and scales are
 * those of the rule above, bit for bit, for every finite or infinite input;
 * a NaN input value stores an unspecified code (its group's scale ignores it).
 * Errors: PKV_ERR_INVALID_ARG (not an 8-bit pool, alignment),
 * PKV_ERR_UNSUPPORTED (head_dim other than 128 or block_size other than 16),
 * PKV_ERR_CUDA.  Slots outside the pool: PKV_DEV_BAD_SLOT. */
int kv_cache_write_q8(const pkv_pool *pool, const void *k_new, const void *v_new,
                      const int64_t *slot_mapping, int32_t num_tokens, void *kv_q8,
                      int32_t *d_status, void *stream);

/* Paged decode attention over an 8-bit cache: the result of
 * paged_decode_attention with K and V taken as code * scale.  q and out in the
 * pool's query type (bf16 for PKV_Q8_BF16, fp16 for PKV_Q8_F16); workspace as
 * paged_decode_workspace_bytes(...); head_dim 128, G <= 8 (PKV_ERR_UNSUPPORTED
 * otherwise).  Errors as paged_decode_attention. */
int paged_decode_attention_q8(const pkv_pool *pool, void *out, const void *q, const void *kv_q8,
                              const int32_t *block_tables, int32_t max_blocks_per_seq,
                              const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                              float scale, void *workspace, size_t workspace_bytes,
                              int32_t *d_status, void *stream);

/* -------------------------------------------------------------- swap to host */

/* Swapping ("vLLM-and-PagedAttention-KR", "Scheduling": when blocks run out, a
 * whole sequence -- the latest arrival -- is evicted and its KV blocks move to
 * CPU memory; they come back when space frees up).  The device side packs the
 * blocks into one contiguous staging buffer so the host copy is a single
 * transfer, and unpacks a staging buffer into (other) blocks on the way back.
 * staging layout: [n][2 (K, V)][num_kv_heads][block_size][head_dim], pool dtype,
 * device memory, 16-byte aligned, 2 * n * block bytes.  8-bit pools: k_pool is
 * the record pool, v_pool is ignored (may be NULL), staging is
 * [n][num_kv_heads][PKV_Q8_SLAB_BYTES] bytes.  ids: device int32 [n].
 * Ids outside the pool are skipped and set PKV_DEV_BAD_BLOCK.  Asynchronous.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_CUDA. */
int kv_gather_blocks(const pkv_pool *pool, const int32_t *ids, int32_t n, const void *k_pool,
                     const void *v_pool, void *staging, int32_t *d_status, void *stream);
int kv_scatter_blocks(const pkv_pool *pool, const int32_t *ids, int32_t n, const void *staging,
                      void *k_pool, void *v_pool, int32_t *d_status, void *stream);

/* --------------------------------------------------------------- cache write */

/* Store num_tokens new tokens' K and V rows into their slots ("가장 기본적인
 * decoding", steps 3-4: the new token's KV goes after the tokens already in its
 * logical block).  Row t of k_new ([num_tokens][num_kv_heads][head_dim],
 * device) is copied bit for bit to k_pool[slot / bs][h][slot % bs][:] for every
 * kv head h (layout R1), and the same for v.  slot_mapping is device int64
 * [num_tokens]; negative slots are skipped; a slot >= num_blocks * block_size is
 * skipped and sets PKV_DEV_BAD_SLOT in *d_status.  All device pointers must be
 * 16-byte aligned (head_dim * elem_size must be a multiple of 16).
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_CUDA (launch failure). */
int kv_cache_write(const pkv_pool *pool, const void *k_new, const void *v_new,
                   const int64_t *slot_mapping, int32_t num_tokens, void *k_pool,
                   void *v_pool, int32_t *d_status, void *stream);

/* ---------------------------------------------------- paged decode attention */

/* Workspace bytes paged_decode_attention needs for these sizes (split-K
 * partials, work list, merge counters, and room for shared prefixes: up to 4
 * more pieces per sequence and the shared-prefix work list).  0 on a bad
 * argument. */
size_t paged_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim,
                                    int32_t max_blocks_per_seq);

/* Single-query attention for every sequence and query head, gathering each
 * sequence's blocks through its block table ("KV Cache를 블록으로 쪼개다": the
 * PagedAttention kernel collects the blocks by following the table, so
 * attention works although KV is not contiguous):
 *   x_j = scale * <q[s][h], K_s[j][h / G]>,  j < context_lens[s]
 *   out[s][h] = sum_j softmax(x)_j * V_s[j][h / G],   G = num_q_heads / num_kv_heads
 * where K_s[j] lives in block block_tables[s][j / bs] at row j % bs (R1).
 * Work is split along the context into partitions whose (o, max, sum) pieces are
 * merged with the log-sum-exp rule; accumulation is fp32; out is rounded to the
 * pool dtype.  The partition size is chosen on the device from the context
 * lengths: 32, 64 or 128 blocks, the largest that still leaves every resident
 * CTA about five work items (paged_decode_default_split() is the smallest
 * candidate, the one the workspace is sized for).  Requirements: pool
 * block_size 16; head_dim 64 or 128;
 * num_q_heads a multiple of num_kv_heads with G <= 16; q/out/pools 16-byte
 * aligned; workspace of at least paged_decode_workspace_bytes(...) bytes,
 * 256-byte aligned, contents need not be initialised.  d_status: see the bits.
 * Sequences with context_len == 0 get zero rows (R7); a sequence with a bad
 * length or table entry gets a zero row and a status bit.  The result is
 * identical whatever the physical placement of the blocks.
 *
 * Shared prefixes ("PagedAttention 파헤치기", section "같은 블록을 여러 요청이
 * 나눠 쓴다": requests with a common prompt share its physical blocks).  When the
 * pool's ledger holds blocks with a reference count of 2 or more at the time of
 * the call (kv_pool_num_shared > 0), the call looks at the tables on the device:
 * neighbouring sequences whose rows agree on at least 16 leading valid block ids
 * (counted up to the block before each one's last token) are linked, and a run
 * of two or more linked sequences reads its shortest link's blocks once -- one
 * tcgen05 contraction of all members' query rows against those keys, in up to 4
 * key chunks -- while each member's partitions cover only the blocks after
 * them; the pieces merge by the same log-sum-exp rule.  The result is the same
 * attention, within fp32 rounding of a different summation order; sequences
 * outside runs are untouched.  Only the ledger's count decides whether the call
 * looks (a CUDA graph captured while it is 0 never looks); only the tables
 * decide what is shared.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA. */
int paged_decode_attention(const pkv_pool *pool, void *out, const void *q,
                           const void *k_pool, const void *v_pool,
                           const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *context_lens, int32_t num_seqs,
                           int32_t num_q_heads, float scale, void *workspace,
                           size_t workspace_bytes, int32_t *d_status, void *stream);

/* Same operation with an explicit partition size: each (sequence, kv head) is
 * cut into partitions of blocks_per_split blocks (>= 1) that run as separate
 * work items and are merged by log-sum-exp.  paged_decode_attention chooses
 * the size itself; results agree within rounding for any size. */
size_t paged_decode_workspace_bytes_split(int32_t num_seqs, int32_t num_q_heads,
                                          int32_t num_kv_heads, int32_t head_dim,
                                          int32_t max_blocks_per_seq,
                                          int32_t blocks_per_split);
int paged_decode_attention_split(const pkv_pool *pool, void *out, const void *q,
                                 const void *k_pool, const void *v_pool,
                                 const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 const int32_t *context_lens, int32_t num_seqs,
                                 int32_t num_q_heads, float scale, int32_t blocks_per_split,
                                 void *workspace, size_t workspace_bytes,
                                 int32_t *d_status, void *stream);

/* ------------------------------------------------- chunked-prefill attention */

/* Workspace bytes paged_prefill_attention needs.  0 on a bad argument. */
size_t paged_prefill_workspace_bytes(int32_t num_seqs, int32_t num_tokens, int32_t num_q_heads,
                                     int32_t num_kv_heads);

/* Workspace bytes with room for an fp16 copy of V (bf16 pools; an addition of
 * this library, not in the pages).  Given at least this much,
 * paged_prefill_attention over a bf16 pool first copies V of every token it
 * will attend to (2 * head_dim bytes per token and kv head, for
 * num_seqs * max_blocks_per_seq blocks) as fp16, scaled per (sequence, kv
 * head) by a power of two that puts the largest |v| just under 2^16, and then
 * forms P V with one fp16 part of P instead of two bf16 parts.  Every V value
 * within 2^30 of its (sequence, kv head)'s largest converts exactly (when that
 * largest is at least 2^-85; below it the scale stops at 2^100); smaller ones
 * round to fp16's subnormal spacing.  The result meets the same tolerance;
 * fp16 pools ignore the extra room.  Such calls run a kernel with 128-key
 * tiles (the others 64-key tiles); it splits its threads' registers with
 * setmaxnreg and launches only from a build whose kernels got the register
 * count that split assumes (otherwise PKV_ERR_CUDA).  0 on a bad argument. */
size_t paged_prefill_workspace_bytes_staged(int32_t num_seqs, int32_t num_tokens,
                                            int32_t num_q_heads, int32_t num_kv_heads,
                                            int32_t head_dim, int32_t max_blocks_per_seq);

/* Attention of a chunk of prompt tokens per sequence over the paged cache
 * ("vLLM과 Ollama의 차이": chunked prefill cuts a long prompt into chunks that
 * run beside the decoding sequences; "LLM 추론 배칭 전략 정리", section 0).
 * Sequence s's chunk is query rows query_start[s] .. query_start[s+1]-1 of q
 * and out ([num_tokens][num_q_heads][head_dim], pool dtype, device); its K/V is
 * already in the cache, which holds context_lens[s] tokens in total, the chunk
 * last.  Query j of the chunk sits at position context_lens[s] - C_s + j and
 * attends to the sequence's tokens 0..position (causal), gathered through
 * block_tables like paged_decode_attention (a one-token chunk is a decode
 * step).  query_start: device int32 [num_seqs + 1], non-decreasing, last entry
 * num_tokens.  A sequence whose chunk is longer than its context or whose
 * context exceeds its table row gets zero rows and PKV_DEV_BAD_LEN; bad table
 * entries set PKV_DEV_BAD_BLOCK.  Requirements as paged_decode_attention
 * (block_size 16, head_dim 64 or 128, G <= 16); workspace of
 * paged_prefill_workspace_bytes(...) bytes (or ..._staged(...) for the fp16
 * copy of V), 256-byte aligned.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA. */
int paged_prefill_attention(const pkv_pool *pool, void *out, const void *q, const void *k_pool,
                            const void *v_pool, const int32_t *block_tables,
                            int32_t max_blocks_per_seq, const int32_t *query_start,
                            const int32_t *context_lens, int32_t num_seqs, int32_t num_tokens,
                            int32_t num_q_heads, float scale, void *workspace,
                            size_t workspace_bytes, int32_t *d_status, void *stream);

/* ------------------------------------------- decode work planned on the host
 *
 * "LLM 추론 배칭 전략 정리", section 5: the CPU keeps the ledger and hands the
 * GPU its block table every step.  A caller that holds the step's context
 * lengths and tables on the host can also hand over the attention call's work
 * plan -- the one paged_decode_attention's first kernel builds on the device --
 * and save that kernel: paged_decode_plan builds it into host memory,
 * the caller copies its paged_decode_plan_bytes(...) bytes to the start of the
 * workspace (with its other host-to-device copies of the step), then calls
 * paged_decode_attention_planned with the same arguments as
 * paged_decode_attention.  The plan is identical to the device's (partition
 * size, work-list order, shared-prefix runs), so the result is too, bit for
 * bit. */

/* Bytes of the work plan (a prefix of the workspace of
 * paged_decode_workspace_bytes(...)).  0 on a bad argument. */
size_t paged_decode_plan_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_dim, int32_t max_blocks_per_seq);

/* Build the plan into `plan` (host memory, plan_bytes >= paged_decode_plan_bytes)
 * from host copies of context_lens [num_seqs] and block_tables
 * [num_seqs][max_blocks_per_seq] (NULL: no shared-prefix runs are looked for;
 * otherwise they are looked for as on the device, when the ledger holds shared
 * blocks).  *shared_prefix_items (may be NULL) receives the number of
 * shared-prefix work items, to pass to paged_decode_attention_planned.  Needs
 * the CUDA device current (the partition size depends on its SM count).
 * Errors: PKV_ERR_INVALID_ARG (also for a length < 0 or beyond the table row),
 * PKV_ERR_UNSUPPORTED (shapes the 16-bit kernels do not take), PKV_ERR_CUDA. */
int paged_decode_plan(const pkv_pool *pool, const int32_t *context_lens,
                      const int32_t *block_tables, int32_t max_blocks_per_seq, int32_t num_seqs,
                      int32_t num_q_heads, void *plan, size_t plan_bytes,
                      int32_t *shared_prefix_items);

/* paged_decode_attention whose workspace already begins with the plan that
 * paged_decode_plan built for the same lengths and tables (enqueued before this
 * call on the same stream, or on one it waits for); shared_prefix_items as
 * returned there.  A plan built from other lengths or tables gives wrong rows
 * (every access stays inside the workspace, the pools and the tables).
 * Errors: as paged_decode_attention. */
int paged_decode_attention_planned(const pkv_pool *pool, void *out, const void *q,
                                   const void *k_pool, const void *v_pool,
                                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *context_lens, int32_t num_seqs,
                                   int32_t num_q_heads, float scale, int32_t shared_prefix_items,
                                   void *workspace, size_t workspace_bytes, int32_t *d_status,
                                   void *stream);

/* Smallest partition size (blocks) paged_decode_attention considers, the one
 * its workspace is laid out for; the 8-bit decode uses exactly this size. */
int32_t paged_decode_default_split(void);

/* Paged decode attention that allocates nothing and takes no workspace.
 * (An addition of this library: the source pages have no counterpart.)
 *
 * Some callers cannot allocate device memory when they decode: an engine that
 * reserved nearly all free HBM for the KV pool at start-up has none left to
 * give, and a step loop may not afford cudaMalloc's implicit synchronisation.
 * This call computes exactly what paged_decode_attention computes, with the
 * scratch kept in a fixed array inside the library: PKV_NOALLOC_SCRATCH_BYTES
 * of global memory on every device that loads the library, held until the
 * process exits.  The caller still passes all inputs and outputs (out, q, the
 * pools, tables, lengths, status word).
 *   - The first call on a device looks up the array's device address (with that
 *     device current) and caches it; make that first call before any stream
 *     capture.  Resetting the device after that first call (cudaDeviceReset,
 *     or a reset of its primary context) is not supported: the cached address
 *     would then name memory the reloaded module no longer owns.
 *   - The partition size is the default when the scratch fits, otherwise the
 *     smallest number of partitions per sequence that fits.  Shapes that do
 *     not fit even with one partition per sequence are rejected with
 *     PKV_ERR_INVALID_ARG, and nothing is launched.
 *   - Nothing in the array has to start at zero: every launch rewrites the
 *     parts it reads.  The array is shared by every call on the device and keeps
 *     the last call's contents, so calls that overlap on the GPU (concurrent
 *     streams) race; serialise them.
 *   - No cudaMalloc, cudaFree or allocating library routine is called.
 * Errors: as paged_decode_attention, plus PKV_ERR_CUDA if the address lookup
 * fails. */
#define PKV_NOALLOC_SCRATCH_BYTES (32u << 20)
int paged_decode_attention_noalloc(const pkv_pool *pool, void *out, const void *q,
                                   const void *k_pool, const void *v_pool,
                                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *context_lens, int32_t num_seqs,
                                   int32_t num_q_heads, float scale, int32_t *d_status,
                                   void *stream);

/* ------------------------------------------------------------ status word */

/* Wait for the stream, read the device status word into *out_word (may be
 * NULL), clear it, and map it to a status: PKV_OK, PKV_ERR_DEVICE_BOUNDS,
 * PKV_ERR_DEVICE_TIMEOUT, or PKV_ERR_CUDA when the stream itself failed. */
int kv_status_check(int32_t *d_status, void *stream, int32_t *out_word);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
