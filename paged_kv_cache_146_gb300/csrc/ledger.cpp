// Host block ledger: free stack + reference counts, on-demand allocation and
// slot mapping for appended tokens.
//
// Follows "vLLM의 핵심 원리 PagedAttention 파헤치기", section "KV Cache를 블록으로
// 쪼개다" (blocks taken one at a time from a free pool as a sequence grows),
// "vLLM-and-PagedAttention-KR", sections "가장 기본적인 decoding" (logical ->
// physical mapping, fill counts, release at the end) and "Parallel Sampling
// decoding" (reference counts of shared blocks), and "LLM 추론 배칭 전략 정리",
// section 5 (the ledger lives on the CPU and becomes the block table).
//
// Every operation is all-or-nothing: arguments are checked completely before
// any state changes.  O(1) per block taken or released.
#include <cstdlib>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"
#include "pkv_internal.h"

struct pkv_pool {
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    pkv_dtype dtype;
    std::vector<int32_t> stack;   // free blocks; back() is handed out next
    std::vector<int32_t> refs;    // refcount per block, 0 = free
    int64_t shared = 0;           // blocks whose refcount is 2 or more

    // every reference-count change goes through these two, which keep `shared`
    void take(int32_t id) { refs[(size_t)id] = 1; }
    void add_ref(int32_t id)
    {
        if (++refs[(size_t)id] == 2) ++shared;
    }
    // returns the new count
    int32_t drop_ref(int32_t id)
    {
        const int32_t r = --refs[(size_t)id];
        if (r == 1) --shared;
        return r;
    }
};

namespace pkv {
bool pool_geometry(const pkv_pool *p, PoolGeometry *g)
{
    if (!p || !g) return false;
    g->num_blocks = p->num_blocks;
    g->block_size = p->block_size;
    g->num_kv_heads = p->num_kv_heads;
    g->head_dim = p->head_dim;
    g->dtype = p->dtype;
    return true;
}

bool pool_has_shared_blocks(const pkv_pool *p) { return p && p->shared > 0; }
}  // namespace pkv

extern "C" {

int pkv_version(void) { return 10000; }

const char *pkv_status_string(int status)
{
    switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_OUT_OF_BLOCKS: return "out of free blocks";
    case PKV_ERR_BAD_BLOCK: return "bad block id, double free or refcount underflow";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_DEVICE_BOUNDS: return "device data out of range (slot, block id or length)";
    case PKV_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
    case PKV_ERR_SHARED_BLOCK: return "append target block is shared; copy it first";
    case PKV_ERR_UNSUPPORTED: return "shape not supported by the kernels";
    default: return "unknown status";
    }
}

int64_t kv_bytes_per_token(int32_t layers, int32_t kv_heads, int32_t head_dim,
                           int32_t elem_bytes)
{
    if (layers < 0 || kv_heads < 0 || head_dim < 0 || elem_bytes < 0) return -1;
    return (int64_t)layers * 2 * kv_heads * head_dim * elem_bytes;
}

int64_t kv_blocks_for_tokens(int64_t num_tokens, int32_t block_size)
{
    if (num_tokens < 0 || block_size <= 0) return -1;
    return (num_tokens + block_size - 1) / block_size;
}

size_t kv_pool_bytes(int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                     int32_t head_dim, pkv_dtype dtype)
{
    if (num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
    if (dtype == PKV_Q8_BF16 || dtype == PKV_Q8_F16)   // codes + one fp16 scale per 32, K and V
        return head_dim % 32 ? 0
                             : (size_t)num_blocks * num_kv_heads * block_size *
                                   (head_dim + head_dim / 32 * 2) * 2;
    if (dtype != PKV_F16 && dtype != PKV_BF16) return 0;
    return (size_t)num_blocks * num_kv_heads * block_size * head_dim * 2;
}

int kv_pool_create(int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                   int32_t head_dim, pkv_dtype dtype, const int32_t *initial_free_order,
                   pkv_pool **out)
{
    if (!out || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F16 && dtype != PKV_BF16 && dtype != PKV_Q8_BF16 && dtype != PKV_Q8_F16)
        return PKV_ERR_INVALID_ARG;
    *out = nullptr;
    pkv_pool *p = new (std::nothrow) pkv_pool;
    if (!p) return PKV_ERR_INVALID_ARG;
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->num_kv_heads = num_kv_heads;
    p->head_dim = head_dim;
    p->dtype = dtype;
    p->refs.assign((size_t)num_blocks, 0);
    p->stack.resize((size_t)num_blocks);
    if (initial_free_order) {
        std::vector<uint8_t> seen((size_t)num_blocks, 0);
        for (int32_t i = 0; i < num_blocks; ++i) {
            int32_t id = initial_free_order[i];
            if (id < 0 || id >= num_blocks || seen[(size_t)id]) {
                delete p;
                return PKV_ERR_INVALID_ARG;
            }
            seen[(size_t)id] = 1;
        }
        // first element handed out first: it sits at the back of the stack
        for (int32_t i = 0; i < num_blocks; ++i)
            p->stack[(size_t)(num_blocks - 1 - i)] = initial_free_order[i];
    } else {
        for (int32_t i = 0; i < num_blocks; ++i)
            p->stack[(size_t)(num_blocks - 1 - i)] = i;
    }
    *out = p;
    return PKV_OK;
}

int kv_pool_destroy(pkv_pool *pool)
{
    delete pool;
    return PKV_OK;
}

int kv_pool_info(const pkv_pool *pool, int32_t *num_blocks, int32_t *block_size,
                 int32_t *num_kv_heads, int32_t *head_dim, int32_t *dtype)
{
    if (!pool) return PKV_ERR_INVALID_ARG;
    if (num_blocks) *num_blocks = pool->num_blocks;
    if (block_size) *block_size = pool->block_size;
    if (num_kv_heads) *num_kv_heads = pool->num_kv_heads;
    if (head_dim) *head_dim = pool->head_dim;
    if (dtype) *dtype = (int32_t)pool->dtype;
    return PKV_OK;
}

int kv_block_alloc(pkv_pool *pool, int32_t n, int32_t *out_ids)
{
    if (!pool || n < 0 || (n > 0 && !out_ids)) return PKV_ERR_INVALID_ARG;
    if ((size_t)n > pool->stack.size()) return PKV_ERR_OUT_OF_BLOCKS;
    for (int32_t i = 0; i < n; ++i) {
        int32_t id = pool->stack.back();
        pool->stack.pop_back();
        pool->take(id);
        out_ids[i] = id;
    }
    return PKV_OK;
}

int kv_block_ref(pkv_pool *pool, int32_t n, const int32_t *ids)
{
    if (!pool || n < 0 || (n > 0 && !ids)) return PKV_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= pool->num_blocks || pool->refs[(size_t)ids[i]] < 1)
            return PKV_ERR_BAD_BLOCK;
    for (int32_t i = 0; i < n; ++i) pool->add_ref(ids[i]);
    return PKV_OK;
}

int kv_block_free(pkv_pool *pool, int32_t n, const int32_t *ids)
{
    if (!pool || n < 0 || (n > 0 && !ids)) return PKV_ERR_INVALID_ARG;
    // check, counting repeats: take the references away, undo on failure
    for (int32_t i = 0; i < n; ++i) {
        int32_t id = ids[i];
        if (id < 0 || id >= pool->num_blocks || pool->refs[(size_t)id] < 1) {
            for (int32_t k = 0; k < i; ++k) pool->refs[(size_t)ids[k]] += 1;
            return PKV_ERR_BAD_BLOCK;
        }
        pool->refs[(size_t)id] -= 1;
    }
    for (int32_t i = 0; i < n; ++i) pool->refs[(size_t)ids[i]] += 1;
    // apply in argument order: a block joins the free stack when it reaches 0
    for (int32_t i = 0; i < n; ++i) {
        int32_t id = ids[i];
        if (pool->drop_ref(id) == 0) pool->stack.push_back(id);
    }
    return PKV_OK;
}

int kv_block_refcount(const pkv_pool *pool, int32_t id, int32_t *out)
{
    if (!pool || !out) return PKV_ERR_INVALID_ARG;
    if (id < 0 || id >= pool->num_blocks) return PKV_ERR_BAD_BLOCK;
    *out = pool->refs[(size_t)id];
    return PKV_OK;
}

int kv_pool_num_free(const pkv_pool *pool, int32_t *out)
{
    if (!pool || !out) return PKV_ERR_INVALID_ARG;
    *out = (int32_t)pool->stack.size();
    return PKV_OK;
}

int kv_pool_num_shared(const pkv_pool *pool, int64_t *out)
{
    if (!pool || !out) return PKV_ERR_INVALID_ARG;
    *out = pool->shared;
    return PKV_OK;
}

int kv_append_slots(pkv_pool *pool, int32_t num_seqs, const int32_t *seq_lens,
                    const int32_t *num_new, int32_t *block_tables,
                    int32_t max_blocks_per_seq, int64_t *slot_mapping)
{
    if (!pool || num_seqs < 0 || max_blocks_per_seq <= 0) return PKV_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!seq_lens || !num_new || !block_tables)) return PKV_ERR_INVALID_ARG;
    const int64_t bs = pool->block_size;
    int64_t need = 0, total_new = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int64_t n0 = seq_lens[s], k = num_new[s];
        if (n0 < 0 || k < 0) return PKV_ERR_INVALID_ARG;
        if (n0 + k > (int64_t)max_blocks_per_seq * bs) return PKV_ERR_INVALID_ARG;
        if (k > 0 && n0 % bs != 0) {
            int32_t tail = block_tables[(int64_t)s * max_blocks_per_seq + n0 / bs];
            if (tail < 0 || tail >= pool->num_blocks || pool->refs[(size_t)tail] < 1)
                return PKV_ERR_BAD_BLOCK;
            if (pool->refs[(size_t)tail] > 1) return PKV_ERR_SHARED_BLOCK;
        }
        // blocks opened by positions n0 .. n0+k-1: multiples of bs in that range
        need += (n0 + k + bs - 1) / bs - (n0 + bs - 1) / bs;
        total_new += k;
    }
    if (total_new > 0 && !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (need > (int64_t)pool->stack.size()) return PKV_ERR_OUT_OF_BLOCKS;
    int64_t t = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
        int64_t n0 = seq_lens[s];
        for (int64_t pos = n0; pos < n0 + num_new[s]; ++pos) {
            if (pos % bs == 0) {
                int32_t id = pool->stack.back();
                pool->stack.pop_back();
                pool->take(id);
                row[pos / bs] = id;
            }
            slot_mapping[t++] = (int64_t)row[pos / bs] * bs + pos % bs;
        }
    }
    return PKV_OK;
}

int kv_seq_fork(pkv_pool *pool, const int32_t *parent_row, int32_t parent_len,
                int32_t *child_row, int32_t max_blocks_per_seq)
{
    if (!pool || !parent_row || !child_row || parent_len < 0 || max_blocks_per_seq <= 0)
        return PKV_ERR_INVALID_ARG;
    const int64_t nb = (parent_len + (int64_t)pool->block_size - 1) / pool->block_size;
    if (nb > max_blocks_per_seq) return PKV_ERR_INVALID_ARG;
    for (int64_t i = 0; i < nb; ++i) {
        const int32_t id = parent_row[i];
        if (id < 0 || id >= pool->num_blocks || pool->refs[(size_t)id] < 1) return PKV_ERR_BAD_BLOCK;
    }
    for (int64_t i = 0; i < nb; ++i) {
        pool->add_ref(parent_row[i]);
        child_row[i] = parent_row[i];
    }
    for (int64_t i = nb; i < max_blocks_per_seq; ++i) child_row[i] = -1;
    return PKV_OK;
}

int kv_append_slots_cow(pkv_pool *pool, int32_t num_seqs, const int32_t *seq_lens,
                        const int32_t *num_new, int32_t *block_tables,
                        int32_t max_blocks_per_seq, int64_t *slot_mapping, int32_t *copy_src,
                        int32_t *copy_dst, int32_t *num_copies)
{
    if (!pool || num_seqs < 0 || max_blocks_per_seq <= 0 || !num_copies) return PKV_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!seq_lens || !num_new || !block_tables || !copy_src || !copy_dst))
        return PKV_ERR_INVALID_ARG;
    const int64_t bs = pool->block_size;
    // dry run: blocks needed, counting the copies the sharing will force; a
    // shared tail loses one reference per copy taken from it, in sequence order
    std::unordered_map<int32_t, int32_t> taken;
    int64_t need = 0, total_new = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int64_t n0 = seq_lens[s], k = num_new[s];
        if (n0 < 0 || k < 0) return PKV_ERR_INVALID_ARG;
        if (n0 + k > (int64_t)max_blocks_per_seq * bs) return PKV_ERR_INVALID_ARG;
        if (k > 0 && n0 % bs != 0) {
            const int32_t tail = block_tables[(int64_t)s * max_blocks_per_seq + n0 / bs];
            if (tail < 0 || tail >= pool->num_blocks || pool->refs[(size_t)tail] < 1)
                return PKV_ERR_BAD_BLOCK;
            int32_t &t = taken[tail];
            if (pool->refs[(size_t)tail] - t > 1) {
                ++t;
                ++need;
            }
        }
        need += (n0 + k + bs - 1) / bs - (n0 + bs - 1) / bs;
        total_new += k;
    }
    if (total_new > 0 && !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (need > (int64_t)pool->stack.size()) return PKV_ERR_OUT_OF_BLOCKS;
    int64_t t = 0;
    int32_t copies = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
        const int64_t n0 = seq_lens[s];
        if (num_new[s] > 0 && n0 % bs != 0) {
            const int32_t tail = row[n0 / bs];
            if (pool->refs[(size_t)tail] > 1) {   // copy on write
                const int32_t fresh = pool->stack.back();
                pool->stack.pop_back();
                pool->take(fresh);
                pool->drop_ref(tail);
                copy_src[copies] = tail;
                copy_dst[copies] = fresh;
                ++copies;
                row[n0 / bs] = fresh;
            }
        }
        for (int64_t pos = n0; pos < n0 + num_new[s]; ++pos) {
            if (pos % bs == 0) {
                const int32_t id = pool->stack.back();
                pool->stack.pop_back();
                pool->take(id);
                row[pos / bs] = id;
            }
            slot_mapping[t++] = (int64_t)row[pos / bs] * bs + pos % bs;
        }
    }
    *num_copies = copies;
    return PKV_OK;
}

}  // extern "C"
