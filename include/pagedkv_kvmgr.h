/*
 * pagedkv_kvmgr.h -- host-side block manager of libpagedkv: allocation of
 * the paged cache's physical blocks, reference counts, copy-on-write, and a
 * radix tree over block-sized token chunks for prefix reuse.  It emits the
 * block tables, context lengths and slot mappings that pkv_paged_kv_append
 * and pkv_paged_attention take.
 *
 * Follows the pages' statement of the engine side of paged KV:
 *   - inferd README, "Paged KV" phase: a block allocator and a page table per
 *     sequence (core/paged_cache.py); its backlog's "prefix-sharing via
 *     copy-on-write KV blocks".
 *   - lfm25-inference README: "KV pages are managed by the engine rather than
 *     by individual requests", "Radix Tree Prefix Caching" (kv/allocator.rs,
 *     kv/radix.rs in its file list), page size 16.
 * The pages give the roles, not the policies; the policies below are this
 * library's (the oracle's model restates them step by step).
 *
 * Policies (deterministic; block_size 16):
 *   - Free blocks form a stack: a fresh manager hands out 0, 1, 2, ...; a
 *     freed block is handed out again before the ones never used.
 *   - A block's reference count counts the sequences whose table holds it
 *     plus one if the radix tree holds it.  Count 0 = free.
 *   - The radix tree maps a full block's 16 token ids (under the path of the
 *     blocks before it) to the block that holds their K/V.  A sequence added
 *     with a prompt reuses the longest chain of cached full blocks matching
 *     the prompt, leaving at least one prompt token to compute (a prefill
 *     must produce the last token's logits).
 *   - When no block is free, the least recently used leaf of the tree whose
 *     block nobody else holds is evicted (ties: lowest block id); a tree
 *     entry is "used" when a prompt matches it or when it is inserted.
 *   - Writing a token into a partially filled block that another sequence
 *     also holds (after pkv_kvmgr_fork) first copies the block: a fresh
 *     block replaces it in this sequence's table and the copy (source,
 *     destination) is returned for pkv_copy_blocks.
 *   - An operation that runs out of blocks frees what it allocated and
 *     returns PKV_ERR_NO_BLOCKS, leaving the sequence as it was.
 *
 * All pointers are HOST pointers.  A manager is not thread-safe.
 */
#ifndef PAGEDKV_KVMGR_H
#define PAGEDKV_KVMGR_H

#include <stdint.h>

#include "pagedkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_kvmgr pkv_kvmgr;

/* A manager of num_blocks blocks of 16 tokens (NULL if num_blocks < 1 or
 * out of memory).  Destroy with pkv_kvmgr_destroy. */
PKV_API pkv_kvmgr* pkv_kvmgr_create(int64_t num_blocks);
PKV_API void pkv_kvmgr_destroy(pkv_kvmgr* m);

/*
 * Register sequence `seq` (a new id) with its prompt tokens[0..n), n >= 1.
 * *cached_tokens receives how many leading prompt tokens are already in the
 * cache (a multiple of 16, reused from the radix tree; at most n - 1); the
 * slots of the other n - *cached_tokens prompt tokens, in order, go to
 * slots[0..n - *cached_tokens) (the caller appends their K/V there).
 */
PKV_API pkv_status pkv_kvmgr_add_sequence(pkv_kvmgr* m, int64_t seq, const int32_t* tokens, int64_t n,
                                          int64_t* cached_tokens, int64_t* slots);

/*
 * Reserve slots for n >= 1 new tokens of `seq` (tokens[0..n), e.g. a decode
 * step's token or a verify window); their slots go to slots[0..n).  If the
 * sequence's last block was partially filled and shared, it is copied first:
 * copy[0] = source block, copy[1] = destination block, *n_copies = 1 (else
 * 0).  The copy must be made (pkv_copy_blocks) before the new K/V are
 * appended.
 */
PKV_API pkv_status pkv_kvmgr_append(pkv_kvmgr* m, int64_t seq, const int32_t* tokens, int64_t n, int64_t* slots,
                                    int32_t* copy, int32_t* n_copies);

/* Publish the full blocks of `seq` in the radix tree (call once their K/V
 * are written), so later prompts with the same prefix reuse them. */
PKV_API pkv_status pkv_kvmgr_commit(pkv_kvmgr* m, int64_t seq);

/* New sequence `child` (a new id) sharing all of `parent`'s blocks and
 * tokens (copy-on-write for the partially filled last block). */
PKV_API pkv_status pkv_kvmgr_fork(pkv_kvmgr* m, int64_t parent, int64_t child);

/* Drop `seq`: its blocks lose one reference (blocks the tree holds stay
 * cached until evicted). */
PKV_API pkv_status pkv_kvmgr_release(pkv_kvmgr* m, int64_t seq);

/*
 * Block tables and context lengths of n sequences, in the layout
 * pkv_paged_attention takes: block_tables[i * max_blocks + j] = block j of
 * seqs[i] (-1 past its last block), context_lens[i] = its token count.
 * PKV_ERR_INVALID_ARG if a sequence needs more than max_blocks blocks.
 */
PKV_API pkv_status pkv_kvmgr_tables(const pkv_kvmgr* m, const int64_t* seqs, int32_t n, int32_t max_blocks,
                                    int32_t* block_tables, int32_t* context_lens);

/* Counts (for tests and monitoring): free blocks; blocks the radix tree
 * holds; the reference count of one block (-1 if out of range). */
PKV_API int64_t pkv_kvmgr_num_free(const pkv_kvmgr* m);
PKV_API int64_t pkv_kvmgr_num_cached(const pkv_kvmgr* m);
PKV_API int32_t pkv_kvmgr_refcount(const pkv_kvmgr* m, int32_t block);

/*
 * Device side of copy-on-write: copy the K and V pages of every kv-head of
 * block pairs[2i] to block pairs[2i + 1], i < n (pairs: DEVICE int32
 * [n][2]).  For an FP8 cache, k_scales / v_scales (device, the cache's scale
 * arrays, writable) get the same copies (NULL: scales not copied).  A block id
 * out of range skips that pair; a block that is the destination of one pair
 * and the source of another gives undefined contents.  Asynchronous on
 * `stream` (a programmatic dependent launch that waits for the previous
 * kernel before touching the cache).
 */
PKV_API pkv_status pkv_copy_blocks(const pkv_cache* cache, const int32_t* pairs, int32_t n, float* k_scales,
                                   float* v_scales, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_KVMGR_H */
