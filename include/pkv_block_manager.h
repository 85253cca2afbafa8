/*
 * pkv_block_manager.h -- host-side block manager with a prefix cache for the paged KV pool.
 *
 * Host only: no call here touches a GPU.  It hands out the physical block ids that
 * pkv_paged_kv_append writes and that the block tables of pkv_paged_decode_attention list.
 *
 * What it follows:
 *   habr.com/ru/articles/1021832, section 4 (fixed 16-token blocks, a reference count per
 *     physical block, copy-on-write for forked sequences) and section 7 "Тот самый
 *     Cache Read", on Automatic Prefix Caching (every full block is keyed by a hash of
 *     all tokens up to its end; a flat table maps hash -> physical block; a new request
 *     looks its blocks up from block 0 and stops at the first miss; the hits are reused with their reference count raised;
 *     blocks whose count fell to zero stay cached until the pool runs dry, and then the
 *     least recently freed one is evicted; cached blocks are never modified).
 *   gotacat.dev/blog/prompt-caching-kv-cache-vllm, sections "Хэш-цепочка в стиле
 *     git" and "Этот кэш не твой": a block's hash is computed from the parent
 *     block's hash, the block's own token ids and extra keys; the first block's parent is
 *     a fixed seed; a per-tenant salt enters the extra keys of the first block only, so
 *     requests with different salts never share blocks; a lookup is capped at
 *     num_tokens - 1 tokens so that at least the last prompt token is computed.
 *
 * Hash (the one format both sides of a comparison must agree on):
 *   h_0 parent = seed (32 bytes, given at creation), h_i parent = h_{i-1};
 *   h_i = SHA-256( parent[32] || u32le(block_size) || block_size x i32le(token id)
 *                  || u32le(len(extra)) || extra ),
 *   extra = the salt for block 0 and empty for every later block.  Only full blocks get a
 *   hash; a partial last block is never cached.
 *
 * Eviction order: blocks whose count reaches zero join the tail of a free queue; allocation
 * takes the head.  pkv_bm_free releases a sequence's blocks from its last block to its
 * first, so among blocks freed together the end of a chain is evicted before its start (a
 * lookup that stops at the first miss can still reuse the start).
 *
 * Thread safety: a manager is not thread safe; serialise calls on one manager.
 * Errors: every call returns a pkv_status (PKV_OK = 0) and sets pkv_last_error(); a call
 * that fails changes nothing.
 */
#ifndef PKV_BLOCK_MANAGER_H_
#define PKV_BLOCK_MANAGER_H_

#include <stdint.h>

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_block_manager pkv_block_manager;

/* SHA-256 of len bytes (FIPS 180-4) into out[32]. */
void pkv_sha256(const void* data, int64_t len, uint8_t out[32]);

/* Chained hashes of the num_tokens / block_size full blocks of a token sequence:
 * out_hashes[i*32 .. i*32+31] = h_i as defined above.  seed: 32 bytes.  salt may be NULL
 * when salt_len is 0.  Returns PKV_ERR_INVALID_ARG for block_size < 1 or negative sizes. */
pkv_status pkv_bm_chain_hashes(const uint8_t seed[32], int32_t block_size, const int32_t* tokens,
                               int64_t num_tokens, const uint8_t* salt, int64_t salt_len,
                               uint8_t* out_hashes);

/* A manager over physical blocks 0 .. num_blocks-1, all free and uncached; the free queue
 * starts in id order.  seed: 32 bytes (the parent of every chain's first block), or NULL
 * for 32 zero bytes.  *out receives the manager (owned by the caller, see destroy). */
pkv_status pkv_bm_create(int64_t num_blocks, int32_t block_size, const uint8_t* seed,
                         pkv_block_manager** out);
void pkv_bm_destroy(pkv_block_manager* bm);

/* Take n blocks from the head of the free queue (count 1 each); a cached block taken this
 * way is evicted (its hash leaves the table).  Fails with PKV_ERR_WORKSPACE, taking
 * nothing, when fewer than n blocks are free.  out_blocks: n int32 ids. */
pkv_status pkv_bm_allocate(pkv_block_manager* bm, int64_t n, int32_t* out_blocks);

/* Prefix lookup for a new request of num_tokens tokens: hashes its full blocks (salt in
 * block 0), walks them from block 0 while the table has the hash, at most
 * (num_tokens - 1) / block_size blocks, and stops at the first miss.  Every hit is taken
 * (count + 1; a block at count 0 leaves the free queue).  out_blocks: room for
 * max_out ids; *num_hit receives the number of hits (at most max_out; the walk stops there). */
pkv_status pkv_bm_get_computed_blocks(pkv_block_manager* bm, const int32_t* tokens, int64_t num_tokens,
                                      const uint8_t* salt, int64_t salt_len, int32_t* out_blocks,
                                      int64_t max_out, int64_t* num_hit);

/* After the KV of tokens[0 .. num_tokens) is in the pool at the blocks of block_table
 * (table_len entries, logical order), record the hashes of its full blocks.  A block that
 * already holds a hash must hold this one (else PKV_ERR_INVALID_ARG); a hash already owned
 * by another block leaves this block uncached (the table keeps the first owner).  Blocks
 * listed must be held (count > 0).  *num_cached receives how many blocks now carry their
 * hash (may be NULL). */
pkv_status pkv_bm_cache_full_blocks(pkv_block_manager* bm, const int32_t* tokens, int64_t num_tokens,
                                    const uint8_t* salt, int64_t salt_len, const int32_t* block_table,
                                    int64_t table_len, int64_t* num_cached);

/* Drop one reference to each listed block, from the last entry to the first; a block whose
 * count reaches zero joins the free-queue tail (staying cached if it has a hash).  A block
 * listed more often than it is held fails the call (nothing changes). */
pkv_status pkv_bm_free(pkv_block_manager* bm, const int32_t* blocks, int64_t n);

/* One more reference to each listed held block (prefix sharing, fork). */
pkv_status pkv_bm_share(pkv_block_manager* bm, const int32_t* blocks, int64_t n);

/* Before writing into held block `block`: if its count is 1 and it is not cached,
 * *out_block = block and *needs_copy = 0.  Otherwise (shared, or cached and therefore
 * immutable) a fresh block is allocated, one reference to `block` is dropped,
 * *out_block = the fresh id and *needs_copy = 1: the caller copies the KV of `block` into
 * it (pkv_copy_blocks) before writing. */
pkv_status pkv_bm_copy_on_write(pkv_block_manager* bm, int32_t block, int32_t* out_block,
                                int32_t* needs_copy);

/* Queries (no side effects).  A negative return means an invalid manager or id. */
int64_t pkv_bm_num_free(const pkv_block_manager* bm);
int64_t pkv_bm_num_cached(const pkv_block_manager* bm);
int32_t pkv_bm_ref_count(const pkv_block_manager* bm, int32_t block);
/* 1 and the hash in out[32] (may be NULL) if the block carries one, 0 if not. */
int32_t pkv_bm_block_hash(const pkv_block_manager* bm, int32_t block, uint8_t* out);
/* The block the table maps this hash to, or -1. */
int32_t pkv_bm_lookup(const pkv_block_manager* bm, const uint8_t hash[32]);
/* The free queue from head (next evicted) to tail: up to max_out ids; returns the count. */
int64_t pkv_bm_free_queue(const pkv_block_manager* bm, int32_t* out, int64_t max_out);

#ifdef __cplusplus
}
#endif

#endif  // PKV_BLOCK_MANAGER_H_
