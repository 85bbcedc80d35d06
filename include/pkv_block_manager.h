/*
 * pkv_block_manager.h - host-side KV-cache block allocator (C ABI).
 *
 * Produces the block tables and slot mappings the decode path consumes.
 * Rules (MinivLLM guide "HowToApproachvLLM", sections 3.1-3.3 and 4.5;
 * "VLLM-0.7.3 源码" section 3.1):
 *   - The cache is NB physical blocks of block_size token slots; free block
 *     ids wait in a FIFO pool and allocation takes the front.
 *   - A freshly allocated block has ref_count 1 (it is in use at once).
 *   - A block gets a content hash only when it is full; the hash chains the
 *     hash of the previous block (the prefix), so equal tokens under a
 *     different prefix hash differently.
 *   - Prompt allocation (allocate_with_cache) walks the prompt's blocks: a
 *     full block whose chained hash is known AND whose stored token ids are
 *     equal (hash-collision guard) is reused (ref_count + 1); from the first
 *     miss on, every block is newly allocated.
 *   - append: after the token is added, num_tokens % block_size == 1 opens a
 *     new block (the previous one was full); == 0 means the last block just
 *     filled, so it is hashed and registered for reuse.  The new token's
 *     slot is block_table[-1] * block_size + last_block_num_tokens - 1.
 *   - deallocate: every block of the sequence loses one reference; blocks
 *     that reach 0 return to the back of the free pool (their content hash
 *     stays registered until the block is handed out again).
 *
 * Sequences are named by caller-chosen int64 ids.  Token ids are int32.
 * Not thread-safe: one manager per host thread, or external locking.
 * Functions return pkv_status (see pkv.h) unless stated; messages via
 * pkv_last_error().
 */
#ifndef PKV_BLOCK_MANAGER_H_
#define PKV_BLOCK_MANAGER_H_

#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_block_manager pkv_block_manager;

/* New manager over num_blocks blocks of block_size slots (block_size >= 1). */
pkv_status pkv_bm_create(int64_t num_blocks, int block_size, pkv_block_manager **out);
void pkv_bm_destroy(pkv_block_manager *bm);

/* 1 if a prompt of num_tokens tokens can be allocated without cache hits. */
int pkv_bm_can_allocate(const pkv_block_manager *bm, int64_t num_tokens);

/*
 * Allocate a new sequence seq_id holding the prompt tokens[0..n) with prefix
 * caching.  *num_cached_tokens (may be NULL) receives how many leading
 * tokens were found cached (a multiple of block_size); their K/V need not be
 * written again.  Fails with PKV_ERR_INVALID_ARG if seq_id exists or n < 1,
 * and PKV_ERR_WORKSPACE if too few free blocks remain (nothing changes).
 */
pkv_status pkv_bm_allocate(pkv_block_manager *bm, int64_t seq_id, const int32_t *tokens,
                           int64_t n, int64_t *num_cached_tokens);

/* 1 if appending one token to seq_id needs no block or a free one exists. */
int pkv_bm_can_append(const pkv_block_manager *bm, int64_t seq_id);

/*
 * Append token to seq_id (allocating a block when the previous one was
 * full) and return the flat slot for its K/V in *slot.
 */
pkv_status pkv_bm_append(pkv_block_manager *bm, int64_t seq_id, int32_t token, int64_t *slot);

/*
 * Append tokens[i] to seq_ids[i] for i < n (one decode step for a batch;
 * ids must be distinct) and write each new token's slot to slots[i].  All
 * or nothing: if the free blocks do not cover every sequence that needs a
 * new one, nothing changes and PKV_ERR_WORKSPACE is returned.
 */
pkv_status pkv_bm_append_batch(pkv_block_manager *bm, const int64_t *seq_ids,
                               const int32_t *tokens, int n, int64_t *slots);

/* Release seq_id: every block loses one reference; free blocks at 0. */
pkv_status pkv_bm_deallocate(pkv_block_manager *bm, int64_t seq_id);

/* Free blocks in the pool. */
int64_t pkv_bm_num_free_blocks(const pkv_block_manager *bm);

/* Tokens held by seq_id, or -1 if unknown. */
int64_t pkv_bm_seq_len(const pkv_block_manager *bm, int64_t seq_id);

/* ref_count of a block (0 when free), or -1 for an invalid id. */
int32_t pkv_bm_ref_count(const pkv_block_manager *bm, int32_t block_id);

/*
 * Copy seq_id's block table into out[0..cap); returns its length (may be
 * larger than cap; only cap entries are written), or -1 if unknown.
 */
int64_t pkv_bm_block_table(const pkv_block_manager *bm, int64_t seq_id, int32_t *out,
                           int64_t cap);

/*
 * Flat slots of tokens [t0, t1) of seq_id into out[0..t1-t0) (for example
 * the uncached prompt tokens a prefill writes).
 */
pkv_status pkv_bm_slots(const pkv_block_manager *bm, int64_t seq_id, int64_t t0, int64_t t1,
                        int64_t *out);

/*
 * Decode-step arrays for the n sequences seq_ids[0..n), as prepare_decode
 * builds them: block_tables [n, MBS] (row b = the table of seq_ids[b],
 * padded with -1), context_lens [n] (tokens held), and, when slot_mapping is
 * non-NULL, the slot of each sequence's newest token.  Fails if a table is
 * longer than MBS or an id is unknown.
 */
pkv_status pkv_bm_decode_batch(const pkv_block_manager *bm, const int64_t *seq_ids, int n,
                               int MBS, int32_t *block_tables, int32_t *context_lens,
                               int64_t *slot_mapping);

#ifdef __cplusplus
}
#endif

#endif /* PKV_BLOCK_MANAGER_H_ */
