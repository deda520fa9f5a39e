/*
 * pagedkv_block_manager.h -- C ABI of the host-side block manager that feeds
 * the decode step of pagedkv.h: it owns the free list of physical blocks, the
 * per-sequence block tables and the reference counts, and turns "append one
 * token to these sequences" into the slot_mapping of pk_reshape_and_cache
 * and the (src, dst) pairs of pk_copy_blocks.
 *
 * The rules it implements:
 *   - Free list: starts as every block id in increasing order; a block is
 *     taken from its front and a freed block goes to its back ("How vLLM and
 *     PagedAttention Actually Work", §6 Python blueprint; "PagedAttention
 *     Explained", copy-on-write walkthrough).
 *   - Allocate on full: a sequence takes a new block only when the token it
 *     appends starts one, i.e. when its length is a multiple of block_size
 *     ("vLLM — PagedAttention", Block Table Data Structure).
 *   - Copy-on-write: appending into a last block whose reference count is
 *     above one first takes a fresh block, records (old, new) for the block
 *     copy, points this sequence at the copy and drops one reference from the
 *     old block; with a count of one the token is written in place ("vLLM —
 *     PagedAttention", Copy-on-Write Logic).
 *   - fork shares blocks of the parent (each count grows by one); freeing a
 *     sequence drops one reference per block and returns blocks whose count
 *     reaches zero ("vLLM — PagedAttention", Three Core API Methods).
 *   - A token's flat slot is block_id * block_size + offset in block.
 *
 * Memory and threads.  Everything lives in host memory owned by the manager
 * (created by pk_bm_create, released by pk_bm_destroy).  Output arrays are
 * caller-owned host memory (pinned memory is fine and lets the caller copy
 * them to the device asynchronously).  A manager is not thread-safe: use one
 * per scheduler thread or serialise the calls.  Nothing here touches the GPU.
 *
 * Errors.  Every call returns a pk_status (pagedkv.h); on error the manager
 * is unchanged (pk_bm_append_slots undoes the part of the batch it had done).
 */
#ifndef PAGEDKV_BLOCK_MANAGER_H
#define PAGEDKV_BLOCK_MANAGER_H

#include "pagedkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pk_block_manager pk_block_manager;

/* A manager for a pool of num_blocks blocks of block_size tokens (both > 0).
 * Returns NULL if an argument is out of range or memory runs out. */
pk_block_manager *pk_bm_create(int num_blocks, int block_size);
/* Releases the manager; NULL is ignored. */
void pk_bm_destroy(pk_block_manager *bm);

/* Registers an empty sequence (length 0, no blocks).
 * PK_ERR_SEQUENCE_EXISTS if the id is taken. */
int pk_bm_add_sequence(pk_block_manager *bm, int64_t seq_id);

/* Appends one token to each of seq_ids[0..n) in order (an id may repeat: it
 * then gets several tokens) and writes the token's flat slot to slots_out[i].
 * New blocks and copy-on-write copies are taken as the rules above say; the
 * copies are queued for pk_bm_take_copies.  All or nothing: if the pool runs
 * out (PK_ERR_NO_BLOCKS) or an id is unknown, the batch is undone and
 * nothing is written to slots_out. */
int pk_bm_append_slots(pk_block_manager *bm, const int64_t *seq_ids, int n, int64_t *slots_out);

/* Starts `child` sharing the parent's first num_tokens tokens.  num_tokens =
 * -1 shares the whole parent, partial last block included (parallel
 * sampling); otherwise num_tokens must be a multiple of block_size and at
 * most the parent's length (prefix sharing of whole blocks). */
int pk_bm_fork(pk_block_manager *bm, int64_t parent, int64_t child, int64_t num_tokens);

/* Drops the sequence; blocks no other sequence holds return to the back of
 * the free list, in table order. */
int pk_bm_free_sequence(pk_block_manager *bm, int64_t seq_id);

/* Number of copy pairs queued since the last pk_bm_take_copies. */
int pk_bm_num_pending_copies(const pk_block_manager *bm);

/* Moves the queued copy pairs, in the order they were decided, to
 * pairs_out[2*i] = src, pairs_out[2*i+1] = dst and sets *num_out.  If more
 * than max_pairs are queued, returns PK_ERR_SHAPE, sets *num_out to the
 * number queued and moves nothing. */
int pk_bm_take_copies(pk_block_manager *bm, int64_t *pairs_out, int max_pairs, int *num_out);

/* Writes the block tables and lengths of seq_ids[0..n) in the layout
 * pk_paged_attention_decode reads: block_tables[i * max_blocks + j] for
 * j < max_blocks (entries past the sequence's blocks are -1) and
 * seq_lens[i].  PK_ERR_SHAPE (nothing written) if a sequence has more than
 * max_blocks blocks or a length above INT32_MAX. */
int pk_bm_export(const pk_block_manager *bm, const int64_t *seq_ids, int n, int32_t *block_tables,
                 int max_blocks, int32_t *seq_lens);

/* Length (tokens) and block count of one sequence. */
int pk_bm_sequence_info(const pk_block_manager *bm, int64_t seq_id, int64_t *length_out, int *num_blocks_out);

/* Free blocks, and blocks held by at least one sequence (their sum is
 * num_blocks). */
int pk_bm_num_free_blocks(const pk_block_manager *bm);
int pk_bm_blocks_in_use(const pk_block_manager *bm);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_BLOCK_MANAGER_H */
