/*
 * pkv_blocks.h — host block manager of the paged KV cache and the device
 * copy-on-write block copy.
 *
 * Sources (web pages, cited by title and section):
 *   [FN] "Sub-Millisecond Token Scheduling: Inside Disaggregated KV-Cache
 *        Paging for Frontier LLMs", section "Paged KV-Cache with Radix Tree
 *        Prefix Cache": fixed-size physical blocks with reference counts, a
 *        free pool, per-sequence block tables grown one block at a time, an
 *        exhausted pool reported to the scheduler so that it preempts, and
 *        prompt-sharing requests referencing the same blocks through
 *        copy-on-write pointers.
 *   [SC] "LLM inference: prefill, decode, KV cache", sections "PagedAttention
 *        & Memory Management (vLLM)" (on-demand allocation through a block
 *        table) and "9. Failure modes and limitations", item 2 (preemption
 *        when memory is exhausted).
 *
 * The manager is plain host code (no CUDA call, no GPU needed).  It hands out
 * the slot of every new token (block * block_size + offset, the slot_mapping
 * of pkv_append) and the (source, destination) block pairs that must be
 * copied on the device before those slots are written (pkv_copy_blocks).
 *
 * Policy, fixed so that results are reproducible:
 *   - The free pool is a stack; a new manager holds blocks 0..N-1 pushed in
 *     that order, so the first block handed out is N-1.  Freed blocks are
 *     pushed on top and are the next ones handed out.
 *   - Appending to a sequence of length L writes positions L, L+1, ...; a
 *     position that starts a block takes a new block; a position inside the
 *     last block writes into it if its reference count is 1, else the block
 *     is copied first (copy-on-write: a new block is taken, the pair
 *     (old, new) is reported, the old block loses one reference).
 *   - pkv_bm_append over several sequences is all or nothing: when the pool
 *     cannot cover the whole call it returns PKV_ERR_OUT_OF_BLOCKS and
 *     changes nothing; the caller frees or swaps out a sequence and retries.
 *   - pkv_bm_free_sequence drops one reference from each block of the table
 *     in table order, pushing each block whose count reaches zero.
 *
 * Thread safety: every call on one manager takes that manager's lock.
 */
#ifndef PKV_BLOCKS_H_
#define PKV_BLOCKS_H_

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_block_manager pkv_block_manager;

/* num_blocks in [1, 2^31 - 1], block_size >= 1.  *out receives the manager
 * (owned by the caller, released by pkv_bm_destroy). */
pkv_status pkv_bm_create(int64_t num_blocks, int32_t block_size, pkv_block_manager** out);
void pkv_bm_destroy(pkv_block_manager* bm);

/* Blocks on the free pool; -1 for a NULL manager. */
int64_t pkv_bm_num_free(pkv_block_manager* bm);
/* Reference count of a physical block; -1 when out of range. */
int32_t pkv_bm_ref_count(pkv_block_manager* bm, int64_t block);
/* Tokens held by a sequence; -1 for an unknown sequence. */
int64_t pkv_bm_seq_len(pkv_block_manager* bm, int64_t seq_id);
/* Number of live sequences. */
int64_t pkv_bm_num_sequences(pkv_block_manager* bm);

/* Register an empty sequence (PKV_ERR_INVALID_ARG if the id is taken). */
pkv_status pkv_bm_add_sequence(pkv_block_manager* bm, int64_t seq_id);

/* New sequence `child` sharing every block of `parent` (each block gains one
 * reference) with the parent's length: the shared-prompt case. */
pkv_status pkv_bm_fork(pkv_block_manager* bm, int64_t parent_id, int64_t child_id);

/* Drop a sequence and one reference from each of its blocks. */
pkv_status pkv_bm_free_sequence(pkv_block_manager* bm, int64_t seq_id);

/*
 * Reserve n_new[i] token slots at the end of sequence seq_ids[i], for i in
 * [0, n_seqs) in that order (ids distinct, n_new[i] >= 0).
 *   slots     int64 [sum n_new], host memory: the flat slot of each new token,
 *             sequence by sequence, ready to be the slot_mapping of pkv_append.
 *   cow_src, cow_dst  int32 [cow_capacity], host memory: block pairs to copy
 *             (pkv_copy_blocks) before the slots are written; at most one per
 *             sequence, so cow_capacity = n_seqs always suffices.
 *   n_cow     receives the number of pairs.
 * PKV_ERR_OUT_OF_BLOCKS: the free pool cannot cover the call; nothing changed.
 * PKV_ERR_INVALID_ARG: unknown or repeated id, negative count, NULL pointer,
 * or cow_capacity below the pairs needed; nothing changed.
 */
pkv_status pkv_bm_append(pkv_block_manager* bm, int32_t n_seqs, const int64_t* seq_ids,
                         const int32_t* n_new, int64_t* slots, int32_t* cow_src,
                         int32_t* cow_dst, int32_t cow_capacity, int32_t* n_cow);

/* Blocks the same pkv_bm_append call would take from the pool (new blocks
 * plus copies), without changing anything. */
pkv_status pkv_bm_blocks_needed(pkv_block_manager* bm, int32_t n_seqs, const int64_t* seq_ids,
                                const int32_t* n_new, int64_t* blocks_needed);

/*
 * Block tables and lengths of n_seqs sequences, host memory:
 *   block_tables  int32 [n_seqs, max_blocks_per_seq], -1 past each table
 *   context_lens  int32 [n_seqs] (may be NULL)
 * PKV_ERR_INVALID_ARG if a table is longer than max_blocks_per_seq or a
 * length exceeds INT32_MAX.
 */
pkv_status pkv_bm_block_tables(pkv_block_manager* bm, int32_t n_seqs, const int64_t* seq_ids,
                                int32_t max_blocks_per_seq, int32_t* block_tables,
                                int32_t* context_lens);

/*
 * pkv_copy_blocks — device copy-on-write step: for each pair i,
 * k_cache[dst[i]] = k_cache[src[i]] and v_cache[dst[i]] = v_cache[src[i]]
 * (whole blocks: all KV heads, all slots, bit for bit).
 *   src_blocks, dst_blocks  int32 [n_pairs], DEVICE memory.
 *   Destinations must be distinct and no destination may be a source of the
 *   same call (pairs from pkv_bm_append satisfy both).  An id outside
 *   [0, num_blocks) is recorded in the device error word (PKV_DEVERR_BLOCK_ID)
 *   and its pair skipped.  n_pairs == 0 is a no-op.  Caches as pkv_append.
 */
pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                           const int32_t* src_blocks, const int32_t* dst_blocks,
                           int32_t n_pairs, pkv_stream_t stream);

/* ------------------------------------------------------------ host tier
 *
 * A second pool of blocks in host memory, for swapping preempted sequences
 * out of HBM ([SC] "9. Failure modes and limitations", item 2, Swap to CPU)
 * and for moving single blocks between the tiers ([UI] "Architecting
 * Multi-Tier Disaggregated KV-Cache Hierarchies...", "C++ Block Scheduler
 * and Asynchronous Fetch Kernel": promote a block from Tier-2 host memory to
 * Tier-1 HBM, demote it back; "Tier-1 / Tier-2 Double Buffering": fetch the
 * blocks needed a few steps ahead while the current step runs).
 *
 * Every table entry is either a device block id or a host block id.  A
 * sequence with any host entry cannot be appended to, forked or attended
 * (pkv_bm_append / pkv_bm_fork / pkv_bm_block_tables return
 * PKV_ERR_INVALID_ARG) until its entries are staged back.  Host blocks are
 * never shared: demoting a shared device block gives this sequence its own
 * host copy and drops one device reference.
 */

/* Give the manager a host pool of num_host_blocks (once).  The host free
 * pool is a stack like the device one (block num_host_blocks - 1 first). */
pkv_status pkv_bm_set_host_blocks(pkv_block_manager* bm, int64_t num_host_blocks);
int64_t pkv_bm_num_free_host(pkv_block_manager* bm);
/* Host entries of a sequence; -1 for an unknown sequence. */
int64_t pkv_bm_host_entries(pkv_block_manager* bm, int64_t seq_id);

/*
 * Demote (evict) / promote (stage) entries `logical[0..n)` of a sequence
 * (distinct indices inside its table).  Entries already in the target tier
 * are skipped.  The (from, to) block pairs to copy are written to the two
 * arrays (n entries suffice) and their count to *n_pairs; copy them with
 * pkv_copy_blocks_between before the freed blocks are reused.  All or
 * nothing: PKV_ERR_OUT_OF_BLOCKS when the target pool is short.
 */
pkv_status pkv_bm_evict(pkv_block_manager* bm, int64_t seq_id, int32_t n, const int32_t* logical,
                        int32_t* dev_src, int32_t* host_dst, int32_t* n_pairs);
pkv_status pkv_bm_stage(pkv_block_manager* bm, int64_t seq_id, int32_t n, const int32_t* logical,
                        int32_t* host_src, int32_t* dev_dst, int32_t* n_pairs);

/* The raw table of a sequence: ids[j] and on_host[j] (0 / 1) for each entry. */
pkv_status pkv_bm_table_entries(pkv_block_manager* bm, int64_t seq_id, int32_t capacity,
                                int32_t* ids, int32_t* on_host, int32_t* n_entries);

/*
 * Prefetch candidates ([UI] "Predictive
 * Prefetching and Attention-Salience Eviction Policy": an evicted block whose
 * predicted activation exceeds the prefetch threshold is staged some steps
 * ahead of the decode step that needs it): the host entries j of a sequence
 * with activation[j] > threshold, most probable first (ties by index), at
 * most `capacity` and at most the free device blocks, so that staging all of
 * them succeeds.  *n_out is how many were written.
 *   activation  float [entries of the sequence], host memory.
 */
pkv_status pkv_bm_prefetch_candidates(pkv_block_manager* bm, int64_t seq_id, const float* activation,
                                      float threshold, int32_t capacity, int32_t* logical, int32_t* n_out);

/*
 * pkv_copy_blocks_between — pair i copies block src_blocks[i] of the source
 * pool (src_k, src_v; src_num_blocks blocks) to block dst_blocks[i] of the
 * destination pool; both pools have the block geometry and dtype of `cache`
 * (its num_blocks is not used).  Pools and id arrays may be device memory or
 * host memory the GPU can address (pinned with pkv_host_alloc): one kernel
 * moves every block of the call through the GPU's own loads and stores.
 * Ids outside a pool are recorded (PKV_DEVERR_BLOCK_ID) and skipped.
 *   max_ctas  upper bound on the copy's thread blocks; 0 = automatic: 64
 *             when a pool is in host memory, else no bound.  A copy across
 *             the host link saturates the link with a few dozen; bounding it
 *             leaves the other SMs to attention kernels running at the same
 *             time on other streams.
 */
pkv_status pkv_copy_blocks_between(const void* src_k, const void* src_v, int64_t src_num_blocks,
                                   void* dst_k, void* dst_v, int64_t dst_num_blocks,
                                   const pkv_cache_desc* cache, const int32_t* src_blocks,
                                   const int32_t* dst_blocks, int32_t n_pairs, int32_t max_ctas,
                                   pkv_stream_t stream);

/* Page-locked host memory mapped into the GPU's address space (the same
 * pointer works on host and device); pkv_host_free releases it. */
pkv_status pkv_host_alloc(size_t bytes, void** ptr);
pkv_status pkv_host_free(void* ptr);

#ifdef __cplusplus
}
#endif

#endif /* PKV_BLOCKS_H_ */
