/*
 * Host-side block manager of the paged KV cache (part of libpagedattn.so).
 *
 * It owns no device memory.  It decides which physical block of the pool
 * holds each 16-token logical block of every sequence, and from that it
 * produces the block tables, lengths, cu_q_lens and slot mappings that the
 * device calls of pagedattn.h consume.
 *
 * What it does, and where the pages describe it:
 *
 *   - Free list and allocate_slots.  A fixed pool of blocks is handed out
 *     from a free list and returned when a sequence ends ("vLLM 在 CANN 上的
 *     推理优化", "vLLM 的 PagedAttention 数据结构": free_blocks,
 *     allocate_slots; "vLLM-Ascend 原理", section 2.1).
 *   - Prefix caching ("vLLM学习整理", section 三 "Prefix Caching").  Every
 *     logical block that fills up gets a key made of its own token ids, the
 *     key of the block before it, and an extra key (model, adapter, salt).
 *     Blocks with equal keys share one physical block, and a reference count
 *     tracks the holders.  A block whose count drops to 0 goes back to the
 *     free list but keeps its key until the list hands it out again, so a
 *     later request (a preempted one that re-prefills, for instance) can
 *     still hit it.
 *   - Copy-on-write ("vLLM-Ascend 原理", section 2.1).  fork() shares every
 *     block of a sequence.  The first write into a shared block that is not
 *     full moves the writer onto a fresh copy, and the call returns the
 *     (source, destination) pair for pa_copy_blocks.
 *   - Truncation ("vLLM-Ascend 原理", section 4 "推测解码").  Rejected
 *     speculative drafts are dropped by cutting the sequence length; blocks
 *     past the new end go back to the pool.
 *
 * Readings where the pages leave a choice open:
 *
 *   - Keys are compared exactly.  A key is the pair (registration id of the
 *     previous block, token ids), plus the extra key on the first block.
 *     Registration ids are never reused, so a 64-bit hash only picks the
 *     bucket and a collision can never alias two prefixes.
 *   - Blocks come off the free list at its head and go back at its tail
 *     (least recently freed first).  A sequence's blocks are freed last
 *     block first, so a prefix's tail is evicted before its head.
 *   - add_sequence matches full blocks only, and never the block that holds
 *     the prompt's last token: at least one prompt token is always computed.
 *
 * Threading: an instance is not thread-safe; one scheduler thread drives it.
 * Error behaviour: every call validates its arguments and returns a
 * pa_bm_status; a failed call changes nothing.
 */
#ifndef PA_BLOCK_MANAGER_H_
#define PA_BLOCK_MANAGER_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_BM_OK = 0,
    PA_BM_ERR_INVALID_ARG = 1,   /* null pointer, bad size, unknown or duplicate sequence id */
    PA_BM_ERR_NO_SPACE = 5,      /* not enough free blocks: nothing was allocated */
    PA_BM_ERR_CAPACITY = 6       /* an output buffer is too small */
} pa_bm_status;

typedef struct pa_block_manager pa_block_manager;

/* A pool of num_blocks blocks of block_size tokens, all free, numbered
 * 0..num_blocks-1 in free-list order.  prefix_caching != 0 turns on the
 * shared-prefix keys.  NULL on bad arguments or when out of host memory. */
pa_block_manager* pa_bm_create(int32_t num_blocks, int32_t block_size, int32_t prefix_caching);
void pa_bm_destroy(pa_block_manager* bm);

/* Blocks an allocation can take now: unreferenced blocks, cached or not. */
int32_t pa_bm_num_free_blocks(const pa_block_manager* bm);

/*
 * Register a new sequence with its prompt token ids (host array, copied).
 * With prefix caching on, the longest run of the prompt's full blocks whose
 * keys are cached is shared at once.  *num_cached_tokens receives its length
 * in tokens: a multiple of block_size, below prompt_len.  The sequence's
 * length starts there; allocate_slots covers the rest.
 */
int pa_bm_add_sequence(pa_block_manager* bm, int64_t seq_id, uint64_t extra_key, const int32_t* prompt,
                       int32_t prompt_len, int32_t* num_cached_tokens);

/* Append known token ids (sampled or draft tokens) to a sequence's token
 * list; allocate_slots then gives them slots. */
int pa_bm_append_tokens(pa_block_manager* bm, int64_t seq_id, const int32_t* token_ids, int32_t n);

/*
 * Reserve slots for the sequence's next num_new known tokens: its length
 * grows by num_new.  New blocks come from the free list; a shared partial
 * last block is first replaced by a copy (copy-on-write), reported in
 * cow_src[0] / cow_dst[0] with *num_cow = 1 (else *num_cow = 0).  Blocks
 * that become full are registered for prefix caching.  PA_BM_ERR_NO_SPACE
 * when the free list is too short (nothing changes: the caller may preempt
 * and retry).
 */
int pa_bm_allocate_slots(pa_block_manager* bm, int64_t seq_id, int32_t num_new, int32_t* cow_src,
                         int32_t* cow_dst, int32_t* num_cow);

/* Cut a sequence back to new_len tokens (<= its length): later blocks are
 * released, and the token list is cut too. */
int pa_bm_truncate(pa_block_manager* bm, int64_t seq_id, int32_t new_len);

/* New sequence child_id sharing every block (and the token list) of parent_id. */
int pa_bm_fork(pa_block_manager* bm, int64_t parent_id, int64_t child_id);

/* Release every block of the sequence (last block first) and forget it. */
int pa_bm_free_sequence(pa_block_manager* bm, int64_t seq_id);

/* Length (tokens with slots) of a sequence, or -1 when unknown. */
int32_t pa_bm_seq_len(const pa_block_manager* bm, int64_t seq_id);

/* The sequence's block table (physical ids, in logical order) into out[cap];
 * returns the number of blocks, or -1 (unknown sequence or cap too small). */
int32_t pa_bm_block_table(const pa_block_manager* bm, int64_t seq_id, int32_t* out, int32_t cap);

/* Reference count of a physical block (-1 for a bad id), and whether it
 * holds a registered prefix key. */
int32_t pa_bm_block_ref(const pa_block_manager* bm, int32_t block);
int32_t pa_bm_block_cached(const pa_block_manager* bm, int32_t block);

/*
 * Host inputs of one device step for num_seqs sequences, where sequence i
 * contributes its last q_lens[i] positions as new tokens (1 <= q_lens[i] <=
 * its length).  Writes
 *   block_tables  [num_seqs, max_blocks] int32, rows padded with -1
 *   seq_lens      [num_seqs] int32
 *   cu_q_lens     [num_seqs + 1] int32
 *   slot_mapping  [sum q_lens] int64: slot = table[pos / bs] * bs + pos % bs
 * PA_BM_ERR_CAPACITY when a table needs more than max_blocks entries or
 * slot_capacity is below the token count.
 */
int pa_bm_build_step(const pa_block_manager* bm, const int64_t* seq_ids, const int32_t* q_lens, int32_t num_seqs,
                     int32_t* block_tables, int32_t max_blocks, int32_t* seq_lens, int32_t* cu_q_lens,
                     int64_t* slot_mapping, int64_t slot_capacity);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCK_MANAGER_H_ */
