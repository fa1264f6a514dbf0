/*
 * pagedattn.h: C ABI of libpagedattn.so, paged KV attention for GB300 (sm_103a).
 *
 * The operations follow the descriptions of vLLM's PagedAttention in
 * "vLLM-Ascend 原理" (section 2.1 PagedAttention, 2.3 Prefill, 2.4 Decode) and
 * "vLLM 在 CANN 上的推理优化" (section "vLLM 的 PagedAttention 数据结构" and
 * the PagedAttentionKernel sketch in "CANN 上的 PagedAttention 算子").
 *
 * Memory layout (all arrays dense, row-major, on the current CUDA device):
 *   k_cache, v_cache  [num_blocks, block_size, num_kv_heads, head_dim]
 *                     two separate pools, one per K and V, element type
 *                     `dtype`; physical block p, offset o, head h, dim d lives
 *                     at ((p * block_size + o) * num_kv_heads + h) * head_dim + d.
 *   block_tables      int32 [num_seqs, max_blocks_per_seq]; row b maps the
 *                     logical blocks of sequence b to physical blocks.  Entries
 *                     at or past ceil(seq_lens[b] / block_size) are never read.
 *   seq_lens          int32 [num_seqs]; tokens of sequence b, counting the
 *                     tokens this step appends (so a decode query sits at
 *                     position seq_lens[b] - 1 and sees itself).
 *   cu_q_lens         int32 [num_seqs + 1]; sequence b owns query / new-token
 *                     rows cu_q_lens[b] .. cu_q_lens[b+1]-1; these are its last
 *                     positions seq_lens[b] - q_len .. seq_lens[b] - 1.
 *   q, out            [rows, num_q_heads, head_dim], element type `dtype`.
 *   key, value        [num_tokens, num_kv_heads, head_dim] (new tokens).
 *
 * Supported: block_size == 16, head_dim in {64, 128}, dtype fp16 or bf16,
 * num_q_heads % num_kv_heads == 0 with num_q_heads / num_kv_heads <= PA_MAX_GROUP
 * (64: grouped-query and multi-query attention);
 * q head h reads kv head h / (num_q_heads / num_kv_heads).
 *
 * Ownership: the caller owns every buffer.  The library allocates no device
 * memory; calls that need scratch space take a caller-provided workspace
 * whose minimum size the matching *_workspace_bytes function returns.
 *
 * Execution: every call only enqueues work on `stream` (a cudaStream_t; NULL
 * = the legacy default stream) and returns without synchronising, except
 * pa_get_device_error, which waits for the stream.
 *
 * Device state: the library looks up, once per device, the addresses of its
 * own device variables (the error word, the scratch array of
 * pa_paged_attention_decode_noalloc) and keeps them for the life of the
 * process.  They do not survive cudaDeviceReset: after a reset, do not call
 * the library again in that process.
 *
 * Errors: arguments are validated on the host before anything is launched;
 * a rejected call returns a nonzero pa_status and enqueues nothing.  A
 * launch failure returns PA_ERR_CUDA.  The kernels also check every block
 * table entry and slot they use against the pool; an out-of-range entry is
 * skipped (its tokens contribute nothing, its write is dropped) and recorded
 * in a device error word that pa_get_device_error reads.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_BLOCK_SIZE 16
#define PA_DEFAULT_PARTITION 512
/* partition_size 0 means PA_DEFAULT_PARTITION tokens, doubled (up to
 * PA_MAX_AUTO_PARTITION) while a sequence of max_seq_len tokens would have
 * more than PA_AUTO_MAX_PARTS partitions (see pa_decode_partition). */
#define PA_AUTO_MAX_PARTS 64
#define PA_MAX_AUTO_PARTITION 8192
#define PA_MAX_GROUP 64
/* Chunks of at most this many queries (decode rows, speculative-verify rows)
 * run in the decode kernel inside pa_paged_attention_prefill. */
#define PA_VERIFY_MAX_Q 8

typedef enum { PA_F16 = 0, PA_BF16 = 1 } pa_dtype;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,          /* null pointer, negative size, inconsistent shape */
    PA_ERR_UNSUPPORTED = 2,          /* dtype, head_dim, block_size or head grouping */
    PA_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace NULL or below *_workspace_bytes */
    PA_ERR_CUDA = 4                  /* a CUDA runtime call or kernel launch failed */
} pa_status;

/* Device error word bits reported by pa_get_device_error. */
#define PA_DEVERR_BLOCK_ID 1   /* a live block-table entry outside [0, num_blocks) */
#define PA_DEVERR_SLOT 2       /* a slot at or past num_blocks * block_size */
#define PA_DEVERR_SEQ_LEN 4    /* seq_len above max_seq_len or the table's capacity */
#define PA_DEVERR_TIMEOUT 8    /* a bounded wait for a TMA copy ran out (the work was abandoned) */
#define PA_DEVERR_WORKSPACE 16 /* an FP8 prefill chunk's 16-bit copy did not fit (its rows were skipped) */

/* Library ABI version (major * 100 + minor). */
int pa_version(void);

/* Static, human-readable name of a pa_status value. */
const char* pa_status_string(int status);

/*
 * Slot address of every new token ("vLLM 在 CANN 上的推理优化", the read_kv
 * sketch: logical index -> logical block idx / block_size, offset
 * idx % block_size, physical block from the table; slot = physical block *
 * block_size + offset).
 *   slot_mapping  int64 [num_tokens] (out): slot of new-token row r.
 *   cu_q_lens     int32 [num_seqs + 1], or NULL meaning one new token per
 *                 sequence (decode; num_tokens must equal num_seqs).
 * Rows of a sequence whose table entry is out of range get slot -1 and set
 * PA_DEVERR_BLOCK_ID; rows of a sequence whose seq_len is below its new-token
 * count (or above the table's capacity) get slot -1 and set
 * PA_DEVERR_SEQ_LEN.  A decode row (cu_q_lens NULL) with seq_len 0 is a
 * padding row (a batch padded to a fixed size, e.g. a captured graph's
 * bucket): slot -1, nothing flagged; decode attention gives it a zero row.
 */
int pa_slot_mapping(int64_t* slot_mapping, const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* seq_lens, const int32_t* cu_q_lens, int num_seqs,
                    int num_tokens, int num_blocks, int block_size, void* stream);

/*
 * reshape_and_cache: write each new token's k and v into its slot
 * ("vLLM-Ascend 原理", section 2.3 "KV 写缓存" and section 2.4 "KV 追加写").
 *   key, value    [num_tokens, num_kv_heads, head_dim]
 *   k_cache/v_cache are updated in place.
 *   slot_mapping  int64 [num_tokens]; a negative slot means "no write"
 *                 (padding); a slot >= num_blocks * block_size is dropped and
 *                 sets PA_DEVERR_SLOT.
 * The copy is bit-exact.  Two rows naming one slot race (last writer wins).
 */
int pa_paged_kv_write(const void* key, const void* value, void* k_cache, void* v_cache,
                      const int64_t* slot_mapping, int num_tokens, int num_blocks,
                      int num_kv_heads, int head_dim, int block_size, int dtype, void* stream);

/*
 * The partition length (tokens) a decode call with these arguments uses:
 * partition_size itself when nonzero; for 0, PA_DEFAULT_PARTITION doubled
 * while ceil(max_seq_len / partition) > PA_AUTO_MAX_PARTS, at most
 * PA_MAX_AUTO_PARTITION (long contexts merge fewer partials; shorter ones keep
 * more, smaller work items for load balance).  Decode and verify rows of
 * pa_paged_attention_prefill use the value for 0.  Returns -1 for a negative
 * argument or a partition_size that is not a multiple of PA_BLOCK_SIZE.
 */
int pa_decode_partition(int max_seq_len, int partition_size);

/*
 * Workspace for pa_paged_attention_decode: the kernel's work list (one entry
 * per sequence partition) and the split-context partials of num_seqs
 * sequences no longer than max_seq_len, cut into partitions of
 * partition_size tokens (0 = the automatic length of pa_decode_partition).
 * Nonzero whenever num_seqs > 0.
 */
size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int max_seq_len,
                                 int partition_size);

/*
 * Decode attention over the paged cache ("vLLM-Ascend 原理", section 2.4
 * "分页自注意力"; the block loop of the CANN PagedAttentionKernel sketch).
 * One query per sequence: out[b, h] = sum_t softmax_t(scale * q[b, h] . k_t) v_t
 * over positions t = 0 .. seq_lens[b] - 1, k_t and v_t read through the block
 * table, with the softmax merged block by block (online softmax).  Sequences
 * longer than partition_size tokens are split into partitions whose partial
 * (max, sum, accumulator) are merged by a log-sum-exp reduction.
 *   out, q        [num_seqs, num_q_heads, head_dim]
 *   max_seq_len   host-side upper bound of seq_lens (sizes the grid).
 *   num_blocks    pool size in blocks (bounds every table entry).
 *   partition_size tokens per partition, a positive multiple of block_size,
 *                 or 0 for the automatic length (pa_decode_partition).
 *   workspace     device scratch of at least pa_decode_workspace_bytes(...)
 *                 bytes, 256-byte aligned.
 * A sequence with seq_len == 0 gets an all-zero output row.
 */
int pa_paged_attention_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, int max_blocks_per_seq,
                              const int32_t* seq_lens, int num_seqs, int max_seq_len,
                              int num_blocks, float scale, int num_q_heads, int num_kv_heads,
                              int head_dim, int block_size, int partition_size, void* workspace,
                              size_t workspace_bytes, int dtype, void* stream);

/*
 * Test support: gather each sequence's cached K/V through its block table into
 * contiguous rows ("vLLM 在 CANN 上的推理优化", read_kv: position t of a
 * sequence lives at offset t % block_size of block table[t / block_size]).
 * The attention calls never do this (the paged design avoids the gathered
 * copy); it exists to check the index translation byte for byte.
 *   k_out, v_out  [cu_seq_lens[num_seqs], num_kv_heads, head_dim], device
 *   cu_seq_lens   device int32 [num_seqs + 1], exclusive prefix sum of seq_lens
 *   elem_bytes    2 (fp16/bf16 pools, [num_blocks, 16, num_kv_heads, head_dim])
 *                 or 1 (FP8 pools, head-major [num_blocks, num_kv_heads, 16,
 *                 head_dim]); the output rows are token-major either way
 * Row b, t receives cache[table[b][t / 16], t % 16] for t < seq_lens[b]
 * (for FP8 pools, cache[table[b][t / 16], h, t % 16] for each head h).  A
 * table entry outside [0, num_blocks) zero-fills its rows and sets
 * PA_DEVERR_BLOCK_ID; a length that disagrees with cu_seq_lens or exceeds the
 * table sets PA_DEVERR_SEQ_LEN and skips the sequence.
 */
int pa_paged_kv_gather(void* k_out, void* v_out, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                       const int32_t* cu_seq_lens, int num_seqs, int max_seq_len, int num_blocks,
                       int num_kv_heads, int head_dim, int elem_bytes, void* stream);

/*
 * Copy whole blocks of both pools, the copy-on-write step of a shared block
 * ("vLLM-Ascend 原理", section 2.1: sequences that share a prefix point at
 * the same physical blocks and copy before they diverge).  For each i,
 * block pairs[2i+1] of k_cache and v_cache receives the bytes of block
 * pairs[2i].  pairs is a device int32 array [num_pairs, 2]; no destination may
 * also be a source in the same call.  A block is 16 * num_kv_heads * head_dim
 * elements of elem_bytes bytes (2 for fp16/bf16, 1 for an FP8 cache).  Ids
 * outside [0, num_blocks) skip the pair and set PA_DEVERR_BLOCK_ID.
 */
int pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs, int num_blocks,
                   int num_kv_heads, int head_dim, int elem_bytes, void* stream);

/* Workspace for pa_paged_attention_prefill over num_seqs sequences and
 * num_tokens query rows: the chunk tile work list (num_seqs + 1 int32 offsets
 * and a cost-sorted list of num_tokens / 4 + num_seqs int32), the
 * decode kernel's work list, and the split-context partials of up to
 * min(num_tokens, PA_VERIFY_MAX_Q * num_seqs) query rows of decode and verify
 * chunks (partitions of pa_decode_partition(max_seq_len, 0) tokens).  Nonzero whenever
 * num_seqs > 0; 0 for a negative argument. */
size_t pa_prefill_workspace_bytes(int num_seqs, int num_tokens, int num_q_heads, int head_dim,
                                  int max_seq_len);

/*
 * Causal attention of query chunks appended onto a cached prefix, as in
 * chunked prefill ("vLLM-Ascend 原理", section 2.3 "因果自注意力": the query
 * at position i sees positions 0..i; section 2.4: a later chunk reads the KV
 * that earlier chunks wrote).  Query row cu_q_lens[b] + i of sequence b sits
 * at position seq_lens[b] - q_len_b + i.  Sequences with 1 <= q_len <=
 * PA_VERIFY_MAX_Q run through the decode kernel: single-query decodes, and the
 * speculative-decoding verify step, where the k draft tokens and the last
 * accepted one form a mini-prefill of q_len = k + 1 queries ("vLLM-Ascend
 * 原理", section 4 "推测解码").  Longer chunks run through the tensor-core
 * prefill kernel.  The new tokens' k/v must already be in the cache
 * (pa_paged_kv_write first).  Rolling back rejected drafts needs no call:
 * lowering seq_lens[b] hides every position at or past it, and the next
 * write overwrites those slots.
 *   out, q        [num_tokens, num_q_heads, head_dim]; num_tokens = cu_q_lens[num_seqs]
 *   max_q_len, max_seq_len  host-side upper bounds (grid sizing, routing).
 *   workspace     >= pa_prefill_workspace_bytes(num_seqs, num_tokens, ...) bytes,
 *                 256-byte aligned.
 * Errors on the device set PA_DEVERR_SEQ_LEN: a decode/verify chunk longer
 * than its seq_len or than max_q_len gets zero rows; a longer chunk that
 * exceeds its seq_len is left unwritten; a chunk whose rows fall outside
 * 0 .. num_tokens - 1 (cu_q_lens inconsistent with num_tokens) is neither
 * read nor written.
 * The call only enqueues work on `stream` (the prefill and decode kernels may
 * run side by side inside it); work queued after it on the same stream sees
 * every output row.
 */
int pa_paged_attention_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* seq_lens, const int32_t* cu_q_lens, int num_seqs,
                               int num_tokens, int max_q_len, int max_seq_len, int num_blocks,
                               float scale, int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, void* workspace, size_t workspace_bytes, int dtype,
                               void* stream);

/*
 * FP8 (E4M3) KV cache ("vLLM-Ascend 原理", section 4 "量化": k and v are
 * quantised to 8 bits as they are written and dequantised after they are read
 * through the block table; the cache takes half the HBM and half the bytes
 * per decode step).  Codes are OCP E4M3 ("FN"), one byte per element; one
 * fp32 scale per pool: value = code * scale.  head_dim must be 128.
 *
 * FP8 pools are head-major: [num_blocks, num_kv_heads, block_size, head_dim],
 * so the 16 rows of one (block, kv head) tile are one contiguous 2 KB run
 * (a 128-byte row per token would otherwise sit num_kv_heads * 128 bytes
 * from the next).  Slot s = block * 16 + offset holds head h's codes at
 * cache[s / 16][h][s % 16][:].  pa_copy_blocks moves whole blocks and works
 * on either layout; pa_paged_kv_gather reads FP8 pools in this order.
 *
 * pa_paged_kv_write_fp8 stores code = e4m3(float(x) * (1.0f / scale)) for each
 * new element x (fp16/bf16 `src_dtype`): one fp32 multiply, round to nearest
 * even, saturating at +-448, NaN kept.  Other arguments as pa_paged_kv_write.
 */
int pa_paged_kv_write_fp8(const void* key, const void* value, void* k_cache, void* v_cache,
                          const int64_t* slot_mapping, int num_tokens, int num_blocks, int num_kv_heads,
                          int head_dim, int block_size, int src_dtype, float k_scale, float v_scale,
                          void* stream);

/*
 * Decode attention over an FP8 cache: as pa_paged_attention_decode with
 * k_t = code * k_scale and v_t = code * v_scale; q and out keep `dtype`
 * (fp16/bf16); the workspace is sized by pa_decode_workspace_bytes.
 */
int pa_paged_attention_decode_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* seq_lens, int num_seqs, int max_seq_len, int num_blocks,
                                  float scale, float k_scale, float v_scale, int num_q_heads,
                                  int num_kv_heads, int head_dim, int block_size, int partition_size,
                                  void* workspace, size_t workspace_bytes, int dtype, void* stream);

/*
 * A continuous-batching step over an FP8 cache ("vLLM-Ascend 原理", section 4
 * "量化": the cache itself is quantised, so every row kind reads it through
 * the block table and dequantises it; section 4 "推测解码" for the verify
 * rows): as pa_paged_attention_prefill with k_t = code * k_scale and
 * v_t = code * v_scale over the head-major E4M3 pools described above.
 * head_dim must be 128; q and out keep `dtype`.  Rows of at most
 * PA_VERIFY_MAX_Q queries read the codes like pa_paged_attention_decode_fp8.
 * For longer chunks a kernel first widens every block of the chunk's
 * sequence to 16-bit values of `dtype` in the workspace (exact: every E4M3
 * value is an fp16 and a bf16 value; the scales are applied as above), and
 * the tensor-core prefill kernel reads that copy like a 16-bit cache.
 *   workspace  >= pa_prefill_fp8_workspace_bytes(..., chunk_kv_tokens) bytes,
 *              256-byte aligned (pa_prefill_workspace_bytes suffices when
 *              max_q_len <= PA_VERIFY_MAX_Q: there is no chunk to copy).
 *              Chunks take copy blocks in sequence order; from the first
 *              chunk whose blocks do not fit in the rest of the workspace on,
 *              every chunk is skipped (its rows are left unwritten) and
 *              PA_DEVERR_WORKSPACE is set.
 */
/* Workspace bytes for pa_paged_attention_prefill_fp8: those of
 * pa_prefill_workspace_bytes, plus the chunks' 16-bit copy (a table of
 * num_seqs * max_blocks_per_seq block ids, and 2 * 16 * num_kv_heads *
 * head_dim * 2 bytes per copied block).  chunk_kv_tokens = the sum of
 * seq_lens[b] over the sequences with more than PA_VERIFY_MAX_Q new tokens
 * (a chunk copies ceil(seq_len / 16) blocks); any larger value is also fine.
 * 0 for a non-positive size or a negative argument. */
size_t pa_prefill_fp8_workspace_bytes(int num_seqs, int num_tokens, int num_q_heads, int num_kv_heads,
                                      int head_dim, int max_seq_len, int max_blocks_per_seq,
                                      int64_t chunk_kv_tokens);

int pa_paged_attention_prefill_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* seq_lens, const int32_t* cu_q_lens, int num_seqs,
                                   int num_tokens, int max_q_len, int max_seq_len, int num_blocks,
                                   float scale, float k_scale, float v_scale, int num_q_heads,
                                   int num_kv_heads, int head_dim, int block_size, void* workspace,
                                   size_t workspace_bytes, int dtype, void* stream);

/*
 * Decode attention for callers that cannot allocate device memory.
 *
 * No counterpart in the pages: this is a deployment variant of
 * pa_paged_attention_decode.  Some callers cannot call cudaMalloc when they
 * run a step: an inference runtime that handed all remaining HBM to its own
 * pool (the KV block pool usually takes everything left) and so has nothing
 * to give a library, or a plugin inside a host framework whose interface
 * forbids device allocation by extensions.  This entry point takes the same
 * arguments as pa_paged_attention_decode minus the workspace and keeps the
 * split-context partials in a fixed scratch array of PA_NOALLOC_SCRATCH_BYTES
 * that the library holds on each GPU, once reserved there (below), until the
 * process exits.  It calls no cudaMalloc, cudaFree or other allocating
 * routine.
 *
 *  - Sizes whose partials need more than PA_NOALLOC_SCRATCH_BYTES
 *    (pa_decode_workspace_bytes(...) > PA_NOALLOC_SCRATCH_BYTES) are rejected
 *    with PA_ERR_WORKSPACE_TOO_SMALL before anything is launched.
 *  - The first call on a device looks up that device's scratch address
 *    (once per device, with the device current); make that first call before
 *    any stream capture.  Under CUDA's lazy module loading (the default) that
 *    first call is also what reserves the PA_NOALLOC_SCRATCH_BYTES on the
 *    device, so a runtime that later gives all free HBM to its KV pool must
 *    make it before taking the memory.  A call with num_seqs == 0 does this
 *    set-up and nothing else (the other arguments are not read).  With
 *    eager loading the array is reserved when the library's code is loaded
 *    into the device's context.
 *  - Every call on a device shares the one scratch array and it keeps the
 *    last call's contents.  Nothing in it needs to start at zero (each call
 *    writes every partial before reading it), but calls whose work overlaps
 *    on the GPU (two streams, two host threads) race on it: serialise them.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u << 20)

int pa_paged_attention_decode_noalloc(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                                      int max_seq_len, int num_blocks, float scale,
                                      int num_q_heads, int num_kv_heads, int head_dim,
                                      int block_size, int partition_size, int dtype, void* stream);

/*
 * Failure-path self-test.  Enqueues a one-thread kernel that waits on an
 * mbarrier phase nothing ever completes, through the same bounded wait the
 * attention kernels use for their TMA copies and pipeline stages.  The wait
 * gives up after about one second of polling and records PA_DEVERR_TIMEOUT
 * in the device error word (read it with pa_get_device_error); the kernel
 * then returns normally, so the context stays usable.  Returns PA_OK once
 * enqueued.
 */
int pa_selftest_wait_timeout(void* stream);

/*
 * Read the device error word (PA_DEVERR_* bits) of the current device after
 * the work queued on `stream` has finished; `clear` != 0 resets it to 0.
 * This call synchronises the stream.
 */
int pa_get_device_error(int* code, int clear, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PAGEDATTN_H */
