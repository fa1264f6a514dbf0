// Internal (non-ABI) declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

// Device error word bits (mirrors the PA_DEVERR_* values of the public header).
#define PA_DEVERR_BLOCK_ID_ 1u
#define PA_DEVERR_SLOT_ 2u
#define PA_DEVERR_SEQ_LEN_ 4u
#define PA_DEVERR_TIMEOUT_ 8u
#define PA_DEVERR_WORKSPACE_ 16u

namespace pa {

// Launch `kern` with programmatic stream serialization: it may start before
// the preceding kernel of the stream has finished; it must call pdl_wait()
// before touching anything that kernel produces.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Rows of a varlen call whose chunk has 1..PA_VERIFY_MAX_Q_ queries (decode
// rows, speculative-verify rows) run in the decode kernel; longer chunks run
// in the prefill kernels.
#define PA_VERIFY_MAX_Q_ 8


struct DecodeParams {
    void* out;                    // [T, Hq, D] (T = B without cu_q_lens)
    const void* q;                // [T, Hq, D]
    const int32_t* block_tables;  // [B, max_blocks]
    const int32_t* seq_lens;      // [B]
    const int32_t* cu_q_lens;     // [B+1] or nullptr (row b = sequence b, one query each)
    float* ws_m;                  // [max_rows, Hq, max_parts] running max (log2 units)
    float* ws_l;                  // [max_rows, Hq, max_parts] running sum
    float* ws_acc;                // [max_rows, Hq, max_parts, D] unnormalised accumulator
    int32_t* units;               // [B * max_parts] (sequence << 16 | partition) work list
    int32_t* unit_count;          // number of entries in `units`
    int32_t* work_counter;        // next work item to claim (reset by the plan kernel)
    int32_t* row_base;            // [B] first partials row of a split sequence
    int32_t* rows;                // [max_rows] (sequence << 3 | query index) of every partials row
    int32_t* row_count;           // number of entries in `rows` (header of the workspace)
    unsigned int* err;            // device error word
    int num_seqs;
    int max_blocks;
    int max_seq_len;
    int num_blocks;
    int num_q_heads;
    int num_kv_heads;
    int head_dim;
    int group;                    // num_q_heads / num_kv_heads
    int partition_tokens;         // multiple of 16
    int max_parts;                // ceil(max_seq_len / partition_tokens)
    int max_q;                    // largest chunk handled here (1..PA_VERIFY_MAX_Q_)
    int max_rows;                 // partials rows available in the workspace
    int num_rows;                 // rows of q and out (num_seqs without cu_q_lens)
    int col_chunks;               // chunks of 8 or 16 (query, head) columns per (unit, kv head)
    float scale_log2;             // scale * log2(e) (times the K dequantisation scale for FP8)
    float v_scale;                // V dequantisation scale (1 for 16-bit caches)
    // 1: the plan kernel has already run (launched on its own) and the decode
    // kernel is launched right after a prefill kernel that allows dependent
    // launch; everything the decode kernel reads completed before that
    // prefill kernel started, so it does not wait for it
    int overlap;
};

struct PrefillParams {
    void* out;                    // [T, Hq, D]
    const void* q;                // [T, Hq, D]
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const int32_t* cu_q_lens;     // [B+1]
    unsigned int* err;
    int num_seqs;
    int max_blocks;
    int max_seq_len;
    int num_blocks;
    int num_q_heads;
    int num_kv_heads;
    int group;
    int q_per_tile;               // queries per tile: rows = q_per_tile * group <= 128
    float scale_log2;             // scale * log2(e) (times the K dequantisation scale for FP8)
    float v_scale;                // V dequantisation scale (1 for 16-bit caches)
    // when *decode_units > 0 (decode rows will run next to this kernel), only
    // the first overlap_ctas CTAs take prefill work; the others leave their SMs
    const int32_t* decode_units;
    int overlap_ctas;
    int pair_cap;                 // pair-list capacity of the plan (num_tokens / 4 + num_seqs)
};

// FP8 (E4M3) cache: the prefill chunks' blocks widened to a 16-bit copy in
// the workspace, which the tensor-core kernel reads like a 16-bit cache.  The
// plan lists each chunk whose copy fits (`chunk_seq`, with its first copy
// block in `chunk_base`); sequence b's block i goes to copy block
// chunk_base[k] + i, recorded in row b of `table` (-1: not loaded).
struct Fp8Copy {
    int32_t* hdr;                 // [0] chunks listed, [1] copy blocks in use
    int32_t* chunk_seq;           // [num_seqs]
    int32_t* chunk_base;          // [num_seqs]
    int32_t* table;               // [num_seqs, max_blocks] copy block ids (rows of listed chunks)
    void* k16;                    // [cap_blocks, 16, Hkv, D] of the query type
    void* v16;
    int cap_blocks;
    const void* k_codes;          // the caller's E4M3 pools [num_blocks, Hkv, 16, D]
    const void* v_codes;
    const int32_t* src_tables;    // the caller's block table [num_seqs, max_blocks]
    int src_num_blocks;
};

// Launchers (return cudaError_t of the launch).
cudaError_t launch_slot_mapping(int64_t* slots, const int32_t* block_tables, int max_blocks,
                                const int32_t* seq_lens, const int32_t* cu_q_lens, int num_seqs,
                                int num_tokens, int num_blocks, unsigned int* err, cudaStream_t s);
cudaError_t launch_kv_write(const void* key, const void* value, void* k_cache, void* v_cache,
                            const int64_t* slots, int num_tokens, int num_blocks, int num_kv_heads,
                            int head_dim, unsigned int* err, cudaStream_t s);
cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          int head_dim, int dtype, cudaStream_t s);
// The work-list plan alone (for p.overlap launches, which skip it).
cudaError_t launch_decode_plan(const DecodeParams& p, cudaStream_t s);
int sm_count();
// FP8 (E4M3) cache, head_dim 128; q/out of `dtype`.
cudaError_t launch_decode_fp8(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                              int dtype, cudaStream_t s);
cudaError_t launch_kv_write_fp8(const void* key, const void* value, void* k_cache, void* v_cache,
                                const int64_t* slots, int num_tokens, int num_blocks, int num_kv_heads,
                                int src_dtype, float k_inv_scale, float v_inv_scale, unsigned int* err,
                                cudaStream_t s);
// pairs: device int32 [num_pairs, 2] (source block, destination block).
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs, int num_blocks,
                               int64_t block_bytes, unsigned int* err, cudaStream_t s);
cudaError_t launch_kv_gather(void* k_out, void* v_out, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                             const int32_t* cu_seq_lens, int num_seqs, int num_blocks, int64_t row_bytes,
                             int64_t head_major_row_bytes, int max_seq_len, unsigned int* err, cudaStream_t s);
// One-thread kernel whose bounded mbarrier wait runs out (records a timeout).
cudaError_t launch_wait_selftest(unsigned int* err, cudaStream_t s);
// tcgen05 prefill: groups of 1 to PA_MAX_GROUP q heads per kv head; q_per_tile = 128 / group.
// `plan` is device scratch of num_seqs + 1 + 2 * pair_cap int32 (the work list
// of query-tile pairs).  With `copy` (FP8 cache, head_dim 128) the plan also
// lists the chunks' copy blocks, a kernel widens them, and K and V come from
// the copy: p.block_tables = copy->table, p.num_blocks = copy->cap_blocks,
// kmap / vmap over copy->k16 / v16.
cudaError_t launch_prefill_tc(const PrefillParams& p, int32_t* plan, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, const CUtensorMap& qmap, int head_dim, int dtype,
                              int max_q_len, int num_tokens, const Fp8Copy* copy, cudaStream_t s);

}  // namespace pa
