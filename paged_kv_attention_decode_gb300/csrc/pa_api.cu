// C ABI of libpagedattn.so: argument validation, tensor-map set-up, launches.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "pa_internal.h"
#include "pagedattn.h"

namespace {

// Device error word: kernels OR PA_DEVERR_* bits into it.
__device__ unsigned int g_pa_device_error;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_err_addr[kMaxDevices] = {};

unsigned int* error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pa_device_error) != cudaSuccess) return nullptr;
        g_err_addr[dev] = static_cast<unsigned int*>(p);
    }
    return g_err_addr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tensor map over one pool [num_blocks * 16 token rows, Hkv, D] viewed as 4-D
// (64-element row piece, D/64 pieces, head, token slot); one box = one 64-dim
// half of the 16 rows of one (block, head), 128-byte swizzled.
bool make_kv_map(CUtensorMap* map, const void* base, int num_blocks, int num_kv_heads, int head_dim, int dtype) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(head_dim / 64), static_cast<cuuint64_t>(num_kv_heads),
                                static_cast<cuuint64_t>(num_blocks) * 16};
    const cuuint64_t strides[3] = {128, static_cast<cuuint64_t>(head_dim) * 2,
                                   static_cast<cuuint64_t>(num_kv_heads) * head_dim * 2};
    const cuuint32_t box[4] = {64, 1, 1, 16};   // one 64-dim half of a (block, head) tile
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor map over one pool whose box is a whole (16-token block, head) tile:
// dims (64-element row piece, token slot, D/64 pieces, head) with strides
// Hkv*D*2, 128 B and D*2 bytes; one box {64, 16, D/64, 1} lands as
// [piece][token][128 B], 128-byte swizzled -- byte for byte what D/64 boxes
// of make_kv_map would write, in one TMA operation.
bool make_kv_map_block(CUtensorMap* map, const void* base, int num_blocks, int num_kv_heads, int head_dim,
                       int dtype) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(num_blocks) * 16, static_cast<cuuint64_t>(head_dim / 64),
                                static_cast<cuuint64_t>(num_kv_heads)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(num_kv_heads) * head_dim * 2, 128,
                                   static_cast<cuuint64_t>(head_dim) * 2};
    const cuuint32_t box[4] = {64, 16, static_cast<cuuint32_t>(head_dim / 64), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor map over the query rows [T, Hq, D] viewed as 4-D (64-element row
// piece, D/64 pieces, q head, token); one box = one 64-dim half of the `group`
// heads of `q_per_tile` consecutive tokens, i.e. q_per_tile * group <= 128
// rows of 128 bytes whose row index is token * group + head.
bool make_q_map(CUtensorMap* map, const void* q, int num_tokens, int num_q_heads, int head_dim, int group,
                int q_per_tile, int dtype) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(head_dim / 64), static_cast<cuuint64_t>(num_q_heads),
                                static_cast<cuuint64_t>(num_tokens)};
    const cuuint64_t strides[3] = {128, static_cast<cuuint64_t>(head_dim) * 2,
                                   static_cast<cuuint64_t>(num_q_heads) * head_dim * 2};
    const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(q_per_tile)};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                    const_cast<void*>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor map over a head-major FP8 pool [num_blocks, Hkv, 16 token rows, 128
// codes]: one box = the 16 rows of one (block, head), a contiguous 2 KB run,
// landing as 16 rows of 128 bytes, 128-byte swizzled.
bool make_kv_map_fp8(CUtensorMap* map, const void* base, int num_blocks, int num_kv_heads) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {128, 16, static_cast<cuuint64_t>(num_kv_heads), static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[3] = {128, 16 * 128, static_cast<cuuint64_t>(num_kv_heads) * 16 * 128};
    const cuuint32_t box[4] = {128, 16, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
size_t align256(size_t x) { return (x + 255u) & ~static_cast<size_t>(255u); }

constexpr int kMaxGrid = 65535;
// Share of the SMs the tcgen05 prefill keeps while decode rows run beside it.
#ifndef PA_OVERLAP_NUM
#define PA_OVERLAP_NUM 1
#endif
#ifndef PA_OVERLAP_DEN
#define PA_OVERLAP_DEN 4
#endif
constexpr int kOverlapPrefillNum = PA_OVERLAP_NUM;
constexpr int kOverlapPrefillDen = PA_OVERLAP_DEN;
// Over an FP8 cache the decode rows cost less (half the bytes) while the
// chunks cost the same (the kernel reads their 16-bit copy).
#ifndef PA_OVERLAP_NUM_FP8
#define PA_OVERLAP_NUM_FP8 1
#endif
#ifndef PA_OVERLAP_DEN_FP8
#define PA_OVERLAP_DEN_FP8 4
#endif
constexpr int kOverlapPrefillNumFp8 = PA_OVERLAP_NUM_FP8;
constexpr int kOverlapPrefillDenFp8 = PA_OVERLAP_DEN_FP8;
constexpr int kMaxPoolBlocks = (1 << 27) - 1;  // token-row coordinate stays below 2^31

int check_shape(int num_q_heads, int num_kv_heads, int head_dim, int block_size, int dtype, int num_blocks) {
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (block_size != PA_BLOCK_SIZE) return PA_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_kv_heads > kMaxGrid) return PA_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads) return PA_ERR_INVALID_ARG;
    if (num_q_heads / num_kv_heads > PA_MAX_GROUP) return PA_ERR_UNSUPPORTED;
    if (num_blocks <= 0 || num_blocks > kMaxPoolBlocks) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

int parts_for(int max_seq_len, int partition) {
    return max_seq_len > 0 ? (max_seq_len + partition - 1) / partition : 1;
}

// partition_size 0: PA_DEFAULT_PARTITION tokens, doubled (up to
// PA_MAX_AUTO_PARTITION) while a sequence of max_seq_len tokens would have more
// than PA_AUTO_MAX_PARTS partitions: long contexts then merge fewer partials
int effective_partition(int max_seq_len, int partition_size) {
    if (partition_size) return partition_size;
    int part = PA_DEFAULT_PARTITION;
    while (part < PA_MAX_AUTO_PARTITION && parts_for(max_seq_len, part) > PA_AUTO_MAX_PARTS) part *= 2;
    return part;
}

size_t partials_bytes(int num_seqs, int num_q_heads, int head_dim, int parts) {
    const size_t n = static_cast<size_t>(num_seqs) * num_q_heads * parts;
    return 2 * align256(n * sizeof(float)) + align256(n * head_dim * sizeof(float));
}

// Decode workspace:
//   [header 256 B: unit count @0, partials row count @64, work counter @128]
//   [unit list: num_seqs * parts int32]
//   when parts > 1: [row_base: num_seqs int32][rows: max_rows int32][partials of max_rows rows]
size_t decode_ws_bytes(int num_seqs, int max_rows, int num_q_heads, int head_dim, int parts) {
    size_t b = 256 + align256(static_cast<size_t>(num_seqs) * parts * sizeof(int32_t));
    if (parts > 1)
        b += align256(static_cast<size_t>(num_seqs) * sizeof(int32_t)) +
             align256(static_cast<size_t>(max_rows) * sizeof(int32_t)) +
             partials_bytes(max_rows, num_q_heads, head_dim, parts);
    return b;
}

void carve_workspace(pa::DecodeParams& p, void* ws) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    p.unit_count = reinterpret_cast<int32_t*>(base);
    p.row_count = reinterpret_cast<int32_t*>(base + 64);
    p.work_counter = reinterpret_cast<int32_t*>(base + 128);
    p.units = reinterpret_cast<int32_t*>(base + 256);
    base += 256 + align256(static_cast<size_t>(p.num_seqs) * p.max_parts * sizeof(int32_t));
    if (p.max_parts > 1) {
        p.row_base = reinterpret_cast<int32_t*>(base);
        base += align256(static_cast<size_t>(p.num_seqs) * sizeof(int32_t));
        p.rows = reinterpret_cast<int32_t*>(base);
        base += align256(static_cast<size_t>(p.max_rows) * sizeof(int32_t));
        const size_t n = static_cast<size_t>(p.max_rows) * p.num_q_heads * p.max_parts;
        p.ws_m = reinterpret_cast<float*>(base);
        p.ws_l = reinterpret_cast<float*>(base + align256(n * sizeof(float)));
        p.ws_acc = reinterpret_cast<float*>(base + 2 * align256(n * sizeof(float)));
    }
}

// Query rows of a varlen call that can need split-context partials: only
// chunks of at most PA_VERIFY_MAX_Q queries run in the decode kernel.
int verify_rows_bound(int num_seqs, int num_tokens) {
    const long long r = std::min<long long>(num_tokens, static_cast<long long>(num_seqs) * PA_VERIFY_MAX_Q);
    return static_cast<int>(r);
}

float scale_log2(float scale) { return scale * 1.4426950408889634f; }

}  // namespace

extern "C" {

int pa_version(void) { return 100; }

const char* pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_WORKSPACE_TOO_SMALL: return "PA_ERR_WORKSPACE_TOO_SMALL";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        default: return "PA_ERR_UNKNOWN";
    }
}

int pa_slot_mapping(int64_t* slot_mapping, const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* seq_lens, const int32_t* cu_q_lens, int num_seqs, int num_tokens,
                    int num_blocks, int block_size, void* stream) {
    if (num_seqs < 0 || num_tokens < 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
    if (block_size != PA_BLOCK_SIZE) return PA_ERR_UNSUPPORTED;
    if (num_blocks <= 0 || num_blocks > kMaxPoolBlocks) return PA_ERR_INVALID_ARG;
    if (!cu_q_lens && num_tokens != num_seqs) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!slot_mapping || !block_tables || !seq_lens) return PA_ERR_INVALID_ARG;
    unsigned int* err = error_word();
    if (!err) return PA_ERR_CUDA;
    cudaError_t e = pa::launch_slot_mapping(slot_mapping, block_tables, max_blocks_per_seq, seq_lens, cu_q_lens,
                                            num_seqs, num_tokens, num_blocks, err,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_paged_kv_write(const void* key, const void* value, void* k_cache, void* v_cache,
                      const int64_t* slot_mapping, int num_tokens, int num_blocks, int num_kv_heads,
                      int head_dim, int block_size, int dtype, void* stream) {
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (block_size != PA_BLOCK_SIZE) return PA_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0 || num_blocks > kMaxPoolBlocks)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    unsigned int* err = error_word();
    if (!err) return PA_ERR_CUDA;
    cudaError_t e = pa::launch_kv_write(key, value, k_cache, v_cache, slot_mapping, num_tokens, num_blocks,
                                        num_kv_heads, head_dim, err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_decode_partition(int max_seq_len, int partition_size) {
    if (max_seq_len < 0 || partition_size < 0 || partition_size % PA_BLOCK_SIZE) return -1;
    return effective_partition(max_seq_len, partition_size);
}

size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int max_seq_len,
                                 int partition_size) {
    if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_seq_len < 0 || partition_size < 0) return 0;
    const int part = effective_partition(max_seq_len, partition_size);
    return decode_ws_bytes(num_seqs, num_seqs, num_q_heads, head_dim, parts_for(max_seq_len, part));
}

// Everything a decode launch needs, prepared and validated on the host.
struct DecodeCall {
    pa::DecodeParams p;
    CUtensorMap kmap, vmap;
    int head_dim, dtype;
    bool fp8;
};

static int decode_prepare(DecodeCall& c, void* out, const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                          const int32_t* cu_q_lens, int num_seqs, int max_seq_len, int num_blocks, float scale,
                          int num_q_heads, int num_kv_heads, int head_dim, int partition_size, void* workspace,
                          size_t workspace_bytes, int dtype, int max_q, int max_rows, int num_rows, bool fp8 = false,
                          float k_scale = 1.f, float v_scale = 1.f) {
    const int part = effective_partition(max_seq_len, partition_size);
    const int parts = parts_for(max_seq_len, part);
    if (parts > 65535) return PA_ERR_INVALID_ARG;   // partition index is a 16-bit field of the work list
    const size_t need = decode_ws_bytes(num_seqs, max_rows, num_q_heads, head_dim, parts);
    if (!workspace || workspace_bytes < need) return PA_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned256(workspace)) return PA_ERR_INVALID_ARG;
    unsigned int* err = error_word();
    if (!err) return PA_ERR_CUDA;
    const bool maps_ok = fp8 ? make_kv_map_fp8(&c.kmap, k_cache, num_blocks, num_kv_heads) &&
                                   make_kv_map_fp8(&c.vmap, v_cache, num_blocks, num_kv_heads)
                             : make_kv_map_block(&c.kmap, k_cache, num_blocks, num_kv_heads, head_dim, dtype) &&
                                   make_kv_map_block(&c.vmap, v_cache, num_blocks, num_kv_heads, head_dim, dtype);
    if (!maps_ok) return PA_ERR_CUDA;
    pa::DecodeParams& p = c.p;
    p = pa::DecodeParams{};
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.cu_q_lens = cu_q_lens;
    p.err = err;
    p.num_seqs = num_seqs;
    p.max_blocks = max_blocks_per_seq;
    p.max_seq_len = max_seq_len;
    p.num_blocks = num_blocks;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.group = num_q_heads / num_kv_heads;
    p.partition_tokens = part;
    p.max_parts = parts;
    p.max_q = max_q;
    p.max_rows = max_rows;
    p.num_rows = num_rows;
    // (query, head) columns per work item: 8, or 16 once a row can have more
    const int cols = max_q * p.group;
    const int chunk = cols > 8 ? 16 : 8;
    p.col_chunks = (cols + chunk - 1) / chunk;
    p.scale_log2 = scale_log2(scale) * k_scale;
    p.v_scale = v_scale;
    carve_workspace(p, workspace);
    c.head_dim = head_dim;
    c.dtype = dtype;
    c.fp8 = fp8;
    return PA_OK;
}

static int decode_launch(const DecodeCall& c, cudaStream_t stream) {
    cudaError_t e = c.fp8 ? pa::launch_decode_fp8(c.p, c.kmap, c.vmap, c.dtype, stream)
                          : pa::launch_decode(c.p, c.kmap, c.vmap, c.head_dim, c.dtype, stream);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

static int decode_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                       const int32_t* cu_q_lens, int num_seqs, int max_seq_len, int num_blocks, float scale,
                       int num_q_heads, int num_kv_heads, int head_dim, int partition_size, void* workspace,
                       size_t workspace_bytes, int dtype, cudaStream_t stream, int max_q, int max_rows,
                       bool fp8 = false, float k_scale = 1.f, float v_scale = 1.f) {
    DecodeCall c;
    const int rc = decode_prepare(c, out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, cu_q_lens,
                                  num_seqs, max_seq_len, num_blocks, scale, num_q_heads, num_kv_heads, head_dim,
                                  partition_size, workspace, workspace_bytes, dtype, max_q, max_rows, num_seqs, fp8,
                                  k_scale, v_scale);
    return rc ? rc : decode_launch(c, stream);
}

int pa_paged_attention_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                              int num_seqs, int max_seq_len, int num_blocks, float scale, int num_q_heads,
                              int num_kv_heads, int head_dim, int block_size, int partition_size,
                              void* workspace, size_t workspace_bytes, int dtype, void* stream) {
    int rc = check_shape(num_q_heads, num_kv_heads, head_dim, block_size, dtype, num_blocks);
    if (rc) return rc;
    if (num_seqs < 0 || num_seqs > kMaxGrid || max_seq_len < 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
    if (partition_size < 0 || partition_size % PA_BLOCK_SIZE) return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
    return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, nullptr, num_seqs,
                       max_seq_len, num_blocks, scale, num_q_heads, num_kv_heads, head_dim, partition_size,
                       workspace, workspace_bytes, dtype, static_cast<cudaStream_t>(stream), 1, num_seqs);
}

// Prefill workspace: [tile work list, 256-aligned][decode-row partials].
// prefill plan: offsets (num_seqs + 1), the cost-sorted pair list and each
// pair's sequence (pair_cap entries each, pair_cap = num_tokens / 4 +
// num_seqs).  A pair
// is two tiles of at least 2 queries (128 rows / at most PA_MAX_GROUP = 64
// heads), so a chunk of q queries has at most q / 4 + 1 pairs.
static_assert(PA_MAX_GROUP <= 64, "the plan's pair bound assumes tiles of at least 2 queries");
static size_t plan_bytes(int num_seqs, int num_tokens) {
    const size_t pairs = static_cast<size_t>(num_tokens) / 4 + static_cast<size_t>(num_seqs);
    return align256((static_cast<size_t>(num_seqs) + 1 + 2 * pairs) * sizeof(int32_t));
}

int pa_paged_kv_write_fp8(const void* key, const void* value, void* k_cache, void* v_cache,
                          const int64_t* slot_mapping, int num_tokens, int num_blocks, int num_kv_heads,
                          int head_dim, int block_size, int src_dtype, float k_scale, float v_scale, void* stream) {
    if (src_dtype != PA_F16 && src_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (block_size != PA_BLOCK_SIZE || head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0 || num_blocks > kMaxPoolBlocks)
        return PA_ERR_INVALID_ARG;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    unsigned int* err = error_word();
    if (!err) return PA_ERR_CUDA;
    const float k_inv = 1.0f / k_scale;   // one fp32 division, as the quantiser's definition states
    const float v_inv = 1.0f / v_scale;
    cudaError_t e = pa::launch_kv_write_fp8(key, value, k_cache, v_cache, slot_mapping, num_tokens, num_blocks,
                                            num_kv_heads, src_dtype, k_inv, v_inv, err,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_paged_attention_decode_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                                  int num_seqs, int max_seq_len, int num_blocks, float scale, float k_scale,
                                  float v_scale, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                  int partition_size, void* workspace, size_t workspace_bytes, int dtype,
                                  void* stream) {
    int rc = check_shape(num_q_heads, num_kv_heads, head_dim, block_size, dtype, num_blocks);
    if (rc) return rc;
    if (head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_seqs > kMaxGrid || max_seq_len < 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
    if (partition_size < 0 || partition_size % PA_BLOCK_SIZE) return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale)) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
    return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, nullptr, num_seqs,
                       max_seq_len, num_blocks, scale, num_q_heads, num_kv_heads, head_dim, partition_size,
                       workspace, workspace_bytes, dtype, static_cast<cudaStream_t>(stream), 1, num_seqs, true,
                       k_scale, v_scale);
}

size_t pa_prefill_workspace_bytes(int num_seqs, int num_tokens, int num_q_heads, int head_dim, int max_seq_len) {
    if (num_seqs <= 0 || num_tokens < 0 || num_q_heads <= 0 || head_dim <= 0 || max_seq_len < 0) return 0;
    return plan_bytes(num_seqs, num_tokens) + decode_ws_bytes(num_seqs, verify_rows_bound(num_seqs, num_tokens), num_q_heads,
                                                  head_dim,
                                                  parts_for(max_seq_len, effective_partition(max_seq_len, 0)));
}

// FP8 varlen calls: after the 16-bit call's workspace, the chunks' 16-bit
// copy ([256 B header | chunk_seq | chunk_base | table | K copy | V copy],
// every part 256-byte aligned).  Copy blocks hold 16 rows of num_kv_heads *
// head_dim 16-bit values, for K and for V.
static size_t fp8_copy_fixed_bytes(int num_seqs, int max_blocks_per_seq) {
    return 256 + 2 * align256(static_cast<size_t>(num_seqs) * sizeof(int32_t)) +
           align256(static_cast<size_t>(num_seqs) * static_cast<size_t>(max_blocks_per_seq) * sizeof(int32_t));
}

static size_t fp8_copy_block_bytes(int num_kv_heads, int head_dim) {
    return 2 * static_cast<size_t>(PA_BLOCK_SIZE) * num_kv_heads * head_dim * 2;   // K and V
}

size_t pa_prefill_fp8_workspace_bytes(int num_seqs, int num_tokens, int num_q_heads, int num_kv_heads,
                                      int head_dim, int max_seq_len, int max_blocks_per_seq,
                                      int64_t chunk_kv_tokens) {
    if (num_seqs <= 0 || num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        max_seq_len < 0 || max_blocks_per_seq <= 0 || chunk_kv_tokens < 0)
        return 0;
    // each chunk rounds its length up to whole blocks: at most one partial
    // block per chunk, and at most num_tokens / (PA_VERIFY_MAX_Q + 1) chunks
    const int64_t chunks = std::min<int64_t>(num_seqs, num_tokens / (PA_VERIFY_MAX_Q + 1));
    int64_t blocks = (chunk_kv_tokens + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE + chunks;
    blocks = std::min<int64_t>(blocks, static_cast<int64_t>(num_seqs) * max_blocks_per_seq);
    blocks = std::min<int64_t>(blocks, kMaxPoolBlocks);
    return pa_prefill_workspace_bytes(num_seqs, num_tokens, num_q_heads, head_dim, max_seq_len) +
           fp8_copy_fixed_bytes(num_seqs, max_blocks_per_seq) +
           static_cast<size_t>(blocks) * fp8_copy_block_bytes(num_kv_heads, head_dim);
}

// Everything a varlen call does, for either cache type; arguments are
// validated by the entry points.
static int prefill_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                        const int32_t* cu_q_lens, int num_seqs, int num_tokens, int max_q_len, int max_seq_len,
                        int num_blocks, float scale, int num_q_heads, int num_kv_heads, int head_dim,
                        void* workspace, size_t workspace_bytes, int dtype, cudaStream_t s, bool fp8,
                        float k_scale, float v_scale) {
    const size_t pb = plan_bytes(num_seqs, num_tokens);
    const size_t base_bytes = pa_prefill_workspace_bytes(num_seqs, num_tokens, num_q_heads, head_dim, max_seq_len);
    if (!workspace || workspace_bytes < base_bytes) return PA_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned256(workspace)) return PA_ERR_INVALID_ARG;
    // FP8 chunks: room for the 16-bit copy of at least one block
    pa::Fp8Copy copy{};
    if (fp8 && max_q_len > PA_VERIFY_MAX_Q) {
        const size_t fixed = fp8_copy_fixed_bytes(num_seqs, max_blocks_per_seq);
        const size_t per = fp8_copy_block_bytes(num_kv_heads, head_dim);
        if (workspace_bytes < base_bytes + fixed + per) return PA_ERR_WORKSPACE_TOO_SMALL;
        const size_t cap = std::min<size_t>((workspace_bytes - base_bytes - fixed) / per, kMaxPoolBlocks);
        uint8_t* c = static_cast<uint8_t*>(workspace) + base_bytes;
        copy.hdr = reinterpret_cast<int32_t*>(c);
        c += 256;
        copy.chunk_seq = reinterpret_cast<int32_t*>(c);
        c += align256(static_cast<size_t>(num_seqs) * sizeof(int32_t));
        copy.chunk_base = reinterpret_cast<int32_t*>(c);
        c += align256(static_cast<size_t>(num_seqs) * sizeof(int32_t));
        copy.table = reinterpret_cast<int32_t*>(c);
        c += align256(static_cast<size_t>(num_seqs) * static_cast<size_t>(max_blocks_per_seq) * sizeof(int32_t));
        copy.k16 = c;
        copy.v16 = c + cap * (per / 2);
        copy.cap_blocks = static_cast<int>(cap);
        copy.k_codes = k_cache;
        copy.v_codes = v_cache;
        copy.src_tables = block_tables;
        copy.src_num_blocks = num_blocks;
    }
    int32_t* plan = static_cast<int32_t*>(workspace);
    const int group = num_q_heads / num_kv_heads;
    // decode rows (q_len == 1) and speculative-verify rows (q_len <= PA_VERIFY_MAX_Q)
    // through the decode kernel
    const int max_q = std::max(1, std::min(max_q_len, PA_VERIFY_MAX_Q));
    DecodeCall dc;
    int rc = decode_prepare(dc, out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, cu_q_lens,
                            num_seqs, max_seq_len, num_blocks, scale, num_q_heads, num_kv_heads, head_dim, 0,
                            static_cast<uint8_t*>(workspace) + pb, workspace_bytes - pb, dtype, max_q,
                            verify_rows_bound(num_seqs, num_tokens), num_tokens, fp8, k_scale, v_scale);
    if (rc) return rc;
    if (max_q_len <= PA_VERIFY_MAX_Q) return decode_launch(dc, s);
    unsigned int* err = error_word();
    pa::PrefillParams p{};
    p.out = out;
    p.q = q;
    p.block_tables = fp8 ? copy.table : block_tables;
    p.seq_lens = seq_lens;
    p.cu_q_lens = cu_q_lens;
    p.err = err;
    p.num_seqs = num_seqs;
    p.max_blocks = max_blocks_per_seq;
    p.max_seq_len = max_seq_len;
    p.num_blocks = fp8 ? copy.cap_blocks : num_blocks;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = group;
    p.scale_log2 = scale_log2(scale) * k_scale;
    p.v_scale = v_scale;
    CUtensorMap kmap, vmap;
    // tiles of 128 / group queries (every supported grouping) on the tcgen05
    // tensor cores, running beside the decode rows: the decode plan and the
    // prefill kernel go first; the decode kernel then starts on the SMs the
    // prefill kernel leaves free.  K comes in one box per 64-dim half of a
    // block, V in one box per block, from the 16-bit cache or (FP8 cache)
    // from the chunks' 16-bit copy.
    const void* kc = fp8 ? copy.k16 : k_cache;
    const void* vc = fp8 ? copy.v16 : v_cache;
    if (!make_kv_map(&kmap, kc, p.num_blocks, num_kv_heads, head_dim, dtype) ||
        !make_kv_map_block(&vmap, vc, p.num_blocks, num_kv_heads, head_dim, dtype))
        return PA_ERR_CUDA;
    p.q_per_tile = 128 / group;
    p.pair_cap = num_tokens / 4 + num_seqs;
    CUtensorMap qmap;
    if (!make_q_map(&qmap, q, num_tokens, num_q_heads, head_dim, group, p.q_per_tile, dtype)) return PA_ERR_CUDA;
    if (pa::launch_decode_plan(dc.p, s) != cudaSuccess) return PA_ERR_CUDA;
    p.decode_units = dc.p.unit_count;
    p.overlap_ctas = std::max(1, fp8 ? pa::sm_count() * kOverlapPrefillNumFp8 / kOverlapPrefillDenFp8
                                     : pa::sm_count() * kOverlapPrefillNum / kOverlapPrefillDen);
    if (pa::launch_prefill_tc(p, plan, kmap, vmap, qmap, head_dim, dtype, max_q_len, num_tokens,
                              fp8 ? &copy : nullptr, s) !=
        cudaSuccess)
        return PA_ERR_CUDA;
    dc.p.overlap = 1;
    return decode_launch(dc, s);
}

int pa_paged_attention_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                               const int32_t* cu_q_lens, int num_seqs, int num_tokens, int max_q_len,
                               int max_seq_len, int num_blocks, float scale, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size, void* workspace, size_t workspace_bytes, int dtype,
                               void* stream) {
    int rc = check_shape(num_q_heads, num_kv_heads, head_dim, block_size, dtype, num_blocks);
    if (rc) return rc;
    if (num_seqs < 0 || num_seqs > kMaxGrid || num_tokens < 0 || max_q_len < 0 || max_seq_len < 0 ||
        max_blocks_per_seq <= 0)
        return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || num_tokens == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !cu_q_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
    return prefill_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, cu_q_lens, num_seqs,
                        num_tokens, max_q_len, max_seq_len, num_blocks, scale, num_q_heads, num_kv_heads, head_dim,
                        workspace, workspace_bytes, dtype, static_cast<cudaStream_t>(stream), false, 1.f, 1.f);
}

int pa_paged_attention_prefill_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                                   const int32_t* cu_q_lens, int num_seqs, int num_tokens, int max_q_len,
                                   int max_seq_len, int num_blocks, float scale, float k_scale, float v_scale,
                                   int num_q_heads, int num_kv_heads, int head_dim, int block_size, void* workspace,
                                   size_t workspace_bytes, int dtype, void* stream) {
    int rc = check_shape(num_q_heads, num_kv_heads, head_dim, block_size, dtype, num_blocks);
    if (rc) return rc;
    if (head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_seqs > kMaxGrid || num_tokens < 0 || max_q_len < 0 || max_seq_len < 0 ||
        max_blocks_per_seq <= 0)
        return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale)) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || num_tokens == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !cu_q_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
    return prefill_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, cu_q_lens, num_seqs,
                        num_tokens, max_q_len, max_seq_len, num_blocks, scale, num_q_heads, num_kv_heads, head_dim,
                        workspace, workspace_bytes, dtype, static_cast<cudaStream_t>(stream), true, k_scale,
                        v_scale);
}

int pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs, int num_blocks,
                   int num_kv_heads, int head_dim, int elem_bytes, void* stream) {
    if (num_pairs < 0 || num_blocks <= 0 || num_blocks > kMaxPoolBlocks || num_kv_heads <= 0 || head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    if (elem_bytes != 1 && elem_bytes != 2) return PA_ERR_UNSUPPORTED;
    const int64_t block_bytes = static_cast<int64_t>(PA_BLOCK_SIZE) * num_kv_heads * head_dim * elem_bytes;
    if (block_bytes % 16) return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (!k_cache || !v_cache || !pairs || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
    unsigned int* err = error_word();
    if (!err) return PA_ERR_CUDA;
    cudaError_t e = pa::launch_copy_blocks(k_cache, v_cache, pairs, num_pairs, num_blocks, block_bytes, err,
                                           static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_paged_kv_gather(void* k_out, void* v_out, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                       const int32_t* cu_seq_lens, int num_seqs, int max_seq_len, int num_blocks, int num_kv_heads,
                       int head_dim, int elem_bytes, void* stream) {
    if (num_seqs < 0 || num_seqs > kMaxGrid || max_seq_len < 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
    if (num_blocks <= 0 || num_blocks > kMaxPoolBlocks || num_kv_heads <= 0 || head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    if (elem_bytes != 1 && elem_bytes != 2) return PA_ERR_UNSUPPORTED;
    const int64_t row_bytes = static_cast<int64_t>(num_kv_heads) * head_dim * elem_bytes;
    if (row_bytes % 16) return PA_ERR_UNSUPPORTED;
    // FP8 pools are head-major: each head's row of head_dim codes is moved in 16-byte chunks
    const int64_t head_major_row_bytes = elem_bytes == 1 ? head_dim : 0;
    if (head_major_row_bytes % 16) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    if (!k_out || !v_out || !k_cache || !v_cache || !block_tables || !seq_lens || !cu_seq_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(k_out) || !aligned16(v_out) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    unsigned int* err = error_word();
    if (!err) return PA_ERR_CUDA;
    cudaError_t e = pa::launch_kv_gather(k_out, v_out, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                                         cu_seq_lens, num_seqs, num_blocks, row_bytes, head_major_row_bytes,
                                         max_seq_len, err,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_selftest_wait_timeout(void* stream) {
    unsigned int* err = error_word();
    if (!err) return PA_ERR_CUDA;
    return pa::launch_wait_selftest(err, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_get_device_error(int* code, int clear, void* stream) {
    if (!code) return PA_ERR_INVALID_ARG;
    unsigned int* err = error_word();
    if (!err) return PA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int v = 0;
    if (cudaMemcpyAsync(&v, err, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return PA_ERR_CUDA;
    if (clear && cudaMemsetAsync(err, 0, sizeof v, s) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
    *code = static_cast<int>(v);
    return PA_OK;
}

}  // extern "C"
