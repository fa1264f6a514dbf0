// Slot addressing and the KV-cache write (reshape_and_cache).
//
// "vLLM 在 CANN 上的推理优化", section "vLLM 的 PagedAttention 数据结构":
// a token's logical index splits into logical block (index / block_size) and
// offset (index % block_size); the block table gives the physical block; the
// token's slot is physical block * block_size + offset.  "vLLM-Ascend 原理"
// section 2.3 ("KV 写缓存") and 2.4 ("KV 追加写"): each new token's k and v are
// stored into that slot of the separate K and V pools.
#include <algorithm>

#include "pa_device.cuh"

namespace pa {

// One warp per sequence; lanes stride over the sequence's new tokens.
__global__ void __launch_bounds__(128) slot_mapping_kernel(int64_t* __restrict__ slots,
                                                           const int32_t* __restrict__ block_tables,
                                                           int max_blocks, const int32_t* __restrict__ seq_lens,
                                                           const int32_t* __restrict__ cu_q_lens, int num_seqs,
                                                           int num_blocks, unsigned int* err) {
    pdl_trigger();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= num_seqs) return;
    const int b = warp;
    const int n = seq_lens[b];
    int row0, ql;
    if (cu_q_lens) {
        row0 = cu_q_lens[b];
        ql = cu_q_lens[b + 1] - row0;
    } else {
        row0 = b;
        ql = 1;
    }
    if (ql <= 0) return;
    const bool seq_ok = n >= ql && n <= max_blocks * 16;
    // a decode row of length 0 pads a batch (to a captured bucket size): it
    // has no token to place, so its slot is -1 and nothing is flagged
    const bool padding = !cu_q_lens && n == 0;
    if (!seq_ok && !padding && lane == 0) record_error(err, PA_DEVERR_SEQ_LEN_);
    for (int i = lane; i < ql; i += 32) {
        int64_t slot = -1;
        if (seq_ok) {
            const int pos = n - ql + i;
            const int blk = block_tables[static_cast<int64_t>(b) * max_blocks + (pos >> 4)];
            if (blk >= 0 && blk < num_blocks)
                slot = static_cast<int64_t>(blk) * 16 + (pos & 15);
            else
                record_error(err, PA_DEVERR_BLOCK_ID_);
        }
        slots[row0 + i] = slot;
    }
}

// Each thread moves 16-byte chunks; chunk index = ((t * H) + h) * (D / 8) + c.
// K and V are handled by the same thread (two independent streams of loads).
template <int D>
__global__ void __launch_bounds__(256) kv_write_kernel(const uint4* __restrict__ key,
                                                       const uint4* __restrict__ value,
                                                       uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                       const int64_t* __restrict__ slots, int num_tokens,
                                                       int num_kv_heads, int64_t num_slots, unsigned int* err) {
    pdl_trigger();  // a following kernel that only reads inputs may overlap this one
    constexpr int CPR = D / 8;  // 16-byte chunks per (token, head) row
    const int64_t row_chunks = static_cast<int64_t>(num_kv_heads) * CPR;
    const int64_t total = static_cast<int64_t>(num_tokens) * row_chunks;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / row_chunks;
        const int64_t within = i - t * row_chunks;  // h * CPR + c
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (within == 0) record_error(err, PA_DEVERR_SLOT_);
            continue;
        }
        const int64_t dst = slot * row_chunks + within;
        const uint4 kv = __ldg(key + i);
        const uint4 vv = __ldg(value + i);
        k_cache[dst] = kv;
        v_cache[dst] = vv;
    }
}

// Quantising write into an FP8 (E4M3) cache ("vLLM-Ascend 原理", section 4
// "量化": k and v are quantised as they are written).  Each thread turns 16
// source values (fp16/bf16) into 16 codes: code = e4m3(float(x) * inv_scale),
// one fp32 multiply, round to nearest even, saturating at +-448.  The pools
// are head-major, [block][head][offset][128 codes]: the eight threads of one
// (token, head) row still store one whole 128-byte line.
template <typename T>
__global__ void __launch_bounds__(256) kv_write_fp8_kernel(const uint4* __restrict__ key,
                                                           const uint4* __restrict__ value,
                                                           uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                           const int64_t* __restrict__ slots, int num_tokens,
                                                           int num_kv_heads, int64_t num_slots, float k_inv,
                                                           float v_inv, unsigned int* err) {
    pdl_trigger();
    constexpr int D = 128;
    constexpr int CPR = D / 16;  // 16-code chunks per (token, head) row
    const int64_t row_chunks = static_cast<int64_t>(num_kv_heads) * CPR;
    const int64_t total = static_cast<int64_t>(num_tokens) * row_chunks;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / row_chunks;
        const int64_t within = i - t * row_chunks;
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (within == 0) record_error(err, PA_DEVERR_SLOT_);
            continue;
        }
        uint4 out[2];
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
            const uint4* src = kv ? value : key;
            const float inv = kv ? v_inv : k_inv;
            const uint4 a = __ldg(src + 2 * i);
            const uint4 b = __ldg(src + 2 * i + 1);
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            uint32_t codes[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 x0 = Elem<T>::to_float2(w[2 * j]);
                const float2 x1 = Elem<T>::to_float2(w[2 * j + 1]);
                const uint16_t lo = f32x2_to_e4m3x2(__fmul_rn(x0.x, inv), __fmul_rn(x0.y, inv));
                const uint16_t hi = f32x2_to_e4m3x2(__fmul_rn(x1.x, inv), __fmul_rn(x1.y, inv));
                codes[j] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            }
            out[kv] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
        }
        const int64_t h = within / CPR;
        const int64_t dst = (((slot >> 4) * num_kv_heads + h) * 16 + (slot & 15)) * CPR + (within - h * CPR);
        k_cache[dst] = out[0];
        v_cache[dst] = out[1];
    }
}

cudaError_t launch_kv_write_fp8(const void* key, const void* value, void* k_cache, void* v_cache,
                                const int64_t* slots, int num_tokens, int num_blocks, int num_kv_heads,
                                int src_dtype, float k_inv_scale, float v_inv_scale, unsigned int* err,
                                cudaStream_t s) {
    if (num_tokens == 0) return cudaSuccess;
    const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * 8;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 152LL * 16) blocks = 152LL * 16;
    const int64_t num_slots = static_cast<int64_t>(num_blocks) * 16;
    auto args = [&](auto kern) {
        kern<<<static_cast<int>(blocks), threads, 0, s>>>(
            static_cast<const uint4*>(key), static_cast<const uint4*>(value), static_cast<uint4*>(k_cache),
            static_cast<uint4*>(v_cache), slots, num_tokens, num_kv_heads, num_slots, k_inv_scale, v_inv_scale, err);
    };
    if (src_dtype == 0)
        args(kv_write_fp8_kernel<__half>);
    else
        args(kv_write_fp8_kernel<__nv_bfloat16>);
    return cudaGetLastError();
}

cudaError_t launch_slot_mapping(int64_t* slots, const int32_t* block_tables, int max_blocks,
                                const int32_t* seq_lens, const int32_t* cu_q_lens, int num_seqs,
                                int num_tokens, int num_blocks, unsigned int* err, cudaStream_t s) {
    (void)num_tokens;
    if (num_seqs == 0) return cudaSuccess;
    const int threads = 128;
    const int blocks = (num_seqs * 32 + threads - 1) / threads;
    slot_mapping_kernel<<<blocks, threads, 0, s>>>(slots, block_tables, max_blocks, seq_lens, cu_q_lens,
                                                   num_seqs, num_blocks, err);
    return cudaGetLastError();
}

cudaError_t launch_kv_write(const void* key, const void* value, void* k_cache, void* v_cache,
                            const int64_t* slots, int num_tokens, int num_blocks, int num_kv_heads,
                            int head_dim, unsigned int* err, cudaStream_t s) {
    if (num_tokens == 0) return cudaSuccess;
    const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * (head_dim / 8);
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = 152LL * 16;  // a few waves of the GPU; the loop strides the rest
    if (blocks > cap) blocks = cap;
    const int64_t num_slots = static_cast<int64_t>(num_blocks) * 16;
    if (head_dim == 128)
        kv_write_kernel<128><<<static_cast<int>(blocks), threads, 0, s>>>(
            static_cast<const uint4*>(key), static_cast<const uint4*>(value), static_cast<uint4*>(k_cache),
            static_cast<uint4*>(v_cache), slots, num_tokens, num_kv_heads, num_slots, err);
    else
        kv_write_kernel<64><<<static_cast<int>(blocks), threads, 0, s>>>(
            static_cast<const uint4*>(key), static_cast<const uint4*>(value), static_cast<uint4*>(k_cache),
            static_cast<uint4*>(v_cache), slots, num_tokens, num_kv_heads, num_slots, err);
    return cudaGetLastError();
}

// Copy whole blocks of both pools: the copy-on-write step of the block
// manager ("vLLM-Ascend 原理", section 2.1).  pairs[2i] -> pairs[2i+1].
// One CTA row per pair; its threads stride the block's 16-byte chunks of K
// and then of V.
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                          const int32_t* __restrict__ pairs, int num_pairs,
                                                          int num_blocks, int64_t chunks_per_block,
                                                          unsigned int* err) {
    pdl_trigger();
    for (int i = blockIdx.y; i < num_pairs; i += gridDim.y) {
        const int src = pairs[2 * i];
        const int dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (blockIdx.x == 0 && threadIdx.x == 0) record_error(err, PA_DEVERR_BLOCK_ID_);
            continue;
        }
        if (src == dst) continue;
        const int64_t s0 = static_cast<int64_t>(src) * chunks_per_block;
        const int64_t d0 = static_cast<int64_t>(dst) * chunks_per_block;
        for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < chunks_per_block;
             c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
            k_cache[d0 + c] = k_cache[s0 + c];
            v_cache[d0 + c] = v_cache[s0 + c];
        }
    }
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs, int num_blocks,
                               int64_t block_bytes, unsigned int* err, cudaStream_t s) {
    if (num_pairs == 0) return cudaSuccess;
    const int64_t chunks = block_bytes / 16;
    const int threads = 256;
    const int gx = static_cast<int>(std::min<int64_t>((chunks + threads - 1) / threads, 8));
    const int gy = std::min(num_pairs, 65535);
    copy_blocks_kernel<<<dim3(gx, gy), threads, 0, s>>>(static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                                                         pairs, num_pairs, num_blocks, chunks, err);
    return cudaGetLastError();
}

// Gather every live token row of each sequence through its block table into
// contiguous rows: out[cu_seq_lens[b] + t] = cache[table[b][t / 16], t % 16]
// ("vLLM 在 CANN 上的推理优化", read_kv: logical index -> block, offset).  One
// CTA row (blockIdx.y) per sequence; each warp moves whole token rows with
// 16-byte loads.  A table entry outside the pool zero-fills its rows.
// head_chunks > 0 reads a head-major pool ([block][head][offset][...], the
// FP8 layout) whose (token, head) rows are head_chunks 16-byte chunks long;
// 0 reads the token-major layout.
__global__ void __launch_bounds__(256) kv_gather_kernel(uint4* __restrict__ k_out, uint4* __restrict__ v_out,
                                                        const uint4* __restrict__ k_cache,
                                                        const uint4* __restrict__ v_cache,
                                                        const int32_t* __restrict__ block_tables, int max_blocks,
                                                        const int32_t* __restrict__ seq_lens,
                                                        const int32_t* __restrict__ cu_seq_lens, int num_blocks,
                                                        int row_chunks, int head_chunks, unsigned int* err) {
    const int b = blockIdx.y;
    int n = seq_lens[b];
    const int64_t base = cu_seq_lens[b];
    if (n < 0 || n > max_blocks * 16 || cu_seq_lens[b + 1] - base != n) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_error(err, PA_DEVERR_SEQ_LEN_);
        return;
    }
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < n; t += warps) {
        const int phys = block_tables[static_cast<int64_t>(b) * max_blocks + (t >> 4)];
        const bool ok = phys >= 0 && phys < num_blocks;
        if (!ok && lane == 0) record_error(err, PA_DEVERR_BLOCK_ID_);
        const int64_t dst = (base + t) * row_chunks;
        for (int c = lane; c < row_chunks; c += 32) {
            int64_t src;
            if (head_chunks > 0) {
                const int h = c / head_chunks;
                src = ((static_cast<int64_t>(phys) * (row_chunks / head_chunks) + h) * 16 + (t & 15)) * head_chunks +
                      (c - h * head_chunks);
            } else {
                src = (static_cast<int64_t>(phys) * 16 + (t & 15)) * row_chunks + c;
            }
            k_out[dst + c] = ok ? k_cache[src] : make_uint4(0, 0, 0, 0);
            v_out[dst + c] = ok ? v_cache[src] : make_uint4(0, 0, 0, 0);
        }
    }
}

cudaError_t launch_kv_gather(void* k_out, void* v_out, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                             const int32_t* cu_seq_lens, int num_seqs, int num_blocks, int64_t row_bytes,
                             int64_t head_major_row_bytes, int max_seq_len, unsigned int* err, cudaStream_t s) {
    if (num_seqs == 0) return cudaSuccess;
    const int threads = 256;
    const int gx = std::max(1, std::min((max_seq_len + 7) / 8, 64));   // 8 token rows per CTA pass
    kv_gather_kernel<<<dim3(gx, num_seqs), threads, 0, s>>>(
        static_cast<uint4*>(k_out), static_cast<uint4*>(v_out), static_cast<const uint4*>(k_cache),
        static_cast<const uint4*>(v_cache), block_tables, max_blocks, seq_lens, cu_seq_lens, num_blocks,
        static_cast<int>(row_bytes / 16), static_cast<int>(head_major_row_bytes / 16), err);
    return cudaGetLastError();
}

// Failure-path self-test: one thread waits on an mbarrier phase that nothing
// ever completes, through the same bounded wait as the attention kernels.
// The wait gives up (about a second) and the kernel records the timeout and
// returns normally.
__global__ void wait_selftest_kernel(unsigned int* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        if (!mbar_wait(&bar, 0)) record_error(err, PA_DEVERR_TIMEOUT_);
    }
}

cudaError_t launch_wait_selftest(unsigned int* err, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(err);
    return cudaGetLastError();
}

}  // namespace pa
