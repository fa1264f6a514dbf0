// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05).
//
// Causal attention of query chunks on their cached prefix ("vLLM-Ascend 原理",
// section 2.3 "因果自注意力": query at position i sees positions 0..i; section
// 2.4: a later chunk reads the KV earlier chunks wrote), for query groups of
// 1 to 64 heads per kv head (a tile holds 128 / G queries of G heads).
//
// One persistent CTA per SM.  A work item is a pair of adjacent 128-row query
// tiles, A and B (rows = (query, q head) pairs of one kv group; TMEM lane r =
// row r), that share one stream of 128-key K/V tiles: every K/V byte loaded
// feeds two tiles of MMAs.  A plan kernel sorts the pairs by cost and the
// CTAs deal them out in a snake (even totals); beside decode rows they take
// them round-robin instead.  One role per warpgroup for the whole kernel:
//   * warps 0-3: softmax of tile A, warps 4-7: softmax of tile B (thread r of
//     a group = row r), with 224 registers each (setmaxnreg) so that a row's
//     128 scores stay in registers;
//   * warp 8: every tcgen05.mma and tcgen05.commit, issued by one elected
//     lane of the converged warp (every lane computes the descriptors), and
//     each item's query tiles (TMA, once the previous item's MMAs are done);
//   * warps 9-11: the K and V tiles, gathered block by block through the
//     block table into a ring of K stages and a ring of V stages.  Each stage
//     belongs to one loader warp, whose eight lanes issue the boxes of a
//     tile's eight blocks together.  Warps 8-11 keep 56 registers.
// Tensor memory (512 columns): S_A | S_B (128 columns each) | O_A | O_B.
// Per key tile j and query tile X:
//   S_X(j) = Q_X K(j)^T   M=128 N=128, eight MMAs of K=16;
//   softmax_X(j)          one tcgen05.ld wait for the S row, exponentials
//                          against the running reference m_ref with paired
//                          fp32 instructions and the sum l (the row maximum
//                          only when the reference may have to move); P
//                          (bf16/fp16) is stored over the row's S;
//   O_X += P_X(j) V(j)    M=128 N=D, eight MMAs of K=16, A read from tensor
//                          memory.
// 128-key tiles (N=128 for S) halve the instructions, barrier waits and
// commits per key of 64-key ones.  S_X is single-buffered: S_X(j+1) is issued
// right behind P_X(j) V(j), which reads P_X(j) from the same columns (the
// MMAs of one thread execute in issue order), so while one tile's softmax
// runs, the tensor pipe works on the other tile (ping-pong).  K(j)'s
// stage is refilled once both S(j) are done, V(j)'s once both P V are
// (k_free / v_free, committed by the MMA warp).
// A row rescales O and l only when its maximum exceeds m_ref by more than 2^8
// (so P <= 256).  Only tiles that cross the causal diagonal are masked; V rows
// past the pair's last query position (or in blocks outside the pool) are
// cleared so that 0 * NaN cannot reach O.
#include <algorithm>
#include <type_traits>

#include "pa_device.cuh"

namespace pa {

namespace {

constexpr int kTcSoftmaxWarps = 4;                                   // per query tile
constexpr int kTcTiles = 2;                                          // query tiles per item (A, B)
constexpr int kTcMmaWarp = kTcTiles * kTcSoftmaxWarps;                // warp 8
constexpr int kTcLoaders = 3;                                        // warps 9-11
constexpr int kTcThreads = (kTcMmaWarp + 1 + kTcLoaders) * 32;      // 384
// Registers per thread: 168 at launch (65536 / 384, in steps of 8); the MMA
// and loader warpgroup gives up all but kTcOtherRegs, and the two softmax
// warpgroups take them (a whole row of 128 fp32 scores stays in registers).
constexpr int kTcLaunchRegs = 168;
constexpr int kTcOtherRegs = 56;
constexpr int kTcSoftmaxRegs = (kTcLaunchRegs * kTcThreads - kTcOtherRegs * (kTcThreads - 256)) / 256 / 8 * 8;   // 224
static_assert(kTcSoftmaxRegs * 256 + kTcOtherRegs * (kTcThreads - 256) <= kTcLaunchRegs * kTcThreads,
              "the warpgroups' registers must fit the launch pool");
constexpr int kTcKeys = 128;                                         // keys per K/V tile
constexpr int kTcBlocks = kTcKeys / 16;                               // cache blocks per tile
constexpr uint32_t kTmemCols = 512;  // S_A | S_B (128 each) | O_A | O_B
constexpr float kRescaleLog2 = 8.f;
constexpr float kPLazyMax = 256.f;   // 2^kRescaleLog2: a tile's sum of P below it needs no row maximum
constexpr unsigned kFullMask = 0xffffffffu;

template <int D>
struct TcShape {
    static constexpr int kKeyHalf = kTcKeys * 128;          // 128 keys x one 64-dim half
    // K or V of one tile: K as [half][key][128 B] (the S MMA's N = 128 keys
    // need one stride between 8-key groups), V as [block][half][16 keys][128 B]
    // (a P V MMA's K = 16 keys are one block: one box per block)
    static constexpr int kKV = (D / 64) * kKeyHalf;
    static constexpr int kQHalf = 128 * 128;                // 128 rows x one half
    static constexpr int kQ = (D / 64) * kQHalf;            // one query tile
    static constexpr int kBudget = 227 * 1024 - 1024;      // dynamic shared memory less alignment slack
    static constexpr int kRingFit = (kBudget - kTcTiles * kQ) / kKV;   // K and V stages together
    // K is needed one softmax earlier than V: the K ring gets the odd stage
    static constexpr int kVStages = kRingFit / 2 > 4 ? 4 : kRingFit / 2;          // 2 at D = 128, 4 at D = 64
    static constexpr int kKStages = kRingFit - kVStages > 4 ? 4 : kRingFit - kVStages;   // 3 at D = 128
    static constexpr int kSmem = kTcTiles * kQ + (kKStages + kVStages) * kKV + 1024;
};

// Per-warpgroup register budgets (every warp of the warpgroup executes the
// same call).  An increase waits until the CTA's pool (its threads x the
// registers per thread it was launched with) has the registers free.
template <uint32_t N>
__device__ __forceinline__ void reg_alloc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void reg_dealloc() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N));
}

// One elected lane of a converged warp issues (every lane computes the
// operands, so they stay warp-uniform).
__device__ __forceinline__ void el_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void el_mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void el_commit(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void el_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(smem_addr(bar)), "r"(bytes)
        : "memory");
}
__device__ __forceinline__ void el_tma_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                          int c3) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];\n\t}" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// Bounded mbarrier wait that also gives up when another thread of the CTA has
// already recorded a failure.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    uint64_t t0 = 0;
    for (uint32_t i = 0; i < kMaxWaitIters; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (wait_timed_out(i, t0)) return false;
        if ((i & 1023u) == 1023u && *abort_flag) return false;
    }
    return false;
}

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// Paired fp32 arithmetic (one instruction for two values on sm_100 and
// later), rounded to nearest like the scalar operations:
// (x, y) <- (x * s, y * s), (x + a, y + b), (x * s + a, y * s + a).
__device__ __forceinline__ void mul2(float& x, float& y, float s) {
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%0, %1};\n\tmov.b64 b, {%2, %2};\n\t"
        "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "+f"(x), "+f"(y)
        : "f"(s));
}
__device__ __forceinline__ void add2(float& x, float& y, float a, float b) {
    asm("{\n\t.reg .b64 p, q, d;\n\tmov.b64 p, {%0, %1};\n\tmov.b64 q, {%2, %3};\n\t"
        "add.rn.f32x2 d, p, q;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "+f"(x), "+f"(y)
        : "f"(a), "f"(b));
}
__device__ __forceinline__ void fma2(float& x, float& y, float s, float a) {
    asm("{\n\t.reg .b64 p, q, r, d;\n\tmov.b64 p, {%0, %1};\n\tmov.b64 q, {%2, %2};\n\t"
        "mov.b64 r, {%3, %3};\n\tfma.rn.f32x2 d, p, q, r;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "+f"(x), "+f"(y)
        : "f"(s), "f"(a));
}

// Key tiles a query-tile pair of a chunk reads: those of its last tile.
// Pair pr of a chunk of ql queries on a sequence of n tokens (tiles of qt rows).
__device__ __forceinline__ int pair_key_tiles(int n, int ql, int qt, int pr) {
    const int ntiles = (ql + qt - 1) / qt;
    const int last = min(2 * pr + 1, ntiles - 1);                 // the pair's last query tile
    const int q_last = min(ql, (last + 1) * qt) - 1;
    return (n - ql + q_last + kTcKeys) / kTcKeys;
}

// One 16-byte run of E4M3 codes (16 elements) widened to 16-bit values of
// type T: two 16-byte runs (exact: every E4M3 value is an fp16 and a bf16
// value).
template <typename T>
__device__ __forceinline__ void widen16(const uint4& in, uint4& lo, uint4& hi) {
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t h01 = e4m3x2_to_f16x2(static_cast<uint16_t>(w[j] & 0xffffu));
        const uint32_t h23 = e4m3x2_to_f16x2(static_cast<uint16_t>(w[j] >> 16));
        if constexpr (std::is_same<T, __half>::value) {
            o[2 * j] = h01;
            o[2 * j + 1] = h23;
        } else {
            const float2 a = Elem<__half>::to_float2(h01);
            const float2 b = Elem<__half>::to_float2(h23);
            o[2 * j] = Elem<T>::pack(a.x, a.y);
            o[2 * j + 1] = Elem<T>::pack(b.x, b.y);
        }
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Exclusive prefix sum of one value per thread over a 1024-thread block, plus
// the running total `carry` of earlier calls (updated).  Every thread calls.
__device__ __forceinline__ int block_exclusive_scan_1024(int v, int* warp_tot, int* carry) {
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(kFullMask, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int t = warp_tot[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(kFullMask, t, off);
            if (lane >= off) t += y;
        }
        warp_tot[lane] = t;  // inclusive over warps
    }
    __syncthreads();
    const int before = *carry + (warp > 0 ? warp_tot[warp - 1] : 0);
    __syncthreads();
    if (tid == 1023) *carry = before + incl;
    __syncthreads();
    return before + incl - v;
}

// Cost classes of the plan's counting sort (key tiles of a pair, clamped).
constexpr int kPlanBuckets = 2048;
static_assert(kPlanBuckets == 2 * 1024, "the plan's class scan takes two classes per thread");

// Work list of the chunked-prefill items.  offsets[b] = number of query-tile
// pairs (two 128-row tiles) of sequences 0..b-1 whose chunk is longer than
// PA_VERIFY_MAX_Q_ tokens (shorter chunks are decode or speculative-verify
// rows and belong to the decode kernel); offsets[B] = total.  order[0 ..
// total) = the global pair indices sorted by the number of key tiles they
// read, longest first (a counting sort; the order within a cost class is
// arbitrary and does not affect any result).  seq_of_pair[l] = the sequence
// of global pair l, so that an item finds its sequence with one load.  The
// pair lists hold at most pair_cap = num_tokens / 4 + num_seqs entries.
// With an FP8 copy (copy.hdr non-null) each chunk with pairs also gets
// ceil(seq_len / 16) consecutive copy blocks, in sequence order; a chunk
// whose blocks would pass copy.cap_blocks (and so every later chunk) gets
// neither blocks nor pairs (its rows are left unwritten) and sets
// PA_DEVERR_WORKSPACE.
// One CTA.
__global__ void __launch_bounds__(1024) prefill_plan_kernel(const int32_t* __restrict__ cu_q_lens,
                                                            const int32_t* __restrict__ seq_lens, int num_seqs,
                                                            int num_tokens, int q_per_tile,
                                                            int32_t* __restrict__ offsets, int pair_cap,
                                                            unsigned int* err, const Fp8Copy copy, int max_seq_len,
                                                            int max_blocks) {
    __shared__ int warp_tot[32];
    __shared__ int carry, blk_carry, chunk_carry, blk_end;
    __shared__ int hist[kPlanBuckets];
    int32_t* order = offsets + num_seqs + 1;
    int32_t* seq_of_pair = order + pair_cap;
    const int tid = threadIdx.x;
    if (tid == 0) carry = blk_carry = chunk_carry = blk_end = 0;
    for (int i = tid; i < kPlanBuckets; i += 1024) hist[i] = 0;
    __syncthreads();
    // the pairs of sequence b: count them (offsets) and their cost classes
    // (a chunk outside the num_tokens query rows has none: its rows cannot be
    // written, and the pair list stays within num_tokens / 4 + num_seqs)
    auto pairs_of = [&](int b, int& ql, int& n) {
        const int c0 = cu_q_lens[b], c1 = cu_q_lens[b + 1];
        ql = c1 - c0;
        n = seq_lens[b];
        if (c0 < 0 || c1 < c0 || c1 > num_tokens) {
            ql = 0;
            return 0;
        }
        const int tiles = ql > PA_VERIFY_MAX_Q_ ? (ql + q_per_tile - 1) / q_per_tile : 0;
        return (tiles + kTcTiles - 1) / kTcTiles;
    };
    auto bucket = [&](int n, int ql, int pr) {
        // a malformed sequence (skipped by the kernel) goes to class 0
        const int c = (n >= ql && ql > 0) ? pair_key_tiles(n, ql, q_per_tile, pr) : 0;
        return kPlanBuckets - 1 - max(0, min(c, kPlanBuckets - 1));   // longest first
    };
    for (int base = 0; base < num_seqs; base += 1024) {
        const int b = base + tid;
        int v = 0, ql = 0, n = 0;
        if (b < num_seqs) {
            v = pairs_of(b, ql, n);
            if (ql == 0 && cu_q_lens[b + 1] != cu_q_lens[b]) record_error(err, PA_DEVERR_SEQ_LEN_);
        }
        if (copy.hdr) {
            // the copy blocks of a chunk the kernel will read (a malformed
            // length is skipped there, and needs none)
            int nb = (v > 0 && n >= ql && n <= max_seq_len && n <= max_blocks * 16) ? (n + 15) >> 4 : 0;
            const int first = block_exclusive_scan_1024(nb, warp_tot, &blk_carry);
            if (nb > 0 && first + nb > copy.cap_blocks) {
                record_error(err, PA_DEVERR_WORKSPACE_);
                nb = 0;
                v = 0;
            }
            const int k = block_exclusive_scan_1024(nb > 0 ? 1 : 0, warp_tot, &chunk_carry);
            if (nb > 0) {
                copy.chunk_seq[k] = b;
                copy.chunk_base[k] = first;
                atomicMax(&blk_end, first + nb);
            }
        }
        if (b < num_seqs)
            for (int pr = 0; pr < v; ++pr) atomicAdd(&hist[bucket(n, ql, pr)], 1);
        const int start = block_exclusive_scan_1024(v, warp_tot, &carry);
        if (b < num_seqs) {
            offsets[b] = start;
            for (int pr = 0; pr < v; ++pr) seq_of_pair[start + pr] = b;
        }
    }
    if (tid == 0) {
        offsets[num_seqs] = carry;
        if (copy.hdr) {
            copy.hdr[0] = chunk_carry;
            copy.hdr[1] = blk_end;
        }
    }
    __syncthreads();
    // bucket starts (exclusive scan of the histogram, two classes per thread)
    if (tid == 0) carry = 0;
    __syncthreads();
    {
        const int h0 = hist[2 * tid], h1 = hist[2 * tid + 1];
        const int start = block_exclusive_scan_1024(h0 + h1, warp_tot, &carry);
        __syncthreads();
        hist[2 * tid] = start;
        hist[2 * tid + 1] = start + h0;
    }
    __syncthreads();
    // scatter each pair's global index to its class (the pair counts from
    // offsets: a chunk without copy blocks has none)
    for (int b = tid; b < num_seqs; b += 1024) {
        int ql = 0, n = 0;
        (void)pairs_of(b, ql, n);
        const int first = offsets[b];
        const int v = offsets[b + 1] - first;
        for (int pr = 0; pr < v; ++pr) {
            // the kernel's pair index l within the sequence counts from the last pair
            const int l = first + (v - 1 - pr);
            order[atomicAdd(&hist[bucket(n, ql, pr)], 1)] = l;
        }
    }
}

// FP8 (E4M3) cache: the blocks of the chunks the plan listed, widened to
// 16-bit rows of the query type in the workspace copy [cap, 16, Hkv, D]
// (token-major, like a 16-bit cache), which the kernel below then reads
// through copy.table.  The conversion is exact (every E4M3 value is an fp16
// and a bf16 value); the scales stay folded into the softmax scale and the
// epilogue.  Copy block u belongs to the last listed chunk k with
// chunk_base[k] <= u; one CTA widens its K and V rows of every kv head (the
// (block, kv head) runs of the head-major pools are 2 KB apart).
constexpr int kWidenThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kWidenThreads) widen_chunk_blocks_kernel(const Fp8Copy c,
                                                                           const int32_t* __restrict__ seq_lens,
                                                                           int max_blocks, int num_kv_heads) {
    constexpr int D = 128;
    const int nchunks = c.hdr[0];
    const int used = min(c.hdr[1], c.cap_blocks);
    const int runs = num_kv_heads * 16 * (D / 16);   // 16-code runs per block and pool
    for (int u = blockIdx.x; u < used && nchunks > 0; u += gridDim.x) {
        int lo = 0, hi = nchunks - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (c.chunk_base[mid] <= u) lo = mid;
            else hi = mid - 1;
        }
        const int b = c.chunk_seq[lo];
        const int i = u - c.chunk_base[lo];
        if (i < 0 || i >= ((seq_lens[b] + 15) >> 4)) continue;
        const int src = c.src_tables[static_cast<int64_t>(b) * max_blocks + i];
        const bool ok = src >= 0 && src < c.src_num_blocks;   // else the kernel flags and masks it
        if (threadIdx.x == 0) c.table[static_cast<int64_t>(b) * max_blocks + i] = ok ? u : -1;
        if (!ok) continue;
        const int64_t src_off = static_cast<int64_t>(src) * num_kv_heads * 16 * D;
        const int64_t dst_off = static_cast<int64_t>(u) * 16 * num_kv_heads * D;
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
            const uint8_t* sp = static_cast<const uint8_t*>(kv ? c.v_codes : c.k_codes) + src_off;
            T* dp = static_cast<T*>(kv ? c.v16 : c.k16) + dst_off;
            for (int x = threadIdx.x; x < runs; x += kWidenThreads) {
                const int row = x >> 3, ch = x & 7;     // row = h * 16 + t of the head-major block
                const int h = row >> 4, t = row & 15;
                const uint4 in = __ldcs(reinterpret_cast<const uint4*>(sp + row * D + ch * 16));
                uint4 lo4, hi4;
                widen16<T>(in, lo4, hi4);
                uint4* o = reinterpret_cast<uint4*>(dp + (t * num_kv_heads + h) * D + ch * 16);
                o[0] = lo4;
                o[1] = hi4;
            }
        }
    }
}

// Persistent: work item w = (rank, kv head) is pair order[rank] of the plan
// (pairs sorted by cost, longest first) for kv head w % num_kv_heads.  The
// CTAs deal the items out like cards in a snake: round k gives CTA i item
// k * C + i for even k and k * C + C - 1 - i for odd k, so the CTAs' total
// costs stay even.  (Beside decode rows: pair w / num_kv_heads of the plan's
// own order, round-robin.)
template <typename T, int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const PrefillParams p, const int32_t* __restrict__ plan,
                      const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap qmap) {
    using Sh = TcShape<D>;
    constexpr int NK = Sh::kKStages;
    constexpr int NV = Sh::kVStages;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t kIdescS = mma_idesc_f16(128, kTcKeys, kBf16, false);
    constexpr uint32_t kIdescPV = mma_idesc_f16(128, D, kBf16, true);

    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t k_full[NK];               // K tile landed (one arrival, by the stage's loader)
    __shared__ uint64_t v_full[NV];               // V tile landed (one arrival, by the stage's loader)
    __shared__ uint64_t k_free[NK];               // every S of the stage's tile complete
    __shared__ uint64_t v_free[NV];               // every P V of the stage's tile complete
    __shared__ uint64_t q_full;                   // the item's query tiles landed
    __shared__ uint64_t item_done;                // every MMA of an item complete
    // S_X(j) complete (one phase per tile of X).  S_X(j+1) is issued only
    // after P_X(j) was stored, which needs the softmax of tile j, so the
    // barrier never runs more than one phase ahead of a waiter.
    __shared__ uint64_t s_full[kTcTiles];
    // P_X(j) stored: one arrival per softmax warp.  A warp reaches tile j+1
    // only after S_X(j+1), which the MMA warp issues after it saw this phase
    // complete, so no warp arrives twice in one phase.
    __shared__ uint64_t p_full[kTcTiles];
    // o_done[X][0]: the last P_X V of an item complete, one phase per item
    // that has a tile X (its epilogue is the only waiter; an item's next phase
    // needs this item's softmax, which comes after the epilogue, so the
    // barrier never runs two phases ahead).  o_done[0][1]: drains every MMA in
    // flight on the abort path.
    __shared__ uint64_t o_done[kTcTiles][2];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int G = p.group;
    const int QT = p.q_per_tile;  // 128 / G
    // a decode kernel launched after this one may start now (it reads
    // nothing this kernel writes); when it has work, only overlap_ctas CTAs
    // stay, so that it gets the other SMs
    pdl_trigger();
    int ctas = static_cast<int>(gridDim.x);
    // Alone on the GPU, the CTAs take the items in the cost-sorted snake order
    // (even totals, the kernel ends together).  Beside decode rows, they take
    // them round-robin in plan order: CTAs that finish early hand their SMs to
    // the HBM-bound decode kernel sooner, which shortens the step more.
    const bool snake = !(p.decode_units && *p.decode_units > 0);
    if (!snake) ctas = min(ctas, p.overlap_ctas);
    const int total_items = plan[p.num_seqs] * p.num_kv_heads;
    if (static_cast<int>(blockIdx.x) >= total_items || static_cast<int>(blockIdx.x) >= ctas) return;

    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    auto qs = [&](int x) { return smem + x * Sh::kQ; };
    auto kst = [&](int s) { return smem + kTcTiles * Sh::kQ + s * Sh::kKV; };
    auto vst = [&](int s) { return smem + kTcTiles * Sh::kQ + (NK + s) * Sh::kKV; };

    // A tile holds q_per_tile queries x G heads <= 128 rows (fewer when G does
    // not divide 128).  The rows past them are never loaded: zero them once,
    // so their scores stay finite and quiet.
    const int q_rows = QT * G;
    const int q_tile_bytes = q_rows * 128 * (D / 64);
    if (q_rows < 128) {
        const int n16 = (128 - q_rows) * 8;   // 16-byte chunks past the loaded rows, per 64-dim half
        for (int i = tid; i < kTcTiles * (D / 64) * n16; i += kTcThreads) {
            const int half = i / n16;         // (tile, half) = smem + half * kQHalf
            reinterpret_cast<uint4*>(smem + half * Sh::kQHalf + q_rows * 128)[i - half * n16] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < NK; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_free[s], 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_free[s], 1);
        }
        mbar_init(&q_full, 1);
        mbar_init(&item_done, 1);
        for (int x = 0; x < kTcTiles; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], kTcSoftmaxWarps);
            mbar_init(&o_done[x][0], 1);
            mbar_init(&o_done[x][1], 1);
        }
        abort_flag = 0;
        fence_barrier_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;
    volatile int* abort_v = &abort_flag;

    // Work item w: (tile pair, kv head) of the plan; within a sequence the
    // pairs nearest the end (the longest key ranges) come first.  Query
    // tiles A (x = 0) and B (x = 1, absent past the chunk's last tile).
    struct Item {
        int g, row0, qlen, n, nkt, pos_pair, nblk_live;
        int q0[kTcTiles], nkx[kTcTiles], pos_lo[kTcTiles], pos_hi[kTcTiles];
        const int32_t* bt;
    };
    // false when the sequence is malformed: every role skips the item
    auto decode_item = [&](int w, Item& it) -> bool {
        it.g = w % p.num_kv_heads;
        const int l = snake ? plan[p.num_seqs + 1 + w / p.num_kv_heads] : w / p.num_kv_heads;
        const int b = plan[p.num_seqs + 1 + p.pair_cap + l];   // the pair's sequence
        it.row0 = p.cu_q_lens[b];
        it.qlen = p.cu_q_lens[b + 1] - it.row0;
        const int ntiles = (it.qlen + QT - 1) / QT;
        const int npairs = (ntiles + kTcTiles - 1) / kTcTiles;
        const int pr = npairs - 1 - (l - plan[b]);
        it.n = p.seq_lens[b];
        if (it.n < it.qlen || it.n > p.max_seq_len || it.n > p.max_blocks * 16) {
            if (pr == npairs - 1 && it.g == 0 && tid == 0) record_error(p.err, PA_DEVERR_SEQ_LEN_);
            return false;
        }
#pragma unroll
        for (int x = 0; x < kTcTiles; ++x) {
            const int qt = pr * kTcTiles + x;
            it.q0[x] = qt * QT;
            if (qt < ntiles) {
                const int q_last = min(it.qlen, it.q0[x] + QT) - 1;
                it.pos_lo[x] = it.n - it.qlen + it.q0[x];
                it.pos_hi[x] = it.n - it.qlen + q_last;
                it.nkx[x] = (it.pos_hi[x] + kTcKeys) / kTcKeys;
            } else {
                it.pos_lo[x] = it.pos_hi[x] = 0;
                it.nkx[x] = 0;
            }
        }
        it.nkt = max(it.nkx[0], it.nkx[1]);                          // key tiles of the pair
        it.pos_pair = it.nkx[1] ? it.pos_hi[1] : it.pos_hi[0];      // the pair's last query position
        it.nblk_live = (it.pos_pair + 16) >> 4;
        it.bt = p.block_tables + static_cast<int64_t>(b) * p.max_blocks;
        return true;
    };

    // the CTA's k-th item: kNoMoreItems past the end, -1 when round k has
    // none for this CTA (a partial last round)
    constexpr int kNoMoreItems = -2;
    auto item_at = [&](int k) -> int {
        const long long base = static_cast<long long>(k) * ctas;
        if (base >= total_items) return kNoMoreItems;
        const int i = static_cast<int>(blockIdx.x);
        const long long w = (snake && (k & 1)) ? base + ctas - 1 - i : base + i;
        return w < total_items ? static_cast<int>(w) : -1;
    };

    // running counters (identical in every role): key tiles loaded so far (the
    // ring position), tiles processed so far per query-tile slot, items so far
    int kv0 = 0;
    int t0[kTcTiles] = {0, 0};
    int items = 0;
    bool ok = true;
    auto next_item = [&](const Item& it) {
        kv0 += it.nkt;
        t0[0] += it.nkx[0];
        t0[1] += it.nkx[1];
        ++items;
        if (*abort_v) ok = false;
    };

    if (warp < kTcMmaWarp) {
        // ============================ softmax rows ============================
        // (warpgroups 0 and 1: the registers of a whole 128-score row)
        reg_alloc<kTcSoftmaxRegs>();
        const int x = warp / kTcSoftmaxWarps;
        const int wq = warp % kTcSoftmaxWarps;
        const int r = wq * 32 + lane;                       // row = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t s_tm = tmem + lane_base + static_cast<uint32_t>(x * kTcKeys);
        const uint32_t o_tm = tmem + lane_base + static_cast<uint32_t>(kTcTiles * kTcKeys + x * D);
        const bool fold = p.scale_log2 > 0.f;   // scale folded into the exponent's FMA
        int n_items_x = 0;   // items of this tile so far (o_done phases)
        for (int k = 0; ok; ++k) {
            const int w0 = item_at(k);
            if (w0 == kNoMoreItems) break;
            Item it;
            if (w0 < 0 || !decode_item(w0, it)) continue;
            const int nk = x ? it.nkx[1] : it.nkx[0];
            const int nk_a = it.nkx[0];
            const int q0 = x ? it.q0[1] : it.q0[0];
            const int pos_lo = x ? it.pos_lo[1] : it.pos_lo[0];
            const int pos_hi = x ? it.pos_hi[1] : it.pos_hi[0];
            const int tx0 = x ? t0[1] : t0[0];
            if (nk > 0) {
                const int qi_row = q0 + r / G;
                const bool row_ok = r < QT * G && qi_row < it.qlen;
                const int pos_row = row_ok ? it.n - it.qlen + qi_row : pos_hi;
                // does the item's live table hold an id outside the pool?  (One
                // scan per item keeps table loads off the per-tile path.)
                bool any_bad = false;
                for (int blk = lane; blk < it.nblk_live; blk += 32) {
                    const int id = it.bt[blk];
                    any_bad |= id < 0 || id >= p.num_blocks;
                }
                any_bad = __any_sync(kFullMask, any_bad);
                float m_ref = -INFINITY, l_run = 0.f;
                for (int j = 0; j < nk; ++j) {
                    const int Tx = tx0 + j;
                    const int J = kv0 + j;
                    // blocks of this tile outside the pool (their keys are masked
                    // and their V rows cleared), from the table as the producer saw it
                    uint32_t bad = 0;
                    if (any_bad) {
#pragma unroll
                        for (int jb = 0; jb < kTcBlocks; ++jb) {
                            const int blk = j * kTcBlocks + jb;
                            if (blk < it.nblk_live) {
                                const int id = it.bt[blk];
                                if (id < 0 || id >= p.num_blocks) bad |= 1u << jb;
                            }
                        }
                    }
                    if (!__all_sync(kFullMask, wait_or_abort(&s_full[x], Tx & 1, abort_v))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const int key0 = j * kTcKeys;
                    // The row maximum only decides the lazy rescale below, so a
                    // first pass takes the exponentials against the current
                    // reference m_ref without it.  When the tile's sum of P stays
                    // below 2^8, so does every P: the maximum is then at most
                    // m_ref + 8, the rule would keep m_ref, and the tile is done.
                    // Otherwise (and on an item's first tile, or while a row has
                    // no reference yet) a second pass reloads S, which stays in
                    // tensor memory until P is stored, and takes the maximum
                    // first.  Either way P is what taking the maximum every time
                    // gives.  (Warp-wide decisions: tcgen05.ld/st are collective.)
                    bool need_max = __any_sync(kFullMask, m_ref == -INFINITY);
                    float sv[kTcKeys];
                    float l_tile;
#pragma unroll 1
                    for (;;) {
                        // the row's 128 scores, all in flight before one wait
                        {
                            uint32_t r0[32], r1[32], r2[32], r3[32];
                            tmem_ld32(s_tm, r0);
                            tmem_ld32(s_tm + 32, r1);
                            tmem_ld32(s_tm + 64, r2);
                            tmem_ld32(s_tm + 96, r3);
                            tmem_ld_wait();
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                sv[c] = __uint_as_float(r0[c]);
                                sv[32 + c] = __uint_as_float(r1[c]);
                                sv[64 + c] = __uint_as_float(r2[c]);
                                sv[96 + c] = __uint_as_float(r3[c]);
                            }
                        }
                        // A positive scale is applied after the row maximum (the
                        // maximum of the scaled scores is the scaled maximum, as
                        // rounding is monotonic), fused with the subtraction of
                        // the exponent.
                        if (!fold) {
#pragma unroll
                            for (int c = 0; c < kTcKeys; c += 2) mul2(sv[c], sv[c + 1], p.scale_log2);
                        }
                        if ((key0 + kTcKeys - 1 > pos_lo) || bad) {
#pragma unroll
                            for (int c = 0; c < kTcKeys; ++c) {
                                const bool dead = key0 + c > pos_row || ((bad >> (c >> 4)) & 1u);
                                sv[c] = dead ? -INFINITY : sv[c];
                            }
                        }
                        if (need_max) {
                            // the row maximum: four chains of three-input maxima
                            float mx;
                            {
                                float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                                for (int c = 0; c < kTcKeys; c += 8) {
#pragma unroll
                                    for (int u = 0; u < 4; ++u)
                                        mq[u] = fmax3(mq[u], sv[c + 2 * u], sv[c + 2 * u + 1]);
                                }
                                mx = fmax3(fmaxf(mq[0], mq[1]), mq[2], mq[3]);
                                if (fold) mx *= p.scale_log2;
                            }
                            // lazy rescale: move the reference only when the
                            // maximum has grown by more than 2^8.  P V(j-1) is
                            // complete (S(j) was issued after it), so O can be
                            // rescaled in place.
                            if (__any_sync(kFullMask, mx > m_ref + kRescaleLog2)) {
                                const float new_ref = fmaxf(m_ref, mx);
                                const float alpha = new_ref == -INFINITY ? 1.f : fast_exp2(m_ref - new_ref);
                                if (j > 0) {
#pragma unroll 1
                                    for (int c0 = 0; c0 < D / 32; ++c0) {   // (rare: kept rolled)
                                        uint32_t rr[32];
                                        tmem_ld32(o_tm + static_cast<uint32_t>(c0 * 32), rr);
                                        tmem_ld_wait();
#pragma unroll
                                        for (int u = 0; u < 32; ++u)
                                            rr[u] = __float_as_uint(__uint_as_float(rr[u]) * alpha);
                                        tmem_st32(o_tm + static_cast<uint32_t>(c0 * 32), rr);
                                    }
                                    tmem_st_wait();
                                }
                                l_run *= alpha;
                                m_ref = new_ref;
                            }
                        }
                        // P = 2^(s - m_ref) (in place) and its sum
                        {
                            const float ref = m_ref == -INFINITY ? 0.f : m_ref;
                            // s * 1 + (-ref) rounds once, like s - ref: one loop for both
                            const float mul = fold ? p.scale_log2 : 1.f;
#pragma unroll
                            for (int c = 0; c < kTcKeys; c += 2) fma2(sv[c], sv[c + 1], mul, -ref);
#pragma unroll
                            for (int c = 0; c < kTcKeys; ++c) sv[c] = fast_exp2(sv[c]);
                            float sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int c = 0; c < kTcKeys; c += 4) {
                                add2(sq[0], sq[1], sv[c], sv[c + 1]);
                                add2(sq[2], sq[3], sv[c + 2], sv[c + 3]);
                            }
                            l_tile = (sq[0] + sq[1]) + (sq[2] + sq[3]);
                        }
                        // (a NaN sum also takes the second pass)
                        if (need_max || !__any_sync(kFullMask, !(l_tile < kPLazyMax))) break;
                        need_max = true;
                    }
                    l_run += l_tile;
                    // P goes over the row's first 64 columns (two 16-bit values
                    // per column, keys in order)
                    {
                        uint32_t pw0[32], pw1[32];
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            pw0[c] = Elem<T>::pack(sv[2 * c], sv[2 * c + 1]);
                            pw1[c] = Elem<T>::pack(sv[64 + 2 * c], sv[64 + 2 * c + 1]);
                        }
                        tmem_st32(s_tm, pw0);
                        tmem_st32(s_tm + 32, pw1);
                    }
                    // V rows that must contribute nothing (past the pair's last
                    // query position, or in a block outside the pool) may hold
                    // anything, NaN included: the first tile of the pair that
                    // reads this key tile clears them before its P V (the other
                    // tile's P V is issued after it)
                    const bool clearer = x == 0 || j >= nk_a;
                    if (clearer && (j == it.nkt - 1 || bad)) {
                        if (!__all_sync(kFullMask, wait_or_abort(&v_full[J % NV], (J / NV) & 1, abort_v))) {
                            ok = false;
                            break;
                        }
                        constexpr int CPR = D / 8;
                        uint8_t* vt = vst(J % NV);
                        for (int idx = r; idx < kTcKeys * CPR; idx += kTcSoftmaxWarps * 32) {
                            const int key = idx / CPR;
                            const int c = idx - key * CPR;
                            if (key0 + key > it.pos_pair || ((bad >> (key >> 4)) & 1u))
                                *reinterpret_cast<uint4*>(vt + (key >> 4) * (D / 64) * 2048 + (c >> 3) * 2048 +
                                                          (key & 15) * 128 + (((c & 7) ^ (key & 7)) << 4)) =
                                    make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                    }
                    tmem_st_wait();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&p_full[x]);
                }
                if (ok) {
                    const bool got = wait_or_abort(&o_done[x][0], n_items_x & 1, abort_v);
                    if (__all_sync(kFullMask, got)) {
                        tc_fence_after_sync();
                        const float inv = l_run > 0.f ? p.v_scale / l_run : 0.f;
                        const int64_t grow =
                            static_cast<int64_t>(it.row0 + qi_row) * p.num_q_heads + it.g * G + (r % G);
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + grow * D);
#pragma unroll 1
                        for (int c0 = 0; c0 < D / 32; ++c0) {   // (once per item: kept rolled)
                            uint32_t rr[32];
                            tmem_ld32(o_tm + static_cast<uint32_t>(c0 * 32), rr);
                            tmem_ld_wait();
                            if (row_ok) {
#pragma unroll
                                for (int c = 0; c < 4; ++c) {
                                    uint4 v4;
                                    v4.x = Elem<T>::pack(__uint_as_float(rr[8 * c + 0]) * inv,
                                                         __uint_as_float(rr[8 * c + 1]) * inv);
                                    v4.y = Elem<T>::pack(__uint_as_float(rr[8 * c + 2]) * inv,
                                                         __uint_as_float(rr[8 * c + 3]) * inv);
                                    v4.z = Elem<T>::pack(__uint_as_float(rr[8 * c + 4]) * inv,
                                                         __uint_as_float(rr[8 * c + 5]) * inv);
                                    v4.w = Elem<T>::pack(__uint_as_float(rr[8 * c + 6]) * inv,
                                                         __uint_as_float(rr[8 * c + 7]) * inv);
                                    dst[c0 * 4 + c] = v4;
                                }
                            }
                        }
                        tc_fence_before_sync();
                    } else {
                        ok = false;
                    }
                }
                ++n_items_x;
            }
            if (!ok) *abort_v = 1;
            next_item(it);
        }
        if (!ok || *abort_v) {
            if (tid == 0) record_error(p.err, PA_DEVERR_TIMEOUT_);
        }
    } else if (warp == kTcMmaWarp) {
        // ============================== MMA issuer ==============================
        reg_dealloc<kTcOtherRegs>();
        int s_issued[kTcTiles] = {0, 0}, pv_issued[kTcTiles] = {0, 0};   // for the abort path
        for (int k = 0; ok; ++k) {
            const int w0 = item_at(k);
            if (w0 == kNoMoreItems) break;
            Item it;
            if (w0 < 0 || !decode_item(w0, it)) continue;
            // S_X(j) into S_X: eight MMAs of K=16 over the head dimension
            auto mma_s = [&](int x, int j) {
                const uint32_t d_tm = tmem + static_cast<uint32_t>(x * kTcKeys);
                const uint64_t a0 = smem_desc_sw128(smem_addr(qs(x)), 16, 1024);
                const uint64_t b0 = smem_desc_sw128(smem_addr(kst((kv0 + j) % NK)), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    // the start-address field (bits 0-13, 16-byte units) never carries out
                    const uint64_t a = a0 + static_cast<uint64_t>(((kk >> 2) * Sh::kQHalf + (kk & 3) * 32) >> 4);
                    const uint64_t bd = b0 + static_cast<uint64_t>(((kk >> 2) * Sh::kKeyHalf + (kk & 3) * 32) >> 4);
                    el_mma(d_tm, a, bd, kIdescS, kk > 0 ? 1u : 0u);
                }
                el_commit(&s_full[x]);
                ++s_issued[x];
            };
            // O_X += P_X(j) V(j): P is read from tensor memory, where the softmax
            // stored it over the first 64 columns of S_X; MMA kp reads block kp
            // of the V tile (its two 64-dim halves 2 KB apart)
            auto mma_pv = [&](int x, int j) {
                const uint32_t p_tm = tmem + static_cast<uint32_t>(x * kTcKeys);
                const uint32_t o_tm = tmem + static_cast<uint32_t>(kTcTiles * kTcKeys + x * D);
                const uint64_t v0 = smem_desc_sw128(smem_addr(vst((kv0 + j) % NV)), 2048, 1024);
#pragma unroll
                for (int kp = 0; kp < kTcKeys / 16; ++kp) {
                    const uint64_t bd = v0 + static_cast<uint64_t>((kp * (D / 64) * 2048) >> 4);
                    el_mma_ta(o_tm, p_tm + static_cast<uint32_t>(kp * 8), bd, kIdescPV, (j > 0 || kp > 0) ? 1u : 0u);
                }
                if (j + 1 == it.nkx[x]) el_commit(&o_done[x][0]);   // the item's last P V of tile x
                ++pv_issued[x];
            };
            auto commit = [&](uint64_t* bar) { el_commit(bar); };
            auto wait_all = [&](uint64_t* bar, uint32_t parity) {
                return __all_sync(kFullMask, wait_or_abort(bar, parity, abort_v));
            };
            // the previous item's MMAs must be complete: its S/P buffers and
            // accumulators are reused
            if (items > 0) ok = wait_all(&item_done, (items - 1) & 1);
            if (ok) {
                // the item's query tiles (the previous item's MMAs are done with theirs)
                el_expect_tx(&q_full, static_cast<uint32_t>((it.nkx[1] ? 2 : 1) * q_tile_bytes));
#pragma unroll
                for (int x = 0; x < kTcTiles; ++x) {
                    if (!it.nkx[x]) continue;
#pragma unroll
                    for (int h = 0; h < D / 64; ++h)
                        el_tma_4d(qs(x) + h * Sh::kQHalf, &qmap, &q_full, 0, h, it.g * G, it.row0 + it.q0[x]);
                }
            }
            if (ok) ok = wait_all(&q_full, items & 1) && wait_all(&k_full[kv0 % NK], (kv0 / NK) & 1);
            if (ok) {
                tc_fence_after_sync();
#pragma unroll
                for (int x = 0; x < kTcTiles; ++x)
                    if (it.nkx[x]) mma_s(x, 0);
                commit(&k_free[kv0 % NK]);
            }
            for (int j = 0; ok && j < it.nkt; ++j) {
                const int J = kv0 + j;
                ok = wait_all(&v_full[J % NV], (J / NV) & 1);
                if (!ok) break;
                bool k_next = false;   // K(j+1) seen landed
                // per tile: P V(j) once its softmax stored P, then S(j+1) into
                // the same columns right behind it (tcgen05.mma operations of
                // one thread execute in issue order, so P V(j) has read P
                // before S(j+1) overwrites it); the other tile's softmax runs
                // meanwhile
#pragma unroll
                for (int x = 0; x < kTcTiles; ++x) {
                    if (j >= it.nkx[x]) continue;
                    const int Tx = t0[x] + j;
                    if (!(ok = wait_all(&p_full[x], Tx & 1))) break;
                    tc_fence_after_sync();
                    mma_pv(x, j);
                    if (j + 1 >= it.nkx[x]) continue;
                    if (!k_next) {
                        if (!(ok = wait_all(&k_full[(J + 1) % NK], ((J + 1) / NK) & 1))) break;
                        k_next = true;
                    }
                    mma_s(x, j + 1);
                }
                if (!ok) break;
                commit(&v_free[J % NV]);                              // V(j)'s stage, once both P V are done
                if (j + 1 < it.nkt) commit(&k_free[(J + 1) % NK]);    // K(j+1)'s, once both S are done
            }
            if (ok) commit(&item_done);
            if (!ok && lane == 0) *abort_v = 1;
            next_item(it);
        }
        if (__any_sync(kFullMask, !ok || *abort_v)) {
            // let MMAs still in flight finish before the CTA's memory is reused
            // (the commit comes from the lane that issued them)
            el_commit(&o_done[0][1]);
            if (lane == 0) {
                (void)mbar_wait(&o_done[0][1], 0);
#pragma unroll
                for (int x = 0; x < kTcTiles; ++x) {
                    if (s_issued[x]) (void)mbar_wait(&s_full[x], (s_issued[x] - 1) & 1);
                    (void)pv_issued[x];
                }
            }
        }
    } else {
        // ================================ loaders ===============================
        // Each ring stage has one loader: K stage s and V stage s belong to
        // loader s % 3, which therefore sees every phase of the stage's
        // k_free / v_free barrier (a parity wait is sound only for the phase
        // after the last one its waiter saw).  A loader walks the key tiles J
        // = kv0 + j in order and issues K(J) and V(J) when it owns their
        // stages, eight lanes at once: lane l < 8 reads block l's id (one
        // coalesced load) and issues that block's boxes (K: one per 64-dim
        // half; V: one).  The MMA warp loads the query tiles.
        reg_dealloc<kTcOtherRegs>();
        const int li = warp - kTcMmaWarp - 1;
        constexpr int kHalves = D / 64;
        int k_last[NK], v_last[NV];   // ring index of the last tile issued per owned stage
#pragma unroll
        for (int s = 0; s < NK; ++s) k_last[s] = -1;
#pragma unroll
        for (int s = 0; s < NV; ++s) v_last[s] = -1;
        for (int k = 0; ok; ++k) {
            const int w0 = item_at(k);
            if (w0 == kNoMoreItems) break;
            Item it;
            if (w0 < 0 || !decode_item(w0, it)) continue;
            for (int j = 0; ok && j < it.nkt; ++j) {
                const int J = kv0 + j;
                const int sk = J % NK, sv = J % NV;
                const bool do_k = sk % kTcLoaders == li, do_v = sv % kTcLoaders == li;
                if (!do_k && !do_v) continue;
                int id = -1;
                if (lane < kTcBlocks && j * kTcBlocks + lane < it.nblk_live) {
                    id = it.bt[j * kTcBlocks + lane];
                    if (id < 0 || id >= p.num_blocks) {
                        if (do_k) record_error(p.err, PA_DEVERR_BLOCK_ID_);
                        id = -1;
                    }
                }
                const uint32_t live = static_cast<uint32_t>(__popc(__ballot_sync(kFullMask, id >= 0)));
                bool r = true;
                if (do_k) {
                    // K(J): free once both S(J - NK) are done
                    if (lane == 0 && J >= NK) r = wait_or_abort(&k_free[sk], ((J - NK) / NK) & 1, abort_v);
                    if (!(ok = __shfl_sync(kFullMask, r ? 1 : 0, 0) != 0)) break;
                    if (lane == 0) mbar_arrive_expect_tx(&k_full[sk], live * kHalves * 2048);
                    __syncwarp();
#pragma unroll
                    for (int h = 0; h < kHalves; ++h)
                        if (id >= 0)
                            tma_load_4d(kst(sk) + h * Sh::kKeyHalf + lane * 2048, &kmap, &k_full[sk], 0, h, it.g, id * 16);
                    k_last[sk] = J;
                }
                if (do_v) {
                    // V(J): free once both P V(J - NV) are done
                    if (lane == 0 && J >= NV) r = wait_or_abort(&v_free[sv], ((J - NV) / NV) & 1, abort_v);
                    if (!(ok = __shfl_sync(kFullMask, r ? 1 : 0, 0) != 0)) break;
                    if (lane == 0) mbar_arrive_expect_tx(&v_full[sv], live * kHalves * 2048);
                    __syncwarp();
                    if (id >= 0) tma_load_4d(vst(sv) + lane * kHalves * 2048, &vmap, &v_full[sv], 0, id * 16, 0, it.g);
                    v_last[sv] = J;
                }
            }
            if (!ok && lane == 0) *abort_v = 1;
            next_item(it);
        }
        if (__any_sync(kFullMask, !ok || *abort_v) && lane == 0) {
            // this loader's copies still in flight: the last phase of each stage it filled
            for (int s = 0; s < NK; ++s)
                if (k_last[s] >= 0) (void)mbar_wait(&k_full[s], (k_last[s] / NK) & 1);
            for (int s = 0; s < NV; ++s)
                if (v_last[s] >= 0) (void)mbar_wait(&v_full[s], (v_last[s] / NV) & 1);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}


template <typename T, int D>
cudaError_t launch_t(const PrefillParams& p, int32_t* plan, const CUtensorMap& kmap, const CUtensorMap& vmap,
                     const CUtensorMap& qmap, int max_q_len, int num_tokens, const Fp8Copy* copy, cudaStream_t s) {
    constexpr int smem = TcShape<D>::kSmem;
    auto kern = prefill_tc_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // the softmax warpgroups' register increase is granted from the pool the
    // CTA is launched with: refuse to launch if the build gave it fewer
    static const int launch_regs = [&] {
        cudaFuncAttributes fa{};
        return cudaFuncGetAttributes(&fa, kern) == cudaSuccess ? fa.numRegs : 0;
    }();
    if (launch_regs < kTcLaunchRegs) return cudaErrorInvalidConfiguration;
    const Fp8Copy none{};
    prefill_plan_kernel<<<1, 1024, 0, s>>>(p.cu_q_lens, p.seq_lens, p.num_seqs, num_tokens, p.q_per_tile, plan,
                                           p.pair_cap, p.err, copy ? *copy : none, p.max_seq_len, p.max_blocks);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (copy && copy->cap_blocks > 0) {
        // a few CTAs per SM stream the copy blocks (at most cap_blocks of them)
        const int wgrid = std::max(1, std::min(copy->cap_blocks, 8 * sm_count()));
        widen_chunk_blocks_kernel<T><<<wgrid, kWidenThreads, 0, s>>>(*copy, p.seq_lens, p.max_blocks,
                                                                     p.num_kv_heads);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // upper bound on the work items: each listed chunk (length > 8) has at
    // most ceil(len / q_per_tile) <= len / 2 tiles, and there are at most
    // max_q_len tokens per chunk; an item is a pair of tiles.  One CTA per SM.
    const long long bound_tiles = std::min<long long>(static_cast<long long>(num_tokens) / 2 + 1,
                                                      static_cast<long long>(p.num_seqs) *
                                                          ((max_q_len + p.q_per_tile - 1) / p.q_per_tile));
    const long long items = (bound_tiles + p.num_seqs) / kTcTiles * p.num_kv_heads + p.num_kv_heads;
    const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(items, sm_count())));
    kern<<<grid, kTcThreads, smem, s>>>(p, plan, kmap, vmap, qmap);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillParams& p, int32_t* plan, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, const CUtensorMap& qmap, int head_dim, int dtype,
                              int max_q_len, int num_tokens, const Fp8Copy* copy, cudaStream_t s) {
    if (p.num_seqs == 0 || max_q_len <= PA_VERIFY_MAX_Q_) return cudaSuccess;
    if (copy && head_dim != 128) return cudaErrorInvalidValue;
    if (dtype == 0)
        return head_dim == 128 ? launch_t<__half, 128>(p, plan, kmap, vmap, qmap, max_q_len, num_tokens, copy, s)
                               : launch_t<__half, 64>(p, plan, kmap, vmap, qmap, max_q_len, num_tokens, copy, s);
    return head_dim == 128
               ? launch_t<__nv_bfloat16, 128>(p, plan, kmap, vmap, qmap, max_q_len, num_tokens, copy, s)
               : launch_t<__nv_bfloat16, 64>(p, plan, kmap, vmap, qmap, max_q_len, num_tokens, copy, s);
}

}  // namespace pa
