// Decode attention over the paged KV cache, plus the split-context reduction.
//
// What is computed ("vLLM-Ascend 原理", section 2.4 "分页自注意力"; the block
// loop of the CANN PagedAttentionKernel sketch): for each sequence the single
// new query attends to every cached position 0..seq_len-1; K and V are read
// block by block through the block table, and because the blocks are not
// contiguous the softmax is merged block by block (online softmax: running
// max m, running sum l, running weighted sum acc).  Long contexts are cut into
// partitions of `partition_tokens`; each partition leaves (m, l, acc) in the
// workspace and a second kernel merges them by log-sum-exp.
//
// GB300 design:
//  * a one-CTA plan kernel lists the (sequence, partition) units; the decode
//    kernel is persistent and gives each work item (unit, kv head) to one
//    warp, which handles the `group` query heads that share the kv head, so
//    every K/V byte is read once and no CTA is launched without work.
//  * each warp owns a private ring of STAGES shared-memory slots; its lane 0
//    fetches whole (16-token block, kv head) tiles of K and V with one 4-D
//    TMA load each (both 64-dim halves, 128-byte swizzle: a TMA issue costs
//    the issuing thread hundreds of cycles, so one box per tile), completing
//    on a per-slot mbarrier, and keeps fetching ahead across the warp's items.
//  * MHA (group 1): fp32 FMA dot products, a 16-way transpose-reduction
//    across the warp (16 shuffles per block), register-resident (m, l, acc).
//  * GQA (group 2..8): the query group x K-block product is a dense
//    contraction: S^T[16 tokens x 8 heads] = K Q^T and O^T += V^T P^T with
//    mma.sync m16n8k16 (fp32 accumulate); M = 16 tokens matches the block.
//  * FP8 (E4M3) pools are head-major, so a (block, kv head) tile is one
//    contiguous 2 KB box; MHA converts codes in registers, GQA converts the
//    tile to 16-bit in shared memory for the MMA.
//  * a warp writes its item's output row, or the partition's (m, l, acc)
//    for the log-sum-exp reduction kernel.
#include <algorithm>
#include <atomic>
#include <type_traits>

#include "pa_device.cuh"

namespace pa {

namespace {

constexpr int kDecodeWarps = 4;
constexpr unsigned kFull = 0xffffffffu;
// The tensor-core path keeps a column's reference max until a score exceeds
// it by this much (log2 units), so softmax weights stay within [0, 2^8].
constexpr float kLazyRescaleLog2 = 8.f;

// Per-warp shared memory: a ring of kStages (K tile, V tile) slots.  A warp
// handles one block at a time, so it moves bytes at (tile bytes) / (block
// latency); FP8 tiles are half the bytes, so the FP8 MHA kernel keeps small
// rings and runs more CTAs (warps) per SM instead.
template <int D, bool kFp8, bool kMma, int kMaxNT = 1>
struct DecodeShape {
    static constexpr int kTileBytes = 16 * D * (kFp8 ? 1 : 2);  // one (block, kv head) tile
    static constexpr int kStageBytes = 2 * kTileBytes;          // K tile + V tile
    // The 16-bit tensor-core kernels are bound by instruction latency per
    // warp: the single-tile one (group heads of decode rows) runs best with
    // 2-stage rings and 3 CTAs (12 warps) per SM; the two-tile one (verify
    // rows, 16 columns) with 3-stage rings and 2 CTAs per SM.  The FP8 MHA
    // kernel keeps 5 CTAs (20 warps) per SM: registers capped at 96.  The FP8
    // tensor-core kernels keep 3 (registers capped at 168; the two-tile one,
    // which also serves the decode rows of a varlen call, would take 207).
    static constexpr int kStages = kFp8 ? (kMma ? 4 : 2) : (kMma ? (kMaxNT > 1 ? 3 : 2) : 3);
    static constexpr int kMinCtasPerSm = (kMma && !kFp8) ? (kMaxNT > 1 ? 2 : 3) : (kFp8 && !kMma ? 5 : 3);
    static constexpr int kWarpBytes = kStages * kStageBytes;
    static constexpr int kSmemBytes = kDecodeWarps * kWarpBytes + 1024;  // + alignment slack
};

// Per-warp TMA producer state for one CTA's partition.
struct WarpRing {
    uint8_t* base;      // this warp's STAGES slots
    uint64_t* bars;     // STAGES mbarriers
};

template <int D, bool kFp8, bool kMma, int kMaxNT>
__device__ __forceinline__ void issue_tile(const WarpRing& ring, int slot, int phys, int kv_head,
                                          const CUtensorMap* kmap, const CUtensorMap* vmap) {
    using Shape = DecodeShape<D, kFp8, kMma, kMaxNT>;
    uint8_t* dst = ring.base + slot * Shape::kStageBytes;
    mbar_arrive_expect_tx(&ring.bars[slot], Shape::kStageBytes);
    if constexpr (kFp8) {
        // head-major FP8 pool: the (block, head) tile is one contiguous 2 KB box
        tma_load_4d(dst, kmap, &ring.bars[slot], 0, 0, kv_head, phys);
        tma_load_4d(dst + Shape::kTileBytes, vmap, &ring.bars[slot], 0, 0, kv_head, phys);
    } else {
        // one box per tile: both 64-dim halves of the 16 rows (block tensor map)
        tma_load_4d(dst, kmap, &ring.bars[slot], 0, phys * 16, 0, kv_head);
        tma_load_4d(dst + Shape::kTileBytes, vmap, &ring.bars[slot], 0, phys * 16, 0, kv_head);
    }
}

// q . k for two 16-bit pairs of type T: s + q0 k0 + q1 k1, each a fused
// multiply-add in fp32 of two 16-bit operands (exact products, one rounding
// per step, as fmaf on the converted values).
template <typename T>
__device__ __forceinline__ float dot2_mixed(float s, uint32_t q01, uint32_t k01) {
    if constexpr (std::is_same<T, __half>::value) {
        asm("{\n\t.reg .f16 q0, q1, k0, k1;\n\tmov.b32 {q0, q1}, %1;\n\tmov.b32 {k0, k1}, %2;\n\t"
            "fma.rn.f32.f16 %0, q0, k0, %0;\n\tfma.rn.f32.f16 %0, q1, k1, %0;\n\t}"
            : "+f"(s)
            : "r"(q01), "r"(k01));
    } else {
        asm("{\n\t.reg .b16 q0, q1, k0, k1;\n\tmov.b32 {q0, q1}, %1;\n\tmov.b32 {k0, k1}, %2;\n\t"
            "fma.rn.f32.bf16 %0, q0, k0, %0;\n\tfma.rn.f32.bf16 %0, q1, k1, %0;\n\t}"
            : "+f"(s)
            : "r"(q01), "r"(k01));
    }
    return s;
}

// ---------------------------------------------------------------------------
// MHA block step: fp32 dot products on the ALU.
// Lane l owns head dims [l*DPL, (l+1)*DPL).
// The scores (kMixedK: 16-bit caches, and FP8 caches with fp16 queries)
// multiply the query's and the key's 16-bit pairs in fp32 directly
// (mixed-precision FMA; E4M3 codes as fp16 pairs straight from their
// conversion), and the score scale is applied once to each finished dot
// product.  FP8 caches with bf16 queries convert the codes to fp32 first.
// With an FP8 cache and fp16 queries (kTokenK) the scores are computed token
// by token instead: lanes 2t and 2t+1 each take half of token t's 128 dims
// (four 16-byte loads of codes, no transpose-reduction), which leaves the
// scores in the same lanes as the reduction does.
// ---------------------------------------------------------------------------
template <typename T, int D, bool kFp8 = false>
struct AluState {
    static constexpr int DPL = D / 32;
    static constexpr bool kMixedK = !kFp8 || std::is_same<T, __half>::value;
    static constexpr bool kTokenK = kFp8 && std::is_same<T, __half>::value;
    uint32_t qk[kTokenK ? 32 : 1];   // this lane's 64 query dims as fp16 pairs (kTokenK)
    float q[DPL];        // scaled fp32 query dims (all but kMixedK)
    uint32_t qh[DPL / 2];  // 16-bit query pairs (kMixedK)
    float qscale;        // score scale applied after the dot product (kMixedK)
    float acc[DPL];
    float m;
    float l;  // this lane's share (even lanes only)

    __device__ __forceinline__ void load_dims(const uint8_t* tile, int tok, int lane, float* x) const {
        if constexpr (kFp8) {
            // four E4M3 codes (head_dim 128, one 128-byte row per token)
            const uint32_t raw = *reinterpret_cast<const uint32_t*>(tile + fp8_off(tok, lane * 4));
            const float2 a = Elem<__half>::to_float2(e4m3x2_to_f16x2(static_cast<uint16_t>(raw & 0xffffu)));
            const float2 b = Elem<__half>::to_float2(e4m3x2_to_f16x2(static_cast<uint16_t>(raw >> 16)));
            x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
        } else if constexpr (DPL == 4) {
            const uint2 raw = *reinterpret_cast<const uint2*>(tile + tile_off<D>(tok, lane * 4));
            const float2 a = Elem<T>::to_float2(raw.x), b = Elem<T>::to_float2(raw.y);
            x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
        } else {
            const uint32_t raw = *reinterpret_cast<const uint32_t*>(tile + tile_off<D>(tok, lane * 2));
            const float2 a = Elem<T>::to_float2(raw);
            x[0] = a.x; x[1] = a.y;
        }
    }

    __device__ __forceinline__ void step(const uint8_t* kt, const uint8_t* vt, int nvalid, int lane) {
        float s;
        if constexpr (kTokenK) {
            // lanes 2t and 2t+1 each take one half of token t's 128 dims
            const int t = lane >> 1, h = lane & 1;
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 raw = *reinterpret_cast<const uint4*>(kt + fp8_off(t, h * 64 + k * 16));
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t k01 = e4m3x2_to_f16x2(static_cast<uint16_t>(w[j] & 0xffffu));
                    const uint32_t k23 = e4m3x2_to_f16x2(static_cast<uint16_t>(w[j] >> 16));
                    s0 = dot2_mixed<T>(s0, qk[8 * k + 2 * j], k01);
                    s1 = dot2_mixed<T>(s1, qk[8 * k + 2 * j + 1], k23);
                }
            }
            s = s0 + s1;
            s += __shfl_xor_sync(kFull, s, 1);
            s *= qscale;
        } else {
            float part[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                float s = 0.f;
                if constexpr (kMixedK) {
                    uint32_t kw[DPL / 2];
                    if constexpr (kFp8) {
                        static_assert(DPL == 4, "FP8 tiles hold head_dim 128");
                        const uint32_t raw = *reinterpret_cast<const uint32_t*>(kt + fp8_off(t, lane * 4));
                        kw[0] = e4m3x2_to_f16x2(static_cast<uint16_t>(raw & 0xffffu));
                        kw[1] = e4m3x2_to_f16x2(static_cast<uint16_t>(raw >> 16));
                    } else if constexpr (DPL == 4) {
                        const uint2 raw = *reinterpret_cast<const uint2*>(kt + tile_off<D>(t, lane * 4));
                        kw[0] = raw.x;
                        kw[1] = raw.y;
                    } else {
                        kw[0] = *reinterpret_cast<const uint32_t*>(kt + tile_off<D>(t, lane * 2));
                    }
#pragma unroll
                    for (int j = 0; j < DPL / 2; ++j) s = dot2_mixed<T>(s, qh[j], kw[j]);
                } else {
                    float k[DPL];
                    load_dims(kt, t, lane, k);
#pragma unroll
                    for (int j = 0; j < DPL; ++j) s = fmaf(q[j], k[j], s);
                }
                part[t] = s;
            }
            // transpose-reduce: after the five exchange rounds lane l holds the full
            // dot product of token l >> 1 (lanes 2t and 2t+1 hold the same value).
            {
                const bool hi = lane & 16;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float send = hi ? part[j] : part[j + 8];
                    const float keep = hi ? part[j + 8] : part[j];
                    part[j] = keep + __shfl_xor_sync(kFull, send, 16);
                }
            }
            {
                const bool hi = lane & 8;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float send = hi ? part[j] : part[j + 4];
                    const float keep = hi ? part[j + 4] : part[j];
                    part[j] = keep + __shfl_xor_sync(kFull, send, 8);
                }
            }
            {
                const bool hi = lane & 4;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float send = hi ? part[j] : part[j + 2];
                    const float keep = hi ? part[j + 2] : part[j];
                    part[j] = keep + __shfl_xor_sync(kFull, send, 4);
                }
            }
            {
                const bool hi = lane & 2;
                const float send = hi ? part[0] : part[1];
                const float keep = hi ? part[1] : part[0];
                part[0] = keep + __shfl_xor_sync(kFull, send, 2);
            }
            s = part[0] + __shfl_xor_sync(kFull, part[0], 1);
            if constexpr (kMixedK) s *= qscale;
        }
        const int tok = lane >> 1;
        s = tok < nvalid ? s : -INFINITY;
        float mb = s;
        mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 2));
        mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 4));
        mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 8));
        mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 16));
        const float m_new = fmaxf(m, mb);
        const float alpha = fast_exp2(m - m_new);
        const float p = fast_exp2(s - m_new);
        m = m_new;
        l = l * alpha + ((lane & 1) ? 0.f : p);
#pragma unroll
        for (int j = 0; j < DPL; ++j) acc[j] *= alpha;
        if (nvalid == 16) {
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const float pt = __shfl_sync(kFull, p, 2 * t);
                float v[DPL];
                load_dims(vt, t, lane, v);
#pragma unroll
                for (int j = 0; j < DPL; ++j) acc[j] = fmaf(pt, v[j], acc[j]);
            }
        } else {
            for (int t = 0; t < nvalid; ++t) {
                const float pt = __shfl_sync(kFull, p, 2 * t);
                float v[DPL];
                load_dims(vt, t, lane, v);
#pragma unroll
                for (int j = 0; j < DPL; ++j) acc[j] = fmaf(pt, v[j], acc[j]);
            }
        }
    }
};

// Two E4M3 codes (low byte first) as a 16-bit pair of type T (exact).
template <typename T>
__device__ __forceinline__ uint32_t codes_to(uint16_t codes) {
    const uint32_t h = e4m3x2_to_f16x2(codes);
    if constexpr (std::is_same<T, __half>::value) {
        return h;
    } else {
        const float2 f = Elem<__half>::to_float2(h);
        return Elem<T>::pack(f.x, f.y);
    }
}

// ---------------------------------------------------------------------------
// Query-group x K-block step on the tensor cores (mma.sync m16n8k16, fp32
// accumulate).  The columns are (query, head) pairs that share one kv head:
// the `group` heads of a decode row, or q_len x group pairs of a
// speculative-verify row, in NT tiles of 8 columns.
// S^T = K Q^T: rows = the 16 tokens of the block.  Lane l holds S^T rows l/4
// and l/4+8 of columns 8*nt + 2*(l%4) + {0,1}; O^T (head_dim x columns) uses
// the same columns, so the per-column rescale needs no data movement.  Column
// j sees the tokens below lim[nt][e]: its query's causal limit, capped at the
// partition end.
// ---------------------------------------------------------------------------
// FP8 (E4M3) tiles (kFp8, head_dim 128) are read without a 16-bit copy:
// ldmatrix treats two codes as one 16-bit element.  For S^T, lane (g, c) then
// holds codes 4c .. 4c+3 of a 16-dim chunk of tokens g and g+8; within each
// k-step the dims are taken in the order 4c, 4c+1 | 4c+2, 4c+3 for the
// logical columns 2c, 2c+1 | 2c+8, 2c+9, and Q^T is loaded in the same order
// (a dot product does not depend on the order of its terms).  For O^T the
// transposing ldmatrix gives lane (g, c) dims 2g, 2g+1 of tokens 2c, 2c+1 of a
// chunk; one byte permute pairs the tokens of each dim, so the m-tile's rows
// g and g+8 are dims 2g and 2g+1 of the chunk (undone when O^T is written).
// P and the converted V are fp16 (every E4M3 value is an fp16 value; P <= 2^8).
template <typename T, int D, int NT, bool kFp8 = false>
struct MmaState {
    static constexpr int KS = D / 16;
    uint32_t qb[KS][NT][2];   // Q^T as the B operand, per 16-dim k-step and column tile
    float o[KS][NT][4];       // O^T accumulator, per 16-dim m-tile and column tile
    float m[NT][2];
    float l[NT][2];
    int lim[NT][2];           // first token the column may not see

    // `masked`: some column of this block has a limit inside it (else every
    // token of the block is visible to every column).  Rows at or past
    // `nvalid` lie beyond the partition end.
    __device__ __forceinline__ void step(uint8_t* kt, uint8_t* vt, int base, int nvalid, bool masked, int lane,
                                         float scale_log2) {
        const uint32_t ka = smem_addr(kt);
        const uint32_t va = smem_addr(vt);
        float c[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) c[nt][e] = 0.f;
        {
            const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int dsub = ((lane >> 4) & 1) * 8;
            // two independent accumulation chains (even and odd k-steps)
            float c2[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) c2[nt][e] = 0.f;
            if constexpr (kFp8) {
                // lane l addresses row l % 8 of matrix l / 8: tokens 0-7 / 8-15
                // of chunks 2kp and 2kp + 1
                const int ft = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                for (int kp = 0; kp < KS / 2; ++kp) {
                    const int chunk = 2 * kp + (lane >> 4);
                    uint32_t x[4];
                    ldsm_x4(ka + ft * 128 + ((chunk ^ (ft & 7)) << 4), x[0], x[1], x[2], x[3]);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int kk = 2 * kp + h;
                        uint32_t a[4];
                        a[0] = codes_to<T>(static_cast<uint16_t>(x[2 * h] & 0xffffu));
                        a[1] = codes_to<T>(static_cast<uint16_t>(x[2 * h + 1] & 0xffffu));
                        a[2] = codes_to<T>(static_cast<uint16_t>(x[2 * h] >> 16));
                        a[3] = codes_to<T>(static_cast<uint16_t>(x[2 * h + 1] >> 16));
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            if (kk & 1) Mma<T>::run(c2[nt], a, qb[kk][nt][0], qb[kk][nt][1]);
                            else Mma<T>::run(c[nt], a, qb[kk][nt][0], qb[kk][nt][1]);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    uint32_t a[4];
                    ldsm_x4(ka + tile_off<D>(tok, kk * 16 + dsub), a[0], a[1], a[2], a[3]);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (kk & 1) Mma<T>::run(c2[nt], a, qb[kk][nt][0], qb[kk][nt][1]);
                        else Mma<T>::run(c[nt], a, qb[kk][nt][0], qb[kk][nt][1]);
                    }
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) c[nt][e] += c2[nt][e];
        }
        const int r0 = lane >> 2;
        float s[NT][4];
        bool grow = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const bool v0 = !masked || base + r0 < lim[nt][e];
                const bool v8 = !masked || base + r0 + 8 < lim[nt][e];
                s[nt][e] = v0 ? c[nt][e] * scale_log2 : -INFINITY;
                s[nt][2 + e] = v8 ? c[nt][2 + e] * scale_log2 : -INFINITY;
            }
            float mx0 = fmaxf(s[nt][0], s[nt][2]), mx1 = fmaxf(s[nt][1], s[nt][3]);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, off));
            }
            c[nt][0] = mx0;   // the block maxima, kept for the rescale below
            c[nt][1] = mx1;
            // lazy rescale: a column's reference max m moves only when a score
            // exceeds it by more than kLazyRescaleLog2 (weights stay <= 2^8)
            grow |= mx0 > m[nt][0] + kLazyRescaleLog2 || mx1 > m[nt][1] + kLazyRescaleLog2;
        }
        if (__any_sync(kFull, grow)) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float mx = c[nt][e];
                    if (!(mx > m[nt][e] + kLazyRescaleLog2)) continue;
                    // a column that saw no token yet has m = -inf: al = 0
                    const float al = fast_exp2(m[nt][e] - mx);
                    m[nt][e] = mx;
                    l[nt][e] *= al;
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        o[mt][nt][e] *= al;
                        o[mt][nt][2 + e] *= al;
                    }
                }
            }
        }
        uint32_t b0[NT], b1[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            // a column that has seen no visible token keeps m = -inf; its
            // weights are then exp2(-inf - 0) = 0, never exp2(-inf + inf)
            const float mu0 = m[nt][0] == -INFINITY ? 0.f : m[nt][0];
            const float mu1 = m[nt][1] == -INFINITY ? 0.f : m[nt][1];
            const float p0 = fast_exp2(s[nt][0] - mu0), p1 = fast_exp2(s[nt][1] - mu1);
            const float p2 = fast_exp2(s[nt][2] - mu0), p3 = fast_exp2(s[nt][3] - mu1);
            l[nt][0] += p0 + p2;
            l[nt][1] += p1 + p3;
            // P^T as the B operand: lane l needs P[token 2*(l%4)+e (+8)][column l/4].
            using PT = typename std::conditional<kFp8, __half, T>::type;
            const uint32_t lo = Elem<PT>::pack(p0, p1);
            const uint32_t hi = Elem<PT>::pack(p2, p3);
            const int src0 = ((lane & 3) << 3) + (lane >> 3);
            const uint32_t x0 = __shfl_sync(kFull, lo, src0);
            const uint32_t x1 = __shfl_sync(kFull, lo, src0 + 4);
            const uint32_t y0 = __shfl_sync(kFull, hi, src0);
            const uint32_t y1 = __shfl_sync(kFull, hi, src0 + 4);
            const uint32_t sel = ((lane >> 2) & 1) ? 0x7632u : 0x5410u;
            b0[nt] = __byte_perm(x0, x1, sel);
            b1[nt] = __byte_perm(y0, y1, sel);
        }
        if (nvalid < 16) {
            // rows past the sequence end may hold anything (even NaN): p = 0
            // there, but 0 * NaN would poison the product, so clear them.
            // (Rows before the end that a column may not see are cache data
            // of the sequence: finite.)
            const int nchunks = (16 - nvalid) * 8;   // 16-byte chunks per half (per FP8 tile)
            if constexpr (kFp8) {
                uint4* z = reinterpret_cast<uint4*>(vt + nvalid * 128);
                for (int i = lane; i < nchunks; i += 32) z[i] = make_uint4(0, 0, 0, 0);
            } else {
#pragma unroll
                for (int h = 0; h < D / 64; ++h) {
                    uint4* z = reinterpret_cast<uint4*>(vt + h * TileGeom<D>::kHalfBytes + nvalid * 128);
                    for (int i = lane; i < nchunks; i += 32) z[i] = make_uint4(0, 0, 0, 0);
                }
            }
            __syncwarp();
        }
        if constexpr (kFp8) {
            const int ft = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int mp = 0; mp < KS / 2; ++mp) {
                const int chunk = 2 * mp + (lane >> 4);
                uint32_t x[4];
                ldsm_x4_t(va + ft * 128 + ((chunk ^ (ft & 7)) << 4), x[0], x[1], x[2], x[3]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // [dim 2g: tokens 2c, 2c+1 | dim 2g+1: tokens 2c, 2c+1] of tokens 0-7 and 8-15
                    const uint32_t y0 = __byte_perm(x[2 * h], 0u, 0x3120u);
                    const uint32_t y1 = __byte_perm(x[2 * h + 1], 0u, 0x3120u);
                    uint32_t a[4];
                    a[0] = e4m3x2_to_f16x2(static_cast<uint16_t>(y0 & 0xffffu));
                    a[1] = e4m3x2_to_f16x2(static_cast<uint16_t>(y0 >> 16));
                    a[2] = e4m3x2_to_f16x2(static_cast<uint16_t>(y1 & 0xffffu));
                    a[3] = e4m3x2_to_f16x2(static_cast<uint16_t>(y1 >> 16));
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) Mma<__half>::run(o[2 * mp + h][nt], a, b0[nt], b1[nt]);
                }
            }
        } else {
            const int tok = (lane & 7) + ((lane >> 4) & 1) * 8;
            const int dsub = ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                uint32_t a[4];
                ldsm_x4_t(va + tile_off<D>(tok, mt * 16 + dsub), a[0], a[1], a[2], a[3]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) Mma<T>::run(o[mt][nt], a, b0[nt], b1[nt]);
            }
        }
    }
};

// ---------------------------------------------------------------------------
// work list: one unit per (sequence, partition) of every decode or verify row
// ---------------------------------------------------------------------------
// units[k] = (b << 16) | partition; *unit_count = total.  A row here is a
// sequence whose chunk has 1..max_q queries (one query without cu_q_lens).
// A sequence of length 0 (or one rejected by the bounds checks) gets no unit:
// its zero output rows are written here.  Longer chunks of a varlen batch
// belong to the prefill kernels and get none.  Every query of a sequence that
// is split into several partitions gets a partials row, listed in `rows` as
// (b << 3) | query index from row_base[b] on.  Also resets the work counter.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* carry, int& chunk_total) {
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int t = warp_tot[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(kFull, t, off);
            if (lane >= off) t += y;
        }
        warp_tot[lane] = t;
    }
    __syncthreads();
    const int excl = *carry + (warp > 0 ? warp_tot[warp - 1] : 0) + incl - v;
    chunk_total = warp_tot[31];
    __syncthreads();
    if (tid == 0) *carry += chunk_total;
    __syncthreads();
    return excl;
}

// Units are listed longest first: every sequence's full partitions, then the
// shorter last partitions, so the items claimed at the end of a launch are
// the small ones.
__global__ void __launch_bounds__(1024) decode_plan_kernel(const DecodeParams p) {
    __shared__ int warp_tot[32];
    __shared__ int carry_u;
    __shared__ int carry_r;
    const int tid = threadIdx.x;
    // the decode kernel may launch now; it waits for this grid to complete
    // before it reads the list
    pdl_trigger();
    const int P = p.partition_tokens;
    // (length, queries) of row b; queries = 0 when the row is not handled here
    auto row_of = [&](int b, bool record, int& qlen) -> int {
        qlen = 1;
        if (p.cu_q_lens) {
            const int c0 = p.cu_q_lens[b], c1 = p.cu_q_lens[b + 1];
            qlen = c1 - c0;
            if (c0 < 0 || c1 > p.num_rows) {
                // rows outside q / out: none of them is read or written
                if (record && qlen >= 1 && qlen <= PA_VERIFY_MAX_Q_) record_error(p.err, PA_DEVERR_SEQ_LEN_);
                qlen = 0;
                return 0;
            }
            if (qlen < 1 || qlen > PA_VERIFY_MAX_Q_) {
                qlen = 0;
                return 0;
            }
        }
        int n = p.seq_lens[b];
        const bool bad = n < 0 || n > p.max_seq_len || n > p.max_blocks * 16 || qlen > p.max_q ||
                         (qlen > 1 && n < qlen);
        if (bad) {
            if (record) record_error(p.err, PA_DEVERR_SEQ_LEN_);
            n = 0;
        }
        return n;
    };
    int chunk_total = 0;
    // Only inputs are read before the wait: the first 1024 rows' lengths.
    // Every global write comes after it, because the preceding kernel of the
    // stream may still be running -- a previous decode call's kernel allows
    // dependent launch as soon as it starts, and it reads the work list, the
    // counter and the output rows that this plan is about to rewrite.
    int qlen0 = 0;
    const int n0 = tid < p.num_seqs ? row_of(tid, true, qlen0) : 0;
    pdl_wait();
    // pass 1: full partitions, partials rows (and the zero rows of empty sequences)
    if (tid == 0) {
        carry_u = 0;
        carry_r = 0;
    }
    __syncthreads();
    for (int base = 0; base < p.num_seqs; base += 1024) {
        const int b = base + tid;
        int v = 0, vr = 0, qlen = 0;
        if (b < p.num_seqs) {
            int n = n0;
            qlen = qlen0;
            if (base > 0) n = row_of(b, true, qlen);
            if (n > 0) {
                v = n / P;
                vr = n > P ? qlen : 0;
            } else if (qlen > 0) {
                // an empty (or rejected) sequence gets zero rows here
                const int qrow = p.cu_q_lens ? p.cu_q_lens[b] : b;
                uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                                    static_cast<int64_t>(qrow) * p.num_q_heads * p.head_dim);
                for (int i = 0; i < qlen * p.num_q_heads * p.head_dim / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
            }
        }
        const int start = block_exclusive_scan(v, warp_tot, &carry_u, chunk_total);
        for (int i = 0; i < v; ++i)
            p.units[start + i] = static_cast<int32_t>((static_cast<uint32_t>(b) << 16) | static_cast<uint32_t>(i));
        const int rstart = block_exclusive_scan(vr, warp_tot, &carry_r, chunk_total);
        if (vr) {
            p.row_base[b] = rstart;
            for (int i = 0; i < vr; ++i) p.rows[rstart + i] = static_cast<int32_t>((static_cast<uint32_t>(b) << 3) | i);
        }
    }
    // pass 2: the partial last partitions
    for (int base = 0; base < p.num_seqs; base += 1024) {
        const int b = base + tid;
        int v = 0, last = 0, qlen = 0;
        if (b < p.num_seqs) {
            int n = n0;
            if (base > 0) n = row_of(b, false, qlen);
            if (n > 0 && n % P) {
                v = 1;
                last = n / P;
            }
        }
        const int start = block_exclusive_scan(v, warp_tot, &carry_u, chunk_total);
        if (v) p.units[start] = static_cast<int32_t>((static_cast<uint32_t>(b) << 16) | static_cast<uint32_t>(last));
    }
    if (tid == 0) {
        *p.unit_count = carry_u;
        *p.work_counter = 0;
        if (p.row_count) *p.row_count = carry_r;
    }
    // this grid completed only after the previous kernel of the stream (the
    // wait above), so the decode kernel's wait on this grid covers that
    // kernel too (the KV write of the step)
}

// ---------------------------------------------------------------------------
// the decode kernel
// ---------------------------------------------------------------------------
// Persistent, warp-granular: work item w = (unit, kv head, column chunk) is
// one partition of one sequence for one kv head, handled start to finish by a
// single warp, for up to 16 of the (query, head) pairs that read that kv head
// (kMaxNT = 2; 8 when kMaxNT = 1).  Warps claim items from a global counter as
// they go (dynamic balance).  Each warp streams the 16-token blocks of its
// items, in order, through its own ring of shared-memory slots: lane 0 keeps
// the TMA fetches STAGES blocks ahead of the block being computed, claiming
// the next item as soon as the fetches reach the end of the current one, so
// the warp's HBM pipeline never drains between items.  Warps never wait for
// one another.
template <typename T, int D, bool kMma, bool kFp8, int kMaxNT>
__global__ void __launch_bounds__(kDecodeWarps * 32, DecodeShape<D, kFp8, kMma, kMaxNT>::kMinCtasPerSm)
    decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap) {
    static_assert(kMma || kMaxNT == 1, "the FMA path handles one query per row");
    using Shape = DecodeShape<D, kFp8, kMma, kMaxNT>;
    constexpr int kDecodeStages = Shape::kStages;
    constexpr int kQueue = 8;  // claimed items not yet computed (<= STAGES + 1 in use)
    constexpr int kChunkCols = 8 * kMaxNT;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bars[kDecodeWarps * kDecodeStages];
    __shared__ int claimed[kDecodeWarps][kQueue];
    __shared__ uint8_t slot_ok[kDecodeWarps][kDecodeStages];   // the slot's block id was inside the pool

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.group;
    const int H = p.num_kv_heads;
    const int C = p.col_chunks;
    const int P = p.partition_tokens;

    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    WarpRing ring{smem + warp * Shape::kWarpBytes, bars + warp * kDecodeStages};
    if (lane == 0) {
        for (int s = 0; s < kDecodeStages; ++s) mbar_init(&ring.bars[s], 1);
        fence_barrier_init();
    }
    __syncwarp();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    // the work list (and, through it, the KV write) is complete; with
    // p.overlap the preceding kernel is a prefill kernel this one runs beside,
    // and the list was built before that kernel started, so the wait moves to
    // the kernel's exit (below)
    if (!p.overlap) pdl_wait();
    // a reduce launched with programmatic dependent launch may be scheduled
    // now: its CTAs wait on chip for this grid to complete
    pdl_trigger();
    const int total = *p.unit_count * H * C;
    if (total == 0) {
        if (p.overlap) pdl_wait();
        return;
    }
    int* queue = claimed[warp];

    struct Item {
        int b, g, part, n, qlen, qrow0, col0, ncols, tok1, lim_min, blk0, nblk;
        const int32_t* bt;
    };
    auto load_item = [&](int w, Item& it) {
        const int ug = w / C;
        const uint32_t unit = static_cast<uint32_t>(p.units[ug / H]);
        it.g = ug % H;
        it.b = static_cast<int>(unit >> 16);
        it.part = static_cast<int>(unit & 0xffffu);
        it.qlen = 1;
        it.qrow0 = it.b;
        if (p.cu_q_lens) {
            it.qrow0 = p.cu_q_lens[it.b];
            it.qlen = p.cu_q_lens[it.b + 1] - it.qrow0;
        }
        int n = p.seq_lens[it.b];
        if (n < it.qlen || n > p.max_seq_len || n > p.max_blocks * 16 || it.qlen < 1 || it.qlen > p.max_q ||
            it.qrow0 < 0 || it.qrow0 + it.qlen > p.num_rows)
            n = 0;
        it.n = n;
        it.col0 = (w % C) * kChunkCols;
        it.ncols = min(kChunkCols, it.qlen * G - it.col0);
        const int tok0 = it.part * P;
        it.tok1 = min(n, tok0 + P);
        // query q (position n - qlen + q) sees the tokens below n - qlen + q + 1
        it.lim_min = min(it.tok1, n - it.qlen + 1 + it.col0 / G);
        it.blk0 = tok0 >> 4;
        it.nblk = (n > 0 && it.ncols > 0) ? ((it.tok1 + 15) >> 4) - it.blk0 : 0;
        it.bt = p.block_tables + static_cast<int64_t>(it.b) * p.max_blocks + it.blk0;
    };
    // this lane's Q^T words of column tiles 0..NT-1 of an item
    auto load_q_mma = [&](const Item& it, uint32_t* dst, int nt_count) {
        const uint16_t* qbase = static_cast<const uint16_t*>(p.q);
        for (int nt = 0; nt < nt_count; ++nt) {
            const int cl = nt * 8 + (lane >> 2);
            const bool ok = cl < it.ncols;
            const int c = it.col0 + cl;
            const int qi = ok ? c / G : 0;
            const int h = ok ? c - qi * G : 0;
            const uint16_t* qq =
                qbase + (static_cast<int64_t>(it.qrow0 + qi) * p.num_q_heads + it.g * G + h) * D;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                // logical k rows 2c, 2c+1 | 2c+8, 2c+9: dims 2c, 2c+1 | 2c+8, 2c+9
                // (16-bit tiles) or 4c, 4c+1 | 4c+2, 4c+3 (FP8 tiles) of the k-step
                const int d = kk * 16 + (kFp8 ? 4 : 2) * (lane & 3);
                const int d2 = d + (kFp8 ? 2 : 8);
                dst[(kk * nt_count + nt) * 2] = ok ? *reinterpret_cast<const uint32_t*>(qq + d) : 0u;
                dst[(kk * nt_count + nt) * 2 + 1] = ok ? *reinterpret_cast<const uint32_t*>(qq + d2) : 0u;
            }
        }
    };

    // ---- fetch cursor: claims items, loads their blocks ahead ----------------
    uint32_t q_tail = 0, q_head = 0;  // queue of claimed item ids (uniform across lanes)
    Item fi;
    int fblk = 0;
    bool fvalid = false;
    // this lane's query words of the most recently claimed item, loaded at
    // claim time so that they have arrived when the item's compute starts
    // (single-tile kernels only: a wider tile's words stay in memory)
    constexpr bool kPrefetchQ = kMaxNT == 1;
    constexpr int kQWords = kMma ? 2 * (D / 16) : D / 64;
    uint32_t qpre[kQWords];
    int qpre_item = -1;
    auto load_q = [&](const Item& it, uint32_t (&dst)[kQWords]) {
        if constexpr (!kMma) {
            const uint16_t* qq = static_cast<const uint16_t*>(p.q) +
                                 (static_cast<int64_t>(it.qrow0) * p.num_q_heads + it.g) * D;
#pragma unroll
            for (int j = 0; j < kQWords; ++j)
                dst[j] = *reinterpret_cast<const uint32_t*>(qq + lane * AluState<T, D>::DPL + 2 * j);
        } else {
            load_q_mma(it, dst, 1);
        }
    };
    auto claim_next = [&]() {
        for (;;) {
            int w = 0;
            if (lane == 0) w = atomicAdd(p.work_counter, 1);
            w = __shfl_sync(kFull, w, 0);
            if (w >= total) {
                fvalid = false;
                return;
            }
            load_item(w, fi);
            if (fi.nblk == 0) continue;  // a column chunk past the row's last (query, head) pair
            if (lane == 0) queue[q_tail % kQueue] = w;
            ++q_tail;
            if constexpr (kPrefetchQ) {
                load_q(fi, qpre);
                qpre_item = w;
            }
            fblk = 0;
            fvalid = true;
            return;
        }
    };
    uint32_t kf = 0;  // blocks issued so far
    auto issue_next = [&]() {
        if (!fvalid) return;
        const int slot = static_cast<int>(kf % kDecodeStages);
        if (lane == 0) {
            const int phys = fi.bt[fblk];
            slot_ok[warp][slot] = phys >= 0 && phys < p.num_blocks;
            if (phys >= 0 && phys < p.num_blocks) {
                issue_tile<D, kFp8, kMma, kMaxNT>(ring, slot, phys, fi.g, &kmap, &vmap);
            } else {
                record_error(p.err, PA_DEVERR_BLOCK_ID_);
                mbar_arrive(&ring.bars[slot]);  // complete the phase without data
            }
        }
        ++kf;
        if (++fblk >= fi.nblk) claim_next();
    };
    claim_next();
#pragma unroll
    for (int s = 0; s < kDecodeStages; ++s) issue_next();

    // ---- compute: the claimed items in order, their blocks in order ---------
    uint32_t kc = 0;  // blocks consumed so far
    // Walk the item's blocks through the ring; `step(kt, vt, base, nvalid)`
    // consumes one landed block.  False when a wait gave up.
    auto for_each_block = [&](const Item& it, auto&& step) -> bool {
        for (int blk = 0; blk < it.nblk; ++blk, ++kc) {
            const int slot = static_cast<int>(kc % kDecodeStages);
            const bool got = mbar_wait(&ring.bars[slot], (kc / kDecodeStages) & 1u);
            if (__any_sync(kFull, !got)) return false;
            const bool valid = slot_ok[warp][slot];   // written by lane 0 before the slot's TMA
            if (valid) {
                uint8_t* kt = ring.base + slot * Shape::kStageBytes;
                uint8_t* vt = kt + Shape::kTileBytes;
                const int base = (it.blk0 + blk) * 16;
                step(kt, vt, base, min(16, it.tok1 - base));
            }
            // the slot is free again: refill it with the block STAGES ahead
            fence_proxy_async_smem();
            __syncwarp();
            issue_next();
        }
        return true;
    };

    // MHA decode row: fp32 FMA path
    auto run_alu = [&](const Item& it, const uint32_t (&qw)[kQWords]) -> bool {
        AluState<T, D, kFp8> alu;
#pragma unroll
        for (int j = 0; j < kQWords; ++j) {
            if constexpr (AluState<T, D, kFp8>::kMixedK) {
                alu.qh[j] = qw[j];
            } else {
                const float2 f = Elem<T>::to_float2(qw[j]);
                alu.q[2 * j] = f.x * p.scale_log2;
                alu.q[2 * j + 1] = f.y * p.scale_log2;
            }
            alu.acc[2 * j] = 0.f;
            alu.acc[2 * j + 1] = 0.f;
        }
        if constexpr (AluState<T, D, kFp8>::kMixedK) alu.qscale = p.scale_log2;
        if constexpr (AluState<T, D, kFp8>::kTokenK) {
            const uint4* qq = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                             (static_cast<int64_t>(it.qrow0) * p.num_q_heads + it.g) * D +
                                                             (lane & 1) * 64);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint4 v = qq[i];
                alu.qk[4 * i] = v.x; alu.qk[4 * i + 1] = v.y; alu.qk[4 * i + 2] = v.z; alu.qk[4 * i + 3] = v.w;
            }
        }
        alu.m = -INFINITY;
        alu.l = 0.f;
        if (!for_each_block(it, [&](uint8_t* kt, uint8_t* vt, int, int nvalid) { alu.step(kt, vt, nvalid, lane); }))
            return false;
        constexpr int DPL = AluState<T, D>::DPL;
#pragma unroll
        for (int j = 0; j < DPL; ++j) alu.acc[j] *= p.v_scale;
        float lsum = alu.l;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) lsum += __shfl_xor_sync(kFull, lsum, off);
        const int hq = it.g;
        if (it.n <= P) {
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            uint16_t* o = static_cast<uint16_t*>(p.out) + (static_cast<int64_t>(it.qrow0) * p.num_q_heads + hq) * D +
                          lane * DPL;
            if constexpr (DPL == 4) {
                uint2 v;
                v.x = Elem<T>::pack(alu.acc[0] * inv, alu.acc[1] * inv);
                v.y = Elem<T>::pack(alu.acc[2] * inv, alu.acc[3] * inv);
                *reinterpret_cast<uint2*>(o) = v;
            } else {
                *reinterpret_cast<uint32_t*>(o) = Elem<T>::pack(alu.acc[0] * inv, alu.acc[1] * inv);
            }
        } else {
            const int64_t pi = (static_cast<int64_t>(p.row_base[it.b]) * p.num_q_heads + hq) * p.max_parts + it.part;
            if (lane == 0) {
                p.ws_m[pi] = alu.m;
                p.ws_l[pi] = lsum;
            }
#pragma unroll
            for (int j = 0; j < DPL; ++j) p.ws_acc[pi * D + lane * DPL + j] = alu.acc[j];
        }
        return true;
    };

    // (query, head) columns of a decode or verify row: tensor-core path
    auto run_mma = [&](auto nt_tag, const Item& it, int w) -> bool {
        constexpr int NT = decltype(nt_tag)::value;
        MmaState<T, D, NT, kFp8> mma;
        if (kPrefetchQ && NT == 1 && qpre_item == w) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                mma.qb[kk][0][0] = qpre[2 * kk];
                mma.qb[kk][0][1] = qpre[2 * kk + 1];
            }
        } else {
            load_q_mma(it, &mma.qb[0][0][0], NT);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
                for (int e = 0; e < 4; ++e) mma.o[kk][nt][e] = 0.f;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                mma.m[nt][e] = -INFINITY;
                mma.l[nt][e] = 0.f;
                const int cl = nt * 8 + 2 * (lane & 3) + e;
                mma.lim[nt][e] = cl < it.ncols ? min(it.tok1, it.n - it.qlen + 1 + (it.col0 + cl) / G) : 0;
            }
        }
        const bool ok = for_each_block(it, [&](uint8_t* kt, uint8_t* vt, int base, int nvalid) {
            const bool masked = base + 16 > it.lim_min;
            mma.step(kt, vt, base, nvalid, masked, lane, p.scale_log2);
        });
        if (!ok) return false;
        const bool split = it.n > P;
        const int prow = split ? p.row_base[it.b] : 0;
        const int dr = lane >> 2;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float lh = mma.l[nt][e];
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) lh += __shfl_xor_sync(kFull, lh, off);
                const int cl = nt * 8 + 2 * (lane & 3) + e;
                if (cl >= it.ncols) continue;
                const int c = it.col0 + cl;
                const int qi = c / G;
                const int hq = it.g * G + (c - qi * G);
                if (!split) {
                    const float inv = lh > 0.f ? p.v_scale / lh : 0.f;
                    uint16_t* o = static_cast<uint16_t*>(p.out) +
                                  (static_cast<int64_t>(it.qrow0 + qi) * p.num_q_heads + hq) * D;
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        if constexpr (kFp8) {   // rows dr, dr + 8 of the m-tile are dims 2 dr, 2 dr + 1
                            *reinterpret_cast<uint32_t*>(o + mt * 16 + 2 * dr) =
                                Elem<T>::pack(mma.o[mt][nt][e] * inv, mma.o[mt][nt][2 + e] * inv);
                        } else {
                            o[mt * 16 + dr] = Elem<T>::from_float(mma.o[mt][nt][e] * inv);
                            o[mt * 16 + dr + 8] = Elem<T>::from_float(mma.o[mt][nt][2 + e] * inv);
                        }
                    }
                } else {
                    const int64_t pi =
                        (static_cast<int64_t>(prow + qi) * p.num_q_heads + hq) * p.max_parts + it.part;
                    if (dr == 0) {
                        p.ws_m[pi] = mma.m[nt][e];
                        p.ws_l[pi] = lh;
                    }
                    float* a = p.ws_acc + pi * D;
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        if constexpr (kFp8) {
                            *reinterpret_cast<float2*>(a + mt * 16 + 2 * dr) =
                                make_float2(mma.o[mt][nt][e] * p.v_scale, mma.o[mt][nt][2 + e] * p.v_scale);
                        } else {
                            a[mt * 16 + dr] = mma.o[mt][nt][e] * p.v_scale;
                            a[mt * 16 + dr + 8] = mma.o[mt][nt][2 + e] * p.v_scale;
                        }
                    }
                }
            }
        }
        return true;
    };

    bool failed = false;
    while (q_head != q_tail) {
        __syncwarp();
        const int w = queue[q_head % kQueue];
        ++q_head;
        Item it;
        load_item(w, it);
        bool ok;
        if constexpr (!kMma) {
            uint32_t qw[kQWords];
            if (qpre_item == w) {
#pragma unroll
                for (int j = 0; j < kQWords; ++j) qw[j] = qpre[j];
            } else {
                load_q(it, qw);  // the fetch cursor has moved past this item already
            }
            ok = run_alu(it, qw);
        } else if constexpr (kMaxNT == 1) {
            ok = run_mma(std::integral_constant<int, 1>{}, it, w);
        } else {
            ok = it.ncols <= 8 ? run_mma(std::integral_constant<int, 1>{}, it, w)
                               : run_mma(std::integral_constant<int, 2>{}, it, w);
        }
        if (!ok) {
            failed = true;
            break;
        }
    }
    if (failed) {
        if (lane == 0) record_error(p.err, PA_DEVERR_TIMEOUT_);
        // let copies still in flight land before the CTA's memory is reused
        for (uint32_t k = kc; k < kf; ++k) (void)mbar_wait(&ring.bars[k % kDecodeStages], (k / kDecodeStages) & 1u);
    }
    // Beside a prefill kernel (p.overlap) this grid must not complete before
    // that kernel does: whatever the stream runs next (the reduce, the next
    // call) is ordered after this grid only, and may rewrite the output rows
    // or cache blocks the prefill kernel is still using.
    if (p.overlap) pdl_wait();
}

// Merge the partitions of each (query row, q head):
// out = sum_p acc_p 2^(m_p - M) / sum_p l_p 2^(m_p - M), M = max_p m_p.
// One warp per (listed partials row, q head); persistent CTAs of 8 warps
// stride over all of them.  A warp forms its partition weights once in shared
// memory (in passes of kReducePass partitions), then each lane streams
// D / 32 dimensions of every partition's accumulator with vector loads.
constexpr int kReduceWarps = 8;
constexpr int kReducePass = 256;   // partition weights staged per warp per pass

template <typename T, int D>
__global__ void __launch_bounds__(kReduceWarps * 32) decode_reduce_kernel(const DecodeParams p) {
    constexpr int DPL = D / 32;
    __shared__ float sc_all[kReduceWarps][kReducePass];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    float* sc = sc_all[warp];
    pdl_wait();   // the decode kernel's partials (launched with programmatic dependent launch)
    const int P = p.partition_tokens;
    const int64_t pairs = static_cast<int64_t>(*p.row_count) * p.num_q_heads;
    for (int64_t w = static_cast<int64_t>(blockIdx.x) * kReduceWarps + warp; w < pairs;
         w += static_cast<int64_t>(gridDim.x) * kReduceWarps) {
        const int k = static_cast<int>(w / p.num_q_heads);
        const int hq = static_cast<int>(w - static_cast<int64_t>(k) * p.num_q_heads);
        const uint32_t entry = static_cast<uint32_t>(p.rows[k]);
        const int b = static_cast<int>(entry >> 3);
        const int qrow = (p.cu_q_lens ? p.cu_q_lens[b] : b) + static_cast<int>(entry & 7u);
        int n = p.seq_lens[b];
        if (n < 0 || n > p.max_seq_len || n > p.max_blocks * 16) n = 0;
        const int nparts = n > 0 ? (n + P - 1) / P : 1;
        const int64_t base = (static_cast<int64_t>(k) * p.num_q_heads + hq) * p.max_parts;
        const float* wm = p.ws_m + base;
        const float* wl = p.ws_l + base;
        const float* wa = p.ws_acc + base * D + lane * DPL;

        float M = -INFINITY;
        for (int i = lane; i < nparts; i += 32) M = fmaxf(M, wm[i]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));

        float L = 0.f, acc[DPL];
#pragma unroll
        for (int j = 0; j < DPL; ++j) acc[j] = 0.f;
        if (M != -INFINITY) {
            for (int p0 = 0; p0 < nparts; p0 += kReducePass) {
                const int np = min(kReducePass, nparts - p0);
                float lpart = 0.f;
                for (int i = lane; i < np; i += 32) {
                    const float s = fast_exp2(wm[p0 + i] - M);
                    sc[i] = s;
                    lpart = fmaf(wl[p0 + i], s, lpart);
                }
                L += lpart;
                __syncwarp();
                const float* a = wa + static_cast<int64_t>(p0) * D;
#pragma unroll 4
                for (int i = 0; i < np; ++i) {
                    const float s = sc[i];
                    if constexpr (DPL == 4) {
                        const float4 x = *reinterpret_cast<const float4*>(a + static_cast<int64_t>(i) * D);
                        acc[0] = fmaf(x.x, s, acc[0]);
                        acc[1] = fmaf(x.y, s, acc[1]);
                        acc[2] = fmaf(x.z, s, acc[2]);
                        acc[3] = fmaf(x.w, s, acc[3]);
                    } else {
                        const float2 x = *reinterpret_cast<const float2*>(a + static_cast<int64_t>(i) * D);
                        acc[0] = fmaf(x.x, s, acc[0]);
                        acc[1] = fmaf(x.y, s, acc[1]);
                    }
                }
                __syncwarp();   // sc is rewritten by the next pass or pair
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        uint16_t* o = reinterpret_cast<uint16_t*>(p.out) + (static_cast<int64_t>(qrow) * p.num_q_heads + hq) * D +
                      lane * DPL;
        if constexpr (DPL == 4) {
            uint2 v;
            v.x = Elem<T>::pack(acc[0] * inv, acc[1] * inv);
            v.y = Elem<T>::pack(acc[2] * inv, acc[3] * inv);
            *reinterpret_cast<uint2*>(o) = v;
        } else {
            *reinterpret_cast<uint32_t*>(o) = Elem<T>::pack(acc[0] * inv, acc[1] * inv);
        }
    }
}

// The same merge with a whole CTA per (listed partials row, q head): for
// launches with few pairs and many partitions (long contexts), where one warp
// per pair would leave most SMs idle.  The per-partition weights are formed
// once in shared memory; each thread then streams one head dimension of every
// partition's accumulator.
constexpr int kReduceMaxParts = 1024;   // partitions staged in shared memory per pass
constexpr int kReduceMaxRowsPerLaunch = 2048;
// below this many (row, q head) pairs a whole CTA merges each pair
constexpr long long kReduceWarpPairsMin = 1024;

template <typename T, int D>
__global__ void __launch_bounds__(D) decode_reduce_cta_kernel(const DecodeParams p) {
    __shared__ float sc[kReduceMaxParts];
    __shared__ float red[D / 32];
    const int hq = blockIdx.x;
    const int d = threadIdx.x;
    const int P = p.partition_tokens;
    const int nrows = *p.row_count;
    for (int k = blockIdx.y; k < nrows; k += gridDim.y) {
        const uint32_t entry = static_cast<uint32_t>(p.rows[k]);
        const int b = static_cast<int>(entry >> 3);
        const int qrow = (p.cu_q_lens ? p.cu_q_lens[b] : b) + static_cast<int>(entry & 7u);
        int n = p.seq_lens[b];
        if (n < 0 || n > p.max_seq_len || n > p.max_blocks * 16) n = 0;
        const int nparts = n > 0 ? (n + P - 1) / P : 1;
        const int64_t base = (static_cast<int64_t>(k) * p.num_q_heads + hq) * p.max_parts;
        const float* wm = p.ws_m + base;
        const float* wl = p.ws_l + base;
        const float* wa = p.ws_acc + base * D;

        // M = max_p m_p (block reduction)
        float M = -INFINITY;
        for (int i = d; i < nparts; i += D) M = fmaxf(M, wm[i]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
        if ((d & 31) == 0) red[d >> 5] = M;
        __syncthreads();
        M = red[0];
#pragma unroll
        for (int w = 1; w < D / 32; ++w) M = fmaxf(M, red[w]);
        __syncthreads();

        float L = 0.f, A = 0.f;
        if (M != -INFINITY) {
            for (int p0 = 0; p0 < nparts; p0 += kReduceMaxParts) {
                const int np = min(kReduceMaxParts, nparts - p0);
                float lpart = 0.f;
                for (int i = d; i < np; i += D) {
                    const float s = fast_exp2(wm[p0 + i] - M);
                    sc[i] = s;
                    lpart = fmaf(wl[p0 + i], s, lpart);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) lpart += __shfl_xor_sync(kFull, lpart, off);
                if ((d & 31) == 0) red[d >> 5] = lpart;
                __syncthreads();
#pragma unroll
                for (int w = 0; w < D / 32; ++w) L += red[w];
                const float* a = wa + static_cast<int64_t>(p0) * D + d;
                int i = 0;
                for (; i + 8 <= np; i += 8) {
                    float x[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) x[u] = a[static_cast<int64_t>(i + u) * D];
#pragma unroll
                    for (int u = 0; u < 8; ++u) A = fmaf(x[u], sc[i + u], A);
                }
                for (; i < np; ++i) A = fmaf(a[static_cast<int64_t>(i) * D], sc[i], A);
                __syncthreads();
            }
        }
        const float v = L > 0.f ? A / L : 0.f;
        reinterpret_cast<uint16_t*>(p.out)[(static_cast<int64_t>(qrow) * p.num_q_heads + hq) * D + d] =
            Elem<T>::from_float(v);
    }
}


template <typename T, int D, bool kMma, bool kFp8 = false, int kMaxNT = 1>
cudaError_t launch_decode_t(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                            cudaStream_t s) {
    constexpr int smem = DecodeShape<D, kFp8, kMma, kMaxNT>::kSmemBytes;
    auto kern = decode_kernel<T, D, kMma, kFp8, kMaxNT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (!p.overlap) {
        e = launch_pdl(decode_plan_kernel, dim3(1), dim3(1024), 0, s, p);
        if (e != cudaSuccess) return e;
    }
    // persistent: as many CTAs as are resident on every SM at once (shared
    // memory and registers), fewer when there cannot be that many items; a
    // CTA beyond that would only start once the work is nearly gone
    static const int ctas_per_sm = [&] {   // once per kernel variant (thread-safe)
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kDecodeWarps * 32, smem) != cudaSuccess || n < 1)
            n = 1;
        return n;
    }();
    const long long max_items =
        static_cast<long long>(p.num_seqs) * p.max_parts * p.num_kv_heads * p.col_chunks;
    const long long want = (max_items + kDecodeWarps - 1) / kDecodeWarps;
    const int grid = static_cast<int>(
        std::max<long long>(1, std::min<long long>(want, static_cast<long long>(ctas_per_sm) * sm_count())));
    e = launch_pdl(kern, dim3(grid), dim3(kDecodeWarps * 32), smem, s, p, kmap, vmap);
    if (e != cudaSuccess) return e;
    if (p.max_parts > 1) {
        const long long pairs = static_cast<long long>(p.max_rows) * p.num_q_heads;
        if (pairs >= kReduceWarpPairsMin) {
            // persistent: a few waves of 8-warp CTAs, one warp per pair
            const int rgrid = static_cast<int>(std::max<long long>(
                1, std::min<long long>((pairs + kReduceWarps - 1) / kReduceWarps, 8LL * sm_count())));
            // scheduled while the decode grid drains (its CTAs wait on chip);
            // the CTA-per-pair layout below has too many CTAs for that to pay
            e = launch_pdl(decode_reduce_kernel<T, D>, dim3(rgrid), dim3(kReduceWarps * 32), 0, s, p);
        } else {
            dim3 rgrid(p.num_q_heads, std::min(p.max_rows, kReduceMaxRowsPerLaunch));
            decode_reduce_cta_kernel<T, D><<<rgrid, D, 0, s>>>(p);
            e = cudaGetLastError();
        }
    }
    return e;
}

}  // namespace

int sm_count() {
    static std::atomic<int> count[64];   // per device, 0 until first asked
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int c = count[dev].load(std::memory_order_relaxed);
    if (!c) {
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) c = 148;
        count[dev].store(c, std::memory_order_relaxed);
    }
    return c;
}

cudaError_t launch_decode_plan(const DecodeParams& p, cudaStream_t s) {
    if (p.num_seqs == 0) return cudaSuccess;
    decode_plan_kernel<<<1, 1024, 0, s>>>(p);
    return cudaGetLastError();
}

// FP8 cache: one query per row and one q head per kv head on the FMA path;
// several (query, head) columns per kv head (GQA, or the queries of a
// speculative-verify row) on the tensor cores, with a second column tile
// once a row has more than 8 columns.
template <typename T>
cudaError_t launch_decode_fp8_t(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                cudaStream_t s) {
    if (p.max_q * p.group > 8) return launch_decode_t<T, 128, true, true, 2>(p, kmap, vmap, s);
    if (p.group > 1 || p.max_q > 1) return launch_decode_t<T, 128, true, true, 1>(p, kmap, vmap, s);
    return launch_decode_t<T, 128, false, true, 1>(p, kmap, vmap, s);
}

cudaError_t launch_decode_fp8(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                              int dtype, cudaStream_t s) {
    if (p.num_seqs == 0) return cudaSuccess;
    return dtype == 0 ? launch_decode_fp8_t<__half>(p, kmap, vmap, s)
                      : launch_decode_fp8_t<__nv_bfloat16>(p, kmap, vmap, s);
}

template <typename T, int D>
cudaError_t launch_decode_d(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                            cudaStream_t s) {
    if (p.max_q * p.group > 8) return launch_decode_t<T, D, true, false, 2>(p, kmap, vmap, s);
    if (p.group > 1 || p.max_q > 1) return launch_decode_t<T, D, true, false, 1>(p, kmap, vmap, s);
    return launch_decode_t<T, D, false, false, 1>(p, kmap, vmap, s);
}

cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          int head_dim, int dtype, cudaStream_t s) {
    if (p.num_seqs == 0) return cudaSuccess;
    if (dtype == 0)
        return head_dim == 128 ? launch_decode_d<__half, 128>(p, kmap, vmap, s)
                               : launch_decode_d<__half, 64>(p, kmap, vmap, s);
    return head_dim == 128 ? launch_decode_d<__nv_bfloat16, 128>(p, kmap, vmap, s)
                           : launch_decode_d<__nv_bfloat16, 64>(p, kmap, vmap, s);
}

}  // namespace pa
