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
//  * grid (partition, kv head, sequence); a CTA handles the `group` query
//    heads that share one kv head, so every K/V byte is read once.
//  * each warp owns a private ring of STAGES shared-memory slots; its lane 0
//    fetches whole (16-token block, kv head) tiles of K and V with 4-D TMA
//    loads (one per 64-dim half, 128-byte swizzle), completing on a per-slot
//    mbarrier.
//  * MHA (group 1): fp32 FMA dot products, a 16-way transpose-reduction
//    across the warp (16 shuffles per block), register-resident (m, l, acc).
//  * GQA (group 2..8): the query group x K-block product is a dense
//    contraction: S^T[16 tokens x 8 heads] = K Q^T and O^T += V^T P^T with
//    mma.sync m16n8k16 (fp32 accumulate); M = 16 tokens matches the block.
//  * warps of a CTA merge their states through shared memory at the end.
#include "pa_device.cuh"

namespace pa {

namespace {

constexpr int kDecodeWarps = 4;
constexpr int kDecodeStages = 3;
constexpr unsigned kFull = 0xffffffffu;

template <int D>
struct DecodeShape {
    static constexpr int kTileBytes = 16 * D * 2;         // one (block, kv head) tile
    static constexpr int kStageBytes = 2 * kTileBytes;    // K tile + V tile
    static constexpr int kWarpBytes = kDecodeStages * kStageBytes;
    static constexpr int kSmemBytes = kDecodeWarps * kWarpBytes + 1024;  // + alignment slack
};

// Per-warp TMA producer state for one CTA's partition.
struct WarpRing {
    uint8_t* base;      // this warp's STAGES slots
    uint64_t* bars;     // STAGES mbarriers
};

template <int D>
__device__ __forceinline__ void issue_tile(const WarpRing& ring, int slot, int phys, int kv_head,
                                          const CUtensorMap* kmap, const CUtensorMap* vmap) {
    uint8_t* dst = ring.base + slot * DecodeShape<D>::kStageBytes;
    mbar_arrive_expect_tx(&ring.bars[slot], DecodeShape<D>::kStageBytes);
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
        tma_load_4d(dst + h * TileGeom<D>::kHalfBytes, kmap, &ring.bars[slot], 0, h, kv_head, phys * 16);
        tma_load_4d(dst + DecodeShape<D>::kTileBytes + h * TileGeom<D>::kHalfBytes, vmap, &ring.bars[slot], 0, h,
                    kv_head, phys * 16);
    }
}

// ---------------------------------------------------------------------------
// MHA block step: fp32 dot products on the ALU.
// Lane l owns head dims [l*DPL, (l+1)*DPL).
// ---------------------------------------------------------------------------
template <typename T, int D>
struct AluState {
    static constexpr int DPL = D / 32;
    float q[DPL];
    float acc[DPL];
    float m;
    float l;  // this lane's share (even lanes only)

    __device__ __forceinline__ void load_dims(const uint8_t* tile, int tok, int lane, float* x) const {
        if constexpr (DPL == 4) {
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
        float part[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            float k[DPL];
            load_dims(kt, t, lane, k);
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < DPL; ++j) s = fmaf(q[j], k[j], s);
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
        float s = part[0] + __shfl_xor_sync(kFull, part[0], 1);
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

// ---------------------------------------------------------------------------
// GQA block step on the tensor cores (mma.sync m16n8k16, fp32 accumulate).
// S^T = K Q^T: rows = 16 tokens of the block, cols = 8 (padded) query heads.
// Lane l holds S^T rows l/4 and l/4+8, head columns 2*(l%4) and 2*(l%4)+1;
// O^T (head_dim x heads) uses the same columns, so the per-head rescale needs
// no data movement.
// ---------------------------------------------------------------------------
template <typename T, int D>
struct MmaState {
    static constexpr int KS = D / 16;
    uint32_t qb[KS][2];   // Q^T as the B operand, per 16-dim k-step
    float o[KS][4];       // O^T accumulator, per 16-dim m-tile
    float m[2];
    float l[2];

    __device__ __forceinline__ void step(uint8_t* kt, uint8_t* vt, int nvalid, int lane, float scale_log2) {
        const uint32_t ka = smem_addr(kt);
        const uint32_t va = smem_addr(vt);
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int dsub = ((lane >> 4) & 1) * 8;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                uint32_t a[4];
                ldsm_x4(ka + tile_off<D>(tok, kk * 16 + dsub), a[0], a[1], a[2], a[3]);
                Mma<T>::run(c, a, qb[kk][0], qb[kk][1]);
            }
        }
        const int r0 = lane >> 2;
        float s0 = r0 < nvalid ? c[0] * scale_log2 : -INFINITY;
        float s1 = r0 < nvalid ? c[1] * scale_log2 : -INFINITY;
        float s2 = r0 + 8 < nvalid ? c[2] * scale_log2 : -INFINITY;
        float s3 = r0 + 8 < nvalid ? c[3] * scale_log2 : -INFINITY;
        float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, off));
        }
        const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
        const float al0 = fast_exp2(m[0] - mn0), al1 = fast_exp2(m[1] - mn1);
        m[0] = mn0;
        m[1] = mn1;
        const float p0 = fast_exp2(s0 - mn0), p1 = fast_exp2(s1 - mn1);
        const float p2 = fast_exp2(s2 - mn0), p3 = fast_exp2(s3 - mn1);
        l[0] = l[0] * al0 + p0 + p2;
        l[1] = l[1] * al1 + p1 + p3;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            o[mt][0] *= al0;
            o[mt][1] *= al1;
            o[mt][2] *= al0;
            o[mt][3] *= al1;
        }
        // P^T as the B operand: lane l needs P[token 2*(l%4)+e (+8)][head l/4].
        const uint32_t lo = Elem<T>::pack(p0, p1);
        const uint32_t hi = Elem<T>::pack(p2, p3);
        const int src0 = ((lane & 3) << 3) + (lane >> 3);
        const uint32_t x0 = __shfl_sync(kFull, lo, src0);
        const uint32_t x1 = __shfl_sync(kFull, lo, src0 + 4);
        const uint32_t y0 = __shfl_sync(kFull, hi, src0);
        const uint32_t y1 = __shfl_sync(kFull, hi, src0 + 4);
        const uint32_t sel = ((lane >> 2) & 1) ? 0x7632u : 0x5410u;
        const uint32_t b0 = __byte_perm(x0, x1, sel);
        const uint32_t b1 = __byte_perm(y0, y1, sel);
        if (nvalid < 16) {
            // rows past the sequence end may hold anything (even NaN): p = 0
            // there, but 0 * NaN would poison the product, so clear them.
            const int nchunks = (16 - nvalid) * 8;   // 16-byte chunks per half
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                uint4* z = reinterpret_cast<uint4*>(vt + h * TileGeom<D>::kHalfBytes + nvalid * 128);
                for (int i = lane; i < nchunks; i += 32) z[i] = make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
        }
        {
            const int tok = (lane & 7) + ((lane >> 4) & 1) * 8;
            const int dsub = ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                uint32_t a[4];
                ldsm_x4_t(va + tile_off<D>(tok, mt * 16 + dsub), a[0], a[1], a[2], a[3]);
                Mma<T>::run(o[mt], a, b0, b1);
            }
        }
    }
};

// ---------------------------------------------------------------------------
// the decode kernel
// ---------------------------------------------------------------------------
template <typename T, int D, bool kMma>
__global__ void __launch_bounds__(kDecodeWarps * 32)
    decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap) {
    using Shape = DecodeShape<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bars[kDecodeWarps * kDecodeStages];
    __shared__ int any_timeout;

    const int part = blockIdx.x;
    const int g = blockIdx.y;
    const int b = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.group;

    int qrow = b;
    if (p.cu_q_lens) {
        const int r0 = p.cu_q_lens[b];
        if (p.cu_q_lens[b + 1] - r0 != 1) return;  // not a decode row
        qrow = r0;
    }
    int n = p.seq_lens[b];
    if (n < 0 || n > p.max_seq_len || n > p.max_blocks * 16) {
        if (part == 0 && g == 0 && threadIdx.x == 0) record_error(p.err, PA_DEVERR_SEQ_LEN_);
        n = 0;  // defined result: a zero row
    }
    const int P = p.partition_tokens;
    const int nparts = n > 0 ? (n + P - 1) / P : 1;
    if (part >= nparts) return;
    const int tok0 = part * P;
    const int tok1 = min(n, tok0 + P);
    const int blk0 = tok0 >> 4;
    const int nblk = n > 0 ? ((tok1 + 15) >> 4) - blk0 : 0;
    const int32_t* bt = p.block_tables + static_cast<int64_t>(b) * p.max_blocks + blk0;

    // 1024-byte aligned slot area (the 128-byte swizzle pattern repeats every 1 KiB)
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kDecodeWarps * kDecodeStages; ++i) mbar_init(&bars[i], 1);
        any_timeout = 0;
        fence_barrier_init();
    }
    __syncthreads();

    WarpRing ring{smem + warp * Shape::kWarpBytes, bars + warp * kDecodeStages};
    const int64_t q_base = (static_cast<int64_t>(qrow) * p.num_q_heads + g * G) * D;
    const T* q = static_cast<const T*>(p.q) + q_base;

    // prologue: fill the ring
    uint32_t inflight = 0;
#pragma unroll
    for (int s = 0; s < kDecodeStages; ++s) {
        const int i = warp + s * kDecodeWarps;
        if (i < nblk) {
            const int phys = bt[i];
            if (phys >= 0 && phys < p.num_blocks) {
                inflight |= 1u << s;
                if (lane == 0) issue_tile<D>(ring, s, phys, g, &kmap, &vmap);
            } else if (lane == 0) {
                record_error(p.err, PA_DEVERR_BLOCK_ID_);
            }
        }
    }

    AluState<T, D> alu;
    MmaState<T, D> mma;
    if constexpr (!kMma) {
        const uint16_t* qq = reinterpret_cast<const uint16_t*>(q);
#pragma unroll
        for (int j = 0; j < AluState<T, D>::DPL; j += 2) {
            const uint32_t raw = *reinterpret_cast<const uint32_t*>(qq + lane * AluState<T, D>::DPL + j);
            const float2 f = Elem<T>::to_float2(raw);
            alu.q[j] = f.x * p.scale_log2;
            alu.q[j + 1] = f.y * p.scale_log2;
            alu.acc[j] = 0.f;
            alu.acc[j + 1] = 0.f;
        }
        alu.m = -INFINITY;
        alu.l = 0.f;
    } else {
        const int hh = lane >> 2;
        const uint16_t* qq = reinterpret_cast<const uint16_t*>(q);
#pragma unroll
        for (int kk = 0; kk < MmaState<T, D>::KS; ++kk) {
            const int d = kk * 16 + 2 * (lane & 3);
            mma.qb[kk][0] = hh < G ? *reinterpret_cast<const uint32_t*>(qq + hh * D + d) : 0u;
            mma.qb[kk][1] = hh < G ? *reinterpret_cast<const uint32_t*>(qq + hh * D + d + 8) : 0u;
#pragma unroll
            for (int e = 0; e < 4; ++e) mma.o[kk][e] = 0.f;
        }
        mma.m[0] = mma.m[1] = -INFINITY;
        mma.l[0] = mma.l[1] = 0.f;
    }

    uint32_t phases = 0;
    bool timed_out = false;
    for (int it = 0;; ++it) {
        const int i = warp + it * kDecodeWarps;
        if (i >= nblk) break;
        const int s = it % kDecodeStages;
        if (inflight & (1u << s)) {
            const bool got = mbar_wait(&ring.bars[s], (phases >> s) & 1u);
            if (__any_sync(kFull, !got)) {
                timed_out = true;
                break;
            }
            phases ^= 1u << s;
            inflight &= ~(1u << s);
            uint8_t* kt = ring.base + s * Shape::kStageBytes;
            uint8_t* vt = kt + Shape::kTileBytes;
            const int nvalid = min(16, tok1 - (blk0 + i) * 16);
            if constexpr (!kMma)
                alu.step(kt, vt, nvalid, lane);
            else
                mma.step(kt, vt, nvalid, lane, p.scale_log2);
        }
        // refill this slot with the warp's block STAGES iterations ahead
        const int i2 = i + kDecodeStages * kDecodeWarps;
        if (i2 < nblk) {
            const int phys = bt[i2];
            fence_proxy_async_smem();
            __syncwarp();
            if (phys >= 0 && phys < p.num_blocks) {
                inflight |= 1u << s;
                if (lane == 0) issue_tile<D>(ring, s, phys, g, &kmap, &vmap);
            } else if (lane == 0) {
                record_error(p.err, PA_DEVERR_BLOCK_ID_);
            }
        }
    }
    if (timed_out) {
        if (lane == 0) {
            record_error(p.err, PA_DEVERR_TIMEOUT_);
            atomicOr(&any_timeout, 1);
        }
        // let copies still in flight land before the CTA's memory is reused
        for (int s = 0; s < kDecodeStages; ++s)
            if (inflight & (1u << s)) (void)mbar_wait(&ring.bars[s], (phases >> s) & 1u);
    }

    // ---- merge the warps' (m, l, acc) -------------------------------------
    __syncthreads();
    float* red_m = reinterpret_cast<float*>(smem);                   // [NW][8]
    float* red_l = red_m + kDecodeWarps * 8;                         // [NW][8]
    float* red_acc = red_l + kDecodeWarps * 8;                       // [NW][8][D]
    if constexpr (!kMma) {
        float lsum = alu.l;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) lsum += __shfl_xor_sync(kFull, lsum, off);
        if (lane == 0) {
            red_m[warp * 8] = alu.m;
            red_l[warp * 8] = lsum;
        }
#pragma unroll
        for (int j = 0; j < AluState<T, D>::DPL; ++j) red_acc[(warp * 8) * D + lane * AluState<T, D>::DPL + j] = alu.acc[j];
    } else {
        float l0 = mma.l[0], l1 = mma.l[1];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(kFull, l0, off);
            l1 += __shfl_xor_sync(kFull, l1, off);
        }
        const int h0 = 2 * (lane & 3);
        if (lane < 4) {
            red_m[warp * 8 + h0] = mma.m[0];
            red_m[warp * 8 + h0 + 1] = mma.m[1];
            red_l[warp * 8 + h0] = l0;
            red_l[warp * 8 + h0 + 1] = l1;
        }
        const int dr = lane >> 2;
#pragma unroll
        for (int mt = 0; mt < MmaState<T, D>::KS; ++mt) {
            red_acc[(warp * 8 + h0) * D + mt * 16 + dr] = mma.o[mt][0];
            red_acc[(warp * 8 + h0 + 1) * D + mt * 16 + dr] = mma.o[mt][1];
            red_acc[(warp * 8 + h0) * D + mt * 16 + dr + 8] = mma.o[mt][2];
            red_acc[(warp * 8 + h0 + 1) * D + mt * 16 + dr + 8] = mma.o[mt][3];
        }
    }
    __syncthreads();
    if (any_timeout) return;

    const int heads = kMma ? G : 1;
    for (int idx = threadIdx.x; idx < heads * D; idx += kDecodeWarps * 32) {
        const int h = idx / D;
        const int d = idx - h * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, red_m[w * 8 + h]);
        float L = 0.f, A = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kDecodeWarps; ++w) {
                const float sc = fast_exp2(red_m[w * 8 + h] - M);
                L = fmaf(red_l[w * 8 + h], sc, L);
                A = fmaf(red_acc[(w * 8 + h) * D + d], sc, A);
            }
        }
        const int hq = g * G + h;
        if (nparts == 1) {
            const float v = L > 0.f ? A / L : 0.f;
            reinterpret_cast<uint16_t*>(p.out)[(static_cast<int64_t>(qrow) * p.num_q_heads + hq) * D + d] =
                Elem<T>::from_float(v);
        } else {
            const int64_t pi = (static_cast<int64_t>(b) * p.num_q_heads + hq) * p.max_parts + part;
            if (d == 0) {
                p.ws_m[pi] = M;
                p.ws_l[pi] = L;
            }
            p.ws_acc[pi * D + d] = A;
        }
    }
}

// Merge the partitions of each (sequence, q head):
// out = sum_p acc_p 2^(m_p - M) / sum_p l_p 2^(m_p - M), M = max_p m_p.
// The per-partition weights are formed once in shared memory; each thread then
// streams one head dimension of every partition's accumulator.
constexpr int kReduceMaxParts = 1024;   // partitions staged in shared memory per pass

template <typename T, int D>
__global__ void __launch_bounds__(D) decode_reduce_kernel(const DecodeParams p) {
    __shared__ float sc[kReduceMaxParts];
    __shared__ float red[D / 32];
    const int hq = blockIdx.x;
    const int b = blockIdx.y;
    const int d = threadIdx.x;
    int qrow = b;
    if (p.cu_q_lens) {
        const int r0 = p.cu_q_lens[b];
        if (p.cu_q_lens[b + 1] - r0 != 1) return;
        qrow = r0;
    }
    int n = p.seq_lens[b];
    if (n < 0 || n > p.max_seq_len || n > p.max_blocks * 16) n = 0;
    const int P = p.partition_tokens;
    const int nparts = n > 0 ? (n + P - 1) / P : 1;
    if (nparts <= 1) return;
    const int64_t base = (static_cast<int64_t>(b) * p.num_q_heads + hq) * p.max_parts;
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

template <typename T, int D, bool kMma>
cudaError_t launch_decode_t(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                            cudaStream_t s) {
    constexpr int smem = DecodeShape<D>::kSmemBytes;
    auto kern = decode_kernel<T, D, kMma>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.max_parts, p.num_kv_heads, p.num_seqs);
    kern<<<grid, kDecodeWarps * 32, smem, s>>>(p, kmap, vmap);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (p.max_parts > 1) {
        dim3 rgrid(p.num_q_heads, p.num_seqs);
        decode_reduce_kernel<T, D><<<rgrid, D, 0, s>>>(p);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          int head_dim, int dtype, cudaStream_t s) {
    if (p.num_seqs == 0) return cudaSuccess;
    const bool mma = p.group > 1;
    if (dtype == 0) {
        if (head_dim == 128)
            return mma ? launch_decode_t<__half, 128, true>(p, kmap, vmap, s)
                       : launch_decode_t<__half, 128, false>(p, kmap, vmap, s);
        return mma ? launch_decode_t<__half, 64, true>(p, kmap, vmap, s)
                   : launch_decode_t<__half, 64, false>(p, kmap, vmap, s);
    }
    if (head_dim == 128)
        return mma ? launch_decode_t<__nv_bfloat16, 128, true>(p, kmap, vmap, s)
                   : launch_decode_t<__nv_bfloat16, 128, false>(p, kmap, vmap, s);
    return mma ? launch_decode_t<__nv_bfloat16, 64, true>(p, kmap, vmap, s)
               : launch_decode_t<__nv_bfloat16, 64, false>(p, kmap, vmap, s);
}

}  // namespace pa
