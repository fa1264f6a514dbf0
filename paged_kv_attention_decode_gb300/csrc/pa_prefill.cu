// Chunked-prefill attention over the paged KV cache.
//
// What is computed ("vLLM-Ascend 原理", section 2.3 "因果自注意力": the query
// at position i attends to positions 0..i; section 2.4: once a prompt is
// chunked, a later chunk's attention reads the KV that earlier chunks wrote):
// query row i of sequence b sits at position seq_len - q_len + i and attends,
// through the block table, to every cached position up to its own.  The
// score matrix never leaves the chip (the fused-attention principle of the
// same page, section 4 "ATB 算子").
//
// GB300 design: one CTA per (query tile, kv head, sequence).  Its 64 rows are
// (query, q head) pairs of one kv-head group, so a K/V tile is loaded once for
// all the group's heads.  A producer warp gathers 64-token K/V tiles (four
// 16-token blocks, 4-D TMA loads per 64-dim half, 128-byte swizzle) into a
// two-stage ring;
// four consumer warps run Q K^T and P V on the tensor cores (mma.sync
// m16n8k16, fp32 accumulate) with an online softmax per row.  Only tiles on
// the causal diagonal are masked.
#include "pa_device.cuh"

namespace pa {

namespace {

constexpr int kPreConsumers = 4;
constexpr int kPreThreads = (kPreConsumers + 1) * 32;
constexpr int kPreRows = 64;
constexpr int kPreKeys = 64;
constexpr int kPreStages = 2;
constexpr unsigned kFull = 0xffffffffu;

template <int D>
struct PrefillShape {
    static constexpr int kBlockTile = 16 * D * 2;
    static constexpr int kHalf = 4 * kBlockTile;           // 64 keys of K (or V)
    static constexpr int kStageBytes = 2 * kHalf;
    static constexpr int kQBytes = kPreRows * D * 2;
    static constexpr int kSmemBytes = kPreStages * kStageBytes + kQBytes + 1024;
};

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kPreConsumers * 32) : "memory");
}

template <typename T, int D>
__global__ void __launch_bounds__(kPreThreads, 2)
    prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap) {
    using Shape = PrefillShape<D>;
    constexpr int KS = D / 16;   // k-steps over head dims
    constexpr int NT = D / 8;    // n-tiles over head dims (P V)
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full_bar[kPreStages];
    __shared__ uint64_t empty_bar[kPreStages];
    __shared__ uint32_t bad_mask[kPreStages];
    __shared__ int abort_flag;

    const int b = blockIdx.z;
    const int g = blockIdx.y;
    const int qt = gridDim.x - 1 - blockIdx.x;  // heaviest tiles first
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.group;
    const int QT = p.q_per_tile;

    const int row0 = p.cu_q_lens[b];
    const int qlen = p.cu_q_lens[b + 1] - row0;
    if (qlen <= PA_VERIFY_MAX_Q_) return;  // decode and verify rows run in the decode kernel
    const int q0 = qt * QT;
    if (q0 >= qlen) return;
    const int n = p.seq_lens[b];
    if (n < qlen || n > p.max_seq_len || n > p.max_blocks * 16) {
        if (qt == 0 && g == 0 && threadIdx.x == 0) record_error(p.err, PA_DEVERR_SEQ_LEN_);
        return;
    }
    const int q_last = min(qlen, q0 + QT) - 1;       // last query of this tile
    const int pos_min = n - qlen + q0;
    const int pos_max = n - qlen + q_last;
    const int n_keys = pos_max + 1;
    const int nkt = (n_keys + kPreKeys - 1) / kPreKeys;
    const int nblk_live = (n_keys + 15) >> 4;
    const int32_t* bt = p.block_tables + static_cast<int64_t>(b) * p.max_blocks;

    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* qs = smem + kPreStages * Shape::kStageBytes;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPreStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], kPreConsumers);
        }
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kPreConsumers) {
        // ----------------------------- producer -----------------------------
        if (lane == 0) {
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
            for (int kt = 0; kt < nkt; ++kt) {
                const int s = kt % kPreStages;
                if (kt >= kPreStages) {
                    if (!mbar_wait(&empty_bar[s], ((kt / kPreStages) - 1) & 1)) {
                        record_error(p.err, PA_DEVERR_TIMEOUT_);
                        atomicOr(&abort_flag, 1);
                        break;
                    }
                }
                if (*(volatile int*)&abort_flag) break;
                uint32_t bytes = 0, bad = 0;
                int phys[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int blk = kt * 4 + j;
                    phys[j] = -1;
                    if (blk < nblk_live) {
                        const int id = bt[blk];
                        if (id >= 0 && id < p.num_blocks) {
                            phys[j] = id;
                            bytes += 2 * Shape::kBlockTile;
                        } else {
                            bad |= 1u << j;
                            record_error(p.err, PA_DEVERR_BLOCK_ID_);
                        }
                    }
                }
                bad_mask[s] = bad;
                uint8_t* st = smem + s * Shape::kStageBytes;
                mbar_arrive_expect_tx(&full_bar[s], bytes);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (phys[j] >= 0) {
#pragma unroll
                        for (int h = 0; h < D / 64; ++h) {
                            tma_load_4d(st + j * Shape::kBlockTile + h * TileGeom<D>::kHalfBytes, &kmap,
                                        &full_bar[s], 0, h, g, phys[j] * 16);
                            tma_load_4d(st + Shape::kHalf + j * Shape::kBlockTile + h * TileGeom<D>::kHalfBytes,
                                        &vmap, &full_bar[s], 0, h, g, phys[j] * 16);
                        }
                    }
                }
            }
        }
        return;
    }

    // ------------------------------ consumers -------------------------------
    // Q tile -> shared memory (same swizzled row format as the K/V tiles)
    {
        constexpr int CPR = D / 8;  // 16-byte chunks per row
        const T* qg = static_cast<const T*>(p.q);
        for (int idx = threadIdx.x; idx < kPreRows * CPR; idx += kPreConsumers * 32) {
            const int r = idx / CPR;
            const int c = idx - r * CPR;
            const int qi = q0 + r / G;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < QT * G && qi < qlen) {
                const int64_t grow = static_cast<int64_t>(row0 + qi) * p.num_q_heads + g * G + (r % G);
                v = *reinterpret_cast<const uint4*>(qg + grow * D + c * 8);
            }
            *reinterpret_cast<uint4*>(qs + tile_off<D>(r, c * 8)) = v;
        }
    }
    consumer_sync();

    uint32_t qa[KS][4];
    {
        const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int dsub = ((lane >> 4) & 1) * 8;
        const uint32_t qaddr = smem_addr(qs);
#pragma unroll
        for (int kk = 0; kk < KS; ++kk)
            ldsm_x4(qaddr + tile_off<D>(r, kk * 16 + dsub), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
    }

    // this lane's two rows (CTA rows warp*16 + lane/4 and +8) and their positions
    int pos_r[2];
    bool row_ok[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int R = warp * 16 + (lane >> 2) + h * 8;
        const int qi = q0 + R / G;
        row_ok[h] = R < QT * G && qi < qlen;
        pos_r[h] = row_ok[h] ? n - qlen + qi : pos_max;
    }

    float o[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY};
    float l_r[2] = {0.f, 0.f};

    for (int kt = 0; kt < nkt; ++kt) {
        const int s = kt % kPreStages;
        const bool got = mbar_wait(&full_bar[s], (kt / kPreStages) & 1);
        if (__any_sync(kFull, !got)) {
            if (lane == 0) {
                record_error(p.err, PA_DEVERR_TIMEOUT_);
                atomicOr(&abort_flag, 1);
            }
            break;
        }
        uint8_t* ks = smem + s * Shape::kStageBytes;
        uint8_t* vs = ks + Shape::kHalf;
        const int key0 = kt * kPreKeys;
        const uint32_t bad = bad_mask[s];
        const bool last = kt == nkt - 1;
        if (last || bad) {
            // clear V rows that must contribute nothing: keys past the tile's
            // last query position (not loaded, or past the sequence end, may
            // hold anything) and keys of blocks with an invalid table entry.
            // Every warp clears all of them itself (identical zero stores), so
            // no cross-warp barrier is needed before its own P V.
            constexpr int CPR = D / 8;
            for (int idx = lane; idx < kPreKeys * CPR; idx += 32) {
                const int kk = idx / CPR;
                if (key0 + kk > pos_max || ((bad >> (kk >> 4)) & 1u))
                    *reinterpret_cast<uint4*>(vs + tile_off<D>(kk, (idx - kk * CPR) * 8)) = make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
        }

        // S = Q K^T for this warp's 16 rows x 64 keys
        float sc[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
        {
            const uint32_t kaddr = smem_addr(ks);
            const int krow = (lane & 7) + ((lane >> 4) & 1) * 8;
            const int dsub = ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(kaddr + tile_off<D>(j * 8 + krow, kk * 16 + dsub), r0, r1, r2, r3);
                    Mma<T>::run(sc[j], qa[kk], r0, r1);
                    Mma<T>::run(sc[j + 1], qa[kk], r2, r3);
                }
            }
        }
        // scale, causal / validity mask, online softmax
        const bool need_mask = (key0 + kPreKeys - 1 > pos_min) || bad;
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int h = e >> 1;
                float v = sc[j][e] * p.scale_log2;
                if (need_mask) {
                    const int key = key0 + j * 8 + 2 * (lane & 3) + (e & 1);
                    const bool dead = key > pos_r[h] || ((bad >> ((j * 8) >> 4)) & 1u);
                    v = dead ? -INFINITY : v;
                }
                sc[j][e] = v;
                mx[h] = fmaxf(mx[h], v);
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFull, mx[h], 1));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFull, mx[h], 2));
        }
        float alpha[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float mn = fmaxf(m_r[h], mx[h]);
            // a row whose keys so far are all masked keeps m = -inf; use 0 as
            // the reference so that 2^(-inf - ref) = 0 instead of NaN
            const float ref = mn == -INFINITY ? 0.f : mn;
            alpha[h] = fast_exp2(m_r[h] - ref);
            m_r[h] = mn;
            mx[h] = ref;
        }
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float pe = fast_exp2(sc[j][e] - mx[e >> 1]);
                sc[j][e] = pe;
                rs[e >> 1] += pe;
            }
        }
        l_r[0] = l_r[0] * alpha[0] + rs[0];
        l_r[1] = l_r[1] * alpha[1] + rs[1];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            o[j][0] *= alpha[0];
            o[j][1] *= alpha[0];
            o[j][2] *= alpha[1];
            o[j][3] *= alpha[1];
        }
        // O += P V
        {
            const uint32_t vaddr = smem_addr(vs);
            const int vrow = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int dsub = ((lane >> 4) & 1) * 8;
#pragma unroll
            for (int kp = 0; kp < kPreKeys / 16; ++kp) {
                uint32_t pa[4];
                pa[0] = Elem<T>::pack(sc[2 * kp][0], sc[2 * kp][1]);
                pa[1] = Elem<T>::pack(sc[2 * kp][2], sc[2 * kp][3]);
                pa[2] = Elem<T>::pack(sc[2 * kp + 1][0], sc[2 * kp + 1][1]);
                pa[3] = Elem<T>::pack(sc[2 * kp + 1][2], sc[2 * kp + 1][3]);
#pragma unroll
                for (int j = 0; j < NT; j += 2) {
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4_t(vaddr + tile_off<D>(kp * 16 + vrow, j * 8 + dsub), r0, r1, r2, r3);
                    Mma<T>::run(o[j], pa, r0, r1);
                    Mma<T>::run(o[j + 1], pa, r2, r3);
                }
            }
        }
        // release the slot to the producer
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
    if (*(volatile int*)&abort_flag) return;

    // normalise and store
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        l_r[h] += __shfl_xor_sync(kFull, l_r[h], 1);
        l_r[h] += __shfl_xor_sync(kFull, l_r[h], 2);
    }
    uint16_t* og = static_cast<uint16_t*>(p.out);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (!row_ok[h]) continue;
        const int R = warp * 16 + (lane >> 2) + h * 8;
        const int qi = q0 + R / G;
        const int64_t grow = static_cast<int64_t>(row0 + qi) * p.num_q_heads + g * G + (R % G);
        const float inv = l_r[h] > 0.f ? 1.f / l_r[h] : 0.f;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int d = j * 8 + 2 * (lane & 3);
            *reinterpret_cast<uint32_t*>(og + grow * D + d) =
                Elem<T>::pack(o[j][2 * h] * inv, o[j][2 * h + 1] * inv);
        }
    }
}

template <typename T, int D>
cudaError_t launch_prefill_t(const PrefillParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             int max_q_len, cudaStream_t s) {
    constexpr int smem = PrefillShape<D>::kSmemBytes;
    auto kern = prefill_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int tiles = (max_q_len + p.q_per_tile - 1) / p.q_per_tile;
    dim3 grid(tiles, p.num_kv_heads, p.num_seqs);
    kern<<<grid, kPreThreads, smem, s>>>(p, kmap, vmap);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           int head_dim, int dtype, int max_q_len, cudaStream_t s) {
    if (p.num_seqs == 0 || max_q_len <= PA_VERIFY_MAX_Q_) return cudaSuccess;
    if (dtype == 0)
        return head_dim == 128 ? launch_prefill_t<__half, 128>(p, kmap, vmap, max_q_len, s)
                               : launch_prefill_t<__half, 64>(p, kmap, vmap, max_q_len, s);
    return head_dim == 128 ? launch_prefill_t<__nv_bfloat16, 128>(p, kmap, vmap, max_q_len, s)
                           : launch_prefill_t<__nv_bfloat16, 64>(p, kmap, vmap, max_q_len, s);
}

}  // namespace pa
