// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05).
//
// Same operation as prefill_kernel in pa_prefill.cu ("vLLM-Ascend 原理",
// section 2.3 "因果自注意力": query at position i sees positions 0..i; section
// 2.4: a later chunk reads the KV earlier chunks wrote), for query groups of
// 1, 2, 4 or 8 heads per kv head.
//
// One CTA = 128 rows = (query, q head) pairs of one kv group; TMEM lane r
// holds row r.  Warp specialisation:
//   * warp 4, lane 0: TMA (Q once; K/V 64-key tiles gathered block by block
//     through the block table into a ring of stages) and every tcgen05.mma;
//   * warps 0-3, thread r = row r: the softmax of its row.
// Per 64-key tile j:
//   S(j) = Q K^T     M=128 N=64 K=16 x D/16 into one of two TMEM S buffers,
//                    issued as soon as K(j) has landed, so it overlaps the
//                    softmax of tile j-1;
//   softmax(j)       tcgen05.ld of the S row, running reference m_ref and sum
//                    l, P row (bf16/fp16) into shared memory, 128-byte swizzled;
//   O += P(j) V(j)   M=128 N=D K=16 x 4 (V read MN-major), accumulated in TMEM.
// O stays in TMEM for the whole key range.  A row rescales O and l only when
// its running maximum exceeds m_ref by more than 2^8 (so P <= 256); then the
// row's O is read, scaled and written back in TMEM before P(j) V is issued.
// Only the tiles that cross the causal diagonal are masked; V rows past the
// tile's last query position are cleared so that 0 * NaN cannot reach O.
#include <algorithm>
#include <type_traits>

#include "pa_device.cuh"

namespace pa {

namespace {

constexpr int kTcSoftmaxWarps = 4;
constexpr int kTcThreads = (kTcSoftmaxWarps + 1) * 32;
constexpr int kTcKeys = 64;
constexpr uint32_t kTmemCols = 256;  // S0 (64) | S1 (64) | O (<= 128)
constexpr float kRescaleLog2 = 8.f;
constexpr unsigned kFullMask = 0xffffffffu;

template <int D, int ST>
struct TcShape {
    static constexpr int kKeyHalf = kTcKeys * 128;          // 64 keys x one 64-dim half
    static constexpr int kKV = (D / 64) * kKeyHalf;         // K (or V) of one stage: [half][key][128 B]
    static constexpr int kStage = 2 * kKV;
    static constexpr int kQHalf = 128 * 128;                // 128 rows x one half
    static constexpr int kQ = (D / 64) * kQHalf;
    static constexpr int kP = 128 * 128;                    // 128 rows x 64 keys x 2 B
    static constexpr bool kPInK = kKV >= kP;                // P(j) reuses the K region of its stage
    static constexpr int kSmem = kQ + ST * kStage + (kPInK ? 0 : ST * kP) + 1024;
};

// Bounded mbarrier wait that also gives up when another thread of the CTA has
// already recorded a failure.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    for (uint32_t i = 0; i < kMaxWaitIters; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 1023u) == 1023u && *abort_flag) return false;
    }
    return false;
}

// Work list of the chunked-prefill tiles: offsets[b] = number of 128-row tiles
// of sequences 0..b-1 whose chunk is longer than PA_VERIFY_MAX_Q_ tokens
// (shorter chunks are decode or speculative-verify rows and belong to the
// decode kernel); offsets[B] = total.  One CTA.
__global__ void __launch_bounds__(1024) prefill_plan_kernel(const int32_t* __restrict__ cu_q_lens, int num_seqs,
                                                            int q_per_tile, int32_t* __restrict__ offsets) {
    __shared__ int warp_tot[32];
    __shared__ int carry;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < num_seqs; base += 1024) {
        const int b = base + tid;
        int v = 0;
        if (b < num_seqs) {
            const int ql = cu_q_lens[b + 1] - cu_q_lens[b];
            v = ql > PA_VERIFY_MAX_Q_ ? (ql + q_per_tile - 1) / q_per_tile : 0;
        }
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
        const int before = carry + (warp > 0 ? warp_tot[warp - 1] : 0);
        if (b < num_seqs) offsets[b] = before + incl - v;
        __syncthreads();
        if (tid == 1023) carry = before + incl;
        __syncthreads();
    }
    if (tid == 0) offsets[num_seqs] = carry;
}

// Persistent: each CTA walks work items w = blockIdx.x, blockIdx.x + gridDim.x, ...
// over (tile, kv head) pairs of the plan; within a sequence the tiles nearest
// the end (the longest key ranges) come first.
// Two CTAs share an SM: ten warps, so one SM sub-partition runs three of them
// and its 16K registers allow at most 168 per thread.
template <typename T, int D, int ST>
__global__ void __maxnreg__(168)
    prefill_tc_kernel(const PrefillParams p, const int32_t* __restrict__ plan,
                      const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap qmap) {
    using Sh = TcShape<D, ST>;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t kIdescS = mma_idesc_f16(128, kTcKeys, kBf16, false);
    constexpr uint32_t kIdescPV = mma_idesc_f16(128, D, kBf16, true);

    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full_bar[ST];
    __shared__ uint64_t s_full[2];
    __shared__ uint64_t p_full[2];   // per tile parity: one arrival per softmax warp
    __shared__ uint64_t o_done;
    __shared__ uint32_t bad_mask[ST];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int G = p.group;
    const int QT = p.q_per_tile;  // 128 / G
    const int total_items = plan[p.num_seqs] * p.num_kv_heads;
    if (static_cast<int>(blockIdx.x) >= total_items) return;

    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* qs = smem;
    auto kst = [&](int s) { return smem + Sh::kQ + s * Sh::kStage; };
    auto vst = [&](int s) { return smem + Sh::kQ + s * Sh::kStage + Sh::kKV; };
    auto pst = [&](int s) { return Sh::kPInK ? kst(s) : smem + Sh::kQ + ST * Sh::kStage + s * Sh::kP; };

    if (warp == 0) {
        tmem_alloc(&tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < ST; ++s) mbar_init(&full_bar[s], 1);
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        mbar_init(&p_full[0], kTcSoftmaxWarps);
        mbar_init(&p_full[1], kTcSoftmaxWarps);
        mbar_init(&o_done, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const uint32_t o_tm = tmem + 128;
    volatile int* abort_v = &abort_flag;

    // per-CTA running counters (identical in every role): tiles processed so far
    int J0 = 0;
    bool ok = true;
    // producer bookkeeping for the abort path
    int s_issued = 0, pv_issued = 0, kv_issued = 0, kv_seen = 0;

    for (int w = blockIdx.x; ok && w < total_items; w += gridDim.x) {
        // ---- decode the work item -------------------------------------------
        const int g = w % p.num_kv_heads;
        const int l = w / p.num_kv_heads;
        int lo = 0, hi = p.num_seqs - 1;  // last b with plan[b] <= l
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (plan[mid] <= l) lo = mid; else hi = mid - 1;
        }
        const int b = lo;
        const int row0 = p.cu_q_lens[b];
        const int qlen = p.cu_q_lens[b + 1] - row0;
        const int ntiles = (qlen + QT - 1) / QT;
        const int qt = ntiles - 1 - (l - plan[b]);
        const int n = p.seq_lens[b];
        if (n < qlen || n > p.max_seq_len || n > p.max_blocks * 16) {
            if (qt == ntiles - 1 && g == 0 && tid == 0) record_error(p.err, PA_DEVERR_SEQ_LEN_);
            continue;
        }
        const int q0 = qt * QT;
        const int q_last = min(qlen, q0 + QT) - 1;
        const int pos_min = n - qlen + q0;
        const int pos_max = n - qlen + q_last;
        const int nkt = (pos_max + kTcKeys) / kTcKeys;
        const int nblk_live = (pos_max + 16) >> 4;
        const int32_t* bt = p.block_tables + static_cast<int64_t>(b) * p.max_blocks;

        if (warp == kTcSoftmaxWarps) {
            // ===================== producer / MMA issuer =====================
            if (lane == 0) {
                auto issue_kv = [&](int j, bool with_q) {
                    const int s = (J0 + j) % ST;
                    uint32_t bytes = with_q ? static_cast<uint32_t>(Sh::kQ) : 0u;
                    uint32_t bad = 0;
                    int phys[4];
#pragma unroll
                    for (int jb = 0; jb < 4; ++jb) {
                        const int blk = j * 4 + jb;
                        phys[jb] = -1;
                        if (blk < nblk_live) {
                            const int id = bt[blk];
                            if (id >= 0 && id < p.num_blocks) {
                                phys[jb] = id;
                                bytes += 2 * (D / 64) * 2048;
                            } else {
                                bad |= 1u << jb;
                                record_error(p.err, PA_DEVERR_BLOCK_ID_);
                            }
                        }
                    }
                    bad_mask[s] = bad;
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(&full_bar[s], bytes);
                    if (with_q) {
#pragma unroll
                        for (int h = 0; h < D / 64; ++h)
                            tma_load_4d(qs + h * Sh::kQHalf, &qmap, &full_bar[s], 0, h, g * G, row0 + q0);
                    }
#pragma unroll
                    for (int jb = 0; jb < 4; ++jb) {
                        if (phys[jb] < 0) continue;
#pragma unroll
                        for (int h = 0; h < D / 64; ++h) {
                            tma_load_4d(kst(s) + h * Sh::kKeyHalf + jb * 2048, &kmap, &full_bar[s], 0, h, g,
                                        phys[jb] * 16);
                            tma_load_4d(vst(s) + h * Sh::kKeyHalf + jb * 2048, &vmap, &full_bar[s], 0, h, g,
                                        phys[jb] * 16);
                        }
                    }
                    ++kv_issued;
                };
                auto issue_s = [&](int j) {
                    const int J = J0 + j;
                    const uint32_t qa = smem_addr(qs);
                    const uint32_t ka = smem_addr(kst(J % ST));
                    const uint32_t d_tm = tmem + static_cast<uint32_t>((J & 1) * kTcKeys);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t a = smem_desc_sw128(qa + (kk >> 2) * Sh::kQHalf + (kk & 3) * 32, 16, 1024);
                        const uint64_t bd =
                            smem_desc_sw128(ka + (kk >> 2) * Sh::kKeyHalf + (kk & 3) * 32, 16, 1024);
                        tc_mma_f16(d_tm, a, bd, kIdescS, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(&s_full[J & 1]);
                    ++s_issued;
                };
                auto issue_pv = [&](int j) {
                    const int s = (J0 + j) % ST;
                    const uint32_t pa = smem_addr(pst(s));
                    const uint32_t va = smem_addr(vst(s));
#pragma unroll
                    for (int kp = 0; kp < kTcKeys / 16; ++kp) {
                        const uint64_t a = smem_desc_sw128(pa + kp * 32, 16, 1024);
                        const uint64_t bd = smem_desc_sw128(va + kp * 2048, Sh::kKeyHalf, 1024);
                        tc_mma_f16(o_tm, a, bd, kIdescPV, (j > 0 || kp > 0) ? 1u : 0u);
                    }
                    tc_commit(&o_done);
                    ++pv_issued;
                };

                // the previous item's last P V must be done before Q and the
                // stages are overwritten
                if (J0 > 0) ok = wait_or_abort(&o_done, (J0 - 1) & 1, abort_v);
                if (ok) {
                    for (int t = 0; t < ST && t < nkt; ++t) issue_kv(t, t == 0);
                    ok = wait_or_abort(&full_bar[J0 % ST], (J0 / ST) & 1, abort_v);
                }
                if (ok) {
                    ++kv_seen;
                    tc_fence_after_sync();
                    issue_s(0);
                }
                for (int j = 0; ok && j < nkt; ++j) {
                    const int J = J0 + j;
                    if (j + 1 < nkt) {
                        // S(j+1): its K has to be in; its TMEM buffer was last read
                        // by the softmax of tile J-1, whose P we already waited for
                        ok = wait_or_abort(&full_bar[(J + 1) % ST], ((J + 1) / ST) & 1, abort_v);
                        if (!ok) break;
                        ++kv_seen;
                        tc_fence_after_sync();
                        issue_s(j + 1);
                    }
                    // two barriers by tile parity: S(J+1) is already issued, so the
                    // softmax warps may finish tiles J and J+1 before this wait; a
                    // single barrier would then be two phases ahead of it
                    ok = wait_or_abort(&p_full[J & 1], (J >> 1) & 1, abort_v);
                    if (!ok) break;
                    tc_fence_after_sync();
                    issue_pv(j);
                    if (j + ST < nkt) {
                        // the stage is free once P(j) V(j) has completed
                        ok = wait_or_abort(&o_done, J & 1, abort_v);
                        if (!ok) break;
                        issue_kv(j + ST, false);
                    }
                }
                if (!ok) *abort_v = 1;
            }
        } else {
            // ========================== softmax rows ==========================
            const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
            const int qi_row = q0 + tid / G;
            const bool row_ok = tid < QT * G && qi_row < qlen;
            const int pos_row = row_ok ? n - qlen + qi_row : pos_max;
            float m_ref = -INFINITY, l_run = 0.f;
            for (int j = 0; j < nkt; ++j) {
                const int J = J0 + j;
                const int s = J % ST;
                // p_full counts one arrival per softmax warp per tile: a warp may
                // start tile J only after every warp has arrived for tile J-2 (the
                // previous use of the same barrier), or its arrival could be
                // counted towards J-2; waiting for J-1 covers that.
                bool got = (J == 0 || wait_or_abort(&p_full[(J - 1) & 1], ((J - 1) >> 1) & 1, abort_v)) &&
                           wait_or_abort(&s_full[J & 1], (J >> 1) & 1, abort_v) &&
                           wait_or_abort(&full_bar[s], (J / ST) & 1, abort_v);
                if (!__all_sync(kFullMask, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                float sv[kTcKeys];
                {
                    uint32_t r[32];
                    const uint32_t s_tm = tmem + lane_base + static_cast<uint32_t>((J & 1) * kTcKeys);
                    tmem_ld32(s_tm, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) sv[c] = __uint_as_float(r[c]);
                    tmem_ld32(s_tm + 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) sv[32 + c] = __uint_as_float(r[c]);
                }
                const int key0 = j * kTcKeys;
                const uint32_t bad = bad_mask[s];
                const bool need_mask = (key0 + kTcKeys - 1 > pos_min) || bad;
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < kTcKeys; ++c) {
                    float v = sv[c] * p.scale_log2;
                    if (need_mask) {
                        const bool dead = key0 + c > pos_row || ((bad >> (c >> 4)) & 1u);
                        v = dead ? -INFINITY : v;
                    }
                    sv[c] = v;
                    mx = fmaxf(mx, v);
                }
                // lazy rescale: move the reference only when the maximum has
                // grown by more than 2^8 (warp-wide: tcgen05.ld/st are collective)
                if (__any_sync(kFullMask, mx > m_ref + kRescaleLog2)) {
                    const float new_ref = fmaxf(m_ref, mx);
                    const float alpha = new_ref == -INFINITY ? 1.f : fast_exp2(m_ref - new_ref);
                    if (j > 0) {
                        got = wait_or_abort(&o_done, (J - 1) & 1, abort_v);
                        if (!__all_sync(kFullMask, got)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
#pragma unroll
                        for (int c0 = 0; c0 < D / 32; ++c0) {
                            uint32_t r[32];
                            tmem_ld32(o_tm + lane_base + static_cast<uint32_t>(c0 * 32), r);
                            tmem_ld_wait();
#pragma unroll
                            for (int u = 0; u < 32; ++u) r[u] = __float_as_uint(__uint_as_float(r[u]) * alpha);
                            tmem_st32(o_tm + lane_base + static_cast<uint32_t>(c0 * 32), r);
                        }
                        tmem_st_wait();
                    }
                    l_run *= alpha;
                    m_ref = new_ref;
                }
                const float ref = m_ref == -INFINITY ? 0.f : m_ref;
                float rs = 0.f;
#pragma unroll
                for (int c = 0; c < kTcKeys; ++c) {
                    const float e = fast_exp2(sv[c] - ref);
                    sv[c] = e;
                    rs += e;
                }
                l_run += rs;
                {
                    // P row -> shared memory: K-major, 128-byte swizzled, 128 B per row
                    uint8_t* prow = pst(s) + tid * 128;
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        uint4 v4;
                        v4.x = Elem<T>::pack(sv[8 * c8 + 0], sv[8 * c8 + 1]);
                        v4.y = Elem<T>::pack(sv[8 * c8 + 2], sv[8 * c8 + 3]);
                        v4.z = Elem<T>::pack(sv[8 * c8 + 4], sv[8 * c8 + 5]);
                        v4.w = Elem<T>::pack(sv[8 * c8 + 6], sv[8 * c8 + 7]);
                        *reinterpret_cast<uint4*>(prow + ((c8 ^ (tid & 7)) << 4)) = v4;
                    }
                }
                if (j == nkt - 1 || bad) {
                    // V rows that must contribute nothing (past the tile's last
                    // query position, or in a block with an invalid table entry)
                    // may hold anything, NaN included: clear them.
                    constexpr int CPR = D / 8;
                    for (int idx = tid; idx < kTcKeys * CPR; idx += kTcSoftmaxWarps * 32) {
                        const int key = idx / CPR;
                        const int c = idx - key * CPR;
                        if (key0 + key > pos_max || ((bad >> (key >> 4)) & 1u))
                            *reinterpret_cast<uint4*>(vst(s) + (c >> 3) * Sh::kKeyHalf + key * 128 +
                                                      (((c & 7) ^ (key & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[J & 1]);
            }
            if (ok) {
                const bool got = wait_or_abort(&o_done, (J0 + nkt - 1) & 1, abort_v);
                if (__all_sync(kFullMask, got)) {
                    tc_fence_after_sync();
                    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                    const int64_t grow = static_cast<int64_t>(row0 + qi_row) * p.num_q_heads + g * G + (tid % G);
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + grow * D);
#pragma unroll
                    for (int c0 = 0; c0 < D / 32; ++c0) {
                        uint32_t r[32];
                        tmem_ld32(o_tm + lane_base + static_cast<uint32_t>(c0 * 32), r);
                        tmem_ld_wait();
                        if (row_ok) {
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                uint4 v4;
                                v4.x = Elem<T>::pack(__uint_as_float(r[8 * c + 0]) * inv,
                                                     __uint_as_float(r[8 * c + 1]) * inv);
                                v4.y = Elem<T>::pack(__uint_as_float(r[8 * c + 2]) * inv,
                                                     __uint_as_float(r[8 * c + 3]) * inv);
                                v4.z = Elem<T>::pack(__uint_as_float(r[8 * c + 4]) * inv,
                                                     __uint_as_float(r[8 * c + 5]) * inv);
                                v4.w = Elem<T>::pack(__uint_as_float(r[8 * c + 6]) * inv,
                                                     __uint_as_float(r[8 * c + 7]) * inv);
                                dst[c0 * 4 + c] = v4;
                            }
                        }
                    }
                    tc_fence_before_sync();
                } else {
                    ok = false;
                }
            }
            if (!ok) *abort_v = 1;
        }
        J0 += nkt;
        if (*abort_v) ok = false;
    }

    if (!ok || *abort_v) {
        if (tid == 0) record_error(p.err, PA_DEVERR_TIMEOUT_);
        if (warp == kTcSoftmaxWarps && lane == 0) {
            // let work still in flight finish before the CTA's memory is reused
            if (s_issued) (void)mbar_wait(&s_full[(s_issued - 1) & 1], ((s_issued - 1) >> 1) & 1);
            if (pv_issued) (void)mbar_wait(&o_done, (pv_issued - 1) & 1);
            for (int t = kv_seen; t < kv_issued; ++t) (void)mbar_wait(&full_bar[t % ST], (t / ST) & 1);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

int sm_count() {
    static int count[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!count[dev]) {
        int c = 0;
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) c = 148;
        count[dev] = c;
    }
    return count[dev];
}

template <typename T, int D, int ST>
cudaError_t launch_t(const PrefillParams& p, int32_t* plan, const CUtensorMap& kmap, const CUtensorMap& vmap,
                     const CUtensorMap& qmap, int max_q_len, int num_tokens, cudaStream_t s) {
    constexpr int smem = TcShape<D, ST>::kSmem;
    auto kern = prefill_tc_kernel<T, D, ST>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    prefill_plan_kernel<<<1, 1024, 0, s>>>(p.cu_q_lens, p.num_seqs, p.q_per_tile, plan);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // upper bound on the work items: each listed chunk (length > 8) has at
    // most ceil(len / q_per_tile) <= len / 2 tiles, and there are at most max_q_len
    // tokens per chunk
    const long long bound_tiles = std::min<long long>(static_cast<long long>(num_tokens) / 2 + 1,
                                                      static_cast<long long>(p.num_seqs) *
                                                          ((max_q_len + p.q_per_tile - 1) / p.q_per_tile));
    const long long items = bound_tiles * p.num_kv_heads;
    const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(items, 2LL * sm_count())));
    kern<<<grid, kTcThreads, smem, s>>>(p, plan, kmap, vmap, qmap);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillParams& p, int32_t* plan, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, const CUtensorMap& qmap, int head_dim, int dtype,
                              int max_q_len, int num_tokens, cudaStream_t s) {
    if (p.num_seqs == 0 || max_q_len <= PA_VERIFY_MAX_Q_) return cudaSuccess;
    if (dtype == 0)
        return head_dim == 128 ? launch_t<__half, 128, 2>(p, plan, kmap, vmap, qmap, max_q_len, num_tokens, s)
                               : launch_t<__half, 64, 2>(p, plan, kmap, vmap, qmap, max_q_len, num_tokens, s);
    return head_dim == 128 ? launch_t<__nv_bfloat16, 128, 2>(p, plan, kmap, vmap, qmap, max_q_len, num_tokens, s)
                           : launch_t<__nv_bfloat16, 64, 2>(p, plan, kmap, vmap, qmap, max_q_len, num_tokens, s);
}

}  // namespace pa
