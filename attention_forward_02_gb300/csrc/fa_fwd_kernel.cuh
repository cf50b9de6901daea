// fa_fwd_kernel.cuh -- the sm_103a attention-forward kernel.
//
// What it computes: for one (batch*head, Q tile) per CTA,
//   O_tile = softmax(Q_tile K^T * scale) V,  LSE_tile = m * scale + ln(l)
// with the online-softmax recurrence of "3.6 어텐션 I — 메모리 문제·
// FlashAttention 원리", section 3.6.4 (state m, l, O kept on chip; alpha =
// exp(m_old - m_new) rescales both l and O; one division by l at the end),
// and the tile loop of section 3.6.6 (Q block fixed per CTA, K/V blocks
// streamed; causal skips blocks above the diagonal and masks the diagonal).
// The grid follows "Triton으로 FlashAttention 1·2 forward 구현하기", section
// "병렬화 단위": one CTA per (Q block, batch*head).
//
// GB300 mapping (differs from the pages' A100 cp.async / ldmatrix / mma.sync
// design; see the design notes for the reasons):
//   warp 4      : TMA producer.  Q tile once; K_j and V_j through a STAGES-deep
//                 ring of 128B-swizzled shared-memory tiles (full/empty mbarriers).
//   warp 5      : MMA issuer (one thread).  S_j = Q K_j^T into one of two TMEM
//                 score buffers (tcgen05.mma, fp32 accumulate), then
//                 O += P_{j-1} V_{j-1} into the TMEM output accumulator.
//                 V is read as an MN-major B operand, so no transpose copy.
//   warps 0..3  : softmax + correction + epilogue.  Thread t owns query row t
//                 = TMEM lane t, so row max / row sum need no shuffles.  exp2
//                 with scale*log2(e) folded into one FMA; P rounded to the input
//                 dtype into a swizzled shared tile for the second MMA; O rescaled
//                 in TMEM by alpha (skipped when the whole warp has alpha == 1);
//                 epilogue O / l staged through shared memory and written with
//                 coalesced 16-byte stores, LSE as one coalesced fp32 per row.
// Every mbarrier wait is bounded: on expiry the CTA records a timeout in the
// device status word, stops, waits (bounded) for its own copies and MMAs,
// frees its TMEM and exits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "sm100_ptx.cuh"

namespace fa {

// Device status word (one per device that loads the library): bit 0 = a
// bounded wait expired.
__device__ unsigned int g_fa_status;
constexpr unsigned int kStatusTimeout = 1u;

constexpr int kBM = 128;  // query rows per CTA: one M = 128 MMA, one TMEM lane per row
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kNumThreads = 192;
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;  // S0 @ 0, S1 @ 128, O @ 256
constexpr uint32_t kTmemO = 256;
constexpr long long kWaitLimitCycles = 1ll << 31;  // about one second at 2 GHz
constexpr int kSwAtomBytes = 128 * 128;             // one [128 rows x 64 cols] 16-bit swizzle block

template <int D>
struct KCfg {
    static constexpr int STAGES = (D == 64) ? 3 : 2;
    static constexpr int TILE = 128 * D * 2;  // bytes of one [128, D] 16-bit tile
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + TILE;
    static constexpr int V_OFF = K_OFF + STAGES * TILE;
    static constexpr int P_OFF = V_OFF + STAGES * TILE;
    static constexpr int P_BYTES = 128 * 128 * 2;
    static constexpr int BAR_OFF = P_OFF + P_BYTES;
    // barrier slots
    static constexpr int B_QFULL = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_KEMPTY = B_KFULL + STAGES;
    static constexpr int B_VFULL = B_KEMPTY + STAGES;
    static constexpr int B_VEMPTY = B_VFULL + STAGES;
    static constexpr int B_SFULL = B_VEMPTY + STAGES;  // two
    static constexpr int B_PFULL = B_SFULL + 2;
    static constexpr int B_ODONE = B_PFULL + 1;
    static constexpr int B_DRAIN = B_ODONE + 1;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr int SLOT_OFF = BAR_OFF + 8 * NUM_BARS;  // TMEM base address, abort flag
    static constexpr int SMEM_USED = SLOT_OFF + 16;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack for 1024-byte alignment
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

template <typename T>
struct DTypeTraits;
template <>
struct DTypeTraits<__half> {
    static constexpr bool kBF16 = false;
    static __device__ __forceinline__ uint32_t pack(float a, float b)
    {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};
template <>
struct DTypeTraits<__nv_bfloat16> {
    static constexpr bool kBF16 = true;
    static __device__ __forceinline__ uint32_t pack(float a, float b)
    {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};

// Bounded wait.  Returns false if the CTA is aborting or the limit expired
// (then the abort flag and the device status word are set).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *abort_flag = 1;
            atomicOr(&g_fa_status, kStatusTimeout);
            return false;
        }
    }
}

// Bounded wait used on the way out (ignores the abort flag: it waits for
// work this thread itself started).
__device__ __forceinline__ void drain_bounded(uint32_t bar, uint32_t parity)
{
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitLimitCycles) {
            atomicOr(&g_fa_status, kStatusTimeout);
            return;
        }
    }
}

// Byte offset of 16-byte chunk `chunk` (0..D/8-1) of row `row` in a [128, D]
// 16-bit tile laid out as D/64 column blocks of [128 rows x 128 B], each
// 128B-swizzled (chunk index XOR row % 8) -- the layout TMA SWIZZLE_128B
// writes and the tcgen05 SW128 descriptors read.
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk)
{
    return static_cast<uint32_t>((chunk >> 3) * kSwAtomBytes + row * 128 +
                                 (((chunk & 7) ^ (row & 7)) << 4));
}

template <int D, bool CAUSAL, typename T>
__global__ void __launch_bounds__(kNumThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, T *__restrict__ out,
                  float *__restrict__ lse, int N, int num_q_tiles, float scale, float scale_log2)
{
    using C = KCfg<D>;
    constexpr int ST = C::STAGES;
    constexpr int KSTEPS_QK = D / 16;   // UMMA_K = 16 for 16-bit operands
    constexpr int KSTEPS_PV = kBN / 16;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int q_tile = num_q_tiles - 1 - static_cast<int>(blockIdx.y);  // heavy causal tiles first
    const int row0 = q_tile * kBM;
    const int num_k_tiles = (N + kBN - 1) / kBN;
    const int nk = CAUSAL ? min(q_tile + 1, num_k_tiles) : num_k_tiles;

    auto bar = [&](int idx) -> uint32_t { return sbase + C::BAR_OFF + 8u * idx; };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + C::SLOT_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::SLOT_OFF + 4);

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_QFULL), 1);
        for (int s = 0; s < ST; ++s) {
            mbar_init(bar(C::B_KFULL + s), 1);
            mbar_init(bar(C::B_KEMPTY + s), 1);
            mbar_init(bar(C::B_VFULL + s), 1);
            mbar_init(bar(C::B_VEMPTY + s), 1);
        }
        mbar_init(bar(C::B_SFULL + 0), 1);
        mbar_init(bar(C::B_SFULL + 1), 1);
        mbar_init(bar(C::B_PFULL), 4 * 32);
        mbar_init(bar(C::B_ODONE), 1);
        mbar_init(bar(C::B_DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTmaWarp) {
        if (lane == 0) {
            // ---------------- producer ----------------
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            mbar_arrive_expect_tx(bar(C::B_QFULL), C::TILE);
            for (int b = 0; b < D / 64; ++b)
                tma_load_3d(sbase + C::Q_OFF + b * kSwAtomBytes, &tm_q, bar(C::B_QFULL), b * 64, row0,
                            bh, pol_q);
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < nk; ++j) {
                const int s = j % ST;
                const uint32_t ph = (j / ST) & 1;
                if (j >= ST && !wait_bounded(bar(C::B_KEMPTY + s), ph ^ 1, abort_flag))
                    break;
                mbar_arrive_expect_tx(bar(C::B_KFULL + s), C::TILE);
                for (int b = 0; b < D / 64; ++b)
                    tma_load_3d(sbase + C::K_OFF + s * C::TILE + b * kSwAtomBytes, &tm_k,
                                bar(C::B_KFULL + s), b * 64, j * kBN, bh, pol_kv);
                ++k_issued;
                if (j >= ST && !wait_bounded(bar(C::B_VEMPTY + s), ph ^ 1, abort_flag))
                    break;
                mbar_arrive_expect_tx(bar(C::B_VFULL + s), C::TILE);
                for (int b = 0; b < D / 64; ++b)
                    tma_load_3d(sbase + C::V_OFF + s * C::TILE + b * kSwAtomBytes, &tm_v,
                                bar(C::B_VFULL + s), b * 64, j * kBN, bh, pol_kv);
                ++v_issued;
            }
            // Wait for every copy this thread issued (immediate on the normal
            // path, where each one was consumed).  The last load into stage s
            // was use number (issued - 1 - s) / ST of that stage.
            drain_bounded(bar(C::B_QFULL), 0);
            for (int s = 0; s < ST; ++s) {
                if (k_issued > s)
                    drain_bounded(bar(C::B_KFULL + s), ((k_issued - 1 - s) / ST) & 1);
                if (v_issued > s)
                    drain_bounded(bar(C::B_VFULL + s), ((v_issued - 1 - s) / ST) & 1);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t idesc_s = make_idesc_f16(DTypeTraits<T>::kBF16, kBM, kBN, false, false);
            constexpr uint32_t idesc_o = make_idesc_f16(DTypeTraits<T>::kBF16, kBM, D, false, true);
            bool ok = wait_bounded(bar(C::B_QFULL), 0, abort_flag);
            tc_fence_after();
            for (int j = 0; ok && j <= nk; ++j) {
                if (j < nk) {
                    const int s = j % ST;
                    const uint32_t ph = (j / ST) & 1;
                    ok = wait_bounded(bar(C::B_KFULL + s), ph, abort_flag);
                    if (!ok)
                        break;
                    tc_fence_after();
                    const uint32_t d_s = tmem + static_cast<uint32_t>(j & 1) * kBN;
                    const uint32_t kt = sbase + C::K_OFF + s * C::TILE;
#pragma unroll
                    for (int kk = 0; kk < KSTEPS_QK; ++kk) {
                        const uint32_t koff = (kk >> 2) * kSwAtomBytes + (kk & 3) * 32;
                        const uint64_t ad = make_sdesc_sw128(sbase + C::Q_OFF + koff, 16, 1024);
                        const uint64_t bd = make_sdesc_sw128(kt + koff, 16, 1024);
                        umma_f16_ss(d_s, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(bar(C::B_SFULL + (j & 1)));
                    umma_commit(bar(C::B_KEMPTY + s));
                }
                if (j >= 1) {
                    const int i = j - 1;
                    const int s = i % ST;
                    const uint32_t ph = (i / ST) & 1;
                    ok = wait_bounded(bar(C::B_PFULL), i & 1, abort_flag);
                    if (!ok)
                        break;
                    ok = wait_bounded(bar(C::B_VFULL + s), ph, abort_flag);
                    if (!ok)
                        break;
                    tc_fence_after();
                    const uint32_t vt = sbase + C::V_OFF + s * C::TILE;
#pragma unroll
                    for (int kk = 0; kk < KSTEPS_PV; ++kk) {
                        const uint32_t poff = (kk >> 2) * kSwAtomBytes + (kk & 3) * 32;
                        const uint64_t ad = make_sdesc_sw128(sbase + C::P_OFF + poff, 16, 1024);
                        // V tile: MN-major; 16 key rows (2048 B) per K step, the
                        // two 64-column blocks of d = 128 are kSwAtomBytes apart.
                        const uint64_t bd = make_sdesc_sw128(vt + kk * 2048, kSwAtomBytes, 1024);
                        umma_f16_ss(tmem + kTmemO, ad, bd, idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(bar(C::B_ODONE));
                    umma_commit(bar(C::B_VEMPTY + s));
                }
            }
            // every MMA issued above has completed once this arrives
            umma_commit(bar(C::B_DRAIN));
            drain_bounded(bar(C::B_DRAIN), 0);
        }
    } else {
        // ---------------- softmax / correction / epilogue (warps 0..3) ----------------
        const int r = threadIdx.x;  // row within the tile == TMEM lane
        const int qrow = row0 + r;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        float m = -INFINITY;  // running max of raw scores (scale >= 0)
        float l = 0.f;
        bool ok = true;
        for (int j = 0; j < nk; ++j) {
            ok = wait_bounded(bar(C::B_SFULL + (j & 1)), (j >> 1) & 1, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok)
                break;
            tc_fence_after();
            float p[kBN];
            {
                uint32_t u[32];
#pragma unroll
                for (int c4 = 0; c4 < kBN / 32; ++c4) {
                    tmem_ld32(tmem + lane_base + static_cast<uint32_t>(j & 1) * kBN + c4 * 32, u);
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        p[c4 * 32 + c] = __uint_as_float(u[c]);
                }
            }
            const int kbase = j * kBN;
            int limit = kBN;  // keys [kbase, kbase + limit) are allowed for this row
            if (kbase + kBN > N)
                limit = N - kbase;
            if (CAUSAL && j == nk - 1)
                limit = min(limit, qrow - kbase + 1);
            const bool masked = __any_sync(0xffffffffu, limit < kBN);
            if (masked) {
#pragma unroll
                for (int c = 0; c < kBN; ++c)
                    if (c >= limit)
                        p[c] = -INFINITY;
            }
            float mt = p[0];
#pragma unroll
            for (int c = 1; c < kBN; ++c)
                mt = fmaxf(mt, p[c]);
            const float m_new = fmaxf(m, mt);
            // alpha = exp(m_old - m_new); 0 while no score has been seen (m = -inf),
            // which also covers scale == 0 where (-inf) * 0 would be NaN.
            const float alpha = (m == -INFINITY) ? 0.f : ex2_approx((m - m_new) * scale_log2);
            const float neg_mc = (m_new == -INFINITY) ? 0.f : -m_new * scale_log2;
            float rsum = 0.f;
            if (masked) {
#pragma unroll
                for (int c = 0; c < kBN; ++c) {
                    const float e = (c < limit) ? ex2_approx(fmaf(p[c], scale_log2, neg_mc)) : 0.f;
                    p[c] = e;
                    rsum += e;
                }
            } else {
#pragma unroll
                for (int c = 0; c < kBN; ++c) {
                    const float e = ex2_approx(fmaf(p[c], scale_log2, neg_mc));
                    p[c] = e;
                    rsum += e;
                }
            }
            l = l * alpha + rsum;
            m = m_new;

            if (j > 0) {
                // PV_{j-1} must be complete: it read the P buffer and wrote O.
                ok = wait_bounded(bar(C::B_ODONE), (j - 1) & 1, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok)
                    break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                    for (int c4 = 0; c4 < D / 32; ++c4) {
                        uint32_t u[32];
                        const uint32_t ta = tmem + lane_base + kTmemO + c4 * 32;
                        tmem_ld32(ta, u);
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            u[c] = __float_as_uint(__uint_as_float(u[c]) * alpha);
                        tmem_st32(ta, u);
                    }
                    tmem_wait_st();
                }
            }
            // P_j (rounded to the input dtype) into the swizzled K-major tile.
            const uint32_t prow = sbase + C::P_OFF;
#pragma unroll
            for (int ch = 0; ch < kBN / 8; ++ch) {
                const uint32_t w0 = DTypeTraits<T>::pack(p[ch * 8 + 0], p[ch * 8 + 1]);
                const uint32_t w1 = DTypeTraits<T>::pack(p[ch * 8 + 2], p[ch * 8 + 3]);
                const uint32_t w2 = DTypeTraits<T>::pack(p[ch * 8 + 4], p[ch * 8 + 5]);
                const uint32_t w3 = DTypeTraits<T>::pack(p[ch * 8 + 6], p[ch * 8 + 7]);
                st_shared_v4(prow + sw128_offset(r, ch), w0, w1, w2, w3);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(C::B_PFULL));
        }

        // ---------------- epilogue ----------------
        // Every softmax thread reaches the named barrier below, whatever
        // happened; a warp that gave up has set the abort flag first, so after
        // the barrier all four warps agree on whether the staged tile is whole.
        if (ok) {
            ok = wait_bounded(bar(C::B_ODONE), (nk - 1) & 1, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
        }
        const uint32_t stage = sbase + C::Q_OFF;  // Q tile is dead: every S MMA completed
        if (ok) {
            tc_fence_after();
            const float inv_l = 1.f / l;
#pragma unroll
            for (int c4 = 0; c4 < D / 32; ++c4) {
                uint32_t u[32];
                tmem_ld32(tmem + lane_base + kTmemO + c4 * 32, u);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int ch = c4 * 4 + q4;
                    const float *f = reinterpret_cast<const float *>(u) + q4 * 8;
                    st_shared_v4(stage + sw128_offset(r, ch),
                                 DTypeTraits<T>::pack(f[0] * inv_l, f[1] * inv_l),
                                 DTypeTraits<T>::pack(f[2] * inv_l, f[3] * inv_l),
                                 DTypeTraits<T>::pack(f[4] * inv_l, f[5] * inv_l),
                                 DTypeTraits<T>::pack(f[6] * inv_l, f[7] * inv_l));
                }
            }
            if (lse != nullptr && qrow < N)
                lse[static_cast<size_t>(bh) * N + qrow] = m * scale + logf(l);
        }
        named_bar_sync(1, 4 * 32);
        if (*abort_flag == 0) {
            constexpr int CHUNKS_PER_ROW = D / 8;
            uint8_t *obase = reinterpret_cast<uint8_t *>(out) +
                             (static_cast<size_t>(bh) * N + row0) * D * sizeof(T);
#pragma unroll 4
            for (int idx = r; idx < kBM * CHUNKS_PER_ROW; idx += 4 * 32) {
                const int row = idx / CHUNKS_PER_ROW;
                const int ch = idx % CHUNKS_PER_ROW;
                const uint4 val = ld_shared_v4(stage + sw128_offset(row, ch));
                if (row0 + row < N)
                    *reinterpret_cast<uint4 *>(obase + (static_cast<size_t>(row) * D + ch * 8) *
                                                           sizeof(T)) = val;
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace fa
