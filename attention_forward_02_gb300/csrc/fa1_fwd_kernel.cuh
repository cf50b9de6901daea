// fa1_fwd_kernel.cuh -- the FA1-structured attention forward, the baseline the
// pages compare FA2 against ("Triton으로 FlashAttention 1·2 forward 구현하기",
// sections "병렬화 단위" and "출력 누적 방식").
//
// Same result as fa_fwd (O = softmax(Q K^T * scale) V, LSE), different loop
// nest: one CTA per (batch, head) -- grid = B * H -- with the K/V block as the
// OUTER loop and the Q blocks as the inner loop.  After every K/V block the
// normalised output and the row statistics (m, l) of each Q block go back to
// global memory in fp32 (a caller-provided workspace) and are read again for
// the next K/V block; the output is converted to the 16-bit dtype only after
// the last block of a row.  With the online-softmax algebra of "3.6 어텐션 I",
// section 3.6.4, one (Q block i, K/V block j) step is
//     m_new = max(m_old, rowmax S_ij),  alpha = exp(m_old - m_new),
//     p = exp(S_ij - m_new),            l_new = alpha * l_old + sum p,
//     O_new = (alpha * l_old * O_old + p V_j) / l_new.
// Causal: Q block i meets K/V blocks j <= i only; the diagonal block is masked
// and is the last one a Q block sees.
//
// GB300 mapping: warp 4 TMA producer (K_j, V_j double-buffered; Q_i through a
// two-slot ring), warp 5 MMA issuer (S = Q_i K_j^T and P V_j on tcgen05 with
// TMEM accumulators), warps 0-3 the softmax / update warpgroup (thread t owns
// row t of the Q block; it reads and writes its fp32 output row, m and l).
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {
namespace fa1 {

constexpr int kBlock = 128;          // rows per Q block = keys per K/V block
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4;
constexpr int kIssuerWarp = 5;
constexpr uint32_t kCols = 512;      // S @ 0 (128), P V @ 128 (D), P @ 128 + D (64)

template <int D>
struct Cfg {
    static_assert(D == 32 || D == 64 || D == 96 || D == 128, "head dims 32, 64, 96, 128");
    static constexpr int TILE = 128 * col_blocks<D>() * 128;  // whole 128-byte swizzle blocks per row
    static constexpr int K_OFF = 0;                  // two stages
    static constexpr int V_OFF = K_OFF + 2 * TILE;   // two stages
    static constexpr int Q_OFF = V_OFF + 2 * TILE;   // two slots
    static constexpr int BAR_OFF = Q_OFF + 2 * TILE;
    static constexpr int B_KFULL = 0, B_VFULL = 2, B_KVEMPTY = 4, B_QFULL = 6, B_QEMPTY = 8;
    static constexpr int B_SFULL = 10, B_SFREE = 11, B_PFULL = 12, B_OFULL = 13, B_OFREE = 14;
    static constexpr int B_DRAIN = 15;
    static constexpr int NUM_BARS = 16;
    static constexpr int SLOT_OFF = BAR_OFF + 8 * NUM_BARS;
    static constexpr int SMEM_USED = SLOT_OFF + 16;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
    static constexpr uint32_t TM_S = 0, TM_PV = 128, TM_P = 128 + D;
};

// Workspace (fp32): O [BH, N, D], then m [BH, N], then l [BH, N].
__host__ __device__ constexpr size_t workspace_floats(long long BH, long long N, int D)
{
    return static_cast<size_t>(BH) * static_cast<size_t>(N) * static_cast<size_t>(D + 2);
}

template <int D, bool CAUSAL, typename T>
__global__ void __launch_bounds__(kThreads, 1)
    fa1_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, T *__restrict__ out,
                   float *__restrict__ lse, float *__restrict__ ws, int N, float scale,
                   float scale_log2)
{
    using C = Cfg<D>;
    constexpr int KSTEPS_QK = D / 16;
    constexpr int KSTEPS_PV = kBlock / 16;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int nt = (N + kBlock - 1) / kBlock;  // Q blocks = K/V blocks
    // steps: for j in [0, nt): for i in [CAUSAL ? j : 0, nt)
    auto first_i = [&](int j) { return CAUSAL ? j : 0; };

    auto bar = [&](int idx) -> uint32_t { return sbase + C::BAR_OFF + 8u * idx; };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + C::SLOT_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::SLOT_OFF + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(C::B_KFULL + s), 1);
            mbar_init(bar(C::B_VFULL + s), 1);
            mbar_init(bar(C::B_KVEMPTY + s), 1);
            mbar_init(bar(C::B_QFULL + s), 1);
            mbar_init(bar(C::B_QEMPTY + s), 1);
        }
        mbar_init(bar(C::B_SFULL), 1);
        mbar_init(bar(C::B_SFREE), 4 * 32);
        mbar_init(bar(C::B_PFULL), 4 * 32);
        mbar_init(bar(C::B_OFULL), 1);
        mbar_init(bar(C::B_OFREE), 4 * 32);
        mbar_init(bar(C::B_DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kIssuerWarp) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            // ---------------- producer: K_j, V_j, then the Q blocks of step j ----------------
            const uint64_t pol = l2_policy_evict_last();
            int kv_issued = 0, q_issued = 0;
            bool ok = true;
            for (int j = 0; ok && j < nt; ++j) {
                const int s = j & 1;
                if (j >= 2 && !(ok = wait_bounded(bar(C::B_KVEMPTY + s), ((j >> 1) - 1) & 1, abort_flag)))
                    break;
                mbar_arrive_expect_tx(bar(C::B_KFULL + s), C::TILE);
                for (int b = 0; b < col_blocks<D>(); ++b)
                    tma_load_3d(sbase + C::K_OFF + s * C::TILE + b * kSwAtomBytes, &tm_k,
                                bar(C::B_KFULL + s), b * 64, j * kBlock, bh, pol);
                mbar_arrive_expect_tx(bar(C::B_VFULL + s), C::TILE);
                for (int b = 0; b < col_blocks<D>(); ++b)
                    tma_load_3d(sbase + C::V_OFF + s * C::TILE + b * kSwAtomBytes, &tm_v,
                                bar(C::B_VFULL + s), b * 64, j * kBlock, bh, pol);
                ++kv_issued;
                for (int i = first_i(j); i < nt; ++i) {
                    const int t = q_issued, qs = t & 1;
                    if (t >= 2 && !(ok = wait_bounded(bar(C::B_QEMPTY + qs), ((t >> 1) - 1) & 1, abort_flag)))
                        break;
                    mbar_arrive_expect_tx(bar(C::B_QFULL + qs), C::TILE);
                    for (int b = 0; b < col_blocks<D>(); ++b)
                        tma_load_3d(sbase + C::Q_OFF + qs * C::TILE + b * kSwAtomBytes, &tm_q,
                                    bar(C::B_QFULL + qs), b * 64, i * kBlock, bh, pol);
                    ++q_issued;
                }
            }
            // wait for every copy issued here (immediate on the normal path)
            for (int s = 0; s < 2; ++s) {
                if (kv_issued > s) {
                    drain_bounded(bar(C::B_KFULL + s), ((kv_issued - 1 - s) >> 1) & 1);
                    drain_bounded(bar(C::B_VFULL + s), ((kv_issued - 1 - s) >> 1) & 1);
                }
                if (q_issued > s)
                    drain_bounded(bar(C::B_QFULL + s), ((q_issued - 1 - s) >> 1) & 1);
            }
        }
    } else if (warp == kIssuerWarp) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t idesc_s = make_idesc_f16(DTypeTraits<T>::kBF16, kBlock, kBlock, false, false);
            constexpr uint32_t idesc_o = make_idesc_f16(DTypeTraits<T>::kBF16, kBlock, D, false, true);
            bool ok = true;
            int t = 0;  // step counter
            for (int j = 0; ok && j < nt; ++j) {
                const int s = j & 1;
                const uint32_t kvpar = (j >> 1) & 1;
                ok = wait_bounded(bar(C::B_KFULL + s), kvpar, abort_flag) &&
                     wait_bounded(bar(C::B_VFULL + s), kvpar, abort_flag);
                for (int i = first_i(j); ok && i < nt; ++i, ++t) {
                    const int qs = t & 1;
                    // S is reused: the softmax must have read the previous one
                    ok = wait_bounded(bar(C::B_QFULL + qs), (t >> 1) & 1, abort_flag) &&
                         (t == 0 || wait_bounded(bar(C::B_SFREE), (t - 1) & 1, abort_flag));
                    if (!ok)
                        break;
                    tc_fence_after();
                    const uint32_t qt = sbase + C::Q_OFF + qs * C::TILE;
                    const uint32_t kt = sbase + C::K_OFF + s * C::TILE;
#pragma unroll
                    for (int kk = 0; kk < KSTEPS_QK; ++kk) {
                        const uint32_t koff = (kk >> 2) * kSwAtomBytes + (kk & 3) * 32;
                        umma_f16_ss(tmem + C::TM_S, make_sdesc_sw128(qt + koff, 16, 1024),
                                    make_sdesc_sw128(kt + koff, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(bar(C::B_SFULL));
                    umma_commit(bar(C::B_QEMPTY + qs));
                    // the P V accumulator is reused: the update must have read it
                    ok = wait_bounded(bar(C::B_PFULL), t & 1, abort_flag) &&
                         (t == 0 || wait_bounded(bar(C::B_OFREE), (t - 1) & 1, abort_flag));
                    if (!ok)
                        break;
                    tc_fence_after();
                    const uint32_t vt = sbase + C::V_OFF + s * C::TILE;
#pragma unroll
                    for (int kk = 0; kk < KSTEPS_PV; ++kk)
                        umma_f16_ts(tmem + C::TM_PV, tmem + C::TM_P + kk * 8,
                                    make_sdesc_sw128(vt + kk * 2048, kSwAtomBytes, 1024), idesc_o,
                                    kk > 0 ? 1u : 0u);
                    umma_commit(bar(C::B_OFULL));
                }
                if (ok)
                    umma_commit(bar(C::B_KVEMPTY + s));
            }
            umma_commit(bar(C::B_DRAIN));
            drain_bounded(bar(C::B_DRAIN), 0);
        }
    } else {
        // ---------------- softmax / update warpgroup (warps 0..3) ----------------
        const int r = threadIdx.x;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        float *ws_o = ws;
        float *ws_m = ws + static_cast<size_t>(gridDim.x) * N * D;
        float *ws_l = ws_m + static_cast<size_t>(gridDim.x) * N;
        bool ok = true;
        int t = 0;
        for (int j = 0; ok && j < nt; ++j) {
            for (int i = first_i(j); i < nt; ++i, ++t) {
                const int qrow = i * kBlock + r;
                const bool live = qrow < N;
                const size_t row = static_cast<size_t>(bh) * N + (live ? qrow : 0);
                // previous state of this row (none before its first K/V block)
                float m_old = -INFINITY, l_old = 0.f;
                if (j > 0 && live) {
                    m_old = ws_m[row];
                    l_old = ws_l[row];
                }
                ok = wait_bounded(bar(C::B_SFULL), t & 1, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok)
                    break;
                tc_fence_after();
                float s[kBlock];
                tmem_ld128(tmem + lane_base + C::TM_S, s);
                tc_fence_before();
                mbar_arrive(bar(C::B_SFREE));
                const int kbase = j * kBlock;
                int limit = min(kBlock, N - kbase);
                if (CAUSAL)
                    limit = min(limit, qrow - kbase + 1);
                const bool masked = __any_sync(0xffffffffu, limit < kBlock);
                if (masked)
                    mask_tail(s, limit);
                const float m_new = fmaxf(m_old, row_max(s));
                const float alpha = (m_old == -INFINITY) ? 0.f : ex2_approx((m_old - m_new) * scale_log2);
                const float rsum = masked ? exp_tile<true>(s, limit, scale_log2, -m_new * scale_log2)
                                          : exp_tile<false>(s, limit, scale_log2, -m_new * scale_log2);
                const float l_new = alpha * l_old + rsum;
                {
                    uint32_t w[64];
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        w[c] = DTypeTraits<T>::pack(s[2 * c], s[2 * c + 1]);
                    tmem_st64(tmem + lane_base + C::TM_P, w);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(C::B_PFULL));
                ok = wait_bounded(bar(C::B_OFULL), t & 1, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok)
                    break;
                tc_fence_after();
                // O_new = (alpha * l_old * O_old + P V) / l_new, in D/32 chunks
                const bool last = CAUSAL ? (j == i) : (j == nt - 1);
                const float keep = alpha * l_old;
                const float inv_l = 1.f / l_new;
                float *orow = ws_o + row * D;
                T *out_row = out + row * D;
#pragma unroll 1
                for (int c4 = 0; c4 < D / 32; ++c4) {
                    uint32_t u[32];
                    tmem_ld32(tmem + lane_base + C::TM_PV + c4 * 32, u);
                    float o[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        o[c] = __uint_as_float(u[c]);
                    if (j > 0 && live) {
                        const float4 *src = reinterpret_cast<const float4 *>(orow + c4 * 32);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 x = src[q];
                            o[4 * q + 0] = fmaf(keep, x.x, o[4 * q + 0]);
                            o[4 * q + 1] = fmaf(keep, x.y, o[4 * q + 1]);
                            o[4 * q + 2] = fmaf(keep, x.z, o[4 * q + 2]);
                            o[4 * q + 3] = fmaf(keep, x.w, o[4 * q + 3]);
                        }
                    }
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        o[c] *= inv_l;
                    if (live) {
                        if (last) {
                            uint4 *dst = reinterpret_cast<uint4 *>(out_row + c4 * 32);
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                dst[q] = make_uint4(DTypeTraits<T>::pack(o[8 * q + 0], o[8 * q + 1]),
                                                    DTypeTraits<T>::pack(o[8 * q + 2], o[8 * q + 3]),
                                                    DTypeTraits<T>::pack(o[8 * q + 4], o[8 * q + 5]),
                                                    DTypeTraits<T>::pack(o[8 * q + 6], o[8 * q + 7]));
                        } else {
                            float4 *dst = reinterpret_cast<float4 *>(orow + c4 * 32);
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                dst[q] = make_float4(o[4 * q + 0], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(bar(C::B_OFREE));
                if (live) {
                    if (last) {
                        if (lse != nullptr)
                            lse[row] = m_new * scale + logf(l_new);
                    } else {
                        ws_m[row] = m_new;
                        ws_l[row] = l_new;
                    }
                }
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == kIssuerWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kCols);
    }
}

}  // namespace fa1
}  // namespace fa
