// fa_decode_tc_kernel.cuh -- decoding attention for up to 16 queries per
// head with the two products on the tensor cores (fa_decode uses it from 3
// queries on, and from 2 at d = 128).
//
// It computes what fa_decode_split_kernel computes (the same split-KV items,
// the same per-chunk partials m, l, O for fa_decode_combine_kernel): the
// online softmax of "3.6 어텐션 I — 메모리 문제·FlashAttention 원리",
// section 3.6.4, over the chunk's 128-key tiles, for the queries at the end
// of the sequence (section 3.6.9: decoding needs its own parallelisation).
// With several queries per head the CUDA-core version spends more time on
// the products than HBM needs to deliver K and V; here, per tile,
//   S^T = K Q^T    tcgen05.mma M = 128 keys, N = 16 (queries, zero-padded),
//                  K = d; A = the K tile (K-major), B = the Q tile (K-major)
//   O^T += V^T P^T tcgen05.mma M = 128 (d, zero-padded: the V tile always
//                  has two 64-column blocks, and the columns past d hold
//                  zeros), N = 16, K = 128 keys; A = the V tile read MN-major
//                  (no transpose copy), B = P^T written to shared memory by
//                  the softmax warps
// with fp32 accumulators in TMEM (S^T in two buffers, so the next tile's
// product runs while this tile's softmax does).
//
// Warp roles (192 threads): warps 0-3 softmax (thread t = TMEM lane t: key t
// of S^T, dimension t of O^T), warp 4 TMA producer (Q once per item into one
// of two buffers, K and V per tile through a ring), warp 5 MMA issuer (one
// thread; also allocates TMEM).  The reference max of each query moves only
// when one of its scores outgrows it by more than 2^8 (O^T and l are then
// rescaled, as in the forward kernel); the tile's maxima are exchanged only
// then.  The partial m, l, O of a chunk are consistent with whatever
// reference was used, which the combine step needs.
// Every mbarrier wait is bounded.
#pragma once

#include "fa_common.cuh"
#include "fa_decode_kernel.cuh"

namespace fa {
namespace dectc {

constexpr int kKeys = 128;       // keys per tile
constexpr int kNP = 16;          // queries per product (Nq padded)
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 64;  // S^T buffers at 0 and 16, O^T at 32
constexpr uint32_t kTmO = 32;
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct Cfg {
    static_assert(D == 32 || D == 64 || D == 96 || D == 128, "head dims 32, 64, 96, 128");
    static constexpr int CB = (D + 63) / 64;            // 64-column blocks of a K, V or Q row
    static constexpr int KTILE = kKeys * CB * 128;      // one K tile (TMA fills columns past D with zeros)
    static constexpr int VTILE = kKeys * 2 * 128;       // one V tile: always two blocks (M = 128); with
                                                        // D <= 64 the second holds zeros, written once
    static constexpr int STAGE = KTILE + VTILE;
    static constexpr int STAGES = D <= 64 ? 4 : 3;
    static constexpr int QBLK = kNP * 128;              // one 64-column block of the Q tile (16 rows x 128 B)
    static constexpr int QTILE = CB * QBLK;             // [16 x 64 CB] 16-bit
    static constexpr int PTILE = 2 * QBLK;              // P^T [16 queries x 128 keys] 16-bit
    static constexpr int KV_OFF = 0;                    // stage s: K at s STAGE, V at s STAGE + KTILE
    static constexpr int Q_OFF = KV_OFF + STAGES * STAGE;  // two Q tiles (item parity)
    static constexpr int P_OFF = Q_OFF + 2 * QTILE;           // two P^T tiles (tile parity)
    static constexpr int RED_OFF = P_OFF + 2 * PTILE;          // fp32 [2][4 warps][16] maxima
    static constexpr int LSUM_OFF = RED_OFF + 2 * 4 * kNP * 4; // fp32 [4 warps][16] row sums
    static constexpr int BAR_OFF = LSUM_OFF + 4 * kNP * 4;
    static constexpr int B_FULL = 0;                    // STAGES: K and V of a tile landed
    static constexpr int B_EMPTY = B_FULL + STAGES;     // STAGES: both products have read them
    static constexpr int B_QFULL = B_EMPTY + STAGES;    // 2
    static constexpr int B_QEMPTY = B_QFULL + 2;        // 2
    static constexpr int B_SFULL = B_QEMPTY + 2;        // 2: S^T buffer ready
    static constexpr int B_SFREE = B_SFULL + 2;         // 2: S^T buffer read
    static constexpr int B_PFULL = B_SFREE + 2;         // 2: P^T tile written
    static constexpr int B_ODONE = B_PFULL + 2;         // 2: the O^T product of that P^T tile done
    static constexpr int B_OFREE = B_ODONE + 2;         // O^T read out at an item's end
    static constexpr int B_DRAIN = B_OFREE + 1;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr int SLOT_OFF = BAR_OFF + 8 * NUM_BARS;  // TMEM base address, abort flag
    static constexpr int SMEM_USED = SLOT_OFF + 16;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
    static_assert(QBLK % 1024 == 0 && Q_OFF % 1024 == 0 && P_OFF % 1024 == 0 && STAGE % 1024 == 0 &&
                      KTILE % 1024 == 0,
                  "1024-byte aligned operand tiles");
};

// Byte offset of 16-bit element (row, col) of a [16 rows x 128] tile stored as
// two 64-column blocks of 16 rows x 128 B, 128B-swizzled (16-byte chunk index
// XOR row % 8): the K-major operand layout of the Q and P^T tiles.
__device__ __forceinline__ uint32_t small_tile_offset(int row, int col)
{
    const int chunk = (col & 63) >> 3;
    return static_cast<uint32_t>((col >> 6) * (kNP * 128) + row * 128 + (((chunk ^ (row & 7)) << 4)) + (col & 7) * 2);
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v)
{
    if (!smem_ok(addr, 2, 2))
        return;
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

template <typename T>
__device__ __forceinline__ uint16_t to16(float x)
{
    const uint32_t w = DTypeTraits<T>::pack(x, 0.f);
    return static_cast<uint16_t>(w & 0xFFFFu);
}

template <int D, typename T>
__global__ void __launch_bounds__(kThreads, 1)
    fa_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, dec::Partials part, int Nq, int Nk, int splits,
                        int tiles_per_split, int num_items, int causal, float scale_log2)
{
    using C = Cfg<D>;
    constexpr int STAGES = C::STAGES;
    constexpr int KSTEPS = D / 16;      // S^T: K = d
    constexpr int PSTEPS = kKeys / 16;  // O^T: K = keys

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    auto bar = [&](int idx) -> uint32_t {
        FA_CHECK(idx >= 0 && idx < C::NUM_BARS);
        return sbase + C::BAR_OFF + 8u * idx;
    };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + C::SLOT_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::SLOT_OFF + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_tiles = (Nk + kKeys - 1) / kKeys;
    // item w = (bh, chunk): key tiles [t0, t0 + count) of head bh
    auto item_tiles = [&](int w, int &bh, int &split, int &t0) -> int {
        bh = w / splits;
        split = w % splits;
        t0 = split * tiles_per_split;
        return max(0, min(num_tiles, t0 + tiles_per_split) - t0);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(C::B_FULL + s), 1);
            mbar_init(bar(C::B_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(C::B_QFULL + b), 1);
            mbar_init(bar(C::B_QEMPTY + b), 1);
            mbar_init(bar(C::B_SFULL + b), 1);
            mbar_init(bar(C::B_SFREE + b), 128);
            mbar_init(bar(C::B_PFULL + b), 128);
            mbar_init(bar(C::B_ODONE + b), 1);
        }
        mbar_init(bar(C::B_OFREE), 128);
        mbar_init(bar(C::B_DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
        tmem_relinquish();
    }
    if constexpr (C::CB == 1) {
        // the second 64-column block of every V tile: zeros for the O^T
        // product's rows past D (no load ever writes it)
        if (warp < 4) {
            for (int i = threadIdx.x; i < STAGES * (kSwAtomBytes / 16); i += 128) {
                const int st = i / (kSwAtomBytes / 16), ch = i % (kSwAtomBytes / 16);
                st_shared_v4(sbase + C::KV_OFF + st * C::STAGE + C::KTILE + kSwAtomBytes + ch * 16, 0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();  // read by the tensor core
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            // ---------------- producer ----------------
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const uint64_t pol = l2_policy_evict_first();  // K and V are read once
            int L = 0, items = 0;
            bool ok = true;
            for (int w = blockIdx.x; ok && w < num_items; w += gridDim.x, ++items) {
                int bh, split, t0;
                const int nt = item_tiles(w, bh, split, t0);
                // Q of the item into buffer items % 2 (rows past Nq read as zeros)
                const int qb = items & 1;
                if (items >= 2 && !(ok = wait_bounded(bar(C::B_QEMPTY + qb), ((items / 2) - 1) & 1, abort_flag)))
                    break;
                mbar_arrive_expect_tx(bar(C::B_QFULL + qb), C::QTILE);
                for (int b = 0; b < C::CB; ++b)
                    tma_load_3d(sbase + C::Q_OFF + qb * C::QTILE + b * C::QBLK, &tm_q, bar(C::B_QFULL + qb),
                                b * 64, 0, bh, pol);
                for (int i = 0; i < nt; ++i, ++L) {
                    const int s = L % STAGES;
                    if (L >= STAGES && !(ok = wait_bounded(bar(C::B_EMPTY + s), ((L / STAGES) - 1) & 1, abort_flag)))
                        break;
                    const uint32_t kdst = sbase + C::KV_OFF + s * C::STAGE;
                    mbar_arrive_expect_tx(bar(C::B_FULL + s), 2 * C::CB * kSwAtomBytes);
                    for (int b = 0; b < C::CB; ++b) {
                        tma_load_3d(kdst + b * kSwAtomBytes, &tm_k, bar(C::B_FULL + s), b * 64, (t0 + i) * kKeys,
                                    bh, pol);
                        tma_load_3d(kdst + C::KTILE + b * kSwAtomBytes, &tm_v, bar(C::B_FULL + s), b * 64,
                                    (t0 + i) * kKeys, bh, pol);
                    }
                }
            }
            // wait for every copy this thread issued
            for (int b = 0; b < 2; ++b)
                if (items > b)
                    drain_bounded(bar(C::B_QFULL + b), ((items - 1 - b) / 2) & 1);
            for (int s = 0; s < STAGES; ++s)
                if (L > s)
                    drain_bounded(bar(C::B_FULL + s), ((L - 1 - s) / STAGES) & 1);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            // Global tile g: S^T_g into buffer g % 2, then the O^T product of
            // tile g - 1 (whose P^T the softmax writes meanwhile).
            constexpr bool BF = DTypeTraits<T>::kBF16;
            constexpr uint32_t idesc_s = make_idesc_f16(BF, kKeys, kNP, false, false);
            constexpr uint32_t idesc_o = make_idesc_f16(BF, 128, kNP, true, false);
            const uint64_t desc_k0 = make_sdesc_sw128(sbase + C::KV_OFF, 16, 1024);
            const uint64_t desc_v0 = make_sdesc_sw128(sbase + C::KV_OFF + C::KTILE, kSwAtomBytes, 1024);
            const uint64_t desc_q0 = make_sdesc_sw128(sbase + C::Q_OFF, 16, 1024);
            const uint64_t desc_p0 = make_sdesc_sw128(sbase + C::P_OFF, 16, 1024);
            // the O^T product of global tile gp (item-local tile jp, CTA item ip)
            auto issue_o = [&](int gp, int jp, int ip) -> bool {
                const int b = gp & 1;
                if (!wait_bounded(bar(C::B_PFULL + b), static_cast<uint32_t>((gp >> 1) & 1), abort_flag))
                    return false;
                // an item's first product overwrites O^T, which the previous
                // item's end must have read
                if (jp == 0 && ip > 0 &&
                    !wait_bounded(bar(C::B_OFREE), static_cast<uint32_t>((ip - 1) & 1), abort_flag))
                    return false;
                tc_fence_after();
                const int s = gp % STAGES;
                const uint64_t vd = desc_v0 + static_cast<uint32_t>((s * C::STAGE) >> 4);
                const uint64_t pd = desc_p0 + static_cast<uint32_t>((b * C::PTILE) >> 4);
#pragma unroll
                for (int kk = 0; kk < PSTEPS; ++kk) {
                    const uint32_t voff = static_cast<uint32_t>((kk * 2048) >> 4);   // 16 keys of 128 B
                    const uint32_t poff = static_cast<uint32_t>(((kk >> 2) * C::QBLK + (kk & 3) * 32) >> 4);
                    umma_f16_ss(tmem + kTmO, vd + voff, pd + poff, idesc_o, (jp > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(bar(C::B_ODONE + b));
                umma_commit(bar(C::B_EMPTY + s));  // K and V of tile gp are no longer read
                return true;
            };
            int g = 0;                     // global tile
            int gp = -1, jp = 0, ip = 0;   // the tile whose O^T product is pending
            int items = 0;
            bool ok = true;
            for (int w = blockIdx.x; ok && w < num_items; w += gridDim.x, ++items) {
                int bh, split, t0;
                const int nt = item_tiles(w, bh, split, t0);
                (void)bh;
                (void)t0;
                const int qb = items & 1;
                for (int j = 0; ok && j < nt; ++j, ++g) {
                    if (j == 0 && !(ok = wait_bounded(bar(C::B_QFULL + qb), (items / 2) & 1, abort_flag)))
                        break;
                    const int s = g % STAGES;
                    ok = wait_bounded(bar(C::B_FULL + s), (g / STAGES) & 1, abort_flag) &&
                         (g < 2 || wait_bounded(bar(C::B_SFREE + (g & 1)), static_cast<uint32_t>(((g >> 1) - 1) & 1),
                                                abort_flag));
                    if (!ok)
                        break;
                    tc_fence_after();
                    const uint64_t kd = desc_k0 + static_cast<uint32_t>((s * C::STAGE) >> 4);
                    const uint64_t qd = desc_q0 + static_cast<uint32_t>((qb * C::QTILE) >> 4);
#pragma unroll
                    for (int kk = 0; kk < KSTEPS; ++kk) {
                        const uint32_t koff = static_cast<uint32_t>(((kk >> 2) * kSwAtomBytes + (kk & 3) * 32) >> 4);
                        const uint32_t qoff = static_cast<uint32_t>(((kk >> 2) * C::QBLK + (kk & 3) * 32) >> 4);
                        umma_f16_ss(tmem + (g & 1) * kNP, kd + koff, qd + qoff, idesc_s, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(bar(C::B_SFULL + (g & 1)));
                    if (j + 1 == nt)
                        umma_commit(bar(C::B_QEMPTY + qb));  // every product reading this Q is issued
                    if (gp >= 0 && !(ok = issue_o(gp, jp, ip)))
                        break;
                    gp = g;
                    jp = j;
                    ip = items;
                }
            }
            if (ok && gp >= 0)
                ok = issue_o(gp, jp, ip);
            // every MMA this thread issued has completed once this arrives
            umma_commit(bar(C::B_DRAIN));
            drain_bounded(bar(C::B_DRAIN), 0);
        }
    } else {
        // ---------------- softmax warps 0-3 ----------------
        const int t = threadIdx.x;  // key t of a tile (S^T lane), dimension t of O^T
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        float *red = reinterpret_cast<float *>(smem + C::RED_OFF);    // [2][4][16]
        float *lsum = reinterpret_cast<float *>(smem + C::LSUM_OFF);  // [4][16]
        int g = 0;
        int items = 0;
        bool ok = true;
        for (int w = blockIdx.x; ok && w < num_items; w += gridDim.x, ++items) {
            int bh, split, t0;
            const int nt = item_tiles(w, bh, split, t0);
            float m_ref[kNP], l[kNP];
#pragma unroll
            for (int q = 0; q < kNP; ++q) {
                m_ref[q] = -INFINITY;
                l[q] = 0.f;
            }
            for (int j = 0; j < nt; ++j, ++g) {
                const int b = g & 1;
                ok = wait_warp(bar(C::B_SFULL + b), static_cast<uint32_t>((g >> 1) & 1), abort_flag);
                tc_fence_after();
                uint32_t su[kNP];
                tmem_ld16(tmem + lane_base + b * kNP, su);  // (read whatever the wait gave)
                tc_fence_before();
                if (ok)
                    mbar_arrive(bar(C::B_SFREE + b));
                // scaled scores of key t (log2 units); masked: keys past the
                // last one query q may see, and the padding queries
                const int key = (t0 + j) * kKeys + t;
                float x[kNP];
                bool grow = false;  // some score of this thread outgrows its query's reference
#pragma unroll
                for (int q = 0; q < kNP; ++q) {
                    const int last = causal ? Nk - Nq + q : Nk - 1;
                    x[q] = (q < Nq && key <= last) ? __uint_as_float(su[q]) * scale_log2 : -INFINITY;
                    grow = grow || (x[q] - m_ref[q] > kRescaleLog2);  // (-inf: never; reference -inf: any visible key)
                }
                // The references move only when a score outgrows one by more than
                // 2^kRescaleLog2 (the first visible key of a query always does):
                // one barrier tells every thread whether any did, or whether the
                // CTA stops; only then are the tile's maxima exchanged.
                float alpha[kNP];
#pragma unroll
                for (int q = 0; q < kNP; ++q)
                    alpha[q] = 1.f;
                bool moved = false;  // an earlier reference moved: O^T is rescaled
                if (named_bar_or(1, 128, !ok || *abort_flag != 0 || grow)) {
                    if (named_bar_or(1, 128, !ok || *abort_flag != 0)) {
                        ok = false;
                        break;
                    }
                    // tile maxima per query: warp shuffles, then the four warps
                    float *rb = red + b * 4 * kNP;
#pragma unroll
                    for (int q = 0; q < kNP; ++q) {
                        float v = x[q];
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1)
                            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
                        if (lane == 0)
                            rb[warp * kNP + q] = v;
                    }
                    named_bar_sync(1, 128);
                    // (every thread computes the same maxima and references)
#pragma unroll
                    for (int q = 0; q < kNP; ++q) {
                        const float tmax =
                            fmaxf(fmaxf(rb[q], rb[kNP + q]), fmaxf(rb[2 * kNP + q], rb[3 * kNP + q]));
                        // the reference moves on the first visible key and when the
                        // tile's max outgrows it by more than 2^kRescaleLog2
                        if (tmax != -INFINITY && (m_ref[q] == -INFINITY || tmax - m_ref[q] > kRescaleLog2)) {
                            moved = moved || (j > 0 && m_ref[q] != -INFINITY);
                            alpha[q] = m_ref[q] == -INFINITY ? 0.f : ex2_approx(m_ref[q] - tmax);
                            m_ref[q] = tmax;
                        }
                    }
                }
                float p[kNP];
#pragma unroll
                for (int q = 0; q < kNP; ++q) {
                    p[q] = m_ref[q] == -INFINITY ? 0.f : ex2_approx(x[q] - m_ref[q]);
                    l[q] = l[q] * alpha[q] + p[q];
                }
                // A failed wait below skips the rest of the tile; the next
                // tile's barrier (or the item's end) stops all four warps together.
                // O^T columns of the queries whose reference moved (rare): the
                // previous O^T product (of tile g - 1) must be done
                if (moved) {
                    ok = wait_warp(bar(C::B_ODONE + (b ^ 1)), static_cast<uint32_t>(((g - 1) >> 1) & 1), abort_flag);
                    if (ok) {
                        tc_fence_after();
                        uint32_t ou[kNP];
                        tmem_ld16(tmem + lane_base + kTmO, ou);
#pragma unroll
                        for (int q = 0; q < kNP; ++q)
                            ou[q] = __float_as_uint(__uint_as_float(ou[q]) * alpha[q]);
                        tmem_st16(tmem + lane_base + kTmO, ou);
                        tmem_wait_st();
                    }
                }
                // P^T tile b is free once the O^T product of tile g - 2 is done
                if (ok && g >= 2)
                    ok = wait_warp(bar(C::B_ODONE + b), static_cast<uint32_t>(((g >> 1) - 1) & 1), abort_flag);
                if (ok) {
                    const uint32_t pt = sbase + C::P_OFF + b * C::PTILE;
#pragma unroll
                    for (int q = 0; q < kNP; ++q)
                        st_shared_u16(pt + small_tile_offset(q, t), to16<T>(p[q]));
                    fence_proxy_async_smem();  // generic-proxy writes, read by the tensor core
                    tc_fence_before();
                    mbar_arrive(bar(C::B_PFULL + b));
                }
            }
            // (a tile that failed after its barrier leaves ok false: the item's
            // end barrier below stops every warp)
            // ---------------- the item's partial m, l, O ----------------
            // l: sum over the 128 keys' threads
#pragma unroll
            for (int q = 0; q < kNP; ++q) {
                float v = l[q];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane == 0)
                    lsum[warp * kNP + q] = v;
            }
            // the last O^T product of the item
            if (ok)
                ok = wait_warp(bar(C::B_ODONE + ((g - 1) & 1)), static_cast<uint32_t>(((g - 1) >> 1) & 1),
                               abort_flag);
            if (named_bar_or(1, 128, !ok || *abort_flag != 0)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t ou[kNP];
            tmem_ld16(tmem + lane_base + kTmO, ou);
            tc_fence_before();
            mbar_arrive(bar(C::B_OFREE));  // the next item's first product may overwrite O^T
            const size_t base = (static_cast<size_t>(bh) * splits + split) * Nq;
            if (t < D) {
#pragma unroll
                for (int q = 0; q < kNP; ++q)
                    if (q < Nq)
                        part.o[(base + q) * D + t] = __uint_as_float(ou[q]);
            }
            if (t < Nq) {
                float lq = 0.f, mq = 0.f;
#pragma unroll
                for (int q = 0; q < kNP; ++q)
                    if (q == t) {
                        lq = lsum[q] + lsum[kNP + q] + lsum[2 * kNP + q] + lsum[3 * kNP + q];
                        mq = m_ref[q];
                    }
                part.l[base + t] = lq;
                part.m[base + t] = mq;
            }
            // the row-sum area is read before the next item writes it
            named_bar_sync(1, 128);
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

}  // namespace dectc
}  // namespace fa
