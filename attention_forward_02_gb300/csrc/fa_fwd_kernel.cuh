// fa_fwd_kernel.cuh -- the sm_103a attention-forward kernel.
//
// What it computes, for one (batch*head, 256-row Q block) per CTA:
//   O = softmax(Q K^T * scale) V,   LSE = m * scale + ln(l)
// with the online-softmax recurrence of "3.6 어텐션 I — 메모리 문제·
// FlashAttention 원리", section 3.6.4 (state m, l, O on chip; alpha rescales
// both l and O; one division by l at the end) and the tile loop of section
// 3.6.6 (Q block fixed per CTA, K/V blocks streamed; causal skips blocks above
// the diagonal and masks the diagonal block).  The grid is FA2's: "Triton으로
// FlashAttention 1·2 forward 구현하기", section "병렬화 단위" -- one CTA per
// (Q block, batch*head); the Q blocks of one head are launched next to each
// other so that their shared K/V stream stays in L2.
//
// GB300 mapping (the pages' A100 design used cp.async, ldmatrix and mma.sync):
//   The CTA's Q block is two 128-row sub-tiles h = 0, 1 (one M = 128 tcgen05
//   MMA each) whose softmax work ping-pongs with the tensor core: while
//   sub-tile h runs the softmax of key tile j, the tensor core runs the other
//   sub-tile's P V and Q K^T products.
//   warp 17      TMA producer: Q0, Q1 once; then K_0, V_0, K_1, V_1, ... through
//                a SLOTS-deep ring of 128B-swizzled shared tiles.
//   warp 16      MMA issuer (one thread), per key tile j and sub-tile h:
//                O_h += P_h,j V_j  then  S_h,j+1 = Q_h K_{j+1}^T  (tcgen05.mma,
//                fp32 accumulators in TMEM).  V is an MN-major B operand.
//   warps 0-15   softmax: sub-tile h = warp / 8 uses warps 8h .. 8h+7.  Query
//                row r of the sub-tile is TMEM lane r; its 128 scores are split
//                between two threads -- half a = 0 takes keys 0-63 (warp
//                8h + r/32), half a = 1 keys 64-127 (warp 8h + 4 + r/32).  The
//                two halves run on the same SM sub-partition and hide each
//                other's latency; they exchange partial row maxima (and, at the
//                end, partial sums) through shared memory.
// Per key tile each thread loads its 64 scores, masks, takes the partial row
// max, exponentiates p = 2^(s*c - m*c) (one packed FMA per pair + ex2) against
// the current reference max, sums, and writes P (rounded to the input dtype)
// into TMEM for the second product.  The reference max moves only when the row
// max grows by more than kRescaleLog2 (log2 units), which is rare; then the
// tile is redone against the new max and l and O are rescaled by alpha.  O and
// l always share the same reference, so O / l and LSE are unchanged (any
// common reference cancels, the algebra of section 3.6.4); p <= 2^kRescaleLog2.
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

constexpr int kSubM = 128;       // rows per sub-tile (one M = 128 MMA; one TMEM lane per row)
constexpr int kBM = 2 * kSubM;   // query rows per CTA
constexpr int kBN = 128;         // keys per K/V tile
constexpr int kHalf = kBN / 2;   // keys per softmax thread
// Five warpgroups: four softmax warpgroups (warps 0-15) and a control
// warpgroup (warp 16 MMA issuer, warp 17 TMA producer, warps 18-19 idle).
// Launched at 96 registers per thread (640 x 96 = 61440); the control
// warpgroup drops to kRegsControl and the softmax warps rise to kRegsSoftmax.
constexpr int kNumThreads = 640;
constexpr int kNumSoftmaxThreads = 512;
constexpr int kMmaWarp = 16;
constexpr int kTmaWarp = 17;
constexpr uint32_t kLaunchRegs = 96;
constexpr uint32_t kRegsSoftmax = 104;
constexpr uint32_t kRegsControl = 64;
static_assert(kNumSoftmaxThreads * kRegsSoftmax + 128 * kRegsControl <= kNumThreads * kLaunchRegs,
              "register split");
// TMEM columns: S0 @ 0, S1 @ 128, O0 @ 256, O1 @ 256 + D.  P_h (16-bit, two
// per column) takes 64 columns: for D = 64 the spare columns 384 + 64 h, for
// D = 128 the first half of S_h (the next S_h product is issued after the
// P_h V product that reads it, and tcgen05.mma ops of one thread execute in
// issue order).
constexpr uint32_t kTmemCols = 512;
template <int D>
__host__ __device__ constexpr uint32_t tmem_p_col(int h)
{
    return D == 64 ? 384u + 64u * h : 128u * h;
}
constexpr float kRescaleLog2 = 8.0f;
constexpr long long kWaitLimitCycles = 1ll << 31;  // about one second at 2 GHz
constexpr int kSwAtomBytes = 128 * 128;             // [128 rows x 64 cols] 16-bit swizzle block

template <int D>
struct KCfg {
    static constexpr int TILE = 128 * D * 2;  // bytes of one [128, D] 16-bit tile
    static constexpr int SLOTS = D == 64 ? 6 : 4;
    static constexpr int Q_OFF = 0;           // Q0, Q1 (later the O staging of each sub-tile)
    static constexpr int KV_OFF = Q_OFF + 2 * TILE;
    static constexpr int X_OFF = KV_OFF + SLOTS * TILE;  // float [2 parity][2 h][2 half][128 rows]
    static constexpr int X_BYTES = 2 * 2 * 2 * 128 * 4;
    static constexpr int BAR_OFF = X_OFF + X_BYTES;
    static constexpr int B_QFULL = 0;
    static constexpr int B_KVFULL = 1;
    static constexpr int B_KVEMPTY = B_KVFULL + SLOTS;
    static constexpr int B_SFULL = B_KVEMPTY + SLOTS;  // two
    static constexpr int B_PFULL = B_SFULL + 2;        // two
    static constexpr int B_OFINAL = B_PFULL + 2;       // two
    static constexpr int B_DRAIN = B_OFINAL + 2;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr int SLOT_OFF = BAR_OFF + 8 * NUM_BARS;  // TMEM base address, abort flag
    static constexpr int SMEM_USED = SLOT_OFF + 16;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack for 1024-byte alignment
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
    static_assert(256 + 2 * D <= static_cast<int>(kTmemCols), "TMEM budget");
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

// Byte offset of 16-byte chunk `chunk` of row `row` in a [128, 64*k] 16-bit
// tile stored as k column blocks of [128 rows x 128 B], each 128B-swizzled
// (chunk index XOR row % 8): the layout TMA SWIZZLE_128B writes and the
// tcgen05 SW128 descriptors read.
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk)
{
    return static_cast<uint32_t>((chunk >> 3) * kSwAtomBytes + row * 128 +
                                 (((chunk & 7) ^ (row & 7)) << 4));
}

// Masks keys c >= limit of one half-row of scores (set to -inf).
__device__ __forceinline__ void mask_tail(float (&s)[kHalf], int limit)
{
#pragma unroll
    for (int c = 0; c < kHalf; ++c)
        if (c >= limit)
            s[c] = -INFINITY;
}

// Maximum of 64 scores: eight independent three-input max chains.
__device__ __forceinline__ float half_max(const float (&s)[kHalf])
{
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        a[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
    for (int c = 16; c < kHalf; c += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i)
            a[i] = fmax3(a[i], s[c + 2 * i], s[c + 2 * i + 1]);
    return fmaxf(fmax3(a[0], a[1], a[2]), fmax3(fmax3(a[3], a[4], a[5]), a[6], a[7]));
}

// In place: s[c] <- 2^(s[c] * c2 + neg_mc) (0 for masked keys c >= limit);
// returns the sum, accumulated as four packed pairs.
template <bool MASKED>
__device__ __forceinline__ float exp_half(float (&s)[kHalf], int limit, float c2, float neg_mc)
{
    float2 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        acc[i] = make_float2(0.f, 0.f);
    const float2 cc = make_float2(c2, c2);
    const float2 nn = make_float2(neg_mc, neg_mc);
#pragma unroll
    for (int c = 0; c < kHalf; c += 2) {
        const float2 x = ffma2(make_float2(s[c], s[c + 1]), cc, nn);
        float e0 = ex2_approx(x.x);
        float e1 = ex2_approx(x.y);
        if (MASKED) {
            e0 = (c < limit) ? e0 : 0.f;
            e1 = (c + 1 < limit) ? e1 : 0.f;
        }
        s[c] = e0;
        s[c + 1] = e1;
        acc[(c >> 1) & 3] = fadd2(acc[(c >> 1) & 3], make_float2(e0, e1));
    }
    const float2 t = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
    return t.x + t.y;
}

template <int D, bool CAUSAL, typename T>
__global__ void __launch_bounds__(kNumThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, T *__restrict__ out,
                  float *__restrict__ lse, int N, int num_q_blocks, float scale, float scale_log2)
{
    using C = KCfg<D>;
    constexpr int SLOTS = C::SLOTS;
    constexpr int KSTEPS_QK = D / 16;  // UMMA_K = 16 for 16-bit operands
    constexpr int KSTEPS_PV = kBN / 16;
    constexpr uint32_t kTmemO = 256;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Q blocks of one head are adjacent in launch order (shared K/V stays in
    // L2); within a head the heaviest causal blocks go first.
    const int bh = static_cast<int>(blockIdx.x / static_cast<unsigned>(num_q_blocks));
    const int qb = num_q_blocks - 1 - static_cast<int>(blockIdx.x % static_cast<unsigned>(num_q_blocks));
    const int row0 = qb * kBM;
    const int num_k_tiles = (N + kBN - 1) / kBN;
    const int nk0 = CAUSAL ? min(2 * qb + 1, num_k_tiles) : num_k_tiles;  // sub-tile 0
    const int nk1 = CAUSAL ? min(2 * qb + 2, num_k_tiles) : num_k_tiles;  // sub-tile 1 (>= nk0)

    auto bar = [&](int idx) -> uint32_t { return sbase + C::BAR_OFF + 8u * idx; };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + C::SLOT_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::SLOT_OFF + 4);

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_QFULL), 1);
        for (int s = 0; s < SLOTS; ++s) {
            mbar_init(bar(C::B_KVFULL + s), 1);
            mbar_init(bar(C::B_KVEMPTY + s), 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(bar(C::B_SFULL + h), 1);
            mbar_init(bar(C::B_PFULL + h), 2 * kSubM);
            mbar_init(bar(C::B_OFINAL + h), 1);
        }
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

    if (warp >= kMmaWarp) {
        reg_dealloc<kRegsControl>();
        if (warp == kTmaWarp && lane == 0) {
            // ---------------- producer ----------------
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            mbar_arrive_expect_tx(bar(C::B_QFULL), 2 * C::TILE);
            for (int h = 0; h < 2; ++h)
                for (int b = 0; b < D / 64; ++b)
                    tma_load_3d(sbase + C::Q_OFF + h * C::TILE + b * kSwAtomBytes, &tm_q,
                                bar(C::B_QFULL), b * 64, row0 + h * kSubM, bh, pol_q);
            int issued = 0;  // loads into the ring: K_j = load 2j, V_j = load 2j + 1
            for (int L = 0; L < 2 * nk1; ++L) {
                const int s = L % SLOTS;
                if (L >= SLOTS && !wait_bounded(bar(C::B_KVEMPTY + s), ((L / SLOTS) - 1) & 1, abort_flag))
                    break;
                const CUtensorMap *map = (L & 1) ? &tm_v : &tm_k;
                mbar_arrive_expect_tx(bar(C::B_KVFULL + s), C::TILE);
                for (int b = 0; b < D / 64; ++b)
                    tma_load_3d(sbase + C::KV_OFF + s * C::TILE + b * kSwAtomBytes, map,
                                bar(C::B_KVFULL + s), b * 64, (L >> 1) * kBN, bh, pol_kv);
                ++issued;
            }
            // Wait for every copy this thread issued (immediate on the normal
            // path, where each one was consumed).
            drain_bounded(bar(C::B_QFULL), 0);
            for (int s = 0; s < SLOTS; ++s)
                if (issued > s)
                    drain_bounded(bar(C::B_KVFULL + s), ((issued - 1 - s) / SLOTS) & 1);
        } else if (warp == kMmaWarp && lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t idesc_s = make_idesc_f16(DTypeTraits<T>::kBF16, kSubM, kBN, false, false);
            constexpr uint32_t idesc_o = make_idesc_f16(DTypeTraits<T>::kBF16, kSubM, D, false, true);
            auto slot_of = [](int L) { return L % SLOTS; };
            auto par_of = [](int L) { return static_cast<uint32_t>((L / SLOTS) & 1); };
            // Descriptors of the ring's first tile and of Q0; a tile at byte
            // offset x from them is the same descriptor plus x >> 4 (the start
            // address field; shared addresses stay below 256 KiB, so no carry).
            const uint64_t kv_desc_k = make_sdesc_sw128(sbase + C::KV_OFF, 16, 1024);
            const uint64_t kv_desc_v = make_sdesc_sw128(sbase + C::KV_OFF, kSwAtomBytes, 1024);
            const uint64_t q_desc = make_sdesc_sw128(sbase + C::Q_OFF, 16, 1024);
            auto issue_s = [&](int h, int j) {
                const uint64_t kd = kv_desc_k + ((slot_of(2 * j) * C::TILE) >> 4);
                const uint64_t qd = q_desc + ((h * C::TILE) >> 4);
#pragma unroll
                for (int kk = 0; kk < KSTEPS_QK; ++kk) {
                    const uint32_t koff = ((kk >> 2) * kSwAtomBytes + (kk & 3) * 32) >> 4;
                    umma_f16_ss(tmem + h * kBN, qd + koff, kd + koff, idesc_s, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int h, int j) {
                const uint64_t vd = kv_desc_v + ((slot_of(2 * j + 1) * C::TILE) >> 4);
                const uint32_t od = tmem + kTmemO + h * D;
#pragma unroll
                for (int kk = 0; kk < KSTEPS_PV; ++kk) {
                    // V: MN-major; 16 key rows (2048 B) per K step; the two
                    // 64-column blocks of D = 128 are kSwAtomBytes apart.
                    // P_h,j: 16-bit in TMEM, two per column, 8 columns per K step.
                    umma_f16_ts(od, tmem + tmem_p_col<D>(h) + kk * 8, vd + ((kk * 2048) >> 4), idesc_o,
                                (j > 0 || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = wait_bounded(bar(C::B_QFULL), 0, abort_flag) &&
                      wait_bounded(bar(C::B_KVFULL + slot_of(0)), par_of(0), abort_flag);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                umma_commit(bar(C::B_SFULL + 0));
                issue_s(1, 0);
                umma_commit(bar(C::B_SFULL + 1));
                umma_commit(bar(C::B_KVEMPTY + slot_of(0)));
            }
            for (int j = 0; ok && j < nk1; ++j) {
                ok = wait_bounded(bar(C::B_KVFULL + slot_of(2 * j + 1)), par_of(2 * j + 1), abort_flag);
                bool have_next_k = false;
                for (int h = 0; ok && h < 2; ++h) {
                    const int nkh = h == 0 ? nk0 : nk1;
                    if (j >= nkh)
                        continue;
                    ok = wait_bounded(bar(C::B_PFULL + h), j & 1, abort_flag);
                    if (!ok)
                        break;
                    tc_fence_after();
                    issue_pv(h, j);
                    if (j + 1 < nkh) {
                        if (!have_next_k) {
                            ok = wait_bounded(bar(C::B_KVFULL + slot_of(2 * j + 2)), par_of(2 * j + 2),
                                              abort_flag);
                            if (!ok)
                                break;
                            tc_fence_after();
                            have_next_k = true;
                        }
                        issue_s(h, j + 1);
                        umma_commit(bar(C::B_SFULL + h));
                    } else {
                        umma_commit(bar(C::B_OFINAL + h));
                    }
                }
                if (!ok)
                    break;
                umma_commit(bar(C::B_KVEMPTY + slot_of(2 * j + 1)));  // V_j: both P V products issued
                if (have_next_k)
                    umma_commit(bar(C::B_KVEMPTY + slot_of(2 * j + 2)));  // K_{j+1}: both S products
            }
            // every MMA issued above has completed once this arrives
            umma_commit(bar(C::B_DRAIN));
            drain_bounded(bar(C::B_DRAIN), 0);
        }
    } else {
        reg_alloc<kRegsSoftmax>();
        // ---------------- softmax: sub-tile h, key half a ----------------
        const int h = warp >> 3;
        const int a = (warp >> 2) & 1;
        const int r = ((warp & 3) << 5) | lane;  // row within the sub-tile == TMEM lane
        const int qrow = row0 + h * kSubM + r;
        const int nkh = h == 0 ? nk0 : nk1;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t s_tm = tmem + lane_base + static_cast<uint32_t>(h * kBN + a * kHalf);
        const uint32_t o_tm = tmem + lane_base + kTmemO + static_cast<uint32_t>(h * D + a * (D / 2));
        const uint32_t p_tm = tmem + lane_base + tmem_p_col<D>(h) + static_cast<uint32_t>(a * kHalf / 2);
        // partial-max exchange: [parity][h][half][row]
        float *xch = reinterpret_cast<float *>(smem + C::X_OFF);
        auto xslot = [&](int par, int half) { return xch + ((par * 2 + h) * 2 + half) * 128 + r; };
        const uint32_t pair_bar = 1 + (h << 2) + (warp & 3);  // the two warps sharing these rows
        float m_ref = -INFINITY;  // reference max (raw score units; scale >= 0)
        float l = 0.f;            // this half's share of the row sum
        bool ok = true;
        for (int j = 0; j < nkh; ++j) {
            // The two warps of a pair pass the same named barriers in the same
            // order: each reaches the exchange below even when its wait failed
            // (it then posts NaN), and both leave the loop together after it.
            ok = wait_bounded(bar(C::B_SFULL + h), j & 1, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            float s[kHalf];
            float mh = NAN;
            float rsum = 0.f;
            // keys [kbase, kbase + limit) of this half are allowed (limit may be <= 0)
            const int kbase = j * kBN + a * kHalf;
            int limit = min(kHalf, N - kbase);
            if (CAUSAL)
                limit = min(limit, qrow - kbase + 1);
            const bool masked = __any_sync(0xffffffffu, limit < kHalf);
            if (ok) {
                tc_fence_after();
                tmem_ld64(s_tm, s);
                if (masked)
                    mask_tail(s, limit);
                // Tile 0 sets the reference max from the exchanged row max.
                // Later tiles exponentiate against the current reference while
                // the row max is taken and exchanged; only a row max that
                // outgrows the reference by more than kRescaleLog2 (rare) sends
                // the two warps down the redo path.
                mh = half_max(s);
                if (j > 0)
                    rsum = masked ? exp_half<true>(s, limit, scale_log2, -m_ref * scale_log2)
                                  : exp_half<false>(s, limit, scale_log2, -m_ref * scale_log2);
            }
            *xslot(j & 1, a) = mh;
            named_bar_sync(pair_bar, 64);
            const float mo = *xslot(j & 1, a ^ 1);
            ok = __all_sync(0xffffffffu, ok && !isnan(mo));
            if (!ok)
                break;
            const float mt = fmaxf(mh, mo);
            float alpha = 1.f;
            if (j == 0) {
                m_ref = mt;
                alpha = 0.f;
                rsum = masked ? exp_half<true>(s, limit, scale_log2, -m_ref * scale_log2)
                              : exp_half<false>(s, limit, scale_log2, -m_ref * scale_log2);
            } else {
                // identical decision in both halves: mt and m_ref are shared
                const bool grow = (mt - m_ref) * scale_log2 > kRescaleLog2;
                if (__any_sync(0xffffffffu, grow)) {
                    if (grow) {
                        alpha = ex2_approx((m_ref - mt) * scale_log2);
                        m_ref = mt;
                    }
                    // S_h is intact until P_h is written below: redo the tile
                    tmem_ld64(s_tm, s);
                    if (masked)
                        mask_tail(s, limit);
                    rsum = masked ? exp_half<true>(s, limit, scale_log2, -m_ref * scale_log2)
                                  : exp_half<false>(s, limit, scale_log2, -m_ref * scale_log2);
                }
            }
            l = l * alpha + rsum;

            // P_h,j (this half's 64 keys) rounded to the input dtype
            {
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    w[c] = DTypeTraits<T>::pack(s[2 * c], s[2 * c + 1]);
                tmem_st32(p_tm, w);
            }
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                // O_h holds P V up to tile j-1 (the S_h,j product, issued after
                // P_h,j-1 V_{j-1}, has completed) and P_h,j V_j is not issued
                // before both halves arrive below.  Each half rescales D/2 columns.
#pragma unroll 1
                for (int c4 = 0; c4 < D / 64; ++c4) {
                    uint32_t u[32];
                    tmem_ld32(o_tm + c4 * 32, u);
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const float2 v = fmul2(make_float2(__uint_as_float(u[c]), __uint_as_float(u[c + 1])),
                                               make_float2(alpha, alpha));
                        u[c] = __float_as_uint(v.x);
                        u[c + 1] = __float_as_uint(v.y);
                    }
                    tmem_st32(o_tm + c4 * 32, u);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(C::B_PFULL + h));
        }

        // ---------------- epilogue of sub-tile h ----------------
        // Every softmax thread of the sub-tile reaches both barriers below; a
        // warp that gave up has set the abort flag first, so after the
        // sub-tile barrier its eight warps agree on whether the tile is whole.
        if (ok) {
            ok = wait_bounded(bar(C::B_OFINAL + h), 0, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
        }
        // parity nkh & 1 was last read before the final tile's exchange
        *xslot(nkh & 1, a) = l;
        named_bar_sync(pair_bar, 64);
        const float l_row = l + *xslot(nkh & 1, a ^ 1);
        // Q_h is dead: every product that read it has completed.
        const uint32_t stage = sbase + C::Q_OFF + h * C::TILE;
        if (ok) {
            tc_fence_after();
            const float inv_l = 1.f / l_row;
#pragma unroll 1
            for (int c4 = 0; c4 < D / 64; ++c4) {
                uint32_t u[32];
                tmem_ld32(o_tm + c4 * 32, u);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const float *f = reinterpret_cast<const float *>(u) + q4 * 8;
                    st_shared_v4(stage + sw128_offset(r, a * (D / 16) + c4 * 4 + q4),
                                 DTypeTraits<T>::pack(f[0] * inv_l, f[1] * inv_l),
                                 DTypeTraits<T>::pack(f[2] * inv_l, f[3] * inv_l),
                                 DTypeTraits<T>::pack(f[4] * inv_l, f[5] * inv_l),
                                 DTypeTraits<T>::pack(f[6] * inv_l, f[7] * inv_l));
                }
            }
            if (a == 0 && lse != nullptr && qrow < N)
                lse[static_cast<size_t>(bh) * N + qrow] = m_ref * scale + logf(l_row);
        }
        named_bar_sync(9 + h, 2 * kSubM);
        if (*abort_flag == 0) {
            constexpr int CHUNKS_PER_ROW = D / 8;
            const int srow0 = row0 + h * kSubM;
            const int t = a * kSubM + r;  // 0 .. 255 within the sub-tile
            uint8_t *obase = reinterpret_cast<uint8_t *>(out) +
                             (static_cast<size_t>(bh) * N + srow0) * D * sizeof(T);
#pragma unroll 4
            for (int idx = t; idx < kSubM * CHUNKS_PER_ROW; idx += 2 * kSubM) {
                const int row = idx / CHUNKS_PER_ROW;
                const int ch = idx % CHUNKS_PER_ROW;
                const uint4 val = ld_shared_v4(stage + sw128_offset(row, ch));
                if (srow0 + row < N)
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
