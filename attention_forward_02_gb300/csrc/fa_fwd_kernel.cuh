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
//   warpgroup h runs the softmax of tile j, the tensor core runs the other
//   sub-tile's P V and Q K^T products.
//   warp 9       TMA producer: Q0, Q1 once; then K_0, V_0, K_1, V_1, ... through
//                a SLOTS-deep ring of 128B-swizzled shared tiles.  With D <= 64
//                the softmax warpgroups free the ring slots (K_j once their
//                S_h,j is complete, V_j once P_h,j V_j is), which keeps those
//                commits off the MMA issuers; with D > 64 the issuer does.
//   warps 8, 10  MMA issuers of sub-tiles 0 and 1 (one thread each), per key
//                tile j: O_h += P_h,j V_j and S_h,j+1 = Q_h K_{j+1}^T
//                (tcgen05.mma, fp32 accumulators in TMEM).  V is an MN-major
//                B operand.
//   warps 4h..4h+3  softmax warpgroup of sub-tile h: thread t owns query row t
//                = TMEM lane t.  It loads S, masks, takes the row max (D <= 64,
//                non-causal: only when the tile's sum shows the reference may
//                have to move), updates the reference max, rescales l and O
//                (in TMEM) by alpha, forms
//                p = 2^(s*c - m*c) with one FMA + ex2, sums l in fp32, rounds P
//                to the input dtype (D <= 64: in the same loop) into TMEM, and
//                finally stages O / l in shared memory (D <= 64: one TMA
//                tensor store writes it out) and writes LSE.
// The reference max moves only when the row max grows by more than
// kRescaleLog2 (in log2 units).  O and l always share the same reference, so
// the final O / l and LSE are unchanged (the same algebra as section 3.6.4:
// any common reference cancels in O / l); p stays <= 2^kRescaleLog2.
// Every mbarrier wait is bounded: on expiry the CTA records a timeout in the
// device status word, stops, waits (bounded) for its own copies and MMAs,
// frees its TMEM and exits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "fa_common.cuh"

namespace fa {

constexpr int kSubM = 128;          // rows per sub-tile (one M = 128 MMA; one TMEM lane per row)
constexpr int kBM = 2 * kSubM;      // query rows per CTA
constexpr int kBN = 128;            // keys per K/V tile
// Three warpgroups: two softmax warpgroups (warps 0-7) and a control
// warpgroup (warps 8 and 10 MMA issuers of sub-tiles 0 and 1, warp 9 TMA
// producer, warp 11 idle).
// Launched at 168 registers per thread (384 x 168 = 64512); the control
// warpgroup drops to 72 and the softmax warpgroups rise to 216 for the
// non-causal D <= 64 launch (96 and 200 otherwise, measured faster there):
// 256 x 216 + 128 x 72 = 64512.
constexpr int kNumThreads = 384;
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr uint32_t kRegsSoftmax = 216;  // D <= 64, non-causal (S and P of a tile live at once)
constexpr uint32_t kRegsControl = 72;
constexpr uint32_t kRegsSoftmaxWide = 200;
constexpr uint32_t kRegsControlWide = 96;
static_assert(256 * kRegsSoftmax + 128 * kRegsControl <= 384 * 168, "register split");
static_assert(256 * kRegsSoftmaxWide + 128 * kRegsControlWide <= 384 * 168, "register split");
// TMEM columns: S0 @ 0, S1 @ 128, O0 @ 256, O1 @ 256 + D.  P_h (16-bit, two
// per column) takes 64 columns: for D <= 64 the spare columns 256 + 2D + 64 h,
// for D > 64 the first half of S_h (the next S_h product is issued after the
// P_h V product that reads it, and tcgen05.mma ops of one thread execute in
// issue order).
constexpr uint32_t kTmemCols = 512;
template <int D>
__host__ __device__ constexpr uint32_t tmem_p_col(int h)
{
    return D <= 64 ? 256u + 2u * D + 64u * h : 128u * h;
}
// Head dims 32 and 96 use the same tiles as 64 and 128: every row of a Q, K
// or V tile is a whole number of 64-column (128-byte) swizzle blocks, and TMA
// fills the columns past D with zeros (nothing past D is read from memory).
// One 128-byte swizzle for every head dim, as "FlashAttention-2를 CuTe로
// 밑바닥부터 구현하며 겪은 GPU 커널 지옥기" (section "V copy와 이상한 no-op
// 이야기") suggests instead of a per-head-dim pattern.
template <int D>
__host__ __device__ constexpr int col_blocks()
{
    return (D + 63) / 64;
}
constexpr float kRescaleLog2 = 8.0f;
constexpr float kRescaleBound = 256.0f;  // 2^kRescaleLog2

template <int D>
struct KCfg {
    static_assert(D == 32 || D == 64 || D == 96 || D == 128, "head dims 32, 64, 96, 128");
    static constexpr int TILE = 128 * col_blocks<D>() * 128;  // bytes of one [128, D] 16-bit tile
    // D <= 64: a 6-slot K/V ring, O staging tiles of their own and two Q
    // buffers per sub-tile, so that the next item's Q lands while this item
    // still runs and its first S product can follow this item's last S.
    // D > 64: a 4-slot ring; O is staged in the sub-tile's only Q tile, which
    // the next item's Q then waits for (its items are long, so that wait
    // matters little).
    static constexpr bool STAGE_IN_Q = D > 64;
    static constexpr int QBUF = STAGE_IN_Q ? 1 : 2;
    static constexpr int SLOTS = D <= 64 ? 6 : 4;
    static constexpr int Q_OFF = 0;                      // Q tile (h, buffer b) at h + 2 b
    static constexpr int KV_OFF = Q_OFF + 2 * QBUF * TILE;  // K/V ring
    static constexpr int OST_OFF = STAGE_IN_Q ? Q_OFF : KV_OFF + SLOTS * TILE;  // O staging
    static constexpr int BAR_OFF = KV_OFF + SLOTS * TILE + (STAGE_IN_Q ? 0 : 2 * TILE);
    static constexpr int B_QFULL = 0;                    // 2 QBUF, (h, b) at h + 2 b
    static constexpr int B_QEMPTY = B_QFULL + 2 * QBUF;  // 2 QBUF
    static constexpr int B_KVFULL = B_QEMPTY + 2 * QBUF;
    static constexpr int B_KVEMPTY = B_KVFULL + SLOTS;
    static constexpr int B_SFULL = B_KVEMPTY + SLOTS;  // two
    static constexpr int B_PFULL = B_SFULL + 2;        // two
    static constexpr int B_OFINAL = B_PFULL + 2;       // two
    static constexpr int B_SFREE = B_OFINAL + 2;       // two (early-S order only)
    static constexpr int B_OREADY = B_SFREE + 2;       // two (early-S order only)
    static constexpr int B_OFREE = B_OREADY + 2;       // two
    static constexpr int B_DRAIN = B_OFREE + 2;        // two (one per MMA issuer)
    static constexpr int NUM_BARS = B_DRAIN + 2;
    static constexpr int SLOT_OFF = BAR_OFF + 8 * NUM_BARS;  // TMEM base address, abort flag
    static constexpr int SMEM_USED = SLOT_OFF + 16;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack for 1024-byte alignment
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
    static_assert(256 + 2 * D <= static_cast<int>(kTmemCols), "TMEM budget");
};

// Masks keys c >= limit of one row of scores (set to -inf).
__device__ __forceinline__ void mask_tail(float (&s)[kBN], int limit)
{
#pragma unroll
    for (int c = 0; c < kBN; ++c)
        if (c >= limit)
            s[c] = -INFINITY;
}

// Row maximum of 128 scores: eight independent three-input max chains.
__device__ __forceinline__ float row_max(const float (&s)[kBN])
{
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        a[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
    for (int c = 16; c < kBN; c += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i)
            a[i] = fmax3(a[i], s[c + 2 * i], s[c + 2 * i + 1]);
    return fmaxf(fmax3(a[0], a[1], a[2]), fmax3(fmax3(a[3], a[4], a[5]), a[6], a[7]));
}

// In place: s[c] <- 2^(s[c] * c2 + neg_mc) (0 for masked keys c >= limit);
// returns the row sum, accumulated as four packed pairs.
template <bool MASKED>
__device__ __forceinline__ float exp_tile(float (&s)[kBN], int limit, float c2, float neg_mc)
{
    float2 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        acc[i] = make_float2(0.f, 0.f);
    const float2 cc = make_float2(c2, c2);
    const float2 nn = make_float2(neg_mc, neg_mc);
#pragma unroll
    for (int c = 0; c < kBN; c += 2) {
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

// As exp_tile, but each pair of exponentials is rounded to 16 bits in the
// same loop (pw[c] = keys 2c, 2c + 1), so the conversions run beside the
// ex2 work instead of after it; s is left as it was.  Returns the fp32 row sum.
template <bool MASKED, typename T>
__device__ __forceinline__ float exp_pack_tile(const float (&s)[kBN], uint32_t (&pw)[kBN / 2], int limit, float c2,
                                               float neg_mc)
{
    float2 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        acc[i] = make_float2(0.f, 0.f);
    const float2 cc = make_float2(c2, c2);
    const float2 nn = make_float2(neg_mc, neg_mc);
#pragma unroll
    for (int c = 0; c < kBN; c += 2) {
        const float2 x = ffma2(make_float2(s[c], s[c + 1]), cc, nn);
        float e0 = ex2_approx(x.x);
        float e1 = ex2_approx(x.y);
        if (MASKED) {
            e0 = (c < limit) ? e0 : 0.f;
            e1 = (c + 1 < limit) ? e1 : 0.f;
        }
        pw[c >> 1] = DTypeTraits<T>::pack(e0, e1);
        acc[(c >> 1) & 3] = fadd2(acc[(c >> 1) & 3], make_float2(e0, e1));
    }
    const float2 t = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
    return t.x + t.y;
}

// Work item w (a 256-row Q block of one head) of a launch with BH heads and
// nqb Q blocks per head.  Non-causal: head-major, so the CTAs working at the
// same time share few heads' K/V in L2.  Causal: heaviest blocks (highest qb)
// of every head first.
template <bool CAUSAL>
__device__ __forceinline__ void item_coords(int w, int BH, int nqb, int &bh, int &qb)
{
    if (CAUSAL) {
        qb = nqb - 1 - w / BH;
        bh = w % BH;
    } else {
        bh = w / nqb;
        qb = w % nqb;
    }
}

// The it-th work item of this CTA: round-robin over the grid; for causal
// launches the direction alternates every round (heavy and light items even out).
template <bool CAUSAL>
__device__ __forceinline__ int item_of(int it)
{
    const int c = (CAUSAL && (it & 1)) ? static_cast<int>(gridDim.x - 1 - blockIdx.x)
                                       : static_cast<int>(blockIdx.x);
    return it * static_cast<int>(gridDim.x) + c;
}

template <int D, bool CAUSAL, typename T>
__global__ void __launch_bounds__(kNumThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  T *__restrict__ out, float *__restrict__ lse, int N, int BH, int num_q_blocks, float scale,
                  float scale_log2)
{
    using C = KCfg<D>;
    // Early-S order (D = 64, where P has TMEM columns of its own): S_h,j+1 is
    // issued as soon as sub-tile h's softmax has finished with S_h,j, ahead of
    // P_h,j V_j, so the two softmax warpgroups need not wait for each other's
    // products.  With D = 128, P overwrites S_h, so S_h,j+1 follows P_h,j V_j.
    constexpr bool EARLY_S = D <= 64;
    constexpr int NUM_ISSUERS = EARLY_S ? 2 : 1;
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
    const int num_items = BH * num_q_blocks;
    const int num_k_tiles = (N + kBN - 1) / kBN;
    // key tiles of row half hr (rows qb kBM + hr kSubM ...) of Q block qb
    auto nk_sub = [&](int qb, int hr) {
        return CAUSAL ? min(2 * qb + 1 + hr, num_k_tiles) : num_k_tiles;
    };
    // Causal: the lower row half sees one key tile more.  Sub-tile h takes row
    // half h ^ swap_of(it), so the extra tile alternates between the two
    // softmax warpgroups from one item of a CTA to the next and neither runs
    // ahead of the other by more than a tile (the K/V ring would stop it).
    auto swap_of = [](int it) { return CAUSAL ? (it & 1) : 0; };

    auto bar = [&](int idx) -> uint32_t {
        FA_CHECK(idx >= 0 && idx < C::NUM_BARS);
        return sbase + C::BAR_OFF + 8u * idx;
    };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + C::SLOT_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::SLOT_OFF + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < SLOTS; ++s) {
            mbar_init(bar(C::B_KVFULL + s), 1);
            // released by the two softmax warpgroups (early-S order) or by
            // each MMA issuer
            mbar_init(bar(C::B_KVEMPTY + s), EARLY_S ? 2 : NUM_ISSUERS);
        }
        for (int q = 0; q < 2 * C::QBUF; ++q) {
            mbar_init(bar(C::B_QFULL + q), 1);
            // released by the products that read Q_h (one commit) and, when O
            // is staged in Q_h, by the epilogue's copy-out (128 arrivals)
            mbar_init(bar(C::B_QEMPTY + q), 1 + (C::STAGE_IN_Q ? 4 * 32 : 0));
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(bar(C::B_SFULL + h), 1);
            mbar_init(bar(C::B_PFULL + h), 4 * 32);
            mbar_init(bar(C::B_OFINAL + h), 1);
            mbar_init(bar(C::B_SFREE + h), 4 * 32);
            mbar_init(bar(C::B_OREADY + h), 1);
            mbar_init(bar(C::B_OFREE + h), 4 * 32);
            mbar_init(bar(C::B_DRAIN + h), 1);
        }
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
      reg_dealloc<((D <= 64 && !CAUSAL) ? kRegsControl : kRegsControlWide)>();
      if (warp == kTmaWarp && lane == 0) {
            // ---------------- producer: per work item Q0, Q1, then K_0, V_0, K_1, V_1, ... ----------------
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            int L = 0;  // loads into the ring so far (all items)
            int items = 0;
            bool ok = true;
            for (int it = 0; ok; ++it) {
                const int w = item_of<CAUSAL>(it);
                if (w >= num_items)
                    break;
                int bh, qb;
                item_coords<CAUSAL>(w, BH, num_q_blocks, bh, qb);
                // Q buffer it % QBUF, used for the (it / QBUF)-th time
                const int qt0 = 2 * (it % C::QBUF), use = it / C::QBUF;
                for (int h = 0; ok && h < 2; ++h) {
                    // Q_h of the item that last used this buffer: every product
                    // that read it is done
                    if (use > 0 && !(ok = wait_bounded(bar(C::B_QEMPTY + qt0 + h), (use - 1) & 1, abort_flag)))
                        break;
                    mbar_arrive_expect_tx(bar(C::B_QFULL + qt0 + h), C::TILE);
                    for (int b = 0; b < col_blocks<D>(); ++b)
                        tma_load_3d(sbase + C::Q_OFF + (qt0 + h) * C::TILE + b * kSwAtomBytes, &tm_q,
                                    bar(C::B_QFULL + qt0 + h), b * 64, qb * kBM + (h ^ swap_of(it)) * kSubM, bh,
                                    pol_q);
                }
                if (!ok)
                    break;
                ++items;
                const int nloads = 2 * nk_sub(qb, 1);  // K_j = load 2j, V_j = load 2j + 1
                for (int Ll = 0; Ll < nloads; ++Ll, ++L) {
                    const int s = L % SLOTS;
                    FA_CHECK(s >= 0 && s < SLOTS && qt0 + 1 < 2 * C::QBUF);
                    if (L >= SLOTS && !(ok = wait_bounded(bar(C::B_KVEMPTY + s), ((L / SLOTS) - 1) & 1, abort_flag)))
                        break;
                    const CUtensorMap *map = (Ll & 1) ? &tm_v : &tm_k;
                    mbar_arrive_expect_tx(bar(C::B_KVFULL + s), C::TILE);
                    for (int b = 0; b < col_blocks<D>(); ++b)
                        tma_load_3d(sbase + C::KV_OFF + s * C::TILE + b * kSwAtomBytes, map,
                                    bar(C::B_KVFULL + s), b * 64, (Ll >> 1) * kBN, bh, pol_kv);
                }
            }
            // Wait for every copy this thread issued (immediate on the normal
            // path, where each one was consumed).
            for (int q = 0; q < 2 * C::QBUF; ++q) {
                const int b = q / 2;                                 // buffer of Q tile q
                const int uses = (items - b + C::QBUF - 1) / C::QBUF;  // items that loaded it
                if (items > b)
                    drain_bounded(bar(C::B_QFULL + q), (uses - 1) & 1);
            }
            for (int s = 0; s < SLOTS; ++s)
                if (L > s)
                    drain_bounded(bar(C::B_KVFULL + s), ((L - 1 - s) / SLOTS) & 1);
      } else if (lane == 0 && (warp == kMmaWarp || (NUM_ISSUERS == 2 && warp == kMmaWarp + 2))) {
            // ---------------- MMA issuer(s) ----------------
            // A thread that issues tcgen05.mma is held for about the product's
            // execution time, so its own barrier waits leave the tensor core
            // idle.  With D = 64 (short products, early-S order) each sub-tile
            // gets its own issuer (warps 8 and 10), so one issues while the
            // other waits.  With D = 128 one issuer serves both sub-tiles in a
            // fixed ping-pong order, which keeps each sub-tile's products
            // together, and releases every K/V load once (after its products
            // read it).  With D = 64 the softmax warpgroups release them.
            const int me = (warp == kMmaWarp) ? 0 : 1;
            const int h_lo = NUM_ISSUERS == 2 ? me : 0;
            const int h_hi = NUM_ISSUERS == 2 ? me + 1 : 2;
            constexpr uint32_t idesc_s = make_idesc_f16(DTypeTraits<T>::kBF16, kSubM, kBN, false, false);
            constexpr uint32_t idesc_o = make_idesc_f16(DTypeTraits<T>::kBF16, kSubM, D, false, true);
            auto slot_of = [](int L) {
                FA_CHECK(L >= 0);
                return L % SLOTS;
            };
            auto par_of = [](int L) { return static_cast<uint32_t>((L / SLOTS) & 1); };
            // Descriptors of the ring's first tile and of Q0: a tile at byte
            // offset x from them is the same descriptor plus x >> 4 (the start
            // address field; shared addresses stay below 256 KiB, no carry).
            const uint64_t desc_k0 = make_sdesc_sw128(sbase + C::KV_OFF, 16, 1024);
            const uint64_t desc_v0 = make_sdesc_sw128(sbase + C::KV_OFF, kSwAtomBytes, 1024);
            const uint64_t desc_q0 = make_sdesc_sw128(sbase + C::Q_OFF, 16, 1024);
            int Lb = 0;              // ring index of the current item's K_0
            int qt0 = 0;             // Q tile of the current item's sub-tile 0
            // key tiles of sub-tile 0 / 1 in earlier items (scalars, not an
            // array: a runtime-indexed array would live in local memory)
            int done0 = 0, done1 = 0;
            auto issue_s = [&](int h, int j) {
                const uint64_t kd = desc_k0 + static_cast<uint32_t>((slot_of(Lb + 2 * j) * C::TILE) >> 4);
                const uint64_t qd = desc_q0 + static_cast<uint32_t>(((qt0 + h) * C::TILE) >> 4);
#pragma unroll
                for (int kk = 0; kk < KSTEPS_QK; ++kk) {
                    const uint32_t koff = static_cast<uint32_t>(((kk >> 2) * kSwAtomBytes + (kk & 3) * 32) >> 4);
                    umma_f16_ss(tmem + h * kBN, qd + koff, kd + koff, idesc_s, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int h, int j) {
                const uint64_t vd = desc_v0 + static_cast<uint32_t>((slot_of(Lb + 2 * j + 1) * C::TILE) >> 4);
                const uint32_t d_o = tmem + kTmemO + h * D;
#pragma unroll
                for (int kk = 0; kk < KSTEPS_PV; ++kk) {
                    // V: MN-major; 16 key rows (2048 B) per K step; the two
                    // 64-column blocks of D = 128 are kSwAtomBytes apart.
                    // P_h,j: 16-bit in TMEM, two per column; 8 columns per K step.
                    umma_f16_ts(d_o, tmem + tmem_p_col<D>(h) + kk * 8,
                                vd + static_cast<uint32_t>((kk * 2048) >> 4), idesc_o,
                                (j > 0 || kk > 0) ? 1u : 0u);
                }
            };
            auto wait_load = [&](int l) {
                return wait_bounded(bar(C::B_KVFULL + slot_of(Lb + l)), par_of(Lb + l), abort_flag);
            };
            // Releases load l of this item: after this issuer's products that
            // read it (commit), or, when none did, as soon as it has landed.
            auto release = [&](int l, bool used) -> bool {
                if (used) {
                    umma_commit(bar(C::B_KVEMPTY + slot_of(Lb + l)));
                    return true;
                }
                if (!wait_load(l))
                    return false;
                mbar_arrive(bar(C::B_KVEMPTY + slot_of(Lb + l)));
                return true;
            };
            // the first P V product of an item overwrites O_h: the previous
            // item's epilogue must have read it
            auto o_free = [&](int h, int it) {
                return it == 0 || wait_bounded(bar(C::B_OFREE + h), (it - 1) & 1, abort_flag);
            };
            bool ok = true;
            for (int it = 0; ok; ++it) {
                const int w = item_of<CAUSAL>(it);
                if (w >= num_items)
                    break;
                int bh, qb;
                item_coords<CAUSAL>(w, BH, num_q_blocks, bh, qb);
                (void)bh;
                // key tiles of sub-tile 0 / 1, and of the longer one (the loads)
                const int nk0 = nk_sub(qb, swap_of(it)), nk1 = nk_sub(qb, 1 ^ swap_of(it));
                const int nkmax = nk_sub(qb, 1);
                auto nk_of = [&](int h) { return h == 0 ? nk0 : nk1; };
                auto done_of = [&](int h) { return h == 0 ? done0 : done1; };
                qt0 = 2 * (it % C::QBUF);
                for (int h = h_lo; ok && h < h_hi; ++h) {
                    ok = wait_bounded(bar(C::B_QFULL + qt0 + h), (it / C::QBUF) & 1, abort_flag);
                    // early-S: S_h,0 overwrites S_h, which the previous item's
                    // last softmax step must have finished reading
                    if (ok && EARLY_S && it > 0)
                        ok = wait_bounded(bar(C::B_SFREE + h), (done_of(h) - 1) & 1, abort_flag);
                }
                ok = ok && wait_load(0);
                if (!ok)
                    break;
                tc_fence_after();
                for (int h = h_lo; h < h_hi; ++h) {
                    issue_s(h, 0);
                    umma_commit(bar(C::B_SFULL + h));
                }
                if constexpr (!EARLY_S)
                    release(0, true);
                for (int j = 0; ok && j < nkmax; ++j) {
                    if constexpr (EARLY_S) {
                        // next S products first, then this tile's P V products
                        for (int h = h_lo; ok && h < h_hi; ++h) {
                            if (j + 1 >= nk_of(h))
                                continue;
                            ok = wait_bounded(bar(C::B_SFREE + h), (done_of(h) + j) & 1, abort_flag) &&
                                 wait_load(2 * j + 2);
                            if (!ok)
                                break;
                            tc_fence_after();
                            issue_s(h, j + 1);
                            umma_commit(bar(C::B_SFULL + h));
                        }
                        for (int h = h_lo; ok && h < h_hi; ++h) {
                            if (j >= nk_of(h))
                                continue;
                            ok = wait_load(2 * j + 1) &&
                                 wait_bounded(bar(C::B_PFULL + h), (done_of(h) + j) & 1, abort_flag) &&
                                 (j > 0 || o_free(h, it));
                            if (!ok)
                                break;
                            tc_fence_after();
                            issue_pv(h, j);
                            umma_commit(bar(C::B_OREADY + h));
                            if (j + 1 == nk_of(h))
                                umma_commit(bar(C::B_OFINAL + h));
                        }
                    } else {
                        // per sub-tile: P V of this tile, then the next S product
                        bool v_used = false, k_used = false;
                        for (int h = h_lo; ok && h < h_hi; ++h) {
                            if (j >= nk_of(h))
                                continue;
                            ok = (v_used || wait_load(2 * j + 1)) &&
                                 wait_bounded(bar(C::B_PFULL + h), (done_of(h) + j) & 1, abort_flag) &&
                                 (j > 0 || o_free(h, it));
                            if (!ok)
                                break;
                            tc_fence_after();
                            issue_pv(h, j);
                            v_used = true;
                            if (j + 1 < nk_of(h)) {
                                ok = k_used || wait_load(2 * j + 2);
                                if (!ok)
                                    break;
                                tc_fence_after();
                                issue_s(h, j + 1);
                                umma_commit(bar(C::B_SFULL + h));
                                k_used = true;
                            } else {
                                umma_commit(bar(C::B_OFINAL + h));
                            }
                        }
                        if (ok)
                            ok = release(2 * j + 1, v_used);
                        if (ok && j + 1 < nkmax)
                            ok = release(2 * j + 2, k_used);
                    }
                }
                if (!ok)
                    break;
                // every product reading Q_h of this item has been issued
                for (int h = h_lo; h < h_hi; ++h)
                    umma_commit(bar(C::B_QEMPTY + qt0 + h));
                done0 += nk0;
                done1 += nk1;
                Lb += 2 * nkmax;
            }
            // every MMA this thread issued has completed once this arrives
            umma_commit(bar(C::B_DRAIN + me));
            drain_bounded(bar(C::B_DRAIN + me), 0);
      }
    } else {
        reg_alloc<((D <= 64 && !CAUSAL) ? kRegsSoftmax : kRegsSoftmaxWide)>();
        // ---------------- softmax warpgroup h (warps 4h .. 4h+3) ----------------
        const int h = warp >> 2;
        const int r = threadIdx.x & 127;  // row within the sub-tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t s_tm = tmem + lane_base + static_cast<uint32_t>(h * kBN);
        const uint32_t o_tm = tmem + lane_base + kTmemO + static_cast<uint32_t>(h * D);
        const uint32_t p_tm = tmem + lane_base + tmem_p_col<D>(h);
        const uint32_t stage = sbase + C::OST_OFF + h * C::TILE;
        int done = 0;  // key tiles of this sub-tile in earlier items
        int Lr = 0;    // ring index of the current item's K_0
        // Early-S order: one thread per warpgroup frees the K/V ring slots
        // (both warpgroups must have freed a slot before it is loaded again).
        const bool rel = EARLY_S && r == 0;
        auto kv_free = [&](int l) {
            if (rel)
                mbar_arrive(bar(C::B_KVEMPTY + (Lr + l) % SLOTS));
        };
        for (int it = 0;; ++it) {
            const int w = item_of<CAUSAL>(it);
            if (w >= num_items)
                break;
            int bh, qb;
            item_coords<CAUSAL>(w, BH, num_q_blocks, bh, qb);
            const int row0 = qb * kBM + (h ^ swap_of(it)) * kSubM;
            const int qrow = row0 + r;
            const int nkh = nk_sub(qb, h ^ swap_of(it));
            float m_ref = -INFINITY;  // reference max (raw score units; scale >= 0)
            float l = 0.f;
            bool ok = true;
            for (int j = 0; j < nkh; ++j) {
                const uint32_t ph = static_cast<uint32_t>((done + j) & 1);
                ok = wait_warp(bar(C::B_SFULL + h), ph, abort_flag);
                if (!ok)
                    break;
                kv_free(2 * j);  // S_h,j has read K_j
                tc_fence_after();
                float s[kBN];
                tmem_ld128(s_tm, s);
                // keys [kbase, kbase + limit) are allowed for this row (limit >= 1)
                const int kbase = j * kBN;
                int limit = min(kBN, N - kbase);
                if (CAUSAL)
                    limit = min(limit, qrow - kbase + 1);
                const bool masked = __any_sync(0xffffffffu, limit < kBN);
                if (masked)
                    mask_tail(s, limit);
                // Tile 0 sets the reference max from its own row max; the reference
                // moves only when a row max outgrows it by more than kRescaleLog2
                // (rare).  D <= 64 takes the row max before the exponentials; D >
                // 64 exponentiates against the current reference while the row max
                // is taken, and redoes the tile from S when the reference moves.
                float alpha = 1.f;
                float rsum;
                uint32_t pw[64];  // P_h,j rounded to the input dtype, two per word
                if constexpr (EARLY_S) {
                    // S_h,j is in registers: let the next S_h product in now, so
                    // that it runs during this tile's exponentials.
                    tc_fence_before();
                    mbar_arrive(bar(C::B_SFREE + h));
                    if (CAUSAL || j == 0) {
                        // causal: the row max first (its launch keeps the
                        // smaller register budget, which the check's second
                        // copy of the tile would exceed)
                        const float mt = row_max(s);
                        if (j == 0) {
                            m_ref = mt;
                            alpha = 0.f;
                        } else {
                            const bool grow = (mt - m_ref) * scale_log2 > kRescaleLog2;
                            if (__any_sync(0xffffffffu, grow) && grow) {
                                alpha = ex2_approx((m_ref - mt) * scale_log2);
                                m_ref = mt;
                            }
                        }
                        rsum = masked ? exp_pack_tile<true, T>(s, pw, limit, scale_log2, -m_ref * scale_log2)
                                      : exp_pack_tile<false, T>(s, pw, limit, scale_log2, -m_ref * scale_log2);
                    } else {
                        // Against the current reference first.  The reference
                        // must move only if some p exceeds 2^kRescaleLog2, and
                        // the largest p is at most the row sum, so the row max
                        // is needed only when the sum exceeds that bound (or is
                        // not finite); the tile is then redone from the scores,
                        // which are still in registers.  Same results as taking
                        // the row max first.
                        rsum = masked ? exp_pack_tile<true, T>(s, pw, limit, scale_log2, -m_ref * scale_log2)
                                      : exp_pack_tile<false, T>(s, pw, limit, scale_log2, -m_ref * scale_log2);
                        const bool check = !(rsum <= kRescaleBound);
                        if (__any_sync(0xffffffffu, check)) {
                            const float mt = row_max(s);
                            const bool grow = (mt - m_ref) * scale_log2 > kRescaleLog2;
                            if (__any_sync(0xffffffffu, grow)) {
                                if (grow) {
                                    alpha = ex2_approx((m_ref - mt) * scale_log2);
                                    m_ref = mt;
                                }
                                rsum = masked
                                           ? exp_pack_tile<true, T>(s, pw, limit, scale_log2, -m_ref * scale_log2)
                                           : exp_pack_tile<false, T>(s, pw, limit, scale_log2, -m_ref * scale_log2);
                            }
                        }
                    }
                } else if (j == 0) {
                    m_ref = row_max(s);
                    alpha = 0.f;
                    rsum = masked ? exp_tile<true>(s, limit, scale_log2, -m_ref * scale_log2)
                                  : exp_tile<false>(s, limit, scale_log2, -m_ref * scale_log2);
                } else {
                    const float mt = row_max(s);
                    rsum = masked ? exp_tile<true>(s, limit, scale_log2, -m_ref * scale_log2)
                                  : exp_tile<false>(s, limit, scale_log2, -m_ref * scale_log2);
                    const bool grow = (mt - m_ref) * scale_log2 > kRescaleLog2;
                    if (__any_sync(0xffffffffu, grow)) {
                        if (grow) {
                            alpha = ex2_approx((m_ref - mt) * scale_log2);
                            m_ref = mt;
                        }
                        // S_h is intact until P_h is written below: redo the tile
                        tmem_ld128(s_tm, s);
                        if (masked)
                            mask_tail(s, limit);
                        rsum = masked ? exp_tile<true>(s, limit, scale_log2, -m_ref * scale_log2)
                                      : exp_tile<false>(s, limit, scale_log2, -m_ref * scale_log2);
                    }
                }
                l = l * alpha + rsum;
                if constexpr (EARLY_S) {
                    // P_h,j-1 V_{j-1} must have read P_h before it is overwritten
                    // (and O_h must be complete before a rescale below).  For
                    // j = 0 the previous item's last product has completed: this
                    // warpgroup waited for it before its epilogue.
                    if (j > 0) {
                        ok = wait_warp(bar(C::B_OREADY + h), ph ^ 1u, abort_flag);
                        if (!ok)
                            break;
                        kv_free(2 * j - 1);  // P_h,j-1 V_j-1 has read V_j-1
                        tc_fence_after();
                    }
                }
                // P_h,j rounded to the input dtype (early-S order: done above)
                if constexpr (!EARLY_S) {
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        pw[c] = DTypeTraits<T>::pack(s[2 * c], s[2 * c + 1]);
                }
                tmem_st64(p_tm, pw);
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    // O_h must hold P V up to tile j-1, and P_h,j V_j is not issued
                    // before this warpgroup arrives below.  In the early-S order
                    // that product was awaited above; in the other order the S_h,j
                    // product, issued after it, has completed.
#pragma unroll
                    for (int c4 = 0; c4 < D / 32; ++c4) {
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
            // The named barriers below are reached by all four warps, whatever
            // happened; their OR-reductions give every warp the same decision.
            if constexpr (!C::STAGE_IN_Q) {
                // the previous item's tensor store has read the staging tile
                // (waited for here, an item later, rather than right after it)
                if (r == 0)
                    bulk_wait_group_read<0>();
                named_bar_sync(1 + h, 4 * 32);
            }
            if (ok) {
                ok = wait_warp(bar(C::B_OFINAL + h), it & 1, abort_flag);
            }
            if (ok) {
                tc_fence_after();
                if (rel) {
                    kv_free(2 * nkh - 1);  // the last P V product has read V
                    // key tiles this sub-tile skips (causal, the upper row
                    // half): freed once they have landed (so that no slot is
                    // freed early)
                    const int nk1 = nk_sub(qb, 1);
                    for (int ll = 2 * nkh; ok && ll < 2 * nk1; ++ll) {
                        const int L = Lr + ll;
                        ok = wait_bounded(bar(C::B_KVFULL + L % SLOTS), static_cast<uint32_t>((L / SLOTS) & 1),
                                          abort_flag);
                        if (ok)
                            kv_free(ll);
                    }
                }
                const float inv_l = 1.f / l;
#pragma unroll
                for (int c4 = 0; c4 < D / 32; ++c4) {
                    uint32_t u[32];
                    tmem_ld32(o_tm + c4 * 32, u);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const float *f = reinterpret_cast<const float *>(u) + q4 * 8;
                        st_shared_v4(stage + sw128_offset(r, c4 * 4 + q4),
                                     DTypeTraits<T>::pack(f[0] * inv_l, f[1] * inv_l),
                                     DTypeTraits<T>::pack(f[2] * inv_l, f[3] * inv_l),
                                     DTypeTraits<T>::pack(f[4] * inv_l, f[5] * inv_l),
                                     DTypeTraits<T>::pack(f[6] * inv_l, f[7] * inv_l));
                    }
                }
                // the staged tile goes out through the TMA engine (async proxy)
                fence_proxy_async_smem();
                // O_h has been read: the next item's first P V product may overwrite it
                tc_fence_before();
                mbar_arrive(bar(C::B_OFREE + h));
                if (lse != nullptr && qrow < N)
                    lse[static_cast<size_t>(bh) * N + qrow] = m_ref * scale + logf(l);
            }
            const bool bad = named_bar_or(1 + h, 4 * 32, !ok || *abort_flag != 0);
            if constexpr (!C::STAGE_IN_Q) {
                // one tensor store per 64-column block; rows past N and columns
                // past D lie outside the tensor and are not written
                if (r == 0 && !bad) {
                    for (int b = 0; b < col_blocks<D>(); ++b)
                        tma_store_3d(&tm_o, stage + b * kSwAtomBytes, b * 64, row0, bh);
                    bulk_commit_group();
                }
            } else {
                // O staged in Q_h: the warpgroup copies it out itself (16-byte
                // coalesced stores), which frees Q_h for the next item's Q
                // sooner than a tensor store that one thread waits for
                if (!bad) {
                    constexpr int CHUNKS_PER_ROW = D / 8;
                    uint8_t *obase = reinterpret_cast<uint8_t *>(out) +
                                     (static_cast<size_t>(bh) * N + row0) * D * sizeof(T);
#pragma unroll 4
                    for (int idx = r; idx < kSubM * CHUNKS_PER_ROW; idx += 4 * 32) {
                        const int row = idx / CHUNKS_PER_ROW;
                        const int ch = idx % CHUNKS_PER_ROW;
                        const uint4 val = ld_shared_v4(stage + sw128_offset(row, ch));
                        if (row0 + row < N)
                            *reinterpret_cast<uint4 *>(obase + (static_cast<size_t>(row) * D + ch * 8) *
                                                                   sizeof(T)) = val;
                    }
                }
                mbar_arrive(bar(C::B_QEMPTY + h));  // the next item's Q_h may land
            }
            // stop together if anything failed (D > 64: the copy-out has read
            // the staging tile, which the next item's Q may now overwrite)
            if (named_bar_or(1 + h, 4 * 32, bad || *abort_flag != 0))
                break;
            done += nkh;
            Lr += 2 * nk_sub(qb, 1);
        }
        if constexpr (!C::STAGE_IN_Q) {
            if (r == 0)
                bulk_wait_group<0>();  // the last tensor store is complete
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

// Failure-path self-test: one warp waits on an mbarrier that nothing ever
// arrives on.  The bounded wait must give up after limit_cycles, set the CTA
// abort flag and record kStatusTimeout in the device status word.
__global__ void fa_selftest_wait_kernel(long long limit_cycles)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const bool ok = wait_bounded(smem_u32(&bar), 0, &abort_flag, limit_cycles);
        if (ok || abort_flag != 1)
            atomicOr(&g_fa_status, kStatusSelftest);  // the wait did not behave as required
    }
}

// Self-test of the checked build's address checks: asks them about
// addresses just inside and just outside the shared window (1 KB of dynamic
// shared memory) and the tensor-memory columns, performing no access.  The
// outside ones record kStatusBounds; an inside one that fails, or an outside
// one that passes, records kStatusSelftest.
__global__ void fa_selftest_bounds_kernel()
{
    extern __shared__ uint8_t smem_raw[];
    if (threadIdx.x != 32)  // warp 1: lane quarter 32..63
        return;
    const uint32_t base = smem_u32(smem_raw);
    const uint32_t end = smem_window_end();
    bool good = smem_ok<true>(base, 1024, 16) && smem_ok<true>(end - 16, 16, 16) &&
                tmem_ok<true>((32u << 16) | 480u, 32, true) && tmem_ok<true>(384u, 128, false);
    good = good && !smem_ok<true>(end - 8, 16, 8);           // runs past the window
    good = good && !smem_ok<true>(base + 4, 16, 16);         // misaligned
    good = good && !tmem_ok<true>((32u << 16) | 496u, 32, true);  // past column 511
    good = good && !tmem_ok<true>(480u, 32, true);           // another warp's lanes
    if (!good)
        atomicOr(&g_fa_status, kStatusSelftest);
}

}  // namespace fa
