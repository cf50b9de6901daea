// fa_bwd_kernel.cuh -- the sm_103a attention-backward kernels.
//
// What they compute: for one head with S = scale Q K^T (causal: key j > query
// i masked), P = softmax(S) row by row, O = P V, and an upstream gradient dO,
//   dV = P^T dO
//   dP = dO V^T
//   dS = P o (dP - D),  D_i = sum_c dO_ic O_ic  (= sum_j P_ij dP_ij)
//   dQ = scale dS K,   dK = scale dS^T Q.
// "3.6 어텐션 I — 메모리 문제·FlashAttention 원리", section 3.6.7: the backward
// pass does not read a stored S or P; it recomputes them block by block from
// Q, K and the row statistic L = m + log l that the forward pass saved
// (P_ij = exp(S_ij - L_i)).
//
// Three launches:
//   fa_bwd_prep_kernel  D_i and L_i * log2(e) into a padded per-head layout,
//                       and zeroes the fp32 dQ accumulator.
//   fa_bwd_kernel       persistent, one CTA per SM; a work item is one
//                       (batch*head, 128-key block n): K_n and V_n stay in
//                       shared memory while the CTA walks the query blocks m
//                       (all of them, or m >= n when causal) and keeps dK_n
//                       and dV_n in TMEM for the whole walk.  The next item's
//                       K, V and first Q, dO loads overlap the epilogue that
//                       writes dK_n and dV_n.  Per query block:
//                         S^T  = K_n Q_m^T           (tcgen05, TMEM)
//                         dP^T = V_n dO_m^T          (tcgen05, TMEM)
//                         P^T  = 2^(S^T scale log2e - L_m log2e)   (warps 0-7)
//                         dS^T = P^T o (dP^T - D_m)                (warps 0-7)
//                         dV_n += P^T dO_m           (P^T read from TMEM)
//                         dK_n += dS^T Q_m           (dS^T read from TMEM)
//                         dQ_m  = dS K_n             (dS^T also in shared memory,
//                                                     read as an MN-major operand)
//                       (the factor scale of dK and dQ is applied once, when
//                       dK_n is written and when dQ is rounded);
//                       and warps 8-11 add dQ_m into the fp32 accumulator with
//                       TMA reduce-add (other key blocks add to the same rows).
//   fa_bwd_dq_kernel    rounds the fp32 accumulator to dQ in the input dtype.
//
// Warp roles in fa_bwd_kernel (512 threads):
//   warps 0-3, 4-7  compute warpgroups c = 0, 1: thread r owns key row r (TMEM
//                   lane r) for query columns [64c, 64c + 64) of the block.
//   warps 8-11      dQ warpgroup: thread r owns query row r of dQ_m.
//   warp 12         TMA producer; warp 13 MMA issuer (one thread).
// Every mbarrier wait is bounded, as in the forward kernel.
#pragma once

#include "fa_common.cuh"

namespace fa {
namespace bwd {

constexpr int kBlk = 128;  // keys per CTA, queries per step
constexpr int kThreads = 512;
constexpr int kDqWarp0 = 8;
constexpr int kTmaWarp = 12;
constexpr int kMmaWarp = 13;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S^T @ 0 (P^T, 16-bit, over its first columns), dP^T @ 128,
// dV @ 256, dK @ 256 + D.  D <= 64: dQ @ 256 + 2D and dS^T (16-bit) @ 448, so
// that dP^T of the next query block can be computed while dK and dQ of this
// one still read dS^T.  D > 64 (no spare columns): dS^T over the first dP^T
// columns and dQ_m over all of them, which the compute warps have finished
// reading when dK and dQ_m are issued; the next dP^T waits for dQ_m to be read.
// Head dims 32 and 96 use tiles of whole 64-column swizzle blocks (TMA fills
// the columns past D with zeros), as the forward kernel does.
constexpr uint32_t kTmS = 0;
constexpr uint32_t kTmDP = 128;
constexpr uint32_t kTmDV = 256;
template <int D>
__host__ __device__ constexpr uint32_t col_dk()
{
    return 256u + D;
}
template <int D>
__host__ __device__ constexpr uint32_t col_dq()
{
    return D <= 64 ? 256u + 2u * D : kTmDP;
}
template <int D>
__host__ __device__ constexpr uint32_t col_ds()
{
    return D <= 64 ? 448u : kTmDP;
}
template <int D>
__host__ __device__ constexpr int col_blocks()
{
    return (D + 63) / 64;
}
// Column distance between the two compute warpgroups' halves of a 16-bit
// P^T / dS^T tile (each half: 64 queries, two per column = 32 columns).  Over
// a 128-column fp32 source (P^T over S^T; dS^T over dP^T for D = 128) each
// half sits on the source columns of its own queries: 64 apart.  In the
// dedicated 64-column dS^T area of D = 64 the halves are adjacent: 32 apart.
template <int D>
__host__ __device__ constexpr uint32_t ds_half()
{
    return D <= 64 ? 32u : 64u;
}
static_assert(448u + 2 * 32u <= kTmemCols && 128u + 64u + 32u <= 256u, "dS^T columns inside their area");
// TMEM column, relative to the start of the P^T or dS^T area, of K step t
// (queries 16t .. 16t + 15) of those 16-bit tiles, whose warpgroup halves are
// `half` columns apart: compute warpgroup c writes the values of its queries
// [64c, 64c + 64) to columns [half c, half c + 32).
__host__ __device__ constexpr uint32_t tm_p_step(int t, uint32_t half)
{
    return half * (t >> 2) + 8u * (t & 3);
}

template <int D>
struct Cfg {
    static_assert(D == 32 || D == 64 || D == 96 || D == 128, "head dims 32, 64, 96, 128");
    static constexpr int TILE = kBlk * col_blocks<D>() * 128;  // one [128, D] 16-bit tile
    // D <= 64 (CONT): two K/V buffers, so the next item's first S^T and dP^T
    // products follow this item's last dV product like any other block's, and
    // the dQ warpgroup writes dK_n, dV_n while the compute warps go on.
    // D > 64: one K/V buffer (no room for two), reloaded once the item's
    // products are done; the compute warps write dK_n, dV_n.
    static constexpr bool CONT = D <= 64;
    static constexpr int KVBUF = CONT ? 2 : 1;
    static constexpr int QST = D <= 64 ? 3 : 2;   // Q (+ L) ring
    static constexpr int DOST = D <= 64 ? 2 : 1;  // dO (+ D) ring
    // dQ goes to the fp32 accumulator in chunks of DQ_COLS columns through two
    // staging buffers, so that one reduce-add can read its buffer while the
    // next chunk is staged: [128 rows x 32 fp32] 128B-swizzled (D <= 64, where
    // the buffers also carry dV_n, dK_n), [128 rows x 16 fp32] 64B-swizzled
    // (D > 64, where shared memory has room for 16 KB of staging only).
    static constexpr int NSTG = 2;
    static constexpr int DQ_COLS = D <= 64 ? 32 : 16;
    static constexpr int STG_BYTES = kBlk * DQ_COLS * 4;
    static constexpr bool DQ_ALIAS = D > 64;  // dQ (and dS^T) over the dP^T columns
    static constexpr int KV_OFF = 0;  // buffer b: K at 2 b TILE, V at (2 b + 1) TILE
    static constexpr int Q_OFF = KV_OFF + 2 * KVBUF * TILE;
    static constexpr int DO_OFF = Q_OFF + QST * TILE;
    static constexpr int DS_OFF = DO_OFF + DOST * TILE;  // dS^T [128 keys x 128 queries]
    static constexpr int STG_OFF = DS_OFF + kBlk * kBlk * 2;
    static constexpr int L_OFF = STG_OFF + NSTG * STG_BYTES;  // QST x 128 fp32
    static constexpr int DD_OFF = L_OFF + QST * kBlk * 4;      // DOST x 128 fp32
    static constexpr int BAR_OFF = DD_OFF + DOST * kBlk * 4;
    static constexpr int B_KVFULL = 0;
    static constexpr int B_KVEMPTY = B_KVFULL + KVBUF;
    static constexpr int B_QFULL = B_KVEMPTY + KVBUF;
    static constexpr int B_QEMPTY = B_QFULL + QST;
    static constexpr int B_DOFULL = B_QEMPTY + QST;
    static constexpr int B_DOEMPTY = B_DOFULL + DOST;
    static constexpr int B_SFULL = B_DOEMPTY + DOST;
    static constexpr int B_DPFULL = B_SFULL + 1;
    static constexpr int B_PFULL = B_DPFULL + 1;
    static constexpr int B_DSFULL = B_PFULL + 1;
    static constexpr int B_DQFULL = B_DSFULL + 1;
    static constexpr int B_DQFREE = B_DQFULL + 1;
    static constexpr int B_DKVFULL = B_DQFREE + 1;
    static constexpr int B_DKVFREE = B_DKVFULL + 1;  // CONT: dK_n, dV_n read out of TMEM
    static constexpr int B_DRAIN = B_DKVFREE + 1;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr int SLOT_OFF = BAR_OFF + 8 * NUM_BARS;  // TMEM base address, abort flag
    static constexpr int SMEM_USED = SLOT_OFF + 16;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
    static_assert(DS_OFF % 1024 == 0 && STG_OFF % 1024 == 0, "swizzled tiles need 1024-byte alignment");
    static_assert(!CONT || (NSTG == 2 && STG_BYTES == kBlk * 128), "dV_n, dK_n staged in the two dQ buffers");
    static_assert(32 % DQ_COLS == 0, "a 32-column TMEM load covers whole chunks");
};

// Work item number w: (head bh, key block n).  Causal: the heads go in
// groups of hg (the last group may be smaller); inside a group the heaviest
// key blocks (low n, which see the most query blocks) of every head come
// first, so that the CTAs running at one time share the Q, dO and dQ
// accumulator of a few heads in L2.  Non-causal: head-major, for the same
// reason.
template <bool CAUSAL>
__device__ __forceinline__ void item_coords(int w, int BH, int nb, int hg, int &bh, int &n)
{
    if (CAUSAL) {
        const int g = w / (hg * nb);
        const int h0 = g * hg;
        const int gs = min(hg, BH - h0);  // heads in this group
        const int r = w - h0 * nb;
        n = r / gs;
        bh = h0 + r % gs;
    } else {
        bh = w / nb;
        n = w % nb;
    }
}

// Item k of this CTA (the kernel is persistent: gridDim.x CTAs, at most one
// per SM).  Round k deals items [k G, k G + G) out to the G CTAs, every other
// round in reverse CTA order, so that the heavy and light causal items of
// consecutive rounds even out per CTA.  False past the last item.
template <bool CAUSAL>
__device__ __forceinline__ bool item_of(int k, int BH, int nb, int hg, int &bh, int &n)
{
    // (the host keeps BH * nb + gridDim.x within int range)
    const int G = static_cast<int>(gridDim.x);
    const int cta = static_cast<int>(blockIdx.x);
    const int w = k * G + ((k & 1) ? G - 1 - cta : cta);
    if (w >= BH * nb)
        return false;
    item_coords<CAUSAL>(w, BH, nb, hg, bh, n);
    return true;
}

template <int D, bool CAUSAL, typename T>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                  const __grid_constant__ CUtensorMap tm_dqacc, const float *__restrict__ lse2,
                  const float *__restrict__ dvec, int N, int Npad, int BH, int nb, int hg, float scale,
                  float scale_log2)
{
    using C = Cfg<D>;
    constexpr bool CONT = C::CONT;
    constexpr int KVBUF = C::KVBUF;
    constexpr int QST = C::QST;
    constexpr int DOST = C::DOST;
    constexpr int NSTG = C::NSTG;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Every role walks the same item sequence; g counts the query blocks of
    // all earlier items (the ring slots and barrier phases run on across items).
    int bh = 0, n = 0;

    auto bar = [&](int idx) -> uint32_t {
        FA_CHECK(idx >= 0 && idx < C::NUM_BARS);
        return sbase + C::BAR_OFF + 8u * idx;
    };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + C::SLOT_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::SLOT_OFF + 4);

    if (threadIdx.x == 0) {
        for (int b = 0; b < KVBUF; ++b) {
            mbar_init(bar(C::B_KVFULL + b), 1);
            mbar_init(bar(C::B_KVEMPTY + b), 1);
        }
        for (int s = 0; s < QST; ++s) {
            mbar_init(bar(C::B_QFULL + s), 1);
            mbar_init(bar(C::B_QEMPTY + s), 1);
        }
        for (int s = 0; s < DOST; ++s) {
            mbar_init(bar(C::B_DOFULL + s), 1);
            mbar_init(bar(C::B_DOEMPTY + s), 1);
        }
        mbar_init(bar(C::B_SFULL), 1);
        mbar_init(bar(C::B_DPFULL), 1);
        mbar_init(bar(C::B_PFULL), 2 * 128);
        mbar_init(bar(C::B_DSFULL), 2 * 128);
        mbar_init(bar(C::B_DQFULL), 1);
        mbar_init(bar(C::B_DQFREE), 128);
        mbar_init(bar(C::B_DKVFULL), 1);
        mbar_init(bar(C::B_DKVFREE), 128);
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
            tma_prefetch_desc(&tm_do);
            // K_n, V_n are read by this CTA only; Q_m, dO_m by every key block
            // of the head.
            const uint64_t pol_kv = l2_policy_evict_first();
            const uint64_t pol_q = l2_policy_evict_last();
            int nq = 0, ndo = 0, nkv = 0;
            // Q_m (+ L_m) and dO_m (+ D_m) of global query block nq into their ring slots
            auto load_block = [&](int m) -> bool {
                const size_t row0 = static_cast<size_t>(bh) * Npad + static_cast<size_t>(m) * kBlk;
                const int s = nq % QST;
                if (nq >= QST && !wait_bounded(bar(C::B_QEMPTY + s), ((nq / QST) - 1) & 1, abort_flag))
                    return false;
                mbar_arrive_expect_tx(bar(C::B_QFULL + s), C::TILE + kBlk * 4);
                for (int b = 0; b < col_blocks<D>(); ++b)
                    tma_load_3d(sbase + C::Q_OFF + s * C::TILE + b * kSwAtomBytes, &tm_q, bar(C::B_QFULL + s),
                                b * 64, m * kBlk, bh, pol_q);
                bulk_load(sbase + C::L_OFF + s * kBlk * 4, lse2 + row0, kBlk * 4, bar(C::B_QFULL + s));
                ++nq;
                const int ds = ndo % DOST;
                if (ndo >= DOST && !wait_bounded(bar(C::B_DOEMPTY + ds), ((ndo / DOST) - 1) & 1, abort_flag))
                    return false;
                mbar_arrive_expect_tx(bar(C::B_DOFULL + ds), C::TILE + kBlk * 4);
                for (int b = 0; b < col_blocks<D>(); ++b)
                    tma_load_3d(sbase + C::DO_OFF + ds * C::TILE + b * kSwAtomBytes, &tm_do,
                                bar(C::B_DOFULL + ds), b * 64, m * kBlk, bh, pol_q);
                bulk_load(sbase + C::DD_OFF + ds * kBlk * 4, dvec + row0, kBlk * 4, bar(C::B_DOFULL + ds));
                ++ndo;
                return true;
            };
            bool ok = true;
            for (int k = 0; ok && item_of<CAUSAL>(k, BH, nb, hg, bh, n); ++k) {
                const int m0 = CAUSAL ? n : 0;  // first query block that sees key block n
                const int cnt = nb - m0;        // query blocks walked (>= 1)
                // the first query block ahead of K_n, V_n: its ring slots free up
                // before the products of the item that last used this K/V buffer
                // have all read K and V
                if (!(ok = load_block(m0)))
                    break;
                const int kb = k % KVBUF;
                if (k >= KVBUF && !(ok = wait_bounded(bar(C::B_KVEMPTY + kb), ((k / KVBUF) - 1) & 1, abort_flag)))
                    break;
                mbar_arrive_expect_tx(bar(C::B_KVFULL + kb), 2 * C::TILE);
                for (int b = 0; b < col_blocks<D>(); ++b) {
                    tma_load_3d(sbase + C::KV_OFF + (2 * kb) * C::TILE + b * kSwAtomBytes, &tm_k,
                                bar(C::B_KVFULL + kb), b * 64, n * kBlk, bh, pol_kv);
                    tma_load_3d(sbase + C::KV_OFF + (2 * kb + 1) * C::TILE + b * kSwAtomBytes, &tm_v,
                                bar(C::B_KVFULL + kb), b * 64, n * kBlk, bh, pol_kv);
                }
                ++nkv;
                for (int i = 1; ok && i < cnt; ++i)
                    ok = load_block(m0 + i);
            }
            // wait for every copy this thread issued
            for (int b = 0; b < KVBUF; ++b)
                if (nkv > b)
                    drain_bounded(bar(C::B_KVFULL + b), ((nkv - 1 - b) / KVBUF) & 1);
            for (int s = 0; s < QST; ++s)
                if (nq > s)
                    drain_bounded(bar(C::B_QFULL + s), ((nq - 1 - s) / QST) & 1);
            for (int s = 0; s < DOST; ++s)
                if (ndo > s)
                    drain_bounded(bar(C::B_DOFULL + s), ((ndo - 1 - s) / DOST) & 1);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr bool BF = DTypeTraits<T>::kBF16;
            constexpr uint32_t idesc_s = make_idesc_f16(BF, kBlk, kBlk, false, false);
            constexpr uint32_t idesc_acc = make_idesc_f16(BF, kBlk, D, false, true);
            constexpr uint32_t idesc_dq = make_idesc_f16(BF, kBlk, D, true, true);
            // K-major views (operands whose contraction runs along the row) and
            // MN-major views (contraction down the rows) of the same tiles; K/V
            // buffer b is 2 b TILE bytes further on.
            const uint64_t k_kmaj = make_sdesc_sw128(sbase + C::KV_OFF, 16, 1024);
            const uint64_t k_mn = make_sdesc_sw128(sbase + C::KV_OFF, kSwAtomBytes, 1024);
            const uint64_t v_kmaj = make_sdesc_sw128(sbase + C::KV_OFF + C::TILE, 16, 1024);
            const uint64_t q_kmaj = make_sdesc_sw128(sbase + C::Q_OFF, 16, 1024);
            const uint64_t q_mn = make_sdesc_sw128(sbase + C::Q_OFF, kSwAtomBytes, 1024);
            const uint64_t do_kmaj = make_sdesc_sw128(sbase + C::DO_OFF, 16, 1024);
            const uint64_t do_mn = make_sdesc_sw128(sbase + C::DO_OFF, kSwAtomBytes, 1024);
            const uint64_t ds_mn = make_sdesc_sw128(sbase + C::DS_OFF, kSwAtomBytes, 1024);
            // K step kk: 16 elements along the row (K-major: 32 bytes inside a
            // 64-column swizzle block, then the next block), or 16 rows
            // (MN-major: 2048 bytes).
            auto kmaj = [](int kk) -> uint32_t {
                return static_cast<uint32_t>(((kk >> 2) * kSwAtomBytes + (kk & 3) * 32) >> 4);
            };
            auto mn = [](int kk) -> uint32_t { return static_cast<uint32_t>((kk * 2048) >> 4); };
            auto tile = [](int slot) -> uint32_t {
                FA_CHECK(slot >= 0 && slot < (QST > DOST ? QST : DOST));
                return static_cast<uint32_t>((slot * C::TILE) >> 4);
            };
            auto kvbuf = [](int b) -> uint32_t {
                FA_CHECK(b >= 0 && b < KVBUF);
                return static_cast<uint32_t>((2 * b * C::TILE) >> 4);
            };

            auto issue_s = [&](int s, int b) {  // S^T = K Q^T
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    umma_f16_ss(tmem + kTmS, k_kmaj + kvbuf(b) + kmaj(kk), q_kmaj + tile(s) + kmaj(kk), idesc_s,
                                kk > 0 ? 1u : 0u);
            };
            auto issue_dp = [&](int s, int b) {  // dP^T = V dO^T
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    umma_f16_ss(tmem + kTmDP, v_kmaj + kvbuf(b) + kmaj(kk), do_kmaj + tile(s) + kmaj(kk), idesc_s,
                                kk > 0 ? 1u : 0u);
            };
            auto issue_dv = [&](int s, bool acc) {  // dV += P^T dO
#pragma unroll
                for (int kk = 0; kk < kBlk / 16; ++kk)
                    umma_f16_ts(tmem + kTmDV, tmem + kTmS + tm_p_step(kk, 64), do_mn + tile(s) + mn(kk), idesc_acc,
                                (acc || kk > 0) ? 1u : 0u);
            };
            auto issue_dk = [&](int s, bool acc) {  // dK += dS^T Q (dS^T from TMEM)
#pragma unroll
                for (int kk = 0; kk < kBlk / 16; ++kk)
                    umma_f16_ts(tmem + col_dk<D>(), tmem + col_ds<D>() + tm_p_step(kk, ds_half<D>()), q_mn + tile(s) + mn(kk),
                                idesc_acc, (acc || kk > 0) ? 1u : 0u);
            };
            auto issue_dq = [&](int b) {  // dQ = dS K
#pragma unroll
                for (int kk = 0; kk < kBlk / 16; ++kk)
                    umma_f16_ss(tmem + col_dq<D>(), ds_mn + mn(kk), k_mn + kvbuf(b) + mn(kk), idesc_dq,
                                kk > 0 ? 1u : 0u);
            };
            // S^T and dP^T of global block gq, whose K/V sit in buffer b.  The
            // previous block's dV product, issued earlier, has read P^T from
            // the S^T columns; D > 64: the previous block's dQ, in the dP^T
            // columns, must have been read out first.
            auto start_block = [&](int gq, int b) -> bool {
                if (!wait_bounded(bar(C::B_QFULL + gq % QST), (gq / QST) & 1, abort_flag))
                    return false;
                tc_fence_after();
                issue_s(gq % QST, b);
                umma_commit(bar(C::B_SFULL));
                return true;
            };
            auto start_dp = [&](int gq, int b) -> bool {
                if (!((!C::DQ_ALIAS || gq == 0 || wait_bounded(bar(C::B_DQFREE), (gq - 1) & 1, abort_flag)) &&
                      wait_bounded(bar(C::B_DOFULL + gq % DOST), (gq / DOST) & 1, abort_flag)))
                    return false;
                tc_fence_after();
                issue_dp(gq % DOST, b);
                umma_commit(bar(C::B_DPFULL));
                return true;
            };

            bool ok = true;
            int g = 0;
            bool have = item_of<CAUSAL>(0, BH, nb, hg, bh, n);
            // the first item's first block (CONT: every later item's first
            // block starts inside the previous item's last block)
            if (have)
                ok = wait_bounded(bar(C::B_KVFULL), 0, abort_flag) && start_block(0, 0) && start_dp(0, 0);
            for (int k = 0; ok && have; ++k) {
                const int cnt = nb - (CAUSAL ? n : 0);
                const int kb = k % KVBUF;
                int bh1 = 0, n1 = 0;
                const bool have_next = item_of<CAUSAL>(k + 1, BH, nb, hg, bh1, n1);
                for (int i = 0; ok && i < cnt; ++i) {
                    const int gi = g + i;
                    const int s = gi % QST, ds = gi % DOST;
                    const uint32_t ph = static_cast<uint32_t>(gi & 1);
                    // next block: in this item, or (CONT) the next item's first
                    const bool next_here = i + 1 < cnt;
                    const bool next_cross = CONT && !next_here && have_next;
                    const int kb1 = next_here ? kb : (k + 1) % KVBUF;
                    if (!(ok = wait_bounded(bar(C::B_PFULL), ph, abort_flag)))
                        break;
                    // CONT, block 0: dV_n, dK_n of the previous item are read
                    // out of TMEM before this item's first products reset them
                    // (otherwise the compute warps' epilogue, ahead of this P^T,
                    // has read them)
                    if (CONT && i == 0 && k > 0 && !(ok = wait_bounded(bar(C::B_DKVFREE), (k - 1) & 1, abort_flag)))
                        break;
                    tc_fence_after();
                    issue_dv(ds, i > 0);
                    if (next_here || next_cross) {
                        // S^T of the next block overwrites P^T, after the dV product
                        // above has read it (one thread's MMAs run in issue order)
                        if (next_cross &&
                            !(ok = wait_bounded(bar(C::B_KVFULL + kb1), ((k + 1) / KVBUF) & 1, abort_flag)))
                            break;
                        if (!(ok = start_block(gi + 1, kb1)))
                            break;
                    }
                    if (!(ok = wait_bounded(bar(C::B_DSFULL), ph, abort_flag)))
                        break;
                    tc_fence_after();
                    // the compute warps are done with D_m; dP^T and dV have read dO_m
                    umma_commit(bar(C::B_DOEMPTY + ds));
                    if (!C::DQ_ALIAS && (next_here || next_cross)) {
                        // D <= 64: dP^T of the next block first (its columns are
                        // free: dS^T has columns of its own), so the compute warps
                        // can go on
                        if (!(ok = start_dp(gi + 1, kb1)))
                            break;
                    }
                    // D > 64: dK reads dS^T from the dP^T columns before dQ writes
                    // them (one thread's MMAs run in issue order)
                    issue_dk(s, i > 0);
                    // CONT: dK_n, dV_n are final once this dK product is done; the
                    // dQ warpgroup writes them while dQ_m runs
                    if (CONT && !next_here)
                        umma_commit(bar(C::B_DKVFULL));
                    if (!C::DQ_ALIAS && gi > 0) {
                        if (!(ok = wait_bounded(bar(C::B_DQFREE), (gi - 1) & 1, abort_flag)))
                            break;
                        tc_fence_after();
                    }
                    issue_dq(kb);
                    umma_commit(bar(C::B_DQFULL));
                    umma_commit(bar(C::B_QEMPTY + s));
                    if (C::DQ_ALIAS && next_here) {
                        // dQ_m sits in the dP^T columns: start_dp waits until it is read out
                        if (!(ok = start_dp(gi + 1, kb)))
                            break;
                    }
                }
                if (!ok)
                    break;
                // dK_n, dV_n are final (D > 64: the compute warps then stage them
                // in the dS^T tile, which the last dQ product has read); K_n, V_n
                // are no longer read
                if (!CONT)
                    umma_commit(bar(C::B_DKVFULL));
                umma_commit(bar(C::B_KVEMPTY + kb));
                g += cnt;
                if (!CONT && have_next) {
                    // the next item's K, V land once the products above are done
                    bh = bh1;
                    n = n1;
                    ok = wait_bounded(bar(C::B_KVFULL), (k + 1) & 1, abort_flag) && start_block(g, 0) &&
                         start_dp(g, 0);
                }
                bh = bh1;
                n = n1;
                have = have_next;
            }
            // every MMA this thread issued has completed once this arrives
            umma_commit(bar(C::B_DRAIN));
            drain_bounded(bar(C::B_DRAIN), 0);
        }
    } else if (warp >= kDqWarp0 && warp < kDqWarp0 + 4) {
        // ---------------- dQ warpgroup (CONT: also dK_n, dV_n) ----------------
        const int r = threadIdx.x & 127;  // query row of the block == TMEM lane (dK/dV: key row)
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t dq_tm = tmem + lane_base + col_dq<D>();
        const bool leader = threadIdx.x == kDqWarp0 * 32;
        int chunk = 0, g = 0;
        bool ok = true;
        for (int k = 0; ok && item_of<CAUSAL>(k, BH, nb, hg, bh, n); ++k) {
            const int m0 = CAUSAL ? n : 0;
            const int cnt = nb - m0;
            for (int i = 0; i < cnt; ++i) {
                bool after_epilogue = false;
                if (CONT && i + 1 == cnt) {
                    // ---- dV_n and dK_n of the item (one 64-column block each),
                    // final once the last dK product is done (before the last dQ) ----
                    bool w = wait_bounded(bar(C::B_DKVFULL), static_cast<uint32_t>(k & 1), abort_flag);
                    w = __all_sync(0xffffffffu, w);
                    if (named_bar_or(3, 128, !w)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // staged in the two dQ buffers once the earlier reduces have
                    // read them, 32 columns at a time, rounded (dK = scale dS^T Q:
                    // dS was kept without the scale); then TMEM is free for the
                    // next item's first products
                    const uint32_t sv = sbase + C::STG_OFF;
                    const uint32_t sk = sv + C::STG_BYTES;
                    if (leader)
                        bulk_wait_group_read<0>();
                    named_bar_sync(3, 128);
#pragma unroll 1
                    for (int t = 0; t < 2 * (D / 32); ++t) {
                        const int c4 = t >> 1;
                        const bool is_k = (t & 1) != 0;
                        const float mul = is_k ? scale : 1.f;
                        uint32_t u[32];
                        tmem_ld32(tmem + lane_base + (is_k ? col_dk<D>() : kTmDV) + 32 * c4, u);
                        const uint32_t dst = is_k ? sk : sv;
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            st_shared_v4(dst + sw128_offset(r, 4 * c4 + q4),
                                         DTypeTraits<T>::pack(__uint_as_float(u[8 * q4 + 0]) * mul, __uint_as_float(u[8 * q4 + 1]) * mul),
                                         DTypeTraits<T>::pack(__uint_as_float(u[8 * q4 + 2]) * mul, __uint_as_float(u[8 * q4 + 3]) * mul),
                                         DTypeTraits<T>::pack(__uint_as_float(u[8 * q4 + 4]) * mul, __uint_as_float(u[8 * q4 + 5]) * mul),
                                         DTypeTraits<T>::pack(__uint_as_float(u[8 * q4 + 6]) * mul, __uint_as_float(u[8 * q4 + 7]) * mul));
                    }
                    tc_fence_before();
                    mbar_arrive(bar(C::B_DKVFREE));
                    fence_proxy_async_smem();
                    named_bar_sync(3, 128);
                    if (leader) {
                        tma_store_3d(&tm_dv, sv, 0, n * kBlk, bh);
                        tma_store_3d(&tm_dk, sk, 0, n * kBlk, bh);
                        bulk_commit_group();
                    }
                    after_epilogue = true;  // the next staging waits for these stores
                }
                bool w = wait_bounded(bar(C::B_DQFULL), static_cast<uint32_t>((g + i) & 1), abort_flag);
                w = __all_sync(0xffffffffu, w);
                if (named_bar_or(3, 128, !w)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int m = m0 + i;
#pragma unroll 1
                for (int c4 = 0; c4 < D / 32; ++c4) {
                    uint32_t u[32];
                    tmem_ld32(dq_tm + 32 * c4, u);
                    if (c4 == D / 32 - 1) {
                        // dQ_m has been read out: its TMEM columns are free
                        tc_fence_before();
                        mbar_arrive(bar(C::B_DQFREE));
                    }
#pragma unroll
                    for (int hh = 0; hh < 32 / C::DQ_COLS; ++hh, ++chunk) {
                        const int stg = chunk % NSTG;
                        const uint32_t sbuf = sbase + C::STG_OFF + stg * C::STG_BYTES;
                        // the reduce (or, right after the epilogue, the dV_n / dK_n
                        // stores) that last read this staging buffer has finished reading
                        if (leader && after_epilogue && c4 == 0 && hh == 0)
                            bulk_wait_group_read<0>();
                        else if (leader && chunk >= NSTG)
                            bulk_wait_group_read<NSTG - 1>();
                        named_bar_sync(3, 128);
                        if constexpr (C::DQ_COLS == 32) {
                            // 128-byte rows, 16-byte chunk k at k ^ (r % 8)
#pragma unroll
                            for (int k8 = 0; k8 < 8; ++k8)
                                st_shared_v4(sbuf + r * 128 + (((k8 ^ (r & 7)) & 7) << 4), u[4 * k8], u[4 * k8 + 1],
                                             u[4 * k8 + 2], u[4 * k8 + 3]);
                        } else {
                            // 64-byte rows, 16-byte chunk k at k ^ ((r / 2) % 4)
#pragma unroll
                            for (int k4 = 0; k4 < 4; ++k4)
                                st_shared_v4(sbuf + r * 64 + (((k4 ^ (r >> 1)) & 3) << 4), u[16 * hh + 4 * k4],
                                             u[16 * hh + 4 * k4 + 1], u[16 * hh + 4 * k4 + 2], u[16 * hh + 4 * k4 + 3]);
                        }
                        fence_proxy_async_smem();
                        named_bar_sync(3, 128);
                        if (leader) {
                            tma_reduce_add_3d(&tm_dqacc, sbuf, 32 * c4 + C::DQ_COLS * hh, m * kBlk, bh);
                            bulk_commit_group();
                        }
                    }
                }
            }
            g += cnt;
        }
        if (leader)
            bulk_wait_group<0>();
    } else if (warp < 8) {
        // ---------------- compute warpgroup c ----------------
        const int c = warp >> 2;
        const int r = threadIdx.x & 127;  // key row of the block == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tm_row = tmem + lane_base;  // TMEM lane of this key row, column 0
        // this warpgroup's 64 query columns of the dS^T tile (one swizzle block)
        const uint32_t ds_half_smem = sbase + C::DS_OFF + c * kSwAtomBytes;
        const float2 c2 = make_float2(scale_log2, scale_log2);
        bool ok = true;
        int g = 0;
        for (int k = 0; ok && item_of<CAUSAL>(k, BH, nb, hg, bh, n); ++k) {
            const int m0 = CAUSAL ? n : 0;
            const int cnt = nb - m0;
            const bool row_valid = n * kBlk + r < N;
            for (int i = 0; i < cnt; ++i) {
                const int gi = g + i;
                const int s = gi % QST, ds = gi % DOST;
                const uint32_t ph = static_cast<uint32_t>(gi & 1);
                ok = wait_bounded(bar(C::B_SFULL), ph, abort_flag) &&
                     wait_bounded(bar(C::B_QFULL + s), (gi / QST) & 1, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok)
                    break;
                tc_fence_after();
                // ---- P^T for queries [64c, 64c + 64) of this key row ----
                // causal: the walk starts at the diagonal block m = n, where
                // keys above the query are masked
                const bool diag = CAUSAL && i == 0;
                const float *lrow = reinterpret_cast<const float *>(smem + C::L_OFF + s * kBlk * 4);
                uint32_t pk[32];
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    uint32_t u[32];
                    tmem_ld32(tm_row + kTmS + 64 * c + 32 * ch, u);
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const int q = 64 * c + 32 * ch + j;
                        const float4 l4 = *reinterpret_cast<const float4 *>(lrow + (q & ~3));
                        const float2 l2 = (q & 2) ? make_float2(l4.z, l4.w) : make_float2(l4.x, l4.y);
                        const float2 x = ffma2(make_float2(__uint_as_float(u[j]), __uint_as_float(u[j + 1])), c2,
                                               make_float2(-l2.x, -l2.y));
                        float e0 = ex2_approx(x.x);
                        float e1 = ex2_approx(x.y);
                        if (diag) {
                            e0 = (q >= r) ? e0 : 0.f;
                            e1 = (q + 1 >= r) ? e1 : 0.f;
                        }
                        pk[16 * ch + j / 2] = DTypeTraits<T>::pack(e0, e1);
                    }
                    if (!row_valid) {
                        // key past the sequence end (K row read as zeros): no weight
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            pk[16 * ch + j] = 0u;
                    }
                    tmem_st16(tm_row + kTmS + 64 * c + 16 * ch, reinterpret_cast<const uint32_t(&)[16]>(pk[16 * ch]));
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(C::B_PFULL));

                // ---- dS^T = P^T o (dP^T - D), into TMEM and shared memory ----
                // D <= 64: dK and dQ of the previous block (issued after this
                // dP^T) must have finished reading dS^T before it is overwritten
                ok = wait_bounded(bar(C::B_DPFULL), ph, abort_flag) &&
                     wait_bounded(bar(C::B_DOFULL + ds), (gi / DOST) & 1, abort_flag) &&
                     (C::DQ_ALIAS || gi == 0 || wait_bounded(bar(C::B_DQFULL), ph ^ 1u, abort_flag));
                ok = __all_sync(0xffffffffu, ok);
                if (!ok)
                    break;
                tc_fence_after();
                const float *drow = reinterpret_cast<const float *>(smem + C::DD_OFF + ds * kBlk * 4);
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    uint32_t u[32];
                    tmem_ld32(tm_row + kTmDP + 64 * c + 32 * ch, u);
                    uint32_t w[16];
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const int q = 64 * c + 32 * ch + j;
                        const float4 d4 = *reinterpret_cast<const float4 *>(drow + (q & ~3));
                        const float2 dd = (q & 2) ? make_float2(d4.z, d4.w) : make_float2(d4.x, d4.y);
                        const float2 p = DTypeTraits<T>::unpack(pk[16 * ch + j / 2]);
                        const float2 t = fadd2(make_float2(__uint_as_float(u[j]), __uint_as_float(u[j + 1])),
                                               make_float2(-dd.x, -dd.y));
                        // dS without the scale factor: dK and dQ apply it once at the end
                        const float2 gr = fmul2(p, t);
                        w[j / 2] = DTypeTraits<T>::pack(gr.x, gr.y);
                    }
                    // dS^T into TMEM (A operand of dK) and into shared memory
                    // (MN-major A operand of dQ): 16-byte chunk 4 ch + k of this row
                    // (8 queries each)
                    tmem_st16(tm_row + col_ds<D>() + ds_half<D>() * c + 16 * ch, w);
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4)
                        st_shared_v4(ds_half_smem + r * 128 + ((((4 * ch + k4) ^ (r & 7)) & 7) << 4), w[4 * k4], w[4 * k4 + 1],
                                     w[4 * k4 + 2], w[4 * k4 + 3]);
                }
                fence_proxy_async_smem();
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(C::B_DSFULL));
            }
            g += cnt;
            if constexpr (!CONT) {
                // ---------------- epilogue of the item: dV_n and dK_n ----------------
                if (ok) {
                    ok = wait_bounded(bar(C::B_DKVFULL), static_cast<uint32_t>(k & 1), abort_flag);
                    ok = __all_sync(0xffffffffu, ok);
                }
                if (named_bar_or(1 + c, 128, !ok || *abort_flag != 0)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // Round 32-column chunks [c0, c0 + nch) of a TMEM accumulator, stage
                // them in this warpgroup's half of the dS^T tile (free: every product
                // has completed, the last dQ included) and store them from column
                // 32 c0.  The tile is reused by the next item's dS^T only after the
                // store has finished reading it.
                auto store_acc = [&](const CUtensorMap *map, uint32_t acc_col, int c0, int nch, float mul) {
                    for (int c4 = 0; c4 < nch; ++c4) {
                        uint32_t u[32];
                        tmem_ld32(tm_row + acc_col + 32 * (c0 + c4), u);
                        float f[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            f[j] = __uint_as_float(u[j]) * mul;
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            st_shared_v4(ds_half_smem + sw128_offset(r, c4 * 4 + q4),
                                         DTypeTraits<T>::pack(f[8 * q4 + 0], f[8 * q4 + 1]),
                                         DTypeTraits<T>::pack(f[8 * q4 + 2], f[8 * q4 + 3]),
                                         DTypeTraits<T>::pack(f[8 * q4 + 4], f[8 * q4 + 5]),
                                         DTypeTraits<T>::pack(f[8 * q4 + 6], f[8 * q4 + 7]));
                    }
                    fence_proxy_async_smem();
                    named_bar_sync(1 + c, 128);
                    if (r == 0) {
                        tma_store_3d(map, ds_half_smem, 32 * c0, n * kBlk, bh);
                        bulk_commit_group();
                        bulk_wait_group_read<0>();
                    }
                    named_bar_sync(1 + c, 128);
                };
                // dK = scale dS^T Q (dS was kept without the scale); dV as is.
                // Warpgroup c writes columns [64c, 64c + 64) of both.
                const int nch = (D / 32 - 2 * c) < 2 ? (D / 32 - 2 * c) : 2;
                store_acc(&tm_dv, kTmDV, 2 * c, nch, 1.f);
                store_acc(&tm_dk, col_dk<D>(), 2 * c, nch, scale);
            }
        }
        if (!CONT && r == 0)
            bulk_wait_group<0>();
        tc_fence_before();
    }

    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// D_i = sum_c dO_ic O_ic and L_i log2(e) for every row of a padded
// [BH, Npad] layout (padding rows: D = 0, L = +inf, so P = 0 there), and the
// fp32 dQ accumulator [BH, Npad, D] set to zero.  D / 8 threads per row, 8
// elements (16 bytes) each.
template <int D, typename T>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const T *__restrict__ o, const T *__restrict__ dout,
                                                          const float *__restrict__ lse,
                                                          float *__restrict__ lse2, float *__restrict__ dvec,
                                                          float *__restrict__ dqacc, int N, int Npad,
                                                          long long rows)
{
    // threads per row: D / 8 rounded up to a power of two (so a row's threads
    // sit in one warp); the parts past D have nothing to read
    constexpr int TPR = D <= 32 ? 4 : D <= 64 ? 8 : 16;
    const long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long row = g / TPR;
    const int part = static_cast<int>(g % TPR);
    const bool valid = row < rows;
    const long long bh = valid ? row / Npad : 0;
    const int i = valid ? static_cast<int>(row % Npad) : 0;
    const bool live = valid && i < N;
    const bool has_part = part * 8 < D;
    float acc = 0.f;
    if (live && has_part) {
        const size_t off = (static_cast<size_t>(bh) * N + i) * D + part * 8;
        const uint4 a = *reinterpret_cast<const uint4 *>(o + off);
        const uint4 b = *reinterpret_cast<const uint4 *>(dout + off);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
        const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 x = DTypeTraits<T>::unpack(aw[k]);
            const float2 y = DTypeTraits<T>::unpack(bw[k]);
            acc = fmaf(x.x, y.x, acc);
            acc = fmaf(x.y, y.y, acc);
        }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (valid) {
        if (part == 0) {
            dvec[row] = live ? acc : 0.f;
            lse2[row] = live ? lse[static_cast<size_t>(bh) * N + i] * 1.4426950408889634f : INFINITY;
        }
        if (has_part) {
            float4 *z = reinterpret_cast<float4 *>(dqacc + static_cast<size_t>(row) * D + part * 8);
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

// dQ [BH, N, D] = scale x the fp32 accumulator [BH, Npad, D] (which holds
// dS K without the scale), rounded to the input dtype.
template <int D, typename T>
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const float *__restrict__ dqacc, T *__restrict__ dq,
                                                        int N, int Npad, long long chunks, float scale)
{
    constexpr int CPR = D / 8;  // 8-element chunks per row
    for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < chunks;
         g += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = g / CPR;  // row of [BH * N]
        const int part = static_cast<int>(g % CPR);
        const long long bh = row / N;
        const int i = static_cast<int>(row % N);
        const float4 *src = reinterpret_cast<const float4 *>(
            dqacc + (static_cast<size_t>(bh) * Npad + i) * D + part * 8);
        float4 a = src[0], b = src[1];
        a.x *= scale, a.y *= scale, a.z *= scale, a.w *= scale;
        b.x *= scale, b.y *= scale, b.z *= scale, b.w *= scale;
        *reinterpret_cast<uint4 *>(dq + static_cast<size_t>(row) * D + part * 8) =
            make_uint4(DTypeTraits<T>::pack(a.x, a.y), DTypeTraits<T>::pack(a.z, a.w),
                       DTypeTraits<T>::pack(b.x, b.y), DTypeTraits<T>::pack(b.z, b.w));
    }
}

}  // namespace bwd
}  // namespace fa
