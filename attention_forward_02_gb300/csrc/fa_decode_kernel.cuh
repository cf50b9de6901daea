// fa_decode_kernel.cuh -- attention for decoding on sm_103a: a few queries
// (1 <= Nq <= 16) per head against a long key sequence (Nk keys).
//
// What it computes is the attention of the forward kernel, O = softmax(Q K^T
// scale) V and LSE, for Nq query rows that sit at the end of the sequence
// (causal: query i attends to keys 0 .. Nk - Nq + i).  "3.6 어텐션 I —
// 메모리 문제·FlashAttention 원리", section 3.6.9 notes that decoding (one
// query) needs a different parallelisation: with one query per head there is
// no Q block to spread over the SMs, and the work is a single pass over K and
// V (about Nq flop per byte, far below the tensor-core ridge), so the time is
// the time to stream K and V from HBM.
//
// Split-KV: the keys of each head are cut into chunks of whole 128-key tiles;
//   fa_decode_split_kernel   persistent, one CTA per SM walking (batch*head,
//                            chunk) items; the producer streams the K/V tiles
//                            of its items back to back through a TMA ring;
//                            per item the compute warps run the online
//                            softmax of section 3.6.4 over them (running max
//                            m, per-thread partial sums l, unnormalised O),
//                            leaving (m, l, O) of the chunk in a workspace;
//   fa_decode_combine_kernel merges the chunks of each query with the same
//                            algebra (the result does not depend on how the
//                            keys are cut, section 3.6.4), and writes O / l and
//                            LSE.
// The arithmetic is on the CUDA cores (fp32); tensor cores would idle on a
// 1..16-row product that HBM cannot feed anyway.
//
// Warp roles of the split kernel (288 threads): warps 0-7 compute, warp 8 TMA
// producer.  Per tile and query:
//   scores   lanes l and l + 16 of warp w take key 16 w + l of the tile, half
//            of d each (so every 8-lane quarter of a 128-bit shared load reads
//            8 consecutive rows: no bank conflict under the 128B swizzle):
//            s' = (q scale log2 e) . k_r in packed fp32 FMAs, halves summed by
//            a lane shuffle;
//   max      warp shuffles, then the eight warps' maxima through shared memory;
//   p        p_r = 2^(s' - m_new), l_r = l_r alpha + p_r (alpha = 2^(m_old - m_new)),
//            written to shared memory for the next phase;
//   P V      thread t takes a column pair of V and a group of the tile's keys:
//            o = o alpha + sum_j p_j v_j (fp32), a fully unrolled loop whose
//            swizzled shared-memory offsets are compile-time constants.
// The number of queries is a template parameter NQ in {1, 2, 4, 8, 16} (the
// launch rounds Nq up; rows past Nq are computed on zero queries and dropped).
// Every mbarrier wait is bounded, as in the other kernels.
#pragma once

#include "fa_common.cuh"

namespace fa {
namespace dec {

constexpr int kTileKeys = 128;
constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = 32 * kComputeWarps;
constexpr int kProducerWarp = kComputeWarps;
constexpr int kThreads = kComputeThreads + 32;
constexpr int kMaxNq = 16;

// Head dims 32 and 96 use tiles of whole 64-column swizzle blocks (TMA fills
// the columns past D with zeros), as the forward kernel does.
template <int D>
__host__ __device__ constexpr int col_blocks()
{
    return (D + 63) / 64;
}

template <int D, int NQ>
struct Cfg {
    static_assert(D == 32 || D == 64 || D == 96 || D == 128, "head dims 32, 64, 96, 128");
    static constexpr int TILE = kTileKeys * col_blocks<D>() * 128;  // one [128, D] 16-bit K or V tile
    static constexpr int PAIRS = D / 2;              // column pairs of the P V phase
    // key groups of the P V phase (D = 96: 48 pairs x 4 groups, 64 threads idle there)
    static constexpr int GROUPS = D == 96 ? 4 : kComputeThreads / PAIRS;
    static constexpr int PV_THREADS = GROUPS * PAIRS;
    static constexpr int KEYS_PER_GROUP = kTileKeys / GROUPS;
    // per-CTA areas besides the ring (q, p, warp maxima, O reduction, barriers, slack)
    static constexpr int EXTRA = NQ * D * 4 + NQ * kTileKeys * 4 + NQ * kComputeWarps * 4 +
                                 GROUPS * NQ * D * 4 + 8 * 2 * 6 + 16 + 1024;
    // up to 192 KiB of K/V in flight per SM, as far as the budget allows
    static constexpr int MAX_STAGES = (227 * 1024 - EXTRA) / (2 * TILE);
    static constexpr int STAGES = (D == 64 ? 6 : 3) < MAX_STAGES ? (D == 64 ? 6 : 3) : MAX_STAGES;
    static_assert(STAGES >= 2, "at least a double-buffered ring");
    static constexpr int KV_OFF = 0;                 // stage s: K at 2 s TILE, V at (2 s + 1) TILE
    static constexpr int QF_OFF = KV_OFF + STAGES * 2 * TILE;     // fp32 [NQ][D]
    static constexpr int PS_OFF = QF_OFF + NQ * D * 4;            // fp32 [NQ][kTileKeys]
    static constexpr int WM_OFF = PS_OFF + NQ * kTileKeys * 4;    // fp32 [NQ][kComputeWarps]
    static constexpr int RO_OFF = WM_OFF + NQ * kComputeWarps * 4;  // fp32 [GROUPS][NQ][D] O reduction
    static constexpr int BAR_OFF = RO_OFF + GROUPS * NQ * D * 4;
    static constexpr int B_FULL = 0;
    static constexpr int B_EMPTY = STAGES;
    static constexpr int NUM_BARS = 2 * STAGES;
    static constexpr int SLOT_OFF = BAR_OFF + 8 * NUM_BARS;  // abort flag
    static constexpr int SMEM_USED = SLOT_OFF + 16;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;
    static_assert(KEYS_PER_GROUP % 8 == 0 && KEYS_PER_GROUP * GROUPS == kTileKeys,
                  "key groups start on a swizzle period and cover the tile");
    static_assert(PV_THREADS <= kComputeThreads, "P V threads");
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

// 128-bit shared load of 8 16-bit values, widened to fp32.
template <typename T>
__device__ __forceinline__ void load8(uint32_t addr, float (&f)[8])
{
    const uint4 x = ld_shared_v4(addr);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = DTypeTraits<T>::unpack(w[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr)
{
    float v;
    if (!smem_ok(addr, 4, 4))
        return 0.f;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr)
{
    uint32_t v;
    if (!smem_ok(addr, 4, 4))
        return 0u;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v)
{
    if (!smem_ok(addr, 4, 4))
        return;
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Workspace of one launch: for every (batch*head, chunk, query) the chunk's
// running max m (log2 units of the scaled score), sum l and unnormalised O.
struct Partials {
    float *o;  // [BH, splits, Nq, D]
    float *m;  // [BH, splits, Nq]
    float *l;  // [BH, splits, Nq]
};

template <int D, int NQ, typename T>
__global__ void __launch_bounds__(kThreads, 1)
    fa_decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                           const T *__restrict__ q, Partials part, int Nq, int Nk, int splits,
                           int tiles_per_split, int num_items, int causal, float scale_log2)
{
    using C = Cfg<D, NQ>;
    constexpr int STAGES = C::STAGES;
    constexpr int HALF_CHUNKS = D / 16;  // 16-byte chunks in half a key row

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    auto bar = [&](int idx) -> uint32_t { return sbase + C::BAR_OFF + 8u * idx; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::SLOT_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_tiles = (Nk + kTileKeys - 1) / kTileKeys;
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
            mbar_init(bar(C::B_EMPTY + s), kComputeThreads);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kProducerWarp) {
        if (lane == 0) {
            // ---------------- producer: the tiles of every item, back to back ----------------
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const uint64_t pol = l2_policy_evict_first();  // K and V are read once
            int L = 0;  // loads into the ring so far
            bool ok = true;
            for (int w = blockIdx.x; ok && w < num_items; w += gridDim.x) {
                int bh, split, t0;
                const int nt = item_tiles(w, bh, split, t0);
                for (int i = 0; i < nt; ++i, ++L) {
                    const int s = L % STAGES;
                    if (L >= STAGES && !(ok = wait_bounded(bar(C::B_EMPTY + s), ((L / STAGES) - 1) & 1, abort_flag)))
                        break;
                    const uint32_t kdst = sbase + C::KV_OFF + (2 * s) * C::TILE;
                    mbar_arrive_expect_tx(bar(C::B_FULL + s), 2 * C::TILE);
                    for (int b = 0; b < col_blocks<D>(); ++b) {
                        tma_load_3d(kdst + b * kSwAtomBytes, &tm_k, bar(C::B_FULL + s), b * 64,
                                    (t0 + i) * kTileKeys, bh, pol);
                        tma_load_3d(kdst + C::TILE + b * kSwAtomBytes, &tm_v, bar(C::B_FULL + s), b * 64,
                                    (t0 + i) * kTileKeys, bh, pol);
                    }
                }
            }
            for (int s = 0; s < STAGES; ++s)
                if (L > s)
                    drain_bounded(bar(C::B_FULL + s), ((L - 1 - s) / STAGES) & 1);
        }
    } else {
        // ---------------- compute warps ----------------
        const int t = threadIdx.x;
        const int key_r = warp * 16 + (lane & 15);  // score phase: key of the tile ...
        const int half = lane >> 4;                 // ... and which half of d
        const int pair = t % C::PAIRS;      // P V phase: column pair ...
        const int grp = t / C::PAIRS;       // ... and key group
        // score phase: byte offset of 16-byte chunk c of this thread's half row
        // (16-byte chunks XOR-swizzled by row % 8 inside 128-byte rows; the two
        // 64-column blocks of D = 128 are kSwAtomBytes apart)
        const uint32_t krow = static_cast<uint32_t>(key_r) * 128u;
        // P V phase: the column pair's 16-byte chunk and its offset inside it
        const int pc8 = (2 * pair) >> 3;
        const uint32_t pv_col = static_cast<uint32_t>((pc8 >> 3) * kSwAtomBytes) + (static_cast<uint32_t>((2 * pair) & 7) * 2u);
        int L = 0;  // tiles consumed so far (all items)
        bool ok = true;
        for (int w = blockIdx.x; ok && w < num_items; w += gridDim.x) {
            int bh, split, t0;
            const int nt = item_tiles(w, bh, split, t0);
            // q of this head, pre-multiplied by scale * log2(e), as fp32; rows
            // past Nq are zero (the previous item's last barrier has retired
            // every read of this area)
            for (int x = t; x < NQ * D; x += kComputeThreads) {
                float val = 0.f;
                if (x < Nq * D) {
                    const uint16_t bits = reinterpret_cast<const uint16_t *>(q)[static_cast<size_t>(bh) * Nq * D + x];
                    val = DTypeTraits<T>::unpack(static_cast<uint32_t>(bits)).x * scale_log2;
                }
                st_shared_f32(sbase + C::QF_OFF + 4u * x, val);
            }
            named_bar_sync(1, kComputeThreads);
            float m[NQ], l[NQ];
            float2 o[NQ];
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                m[qi] = -INFINITY;
                l[qi] = 0.f;
                o[qi] = make_float2(0.f, 0.f);
            }
            for (int i = 0; i < nt; ++i, ++L) {
                const int s = L % STAGES;
                ok = wait_bounded(bar(C::B_FULL + s), (L / STAGES) & 1, abort_flag);
                // one decision for all eight warps: the named barriers below need them all
                if (named_bar_or(3, kComputeThreads, !ok || *abort_flag != 0)) {
                    ok = false;
                    break;
                }
                const uint32_t ktile = sbase + C::KV_OFF + (2 * s) * C::TILE;
                const uint32_t vtile = ktile + C::TILE;
                const int key = (t0 + i) * kTileKeys + key_r;
                // ---- scores: this thread's half of key key_r against every query ----
                float2 acc[NQ];
#pragma unroll
                for (int qi = 0; qi < NQ; ++qi)
                    acc[qi] = make_float2(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < HALF_CHUNKS; ++c) {
                    const int chunk = half * HALF_CHUNKS + c;  // 16-byte chunk of the row
                    const uint32_t addr = ktile + static_cast<uint32_t>((chunk >> 3) * kSwAtomBytes) + krow +
                                          ((static_cast<uint32_t>((chunk & 7) ^ (key_r & 7))) << 4);
                    const uint4 kx = ld_shared_v4(addr);
                    const float2 k0 = DTypeTraits<T>::unpack(kx.x), k1 = DTypeTraits<T>::unpack(kx.y);
                    const float2 k2 = DTypeTraits<T>::unpack(kx.z), k3 = DTypeTraits<T>::unpack(kx.w);
#pragma unroll
                    for (int qi = 0; qi < NQ; ++qi) {
                        const float4 a = *reinterpret_cast<const float4 *>(smem + C::QF_OFF + 4 * (qi * D + 8 * chunk));
                        const float4 b = *reinterpret_cast<const float4 *>(smem + C::QF_OFF + 4 * (qi * D + 8 * chunk + 4));
                        acc[qi] = ffma2(make_float2(a.x, a.y), k0, acc[qi]);
                        acc[qi] = ffma2(make_float2(a.z, a.w), k1, acc[qi]);
                        acc[qi] = ffma2(make_float2(b.x, b.y), k2, acc[qi]);
                        acc[qi] = ffma2(make_float2(b.z, b.w), k3, acc[qi]);
                    }
                }
                // ---- both halves, masks, tile maxima ----
                float sc[NQ];
#pragma unroll
                for (int qi = 0; qi < NQ; ++qi) {
                    float v = acc[qi].x + acc[qi].y;
                    v += __shfl_xor_sync(0xffffffffu, v, 16);
                    const int last = causal ? Nk - Nq + qi : Nk - 1;  // last key query qi may see
                    if (key > last)
                        v = -INFINITY;
                    sc[qi] = v;
                    float wm = v;
#pragma unroll
                    for (int off = 8; off > 0; off >>= 1)  // lanes l, l + 16 hold the same score
                        wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, off));
                    if (lane == 0)
                        st_shared_f32(sbase + C::WM_OFF + 4u * (qi * kComputeWarps + warp), wm);
                }
                named_bar_sync(1, kComputeThreads);
                float alpha[NQ];
#pragma unroll
                for (int qi = 0; qi < NQ; ++qi) {
                    const float4 w0 = *reinterpret_cast<const float4 *>(smem + C::WM_OFF + 4 * (qi * kComputeWarps));
                    const float4 w1 = *reinterpret_cast<const float4 *>(smem + C::WM_OFF + 4 * (qi * kComputeWarps + 4));
                    const float tmax = fmaxf(fmax3(w0.x, w0.y, w0.z), fmax3(fmax3(w0.w, w1.x, w1.y), w1.z, w1.w));
                    const float m_new = fmaxf(m[qi], tmax);
                    float p = 0.f;
                    alpha[qi] = 1.f;
                    if (m_new != -INFINITY) {  // some key of this query seen so far
                        alpha[qi] = ex2_approx(m[qi] - m_new);
                        p = ex2_approx(sc[qi] - m_new);
                        m[qi] = m_new;
                    }
                    if (half == 0) {
                        l[qi] = l[qi] * alpha[qi] + p;
                        st_shared_f32(sbase + C::PS_OFF + 4u * (qi * kTileKeys + key_r), p);
                    }
                }
                named_bar_sync(1, kComputeThreads);
                // ---- P V: column pair `pair`, keys [grp KEYS_PER_GROUP, +KEYS_PER_GROUP) ----
#pragma unroll
                for (int qi = 0; qi < NQ; ++qi)
                    o[qi] = fmul2(o[qi], make_float2(alpha[qi], alpha[qi]));
                const uint32_t vbase = vtile + pv_col + static_cast<uint32_t>(grp * C::KEYS_PER_GROUP) * 128u;
                const uint8_t *pbase = smem + C::PS_OFF + 4 * (grp * C::KEYS_PER_GROUP);
#pragma unroll
                for (int j4 = 0; j4 < C::KEYS_PER_GROUP; j4 += 4) {
                    if (C::PV_THREADS < kComputeThreads && t >= C::PV_THREADS)
                        break;
                    float4 pq[NQ];
#pragma unroll
                    for (int qi = 0; qi < NQ; ++qi)
                        pq[qi] = *reinterpret_cast<const float4 *>(pbase + 4 * (qi * kTileKeys + j4));
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int jj = j4 + u;  // key of the group; its row % 8 is jj % 8
                        const uint32_t va = vbase + static_cast<uint32_t>(jj) * 128u +
                                            ((static_cast<uint32_t>((pc8 & 7) ^ (jj & 7))) << 4);
                        const float2 vv = DTypeTraits<T>::unpack(ld_shared_u32(va));
#pragma unroll
                        for (int qi = 0; qi < NQ; ++qi) {
                            const float pj = u == 0 ? pq[qi].x : u == 1 ? pq[qi].y : u == 2 ? pq[qi].z : pq[qi].w;
                            o[qi] = ffma2(make_float2(pj, pj), vv, o[qi]);
                        }
                    }
                }
                // the stage (K and V) is free again; the p buffer and the warp
                // maxima are free once every thread has passed this barrier
                mbar_arrive(bar(C::B_EMPTY + s));
                named_bar_sync(1, kComputeThreads);
            }
            if (!ok)
                break;
            // ---------------- the item's (m, l, O) ----------------
            // l: sum over the threads (keys); O: sum over the key groups
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                float ws = l[qi];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    ws += __shfl_xor_sync(0xffffffffu, ws, off);
                if (lane == 0)
                    st_shared_f32(sbase + C::WM_OFF + 4u * (qi * kComputeWarps + warp), ws);
                if (t < C::PV_THREADS) {
                    const uint32_t oa = sbase + C::RO_OFF + 4u * ((grp * NQ + qi) * D + 2 * pair);
                    st_shared_f32(oa, o[qi].x);
                    st_shared_f32(oa + 4, o[qi].y);
                }
            }
            named_bar_sync(1, kComputeThreads);
            const size_t base = (static_cast<size_t>(bh) * splits + split) * Nq;
            for (int x = t; x < Nq * D; x += kComputeThreads) {
                const int qi = x / D, c = x % D;
                float sum = 0.f;
                for (int g = 0; g < C::GROUPS; ++g)
                    sum += ld_shared_f32(sbase + C::RO_OFF + 4u * ((g * NQ + qi) * D + c));
                part.o[(base + qi) * D + c] = sum;
            }
            if (t < Nq) {
                float sum = 0.f;
                for (int wi = 0; wi < kComputeWarps; ++wi)
                    sum += ld_shared_f32(sbase + C::WM_OFF + 4u * (t * kComputeWarps + wi));
                part.l[base + t] = sum;
#pragma unroll
                for (int qi = 0; qi < NQ; ++qi)
                    if (qi == t)
                        part.m[base + t] = m[qi];
            }
            // every read of the reduction areas and of q is done before the next item
            named_bar_sync(1, kComputeThreads);
        }
    }
    __syncthreads();
}

// Merges the chunks of every (batch*head, query): M = max_s m_s,
// L = sum_s l_s 2^(m_s - M), O = sum_s O_s 2^(m_s - M) / L, LSE = (M + log2 L) ln 2.
// One warp per (batch*head, query).
template <int D, typename T>
__global__ void __launch_bounds__(256) fa_decode_combine_kernel(Partials part, T *__restrict__ out,
                                                                float *__restrict__ lse, long long rows, int Nq,
                                                                int splits)
{
    const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows)
        return;
    const long long bh = row / Nq;
    const int qi = static_cast<int>(row % Nq);
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s)
        M = fmaxf(M, part.m[(bh * splits + s) * Nq + qi]);
    // column pairs 2 pr, 2 pr + 1 for pr = lane, lane + 32, ... (< D / 2)
    constexpr int PAIRS = D / 2;
    constexpr int PPL = (PAIRS + 31) / 32;
    float2 acc[PPL];
#pragma unroll
    for (int k = 0; k < PPL; ++k)
        acc[k] = make_float2(0.f, 0.f);
    float L = 0.f;
    for (int s = 0; s < splits; ++s) {
        const size_t idx = (static_cast<size_t>(bh) * splits + s) * Nq + qi;
        const float ms = part.m[idx];
        if (ms == -INFINITY)
            continue;  // a chunk with no key this query may see
        const float w = ex2_approx(ms - M);
        L = fmaf(part.l[idx], w, L);
#pragma unroll
        for (int k = 0; k < PPL; ++k) {
            const int pr = lane + 32 * k;
            if (pr < PAIRS) {
                const float2 v = *reinterpret_cast<const float2 *>(part.o + idx * D + 2 * pr);
                acc[k] = make_float2(fmaf(v.x, w, acc[k].x), fmaf(v.y, w, acc[k].y));
            }
        }
    }
    const float inv = 1.f / L;
    T *dst = out + static_cast<size_t>(row) * D;
#pragma unroll
    for (int k = 0; k < PPL; ++k) {
        const int pr = lane + 32 * k;
        if (pr < PAIRS)
            *reinterpret_cast<uint32_t *>(dst + 2 * pr) = DTypeTraits<T>::pack(acc[k].x * inv, acc[k].y * inv);
    }
    if (lse != nullptr && lane == 0)
        lse[row] = (M + __log2f(L)) * 0.6931471805599453f;
}

}  // namespace dec
}  // namespace fa
