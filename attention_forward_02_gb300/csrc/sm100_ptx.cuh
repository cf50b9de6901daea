// sm100_ptx.cuh -- thin inline-PTX wrappers for the Blackwell (sm_100 family,
// built here for sm_103a) features the attention kernel uses: mbarriers,
// TMA tensor loads, tcgen05 MMA / TMEM allocation / TMEM loads and stores,
// and the proxy / tcgen05 ordering fences.  Written from the PTX ISA
// descriptions of these instructions.  Also the bulk copies (plain, tensor
// store, tensor reduce-add) the backward kernel uses.
#pragma once

#include <cstdint>

namespace fa {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// Device status word and the checked build
//
// Device status word, one per device and translation unit (the host side of
// each unit reads and clears its own): bit 0 = a bounded wait expired, bit 1 =
// the wait self-test misbehaved, bit 2 = an address check of the checked build
// failed.
static __device__ unsigned int g_fa_status;
constexpr unsigned int kStatusTimeout = 1u;
constexpr unsigned int kStatusSelftest = 2u;
constexpr unsigned int kStatusBounds = 4u;

// Checked build (compiled with -DFA_BOUNDS_CHECK, a second library beside the
// product one).  Every wrapper below that names a shared-memory or tensor-
// memory address checks it first: shared addresses must lie inside the
// block's shared window with their alignment, tensor-memory accesses inside
// the 512 columns (and, for a warp's loads and stores, in that warp's lane
// quarter), and the footprint of every MMA operand and accumulator inside its
// memory.  A failed check records kStatusBounds in the status word and skips
// the access (no trap): the kernel's bounded waits then end the launch, and
// the host reads FA_ERR_BOUNDS.  In the product build the checks compile away.
#ifdef FA_BOUNDS_CHECK
constexpr bool kBoundsCheck = true;
#else
constexpr bool kBoundsCheck = false;
#endif
constexpr uint32_t kTmemColumns = 512;

static __device__ __noinline__ void bounds_fail() { atomicOr(&g_fa_status, kStatusBounds); }

// One past the last shared-memory byte of the block (static + dynamic; the
// dynamic area follows the static one).
__device__ __forceinline__ uint32_t smem_window_end()
{
    extern __shared__ uint8_t fa_dynamic_smem[];
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    return smem_u32(fa_dynamic_smem) + dyn;
}

// The check itself (FORCE: evaluated in either build; used by the self-test).
template <bool FORCE = false>
__device__ __forceinline__ bool smem_ok(uint32_t addr, uint32_t bytes, uint32_t align)
{
    if (!kBoundsCheck && !FORCE)
        return true;
    const uint32_t end = smem_window_end();
    const bool ok = (addr & (align - 1u)) == 0u && addr < end && bytes <= end - addr;
    if (!ok)
        bounds_fail();
    return ok;
}

// Columns [col, col + ncols) of tensor memory; lane_quarter: the address is
// used by this warp's tcgen05.ld / st, whose lanes are 32 (warp % 4) + 0..31.
template <bool FORCE = false>
__device__ __forceinline__ bool tmem_ok(uint32_t taddr, uint32_t ncols, bool lane_quarter)
{
    if (!kBoundsCheck && !FORCE)
        return true;
    const uint32_t col = taddr & 0xFFFFu, lanes = taddr >> 16;
    bool ok = col < kTmemColumns && ncols <= kTmemColumns - col;
    if (lane_quarter)
        ok = ok && lanes == 32u * ((threadIdx.x >> 5) & 3u);
    else
        ok = ok && lanes == 0u;
    if (!ok)
        bounds_fail();
    return ok;
}

// Footprint of a 128B-swizzled operand tile named by a shared-memory matrix
// descriptor: `rows` rows of the M or N dimension (K-major: 8-row groups SBO
// apart, each inside one aligned 1024-byte block; MN-major: 64-element
// column blocks LBO apart, one K step = 16 rows of 128 bytes).
template <bool FORCE = false>
__device__ __forceinline__ bool sdesc_ok(uint64_t desc, uint32_t rows, bool mn_major)
{
    if (!kBoundsCheck && !FORCE)
        return true;
    const uint32_t start = static_cast<uint32_t>(desc & 0x3FFFu) << 4;
    const uint32_t lbo = static_cast<uint32_t>((desc >> 16) & 0x3FFFu) << 4;
    const uint32_t sbo = static_cast<uint32_t>((desc >> 32) & 0x3FFFu) << 4;
    if (mn_major)
        return smem_ok<FORCE>(start, ((rows + 63u) / 64u - 1u) * lbo + 16u * 128u, 128u);
    const uint32_t base = start & ~1023u;
    return smem_ok<FORCE>(base, (rows / 8u - 1u) * sbo + 1024u, 1024u);
}

// Index check of the checked build (ring slots, buffers, barrier numbers):
// records kStatusBounds when the condition is false.
#define FA_CHECK(cond)                            \
    do {                                          \
        if (::fa::kBoundsCheck && !(cond))        \
            ::fa::bounds_fail();                  \
    } while (0)

// Makes a warp-collective decision uniform (every lane skips or none).
__device__ __forceinline__ bool warp_all(bool v)
{
    return kBoundsCheck ? __all_sync(0xffffffffu, v) : v;
}

// ---------------------------------------------------------------------------
// mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    if (!smem_ok(bar, 8, 8))
        return;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes the initialised barriers visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    if (!smem_ok(bar, 8, 8))
        return;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    if (!smem_ok(bar, 8, 8))
        return;
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// True once the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    if (!smem_ok(bar, 8, 8))
        return false;
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// ---------------------------------------------------------------------------
// TMA (bulk tensor copy global -> shared, completion counted on an mbarrier)

__device__ __forceinline__ void tma_prefetch_desc(const void *tmap)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, uint32_t bar, int x,
                                            int y, int z, uint64_t policy)
{
    // every box here is at least 1 KB and 128-byte aligned
    if (!smem_ok(dst, 1024, 128) || !smem_ok(bar, 8, 8))
        return;
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(policy)
        : "memory");
}

// Plain bulk copy global -> shared of `bytes` (a multiple of 16; both
// addresses 16-byte aligned), completion counted on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    if (!smem_ok(dst, bytes, 16) || !smem_ok(bar, 8, 8))
        return;
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// Tensor store shared -> global of one box (rows outside the tensor are not
// written), tracked by the issuing thread's bulk async-group.
__device__ __forceinline__ void tma_store_3d(const void *tmap, uint32_t src, int x, int y, int z)
{
    if (!smem_ok(src, 1024, 128))
        return;
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(tmap)),
        "r"(src), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// Tensor reduce-add shared -> global of one box: global += shared, element
// by element, performed in L2 (atomic with respect to other reductions).
__device__ __forceinline__ void tma_reduce_add_3d(const void *tmap, uint32_t src, int x, int y, int z)
{
    if (!smem_ok(src, 1024, 128))
        return;
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(tmap)),
        "r"(src), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// At most N of this thread's bulk groups still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// At most N of this thread's bulk groups not yet complete.
template <int N>
__device__ __forceinline__ void bulk_wait_group()
{
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// L2 eviction-priority policies for the cache hint above.
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------------------
// Fences

// Generic-proxy shared-memory writes become visible to the async proxy
// (tcgen05.mma operand reads).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Named barrier that also ORs a predicate across the participating threads:
// every thread gets the same result.
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t nthreads, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Named barrier over a subset of the CTA's warps.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Per-warpgroup register budget change (all four warps of a warpgroup execute
// it).  The shares of all warpgroups must add up to at most the registers the
// block was launched with.
template <uint32_t R>
__device__ __forceinline__ void reg_alloc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}
template <uint32_t R>
__device__ __forceinline__ void reg_dealloc()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}

// ---------------------------------------------------------------------------
// TMEM allocation (one full warp executes each of these)

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 MMA, kind::f16 (fp16 or bf16 operands, fp32 accumulator in TMEM)

// Instruction descriptor: D fp32, A/B fp16 (0) or bf16 (1), dense, no negate;
// a_mn / b_mn select MN-major operands; N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t make_idesc_f16(bool bf16, int M, int N, bool a_mn, bool b_mn)
{
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile:
// start address, leading- and stride-dimension byte offsets (all >> 4),
// descriptor version 1 (bits 46-47), layout SWIZZLE_128B (2 at bits 61-63).
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                     uint32_t sbo_bytes)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_f16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate)
{
    if (kBoundsCheck) {
        const uint32_t m = ((idesc >> 24) & 0x1Fu) << 4, n = ((idesc >> 17) & 0x3Fu) << 3;
        if (!(tmem_ok(d_tmem, n, false) && sdesc_ok(adesc, m, (idesc >> 15) & 1u) &&
              sdesc_ok(bdesc, n, (idesc >> 16) & 1u)))
            return;
    }
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T: A (M = 128 rows = lanes, 16-bit elements
// packed two per 32-bit column along K) is read from tensor memory.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate)
{
    if (kBoundsCheck) {
        const uint32_t n = ((idesc >> 17) & 0x3Fu) << 3;
        // A: 128 lanes x 16 elements of 16 bits = 8 columns
        if (!(tmem_ok(d_tmem, n, false) && tmem_ok(a_tmem, 8, false) &&
              sdesc_ok(bdesc, n, (idesc >> 16) & 1u)))
            return;
    }
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The mbarrier receives one arrive when every tcgen05 op this thread issued
// before the commit has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    if (!smem_ok(bar, 8, 8))
        return;
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// ---------------------------------------------------------------------------
// TMEM <-> registers, shape 32x32b: thread t of the warp reads/writes TMEM
// lane (warp's lane quarter base + t); .x32 covers 32 consecutive columns.
// The load and its wait are one asm statement, so no use of the results can
// be scheduled before the data has arrived.

#define FA_R32(a)                                                                              \
    "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]),         \
        "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), \
        "=r"(a[14]), "=r"(a[15]), "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]),           \
        "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]), "=r"(a[25]),           \
        "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31])
#define FA_W32(a)                                                                              \
    "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]),    \
        "r"(a[8]), "r"(a[9]), "r"(a[10]), "r"(a[11]), "r"(a[12]), "r"(a[13]), "r"(a[14]),      \
        "r"(a[15]), "r"(a[16]), "r"(a[17]), "r"(a[18]), "r"(a[19]), "r"(a[20]), "r"(a[21]),    \
        "r"(a[22]), "r"(a[23]), "r"(a[24]), "r"(a[25]), "r"(a[26]), "r"(a[27]), "r"(a[28]),    \
        "r"(a[29]), "r"(a[30]), "r"(a[31])

// 16 consecutive columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    if (!warp_all(tmem_ok(taddr, 16, true))) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            r[i] = 0;
        return;
    }
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    if (!warp_all(tmem_ok(taddr, 32, true))) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            r[i] = 0;
        return;
    }
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : FA_R32(r)
        : "r"(taddr)
        : "memory");
}

// 64 consecutive columns: two .x32 loads, one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&f)[64])
{
    if (!warp_all(tmem_ok(taddr, 64, true))) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
            f[i] = 0;
        return;
    }
    uint32_t(&r)[64] = reinterpret_cast<uint32_t(&)[64]>(f);
    asm volatile(
        "{\n\t.reg .b32 t;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
        "add.u32 t, %64, 32;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [t];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t}"
        : FA_R32(r), FA_R32((r + 32))
        : "r"(taddr)
        : "memory");
}

// 128 consecutive columns: four .x32 loads, one wait.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&f)[128])
{
    if (!warp_all(tmem_ok(taddr, 128, true))) {
#pragma unroll
        for (int i = 0; i < 128; ++i)
            f[i] = 0;
        return;
    }
    uint32_t(&r)[128] = reinterpret_cast<uint32_t(&)[128]>(f);
    asm volatile(
        "{\n\t.reg .b32 t;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%128];\n\t"
        "add.u32 t, %128, 32;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [t];\n\t"
        "add.u32 t, %128, 64;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, "
        "%80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95}, [t];\n\t"
        "add.u32 t, %128, 96;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, "
        "%111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, "
        "%126, %127}, [t];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t}"
        : FA_R32(r), FA_R32((r + 32)), FA_R32((r + 64)), FA_R32((r + 96))
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    if (!warp_all(tmem_ok(taddr, 16, true)))
        return;
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    if (!warp_all(tmem_ok(taddr, 32, true)))
        return;
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        FA_W32(r)
        : "memory");
}

__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[64])
{
    if (!warp_all(tmem_ok(taddr, 64, true)))
        return;
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, "
        "%33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, "
        "%49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};" ::"r"(
            taddr),
        FA_W32(r), FA_W32((r + 32))
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d)
{
    if (!smem_ok(addr, 16, 16))
        return;
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    if (!smem_ok(addr, 16, 16))
        return make_uint4(0, 0, 0, 0);
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Packed fp32 pair arithmetic (one instruction for two lanes of data).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
// Three-input maximum.
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace fa
