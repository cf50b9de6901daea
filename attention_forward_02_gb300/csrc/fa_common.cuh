// fa_common.cuh -- device pieces shared by the forward and backward kernels:
// bounded mbarrier waits, the 16-bit dtype traits and
// the 128B-swizzle tile addressing.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "sm100_ptx.cuh"

namespace fa {

constexpr long long kWaitLimitCycles = 1ll << 31;  // about one second at 2 GHz
constexpr int kSwAtomBytes = 128 * 128;             // [128 rows x 64 cols] 16-bit swizzle block

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
    static __device__ __forceinline__ float2 unpack(uint32_t w)
    {
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
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
    static __device__ __forceinline__ float2 unpack(uint32_t w)
    {
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
    }
};

// Bounded wait.  Returns false if the CTA is aborting or the limit expired
// (then the abort flag and the device status word are set).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             long long limit_cycles = kWaitLimitCycles)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (clock64() - t0 > limit_cycles) {
            *abort_flag = 1;
            atomicOr(&g_fa_status, kStatusTimeout);
            return false;
        }
    }
}

// Warp-wide bounded wait (every lane of the warp calls it, on the same
// barrier and parity): one try_wait and one vote when the phase has already
// completed, the bounded loop otherwise.  Every lane gets the same result.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag)
{
    if (__builtin_expect(__all_sync(0xffffffffu, mbar_try_wait(bar, parity)), 1))
        return true;
    return __all_sync(0xffffffffu, wait_bounded(bar, parity, abort_flag));
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

}  // namespace fa
