// fa_host.h -- host-side helpers shared by the library's translation units
// (forward entry points in fa_fwd.cu, backward in fa_bwd.cu, decoding in
// fa_decode.cu).  Internal: not
// part of the C ABI (the library is built with hidden visibility).
#pragma once

#include <cuda.h>

#include <cstddef>
#include <cstdint>

#include "fa.h"

namespace fa_host {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;

inline bool overlaps(uintptr_t a, size_t na, uintptr_t b, size_t nb) { return a < b + nb && b < a + na; }

// The current device's TMA encoder and SM count (initialised once per device;
// fails with FA_ERR_UNSUPPORTED on anything but sm_103).
fa_status_t encoder(EncodeTiledFn *fn, int *num_sms);

// 3-D view [BH, N, d] of a contiguous [B, H, N, d] 16-bit tensor; box = 64
// columns x 128 rows x 1 head, SWIZZLE_128B, rows past N read as zeros (and
// are not written by stores).
fa_status_t encode_qkv_map(EncodeTiledFn encode, CUtensorMap *map, const void *ptr, int BH, int N,
                           int d, fa_dtype_t dtype);

// Argument checks shared by the forward entry points (no CUDA calls).  Sets
// *empty for a problem with nothing to compute.
fa_status_t check_args(const void *q, const void *k, const void *v, const void *o, const float *lse,
                       int B, int H, int N, int d, float scale, int causal, fa_dtype_t dtype,
                       bool *empty);

// Read and clear the backward / decoding units' device status words (bit 0:
// a bounded wait expired); 0 when nothing was recorded.
fa_status_t take_bwd_status(unsigned int *word);
fa_status_t take_decode_status(unsigned int *word);

}  // namespace fa_host
