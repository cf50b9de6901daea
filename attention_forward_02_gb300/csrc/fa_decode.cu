// fa_decode.cu -- host side of the decoding entry points declared in
// include/fa.h: argument checks, the split-KV plan, TMA descriptors, and the
// two launches (per-chunk partials on the CUDA cores for a few queries, on
// the tensor cores for more; then the combine).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <functional>
#include <mutex>

#include "fa.h"
#include "fa_decode_kernel.cuh"
#include "fa_decode_tc_kernel.cuh"
#include "fa_host.h"

namespace {

using fa_host::EncodeTiledFn;
using fa_host::kMaxDevices;
using fa_host::overlaps;

struct DecState {
    std::once_flag once;
    cudaError_t err = cudaErrorUnknown;
};
DecState g_dec[kMaxDevices];

template <int D, int NQ, typename T>
cudaError_t set_smem_attr()
{
    return cudaFuncSetAttribute(fa::dec::fa_decode_split_kernel<D, NQ, T>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, fa::dec::Cfg<D, NQ>::SMEM_ALLOC);
}

template <int D, typename T>
cudaError_t set_smem_attr_all()
{
    cudaError_t e = set_smem_attr<D, 1, T>();
    if (e == cudaSuccess) e = set_smem_attr<D, 2, T>();
    if (e == cudaSuccess) e = set_smem_attr<D, 4, T>();
    if (e == cudaSuccess) e = set_smem_attr<D, 8, T>();
    if (e == cudaSuccess) e = set_smem_attr<D, 16, T>();
    return e;
}

template <int D, typename T>
cudaError_t set_smem_attr_tc()
{
    return cudaFuncSetAttribute(fa::dectc::fa_decode_tc_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                fa::dectc::Cfg<D>::SMEM_ALLOC);
}

void init_dec(DecState &st)
{
    cudaError_t e = set_smem_attr_tc<32, __half>();
    if (e == cudaSuccess) e = set_smem_attr_tc<64, __half>();
    if (e == cudaSuccess) e = set_smem_attr_tc<96, __half>();
    if (e == cudaSuccess) e = set_smem_attr_tc<128, __half>();
    if (e == cudaSuccess) e = set_smem_attr_tc<32, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr_tc<64, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr_tc<96, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr_tc<128, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr_all<32, __half>();
    if (e == cudaSuccess) e = set_smem_attr_all<64, __half>();
    if (e == cudaSuccess) e = set_smem_attr_all<96, __half>();
    if (e == cudaSuccess) e = set_smem_attr_all<128, __half>();
    if (e == cudaSuccess) e = set_smem_attr_all<32, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr_all<64, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr_all<96, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr_all<128, __nv_bfloat16>();
    st.err = e;
}

long long key_tiles(int Nk) { return (static_cast<long long>(Nk) + fa::dec::kTileKeys - 1) / fa::dec::kTileKeys; }

// Split plan: enough (head, chunk) items for about eight per SM, chunks of
// whole 128-key tiles, every chunk non-empty.
void plan(long long BH, int Nk, int num_sms, int *splits, int *tiles_per_split)
{
    const long long tiles = key_tiles(Nk);
    long long want = (8LL * num_sms + BH - 1) / BH;
    if (want < 1)
        want = 1;
    if (want > tiles)
        want = tiles;
    const long long per = (tiles + want - 1) / want;
    *tiles_per_split = static_cast<int>(per);
    *splits = static_cast<int>((tiles + per - 1) / per);
}

template <int D, int NQ, typename T>
fa_status_t launch_nq(const CUtensorMap &mk, const CUtensorMap &mv, const void *q, void *o, float *lse, float *ws,
                      int BH, int Nq, int Nk, float scale, int causal, int num_sms, cudaStream_t stream)
{
    using namespace fa::dec;
    int splits = 1, per = 1;
    plan(BH, Nk, num_sms, &splits, &per);
    Partials part;
    part.o = ws;
    part.m = ws + static_cast<size_t>(BH) * splits * Nq * D;
    part.l = part.m + static_cast<size_t>(BH) * splits * Nq;
    const int items = BH * splits;
    const unsigned grid = static_cast<unsigned>(items < num_sms ? items : num_sms);
    const float scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    fa_decode_split_kernel<D, NQ, T><<<grid, kThreads, Cfg<D, NQ>::SMEM_ALLOC, stream>>>(
        mk, mv, static_cast<const T *>(q), part, Nq, Nk, splits, per, items, causal, scale_log2);
    const long long rows = static_cast<long long>(BH) * Nq;
    fa_decode_combine_kernel<D, T><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
        part, static_cast<T *>(o), lse, rows, Nq, splits);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

bool use_tensor_cores(int Nq, int d) { return Nq >= 3 || (Nq == 2 && d == 128); }

// Q of the tensor-core path as [BH, Nq, d] 16-bit: one box is 16 query rows
// x 64 columns (rows past Nq and columns past d read as zeros), 128B-swizzled,
// the K-major operand of S^T = K Q^T.
fa_status_t encode_q16_map(EncodeTiledFn encode, CUtensorMap *map, const void *q, int BH, int Nq, int d,
                           fa_dtype_t dtype)
{
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Nq), static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(Nq) * d * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(fa::dectc::kNP), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(map, dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                        const_cast<void *>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// 3-16 queries: both products on the tensor cores.
template <int D, typename T>
fa_status_t launch_tc(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, void *o, float *lse,
                      float *ws, int BH, int Nq, int Nk, float scale, int causal, int num_sms, cudaStream_t stream)
{
    using fa::dec::Partials;
    int splits = 1, per = 1;
    plan(BH, Nk, num_sms, &splits, &per);
    Partials part;
    part.o = ws;
    part.m = ws + static_cast<size_t>(BH) * splits * Nq * D;
    part.l = part.m + static_cast<size_t>(BH) * splits * Nq;
    const int items = BH * splits;
    const unsigned grid = static_cast<unsigned>(items < num_sms ? items : num_sms);
    const float scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    fa::dectc::fa_decode_tc_kernel<D, T><<<grid, fa::dectc::kThreads, fa::dectc::Cfg<D>::SMEM_ALLOC, stream>>>(
        mq, mk, mv, part, Nq, Nk, splits, per, items, causal, scale_log2);
    const long long rows = static_cast<long long>(BH) * Nq;
    fa::dec::fa_decode_combine_kernel<D, T><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
        part, static_cast<T *>(o), lse, rows, Nq, splits);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// The query count rounds up to the next compiled one (1, 2, 4, 8, 16).
template <int D, typename T>
fa_status_t launch(const CUtensorMap &mk, const CUtensorMap &mv, const void *q, void *o, float *lse, float *ws,
                   int BH, int Nq, int Nk, float scale, int causal, int num_sms, cudaStream_t stream)
{
    if (Nq <= 1)
        return launch_nq<D, 1, T>(mk, mv, q, o, lse, ws, BH, Nq, Nk, scale, causal, num_sms, stream);
    if (Nq <= 2)
        return launch_nq<D, 2, T>(mk, mv, q, o, lse, ws, BH, Nq, Nk, scale, causal, num_sms, stream);
    if (Nq <= 4)
        return launch_nq<D, 4, T>(mk, mv, q, o, lse, ws, BH, Nq, Nk, scale, causal, num_sms, stream);
    if (Nq <= 8)
        return launch_nq<D, 8, T>(mk, mv, q, o, lse, ws, BH, Nq, Nk, scale, causal, num_sms, stream);
    return launch_nq<D, 16, T>(mk, mv, q, o, lse, ws, BH, Nq, Nk, scale, causal, num_sms, stream);
}

}  // namespace

namespace fa_host {

fa_status_t take_decode_status(unsigned int *word)
{
    *word = 0;
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(word, fa::g_fa_status, sizeof(*word)) != cudaSuccess)
        return FA_ERR_CUDA;
    if (cudaMemcpyToSymbol(fa::g_fa_status, &zero, sizeof(zero)) != cudaSuccess)
        return FA_ERR_CUDA;
    return FA_OK;
}

}  // namespace fa_host

extern "C" {

size_t fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d)
{
    if (B < 0 || H < 0 || Nq < 1 || Nq > fa::dec::kMaxNq || Nk < Nq || (d != 32 && d != 64 && d != 96 && d != 128))
        return 0;
    // at most one chunk per key tile
    const size_t rows = static_cast<size_t>(B) * H * static_cast<size_t>(key_tiles(Nk)) * Nq;
    return rows * (static_cast<size_t>(d) + 2) * sizeof(float);
}

fa_status_t fa_decode(const void *q, const void *k, const void *v, void *o, float *lse, void *workspace,
                      size_t workspace_bytes, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                      fa_dtype_t dtype, void *stream)
{
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0)
        return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1)
        return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale))
        return FA_ERR_INVALID_ARG;
    if (dtype != FA_FP16 && dtype != FA_BF16)
        return FA_ERR_UNSUPPORTED;
    if (d != 32 && d != 64 && d != 96 && d != 128)
        return FA_ERR_UNSUPPORTED;
    if (scale < 0.f)
        return FA_ERR_UNSUPPORTED;
    if (B == 0 || H == 0)
        return FA_OK;  // empty problem
    if (Nq < 1 || Nq > fa::dec::kMaxNq)
        return FA_ERR_UNSUPPORTED;
    if (Nk < Nq)
        return FA_ERR_INVALID_ARG;
    if (!q || !k || !v || !o || !workspace)
        return FA_ERR_INVALID_ARG;
    const long long BH = static_cast<long long>(B) * H;
    if (BH * key_tiles(Nk) > 0x7fffffffLL)
        return FA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
         reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(workspace)) & 15u)
        return FA_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(lse) & 3u)
        return FA_ERR_MISALIGNED;
    const size_t need = fa_decode_workspace_size(B, H, Nq, Nk, d);
    if (workspace_bytes < need)
        return FA_ERR_INVALID_ARG;
    const size_t qbytes = static_cast<size_t>(BH) * Nq * d * 2;
    const size_t kbytes = static_cast<size_t>(BH) * Nk * d * 2;
    const size_t lbytes = static_cast<size_t>(BH) * Nq * sizeof(float);
    const uintptr_t uo = reinterpret_cast<uintptr_t>(o), uw = reinterpret_cast<uintptr_t>(workspace);
    const uintptr_t ins[3] = {reinterpret_cast<uintptr_t>(q), reinterpret_cast<uintptr_t>(k),
                              reinterpret_cast<uintptr_t>(v)};
    const size_t in_bytes[3] = {qbytes, kbytes, kbytes};
    for (int a = 0; a < 3; ++a)
        if (overlaps(uo, qbytes, ins[a], in_bytes[a]) || overlaps(uw, need, ins[a], in_bytes[a]) ||
            (lse && overlaps(reinterpret_cast<uintptr_t>(lse), lbytes, ins[a], in_bytes[a])))
            return FA_ERR_INVALID_ARG;
    if (overlaps(uo, qbytes, uw, need) ||
        (lse && (overlaps(reinterpret_cast<uintptr_t>(lse), lbytes, uo, qbytes) ||
                 overlaps(reinterpret_cast<uintptr_t>(lse), lbytes, uw, need))))
        return FA_ERR_INVALID_ARG;

    EncodeTiledFn encode = nullptr;
    int sms = 0;
    fa_status_t s = fa_host::encoder(&encode, &sms);
    if (s != FA_OK)
        return s;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FA_ERR_CUDA;
    DecState &st = g_dec[dev];
    std::call_once(st.once, init_dec, std::ref(st));
    if (st.err != cudaSuccess)
        return FA_ERR_CUDA;
    const int bh = static_cast<int>(BH);
    CUtensorMap mk, mv;
    if ((s = fa_host::encode_qkv_map(encode, &mk, k, bh, Nk, d, dtype)) != FA_OK) return s;
    if ((s = fa_host::encode_qkv_map(encode, &mv, v, bh, Nk, d, dtype)) != FA_OK) return s;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    float *ws = static_cast<float *>(workspace);
    // The tensor-core kernel from 3 queries on, and from 2 at d = 128
    // (measured: with one query, and with two at d < 128, the CUDA-core
    // kernel is as fast or faster; beyond, its query loops grow with Nq)
    if (use_tensor_cores(Nq, d)) {
        CUtensorMap mq;
        if ((s = encode_q16_map(encode, &mq, q, bh, Nq, d, dtype)) != FA_OK)
            return s;
#define FA_DEC_TC(DD)                                                                                      \
    if (d == DD)                                                                                           \
        return dtype == FA_FP16                                                                            \
                   ? launch_tc<DD, __half>(mq, mk, mv, o, lse, ws, bh, Nq, Nk, scale, causal, sms, cs)     \
                   : launch_tc<DD, __nv_bfloat16>(mq, mk, mv, o, lse, ws, bh, Nq, Nk, scale, causal, sms, cs);
        FA_DEC_TC(32)
        FA_DEC_TC(64)
        FA_DEC_TC(96)
        FA_DEC_TC(128)
#undef FA_DEC_TC
        return FA_ERR_UNSUPPORTED;
    }
#define FA_DEC_D(DD, TT)                                                                                  \
    if (d == DD)                                                                                          \
        return launch<DD, TT>(mk, mv, q, o, lse, ws, bh, Nq, Nk, scale, causal, sms, cs);
    if (dtype == FA_FP16) {
        FA_DEC_D(32, __half)
        FA_DEC_D(64, __half)
        FA_DEC_D(96, __half)
        FA_DEC_D(128, __half)
    } else {
        FA_DEC_D(32, __nv_bfloat16)
        FA_DEC_D(64, __nv_bfloat16)
        FA_DEC_D(96, __nv_bfloat16)
        FA_DEC_D(128, __nv_bfloat16)
    }
#undef FA_DEC_D
    return FA_ERR_UNSUPPORTED;
}

}  // extern "C"
