// fa_bwd.cu -- host side of the backward entry points declared in
// include/fa.h: argument checks, workspace layout, TMA descriptors, and the
// three launches (row terms, main kernel, dQ rounding).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <functional>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "fa.h"
#include "fa_bwd_kernel.cuh"
#include "fa_host.h"

namespace {

using fa_host::EncodeTiledFn;
using fa_host::kMaxDevices;
using fa_host::overlaps;

struct BwdState {
    std::once_flag once;
    cudaError_t err = cudaErrorUnknown;
};
BwdState g_bwd[kMaxDevices];

template <int D, bool CAUSAL, typename T>
cudaError_t set_smem_attr()
{
    return cudaFuncSetAttribute(fa::bwd::fa_bwd_kernel<D, CAUSAL, T>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, fa::bwd::Cfg<D>::SMEM_ALLOC);
}

void init_bwd(BwdState &st)
{
    cudaError_t e = cudaSuccess;
#define FA_BWD_ATTR(DD)                                                                                   \
    if (e == cudaSuccess) e = set_smem_attr<DD, false, __half>();                                         \
    if (e == cudaSuccess) e = set_smem_attr<DD, true, __half>();                                          \
    if (e == cudaSuccess) e = set_smem_attr<DD, false, __nv_bfloat16>();                                  \
    if (e == cudaSuccess) e = set_smem_attr<DD, true, __nv_bfloat16>();
    FA_BWD_ATTR(32)
    FA_BWD_ATTR(64)
    FA_BWD_ATTR(96)
    FA_BWD_ATTR(128)
#undef FA_BWD_ATTR
    st.err = e;
}

long long padded_rows(int N) { return (static_cast<long long>(N) + fa::bwd::kBlk - 1) / fa::bwd::kBlk * fa::bwd::kBlk; }

// fp32 accumulator [BH, Npad, d], in the layout the dQ warps stage: box
// 32 columns (128 bytes) x 128 rows x 1 with SWIZZLE_128B for d <= 64, box
// 16 columns (64 bytes) x 128 rows x 1 with SWIZZLE_64B for d > 64.
fa_status_t encode_acc_map(EncodeTiledFn encode, CUtensorMap *map, float *ptr, int BH, long long Npad, int d)
{
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Npad),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                                   static_cast<cuuint64_t>(Npad) * static_cast<cuuint64_t>(d) * 4};
    const bool narrow = d > 64;
    const cuuint32_t box[3] = {narrow ? 16u : 32u, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        narrow ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

struct Maps {
    CUtensorMap q, k, v, dout, dk, dv, acc;
};

// Longest per-CTA load when the causal items, heads in groups of hg and the
// heaviest key blocks first inside each group, are dealt out as the kernel
// deals them (round r: items [r G, r G + G), every other round in reverse CTA
// order).  An item costs its query blocks plus half a block of set-up.
double causal_makespan(int BH, int nb, int G, int hg, std::vector<double> &load)
{
    load.assign(static_cast<size_t>(G), 0.0);
    const long long W = static_cast<long long>(BH) * nb;
    for (long long w = 0; w < W; ++w) {
        const long long r = w / G, c = w % G;
        const long long cta = (r & 1) ? G - 1 - c : c;
        const long long g = w / (static_cast<long long>(hg) * nb);
        const long long h0 = g * hg;
        const long long gs = std::min<long long>(hg, BH - h0);
        const long long n = (w - h0 * nb) / gs;
        load[static_cast<size_t>(cta)] += static_cast<double>(nb - n) + 0.5;
    }
    return *std::max_element(load.begin(), load.end());
}

// Head-group size of the causal walk.  Heaviest-first across all heads keeps
// the CTAs balanced but has every head's Q, dO and fp32 dQ accumulator in
// flight at once; when those exceed what L2 keeps, groups of a few heads cut
// the re-reads from DRAM (base causal shape: 771 MB of DRAM traffic per
// launch across all 128 heads).  Among the group sizes whose simulated
// makespan is within 3 % of the best, the smallest is taken.  Cached per
// shape.
int causal_head_group(int BH, int nb, int G, int d)
{
    const double head_bytes = static_cast<double>(nb) * 128.0 * d * (2 + 2 + 4);  // Q, dO, accumulator
    if (BH <= 1 || head_bytes * BH <= 64.0 * (1 << 20))
        return BH;
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int>, int> cache;
    const auto key = std::make_tuple(BH, nb, G, d);
    {
        std::lock_guard<std::mutex> lock(mu);
        const auto it = cache.find(key);
        if (it != cache.end())
            return it->second;
    }
    std::vector<double> load;
    // candidates: every group of one to eight rounds of items, and all heads
    std::vector<int> cand{BH};
    for (int hg = 1; hg < BH; ++hg) {
        const long long items = static_cast<long long>(hg) * nb;
        if (items >= G && items <= 8LL * G && head_bytes * hg <= 64.0 * (1 << 20))
            cand.push_back(hg);
    }
    std::vector<double> span(cand.size());
    double best = 0.0;
    for (size_t i = 0; i < cand.size(); ++i) {
        span[i] = causal_makespan(BH, nb, G, cand[i], load);
        best = i == 0 ? span[i] : std::min(best, span[i]);
    }
    int hg = BH;
    for (size_t i = 0; i < cand.size(); ++i)
        if (span[i] <= 1.03 * best && cand[i] < hg)
            hg = cand[i];
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = hg;
    return hg;
}

template <int D, bool CAUSAL, typename T>
fa_status_t launch(const Maps &mp, const void *o, const float *lse, const void *dout, void *dq, float *acc,
                   float *lse2, float *dvec, int BH, int N, float scale, int num_sms, cudaStream_t stream)
{
    using namespace fa::bwd;
    const long long Npad = padded_rows(N);
    const int nb = static_cast<int>(Npad / kBlk);
    const long long rows = static_cast<long long>(BH) * Npad;
    {
        const long long threads = rows * (D <= 32 ? 4 : D <= 64 ? 8 : 16);
        const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
        fa_bwd_prep_kernel<D, T><<<grid, 256, 0, stream>>>(static_cast<const T *>(o),
                                                            static_cast<const T *>(dout), lse, lse2, dvec,
                                                            acc, N, static_cast<int>(Npad), rows);
    }
    const float scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    // persistent: one CTA per SM (shared memory and TMEM allow no more), each
    // walking its share of the BH * nb (head, key block) items
    const long long items = static_cast<long long>(BH) * nb;
    const unsigned grid = static_cast<unsigned>(items < num_sms ? items : num_sms);
    const int hg = CAUSAL ? causal_head_group(BH, nb, static_cast<int>(grid), D) : BH;
    fa_bwd_kernel<D, CAUSAL, T><<<grid, kThreads, Cfg<D>::SMEM_ALLOC, stream>>>(
        mp.q, mp.k, mp.v, mp.dout, mp.dk, mp.dv, mp.acc, lse2, dvec, N, static_cast<int>(Npad), BH, nb, hg,
        scale, scale_log2);
    {
        const long long chunks = static_cast<long long>(BH) * N * (D / 8);
        long long blocks = (chunks + 255) / 256;
        if (blocks > 65535LL * 16)
            blocks = 65535LL * 16;
        fa_bwd_dq_kernel<D, T><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(acc, static_cast<T *>(dq), N,
                                                                                 static_cast<int>(Npad), chunks,
                                                                                 scale);
    }
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

namespace fa_host {

fa_status_t take_bwd_status(unsigned int *word)
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

size_t fa_bwd_workspace_size(int B, int H, int N, int d)
{
    if (B < 0 || H < 0 || N < 0 || (d != 32 && d != 64 && d != 96 && d != 128))
        return 0;
    const size_t rows = static_cast<size_t>(B) * H * static_cast<size_t>(padded_rows(N));
    return rows * (static_cast<size_t>(d) + 2) * sizeof(float);
}

fa_status_t fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                   const void *dout, void *dq, void *dk, void *dv, void *workspace, size_t workspace_bytes,
                   int B, int H, int N, int d, float scale, int causal, fa_dtype_t dtype, void *stream)
{
    bool empty = false;
    // q, k, v, o as in the forward (o is an input here; the overlap check
    // against q, k, v still applies: they are distinct tensors)
    fa_status_t s = fa_host::check_args(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, &empty);
    if (s != FA_OK || empty)
        return s;
    if (!lse || !dout || !dq || !dk || !dv)
        return FA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) | reinterpret_cast<uintptr_t>(dk) |
         reinterpret_cast<uintptr_t>(dv) | reinterpret_cast<uintptr_t>(workspace)) & 15u)
        return FA_ERR_MISALIGNED;
    const size_t need = fa_bwd_workspace_size(B, H, N, d);
    if (!workspace || workspace_bytes < need)
        return FA_ERR_INVALID_ARG;
    const long long BH = static_cast<long long>(B) * H;
    const long long Npad = padded_rows(N);
    if (BH * (Npad / fa::bwd::kBlk) > 0x7fffffffLL - 65536)
        return FA_ERR_UNSUPPORTED;  // item numbers (plus one round of CTAs) are 32-bit
    const size_t bytes = static_cast<size_t>(BH) * N * d * 2;
    const size_t lbytes = static_cast<size_t>(BH) * N * sizeof(float);
    const uintptr_t outs[4] = {reinterpret_cast<uintptr_t>(dq), reinterpret_cast<uintptr_t>(dk),
                               reinterpret_cast<uintptr_t>(dv), reinterpret_cast<uintptr_t>(workspace)};
    const size_t out_bytes[4] = {bytes, bytes, bytes, need};
    const uintptr_t ins[6] = {reinterpret_cast<uintptr_t>(q), reinterpret_cast<uintptr_t>(k),
                              reinterpret_cast<uintptr_t>(v), reinterpret_cast<uintptr_t>(o),
                              reinterpret_cast<uintptr_t>(dout), reinterpret_cast<uintptr_t>(lse)};
    const size_t in_bytes[6] = {bytes, bytes, bytes, bytes, bytes, lbytes};
    for (int a = 0; a < 4; ++a) {
        for (int b = a + 1; b < 4; ++b)
            if (overlaps(outs[a], out_bytes[a], outs[b], out_bytes[b]))
                return FA_ERR_INVALID_ARG;
        for (int b = 0; b < 6; ++b)
            if (overlaps(outs[a], out_bytes[a], ins[b], in_bytes[b]))
                return FA_ERR_INVALID_ARG;
    }

    EncodeTiledFn encode = nullptr;
    int num_sms = 0;
    if ((s = fa_host::encoder(&encode, &num_sms)) != FA_OK)
        return s;
    if (num_sms < 1)
        return FA_ERR_CUDA;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FA_ERR_CUDA;
    BwdState &st = g_bwd[dev];
    std::call_once(st.once, init_bwd, std::ref(st));
    if (st.err != cudaSuccess)
        return FA_ERR_CUDA;

    const int bh = static_cast<int>(BH);
    float *acc = static_cast<float *>(workspace);
    float *lse2 = acc + static_cast<size_t>(BH) * Npad * d;
    float *dvec = lse2 + static_cast<size_t>(BH) * Npad;
    Maps mp;
    if ((s = fa_host::encode_qkv_map(encode, &mp.q, q, bh, N, d, dtype)) != FA_OK) return s;
    if ((s = fa_host::encode_qkv_map(encode, &mp.k, k, bh, N, d, dtype)) != FA_OK) return s;
    if ((s = fa_host::encode_qkv_map(encode, &mp.v, v, bh, N, d, dtype)) != FA_OK) return s;
    if ((s = fa_host::encode_qkv_map(encode, &mp.dout, dout, bh, N, d, dtype)) != FA_OK) return s;
    if ((s = fa_host::encode_qkv_map(encode, &mp.dk, dk, bh, N, d, dtype)) != FA_OK) return s;
    if ((s = fa_host::encode_qkv_map(encode, &mp.dv, dv, bh, N, d, dtype)) != FA_OK) return s;
    if ((s = encode_acc_map(encode, &mp.acc, acc, bh, Npad, d)) != FA_OK) return s;

    cudaStream_t cs = static_cast<cudaStream_t>(stream);
#define FA_BWD_ARGS mp, o, lse, dout, dq, acc, lse2, dvec, bh, N, scale, num_sms, cs
#define FA_BWD_D(DD, TT)                                                                                  \
    if (d == DD)                                                                                          \
        return causal ? launch<DD, true, TT>(FA_BWD_ARGS) : launch<DD, false, TT>(FA_BWD_ARGS);
    if (dtype == FA_FP16) {
        FA_BWD_D(32, __half)
        FA_BWD_D(64, __half)
        FA_BWD_D(96, __half)
        FA_BWD_D(128, __half)
    } else {
        FA_BWD_D(32, __nv_bfloat16)
        FA_BWD_D(64, __nv_bfloat16)
        FA_BWD_D(96, __nv_bfloat16)
        FA_BWD_D(128, __nv_bfloat16)
    }
    return FA_ERR_UNSUPPORTED;
#undef FA_BWD_D
#undef FA_BWD_ARGS
}

}  // extern "C"
