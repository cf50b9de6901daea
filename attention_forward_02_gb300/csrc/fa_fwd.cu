// fa_fwd.cu -- host side of the C ABI declared in include/fa.h: argument
// checks, TMA descriptor encoding, and the launch of the sm_103a kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>

#include "fa.h"
#include "fa1_fwd_kernel.cuh"
#include "fa_fwd_kernel.cuh"
#include "fa_host.h"

using fa_host::EncodeTiledFn;
using fa_host::kMaxDevices;
using fa_host::overlaps;

namespace {

struct DeviceState {
    std::once_flag once;
    fa_status_t init_status = FA_ERR_CUDA;
    EncodeTiledFn encode = nullptr;
    int num_sms = 0;
};
DeviceState g_dev[kMaxDevices];

template <int D, bool CAUSAL, typename T>
cudaError_t set_smem_attr()
{
    return cudaFuncSetAttribute(fa::fa_fwd_kernel<D, CAUSAL, T>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, fa::KCfg<D>::SMEM_ALLOC);
}

template <int D, bool CAUSAL, typename T>
cudaError_t set_smem_attr_fa1()
{
    return cudaFuncSetAttribute(fa::fa1::fa1_fwd_kernel<D, CAUSAL, T>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                fa::fa1::Cfg<D>::SMEM_ALLOC);
}

void init_device(int dev, DeviceState &st)
{
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
        st.init_status = FA_ERR_CUDA;
        return;
    }
    // tcgen05 / TMEM kernels are built for sm_103a only.
    if (prop.major != 10 || prop.minor != 3) {
        st.init_status = FA_ERR_UNSUPPORTED;
        return;
    }
    st.num_sms = prop.multiProcessorCount;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
        st.init_status = FA_ERR_CUDA;
        return;
    }
    st.encode = reinterpret_cast<EncodeTiledFn>(fn);
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = set_smem_attr<32, false, __half>();
    if (e == cudaSuccess) e = set_smem_attr<32, true, __half>();
    if (e == cudaSuccess) e = set_smem_attr<96, false, __half>();
    if (e == cudaSuccess) e = set_smem_attr<96, true, __half>();
    if (e == cudaSuccess) e = set_smem_attr<32, false, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr<32, true, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr<96, false, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr<96, true, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr<64, false, __half>();
    if (e == cudaSuccess) e = set_smem_attr<64, true, __half>();
    if (e == cudaSuccess) e = set_smem_attr<128, false, __half>();
    if (e == cudaSuccess) e = set_smem_attr<128, true, __half>();
    if (e == cudaSuccess) e = set_smem_attr<64, false, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr<64, true, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr<128, false, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr<128, true, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr_fa1<32, false, __half>();
    if (e == cudaSuccess) e = set_smem_attr_fa1<32, true, __half>();
    if (e == cudaSuccess) e = set_smem_attr_fa1<96, false, __half>();
    if (e == cudaSuccess) e = set_smem_attr_fa1<96, true, __half>();
    if (e == cudaSuccess) e = set_smem_attr_fa1<32, false, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr_fa1<32, true, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr_fa1<96, false, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr_fa1<96, true, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr_fa1<64, false, __half>();
    if (e == cudaSuccess) e = set_smem_attr_fa1<64, true, __half>();
    if (e == cudaSuccess) e = set_smem_attr_fa1<128, false, __half>();
    if (e == cudaSuccess) e = set_smem_attr_fa1<128, true, __half>();
    if (e == cudaSuccess) e = set_smem_attr_fa1<64, false, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr_fa1<64, true, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr_fa1<128, false, __nv_bfloat16>();
    if (e == cudaSuccess) e = set_smem_attr_fa1<128, true, __nv_bfloat16>();
    st.init_status = (e == cudaSuccess) ? FA_OK : FA_ERR_CUDA;
}



// Persistent launch: one CTA per SM (TMEM and shared memory allow one), each
// walking its share of the (batch*head, 256-row Q block) work items.
template <int D, bool CAUSAL, typename T>
fa_status_t launch(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mo,
                   void *o, float *lse, int BH, int N, float scale, int num_sms, cudaStream_t stream)
{
    const int num_q_blocks = (N + fa::kBM - 1) / fa::kBM;
    const long long items = static_cast<long long>(BH) * num_q_blocks;
    const float scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    const unsigned grid = static_cast<unsigned>(items < num_sms ? items : num_sms);
    fa::fa_fwd_kernel<D, CAUSAL, T><<<grid, fa::kNumThreads, fa::KCfg<D>::SMEM_ALLOC, stream>>>(
        mq, mk, mv, mo, static_cast<T *>(o), lse, N, BH, num_q_blocks, scale, scale_log2);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Head-dim and causal dispatch of the FA2 launch.
template <typename T>
fa_status_t launch_d(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mo,
                     void *o, float *lse, int BH, int N, int d, float scale, int causal, int num_sms,
                     cudaStream_t stream)
{
#define FA_LAUNCH_D(DD)                                                                                  \
    if (d == DD)                                                                                         \
        return causal ? launch<DD, true, T>(mq, mk, mv, mo, o, lse, BH, N, scale, num_sms, stream)       \
                      : launch<DD, false, T>(mq, mk, mv, mo, o, lse, BH, N, scale, num_sms, stream);
    FA_LAUNCH_D(32)
    FA_LAUNCH_D(64)
    FA_LAUNCH_D(96)
    FA_LAUNCH_D(128)
#undef FA_LAUNCH_D
    return FA_ERR_UNSUPPORTED;
}

template <int D, bool CAUSAL, typename T>
fa_status_t launch_fa1(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, void *o,
                       float *lse, float *ws, int BH, int N, float scale, cudaStream_t stream);

// Head-dim, causal and dtype dispatch of the FA1 launch.
fa_status_t launch_fa1_any(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, void *o,
                           float *lse, float *ws, int BH, int N, int d, float scale, int causal, fa_dtype_t dtype,
                           cudaStream_t stream)
{
#define FA1_D(DD, TT)                                                                                     \
    if (d == DD)                                                                                          \
        return causal ? launch_fa1<DD, true, TT>(mq, mk, mv, o, lse, ws, BH, N, scale, stream)            \
                      : launch_fa1<DD, false, TT>(mq, mk, mv, o, lse, ws, BH, N, scale, stream);
    if (dtype == FA_FP16) {
        FA1_D(32, __half)
        FA1_D(64, __half)
        FA1_D(96, __half)
        FA1_D(128, __half)
    } else {
        FA1_D(32, __nv_bfloat16)
        FA1_D(64, __nv_bfloat16)
        FA1_D(96, __nv_bfloat16)
        FA1_D(128, __nv_bfloat16)
    }
#undef FA1_D
    return FA_ERR_UNSUPPORTED;
}

template <int D, bool CAUSAL, typename T>
fa_status_t launch_fa1(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, void *o,
                       float *lse, float *ws, int BH, int N, float scale, cudaStream_t stream)
{
    const float scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    fa::fa1::fa1_fwd_kernel<D, CAUSAL, T>
        <<<static_cast<unsigned>(BH), fa::fa1::kThreads, fa::fa1::Cfg<D>::SMEM_ALLOC, stream>>>(
            mq, mk, mv, static_cast<T *>(o), lse, ws, N, scale, scale_log2);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}



}  // namespace

namespace fa_host {

fa_status_t device_state(DeviceState **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FA_ERR_CUDA;
    DeviceState &st = g_dev[dev];
    std::call_once(st.once, init_device, dev, std::ref(st));
    *out = &st;
    return st.init_status;
}

// 3-D view [BH, N, d] of a contiguous [B, H, N, d] tensor; box = 64 columns
// (128 bytes, one swizzle span) x 128 rows x 1 head, SWIZZLE_128B, rows past N
// read as zeros.
fa_status_t encode_qkv_map(EncodeTiledFn encode, CUtensorMap *map, const void *ptr, int BH, int N,
                           int d, fa_dtype_t dtype)
{
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                   static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(map,
                        dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        3, const_cast<void *>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// Checks shared by the entry points; nothing here calls CUDA.  Sets *empty for
// a problem with nothing to compute.
fa_status_t check_args(const void *q, const void *k, const void *v, const void *o, const float *lse,
                       int B, int H, int N, int d, float scale, int causal, fa_dtype_t dtype,
                       bool *empty)
{
    *empty = false;
    if (B < 0 || H < 0 || N < 0)
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
    if (B == 0 || H == 0 || N == 0) {
        *empty = true;  // empty problem
        return FA_OK;
    }
    if (!q || !k || !v || !o)
        return FA_ERR_INVALID_ARG;
    const long long BH = static_cast<long long>(B) * H;
    if (BH > 0x7fffffffLL)
        return FA_ERR_UNSUPPORTED;
    if (BH * ((N + fa::kBM - 1) / fa::kBM) > 0x7fffffffLL)
        return FA_ERR_UNSUPPORTED;  // grid.x limit
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
         reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o)) & 15u)
        return FA_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(lse) & 3u)
        return FA_ERR_MISALIGNED;
    const size_t bytes = static_cast<size_t>(BH) * N * d * 2;
    const uintptr_t uo = reinterpret_cast<uintptr_t>(o);
    if (overlaps(uo, bytes, reinterpret_cast<uintptr_t>(q), bytes) ||
        overlaps(uo, bytes, reinterpret_cast<uintptr_t>(k), bytes) ||
        overlaps(uo, bytes, reinterpret_cast<uintptr_t>(v), bytes))
        return FA_ERR_INVALID_ARG;
    if (lse) {
        const size_t lbytes = static_cast<size_t>(BH) * N * sizeof(float);
        const uintptr_t ul = reinterpret_cast<uintptr_t>(lse);
        if (overlaps(ul, lbytes, uo, bytes) || overlaps(ul, lbytes, reinterpret_cast<uintptr_t>(q), bytes) ||
            overlaps(ul, lbytes, reinterpret_cast<uintptr_t>(k), bytes) ||
            overlaps(ul, lbytes, reinterpret_cast<uintptr_t>(v), bytes))
            return FA_ERR_INVALID_ARG;
    }
    return FA_OK;
}

fa_status_t encoder(EncodeTiledFn *fn, int *num_sms)
{
    DeviceState *st = nullptr;
    fa_status_t s = device_state(&st);
    if (s != FA_OK)
        return s;
    *fn = st->encode;
    if (num_sms)
        *num_sms = st->num_sms;
    return FA_OK;
}

}  // namespace fa_host

namespace {

using fa_host::check_args;
using fa_host::device_state;
using fa_host::encode_qkv_map;

// Device state plus the three TMA descriptors of Q, K, V.
fa_status_t prepare(const void *q, const void *k, const void *v, int BH, int N, int d,
                    fa_dtype_t dtype, CUtensorMap *mq, CUtensorMap *mk, CUtensorMap *mv,
                    int *num_sms = nullptr)
{
    DeviceState *st = nullptr;
    fa_status_t s = device_state(&st);
    if (s != FA_OK)
        return s;
    if (num_sms)
        *num_sms = st->num_sms;
    if ((s = encode_qkv_map(st->encode, mq, q, BH, N, d, dtype)) != FA_OK) return s;
    if ((s = encode_qkv_map(st->encode, mk, k, BH, N, d, dtype)) != FA_OK) return s;
    return encode_qkv_map(st->encode, mv, v, BH, N, d, dtype);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of fa1_fwd: its scratch lives in this fixed device
// array instead of a caller workspace.  Every device that loads the library
// holds the array until the process exits.
constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB
static __device__ __align__(256) float g_fa1_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

struct NoAllocState {
    std::once_flag once;
    cudaError_t err = cudaErrorUnknown;
    float *scratch = nullptr;  // device address of g_fa1_noalloc_scratch
};
NoAllocState g_noalloc[kMaxDevices];

// Once per device, with that device current: look up the array's device
// address (its name in host code is only a host-side stand-in).
void init_noalloc(NoAllocState &st)
{
    void *ptr = nullptr;
    st.err = cudaGetSymbolAddress(&ptr, g_fa1_noalloc_scratch);
    st.scratch = (st.err == cudaSuccess) ? static_cast<float *>(ptr) : nullptr;
}

}  // namespace

extern "C" {

fa_status_t fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                   int N, int d, float scale, int causal, fa_dtype_t dtype, void *stream)
{
    bool empty = false;
    fa_status_t s = check_args(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, &empty);
    if (s != FA_OK || empty)
        return s;
    const int bh = B * H;
    CUtensorMap mq, mk, mv, mo;
    int sms = 0;
    if ((s = prepare(q, k, v, bh, N, d, dtype, &mq, &mk, &mv, &sms)) != FA_OK)
        return s;
    // O has Q's layout; the epilogue writes it through a map of the same shape
    EncodeTiledFn enc = nullptr;
    if ((s = fa_host::encoder(&enc, nullptr)) != FA_OK || (s = encode_qkv_map(enc, &mo, o, bh, N, d, dtype)) != FA_OK)
        return s;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    return dtype == FA_FP16 ? launch_d<__half>(mq, mk, mv, mo, o, lse, bh, N, d, scale, causal, sms, cs)
                            : launch_d<__nv_bfloat16>(mq, mk, mv, mo, o, lse, bh, N, d, scale, causal, sms, cs);
}

size_t fa1_fwd_workspace_size(int B, int H, int N, int d)
{
    if (B < 0 || H < 0 || N < 0 || (d != 32 && d != 64 && d != 96 && d != 128))
        return 0;
    return fa::fa1::workspace_floats(static_cast<long long>(B) * H, N, d) * sizeof(float);
}

fa_status_t fa1_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                    void *workspace, size_t workspace_bytes, int B, int H, int N, int d,
                    float scale, int causal, fa_dtype_t dtype, void *stream)
{
    bool empty = false;
    fa_status_t s = check_args(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, &empty);
    if (s != FA_OK || empty)
        return s;
    const size_t need = fa1_fwd_workspace_size(B, H, N, d);
    if (!workspace || workspace_bytes < need)
        return FA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 15u)
        return FA_ERR_MISALIGNED;
    const size_t bytes = static_cast<size_t>(B) * H * N * d * 2;
    const uintptr_t uw = reinterpret_cast<uintptr_t>(workspace);
    if (overlaps(uw, need, reinterpret_cast<uintptr_t>(q), bytes) ||
        overlaps(uw, need, reinterpret_cast<uintptr_t>(k), bytes) ||
        overlaps(uw, need, reinterpret_cast<uintptr_t>(v), bytes) ||
        overlaps(uw, need, reinterpret_cast<uintptr_t>(o), bytes) ||
        (lse && overlaps(uw, need, reinterpret_cast<uintptr_t>(lse),
                         static_cast<size_t>(B) * H * N * sizeof(float))))
        return FA_ERR_INVALID_ARG;
    const int bh = B * H;
    CUtensorMap mq, mk, mv;
    if ((s = prepare(q, k, v, bh, N, d, dtype, &mq, &mk, &mv)) != FA_OK)
        return s;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    float *ws = static_cast<float *>(workspace);
    return launch_fa1_any(mq, mk, mv, o, lse, ws, bh, N, d, scale, causal, dtype, cs);
}

fa_status_t fa1_fwd_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                            int B, int H, int N, int d, float scale, int causal, fa_dtype_t dtype,
                            void *stream)
{
    bool empty = false;
    fa_status_t s = check_args(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, &empty);
    if (s != FA_OK || empty)
        return s;
    if (fa1_fwd_workspace_size(B, H, N, d) > kNoAllocScratchBytes)
        return FA_ERR_UNSUPPORTED;  // problem needs more scratch than the fixed array holds
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FA_ERR_CUDA;
    NoAllocState &na = g_noalloc[dev];
    std::call_once(na.once, init_noalloc, std::ref(na));
    if (na.err != cudaSuccess || na.scratch == nullptr)
        return FA_ERR_CUDA;
    const int bh = B * H;
    CUtensorMap mq, mk, mv;
    if ((s = prepare(q, k, v, bh, N, d, dtype, &mq, &mk, &mv)) != FA_OK)
        return s;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    float *ws = na.scratch;
    return launch_fa1_any(mq, mk, mv, o, lse, ws, bh, N, d, scale, causal, dtype, cs);
}

fa_status_t fa_last_device_status(void *stream)
{
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(cs) != cudaSuccess)
        return FA_ERR_CUDA;
    unsigned int word = 0;
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(&word, fa::g_fa_status, sizeof(word)) != cudaSuccess)
        return FA_ERR_CUDA;
    if (cudaMemcpyToSymbol(fa::g_fa_status, &zero, sizeof(zero)) != cudaSuccess)
        return FA_ERR_CUDA;
    unsigned int bwd_word = 0, dec_word = 0;
    if (fa_host::take_bwd_status(&bwd_word) != FA_OK || fa_host::take_decode_status(&dec_word) != FA_OK)
        return FA_ERR_CUDA;
    word |= bwd_word | dec_word;
    if (word & fa::kStatusSelftest)
        return FA_ERR_CUDA;  // a self-test did not behave as required
    if (word & fa::kStatusBounds)
        return FA_ERR_BOUNDS;
    return (word & fa::kStatusTimeout) ? FA_ERR_TIMEOUT : FA_OK;
}

fa_status_t fa_selftest_wait_timeout(int limit_us, void *stream)
{
    if (limit_us < 1 || limit_us > 1000000)
        return FA_ERR_INVALID_ARG;
    int dev = -1;
    int clock_khz = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&clock_khz, cudaDevAttrClockRate, dev) != cudaSuccess)
        return FA_ERR_CUDA;
    if (clock_khz <= 0)
        clock_khz = 2000000;
    const long long cycles = static_cast<long long>(limit_us) * (clock_khz / 1000);
    fa::fa_selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(cycles);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t fa_selftest_bounds_check(void *stream)
{
    fa::fa_selftest_bounds_kernel<<<1, 128, 1024, static_cast<cudaStream_t>(stream)>>>();
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_checked_build(void) { return fa::kBoundsCheck ? 1 : 0; }

const char *fa_status_str(fa_status_t status)
{
    switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    case FA_ERR_BOUNDS: return "FA_ERR_BOUNDS";
    }
    return "FA_ERR_UNKNOWN";
}

int fa_abi_version(void) { return FA_ABI_VERSION; }

}  // extern "C"
