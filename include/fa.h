/*
 * fa.h -- C ABI of the GB300 (sm_103a) attention library.
 *
 * The main operation: the FlashAttention-2 style tiled attention forward
 *
 *     O = softmax(Q K^T * scale) V,     LSE = log(sum_j exp(scale * q_i . k_j))
 *
 * computed per (batch, head) with an online softmax whose running max m,
 * running sum l and unnormalised output accumulator stay on chip for the
 * whole K/V loop; the N x N score matrix is never written to device memory.
 *
 * Sources (page title, section):
 *  - "3.6 어텐션 I — 메모리 문제·FlashAttention 원리": 3.6.4 (online softmax
 *    recurrence, alpha = exp(m_old - m_new), one final division by l), 3.6.6
 *    (the FA2 tile loop: Q block outer / parallel, K/V blocks inner; causal
 *    skips key blocks j > i and masks the diagonal block), 3.6.7 (row
 *    statistic L = m + log l saved for the backward pass; the backward
 *    pass, fa_bwd, recomputes S and P from it).
 *  - "Triton으로 FlashAttention 1·2 forward 구현하기", section "병렬화 단위":
 *    grid = (cdiv(N, BLOCK_M), B * H), one program per Q block.
 *  - "FlashAttention-2를 CuTe로 밑바닥부터 구현하며 겪은 GPU 커널 지옥기",
 *    section "커널 구조는 단순한데, 디테일이 지옥임": P = QK^T / sqrt(d_h).
 *
 * All functions are plain C, thread-safe, and never throw.  No torch or
 * CUDA types appear in the signatures: device buffers are plain pointers and
 * the stream is a cudaStream_t passed as void* (NULL = the legacy default
 * stream of the calling thread's current device).
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FA_ABI_VERSION 4

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

/* Status codes.  Every entry point returns one of these. */
typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* a NULL buffer, a negative size, causal not 0/1, a
                               non-finite scale, overlapping output and input */
    FA_ERR_UNSUPPORTED = 2, /* d not supported, negative scale, dtype unknown,
                               N beyond the grid limit, device not sm_103 */
    FA_ERR_MISALIGNED = 3,  /* q, k, v or o not 16-byte aligned; lse not 4-byte */
    FA_ERR_CUDA = 4,        /* a CUDA runtime/driver call or the launch failed */
    FA_ERR_TIMEOUT = 5,     /* a kernel wait gave up (reported by
                               fa_last_device_status after the stream drained) */
    FA_ERR_BOUNDS = 6       /* checked build only: a device-side address check
                               failed and the access was skipped (reported by
                               fa_last_device_status) */
} fa_status_t;

/* Element type of Q, K, V and O (all four share it); accumulation is fp32. */
typedef enum { FA_FP16 = 0, FA_BF16 = 1 } fa_dtype_t;

/*
 * fa_fwd -- attention forward on the caller's stream (asynchronous).
 *
 *  q, k, v : device pointers, contiguous [B, H, N, d] tensors of `dtype`
 *            (row stride d elements), 16-byte aligned.  Read only.
 *  o       : device pointer, contiguous [B, H, N, d] of `dtype`, 16-byte
 *            aligned; must not overlap q, k or v.  Written: O rounded to
 *            nearest from fp32.
 *  lse     : device pointer to [B, H, N] fp32 (4-byte aligned), or NULL to
 *            skip it.  Written: lse = m * scale + ln(l), the natural log of
 *            sum_j exp(scale * q_i . k_j) over the allowed keys.
 *  B, H, N : batch, heads, sequence length (queries = keys = N).  Any of them
 *            0 is an empty problem: FA_OK, nothing launched.  Ragged N (not a
 *            multiple of the 128-row tile) is supported.
 *  d       : head dimension, 32, 64, 96 or 128.
 *  scale   : score scale (1/sqrt(d) for standard attention); finite, >= 0.
 *  causal  : 0 = every key; 1 = query i attends to keys j <= i.
 *  dtype   : FA_FP16 or FA_BF16.
 *  stream  : cudaStream_t (as void*), or NULL.
 *
 * Ownership: the caller owns every buffer; the library allocates no device
 * memory.  Argument errors are detected before anything is launched and leave
 * the outputs untouched.  A launch failure returns FA_ERR_CUDA.  A kernel
 * whose internal wait times out finishes early, leaves O/LSE partially
 * written, and records FA_ERR_TIMEOUT for fa_last_device_status.
 */
FA_API fa_status_t fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                   int B, int H, int N, int d, float scale, int causal,
                   fa_dtype_t dtype, void *stream);

/*
 * fa1_fwd_workspace_size -- bytes of device workspace fa1_fwd needs for a
 * problem: B*H*N*(d+2) fp32 values (the running output, max and sum of every
 * row).  0 for invalid sizes.
 */
FA_API size_t fa1_fwd_workspace_size(int B, int H, int N, int d);

/*
 * fa1_fwd -- the same attention forward computed with the FlashAttention-1
 * loop nest that "Triton으로 FlashAttention 1·2 forward 구현하기" (sections
 * "병렬화 단위", "출력 누적 방식") compares FA2 against: one CTA per (batch,
 * head), K/V blocks in the outer loop, Q blocks inside; after each K/V block
 * the normalised output and the statistics (m, l) of every row go to global
 * memory in fp32 and come back for the next block.  A baseline for the FA2
 * kernel above, not a faster path.
 *
 *  q, k, v, o, lse, B, H, N, d, scale, causal, dtype, stream: as for fa_fwd,
 *            with the same checks and results (up to rounding order).
 *  workspace: device pointer, 16-byte aligned, at least
 *            fa1_fwd_workspace_size(B, H, N, d) bytes, not overlapping any
 *            other buffer; owned by the caller; its contents on entry do not
 *            matter and on return are scratch.  Calls that share a workspace
 *            must not run concurrently.
 * Errors: as fa_fwd, plus FA_ERR_INVALID_ARG for a missing, short or
 * overlapping workspace and FA_ERR_MISALIGNED for a misaligned one.
 */
FA_API fa_status_t fa1_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                           void *workspace, size_t workspace_bytes, int B, int H, int N, int d,
                           float scale, int causal, fa_dtype_t dtype, void *stream);

/*
 * fa1_fwd_noalloc -- fa1_fwd without a workspace argument, for callers that
 * cannot allocate device memory on their own: code running where cudaMalloc
 * is unavailable or forbidden (a plugin or runtime that hands out only fixed
 * input/output buffers, a latency path that must not call into the
 * allocator).  The pages have no counterpart; this is a convenience of the
 * library.
 *
 *  Arguments and results: as fa1_fwd, without workspace / workspace_bytes.
 *  Scratch: a fixed 16 MiB device array inside the library, held by every
 *            device that loads the library until the process exits.  Problems
 *            needing more than that (fa1_fwd_workspace_size(B,H,N,d) > 16 MiB)
 *            return FA_ERR_UNSUPPORTED before anything is launched.
 *  No allocation: the call never calls cudaMalloc, cudaFree or any allocating
 *            routine.  The first call on each device looks up the array's
 *            device address (cudaGetSymbolAddress) with that device current;
 *            make that first call before any stream capture.
 *  Sharing: every call uses the same array and leaves its last contents in
 *            it; the kernel writes each scratch value before reading it, so
 *            nothing has to be cleared.  Calls that overlap on the GPU (other
 *            streams, other threads) race on the array: serialise them.
 */
FA_API fa_status_t fa1_fwd_noalloc(const void *q, const void *k, const void *v, void *o,
                                   float *lse, int B, int H, int N, int d, float scale, int causal,
                                   fa_dtype_t dtype, void *stream);

/*
 * fa_bwd_workspace_size -- bytes of device workspace fa_bwd needs: with
 * Npad = N rounded up to a multiple of 128, an fp32 dQ accumulator
 * [B*H, Npad, d] followed by two fp32 row vectors [B*H, Npad] (L log2(e) and
 * D, see fa_bwd).  0 for invalid sizes.
 */
FA_API size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * fa_bwd -- attention backward on the caller's stream (asynchronous): the
 * gradients of a loss with respect to q, k, v given its gradient dout with
 * respect to the forward output o.  With S = scale Q K^T (causal: keys j > i
 * masked), P = softmax(S), O = P V:
 *     dV = P^T dO,   dP = dO V^T,   dS = P o (dP - D),  D_i = sum_c dO_ic O_ic,
 *     dQ = scale dS K,   dK = scale dS^T Q.
 * Following "3.6 어텐션 I — 메모리 문제·FlashAttention 원리", section 3.6.7,
 * S and P are never read from memory: each 128 x 128 block is recomputed
 * from Q, K and the forward pass's saved row statistic (P = exp(S - lse)).
 *
 *  q, k, v : the forward inputs; device, contiguous [B, H, N, d] of `dtype`,
 *            16-byte aligned.  Read only.
 *  o       : the forward output fa_fwd wrote for them (same layout).  Read only.
 *  lse     : the forward's lse output, [B, H, N] fp32, 4-byte aligned; must
 *            not be NULL.  Read only.
 *  dout    : dL/dO, contiguous [B, H, N, d] of `dtype`, 16-byte aligned.
 *  dq, dk, dv : outputs, contiguous [B, H, N, d] of `dtype`, 16-byte aligned;
 *            must not overlap each other, the inputs or the workspace.
 *            Written: the gradients rounded to nearest from fp32.
 *  workspace : device pointer, 16-byte aligned, at least
 *            fa_bwd_workspace_size(B, H, N, d) bytes, not overlapping any
 *            other buffer; owned by the caller; contents on entry do not
 *            matter (the call clears what it accumulates into).  Calls that
 *            share a workspace must not run concurrently.
 *  B, H, N, d, scale, causal, dtype, stream : as for fa_fwd (the same
 *            values the forward call used).
 *
 * Three kernels run in order on `stream`: the row terms D and L log2(e) plus
 * clearing the accumulator; the main kernel (one CTA per head and 128-key
 * block, dK and dV kept on chip, dQ added into the fp32 accumulator); the
 * rounding of dQ.  Errors: as fa_fwd, plus FA_ERR_INVALID_ARG for a NULL lse
 * or dout/dq/dk/dv, or a missing, short or overlapping workspace, and
 * FA_ERR_MISALIGNED for a misaligned buffer.
 */
FA_API fa_status_t fa_bwd(const void *q, const void *k, const void *v, const void *o,
                          const float *lse, const void *dout, void *dq, void *dk, void *dv,
                          void *workspace, size_t workspace_bytes, int B, int H, int N, int d,
                          float scale, int causal, fa_dtype_t dtype, void *stream);

/*
 * fa_decode_workspace_size -- bytes of device workspace fa_decode needs: at
 * most one key chunk per 128 keys, each with an fp32 (m, l, O[d]) per query:
 * B*H*ceil(Nk/128)*Nq*(d+2)*4.  0 for invalid sizes.
 */
FA_API size_t fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d);

/*
 * fa_decode -- attention for decoding (asynchronous): Nq query rows per head
 * (1 <= Nq <= 16) against Nk >= Nq keys,
 *     O = softmax(Q K^T * scale) V,   LSE = log(sum_j exp(scale * q_i . k_j)),
 * with causal = 1 placing the queries at the end of the sequence (query i
 * attends to keys 0 .. Nk - Nq + i; with Nq = 1 that is every key).  "3.6
 * 어텐션 I — 메모리 문제·FlashAttention 원리", section 3.6.9: decoding needs a
 * different parallelisation than the Q-block grid of fa_fwd.  Split-KV: each
 * head's keys are cut into chunks that run the online softmax of section
 * 3.6.4 in parallel; a second launch merges the chunks' (m, l, O) with the
 * same rescaling (the result does not depend on the cut).
 *
 *  q       : device, contiguous [B, H, Nq, d] of `dtype`, 16-byte aligned.
 *  k, v    : device, contiguous [B, H, Nk, d] of `dtype` (a KV cache),
 *            16-byte aligned.
 *  o       : device, contiguous [B, H, Nq, d] of `dtype`, 16-byte aligned.
 *  lse     : [B, H, Nq] fp32 (natural log, as fa_fwd), or NULL.
 *  workspace : device, 16-byte aligned, >= fa_decode_workspace_size bytes,
 *            not overlapping any other buffer; contents do not matter.  Calls
 *            that share a workspace must not run concurrently.
 *  B, H, d, scale, dtype, stream : as for fa_fwd.
 * Errors: as fa_fwd, plus FA_ERR_UNSUPPORTED for Nq outside 1..16 and
 * FA_ERR_INVALID_ARG for Nk < Nq or a missing, short or overlapping workspace.
 */
FA_API fa_status_t fa_decode(const void *q, const void *k, const void *v, void *o, float *lse,
                             void *workspace, size_t workspace_bytes, int B, int H, int Nq, int Nk,
                             int d, float scale, int causal, fa_dtype_t dtype, void *stream);

/*
 * fa_last_device_status -- synchronise `stream`, read and clear the device
 * status word of the current device.  Returns FA_ERR_BOUNDS if a kernel of
 * the checked build (below) failed an address check, else FA_ERR_TIMEOUT if
 * any kernel launched since the last call gave up on a wait, FA_ERR_CUDA if
 * the stream reports an error, else FA_OK.  Not for use during CUDA graph
 * capture.
 *
 * Checked build.  The same sources compiled with FA_BOUNDS_CHECK give a second
 * library (libfa_gb300_checked.so) with the same entry points, for testing in
 * place of a memory checker: before every shared-memory and tensor-memory
 * access (TMA copies, MMA operands and accumulators, tensor-memory loads and
 * stores, mbarrier operations, shared loads and stores) its kernels check the
 * address against the block's shared window and the 512 tensor-memory
 * columns (and a warp's own lane quarter), and check ring-slot, buffer and
 * barrier indices.  A failed check skips the access and sets a bit that
 * fa_last_device_status reports as FA_ERR_BOUNDS; nothing traps.  The product
 * library compiles the checks away.
 */
FA_API fa_status_t fa_last_device_status(void *stream);

/*
 * fa_selftest_wait_timeout -- exercises the failure path without a GPU fault.
 * Launches one small kernel on `stream` whose bounded mbarrier wait (the same
 * wait the attention kernels use) waits on a barrier that nothing arrives on.
 * After about limit_us microseconds (1 .. 1e6) the wait gives up and records a
 * timeout in the device status word; fa_last_device_status then returns
 * FA_ERR_TIMEOUT (or FA_ERR_CUDA if the wait misbehaved).  Nothing hangs or
 * traps, and the CUDA context stays usable.  Returns FA_OK once launched.
 */
FA_API fa_status_t fa_selftest_wait_timeout(int limit_us, void *stream);

/*
 * fa_selftest_bounds_check -- exercises the checked build's address checks
 * without touching memory.  Launches one small kernel on `stream` that asks
 * the same check functions about addresses inside and outside the shared
 * window and the tensor-memory columns, in either build, and performs no
 * access with them.  The outside ones must fail, which records the
 * FA_ERR_BOUNDS bit; an inside one that failed records a self-test fault.
 * fa_last_device_status then returns FA_ERR_BOUNDS (or FA_ERR_CUDA if a check
 * misbehaved).  Returns FA_OK once launched.  The pages have no counterpart:
 * this is test support.
 */
FA_API fa_status_t fa_selftest_bounds_check(void *stream);

/* 1 if this library was built with the device-side address checks, else 0. */
FA_API int fa_checked_build(void);

/* Human-readable name of a status code (static storage; never NULL). */
FA_API const char *fa_status_str(fa_status_t status);

/* FA_ABI_VERSION of the built library. */
FA_API int fa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
