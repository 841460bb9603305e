/*
 * exattn -- exact fused multi-head attention (forward and backward) on one
 * GB300 GPU (sm_103a).  Plain C ABI: device pointers, sizes and a stream; no
 * framework types.
 *
 * What is computed (per batch b and head h, all tensors contiguous row-major):
 *   S = scale * Q K^T                         [Nq x Nk]
 *   S_qk = -inf where causal and k > q         (top-left aligned mask)
 *   P = softmax_row(S),  O = P V              [Nq x d]
 *   LSE_q = ln sum_k exp(S_qk)                 (natural log, scaled scores)
 * -- SparkAttention (arXiv 2502.12784), Equation 1 and the masked decoder MHA
 * of Figure 1; CANN ops-transformer MHA article, section 1 (scale 1/sqrt(d_k)).
 * The score matrix never reaches global memory: the forward is tiled with an
 * online (running max / running sum) softmax, SparkAttention Figure 6, and is
 * parallel over batch x heads x query-row blocks ("Fast Transformer training
 * with long sequences", attention parallelism section).
 *
 * Layouts:
 *   Q, O, dO, dQ : [B][H][Nq][d]   16-bit (bf16 or fp16, see attn_dtype)
 *   K, V, dK, dV : [B][H][Nk][d]   16-bit
 *   LSE          : [B][H][Nq]      fp32
 * All pointers are device pointers owned by the caller and must be 16-byte
 * aligned.  d must be 64 or 128.  All arithmetic accumulates in fp32; outputs
 * are rounded to nearest even into the input dtype.
 *
 * Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 * stream) and allocate no device memory.  Arguments are validated before any
 * launch; on an error status nothing is launched and no output is written.
 * Every device-side wait is bounded: if one expires the kernel records
 * ATTN_ERR_TIMEOUT in a per-device error word and exits; attn_check_device_error
 * (or EXATTN_CHECKED=1 in the environment, which synchronises after each call)
 * reports it.
 */
#ifndef EXATTN_H
#define EXATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,     /* null pointer, non-positive size, bad scale, bad dtype */
  ATTN_ERR_UNSUPPORTED = 2,     /* d not in {64, 128}, or no sm_103a device */
  ATTN_ERR_MISALIGNED = 3,      /* a pointer is not 16-byte aligned */
  ATTN_ERR_CUDA = 4,            /* a CUDA runtime/driver call or launch failed */
  ATTN_ERR_TIMEOUT = 5,         /* a bounded device wait expired (kernel exited early) */
  ATTN_ERR_WORKSPACE = 6,       /* workspace null or smaller than attn_bwd_workspace_size */
  ATTN_ERR_NOT_IMPLEMENTED = 7
} attn_status;

typedef enum { ATTN_BF16 = 0, ATTN_FP16 = 1 } attn_dtype;

/*
 * Forward.  Writes O and LSE.
 *   Q [B,H,Nq,d], K [B,H,Nk,d], V [B,H,Nk,d] inputs; O [B,H,Nq,d] and
 *   LSE [B,H,Nq] (fp32) outputs.  causal != 0 applies the top-left mask
 *   (query q sees keys k <= q).  scale > 0 and finite multiplies Q K^T.
 * Tiling, online softmax and per-block output as in SparkAttention Figure 6
 * (read Q once, stream K/V tiles, write O once); LSE is the saved row
 * statistic of the StreamKL summary, Methodology 1-2 (LSE = m + log l).
 */
attn_status attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                     int B, int H, int Nq, int Nk, int d, int causal, float scale,
                     attn_dtype dtype, void* stream);

/*
 * Bytes of device workspace attn_bwd needs for this shape: an fp32 dQ
 * accumulator [B,H,ceil(Nq/128)*128,d] plus two fp32 row vectors of the same
 * padded length (D = rowsum(dO o O) and the base-2 LSE).  Returns 0 for
 * invalid sizes.
 */
size_t attn_bwd_workspace_size(int B, int H, int Nq, int d);

/*
 * Backward of the loss sum(O o dO).  Inputs Q, K, V, O, dO (16-bit) and LSE
 * (fp32, as written by attn_fwd); outputs dQ [B,H,Nq,d], dK, dV [B,H,Nk,d].
 * workspace: caller-owned device memory of at least
 * attn_bwd_workspace_size(B,H,Nq,d) bytes, 256-byte aligned; its contents on
 * entry do not matter.
 * Steps (SparkAttention Figure 9 / Equation 4, "Fast Transformer training
 * with long sequences" backward parallelisation, StreamKL Methodology 2):
 *   D = rowsum(dO o O) ("dPsum"); per key/value block (parallel over blocks
 *   of columns of the attention matrix) recompute P = exp(S - LSE),
 *   dV += P^T dO, dP = dO V^T, dS = P o (dP - D), dK += scale dS^T Q, and
 *   dQ += scale dS K accumulated across blocks with fp32 atomics.
 * The dQ summation order across key blocks is not fixed, so dQ may differ
 * between runs by fp32 rounding.
 */
attn_status attn_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* LSE, void* dQ, void* dK, void* dV,
                     int B, int H, int Nq, int Nk, int d, int causal, float scale,
                     attn_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The three steps attn_bwd launches, callable one at a time (same arguments
 * and validation as attn_bwd; attn_bwd is exactly these three in this order on
 * `stream`, sharing `workspace`):
 *   attn_bwd_preprocess  D = rowsum(dO o O) and the base-2 LSE into the
 *                        workspace; zeroes the workspace's fp32 dQ accumulator
 *                        (SparkAttention Figure 9, the dPsum term).
 *   attn_bwd_kv_blocks   the fused pass over key/value blocks: writes dK and
 *                        dV and adds every block's dQ contribution into the
 *                        accumulator ("Fast Transformer training with long
 *                        sequences", backward parallelisation over columns).
 *   attn_bwd_dq_convert  dQ = scale * accumulator, rounded to the dtype.
 * Each step reads what the previous one left in `workspace`; calling them out
 * of order gives undefined results (no fault).
 */
attn_status attn_bwd_preprocess(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                                const float* LSE, void* dQ, void* dK, void* dV,
                                int B, int H, int Nq, int Nk, int d, int causal, float scale,
                                attn_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);
attn_status attn_bwd_kv_blocks(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                               const float* LSE, void* dQ, void* dK, void* dV,
                               int B, int H, int Nq, int Nk, int d, int causal, float scale,
                               attn_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);
attn_status attn_bwd_dq_convert(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                                const float* LSE, void* dQ, void* dK, void* dV,
                                int B, int H, int Nq, int Nk, int d, int causal, float scale,
                                attn_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward for callers that cannot allocate device memory -- for example a
 * plugin inside an engine that owns all device memory and forbids allocation
 * while it runs, or a latency-bound loop that cannot risk an allocator call
 * (or its failure) on every step.  The paper has no counterpart: this is a
 * deployment convenience of this library.
 *
 * Same arguments, layouts and results as attn_bwd, minus the workspace: the
 * scratch comes from one fixed array of ATTN_BWD_NOALLOC_MAX_WORKSPACE_BYTES
 * built into the library, which every GPU that loads the library reserves
 * until the process exits.  Nothing is allocated by this call.
 *   - Shapes whose attn_bwd_workspace_size exceeds the maximum are rejected
 *     with ATTN_ERR_WORKSPACE (attn_last_error gives the sizes); nothing runs.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture begins.
 *   - All calls share the one array, which keeps the last call's contents;
 *     each call clears what must start at zero.  Calls whose executions
 *     overlap on the GPU (different streams, or different host threads on
 *     the same device) race on the array and give wrong results: serialise
 *     them.
 */
#define ATTN_BWD_NOALLOC_MAX_WORKSPACE_BYTES ((size_t)64 << 20)
attn_status attn_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                             const float* LSE, void* dQ, void* dK, void* dV,
                             int B, int H, int Nq, int Nk, int d, int causal, float scale,
                             attn_dtype dtype, void* stream);

/* Static description of a status code. */
const char* attn_status_string(attn_status status);

/*
 * Describes, on the calling host thread, the most recent failure inside this
 * library (which CUDA call failed and its error string); "" if none.  The
 * pointer stays valid until the thread's next call into the library.
 */
const char* attn_last_error(void);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns ATTN_ERR_TIMEOUT if a kernel's bounded wait expired since the
 * last check, ATTN_ERR_CUDA if synchronisation failed, else ATTN_OK.
 */
attn_status attn_check_device_error(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* EXATTN_H */
