/*
 * exattn -- exact fused multi-head attention (forward and backward) on one
 * GB300 GPU (sm_103a).  Plain C ABI: device pointers, sizes and a stream; no
 * framework types.
 *
 * What is computed (per batch b and head h):
 *   S = scale * Q K^T                         [Nq x Nk]
 *   S_qk = -inf where the causal mask hides k from q (see attn_mask)
 *   P = softmax_row(S),  O = P V              [Nq x d]
 *   LSE_q = ln sum_k exp(S_qk)                 (natural log, scaled scores)
 * A query row that sees no key (only possible with the bottom-right mask and
 * Nq > Nk) gets O = 0, LSE = -inf and zero gradients.
 * -- SparkAttention (arXiv 2502.12784), Equation 1 and the masked decoder MHA
 * of Figure 1; CANN ops-transformer MHA article, section 1 (scale 1/sqrt(d_k)).
 * The score matrix never reaches global memory: the forward is tiled with an
 * online (running max / running sum) softmax, SparkAttention Figure 6, and is
 * parallel over batch x heads x query-row blocks ("Fast Transformer training
 * with long sequences", attention parallelism section).
 *
 * Layouts (the plain entry points; the *_strided ones take any strides, see
 * attn_strides):
 *   Q, O, dO, dQ : [B][H][Nq][d]   16-bit (bf16 or fp16, see attn_dtype), contiguous
 *   K, V, dK, dV : [B][H][Nk][d]   16-bit, contiguous
 *   LSE          : [B][H][Nq]      fp32, contiguous (always)
 * All pointers are device pointers owned by the caller and must be 16-byte
 * aligned.  d must be 64 or 128.  All arithmetic accumulates in fp32; outputs
 * are rounded to nearest even into the input dtype.
 *
 * Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 * stream) and allocate no device memory.  The library keeps per-device state
 * (the device address of its error word, the device's SM count and L2 size)
 * from the first call on a device to process exit: do not reset a device
 * (cudaDeviceReset) while the library is in use on it.  Arguments are
 * validated before any launch; on an error status nothing is launched and no
 * output is written.
 * The backward's kernels are dependent launches (programmatic stream
 * serialisation): each may start before the work ahead of it on the stream
 * has finished, but waits for that work before it reads or writes anything
 * the work could touch, so stream order holds as for ordinary launches.
 * Every wait between warp roles (an mbarrier) is bounded: if one expires the
 * kernel records ATTN_ERR_TIMEOUT in a per-device error word and exits;
 * attn_check_device_error (or EXATTN_CHECKED=1 in the environment, which
 * synchronises after each call) reports it.
 */
#ifndef EXATTN_H
#define EXATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,     /* null pointer, non-positive size, bad scale, dtype, mask or strides;
                                   sizes past the launch limits: ceil(Nq/256) or ceil(Nk/128) above
                                   65535, or B*H*ceil(Nk/128) above 2^31 - 1 */
  ATTN_ERR_UNSUPPORTED = 2,     /* d not in {64, 128}, or no sm_103a device */
  ATTN_ERR_MISALIGNED = 3,      /* a pointer is not 16-byte aligned */
  ATTN_ERR_CUDA = 4,            /* a CUDA runtime/driver call or launch failed */
  ATTN_ERR_TIMEOUT = 5,         /* a bounded device wait expired (kernel exited early) */
  ATTN_ERR_WORKSPACE = 6,       /* workspace null or smaller than attn_bwd_workspace_size */
  ATTN_ERR_NOT_IMPLEMENTED = 7
} attn_status;

typedef enum { ATTN_BF16 = 0, ATTN_FP16 = 1 } attn_dtype;

/*
 * Values of the `causal` argument (any other value is ATTN_ERR_INVALID_ARG).
 *   ATTN_MASK_NONE                 every query sees every key.
 *   ATTN_MASK_CAUSAL               top-left alignment: query q sees keys k <= q.
 *   ATTN_MASK_CAUSAL_BOTTOM_RIGHT  the Nq queries are the last Nq positions of
 *                                  the Nk-long sequence (a decoder continuing a
 *                                  cached prefix): query q sees keys
 *                                  k <= q + Nk - Nq.
 * Both causal forms are the masked decoder self-attention of SparkAttention
 * Figure 1 (a position attends to itself and the positions before it); they
 * differ only when Nq != Nk.
 */
typedef enum {
  ATTN_MASK_NONE = 0,
  ATTN_MASK_CAUSAL = 1,
  ATTN_MASK_CAUSAL_BOTTOM_RIGHT = 2
} attn_mask;

/*
 * Element strides of a 16-bit [B][H][N][d] view whose d elements are
 * contiguous (stride 1): element (b, h, n, c) is at
 * base + b*batch + h*head + n*row + c.
 *   contiguous [B][H][N][d]:          {H*N*d, N*d, d}
 *   [B][N][H][d] (rows of [S, H*D]):  {N*H*d, d, H*d}
 * Rules (ATTN_ERR_INVALID_ARG otherwise): row >= d; every stride a positive
 * multiple of 8 elements (16 bytes, a tensor-copy requirement) below 2^39;
 * the stride of a dimension of extent 1 is ignored.  Outputs must not overlap
 * one another or any input.  The CANN ops-transformer MHA article, section 1,
 * stores attention inputs as [S, H*D] rows; this struct admits that layout
 * and the per-head [N][d] matrices alike.
 */
typedef struct attn_strides {
  long long batch;
  long long head;
  long long row;
} attn_strides;

/*
 * Forward.  Writes O and LSE.
 *   Q [B,H,Nq,d], K [B,H,Nk,d], V [B,H,Nk,d] inputs; O [B,H,Nq,d] and
 *   LSE [B,H,Nq] (fp32) outputs.  causal is an attn_mask value.  scale > 0
 *   and finite multiplies Q K^T.
 * Tiling, online softmax and per-block output as in SparkAttention Figure 6
 * (read Q once, stream K/V tiles, write O once); LSE is the saved row
 * statistic of the StreamKL summary, Methodology 1-2 (LSE = m + log l).
 */
attn_status attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                     int B, int H, int Nq, int Nk, int d, int causal, float scale,
                     attn_dtype dtype, void* stream);

/*
 * attn_fwd on strided views: each 16-bit tensor comes with its attn_strides
 * (Q and O over Nq rows, K and V over Nk rows).  LSE stays contiguous
 * [B][H][Nq].  Same results and errors as attn_fwd, plus ATTN_ERR_INVALID_ARG
 * for strides that break the attn_strides rules.
 */
attn_status attn_fwd_strided(const void* Q, attn_strides q_strides, const void* K, attn_strides k_strides,
                             const void* V, attn_strides v_strides, void* O, attn_strides o_strides,
                             float* LSE, int B, int H, int Nq, int Nk, int d, int causal, float scale,
                             attn_dtype dtype, void* stream);

/*
 * Split-KV forward for few query rows (autoregressive decoding: Nq = 1 up to a
 * few hundred).  Same inputs, outputs, masks and results as attn_fwd (exact up
 * to fp32 rounding order).  With few query rows the plain forward has only
 * B*H*ceil(Nq/256) blocks of work; here the key dimension is also divided across
 * blocks (the "Split-K variant" of the StreamKL summary, GPU kernel
 * optimisations): block (b*H+h, query tile, s) runs the online softmax of one
 * 128-row query tile over the s-th contiguous slice of the key tiles it sees,
 * and a second kernel merges the slices of each row by their log-sum-exp:
 *   LSE = ln sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s.
 * num_splits: 1..256 slices per query tile, or 0 to let the library choose
 * (attn_fwd_splitkv_num_splits); when it chooses 1 this is exactly attn_fwd
 * and needs no workspace.  workspace: at least
 * attn_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, num_splits) bytes of device
 * memory, 256-byte aligned, contents on entry irrelevant (fp32 partial O and
 * LSE of every slice).  Errors as attn_fwd, plus ATTN_ERR_INVALID_ARG for
 * num_splits outside [0, 256] and ATTN_ERR_WORKSPACE for a missing or small
 * workspace.
 */
attn_status attn_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE,
                             int B, int H, int Nq, int Nk, int d, int causal, float scale,
                             attn_dtype dtype, int num_splits, void* workspace, size_t workspace_bytes,
                             void* stream);

/* attn_fwd_splitkv on strided views (see attn_strides and attn_fwd_strided). */
attn_status attn_fwd_splitkv_strided(const void* Q, attn_strides q_strides, const void* K, attn_strides k_strides,
                                     const void* V, attn_strides v_strides, void* O, attn_strides o_strides,
                                     float* LSE, int B, int H, int Nq, int Nk, int d, int causal, float scale,
                                     attn_dtype dtype, int num_splits, void* workspace, size_t workspace_bytes,
                                     void* stream);

/*
 * The number of slices attn_fwd_splitkv uses for num_splits = 0: 1 when the
 * B*H*ceil(Nq/128) query tiles alone fill sm_count SMs; otherwise the count
 * that minimises (waves of blocks over sm_count SMs, with two resident blocks
 * per SM at d = 64 and one at d = 128) x (key tiles per block + one tile of
 * fixed cost), kept at 1 unless a split wins by more than 2 %.  sm_count <= 0 asks the current device.  Returns 0
 * for invalid sizes (or when no device answers for sm_count <= 0).  The
 * StreamKL summary names the split-K variant for small N_Q without a rule for
 * the number of slices; this one is the library's own.
 */
int attn_fwd_splitkv_num_splits(int B, int H, int Nq, int Nk, int d, int sm_count);

/*
 * Workspace bytes of attn_fwd_splitkv for num_splits (0: the library's choice
 * on the current device, which may need none): fp32 partial O
 * [splits][B*H][Nq][d] and partial base-2 LSE [splits][B*H][Nq], each part
 * 256-byte aligned.  0 for invalid arguments.  The partial results are the
 * per-slice state of the StreamKL summary's split-K variant; the pages do not
 * size them (the caller owns all device memory).
 */
size_t attn_fwd_splitkv_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits);

/*
 * Attention KL divergence (the StreamKL summary, Methodology 1): a teacher
 * distribution P1 = softmax(scale Q1 K1^T) and a student P2 = softmax(scale
 * Q2 K2^T) over the same key positions (and the same attn_mask), and the
 * row-wise divergence of the student from the teacher
 *   KL_q = sum_k P1_qk (log P1_qk - log P2_qk)
 * computed in one pass with five running scalars per row, without forming
 * either distribution.  Q1, Q2 [B,H,Nq,d] and K1, K2 [B,H,Nk,d] 16-bit,
 * contiguous; outputs KL, LSE1, LSE2 [B,H,Nq] fp32 (LSE_t in natural-log
 * units, as attn_fwd).  A row that sees no key gets KL = 0 and LSE = -inf.
 * Errors as attn_fwd.
 */
attn_status attn_kl_fwd(const void* Q1, const void* K1, const void* Q2, const void* K2, float* KL, float* LSE1,
                        float* LSE2, int B, int H, int Nq, int Nk, int d, int causal, float scale,
                        attn_dtype dtype, void* stream);

/*
 * attn_kl_fwd for few query rows (the StreamKL summary's split-K variant, GPU
 * kernel optimisations): the key tiles each query tile sees are divided into
 * num_splits contiguous slices processed by separate blocks; each writes its
 * slice's five running scalars and a second kernel merges them (maxima
 * combined, sums and the weighted logit difference rescaled to the common
 * maxima).  Same results as attn_kl_fwd up to fp32 rounding.  num_splits:
 * 1..256, or 0 for the library's choice (the rule of
 * attn_fwd_splitkv_num_splits with one resident block per SM at either d;
 * when it is 1 this is exactly attn_kl_fwd and needs no workspace).
 * workspace: at least attn_kl_fwd_splitkv_workspace_size(B, H, Nq, Nk, d,
 * num_splits) bytes, 256-byte aligned, contents on entry irrelevant.  Errors as attn_kl_fwd, plus
 * ATTN_ERR_INVALID_ARG for num_splits outside [0, 256] and ATTN_ERR_WORKSPACE
 * for a missing or small workspace.
 */
attn_status attn_kl_fwd_splitkv(const void* Q1, const void* K1, const void* Q2, const void* K2, float* KL,
                                float* LSE1, float* LSE2, int B, int H, int Nq, int Nk, int d, int causal,
                                float scale, attn_dtype dtype, int num_splits, void* workspace,
                                size_t workspace_bytes, void* stream);

/* Workspace bytes of attn_kl_fwd_splitkv for num_splits (0: the library's
 * choice, which may need none): the five running scalars of the StreamKL
 * summary's Methodology 1, per slice and query row, in fp32.  The pages do not
 * size them (the caller owns all device memory). */
size_t attn_kl_fwd_splitkv_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits);

/*
 * Gradients of sum_q G_q KL_q (Methodology 2: probabilities regenerated from
 * the stored LSEs) for one distribution:
 *   setting 1, the student is trained (teacher fixed):
 *     dS = G (P2 - P1);                 dQ, dK are gradients w.r.t. Q2, K2
 *   setting 2, the teacher is trained (student fixed):
 *     dS = G P1 (log P1 - log P2 - KL); dQ, dK are gradients w.r.t. Q1, K1
 * with dQ = scale dS K and dK = scale dS^T Q of that distribution.  KL, LSE1,
 * LSE2 as written by attn_kl_fwd; G [B,H,Nq] fp32; dQ [B,H,Nq,d] and dK
 * [B,H,Nk,d] 16-bit outputs.  Two launches: dQ over query tiles and dK over
 * key tiles, each visiting every (query tile, key tile) pair once, no atomics:
 * the same bits on every run.  Errors as attn_fwd, plus ATTN_ERR_INVALID_ARG
 * for a setting other than 1 or 2.
 */
attn_status attn_kl_bwd(const void* Q1, const void* K1, const void* Q2, const void* K2, const float* KL,
                        const float* LSE1, const float* LSE2, const float* G, int setting, void* dQ, void* dK,
                        int B, int H, int Nq, int Nk, int d, int causal, float scale, attn_dtype dtype,
                        void* stream);

/*
 * Bytes of device workspace attn_kl_bwd_ex needs in the one-pass mode: an fp32
 * dQ accumulator [B,H,ceil(Nq/128)*128,d] plus three fp32 row vectors of that
 * padded length.  Returns 0 for invalid sizes.  The accumulator is the
 * buffer of the StreamKL summary's fused backward ("atomics while the buffer
 * fits in L2"); the pages do not size it (the caller owns all device memory).
 */
size_t attn_kl_bwd_workspace_size(int B, int H, int Nq, int d);

/*
 * attn_kl_bwd with a choice of how dQ is produced (dq_mode, an attn_dq_mode
 * value).  ATTN_DQ_DETERMINISTIC is attn_kl_bwd: two launches, no atomics, the
 * same bits on every run; the workspace is unused and may be NULL.
 * ATTN_DQ_ATOMIC and ATTN_DQ_AUTO take the StreamKL summary's one-pass form
 * (Methodology 2, fusion choice): one block per key tile recomputes both
 * distributions' scores once, accumulates dK on chip and adds its dQ
 * contribution into an fp32 accumulator in the workspace (copy-engine
 * reduce-adds through L2); a last launch writes dQ = scale * accumulator.
 * Four score-sized products per (query tile, key tile) pair instead of six.
 * dK is the same bits on every run; dQ's summation order across key tiles is
 * not fixed.  workspace: at least attn_kl_bwd_workspace_size(B,H,Nq,d) bytes,
 * 256-byte aligned, contents on entry irrelevant.  Errors as attn_kl_bwd, plus
 * ATTN_ERR_INVALID_ARG for an unknown dq_mode, ATTN_ERR_WORKSPACE for a
 * missing or small workspace and ATTN_ERR_MISALIGNED for a workspace that is
 * not 256-byte aligned (one-pass modes).
 */
attn_status attn_kl_bwd_ex(const void* Q1, const void* K1, const void* Q2, const void* K2, const float* KL,
                           const float* LSE1, const float* LSE2, const float* G, int setting, void* dQ, void* dK,
                           int B, int H, int Nq, int Nk, int d, int causal, float scale, attn_dtype dtype,
                           int dq_mode, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace attn_bwd needs for this shape: an fp32 dQ
 * accumulator [B,H,ceil(Nq/128)*128,d] plus two fp32 row vectors of the same
 * padded length (D = rowsum(dO o O) and the negated base-2 LSE).  Returns 0 for
 * invalid sizes.  The accumulator is the buffer that the thread blocks of
 * SparkAttention Figure 9 (and the column-block backward of "Fast Transformer
 * training with long sequences") add their dQ contributions into; D is that
 * figure's dPsum term.  The pages do not size it: this helper exists because
 * the caller owns all device memory.
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
 *   dQ += scale dS K accumulated across blocks by fp32 reductions into the
 *   workspace (ATTN_DQ_ATOMIC of attn_bwd_ex).
 * The dQ summation order across key blocks is not fixed, so dQ may differ
 * between runs by fp32 rounding; attn_bwd_ex with ATTN_DQ_DETERMINISTIC
 * gives the same bits on every run.  dK and dV are the same bits on every
 * run in either mode.
 */
attn_status attn_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* LSE, void* dQ, void* dK, void* dV,
                     int B, int H, int Nq, int Nk, int d, int causal, float scale,
                     attn_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_bwd on strided views (see attn_strides): Q, O, dO, dQ over Nq rows,
 * K, V, dK, dV over Nk rows; LSE contiguous [B][H][Nq]; the workspace as for
 * attn_bwd.  Same results and errors as attn_bwd, plus ATTN_ERR_INVALID_ARG
 * for strides that break the attn_strides rules.
 */
attn_status attn_bwd_strided(const void* Q, attn_strides q_strides, const void* K, attn_strides k_strides,
                             const void* V, attn_strides v_strides, const void* O, attn_strides o_strides,
                             const void* dO, attn_strides do_strides, const float* LSE, void* dQ,
                             attn_strides dq_strides, void* dK, attn_strides dk_strides, void* dV,
                             attn_strides dv_strides, int B, int H, int Nq, int Nk, int d, int causal,
                             float scale, attn_dtype dtype, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * How the backward produces dQ (attn_bwd_ex, attn_bwd_strided_ex).
 *   ATTN_DQ_ATOMIC         every key/value block adds its dQ contribution into
 *                          an fp32 accumulator (copy-engine reduce-adds of
 *                          shared-memory tiles); the order
 *                          of the additions varies, so dQ may differ between
 *                          runs in its last bits.  This is attn_bwd.  While
 *                          the accumulator fits in half the L2 cache (a
 *                          quarter with no mask) the key blocks are launched
 *                          heads fastest (the heavy low causal blocks of
 *                          every head start first); past that, in groups of
 *                          a few heads, so the blocks adding into one head's
 *                          rows run close together and find them still in
 *                          L2.
 *   ATTN_DQ_DETERMINISTIC  the key/value blocks produce dK and dV only; a
 *                          second kernel, parallel over 128-row query tiles,
 *                          recomputes S, P, dP and dS for each key tile the
 *                          tile sees, in increasing key order, and accumulates
 *                          dQ on chip.  dQ, dK and dV are the same bits on
 *                          every run; S and dP are computed twice (seven
 *                          tile products per key/query tile pair instead of
 *                          five).
 *   ATTN_DQ_AUTO           the faster of the two for the shape, as
 *                          attn_bwd_auto_dq_mode decides.  The StreamKL
 *                          summary (backward, kernel fusion) picks atomics
 *                          while the buffer fits in L2 and separate kernels
 *                          when contention on it grows; with the launch order
 *                          above, a head's additions stay in L2 whatever the
 *                          accumulator's size, and on GB300 the reductions
 *                          measured faster on every shape tried.
 * SparkAttention Figure 9 adds dQ across thread blocks atomically.
 */
typedef enum {
  ATTN_DQ_ATOMIC = 0,
  ATTN_DQ_DETERMINISTIC = 1,
  ATTN_DQ_AUTO = 2
} attn_dq_mode;

/*
 * How attn_fwd spreads a causal forward over the SMs.  The forward's work is
 * in 256-row query blocks, block = bh * ceil(Nq/256) + qb, and under a causal
 * mask a block's work grows with its position qb.  Where launching one CTA per
 * block (heaviest first) would leave SMs idle at the end, attn_fwd instead
 * runs one CTA per SM over lists of blocks that the host packs so that the
 * CTAs' work is even.  Returns the number of lists (CTAs), with the lists in
 * blocks[begin[i] .. begin[i+1]) for i < that number, or 0 when no lists
 * are used: no mask; d = 64 with Nk <= 2048, where attn_fwd runs one 128-row
 * query tile per CTA, two CTAs per SM; one wave or less; more than 2048
 * blocks; or a packing that would not shorten the busiest SM by 3 % after the
 * hand-over cost between a CTA's blocks.  blocks_cap and begin_cap are the capacities
 * of the two caller-owned host arrays.  sm_count <= 0 takes the current
 * device's.  Returns -1 for sizes attn_fwd rejects, arrays too small, or a
 * device count that is needed and cannot be read.  The pages parallelise the
 * forward over batch x heads x row blocks ("Fast Transformer training with
 * long sequences", attention parallelism); packing the blocks onto the SMs is
 * this library's own scheduling, with no counterpart there.
 */
int attn_fwd_schedule(int B, int H, int Nq, int Nk, int d, int causal, int sm_count, uint32_t* blocks,
                      int blocks_cap, int* begin, int begin_cap);

/*
 * Heads per launch group of the key/value-block kernels when dQ is reduced
 * into the fp32 accumulator (ATTN_DQ_ATOMIC, and the one-pass KL backward).
 * The blocks (one per head and 128-row key block) are numbered in groups of
 * this many heads, heads fastest within a group, the last group also taking
 * the B*H mod G heads left over.  G = B*H (plain heads-fastest order) while
 * the accumulator, B*H*ceil(Nq/128)*128*d*4 bytes, is at most a quarter of
 * l2_bytes with no mask, or half of it under a causal mask.  Otherwise G is
 * the number of heads whose accumulator rows fit in l2_bytes/16 (at least
 * 1); under a causal mask it is at least ceil(2*sm_count / ceil(Nk/128)); and
 * it is at most B*H.  sm_count <= 0 or l2_bytes = 0 take the current
 * device's values.  Returns -1 for sizes the backward rejects, or when a
 * device value is needed and cannot be read.  The rule serves the StreamKL
 * summary's condition for atomics (the buffer in use fits in L2); the launch
 * order itself has no counterpart on the pages.
 */
int attn_bwd_head_group(int B, int H, int Nq, int Nk, int d, int causal, int sm_count, size_t l2_bytes);

/*
 * The mode ATTN_DQ_AUTO resolves to for a backward of this shape (causal: an
 * attn_mask value): ATTN_DQ_ATOMIC.  On GB300 the reductions measured 1.3x to
 * 1.6x faster than the query-tile kernel on every shape tried (20 shapes with
 * 16 MiB to 512 MiB of accumulator, causal and not, d = 64 and 128): the
 * query-tile kernel recomputes S and dP, and with the launch order of
 * ATTN_DQ_ATOMIC the reductions' working set stays in L2.  Returns -1 for
 * invalid sizes.  Needs no device.  This is the choice the StreamKL summary
 * makes in its backward (atomics while the buffer fits in L2, separate
 * kernels under contention), measured on GB300.
 */
int attn_bwd_auto_dq_mode(int B, int H, int Nq, int Nk, int d, int causal);

/*
 * attn_bwd with a dQ mode (attn_dq_mode; other values are
 * ATTN_ERR_INVALID_ARG).  The workspace is sized by attn_bwd_workspace_size
 * for every mode (the deterministic mode leaves the accumulator part unused).
 */
attn_status attn_bwd_ex(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                        const float* LSE, void* dQ, void* dK, void* dV,
                        int B, int H, int Nq, int Nk, int d, int causal, float scale,
                        attn_dtype dtype, int dq_mode, void* workspace, size_t workspace_bytes, void* stream);

/* attn_bwd_strided with a dQ mode (see attn_bwd_ex). */
attn_status attn_bwd_strided_ex(const void* Q, attn_strides q_strides, const void* K, attn_strides k_strides,
                                const void* V, attn_strides v_strides, const void* O, attn_strides o_strides,
                                const void* dO, attn_strides do_strides, const float* LSE, void* dQ,
                                attn_strides dq_strides, void* dK, attn_strides dk_strides, void* dV,
                                attn_strides dv_strides, int B, int H, int Nq, int Nk, int d, int causal,
                                float scale, attn_dtype dtype, int dq_mode, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * The three steps attn_bwd launches, callable one at a time (same arguments
 * and validation as attn_bwd; attn_bwd is exactly these three in this order on
 * `stream`, sharing `workspace`):
 *   attn_bwd_preprocess  D = rowsum(dO o O) and the negated base-2 LSE into the
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
 * Self-test of the bounded device waits.  Launches one block whose thread
 * waits, through the same bounded wait the attention kernels use on their
 * pipelines, on a shared-memory barrier that nothing ever arrives at.  After
 * timeout_ms milliseconds the wait gives up, the kernel records
 * ATTN_ERR_TIMEOUT in the device error word and returns normally: no fault,
 * no trap, and the context stays usable.  The call then synchronises `stream`
 * and returns what attn_check_device_error reports, so a working library
 * returns ATTN_ERR_TIMEOUT (and clears the error word).  timeout_ms must be
 * in [1, 10000] (ATTN_ERR_INVALID_ARG otherwise).  The pages have no
 * counterpart: this is a check of the library's own failure detection.
 */
attn_status attn_selftest_wait_timeout(int timeout_ms, void* stream);

/*
 * Backward for callers that cannot allocate device memory -- for example a
 * plugin inside an engine that owns all device memory and forbids allocation
 * while it runs, or a latency-bound loop that cannot risk an allocator call
 * (or its failure) on every step.  The paper has no counterpart: this is a
 * deployment convenience of this library.
 *
 * Same arguments, layouts and results as attn_bwd, minus the workspace: the
 * scratch comes from one fixed array of ATTN_BWD_NOALLOC_MAX_WORKSPACE_BYTES
 * built into the library.  A GPU reserves the array when the library's module
 * that holds it is loaded there -- with CUDA's default lazy module loading at
 * the first attn_bwd_noalloc call on that device, with eager loading
 * (CUDA_MODULE_LOADING=EAGER) when the library's code is loaded -- and keeps
 * it until the process exits.  Nothing is allocated by this call.
 *   - Shapes whose attn_bwd_workspace_size exceeds the maximum are rejected
 *     with ATTN_ERR_WORKSPACE (attn_last_error gives the sizes); nothing runs.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture begins.  The address is kept for the life
 *     of the process, so do not reset the device (cudaDeviceReset) between
 *     calls: the library's per-device state, this address included, would
 *     then name memory of a context that no longer exists.
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

/* Static description of a status code (a diagnostic of this library; the
 * pages have no counterpart).  Never NULL: unknown codes give
 * "unknown status". */
const char* attn_status_string(attn_status status);

/*
 * Describes, on the calling host thread, the most recent failure inside this
 * library (which CUDA call failed and its error string); "" if none.  The
 * pointer stays valid until the thread's next call into the library.  A
 * diagnostic of this library; the pages have no counterpart.
 */
const char* attn_last_error(void);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns ATTN_ERR_TIMEOUT if a kernel's bounded wait expired since the
 * last check, ATTN_ERR_CUDA if synchronisation failed, else ATTN_OK.  A
 * diagnostic of this library's failure detection; the pages have no
 * counterpart.
 */
attn_status attn_check_device_error(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* EXATTN_H */
