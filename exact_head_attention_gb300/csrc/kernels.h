// Internal interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public header.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace exattn {

constexpr int kTileRows = 128;   // query rows per MMA tile (tcgen05 M) and key rows per K/V tile
constexpr int kFwdSubTiles = 2;  // query tiles per forward CTA (256 rows)

// The causal forward at d = 64 over at most this many keys runs one 128-row query tile per CTA, two CTAs
// per SM (fwd_tile_kernel) instead of 256-row blocks.
constexpr int kTileKernelMaxKeys = 2048;
inline bool fwd_uses_tile_kernel(int d, bool causal, int Nk) { return d == 64 && causal && Nk <= kTileKernelMaxKeys; }

// Element strides of a [B][H][N][d] view whose d elements are contiguous.
struct RowStrides {
  long long b, h, n;
};

// Causal masks: query q sees keys k <= q + causal_off, where causal_off is 0 (top-left alignment) or
// Nk - Nq (bottom-right alignment).

struct FwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_o;  // 4-D maps {d, N, H, B}, box {64, 128, 1, 1}, 128-byte swizzle
  float* lse;                          // [B*H][Nq]
  uint32_t* err_word;
  int sm_count;                        // of the device (the persistent causal launch runs one CTA per SM)
  int bh_count, heads, Nq, Nk, d;
  bool causal, bf16;
  int causal_off;
  float scale;
  uint64_t timeout_ns;
};

struct BwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do, tm_dk, tm_dv, tm_dq;
  CUtensorMap tm_dqacc;  // d = 64: 2-D fp32 map {d, B*H*Nq_pad} over dq_acc, box {32, 128}, 128-byte swizzle
  const void* o;       // [B][H][Nq][d] 16-bit, strides so
  const void* dout;    // [B][H][Nq][d] 16-bit, strides sdo
  const float* lse;    // [B*H][Nq]
  void* dq;            // [B][H][Nq][d] 16-bit, strides sdq
  RowStrides so, sdo, sdq;
  float* dq_acc;       // [B*H][Nq_pad][d] fp32 workspace (nullptr: deterministic dQ)
  float* nlse2;        // [B*H][Nq_pad] fp32 workspace: -LSE * log2(e), -inf on padding rows and rows without keys
  float* dsum;         // [B*H][Nq_pad] fp32 workspace: rowsum(dO o O), 0 on padding rows
  uint32_t* err_word;
  int bh_count, heads, Nq, Nq_pad, Nk, d;
  bool causal, bf16;
  int head_group;  // heads per launch group of the key/value blocks (kv_order.cuh)
  int causal_off;
  float scale;
  uint64_t timeout_ns;
};

// Split-KV forward: each CTA covers one 128-row query tile and one contiguous slice of the key tiles
// it sees; a second kernel merges the slices' partial results by their LSE.
struct SplitArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // as in FwdArgs
  float* o_part;                 // [splits][B*H][Nq][d] fp32: O of each slice, normalised by its own sum
  float* l_part;                 // [splits][B*H][Nq] fp32: base-2 LSE of each slice (-inf: no key seen)
  void* o;                       // merged O, 16-bit, strides so
  RowStrides so;
  float* lse;                    // [B*H][Nq], natural log
  uint32_t* err_word;
  int bh_count, heads, Nq, Nk, d, splits;
  bool causal, bf16;
  int causal_off;
  float scale;
  uint64_t timeout_ns;
};

// Query-tile gradient kernel: for one 128-row query tile, over the key tiles it sees in increasing order,
//   S_a = Q_a K_a^T, S_b = Q_b K_b^T, dS = f(S_a, S_b, per-row values), dQ += dS K_dq,
// with dQ accumulated on chip and stored once (times scale): the same bits on every run.  Used by the
// attention backward's deterministic mode (a = (Q, K), b = (dO, V), K_dq = K) and by the attention-KL
// backward (a = teacher, b = student, K_dq = the trained distribution's keys).
constexpr int kPairAttn = 0, kPairKlStudent = 1, kPairKlTeacher = 2;

struct PairDqArgs {
  CUtensorMap tm_qa, tm_ka, tm_qb, tm_kb, tm_dq;
  // per-row values, [B*H][rv_stride]: attention: base-2 LSE, D; KL: LSE1, LSE2, KL, upstream gradient g
  const float* rv[4];
  int rv_stride;
  uint32_t* err_word;
  int bh_count, heads, Nq, Nk, d;
  bool causal, bf16;
  int causal_off;
  float scale;
  int op;  // kPairAttn, kPairKlStudent, kPairKlTeacher
  uint64_t timeout_ns;
};

// Attention KL divergence (teacher a = (Q1, K1), student b = (Q2, K2)).
struct KlArgs {
  CUtensorMap tm_qa, tm_ka, tm_qb, tm_kb;  // 4-D maps as in FwdArgs
  CUtensorMap tm_dk;                       // backward: dK of the trained distribution
  float* kl;                               // [B*H][Nq]: forward output, backward input
  float* lse1;                             // [B*H][Nq]
  float* lse2;                             // [B*H][Nq]
  const float* g;                          // [B*H][Nq]: upstream gradient (backward)
  float* part;                             // forward, splits > 1: [5][splits][B*H][Nq] per-slice state
  int splits;                              // forward: key slices per query tile (1: none)
  // fused backward (atomic dQ): fp32 accumulator [B*H][Nq_pad][d], its 2-D map (d = 64, as in
  // BwdArgs), and three planes of per-row values [3][B*H][Nq_pad]
  float* dq_acc;
  CUtensorMap tm_dqacc;
  float* rowv;
  int Nq_pad;
  int head_group;  // as in BwdArgs
  uint32_t* err_word;
  int bh_count, heads, Nq, Nk, d;
  bool causal, bf16;
  int causal_off;
  float scale;
  int op;  // backward: kPairKlStudent or kPairKlTeacher
  uint64_t timeout_ns;
};

// Backward steps (bit mask for launch_bwd).  The atomic dQ mode runs pre, main, convert; the
// deterministic mode (dq_acc == nullptr) runs pre, main (dK and dV only), then the dQ kernel.
constexpr int kBwdPre = 1, kBwdMain = 2, kBwdConvert = 4, kBwdAll = 7, kBwdDq = 8;
constexpr int kBwdDeterministic = kBwdPre | kBwdMain | kBwdDq;

// Sets the message attn_last_error returns on this host thread.
void set_last_error(const char* msg);

// Each returns cudaSuccess or the launch error.
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_fwd_split(const SplitArgs& a, cudaStream_t stream);
cudaError_t launch_bwd(const BwdArgs& a, int steps, cudaStream_t stream);
cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_pair_dq(const PairDqArgs& a, cudaStream_t stream);
cudaError_t launch_kl_fwd(const KlArgs& a, cudaStream_t stream);
cudaError_t launch_kl_dk(const KlArgs& a, cudaStream_t stream);
// Row values + zeroed accumulator, then the one-pass key-tile kernel (dK and the dQ reduce-adds); the
// caller converts the accumulator with the attention backward's kBwdConvert step.
cudaError_t launch_kl_bwd_fused(const KlArgs& a, cudaStream_t stream);

}  // namespace exattn
