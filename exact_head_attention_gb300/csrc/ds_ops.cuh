// Element policies for the gradient of the scores, dS = f(S_a, S_b, per-row values), shared by the
// query-tile gradient kernel and the attention-KL key-tile kernel.  Per-row values come from four
// row vectors: attention: base-2 LSE, D; attention KL: LSE1, LSE2, KL, upstream gradient g.
#pragma once

#include <cstddef>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace exattn {

template <bool BF16>
__device__ __forceinline__ float round16(float x) {
  return unpack_lo<BF16>(pack2<BF16>(x, 0.f));
}

// dS policies: per-row values loaded once, then dS of one element from the two raw scores (unscaled
// dot products).  A row past Nq, or one that sees no key, gets values that make every dS exactly 0.
template <int OP, bool BF16>
struct DsOp;

template <bool BF16>
struct DsOp<kPairAttn, BF16> {
  float lse2, dsum;  // base-2 LSE (+inf on rows without keys and on padding), D = rowsum(dO o O)
  __device__ void load(const float* const (&rv)[4], size_t r, bool valid) {
    lse2 = valid ? rv[0][r] : INFINITY;
    dsum = valid ? rv[1][r] : 0.f;
  }
  __device__ float operator()(float sa, float sb, float c_log2, float) const {
    const float p = round16<BF16>(ex2_approx(fmaf(sa, c_log2, -lse2)));
    return p * (sb - dsum);
  }
};

template <bool BF16>
struct DsOp<kPairKlStudent, BF16> {
  float l1, l2, g;  // base-2 LSEs of teacher and student, upstream gradient
  __device__ void load(const float* const (&rv)[4], size_t r, bool valid) {
    const float lse1 = valid ? rv[0][r] : -INFINITY;
    const bool empty = lse1 == -INFINITY;
    l1 = empty ? INFINITY : lse1 * 1.4426950408889634f;
    l2 = empty ? INFINITY : rv[1][r] * 1.4426950408889634f;
    g = empty ? 0.f : rv[3][r];
  }
  __device__ float operator()(float sa, float sb, float c_log2, float) const {
    return g * (ex2_approx(fmaf(sb, c_log2, -l2)) - ex2_approx(fmaf(sa, c_log2, -l1)));
  }
};

template <bool BF16>
struct DsOp<kPairKlTeacher, BF16> {
  float l1, g, cst;  // base-2 teacher LSE, upstream gradient, LSE_b - LSE_a - KL (natural)
  __device__ void load(const float* const (&rv)[4], size_t r, bool valid) {
    const float lse1 = valid ? rv[0][r] : -INFINITY;
    const bool empty = lse1 == -INFINITY;
    l1 = empty ? INFINITY : lse1 * 1.4426950408889634f;
    g = empty ? 0.f : rv[3][r];
    cst = empty ? 0.f : rv[1][r] - lse1 - rv[2][r];
  }
  __device__ float operator()(float sa, float sb, float c_log2, float scale) const {
    return g * ex2_approx(fmaf(sa, c_log2, -l1)) * fmaf(scale, sa - sb, cst);
  }
};

}  // namespace exattn
