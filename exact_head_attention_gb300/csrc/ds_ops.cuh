// Element policies for the gradient of the scores, dS = f(S_a, S_b, per-row values), shared by the
// query-tile gradient kernel and the attention-KL key-tile kernel.  Per-row values come from four
// row vectors: attention: negated base-2 LSE, D; attention KL: LSE1, LSE2, KL, upstream gradient g.
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
// dot products), or of two neighbouring key columns at once with fp32 pairs (`pair`: the same
// per-element arithmetic, so the same bits).  A row past Nq, or one that sees no key, gets values that
// make every dS exactly 0.
template <int OP, bool BF16>
struct DsOp;

template <bool BF16>
struct DsOp<kPairAttn, BF16> {
  float nlse2, dsum;  // -(base-2 LSE) (-inf on rows without keys and on padding), D = rowsum(dO o O)
  __device__ void load(const float* const (&rv)[4], size_t r, bool valid) {
    nlse2 = valid ? rv[0][r] : -INFINITY;
    dsum = valid ? rv[1][r] : 0.f;
  }
  __device__ float operator()(float sa, float sb, float c_log2, float) const {
    const float p = round16<BF16>(ex2_approx(fmaf(sa, c_log2, nlse2)));
    return p * (sb - dsum);
  }
  __device__ void pair(float sa0, float sa1, float sb0, float sb1, float c_log2, float, float& ds0, float& ds1) const {
    float x0, x1;
    f2_unpack(f2_fma(f2_pack(sa0, sa1), f2_pack(c_log2, c_log2), f2_pack(nlse2, nlse2)), x0, x1);
    const uint32_t pp = pack2<BF16>(ex2_approx(x0), ex2_approx(x1));  // P rounded to 16 bits
    const uint64_t p2 = f2_pack(unpack_lo<BF16>(pp), unpack_hi<BF16>(pp));
    f2_unpack(f2_mul(p2, f2_sub(f2_pack(sb0, sb1), f2_pack(dsum, dsum))), ds0, ds1);
  }
};

template <bool BF16>
struct DsOp<kPairKlStudent, BF16> {
  float nl1, nl2, g;  // negated base-2 LSEs of teacher and student, upstream gradient
  __device__ void load(const float* const (&rv)[4], size_t r, bool valid) {
    const float lse1 = valid ? rv[0][r] : -INFINITY;
    const bool empty = lse1 == -INFINITY;
    nl1 = empty ? -INFINITY : -lse1 * 1.4426950408889634f;
    nl2 = empty ? -INFINITY : -rv[1][r] * 1.4426950408889634f;
    g = empty ? 0.f : rv[3][r];
  }
  __device__ float operator()(float sa, float sb, float c_log2, float) const {
    return g * (ex2_approx(fmaf(sb, c_log2, nl2)) - ex2_approx(fmaf(sa, c_log2, nl1)));
  }
  __device__ void pair(float sa0, float sa1, float sb0, float sb1, float c_log2, float, float& ds0, float& ds1) const {
    const uint64_t c2 = f2_pack(c_log2, c_log2);
    float xa0, xa1, xb0, xb1;
    f2_unpack(f2_fma(f2_pack(sa0, sa1), c2, f2_pack(nl1, nl1)), xa0, xa1);
    f2_unpack(f2_fma(f2_pack(sb0, sb1), c2, f2_pack(nl2, nl2)), xb0, xb1);
    const uint64_t d = f2_sub(f2_pack(ex2_approx(xb0), ex2_approx(xb1)), f2_pack(ex2_approx(xa0), ex2_approx(xa1)));
    f2_unpack(f2_mul(f2_pack(g, g), d), ds0, ds1);
  }
};

template <bool BF16>
struct DsOp<kPairKlTeacher, BF16> {
  float nl1, g, cst;  // negated base-2 teacher LSE, upstream gradient, LSE_b - LSE_a - KL (natural)
  __device__ void load(const float* const (&rv)[4], size_t r, bool valid) {
    const float lse1 = valid ? rv[0][r] : -INFINITY;
    const bool empty = lse1 == -INFINITY;
    nl1 = empty ? -INFINITY : -lse1 * 1.4426950408889634f;
    g = empty ? 0.f : rv[3][r];
    cst = empty ? 0.f : rv[1][r] - lse1 - rv[2][r];
  }
  __device__ float operator()(float sa, float sb, float c_log2, float scale) const {
    return g * ex2_approx(fmaf(sa, c_log2, nl1)) * fmaf(scale, sa - sb, cst);
  }
  __device__ void pair(float sa0, float sa1, float sb0, float sb1, float c_log2, float scale, float& ds0,
                       float& ds1) const {
    const uint64_t sa2 = f2_pack(sa0, sa1);
    float x0, x1;
    f2_unpack(f2_fma(sa2, f2_pack(c_log2, c_log2), f2_pack(nl1, nl1)), x0, x1);
    const uint64_t ge = f2_mul(f2_pack(g, g), f2_pack(ex2_approx(x0), ex2_approx(x1)));
    const uint64_t t = f2_fma(f2_pack(scale, scale), f2_sub(sa2, f2_pack(sb0, sb1)), f2_pack(cst, cst));
    f2_unpack(f2_mul(ge, t), ds0, ds1);
  }
};

}  // namespace exattn
