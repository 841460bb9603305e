// The online-softmax step shared by the forward kernels (one query row per thread,
// scores in TMEM): running max / running sum with lazy rescaling of the O row.
// The StreamKL summary, Methodology 1, restates the running pair (m, l) with
// LSE = m + log l; SparkAttention Figure 6 (step 2) is the same tile-wise update.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace exattn {

// One key tile of the online softmax for this thread's query row (= TMEM lane).  Reads the 128
// scores of S once, updates the running max m (base-2 units of the scaled scores) and sum l,
// rescales the O row in TMEM when the max grows by more than 2^8 (the final O / l is exact with a
// stale max), and writes P = exp2(s * c_log2 - m) over the first 64 S columns as packed 16-bit
// pairs: scores [64h, 64h + 64) become packed columns [32h, 32h + 32), the A operand of the PV
// MMA (every score is in registers before the first packed column is written).  With MASKED,
// columns at or past `lim` count as -inf.  The exponent argument and the sums use paired fp32
// instructions.  `before_rescale()` runs (warp-uniformly) before O is read for a rescale: a caller
// whose previous P V product may still be in flight waits for it there.
//
// softmax_tile_to is the same step with P written to its own 64 TMEM columns at tP instead of over S,
// and two more warp-uniform hooks: `after_load()` once every score is in registers (S may then be
// overwritten by the next score product), and `before_p()` before the first packed column of P is
// written (a caller whose previous P V product may still read the P columns waits there).
template <int D, bool MASKED, bool BF16, typename AfterLoad, typename BeforeRescale, typename BeforeP>
__device__ __forceinline__ void softmax_tile_to(uint32_t tS, uint32_t tP, uint32_t tO, int lim, float c_log2,
                                                bool first, float& m, float& l, AfterLoad&& after_load,
                                                BeforeRescale&& before_rescale, BeforeP&& before_p) {
  uint32_t sr[4][32];
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
  tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < 4; ++c) reg_fence32(sr[c]);
  after_load();
  if constexpr (MASKED) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (c * 32 + i >= lim) sr[c][i] = __float_as_uint(-INFINITY);
  }
  float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // independent chains
#pragma unroll
  for (int p = 0; p < 64; ++p)
    mx4[p & 3] = max3(mx4[p & 3], __uint_as_float(sr[p >> 4][(2 * p) & 31]), __uint_as_float(sr[p >> 4][(2 * p + 1) & 31]));
  const float m_new = fmaxf(m, max3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3])) * c_log2);
  if (first) {
    m = m_new;
  } else {
    const bool need = m_new > m + 8.0f;
    if (__any_sync(0xffffffffu, need)) {
      before_rescale();
      // O is complete for the previous key tile: its last MMA was issued before this tile's S.
      const float alpha = need ? ex2_approx(m - m_new) : 1.0f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_wait_ld();
        reg_fence32(o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st32(tO + c * 32, o);
      }
      tmem_wait_st();
      l *= alpha;
      if (need) m = m_new;
    }
  }
  before_p();
  const float ms = (m == -INFINITY) ? 0.f : m;
  const uint64_t c2 = f2_pack(c_log2, c_log2), nm2 = f2_pack(-ms, -ms);
  uint64_t acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = f2_pack(0.f, 0.f);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t pk[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int p = h * 32 + i;  // score pair (2p, 2p + 1)
      const uint64_t x = f2_fma(f2_pack(__uint_as_float(sr[p >> 4][(2 * p) & 31]), __uint_as_float(sr[p >> 4][(2 * p + 1) & 31])),
                                c2, nm2);
      float x0, x1;
      f2_unpack(x, x0, x1);
      const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
      acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
      pk[i] = pack2<BF16>(p0, p1);
    }
    tmem_st32(tP + h * 32, pk);
  }
  float s0, s1, s2, s3;
  f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), s0, s1);
  (void)s2;
  (void)s3;
  l += s0 + s1;
}

template <int D, bool MASKED, bool BF16, typename BeforeRescale>
__device__ __forceinline__ void softmax_tile(uint32_t tS, uint32_t tO, int lim, float c_log2, bool first, float& m,
                                             float& l, BeforeRescale&& before_rescale) {
  softmax_tile_to<D, MASKED, BF16>(tS, tS, tO, lim, c_log2, first, m, l, [] {}, before_rescale, [] {});
}

}  // namespace exattn
