// Attention KL divergence on sm_103a: a fused one-pass forward and the key-tile half of the backward.
//
// Teacher (a) and student (b) attention distributions over the same key positions,
//     P_t = softmax(scale Q_t K_t^T),  KL_q = sum_k P_a,qk (log P_a,qk - log P_b,qk),
// never materialised.  Forward (StreamKL summary, Methodology 1): per query row,
// five running scalars m_a, m_b (running maxima), l_a, l_b (sums of exponentials)
// and acc (the exp-weighted logit difference) are updated tile by tile:
//     acc = sum_k exp(S_a,k - m_a) (S_a,k - S_b,k),   KL = acc / l_a + LSE_b - LSE_a,
// with LSE_t = m_t + log l_t; both LSEs are stored for the backward.  Causal key
// tiles past a query tile's frontier are skipped.
//
// Backward (Methodology 2): the probabilities are regenerated from the stored
// LSEs, and for the distribution being trained (student: dS = g (P_b - P_a);
// teacher: dS = g P_a (log P_a - log P_b - KL)) dQ comes from the query-tile
// kernel and dK from kl_dk_kernel below: one CTA per 128-row key tile, over the
// query tiles that see it, dK += dS^T Q with dS staged in shared memory.  Each
// (query tile, key tile) pair is visited once by each kernel, and neither uses
// atomics ("separate kernels" in the summary's fusion choice).
//
// Forward warp roles (384 threads, registers re-split per warpgroup): warps 0-3
// and 4-7 are two compute warpgroups taking alternate key tiles (thread = query
// row), each with its own five scalars, merged through shared memory at the end;
// warp 8 is the TMA producer; warp 9 the MMA issuer and TMEM owner; warps 10-11
// complete the control warpgroup.  TMEM: buffer b in {0, 1} holds
// S_a at [256b, 256b+128) and S_b at [256b+128, 256b+256).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ds_ops.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace exattn {
namespace {

constexpr uint32_t kChunkBytes = 128 * 128;

// ====================================================================== forward

constexpr int kKlFwdThreads = 384;
// Register shares after reallocation (launch: 168 each); one warp of each warpgroup per SM sub-partition.
constexpr uint32_t kKlRegsCompute = 208, kKlRegsControl = 88;
static_assert(2 * kKlRegsCompute + kKlRegsControl == 3 * 168, "register split must match the launch");

template <int D>
struct KlFwdCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = kTileRows * D * 2;
  static constexpr int NS = (D == 64) ? 4 : 2;  // ring slots, each K_a and K_b of one key tile
  static constexpr uint32_t OFF_QA = 0;
  static constexpr uint32_t OFF_QB = TILE;
  static constexpr uint32_t OFF_RING = 2 * TILE;
  static constexpr uint32_t OFF_MERGE = OFF_RING + NS * 2 * TILE;  // 5 x 128 floats
  static constexpr uint32_t OFF_BAR = OFF_MERGE + 5 * 128 * 4;
  // q_full, k_full[NS], k_empty[NS], s_full[2], s_free[2], mma_done
  static constexpr int NBAR = 1 + 2 * NS + 5;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
};

struct KlFwdBars {
  uint32_t base;
  int ns;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t k_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t k_empty(int s) const { return base + 8 * (1 + ns + s); }
  __device__ uint32_t s_full(int b) const { return base + 8 * (1 + 2 * ns + b); }
  __device__ uint32_t s_free(int b) const { return base + 8 * (3 + 2 * ns + b); }
  __device__ uint32_t mma_done() const { return base + 8 * (5 + 2 * ns); }
};

// exp2(x - m) with m = -inf (a row without a visible key so far) treated as 0; masked x are -inf.
__device__ __forceinline__ float base_of(float m) { return m == -INFINITY ? 0.f : m; }

// One key tile of the five-scalar update for this thread's query row: reads the tile's raw teacher and
// student scores from TMEM twice (tile maxima, then sums), rescales l_a, acc (by the teacher's max
// change) and l_b (the student's), and adds
//     l_a += sum exp2(s_a c - m_a),  l_b += sum exp2(s_b c - m_b),  acc += sum exp2(s_a c - m_a) (s_a - s_b)
// (c = scale log2 e; acc in raw score units).  With MASKED, columns at or past `lim` take no part.
// Neighbouring columns travel as fp32 pairs.
template <bool MASKED>
__device__ __forceinline__ void kl_tile(uint32_t tA, uint32_t tB, int lim, float c_log2, float& ma, float& mb,
                                        float& la, float& lb, float& acc) {
  float xa[2] = {-INFINITY, -INFINITY}, xb[2] = {-INFINITY, -INFINITY};
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t va[32], vb[32];
    tmem_ld32(tA + c * 32, va);
    tmem_ld32(tB + c * 32, vb);
    tmem_wait_ld();
    reg_fence32(va);
    reg_fence32(vb);
    if constexpr (MASKED) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (c * 32 + i >= lim) va[i] = vb[i] = __float_as_uint(-INFINITY);
    }
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      xa[p & 1] = max3(xa[p & 1], __uint_as_float(va[2 * p]), __uint_as_float(va[2 * p + 1]));
      xb[p & 1] = max3(xb[p & 1], __uint_as_float(vb[2 * p]), __uint_as_float(vb[2 * p + 1]));
    }
  }
  const float na = fmaxf(ma, fmaxf(xa[0], xa[1]) * c_log2), nb = fmaxf(mb, fmaxf(xb[0], xb[1]) * c_log2);
  const float alpha_a = na == ma ? 1.f : ex2_approx(ma - na), alpha_b = nb == mb ? 1.f : ex2_approx(mb - nb);
  la *= alpha_a;
  acc *= alpha_a;
  lb *= alpha_b;
  ma = na;
  mb = nb;
  // Pairs of neighbouring columns of one distribution travel together: (s[2p], s[2p+1]) of the teacher
  // and of the student each form one fp32 pair, so the exponent arguments, the two sums, the score
  // difference and the weighted difference take one paired instruction per two columns.
  const uint64_t c2 = f2_pack(c_log2, c_log2);
  const uint64_t na2 = f2_pack(-base_of(ma), -base_of(ma)), nb2 = f2_pack(-base_of(mb), -base_of(mb));
  uint64_t la2 = f2_pack(0.f, 0.f), lb2 = f2_pack(0.f, 0.f), ac2 = f2_pack(0.f, 0.f);
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t va[32], vb[32];
    tmem_ld32(tA + c * 32, va);
    tmem_ld32(tB + c * 32, vb);
    tmem_wait_ld();
    reg_fence32(va);
    reg_fence32(vb);
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      const uint64_t a2 = f2_pack(__uint_as_float(va[2 * p]), __uint_as_float(va[2 * p + 1]));
      const uint64_t b2 = f2_pack(__uint_as_float(vb[2 * p]), __uint_as_float(vb[2 * p + 1]));
      float xa0, xa1, xb0, xb1;
      f2_unpack(f2_fma(a2, c2, na2), xa0, xa1);
      f2_unpack(f2_fma(b2, c2, nb2), xb0, xb1);
      float ea0 = ex2_approx(xa0), ea1 = ex2_approx(xa1), eb0 = ex2_approx(xb0), eb1 = ex2_approx(xb1);
      uint64_t df2 = f2_sub(a2, b2);
      if constexpr (MASKED) {
        const int col = c * 32 + 2 * p;
        if (col >= lim || col + 1 >= lim) {  // masked columns take no part (their difference may be NaN)
          float d0, d1;
          f2_unpack(df2, d0, d1);
          if (col >= lim) ea0 = eb0 = d0 = 0.f;
          if (col + 1 >= lim) ea1 = eb1 = d1 = 0.f;
          df2 = f2_pack(d0, d1);
        }
      }
      const uint64_t e_a = f2_pack(ea0, ea1);
      la2 = f2_add(la2, e_a);
      lb2 = f2_add(lb2, f2_pack(eb0, eb1));
      ac2 = f2_fma(e_a, df2, ac2);
    }
  }
  float a0, a1, b0, b1, d0, d1;
  f2_unpack(la2, a0, a1);
  f2_unpack(lb2, b0, b1);
  f2_unpack(ac2, d0, d1);
  la += a0 + a1;
  lb += b0 + b1;
  acc += d0 + d1;
}

// SPLIT: the grid's z dimension divides the key tiles a query tile sees into a.splits contiguous
// slices (the summary's split-K variant for few query rows); each block writes its slice's merged five
// scalars to a.part and kl_combine_kernel forms KL and the LSEs.
template <int D, bool CAUSAL, bool BF16, bool SPLIT>
__global__ void __launch_bounds__(kKlFwdThreads, 1) kl_fwd_kernel(const __grid_constant__ KlArgs a) {
  using C = KlFwdCfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  if (!smem_base_aligned(sbase, a.err_word)) return;
  uint8_t* gbase = smem_raw;
  const uint32_t sQa = sbase + C::OFF_QA, sQb = sbase + C::OFF_QB, sRing = sbase + C::OFF_RING;
  const KlFwdBars bars{sbase + C::OFF_BAR, NS};
  float* merge = reinterpret_cast<float*>(gbase + C::OFF_MERGE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + C::OFF_MISC + 4);
  const WaitCtx wc{abort_flag, a.err_word, a.timeout_ns};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int head = bh % a.heads, batch = bh / a.heads;
  const int qt = gridDim.y - 1 - blockIdx.y;  // heaviest (causal) query tiles first
  const int q0 = qt * kTileRows;
  const int nkv = (a.Nk + kTileRows - 1) / kTileRows;
  const int coff = CAUSAL ? a.causal_off : 0;
  int nvis = nkv;  // key tiles this query tile sees
  if (CAUSAL) {
    const int last_key = q0 + kTileRows - 1 + coff;
    nvis = last_key < 0 ? 0 : min(nkv, last_key / kTileRows + 1);
  }
  // this block's key tiles [j0, j0 + n): all of them, or one slice (slices differ by at most one tile)
  const int split = SPLIT ? static_cast<int>(blockIdx.z) : 0, nsplit = SPLIT ? a.splits : 1;
  const int j0 = static_cast<int>(static_cast<long long>(split) * nvis / nsplit);
  const int n = static_cast<int>(static_cast<long long>(split + 1) * nvis / nsplit) - j0;

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    mbar_init(bars.q_full(), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bars.k_full(s), 1);
      mbar_init(bars.k_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.s_full(b), 1);
      mbar_init(bars.s_free(b), kTileRows);
    }
    mbar_init(bars.mma_done(), 1);
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) regs_decrease<kKlRegsControl>();
  else regs_increase<kKlRegsCompute>();
  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0) {
      prefetch_tmap(&a.tm_qa);
      prefetch_tmap(&a.tm_qb);
      prefetch_tmap(&a.tm_ka);
      prefetch_tmap(&a.tm_kb);
      mbar_arrive_expect_tx(bars.q_full(), 2 * C::TILE);
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_4d(sQa + c * kChunkBytes, &a.tm_qa, c * 64, q0, head, batch, bars.q_full());
        tma_load_4d(sQb + c * kChunkBytes, &a.tm_qb, c * 64, q0, head, batch, bars.q_full());
      }
      int issued = 0;
      for (int j = 0; j < n; ++j) {
        const int s = j % NS;
        if (!mbar_wait(bars.k_empty(s), ((j / NS) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(bars.k_full(s), 2 * C::TILE);
        const uint32_t dst = sRing + s * 2 * C::TILE;
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_4d(dst + c * kChunkBytes, &a.tm_ka, c * 64, (j0 + j) * kTileRows, head, batch, bars.k_full(s));
          tma_load_4d(dst + C::TILE + c * kChunkBytes, &a.tm_kb, c * 64, (j0 + j) * kTileRows, head, batch,
                      bars.k_full(s));
        }
        ++issued;
      }
      if (*abort_flag) {
        for (int j = max(0, issued - NS); j < issued; ++j) mbar_drain(bars.k_full(j % NS), (j / NS) & 1, a.timeout_ns);
        mbar_drain(bars.q_full(), 0, a.timeout_ns);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idS = idesc_f16(128, 128, BF16, false, false);
      constexpr uint32_t kTileLo = C::TILE >> 4;
      const uint32_t qa_lo = sdesc_lo(sQa, 16), qb_lo = sdesc_lo(sQb, 16), ring_lo = sdesc_lo(sRing, 16);
      auto scores = [&](uint32_t d, uint32_t q_lo, uint32_t b_lo) {
        mma_ss_lo<false>(d, q_lo, b_lo, idS);
#pragma unroll
        for (int k = 1; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * kChunkBytes + (k & 3) * 32) >> 4;
          mma_ss_lo<true>(d, q_lo + off, b_lo + off, idS);
        }
      };
      bool ok = mbar_wait(bars.q_full(), 0, wc);
      for (int j = 0; ok && j < n; ++j) {
        const int b = j & 1, s = j % NS;
        // buffer b was last read by its warpgroup for tile j - 2
        if (j >= 2 && !(ok = mbar_wait(bars.s_free(b), ((j >> 1) - 1) & 1, wc))) break;
        if (!(ok = mbar_wait(bars.k_full(s), (j / NS) & 1, wc))) break;
        tc_fence_after();
        scores(tmem + b * 256, qa_lo, ring_lo + (2 * s) * kTileLo);
        scores(tmem + b * 256 + 128, qb_lo, ring_lo + (2 * s + 1) * kTileLo);
        mma_commit(bars.s_full(b));
        mma_commit(bars.k_empty(s));
      }
      mma_commit(bars.mma_done());
      mbar_drain(bars.mma_done(), 0, a.timeout_ns);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ compute: warpgroup t takes tiles j = t (mod 2)
    const int t = warp >> 2, quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row inside the tile = TMEM lane
    const int row = q0 + r;
    const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tA = tmem + t * 256 + lane_bits, tB = tA + 128;
    const float c_log2 = a.scale * 1.4426950408889634f;
    // running state: maxima in base-2 units of the scaled scores; acc in raw (unscaled) score units
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f, acc = 0.f;
    bool ok = true;
    for (int j = t; ok && j < n; j += 2) {
      if (!(ok = mbar_wait_warp(bars.s_full(t), (j >> 1) & 1, wc))) break;
      tc_fence_after();
      const int jg = j0 + j;  // key tile index
      const bool need_mask =
          ((jg + 1) * kTileRows > a.Nk) || (CAUSAL && jg * kTileRows + kTileRows - 1 > q0 + coff);
      const int lim = need_mask ? (CAUSAL ? min(a.Nk, row + coff + 1) : a.Nk) - jg * kTileRows : kTileRows;
      if (need_mask)
        kl_tile<true>(tA, tB, lim, c_log2, ma, mb, la, lb, acc);
      else
        kl_tile<false>(tA, tB, lim, c_log2, ma, mb, la, lb, acc);
      tc_fence_before();
      mbar_arrive(bars.s_free(t));  // both score tiles were read: the buffer may be refilled
    }

    // ------------------------------------------------------------ merge the two warpgroups' states
    if (t == 1) {
      merge[0 * 128 + r] = ma;
      merge[1 * 128 + r] = mb;
      merge[2 * 128 + r] = la;
      merge[3 * 128 + r] = lb;
      merge[4 * 128 + r] = acc;
    }
    named_bar_sync(1, 256);
    if (t == 0 && ok && !*abort_flag && row < a.Nq) {
      const float ma1 = merge[r], mb1 = merge[128 + r], la1 = merge[256 + r], lb1 = merge[384 + r], ac1 = merge[512 + r];
      const float Ma = fmaxf(ma, ma1), Mb = fmaxf(mb, mb1);
      const float w0 = ma == -INFINITY ? 0.f : ex2_approx(ma - Ma), w1 = ma1 == -INFINITY ? 0.f : ex2_approx(ma1 - Ma);
      const float v0 = mb == -INFINITY ? 0.f : ex2_approx(mb - Mb), v1 = mb1 == -INFINITY ? 0.f : ex2_approx(mb1 - Mb);
      const float L_a = la * w0 + la1 * w1, L_b = lb * v0 + lb1 * v1, A = acc * w0 + ac1 * w1;
      const size_t o = static_cast<size_t>(bh) * a.Nq + row;
      if constexpr (SPLIT) {
        // the slice's state: maxima (base 2), sums and acc, one plane each
        const size_t plane = static_cast<size_t>(a.splits) * a.bh_count * a.Nq;
        const size_t e = static_cast<size_t>(split) * a.bh_count * a.Nq + o;
        a.part[e] = Ma;
        a.part[plane + e] = Mb;
        a.part[2 * plane + e] = L_a;
        a.part[3 * plane + e] = L_b;
        a.part[4 * plane + e] = A;
      } else if (L_a > 0.f) {
        const float lse_a = (Ma + __log2f(L_a)) * 0.6931471805599453f;
        const float lse_b = (Mb + __log2f(L_b)) * 0.6931471805599453f;
        a.lse1[o] = lse_a;
        a.lse2[o] = lse_b;
        a.kl[o] = a.scale * A / L_a + lse_b - lse_a;
      } else {  // the row sees no key
        a.lse1[o] = -INFINITY;
        a.lse2[o] = -INFINITY;
        a.kl[o] = 0.f;
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ====================================================================== backward: dK over key tiles

constexpr int kKlDkThreads = 192;

template <int D>
struct KlDkCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = kTileRows * D * 2;
  static constexpr int NS = (D == 64) ? 4 : 2;  // ring slots, each Q_a and Q_b of one query tile
  static constexpr uint32_t OFF_KA = 0;
  static constexpr uint32_t OFF_KB = TILE;
  static constexpr uint32_t OFF_DS = 2 * TILE;                 // dS [query][key] 16-bit, 32 KB
  static constexpr uint32_t OFF_RING = OFF_DS + 128 * 128 * 2;
  static constexpr uint32_t OFF_BAR = OFF_RING + NS * 2 * TILE;
  // kv_full, q_full[NS], q_empty[NS], s_full, s_used, ds_ready, ds_free, done, mma_done
  static constexpr int NBAR = 1 + 2 * NS + 6;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
};

struct KlDkBars {
  uint32_t base;
  int ns;
  __device__ uint32_t kv_full() const { return base; }
  __device__ uint32_t q_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t q_empty(int s) const { return base + 8 * (1 + ns + s); }
  __device__ uint32_t at(int k) const { return base + 8 * (1 + 2 * ns + k); }
  __device__ uint32_t s_full() const { return at(0); }
  __device__ uint32_t s_used() const { return at(1); }
  __device__ uint32_t ds_ready() const { return at(2); }
  __device__ uint32_t ds_free() const { return at(3); }
  __device__ uint32_t done() const { return at(4); }
  __device__ uint32_t mma_done() const { return at(5); }
};

// One CTA per 128-row key tile j of one head.  For every query tile i that sees it:
//   S_a = Q_a,i K_a,j^T and S_b = Q_b,i K_b,j^T (TMEM, lane = query row), dS by the policy (thread =
//   query row, its row values in registers), dS stored [query][key] into shared memory, and
//   dK_j += dS^T Q_t,i with dS^T read MN-major from that tile (t = the trained distribution).
// Issue order per tile: S_i | (S_i read) S_{i+1} | (dS_i stored) dK_i: the next scores overlap this
// tile's element work.  TMEM: S_a [0,128), S_b [128,256), dK [256,256+d).
template <int D, bool CAUSAL, bool BF16, int OP>
__global__ void __launch_bounds__(kKlDkThreads, 1) kl_dk_kernel(const __grid_constant__ KlArgs a) {
  using C = KlDkCfg<D>;
  constexpr int NS = C::NS;
  constexpr bool STUDENT = (OP == kPairKlStudent);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  if (!smem_base_aligned(sbase, a.err_word)) return;
  uint8_t* gbase = smem_raw;
  const uint32_t sKa = sbase + C::OFF_KA, sKb = sbase + C::OFF_KB, sDS = sbase + C::OFF_DS;
  const uint32_t sRing = sbase + C::OFF_RING;
  const KlDkBars bars{sbase + C::OFF_BAR, NS};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + C::OFF_MISC + 4);
  const WaitCtx wc{abort_flag, a.err_word, a.timeout_ns};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int head = bh % a.heads, batch = bh / a.heads;
  const int jb = blockIdx.y;  // key tile; causal work decreases with jb
  const int k0 = jb * kTileRows;
  const int nq_tiles = (a.Nq + kTileRows - 1) / kTileRows;
  const int coff = CAUSAL ? a.causal_off : 0;
  const int i_start = CAUSAL ? max(0, k0 - coff) / kTileRows : 0;  // first query tile with a row that sees key k0
  const int n = max(0, nq_tiles - i_start);

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    mbar_init(bars.kv_full(), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bars.q_full(s), 1);
      mbar_init(bars.q_empty(s), 1);
    }
    mbar_init(bars.s_full(), 1);
    mbar_init(bars.s_used(), kTileRows);
    mbar_init(bars.ds_ready(), kTileRows);
    mbar_init(bars.ds_free(), 1);
    mbar_init(bars.done(), 1);
    mbar_init(bars.mma_done(), 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tSa = tmem, tSb = tmem + 128, tdK = tmem + 256;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0) {
      prefetch_tmap(&a.tm_qa);
      prefetch_tmap(&a.tm_qb);
      mbar_arrive_expect_tx(bars.kv_full(), 2 * C::TILE);
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_4d(sKa + c * kChunkBytes, &a.tm_ka, c * 64, k0, head, batch, bars.kv_full());
        tma_load_4d(sKb + c * kChunkBytes, &a.tm_kb, c * 64, k0, head, batch, bars.kv_full());
      }
      int issued = 0;
      for (int it = 0; it < n; ++it) {
        const int s = it % NS;
        if (!mbar_wait(bars.q_empty(s), ((it / NS) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(bars.q_full(s), 2 * C::TILE);
        const uint32_t dst = sRing + s * 2 * C::TILE;
        const int q_row = (i_start + it) * kTileRows;
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_4d(dst + c * kChunkBytes, &a.tm_qa, c * 64, q_row, head, batch, bars.q_full(s));
          tma_load_4d(dst + C::TILE + c * kChunkBytes, &a.tm_qb, c * 64, q_row, head, batch, bars.q_full(s));
        }
        ++issued;
      }
      if (*abort_flag) {
        for (int it = max(0, issued - NS); it < issued; ++it) mbar_drain(bars.q_full(it % NS), (it / NS) & 1, a.timeout_ns);
        mbar_drain(bars.kv_full(), 0, a.timeout_ns);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idS = idesc_f16(128, 128, BF16, false, false);  // Q K-major x K K-major
      constexpr uint32_t idK = idesc_f16(128, D, BF16, true, true);      // A = dS^T MN-major, B = Q MN-major
      constexpr uint32_t kTileLo = C::TILE >> 4;
      const uint32_t ka_kmaj = sdesc_lo(sKa, 16), kb_kmaj = sdesc_lo(sKb, 16);
      const uint32_t ring_kmaj = sdesc_lo(sRing, 16), ring_mn = sdesc_lo(sRing, kChunkBytes);
      const uint32_t ds_mn = sdesc_lo(sDS, kChunkBytes);
      auto scores = [&](uint32_t d, uint32_t q_lo, uint32_t b_lo) {
        mma_ss_lo<false>(d, q_lo, b_lo, idS);
#pragma unroll
        for (int k = 1; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * kChunkBytes + (k & 3) * 32) >> 4;
          mma_ss_lo<true>(d, q_lo + off, b_lo + off, idS);
        }
      };
      auto issue_S = [&](int it) -> bool {
        const int s = it % NS;
        if (!mbar_wait(bars.q_full(s), (it / NS) & 1, wc)) return false;
        tc_fence_after();
        scores(tSa, ring_kmaj + (2 * s) * kTileLo, ka_kmaj);
        scores(tSb, ring_kmaj + (2 * s + 1) * kTileLo, kb_kmaj);
        mma_commit(bars.s_full());
        return true;
      };
      bool ok = mbar_wait(bars.kv_full(), 0, wc);
      if (ok) ok = issue_S(0);
      for (int it = 0; ok && it < n; ++it) {
        // the next scores overwrite S_a/S_b once this tile's are in registers
        if (it + 1 < n) {
          if (!(ok = mbar_wait(bars.s_used(), it & 1, wc))) break;
          tc_fence_after();
          if (!(ok = issue_S(it + 1))) break;
        }
        if (!(ok = mbar_wait(bars.ds_ready(), it & 1, wc))) break;
        tc_fence_after();
        // dK += dS^T Q_t  (A: dS^T [key][query] read MN-major from the dS tile; B: Q_t [query][d] MN-major;
        // 16 query rows per K step)
        const int s = it % NS;
        const uint32_t q_lo = ring_mn + (2 * s + (STUDENT ? 1 : 0)) * kTileLo;
        mma_ss_lo_rt(tdK, ds_mn, q_lo, idK, it > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 1; k < 128 / 16; ++k) mma_ss_lo<true>(tdK, ds_mn + k * (2048 >> 4), q_lo + k * (2048 >> 4), idK);
        mma_commit(bars.ds_free());
        mma_commit(bars.q_empty(s));
      }
      if (ok) mma_commit(bars.done());
      mma_commit(bars.mma_done());
      mbar_drain(bars.mma_done(), 0, a.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ compute (thread = query row)
    const int r = warp * 32 + lane;
    const uint32_t lane_bits = static_cast<uint32_t>(warp * 32) << 16;
    const float c_log2 = a.scale * 1.4426950408889634f;
    const float* rv[4] = {a.lse1, a.lse2, a.kl, a.g};
    const bool ragged_kv = k0 + kTileRows > a.Nk;
    bool ok = true;
    for (int it = 0; ok && it < n; ++it) {
      const int q0 = (i_start + it) * kTileRows, row = q0 + r;
      DsOp<OP, BF16> op;
      op.load(rv, static_cast<size_t>(bh) * a.Nq + row, row < a.Nq);
      if (!(ok = mbar_wait_warp(bars.s_full(), it & 1, wc))) break;
      tc_fence_after();
      const bool need_mask = ragged_kv || (CAUSAL && q0 + coff < k0 + kTileRows - 1);
      const int lim = need_mask ? (CAUSAL ? min(a.Nk, row + coff + 1) : a.Nk) - k0 : kTileRows;
      uint32_t pk[2][32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // key columns [64h, 64h + 64)
        uint32_t va[2][32], vb[2][32];
        tmem_ld32(tSa + lane_bits + h * 64, va[0]);
        tmem_ld32(tSa + lane_bits + h * 64 + 32, va[1]);
        tmem_ld32(tSb + lane_bits + h * 64, vb[0]);
        tmem_ld32(tSb + lane_bits + h * 64 + 32, vb[1]);
        tmem_wait_ld();
        reg_fence32(va[0]);
        reg_fence32(va[1]);
        reg_fence32(vb[0]);
        reg_fence32(vb[1]);
        if (h == 1) {
          tc_fence_before();
          mbar_arrive(bars.s_used());  // both score tiles are in registers: the next ones may go
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c0 = 2 * i, c1 = 2 * i + 1;
          float d0, d1;
          op.pair(__uint_as_float(va[c0 >> 5][c0 & 31]), __uint_as_float(va[c1 >> 5][c1 & 31]),
                  __uint_as_float(vb[c0 >> 5][c0 & 31]), __uint_as_float(vb[c1 >> 5][c1 & 31]), c_log2, a.scale, d0, d1);
          if (need_mask) {
            if (h * 64 + c0 >= lim) d0 = 0.f;
            if (h * 64 + c1 >= lim) d1 = 0.f;
          }
          pk[h][i] = pack2<BF16>(d0, d1);
        }
      }
      // the previous dK MMA must have read the dS tile
      if (it > 0 && !(ok = mbar_wait_warp(bars.ds_free(), (it - 1) & 1, wc))) break;
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int u = 0; u < 8; ++u)
          st_shared_v4(sDS + h * kChunkBytes + sw128_offset(r, u), pk[h][4 * u], pk[h][4 * u + 1], pk[h][4 * u + 2],
                       pk[h][4 * u + 3]);
      fence_proxy_async_smem();
      mbar_arrive(bars.ds_ready());
    }

    // ------------------------------------------------------------ epilogue: dK * scale, staged in the K_a tile
    if (ok && n > 0) ok = mbar_wait_warp(bars.done(), 0, wc);
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < C::NCH; ++ch) {
        uint32_t o[2][32];
        if (n > 0) {
          tmem_ld32(tdK + lane_bits + ch * 64, o[0]);
          tmem_ld32(tdK + lane_bits + ch * 64 + 32, o[1]);
          tmem_wait_ld();
          reg_fence32(o[0]);
          reg_fence32(o[1]);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[0][i] = o[1][i] = 0u;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int hh = u >> 2, b = (u & 3) * 8;
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack2<BF16>(__uint_as_float(o[hh][b + 2 * e]) * a.scale, __uint_as_float(o[hh][b + 2 * e + 1]) * a.scale);
          st_shared_v4(sKa + ch * kChunkBytes + sw128_offset(r, u), w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (ok && r == 0 && !*abort_flag) {
      for (int ch = 0; ch < C::NCH; ++ch) tma_store_4d(&a.tm_dk, sKa + ch * kChunkBytes, ch * 64, k0, head, batch);
      tma_store_commit();
      tma_store_wait_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge of the slices' five scalars, one thread per query row:
//   M_t = max_s m_t,s,  l_t = sum_s l_t,s 2^(m_t,s - M_t),  acc = sum_s acc_s 2^(m_a,s - M_a),
// then LSE_t = (M_t + log2 l_t) ln 2 and KL = scale acc / l_a + LSE_b - LSE_a.
__global__ void __launch_bounds__(256) kl_combine_kernel(const __grid_constant__ KlArgs a) {
  const size_t rows = static_cast<size_t>(a.bh_count) * a.Nq;
  const size_t o = static_cast<size_t>(blockIdx.x) * 256 + threadIdx.x;
  if (o >= rows) return;
  const size_t plane = static_cast<size_t>(a.splits) * rows;
  float Ma = -INFINITY, Mb = -INFINITY;
  for (int s = 0; s < a.splits; ++s) {
    Ma = fmaxf(Ma, a.part[s * rows + o]);
    Mb = fmaxf(Mb, a.part[plane + s * rows + o]);
  }
  float La = 0.f, Lb = 0.f, A = 0.f;
  for (int s = 0; s < a.splits; ++s) {
    const size_t e = s * rows + o;
    const float ma = a.part[e], mb = a.part[plane + e];
    if (ma != -INFINITY) {
      const float w = ex2_approx(ma - Ma);
      La = fmaf(a.part[2 * plane + e], w, La);
      A = fmaf(a.part[4 * plane + e], w, A);
    }
    if (mb != -INFINITY) Lb = fmaf(a.part[3 * plane + e], ex2_approx(mb - Mb), Lb);
  }
  if (La > 0.f) {
    const float lse_a = (Ma + __log2f(La)) * 0.6931471805599453f;
    const float lse_b = (Mb + __log2f(Lb)) * 0.6931471805599453f;
    a.lse1[o] = lse_a;
    a.lse2[o] = lse_b;
    a.kl[o] = a.scale * A / La + lse_b - lse_a;
  } else {
    a.lse1[o] = -INFINITY;
    a.lse2[o] = -INFINITY;
    a.kl[o] = 0.f;
  }
}

// ====================================================================== launchers

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_kl_fwd_t(const KlArgs& a, cudaStream_t stream) {
  using C = KlFwdCfg<D>;
  const bool split = a.splits > 1;
  auto kern = split ? kl_fwd_kernel<D, CAUSAL, BF16, true> : kl_fwd_kernel<D, CAUSAL, BF16, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(a.bh_count, (a.Nq + kTileRows - 1) / kTileRows, split ? a.splits : 1);
  kern<<<grid, kKlFwdThreads, C::BYTES, stream>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess || !split) return e;
  const size_t rows = static_cast<size_t>(a.bh_count) * a.Nq;
  kl_combine_kernel<<<static_cast<unsigned>((rows + 255) / 256), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

template <int D, bool CAUSAL, bool BF16, int OP>
cudaError_t launch_kl_dk_t(const KlArgs& a, cudaStream_t stream) {
  using C = KlDkCfg<D>;
  auto kern = kl_dk_kernel<D, CAUSAL, BF16, OP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(a.bh_count, (a.Nk + kTileRows - 1) / kTileRows, 1);
  kern<<<grid, kKlDkThreads, C::BYTES, stream>>>(a);
  return cudaGetLastError();
}

template <int OP>
cudaError_t launch_kl_dk_op(const KlArgs& a, cudaStream_t stream) {
  if (a.d == 64) {
    if (a.causal) return a.bf16 ? launch_kl_dk_t<64, true, true, OP>(a, stream) : launch_kl_dk_t<64, true, false, OP>(a, stream);
    return a.bf16 ? launch_kl_dk_t<64, false, true, OP>(a, stream) : launch_kl_dk_t<64, false, false, OP>(a, stream);
  }
  if (a.causal) return a.bf16 ? launch_kl_dk_t<128, true, true, OP>(a, stream) : launch_kl_dk_t<128, true, false, OP>(a, stream);
  return a.bf16 ? launch_kl_dk_t<128, false, true, OP>(a, stream) : launch_kl_dk_t<128, false, false, OP>(a, stream);
}

}  // namespace

cudaError_t launch_kl_fwd(const KlArgs& a, cudaStream_t stream) {
  if (a.d == 64) {
    if (a.causal) return a.bf16 ? launch_kl_fwd_t<64, true, true>(a, stream) : launch_kl_fwd_t<64, true, false>(a, stream);
    return a.bf16 ? launch_kl_fwd_t<64, false, true>(a, stream) : launch_kl_fwd_t<64, false, false>(a, stream);
  }
  if (a.causal) return a.bf16 ? launch_kl_fwd_t<128, true, true>(a, stream) : launch_kl_fwd_t<128, true, false>(a, stream);
  return a.bf16 ? launch_kl_fwd_t<128, false, true>(a, stream) : launch_kl_fwd_t<128, false, false>(a, stream);
}

cudaError_t launch_kl_dk(const KlArgs& a, cudaStream_t stream) {
  return a.op == kPairKlStudent ? launch_kl_dk_op<kPairKlStudent>(a, stream) : launch_kl_dk_op<kPairKlTeacher>(a, stream);
}

}  // namespace exattn
