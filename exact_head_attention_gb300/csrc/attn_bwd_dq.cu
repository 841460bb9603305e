// Query-tile gradient kernel for sm_103a: dQ of one 128-row query tile, keys in a fixed order.
//
// The attention backward parallel over key/value blocks sums every block's dQ
// contribution with atomics, so the summation order (and dQ's last bits) varies
// from run to run.  The StreamKL summary (backward, kernel fusion) names the
// alternative: a separate kernel for dQ.  Here the grid is parallel over query
// tiles (B*H x ceil(Nq/128)); the CTA of tile i walks the key tiles it sees in
// increasing order and recomputes, for each, two score tiles
//     S_a = Q_a K_a^T,  S_b = Q_b K_b^T
// and the gradient of the scores dS = f(S_a, S_b, row values), then adds
// dQ_i += dS K_dq on chip and stores dQ_i (times scale) once: the same bits on
// every run.  The element function f is a policy:
//   attention (SparkAttention Figure 9 terms; a = (Q, K), b = (dO, V), K_dq = K):
//       P = exp2(S_a*scale*log2e - LSE2), rounded to the input dtype as in the
//       key/value-block kernel, and dS = P o (S_b - D)
//   attention KL (StreamKL summary, Methodology 2; a = teacher, b = student):
//       student trained: dS = g (P_b - P_a), K_dq = K_b
//       teacher trained: dS = g P_a (scale (S_a - S_b) + LSE_b - LSE_a - KL), K_dq = K_a
//
// Warp roles (192 threads):
//   warps 0-3  compute (thread = query row = TMEM lane; its row values are registers)
//   warp  4    TMA producer: Q_a and Q_b once, K_a / K_b into two rings; the ring
//              that feeds the dQ MMA is one slot deeper, since its slots are
//              released only after dQ
//   warp  5    MMA issuer (one thread) and TMEM owner
// Tensor memory: S_a double buffer [0,128) / [384,512) (dS packed in pairs over
// the first 64 columns of its S_a), S_b [128,256), dQ [256,256+d).
// Issue order: S_a0 S_b0 S_a1 | (dS_0 ready) S_b1 dQ_0 S_a2 | (dS_1 ready) S_b2 dQ_1 S_a3 | ...:
// the compute warps start on tile j+1 as soon as S_b(j+1) lands, while dQ_j runs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ds_ops.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace exattn {
namespace {

constexpr int kDqThreads = 192;
constexpr uint32_t kChunkBytes = 128 * 128;

// Ring `a` feeds the dQ MMA unless the student's keys do (KL, student trained).
template <int OP>
constexpr bool kDqFromB = (OP == kPairKlStudent);

template <int D, int OP>
struct DqCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = kTileRows * D * 2;
  static constexpr int NS_DQ = (D == 64) ? 4 : 3;     // ring feeding dQ: slots freed after the dQ MMA
  static constexpr int NS_OTHER = (D == 64) ? 4 : 2;  // other ring: slots freed after its score MMA
  static constexpr int NS_A = kDqFromB<OP> ? NS_OTHER : NS_DQ;
  static constexpr int NS_B = kDqFromB<OP> ? NS_DQ : NS_OTHER;
  static constexpr uint32_t OFF_QA = 0;
  static constexpr uint32_t OFF_QB = OFF_QA + TILE;
  static constexpr uint32_t OFF_KA = OFF_QB + TILE;
  static constexpr uint32_t OFF_KB = OFF_KA + NS_A * TILE;
  static constexpr uint32_t OFF_BAR = OFF_KB + NS_B * TILE;
  // q_full, a_full[NS_A], a_empty[NS_A], b_full[NS_B], b_empty[NS_B], s_full[2], sb_full, ds_ready, dq_done, mma_done
  static constexpr int NBAR = 1 + 2 * NS_A + 2 * NS_B + 6;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
};

struct DqBars {
  uint32_t base;
  int na, nb;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t a_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t a_empty(int s) const { return base + 8 * (1 + na + s); }
  __device__ uint32_t b_full(int s) const { return base + 8 * (1 + 2 * na + s); }
  __device__ uint32_t b_empty(int s) const { return base + 8 * (1 + 2 * na + nb + s); }
  __device__ uint32_t at(int k) const { return base + 8 * (1 + 2 * na + 2 * nb + k); }
  __device__ uint32_t s_full(int b) const { return at(b); }
  __device__ uint32_t sb_full() const { return at(2); }
  __device__ uint32_t ds_ready() const { return at(3); }
  __device__ uint32_t dq_done() const { return at(4); }
  __device__ uint32_t mma_done() const { return at(5); }
};

constexpr uint32_t kColSa0 = 0, kColSb = 128, kColDQ = 256, kColSa1 = 384;
__device__ __forceinline__ uint32_t sa_col(int j) { return (j & 1) ? kColSa1 : kColSa0; }

template <int D, bool CAUSAL, bool BF16, int OP>
__global__ void __launch_bounds__(kDqThreads, 1) pair_dq_kernel(const __grid_constant__ PairDqArgs a) {
  using C = DqCfg<D, OP>;
  constexpr int NA = C::NS_A, NB = C::NS_B;
  constexpr bool FROM_B = kDqFromB<OP>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  if (!smem_base_aligned(sbase, a.err_word)) return;
  uint8_t* gbase = smem_raw;
  const uint32_t sQa = sbase + C::OFF_QA, sQb = sbase + C::OFF_QB, sKa = sbase + C::OFF_KA, sKb = sbase + C::OFF_KB;
  const DqBars bars{sbase + C::OFF_BAR, NA, NB};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + C::OFF_MISC + 4);
  const WaitCtx wc{abort_flag, a.err_word, a.timeout_ns};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int head = bh % a.heads, batch = bh / a.heads;
  const int qt = gridDim.y - 1 - blockIdx.y;  // heaviest (causal) query tiles are scheduled first
  const int q0 = qt * kTileRows;
  const int nkv = (a.Nk + kTileRows - 1) / kTileRows;
  const int coff = CAUSAL ? a.causal_off : 0;
  int n = nkv;  // key tiles this query tile sees
  if (CAUSAL) {
    const int last_key = q0 + kTileRows - 1 + coff;
    n = last_key < 0 ? 0 : min(nkv, last_key / kTileRows + 1);
  }

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    mbar_init(bars.q_full(), 1);
    for (int s = 0; s < NA; ++s) {
      mbar_init(bars.a_full(s), 1);
      mbar_init(bars.a_empty(s), 1);
    }
    for (int s = 0; s < NB; ++s) {
      mbar_init(bars.b_full(s), 1);
      mbar_init(bars.b_empty(s), 1);
    }
    mbar_init(bars.s_full(0), 1);
    mbar_init(bars.s_full(1), 1);
    mbar_init(bars.sb_full(), 1);
    mbar_init(bars.ds_ready(), kTileRows);
    mbar_init(bars.dq_done(), 1);
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

  if (warp == 4) {
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
      int issued_a = 0, issued_b = 0;
      for (int j = 0; j < n; ++j) {
        const int sa = j % NA, sb = j % NB;
        if (!mbar_wait(bars.a_empty(sa), ((j / NA) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(bars.a_full(sa), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_4d(sKa + sa * C::TILE + c * kChunkBytes, &a.tm_ka, c * 64, j * kTileRows, head, batch, bars.a_full(sa));
        ++issued_a;
        if (!mbar_wait(bars.b_empty(sb), ((j / NB) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(bars.b_full(sb), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_4d(sKb + sb * C::TILE + c * kChunkBytes, &a.tm_kb, c * 64, j * kTileRows, head, batch, bars.b_full(sb));
        ++issued_b;
      }
      if (*abort_flag) {
        for (int j = max(0, issued_a - NA); j < issued_a; ++j) mbar_drain(bars.a_full(j % NA), (j / NA) & 1, a.timeout_ns);
        for (int j = max(0, issued_b - NB); j < issued_b; ++j) mbar_drain(bars.b_full(j % NB), (j / NB) & 1, a.timeout_ns);
        mbar_drain(bars.q_full(), 0, a.timeout_ns);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idS = idesc_f16(128, 128, BF16, false, false);  // K-major x K-major
      constexpr uint32_t idQ = idesc_f16(128, D, BF16, false, true);     // A = dS (TMEM), B = keys MN-major
      constexpr uint32_t kTileLo = C::TILE >> 4;
      const uint32_t qa_lo = sdesc_lo(sQa, 16), qb_lo = sdesc_lo(sQb, 16);
      const uint32_t ka_kmaj = sdesc_lo(sKa, 16), kb_kmaj = sdesc_lo(sKb, 16);
      const uint32_t kdq_mn = sdesc_lo(FROM_B ? sKb : sKa, kChunkBytes);
      auto scores = [&](uint32_t d, uint32_t q_lo, uint32_t b_lo) {
        mma_ss_lo<false>(d, q_lo, b_lo, idS);
#pragma unroll
        for (int k = 1; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * kChunkBytes + (k & 3) * 32) >> 4;
          mma_ss_lo<true>(d, q_lo + off, b_lo + off, idS);
        }
      };
      // S_a(j) into its buffer
      auto issue_Sa = [&](int j) -> bool {
        const int s = j % NA;
        if (!mbar_wait(bars.a_full(s), (j / NA) & 1, wc)) return false;
        tc_fence_after();
        scores(tmem + sa_col(j), qa_lo, ka_kmaj + s * kTileLo);
        mma_commit(bars.s_full(j & 1));
        if (FROM_B) mma_commit(bars.a_empty(s));
        return true;
      };
      // S_b(j)
      auto issue_Sb = [&](int j) -> bool {
        const int s = j % NB;
        if (!mbar_wait(bars.b_full(s), (j / NB) & 1, wc)) return false;
        tc_fence_after();
        scores(tmem + kColSb, qb_lo, kb_kmaj + s * kTileLo);
        mma_commit(bars.sb_full());
        if (!FROM_B) mma_commit(bars.b_empty(s));
        return true;
      };
      bool ok = mbar_wait(bars.q_full(), 0, wc);
      if (ok) ok = issue_Sa(0);
      if (ok) ok = issue_Sb(0);
      if (ok && n > 1) ok = issue_Sa(1);
      for (int j = 0; ok && j < n; ++j) {
        if (!(ok = mbar_wait(bars.ds_ready(), j & 1, wc))) break;  // dS_j packed in TMEM, S_b(j) read
        tc_fence_after();
        if (j + 1 < n && !(ok = issue_Sb(j + 1))) break;
        // dQ += dS_j K_dq(j)  (A: dS_j packed in its S_a buffer; B: keys [key][d], 16 keys per K step)
        const int s = j % (FROM_B ? NB : NA);
        const uint32_t pa = tmem + sa_col(j), b_lo = kdq_mn + s * kTileLo;
        mma_ts_lo_rt(tmem + kColDQ, pa, b_lo, idQ, j > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 1; k < kTileRows / 16; ++k) mma_ts_lo<true>(tmem + kColDQ, pa + k * 8, b_lo + k * (2048 >> 4), idQ);
        mma_commit(FROM_B ? bars.b_empty(s) : bars.a_empty(s));
        if (j == n - 1) mma_commit(bars.dq_done());
        // S_a(j+2) overwrites buffer j & 1 after dQ_j has read dS_j from it (one thread's MMAs run in order)
        if (j + 2 < n && !(ok = issue_Sa(j + 2))) break;
      }
      mma_commit(bars.mma_done());
      mbar_drain(bars.mma_done(), 0, a.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ compute
    const int r = warp * 32 + lane;  // query row inside the tile = TMEM lane
    const int row = q0 + r;
    const uint32_t lane_bits = static_cast<uint32_t>(warp * 32) << 16;
    const float c_log2 = a.scale * 1.4426950408889634f;
    DsOp<OP, BF16> op;
    op.load(a.rv, static_cast<size_t>(bh) * a.rv_stride + row, row < a.Nq);
    bool ok = true;
    for (int j = 0; ok && j < n; ++j) {
      if (!(ok = mbar_wait_warp(bars.s_full(j & 1), (j >> 1) & 1, wc))) break;
      if (!(ok = mbar_wait_warp(bars.sb_full(), j & 1, wc))) break;
      tc_fence_after();
      const uint32_t tSa = tmem + sa_col(j) + lane_bits, tSb = tmem + kColSb + lane_bits;
      // keys at or past `lim` are masked (ragged last key tile, tiles the causal diagonal crosses)
      const bool need_mask =
          ((j + 1) * kTileRows > a.Nk) || (CAUSAL && j * kTileRows + kTileRows - 1 > q0 + coff);
      const int lim = need_mask ? (CAUSAL ? min(a.Nk, row + coff + 1) : a.Nk) - j * kTileRows : kTileRows;
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // key columns [64h, 64h + 64) -> packed columns [32h, 32h + 32)
        uint32_t va[2][32], vb[2][32];
        tmem_ld32(tSa + h * 64, va[0]);
        tmem_ld32(tSa + h * 64 + 32, va[1]);
        tmem_ld32(tSb + h * 64, vb[0]);
        tmem_ld32(tSb + h * 64 + 32, vb[1]);
        tmem_wait_ld();
        reg_fence32(va[0]);
        reg_fence32(va[1]);
        reg_fence32(vb[0]);
        reg_fence32(vb[1]);
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c0 = 2 * i, c1 = 2 * i + 1;  // columns inside this half
          float ds0, ds1;
          op.pair(__uint_as_float(va[c0 >> 5][c0 & 31]), __uint_as_float(va[c1 >> 5][c1 & 31]),
                  __uint_as_float(vb[c0 >> 5][c0 & 31]), __uint_as_float(vb[c1 >> 5][c1 & 31]), c_log2, a.scale, ds0, ds1);
          if (need_mask) {
            if (h * 64 + c0 >= lim) ds0 = 0.f;
            if (h * 64 + c1 >= lim) ds1 = 0.f;
          }
          pk[i] = pack2<BF16>(ds0, ds1);
        }
        tmem_st32(tSa + h * 32, pk);  // packed columns [32h, 32h + 32): scores there were read already
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bars.ds_ready());
    }

    // ------------------------------------------------------------ epilogue: dQ * scale, staged in the Q_a tile
    // (n == 0: nothing was loaded or accumulated; the tile's dQ is zero.)
    if (ok && n > 0) ok = mbar_wait_warp(bars.dq_done(), 0, wc);
    if (ok) {
      tc_fence_after();
      const uint32_t tQ = tmem + kColDQ + lane_bits;
#pragma unroll
      for (int ch = 0; ch < C::NCH; ++ch) {
        uint32_t o[2][32];
        if (n > 0) {
          tmem_ld32(tQ + ch * 64, o[0]);
          tmem_ld32(tQ + ch * 64 + 32, o[1]);
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
          st_shared_v4(sQa + ch * kChunkBytes + sw128_offset(r, u), w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (ok && r == 0 && !*abort_flag) {
      for (int ch = 0; ch < C::NCH; ++ch) tma_store_4d(&a.tm_dq, sQa + ch * kChunkBytes, ch * 64, q0, head, batch);
      tma_store_commit();
      tma_store_wait_all();
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL, bool BF16, int OP>
cudaError_t launch_pair_t(const PairDqArgs& a, cudaStream_t stream) {
  using C = DqCfg<D, OP>;
  auto kern = pair_dq_kernel<D, CAUSAL, BF16, OP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(a.bh_count, (a.Nq + kTileRows - 1) / kTileRows, 1);
  kern<<<grid, kDqThreads, C::BYTES, stream>>>(a);
  return cudaGetLastError();
}

template <int OP>
cudaError_t launch_pair_op(const PairDqArgs& a, cudaStream_t stream) {
  if (a.d == 64) {
    if (a.causal) return a.bf16 ? launch_pair_t<64, true, true, OP>(a, stream) : launch_pair_t<64, true, false, OP>(a, stream);
    return a.bf16 ? launch_pair_t<64, false, true, OP>(a, stream) : launch_pair_t<64, false, false, OP>(a, stream);
  }
  if (a.causal) return a.bf16 ? launch_pair_t<128, true, true, OP>(a, stream) : launch_pair_t<128, true, false, OP>(a, stream);
  return a.bf16 ? launch_pair_t<128, false, true, OP>(a, stream) : launch_pair_t<128, false, false, OP>(a, stream);
}

}  // namespace

cudaError_t launch_pair_dq(const PairDqArgs& a, cudaStream_t stream) {
  switch (a.op) {
    case kPairAttn: return launch_pair_op<kPairAttn>(a, stream);
    case kPairKlStudent: return launch_pair_op<kPairKlStudent>(a, stream);
    case kPairKlTeacher: return launch_pair_op<kPairKlTeacher>(a, stream);
  }
  return cudaErrorInvalidValue;
}

// The attention backward's deterministic dQ: a = (Q, K), b = (dO, V); per-row values from the
// preprocess (base-2 LSE with +inf on rows without keys, D).
cudaError_t launch_bwd_dq(const BwdArgs& b, cudaStream_t stream) {
  PairDqArgs a;
  a.tm_qa = b.tm_q;
  a.tm_ka = b.tm_k;
  a.tm_qb = b.tm_do;
  a.tm_kb = b.tm_v;
  a.tm_dq = b.tm_dq;
  a.rv[0] = b.nlse2;
  a.rv[1] = b.dsum;
  a.rv[2] = nullptr;
  a.rv[3] = nullptr;
  a.rv_stride = b.Nq_pad;
  a.err_word = b.err_word;
  a.bh_count = b.bh_count;
  a.heads = b.heads;
  a.Nq = b.Nq;
  a.Nk = b.Nk;
  a.d = b.d;
  a.causal = b.causal;
  a.bf16 = b.bf16;
  a.causal_off = b.causal_off;
  a.scale = b.scale;
  a.op = kPairAttn;
  a.timeout_ns = b.timeout_ns;
  return launch_pair_dq(a, stream);
}

}  // namespace exattn
