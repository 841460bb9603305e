// Deterministic dQ for sm_103a: one CTA per 128-row query tile, keys in a fixed order.
//
// The backward pass parallel over key/value blocks sums every block's dQ
// contribution with atomics, so the summation order (and dQ's last bits) varies
// from run to run.  The StreamKL summary (backward, kernel fusion) names the
// alternative: a separate kernel for dQ.  Here the grid is parallel over query
// tiles (B*H x ceil(Nq/128)); the CTA of tile i walks the key tiles it sees in
// increasing order and recomputes, for each (SparkAttention Figure 9 terms):
//     S = Q_i K_j^T,  P = exp2(S*scale*log2e - LSE2_i),  dP = dO_i V_j^T,
//     dS = P o (dP - D_i),  dQ_i += dS K_j
// with dQ_i accumulated in TMEM and stored once (times scale): the result is
// the same bits on every run.  P is rounded to the input dtype before dS, as in
// the key/value-block kernel, so both modes use the same dS.
//
// Warp roles (192 threads):
//   warps 0-3  compute (thread = query row = TMEM lane; its LSE2 and D are scalars)
//   warp  4    TMA producer: Q_i and dO_i once, K_j / V_j into NS-deep rings
//   warp  5    MMA issuer (one thread) and TMEM owner
// Tensor memory: S double buffer [0,128) / [384,512) (dS packed in pairs over
// the first 64 columns of its S), dP [128,256), dQ [256,256+d).
// Issue order: S_0 dP_0 S_1 | (dS_0 ready) dP_1 dQ_0 S_2 | (dS_1 ready) dP_2 dQ_1 S_3 | ...:
// the compute warps start on tile j+1 as soon as dP_{j+1} lands, while dQ_j runs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace exattn {
namespace {

constexpr int kDqThreads = 192;
constexpr uint32_t kChunkBytes = 128 * 128;

template <int D>
struct DqCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = kTileRows * D * 2;
  static constexpr int NS = (D == 64) ? 4 : 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_DO = OFF_Q + TILE;
  static constexpr uint32_t OFF_K = OFF_DO + TILE;
  static constexpr uint32_t OFF_V = OFF_K + NS * TILE;
  static constexpr uint32_t OFF_BAR = OFF_V + NS * TILE;
  // q_full, k_full[NS], k_empty[NS], v_full[NS], v_empty[NS], s_full[2], dp_full, ds_ready, dq_done, mma_done
  static constexpr int NBAR = 1 + 4 * NS + 6;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
};

struct DqBars {
  uint32_t base;
  int ns;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t k_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t k_empty(int s) const { return base + 8 * (1 + ns + s); }
  __device__ uint32_t v_full(int s) const { return base + 8 * (1 + 2 * ns + s); }
  __device__ uint32_t v_empty(int s) const { return base + 8 * (1 + 3 * ns + s); }
  __device__ uint32_t s_full(int b) const { return base + 8 * (1 + 4 * ns + b); }
  __device__ uint32_t dp_full() const { return base + 8 * (3 + 4 * ns); }
  __device__ uint32_t ds_ready() const { return base + 8 * (4 + 4 * ns); }
  __device__ uint32_t dq_done() const { return base + 8 * (5 + 4 * ns); }
  __device__ uint32_t mma_done() const { return base + 8 * (6 + 4 * ns); }
};

constexpr uint32_t kColS0 = 0, kColDP = 128, kColDQ = 256, kColS1 = 384;
__device__ __forceinline__ uint32_t s_col(int j) { return (j & 1) ? kColS1 : kColS0; }

template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kDqThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdArgs a) {
  using C = DqCfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  if (!smem_base_aligned(sbase, a.err_word)) return;
  uint8_t* gbase = smem_raw;
  const uint32_t sQ = sbase + C::OFF_Q, sDO = sbase + C::OFF_DO, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  const DqBars bars{sbase + C::OFF_BAR, NS};
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
    for (int s = 0; s < NS; ++s) {
      mbar_init(bars.k_full(s), 1);
      mbar_init(bars.k_empty(s), 1);
      mbar_init(bars.v_full(s), 1);
      mbar_init(bars.v_empty(s), 1);
    }
    mbar_init(bars.s_full(0), 1);
    mbar_init(bars.s_full(1), 1);
    mbar_init(bars.dp_full(), 1);
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
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_do);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      mbar_arrive_expect_tx(bars.q_full(), 2 * C::TILE);
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_4d(sQ + c * kChunkBytes, &a.tm_q, c * 64, q0, head, batch, bars.q_full());
        tma_load_4d(sDO + c * kChunkBytes, &a.tm_do, c * 64, q0, head, batch, bars.q_full());
      }
      int issued_k = 0, issued_v = 0;
      for (int j = 0; j < n; ++j) {
        const int s = j % NS;
        const uint32_t ph = (j / NS) & 1;
        if (!mbar_wait(bars.k_empty(s), ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(bars.k_full(s), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_4d(sK + s * C::TILE + c * kChunkBytes, &a.tm_k, c * 64, j * kTileRows, head, batch, bars.k_full(s));
        ++issued_k;
        if (!mbar_wait(bars.v_empty(s), ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(bars.v_full(s), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_4d(sV + s * C::TILE + c * kChunkBytes, &a.tm_v, c * 64, j * kTileRows, head, batch, bars.v_full(s));
        ++issued_v;
      }
      if (*abort_flag) {
        for (int j = max(0, issued_k - NS); j < issued_k; ++j) mbar_drain(bars.k_full(j % NS), (j / NS) & 1, a.timeout_ns);
        for (int j = max(0, issued_v - NS); j < issued_v; ++j) mbar_drain(bars.v_full(j % NS), (j / NS) & 1, a.timeout_ns);
        mbar_drain(bars.q_full(), 0, a.timeout_ns);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idS = idesc_f16(128, 128, BF16, false, false);  // K-major x K-major
      constexpr uint32_t idQ = idesc_f16(128, D, BF16, false, true);     // A = dS (TMEM), B = K MN-major
      constexpr uint32_t kTileLo = C::TILE >> 4;
      const uint32_t q_lo = sdesc_lo(sQ, 16), do_lo = sdesc_lo(sDO, 16);
      const uint32_t k_kmaj = sdesc_lo(sK, 16), v_kmaj = sdesc_lo(sV, 16), k_mn = sdesc_lo(sK, kChunkBytes);
      // S_j = Q K_j^T into its buffer (the same operands as the forward's scores)
      auto issue_S = [&](int j) -> bool {
        const int s = j % NS;
        if (!mbar_wait(bars.k_full(s), (j / NS) & 1, wc)) return false;
        tc_fence_after();
        const uint32_t d = tmem + s_col(j), b_lo = k_kmaj + s * kTileLo;
        mma_ss_lo<false>(d, q_lo, b_lo, idS);
#pragma unroll
        for (int k = 1; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * kChunkBytes + (k & 3) * 32) >> 4;
          mma_ss_lo<true>(d, q_lo + off, b_lo + off, idS);
        }
        mma_commit(bars.s_full(j & 1));
        return true;
      };
      // dP_j = dO V_j^T
      auto issue_dP = [&](int j) -> bool {
        const int s = j % NS;
        if (!mbar_wait(bars.v_full(s), (j / NS) & 1, wc)) return false;
        tc_fence_after();
        const uint32_t d = tmem + kColDP, b_lo = v_kmaj + s * kTileLo;
        mma_ss_lo<false>(d, do_lo, b_lo, idS);
#pragma unroll
        for (int k = 1; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * kChunkBytes + (k & 3) * 32) >> 4;
          mma_ss_lo<true>(d, do_lo + off, b_lo + off, idS);
        }
        mma_commit(bars.dp_full());
        mma_commit(bars.v_empty(s));
        return true;
      };
      bool ok = mbar_wait(bars.q_full(), 0, wc);
      if (ok) ok = issue_S(0);
      if (ok) ok = issue_dP(0);
      if (ok && n > 1) ok = issue_S(1);
      for (int j = 0; ok && j < n; ++j) {
        if (!(ok = mbar_wait(bars.ds_ready(), j & 1, wc))) break;  // dS_j packed in TMEM, dP_j read
        tc_fence_after();
        if (j + 1 < n && !(ok = issue_dP(j + 1))) break;
        // dQ += dS_j K_j  (A: dS_j packed in its S buffer; B: K_j [key][d], 16 keys per K step)
        const int s = j % NS;
        const uint32_t pa = tmem + s_col(j), b_lo = k_mn + s * kTileLo;
        mma_ts_lo_rt(tmem + kColDQ, pa, b_lo, idQ, j > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 1; k < kTileRows / 16; ++k) mma_ts_lo<true>(tmem + kColDQ, pa + k * 8, b_lo + k * (2048 >> 4), idQ);
        mma_commit(bars.k_empty(s));
        if (j == n - 1) mma_commit(bars.dq_done());
        // S_{j+2} overwrites buffer j & 1 after dQ_j has read dS_j from it (one thread's MMAs run in order)
        if (j + 2 < n && !(ok = issue_S(j + 2))) break;
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
    const size_t vrow = static_cast<size_t>(bh) * a.Nq_pad + row;  // rows past Nq: LSE2 = +inf, D = 0
    const float lse2 = a.lse2[vrow], dsum = a.dsum[vrow];
    bool ok = true;
    for (int j = 0; ok && j < n; ++j) {
      if (!(ok = mbar_wait_warp(bars.s_full(j & 1), (j >> 1) & 1, wc))) break;
      if (!(ok = mbar_wait_warp(bars.dp_full(), j & 1, wc))) break;
      tc_fence_after();
      const uint32_t tS = tmem + s_col(j) + lane_bits, tP = tmem + kColDP + lane_bits;
      // keys at or past `lim` are masked (ragged last key tile, tiles the causal diagonal crosses)
      const bool need_mask =
          ((j + 1) * kTileRows > a.Nk) || (CAUSAL && j * kTileRows + kTileRows - 1 > q0 + coff);
      const int lim = need_mask ? (CAUSAL ? min(a.Nk, row + coff + 1) : a.Nk) - j * kTileRows : kTileRows;
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // key columns [64h, 64h + 64) -> packed columns [32h, 32h + 32)
        uint32_t sv[2][32], pv[2][32];
        tmem_ld32(tS + h * 64, sv[0]);
        tmem_ld32(tS + h * 64 + 32, sv[1]);
        tmem_ld32(tP + h * 64, pv[0]);
        tmem_ld32(tP + h * 64 + 32, pv[1]);
        tmem_wait_ld();
        reg_fence32(sv[0]);
        reg_fence32(sv[1]);
        reg_fence32(pv[0]);
        reg_fence32(pv[1]);
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c0 = 2 * i, c1 = 2 * i + 1;  // columns inside this half
          float p0 = ex2_approx(fmaf(__uint_as_float(sv[c0 >> 5][c0 & 31]), c_log2, -lse2));
          float p1 = ex2_approx(fmaf(__uint_as_float(sv[c1 >> 5][c1 & 31]), c_log2, -lse2));
          if (need_mask) {
            if (h * 64 + c0 >= lim) p0 = 0.f;
            if (h * 64 + c1 >= lim) p1 = 0.f;
          }
          // P rounded to the input dtype, as the key/value-block kernel uses it
          const uint32_t pp = pack2<BF16>(p0, p1);
          const float ds0 = unpack_lo<BF16>(pp) * (__uint_as_float(pv[c0 >> 5][c0 & 31]) - dsum);
          const float ds1 = unpack_hi<BF16>(pp) * (__uint_as_float(pv[c1 >> 5][c1 & 31]) - dsum);
          pk[i] = pack2<BF16>(ds0, ds1);
        }
        tmem_st32(tS + h * 32, pk);  // packed columns [32h, 32h + 32): scores there were read already
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bars.ds_ready());
    }

    // ------------------------------------------------------------ epilogue: dQ * scale, staged in the Q tile
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
          st_shared_v4(sQ + ch * kChunkBytes + sw128_offset(r, u), w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (ok && r == 0 && !*abort_flag) {
      for (int ch = 0; ch < C::NCH; ++ch) tma_store_4d(&a.tm_dq, sQ + ch * kChunkBytes, ch * 64, q0, head, batch);
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

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_dq_t(const BwdArgs& a, cudaStream_t stream) {
  using C = DqCfg<D>;
  auto kern = bwd_dq_kernel<D, CAUSAL, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(a.bh_count, (a.Nq + kTileRows - 1) / kTileRows, 1);
  kern<<<grid, kDqThreads, C::BYTES, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t stream) {
  if (a.d == 64) {
    if (a.causal) return a.bf16 ? launch_dq_t<64, true, true>(a, stream) : launch_dq_t<64, true, false>(a, stream);
    return a.bf16 ? launch_dq_t<64, false, true>(a, stream) : launch_dq_t<64, false, false>(a, stream);
  }
  if (a.causal) return a.bf16 ? launch_dq_t<128, true, true>(a, stream) : launch_dq_t<128, true, false>(a, stream);
  return a.bf16 ? launch_dq_t<128, false, true>(a, stream) : launch_dq_t<128, false, false>(a, stream);
}

}  // namespace exattn
