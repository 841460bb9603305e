// Split-KV forward for few query rows (decoding: Nq = 1 .. a few hundred) on sm_103a.
//
// With few query rows, B*H*ceil(Nq/256) forward blocks leave most SMs idle.
// The StreamKL summary (GPU kernel optimisations, "Split-K variant") restores
// the parallelism by dividing the key dimension across thread blocks: here the
// grid is (B*H, ceil(Nq/128), splits), and block (bh, qt, s) runs the online
// softmax of query tile qt over the s-th contiguous slice of the key tiles that
// tile sees.  It writes the slice's O, normalised by the slice's own sum, and the
// slice's base-2 LSE to fp32 workspace.  fwd_combine_kernel then merges the
// slices of every query row:
//     L = log2 sum_s 2^{L_s},  O = sum_s 2^{L_s - L} O_s,  LSE = L ln 2,
// exact up to rounding (a slice that saw no key has L_s = -inf and weight 0).
// The merge is a dependent launch: it starts while the last slice blocks run
// and waits for the slice kernel before it reads anything.
//
// At d = 64 the slices run on the one-tile body of fwd_tile.cuh (two slice
// blocks per SM).  At d = 128, warp roles of the slice kernel (192 threads):
//   warps 0-3  softmax warpgroup (thread = query row = TMEM lane)
//   warp  4    TMA producer: Q once, then K_j / V_j into NS-deep rings
//   warp  5    MMA issuer (one thread) and TMEM owner
// Tensor memory: S double buffer [0,128) / [128,256) (P packed over the first
// 64 columns of its S), O accumulator [256, 256+d).  Issue order S_0 S_1 |
// PV_0 S_2 | PV_1 S_3 | ...: the next tile's scores are ready while the softmax
// works on this one.  Because S_{i+1} is issued before PV_i, a rescale of O at
// tile i+1 first waits for PV_i (pv_done); o_full marks the last PV.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fwd_tile.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "softmax.cuh"

namespace exattn {
namespace {

constexpr int kSplitThreads = 192;
constexpr uint32_t kChunkBytes = 128 * 128;  // 128 rows x 128 bytes

template <int D>
struct SplitCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = kTileRows * D * 2;
  static constexpr int NS = (D == 64) ? 6 : 3;  // K and V ring depth (K/V bytes in flight per SM)
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + TILE;
  static constexpr uint32_t OFF_V = OFF_K + NS * TILE;
  static constexpr uint32_t OFF_BAR = OFF_V + NS * TILE;
  // q_full, k_full[NS], k_empty[NS], v_full[NS], v_empty[NS], s_full[2], p_full[2], pv_done, o_full, mma_done
  static constexpr int NBAR = 1 + 4 * NS + 7;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;  // tmem slot (4 B) + abort flag (4 B)
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
  static_assert(TILE % 1024 == 0, "operand tiles stay 1024-byte aligned");
};

struct SplitBars {
  uint32_t base;
  int ns;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t k_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t k_empty(int s) const { return base + 8 * (1 + ns + s); }
  __device__ uint32_t v_full(int s) const { return base + 8 * (1 + 2 * ns + s); }
  __device__ uint32_t v_empty(int s) const { return base + 8 * (1 + 3 * ns + s); }
  __device__ uint32_t s_full(int b) const { return base + 8 * (1 + 4 * ns + b); }
  __device__ uint32_t p_full(int b) const { return base + 8 * (3 + 4 * ns + b); }
  __device__ uint32_t pv_done() const { return base + 8 * (5 + 4 * ns); }
  __device__ uint32_t o_full() const { return base + 8 * (6 + 4 * ns); }
  __device__ uint32_t mma_done() const { return base + 8 * (7 + 4 * ns); }
};

template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kSplitThreads, 1) fwd_split_kernel(const __grid_constant__ SplitArgs a) {
  // The merge kernel is a dependent launch: it may start once every slice block is running, and waits
  // for this kernel to finish before it reads the slices.
  griddep_launch_dependents();
  using C = SplitCfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  if (!smem_base_aligned(sbase, a.err_word)) return;
  uint8_t* gbase = smem_raw;
  const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  const SplitBars bars{sbase + C::OFF_BAR, NS};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + C::OFF_MISC + 4);
  const WaitCtx wc{abort_flag, a.err_word, a.timeout_ns};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int head = bh % a.heads, batch = bh / a.heads;
  const int q0 = blockIdx.y * kTileRows;
  const int split = blockIdx.z;
  const int nkv = (a.Nk + kTileRows - 1) / kTileRows;
  const int coff = CAUSAL ? a.causal_off : 0;
  // key tiles this query tile sees (causal: through the tile of the last key its last row sees)
  int nvis = nkv;
  if (CAUSAL) {
    const int last_key = q0 + kTileRows - 1 + coff;
    nvis = last_key < 0 ? 0 : min(nkv, last_key / kTileRows + 1);
  }
  // this block's slice [j0, j0 + n): slices differ in length by at most one tile
  const int j0 = static_cast<int>(static_cast<long long>(split) * nvis / a.splits);
  const int n = static_cast<int>(static_cast<long long>(split + 1) * nvis / a.splits) - j0;

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    mbar_init(bars.q_full(), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bars.k_full(s), 1);
      mbar_init(bars.k_empty(s), 1);
      mbar_init(bars.v_full(s), 1);
      mbar_init(bars.v_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.s_full(b), 1);
      mbar_init(bars.p_full(b), kTileRows);
    }
    mbar_init(bars.pv_done(), 1);
    mbar_init(bars.o_full(), 1);
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
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      mbar_arrive_expect_tx(bars.q_full(), C::TILE);
      for (int c = 0; c < C::NCH; ++c)
        tma_load_4d(sQ + c * kChunkBytes, &a.tm_q, c * 64, q0, head, batch, bars.q_full());
      int issued_k = 0, issued_v = 0;
      for (int i = 0; i < n; ++i) {
        const int s = i % NS;
        const uint32_t ph = (i / NS) & 1;
        const int row = (j0 + i) * kTileRows;
        if (!mbar_wait(bars.k_empty(s), ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(bars.k_full(s), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_4d(sK + s * C::TILE + c * kChunkBytes, &a.tm_k, c * 64, row, head, batch, bars.k_full(s));
        ++issued_k;
        if (!mbar_wait(bars.v_empty(s), ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(bars.v_full(s), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_4d(sV + s * C::TILE + c * kChunkBytes, &a.tm_v, c * 64, row, head, batch, bars.v_full(s));
        ++issued_v;
      }
      // On abort, every load this thread issued must land before the CTA exits.
      if (*abort_flag) {
        for (int i = max(0, issued_k - NS); i < issued_k; ++i) mbar_drain(bars.k_full(i % NS), (i / NS) & 1, a.timeout_ns);
        for (int i = max(0, issued_v - NS); i < issued_v; ++i) mbar_drain(bars.v_full(i % NS), (i / NS) & 1, a.timeout_ns);
        mbar_drain(bars.q_full(), 0, a.timeout_ns);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idS = idesc_f16(128, 128, BF16, false, false);
      constexpr uint32_t idPV = idesc_f16(128, D, BF16, false, true);
      constexpr uint32_t kTileLo = C::TILE >> 4;
      const uint32_t q_lo = sdesc_lo(sQ, 16), k_lo = sdesc_lo(sK, 16), v_lo = sdesc_lo(sV, kChunkBytes);
      // S_i = Q K_i^T into buffer i & 1
      auto issue_S = [&](int i) -> bool {
        const int s = i % NS;
        if (!mbar_wait(bars.k_full(s), (i / NS) & 1, wc)) return false;
        tc_fence_after();
        const uint32_t d = tmem + (i & 1) * 128, b_lo = k_lo + s * kTileLo;
        mma_ss_lo<false>(d, q_lo, b_lo, idS);
#pragma unroll
        for (int k = 1; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * kChunkBytes + (k & 3) * 32) >> 4;
          mma_ss_lo<true>(d, q_lo + off, b_lo + off, idS);
        }
        mma_commit(bars.s_full(i & 1));
        mma_commit(bars.k_empty(s));
        return true;
      };
      // O += P_i V_i, P_i read from TMEM buffer i & 1
      auto issue_PV = [&](int i) -> bool {
        const int s = i % NS;
        if (!mbar_wait(bars.v_full(s), (i / NS) & 1, wc)) return false;
        if (!mbar_wait(bars.p_full(i & 1), (i >> 1) & 1, wc)) return false;
        tc_fence_after();
        const uint32_t d = tmem + 256, pa = tmem + (i & 1) * 128, b_lo = v_lo + s * kTileLo;
        mma_ts_lo_rt(d, pa, b_lo, idPV, i > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 1; k < kTileRows / 16; ++k) mma_ts_lo<true>(d, pa + k * 8, b_lo + k * (2048 >> 4), idPV);
        mma_commit(bars.v_empty(s));
        mma_commit(bars.pv_done());
        return true;
      };
      bool ok = mbar_wait(bars.q_full(), 0, wc);
      if (ok) ok = issue_S(0);
      if (ok && n > 1) ok = issue_S(1);
      for (int i = 0; ok && i < n; ++i) {
        if (!(ok = issue_PV(i))) break;
        if (i == n - 1) mma_commit(bars.o_full());
        // S_{i+2} overwrites buffer i & 1 after PV_i has read P_i from it (one thread's MMAs run in order)
        if (i + 2 < n && !(ok = issue_S(i + 2))) break;
      }
      mma_commit(bars.mma_done());
      mbar_drain(bars.mma_done(), 0, a.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = warp * 32 + lane;  // row inside the tile = TMEM lane
    const int row = q0 + r;
    const uint32_t lane_bits = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tO = tmem + 256 + lane_bits;
    const float c_log2 = a.scale * 1.4426950408889634f;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      if (!(ok = mbar_wait_warp(bars.s_full(i & 1), (i >> 1) & 1, wc))) break;
      tc_fence_after();
      const int j = j0 + i;
      const bool need_mask =
          ((j + 1) * kTileRows > a.Nk) || (CAUSAL && j * kTileRows + kTileRows - 1 > q0 + coff);
      const int lim = need_mask ? (CAUSAL ? min(a.Nk, row + coff + 1) : a.Nk) - j * kTileRows : kTileRows;
      const uint32_t tS = tmem + (i & 1) * 128 + lane_bits;
      // PV_{i-1} was issued after S_i: it must have finished before O is rescaled.
      auto wait_pv = [&] {
        if (!mbar_wait_warp(bars.pv_done(), (i - 1) & 1, wc)) ok = false;
        tc_fence_after();
      };
      if (need_mask)
        softmax_tile<D, true, BF16>(tS, tO, lim, c_log2, i == 0, m, l, wait_pv);
      else
        softmax_tile<D, false, BF16>(tS, tO, lim, c_log2, i == 0, m, l, wait_pv);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bars.p_full(i & 1));
      if (!ok) break;
    }

    // ------------------------------------------------------------ slice epilogue
    if (ok && n > 0) ok = mbar_wait_warp(bars.o_full(), 0, wc);
    if (ok) {
      tc_fence_after();
      const size_t prow = (static_cast<size_t>(split) * a.bh_count + bh) * a.Nq + row;
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      if (row < a.Nq) a.l_part[prow] = l > 0.f ? m + __log2f(l) : -INFINITY;
      float4* dst = reinterpret_cast<float4*>(a.o_part + prow * D);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (n > 0) {
          tmem_ld32(tO + c * 32, o);  // warp-collective: every lane loads, only real rows store
          tmem_wait_ld();
          reg_fence32(o);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (row < a.Nq) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[c * 8 + e] = make_float4(__uint_as_float(o[4 * e]) * inv_l, __uint_as_float(o[4 * e + 1]) * inv_l,
                                         __uint_as_float(o[4 * e + 2]) * inv_l, __uint_as_float(o[4 * e + 3]) * inv_l);
        }
      }
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

// The slice kernel at d = 64: one query tile and one slice of its key tiles per CTA, two CTAs per SM
// (fwd_tile.cuh), so two online-softmax chains run per SM where fwd_split_kernel runs one.  The same
// slices, the same per-slice results (O normalised by the slice's own sum, base-2 LSE) and the same merge.
template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(tile::kThreads, 2) fwd_split_tile_kernel(const __grid_constant__ SplitArgs a) {
  griddep_launch_dependents();  // the merge kernel may start; it waits before it reads the slices
  const int bh = blockIdx.x;
  const int split = blockIdx.z;
  tile::Work w;
  w.head = bh % a.heads;
  w.batch = bh / a.heads;
  w.q0 = blockIdx.y * kTileRows;
  const int nkv = (a.Nk + kTileRows - 1) / kTileRows;
  int nvis = nkv;  // key tiles this query tile sees
  if (CAUSAL) {
    const int last_key = w.q0 + kTileRows - 1 + a.causal_off;
    nvis = last_key < 0 ? 0 : min(nkv, last_key / kTileRows + 1);
  }
  // this block's slice [j0, j0 + n): slices differ in length by at most one tile
  w.j0 = static_cast<int>(static_cast<long long>(split) * nvis / a.splits);
  w.n = static_cast<int>(static_cast<long long>(split + 1) * nvis / a.splits) - w.j0;
  auto epilogue = [&](bool ok, float m, float l, int r, uint32_t tO, uint32_t, volatile uint32_t*) {
    if (!ok) return;  // warp-uniform
    const int row = w.q0 + r;
    const size_t prow = (static_cast<size_t>(split) * a.bh_count + bh) * a.Nq + row;
    const float inv_l = l > 0.f ? 1.0f / l : 0.f;
    if (row < a.Nq) a.l_part[prow] = l > 0.f ? m + __log2f(l) : -INFINITY;
    float4* dst = reinterpret_cast<float4*>(a.o_part + prow * D);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      if (w.n > 0) {
        tmem_ld32(tO + c * 32, o);  // warp-collective: every lane loads, only real rows store
        tmem_wait_ld();
        reg_fence32(o);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
      if (row < a.Nq) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          dst[c * 8 + e] = make_float4(__uint_as_float(o[4 * e]) * inv_l, __uint_as_float(o[4 * e + 1]) * inv_l,
                                       __uint_as_float(o[4 * e + 2]) * inv_l, __uint_as_float(o[4 * e + 3]) * inv_l);
      }
    }
  };
  tile::run<D, CAUSAL, BF16>(&a.tm_q, &a.tm_k, &a.tm_v, w, a.Nk, a.causal_off, a.scale, a.err_word, a.timeout_ns,
                             epilogue);
}

// Merge of the slices, one warp per query row: lane holds d/32 consecutive columns.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fwd_combine_kernel(const __grid_constant__ SplitArgs a) {
  griddep_wait();  // a dependent launch: the slices are complete once the slice kernel has finished
  constexpr int V = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long rows = static_cast<long long>(a.bh_count) * a.Nq;
  const long long rid = static_cast<long long>(blockIdx.x) * 8 + warp;
  if (rid >= rows) return;  // warp-uniform
  const size_t split_stride = static_cast<size_t>(rows);
  const float* lp = a.l_part + rid;
  float mx = -INFINITY;
  for (int s = lane; s < a.splits; s += 32) mx = fmaxf(mx, lp[s * split_stride]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < a.splits; ++s) {
      const float w = ex2_approx(lp[s * split_stride] - mx);  // 0 for a slice that saw no key
      if (w > 0.f) {                                           // the same for every lane
        const float* op = a.o_part + (s * split_stride + rid) * D + lane * V;
        if constexpr (V == 4) {
          const float4 x = *reinterpret_cast<const float4*>(op);
          acc[0] = fmaf(w, x.x, acc[0]);
          acc[1] = fmaf(w, x.y, acc[1]);
          acc[2] = fmaf(w, x.z, acc[2]);
          acc[3] = fmaf(w, x.w, acc[3]);
        } else {
          const float2 x = *reinterpret_cast<const float2*>(op);
          acc[0] = fmaf(w, x.x, acc[0]);
          acc[1] = fmaf(w, x.y, acc[1]);
        }
        wsum += w;
      }
    }
  }
  const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
  const long long bh = rid / a.Nq, q = rid % a.Nq;
  const long long b = bh / a.heads, h = bh % a.heads;
  uint16_t* out = static_cast<uint16_t*>(a.o) + b * a.so.b + h * a.so.h + q * a.so.n + lane * V;
  if constexpr (V == 4) {
    const uint2 w = make_uint2(pack2<BF16>(acc[0] * inv, acc[1] * inv), pack2<BF16>(acc[2] * inv, acc[3] * inv));
    *reinterpret_cast<uint2*>(out) = w;
  } else {
    *reinterpret_cast<uint32_t*>(out) = pack2<BF16>(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0) a.lse[rid] = wsum > 0.f ? (mx + __log2f(wsum)) * 0.6931471805599453f : -INFINITY;
}

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_split_t(const SplitArgs& a, cudaStream_t stream) {
  dim3 grid(a.bh_count, (a.Nq + kTileRows - 1) / kTileRows, a.splits);
  cudaError_t e;
  if constexpr (D == 64) {  // two slice CTAs per SM (the library's slice count assumes as much at d = 64)
    using T = tile::Cfg<D>;
    auto kern = fwd_split_tile_kernel<D, CAUSAL, BF16>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_ALLOC)) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
      return e;
    kern<<<grid, tile::kThreads, T::SMEM_ALLOC, stream>>>(a);
  } else {
    using C = SplitCfg<D>;
    auto kern = fwd_split_kernel<D, CAUSAL, BF16>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::BYTES)) != cudaSuccess) return e;
    kern<<<grid, kSplitThreads, C::BYTES, stream>>>(a);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // The merge as a dependent launch (programmatic stream serialisation): its launch overlaps the slice
  // kernel's last blocks.
  const long long rows = static_cast<long long>(a.bh_count) * a.Nq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + 7) / 8));
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fwd_combine_kernel<D, BF16>, a);
}

}  // namespace

cudaError_t launch_fwd_split(const SplitArgs& a, cudaStream_t stream) {
  if (a.d == 64) {
    if (a.causal) return a.bf16 ? launch_split_t<64, true, true>(a, stream) : launch_split_t<64, true, false>(a, stream);
    return a.bf16 ? launch_split_t<64, false, true>(a, stream) : launch_split_t<64, false, false>(a, stream);
  }
  if (a.causal) return a.bf16 ? launch_split_t<128, true, true>(a, stream) : launch_split_t<128, true, false>(a, stream);
  return a.bf16 ? launch_split_t<128, false, true>(a, stream) : launch_split_t<128, false, false>(a, stream);
}

}  // namespace exattn
