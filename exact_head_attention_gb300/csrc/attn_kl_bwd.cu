// Attention-KL backward in one pass over key tiles (atomic dQ mode).
//
// The StreamKL summary (Methodology 2 and its fusion choice) gives two ways to
// produce both gradients of the KL divergence: separate dQ and dK kernels, or
// one pass whose dQ contributions are added across thread blocks with atomics
// while the accumulator fits in L2.  attn_kl.cu and attn_bwd_dq.cu implement
// the first (repeatable, six score-sized products per tile pair); this file
// the second (four products per pair: the two score products, dK and dQ).
//
// kl_bwd_pre_kernel: per query row the three values the score gradient needs,
//   base-2 teacher LSE, then the student's base-2 LSE (student trained) or
//   LSE_b - LSE_a - KL (teacher trained), then the upstream gradient g, with
//   values that make every dS exactly 0 on rows without keys and on padding;
//   and the fp32 dQ accumulator zeroed.
// kl_bwd_fused_kernel: one CTA per 128-row key tile j of one (batch, head),
//   K_a,j and K_b,j resident (teacher a, student b; t = the trained one).  For
//   every query tile i that sees it:
//     S_a^T = K_a Q_a,i^T, S_b^T = K_b Q_b,i^T        (TMEM, lane = key row)
//     dS^T  = f(S_a^T, S_b^T, row values)              (compute warps)
//     dK_t += dS^T Q_t,i                              (TMEM)
//     dQ_t,i += dS K_t  -> copy-engine reduce-add into the fp32 accumulator
//   The attention backward's key/value-block kernel (attn_bwd.cu) is the model:
//   K_b takes V's place, Q_b takes dO's, and S_b^T takes dP^T's, in the
//   columns dV would use (there is no dV here).
// The dQ conversion (dQ = scale * accumulator) is the attention backward's.
//
// Warp roles (320 threads): warps 0-3 and 4-7 compute (thread = key row; query
// columns [0, 64) and [64, 128)), warp 8 TMA producer (K_a, K_b once; per query
// tile the untrained then the trained distribution's Q through an NR-slot ring),
// warp 9 MMA issuer and TMEM owner.
// Tensor memory (512 columns):
//   X  = [0,128)    S_a^T
//   Y  = [128,256)  dQ_i^T (d = 128, lane = d) or dQ_i (d = 64, lane = query row),
//                   and the packed dS^T (the dK MMA's A operand): d = 128 in the
//                   first 32 columns of each warpgroup's half once it has read
//                   dQ_{i-1}^T out of them; d = 64 in [64,128) on even tiles and
//                   in [448,512) on odd tiles
//   W  = [256,384)  S_b^T
//   dK = [384,384+d)
// MMA issue order per tile i: S_{i+1} (once S_i is in registers), dK_i (once
// dS^T_i is in TMEM), dQ_i (once dS^T_i is in shared memory): the next scores
// overlap this tile's element work.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "kv_order.cuh"
#include "ptx.cuh"

namespace exattn {
namespace {

constexpr int kKlBwdThreads = 320;
constexpr uint32_t kChunkBytes = 128 * 128;

template <int D>
struct KlBwdCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = kTileRows * D * 2;
  static constexpr uint32_t PT = 128 * 128 * 2;  // dS^T tile
  static constexpr int NR = (D == 64) ? 6 : 3;   // ring slots (the two distributions' Q_i alternate)
  // fp32 dQ staging, 32 KB, as in the attention backward: d = 128, 64 query rows x 128 d row-major
  // (warpgroup 0; warpgroup 1 uses the dS^T tile); d = 64, two [128 query][32 d] boxes in the
  // accumulator tensor map's 128-byte-swizzled layout.
  static constexpr uint32_t STAGE_BYTES = 32768;
  static constexpr uint32_t OFF_KA = 0;
  static constexpr uint32_t OFF_KB = OFF_KA + TILE;
  static constexpr uint32_t OFF_DS = OFF_KB + TILE;
  static constexpr uint32_t OFF_RING = OFF_DS + PT;
  static constexpr uint32_t OFF_STAGE = OFF_RING + NR * TILE;
  // per warpgroup, the row values of its 64 query columns for the current tile: [3][64] fp32
  static constexpr uint32_t OFF_ROWV = OFF_STAGE + STAGE_BYTES;
  static constexpr uint32_t ROWV_BYTES = 3 * 64 * 4;
  static constexpr uint32_t OFF_BAR = OFF_ROWV + 2 * ROWV_BYTES;
  // kv_full, ring_full[NR], ring_empty[NR], s_full, s_used, pd_ready, dss_ready, mma_done, dq_full,
  // dq_empty, dstile_free, done
  static constexpr int NBAR = 1 + 2 * NR + 9;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
};

struct KlBwdBars {
  uint32_t base;
  int nr;
  __device__ uint32_t kv_full() const { return base; }
  __device__ uint32_t ring_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t ring_empty(int s) const { return base + 8 * (1 + nr + s); }
  __device__ uint32_t at(int k) const { return base + 8 * (1 + 2 * nr + k); }
  __device__ uint32_t s_full() const { return at(0); }       // S_a^T, S_b^T of a tile in TMEM
  __device__ uint32_t s_used() const { return at(1); }       // both read into registers
  __device__ uint32_t pd_ready() const { return at(2); }     // dS^T packed in TMEM (dK may go)
  __device__ uint32_t dss_ready() const { return at(3); }    // dS^T in shared memory (dQ may go)
  // the dQ MMA has read the dS^T tile: the same completion as dq_full, which one commit marks
  __device__ uint32_t ds_empty() const { return dq_full(); }
  __device__ uint32_t dq_full() const { return at(5); }
  __device__ uint32_t dq_empty() const { return at(6); }
  __device__ uint32_t dstile_free() const { return at(7); }  // d = 128: WG1's staged dQ rows read
  __device__ uint32_t done() const { return at(8); }
  __device__ uint32_t mma_done() const { return at(4); }
};

// TMEM column (from the allocation's base) where warpgroup h stores its packed dS^T half on tile
// `it`, and the column of K step k (16 query columns) of the whole operand.
template <int D>
__device__ __forceinline__ uint32_t ds_store_col(int it, int h) {
  return D == 128 ? 128u + 64u * h : ((it & 1) ? 448u : 192u) + 32u * h;
}
template <int D>
__device__ __forceinline__ uint32_t ds_mma_col(int it, int k) {
  if constexpr (D == 128) return 128u + (k < 4 ? k * 8 : 64 + (k - 4) * 8);
  return ((it & 1) ? 448u : 192u) + (k < 4 ? k * 8 : 32 + (k - 4) * 8);
}

// dS of one element from the raw scores (unscaled dot products) and the query row's three values.
// Student trained: g (P_b - P_a).  Teacher trained: g P_a (scale (S_a - S_b) + LSE_b - LSE_a - KL).
template <int OP>
__device__ __forceinline__ float kl_ds(float sa, float sb, float v0, float v1, float g, float c_log2, float scale) {
  if constexpr (OP == kPairKlStudent)
    return g * (ex2_approx(fmaf(sb, c_log2, -v1)) - ex2_approx(fmaf(sa, c_log2, -v0)));
  else
    return g * ex2_approx(fmaf(sa, c_log2, -v0)) * fmaf(scale, sa - sb, v1);
}

// Row values into three planes of a.rowv ([B*H][Nq_pad] each) and the accumulator zeroed; D / 8
// threads per padded row, 8 accumulator floats each.
template <int D, int OP>
__global__ void __launch_bounds__(256) kl_bwd_pre_kernel(const __grid_constant__ KlArgs a) {
  constexpr int TPR = D / 8;
  constexpr int RPB = 256 / TPR;
  const size_t row = static_cast<size_t>(blockIdx.x) * RPB + threadIdx.x / TPR;
  const int sub = threadIdx.x % TPR;
  const size_t total = static_cast<size_t>(a.bh_count) * a.Nq_pad;
  if (row >= total) return;
  float4* z = reinterpret_cast<float4*>(a.dq_acc + row * D + sub * 8);
  z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
  z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (sub != 0) return;
  const size_t bh = row / a.Nq_pad, q = row % a.Nq_pad;
  float v0 = INFINITY, v1 = (OP == kPairKlStudent) ? INFINITY : 0.f, g = 0.f;
  if (q < static_cast<size_t>(a.Nq)) {
    const size_t e = bh * a.Nq + q;
    const float l1 = a.lse1[e];
    if (l1 != -INFINITY) {  // a row that sees no key keeps dS = 0
      v0 = l1 * 1.4426950408889634f;
      v1 = (OP == kPairKlStudent) ? a.lse2[e] * 1.4426950408889634f : a.lse2[e] - l1 - a.kl[e];
      g = a.g[e];
    }
  }
  a.rowv[row] = v0;
  a.rowv[total + row] = v1;
  a.rowv[2 * total + row] = g;
}

template <int D, bool CAUSAL, bool BF16, int OP>
__global__ void __launch_bounds__(kKlBwdThreads, 1) kl_bwd_fused_kernel(const __grid_constant__ KlArgs a) {
  using C = KlBwdCfg<D>;
  constexpr int NR = C::NR;
  constexpr bool STUDENT = (OP == kPairKlStudent);
  // Ring order per query tile: the untrained distribution's queries first (ring position 2i, read by
  // its score product only and released after it), then the trained one's (2i + 1, released after dK_i).
  // S_{i+1} then waits only for slots that S_i or dK_{i-1} release, both issued before it.
  constexpr int PA = STUDENT ? 0 : 1;  // ring parity of Q_a
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  if (!smem_base_aligned(sbase, a.err_word)) return;
  uint8_t* gbase = smem_raw;
  const uint32_t sKa = sbase + C::OFF_KA, sKb = sbase + C::OFF_KB, sDS = sbase + C::OFF_DS;
  const uint32_t sRing = sbase + C::OFF_RING;
  const KlBwdBars bars{sbase + C::OFF_BAR, NR};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + C::OFF_MISC + 4);
  const WaitCtx wc{abort_flag, a.err_word, a.timeout_ns};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (a.Nk + kTileRows - 1) / kTileRows;
  const KvBlock blk = kv_block(blockIdx.x, a.bh_count, a.head_group, nkb);  // launch order as in the attention backward
  const int bh = blk.bh;
  const int head = bh % a.heads, batch = bh / a.heads;
  const int jb = blk.jb;  // key tile; causal work decreases with jb
  const int k0 = jb * kTileRows;
  const int nq_tiles = (a.Nq + kTileRows - 1) / kTileRows;
  const int coff = CAUSAL ? a.causal_off : 0;
  const int i_start = CAUSAL ? max(0, k0 - coff) / kTileRows : 0;  // first query tile with a row that sees key k0
  const int n = max(0, nq_tiles - i_start);                         // query tiles this block visits

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    mbar_init(bars.kv_full(), 1);
    for (int s = 0; s < NR; ++s) {
      mbar_init(bars.ring_full(s), 1);
      mbar_init(bars.ring_empty(s), 1);
    }
    mbar_init(bars.s_full(), 1);
    mbar_init(bars.s_used(), 256);
    mbar_init(bars.pd_ready(), 256);
    mbar_init(bars.dss_ready(), 256);
    mbar_init(bars.dq_full(), 1);
    mbar_init(bars.dq_empty(), 256);
    mbar_init(bars.dstile_free(), 1);
    mbar_init(bars.done(), 1);
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
  const uint32_t tX = tmem, tY = tmem + 128, tW = tmem + 256, tdK = tmem + 384;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0) {
      prefetch_tmap(&a.tm_qa);
      prefetch_tmap(&a.tm_qb);
      mbar_arrive_expect_tx(bars.kv_full(), 2 * C::TILE);
      // both key tiles are read by this block only (evict-first); the dQ reduce-adds are evict-last
      const uint64_t once = l2_evict_first();
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_4d_hint(sKa + c * kChunkBytes, &a.tm_ka, c * 64, k0, head, batch, bars.kv_full(), once);
        tma_load_4d_hint(sKb + c * kChunkBytes, &a.tm_kb, c * 64, k0, head, batch, bars.kv_full(), once);
      }
      int issued = 0;
      for (int L = 0; L < 2 * n; ++L) {
        const int s = L % NR;
        if (!mbar_wait(bars.ring_empty(s), ((L / NR) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(bars.ring_full(s), C::TILE);
        const CUtensorMap* map = ((L & 1) == PA) ? &a.tm_qa : &a.tm_qb;
        const int q_row = (i_start + (L >> 1)) * kTileRows;
        for (int c = 0; c < C::NCH; ++c)
          tma_load_4d(sRing + s * C::TILE + c * kChunkBytes, map, c * 64, q_row, head, batch, bars.ring_full(s));
        ++issued;
      }
      if (*abort_flag) {
        for (int L = max(0, issued - NR); L < issued; ++L) mbar_drain(bars.ring_full(L % NR), (L / NR) & 1, a.timeout_ns);
        mbar_drain(bars.kv_full(), 0, a.timeout_ns);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idS = idesc_f16(128, 128, BF16, false, false);  // K-major x K-major
      constexpr uint32_t idG = idesc_f16(128, D, BF16, false, true);     // dK: A (TMEM) K-major, B MN-major
      constexpr uint32_t idQ = idesc_f16(128, D, BF16, true, true);      // dQ: A = dS MN-major, B = K_t MN-major
      constexpr uint32_t idQT = idesc_f16(D, 128, BF16, true, true);     // dQ^T: A = K_t^T MN-major, B = dS^T MN-major
      auto slot_of = [](int L) { return L % NR; };
      auto phase_of = [](int L) { return static_cast<uint32_t>((L / NR) & 1); };
      constexpr uint32_t kTileLo = C::TILE >> 4;
      const uint32_t ka_kmaj = sdesc_lo(sKa, 16), kb_kmaj = sdesc_lo(sKb, 16), ring_kmaj = sdesc_lo(sRing, 16);
      const uint32_t ring_mn = sdesc_lo(sRing, kChunkBytes), kt_mn = sdesc_lo(STUDENT ? sKb : sKa, kChunkBytes);
      const uint32_t ds_mn = sdesc_lo(sDS, kChunkBytes);
      auto scores = [&](uint32_t d, uint32_t a_lo, uint32_t b_lo) {
        mma_ss_lo<false>(d, a_lo, b_lo, idS);
#pragma unroll
        for (int k = 1; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * kChunkBytes + (k & 3) * 32) >> 4;
          mma_ss_lo<true>(d, a_lo + off, b_lo + off, idS);
        }
      };
      // S_a^T and S_b^T of query tile `it`; the untrained distribution's queries are read by these
      // products only, so their ring slot is released once they complete.
      auto issue_S = [&](int it) -> bool {
        const int La = 2 * it + PA, Lb = 2 * it + 1 - PA;
        if (!mbar_wait(bars.ring_full(slot_of(La)), phase_of(La), wc)) return false;
        if (!mbar_wait(bars.ring_full(slot_of(Lb)), phase_of(Lb), wc)) return false;
        tc_fence_after();
        scores(tX, ka_kmaj, ring_kmaj + slot_of(La) * kTileLo);
        scores(tW, kb_kmaj, ring_kmaj + slot_of(Lb) * kTileLo);
        mma_commit(bars.s_full());
        mma_commit(bars.ring_empty(slot_of(2 * it)));
        return true;
      };

      bool ok = mbar_wait(bars.kv_full(), 0, wc);
      if (ok) ok = issue_S(0);
      for (int it = 0; ok && it < n; ++it) {
        // S_{i+1} overwrites X and W once the compute warps have read S_i; it runs while they form dS_i.
        if (it + 1 < n) {
          if (!(ok = mbar_wait(bars.s_used(), it & 1, wc))) break;
          if (!(ok = issue_S(it + 1))) break;
        }
        if (!(ok = mbar_wait(bars.pd_ready(), it & 1, wc))) break;
        tc_fence_after();
        // dK_t += dS^T Q_t,i   (A: dS^T packed in TMEM; B: Q_t,i [query][d] MN-major, 16 query rows per K step)
        const uint32_t q_lo = ring_mn + slot_of(2 * it + 1) * kTileLo;
        mma_ts_lo_rt(tdK, tmem + ds_mma_col<D>(it, 0), q_lo, idG, it > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 1; k < 128 / 16; ++k) mma_ts_lo<true>(tdK, tmem + ds_mma_col<D>(it, k), q_lo + k * (2048 >> 4), idG);
        mma_commit(bars.ring_empty(slot_of(2 * it + 1)));
        // dQ_i overwrites Y (d = 128: also dS^T_i) after dK_i has read it (MMAs of one thread run in order).
        if (it > 0 && !(ok = mbar_wait(bars.dq_empty(), (it - 1) & 1, wc))) break;
        if (!(ok = mbar_wait(bars.dss_ready(), it & 1, wc))) break;
        tc_fence_after();
        if constexpr (D == 128) {
          // dQ_i^T = K_t^T dS^T  (A: K_t^T [d][key] MN-major from the K_t tile; B: dS^T MN-major)
          mma_ss_lo<false>(tY, kt_mn, ds_mn, idQT);
#pragma unroll
          for (int k = 1; k < 128 / 16; ++k) mma_ss_lo<true>(tY, kt_mn + k * (2048 >> 4), ds_mn + k * (2048 >> 4), idQT);
        } else {
          // dQ_i = dS K_t  (A: dS [query][key] MN-major from the dS^T tile; B: K_t [key][d] MN-major)
          mma_ss_lo<false>(tY, ds_mn, kt_mn, idQ);
#pragma unroll
          for (int k = 1; k < 128 / 16; ++k) mma_ss_lo<true>(tY, ds_mn + k * (2048 >> 4), kt_mn + k * (2048 >> 4), idQ);
        }
        mma_commit(bars.dq_full());  // also frees the dS^T tile (ds_empty)
      }
      if (ok) mma_commit(bars.done());
      mma_commit(bars.mma_done());
      mbar_drain(bars.mma_done(), 0, a.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ compute
    const int h = warp >> 2;             // query half: columns [64h, 64h + 64)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;   // TMEM lane: key row of S^T; d (d = 128) or query row of dQ
    const int kv = k0 + r;
    const bool kv_valid = kv < a.Nk;
    const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
    const float c_log2 = a.scale * 1.4426950408889634f;
    const uint32_t ds_row = sDS + h * kChunkBytes;
    const size_t plane = static_cast<size_t>(a.bh_count) * a.Nq_pad;
    const float* rv0 = a.rowv + static_cast<size_t>(bh) * a.Nq_pad;
    const float* srow = reinterpret_cast<const float*>(gbase + C::OFF_ROWV + h * C::ROWV_BYTES);
    // The warpgroup's 3 x 64 row values of a tile are 48 float4: thread r < 48 fetches vector r / 16,
    // columns 4 (r % 16) .. + 3, one tile ahead, and stores them into shared memory at the tile's start.
    auto fetch_rows = [&](int it) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < 48) v = __ldg(reinterpret_cast<const float4*>(rv0 + (r / 16) * plane + (i_start + it) * kTileRows + h * 64 + 4 * (r % 16)));
      return v;
    };
    float4 rnext = fetch_rows(0);
    // Once a wait has failed (its time limit expired, or another warp raised the abort flag) a compute
    // warp does not leave the tile loop: it skips its remaining waits and runs on, so that every warp
    // of its warpgroup meets the warpgroup's named barriers equally often and in the same order (a warp
    // that left early would release a barrier of the same number for the wrong round).  What it computes
    // after a failure is garbage: the epilogue skips the dK store (it checks the abort flag), and the dQ
    // still added into the accumulator is marked invalid by the error word.  `ok` stays warp-uniform.
    bool ok = true;
    auto wait = [&](uint32_t bar, uint32_t parity) { ok = ok && mbar_wait_warp(bar, parity, wc); };

    // d = 128, dQ_i^T (lane = d, column = query row): this warpgroup reduces query rows [64h, 64h + 64)
    // through a 32 KB row-major buffer (warpgroup 0: the staging tile; warpgroup 1: the dS^T tile, free
    // from the end of the dQ_i MMA until the next dS^T store, which waits for this read: dstile_free),
    // one flat copy-engine reduce-add per warpgroup.  The rows come out of TMEM 32 at a time; with
    // `ds`, this warpgroup's packed dS^T of the next tile goes into the first 32 columns once read.
    auto drain128 = [&](int it, bool with_ds, const uint32_t (&ds)[32]) {
      wait(bars.dq_full(), it & 1);
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(tY + lane_bits + h * 64, v);
      tmem_wait_ld();
      reg_fence32(v);
      if (with_ds) {
        tmem_st32(tmem + lane_bits + ds_store_col<D>(it + 1, h), ds);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bars.pd_ready());  // dK of the next tile may go
      }
      const uint32_t buf_off = h ? C::OFF_DS : C::OFF_STAGE;
      if (h == 0) {
        if (r == 0) tma_store_wait_read_all();  // the previous reduction from the staging tile
        named_bar_sync(1, 128);
      }
      float* buf = reinterpret_cast<float*>(gbase + buf_off);
#pragma unroll
      for (int c = 0; c < 32; ++c) buf[c * D + r] = __uint_as_float(v[c]);
      tmem_ld32(tY + lane_bits + h * 64 + 32, v);
      tmem_wait_ld();
      reg_fence32(v);
      tc_fence_before();
      mbar_arrive(bars.dq_empty());
#pragma unroll
      for (int c = 0; c < 32; ++c) buf[(32 + c) * D + r] = __uint_as_float(v[c]);
      fence_proxy_async_smem();
      named_bar_sync(1 + h, 128);
      if (r == 0) {
        const size_t row0 = static_cast<size_t>(bh) * a.Nq_pad + (i_start + it) * kTileRows + h * 64;
        bulk_reduce_add_f32_hint(a.dq_acc + row0 * D, sbase + buf_off, C::STAGE_BYTES, l2_evict_last());
        tma_store_commit();
      }
    };
    // d = 64, dQ_i (lane = query row): this warpgroup reduces d columns [32h, 32h + 32) as one
    // [128 query][32 d] box written with the accumulator map's 128-byte swizzle, one tensor reduce-add.
    auto drain64 = [&](int it) {
      wait(bars.dq_full(), it & 1);
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(tY + lane_bits + h * 32, v);
      tmem_wait_ld();
      reg_fence32(v);
      tc_fence_before();
      mbar_arrive(bars.dq_empty());
      const uint32_t box = sbase + C::OFF_STAGE + h * (C::STAGE_BYTES / 2);
      if (r == 0) tma_store_wait_read_all();  // this half's previous reduction has read the box
      named_bar_sync(1 + h, 128);
#pragma unroll
      for (int u = 0; u < 8; ++u) st_shared_v4(box + sw128_offset(r, u), v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
      fence_proxy_async_smem();
      named_bar_sync(1 + h, 128);
      if (r == 0) {
        tma_reduce_add_2d_hint(&a.tm_dqacc, box, 32 * h, bh * a.Nq_pad + (i_start + it) * kTileRows, l2_evict_last());
        tma_store_commit();
      }
    };

    const bool ragged_kv = k0 + kTileRows > a.Nk;  // block-uniform
    for (int it = 0; it < n; ++it) {
      const int qb = (i_start + it) * kTileRows + h * 64;  // first query column of this half
      wait(bars.s_full(), it & 1);
      tc_fence_after();
      // This tile's row values into shared memory (the barrier before: every thread of the warpgroup
      // has finished reading the previous tile's), and the next tile's fetched meanwhile.
      named_bar_sync(3 + h, 128);
      if (r < 48) *reinterpret_cast<float4*>(gbase + C::OFF_ROWV + h * C::ROWV_BYTES + ((r / 16) * 64 + 4 * (r % 16)) * 4) = rnext;
      named_bar_sync(3 + h, 128);
      if (it + 1 < n) rnext = fetch_rows(it + 1);
      // Only query tiles the causal diagonal crosses and a ragged last key tile need the mask:
      // columns below `lo` get dS = 0.
      const bool diag = CAUSAL && ((i_start + it) * kTileRows + coff < k0 + kTileRows - 1);
      const int lo = !kv_valid ? 64 : (diag ? kv - coff - qb : 0);
      const bool masked = diag || ragged_kv;
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 2; ++c) {  // 32 query columns at a time
        uint32_t sa[32], sb[32];
        tmem_ld32(tX + lane_bits + h * 64 + 32 * c, sa);
        tmem_ld32(tW + lane_bits + h * 64 + 32 * c, sb);
        tmem_wait_ld();
        reg_fence32(sa);
        reg_fence32(sb);
        if (c == 1) {
          tc_fence_before();
          mbar_arrive(bars.s_used());  // both score tiles are in registers: the next ones may go
        }
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const int col0 = 32 * c + 4 * e4;
          const float4 v0 = *reinterpret_cast<const float4*>(srow + col0);
          const float4 v1 = *reinterpret_cast<const float4*>(srow + 64 + col0);
          const float4 gg = *reinterpret_cast<const float4*>(srow + 128 + col0);
          const float a0[4] = {v0.x, v0.y, v0.z, v0.w}, a1[4] = {v1.x, v1.y, v1.z, v1.w};
          const float ag[4] = {gg.x, gg.y, gg.z, gg.w};
          float ds[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = 4 * e4 + e;
            ds[e] = kl_ds<OP>(__uint_as_float(sa[i]), __uint_as_float(sb[i]), a0[e], a1[e], ag[e], c_log2, a.scale);
            if (masked && col0 + e < lo) ds[e] = 0.f;
          }
          pk[16 * c + 2 * e4] = pack2<BF16>(ds[0], ds[1]);
          pk[16 * c + 2 * e4 + 1] = pack2<BF16>(ds[2], ds[3]);
        }
      }
      // dS^T into TMEM for dK_i: at d = 128 once this warpgroup has read dQ_{i-1}^T out of its half of
      // Y (dQ_{i-1} follows dK_{i-1}, so that has also read dS^T_{i-1}); at d = 64 into the buffer of
      // this tile's parity, which dK_{i-2} read before S_i was issued.
      if (D == 128 && it > 0) {
        drain128(it - 1, true, pk);
      } else {
        tmem_st32(tmem + lane_bits + ds_store_col<D>(it, h), pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bars.pd_ready());  // dK_i may go
      }
      // dS^T into the shared tile for dQ_i, once dQ_{i-1} has read it
      if (it > 0) wait(bars.ds_empty(), (it - 1) & 1);
      if constexpr (D == 128) {
        // The dS^T tile held warpgroup 1's dQ_{i-1} rows; the copy engine must have read them.
        if (it > 0 && h == 1) {
          if (r == 0) tma_store_wait_read_all();
          named_bar_sync(2, 128);
          if (r == 0) mbar_arrive(bars.dstile_free());
        }
        if (it > 0 && h == 0) wait(bars.dstile_free(), (it - 1) & 1);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        st_shared_v4(ds_row + sw128_offset(r, u), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      fence_proxy_async_smem();
      mbar_arrive(bars.dss_ready());  // dQ_i may go
      if (D == 64 && it > 0) drain64(it - 1);
    }
    if (n > 0) {
      if constexpr (D == 128) {
        const uint32_t none[32] = {};
        drain128(n - 1, false, none);
      } else {
        drain64(n - 1);
      }
    }

    // ------------------------------------------------------------ epilogue: dK * scale
    // Warpgroup h writes d columns [64h, 64h + 64), staged in the K_a tile (every MMA has completed).
    if (ok && n > 0) ok = mbar_wait_warp(bars.done(), 0, wc);
    const bool mine = h < C::NCH;
    const uint32_t stage = sKa + h * kChunkBytes;
    if (ok && mine) {
      tc_fence_after();
      uint32_t o[2][32];
      if (n > 0) {
        tmem_ld32(tdK + lane_bits + h * 64, o[0]);
        tmem_ld32(tdK + lane_bits + h * 64 + 32, o[1]);
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
        st_shared_v4(stage + sw128_offset(r, u), w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1 + h, 128);
    if (ok && mine && r == 0 && !*abort_flag) {
      tma_store_4d_hint(&a.tm_dk, stage, h * 64, k0, head, batch, l2_evict_first());  // not read again here
      tma_store_commit();
    }
    if (r == 0) tma_store_wait_all();  // this thread's stores and dQ reductions have completed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL, bool BF16, int OP>
cudaError_t launch_kl_bwd_fused_t(const KlArgs& a, cudaStream_t stream) {
  using C = KlBwdCfg<D>;
  constexpr int RPB = 256 / (D / 8);
  const size_t rows = static_cast<size_t>(a.bh_count) * a.Nq_pad;
  kl_bwd_pre_kernel<D, OP><<<static_cast<unsigned>((rows + RPB - 1) / RPB), 256, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kern = kl_bwd_fused_kernel<D, CAUSAL, BF16, OP>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::BYTES)) != cudaSuccess) return e;
  const unsigned blocks = static_cast<unsigned>(a.bh_count) * ((a.Nk + kTileRows - 1) / kTileRows);
  kern<<<blocks, kKlBwdThreads, C::BYTES, stream>>>(a);
  return cudaGetLastError();
}

template <int OP>
cudaError_t launch_kl_bwd_fused_op(const KlArgs& a, cudaStream_t stream) {
  if (a.d == 64) {
    if (a.causal)
      return a.bf16 ? launch_kl_bwd_fused_t<64, true, true, OP>(a, stream) : launch_kl_bwd_fused_t<64, true, false, OP>(a, stream);
    return a.bf16 ? launch_kl_bwd_fused_t<64, false, true, OP>(a, stream) : launch_kl_bwd_fused_t<64, false, false, OP>(a, stream);
  }
  if (a.causal)
    return a.bf16 ? launch_kl_bwd_fused_t<128, true, true, OP>(a, stream) : launch_kl_bwd_fused_t<128, true, false, OP>(a, stream);
  return a.bf16 ? launch_kl_bwd_fused_t<128, false, true, OP>(a, stream) : launch_kl_bwd_fused_t<128, false, false, OP>(a, stream);
}

}  // namespace

cudaError_t launch_kl_bwd_fused(const KlArgs& a, cudaStream_t stream) {
  return a.op == kPairKlStudent ? launch_kl_bwd_fused_op<kPairKlStudent>(a, stream)
                                : launch_kl_bwd_fused_op<kPairKlTeacher>(a, stream);
}

}  // namespace exattn
