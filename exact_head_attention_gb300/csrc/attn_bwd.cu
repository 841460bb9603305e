// Fused attention backward for sm_103a: three launches on one stream.
//
// 1. bwd_pre_kernel: D_q = rowsum(dO o O) in fp32 (SparkAttention Figure 9,
//    "dPsum"), LSE converted to base 2 and stored negated, the additive term of
//    the exponent (padding rows get -inf so that their recomputed
//    probabilities are exactly 0), and the fp32 dQ accumulator zeroed.
// 2. bwd_main_kernel: one CTA per 128-row key/value block of one (batch,
//    head) -- the backward pass is parallel over blocks of columns of the
//    attention matrix ("Fast Transformer training with long sequences",
//    backward parallelisation).  K_j, V_j stay resident; for every query tile
//    i that sees them (causal: i >= j) it recomputes
//        S^T = K_j Q_i^T,  P^T = exp2(S^T*scale*log2e - LSE2_i)
//        dP^T = V_j dO_i^T, dS^T = P^T o (dP^T - D_i)
//        dV_j += P^T dO_i,  dK_j += dS^T Q_i,  dQ_i += dS K_j
//    (StreamKL summary, Methodology 2: P regenerated tile by tile from the
//    stored LSE), accumulating dK_j, dV_j in TMEM and adding dQ_i into the
//    fp32 accumulator in L2 (SparkAttention: dQ is atomically added across
//    thread blocks; StreamKL: atomics while the buffer fits in L2).  The
//    adds are copy-engine reduce-adds of a shared-memory tile: flat bulk
//    copies of dQ^T's row-major halves at d = 128, 2-D tensor copies of
//    128-byte-swizzled [128 query][32 d] boxes at d = 64.  A template flag drops
//    the dQ work entirely for the deterministic mode, where the query-tile
//    kernel (attn_bwd_dq.cu) produces dQ instead.
// 3. bwd_dq_convert_kernel: dQ = scale * dQacc rounded to the input dtype.
//
// L2: the dQ accumulator's reduce-adds carry an evict-last hint and the loads of K_j, V_j and the
// stores of dK, dV an evict-first one, so that what this kernel touches once does not push the
// accumulator's lines out of L2 between the key blocks that add into them.
//
// Main-kernel warp roles (320 threads):
//   warps 0-3   compute, query columns [0, 64) of each tile (thread = key row),
//               and query rows [0, 64) of the dQ drain
//   warps 4-7   compute, query columns [64, 128), dQ query rows [64, 128)
//   warp  8     TMA producer: K_j, V_j once; Q_i and dO_i through two rings,
//               LSE2_i and D_i through a 2-slot ring
//   warp  9     MMA issuer (one thread) and TMEM owner
// Tensor memory (512 columns):
//   X  = [0,128)    S^T_i, then dP^T_i; then each compute warpgroup h packs its
//                   dS^T half into [64h+32, 64h+64) -- the A operand of the dK MMA
//   Y  = [128,256)  dQ_i (d = 64: lane = query row, 64 columns) or dQ_i^T (d = 128:
//                   lane = d), and the packed P^T (the dV MMA's A operand), written
//                   as soon as the exponentials are done: d = 128 into the columns
//                   each warpgroup has just read dQ_{i-1}^T from, d = 64 into the
//                   64 columns dQ leaves free
//   dV = [256,256+d), dK = [384,384+d)
// Shared memory: K_j, V_j, dS^T (the dQ MMA's operand), the Q/dO ring.
// Per tile i the MMA issue order is dV_i, dK_i, S_{i+1}, dQ_i, dP_{i+1}: dV_i
// queues behind dP^T_i (P^T_i is in Y by then) and overlaps the forming of dS^T_i, the
// exponentials of tile i+1 overlap dQ_i and dP_{i+1}, and the dQ_i reduction
// (issued by the compute warps after they hand over tile i+1) overlaps the
// next tile's MMAs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "kv_order.cuh"
#include "ptx.cuh"

namespace exattn {
namespace {

constexpr int kBwdThreads = 320;
constexpr uint32_t kChunkBytes = 128 * 128;

template <int D>
struct BwdCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = kTileRows * D * 2;
  static constexpr uint32_t PT = 128 * 128 * 2;  // dS^T tile
  // Q/dO ring slots.  d = 128 gives one slot to the dQ staging tile: reducing dQ with the copy
  // engine from shared memory is far cheaper than per-thread atomics, which outweighs the shallower ring.
  static constexpr int NR = (D == 64) ? 6 : 3;
  // The ring is two: NQ slots take Q_i, freed by dK_i (its last reader), and NO slots take dO_i.  At
  // d = 128 the one dO slot is freed by dV_i, a product before dK_i, so the load of dO_{i+1} (needed by
  // dP_{i+1}, three products after dV_i) starts as early as it can.  At d = 64 the rings are deep enough
  // for dO_i's slot to be freed with Q_i's, by one commit per tile.
  static constexpr int NQ = (D == 64) ? 3 : 2;
  static constexpr int NO = NR - NQ;
  static constexpr bool DO_OWN_FREE = (D == 128);
  static_assert(DO_OWN_FREE || NO == NQ, "dO slots freed with the Q slots of the same tile");
  // fp32 dQ staging, 32 KB: d = 128, 64 query rows x 128 d in the accumulator's row-major layout (one
  // half per warpgroup in turn with the dS^T tile); d = 64, two [128 query][32 d] boxes (one per
  // warpgroup) in the 128-byte-swizzled layout of the accumulator's tensor map.
  static constexpr uint32_t STAGE_BYTES = 32768;
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + TILE;
  static constexpr uint32_t OFF_DS = OFF_V + TILE;
  static constexpr uint32_t OFF_RING = OFF_DS + PT;
  static constexpr uint32_t OFF_STAGE = OFF_RING + NR * TILE;
  // two slots of the query tile's row vectors: 128 negated base-2 LSE then 128 D values (fp32)
  static constexpr uint32_t OFF_ROWV = OFF_STAGE + STAGE_BYTES;
  static constexpr uint32_t ROWV_BYTES = 2 * 128 * 4;
  static constexpr uint32_t OFF_BAR = OFF_ROWV + 2 * ROWV_BYTES;
  // kv_full, q_full[NQ], do_full[NO], q_free[NQ], do_free[NO], s_full, s_used, dp_full, pd_ready[0], p_ready,
  // dq_full, dq_empty, done, mma_done, rowv_full[2], rowv_empty[2], dss_ready, dstile_free, pd_ready[1]
  static constexpr int NBAR = 1 + 2 * NR + 16;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  // The operand tiles need 1024-byte alignment; the dynamic shared memory base is checked at entry
  // instead of padding.
  static constexpr uint32_t SMEM_ALLOC = BYTES;
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

struct BwdBars {
  uint32_t base;
  int nr, nq;
  __device__ uint32_t kv_full() const { return base; }
  __device__ uint32_t q_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t do_full(int s) const { return base + 8 * (1 + nq + s); }
  __device__ uint32_t q_free(int s) const { return base + 8 * (1 + nr + s); }        // dK of the slot's tile done
  __device__ uint32_t do_free(int s) const { return base + 8 * (1 + nr + nq + s); }  // dV of the slot's tile done
  __device__ uint32_t at(int k) const { return base + 8 * (1 + 2 * nr + k); }
  __device__ uint32_t s_full() const { return at(0); }
  __device__ uint32_t s_used() const { return at(1); }
  __device__ uint32_t dp_full() const { return at(2); }
  // compute warpgroup h has packed its half of dS^T into TMEM X (the query columns [64h, 64h + 64): dK's
  // K steps 4h .. 4h + 3); at d = 64 pd_ready(0) stands for both warpgroups
  __device__ uint32_t pd_ready(int h) const { return h ? at(15) : at(3); }
  __device__ uint32_t dss_ready() const { return at(13); } // dS^T in shared memory
  // d = 128: the copy engine has read warpgroup 1's dQ rows out of the dS^T tile
  __device__ uint32_t dstile_free() const { return at(14); }
  __device__ uint32_t p_ready() const { return at(4); }    // P^T packed in TMEM Y (dV may go)
  // the dQ MMA has read the dS^T tile: the same completion as dq_full, which one commit marks
  __device__ uint32_t ds_empty() const { return dq_full(); }
  __device__ uint32_t dq_full() const { return at(5); }
  __device__ uint32_t dq_empty() const { return at(6); }
  __device__ uint32_t done() const { return at(7); }
  __device__ uint32_t mma_done() const { return at(8); }
  __device__ uint32_t rowv_full(int s) const { return at(9 + s); }
  __device__ uint32_t rowv_empty(int s) const { return at(11 + s); }
};

// TMEM column of K step k (16 query columns) of the packed dS^T operand in X: query columns [0, 64)
// sit in [32, 64), query columns [64, 128) in [96, 128).
__device__ __forceinline__ uint32_t ds_col(int k) { return (k < 4 ? k * 8 : 64 + (k - 4) * 8) + 32; }

// The packed P^T operand lives in Y, so that it can be written before dP^T lands in X.  Query half h
// (32 packed columns) starts at column p_base<D>() + h * p_stride<D>() of Y: d = 128, the first 32
// columns of the half of dQ_{i-1}^T that warpgroup h has just read out; d = 64, the 64 columns of Y
// that dQ (64 columns) leaves free.
template <int D>
__device__ __forceinline__ constexpr uint32_t p_base() { return D == 64 ? 64u : 0u; }
template <int D>
__device__ __forceinline__ constexpr uint32_t p_stride() { return D == 64 ? 32u : 64u; }
template <int D>
__device__ __forceinline__ uint32_t p_col(int k) { return p_base<D>() + (k < 4 ? k * 8 : p_stride<D>() + (k - 4) * 8); }

// DQ = false: dK and dV only (the deterministic mode computes dQ in pair_dq_kernel (attn_bwd_dq.cu) instead); the dQ
// MMA, the dS^T tile in shared memory and the reductions are left out.
template <int D, bool CAUSAL, bool BF16, bool DQ>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_main_kernel(const __grid_constant__ BwdArgs a) {
  using C = BwdCfg<D>;
  constexpr int NR = C::NR;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  if (!smem_base_aligned(sbase, a.err_word)) return;
  uint8_t* gbase = smem_raw;
  const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sDS = sbase + C::OFF_DS;
  const uint32_t sRing = sbase + C::OFF_RING;
  const uint32_t sRowv = sbase + C::OFF_ROWV;
  const BwdBars bars{sbase + C::OFF_BAR, NR, C::NQ};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + C::OFF_MISC + 4);
  const WaitCtx wc{abort_flag, a.err_word, a.timeout_ns};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (a.Nk + kTileRows - 1) / kTileRows;
  const KvBlock blk = kv_block(blockIdx.x, a.bh_count, a.head_group, nkb);
  const int bh = blk.bh;
  const int head = bh % a.heads, batch = bh / a.heads;
  const int jb = blk.jb;  // key block; causal work decreases with jb
  const int k0 = jb * kTileRows;
  const int nq_tiles = (a.Nq + kTileRows - 1) / kTileRows;
  // Causal: query q sees key k iff k <= q + coff, so the first query tile to visit holds row k0 - coff.
  const int coff = CAUSAL ? a.causal_off : 0;
  const int i_start = CAUSAL ? max(0, k0 - coff) / kTileRows : 0;
  const int n = max(0, nq_tiles - i_start);  // query tiles this block visits

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    mbar_init(bars.kv_full(), 1);
    for (int s = 0; s < C::NQ; ++s) {
      mbar_init(bars.q_full(s), 1);
      mbar_init(bars.q_free(s), 1);
    }
    for (int s = 0; s < C::NO; ++s) {
      mbar_init(bars.do_full(s), 1);
      mbar_init(bars.do_free(s), 1);
    }
    mbar_init(bars.s_full(), 1);
    mbar_init(bars.s_used(), 256);
    mbar_init(bars.dp_full(), 1);
    // d = 64: one hand-over for both warpgroups (pd_ready(0), 256 arrivals); d = 128: one each
    mbar_init(bars.pd_ready(0), D == 128 ? 128 : 256);
    mbar_init(bars.pd_ready(1), 128);
    mbar_init(bars.p_ready(), 256);
    mbar_init(bars.dss_ready(), 256);
    mbar_init(bars.dstile_free(), 1);
    mbar_init(bars.dq_full(), 1);
    mbar_init(bars.dq_empty(), 256);
    mbar_init(bars.done(), 1);
    mbar_init(bars.mma_done(), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bars.rowv_full(s), 1);
      mbar_init(bars.rowv_empty(s), 256);
    }
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
  const uint32_t tX = tmem, tY = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;

  // This kernel may start while the preprocess kernel finishes (dependent launch): K and V are not
  // written by it, so their loads go first; everything else waits for it (LSE2, D, the zeroed
  // accumulator, and through it every earlier kernel).
  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0) {
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_do);
      mbar_arrive_expect_tx(bars.kv_full(), 2 * C::TILE);
      // K_j and V_j are read by this block only: their lines should not push out the dQ accumulator's
      // or the query tiles' (which the other key blocks of the head read too).
      const uint64_t once = l2_evict_first();
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_4d_hint(sK + c * kChunkBytes, &a.tm_k, c * 64, k0, head, batch, bars.kv_full(), once);
        tma_load_4d_hint(sV + c * kChunkBytes, &a.tm_v, c * 64, k0, head, batch, bars.kv_full(), once);
      }
    }
    griddep_wait();
    griddep_launch_dependents();
    if (lane == 0 && n > 0) {
      int issued_q = 0, issued_do = 0, issued_rowv = 0;
      for (int it = 0; it < n; ++it) {
        // LSE2 and D of query tile it into row-vector slot it % 2
        const int rs = it & 1;
        if (!mbar_wait(bars.rowv_empty(rs), ((it >> 1) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(bars.rowv_full(rs), C::ROWV_BYTES);
        const size_t off = static_cast<size_t>(bh) * a.Nq_pad + (i_start + it) * kTileRows;
        bulk_load(sRowv + rs * C::ROWV_BYTES, a.nlse2 + off, 512, bars.rowv_full(rs));
        bulk_load(sRowv + rs * C::ROWV_BYTES + 512, a.dsum + off, 512, bars.rowv_full(rs));
        ++issued_rowv;
        const int q_row = (i_start + it) * kTileRows;
        // Q_it into slot it % NQ, once tile it - NQ's dK has completed (which also frees dO slot it % NO
        // when the dO slots are freed with the Q ones)
        const int sq = it % C::NQ;
        if (!mbar_wait(bars.q_free(sq), ((it / C::NQ) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(bars.q_full(sq), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_4d(sRing + sq * C::TILE + c * kChunkBytes, &a.tm_q, c * 64, q_row, head, batch, bars.q_full(sq));
        ++issued_q;
        // dO_it into slot it % NO, once tile it - NO's dV has completed
        const int so = it % C::NO;
        if (C::DO_OWN_FREE && !mbar_wait(bars.do_free(so), ((it / C::NO) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(bars.do_full(so), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_4d(sRing + (C::NQ + so) * C::TILE + c * kChunkBytes, &a.tm_do, c * 64, q_row, head, batch,
                      bars.do_full(so));
        ++issued_do;
      }
      if (*abort_flag) {
        for (int it = max(0, issued_q - C::NQ); it < issued_q; ++it)
          mbar_drain(bars.q_full(it % C::NQ), (it / C::NQ) & 1, a.timeout_ns);
        for (int it = max(0, issued_do - C::NO); it < issued_do; ++it)
          mbar_drain(bars.do_full(it % C::NO), (it / C::NO) & 1, a.timeout_ns);
        for (int it = max(0, issued_rowv - 2); it < issued_rowv; ++it)
          mbar_drain(bars.rowv_full(it & 1), (it >> 1) & 1, a.timeout_ns);
        mbar_drain(bars.kv_full(), 0, a.timeout_ns);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    griddep_wait();
    if (lane == 0 && n > 0) {
      constexpr uint32_t idS = idesc_f16(128, 128, BF16, false, false);   // K-major x K-major
      constexpr uint32_t idG = idesc_f16(128, D, BF16, false, true);      // dV, dK: A (TMEM) K-major, B MN-major
      constexpr uint32_t idQ = idesc_f16(128, D, BF16, true, true);       // dQ: A = dS MN-major, B = K MN-major
      constexpr uint32_t idQT = idesc_f16(D, 128, BF16, true, true);      // dQ^T: A = K^T MN-major, B = dS^T MN-major
      // ring slot (in tiles from the ring's start) of Q_it and of dO_it
      auto q_slot = [](int it) { return it % C::NQ; };
      auto do_slot = [](int it) { return C::NQ + it % C::NO; };
      // Descriptor low words of the operand bases (K-major: leading offset unused; MN-major: the
      // 64-column chunk stride).  A K step adds a constant, so one thread keeps up with the tensor core.
      constexpr uint32_t kTileLo = C::TILE >> 4;
      const uint32_t k_kmaj = sdesc_lo(sK, 16), v_kmaj = sdesc_lo(sV, 16), ring_kmaj = sdesc_lo(sRing, 16);
      const uint32_t ring_mn = sdesc_lo(sRing, kChunkBytes), k_mn = sdesc_lo(sK, kChunkBytes);
      const uint32_t ds_mn = sdesc_lo(sDS, kChunkBytes);

      // S^T_i = K Q_i^T into X
      auto issue_S = [&](int it) -> bool {
        if (!mbar_wait(bars.q_full(it % C::NQ), (it / C::NQ) & 1, wc)) return false;
        tc_fence_after();
        const uint32_t b_lo = ring_kmaj + q_slot(it) * kTileLo;
        mma_ss_lo<false>(tX, k_kmaj, b_lo, idS);
#pragma unroll
        for (int k = 1; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * kChunkBytes + (k & 3) * 32) >> 4;
          mma_ss_lo<true>(tX, k_kmaj + off, b_lo + off, idS);
        }
        mma_commit(bars.s_full());
        return true;
      };
      // dP^T_i = V dO_i^T into X (after the compute warps have read S^T_i)
      auto issue_dP = [&](int it) -> bool {
        if (!mbar_wait(bars.do_full(it % C::NO), (it / C::NO) & 1, wc)) return false;
        if (!mbar_wait(bars.s_used(), it & 1, wc)) return false;
        tc_fence_after();
        const uint32_t b_lo = ring_kmaj + do_slot(it) * kTileLo;
        mma_ss_lo<false>(tX, v_kmaj, b_lo, idS);
#pragma unroll
        for (int k = 1; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * kChunkBytes + (k & 3) * 32) >> 4;
          mma_ss_lo<true>(tX, v_kmaj + off, b_lo + off, idS);
        }
        mma_commit(bars.dp_full());
        return true;
      };

      bool ok = mbar_wait(bars.kv_full(), 0, wc);
      if (ok) ok = issue_S(0);
      if (ok) ok = issue_dP(0);
      for (int it = 0; ok && it < n; ++it) {
        // dV_i needs only P^T, which is in Y before dP^T_i lands: it queues behind dP^T_i and runs while
        // the compute warps form dS^T.
        if (!(ok = mbar_wait(bars.p_ready(), it & 1, wc))) break;
        tc_fence_after();
        const uint32_t q_lo = ring_mn + q_slot(it) * kTileLo;
        const uint32_t do_lo = ring_mn + do_slot(it) * kTileLo;
        const uint32_t acc0 = it > 0 ? 1u : 0u;
        // dV += P^T dO_i   (A: P^T packed in TMEM Y; B: dO_i [query][d] MN-major, 16 query rows per K step)
        mma_ts_lo_rt(tdV, tY + p_col<D>(0), do_lo, idG, acc0);
#pragma unroll
        for (int k = 1; k < 128 / 16; ++k) mma_ts_lo<true>(tdV, tY + p_col<D>(k), do_lo + k * (2048 >> 4), idG);
        if (C::DO_OWN_FREE) mma_commit(bars.do_free(it % C::NO));  // dO_i's last reader
        // dK += dS^T Q_i   (A: dS^T packed in TMEM X; B: Q_i [query][d] MN-major).  At d = 128 in the two
        // halves of its query (K) dimension, as the two compute warpgroups hand them over: warpgroup 0
        // hands over first (it stages part of its dQ later).  At d = 64 the warpgroups finish together and
        // a wait between the halves only cost time.
        if (!(ok = mbar_wait(bars.pd_ready(0), it & 1, wc))) break;
        tc_fence_after();
        mma_ts_lo_rt(tdK, tX + ds_col(0), q_lo, idG, acc0);
#pragma unroll
        for (int k = 1; k < 4; ++k) mma_ts_lo<true>(tdK, tX + ds_col(k), q_lo + k * (2048 >> 4), idG);
        if (D == 128) {
          if (!(ok = mbar_wait(bars.pd_ready(1), it & 1, wc))) break;
          tc_fence_after();
        }
#pragma unroll
        for (int k = 4; k < 128 / 16; ++k) mma_ts_lo<true>(tdK, tX + ds_col(k), q_lo + k * (2048 >> 4), idG);
        mma_commit(bars.q_free(it % C::NQ));  // Q_i's last reader (and dO_i's, before it)
        // S^T_{i+1} overwrites X after dK_i has read it, and dQ_i overwrites Y after dV_i has read it
        // (MMAs of one thread run in order).
        if (it + 1 < n && !(ok = issue_S(it + 1))) break;
        if constexpr (!DQ) {
          if (it + 1 < n && !(ok = issue_dP(it + 1))) break;
          continue;
        }
        if (it > 0 && !(ok = mbar_wait(bars.dq_empty(), (it - 1) & 1, wc))) break;
        if (!(ok = mbar_wait(bars.dss_ready(), it & 1, wc))) break;
        tc_fence_after();
        if constexpr (D == 128) {
          // dQ_i^T = K^T dS^T  (A: K^T [d][key] read MN-major from the K tile; B: dS^T [query][key] read
          // MN-major from the dS^T tile).  TMEM lane = d, so each warp's reduction covers whole rows.
          mma_ss_lo<false>(tY, k_mn, ds_mn, idQT);
#pragma unroll
          for (int k = 1; k < 128 / 16; ++k) mma_ss_lo<true>(tY, k_mn + k * (2048 >> 4), ds_mn + k * (2048 >> 4), idQT);
        } else {
          // dQ_i = dS K  (A: dS [query][key] read MN-major from the dS^T tile; B: K [key][d] MN-major)
          mma_ss_lo<false>(tY, ds_mn, k_mn, idQ);
#pragma unroll
          for (int k = 1; k < 128 / 16; ++k) mma_ss_lo<true>(tY, ds_mn + k * (2048 >> 4), k_mn + k * (2048 >> 4), idQ);
        }
        // dq_full also frees the dS^T tile (ds_empty).  At d = 64 the compute warps read dQ_i only after
        // dP_{i+1} has landed, whose commit covers dQ_i too: only the last tile's dQ needs its own.
        if (D == 128 || it + 1 == n) mma_commit(bars.dq_full());
        if (it + 1 < n && !(ok = issue_dP(it + 1))) break;
      }
      if (ok) mma_commit(bars.done());
      mma_commit(bars.mma_done());
      mbar_drain(bars.mma_done(), 0, a.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ compute
    griddep_wait();
    const int h = warp >> 2;             // query half: columns [64h, 64h + 64)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;   // TMEM lane: key row of S^T/dP^T; d (d = 128) or query row of dQ
    const int kv = k0 + r;
    const bool kv_valid = kv < a.Nk;
    const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
    const float c_log2 = a.scale * 1.4426950408889634f;
    const uint32_t ds_row = sDS + h * kChunkBytes;
    // Once a wait has failed (its time limit expired, or another warp raised the abort flag) a compute
    // warp does not leave the tile loop: it skips its remaining waits and runs on, so that every warp
    // of its warpgroup meets the warpgroup's named barriers equally often and in the same order.  (A
    // warp that left early would arrive at the epilogue's barrier of the same number while the others
    // wait inside the loop, and the barrier would release both groups in the wrong rounds.)  What the
    // warp computes after a failure is garbage: the epilogue skips the dK/dV stores (it checks the abort
    // flag), and the dQ still added into the accumulator is marked invalid by the error word.  `ok`
    // stays warp-uniform.
    bool ok = true;
    auto wait = [&](uint32_t bar, uint32_t parity) { ok = ok && mbar_wait_warp(bar, parity, wc); };

    // dQ_i from TMEM Y -> fp32 reductions into the accumulator; Y is released as soon as the
    // values are in registers.
    // d = 128: dQ_i^T: lane = d, column = query row.  This warpgroup reduces query rows [64h, 64h + 64):
    // it writes them row-major (the accumulator's layout; a warp's 32 lanes are 32 consecutive floats of
    // a row) into a 32 KB buffer and one thread has the copy engine add that contiguous block into the
    // accumulator.  Warpgroup 0 owns the staging tile (its previous reduction was issued a whole tile
    // ago); warpgroup 1 uses the dS^T tile, free from the end of the dQ_i MMA until the next dS^T store,
    // which waits for this reduction's read (see dstile_free).  The rows come out of TMEM 32 at a time;
    // with `pp`, this warpgroup's P^T of the next tile goes into the first 32 columns once they are read.
    // Part a stages the first 32 rows, part b the other 32 and hands the block to the copy engine.
    // Warpgroup 0 runs part b of dQ_{i-1} only after it has handed over its half of dS^T_i (its staging
    // tile is its own), so the dK half it feeds can start while warpgroup 1 still drains.
    const uint32_t buf_off = h ? C::OFF_DS : C::OFF_STAGE;
    float* const buf = reinterpret_cast<float*>(gbase + buf_off);
    auto drain128_a = [&](int it, bool with_p, const uint32_t (&pp)[32]) {
      wait(bars.dq_full(), it & 1);
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(tY + lane_bits + h * 64, v);
      tmem_wait_ld();
      reg_fence32(v);
      if (with_p) {
        tmem_st32(tY + lane_bits + p_base<D>() + h * p_stride<D>(), pp);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bars.p_ready());  // dV of the next tile may go
      }
      if (h == 0) {
        if (r == 0) tma_store_wait_read_all();  // the previous reduction from the staging tile
        named_bar_sync(1, 128);
      }
#pragma unroll
      for (int c = 0; c < 32; ++c) buf[c * D + r] = __uint_as_float(v[c]);
    };
    auto drain128_b = [&](int it) {
      uint32_t v[32];
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
    auto drain_dq = [&](int it) {
      if constexpr (D == 128) {
        const uint32_t none[32] = {};
        drain128_a(it, false, none);
        drain128_b(it);
      } else {
        // dQ_i is complete: for i < n - 1 the dP^T_{i+1} wait of this iteration showed it (dQ_i was
        // issued before dP_{i+1}); the last tile's dQ has a commit of its own.
        if (it + 1 == n) {
          wait(bars.dq_full(), 0);
          tc_fence_after();
        }
        // dQ_i: lane = query row; this warpgroup reduces d columns [32h, 32h + 32).  Its box [128
        // query][32 d] (128 bytes per row) goes into its half of the staging tile with the 128-byte
        // swizzle of the accumulator's tensor map (a thread writes one row: no bank conflicts), and one
        // thread has the copy engine add the box into the accumulator (a tensor reduce-add).
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
      }
    };

    const bool ragged_kv = k0 + kTileRows > a.Nk;  // block-uniform
    for (int it = 0; it < n; ++it) {
      const int qb = (i_start + it) * kTileRows + h * 64;  // first query column of this half
      const int rs = it & 1;                                // row-vector slot of this query tile
      const float* rowv = reinterpret_cast<const float*>(gbase + C::OFF_ROWV + rs * C::ROWV_BYTES);
      const float* nlse2 = rowv + h * 64;  // -LSE2: the exponent's additive term
      const float* dsum = rowv + 128 + h * 64;
      wait(bars.s_full(), it & 1);
      tc_fence_after();
      uint32_t s[2][32];
      tmem_ld32(tX + lane_bits + h * 64, s[0]);
      tmem_ld32(tX + lane_bits + h * 64 + 32, s[1]);
      tmem_wait_ld();
      reg_fence32(s[0]);
      reg_fence32(s[1]);
      tc_fence_before();
      mbar_arrive(bars.s_used());
      wait(bars.rowv_full(rs), (it >> 1) & 1);

      // P^T = exp2(S^T * scale*log2e - LSE2); masked entries are exactly 0.  Only query tiles the
      // causal diagonal crosses and a ragged last key block need the mask: columns below `lo` are zeroed.
      // Neighbouring query columns travel as fp32 pairs (the workspace holds -LSE2, so one paired FMA
      // forms two exponent arguments).
      const bool diag = CAUSAL && ((i_start + it) * kTileRows + coff < k0 + kTileRows - 1);
      const uint64_t c2 = f2_pack(c_log2, c_log2);
      float p[64];
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(nlse2 + c);
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const int col = c + e;
          const uint64_t s2 = f2_pack(__uint_as_float(s[col >> 5][col & 31]), __uint_as_float(s[col >> 5][(col + 1) & 31]));
          float x0, x1;
          f2_unpack(f2_fma(s2, c2, e ? f2_pack(l4.z, l4.w) : f2_pack(l4.x, l4.y)), x0, x1);
          p[col] = ex2_approx(x0);
          p[col + 1] = ex2_approx(x1);
        }
      }
      if (diag || ragged_kv) {
        const int lo = !kv_valid ? 64 : (diag ? kv - coff - qb : 0);
#pragma unroll
        for (int col = 0; col < 64; ++col)
          if (col < lo) p[col] = 0.f;
      }
      // P^T rounded to 16 bits: the dV MMA's operand, and the P used in dS below (so that dV and dK
      // see the same probabilities).
      uint32_t pp[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) pp[i] = pack2<BF16>(p[2 * i], p[2 * i + 1]);

      // P^T into Y, before dP^T_i lands: at d = 128 once this warpgroup has read dQ_{i-1}^T out of its
      // half of Y (dQ_{i-1} runs just before dP^T_i), at d = 64 straight away.  dV_i then queues behind
      // dP^T_i.  Staging dQ_{i-1} for the copy engine fits before dP^T_i lands.
      if (DQ && D == 128 && it > 0) {
        drain128_a(it - 1, true, pp);
        if (h == 1) drain128_b(it - 1);
      } else {
        tmem_st32(tY + lane_bits + p_base<D>() + h * p_stride<D>(), pp);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bars.p_ready());  // dV_i may go
      }

      wait(bars.dp_full(), it & 1);
      tc_fence_after();
      tmem_ld32(tX + lane_bits + h * 64, s[0]);
      tmem_ld32(tX + lane_bits + h * 64 + 32, s[1]);
      tmem_wait_ld();
      reg_fence32(s[0]);
      reg_fence32(s[1]);
      // dS^T = P^T o (dP^T - D), into the half's last 32 columns of X and into the shared dS^T tile.
      // Neighbouring query columns travel as fp32 pairs (the dP^T registers hold them side by side).
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float4 d4 = *reinterpret_cast<const float4*>(dsum + c);
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const int col = c + e;
          const uint64_t dp2 = f2_pack(__uint_as_float(s[col >> 5][col & 31]), __uint_as_float(s[col >> 5][(col + 1) & 31]));
          const uint64_t d2 = e ? f2_pack(d4.z, d4.w) : f2_pack(d4.x, d4.y);
          const uint64_t p2 = f2_pack(unpack_lo<BF16>(pp[col >> 1]), unpack_hi<BF16>(pp[col >> 1]));
          float ds0, ds1;
          f2_unpack(f2_mul(p2, f2_sub(dp2, d2)), ds0, ds1);
          pk[col >> 1] = pack2<BF16>(ds0, ds1);
        }
      }
      mbar_arrive(bars.rowv_empty(rs));
      tmem_st32(tX + lane_bits + h * 64 + 32, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bars.pd_ready(D == 128 ? h : 0));  // dK_i (at d = 128 this half of it) may go
      if constexpr (!DQ) continue;
      // The dQ_{i-1} MMA has read the dS^T tile.  At d = 64 the dP^T_i wait above showed that already.
      if (D == 128 && it > 0) wait(bars.ds_empty(), (it - 1) & 1);
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

      // The previous tile's dQ is staged and handed to the copy engine after this tile is handed over:
      // at d = 128 warpgroup 0's second half, at d = 64 all of it.
      if (DQ && D == 128 && it > 0 && h == 0) drain128_b(it - 1);
      if (DQ && D == 64 && it > 0) drain_dq(it - 1);
    }
    if (DQ && n > 0) drain_dq(n - 1);

    // ------------------------------------------------------------ epilogue
    // warps 0-3 write dV (staged in the V tile), warps 4-7 write dK * scale (staged in the K tile).
    if (ok && n > 0) ok = mbar_wait_warp(bars.done(), 0, wc);
    const uint32_t stage = h ? sK : sV;
    const uint32_t tacc = (h ? tdK : tdV) + lane_bits;
    const float mul = h ? a.scale : 1.0f;
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < C::NCH; ++ch) {
        uint32_t o[2][32];
        if (n > 0) {
          tmem_ld32(tacc + ch * 64, o[0]);
          tmem_ld32(tacc + ch * 64 + 32, o[1]);
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
            w[e] = pack2<BF16>(__uint_as_float(o[hh][b + 2 * e]) * mul, __uint_as_float(o[hh][b + 2 * e + 1]) * mul);
          st_shared_v4(stage + ch * kChunkBytes + sw128_offset(r, u), w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1 + h, 128);
    if (ok && r == 0 && !*abort_flag) {
      const CUtensorMap* map = h ? &a.tm_dk : &a.tm_dv;
      const uint64_t once = l2_evict_first();  // dK and dV are not read again here
      for (int ch = 0; ch < C::NCH; ++ch) tma_store_4d_hint(map, stage + ch * kChunkBytes, ch * 64, k0, head, batch, once);
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

// D = rowsum(dO o O), -LSE2 = -LSE * log2(e) (-inf on padding rows and on rows that see no key, so
// that their recomputed probabilities are exactly 0; stored negated, the exponent's additive term),
// dQacc = 0.
// TPR threads per row, 8 elements (16 bytes) per thread; a block covers pre_rows<D>() consecutive rows of
// one (batch, head), two per thread, with both rows' loads in flight before the first sum (one row per
// thread measured the same or slower, four and eight slower).  The block's (batch, head) and row range
// come from blockIdx.x by two 32-bit divisions.
constexpr int kPreRowsPerThread = 2;
template <int D>
__host__ __device__ constexpr int pre_rows_per_pass() { return 256 / (D / 8); }
template <int D>
__host__ __device__ constexpr int pre_rows() { return kPreRowsPerThread * pre_rows_per_pass<D>(); }

template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __grid_constant__ BwdArgs a) {
  // O, dO and LSE may come from the kernels just before; the workspace may still be read by the
  // previous backward's kernels.  Only after they are done may the main kernel start (its prologue
  // then overlaps this kernel's tail).
  griddep_wait();
  griddep_launch_dependents();
  constexpr int TPR = D / 8;
  constexpr int RPB = pre_rows_per_pass<D>();
  constexpr int NP = kPreRowsPerThread;
  const unsigned blocks_per_head = static_cast<unsigned>(a.Nq_pad) / pre_rows<D>();
  const unsigned bh = blockIdx.x / blocks_per_head;
  const int q0 = static_cast<int>(blockIdx.x - bh * blocks_per_head) * pre_rows<D>() + static_cast<int>(threadIdx.x) / TPR;
  const unsigned batch = bh / static_cast<unsigned>(a.heads), head = bh - batch * static_cast<unsigned>(a.heads);
  const int sub = threadIdx.x % TPR;
  const uint16_t* o = static_cast<const uint16_t*>(a.o) + batch * a.so.b + head * a.so.h + sub * 8;
  const uint16_t* dout = static_cast<const uint16_t*>(a.dout) + batch * a.sdo.b + head * a.sdo.h + sub * 8;
  uint4 ov[NP], dv[NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const int q = q0 + p * RPB;
    if (q < a.Nq) {
      ov[p] = __ldg(reinterpret_cast<const uint4*>(o + q * a.so.n));
      dv[p] = __ldg(reinterpret_cast<const uint4*>(dout + q * a.sdo.n));
    } else {
      ov[p] = dv[p] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  float acc[NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const uint32_t ow[4] = {ov[p].x, ov[p].y, ov[p].z, ov[p].w}, dw[4] = {dv[p].x, dv[p].y, dv[p].z, dv[p].w};
    acc[p] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc[p] = fmaf(unpack_lo<BF16>(ow[e]), unpack_lo<BF16>(dw[e]), acc[p]);
      acc[p] = fmaf(unpack_hi<BF16>(ow[e]), unpack_hi<BF16>(dw[e]), acc[p]);
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1)
#pragma unroll
    for (int p = 0; p < NP; ++p) acc[p] += __shfl_xor_sync(0xffffffffu, acc[p], off);
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const int q = q0 + p * RPB;
    const size_t row = static_cast<size_t>(bh) * a.Nq_pad + q;
    if (a.dq_acc != nullptr) {  // no accumulator in the deterministic mode
      float4* z = reinterpret_cast<float4*>(a.dq_acc + row * D + sub * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (sub == 0) {
      if (q < a.Nq) {
        const float lse = a.lse[static_cast<size_t>(bh) * a.Nq + q];
        a.nlse2[row] = lse == -INFINITY ? -INFINITY : -lse * 1.4426950408889634f;
        a.dsum[row] = acc[p];
      } else {
        a.nlse2[row] = -INFINITY;
        a.dsum[row] = 0.f;
      }
    }
  }
}

// dQ = scale * dQacc, rounded to the input dtype.  A block covers 2 x 256 chunks of 8 elements of one
// (batch, head); each thread loads both of its chunks before it converts either.  The accumulator's
// rows of one head are contiguous, so a chunk's source is the head's base plus 8 x its index.
constexpr int kConvChunks = 512;
template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const __grid_constant__ BwdArgs a) {
  griddep_wait();  // the accumulator is complete once the main kernel has finished
  constexpr int CPR = D / 8;  // chunks per row
  const int chunks = a.Nq * CPR;
  const unsigned blocks_per_head = static_cast<unsigned>((chunks + kConvChunks - 1) / kConvChunks);
  const unsigned bh = blockIdx.x / blocks_per_head;
  const int c0 = static_cast<int>(blockIdx.x - bh * blocks_per_head) * kConvChunks + static_cast<int>(threadIdx.x);
  const unsigned batch = bh / static_cast<unsigned>(a.heads), head = bh - batch * static_cast<unsigned>(a.heads);
  const float* acc = a.dq_acc + static_cast<size_t>(bh) * a.Nq_pad * D;
  uint16_t* dq = static_cast<uint16_t*>(a.dq) + batch * a.sdq.b + head * a.sdq.h;
  float4 x[2], y[2];
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const int c = c0 + p * 256;
    if (c < chunks) {
      const float4* src = reinterpret_cast<const float4*>(acc + static_cast<size_t>(c) * 8);
      x[p] = src[0];
      y[p] = src[1];
    }
  }
  const float s = a.scale;
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const int c = c0 + p * 256;
    if (c >= chunks) continue;
    uint4 out;
    out.x = pack2<BF16>(x[p].x * s, x[p].y * s);
    out.y = pack2<BF16>(x[p].z * s, x[p].w * s);
    out.z = pack2<BF16>(y[p].x * s, y[p].y * s);
    out.w = pack2<BF16>(y[p].z * s, y[p].w * s);
    const int q = c / CPR, col = (c % CPR) * 8;
    *reinterpret_cast<uint4*>(dq + static_cast<long long>(q) * a.sdq.n + col) = out;
  }
}

// Launches `kern` with programmatic stream serialisation: it may start before the previous kernel on
// the stream has finished, and waits for it with griddep_wait where it must.
template <typename Kern>
cudaError_t launch_dependent(Kern kern, dim3 grid, int threads, uint32_t smem, cudaStream_t stream, const BwdArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// steps: bit 0 = preprocess, bit 1 = main, bit 2 = dQ conversion (launched in that order, each as a
// dependent launch).
template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_bwd_t(const BwdArgs& a, int steps, cudaStream_t stream) {
  using C = BwdCfg<D>;
  if (steps & kBwdPre) {
    static_assert(kTileRows % pre_rows<D>() == 0, "a block's rows lie inside one head's padded rows");
    const size_t blocks = static_cast<size_t>(a.bh_count) * (a.Nq_pad / pre_rows<D>());
    cudaError_t e = launch_dependent(bwd_pre_kernel<D, BF16>, dim3(static_cast<unsigned>(blocks)), 256, 0, stream, a);
    if (e != cudaSuccess) return e;
  }
  if (steps & kBwdMain) {
    // no accumulator: the deterministic mode, where pair_dq_kernel produces dQ
    auto kern = a.dq_acc ? bwd_main_kernel<D, CAUSAL, BF16, true> : bwd_main_kernel<D, CAUSAL, BF16, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    const unsigned blocks = static_cast<unsigned>(a.bh_count) * ((a.Nk + kTileRows - 1) / kTileRows);
    e = launch_dependent(kern, dim3(blocks), kBwdThreads, C::SMEM_ALLOC, stream, a);
    if (e != cudaSuccess) return e;
  }
  if ((steps & kBwdConvert) && a.dq_acc) {
    const size_t per_head = (static_cast<size_t>(a.Nq) * (D / 8) + kConvChunks - 1) / kConvChunks;
    cudaError_t e = launch_dependent(bwd_dq_convert_kernel<D, BF16>, dim3(static_cast<unsigned>(a.bh_count * per_head)), 256,
                                     0, stream, a);
    if (e != cudaSuccess) return e;
  }
  if (steps & kBwdDq) return launch_bwd_dq(a, stream);
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, int steps, cudaStream_t stream) {
  if (a.d == 64) {
    if (a.causal)
      return a.bf16 ? launch_bwd_t<64, true, true>(a, steps, stream) : launch_bwd_t<64, true, false>(a, steps, stream);
    return a.bf16 ? launch_bwd_t<64, false, true>(a, steps, stream) : launch_bwd_t<64, false, false>(a, steps, stream);
  }
  if (a.causal)
    return a.bf16 ? launch_bwd_t<128, true, true>(a, steps, stream) : launch_bwd_t<128, true, false>(a, steps, stream);
  return a.bf16 ? launch_bwd_t<128, false, true>(a, steps, stream) : launch_bwd_t<128, false, false>(a, steps, stream);
}

}  // namespace exattn
