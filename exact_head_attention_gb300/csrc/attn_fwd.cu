// Fused attention forward for sm_103a.
//
// One CTA owns 256 query rows of one (batch, head): two 128-row query tiles
// Q0, Q1 that share every K/V tile it streams (SparkAttention, Figure 6: Q
// read once, K/V streamed, O written once; parallel over batch x heads x
// query-row blocks as in "Fast Transformer training with long sequences").
//
// Warp roles (384 threads, registers re-split per warpgroup):
//   warps 0-3  softmax warpgroup for query tile 0 (thread = query row)
//   warps 4-7  softmax warpgroup for query tile 1
//   warp  8    TMA producer: Q once, then K_j / V_j into NS-deep rings
//   warp  9    MMA issuer (one thread) and TMEM owner
//   warps 10-11 idle (they complete the control warpgroup)
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   [  0,128) S0 = Q0 K_j^T fp32; P0 (16-bit, packed in pairs) overwrites its first 64 columns
//   [128,256) S1 / P1
//   [256,256+d) O0 accumulator, [384,384+d) O1 accumulator
//
// Per key tile j and query tile t the MMA warp issues S_t = Q_t K_j^T, the
// softmax warpgroup turns S_t into P_t = exp2(S_t*scale*log2e - m) with the
// online running max m and running sum l (rescaling O_t in TMEM only when the
// max grows by more than 2^8 -- the final O/l is exact either way), writes P_t
// back into TMEM, and the MMA warp issues O_t += P_t V_j with P_t read from
// TMEM.  Issue order S0[0] S1[0] | PV0[j] S0[j+1] PV1[j] S1[j+1] | ... keeps
// the tensor pipe busy on one tile while the other tile's softmax runs.
// Causal (query q sees keys k <= q + causal_off: 0 for top-left alignment,
// Nk - Nq for bottom-right): key tiles past a query tile's diagonal are skipped
// entirely and only tiles the diagonal crosses (or the ragged last tile) are
// masked.  A query tile that sees no key at all (bottom-right, Nq > Nk) writes
// O = 0 and LSE = -inf without touching the tensor pipe.
//
// Launches: one CTA per 256-row block (grid (B*H, blocks), heaviest causal
// blocks first), or, for causal grids too coarse to balance that way, one CTA
// per SM over host-packed lists of blocks (fwd_schedule.h), walked by the same
// body with the barriers re-armed between blocks.  The causal forward of short
// sequences at d = 64 runs fwd_tile_kernel instead: one query tile per CTA, two
// CTAs per SM (described at that kernel).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fwd_schedule.h"
#include "fwd_tile.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "softmax.cuh"

namespace exattn {
namespace {

constexpr int kFwdThreads = 384;
// Register shares after reallocation (launch: 168 each).  Each SM sub-partition holds one warp of
// each of the three warpgroups, so the shares must sum to 3 x 168 = 504.
constexpr uint32_t kRegsSoftmax = 208, kRegsControl = 88;
static_assert(2 * kRegsSoftmax + kRegsControl == 3 * 168, "register split must match the launch");
constexpr uint32_t kChunkBytes = 128 * 128;  // 128 rows x 128 bytes

template <int D>
struct FwdCfg {
  static constexpr int NCH = D / 64;                      // 128-byte chunks per row
  static constexpr uint32_t TILE = kTileRows * D * 2;     // one 128-row 16-bit tile
  static constexpr int NS = (D == 64) ? 4 : 2;            // K and V ring depth
  // NS = 2: the ring slots are freed by the score commits of query tile 1 (S_1[j] completes after K_j's
  // last read, and after the P V_{j-1} products), so no commit of their own.  Those commits alternate
  // between two barriers by the key tile's parity.  A parity wait finds the completion it means only if
  // the waiter has seen the barrier's previous completion and the next one cannot have happened yet.
  // Before loading K_j and V_j the producer waits for S_1[j-2] and S_1[j-1]: every completion of both
  // barriers in turn, and on each barrier the completion after the awaited one is S_1[j] or S_1[j+1],
  // which needs the K_j or K_{j+1} it has yet to load.  A deeper ring keeps its own empty barriers.
  static constexpr bool FREE_BY_S1 = (NS == 2);
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + 2 * TILE;
  static constexpr uint32_t OFF_V = OFF_K + NS * TILE;
  static constexpr uint32_t OFF_BAR = OFF_V + NS * TILE;
  // barriers: q_full, k_full[NS], k_empty[NS], v_full[NS], v_empty[NS], s_full[2], p_full[2], o_full[2], mma_done,
  // s_full of query tile 1's odd key tiles (FREE_BY_S1)
  static constexpr int NBAR = 1 + 4 * NS + 8;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;  // tmem slot (4 B) + abort flag (4 B)
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static constexpr uint32_t SMEM_ALLOC = BYTES + 1024;      // slack for 1024-byte alignment
};

struct FwdBars {
  uint32_t base;
  int ns;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t k_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t k_empty(int s) const { return base + 8 * (1 + ns + s); }
  __device__ uint32_t v_full(int s) const { return base + 8 * (1 + 2 * ns + s); }
  __device__ uint32_t v_empty(int s) const { return base + 8 * (1 + 3 * ns + s); }
  __device__ uint32_t s_full(int t) const { return base + 8 * (1 + 4 * ns + t); }
  __device__ uint32_t s_full_odd1() const { return base + 8 * (8 + 4 * ns); }
  __device__ uint32_t p_full(int t) const { return base + 8 * (3 + 4 * ns + t); }
  __device__ uint32_t o_full(int t) const { return base + 8 * (5 + 4 * ns + t); }
  __device__ uint32_t mma_done() const { return base + 8 * (7 + 4 * ns); }
};

// The forward of query blocks units[0 .. nunits) of 256 rows each; unit = bh * nqb + qb.  A plain launch
// gives each CTA one block; a persistent launch gives each CTA (one per SM) a list that the host packed
// so that the CTAs' causal work is even.  Between two blocks every role has finished the first (its
// loads consumed, its MMAs drained, its O stored), and the barriers are re-armed.
template <int D, bool CAUSAL, bool BF16, bool MULTI>
__device__ __forceinline__ void fwd_body(const FwdArgs& a, const uint32_t* units, int nunits_arg) {
  const int nunits = MULTI ? nunits_arg : 1;  // a plain launch compiles without the block loop's machinery
  using C = FwdCfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  const FwdBars bars{sbase + C::OFF_BAR, NS};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + C::OFF_MISC + 4);
  const WaitCtx wc{abort_flag, a.err_word, a.timeout_ns};

  // A dependent launch after this kernel (the backward's preprocess) may start once every CTA is
  // running; it waits for this kernel to finish before it reads anything.
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (a.Nq + kFwdSubTiles * kTileRows - 1) / (kFwdSubTiles * kTileRows);
  const int nkv = (a.Nk + kTileRows - 1) / kTileRows;
  const int coff = CAUSAL ? a.causal_off : 0;

  // Query tile t's score commit for key tile j, and the parity of a wait for it (FREE_BY_S1: tile 1's
  // commits alternate between two barriers).
  auto score_bar = [&](int t, int j) { return (C::FREE_BY_S1 && t == 1 && (j & 1)) ? bars.s_full_odd1() : bars.s_full(t); };
  auto score_parity = [&](int t, int j) -> uint32_t { return (C::FREE_BY_S1 && t == 1) ? (j >> 1) & 1 : j & 1; };

  auto init_bars = [&] {
    mbar_init(bars.q_full(), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bars.k_full(s), 1);
      mbar_init(bars.k_empty(s), 1);
      mbar_init(bars.v_full(s), 1);
      mbar_init(bars.v_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bars.s_full(t), 1);
      mbar_init(bars.p_full(t), kTileRows);
      mbar_init(bars.o_full(t), 1);
    }
    mbar_init(bars.s_full_odd1(), 1);
    mbar_init(bars.mma_done(), 1);
    fence_mbar_init();
  };
  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    init_bars();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Start of block ui: after the first, all threads meet (named barrier 3), and unless a wait gave up
  // in an earlier block (then every thread leaves the loop together) thread 0 re-arms the barriers.
  auto next_unit = [&](int ui) -> bool {
    if (!MULTI || ui == 0) return true;
    tc_fence_before();
    named_bar_sync(3, kFwdThreads);
    const bool go = *abort_flag == 0u;
    if (go && threadIdx.x == 0) {
      mbar_inval(bars.q_full());
      for (int s = 0; s < NS; ++s) {
        mbar_inval(bars.k_full(s));
        mbar_inval(bars.k_empty(s));
        mbar_inval(bars.v_full(s));
        mbar_inval(bars.v_empty(s));
      }
      for (int t = 0; t < 2; ++t) {
        mbar_inval(bars.s_full(t));
        mbar_inval(bars.p_full(t));
        mbar_inval(bars.o_full(t));
      }
      mbar_inval(bars.s_full_odd1());
      mbar_inval(bars.mma_done());
      init_bars();
    }
    named_bar_sync(3, kFwdThreads);
    tc_fence_after();
    return go;
  };
  // the block's coordinates and the key tiles its query tiles visit (causal: through the tile holding
  // the last key the tile's last row sees)
  struct Unit {
    int bh, head, batch, q0, ntile0, ntile1;  // ntile1 >= ntile0
  };
  auto unit_of = [&](int ui) {
    Unit u;
    int qb;
    if constexpr (MULTI) {
      u.bh = static_cast<int>(units[ui]) / nqb;
      qb = static_cast<int>(units[ui]) % nqb;
    } else {  // a plain launch: (B*H, blocks) grid, heaviest causal blocks first
      u.bh = blockIdx.x;
      qb = gridDim.y - 1 - blockIdx.y;
    }
    u.head = u.bh % a.heads;
    u.batch = u.bh / a.heads;
    u.q0 = qb * (kFwdSubTiles * kTileRows);
    auto tiles_of = [&](int t) {
      if (!CAUSAL) return nkv;
      const int last_key = u.q0 + t * kTileRows + kTileRows - 1 + coff;
      return last_key < 0 ? 0 : min(nkv, last_key / kTileRows + 1);
    };
    u.ntile0 = tiles_of(0);
    u.ntile1 = tiles_of(1);
    return u;
  };

  if (warp >= 8) {
    // ------------------------------------------------------------ control warpgroup
    // warp 8: TMA producer, warp 9: MMA issuer, warps 10-11: idle.
    regs_decrease<kRegsControl>();
    for (int ui = 0; ui < nunits; ++ui) {
      if (!next_unit(ui)) break;
      const Unit u = unit_of(ui);
      const int bh = u.bh, head = u.head, batch = u.batch, q0 = u.q0, ntile0 = u.ntile0, ntile1 = u.ntile1;
      (void)bh;
      if (warp == 8 && lane == 0 && ntile1 > 0) {
        // ---- producer
        prefetch_tmap(&a.tm_q);
        prefetch_tmap(&a.tm_k);
        prefetch_tmap(&a.tm_v);
        mbar_arrive_expect_tx(bars.q_full(), 2 * C::TILE);
        for (int t = 0; t < 2; ++t)
          for (int c = 0; c < C::NCH; ++c)
            tma_load_4d(sQ + t * C::TILE + c * kChunkBytes, &a.tm_q, c * 64, q0 + t * kTileRows, head, batch, bars.q_full());
        int issued_k = 0, issued_v = 0;
        for (int j = 0; j < ntile1; ++j) {
          const int s = j % NS;
          const uint32_t ph = (j / NS) & 1;
          // K_{j-NS} is free once S_1[j-NS] has completed; V_{j-NS} once S_1[j-NS+1] has (it follows
          // P_1 V_{j-NS}).
          if (C::FREE_BY_S1 ? (j >= NS && !mbar_wait(score_bar(1, j - NS), score_parity(1, j - NS), wc))
                            : !mbar_wait(bars.k_empty(s), ph ^ 1, wc))
            break;
          mbar_arrive_expect_tx(bars.k_full(s), C::TILE);
          for (int c = 0; c < C::NCH; ++c)
            tma_load_4d(sK + s * C::TILE + c * kChunkBytes, &a.tm_k, c * 64, j * kTileRows, head, batch, bars.k_full(s));
          ++issued_k;
          if (C::FREE_BY_S1 ? (j >= NS && !mbar_wait(score_bar(1, j - NS + 1), score_parity(1, j - NS + 1), wc))
                            : !mbar_wait(bars.v_empty(s), ph ^ 1, wc))
            break;
          mbar_arrive_expect_tx(bars.v_full(s), C::TILE);
          for (int c = 0; c < C::NCH; ++c)
            tma_load_4d(sV + s * C::TILE + c * kChunkBytes, &a.tm_v, c * 64, j * kTileRows, head, batch, bars.v_full(s));
          ++issued_v;
        }
        // On abort, every load this thread issued must land before the CTA exits.
        if (*abort_flag) {
          for (int j = max(0, issued_k - NS); j < issued_k; ++j) mbar_drain(bars.k_full(j % NS), (j / NS) & 1, a.timeout_ns);
          for (int j = max(0, issued_v - NS); j < issued_v; ++j) mbar_drain(bars.v_full(j % NS), (j / NS) & 1, a.timeout_ns);
          mbar_drain(bars.q_full(), 0, a.timeout_ns);
        } else if (!C::FREE_BY_S1 && MULTI && nunits > 1) {
          // Before the next block re-arms the barriers, the commits that free the ring slots (the last
          // ones are never waited for otherwise) must all have arrived.  (With FREE_BY_S1 they are the
          // score commits, each of which softmax warpgroup 1 waits for.)
          for (int j = ntile1; j < ntile1 + NS; ++j) {
            if (!mbar_wait(bars.k_empty(j % NS), ((j / NS) & 1) ^ 1, wc)) break;
            if (!mbar_wait(bars.v_empty(j % NS), ((j / NS) & 1) ^ 1, wc)) break;
          }
        }
      } else if (warp == 9 && lane == 0 && ntile1 > 0) {
        // ---- MMA issuer
        constexpr uint32_t idS = idesc_f16(128, 128, BF16, false, false);
        constexpr uint32_t idPV = idesc_f16(128, D, BF16, false, true);
        bool ok = mbar_wait(bars.q_full(), 0, wc);
        // Descriptor low words of the operand bases; a K step adds a constant (the issue loop of a
        // single thread must keep up with one MMA per 64 tensor-core cycles).
        constexpr uint32_t kTileLo = C::TILE >> 4;
        const uint32_t q_lo = sdesc_lo(sQ, 16), k_lo = sdesc_lo(sK, 16), v_lo = sdesc_lo(sV, kChunkBytes);

        auto issue_S = [&](int t, int j) -> bool {
          const int s = j % NS;
          if (!mbar_wait(bars.k_full(s), (j / NS) & 1, wc)) return false;
          tc_fence_after();
          const uint32_t d = tmem + t * 128, a_lo = q_lo + t * kTileLo, b_lo = k_lo + s * kTileLo;
          mma_ss_lo<false>(d, a_lo, b_lo, idS);
  #pragma unroll
          for (int k = 1; k < D / 16; ++k) {
            const uint32_t off = ((k >> 2) * kChunkBytes + (k & 3) * 32) >> 4;
            mma_ss_lo<true>(d, a_lo + off, b_lo + off, idS);
          }
          mma_commit(score_bar(t, j));
          return true;
        };
        auto issue_PV = [&](int t, int j) -> bool {
          const int s = j % NS;
          if (!mbar_wait(bars.v_full(s), (j / NS) & 1, wc)) return false;
          if (!mbar_wait(bars.p_full(t), j & 1, wc)) return false;
          tc_fence_after();
          const uint32_t d = tmem + 256 + t * 128, a = tmem + t * 128, b_lo = v_lo + s * kTileLo;
          mma_ts_lo_rt(d, a, b_lo, idPV, j > 0 ? 1u : 0u);
  #pragma unroll
          for (int k = 1; k < kTileRows / 16; ++k) mma_ts_lo<true>(d, a + k * 8, b_lo + k * (2048 >> 4), idPV);
          return true;
        };

        if (ok && ntile0 > 0) ok = issue_S(0, 0);
        if (ok) ok = issue_S(1, 0);
        if (ok && !C::FREE_BY_S1) mma_commit(bars.k_empty(0));
        for (int j = 0; ok && j < ntile1; ++j) {
          if (j < ntile0) {
            if (!(ok = issue_PV(0, j))) break;
            if (j == ntile0 - 1) mma_commit(bars.o_full(0));
            if (j + 1 < ntile0 && !(ok = issue_S(0, j + 1))) break;
          }
          if (!(ok = issue_PV(1, j))) break;
          if (!C::FREE_BY_S1) mma_commit(bars.v_empty(j % NS));
          if (j == ntile1 - 1) mma_commit(bars.o_full(1));
          if (j + 1 < ntile1) {
            if (!(ok = issue_S(1, j + 1))) break;
            if (!C::FREE_BY_S1) mma_commit(bars.k_empty((j + 1) % NS));
          }
        }
        // Every MMA issued above completes before TMEM can be released.
        mma_commit(bars.mma_done());
        mbar_drain(bars.mma_done(), 0, a.timeout_ns);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    regs_increase<kRegsSoftmax>();
    for (int ui = 0; ui < nunits; ++ui) {
      if (!next_unit(ui)) break;
      const Unit u = unit_of(ui);
      const int bh = u.bh, head = u.head, batch = u.batch, q0 = u.q0, ntile0 = u.ntile0, ntile1 = u.ntile1;
      const int t = warp >> 2;                  // query tile of this warpgroup
      const int quarter = warp & 3;             // TMEM lane quarter this warp may access
      const int r = quarter * 32 + lane;        // row inside the tile = TMEM lane
      const int row = q0 + t * kTileRows + r;   // query index inside the head
      const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
      const uint32_t tS = tmem + t * 128 + lane_bits;
      const uint32_t tO = tmem + 256 + t * 128 + lane_bits;
      const float c_log2 = a.scale * 1.4426950408889634f;  // scale * log2(e)
      const int n = t ? ntile1 : ntile0;
      float m = -INFINITY;  // running max of the scaled scores, base-2 units
      float l = 0.f;        // running sum of exp2(score - m)
      bool ok = true;

      for (int j = 0; j < n; ++j) {
        if (!(ok = mbar_wait_warp(score_bar(t, j), score_parity(t, j), wc))) break;
        tc_fence_after();
        // Columns at or past `lim` are masked (ragged last key tile, causal diagonal tile).
        const bool need_mask =
            ((j + 1) * kTileRows > a.Nk) || (CAUSAL && j * kTileRows + kTileRows - 1 > q0 + t * kTileRows + coff);
        const int lim = need_mask ? (CAUSAL ? min(a.Nk, row + coff + 1) : a.Nk) - j * kTileRows : kTileRows;
        if (need_mask)
          softmax_tile<D, true, BF16>(tS, tO, lim, c_log2, j == 0, m, l, [] {});
        else
          softmax_tile<D, false, BF16>(tS, tO, lim, c_log2, j == 0, m, l, [] {});
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bars.p_full(t));
      }

      // ------------------------------------------------------------ epilogue
      // A row that saw no key (l = 0) gets O = 0 and LSE = -inf.  A tile with no key tiles at all
      // never had its O accumulated; it stages zeros once the Q copy into its staging tile has landed.
      // (With no key tile anywhere in the block nothing was loaded and there is nothing to wait for.)
      if (ok && (n > 0 || ntile1 > 0)) ok = mbar_wait_warp(n > 0 ? bars.o_full(t) : bars.q_full(), 0, wc);
      if (ok) {
        tc_fence_after();
        const float inv_l = l > 0.f ? 1.0f / l : 0.f;
        if (row < a.Nq)
          a.lse[static_cast<size_t>(bh) * a.Nq + row] = l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
        const uint32_t stage = sQ + t * C::TILE;  // Q_t is dead: all of its MMAs completed before o_full
  #pragma unroll
        for (int ch = 0; ch < C::NCH; ++ch) {
          uint32_t o[2][32];
          if (n > 0) {
            tmem_ld32(tO + ch * 64, o[0]);
            tmem_ld32(tO + ch * 64 + 32, o[1]);
            tmem_wait_ld();
            reg_fence32(o[0]);
            reg_fence32(o[1]);
          } else {
  #pragma unroll
            for (int i = 0; i < 32; ++i) o[0][i] = o[1][i] = 0u;
          }
  #pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int h = u >> 2, b = (u & 3) * 8;
            const uint32_t w0 = pack2<BF16>(__uint_as_float(o[h][b + 0]) * inv_l, __uint_as_float(o[h][b + 1]) * inv_l);
            const uint32_t w1 = pack2<BF16>(__uint_as_float(o[h][b + 2]) * inv_l, __uint_as_float(o[h][b + 3]) * inv_l);
            const uint32_t w2 = pack2<BF16>(__uint_as_float(o[h][b + 4]) * inv_l, __uint_as_float(o[h][b + 5]) * inv_l);
            const uint32_t w3 = pack2<BF16>(__uint_as_float(o[h][b + 6]) * inv_l, __uint_as_float(o[h][b + 7]) * inv_l);
            st_shared_v4(stage + ch * kChunkBytes + sw128_offset(r, u), w0, w1, w2, w3);
          }
        }
        fence_proxy_async_smem();
      }
      named_bar_sync(1 + t, 128);
      if (ok && r == 0 && q0 + t * kTileRows < a.Nq && !*abort_flag) {
        for (int ch = 0; ch < C::NCH; ++ch)
          tma_store_4d(&a.tm_o, sQ + t * C::TILE + ch * kChunkBytes, ch * 64, q0 + t * kTileRows, head, batch);
        tma_store_commit();
        tma_store_wait_all();
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

// One 256-row query block per CTA; the grid is (B*H, blocks) with the heaviest causal blocks first.
template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel(const __grid_constant__ FwdArgs a) {
  fwd_body<D, CAUSAL, BF16, false>(a, nullptr, 1);
}

// Persistent: CTA i takes the blocks sch.unit[sch.begin[i] .. sch.begin[i + 1]).
template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel_persistent(const __grid_constant__ FwdArgs a,
                                                                       const __grid_constant__ FwdSchedule sch) {
  const int b = sch.begin[blockIdx.x], e = sch.begin[blockIdx.x + 1];
  fwd_body<D, CAUSAL, BF16, true>(a, sch.unit + b, e - b);
}

// One 128-row query tile per CTA, two CTAs per SM (fwd_tile.cuh): the causal forward of short sequences
// at d = 64.  Where a head has few key tiles, a 256-row block's start (its first loads come from DRAM)
// and drain (the epilogue, and a query tile that finishes early waiting for its partner at the
// teardown) are a large share of its time, and with one CTA per SM nothing hides them.  Grid
// (B*H, ceil(Nq/128)), heaviest causal tiles first.
template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(tile::kThreads, 2) fwd_tile_kernel(const __grid_constant__ FwdArgs a) {
  griddep_launch_dependents();
  const int bh = blockIdx.x;
  tile::Work w;
  w.head = bh % a.heads;
  w.batch = bh / a.heads;
  w.q0 = (gridDim.y - 1 - blockIdx.y) * kTileRows;
  w.j0 = 0;
  const int nkv = (a.Nk + kTileRows - 1) / kTileRows;
  w.n = nkv;  // key tiles the query tile sees (causal: through the tile of its last row's last key)
  if (CAUSAL) {
    const int last_key = w.q0 + kTileRows - 1 + a.causal_off;
    w.n = last_key < 0 ? 0 : min(nkv, last_key / kTileRows + 1);
  }
  // O / l rounded to the dtype, staged in the dead Q tile with the tensor map's swizzle, one TMA store;
  // a row that saw no key (l = 0) gets O = 0 and LSE = -inf.
  auto epilogue = [&](bool ok, float m, float l, int r, uint32_t tO, uint32_t sQ, volatile uint32_t* abort_flag) {
    using C = tile::Cfg<D>;
    const int row = w.q0 + r;
    if (ok) {
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      if (row < a.Nq)
        a.lse[static_cast<size_t>(bh) * a.Nq + row] = l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
#pragma unroll
      for (int ch = 0; ch < C::NCH; ++ch) {
        uint32_t o[2][32];
        if (w.n > 0) {
          tmem_ld32(tO + ch * 64, o[0]);
          tmem_ld32(tO + ch * 64 + 32, o[1]);
          tmem_wait_ld();
          reg_fence32(o[0]);
          reg_fence32(o[1]);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[0][i] = o[1][i] = 0u;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int h = u >> 2, b = (u & 3) * 8;
          const uint32_t w0 = pack2<BF16>(__uint_as_float(o[h][b + 0]) * inv_l, __uint_as_float(o[h][b + 1]) * inv_l);
          const uint32_t w1 = pack2<BF16>(__uint_as_float(o[h][b + 2]) * inv_l, __uint_as_float(o[h][b + 3]) * inv_l);
          const uint32_t w2 = pack2<BF16>(__uint_as_float(o[h][b + 4]) * inv_l, __uint_as_float(o[h][b + 5]) * inv_l);
          const uint32_t w3 = pack2<BF16>(__uint_as_float(o[h][b + 6]) * inv_l, __uint_as_float(o[h][b + 7]) * inv_l);
          st_shared_v4(sQ + ch * tile::kChunkBytes + sw128_offset(r, u), w0, w1, w2, w3);
        }
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (ok && r == 0 && w.q0 < a.Nq && !*abort_flag) {
      for (int ch = 0; ch < C::NCH; ++ch)
        tma_store_4d(&a.tm_o, sQ + ch * tile::kChunkBytes, ch * 64, w.q0, w.head, w.batch);
      tma_store_commit();
      tma_store_wait_all();
    }
  };
  tile::run<D, CAUSAL, BF16>(&a.tm_q, &a.tm_k, &a.tm_v, w, a.Nk, a.causal_off, a.scale, a.err_word, a.timeout_ns,
                             epilogue);
}

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t stream) {
  using C = FwdCfg<D>;
  // The one-tile kernel serves the causal forward at d = 64 when a query tile sees few key tiles: there a
  // two-tile block's start and drain are not hidden by a second resident block, and its two query tiles'
  // work differs.  (With no mask the tiles of a head are alike, and the two-tile kernel, which streams
  // each K/V tile once for two query tiles, measured as fast or faster.)
  if constexpr (D == 64 && CAUSAL) {
    if (fwd_uses_tile_kernel(D, CAUSAL, a.Nk)) {
      using T = tile::Cfg<D>;
      auto kern = fwd_tile_kernel<D, CAUSAL, BF16>;
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_ALLOC);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
      kern<<<dim3(a.bh_count, (a.Nq + kTileRows - 1) / kTileRows, 1), tile::kThreads, T::SMEM_ALLOC, stream>>>(a);
      return cudaGetLastError();
    }
  }
  const int nqb = (a.Nq + kFwdSubTiles * kTileRows - 1) / (kFwdSubTiles * kTileRows);
  const FwdSchedule* sch = CAUSAL ? persistent_schedule(a.bh_count, nqb, a.Nq, a.Nk, a.causal_off, a.sm_count) : nullptr;
  if (sch) {
    auto kern = fwd_kernel_persistent<D, CAUSAL, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    kern<<<sch->ctas, kFwdThreads, C::SMEM_ALLOC, stream>>>(a, *sch);
    return cudaGetLastError();
  }
  auto kern = fwd_kernel<D, CAUSAL, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  dim3 grid(a.bh_count, nqb, 1);
  kern<<<grid, kFwdThreads, C::SMEM_ALLOC, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  if (a.d == 64) {
    if (a.causal) return a.bf16 ? launch_fwd_t<64, true, true>(a, stream) : launch_fwd_t<64, true, false>(a, stream);
    return a.bf16 ? launch_fwd_t<64, false, true>(a, stream) : launch_fwd_t<64, false, false>(a, stream);
  }
  if (a.causal) return a.bf16 ? launch_fwd_t<128, true, true>(a, stream) : launch_fwd_t<128, true, false>(a, stream);
  return a.bf16 ? launch_fwd_t<128, false, true>(a, stream) : launch_fwd_t<128, false, false>(a, stream);
}

}  // namespace exattn
