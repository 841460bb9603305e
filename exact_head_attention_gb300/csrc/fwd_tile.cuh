// One 128-row query tile per CTA, two CTAs per SM: the body shared by the forward of short causal
// sequences at d = 64 (attn_fwd.cu) and the split-KV forward at d = 64 (attn_splitkv.cu).
//
// A CTA holds one query tile (d = 64) in 256 TMEM columns -- S [0, 128), O [128, 192) and P, packed
// 16-bit, [192, 256) -- and 80 KB of shared memory, so two CTAs share an SM: one's start (its first
// loads come from DRAM) and drain overlap the other's products, and two online-softmax chains run per
// SM where one CTA of the split-KV forward runs one.  The per-tile step is the two-tile forward's online
// softmax (the same arithmetic in the same order, so the same results), with P in columns of its own.
//
// Warp roles (256 threads, two warpgroups): warps 0-3 softmax (thread = query row = TMEM lane), warp 4
// TMA producer, warp 5 MMA issuer and TMEM owner, warps 6-7 idle (they complete the control
// warpgroup).  Two CTAs of 256 threads launch with 128 registers a thread; setmaxnreg moves 80 of the
// control warpgroup's to the softmax warpgroup (208 / 48), which holds a whole score row.  Issue order
// S_0 | S_1 PV_0 | S_2 PV_1 ...: S_{i+1} is issued as soon as the softmax warps hold S_i in registers
// (s_used), so it overlaps their exponentials; PV_i once P_i is in TMEM (p_full).  Before the softmax
// of tile i+1 rescales O or writes P_{i+1}, it waits for PV_i (pv_done).
#pragma once

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "softmax.cuh"

namespace exattn {
namespace tile {

constexpr uint32_t kChunkBytes = 128 * 128;  // 128 rows x 128 bytes
constexpr int kThreads = 256;
constexpr uint32_t kRegsSoftmax = 208, kRegsControl = 48;
static_assert(kRegsSoftmax + kRegsControl == 2 * 128, "register split must match the launch (2 CTAs of 256)");

template <int D>
struct Cfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = kTileRows * D * 2;
  static constexpr int NS = 2;  // K and V ring depth (3 measured no faster)
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + TILE;
  static constexpr uint32_t OFF_V = OFF_K + NS * TILE;
  static constexpr uint32_t OFF_BAR = OFF_V + NS * TILE;
  // q_full, k_full[NS], k_empty[NS], v_full[NS], v_empty[NS], s_full, p_full, o_full, mma_done, s_used,
  // pv_done
  static constexpr int NBAR = 1 + 4 * NS + 6;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;  // tmem slot (4 B) + abort flag (4 B)
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  // No alignment slack (two CTAs must fit an SM): the dynamic shared memory base is checked at entry.
  static constexpr uint32_t SMEM_ALLOC = BYTES;
  static_assert(2 * (SMEM_ALLOC + 1024) <= 228 * 1024, "two CTAs per SM (1 KB of each CTA's is reserved)");
};

struct Bars {
  uint32_t base;
  int ns;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t k_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t k_empty(int s) const { return base + 8 * (1 + ns + s); }
  __device__ uint32_t v_full(int s) const { return base + 8 * (1 + 2 * ns + s); }
  __device__ uint32_t v_empty(int s) const { return base + 8 * (1 + 3 * ns + s); }
  __device__ uint32_t s_full() const { return base + 8 * (1 + 4 * ns); }
  __device__ uint32_t p_full() const { return base + 8 * (2 + 4 * ns); }
  __device__ uint32_t o_full() const { return base + 8 * (3 + 4 * ns); }
  __device__ uint32_t mma_done() const { return base + 8 * (4 + 4 * ns); }
  __device__ uint32_t s_used() const { return base + 8 * (5 + 4 * ns); }   // S is in the softmax's registers
  __device__ uint32_t pv_done() const { return base + 8 * (6 + 4 * ns); }  // the last P V product has completed
};

// What one CTA computes: query tile q0 of head (head, batch) against key tiles [j0, j0 + n).
struct Work {
  int head, batch, q0, j0, n;
};

// The whole CTA: set-up, producer, MMA issuer and online softmax over the work's key tiles.  The four
// softmax warps then call epilogue(ok, m, l, r, tO, sQ, abort_flag): ok is false when a wait gave up;
// m and l are the row's running max (base-2 units of the scaled scores) and sum; r is the row in the
// tile (the thread index, 0..127); tO is its O row in TMEM (holding sum_k exp2(s - m) V_k when
// work.n > 0; an epilogue must not read it otherwise); sQ is the Q tile's shared memory, free for
// staging (every MMA has completed).  Then the CTA tears down.  Every wait is bounded.
template <int D, bool CAUSAL, bool BF16, typename Epilogue>
__device__ __forceinline__ void run(const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                    const Work& w, int Nk, int causal_off, float scale, uint32_t* err_word,
                                    uint64_t timeout_ns, Epilogue&& epilogue) {
  static_assert(D == 64, "S, O and a separate P fill the 256 TMEM columns only at d = 64");
  using C = Cfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  if (!smem_base_aligned(sbase, err_word)) return;
  uint8_t* gbase = smem_raw;
  const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  const Bars bars{sbase + C::OFF_BAR, NS};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + C::OFF_MISC + 4);
  const WaitCtx wc{abort_flag, err_word, timeout_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = w.n;

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    mbar_init(bars.q_full(), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bars.k_full(s), 1);
      mbar_init(bars.k_empty(s), 1);
      mbar_init(bars.v_full(s), 1);
      mbar_init(bars.v_empty(s), 1);
    }
    mbar_init(bars.s_full(), 1);
    mbar_init(bars.p_full(), kTileRows);
    mbar_init(bars.o_full(), 1);
    mbar_init(bars.mma_done(), 1);
    mbar_init(bars.s_used(), kTileRows);
    mbar_init(bars.pv_done(), 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 4) {
    regs_decrease<kRegsControl>();
    if (warp == 4 && lane == 0 && n > 0) {
      // ---------------------------------------------------------- producer
      prefetch_tmap(tm_q);
      prefetch_tmap(tm_k);
      prefetch_tmap(tm_v);
      mbar_arrive_expect_tx(bars.q_full(), C::TILE);
      for (int c = 0; c < C::NCH; ++c) tma_load_4d(sQ + c * kChunkBytes, tm_q, c * 64, w.q0, w.head, w.batch, bars.q_full());
      int issued_k = 0, issued_v = 0;
      for (int i = 0; i < n; ++i) {
        const int s = i % NS;
        const uint32_t ph = (i / NS) & 1;
        const int key0 = (w.j0 + i) * kTileRows;
        if (!mbar_wait(bars.k_empty(s), ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(bars.k_full(s), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_4d(sK + s * C::TILE + c * kChunkBytes, tm_k, c * 64, key0, w.head, w.batch, bars.k_full(s));
        ++issued_k;
        if (!mbar_wait(bars.v_empty(s), ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(bars.v_full(s), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_4d(sV + s * C::TILE + c * kChunkBytes, tm_v, c * 64, key0, w.head, w.batch, bars.v_full(s));
        ++issued_v;
      }
      // On abort, every load this thread issued must land before the CTA exits.
      if (*abort_flag) {
        for (int i = max(0, issued_k - NS); i < issued_k; ++i) mbar_drain(bars.k_full(i % NS), (i / NS) & 1, timeout_ns);
        for (int i = max(0, issued_v - NS); i < issued_v; ++i) mbar_drain(bars.v_full(i % NS), (i / NS) & 1, timeout_ns);
        mbar_drain(bars.q_full(), 0, timeout_ns);
      }
    } else if (warp == 5 && lane == 0 && n > 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idS = idesc_f16(128, 128, BF16, false, false);
      constexpr uint32_t idPV = idesc_f16(128, D, BF16, false, true);
      constexpr uint32_t kTileLo = C::TILE >> 4;
      const uint32_t q_lo = sdesc_lo(sQ, 16), k_lo = sdesc_lo(sK, 16), v_lo = sdesc_lo(sV, kChunkBytes);
      auto issue_S = [&](int i) -> bool {
        const int s = i % NS;
        if (!mbar_wait(bars.k_full(s), (i / NS) & 1, wc)) return false;
        tc_fence_after();
        const uint32_t b_lo = k_lo + s * kTileLo;
        mma_ss_lo<false>(tmem, q_lo, b_lo, idS);
#pragma unroll
        for (int k = 1; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * kChunkBytes + (k & 3) * 32) >> 4;
          mma_ss_lo<true>(tmem, q_lo + off, b_lo + off, idS);
        }
        mma_commit(bars.s_full());
        mma_commit(bars.k_empty(s));
        return true;
      };
      auto issue_PV = [&](int i) -> bool {
        const int s = i % NS;
        if (!mbar_wait(bars.v_full(s), (i / NS) & 1, wc)) return false;
        if (!mbar_wait(bars.p_full(), i & 1, wc)) return false;
        tc_fence_after();
        const uint32_t d = tmem + 128, pa = tmem + 192, b_lo = v_lo + s * kTileLo;
        mma_ts_lo_rt(d, pa, b_lo, idPV, i > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 1; k < kTileRows / 16; ++k) mma_ts_lo<true>(d, pa + k * 8, b_lo + k * (2048 >> 4), idPV);
        mma_commit(bars.v_empty(s));
        mma_commit(bars.pv_done());
        return true;
      };
      bool ok = mbar_wait(bars.q_full(), 0, wc);
      if (ok) ok = issue_S(0);
      for (int i = 0; ok && i < n; ++i) {
        // S_{i+1} overwrites S_i once the softmax warps hold S_i in registers
        if (i + 1 < n && !((ok = mbar_wait(bars.s_used(), i & 1, wc)) && (ok = issue_S(i + 1)))) break;
        if (!(ok = issue_PV(i))) break;
        if (i == n - 1) mma_commit(bars.o_full());
      }
      // Every MMA issued above completes before TMEM can be released.
      mma_commit(bars.mma_done());
      mbar_drain(bars.mma_done(), 0, timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ softmax
    regs_increase<kRegsSoftmax>();
    const int r = warp * 32 + lane;  // row inside the tile = TMEM lane
    const int row = w.q0 + r;        // query index inside the head
    const uint32_t lane_bits = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_bits, tO = tmem + 128 + lane_bits, tP = tmem + 192 + lane_bits;
    const float c_log2 = scale * 1.4426950408889634f;
    const int coff = CAUSAL ? causal_off : 0;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      if (!(ok = mbar_wait_warp(bars.s_full(), i & 1, wc))) break;
      tc_fence_after();
      // Columns at or past `lim` are masked (ragged last key tile, causal diagonal tile).
      const int j = w.j0 + i;
      const bool need_mask = ((j + 1) * kTileRows > Nk) || (CAUSAL && j * kTileRows + kTileRows - 1 > w.q0 + coff);
      const int lim = need_mask ? (CAUSAL ? min(Nk, row + coff + 1) : Nk) - j * kTileRows : kTileRows;
      const auto s_read = [&] {
        tc_fence_before();
        mbar_arrive(bars.s_used());  // S_{i+1} may overwrite S
      };
      // PV_{i-1} reads P and adds into O: it must have completed before O is rescaled or P rewritten.
      const auto pv_finished = [&] {
        if (i > 0 && !mbar_wait_warp(bars.pv_done(), (i - 1) & 1, wc)) ok = false;
        tc_fence_after();
      };
      if (need_mask)
        softmax_tile_to<D, true, BF16>(tS, tP, tO, lim, c_log2, i == 0, m, l, s_read, pv_finished, pv_finished);
      else
        softmax_tile_to<D, false, BF16>(tS, tP, tO, lim, c_log2, i == 0, m, l, s_read, pv_finished, pv_finished);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bars.p_full());
      if (!ok) break;
    }
    if (ok && n > 0) ok = mbar_wait_warp(bars.o_full(), 0, wc);
    if (ok) tc_fence_after();
    epilogue(ok, m, l, r, tO, sQ, abort_flag);
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace tile
}  // namespace exattn
