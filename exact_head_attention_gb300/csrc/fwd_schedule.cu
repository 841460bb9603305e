// Host-side packing of causal forward query blocks onto one CTA per SM (see fwd_schedule.h).
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "fwd_schedule.h"
#include "kernels.h"

namespace exattn {
namespace {

constexpr int kUnitFixedCost = 2;     // a block's start and epilogue, in key-tile visits
constexpr int kPersistBlockCost = 2;  // extra per block on a list: the CTA-wide hand-over between blocks

// Longest first onto the least loaded CTA, then moves and swaps that shorten the most loaded CTA.  A
// block's cost is the key tiles its two query tiles visit plus its fixed part.  Returns false (ctas = 0)
// where the lists would not beat the launch order: a list mixes heads and positions, so concurrent
// blocks share fewer K/V tiles in L2 than in launch order, and each listed block costs
// kPersistBlockCost more; lists are used only where, with that, they still shorten the most loaded SM
// by 3 % against longest-first.  Measured: the 8k workload's forward 160 -> 154 us packed; 32k ones,
// already balanced within 2 %, 4-8 % slower packed; 1k blocks (a few key tiles each) 4 % slower.
bool pack(int bh, int nqb, int Nk, int causal_off, int ctas, FwdSchedule* out) {
  const int nkv = (Nk + kTileRows - 1) / kTileRows;
  auto tiles = [&](int qb, int t) {
    const int last_key = qb * kFwdSubTiles * kTileRows + t * kTileRows + kTileRows - 1 + causal_off;
    return last_key < 0 ? 0 : std::min(nkv, last_key / kTileRows + 1);
  };
  std::vector<int> qcost(nqb);
  for (int qb = 0; qb < nqb; ++qb) qcost[qb] = tiles(qb, 0) + tiles(qb, 1) + kUnitFixedCost;
  const uint32_t units = static_cast<uint32_t>(bh) * nqb;
  std::vector<uint32_t> order(units);
  for (uint32_t u = 0; u < units; ++u) order[u] = u;
  auto cost = [&](uint32_t u) { return qcost[u % nqb]; };
  std::stable_sort(order.begin(), order.end(), [&](uint32_t x, uint32_t y) { return cost(x) > cost(y); });
  std::vector<std::vector<uint32_t>> bins(ctas);
  std::vector<long long> load(ctas, 0);
  for (uint32_t u : order) {
    const int b = static_cast<int>(std::min_element(load.begin(), load.end()) - load.begin());
    bins[b].push_back(u);
    load[b] += cost(u);
  }
  const long long lpt_max = *std::max_element(load.begin(), load.end());  // about what launch order gets
  for (int round = 0; round < 4 * ctas; ++round) {
    const int hi = static_cast<int>(std::max_element(load.begin(), load.end()) - load.begin());
    bool improved = false;
    for (int lo = 0; lo < ctas && !improved; ++lo) {
      if (lo == hi) continue;
      for (size_t i = 0; i < bins[hi].size() && !improved; ++i) {
        const int ca = cost(bins[hi][i]);
        if (std::max(load[hi] - ca, load[lo] + ca) < load[hi]) {  // move
          bins[lo].push_back(bins[hi][i]);
          bins[hi].erase(bins[hi].begin() + static_cast<long>(i));
          load[hi] -= ca;
          load[lo] += ca;
          improved = true;
          break;
        }
        for (size_t j = 0; j < bins[lo].size(); ++j) {  // swap for a lighter block
          const int cb = cost(bins[lo][j]);
          if (cb >= ca) continue;
          if (std::max(load[hi] - ca + cb, load[lo] - cb + ca) < load[hi]) {
            std::swap(bins[hi][i], bins[lo][j]);
            load[hi] += cb - ca;
            load[lo] += ca - cb;
            improved = true;
            break;
          }
        }
      }
    }
    if (!improved) break;
  }
  long long packed_max = 0;
  for (int b = 0; b < ctas; ++b)
    packed_max = std::max(packed_max, load[b] + kPersistBlockCost * static_cast<long long>(bins[b].size()));
  out->ctas = 0;
  if (100 * packed_max > 97 * lpt_max) return false;
  int pos = 0;
  for (int b = 0; b < ctas; ++b) {
    std::sort(bins[b].begin(), bins[b].end(), [&](uint32_t x, uint32_t y) { return cost(x) > cost(y); });
    out->begin[b] = static_cast<uint16_t>(pos);
    for (uint32_t u : bins[b]) out->unit[pos++] = u;
  }
  out->begin[ctas] = static_cast<uint16_t>(pos);
  out->ctas = ctas;
  return true;
}

}  // namespace

const FwdSchedule* persistent_schedule(int bh, int nqb, int Nq, int Nk, int causal_off, int sm_count) {
  const long long units = static_cast<long long>(bh) * nqb;
  const int ctas = std::min(sm_count, kPersistMaxCtas);
  if (ctas <= 0 || units <= ctas || units > kPersistMaxUnits) return nullptr;
  using Key = std::tuple<int, int, int, int, int, int>;
  static std::mutex mu;
  static std::map<Key, FwdSchedule> cache;
  const Key key{bh, nqb, Nq, Nk, causal_off, ctas};
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it == cache.end()) {
    if (cache.size() >= 64) cache.clear();
    it = cache.emplace(key, FwdSchedule{}).first;
    pack(bh, nqb, Nk, causal_off, ctas, &it->second);
  }
  if (it->second.ctas == 0) return nullptr;
  // A copy per thread: another thread may clear the cache as soon as the lock is released.
  thread_local FwdSchedule copy;
  copy = it->second;
  return &copy;
}

}  // namespace exattn
