// Packed lists of forward query blocks for the persistent causal launch (host side; the list is passed
// to the kernel as a grid-constant argument).
//
// Under a causal mask a 256-row query block's work grows with its position, from one key tile to the
// whole row.  With one CTA per block the hardware hands blocks to SMs heaviest first (the launch
// order), which for few, coarse blocks leaves part of the SMs' time idle at the end: a tenth of it on
// 12 heads of 32 blocks over 152 SMs.  The persistent launch runs one CTA per SM over a list of blocks
// that the host packs.
#pragma once

#include <cstdint>

namespace exattn {

constexpr int kPersistMaxCtas = 160;
constexpr int kPersistMaxUnits = 2048;

struct FwdSchedule {
  int ctas;                             // 0: the launch order is used
  uint16_t begin[kPersistMaxCtas + 1];  // CTA i runs unit[begin[i] .. begin[i + 1])
  uint32_t unit[kPersistMaxUnits];      // a query block: bh * nqb + qb
};

// The packed lists for a causal forward of bh heads of nqb 256-row blocks (causal_off as in FwdArgs),
// or nullptr when the launch order is used: one wave or less, more blocks than a list holds, or a
// packing that does not beat the launch order clearly.  Cached per shape; the pointer is to this
// thread's copy and stays valid until the thread's next call.
const FwdSchedule* persistent_schedule(int bh, int nqb, int Nq, int Nk, int causal_off, int sm_count);

}  // namespace exattn
