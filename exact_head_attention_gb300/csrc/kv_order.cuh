// Launch order of the key/value-block kernels (attention backward, attention-KL backward).
//
// One CTA per (head, 128-row key block).  Blocks are numbered along grid.x in groups of `head_group`
// heads, the last group also taking the B*H mod head_group heads left over; within a group the heads go
// fastest.  Heads fastest puts the heavy low key blocks of a causal mask first, so the light ones fill
// the group's last wave (a short last group would start its heavy blocks with too few light ones to
// run beside them, hence no group below head_group heads).  Small groups keep the key blocks that add
// into one head's dQ accumulator rows close together in time, so those rows are still in L2 when the
// next block adds into them.  head_group = B*H is the plain heads-fastest order; head_group = 1 runs
// each head's key blocks consecutively.  The host picks the group (api.cu).
#pragma once

namespace exattn {

struct KvBlock {
  int bh;  // flattened batch * heads + head
  int jb;  // key block
};

__device__ __forceinline__ KvBlock kv_block(int block, int bh_count, int head_group, int nkb) {
  const int groups = max(1, bh_count / head_group);
  const int per_group = head_group * nkb;  // fits an int: the host limits B*H*nkb to 2^31 - 1
  const int group = min(block / per_group, groups - 1);
  const int r = block - group * per_group;
  const int heads = group == groups - 1 ? bh_count - group * head_group : head_group;
  const int jb = r / heads;
  return {group * head_group + (r - jb * heads), jb};
}

}  // namespace exattn
