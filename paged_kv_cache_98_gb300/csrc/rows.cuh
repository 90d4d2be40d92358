// Row -> (sequence, number of visible keys) for the attention kernels.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace pkv {

// A decode row is a sequence and sees its whole context.  A prefill row is
// query i of sequence s, at absolute position context_lens[s] - q_len + i,
// and sees keys 0..that position ("第32讲 … Prefill vs Decode …", §5.4).
// Lengths beyond the block table or the launched partitions are clamped and
// flagged, so no access leaves the table.
__device__ __forceinline__ int row_keys(const AttnParams& p, int row, int* seq_out) {
  int s = row, keys;
  if (p.query_start_loc == nullptr) {
    keys = __ldg(p.context_lens + row);
  } else {
    int lo = 0, hi = p.num_seqs - 1;  // largest s with query_start_loc[s] <= row
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (__ldg(p.query_start_loc + mid) <= row) lo = mid; else hi = mid - 1;
    }
    s = lo;
    const int q0 = __ldg(p.query_start_loc + s);
    const int q_len = __ldg(p.query_start_loc + s + 1) - q0;
    keys = __ldg(p.context_lens + s) - q_len + (row - q0) + 1;
  }
  *seq_out = s;
  const int cap_table = p.max_blocks_per_seq * kBlockSize;
  const int cap_launch = p.max_parts * p.partition;
  int cap = cap_table < cap_launch ? cap_table : cap_launch;
  if (keys < 0 || keys > cap) {
    if (threadIdx.x == 0) flag_error(p.errors, PKV_DEVERR_CONTEXT);
    keys = keys < 0 ? 0 : cap;
  }
  return keys;
}

// Cascade decode: first key of sequence s's own part (its shared prefix), for a
// context of `keys` tokens.  The prefix must be whole blocks within the
// context; otherwise it is cut back to one and the error flagged.
__device__ __forceinline__ int cascade_prefix(const AttnParams& p, int s, int keys, bool report) {
  if (p.prefix_lens == nullptr) return 0;
  int pre = __ldg(p.prefix_lens + s);
  if (pre < 0 || pre > keys || (pre & (kBlockSize - 1)) != 0) {
    if (report) flag_error(p.errors, PKV_DEVERR_CONTEXT);
    pre = pre < 0 ? 0 : (pre > keys ? keys : pre);
    pre &= ~(kBlockSize - 1);
  }
  return pre;
}

// Partial slots of the shared-prefix pass that precede sequence s's own: two
// per chunk of the prefix (its even and its odd key tiles).
__device__ __forceinline__ int cascade_slots(const AttnParams& p, int prefix) {
  return p.prefix_chunk > 0 ? 2 * ((prefix + p.prefix_chunk - 1) / p.prefix_chunk) : 0;
}

}  // namespace pkv
