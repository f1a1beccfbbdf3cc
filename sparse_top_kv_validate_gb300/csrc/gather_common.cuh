// gather_common.cuh -- work-unit geometry shared by the gather kernels.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace sa {

// A work unit is (batch, group, query position): the group is a KV head
// (serving its whole GQA group of query heads) or, when every query head has
// its own index row, a single query head.
struct UnitInfo {
  int64_t b, i, kvh, h0, ih;
};

// Unit counts stay below 2^31 (checked on the host), so 32-bit division.
__device__ __forceinline__ UnitInfo unit_info(const GatherArgs& a, int64_t unit) {
  UnitInfo u;
  const uint32_t un = static_cast<uint32_t>(unit);
  const uint32_t sq = static_cast<uint32_t>(a.Sq), ng = static_cast<uint32_t>(a.n_groups);
  const uint32_t r = un / sq;
  u.i = un - r * sq;
  const uint32_t bb = r / ng;
  const uint32_t grp = r - bb * ng;
  u.b = bb;
  if (a.n_groups == a.Hkv) {
    u.kvh = grp;
    u.h0 = static_cast<int64_t>(grp) * a.g;
  } else {
    u.kvh = grp / static_cast<uint32_t>(a.g);
    u.h0 = grp;
  }
  u.ih = (a.I == 1) ? 0 : (a.I == a.Hkv ? u.kvh : u.h0);
  return u;
}

// Per-batch write position of the fused current-token append.
__device__ __forceinline__ int64_t write_pos_of(const GatherArgs& a, int64_t b) {
  return a.write_pos ? a.write_pos[b] : a.T - a.C;
}

}  // namespace sa
