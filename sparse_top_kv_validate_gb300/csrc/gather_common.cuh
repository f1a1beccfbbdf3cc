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

__device__ __forceinline__ UnitInfo unit_info(const GatherArgs& a, int64_t unit) {
  UnitInfo u;
  u.i = unit % a.Sq;
  const int64_t r = unit / a.Sq;
  const int64_t grp = r % a.n_groups;
  u.b = r / a.n_groups;
  if (a.n_groups == a.Hkv) {
    u.kvh = grp;
    u.h0 = grp * a.g;
  } else {
    u.kvh = grp / a.g;
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
