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

// The additive term of logical element (b, h, i, j): an IndexShare bias or an
// ONNX attention mask (bool: 0 where set, -inf where clear; a key at or past
// a short key axis: -inf).
__device__ __forceinline__ float bias_term(const GatherArgs& a, int64_t b, int64_t h, int64_t i,
                                           int64_t j) {
  if (a.bias_key_extent > 0 && j >= a.bias_key_extent) return SA_NEG_INF;
  const int64_t off = b * a.bias_sb + h * a.bias_sh + i * a.bias_si + j * a.bias_sk;
  switch (a.bias_kind) {
    case kBiasF16: return __half2float(__ldg(static_cast<const __half*>(a.bias) + off));
    case kBiasBF16:
      return __bfloat162float(__ldg(static_cast<const __nv_bfloat16*>(a.bias) + off));
    case kBiasBool: return __ldg(static_cast<const uint8_t*>(a.bias) + off) ? 0.0f : SA_NEG_INF;
    default: return __ldg(static_cast<const float*>(a.bias) + off);
  }
}

// Dense source: whether key c of query i of batch b is visible (causal frontier,
// shifted by the padding frontier nonpad[b] - Sq when given; the frontier itself).
__device__ __forceinline__ bool dense_visible(const GatherArgs& a, int64_t b, int64_t i,
                                              int64_t c) {
  int64_t off = a.past_len;
  if (a.dense_nonpad) {
    const int64_t np = __ldg(a.dense_nonpad + b);
    if (np >= 0 && c >= np) return false;
    off = np - a.Sq;
  }
  return !(a.causal && c > off + i);
}

// Per-batch write position of the fused current-token append.
__device__ __forceinline__ int64_t write_pos_of(const GatherArgs& a, int64_t b) {
  return a.write_pos ? a.write_pos[b] : a.T - a.C;
}

}  // namespace sa
