// k_validate.cu -- device validation of selected-index rows.
//
// Semantics: IndexShare (onnx-runtime-ep-cuda src/kernels/index_share.rs),
// `validate_indices` (host) and `validate_index_rows` (device latch).  Each
// row is scanned left to right; -1 is padding; any other value is checked for
// being below -1, after padding, >= bound, equal to / smaller than its
// predecessor, in that order; the first failing column decides the code; a
// row of only -1 is "all padding".
//
// GB300 mapping: one warp per row.  A chunk of 32*E columns sits in
// registers (lane l owns E consecutive columns, loaded with 16-byte vector
// loads when aligned), so every load of a row up to 32*E columns is in flight
// at once.  The left-to-right scan becomes: a per-lane sequential scan of its
// E columns given (a) whether any earlier lane saw a -1 (ballot prefix) and
// (b) the previous lane's last value (shuffle); the row's first failing
// column is the warp-wide minimum.  Codes are bit-identical to the
// definition.
#include "common.cuh"
#include "kernels.h"

namespace sa {

template <int E>
__global__ void __launch_bounds__(256) validate_rows_kernel(ValidateArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= a.rows) return;
  const int64_t K = a.K;
  const int64_t b = row / a.rows_per_batch;
  const int64_t bound = a.bound_per_batch ? a.bound_per_batch[b] : a.bound;
  const int64_t base = row * K;

  bool pad_seen = false;   // a -1 appeared in an earlier chunk
  bool any_kept = false;   // a non -1 value appeared (row not all padding)
  int64_t prev_last = 0;   // value of the column just before this chunk
  int code = 0;

  for (int64_t c0 = 0; c0 < K; c0 += 32 * E) {
    const int64_t lc0 = c0 + static_cast<int64_t>(lane) * E;
    int64_t v[E];
    const bool full = lc0 + E <= K;
    if (full && a.vec_ok) {
      if (a.is_i64) {
        const int4* p = reinterpret_cast<const int4*>(static_cast<const int64_t*>(a.idx) + base + lc0);
#pragma unroll
        for (int e = 0; e < E / 2; ++e) {
          int4 w = __ldg(p + e);
          v[2 * e] = (static_cast<int64_t>(static_cast<uint32_t>(w.y)) << 32) |
                     static_cast<uint32_t>(w.x);
          v[2 * e + 1] = (static_cast<int64_t>(static_cast<uint32_t>(w.w)) << 32) |
                         static_cast<uint32_t>(w.z);
        }
      } else {
        const int4* p = reinterpret_cast<const int4*>(static_cast<const int32_t*>(a.idx) + base + lc0);
#pragma unroll
        for (int e = 0; e < E / 4; ++e) {
          int4 w = __ldg(p + e);
          v[4 * e] = w.x;
          v[4 * e + 1] = w.y;
          v[4 * e + 2] = w.z;
          v[4 * e + 3] = w.w;
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        v[e] = (lc0 + e < K) ? load_index(a.idx, base + lc0 + e, a.is_i64) : -1;
      }
    }
    int n_here = 0;  // columns this lane owns in this chunk
    if (lc0 < K) n_here = static_cast<int>(K - lc0 < E ? K - lc0 : E);
    bool has_pad = false, has_kept = false;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (e < n_here) {
        has_pad |= (v[e] == -1);
        has_kept |= (v[e] != -1);
      }
    }
    const uint32_t pad_mask = __ballot_sync(0xffffffffu, has_pad);
    const uint32_t kept_mask = __ballot_sync(0xffffffffu, has_kept);
    // Value of the column before this lane's first column.
    int64_t before = __shfl_up_sync(0xffffffffu, v[E - 1], 1);
    if (lane == 0) before = prev_last;
    const bool have_before = (lc0 > 0);
    bool p = pad_seen || (pad_mask & ((1u << lane) - 1u)) != 0;

    int my_code = 0;
    int64_t my_col = INT64_MAX;
    int64_t pv = before;
    bool have_pv = have_before;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (e < n_here && my_code == 0) {
        const int64_t x = v[e];
        if (x == -1) {
          p = true;
        } else {
          int c = 0;
          if (x < -1) c = SA_IDX_BELOW_SENTINEL;
          else if (p) c = SA_IDX_AFTER_PADDING;
          else if (x >= bound) c = SA_IDX_OUT_OF_RANGE;
          else if (have_pv && x == pv) c = SA_IDX_DUPLICATE;
          else if (have_pv && x < pv) c = SA_IDX_NOT_INCREASING;
          if (c) {
            my_code = c;
            my_col = lc0 + e;
          }
          pv = x;
          have_pv = true;
        }
      }
    }
    // First failing column across the warp.
    const uint32_t fail_mask = __ballot_sync(0xffffffffu, my_code != 0);
    if (fail_mask) {
      const int first = __ffs(fail_mask) - 1;  // lanes own increasing columns
      code = __shfl_sync(0xffffffffu, my_code, first);
      break;
    }
    pad_seen = pad_seen || pad_mask != 0;
    any_kept = any_kept || kept_mask != 0;
    prev_last = __shfl_sync(0xffffffffu, v[E - 1], 31);
  }
  if (code == 0 && !any_kept) code = SA_IDX_ALL_PADDING;
  if (lane == 0) {
    if (a.row_status) a.row_status[row] = static_cast<uint8_t>(code);
    if (code && a.err_word) atomicOr(a.err_word, static_cast<uint32_t>(code));
  }
}

int launch_validate(const ValidateArgs& a, cudaStream_t st) {
  if (a.rows == 0) return 0;
  const int warps = 8;
  const unsigned grid = static_cast<unsigned>((a.rows + warps - 1) / warps);
  if (a.K <= 32 * 4) {
    validate_rows_kernel<4><<<grid, 32 * warps, 0, st>>>(a);
  } else if (a.K <= 32 * 16) {
    validate_rows_kernel<16><<<grid, 32 * warps, 0, st>>>(a);
  } else if (a.is_i64 || a.K <= 32 * 32) {
    validate_rows_kernel<32><<<grid, 32 * warps, 0, st>>>(a);
  } else {
    validate_rows_kernel<64><<<grid, 32 * warps, 0, st>>>(a);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace sa
