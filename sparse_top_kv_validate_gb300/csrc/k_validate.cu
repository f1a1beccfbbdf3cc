// k_validate.cu -- device validation of selected-index rows.
//
// Semantics: IndexShare (onnx-runtime-ep-cuda src/kernels/index_share.rs),
// `validate_indices` (host) and `validate_index_rows` (device latch).  Each
// row is scanned left to right; -1 is padding; any other value is checked for
// being below -1, after padding, >= bound, equal to / smaller than its
// predecessor, in that order; the first failing column decides the code; a
// row of only -1 is "all padding".
//
// GB300 mapping: the left-to-right scan is evaluated in its exact per-column
// form.  Assuming every earlier column passed, column j fails iff:
//   v < -1                          -> below sentinel
//   j > 0 and v[j-1] == -1          -> after padding
//   v >= bound                      -> out of range
//   j > 0 and v == v[j-1] / v < v[j-1] -> duplicate / not increasing
// (a -1 passes).  The row's status is the code of the smallest failing
// column, and "all padding" when no column fails and v[0] == -1.  Columns are
// therefore independent: one warp per row loads its columns with 16-byte
// vector loads, all in flight at once, and a warp max-reduction of the key
// ~(column << 8 | code) picks the first failure.  Bit-identical codes.
#include "common.cuh"
#include "kernels.h"

namespace sa {

__device__ __forceinline__ int column_rule(int64_t v, int64_t prev, int64_t col, int64_t bound) {
  if (v == -1) return 0;
  if (v < -1) return SA_IDX_BELOW_SENTINEL;
  if (col > 0 && prev == -1) return SA_IDX_AFTER_PADDING;
  if (v >= bound) return SA_IDX_OUT_OF_RANGE;
  if (col > 0 && v == prev) return SA_IDX_DUPLICATE;
  if (col > 0 && v < prev) return SA_IDX_NOT_INCREASING;
  return 0;
}

// E consecutive columns per lane per step; 32*E columns per warp step.
template <int E>
__global__ void __launch_bounds__(256) validate_rows_kernel(ValidateArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= a.rows) return;
  const int64_t K = a.K;
  const int64_t b = row / a.rows_per_batch;
  const int64_t bound = a.bound_per_batch ? a.bound_per_batch[b] : a.bound;
  const int64_t base = row * K;
  unsigned long long best = 0;  // max of ~key over failing columns (0 = none)

#pragma unroll 2
  for (int64_t c0 = static_cast<int64_t>(lane) * E; c0 < K; c0 += 32 * E) {
    int64_t v[E];
    if (c0 + E <= K && a.vec_ok) {
      if (a.is_i64) {
        const int4* p = reinterpret_cast<const int4*>(static_cast<const int64_t*>(a.idx) + base + c0);
#pragma unroll
        for (int e = 0; e < E / 2; ++e) {
          const int4 w = __ldg(p + e);
          v[2 * e] = static_cast<int64_t>((static_cast<uint64_t>(static_cast<uint32_t>(w.y)) << 32) |
                                          static_cast<uint32_t>(w.x));
          v[2 * e + 1] = static_cast<int64_t>(
              (static_cast<uint64_t>(static_cast<uint32_t>(w.w)) << 32) | static_cast<uint32_t>(w.z));
        }
      } else {
        const int4* p = reinterpret_cast<const int4*>(static_cast<const int32_t*>(a.idx) + base + c0);
#pragma unroll
        for (int e = 0; e < E / 4; ++e) {
          const int4 w = __ldg(p + e);
          v[4 * e] = w.x;
          v[4 * e + 1] = w.y;
          v[4 * e + 2] = w.z;
          v[4 * e + 3] = w.w;
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = (c0 + e < K) ? load_index(a.idx, base + c0 + e, a.is_i64) : -1;
    }
    const int64_t before = c0 > 0 ? load_index(a.idx, base + c0 - 1, a.is_i64) : 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int64_t col = c0 + e;
      if (col < K) {
        const int code = column_rule(v[e], e == 0 ? before : v[e - 1], col, bound);
        if (code) {
          const unsigned long long k = ~((static_cast<unsigned long long>(col) << 8) |
                                         static_cast<unsigned long long>(code));
          best = best > k ? best : k;
        }
      }
    }
  }
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, sh);
    best = best > o ? best : o;
  }
  if (lane == 0) {
    int code = best ? static_cast<int>((~best) & 0xff) : 0;
    if (code == 0 && load_index(a.idx, base, a.is_i64) == -1) code = SA_IDX_ALL_PADDING;
    if (a.row_status) a.row_status[row] = static_cast<uint8_t>(code);
    if (code && a.err_word) atomicOr(a.err_word, static_cast<uint32_t>(code));
  }
}

int launch_validate(const ValidateArgs& a, cudaStream_t st) {
  if (a.rows == 0) return 0;
  const int warps = 8;
  const unsigned grid = static_cast<unsigned>((a.rows + warps - 1) / warps);
  if (a.K <= 32 * 4 || a.is_i64) validate_rows_kernel<4><<<grid, 32 * warps, 0, st>>>(a);
  else validate_rows_kernel<8><<<grid, 32 * warps, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace sa
