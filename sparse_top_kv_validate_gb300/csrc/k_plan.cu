// k_plan.cu -- per index row: validation, candidate cache positions, and the
// current-token append, ahead of the streaming gather kernel.
//
// Semantics: IndexShare (onnx-runtime-ep-cuda src/kernels/index_share.rs):
// `validate_indices` / `validate_index_rows` (row rules, first failing column
// decides), `build_present` (present = past ++ current, here the in-place
// append of the current token), and the candidate set of `index_share_row`
// (the valid prefix of a row's selected indices); the dense window of recent
// tokens united with the selected ones as in the compressed sparse attention
// pages (`csa_ratio128_sink_attention`).
//
// GB300 mapping: one 256-thread block per index row (b, ih, i).  Every column
// is checked in its exact per-column form (a column's rule depends only on its
// value and its left neighbour's; the first failing column wins through a
// block max of ~(column << 8 | code)), so the row needs no sequential scan.
// The same pass writes pos[row][c], the cache position of candidate c
// (window positions first, then selected indices) or -1 when masked, padded
// with -1 to whole 16-candidate tiles -- the only thing the gather kernel
// reads per candidate.  Extra blocks copy the current token(s) into the cache.
#include "common.cuh"
#include "kernels.h"

namespace sa {

__device__ __forceinline__ int plan_column_code(int64_t v, int64_t prev, int64_t col,
                                                int64_t bound) {
  if (v == -1) return col == 0 ? SA_IDX_ALL_PADDING : 0;
  if (v < -1) return SA_IDX_BELOW_SENTINEL;
  if (col > 0 && prev == -1) return SA_IDX_AFTER_PADDING;
  if (v >= bound) return SA_IDX_OUT_OF_RANGE;
  if (col > 0 && v == prev) return SA_IDX_DUPLICATE;
  if (col > 0 && v < prev) return SA_IDX_NOT_INCREASING;
  return 0;
}

__global__ void __launch_bounds__(256) plan_rows_kernel(PlanArgs a) {
  pdl_launch_dependents();  // the gather kernel may start its set-up now
  const int64_t irows = a.plan_rows ? a.B * a.I * a.Sq : 0;
  if (static_cast<int64_t>(blockIdx.x) >= irows) {
    // ---- append blocks: cur [B, Hkv, C, D] -> cache rows write_pos[b] + c --------
    const int64_t blk = blockIdx.x - irows;
    const int64_t row_bytes = a.D * a.esz;
    const int64_t n16 = a.B * a.Hkv * a.C * (row_bytes / 16);
    for (int64_t e = blk * blockDim.x + threadIdx.x; e < n16;
         e += static_cast<int64_t>(a.append_blocks) * blockDim.x) {
      const int64_t per_row = row_bytes / 16;
      const int64_t r = e / per_row, cc = e % per_row;   // r = (b*Hkv + h)*C + c
      const int64_t b = r / (a.Hkv * a.C);
      const int64_t wp = a.write_pos ? a.write_pos[b] : a.T - a.C;
      if (wp < 0 || wp + a.C > a.T) {
        if (cc == 0 && a.err_word) atomicOr(a.err_word, SA_ERRBIT_WRITE_POS);
        continue;
      }
      const int64_t bh = r / a.C, c = r % a.C;
      const int64_t dst = (bh * a.T + wp + c) * row_bytes + cc * 16;
      const int64_t src = r * row_bytes + cc * 16;
      *reinterpret_cast<int4*>(static_cast<char*>(a.k_cache) + dst) =
          __ldg(reinterpret_cast<const int4*>(static_cast<const char*>(a.k_cur) + src));
      *reinterpret_cast<int4*>(static_cast<char*>(a.v_cache) + dst) =
          __ldg(reinterpret_cast<const int4*>(static_cast<const char*>(a.v_cur) + src));
    }
    return;
  }
  // ---- index-row blocks ------------------------------------------------------------
  const int64_t irow = blockIdx.x;
  const int64_t i = irow % a.Sq;
  const int64_t b = irow / (a.I * a.Sq);
  const CandRule rule = cand_rule(a.kv_len, b, a.T, a.window, a.causal, a.past_len, i);
  const int64_t len = rule.len;
  int32_t* pos = a.pos + irow * a.n_cand_pad;
  const int64_t ncand = a.window + a.K;

  if (a.write_positions) {
    // window candidates
    for (int64_t c = threadIdx.x; c < a.window; c += blockDim.x) pos[c] = window_pos(rule, c);
    // padding of the last tile
    for (int64_t c = ncand + threadIdx.x; c < a.n_cand_pad; c += blockDim.x) pos[c] = -1;
  }

  // selected columns: 8 consecutive per thread per step, every load of the
  // step issued before any is used
  const int64_t base = irow * a.K;
  unsigned long long best = 0;  // max over failing columns of ~(col << 8 | code)
  for (int64_t c0 = static_cast<int64_t>(threadIdx.x) * 8; c0 < a.K; c0 += blockDim.x * 8) {
    int64_t v[8];
    if (c0 + 8 <= a.K && a.vec_ok) {
      if (a.idx_is_i64) {
        const int4* p = reinterpret_cast<const int4*>(static_cast<const int64_t*>(a.idx) + base + c0);
        int4 w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) w[q] = __ldg(p + q);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          v[2 * q] = static_cast<int64_t>((static_cast<uint64_t>(static_cast<uint32_t>(w[q].y)) << 32) |
                                          static_cast<uint32_t>(w[q].x));
          v[2 * q + 1] = static_cast<int64_t>(
              (static_cast<uint64_t>(static_cast<uint32_t>(w[q].w)) << 32) | static_cast<uint32_t>(w[q].z));
        }
      } else {
        const int4* p = reinterpret_cast<const int4*>(static_cast<const int32_t*>(a.idx) + base + c0);
        const int4 w0 = __ldg(p), w1 = __ldg(p + 1);
        v[0] = w0.x; v[1] = w0.y; v[2] = w0.z; v[3] = w0.w;
        v[4] = w1.x; v[5] = w1.y; v[6] = w1.z; v[7] = w1.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = (c0 + e < a.K) ? load_index(a.idx, base + c0 + e, a.idx_is_i64) : -1;
    }
    const int64_t before = c0 > 0 ? load_index(a.idx, base + c0 - 1, a.idx_is_i64) : 0;
    int32_t out[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int64_t col = c0 + e;
      const int64_t t = v[e];
      if (a.validate && col < a.K) {
        const int code = plan_column_code(t, e == 0 ? before : v[e - 1], col, len);
        if (code) {
          const unsigned long long key =
              ~((static_cast<unsigned long long>(code == SA_IDX_ALL_PADDING ? a.K : col) << 8) |
                static_cast<unsigned long long>(code));
          best = best > key ? best : key;
        }
      }
      out[e] = selected_pos(rule, t);
    }
    if (!a.write_positions) continue;
    int32_t* dst = pos + a.window + c0;
    if (c0 + 8 <= a.K && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0)) {
      reinterpret_cast<int4*>(dst)[0] = make_int4(out[0], out[1], out[2], out[3]);
      reinterpret_cast<int4*>(dst)[1] = make_int4(out[4], out[5], out[6], out[7]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (c0 + e < a.K) dst[e] = out[e];
    }
  }
  if (!a.validate) return;
  // block max of the failure keys
  __shared__ unsigned long long red[8];
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, sh);
    best = best > o ? best : o;
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long m = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) m = m > red[w] ? m : red[w];
    const int code = m ? static_cast<int>((~m) & 0xff) : 0;
    if (a.row_status) a.row_status[irow] = static_cast<uint8_t>(code);
    if (code && a.err_word) atomicOr(a.err_word, static_cast<uint32_t>(code));
  }
}

int launch_plan(const PlanArgs& a, cudaStream_t st) {
  const int64_t irows = a.plan_rows ? a.B * a.I * a.Sq : 0;
  const int64_t blocks = irows + a.append_blocks;
  if (blocks == 0) return 0;
  plan_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace sa
