// k_decode.cu -- split-K gather decode over a KV cache (selected tokens or
// a page table), and the fixed-order combine of the split partials.
//
// Semantics: IndexShare `index_share_row` (onnx-runtime-ep-cuda
// src/kernels/index_share.rs) -- gather the valid prefix of a row's selected
// indices, scaled QK scores, a stable fp32 softmax in which a fully-masked row
// gives 0, probs . V; ONNX Attention `attention_split` / `attention_combine`
// (standard_attention.rs) -- FlashDecoding: each split of the keys yields
// (max, sum, unnormalised P.V) and a log-sum-exp combine merges the splits in
// a fixed order; paged addressing as in ferrum-kernels causal_attention.rs
// (16-token blocks through a table).
//
// What this file holds (the tensor-core gather is gather_stream_kernel in
// k_stream.cu):
//  * unit / candidate resolution shared by the gather kernels: a work unit is
//    (batch, KV head or index head, query) serving every query head that
//    shares its index row and KV head; resolve_candidate maps a candidate to a
//    cache row (index row, window, masks, page table) or -1, never out of
//    bounds.
//  * gather_simt_kernel: the general path for fp32 storage and the shapes the
//    tensor-core kernel does not take.  One CTA per (unit, head, split of
//    `chunk` candidates); warps stride over the candidates, each lane holding
//    DPL dims (d = lane + 32 k), a few candidates' rows loaded at once; fp32
//    FMA and an online softmax; the bias and mask terms of gather_common.cuh.
//    Warps merge in shared memory in warp order.
//  * combine_kernel and combine_flat_kernel: the fixed-order log-sum-exp merge
//    of split partials (max, sum, unnormalised P.V), with the sink logit in
//    the denominator; combine_flat_kernel is one thread per four output dims
//    with every split's partials loaded at once (the FP8 paths).
//  * paged_append_kernel: writes the new token into its page before a paged
//    decode.
// Results are deterministic run to run (fixed warp and split order).
#include "gather_common.cuh"

namespace sa {

// ---------------------------------------------------------------------------
// unit / candidate resolution (shared by the tensor-core and SIMT kernels)
// ---------------------------------------------------------------------------

// Number of candidates of this unit (the per-batch context for paged units).
__device__ __forceinline__ int64_t unit_candidates(const GatherArgs& a, const UnitInfo& u) {
  if (a.source == kPaged) {
    int64_t ctx = a.ctx_len[u.b];
    const int64_t cap = a.max_pages * a.page_tokens;
    if (ctx < 1 || ctx > cap) return 0;
    return ctx;
  }
  return a.n_cand;
}

// Candidate c of the unit -> cache row id (row of D elements in k/v), or -1
// when the candidate is masked or absent.  Never returns an out-of-bounds row.
__device__ __forceinline__ int32_t resolve_candidate(const GatherArgs& a, const UnitInfo& u,
                                                     int64_t c) {
  if (a.source == kPaged) {
    const int64_t ctx = a.ctx_len[u.b];
    if (c >= ctx) return -1;
    const int32_t page = a.block_table[u.b * a.max_pages + c / a.page_tokens];
    if (page < 0 || page >= a.num_pages) {
      if (a.err_word) atomicOr(a.err_word, SA_ERRBIT_PAGE);
      return -1;
    }
    return static_cast<int32_t>((static_cast<int64_t>(page) * a.Hkv + u.kvh) * a.page_tokens +
                                c % a.page_tokens);
  }
  if (a.source == kDense) {
    if (!dense_visible(a, u.b, u.i, c)) return -1;
    return static_cast<int32_t>((u.b * a.Hkv + u.kvh) * a.T + c);
  }
  int64_t len = a.kv_len ? a.kv_len[u.b] : a.T;
  if (len > a.T) len = a.T;
  const int64_t wstart = len - a.window;
  int64_t t;
  if (c < a.window) {
    t = wstart + c;
    if (t < 0) return -1;
  } else {
    const int64_t off = ((u.b * a.I + u.ih) * a.Sq + u.i) * a.K + (c - a.window);
    t = load_index(a.idx, off, a.idx_is_i64);
    if (t < 0 || t >= len) return -1;
    if (a.window > 0 && t >= wstart) return -1;  // already in the window
  }
  if (a.causal && t > a.past_len + u.i) return -1;
  return static_cast<int32_t>((u.b * a.Hkv + u.kvh) * a.T + t);
}

// ---------------------------------------------------------------------------
// SIMT gather kernel (fp32 storage, or shapes the tensor-core kernel skips)
// ---------------------------------------------------------------------------
// One CTA per (unit, head, split); warps stride over candidates; lanes hold
// DPL dims each (d = lane + 32 * k).  fp32 FMA throughout.

template <typename T, int DPL>
__global__ void __launch_bounds__(128) gather_simt_kernel(GatherArgs a) {
  __shared__ float sm_o[4][DPL * 32];
  __shared__ float sm_ml[4][2];
  const int64_t split = blockIdx.x % a.splits;
  const int64_t rest = blockIdx.x / a.splits;
  const int64_t hh = rest % a.hpu;
  const int64_t unit = rest / a.hpu;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const UnitInfo u = unit_info(a, unit);
  const int64_t h = u.h0 + hh;
  const int64_t D = a.D;
  const int64_t n_cand = unit_candidates(a, u);
  const int64_t c0 = split * a.chunk;
  int64_t c1 = c0 + a.chunk;
  if (c1 > n_cand) c1 = n_cand;

  const T* qp = static_cast<const T*>(a.q) + ((u.b * a.Hq + h) * a.Sq + u.i) * D;
  float q[DPL], o[DPL];
#pragma unroll
  for (int k = 0; k < DPL; ++k) {
    const int64_t d = lane + 32 * k;
    q[k] = d < D ? to_f32<T>(qp[d]) : 0.f;
    o[k] = 0.f;
  }
  float m = SA_NEG_INF, l = 0.f;
  const T* kp = static_cast<const T*>(a.k);
  const T* vp = static_cast<const T*>(a.v);
  const float sl2 = a.scale_log2;
  // Warp w takes candidates c0 + w, c0 + w + 4, ... in that order, kU at a
  // time: the kU rows are resolved and their K and V values loaded together
  // (independent loads in flight), then the online softmax takes them in turn.
  constexpr int kU = DPL <= 2 ? 4 : (DPL <= 4 ? 2 : 1);
  for (int64_t cb = c0 + warp; cb < c1; cb += 4 * kU) {
    int32_t rows[kU];
#pragma unroll
    for (int t = 0; t < kU; ++t) {
      const int64_t c = cb + 4 * t;
      rows[t] = c < c1 ? resolve_candidate(a, u, c) : -1;
    }
    float kv[kU][DPL], vv[kU][DPL];
#pragma unroll
    for (int t = 0; t < kU; ++t) {
      const T* kr = kp + static_cast<int64_t>(rows[t] < 0 ? 0 : rows[t]) * D;
      const T* vr = vp + static_cast<int64_t>(rows[t] < 0 ? 0 : rows[t]) * D;
#pragma unroll
      for (int k = 0; k < DPL; ++k) {
        const int64_t d = lane + 32 * k;
        const bool in = rows[t] >= 0 && d < D;
        kv[t][k] = in ? to_f32<T>(kr[d]) : 0.f;
        vv[t][k] = in ? to_f32<T>(vr[d]) : 0.f;
      }
    }
#pragma unroll
    for (int t = 0; t < kU; ++t) {
      const int32_t row = rows[t];
      if (row < 0) continue;
      float dot = 0.f;
#pragma unroll
      for (int k = 0; k < DPL; ++k) {
        const int64_t d = lane + 32 * k;
        if (d < D) dot = fmaf(q[k], kv[t][k], dot);
      }
#pragma unroll
      for (int sh = 16; sh > 0; sh >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, sh);
      float x;
      if (a.softcap != 0.f) x = a.softcap * tanhf(dot * (sl2 / kLog2e) * a.inv_softcap) * kLog2e;
      else x = dot * sl2;
      if (a.bias) {  // [IS] bias_at / [SA] mask_bias, keyed by the cache position
        const int64_t j = row - (u.b * a.Hkv + u.kvh) * a.T;
        x += kLog2e * bias_term(a, u.b, h, u.i, j);
        if (x == SA_NEG_INF) continue;  // a -inf term masks the key
      }
      const float mn = fmaxf(m, x);
      const float al = exp2f(m - mn);  // m == -inf -> 0
      const float p = exp2f(x - mn);
      l = l * al + p;
#pragma unroll
      for (int k = 0; k < DPL; ++k) {
        const int64_t d = lane + 32 * k;
        o[k] = o[k] * al + (d < D ? p * vv[t][k] : 0.f);
      }
      m = mn;
    }
  }
#pragma unroll
  for (int k = 0; k < DPL; ++k) sm_o[warp][lane + 32 * k] = o[k];
  if (lane == 0) {
    sm_ml[warp][0] = m;
    sm_ml[warp][1] = l;
  }
  __syncthreads();
  if (warp != 0) return;
  float M = SA_NEG_INF;
  for (int w = 0; w < 4; ++w) M = fmaxf(M, sm_ml[w][0]);
  float L = 0.f;
  float f[4];
  for (int w = 0; w < 4; ++w) {
    f[w] = (M == SA_NEG_INF) ? 0.f : exp2f(sm_ml[w][0] - M);
    L += sm_ml[w][1] * f[w];
  }
  for (int k = 0; k < DPL; ++k) {
    const int64_t d = lane + 32 * k;
    if (d >= D) continue;
    float acc = 0.f;
    for (int w = 0; w < 4; ++w) acc += sm_o[w][lane + 32 * k] * f[w];
    if (a.splits == 1) {
      float LL = L;
      if (a.sink && M != SA_NEG_INF) LL += exp2f(a.sink[h] * kLog2e - M);
      const float out = (M == SA_NEG_INF || LL == 0.f) ? 0.f : acc / LL;
      static_cast<T*>(a.y)[((u.b * a.Hq + h) * a.Sq + u.i) * D + d] = from_f32<T>(out);
    } else {
      const int64_t pidx = (unit * a.splits + split) * a.hpu + hh;
      a.part_o[pidx * D + d] = acc;
      if (d == 0) {
        a.part_ml[2 * pidx] = M;
        a.part_ml[2 * pidx + 1] = L;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// combine: y = sum_s o_s 2^(m_s - M) / (sum_s l_s 2^(m_s - M) [+ sink term])
// ---------------------------------------------------------------------------

constexpr int kCombineMaxSplits = 512;  // split weights kept in shared memory

template <typename T>
__global__ void __launch_bounds__(128) combine_kernel(GatherArgs a) {
  __shared__ float w_s[kCombineMaxSplits];
  __shared__ float inv_s;
  const int64_t hh = blockIdx.x % a.hpu;
  const int64_t unit = blockIdx.x / a.hpu;
  const UnitInfo u = unit_info(a, unit);
  const int64_t h = u.h0 + hh;
  const int64_t D = a.Dv;
  const int splits = static_cast<int>(a.splits);
  pdl_wait();  // the partials of the kernel before (launched as its dependent)
  const float* ml = a.part_ml + (unit * a.splits * a.hpu + hh) * 2;
  const int64_t mstride = a.hpu * 2;
  // Split weights w_s = 2^(m_s - M) (0 for an empty split) and 1 / L, by warp 0.
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float M = SA_NEG_INF;
    for (int s = lane; s < splits; s += 32) M = fmaxf(M, ml[s * mstride]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int s = lane; s < splits; s += 32) {
      const float ms = ml[s * mstride];
      const float w = (M == SA_NEG_INF || ms == SA_NEG_INF) ? 0.f : ex2(ms - M);
      if (s < kCombineMaxSplits) w_s[s] = w;
      L += ml[s * mstride + 1] * w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) {
      if (a.sink && M != SA_NEG_INF) L += ex2(a.sink[h] * kLog2e - M);
      inv_s = (M == SA_NEG_INF || L == 0.f) ? 0.f : 1.0f / L;
    }
  }
  __syncthreads();
  const float inv = inv_s;
  T* yp = static_cast<T*>(a.y) + ((u.b * a.Hq + h) * a.Sq + u.i) * D;
  const float* po = a.part_o + (unit * a.splits * a.hpu + hh) * D;
  const int64_t pstride = a.hpu * D;  // between splits
  if (splits <= kCombineMaxSplits && (D & 3) == 0) {
    for (int64_t d = 4 * threadIdx.x; d < D; d += 4 * blockDim.x) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = 0; s < splits; ++s) {
        const float w = w_s[s];
        if (w == 0.f) continue;
        const float4 v = *reinterpret_cast<const float4*>(po + s * pstride + d);
        acc.x = fmaf(v.x, w, acc.x);
        acc.y = fmaf(v.y, w, acc.y);
        acc.z = fmaf(v.z, w, acc.z);
        acc.w = fmaf(v.w, w, acc.w);
      }
      yp[d] = from_f32<T>(acc.x * inv);
      yp[d + 1] = from_f32<T>(acc.y * inv);
      yp[d + 2] = from_f32<T>(acc.z * inv);
      yp[d + 3] = from_f32<T>(acc.w * inv);
    }
  } else {
    float M = SA_NEG_INF;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, ml[s * mstride]);
    for (int64_t d = threadIdx.x; d < D; d += blockDim.x) {
      float acc = 0.f;
      for (int s = 0; s < splits; ++s) {
        const float ms = ml[s * mstride];
        if (M == SA_NEG_INF || ms == SA_NEG_INF) continue;
        acc += po[s * pstride + d] * ex2(ms - M);
      }
      yp[d] = from_f32<T>(acc * inv);
    }
  }
}

// ---------------------------------------------------------------------------
// paged: write the new token's K/V into the pool at token ctx - 1
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) paged_append_kernel(PagedAppendArgs a) {
  const int64_t row_bytes = a.D * a.esz;
  const int64_t n = a.B * a.Hkv * row_bytes;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t byte = e % row_bytes;
    const int64_t bh = e / row_bytes;
    const int64_t b = bh / a.Hkv, h = bh % a.Hkv;
    const int64_t ctx = a.ctx_len[b];
    if (ctx < 1 || ctx > a.max_pages * a.page_tokens) {
      if (byte == 0 && h == 0 && a.err_word) atomicOr(a.err_word, SA_ERRBIT_PAGE);
      continue;
    }
    const int64_t t = ctx - 1;
    const int32_t page = a.block_table[b * a.max_pages + t / a.page_tokens];
    if (page < 0 || page >= a.num_pages) {
      if (byte == 0 && h == 0 && a.err_word) atomicOr(a.err_word, SA_ERRBIT_PAGE);
      continue;
    }
    const int64_t dst = ((static_cast<int64_t>(page) * a.Hkv + h) * a.page_tokens +
                         t % a.page_tokens) * row_bytes + byte;
    const int64_t src = bh * row_bytes + byte;
    if (a.k_new)
      static_cast<unsigned char*>(a.k_pool)[dst] = static_cast<const unsigned char*>(a.k_new)[src];
    if (a.v_new)
      static_cast<unsigned char*>(a.v_pool)[dst] = static_cast<const unsigned char*>(a.v_new)[src];
  }
}

int launch_paged_append(const PagedAppendArgs& a, cudaStream_t st) {
  const int64_t n = a.B * a.Hkv * a.D * a.esz;
  if (n == 0) return 0;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  paged_append_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

template <typename T, int DPL>
static int launch_simt(const GatherArgs& a, cudaStream_t st) {
  const int64_t grid = a.units * a.hpu * a.splits;
  gather_simt_kernel<T, DPL><<<static_cast<unsigned>(grid), 128, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

template <typename T>
static int launch_simt_any(const GatherArgs& a, cudaStream_t st) {
  const int64_t dpl = (a.D + 31) / 32;
  if (dpl <= 1) return launch_simt<T, 1>(a, st);
  if (dpl <= 2) return launch_simt<T, 2>(a, st);
  if (dpl <= 4) return launch_simt<T, 4>(a, st);
  if (dpl <= 8) return launch_simt<T, 8>(a, st);
  if (dpl <= 16) return launch_simt<T, 16>(a, st);
  return -2;
}

// Whether the tensor-core kernel serves this request (mirrors the host plan).
bool gather_uses_mma(const GatherArgs& a, int dtype) {
  if (dtype != SA_F16 && dtype != SA_BF16) return false;
  if (!(a.D == 64 || a.D == 128 || a.D == 256)) return false;
  if (a.hpu > 16) return false;
  if (a.D == 256 && a.hpu > 8) return false;
  return true;
}

int launch_gather_simt(const GatherArgs& a, int dtype, cudaStream_t st) {
  if (a.units == 0) return 0;
  if (dtype == SA_F32) return launch_simt_any<float>(a, st);
  if (dtype == SA_F16) return launch_simt_any<__half>(a, st);
  if (dtype == SA_BF16) return launch_simt_any<__nv_bfloat16>(a, st);
  return -2;
}

// The same merge for at most kFlatSplits splits, D % 4 == 0 and y aligned to
// four elements, one thread per four output dims of one head: every split's
// (max, sum) and O values are requested together, so the merge costs one
// round trip to L2.
constexpr int kFlatSplits = 8;

template <typename T>
__device__ __forceinline__ void store4(T* p, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void store4<float>(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}
template <>
__device__ __forceinline__ void store4<__half>(__half* p, float a, float b, float c, float d) {
  *reinterpret_cast<uint2*>(p) = make_uint2(pack2<__half>(a, b), pack2<__half>(c, d));
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float a, float b, float c,
                                                      float d) {
  *reinterpret_cast<uint2*>(p) =
      make_uint2(pack2<__nv_bfloat16>(a, b), pack2<__nv_bfloat16>(c, d));
}

template <typename T>
__global__ void __launch_bounds__(256) combine_flat_kernel(GatherArgs a) {
  pdl_wait();  // the partials of the kernel before (launched as its dependent)
  // item counts stay below 2^31 on this path (checked on the host): 32-bit division
  const uint32_t q4 = static_cast<uint32_t>(a.Dv / 4), hpu = static_cast<uint32_t>(a.hpu);
  const uint32_t item = blockIdx.x * blockDim.x + threadIdx.x;
  if (static_cast<int64_t>(item) >= a.units * a.hpu * q4) return;
  const uint32_t uh = item / q4, d = 4 * (item - uh * q4);
  const uint32_t unit = uh / hpu, hh = uh - unit * hpu;
  const UnitInfo u = unit_info(a, unit);
  const int64_t h = u.h0 + hh;
  const int splits = static_cast<int>(a.splits);
  const int64_t row0 = static_cast<int64_t>(unit) * a.splits * a.hpu + hh;  // (unit, split 0, head)
  float m[kFlatSplits], l[kFlatSplits];
  float4 o[kFlatSplits];
#pragma unroll
  for (int s = 0; s < kFlatSplits; ++s) {
    if (s < splits) {
      const int64_t r = row0 + s * a.hpu;
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.part_ml) + r);
      m[s] = ml.x;
      l[s] = ml.y;
      o[s] = __ldcg(reinterpret_cast<const float4*>(a.part_o + r * a.Dv + d));
    } else {
      m[s] = SA_NEG_INF;
      l[s] = 0.f;
      o[s] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  float M = SA_NEG_INF;
#pragma unroll
  for (int s = 0; s < kFlatSplits; ++s) M = fmaxf(M, m[s]);
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int s = 0; s < kFlatSplits; ++s) {
    const float w = (M == SA_NEG_INF || m[s] == SA_NEG_INF) ? 0.f : ex2(m[s] - M);
    L += l[s] * w;
    acc.x = fmaf(o[s].x, w, acc.x);
    acc.y = fmaf(o[s].y, w, acc.y);
    acc.z = fmaf(o[s].z, w, acc.z);
    acc.w = fmaf(o[s].w, w, acc.w);
  }
  if (a.sink && M != SA_NEG_INF) L += ex2(a.sink[h] * kLog2e - M);
  const float inv = (M == SA_NEG_INF || L == 0.f) ? 0.f : 1.0f / L;
  T* yp = static_cast<T*>(a.y) + ((u.b * a.Hq + h) * a.Sq + u.i) * a.Dv + d;
  store4<T>(yp, acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

// Launched as a programmatic dependent of the partials' kernel: its CTAs may
// be scheduled while that kernel drains, and wait for it (griddepcontrol.wait)
// before reading the partials.
template <typename T>
static int launch_combine_t(const GatherArgs& a, unsigned grid, cudaStream_t st) {
  const int64_t items = a.units * a.hpu * (a.Dv / 4);
  const bool flat = a.splits <= kFlatSplits && a.Dv % 4 == 0 && items < (int64_t(1) << 31) &&
                    reinterpret_cast<uintptr_t>(a.y) % (4 * sizeof(T)) == 0;  // vector stores
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(flat ? static_cast<unsigned>((items + 255) / 256) : grid);
  cfg.blockDim = dim3(flat ? 256 : 128);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, flat ? combine_flat_kernel<T> : combine_kernel<T>, a) ==
                 cudaSuccess
             ? 0
             : -1;
}

int launch_combine(const GatherArgs& a, int dtype, cudaStream_t st) {
  if (a.splits <= 1 || a.units == 0) return 0;
  const unsigned grid = static_cast<unsigned>(a.units * a.hpu);
  if (dtype == SA_F32) return launch_combine_t<float>(a, grid, st);
  if (dtype == SA_F16) return launch_combine_t<__half>(a, grid, st);
  return launch_combine_t<__nv_bfloat16>(a, grid, st);
}

}  // namespace sa
