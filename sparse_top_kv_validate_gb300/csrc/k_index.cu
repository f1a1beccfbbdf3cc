// k_index.cu -- ratio-4 index scoring and deterministic top-k selection: the
// step that produces the selected indices of compressed sparse attention.
//
// Semantics: onnx-runtime-ep-cpu src/kernels/compressed_sparse_attention.rs,
// finalize_index_query / hadamard_bf16 / fp4_roundtrip / select_ratio4_topk,
// and onnx-runtime-ep-cuda compressed_sparse_attention.rs,
// csa_ratio4_index_select / csa_ratio4_index_replicate.  Per (batch, query)
// row: each index head's query is rounded to bf16, Walsh-Hadamard transformed
// (bf16-rounded 1/sqrt(n) scale) and FP4-rounded per block of 32; each causal
// record r < (position + 1) / 4 scores sum_h relu(q_h . k_r) * w_h * c in
// binary32 (dot products in ascending dimension order, heads in ascending
// order, every multiply and add rounded on its own); records are ranked by
// score (Rust total_cmp, higher first), then by record index.
//
// GB300 design:
//  * index_query_kernel: one warp per (row, head).  The butterflies of spans
//    below the elements per lane run in registers, the larger spans through
//    shuffles; then the scale, the bf16 rounding and the OCP MX FP4 block
//    quantizer (scale 2^(floor(log2 amax) - 2)).  The query leaves as signed
//    integers 2 * E2M1 in [-12, 12] (one byte per dimension, in order) with
//    one exponent per block.
//  * index_score_kernel: one thread per record, 256 records per CTA staged in
//    shared memory.  A product of two FP4 values is exact in binary32, so when
//    every partial sum of the serial dot product is exactly representable --
//    the block exponents of query and key within 9 binades of each other and
//    far from underflow and overflow -- the serial binary32 sum IS the exact
//    dot product.  That is computed as one integer dp4a sum per 32-block,
//    combined exactly.  Any other (record, head) runs the serial binary32
//    loop.  Either way the score is the definition's, bit for bit, and the
//    head sum runs serially in ascending head order.
//  * index_topk_kernel: one CTA per row.  Equal scores are found with an
//    open-addressing hash set; an MSB-first radix select over the total-order
//    keys finds the k-th; the selected (key, record) pairs are bitonic-sorted
//    into score order (or record order).
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace sa {

namespace {

constexpr int kScoreThreads = 256;  // records per score CTA
constexpr int kTopkThreads = 1024;
constexpr uint32_t kEmpty = 0xffffffffu;  // hash slot marker (a NaN pattern: never a key)

// Row geometry: the causal record limit of row (b, s).
__device__ __forceinline__ int64_t row_limit(const IndexArgs& a, int64_t row) {
  const int64_t b = row / a.S, s = row % a.S;
  const int64_t p = (a.query_start_b ? __ldg(a.query_start_b + b) : a.query_start) + s;
  int64_t lim = p >= 0 ? (p + 1) / 4 : 0;
  return lim < a.R ? lim : a.R;
}

__device__ __forceinline__ float round_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// 2^e as binary32 for e in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float pow2f(int e) {
  if (e >= -126) return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
  return __uint_as_float(1u << (e + 149));
}

// floor(log2(m)) of a positive finite binary32 value.
__device__ __forceinline__ int floor_log2(float m) {
  const uint32_t u = __float_as_uint(m);
  const int ex = static_cast<int>((u >> 23) & 0xffu);
  if (ex) return ex - 127;
  return (31 - __clz(u & 0x7fffffu)) - 149;
}

// 2 * (nearest E2M1 magnitude to v >= 0), ties to the even code, saturating at 6.
__device__ __forceinline__ int e2m1_twice(float v) {
  if (v <= 0.25f) return 0;
  if (v < 0.75f) return 1;
  if (v <= 1.25f) return 2;
  if (v < 1.75f) return 3;
  if (v <= 2.5f) return 4;
  if (v < 3.5f) return 6;
  if (v <= 5.0f) return 8;
  return 12;
}

}  // namespace

// ---- query finalize ----------------------------------------------------------------------
// Grid: rows * IH warps, 4 warps per CTA.  NB = ID / 32 blocks = elements per lane.
template <int NB>
__global__ void __launch_bounds__(128) index_query_kernel(const IndexArgs a) {
  constexpr int ID = NB * 32;
  const int lane = threadIdx.x & 31;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (w >= a.rows * a.IH) return;
  const float* src = a.query + w * ID;
  float v[NB];
#pragma unroll
  for (int j = 0; j < NB; ++j) v[j] = round_bf16(__ldg(src + lane * NB + j));
  // butterflies: element i = lane * NB + j; spans below NB inside the lane
#pragma unroll
  for (int span = 1; span < NB; span *= 2)
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (!(j & span)) {
        const float l = v[j], r = v[j + span];
        v[j] = __fadd_rn(l, r);
        v[j + span] = __fsub_rn(l, r);
      }
  // spans NB .. ID/2: partner lane = lane ^ (span / NB); the left element's
  // lane takes left + right, the right one's left - right
#pragma unroll
  for (int ld = 1; ld < 32; ld *= 2)
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const float o = __shfl_xor_sync(0xffffffffu, v[j], ld);
      v[j] = (lane & ld) ? __fsub_rn(o, v[j]) : __fadd_rn(v[j], o);
    }
#pragma unroll
  for (int j = 0; j < NB; ++j) v[j] = round_bf16(__fmul_rn(v[j], a.had_scale));

  // FP4 per 32-block: the block's 32 / NB lanes
  constexpr int L = 32 / NB;
  float m = 0.0f;
  bool nf = false;
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    nf |= !isfinite(v[j]);
    m = fmaxf(m, fabsf(v[j]));
  }
#pragma unroll
  for (int o = 1; o < L; o *= 2) {
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    nf |= __shfl_xor_sync(0xffffffffu, nf ? 1 : 0, o) != 0;
  }
  int e = -127;  // all-zero block: scale byte 0
  if (!nf && m > 0.0f) {
    e = floor_log2(m) - 2;
    e = e < -127 ? -127 : (e > 127 ? 127 : e);
  }
  const float inv = pow2f(-e);  // exact: -e in [-127, 127]
  int8_t* qc = a.qcodes + w * ID;
  bool nz = false;
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    const int d = lane * NB + j;
    const float x = __fmul_rn(v[j], inv);
    int c = nf ? 0 : e2m1_twice(fabsf(x));
    if (x < 0.0f) c = -c;
    nz |= c != 0;
    qc[d] = static_cast<int8_t>(c);
  }
#pragma unroll
  for (int o = 1; o < L; o *= 2) nz |= __shfl_xor_sync(0xffffffffu, nz ? 1 : 0, o) != 0;
  // per block: exponent of the integer codes (value = code * 2^(e - 1)),
  // 127 marks a non-finite block
  const int blk = lane / L;
  if (lane % L == 0) a.qexp[w * NB + blk] = static_cast<int8_t>(nf ? 127 : e - 1);
  // per head: min / max exponent over its non-zero blocks, non-finite flag
  int emin = nz && !nf ? e - 1 : 1000, emax = nz && !nf ? e - 1 : -1000;
  int anynf = nf ? 1 : 0;
#pragma unroll
  for (int o = L; o < 32; o *= 2) {
    emin = min(emin, __shfl_xor_sync(0xffffffffu, emin, o));
    emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, o));
    anynf |= __shfl_xor_sync(0xffffffffu, anynf, o);
  }
  if (lane == 0) {
    int meta;
    if (anynf) meta = kQmetaNonfinite;
    else if (emin > emax) meta = kQmetaZero;  // every block zero: the dot is 0
    else meta = ((emin + 256) & 0x3ff) | (((emax + 256) & 0x3ff) << 10);
    a.qmeta[w] = meta;
  }
}

// ---- scores ------------------------------------------------------------------------------

namespace {

// PTX prmt in its default mode: byte i of the result is byte (c_i & 7) of
// {a, b}, or that byte's sign replicated when bit 3 of selector nibble c_i is
// set (the __byte_perm intrinsic ignores that bit).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Signed bytes 2 * E2M1 of the four nibble codes in the low 16 bits of x
// (element i in bits 4i..4i+3, bit 3 of a code its sign): byte i of the result.
__device__ __forceinline__ uint32_t nib4_to_s8(uint32_t x) {
  // select byte (code & 7) of the 8-byte tables: magnitudes 0 1 2 3 4 6 8 12
  // and their negations
  const uint32_t sel = x & 0x7777u;
  const uint32_t pos = prmt(0x03020100u, 0x0c080604u, sel);
  const uint32_t neg = prmt(0xfdfeff00u, 0xf4f8fafcu, sel);
  // sign mask: selector 9 (replicate the sign of byte 1 = 0x80) for a
  // negative code, 0 (byte 0 = 0x00) otherwise
  const uint32_t sgn = x & 0x8888u;
  const uint32_t sm = prmt(0x00008000u, 0u, sgn | (sgn >> 3));
  return (pos & ~sm) | (neg & sm);
}

// Element d's value as binary32 from the dp4a layout: code * 2^ex.
__device__ __forceinline__ float code_value(int code, int ex) {
  return __fmul_rn(static_cast<float>(code), pow2f(ex));
}

}  // namespace

template <int NB>
__global__ void __launch_bounds__(kScoreThreads) index_score_kernel(const IndexArgs a) {
  constexpr int ID = NB * 32;
  // largest block-exponent spread for which ID products of at most 144 units,
  // each shifted by up to the spread, sum below 2^24 units (exact in binary32)
  constexpr int kSpread = NB == 1 ? 11 : NB == 2 ? 10 : NB == 4 ? 9 : 8;
  constexpr int RW = (NB * 17 + 3) / 4 + 1;  // record words read (covers the funnel shifts)
  extern __shared__ __align__(16) unsigned char smem[];
  const int64_t row = blockIdx.y;
  const int64_t limit = row_limit(a, row);
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kScoreThreads;
  if (r0 >= limit) return;
  const int tid = threadIdx.x;
  const int IH = static_cast<int>(a.IH);
  uint32_t* sq = reinterpret_cast<uint32_t*>(smem);                    // [IH][ID / 4]
  int8_t* se = reinterpret_cast<int8_t*>(sq + IH * (ID / 4));           // [IH][NB]
  int* sm = reinterpret_cast<int*>(smem + ((IH * (ID + NB) + 15) / 16) * 16);  // [IH]
  float* sw = reinterpret_cast<float*>(sm + IH);                        // [IH]
  uint32_t* srec = reinterpret_cast<uint32_t*>(sw + IH);                // [256][stride / 4]
  // stage the row's query codes, exponents, metas, weights and 256 records
  pdl_wait();
  {
    const uint4* qsrc = reinterpret_cast<const uint4*>(a.qcodes + row * IH * ID);
    for (int i = tid; i < IH * ID / 16; i += kScoreThreads)
      reinterpret_cast<uint4*>(sq)[i] = qsrc[i];
    for (int i = tid; i < IH * NB; i += kScoreThreads) se[i] = a.qexp[row * IH * NB + i];
    for (int i = tid; i < IH; i += kScoreThreads) {
      sm[i] = a.qmeta[row * IH + i];
      sw[i] = __ldg(a.weight + row * IH + i);
    }
    const int64_t b = row / a.S;
    const int sw4 = static_cast<int>(a.key_stride / 4);
    int64_t nrec = limit - r0;
    if (nrec > kScoreThreads) nrec = kScoreThreads;
    const uint32_t* ksrc = reinterpret_cast<const uint32_t*>(a.keys + (b * a.R + r0) * a.key_stride);
    for (int i = tid; i < nrec * sw4; i += kScoreThreads) srec[i] = __ldg(ksrc + i);
  }
  __syncthreads();
  const int64_t r = r0 + tid;
  if (r >= limit) return;

  // this thread's record: the packed words of each block, realigned
  uint32_t rw[RW];
  const uint32_t* mine = srec + tid * static_cast<int>(a.key_stride / 4);
#pragma unroll
  for (int i = 0; i < RW; ++i) rw[i] = (i * 4 < a.key_stride) ? mine[i] : 0u;
  uint32_t kv[NB][8];  // signed bytes of elements 4j .. 4j + 3 of each block
  int ke[NB];
  int kemin = 1000, kemax = -1000;
  bool knf = false;
#pragma unroll
  for (int bl = 0; bl < NB; ++bl) {
    const int o = 17 * bl;  // scale byte; the block's data bytes start at o + 1
    const uint32_t sbyte = (rw[o / 4] >> (8 * (o % 4))) & 0xffu;
    knf |= sbyte == 0xffu;
    ke[bl] = static_cast<int>(sbyte) - 128;  // value = code * 2^(byte - 128)
    kemin = min(kemin, ke[bl]);
    kemax = max(kemax, ke[bl]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int ob = o + 1 + 4 * k;
      const uint32_t word = __funnelshift_r(rw[ob / 4], rw[ob / 4 + 1], 8 * (ob % 4));
      kv[bl][2 * k] = nib4_to_s8(word);
      kv[bl][2 * k + 1] = nib4_to_s8(word >> 16);
    }
  }
  const int dk = kemax - kemin;

  float score = 0.0f;
  for (int h = 0; h < IH; ++h) {
    const int meta = sm[h];
    float dot = 0.0f;
    if (meta != kQmetaZero) {
      const uint32_t* qh = sq + h * (ID / 4);
      const int8_t* qe = se + h * NB;
      bool fast = !knf && meta != kQmetaNonfinite;
      int qmin = 0, qmax = 0;
      if (fast) {
        qmin = (meta & 0x3ff) - 256;
        qmax = ((meta >> 10) & 0x3ff) - 256;
        const int smin = qmin + kemin, smax = qmax + kemax;
        fast = (qmax - qmin) + dk <= kSpread && smin >= -149 && smax <= 100;
      }
      if (fast) {
        int32_t N = 0;
        const int smin = qmin + kemin;
#pragma unroll
        for (int bl = 0; bl < NB; ++bl) {
          const uint4 q0 = reinterpret_cast<const uint4*>(qh)[bl * 2];
          const uint4 q1 = reinterpret_cast<const uint4*>(qh)[bl * 2 + 1];
          int32_t I = 0;
          I = __dp4a(static_cast<int>(kv[bl][0]), static_cast<int>(q0.x), I);
          I = __dp4a(static_cast<int>(kv[bl][1]), static_cast<int>(q0.y), I);
          I = __dp4a(static_cast<int>(kv[bl][2]), static_cast<int>(q0.z), I);
          I = __dp4a(static_cast<int>(kv[bl][3]), static_cast<int>(q0.w), I);
          I = __dp4a(static_cast<int>(kv[bl][4]), static_cast<int>(q1.x), I);
          I = __dp4a(static_cast<int>(kv[bl][5]), static_cast<int>(q1.y), I);
          I = __dp4a(static_cast<int>(kv[bl][6]), static_cast<int>(q1.z), I);
          I = __dp4a(static_cast<int>(kv[bl][7]), static_cast<int>(q1.w), I);
          if (I != 0) N += I * (1 << (qe[bl] + ke[bl] - smin));  // shift in [0, kSpread]
        }
        dot = __fmul_rn(static_cast<float>(N), pow2f(smin));  // |N| < 2^24: exact
      } else {
        // the definition itself: serial binary32, ascending dimension (the key
        // codes re-read from the staged record: no dynamic register indexing)
        const uint8_t* rb = reinterpret_cast<const uint8_t*>(mine);
#pragma unroll 1
        for (int d = 0; d < ID; ++d) {
          const int bl = d >> 5;
          const int qc = static_cast<int>(reinterpret_cast<const int8_t*>(qh)[d]);
          const uint8_t* blk = rb + 17 * bl;
          const int kb = static_cast<int>(blk[0]) - 128;
          const uint32_t nib = (blk[1 + ((d & 31) >> 1)] >> (4 * (d & 1))) & 0xfu;
          const int kc = static_cast<int>(static_cast<int8_t>(nib4_to_s8(nib) & 0xffu));
          const float qv = qe[bl] == 127 ? __int_as_float(0x7fc00000) : code_value(qc, qe[bl]);
          const float kv_ = kb == 127 ? __int_as_float(0x7fc00000) : code_value(kc, kb);
          dot = __fadd_rn(dot, __fmul_rn(qv, kv_));
        }
      }
    }
    const float relu = fmaxf(dot, 0.0f);
    score = __fadd_rn(score, __fmul_rn(__fmul_rn(relu, sw[h]), a.weight_scale));
  }
  a.scores[row * a.R + r] = score;
  pdl_launch_dependents();
}

// ---- top-k -------------------------------------------------------------------------------

namespace {

// Block-wide exclusive prefix sum of one value per thread (1024 threads).
__device__ __forceinline__ int block_excl_scan(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o *= 2) {
    const int n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o *= 2) {
      const int n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    wsum[lane] = s;  // inclusive totals per warp
  }
  __syncthreads();
  const int before = (warp > 0 ? wsum[warp - 1] : 0) + x - v;
  const int tot = wsum[31];
  __syncthreads();  // wsum reused by the next scan
  *total = tot;
  return before;
}

// Ascending bitonic sort of n (a power of two) 64-bit keys in shared memory.
__device__ void bitonic_sort(unsigned long long* k, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n / 2; i += blockDim.x) {
        const int lo = 2 * stride * (i / stride) + (i % stride);
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const unsigned long long x = k[lo], y = k[hi];
        if ((x > y) == up) {
          k[lo] = y;
          k[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

}  // namespace

// Grid: one CTA per row.  keys / hash: shared memory when they fit
// (a.topk_global == 0), else this row's slices of the workspace.
__global__ void __launch_bounds__(kTopkThreads) index_topk_kernel(const IndexArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_hist[256];
  __shared__ int s_wsum[32];
  __shared__ int s_flags;
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  const int n = static_cast<int>(row_limit(a, row));
  const int P = a.hash_slots;
  uint32_t* keys;
  uint32_t* hash;
  if (a.topk_global) {
    keys = a.gkeys + row * a.R;
    hash = a.ghash + row * static_cast<int64_t>(P);
  } else {
    keys = reinterpret_cast<uint32_t*>(smem);
    hash = keys + ((a.R + 3) / 4) * 4;
  }
  if (tid == 0) s_flags = 0;
  for (int i = tid; i < P; i += kTopkThreads) hash[i] = kEmpty;
  pdl_wait();
  __syncthreads();

  // keys in ascending order of (score descending): d = ~(total-order key)
  int flags = 0;
  const float* sc = a.scores + row * a.R;
  for (int i = tid; i < n; i += kTopkThreads) {
    const float f = sc[i];
    const uint32_t u = __float_as_uint(f);
    const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    keys[i] = ~ord;
    if (!isfinite(f)) flags |= kSelNonfinite;
  }
  __syncthreads();
  // equal scores (binary32 ==: +0 equals -0, NaN equals nothing)
  for (int i = tid; i < n; i += kTopkThreads) {
    const float f = sc[i];
    if (f != f) continue;
    const uint32_t c = (f == 0.0f) ? 0u : __float_as_uint(f);
    uint32_t h = (c * 0x9e3779b1u) >> (32 - a.hash_log2);
    for (int probe = 0; probe < P; ++probe) {
      const uint32_t prev = atomicCAS(hash + h, kEmpty, c);
      if (prev == kEmpty) break;
      if (prev == c) {
        flags |= kSelTie;
        break;
      }
      h = (h + 1) & static_cast<uint32_t>(P - 1);
    }
  }
  if (flags) atomicOr(&s_flags, flags);

  const int k = n < a.topk ? n : static_cast<int>(a.topk);
  // ---- radix select of the k-th smallest key (k >= 1, k < n) ----
  uint32_t prefix = 0, pmask = 0;
  int need = k;  // rank within the keys that match the prefix
  if (k > 0 && k < n) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = tid; i < 256; i += kTopkThreads) s_hist[i] = 0;
      __syncthreads();
      for (int i0 = 0; i0 < n; i0 += kTopkThreads) {
        const int i = i0 + tid;
        const bool in = i < n && (keys[i] & pmask) == prefix;
        const unsigned act = __ballot_sync(0xffffffffu, in);
        if (in) {
          const uint32_t dig = (keys[i] >> shift) & 0xffu;
          const unsigned peers = __match_any_sync(act, dig);
          if ((__ffs(peers) - 1) == (tid & 31)) atomicAdd(&s_hist[dig], __popc(peers));
        }
      }
      __syncthreads();
      if (tid < 32) {
        // the digit holding rank `need`: cumulative counts over 8 bins per lane
        int c[8], tot = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = s_hist[tid * 8 + j];
          tot += c[j];
        }
        int x = tot;
#pragma unroll
        for (int o = 1; o < 32; o *= 2) {
          const int y = __shfl_up_sync(0xffffffffu, x, o);
          if (tid >= o) x += y;
        }
        int cum = x - tot;  // before this lane's bins
        int found = -1, before = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (found < 0 && cum + c[j] >= need) {
            found = tid * 8 + j;
            before = cum;
          }
          cum += c[j];
        }
        const unsigned has = __ballot_sync(0xffffffffu, found >= 0);
        const int src = __ffs(has) - 1;
        const int dg = __shfl_sync(0xffffffffu, found, src);
        const int bf = __shfl_sync(0xffffffffu, before, src);
        if (tid == 0) {
          s_prefix = prefix | (static_cast<uint32_t>(dg) << shift);
          s_need = need - bf;
        }
      }
      __syncthreads();
      prefix = s_prefix;
      need = s_need;
      pmask |= 0xffu << shift;
    }
  }
  // ---- collect: keys below the threshold, and the first `need` equal to it ----
  unsigned long long* sel = reinterpret_cast<unsigned long long*>(hash);  // the hash is done
  const bool all = (k == n);
  const int chunk = (n + kTopkThreads - 1) / kTopkThreads;
  const int c0 = tid * chunk;
  const int c1 = min(n, c0 + chunk);
  int eq = 0, less = 0;
  if (!all)
    for (int i = c0; i < c1; ++i) {
      const uint32_t d = keys[i];
      eq += d == prefix;
      less += d < prefix;
    }
  int tot;
  const int eq_before = block_excl_scan(eq, s_wsum, &tot);
  int take_eq = all ? 0 : max(0, min(eq, need - eq_before));
  const int mine = all ? (c1 > c0 ? c1 - c0 : 0) : less + take_eq;
  int kcount;
  int slot = block_excl_scan(mine, s_wsum, &kcount);
  __syncthreads();  // every thread is past the hash before it is overwritten
  int npad = 1;
  while (npad < kcount) npad <<= 1;
  for (int i = c0; i < c1; ++i) {
    const uint32_t d = keys[i];
    bool take = all || d < prefix;
    if (!take && d == prefix && take_eq > 0) {
      take = true;
      --take_eq;
    }
    if (take)
      sel[slot++] = a.ascending ? (static_cast<unsigned long long>(i) << 32)
                                : ((static_cast<unsigned long long>(d) << 32) | static_cast<uint32_t>(i));
  }
  for (int i = kcount + tid; i < npad; i += kTopkThreads) sel[i] = ~0ull;
  __syncthreads();
  if (kcount > 1) bitonic_sort(sel, npad);
  // ---- write the row (replicated per output head), -1 past the selection ----
  const int64_t b = row / a.S, s = row % a.S;
  for (int o = 0; o < a.out_heads; ++o) {
    int32_t* out = a.selected + ((b * a.out_heads + o) * a.S + s) * a.topk;
    for (int j = tid; j < a.topk; j += kTopkThreads) {
      int32_t v = -1;
      if (j < kcount) {
        const unsigned long long x = sel[j];
        v = a.ascending ? static_cast<int32_t>(x >> 32) : static_cast<int32_t>(x & 0xffffffffu);
      }
      out[j] = v;
    }
  }
  __syncthreads();
  if (tid == 0) {
    const int f = s_flags;
    if (a.row_status) a.row_status[row] = static_cast<uint8_t>(f);
    if (f && a.err_word) atomicOr(a.err_word, static_cast<uint32_t>(f) << kSelErrShift);
  }
}

// ---- host side ---------------------------------------------------------------------------

size_t index_topk_smem_bytes(int64_t R, int hash_slots) {
  return static_cast<size_t>((R + 3) / 4 * 4) * 4 + static_cast<size_t>(hash_slots) * 4;
}

size_t index_score_smem_bytes(int64_t IH, int64_t ID, int64_t key_stride) {
  const int64_t NB = ID / 32;
  return static_cast<size_t>((IH * (ID + NB) + 15) / 16 * 16 + IH * 8 +
                             kScoreThreads * key_stride);
}

template <int NB>
static int launch_index_t(const IndexArgs& a, cudaStream_t st) {
  const unsigned qblocks = static_cast<unsigned>((a.rows * a.IH + 3) / 4);
  index_query_kernel<NB><<<qblocks, 128, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return -1;
  const size_t ss = index_score_smem_bytes(a.IH, a.ID, a.key_stride);
  if (cudaFuncSetAttribute(index_score_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(ss)) != cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = st;
  cfg.gridDim = dim3(static_cast<unsigned>((a.R + kScoreThreads - 1) / kScoreThreads),
                     static_cast<unsigned>(a.rows));
  cfg.blockDim = dim3(kScoreThreads);
  cfg.dynamicSmemBytes = ss;
  mark_event(a.ev_before, st);
  if (cudaLaunchKernelEx(&cfg, index_score_kernel<NB>, a) != cudaSuccess) return -1;
  mark_event(a.ev_after, st);
  const size_t ts = a.topk_global ? 0 : index_topk_smem_bytes(a.R, a.hash_slots);
  if (cudaFuncSetAttribute(index_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(ts)) != cudaSuccess)
    return -1;
  cfg.gridDim = dim3(static_cast<unsigned>(a.rows));
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = ts;
  return cudaLaunchKernelEx(&cfg, index_topk_kernel, a) == cudaSuccess ? 0 : -1;
}

int launch_index_select(const IndexArgs& a, cudaStream_t st) {
  switch (a.ID) {
    case 32: return launch_index_t<1>(a, st);
    case 64: return launch_index_t<2>(a, st);
    case 128: return launch_index_t<4>(a, st);
    case 256: return launch_index_t<8>(a, st);
    default: return -1;
  }
}

}  // namespace sa
