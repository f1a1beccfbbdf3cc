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
//    keys finds the k-th; the selected (key, record) pairs are sorted into
//    score order (or record order): runs of 64 by a bitonic network in each
//    warp's registers, then merge levels found by binary search (merge path).
#include <cmath>

#include "codes.cuh"
#include "common.cuh"
#include "kernels.h"

namespace sa {

namespace {

constexpr int kScoreRecords = 256;  // records per score CTA
constexpr int kTopkThreads = 1024;
constexpr int kTiePartsLog2 = 3;  // CTAs per row sharing the equal-score check
constexpr int kTieParts = 1 << kTiePartsLog2;
constexpr uint32_t kEmpty = 0xffffffffu;  // hash slot marker (a NaN pattern: never a key)

// Row geometry: the causal record limit of row (b, s).
__device__ __forceinline__ int64_t row_limit(const IndexArgs& a, int64_t row) {
  const int64_t b = row / a.S, s = row % a.S;
  const int64_t p = (a.query_start_b ? __ldg(a.query_start_b + b) : a.query_start) + s;
  int64_t lim = p >= 0 ? (p + 1) / 4 : 0;
  return lim < a.R ? lim : a.R;
}

// Rank key of a score: ascending keys = descending scores in Rust's total_cmp
// order (the complement of the order-preserving unsigned image of the bits).
__device__ __forceinline__ uint32_t rank_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? u : ~(u | 0x80000000u);
}

}  // namespace

// ---- query finalize ----------------------------------------------------------------------
// Grid: rows * IH warps, 4 warps per CTA.  NB = ID / 32 blocks = elements per lane.
template <int NB>
__global__ void __launch_bounds__(128) index_query_kernel(const IndexArgs a) {
  constexpr int ID = NB * 32;
  const int lane = threadIdx.x & 31;
  // the per-row tables the later kernels fill: histogram, flags, counters
  {
    const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t i = t0; i < a.rows * 2048; i += nth) a.hist[i] = 0u;
    for (int64_t i = t0; i < a.rows; i += nth) {
      a.rowflags[i] = 0u;
      a.done[i] = 0u;
    }
  }
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
  // per block: exponent of the integer codes (value = code * 2^(e - 1)) and
  // that power of two as binary32; exponent 127 marks a non-finite block
  const int blk = lane / L;
  if (lane % L == 0) {
    a.qexp[w * NB + blk] = static_cast<int8_t>(nf ? 127 : e - 1);
    a.qscale[w * NB + blk] = pow2f(e - 1);
  }
  // per head: exponent range over its non-zero blocks, zero / non-finite flags
  int emin = nz && !nf ? e - 1 : 1000, emax = nz && !nf ? e - 1 : -1000;
  int anynf = nf ? 1 : 0;
#pragma unroll
  for (int o = L; o < 32; o *= 2) {
    emin = min(emin, __shfl_xor_sync(0xffffffffu, emin, o));
    emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, o));
    anynf |= __shfl_xor_sync(0xffffffffu, anynf, o);
  }
  if (lane == 0) {
    int4 info;
    info.x = emax - emin;
    info.y = emin;
    info.z = emax;
    info.w = anynf ? kQinfoNonfinite : (emin > emax ? kQinfoZero : 0);
    a.qinfo[w] = info;
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

// Element value as binary32: code * 2^ex (ex 127: the block is non-finite).
__device__ __forceinline__ float code_value(int code, int ex) {
  if (ex == 127) return __int_as_float(0x7fc00000);
  return __fmul_rn(static_cast<float>(code), pow2f(ex));
}

// One record, unpacked: signed codes of every 4 elements, block exponents and
// their powers of two, the exponent range and whether a scale is NaN.
template <int NB>
struct KeyRec {
  uint32_t kv[NB][8];
  float ks[NB];
  int kemin, kemax;
  bool knf;
  const uint8_t* bytes;  // the staged record (serial path)
};

template <int NB>
__device__ __forceinline__ void unpack_record(const uint32_t* mine, int stride_bytes,
                                              KeyRec<NB>& k) {
  constexpr int RW = (NB * 17 + 3) / 4 + 1;  // words covering the funnel shifts
  uint32_t rw[RW];
#pragma unroll
  for (int i = 0; i < RW; ++i) rw[i] = (i * 4 < stride_bytes) ? mine[i] : 0u;
  k.kemin = 1000;
  k.kemax = -1000;
  k.knf = false;
  k.bytes = reinterpret_cast<const uint8_t*>(mine);
#pragma unroll
  for (int bl = 0; bl < NB; ++bl) {
    const int o = 17 * bl;  // scale byte; the block's data bytes start at o + 1
    const uint32_t sbyte = (rw[o / 4] >> (8 * (o % 4))) & 0xffu;
    k.knf |= sbyte == 0xffu;
    const int ke = static_cast<int>(sbyte) - 128;  // value = code * 2^(byte - 128)
    k.ks[bl] = pow2f(ke);
    k.kemin = min(k.kemin, ke);
    k.kemax = max(k.kemax, ke);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int ob = o + 1 + 4 * w;
      const uint32_t word = __funnelshift_r(rw[ob / 4], rw[ob / 4 + 1], 8 * (ob % 4));
      k.kv[bl][2 * w] = nib4_to_s8(word);
      k.kv[bl][2 * w + 1] = nib4_to_s8(word >> 16);
    }
  }
}

}  // namespace

// RPT records per thread (2 for ID <= 128), 256 records per CTA.
template <int NB, int RPT>
__global__ void __launch_bounds__(kScoreRecords / RPT) index_score_kernel(const IndexArgs a) {
  constexpr int ID = NB * 32;
  constexpr int NT = kScoreRecords / RPT;
  // largest block-exponent spread for which ID products of at most 144 units,
  // each scaled by up to 2^spread, sum below 2^24 units (exact in binary32)
  constexpr int kSpread = NB == 1 ? 11 : NB == 2 ? 10 : NB == 4 ? 9 : 8;
  extern __shared__ __align__(16) unsigned char smem[];
  const int64_t row = blockIdx.y;
  const int64_t limit = row_limit(a, row);
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kScoreRecords;
  if (r0 >= limit) return;
  const int tid = threadIdx.x;
  const int IH = static_cast<int>(a.IH);
  int4* sinfo = reinterpret_cast<int4*>(smem);                        // [IH]
  float* sqs = reinterpret_cast<float*>(sinfo + IH);                   // [IH][NB]
  float* sw = sqs + ((IH * NB + 3) / 4) * 4;                           // [IH]
  uint32_t* sq = reinterpret_cast<uint32_t*>(sw + ((IH + 3) / 4) * 4); // [IH][ID / 4]
  int8_t* se = reinterpret_cast<int8_t*>(sq + IH * (ID / 4));          // [IH][NB]
  uint32_t* srec = reinterpret_cast<uint32_t*>(se + ((IH * NB + 15) / 16) * 16);
  __shared__ uint32_t shist[2048];  // this CTA's counts of the rank keys' top 11 bits
  __shared__ uint32_t sflags;
  for (int i = tid; i < 2048; i += NT) shist[i] = 0u;
  if (tid == 0) sflags = 0u;
  pdl_wait();
  {
    const uint4* qsrc = reinterpret_cast<const uint4*>(a.qcodes + row * IH * ID);
    for (int i = tid; i < IH * ID / 16; i += NT) reinterpret_cast<uint4*>(sq)[i] = qsrc[i];
    for (int i = tid; i < IH * NB; i += NT) {
      se[i] = a.qexp[row * IH * NB + i];
      sqs[i] = a.qscale[row * IH * NB + i];
    }
    for (int i = tid; i < IH; i += NT) {
      sinfo[i] = a.qinfo[row * IH + i];
      sw[i] = __ldg(a.weight + row * IH + i);
    }
    const int64_t b = row / a.S;
    const int sw4 = static_cast<int>(a.key_stride / 4);
    int64_t nrec = limit - r0;
    if (nrec > kScoreRecords) nrec = kScoreRecords;
    const uint32_t* ksrc =
        reinterpret_cast<const uint32_t*>(a.keys + (b * a.R + r0) * a.key_stride);
    for (int i = tid; i < nrec * sw4; i += NT) srec[i] = __ldg(ksrc + i);
  }
  __syncthreads();
  const int stride4 = static_cast<int>(a.key_stride / 4);
  bool live[RPT];
  KeyRec<NB> k[RPT];
  int lim_d[RPT], lim_lo[RPT], lim_hi[RPT];
  float score[RPT];
#pragma unroll
  for (int j = 0; j < RPT; ++j) {
    const int loc = tid + j * NT;
    live[j] = r0 + loc < limit;
    unpack_record<NB>(srec + (live[j] ? loc : 0) * stride4, static_cast<int>(a.key_stride), k[j]);
    // a head takes the exact path when its exponent range fits these bounds
    lim_d[j] = kSpread - (k[j].kemax - k[j].kemin);
    lim_lo[j] = -149 - k[j].kemin;
    lim_hi[j] = 100 - k[j].kemax;
    if (k[j].knf) lim_d[j] = -1;
    score[j] = 0.0f;
  }
  for (int h = 0; h < IH; ++h) {
    const int4 info = sinfo[h];
    const float wh = sw[h];
    const uint4* qh = reinterpret_cast<const uint4*>(sq + h * (ID / 4));
    float qs[NB];
#pragma unroll
    for (int bl = 0; bl < NB; ++bl) qs[bl] = sqs[h * NB + bl];
    int32_t I[RPT][NB];
#pragma unroll
    for (int bl = 0; bl < NB; ++bl) {
      const uint4 q0 = qh[bl * 2], q1 = qh[bl * 2 + 1];
#pragma unroll
      for (int j = 0; j < RPT; ++j) {
        int32_t t = 0;
        t = __dp4a(static_cast<int>(k[j].kv[bl][0]), static_cast<int>(q0.x), t);
        t = __dp4a(static_cast<int>(k[j].kv[bl][1]), static_cast<int>(q0.y), t);
        t = __dp4a(static_cast<int>(k[j].kv[bl][2]), static_cast<int>(q0.z), t);
        t = __dp4a(static_cast<int>(k[j].kv[bl][3]), static_cast<int>(q0.w), t);
        t = __dp4a(static_cast<int>(k[j].kv[bl][4]), static_cast<int>(q1.x), t);
        t = __dp4a(static_cast<int>(k[j].kv[bl][5]), static_cast<int>(q1.y), t);
        t = __dp4a(static_cast<int>(k[j].kv[bl][6]), static_cast<int>(q1.z), t);
        t = __dp4a(static_cast<int>(k[j].kv[bl][7]), static_cast<int>(q1.w), t);
        I[j][bl] = t;
      }
    }
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      float dot = 0.0f;
      if (info.w != kQinfoZero) {
        if (info.w == 0 && info.x <= lim_d[j] && info.y >= lim_lo[j] && info.z <= lim_hi[j]) {
          // every partial sum exact: the block sums times their exact powers
          // of two, added exactly (each fma's result is representable)
#pragma unroll
          for (int bl = 0; bl < NB; ++bl)
            dot = __fmaf_rn(static_cast<float>(I[j][bl]), __fmul_rn(qs[bl], k[j].ks[bl]), dot);
        } else {
          // the definition itself: serial binary32 in ascending dimension
          // (codes re-read from shared memory: no dynamic register indexing)
          const int8_t* qcb = reinterpret_cast<const int8_t*>(qh);
          const int8_t* qe = se + h * NB;
          const uint8_t* rb = k[j].bytes;
#pragma unroll 1
          for (int d = 0; d < ID; ++d) {
            const int bl = d >> 5;
            const uint8_t* blk = rb + 17 * bl;
            const int kb = static_cast<int>(blk[0]) - 128;
            const uint32_t nib = (blk[1 + ((d & 31) >> 1)] >> (4 * (d & 1))) & 0xfu;
            const int kc = static_cast<int>(static_cast<int8_t>(nib4_to_s8(nib) & 0xffu));
            dot = __fadd_rn(dot, __fmul_rn(code_value(qcb[d], qe[bl]), code_value(kc, kb)));
          }
        }
      }
      const float relu = fmaxf(dot, 0.0f);
      score[j] = __fadd_rn(score[j], __fmul_rn(__fmul_rn(relu, wh), a.weight_scale));
    }
  }
  // scores out; their rank keys into the row's histogram (counted here,
  // added to the global one per bin)
  uint32_t flags = 0;
#pragma unroll
  for (int j = 0; j < RPT; ++j) {
    if (!live[j]) continue;
    const float f = score[j];
    a.scores[row * a.R + r0 + tid + j * NT] = f;
    atomicAdd(&shist[rank_key(f) >> 21], 1u);
    if (!isfinite(f)) flags |= kSelNonfinite;
  }
  if (flags) atomicOr(&sflags, flags);
  __syncthreads();
  for (int i = tid; i < 2048; i += NT)
    if (shist[i]) atomicAdd(a.hist + row * 2048 + i, shist[i]);
  if (tid == 0 && sflags) atomicOr(a.rowflags + row, sflags);
  pdl_launch_dependents();
}

// ---- top-k -------------------------------------------------------------------------------

namespace {

// Each warp sorts runs of 64 keys ascending in registers (two keys a lane:
// run positions lane and lane + 32), a bitonic network over the run.
__device__ void warp_sort64(unsigned long long* k, int n) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int c = warp; c < n / 64; c += nw) {
    const int base = c * 64;
    unsigned long long x[2] = {k[base + lane], k[base + 32 + lane]};
#pragma unroll
    for (int sz = 2; sz <= 64; sz <<= 1) {
#pragma unroll
      for (int stride = sz >> 1; stride > 0; stride >>= 1) {
        if (stride == 32) {  // sz == 64: the run's final merge, ascending
          if (x[0] > x[1]) {
            const unsigned long long t = x[0];
            x[0] = x[1];
            x[1] = t;
          }
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, x[h], stride);
            const int e = 32 * h + lane;  // position in the run
            const bool up = sz == 64 || (e & sz) == 0;
            const bool keep_min = ((e & stride) == 0) == up;
            x[h] = keep_min ? (x[h] < o ? x[h] : o) : (x[h] < o ? o : x[h]);
          }
        }
      }
    }
    k[base + lane] = x[0];
    k[base + 32 + lane] = x[1];
  }
}

// One merge level: the sorted runs of L keys in src, taken in pairs, become
// sorted runs of 2 L in dst.  Output rank r of a pair is found by a binary
// search for the number i of keys of the first run among the pair's first r
// outputs (equal keys -- only the padding -- take the second run's first).
__device__ void merge_level(const unsigned long long* src, unsigned long long* dst, int n, int L) {
  for (int o = threadIdx.x; o < n; o += blockDim.x) {
    const int base = o & ~(2 * L - 1), r = o - base;
    const unsigned long long* A = src + base;
    const unsigned long long* Bv = A + L;
    int lo = r > L ? r - L : 0, hi = r < L ? r : L;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (A[mid] < Bv[r - mid - 1]) lo = mid + 1;
      else hi = mid;
    }
    const int j = r - lo;
    const bool take_a = j >= L || (lo < L && A[lo] < Bv[j]);
    dst[o] = take_a ? A[lo] : Bv[j];
  }
}

// Ascending sort of n (a power of two, >= 64) 64-bit keys in shared memory:
// runs of 64 sorted in registers, then log2(n / 64) merge levels between k
// and tmp (n keys of scratch), the result back in k.
__device__ void merge_sort(unsigned long long* k, unsigned long long* tmp, int n) {
  warp_sort64(k, n);
  __syncthreads();
  unsigned long long* src = k;
  unsigned long long* dst = tmp;
  for (int L = 64; L < n; L <<= 1) {
    merge_level(src, dst, n, L);
    __syncthreads();
    unsigned long long* t = src;
    src = dst;
    dst = t;
  }
  if (src != k) {
    for (int o = threadIdx.x; o < n; o += blockDim.x) k[o] = src[o];
    __syncthreads();
  }
}

// Ascending bitonic sort of n (a power of two, below 64) 64-bit keys in
// shared memory, a barrier per stage.
__device__ void bitonic_sort(unsigned long long* k, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n / 2; i += blockDim.x) {
        const int lo = ((i & ~(stride - 1)) << 1) | (i & (stride - 1));
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

// One pass over the bucket of a row: among the keys matching (prefix, pmask),
// the digit (v >> shift) & dmask holding rank `need`; returns the extended
// prefix, updates need to the rank inside that digit and cnt to its count.
__device__ unsigned long long bucket_pass(const unsigned long long* bk, int m,
                                          unsigned long long prefix, unsigned long long pmask,
                                          int shift, unsigned dmask, int& need, int& cnt,
                                          int* hist, unsigned long long* s_prefix, int* s_need,
                                          int* s_cnt) {
  const int tid = threadIdx.x;
  for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int i0 = 0; i0 < m; i0 += blockDim.x) {
    const int i = i0 + tid;
    unsigned long long v = 0;
    bool in = false;
    if (i < m) {
      v = bk[i];
      in = (v & pmask) == prefix;
    }
    const unsigned act = __ballot_sync(0xffffffffu, in);
    if (in) {
      const unsigned dig = static_cast<unsigned>(v >> shift) & dmask;
      const unsigned peers = __match_any_sync(act, dig);
      if ((__ffs(peers) - 1) == (tid & 31)) atomicAdd(&hist[dig], __popc(peers));
    }
  }
  __syncthreads();
  if (tid < 32) {
    int c[8], tot = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c[j] = hist[tid * 8 + j];
      tot += c[j];
    }
    int x = tot;
#pragma unroll
    for (int o = 1; o < 32; o *= 2) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (tid >= o) x += y;
    }
    int cum = x - tot, found = -1, before = 0, cc = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (found < 0 && cum + c[j] >= need) {
        found = tid * 8 + j;
        before = cum;
        cc = c[j];
      }
      cum += c[j];
    }
    const unsigned has = __ballot_sync(0xffffffffu, found >= 0);
    const int src = __ffs(has) - 1;
    const int dg = __shfl_sync(0xffffffffu, found, src);
    const int bf = __shfl_sync(0xffffffffu, before, src);
    const int ct = __shfl_sync(0xffffffffu, cc, src);
    if (tid == 0) {
      *s_prefix = prefix | (static_cast<unsigned long long>(dg) << shift);
      *s_need = need - bf;
      *s_cnt = ct;
    }
  }
  __syncthreads();
  need = *s_need;
  cnt = *s_cnt;
  return *s_prefix;
}

// Inserts this thread's scores f[u] (those with take[u]) into an
// open-addressing hash set of binary32 values (==: +0 equals -0; NaN is never
// passed); slot hs[u] first.  Returns 1 if one of them was already there.
// One probe per round, walking the thread's scores in turn, so that the
// lanes of a warp stay in step.
template <int kPer>
__device__ __forceinline__ int insert_scores(uint32_t* table, const uint32_t (&hc)[kPer],
                                             const uint32_t (&h0)[kPer],
                                             const bool (&take)[kPer], uint32_t hmask) {
  int u = 0, ties = 0;
  bool have = false;
  uint32_t c = 0, hs = 0;
  while (true) {
    while (!have && u < kPer) {
      if (take[u]) {
        c = hc[u];
        hs = h0[u];
        have = true;
      } else {
        ++u;
      }
    }
    if (!have) break;
    const uint32_t prev = atomicCAS(table + hs, kEmpty, c);
    if (prev == kEmpty || prev == c) {
      ties |= prev == c;
      have = false;
      ++u;
    } else {
      hs = (hs + 1) & hmask;
    }
  }
  return ties;
}

}  // namespace

// Equal scores of a row ([CSA-CPU] select_ratio4_topk refuses them): one of
// kTieParts CTAs of the row reads the row's scores and keeps those whose hash
// falls in its part of the slot range, in a hash set in shared memory;
// meeting an equal value flags the row.
__device__ void tie_part(const IndexArgs& a, int64_t row, int part, uint32_t* table) {
  __shared__ int s_tie;
  const int tid = threadIdx.x;
  const int n = static_cast<int>(row_limit(a, row));
  const int slots = a.hash_slots / kTieParts;
  const uint32_t hmask = static_cast<uint32_t>(slots - 1);
  const int shift = a.hash_log2 - kTiePartsLog2;  // low bits: the slot within the part
  for (int i = tid; i < slots; i += kTopkThreads) table[i] = kEmpty;
  if (tid == 0) s_tie = 0;
  __syncthreads();
  const float* sc = a.scores + row * a.R;
  int ties = 0;
  constexpr int kPer = 8;
  for (int r0 = 0; r0 < n; r0 += kPer * kTopkThreads) {
    uint32_t hc[kPer], h0[kPer];
    bool take[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = r0 + u * kTopkThreads + tid;
      const float v = i < n ? sc[i] : 0.0f;
      hc[u] = (v == 0.0f) ? 0u : __float_as_uint(v);
      const uint32_t h = (hc[u] * 0x9e3779b1u) >> (32 - a.hash_log2);
      take[u] = i < n && v == v && static_cast<int>(h >> shift) == part;
      h0[u] = h & hmask;
    }
    ties |= insert_scores<kPer>(table, hc, h0, take, hmask);
  }
  if (ties) s_tie = 1;
  __syncthreads();
  if (tid == 0 && s_tie) atomicOr(a.rowflags + row, static_cast<uint32_t>(kSelTie));
}

// Grid: one CTA per row.  The score kernel left the row's scores, the
// histogram of their rank keys' top 11 bits, and (with the tie kernel) the
// row's flags.
__device__ void topk_row(const IndexArgs& a, int64_t row, unsigned long long* sel) {
  __shared__ int s_hist[256];
  __shared__ uint32_t s_bin[2048];
  __shared__ int s_wsum[32];
  __shared__ int s_slot, s_bslot, s_need, s_cnt, s_digit, s_below;
  __shared__ int s_wt[32], s_wb[32];
  __shared__ unsigned long long s_prefix;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = static_cast<int>(row_limit(a, row));
  const int k = n < a.topk ? n : static_cast<int>(a.topk);
  if (tid == 0) {
    s_slot = 0;
    s_bslot = 0;
  }
  __syncthreads();
  // ---- the threshold bin: the smallest top-11-bit value D whose cumulative
  // count reaches k (every key with a smaller top is selected) ----
  const bool all = (k == n);
  int D = 2048, below = 0;
  if (!all) {
    for (int i = tid; i < 2048; i += kTopkThreads) s_bin[i] = a.hist[row * 2048 + i];
    __syncthreads();
    // two bins per thread, block-wide inclusive scan
    const int c0 = static_cast<int>(s_bin[2 * tid]), c1 = static_cast<int>(s_bin[2 * tid + 1]);
    int x = c0 + c1;
#pragma unroll
    for (int o = 1; o < 32; o *= 2) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int t = s_wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o *= 2) {
        const int y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      s_wsum[lane] = t;
    }
    __syncthreads();
    const int excl = (warp > 0 ? s_wsum[warp - 1] : 0) + x - (c0 + c1);
    if (excl < k && excl + c0 >= k) {
      s_digit = 2 * tid;
      s_below = excl;
    } else if (excl + c0 < k && excl + c0 + c1 >= k) {
      s_digit = 2 * tid + 1;
      s_below = excl + c0;
    }
    __syncthreads();
    D = s_digit;
    below = s_below;
  }
  // ---- one pass over the scores: tops below D are selected, the bin D
  // goes to the bucket ----
  const float* sc = a.scores + row * a.R;
  unsigned long long* bk = a.bucket + row * a.R;
  constexpr int kPer = 16;  // scores per thread per round, loaded before use
  for (int r0 = 0; r0 < n; r0 += kPer * kTopkThreads) {
    float f[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = r0 + u * kTopkThreads + tid;
      f[u] = i < n ? sc[i] : 0.0f;
    }
    // this warp's counts of selected and bucket entries, then one block scan
    // of them: every warp writes at its own offsets (no contended counters)
    int nt = 0, nb = 0;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = r0 + u * kTopkThreads + tid;
      const int top = i < n ? static_cast<int>(rank_key(f[u]) >> 21) : 4096;
      nt += __popc(__ballot_sync(0xffffffffu, all ? i < n : top < D));
      nb += __popc(__ballot_sync(0xffffffffu, !all && top == D));
    }
    if (lane == 0) {
      s_wt[warp] = nt;
      s_wb[warp] = nb;
    }
    __syncthreads();
    if (warp == 0) {
      int xt = s_wt[lane], xb = s_wb[lane];
      const int t0 = xt, b0 = xb;
#pragma unroll
      for (int o = 1; o < 32; o *= 2) {
        const int yt = __shfl_up_sync(0xffffffffu, xt, o), yb = __shfl_up_sync(0xffffffffu, xb, o);
        if (lane >= o) {
          xt += yt;
          xb += yb;
        }
      }
      s_wt[lane] = s_slot + xt - t0;  // exclusive offsets after the earlier rounds
      s_wb[lane] = s_bslot + xb - b0;
      if (lane == 31) {
        s_slot += xt;
        s_bslot += xb;
      }
    }
    __syncthreads();
    int ot = s_wt[warp], ob = s_wb[warp];
    const unsigned before_me = (1u << lane) - 1u;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = r0 + u * kTopkThreads + tid;
      uint32_t d = 0;
      int top = 4096;
      if (i < n) {
        d = rank_key(f[u]);
        top = static_cast<int>(d >> 21);
      }
      const bool take = all ? i < n : top < D;
      const bool inb = !all && top == D;
      const unsigned long long key =
          (static_cast<unsigned long long>(d) << 32) | static_cast<uint32_t>(i);
      const unsigned mt = __ballot_sync(0xffffffffu, take);
      const unsigned mb = __ballot_sync(0xffffffffu, inb);
      if (take)
        sel[ot + __popc(mt & before_me)] =
            a.ascending ? (static_cast<unsigned long long>(i) << 32) : key;
      if (inb) bk[ob + __popc(mb & before_me)] = key;
      ot += __popc(mt);
      ob += __popc(mb);
    }
    __syncthreads();
  }
  __syncthreads();
  // ---- inside the bucket: the (k - below)-th smallest (key, record) ----
  if (!all) {
    const int m = s_bslot;
    int need = k - below, cnt = m;
    unsigned long long prefix = static_cast<unsigned long long>(D) << 53;
    unsigned long long pmask = 0x7ffull << 53;
    unsigned long long thr = ~0ull;
    if (cnt > need) {
      // digits of the remaining 53 bits: 8 bits at a time, the last 5
      for (int shift = 45; shift >= 0; shift -= 8) {
        const int sh = shift < 0 ? 0 : shift;
        const unsigned dmask = 0xffu;
        prefix = bucket_pass(bk, m, prefix, pmask, sh, dmask, need, cnt, s_hist, &s_prefix,
                             &s_need, &s_cnt);
        pmask |= static_cast<unsigned long long>(dmask) << sh;
        if (cnt == need) break;
      }
      if (cnt > need) {  // bits 4..0
        prefix = bucket_pass(bk, m, prefix, pmask, 0, 0x1fu, need, cnt, s_hist, &s_prefix,
                             &s_need, &s_cnt);
        pmask |= 0x1full;
      }
      thr = prefix | ~pmask;  // every key matching the prefix
    }
    for (int i0 = 0; i0 < m; i0 += kTopkThreads) {
      const int i = i0 + tid;
      const bool take = i < m && bk[i] <= thr;
      const unsigned mt = __ballot_sync(0xffffffffu, take);
      int base = 0;
      if (lane == 0 && mt) base = atomicAdd(&s_slot, __popc(mt));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (take) {
        const unsigned long long v = bk[i];
        sel[base + __popc(mt & ((1u << lane) - 1u))] =
            a.ascending ? ((v & 0xffffffffull) << 32) : v;
      }
    }
    __syncthreads();
  }
  const int kcount = s_slot;  // == k
  int npad = 1;
  while (npad < kcount) npad <<= 1;
  for (int i = kcount + tid; i < npad; i += kTopkThreads) sel[i] = ~0ull;
  __syncthreads();
  if (kcount > 1) {
    if (npad >= 64) merge_sort(sel, sel + a.sel_slots, npad);
    else bitonic_sort(sel, npad);
  }
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
}

// Grid (1 + kTieParts, rows): CTA 0 of a row selects its top-k, CTAs 1..
// kTieParts check its scores for equal values, side by side.  The last CTA
// of the row to finish (a per-row counter) writes its status.
__global__ void __launch_bounds__(kTopkThreads) index_select_kernel(const IndexArgs a) {
  extern __shared__ __align__(16) unsigned long long dyn[];
  __shared__ int s_last;
  const int64_t row = blockIdx.y;
  pdl_wait();  // the scores, histogram and flags of the score kernel
  if (blockIdx.x == 0) topk_row(a, row, dyn);
  else tie_part(a, row, static_cast<int>(blockIdx.x) - 1, reinterpret_cast<uint32_t*>(dyn));
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's flags before its count
    s_last = atomicAdd(a.done + row, 1u) == kTieParts;
  }
  __syncthreads();
  if (s_last && threadIdx.x == 0) {
    __threadfence();
    const uint32_t f = atomicOr(a.rowflags + row, 0u);  // every CTA's flags are in
    if (a.row_status) a.row_status[row] = static_cast<uint8_t>(f);
    if (f && a.err_word) atomicOr(a.err_word, f << kSelErrShift);
  }
}

// ---- host side ---------------------------------------------------------------------------

// the selection and the merge sort's scratch
size_t index_topk_smem_bytes(int64_t sel_slots) { return static_cast<size_t>(sel_slots) * 16; }

size_t index_tie_smem_bytes(int hash_slots) {
  return static_cast<size_t>(hash_slots / kTieParts) * 4;
}

size_t index_score_smem_bytes(int64_t IH, int64_t ID, int64_t key_stride) {
  const int64_t NB = ID / 32;
  return static_cast<size_t>(IH * 16 + (IH * NB + 3) / 4 * 16 + (IH + 3) / 4 * 16 + IH * ID +
                             (IH * NB + 15) / 16 * 16 + kScoreRecords * key_stride);
}

template <int NB>
static int launch_index_t(const IndexArgs& a, cudaStream_t st) {
  constexpr int RPT = NB <= 4 ? 2 : 1;
  const unsigned qblocks = static_cast<unsigned>((a.rows * a.IH + 3) / 4);
  index_query_kernel<NB><<<qblocks, 128, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return -1;
  const size_t ss = index_score_smem_bytes(a.IH, a.ID, a.key_stride);
  if (cudaFuncSetAttribute(index_score_kernel<NB, RPT>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(ss)) != cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = st;
  cfg.gridDim = dim3(static_cast<unsigned>((a.R + kScoreRecords - 1) / kScoreRecords),
                     static_cast<unsigned>(a.rows));
  cfg.blockDim = dim3(kScoreRecords / RPT);
  cfg.dynamicSmemBytes = ss;
  mark_event(a.ev_before, st);
  if (cudaLaunchKernelEx(&cfg, index_score_kernel<NB, RPT>, a) != cudaSuccess) return -1;
  mark_event(a.ev_after, st);
  const size_t hs = index_tie_smem_bytes(a.hash_slots);
  const size_t ts = index_topk_smem_bytes(a.sel_slots);
  const size_t ds = hs > ts ? hs : ts;
  if (cudaFuncSetAttribute(index_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(ds)) != cudaSuccess)
    return -1;
  cfg.gridDim = dim3(1 + kTieParts, static_cast<unsigned>(a.rows));
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = ds;
  return cudaLaunchKernelEx(&cfg, index_select_kernel, a) == cudaSuccess ? 0 : -1;
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
