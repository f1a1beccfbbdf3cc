// k_compress.cu -- the CSA compression stages: ratio-4 attention records,
// ratio-4 index keys and ratio-128 attention records, produced from the
// compressor's value and gate rows and the carry of the open block.
//
// Semantics: onnx-runtime-ep-cpu src/kernels/compressed_sparse_attention.rs,
// compress_ratio4_stream / pool_ratio4_record / pool_ratio128_record /
// finalize_attention_record / finalize_index_record / apply_compressed_rope,
// and onnx-runtime-ep-cuda compressed_sparse_attention.rs,
// csa_ratio128_compress / csa_ratio4_main_compress / csa_ratio4_index_compress.
// A record is the per-dimension softmax pool of its candidates (score = gate
// + ape), rounded to bf16, RMS-normalised times a learned scale (bf16), its
// last n_rope dimensions rotated by the compressed RoPE at the block start
// (bf16 per component), then stored as FP8 blocks + a bf16 tail (attention)
// or Hadamard-transformed and stored as FP4 blocks (index keys).
//
// GB300 design.  The pages run one serial thread per sequence that walks the
// carry token by token.  A record depends only on the tokens of its block
// (ratio 4: and of the block before), each found either in this call's rows
// or in the carry, so every record a call closes is computed independently:
//  * compress_r4_kernel: one warp per record; the 8 warps of a CTA take 8
//    sequences at the same record index, so the RoPE rotation (one double
//    sine and cosine per pair) is evaluated once per CTA.  Lanes pool four
//    dimensions at a time from 16-byte loads of the 8 candidates' values and
//    scores, stage the pooled record in shared memory and finalize it there.
//  * compress_r128_kernel: one CTA per record, a thread per dimension pooling
//    the block's 128 tokens, then warp 0 finalizes.
//  * compress_carry_kernel: one thread per (sequence, source dimension)
//    writes the carry the stream holds after the call (runs after the record
//    kernel, which reads the carry of before the call).
// Bit-exactness: every step is the pages' binary32 operation, rounded once,
// in their order (no contraction; RMSNorm's square sum runs in dimension
// order in one lane).  The pool weight e^t is the correctly rounded binary32
// value: Tang's table-driven exponential (ACM TOMS 15(2), 1989) in
// float-float arithmetic, accepted by Ziv's rounding test and otherwise
// evaluated in double and rounded.
#include <cmath>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "codes.cuh"
#include "common.cuh"
#include "kernels.h"

namespace sa {

namespace {

// ---- e^t, t <= 0, correctly rounded to binary32 ------------------------------------------
//
// t = (256 m + j) ln2/256 + r with |r| <= ln2/512: e^t = 2^m 2^(j/256) e^r.
// 2^(j/256) is held as hi + lo (binary32 pair, ~2^-48 relative); r as
// r_hi + r_lo from a three-part ln2/256 (k L1 exact through an FMA residual);
// e^r - 1 - r = r^2/2 + r^3/6 (the r^4 term is below 2^-42).  The error of
// the float-float value is below 2^-38.4 of the result (the largest seen
// over a dense sample is 2^-39.3); it is rounded once and accepted when its
// residual stays 2^-37 clear of a rounding boundary, about 1 input in 8000
// falling back to the double evaluation.

struct ExpTable {
  float2 e[256];  // (hi, lo)
};

__host__ __device__ constexpr double exp_series(double x) {
  double term[32] = {};
  term[0] = 1.0;
  for (int n = 1; n < 32; ++n) term[n] = term[n - 1] * x / n;
  double s = 0.0;
  for (int n = 31; n >= 0; --n) s += term[n];  // smallest terms first
  return s;
}

__host__ __device__ constexpr ExpTable make_exp_table() {
  ExpTable t{};
  for (int j = 0; j < 256; ++j) {
    const double v = exp_series(j * (0.69314718055994530942 / 256.0));
    t.e[j].x = static_cast<float>(v);
    t.e[j].y = static_cast<float>(v - static_cast<double>(t.e[j].x));
  }
  return t;
}

__device__ const ExpTable g_exp_table = make_exp_table();

constexpr float kInvL = 0x1.7153b2p+8f;   // 256 / ln 2
constexpr float kL1 = 0x1.62e43p-9f;      // ln2/256 = kL1 + kL2 + O(2^-61)
constexpr float kL2 = -0x1.05c61p-37f;
constexpr float kSixth = 0x1.555556p-3f;
constexpr float kMargin = 0x1p-37f;
constexpr float kShifter = 0x1.8p23f;     // x + 1.5 * 2^23 rounds x to an integer

__device__ __noinline__ float exp_double(float t) {
  return static_cast<float>(exp(static_cast<double>(t)));
}

// The table evaluation, without branches (so that a caller's independent
// evaluations interleave).  The float-float value y1 + c is within 2^-37 of
// e^t / 2^m; rounding it with c raised and lowered by 2^-37 gives the same
// binary32 number exactly when that number is the correct rounding of e^t /
// 2^m (rounding is monotone), and then `ok` is true.  `ok` is false for t
// outside [-87, 0] (NaN and -inf included); the caller then takes
// exp_double(t).  (Kept scalar: a packed two-lane form of these steps gave
// certified results one ulp off under some instruction schedules.)
__device__ __forceinline__ float exp_table(float t, const float2* tab, bool& ok) {
  const float kb = __fmaf_rn(t, kInvL, kShifter);
  const uint32_t kbits = __float_as_uint(kb);  // 0x4b400000 + k, k = round(t 256 / ln 2)
  const float kf = __fsub_rn(kb, kShifter);
  // a = t - k L1 is exact (t and k L1 within a factor of two for k != 0)
  const float p1 = __fmul_rn(kf, kL1);
  const float e1 = __fmaf_rn(kf, kL1, -p1);
  const float a = __fsub_rn(t, p1);
  const float bsum = __fmaf_rn(kf, kL2, e1);  // r = a - bsum
  const float r = __fsub_rn(a, bsum);
  const float q = __fmul_rn(__fmul_rn(r, r), __fmaf_rn(r, kSixth, 0.5f));
  const float u = __fsub_rn(q, bsum);           // e^r = 1 + a + u
  const float2 T = tab[kbits & 255u];          // 2^(j/256), j = k mod 256
  const float p_hi = __fmul_rn(T.x, a);
  const float p_lo = __fmaf_rn(T.x, a, -p_hi);
  const float w = __fadd_rn(__fmaf_rn(T.x, u, p_lo), __fmaf_rn(T.y, a, T.y));
  const float y1 = __fadd_rn(T.x, p_hi);
  const float c = __fadd_rn(__fsub_rn(p_hi, __fsub_rn(y1, T.x)), w);  // exact low part + w
  const float ya = __fadd_rn(y1, __fadd_rn(c, kMargin));
  const float yb = __fadd_rn(y1, __fsub_rn(c, kMargin));
  ok = t >= -87.0f && t <= 0.0f && ya == yb;
  // times 2^m, m = floor(k / 256), on the exponent field (the result is normal)
  const uint32_t m23 = (kbits & ~255u) << 15;  // (k + 0x4b400000) / 256 * 2^23
  return __uint_as_float(__float_as_uint(ya) + m23 - (__float_as_uint(kShifter) << 15));
}

// ---- shared pieces -------------------------------------------------------------------------

constexpr int kR4Warps = 8;
constexpr int kTableFloats = 512 + 128 + 16;  // exp table, 64 (cos, sin) pairs, scales

__device__ __forceinline__ void load_exp_table(float2* tab) {
  for (int i = threadIdx.x; i < 256; i += blockDim.x) tab[i] = g_exp_table.e[i];
}

// The compressed RoPE rotation at block_start, one (cos, sin) per pair:
// frequency = base (1 - ramp) + (base / 16) ramp, ramp = clamp((i - 15) / 10),
// angle = position * frequency in binary32; sine and cosine of the binary32
// angle are evaluated in double and rounded.
__device__ void rope_rotation(const CompressArgs& a, int64_t block_start, float2* rot,
                              int lane) {
  const float p = __ll2float_rn(block_start);
  for (int i = lane; i < a.n_rope / 2; i += 32) {
    float ramp = __fdiv_rn(__fsub_rn(static_cast<float>(i), 15.0f), 10.0f);
    ramp = fminf(1.0f, fmaxf(0.0f, ramp));
    const float base = a.rope_base[i];
    const float f = __fadd_rn(__fmul_rn(base, __fsub_rn(1.0f, ramp)),
                              __fmul_rn(__fdiv_rn(base, 16.0f), ramp));
    const float ang = __fmul_rn(p, f);
    double s, c;
    sincos(static_cast<double>(ang), &s, &c);
    rot[i] = make_float2(static_cast<float>(c), static_cast<float>(s));
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Exponent of an FP8 block: the smallest e with amax / 2^e <= 448 (0 for
// amax 0), clamped to [-127, 127].  448 = 1.75 * 2^8.
__device__ __forceinline__ int fp8_block_exponent(float amax) {
  if (amax == 0.0f) return 0;
  const uint32_t u = __float_as_uint(amax);
  const bool above = (u & 0x7f800000u) && (u & 0x7fffffu) > 0x600000u;
  const int e = floor_log2(amax) - 8 + (above ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

__device__ __forceinline__ float e4m3_value(uint8_t c) {
  return __half2float(__half(__nv_cvt_fp8_to_halfraw(c, __NV_E4M3)));
}

// RMSNorm's scale of one pooled record rec[D]: the binary32 square sum in
// dimension order (a serial chain, one thread), then 1 / sqrt(sum / D +
// 1e-6).  Returns a negative value when the sum is not finite.
__device__ __forceinline__ float rms_inverse(const float* rec, int D) {
  float sum = 0.0f;
  for (int d = 0; d < D; d += 4) {
    const float4 x = *reinterpret_cast<const float4*>(rec + d);
    sum = __fadd_rn(sum, __fmul_rn(x.x, x.x));
    sum = __fadd_rn(sum, __fmul_rn(x.y, x.y));
    sum = __fadd_rn(sum, __fmul_rn(x.z, x.z));
    sum = __fadd_rn(sum, __fmul_rn(x.w, x.w));
  }
  if (!isfinite(sum)) return -1.0f;
  return __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(sum, static_cast<float>(D)), 1.0e-6f)));
}

// Finalize one record held (pooled, bf16-rounded) in shared memory rec[D],
// by one warp, given its RMSNorm scale: normalisation, RoPE, (index:
// Hadamard), validity, quantize, store.
template <int KIND>
__device__ void finalize_warp(const CompressArgs& a, float* rec, const float2* rot, int64_t b,
                              int64_t k, bool ok, float inv, int lane) {
  const int D = a.D;
  ok = ok && inv >= 0.0f;
  for (int d = lane; d < D; d += 32)
    rec[d] = round_bf16(__fmul_rn(__fmul_rn(rec[d], inv), __ldg(a.norm + d)));
  __syncwarp();
  for (int i = lane; i < a.n_rope / 2; i += 32) {
    const int d = D - a.n_rope + 2 * i;
    const float re = rec[d], im = rec[d + 1];
    const float2 cs = rot[i];
    rec[d] = round_bf16(__fsub_rn(__fmul_rn(re, cs.x), __fmul_rn(im, cs.y)));
    rec[d + 1] = round_bf16(__fadd_rn(__fmul_rn(re, cs.y), __fmul_rn(im, cs.x)));
  }
  __syncwarp();
  if (KIND == kCompressIndex) {
    // Walsh-Hadamard butterflies, span 1, 2, 4, ...: a level's pairs are disjoint
    for (int span = 1; span < D; span *= 2) {
      for (int q = lane; q < D / 2; q += 32) {
        const int i = (q / span) * 2 * span + (q % span);
        const float l = rec[i], r = rec[i + span];
        rec[i] = __fadd_rn(l, r);
        rec[i + span] = __fsub_rn(l, r);
      }
      __syncwarp();
    }
    const float hs = __frcp_rn(__fsqrt_rn(static_cast<float>(D)));
    for (int d = lane; d < D; d += 32) rec[d] = round_bf16(__fmul_rn(rec[d], hs));
    __syncwarp();
  }
  bool fin = true;
  for (int d = lane; d < D; d += 32) fin = fin && isfinite(rec[d]);
  ok = __all_sync(0xffffffffu, ok && fin);

  uint8_t* dst = a.records ? a.records + (b * a.rows + k) * a.record_stride : nullptr;
  float* lg = a.logical ? a.logical + (b * a.rows + k) * static_cast<int64_t>(D) : nullptr;
  if (!ok) {
    if (dst)
      for (int i = lane; i < a.width; i += 32) dst[i] = 0;
    if (lg)
      for (int d = lane; d < D; d += 32) lg[d] = 0.0f;
    if (lane == 0 && a.err_word) atomicOr(a.err_word, static_cast<uint32_t>(SA_ERRBIT_COMPRESS));
    return;
  }
  if (KIND == kCompressAttn) {
    const int nb = (D - a.n_rope) / 64;
    for (int blk = 0; blk < nb; ++blk) {
      const float x0 = rec[64 * blk + lane], x1 = rec[64 * blk + 32 + lane];
      const int e = fp8_block_exponent(warp_max(fmaxf(fabsf(x0), fabsf(x1))));
      const float sc = pow2f(-e);
      const uint8_t c0 = __nv_cvt_float_to_fp8(__fmul_rn(x0, sc), __NV_SATFINITE, __NV_E4M3);
      const uint8_t c1 = __nv_cvt_float_to_fp8(__fmul_rn(x1, sc), __NV_SATFINITE, __NV_E4M3);
      if (dst) {
        if (lane == 0) dst[blk * 65] = static_cast<uint8_t>(e + 127);
        dst[blk * 65 + 1 + lane] = c0;
        dst[blk * 65 + 33 + lane] = c1;
      }
      if (lg) {
        const float s = pow2f(e);
        lg[64 * blk + lane] = __fmul_rn(e4m3_value(c0), s);
        lg[64 * blk + 32 + lane] = __fmul_rn(e4m3_value(c1), s);
      }
    }
    for (int r = lane; r < a.n_rope; r += 32) {
      const float v = rec[D - a.n_rope + r];
      const uint32_t bits = __float_as_uint(v) >> 16;  // v is a bf16 value
      if (dst) {
        dst[nb * 65 + 2 * r] = static_cast<uint8_t>(bits & 0xffu);
        dst[nb * 65 + 2 * r + 1] = static_cast<uint8_t>(bits >> 8);
      }
      if (lg) lg[D - a.n_rope + r] = v;
    }
  } else {
    for (int blk = 0; blk < D / 32; ++blk) {
      const float x = rec[32 * blk + lane];
      const float amax = warp_max(fabsf(x));
      int e = -127;  // an all-zero block: scale byte 0
      if (amax > 0.0f) {
        e = floor_log2(amax) - 2;
        e = e < -127 ? -127 : (e > 127 ? 127 : e);
      }
      const float xs = __fmul_rn(x, pow2f(-e));
      const int tw = e2m1_twice(fabsf(xs));
      int code = e2m1_code(tw);
      if (xs < 0.0f && code) code |= 8;
      const int hi = __shfl_down_sync(0xffffffffu, code, 1);
      if (dst) {
        if (lane == 0) dst[blk * 17] = static_cast<uint8_t>(e + 127);
        if (!(lane & 1)) dst[blk * 17 + 1 + lane / 2] = static_cast<uint8_t>(code | (hi << 4));
      }
      if (lg) {
        const float mag = __fmul_rn(0.5f * static_cast<float>(tw), pow2f(e));
        lg[32 * blk + lane] = (code & 8) ? -mag : mag;
      }
    }
  }
}

// ---- ratio 4 -------------------------------------------------------------------------------

// The weights e^t[c] of 8 candidates (independent evaluations); the rare
// uncertified ones are redone in double (e^-inf = 0 there).
__device__ __forceinline__ void weights8(const float (&t)[8], const float2* tab, float (&w)[8]) {
  bool ok[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) w[c] = exp_table(t[c], tab, ok[c]);
  bool all = true;
#pragma unroll
  for (int c = 0; c < 8; ++c) all = all && ok[c];
  if (!all) {
#pragma unroll
    for (int c = 0; c < 8; ++c)
      if (!ok[c]) w[c] = exp_double(t[c]);
  }
}

// Adds 8 candidates' terms to the pool sums in candidate order: num += w v,
// den += w; a -inf score leaves num unchanged and adds w = 0 to den, which
// leaves it unchanged too (den is never -0).
__device__ __forceinline__ void pool_sums8(const float (&s)[8], const float (&v)[8],
                                           const float (&w)[8], float& num, float& den) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float n2 = __fadd_rn(num, __fmul_rn(w[c], v[c]));
    num = s[c] != SA_NEG_INF ? n2 : num;
    den = __fadd_rn(den, w[c]);
  }
}

// Softmax pool of one dimension over 8 candidates (scores s, values v), in
// candidate order, -inf scores left out; then bf16.
__device__ __forceinline__ float pool_dim8(const float (&s)[8], const float (&v)[8], bool& ok,
                                           const float2* tab) {
  float m = SA_NEG_INF;
#pragma unroll
  for (int c = 0; c < 8; ++c) m = fmaxf(m, s[c]);
  ok = ok && isfinite(m);
  float t[8], w[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) t[c] = __fsub_rn(s[c], m);
  weights8(t, tab, w);
  float num = 0.0f, den = 0.0f;
  pool_sums8(s, v, w, num, den);
  ok = ok && den != 0.0f && isfinite(den) && isfinite(num);
  return round_bf16(__fdiv_rn(num, den));
}

// One warp's pipeline stage: 8 candidates x (value, score) x 32 dimensions.
constexpr int kStageFloats = 8 * 2 * 32;

__device__ __forceinline__ void cp_async16(float* dst, const float* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)),
               "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}

// Record k's candidates (ratio 4): c < 4 the previous block's token 4k - 4 +
// c on source dims [0, D), c >= 4 the block's token 4k + c - 4 on [D, 2D).
// A token of this call is read from kv / gate and scores gate + its phase's
// ape row; an earlier one from its carry slot (the open block's tokens in
// slots 4 + phase, the closed block before it in slots 0..3), its score as
// stored; a token before position 0 is no candidate (value 0, score -inf).
//
// Each lane stages 4 of a stage's 128 16-byte chunks: chunk q = lane + 32 i
// holds candidate q / 16, array (q / 8) % 2 (0 value, 1 score), dims
// 4 (q % 8) .. + 3 of the stage's 32.  `src` are those chunks' sources at
// dim 0 (absent candidates read nothing: zero-filled), `ape_off` per
// candidate the row in the shared ape table whose dim d is added to the
// staged score: the phase row (+ D for c >= 4), a zero row (carry) or a
// -inf row (absent).
struct R4Plan {
  const float* src[4];
  uint32_t valid;  // bit i: chunk i has a source
  int ape_off[8];
};

__device__ __forceinline__ void r4_plan(const CompressArgs& a, int64_t b, int64_t k, int lane,
                                        R4Plan& pl) {
  const int64_t open_from = a.start - (a.start & 3);
  const int W = static_cast<int>(a.W);
  pl.valid = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) pl.src[i] = a.kv;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int64_t P = c < 4 ? 4 * k - 4 + c : 4 * k + c - 4;
    const int half = c < 4 ? 0 : a.D;
    const float* v = nullptr;
    const float* sc = nullptr;
    if (P < 0) {
      pl.ape_off[c] = 4 * W + a.D;  // the -inf row
    } else if (P >= a.start) {
      const int64_t off = (b * a.S + (P - a.start)) * a.W + half;
      v = a.kv + off;
      sc = a.gate + off;
      pl.ape_off[c] = static_cast<int>(P & 3) * W + half;
    } else {
      const int64_t slot = P >= open_from ? 4 + (P & 3) : (P & 3);
      v = a.carry + ((b * 8 + slot) * 2) * a.W + half;
      sc = v + a.W;
      pl.ape_off[c] = 4 * W;  // the zero row
    }
    // this lane's chunks of candidate c: i with 2 i + (lane >= 16) == c
    if ((c & 1) == (lane >= 16 ? 1 : 0) && v) {
      const int i = c >> 1;
      pl.src[i] = (((lane >> 3) & 1) ? sc : v) + 4 * (lane & 7);
      pl.valid |= 1u << i;
    }
  }
}

__device__ __forceinline__ void r4_stage(const CompressArgs& a, const R4Plan& pl, int it,
                                         float* stage, int lane) {
  const int dst = ((lane >= 16 ? 1 : 0) * 2 + ((lane >> 3) & 1)) * 32 + 4 * (lane & 7);
  const bool in_d = 32 * it + 4 * (lane & 7) < a.D;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool valid = ((pl.valid >> i) & 1u) && in_d;
    cp_async16(stage + dst + 128 * i, valid ? pl.src[i] + 32 * it : a.ape, valid);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int KIND>
__global__ void __launch_bounds__(kR4Warps * 32, 3) compress_r4_kernel(const CompressArgs a) {
  extern __shared__ __align__(16) float smem[];
  float2* tab = reinterpret_cast<float2*>(smem);
  float2* rot = reinterpret_cast<float2*>(smem + 512);
  float* invs = smem + 640;                    // [warps] RMSNorm scales
  float* ape_s = smem + kTableFloats;          // [4, W] phase rows, then D zeros, D -inf
  const int W = static_cast<int>(a.W);
  const int rs = a.D + 4;                      // record stride: the RMS lanes hit distinct banks
  float* recs = ape_s + 5 * W;                 // [warps, D + 4]
  float* stages = recs + kR4Warps * rs;        // [warps, 2, kStageFloats]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t k = a.k0 + blockIdx.x;
  load_exp_table(tab);
  for (int i = threadIdx.x; i < W; i += blockDim.x)  // 4 rows of W floats, as float4
    reinterpret_cast<float4*>(ape_s)[i] = __ldg(reinterpret_cast<const float4*>(a.ape) + i);
  for (int i = threadIdx.x; i < W; i += blockDim.x)
    ape_s[4 * W + i] = i < a.D ? 0.0f : SA_NEG_INF;
  __syncthreads();
  const int64_t b = static_cast<int64_t>(blockIdx.y) * kR4Warps + warp;
  const bool active = b < a.B;
  float* rec = recs + warp * rs;
  bool ok = true;
  if (active) {
    R4Plan pl;
    r4_plan(a, b, k, lane, pl);
    float* stg = stages + warp * 2 * kStageFloats;
    const int niter = (a.D + 31) / 32;
    r4_stage(a, pl, 0, stg, lane);
    for (int it = 0; it < niter; ++it) {
      if (it + 1 < niter)
        r4_stage(a, pl, it + 1, stg + ((it + 1) & 1) * kStageFloats, lane);
      else
        asm volatile("cp.async.commit_group;" ::: "memory");
      asm volatile("cp.async.wait_group 1;" ::: "memory");
      __syncwarp();
      const float* cur = stg + (it & 1) * kStageFloats;
      const int d = 32 * it + lane < a.D ? 32 * it + lane : a.D - 1;
      float s[8], v[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        v[c] = cur[(c * 2) * 32 + lane];
        s[c] = __fadd_rn(cur[(c * 2 + 1) * 32 + lane], ape_s[pl.ape_off[c] + d]);
      }
      const float out = pool_dim8(s, v, ok, tab);
      if (32 * it + lane < a.D) rec[32 * it + lane] = out;
      __syncwarp();  // every lane has read this stage before it is refilled
    }
  }
  __syncthreads();
  // off the pooling path, once per CTA: warp 0 the RoPE rotation of this
  // record index, warp 1 the RMSNorm square sums (serial chains, one lane per
  // record, in parallel)
  if (warp == 0) rope_rotation(a, 4 * k, rot, lane);
  if (warp == 1 && lane < kR4Warps && static_cast<int64_t>(blockIdx.y) * kR4Warps + lane < a.B)
    invs[lane] = rms_inverse(recs + lane * rs, a.D);
  __syncthreads();
  if (!active) return;
  ok = __all_sync(0xffffffffu, ok);
  finalize_warp<KIND>(a, rec, rot, b, k, ok, invs[warp], lane);
}

// ---- ratio 128 -----------------------------------------------------------------------------

__global__ void __launch_bounds__(1024) compress_r128_kernel(const CompressArgs a) {
  extern __shared__ __align__(16) float smem[];
  float2* tab = reinterpret_cast<float2*>(smem);
  float2* rot = reinterpret_cast<float2*>(smem + 512);
  float* inv = smem + 640;
  float* rec = smem + kTableFloats;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t k = a.k0 + blockIdx.x;
  const int64_t b = blockIdx.y;
  load_exp_table(tab);
  __syncthreads();
  // candidates: the block's tokens 128k + j; those of this call (j >=
  // first_new) from kv / gate + ape[j], the earlier ones from carry slot j
  const int64_t first_new = a.start - 128 * k;
  const int64_t W = a.W;
  const float* cy = a.carry + b * 128 * 2 * W;
  const int64_t row0 = b * a.S - a.start + 128 * k;  // row of token 128k (may be < b S)
  bool ok = true;
  for (int d = threadIdx.x; d < a.D; d += blockDim.x) {
    auto score = [&](int j) {
      return j >= first_new ? __fadd_rn(__ldg(a.gate + (row0 + j) * W + d),
                                        __ldg(a.ape + j * W + d))
                            : cy[(2 * j + 1) * W + d];
    };
    auto value = [&](int j) {
      return j >= first_new ? __ldg(a.kv + (row0 + j) * W + d) : cy[(2 * j) * W + d];
    };
    float m = SA_NEG_INF;
#pragma unroll 8
    for (int j = 0; j < 128; ++j) m = fmaxf(m, score(j));
    ok = ok && isfinite(m);
    float num = 0.0f, den = 0.0f;
    for (int j0 = 0; j0 < 128; j0 += 8) {
      float sc[8], v[8], t[8], w[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        sc[c] = score(j0 + c);
        v[c] = value(j0 + c);
        t[c] = __fsub_rn(sc[c], m);
      }
      weights8(t, tab, w);
      pool_sums8(sc, v, w, num, den);
    }
    ok = ok && den != 0.0f && isfinite(den) && isfinite(num);
    rec[d] = round_bf16(__fdiv_rn(num, den));
  }
  if (warp == 0) rope_rotation(a, 128 * k, rot, lane);
  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  if (warp != 0) return;
  if (lane == 0) *inv = rms_inverse(rec, a.D);
  __syncwarp();
  finalize_warp<kCompressAttn>(a, rec, rot, b, k, ok, *inv, lane);
}

// ---- the carry after the call --------------------------------------------------------------

__device__ __forceinline__ void carry_from_row(const CompressArgs& a, int64_t b, int64_t q,
                                               int64_t d, float& v, float& s) {
  const int64_t off = (b * a.S + (q - a.start)) * a.W + d;
  v = __ldg(a.kv + off);
  s = __fadd_rn(__ldg(a.gate + off), __ldg(a.ape + (q % a.ratio) * a.W + d));
}

__global__ void __launch_bounds__(256) compress_carry_kernel(const CompressArgs a) {
  const int64_t d = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t b = blockIdx.y;
  if (d >= a.W) return;
  const int64_t W = a.W;
  float* cy = a.carry + b * (a.ratio == 128 ? 128 : 8) * 2 * W;
  const int64_t open_end = a.total - a.total % a.ratio;
  if (a.ratio == 128) {
    for (int j = 0; j < 128; ++j) {
      const int64_t q = open_end + j;
      float v = 0.0f, s = SA_NEG_INF;
      if (q < a.total) {
        if (q < a.start) continue;  // already in its slot
        carry_from_row(a, b, q, d, v, s);
      }
      cy[(2 * j) * W + d] = v;
      cy[(2 * j + 1) * W + d] = s;
    }
    return;
  }
  const int64_t open_from = a.start - a.start % 4;
  float pv[4], ps[4];
  bool pw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // previous-block slots: read everything first
    pv[i] = 0.0f;
    ps[i] = SA_NEG_INF;
    pw[i] = true;
    if (open_end == 0) continue;
    const int64_t q = open_end - 4 + i;
    if (q >= a.start) {
      carry_from_row(a, b, q, d, pv[i], ps[i]);
    } else if (q >= open_from) {  // the block was open before the call: it moves
      pv[i] = cy[((4 + i) * 2) * W + d];
      ps[i] = cy[((4 + i) * 2 + 1) * W + d];
    } else {
      pw[i] = false;  // the closed block before the call stays
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (!pw[i]) continue;
    cy[(i * 2) * W + d] = pv[i];
    cy[(i * 2 + 1) * W + d] = ps[i];
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t q = open_end + i;
    float v = 0.0f, s = SA_NEG_INF;
    if (q < a.total) {
      if (q < a.start) continue;
      carry_from_row(a, b, q, d, v, s);
    }
    cy[((4 + i) * 2) * W + d] = v;
    cy[((4 + i) * 2 + 1) * W + d] = s;
  }
}

__global__ void pool_weight_kernel(const float* t, float* w, int64_t n) {
  __shared__ float2 tab[256];
  load_exp_table(tab);
  __syncthreads();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    const float x = __ldg(t + i);
    bool ok;
    const float y = exp_table(x, tab, ok);
    w[i] = ok ? y : exp_double(x);
  }
}

}  // namespace

// ---- host side ------------------------------------------------------------------------------

size_t compress_smem_bytes(int ratio, int64_t D) {
  if (ratio == 4)  // tables, ape rows (4 x 2D + a zero and a -inf row), records, stages
    return static_cast<size_t>(kTableFloats + 10 * D + kR4Warps * (D + 4) +
                               kR4Warps * 2 * kStageFloats) * sizeof(float);
  return static_cast<size_t>(kTableFloats + D) * sizeof(float);
}

template <typename K>
static int set_smem(K kernel, size_t smem) {
  if (smem <= 48 * 1024) return 0;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(smem)) == cudaSuccess
             ? 0
             : -1;
}

int launch_compress(const CompressArgs& a, cudaStream_t st) {
  if (a.nk > 0) {
    const size_t smem = compress_smem_bytes(static_cast<int>(a.ratio), a.D);
    mark_event(a.ev_before, st);
    if (a.ratio == 4) {
      const dim3 grid(static_cast<unsigned>(a.nk),
                      static_cast<unsigned>((a.B + kR4Warps - 1) / kR4Warps));
      if (a.kind == kCompressAttn) {
        if (set_smem(compress_r4_kernel<kCompressAttn>, smem) != 0) return -1;
        compress_r4_kernel<kCompressAttn><<<grid, kR4Warps * 32, smem, st>>>(a);
      } else {
        if (set_smem(compress_r4_kernel<kCompressIndex>, smem) != 0) return -1;
        compress_r4_kernel<kCompressIndex><<<grid, kR4Warps * 32, smem, st>>>(a);
      }
    } else {
      const int threads = static_cast<int>((a.D + 31) / 32 * 32);
      if (set_smem(compress_r128_kernel, smem) != 0) return -1;
      compress_r128_kernel<<<dim3(static_cast<unsigned>(a.nk), static_cast<unsigned>(a.B)),
                             threads, smem, st>>>(a);
    }
    if (cudaGetLastError() != cudaSuccess) return -1;
    mark_event(a.ev_after, st);
  }
  compress_carry_kernel<<<dim3(static_cast<unsigned>((a.W + 255) / 256),
                               static_cast<unsigned>(a.B)),
                          256, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_pool_weight(const float* t, float* w, int64_t n, cudaStream_t st) {
  if (n <= 0) return 0;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  pool_weight_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(t, w, n);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace sa
