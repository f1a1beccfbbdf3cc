// k_fp8.cu -- selected-token decode over a hybrid FP8 latent cache (MQA).
//
// Semantics: the hybrid record of the compressed sparse attention pages
// (onnx-runtime-ep-cpu compressed_sparse_attention.rs, `CacheFormat::
// Fp8E4m3Block64` and `dequantize_cache`): per record, blocks of [E8M0 scale
// byte, 64 E4M3FN codes] for the non-RoPE dims, then the RoPE dims as
// little-endian bf16; value = e4m3(code) * 2^(scale - 127).  The attention is
// IndexShare's `index_share_row` over the candidate set planned by k_plan.cu
// (a dense window of recent tokens united with the selected indices, as in
// `csa_ratio128_sink_attention`), with K and V both the decoded record.
//
// GB300 design (tensor-core tile, heads split across CTAs):
//  * CTA = (batch, block of 32 query heads, chunk of 16-key tiles); 8 warps =
//    2 head groups of 16 x 4 quarters of the 576 dims.  The 32 x 576 fp32
//    output lives in registers (72 accumulators per thread).
//  * Each tile's raw records arrive by 8-byte cp.async into a double-buffered
//    staging area while the previous tile computes; threads then decode them
//    exactly to bf16 (E4M3 pairs -> f16x2 -> times the power-of-two scale) into
//    a padded shared tile; masked records are zero rows.
//  * Scores: each warp computes S over its dim quarter (m16n8k16, heads as M,
//    keys as N); the four partial S tiles of a head group are summed through
//    shared memory and every warp of the group runs the same online softmax.
//    Then each warp does O += P . V over its quarter, P taken straight from
//    the S accumulators, V through ldmatrix.trans.
//  * Key chunks merge in the fixed-order combine kernel.
#include "e4m3.cuh"
#include "gather_common.cuh"


namespace sa {

namespace {

constexpr int kD = 576, kNope = 512, kRope = 64;
constexpr int kRec = kNope / 64 * 65 + kRope * 2;   // 648 bytes
constexpr int kHeads = 32;                           // query heads per CTA
constexpr int kQuarter = kD / 4;                     // 144 dims per warp
constexpr int kNT = kQuarter / 8;                    // 18 n-tiles of output dims
constexpr int kKS = kQuarter / 16;                   // 9 k-steps per quarter
constexpr int kRowStride = kD * 2 + 16;              // padded bf16 row (1168 B)
constexpr int kRawStage = 16 * kRec;                 // 10368 B
constexpr int kMaxChunkTiles = 64;

// shared-memory layout (bytes)
constexpr int kOffQ = 0;                                   // [32][kRowStride]
constexpr int kOffDec = kOffQ + kHeads * kRowStride;       // [16][kRowStride]
constexpr int kOffRaw = kOffDec + 16 * kRowStride;         // [2][kRawStage]
constexpr int kOffX = kOffRaw + 2 * kRawStage;             // [2 hg][4 q][8 values][32 lanes] f32
constexpr int kOffPos = kOffX + 2 * 4 * 32 * 8 * 4;        // [kMaxChunkTiles * 16] i32
constexpr int kSmem = kOffPos + kMaxChunkTiles * 16 * 4;

__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// E8M0 scale byte -> 2^(b - 127) (255 is NaN in the format; it maps to NaN).
__device__ __forceinline__ float e8m0_to_float(uint32_t b) {
  if (b == 255u) return __int_as_float(0x7fc00000);
  if (b == 0u) return __int_as_float(0x00400000);  // 2^-127, a subnormal float
  return __int_as_float(static_cast<int>(b) << 23);
}

// The decoded tile keeps 16-byte chunk c of a row at chunk c ^ ((c >> 3) & 7)
// (within its group of eight): the decode's stores, 16 lanes of one record
// writing chunks 4p + i, then fall on distinct bank groups, while ldmatrix,
// 8 rows at one chunk, stays conflict-free through the 73-chunk row stride.
__device__ __forceinline__ int dec_chunk(int c) { return c ^ ((c >> 3) & 7); }

}  // namespace

size_t fp8_smem_bytes() { return kSmem; }
int fp8_chunk_tiles_max() { return kMaxChunkTiles; }

// One CTA per (unit = (batch, query position), head block, key chunk).
// grid = B * Sq * (Hq/32) * splits.
__global__ void __launch_bounds__(256, 2) fp8_decode_kernel(GatherArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int hg = warp >> 2;  // head group (16 heads)
  const int qd = warp & 3;   // dim quarter
  const int64_t nhb = a.Hq / kHeads;
  const int64_t split = blockIdx.x % a.splits;
  const int64_t hb = (blockIdx.x / a.splits) % nhb;
  const int64_t unit = blockIdx.x / (a.splits * nhb);  // b * Sq + i
  const int64_t b = unit / a.Sq, qi = unit % a.Sq;
  const int64_t tiles = a.tiles_per_unit;
  const int64_t t0 = split * a.chunk;
  int64_t nt = tiles - t0;
  if (nt > a.chunk) nt = a.chunk;
  if (nt < 0) nt = 0;

  unsigned char* sq = smem + kOffQ;
  unsigned char* sdec = smem + kOffDec;
  unsigned char* sraw = smem + kOffRaw;
  float* sx = reinterpret_cast<float*>(smem + kOffX);
  int32_t* spos = reinterpret_cast<int32_t*>(smem + kOffPos);

  // ---- positions of this chunk, Q of this head block ----------------------------------
  const int32_t* prow = a.pos + unit * a.n_cand_pad + t0 * 16;  // one index row per unit
  for (int64_t e = tid; e < nt * 16; e += 256) spos[e] = __ldg(prow + e);
  {
    const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(a.q);
    for (int e = tid; e < kHeads * kD * 2 / 16; e += 256) {
      const int h = e / (kD * 2 / 16), c = e % (kD * 2 / 16);
      const uint4* qsrc = reinterpret_cast<const uint4*>(
          qb + ((b * a.Hq + hb * kHeads + h) * a.Sq + qi) * kD);
      *reinterpret_cast<uint4*>(sq + h * kRowStride + c * 16) = __ldg(qsrc + c);
    }
  }
  __syncthreads();

  const char* recs = static_cast<const char*>(a.k) + (b * a.Hkv) * a.T * a.record_stride;
  auto issue_raw = [&](int64_t t, int stage) {
    const uint32_t dst0 = smem_u32(sraw + stage * kRawStage);
    for (int w = tid; w < 16 * (kRec / 8); w += 256) {
      const int r = w / (kRec / 8), j = w % (kRec / 8);
      const int32_t p = spos[t * 16 + r];
      if (p >= 0) cp_async8(dst0 + r * kRec + j * 8, recs + static_cast<int64_t>(p) * a.record_stride + j * 8);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  // ---- per-thread state ---------------------------------------------------------------
  float o[kNT][4];
#pragma unroll
  for (int n = 0; n < kNT; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
  float m_run[2] = {SA_NEG_INF, SA_NEG_INF}, l_run[2] = {0.f, 0.f};
  const float sl2 = a.scale_log2;
  const float cap = a.softcap, inv_cap = a.inv_softcap;

  if (nt > 0) issue_raw(0, 0);
  for (int64_t t = 0; t < nt; ++t) {
    if (t + 1 < nt) issue_raw(t + 1, static_cast<int>((t + 1) & 1));
    else asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncthreads();
    // ---- decode tile t: thread (record r, part p) --------------------------------------
    {
      const int r = tid >> 4, p = tid & 15;
      const bool valid = spos[t * 16 + r] >= 0;
      const unsigned char* raw = sraw + (t & 1) * kRawStage + r * kRec;
      unsigned char* drow = sdec + r * kRowStride;
      // FP8: block k = p/2, codes [32h, 32h+32) of the block
      const int k = p >> 1, h = p & 1;
      uint32_t outw[16];
      if (valid) {
        const float sc = e8m0_to_float(raw[65 * k]);
        const unsigned char* codes = raw + 65 * k + 1 + 32 * h;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint16_t two = static_cast<uint16_t>(codes[2 * i] | (codes[2 * i + 1] << 8));
          const float2 f = e4m3x2_to_float2(two);
          outw[i] = pack2<__nv_bfloat16>(f.x * sc, f.y * sc);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) outw[i] = 0u;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<uint4*>(drow + dec_chunk(p * 4 + i) * 16) =
            make_uint4(outw[4 * i], outw[4 * i + 1], outw[4 * i + 2], outw[4 * i + 3]);
      // RoPE tail: 64 little-endian bf16 = 128 bytes, two threads per record
      if (p < 2) {
        const uint2* rsrc = reinterpret_cast<const uint2*>(raw + kNope / 64 * 65 + 64 * p);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint2 lo = valid ? rsrc[2 * i] : make_uint2(0, 0);
          const uint2 hi = valid ? rsrc[2 * i + 1] : make_uint2(0, 0);
          *reinterpret_cast<uint4*>(drow + dec_chunk(kNope / 8 + 4 * p + i) * 16) =
              make_uint4(lo.x, lo.y, hi.x, hi.y);
        }
      }
    }
    __syncthreads();

    // ---- S partial over this warp's dim quarter: 16 heads x 16 keys ------------------------
    float s[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
    {
      const uint32_t qa = smem_u32(sq) + (hg * 16 + (lane & 15)) * kRowStride +
                          (qd * kQuarter + 8 * (lane >> 4)) * 2;
      const int jm = lane >> 3, rr = lane & 7;
      const uint32_t krow = smem_u32(sdec) + (rr + 8 * (jm >> 1)) * kRowStride;
      const int kc0 = (qd * kQuarter) / 8 + (jm & 1);  // this lane's chunk at k-step 0
#pragma unroll
      for (int kk = 0; kk < kKS; ++kk) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(qa + kk * 32, a0, a1, a2, a3);
        ldsm_x4(krow + dec_chunk(kc0 + 2 * kk) * 16, b0, b1, b2, b3);
        mma16816<__nv_bfloat16>(s[0], a0, a1, a2, a3, b0, b1);
        mma16816<__nv_bfloat16>(s[1], a0, a1, a2, a3, b2, b3);
      }
    }
    // sum the four quarters' partial scores of this head group; sx is
    // [hg][quarter][value][lane] so that every access is one word per lane
    float* myx = sx + (hg * 4 + qd) * 8 * 32 + lane;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) myx[(n * 4 + e) * 32] = s[n][e];
    named_bar(1 + hg, 128);
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) acc += sx[((hg * 4 + q) * 8 + n * 4 + e) * 32 + lane];
        s[n][e] = acc;
      }
    // ---- online softmax (rows = heads gid, gid+8; columns = keys) -------------------------
    const int32_t* tp = spos + t * 16;
    float mx[2] = {SA_NEG_INF, SA_NEG_INF};
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      const bool v0 = tp[n * 8 + 2 * tig] >= 0, v1 = tp[n * 8 + 2 * tig + 1] >= 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = s[n][e];
        if (cap != 0.f) x = cap * tanh_fast(x * (sl2 * (1.0f / kLog2e)) * inv_cap) * kLog2e;
        else x = x * sl2;
        if (a.bias) {  // [IS] bias_at, keyed by the key's cache position
          const int32_t j = tp[n * 8 + 2 * tig + (e & 1)];
          const int64_t h = hb * kHeads + hg * 16 + gid + 8 * (e >> 1);
          if (j >= 0) x += kLog2e * bias_term(a, b, h, qi, j);
        }
        s[n][e] = ((e & 1) ? v1 : v0) ? x : SA_NEG_INF;
      }
      mx[0] = fmaxf(mx[0], fmaxf(s[n][0], s[n][1]));
      mx[1] = fmaxf(mx[1], fmaxf(s[n][2], s[n][3]));
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 1));
      mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 2));
    }
    // Lazy running maximum: raised only when the tile's maximum exceeds it by
    // more than 2^8 (probabilities up to 256 are exact enough in bf16), so the
    // O accumulators are rescaled only on such tiles.
    float mu[2], al[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      al[j] = 1.0f;
      if (mx[j] > m_run[j] + 8.0f) {  // also the first finite maximum
        al[j] = ex2(m_run[j] - mx[j]);
        m_run[j] = mx[j];
      }
      mu[j] = (m_run[j] == SA_NEG_INF) ? 0.f : m_run[j];
    }
    const bool rescale = __any_sync(0xffffffffu, al[0] != 1.0f || al[1] != 1.0f);
    float ps[2] = {0.f, 0.f};
    uint32_t pa[4];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      const float p0 = ex2(s[n][0] - mu[0]), p1 = ex2(s[n][1] - mu[0]);
      const float p2 = ex2(s[n][2] - mu[1]), p3 = ex2(s[n][3] - mu[1]);
      ps[0] += p0 + p1;
      ps[1] += p2 + p3;
      pa[2 * n] = pack2<__nv_bfloat16>(p0, p1);      // rows gid, keys 8n + 2tig..
      pa[2 * n + 1] = pack2<__nv_bfloat16>(p2, p3);  // rows gid + 8
    }
    l_run[0] = l_run[0] * al[0] + ps[0];
    l_run[1] = l_run[1] * al[1] + ps[1];
    if (rescale) {
#pragma unroll
      for (int n = 0; n < kNT; ++n) {
        o[n][0] *= al[0];
        o[n][1] *= al[0];
        o[n][2] *= al[1];
        o[n][3] *= al[1];
      }
    }
    // ---- O += P . V over this warp's quarter --------------------------------------------
    {
      const int jm = lane >> 3, rr = lane & 7;
      const uint32_t vrow = smem_u32(sdec) + (rr + 8 * (jm & 1)) * kRowStride;
      const int vc0 = (qd * kQuarter) / 8 + (jm >> 1);
#pragma unroll
      for (int n2 = 0; n2 < kNT / 2; ++n2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vrow + dec_chunk(vc0 + 2 * n2) * 16, b0, b1, b2, b3);
        mma16816<__nv_bfloat16>(o[2 * n2], pa[0], pa[1], pa[2], pa[3], b0, b1);
        mma16816<__nv_bfloat16>(o[2 * n2 + 1], pa[0], pa[1], pa[2], pa[3], b2, b3);
      }
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");

  // ---- row sums, then the chunk's partial (or the final output) ---------------------------
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 1);
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 2);
  }
  const int h_lo = static_cast<int>(hb * kHeads + hg * 16 + gid);  // rows gid and gid + 8
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int h = h_lo + 8 * j;
    if (a.splits == 1) {
      float L = l_run[j];
      const float M = m_run[j];
      if (a.sink && M != SA_NEG_INF) L += ex2(a.sink[h] * kLog2e - M);
      const float inv = (M == SA_NEG_INF || L == 0.f) ? 0.f : 1.0f / L;
      __nv_bfloat16* yp =
          static_cast<__nv_bfloat16*>(a.y) + ((b * a.Hq + h) * a.Sq + qi) * kD + qd * kQuarter;
#pragma unroll
      for (int n = 0; n < kNT; ++n) {
        *reinterpret_cast<uint32_t*>(yp + n * 8 + 2 * tig) =
            pack2<__nv_bfloat16>(o[n][2 * j] * inv, o[n][2 * j + 1] * inv);
      }
    } else {
      const int64_t pidx = (unit * a.splits + split) * a.Hq + h;  // (unit, split, head)
      float* po = a.part_o + pidx * kD + qd * kQuarter;
#pragma unroll
      for (int n = 0; n < kNT; ++n)
        *reinterpret_cast<float2*>(po + n * 8 + 2 * tig) = make_float2(o[n][2 * j], o[n][2 * j + 1]);
      if (qd == 0 && tig == 0) {
        a.part_ml[2 * pidx] = m_run[j];
        a.part_ml[2 * pidx + 1] = l_run[j];
      }
    }
  }
}

int launch_fp8_decode(const GatherArgs& a, cudaStream_t st) {
  if (cudaFuncSetAttribute(fp8_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmem) != cudaSuccess)
    return -1;
  const int64_t grid = a.B * a.Sq * (a.Hq / kHeads) * a.splits;
  fp8_decode_kernel<<<static_cast<unsigned>(grid), 256, kSmem, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace sa
