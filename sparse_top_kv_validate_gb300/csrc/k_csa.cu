// k_csa.cu -- compressed sparse attention (ratio 4) in the pages' own form:
// a separate window store of recent tokens plus the selected compressed
// records, a bias keyed by the candidate slot, a per-head sink.
//
// Semantics: onnx-runtime-ep-cpu src/kernels/compressed_sparse_attention.rs,
// ratio4_attention (and its call in execute_ratio4); onnx-runtime-ep-cuda
// compressed_sparse_attention.rs, csa_ratio4_sink_attention.  For the query
// at position p = total - S + s: dense slots c < dense (128, or min(L, 128)
// when the query block starts at position 0) are the window rows at
// positions max(total - L, p + 1 - 128) + c that are <= p and stored; slot
// dense + k is selected record k (skipped when negative or at or past
// total / 4 records); score = scale * q . row + bias(b, h, s, slot); softmax
// with exp(sink[h] - max) added to the denominator; y = sum p * row (K = V).
//
// GB300 design:
//  * csa_assemble_kernel: one warp per (query, four candidate slots) writes
//    the slots' rows as bf16 into a candidate buffer (window rows converted,
//    hybrid FP8 records decoded exactly: 583-byte records are not even 2-byte
//    aligned, so a warp stages each one in shared memory -- 16-byte loads for
//    its aligned interior, byte loads for the ends, the four records' loads in
//    flight together -- and decodes it from there), with a validity byte; the
//    rows stay in L2 for the attention kernel.
//  * bf16 queries in blocks of 128 heads (D 512): the tcgen05 attention kernel
//    of k_fp8_tc.cu in its 512-dim geometry reads the assembled rows by TMA in
//    128-slot tiles (two CTAs per head block, each owning 256 output dims;
//    the validity bytes mask the slots; the slot bias is added to the log2
//    logits in tensor memory before the maximum is taken).
//  * otherwise csa_attn_kernel: CTA = (query, block of 32 heads, key split); 8 warps =
//    2 head groups of 16 x 4 quarters of the dims.  Candidate tiles of 16 rows
//    arrive by 16-byte cp.async, double-buffered; S over each warp's quarter
//    on the m16n8k16 tensor-core MMA (heads as M, keys as N), the quarters
//    summed through shared memory, an online softmax in the log2 domain with
//    the slot bias, then O += P . V from the same rows.
//  * csa_combine_kernel merges key splits in split order (deterministic).
#include "e4m3.cuh"
#include "gather_common.cuh"


namespace sa {

namespace {

constexpr int kHeads = 32;  // query heads per attention CTA
constexpr int kWindow = 128;

template <int D>
struct CsaGeo {
  static constexpr int kQuarter = D / 4;            // dims per warp
  static constexpr int kNT = kQuarter / 8;          // output n-tiles per warp
  static constexpr int kKS = kQuarter / 16;         // k-steps per warp
  static constexpr int kRowStride = D * 2 + 16;     // padded bf16 row: conflict-free ldmatrix
  static constexpr int kOffQ = 0;                   // [32][kRowStride]
  static constexpr int kOffRows = kOffQ + kHeads * kRowStride;  // [2][16][kRowStride]
  static constexpr int kOffX = kOffRows + 2 * 16 * kRowStride;  // [2 hg][4 q][8][32] f32
  static constexpr int kOffValid = kOffX + 2 * 4 * 8 * 32 * 4;  // [2][16] u8
  static constexpr int kSmem = kOffValid + 64;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Two E4M3FN codes (low byte first) -> two floats, exactly.
__device__ __forceinline__ float2 e4m3_pair(uint32_t two) { return e4m3x2_to_float2(two); }

// E8M0 scale byte -> 2^(b - 127) (0xFF, NaN in the format, maps to NaN).
__device__ __forceinline__ float e8m0(uint32_t b) {
  if (b == 255u) return __int_as_float(0x7fc00000);
  if (b == 0u) return __int_as_float(0x00400000);  // 2^-127
  return __int_as_float(static_cast<int>(b) << 23);
}

// Candidate geometry of query row (b, s).
struct CsaRow {
  int64_t pos, base, dense_start;
  int dense;
};

__device__ __forceinline__ CsaRow csa_row(const CsaArgs& a, int64_t s) {
  CsaRow r;
  r.pos = a.total - a.S + s;
  r.base = a.total - a.L;
  int64_t w = r.pos + 1 - kWindow;
  if (w < 0) w = 0;
  r.dense_start = r.base > w ? r.base : w;
  r.dense = a.dense;
  return r;
}

}  // namespace

// ---- candidate rows ------------------------------------------------------------------------
// grid (c_pad / 8, units), 8 warps: warp w writes candidate slot blockIdx.x * 8 + w.
// Each warp assembles kSlotsPerWarp consecutive candidate slots.  It first
// stages every selected record among them in shared memory -- the 16-byte
// aligned interior with vector loads, the unaligned head and tail (under 16
// bytes each) with byte loads, all issued together and none outside the
// record; byte j of a record sits at stage[(address % 16) + j] -- and then
// decodes and writes the slots in turn.
constexpr int kSlotsPerWarp = 4;

// Shared-memory bytes a warp stages one record in: the record and up to 15
// bytes before it, rounded to 16 (dynamic: the CTA then holds 8 warps x 4).
__host__ __device__ __forceinline__ int csa_stage_bytes(int64_t D, int64_t n_rope) {
  const int nbytes = static_cast<int>((D - n_rope) / 64 * 65 + 2 * n_rope);
  return (15 + nbytes + 15) / 16 * 16;
}

template <int D>
__global__ void __launch_bounds__(256) csa_assemble_kernel(const CsaArgs a) {
  extern __shared__ __align__(16) uint8_t stage_all[];
  const int lane = threadIdx.x & 31;
  const int kStageBytes = csa_stage_bytes(D, a.n_rope);
  uint8_t* stage = stage_all + (threadIdx.x >> 5) * kSlotsPerWarp * kStageBytes;
  const int64_t c0 = (static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * kSlotsPerWarp;
  const int64_t unit = blockIdx.y;  // b * S + s
  const int64_t b = unit / a.S, s = unit % a.S;
  const CsaRow r = csa_row(a, s);
  const int nb = static_cast<int>((D - a.n_rope) / 64);
  const int nbytes = 65 * nb + 2 * static_cast<int>(a.n_rope);
  // the slots' selected records (lane i < kSlotsPerWarp reads slot c0 + i's)
  int32_t mine = -1;
  if (lane < kSlotsPerWarp) {
    const int64_t c = c0 + lane;
    if (c < a.c_pad && c >= r.dense && c < r.dense + a.topk)
      mine = __ldg(a.selected + unit * a.topk + (c - r.dense));
  }
  // phase 1: stage every valid record
#pragma unroll
  for (int i = 0; i < kSlotsPerWarp; ++i) {
    const int32_t rec = __shfl_sync(0xffffffffu, mine, i);
    if (rec < 0 || rec >= a.valid_records) continue;
    const uint8_t* src = a.records + (b * a.R + rec) * a.record_stride;
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), s1 = s0 + nbytes;
    const uintptr_t a0 = (s0 + 15) & ~static_cast<uintptr_t>(15);
    const uintptr_t a1 = s1 & ~static_cast<uintptr_t>(15);
    uint8_t* st = stage + i * kStageBytes + (s0 & 15);
    const int head = static_cast<int>((a0 < s1 ? a0 : s1) - s0);   // bytes before the interior
    const int body = a1 > a0 ? static_cast<int>((a1 - a0) / 16) : 0;  // 16-byte words
    const int tail0 = head + 16 * body;                              // first tail byte
    for (int w = lane; w < body; w += 32)
      *reinterpret_cast<uint4*>(st + head + 16 * w) = __ldg(reinterpret_cast<const uint4*>(a0) + w);
    if (lane < head) st[lane] = __ldg(src + lane);
    if (tail0 + lane < nbytes) st[tail0 + lane] = __ldg(src + tail0 + lane);
  }
  __syncwarp();
  // phase 2: each slot's bf16 row and validity byte
  for (int i = 0; i < kSlotsPerWarp; ++i) {
    const int64_t c = c0 + i;
    if (c >= a.c_pad) break;
    __nv_bfloat16* dst = a.rows + (unit * a.c_pad + c) * D;
    bool valid = false;
    if (c < r.dense) {
      const int64_t absolute = r.dense_start + c;
      const int64_t rel = absolute - r.base;
      valid = absolute <= r.pos && rel < a.L;
      if (valid) {
        // lane l: dims [l * D / 32, (l + 1) * D / 32)
        constexpr int kPer = D / 32;
        uint32_t w[kPer / 2];
        if (a.kv_dtype == SA_BF16) {
          const uint32_t* src = reinterpret_cast<const uint32_t*>(
              static_cast<const __nv_bfloat16*>(a.window) + (b * a.L + rel) * D + lane * kPer);
#pragma unroll
          for (int e = 0; e < kPer / 2; ++e) w[e] = __ldg(src + e);
        } else {
          const float2* src = reinterpret_cast<const float2*>(
              static_cast<const float*>(a.window) + (b * a.L + rel) * D + lane * kPer);
#pragma unroll
          for (int e = 0; e < kPer / 2; ++e) {
            const float2 f = __ldg(src + e);
            w[e] = pack2<__nv_bfloat16>(f.x, f.y);
          }
        }
        if (kPer >= 8) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + lane * kPer);
#pragma unroll
          for (int e = 0; e < kPer / 8; ++e)
            d4[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        } else {
          *reinterpret_cast<uint2*>(dst + lane * kPer) = make_uint2(w[0], w[1]);
        }
      }
    } else if (c < r.dense + a.topk) {
      const int32_t rec = __shfl_sync(0xffffffffu, mine, i);
      if (rec >= a.valid_records && lane == 0 && a.err_word) atomicOr(a.err_word, SA_ERRBIT_RECORD);
      valid = rec >= 0 && rec < a.valid_records;
      if (valid) {
        const uint8_t* src = a.records + (b * a.R + rec) * a.record_stride;
        const uint8_t* st = stage + i * kStageBytes + (reinterpret_cast<uintptr_t>(src) & 15);
        uint32_t* d32 = reinterpret_cast<uint32_t*>(dst);
        for (int k = 0; k < nb; ++k) {
          const uint8_t* blk = st + 65 * k;
          const float sc = e8m0(blk[0]);
          const uint32_t two = static_cast<uint32_t>(blk[1 + 2 * lane]) |
                               (static_cast<uint32_t>(blk[2 + 2 * lane]) << 8);
          const float2 f = e4m3_pair(two);
          d32[32 * k + lane] = pack2<__nv_bfloat16>(f.x * sc, f.y * sc);
        }
        // the RoPE dims: little-endian bf16, copied
        const uint8_t* tl = st + 65 * nb;
        uint16_t* d16 = reinterpret_cast<uint16_t*>(dst + 64 * nb);
        for (int e = lane; e < a.n_rope; e += 32)
          d16[e] = static_cast<uint16_t>(tl[2 * e] | (tl[2 * e + 1] << 8));
      }
    }
    if (!valid) {
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      for (int e = lane; e < D / 8; e += 32) d4[e] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (lane == 0) a.valid[unit * a.c_pad + c] = valid ? 1 : 0;
  }
  pdl_launch_dependents();
}

// ---- attention ------------------------------------------------------------------------------
// One CTA per (unit, head block, key split): blockIdx.x = (unit * hblocks + hb) * splits + split.
template <int D>
__global__ void __launch_bounds__(256, 2) csa_attn_kernel(const CsaArgs a) {
  using G = CsaGeo<D>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int hg = warp >> 2;  // head group (16 heads)
  const int qd = warp & 3;   // dim quarter
  const int64_t hblocks = a.H / kHeads;
  const int64_t split = blockIdx.x % a.splits;
  const int64_t hb = (blockIdx.x / a.splits) % hblocks;
  const int64_t unit = blockIdx.x / (a.splits * hblocks);
  const int64_t b = unit / a.S, s = unit % a.S;
  const int64_t t0 = split * a.chunk_tiles;
  int64_t nt = a.c_pad / 16 - t0;
  if (nt > a.chunk_tiles) nt = a.chunk_tiles;
  if (nt < 0) nt = 0;
  unsigned char* sq = smem + G::kOffQ;
  unsigned char* srows = smem + G::kOffRows;
  float* sx = reinterpret_cast<float*>(smem + G::kOffX);
  uint8_t* svalid = smem + G::kOffValid;

  // Q of this head block (bf16; float queries rounded)
  for (int e = tid; e < kHeads * D / 8; e += 256) {
    const int h = e / (D / 8), c8 = e % (D / 8);
    const int64_t qoff = ((unit * a.H) + hb * kHeads + h) * D + c8 * 8;
    uint4 v;
    if (a.q_dtype == SA_BF16) {
      v = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.query) + qoff));
    } else {
      const float4* f = reinterpret_cast<const float4*>(static_cast<const float*>(a.query) + qoff);
      const float4 x = __ldg(f), y = __ldg(f + 1);
      v = make_uint4(pack2<__nv_bfloat16>(x.x, x.y), pack2<__nv_bfloat16>(x.z, x.w),
                     pack2<__nv_bfloat16>(y.x, y.y), pack2<__nv_bfloat16>(y.z, y.w));
    }
    *reinterpret_cast<uint4*>(sq + h * G::kRowStride + c8 * 16) = v;
  }
  pdl_wait();  // the candidate rows

  const __nv_bfloat16* rows = a.rows + (unit * a.c_pad + t0 * 16) * D;
  const uint8_t* vrow = a.valid + unit * a.c_pad + t0 * 16;
  auto issue = [&](int64_t t, int stage) {
    const uint32_t dst0 = smem_u32(srows + stage * 16 * G::kRowStride);
    for (int w = tid; w < 16 * (D / 8); w += 256) {
      const int r = w / (D / 8), j = w % (D / 8);
      cp_async16(dst0 + r * G::kRowStride + j * 16, rows + (t * 16 + r) * D + j * 8);
    }
    if (tid < 16) svalid[stage * 16 + tid] = vrow[t * 16 + tid];
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  float o[G::kNT][4];
#pragma unroll
  for (int n = 0; n < G::kNT; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
  float m_run[2] = {SA_NEG_INF, SA_NEG_INF}, l_run[2] = {0.f, 0.f};
  const float sl2 = a.scale_log2;
  const int64_t h_lo = hb * kHeads + hg * 16 + gid;  // rows gid and gid + 8

  if (nt > 0) issue(0, 0);
  for (int64_t t = 0; t < nt; ++t) {
    if (t + 1 < nt) issue(t + 1, static_cast<int>((t + 1) & 1));
    else asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncthreads();
    const int stage = static_cast<int>(t & 1);
    const uint32_t kbase = smem_u32(srows + stage * 16 * G::kRowStride);

    // S partial over this warp's quarter: 16 heads x 16 keys
    float sacc[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[n][e] = 0.f;
    {
      const uint32_t qa = smem_u32(sq) + (hg * 16 + (lane & 15)) * G::kRowStride +
                          (qd * G::kQuarter + 8 * (lane >> 4)) * 2;
      const int jm = lane >> 3, rr = lane & 7;
      const uint32_t krow = kbase + (rr + 8 * (jm >> 1)) * G::kRowStride +
                            (qd * G::kQuarter + 8 * (jm & 1)) * 2;
#pragma unroll
      for (int kk = 0; kk < G::kKS; ++kk) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(qa + kk * 32, a0, a1, a2, a3);
        ldsm_x4(krow + kk * 32, b0, b1, b2, b3);
        mma16816<__nv_bfloat16>(sacc[0], a0, a1, a2, a3, b0, b1);
        mma16816<__nv_bfloat16>(sacc[1], a0, a1, a2, a3, b2, b3);
      }
    }
    // the four quarters' sums: sx is [hg][quarter][value][lane]
    float* myx = sx + (hg * 4 + qd) * 8 * 32 + lane;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) myx[(n * 4 + e) * 32] = sacc[n][e];
    named_bar(1 + hg, 128);
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float acc = 0.f;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) acc += sx[((hg * 4 + q4) * 8 + n * 4 + e) * 32 + lane];
        sacc[n][e] = acc;
      }
    // online softmax: rows = heads gid, gid + 8; columns = candidate slots
    const uint8_t* tv = svalid + stage * 16;
    const int64_t slot0 = (t0 + t) * 16;
    float mx[2] = {SA_NEG_INF, SA_NEG_INF};
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = n * 8 + 2 * tig + (e & 1);
        float x = sacc[n][e] * sl2;
        if (a.bias && tv[col])
          x += kLog2e * __ldg(a.bias + b * a.bias_sb + (h_lo + 8 * (e >> 1)) * a.bias_sh +
                              s * a.bias_si + (slot0 + col) * a.bias_sk);
        sacc[n][e] = tv[col] ? x : SA_NEG_INF;
        mx[e >> 1] = fmaxf(mx[e >> 1], sacc[n][e]);
      }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 1));
      mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 2));
    }
    float mu[2], al[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      al[j] = 1.0f;
      if (mx[j] > m_run[j] + 8.0f) {  // lazy maximum (also the first finite one)
        al[j] = ex2(m_run[j] - mx[j]);
        m_run[j] = mx[j];
      }
      mu[j] = (m_run[j] == SA_NEG_INF) ? 0.f : m_run[j];
    }
    float ps[2] = {0.f, 0.f};
    uint32_t pa[4];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      const float p0 = ex2(sacc[n][0] - mu[0]), p1 = ex2(sacc[n][1] - mu[0]);
      const float p2 = ex2(sacc[n][2] - mu[1]), p3 = ex2(sacc[n][3] - mu[1]);
      ps[0] += p0 + p1;
      ps[1] += p2 + p3;
      pa[2 * n] = pack2<__nv_bfloat16>(p0, p1);
      pa[2 * n + 1] = pack2<__nv_bfloat16>(p2, p3);
    }
    l_run[0] = l_run[0] * al[0] + ps[0];
    l_run[1] = l_run[1] * al[1] + ps[1];
    if (al[0] != 1.0f || al[1] != 1.0f) {
#pragma unroll
      for (int n = 0; n < G::kNT; ++n) {
        o[n][0] *= al[0];
        o[n][1] *= al[0];
        o[n][2] *= al[1];
        o[n][3] *= al[1];
      }
    }
    // O += P . V over this warp's quarter
    {
      const int jm = lane >> 3, rr = lane & 7;
      const uint32_t vrow0 = kbase + (rr + 8 * (jm & 1)) * G::kRowStride +
                             (qd * G::kQuarter + 8 * (jm >> 1)) * 2;
#pragma unroll
      for (int n2 = 0; n2 < G::kNT / 2; ++n2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vrow0 + n2 * 32, b0, b1, b2, b3);
        mma16816<__nv_bfloat16>(o[2 * n2], pa[0], pa[1], pa[2], pa[3], b0, b1);
        mma16816<__nv_bfloat16>(o[2 * n2 + 1], pa[0], pa[1], pa[2], pa[3], b2, b3);
      }
    }
    __syncthreads();  // every warp is done with this stage before it refills
  }
  asm volatile("cp.async.wait_all;" ::: "memory");

#pragma unroll
  for (int j = 0; j < 2; ++j) {
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 1);
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 2);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int64_t h = h_lo + 8 * j;
    if (a.splits == 1) {
      float L = l_run[j];
      const float M = m_run[j];
      if (a.sink && M != SA_NEG_INF) L += ex2(a.sink[h] * kLog2e - M);
      const float inv = (M == SA_NEG_INF || L == 0.f) ? 0.f : 1.0f / L;
      const int64_t yoff = ((unit * a.H) + h) * D + qd * G::kQuarter;
#pragma unroll
      for (int n = 0; n < G::kNT; ++n) {
        const float v0 = o[n][2 * j] * inv, v1 = o[n][2 * j + 1] * inv;
        if (a.q_dtype == SA_BF16)
          *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.y) + yoff + n * 8 + 2 * tig) =
              pack2<__nv_bfloat16>(v0, v1);
        else
          *reinterpret_cast<float2*>(static_cast<float*>(a.y) + yoff + n * 8 + 2 * tig) =
              make_float2(v0, v1);
      }
    } else {
      const int64_t pidx = (unit * a.splits + split) * a.H + h;
      float* po = a.part_o + pidx * D + qd * G::kQuarter;
#pragma unroll
      for (int n = 0; n < G::kNT; ++n)
        *reinterpret_cast<float2*>(po + n * 8 + 2 * tig) = make_float2(o[n][2 * j], o[n][2 * j + 1]);
      if (qd == 0 && tig == 0) {
        a.part_ml[2 * pidx] = m_run[j];
        a.part_ml[2 * pidx + 1] = l_run[j];
      }
    }
  }
  pdl_launch_dependents();
}

// ---- split merge ----------------------------------------------------------------------------
// One 128-thread block per (unit, head): y = sum_s o_s 2^(m_s - M) / (sum_s l_s 2^(m_s - M)
// [+ 2^(sink - M)]), splits in order.
template <int D>
__global__ void __launch_bounds__(128) csa_combine_kernel(const CsaArgs a) {
  const int64_t uh = blockIdx.x;  // unit * H + h
  const int64_t unit = uh / a.H, h = uh % a.H;
  pdl_wait();
  float M = SA_NEG_INF;
  for (int64_t sp = 0; sp < a.splits; ++sp)
    M = fmaxf(M, a.part_ml[2 * ((unit * a.splits + sp) * a.H + h)]);
  float L = 0.f;
  for (int64_t sp = 0; sp < a.splits; ++sp) {
    const int64_t pidx = (unit * a.splits + sp) * a.H + h;
    const float ms = a.part_ml[2 * pidx];
    if (M != SA_NEG_INF && ms != SA_NEG_INF) L += a.part_ml[2 * pidx + 1] * ex2(ms - M);
  }
  if (a.sink && M != SA_NEG_INF) L += ex2(a.sink[h] * kLog2e - M);
  const float inv = (M == SA_NEG_INF || L == 0.f) ? 0.f : 1.0f / L;
  for (int d = threadIdx.x; d < D; d += 128) {
    float acc = 0.f;
    for (int64_t sp = 0; sp < a.splits; ++sp) {
      const int64_t pidx = (unit * a.splits + sp) * a.H + h;
      const float ms = a.part_ml[2 * pidx];
      if (M == SA_NEG_INF || ms == SA_NEG_INF) continue;
      acc += a.part_o[pidx * D + d] * ex2(ms - M);
    }
    const float v = acc * inv;
    if (a.q_dtype == SA_BF16) static_cast<__nv_bfloat16*>(a.y)[uh * D + d] = __float2bfloat16_rn(v);
    else static_cast<float*>(a.y)[uh * D + d] = v;
  }
}

// ---- host side ------------------------------------------------------------------------------

size_t csa_attn_smem_bytes(int64_t D) {
  return D == 128 ? CsaGeo<128>::kSmem : CsaGeo<512>::kSmem;
}

template <typename K>
static int launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      const CsaArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a) == cudaSuccess ? 0 : -1;
}

template <int D>
static int launch_csa_t(const CsaArgs& a, cudaStream_t st) {
  using G = CsaGeo<D>;
  constexpr int kSlotsPerCta = 8 * kSlotsPerWarp;
  const size_t stage_smem = static_cast<size_t>(kSlotsPerCta) * csa_stage_bytes(D, a.n_rope);
  csa_assemble_kernel<D><<<dim3(static_cast<unsigned>((a.c_pad + kSlotsPerCta - 1) / kSlotsPerCta),
                               static_cast<unsigned>(a.B * a.S)), 256, stage_smem, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return -1;
  if (a.tc) {  // the tcgen05 kernel over the same rows (k_fp8_tc.cu)
    bool merged = false;
    if (launch_csa_tc(a, st, &merged) != 0) return -1;
    if (!merged)
      return launch_pdl(csa_combine_kernel<D>, dim3(static_cast<unsigned>(a.B * a.S * a.H)),
                        dim3(128), 0, st, a);
    return 0;
  }
  if (cudaFuncSetAttribute(csa_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           G::kSmem) != cudaSuccess)
    return -1;
  const int64_t grid = a.B * a.S * (a.H / kHeads) * a.splits;
  mark_event(a.ev_before, st);
  if (launch_pdl(csa_attn_kernel<D>, dim3(static_cast<unsigned>(grid)), dim3(256), G::kSmem, st,
                 a) != 0)
    return -1;
  mark_event(a.ev_after, st);
  if (a.splits > 1)
    return launch_pdl(csa_combine_kernel<D>, dim3(static_cast<unsigned>(a.B * a.S * a.H)),
                      dim3(128), 0, st, a);
  return 0;
}

int launch_csa(const CsaArgs& a, cudaStream_t st) {
  if (a.D == 512) return launch_csa_t<512>(a, st);
  if (a.D == 128) return launch_csa_t<128>(a, st);
  return -1;
}

}  // namespace sa
