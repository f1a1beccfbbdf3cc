// k_fp8_tc.cu -- selected-token decode over the hybrid FP8 latent cache on the
// fifth-generation tensor cores (tcgen05 + TMEM + TMA), for blocks of 128
// query heads.
//
// Semantics: as k_fp8.cu -- the hybrid record of the compressed sparse
// attention pages (onnx-runtime-ep-cpu compressed_sparse_attention.rs,
// `CacheFormat::Fp8E4m3Block64`, `dequantize_cache`: blocks of [E8M0 scale
// byte, 64 E4M3FN codes] then the RoPE dims as little-endian bf16), and
// IndexShare's `index_share_row` over the candidates planned by k_plan.cu,
// with K and V both the decoded 576-dim record.
//
// GB300 design: two kernels.
//  1. fp8_gather_decode_kernel: each warp takes eight planned candidates,
//     fetches each record as one bulk copy (its 16-byte-aligned 656-byte
//     window) into shared memory and writes the exact bf16 decode (e4m3 x 2^(scale-127);
//     the RoPE tail copied) as row [unit, candidate] of a [units, n_cand_pad,
//     576] bf16 buffer; masked candidates are zero rows.  Each record is
//     decoded once, and the buffer (40 MB for 16 queries of 2176 keys) stays
//     in L2 for the attention kernel.
//  2. fp8_tc05_kernel: the 128 heads of a head block are the M of every MMA.
//     The 128 x 576 fp32 output block (288 KB) is larger than one SM's tensor
//     memory, so three CTAs share each (query position, head block, key
//     split): each owns a third of the output dims (three 64-dim chunks) and
//     computes the full 128-key score tiles itself.
//      * Q (128 heads x 576) stays in shared memory for the whole CTA as nine
//        128-byte-swizzled 64-dim slabs; warp 0's lane streams the decoded
//        keys by TMA into a five-slot ring: for every 128-key tile the nine
//        64-dim chunks for the scores, then the CTA's three chunks again as V.
//      * Warp 1's lane issues S = Q K^T chunk by chunk into one of two TMEM
//        score buffers; warp 2's lane issues O += P V (P from TMEM, V
//        MN-major, N = 64 per chunk).  (Two lanes: tcgen05.mma issue returns
//        only when the tensor core can take the instruction, so each lane
//        should wait only on its own inputs.)
//      * Warps 4-7 are the softmax warpgroup; thread r owns head r (TMEM lane
//        r).  Per tile: the maximum raw score over the valid keys (scale and
//        softcap are monotonic), a running maximum raised only by more than
//        2^8 (O then rescaled in TMEM), then P as bf16 pairs written over the
//        tile's own score columns.  At the end it writes the CTA's 192 output
//        dims, normalised, or a partial (m, l, O) for the split combine.
//      * Every mbarrier wait is bounded: a stalled pipeline sets
//        SA_ERRBIT_TIMEOUT, stops every role and still frees the tensor
//        memory.
//  The same attention kernel, in a 512-dim geometry (eight chunks, two CTAs
//  of 256 output dims), serves the compressed sparse attention rows that
//  k_csa.cu assembles: validity from bytes instead of planned positions, and
//  an optional additive bias per candidate slot (launch_csa_tc).
#include <cuda.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "e4m3.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace sa {

namespace {

constexpr int kD = 576;                  // FP8 latent record: 512 FP8 dims + 64 RoPE dims
constexpr int kRowBytes = kD * 2;        // decoded row: 576 bf16
constexpr int kHeads = 128;              // M of every MMA
constexpr int kKeys = 128;               // keys per tile (N of the score MMA)
constexpr int kChunkBytes = 128 * 128;   // 128 rows x 64 bf16, 128-byte swizzled
constexpr int kStages = 5;               // ring of key chunks
constexpr int kWarpLoad = 0, kWarpS = 1, kWarpPv = 2, kWarpSoftmax = 4;
constexpr int kThreads = 256;
constexpr int kMaxTiles = 48;            // tiles per CTA (validity staged in shared memory)
constexpr int kRecRope = 8 * 65;         // byte offset of the RoPE tail in a record
constexpr float kRescaleLog2 = 8.0f;
// barriers: q_full, full_s[kStages], full_pv[kStages], empty[kStages],
// s_full[2], p_full[2], pv_free[2], o_full, done[2].  A filled slot is
// announced on full_s or full_pv by the lane that will read it: each of those
// barriers then has one waiter that takes its phases in order (one ring
// barrier shared by both lanes would let the PV lane, running ahead of the
// fill, meet a phase two ahead of the barrier's and take it as complete).
constexpr int kBarQ = 0, kBarFullS = 1, kBarFullPv = kBarFullS + kStages,
              kBarEmpty = kBarFullPv + kStages, kBarS = kBarEmpty + kStages,
              kBarP = kBarS + 2, kBarPv = kBarP + 2, kBarO = kBarPv + 2, kBarDone = kBarO + 1,
              kNumBars = kBarDone + 2;
constexpr int kMaxClusterSplits = 8;
// tensor memory: score buffers 0 and 1, then this CTA's output dims
constexpr uint32_t kColS = 0, kColO = 2 * kKeys, kTmemCols = 512;

// Geometry of the attention kernel for a row width D (576: the FP8 latent
// record, three CTAs of 192 output dims per head block; 512: the compressed
// sparse attention rows, two CTAs of 256 output dims).
template <int D>
struct TcGeo {
  static constexpr int kD = D;
  static constexpr int kChunks = D / 64;                       // 64-dim chunks of a row
  static constexpr int kParts = D == 576 ? 3 : 2;              // CTAs sharing the output dims
  static constexpr int kPartChunks = kChunks / kParts;         // output chunks per CTA
  static constexpr int kPartDims = kPartChunks * 64;
  static constexpr int kEntries = kChunks + kPartChunks;       // ring entries per tile
  // shared memory (bytes)
  static constexpr int kOffQ = 0;                              // kChunks slabs [128 heads][64]
  static constexpr int kOffRing = kChunks * kChunkBytes;       // [kStages] key chunks
  static constexpr int kOffValid = kOffRing + kStages * kChunkBytes;  // [kMaxTiles][4] masks
  static constexpr int kOffBar = kOffValid + kMaxTiles * 16;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmem = kOffAbort + 4 + 1024;           // + alignment slack
  // The epilogue and the split merge reuse the Q area and the ring once every
  // MMA has completed: the CTA's O rows (fp32, padded rows), its (max, sum)
  // per row, the merge weights.
  static constexpr int kOStride = kPartDims + 4;               // floats per O row
  static constexpr int kOffMO = kOffQ;
  static constexpr int kOffMMl = kOffMO + kHeads * kOStride * 4;
  static constexpr int kOffMW = kOffMMl + kHeads * 8;
  static_assert(kChunks * 64 == D && kPartChunks * kParts == kChunks, "row geometry");
  static_assert(kOffMW + kHeads * kMaxClusterSplits * 4 <= kOffValid, "merge area");
  static_assert(kSmem <= 232448, "shared memory");
  static_assert(kColO + kPartDims <= kTmemCols, "tensor memory");
};
using GeoFp8 = TcGeo<576>;
using GeoCsa = TcGeo<512>;

struct Fp8TcParams {
  const int32_t* pos;        // [units, n_cand_pad] planned cache positions or -1
  const uint8_t* valid_u8;   // or, when set: [units, n_cand_pad] 1 = a valid candidate
  // nullable additive bias of candidate slot k (natural-log units), unit = b * bias_S + s:
  // element (b, h, s, k) at b * bias_sb + h * bias_sh + s * bias_si + k * bias_sk
  const float* bias;
  int64_t bias_sb, bias_sh, bias_si, bias_sk;
  int bias_S;
  int64_t n_cand_pad;        // multiple of 128
  void* y;                   // [B, Hq, Sq, D] bf16
  float* part_o;             // splits > 1: [units * splits * Hq, D] partial outputs
  float* part_ml;            //             [units * splits * Hq, 2] (max, sum)
  const float* sink;         // nullable [Hq]
  uint32_t* err_word;
  int B, Sq, Hq, hblocks, splits, chunk_tiles, tiles;
  int cluster_merge;         // the splits of an output block form a cluster and merge on chip
  float scale_log2;          // scale * log2(e)
  float k1, c_log2;          // softcap: logit2 = c_log2 * tanh(s * k1)
};

struct DecodeParams {
  const char* recs;          // k_cache base: [B, 1, T, record_stride] bytes
  int64_t record_stride;
  int64_t T;
  const int32_t* pos;        // [units, n_cand_pad]
  int64_t rows;              // units * n_cand_pad
  int64_t n_cand_pad;
  int Sq;
  __nv_bfloat16* kdec;       // [units, n_cand_pad, 576]
  uint32_t* err_word;        // nullable: SA_ERRBIT_TIMEOUT if a copy never lands
  // own_positions: the kernel plans its candidates from the index rows (one
  // latent head, one index head: unit u = b * Sq + i is index row u) and writes
  // them to pos for the attention kernel; else it reads the planned pos.
  int own_positions;
  int after_plan;            // a validation-only plan kernel runs just before this one
  int32_t* pos_out;
  const void* idx;           // [B, 1, Sq, K]
  int idx_is_i64;
  int causal;
  int64_t K, window, past_len;
  const int64_t* kv_len;     // nullable
};

// The ring's entries, in order: the nine score chunks of tile 0, then for
// each tile j: the nine score chunks of tile j + 1 (if any) and the CTA's
// three output chunks of tile j.
template <class G>
__device__ __forceinline__ uint32_t s_entry(int j, int c) {
  return j == 0 ? static_cast<uint32_t>(c)
                : static_cast<uint32_t>(G::kChunks + G::kEntries * (j - 1) + c);
}
template <class G>
__device__ __forceinline__ uint32_t pv_entry(int j, int k, int nt) {
  return static_cast<uint32_t>(G::kChunks + G::kEntries * j + (j + 1 < nt ? G::kChunks : 0) + k);
}
// Entry e -> (tile j, chunk c, read by the score lane?).
template <class G>
__device__ __forceinline__ void entry_of(int e, int nt, int part, int& j, int& c, bool& score) {
  if (e < G::kChunks) {
    j = 0;
    c = e;
    score = true;
    return;
  }
  const int q = e - G::kChunks, blk = q / G::kEntries, rr = q % G::kEntries;
  const bool more = blk + 1 < nt;
  score = more && rr < G::kChunks;
  if (score) {
    j = blk + 1;
    c = rr;
  } else {
    j = blk;
    c = part * G::kPartChunks + (rr - (more ? G::kChunks : 0));
  }
}

// ---- thread-block cluster helpers ----
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster; release / acquire of shared memory.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// This CTA's shared address -> the same offset in cluster CTA `rank`.
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float2 ld_cluster_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}

// Two E4M3FN codes -> two floats, exactly (via the f16x2 conversion).
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t two) { return e4m3x2_to_float2(two); }

// E8M0 scale byte -> 2^(b - 127); 255 is NaN in the format.
__device__ __forceinline__ float e8m0_scale(uint32_t b) {
  if (b == 255u) return __int_as_float(0x7fc00000);
  if (b == 0u) return __int_as_float(0x00400000);  // 2^-127, a subnormal float
  return __int_as_float(static_cast<int>(b) << 23);
}

}  // namespace

namespace {

// ---- kernel 1: gather + exact decode of the planned candidates' records ------------------

constexpr int kDecRecs = 8;  // records per warp, all in flight together
static_assert(128 % kDecRecs == 0, "a warp's rows must lie in one unit");
static_assert(kDecRecs >= 2 && kDecRecs <= 32 && (kDecRecs & (kDecRecs - 1)) == 0,
              "two halves of lanes, a power of two");
// A record is fetched as the 16-byte-aligned window around it: records are
// 8-byte aligned (checked on the host), so the window starts 0 or 8 bytes
// before the record and is 656 bytes long; it never leaves the 16-byte
// granules that hold the record.
constexpr int kDecSlot = 656;
constexpr size_t kDecSmem = 8 * kDecRecs * kDecSlot + 8 * 2 * sizeof(uint64_t);

// Eight decoded bf16 values (16 bytes) of FP8 block c, codes [8g, 8g + 8):
// record bytes 65c + 1 + 8g .. (read as aligned words of the staged window,
// the record starting `off` bytes into it), scaled by the block's E8M0 byte.
__device__ __forceinline__ uint4 decode8(const uint32_t* sw, const unsigned char* sb, int off,
                                         int c, int g) {
  const float sc = e8m0_scale(sb[off + 65 * c]);
  const uint64_t sc2 = f2_pack(sc, sc);
  const int first = off + 65 * c + 1 + 8 * g;
  const int w0 = first >> 2, sh = (first & 3) * 8;
  const uint32_t a = sw[w0], b = sw[w0 + 1], d = sw[w0 + 2];
  const uint32_t lo = sh ? __funnelshift_r(a, b, sh) : a;
  const uint32_t hi = sh ? __funnelshift_r(b, d, sh) : b;
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t codes = i ? hi : lo;
    const float2 x = e4m3x2_to_f2(codes & 0xffffu), y = e4m3x2_to_f2(codes >> 16);
    float a0, a1, b0, b1;
    f2_unpack(f2_mul(f2_pack(x.x, x.y), sc2), a0, a1);
    f2_unpack(f2_mul(f2_pack(y.x, y.y), sc2), b0, b1);
    o[2 * i] = pack2<__nv_bfloat16>(a0, a1);
    o[2 * i + 1] = pack2<__nv_bfloat16>(b0, b1);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// One decoded row (72 x 16 bytes) from a staged record window, or zeros when
// the candidate is masked: lane l writes 16-byte chunks l and l + 32 (FP8
// blocks l / 8 and 4 + l / 8, codes [8 (l % 8), 8 (l % 8) + 8)), so that every
// warp store is 512 contiguous bytes; lanes 0-7 copy the RoPE tail (record
// bytes 520 ..) to chunks 64-71.
__device__ __forceinline__ void decode_row(const unsigned char* slot, int off, uint4* out, int lane,
                                           bool valid) {
  const uint32_t* sw = reinterpret_cast<const uint32_t*>(slot);
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  const uint4 lo = decode8(sw, slot, off, lane >> 3, lane & 7);
  const uint4 hi = decode8(sw, slot, off, 4 + (lane >> 3), lane & 7);
  out[lane] = valid ? lo : z;
  out[32 + lane] = valid ? hi : z;
  if (lane < 8) {
    const uint2* rope = reinterpret_cast<const uint2*>(slot + off + kRecRope);  // 8-byte aligned
    const uint2 r0 = rope[2 * lane], r1 = rope[2 * lane + 1];
    out[64 + lane] = valid ? make_uint4(r0.x, r0.y, r1.x, r1.y) : z;
  }
}

// Each warp decodes kDecRecs consecutive rows [unit, candidate] of the buffer
// (8 warps per CTA): the rows' positions, then one bulk copy per record
// window into shared memory (lanes 0-7; the two halves complete on their own
// mbarriers), then the decodes, the four rows of a half interleaved.  A
// masked candidate is not fetched; its row is written as zeros.
__global__ void __launch_bounds__(256, 4) fp8_gather_decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(16) unsigned char stage[];  // [8 warps][kDecRecs][kDecSlot], barriers
  const int warp = static_cast<int>(threadIdx.x) >> 5, lane = static_cast<int>(threadIdx.x) & 31;
  // rows = units * n_cand_pad is a multiple of kDecRecs: a warp's rows are all in range
  const int64_t row0 = (static_cast<int64_t>(blockIdx.x) * 8 + warp) * kDecRecs;
  // With own positions after the plan kernel, nothing here reads what that
  // kernel writes (the validation); the wait moves to the end, so that this
  // grid completes only after it (the attention kernel waits on this grid).
  const bool wait_late = p.own_positions && p.after_plan;
  if (row0 >= p.rows) {
    if (wait_late) pdl_wait();
    return;
  }
  unsigned char* st = stage + warp * kDecRecs * kDecSlot;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage + 8 * kDecRecs * kDecSlot) + 2 * warp;
  if (lane == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
  }
  fence_proxy_async_smem();
  fence_mbar_init();
  __syncwarp();
  if (!wait_late) pdl_wait();  // the planned positions, or the work before the call
  pdl_launch_dependents();       // the attention kernel may start its set-up
  // The warp's rows share one unit (kDecRecs divides n_cand_pad, a multiple
  // of 128, and row0 is a multiple of kDecRecs): one division per warp.
  const int64_t unit = row0 / p.n_cand_pad;
  const int64_t b = unit / p.Sq;
  int32_t mine = -1;
  if (p.own_positions) {
    if (lane < kDecRecs) {
      const int64_t c = row0 - unit * p.n_cand_pad + lane;
      const CandRule rule =
          cand_rule(p.kv_len, b, p.T, p.window, p.causal, p.past_len, unit - b * p.Sq);
      if (c < p.window) mine = window_pos(rule, c);
      else if (c < p.window + p.K)
        mine = selected_pos(rule, load_index(p.idx, unit * p.K + (c - p.window), p.idx_is_i64));
      p.pos_out[row0 + lane] = mine;
    }
  } else if (lane < kDecRecs) {
    mine = __ldg(p.pos + row0 + lane);
  }
  const char* batch_recs = p.recs + b * p.T * p.record_stride;
  const char* rec = batch_recs + static_cast<int64_t>(mine >= 0 ? mine : 0) * p.record_stride;
  const int off = static_cast<int>(reinterpret_cast<uintptr_t>(rec) & 15u);
  // bytes expected per half: lanes [0, kHalf) hold half 0's records, lanes
  // [kHalf, 2 kHalf) half 1's
  constexpr int kHalf = kDecRecs / 2;
  uint32_t tot = (mine >= 0) ? static_cast<uint32_t>(kDecSlot) : 0u;
#pragma unroll
  for (int sh = 1; sh < kHalf; sh <<= 1) tot += __shfl_xor_sync(0xffffffffu, tot, sh);
  const uint32_t tot1 = __shfl_sync(0xffffffffu, tot, kHalf);
  if (lane == 0) {
    mbar_arrive_expect_tx(&bars[0], tot);
    mbar_arrive_expect_tx(&bars[1], tot1);
  }
  __syncwarp();
  if (mine >= 0) bulk_g2s(st + lane * kDecSlot, rec - off, kDecSlot, &bars[lane / kHalf]);
  uint4* out0 = reinterpret_cast<uint4*>(p.kdec + row0 * kD);  // rows of 72 x 16 bytes
  bool landed[2] = {true, true};
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    landed[half] = mbar_wait(&bars[half], 0u);
#pragma unroll
    for (int rr = 0; rr < kHalf; ++rr) {
      const int r = half * kHalf + rr;
      const bool valid = __shfl_sync(0xffffffffu, mine, r) >= 0;
      const int ro = __shfl_sync(0xffffffffu, off, r);
      decode_row(st + r * kDecSlot, ro, out0 + r * (kRowBytes / 16), lane, valid);
    }
  }
  if (!landed[0] || !landed[1]) {
    // a copy that never landed: report it, and give the copies still in
    // flight one more bounded wait before the warp's shared memory is released
    if (lane == 0 && p.err_word) atomicOr(p.err_word, SA_ERRBIT_TIMEOUT);
    if (!landed[0]) mbar_wait(&bars[0], 0u);
    if (!landed[1]) mbar_wait(&bars[1], 0u);
  }
  if (wait_late) pdl_wait();
}

}  // namespace

namespace {

// ---- kernel 2 roles: the TMA lane, the MMA issue lanes -------------------------------------

// The ring entries in order, each a 128-key x 64-dim box of the decoded buffer
// (Q's nine slabs were requested in the prologue).
template <class G>
__device__ void fp8tc_producer(const CUtensorMap* tk, const Fp8TcParams& p,
                               int unit, int t0, int nt, int part, uint8_t* sm,
                               uint64_t* bars, volatile int* abort_flag) {
  tc05::prefetch_tmap(tk);
  // per slot: armed at all, last fill read by the score lane, its parity;
  // and the parity of the next phase of full_s / full_pv
  uint32_t armed = 0, last_score = 0, last_par = 0, par_s = 0, par_pv = 0;
  const int total = G::kEntries * nt;
  for (int e = 0; e < total; ++e) {
    int j, c;
    bool score;
    entry_of<G>(e, nt, part, j, c, score);
    const uint32_t slot = static_cast<uint32_t>(e) % kStages, use = static_cast<uint32_t>(e) / kStages;
    if (use > 0 && !wait_or_abort(&bars[kBarEmpty + slot], (use - 1) & 1, abort_flag, p.err_word))
      break;
    uint32_t& par = score ? par_s : par_pv;
    const uint32_t ph = (par >> slot) & 1;
    par ^= 1u << slot;
    armed |= 1u << slot;
    last_score = (last_score & ~(1u << slot)) | ((score ? 1u : 0u) << slot);
    last_par = (last_par & ~(1u << slot)) | (ph << slot);
    uint64_t* full = &bars[(score ? kBarFullS : kBarFullPv) + slot];
    mbar_arrive_expect_tx(full, kChunkBytes);
    tc05::tma_load3(sm + G::kOffRing + slot * kChunkBytes, tk, 64 * c, (t0 + j) * kKeys, unit, full);
  }
  // no copy may still be landing when the CTA exits
  mbar_wait(&bars[kBarQ], 0);
  for (int s = 0; s < kStages; ++s)
    if ((armed >> s) & 1)
      mbar_wait(&bars[(((last_score >> s) & 1) ? kBarFullS : kBarFullPv) + s], (last_par >> s) & 1);
}

// Every MMA this lane issued completes before the tensor memory is released.
__device__ __forceinline__ void drain_lane(uint64_t* done) {
  tc05::commit(done);
  mbar_wait(done, 0);
}

// S_j = Q K_j^T into score buffer j & 1, one 64-dim chunk (4 k-steps) at a time.
template <class G>
__device__ void fp8tc_score_lane(const Fp8TcParams& p, int nt, uint8_t* sm, uint64_t* bars,
                                 uint32_t tmem, volatile int* abort_flag) {
  constexpr uint32_t id_s = tc05::idesc_f16(kHeads, kKeys, true, false, false);
  const uint64_t dQ = tc05::sw128_desc(smem_u32(sm + G::kOffQ), 16, 1024);
  const uint64_t dK = tc05::sw128_desc(smem_u32(sm + G::kOffRing), 16, 1024);
  bool ok = wait_or_abort(&bars[kBarQ], 0, abort_flag, p.err_word);
  uint32_t par = 0;  // bit s: parity of the next awaited phase of full_s[s]
  for (int j = 0; ok && j < nt; ++j) {
    const int buf = j & 1;
    // the buffer's previous P (tile j - 2) must have been read by its PV
    if (j >= 2 && !wait_or_abort(&bars[kBarPv + buf], ((j - 2) >> 1) & 1, abort_flag, p.err_word))
      break;
    for (int c = 0; c < G::kChunks; ++c) {
      const uint32_t e = s_entry<G>(j, c), slot = e % kStages;
      if (!wait_or_abort(&bars[kBarFullS + slot], (par >> slot) & 1, abort_flag, p.err_word)) {
        ok = false;
        break;
      }
      par ^= 1u << slot;
      tc05::fence_after_sync();
      const uint64_t a0 = dQ + ((static_cast<uint32_t>(c) * kChunkBytes) >> 4);
      const uint64_t b0 = dK + ((slot * kChunkBytes) >> 4);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc05::mma_ss(tmem + kColS + buf * kKeys, a0 + kk * 2, b0 + kk * 2, id_s,
                     (c > 0 || kk > 0) ? 1u : 0u);
      tc05::commit(&bars[kBarEmpty + slot]);
    }
    if (!ok) break;
    tc05::commit(&bars[kBarS + buf]);
  }
  drain_lane(&bars[kBarDone + 0]);
}

// O[:, 64k .. 64k + 64) += P_j V_j[:, chunk part * 3 + k] for the CTA's three
// output chunks; P_j is the bf16 pairs over score buffer j & 1's first 64
// columns (keys 2i, 2i + 1 in column i).
template <class G>
__device__ void fp8tc_pv_lane(const Fp8TcParams& p, int nt, uint8_t* sm, uint64_t* bars,
                              uint32_t tmem, volatile int* abort_flag) {
  constexpr uint32_t id_o = tc05::idesc_f16(kHeads, 64, true, false, true);
  const uint64_t dV = tc05::sw128_desc(smem_u32(sm + G::kOffRing), kChunkBytes, 1024);
  bool ok = true;
  uint32_t par = 0;  // bit s: parity of the next awaited phase of full_pv[s]
  for (int j = 0; ok && j < nt; ++j) {
    const int buf = j & 1;
    if (!wait_or_abort(&bars[kBarP + buf], (j >> 1) & 1, abort_flag, p.err_word)) break;
    tc05::fence_after_sync();
    for (int k = 0; k < G::kPartChunks; ++k) {
      const uint32_t e = pv_entry<G>(j, k, nt), slot = e % kStages;
      if (!wait_or_abort(&bars[kBarFullPv + slot], (par >> slot) & 1, abort_flag, p.err_word)) {
        ok = false;
        break;
      }
      par ^= 1u << slot;
      tc05::fence_after_sync();
      const uint64_t v0 = dV + ((slot * kChunkBytes) >> 4);
#pragma unroll
      for (int kk = 0; kk < kKeys / 16; ++kk)
        tc05::mma_ts(tmem + kColO + 64 * k, tmem + kColS + buf * kKeys + 8 * kk,
                     v0 + ((kk * 2048) >> 4), id_o, (j > 0 || kk > 0) ? 1u : 0u);
      tc05::commit(&bars[kBarEmpty + slot]);
    }
    if (!ok) break;
    tc05::commit(&bars[kBarPv + buf]);
    if (j == nt - 1) tc05::commit(&bars[kBarO]);
  }
  drain_lane(&bars[kBarDone + 1]);
}

}  // namespace

namespace {

// ---- kernel 2 role: softmax warpgroup (warps 4-7; thread r = head r = TMEM lane r) -------

// kCols columns of this thread's O row *= alpha, in tensor memory (warp-collective).
template <class G>
__device__ __forceinline__ void rescale_o(uint32_t tO, float alpha) {
  const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
  for (int c = 0; c < G::kPartDims / 32; ++c) {
    uint32_t o[32];
    tc05::tmem_ld32(tO + c * 32, o);
    tc05::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float lo, hi;
      f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), a2), lo,
                hi);
      o[2 * i] = __float_as_uint(lo);
      o[2 * i + 1] = __float_as_uint(hi);
    }
    tc05::tmem_st32(tO + c * 32, o);
  }
  tc05::tmem_st_wait();
}

// Log2-domain logit of a raw score.
template <bool kCap>
__device__ __forceinline__ float logit2(float s, const Fp8TcParams& p) {
  return kCap ? p.c_log2 * tanh_approx(s * p.k1) : s * p.scale_log2;
}

template <class G, bool kCap, bool kBias>
__device__ void fp8tc_softmax(const Fp8TcParams& p, int unit, int hb, int split, int nt,
                              int part, const uint32_t* valid, uint64_t* bars, uint32_t tmem,
                              volatile int* abort_flag) {
  const int warp = static_cast<int>(threadIdx.x) >> 5, lane = static_cast<int>(threadIdx.x) & 31;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  float m_run = SA_NEG_INF, l_run = 0.0f;
  bool ok = true;
  // kBias: this head's bias row at candidate slot 0
  const float* brow = nullptr;
  if constexpr (kBias) {
    const int bb = unit / p.bias_S, ss = unit % p.bias_S;
    brow = p.bias + bb * p.bias_sb + static_cast<int64_t>(hb * kHeads + row) * p.bias_sh +
           ss * p.bias_si;
  }
  const int64_t slot_t0 = static_cast<int64_t>(split) * p.chunk_tiles * kKeys;
  for (int j = 0; j < nt; ++j) {
    const int buf = j & 1;
    // validity of the tile's keys 32k + bit (kept in scalars: the loops over k
    // below are not unrolled)
    const uint4 vm = reinterpret_cast<const uint4*>(valid)[j];
    const uint32_t vm0 = vm.x, vm1 = vm.y, vm2 = vm.z, vm3 = vm.w;
    auto valid_bits = [&](int k) { return k == 0 ? vm0 : k == 1 ? vm1 : k == 2 ? vm2 : vm3; };
    if (!wait_or_abort_warp(&bars[kBarS + buf], (j >> 1) & 1, abort_flag, p.err_word)) {
      ok = false;
      break;
    }
    tc05::fence_after_sync();
    const uint32_t tS = tl + kColS + buf * kKeys;
    // pass 1: the largest raw score over the valid keys
    float mx = SA_NEG_INF;
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
      uint32_t s[32];
      tc05::tmem_ld32(tS + 32 * k, s);
      tc05::tmem_ld_wait();
      const uint32_t vk = valid_bits(k);
      if constexpr (kBias) {
        // the biased log2 logits replace the raw scores in tensor memory
        const float* bk = brow + (slot_t0 + j * kKeys + 32 * k) * p.bias_sk;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float x = SA_NEG_INF;
          if ((vk >> i) & 1u)
            x = logit2<kCap>(__uint_as_float(s[i]), p) + kLog2e * __ldg(bk + i * p.bias_sk);
          s[i] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
        tc05::tmem_st32(tS + 32 * k, s);
      } else if (vk == 0xffffffffu) {
#pragma unroll
        for (int i = 0; i < 16; ++i) mx = max3(mx, __uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a = ((vk >> (2 * i)) & 1u) ? __uint_as_float(s[2 * i]) : SA_NEG_INF;
          const float c = ((vk >> (2 * i + 1)) & 1u) ? __uint_as_float(s[2 * i + 1]) : SA_NEG_INF;
          mx = max3(mx, a, c);
        }
      }
    }
    if constexpr (kBias) tc05::tmem_st_wait();
    // the lazy running maximum (log2 units): raised only past 2^8
    const float mt = (kBias || mx == SA_NEG_INF) ? mx : logit2<kCap>(mx, p);
    float alpha = 1.0f;
    if (mt > m_run + kRescaleLog2) {  // also the first finite maximum
      alpha = ex2(m_run - mt);
      m_run = mt;
    }
    const float mu = m_run == SA_NEG_INF ? 0.0f : m_run;
    // O *= alpha before PV_j accumulates into it (PV_(j-1) must be complete)
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
      if (!wait_or_abort_warp(&bars[kBarPv + ((j - 1) & 1)], ((j - 1) >> 1) & 1, abort_flag,
                              p.err_word)) {
        ok = false;
        break;
      }
      tc05::fence_after_sync();
      rescale_o<G>(tl + kColO, alpha);
    }
    // pass 2: P = 2^(logit - mu) as bf16 pairs over the buffer's first 64 columns
    float ls0 = 0.0f, ls1 = 0.0f;
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
      uint32_t s[32];
      tc05::tmem_ld32(tS + 32 * k, s);
      tc05::tmem_ld_wait();
      const uint32_t vk = valid_bits(k);
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float x0 = kBias ? __uint_as_float(s[2 * i]) : logit2<kCap>(__uint_as_float(s[2 * i]), p);
        const float x1 =
            kBias ? __uint_as_float(s[2 * i + 1]) : logit2<kCap>(__uint_as_float(s[2 * i + 1]), p);
        float p0 = ex2(x0 - mu);
        float p1 = ex2(x1 - mu);
        if (!((vk >> (2 * i)) & 1u)) p0 = 0.0f;
        if (!((vk >> (2 * i + 1)) & 1u)) p1 = 0.0f;
        ls0 += p0;
        ls1 += p1;
        pk[i] = pack2<__nv_bfloat16>(p0, p1);
      }
      tc05::tmem_st16(tS + 16 * k, pk);
    }
    tc05::tmem_st_wait();
    l_run = l_run * alpha + (ls0 + ls1);
    tc05::fence_before_sync();
    mbar_arrive(&bars[kBarP + buf]);
  }

  // ---- epilogue: this CTA's 192 output dims of head row ----------------------------------
  pdl_launch_dependents();  // the combine kernel may start launching
  // Each thread stages its row in the Q area (free: every score MMA has
  // completed) and, for y or the partials, copies it out with one bulk copy
  // (row-per-thread global stores would be 48 scattered 16-byte writes each).
  const int h = hb * kHeads + row;
  const int b = unit / p.Sq, i = unit % p.Sq;
  const bool have = nt > 0 && ok && wait_or_abort_warp(&bars[kBarO], 0, abort_flag, p.err_word);
  if (have) tc05::fence_after_sync();
  mbar_wait(&bars[kBarQ], 0);  // (no tile at all: Q's load must have landed before its area is reused)
  uint8_t* sm = reinterpret_cast<uint8_t*>(bars) - G::kOffBar;
  float* orow = reinterpret_cast<float*>(sm + G::kOffMO) + row * G::kOStride;
  if (p.splits == 1) {
    float L = l_run;
    if (p.sink && m_run != SA_NEG_INF) L += ex2(p.sink[h] * kLog2e - m_run);
    const float inv = (!have || m_run == SA_NEG_INF || L == 0.0f) ? 0.0f : 1.0f / L;
    uint32_t* yrow = reinterpret_cast<uint32_t*>(orow);  // 192 bf16 = 384 bytes
#pragma unroll 1
    for (int c = 0; c < G::kPartDims / 32; ++c) {
      uint32_t o[32];
      if (have) {
        tc05::tmem_ld32(tl + kColO + c * 32, o);
        tc05::tmem_ld_wait();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w[e] = pack2<__nv_bfloat16>(__uint_as_float(o[8 * q + 2 * e]) * inv,
                                      __uint_as_float(o[8 * q + 2 * e + 1]) * inv);
        *reinterpret_cast<uint4*>(yrow + c * 16 + 4 * q) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    fence_proxy_async_smem();
    tc05::bulk_s2g(static_cast<__nv_bfloat16*>(p.y) +
                       ((static_cast<int64_t>(b) * p.Hq + h) * p.Sq + i) * G::kD + part * G::kPartDims,
                   yrow, G::kPartDims * 2);
    tc05::bulk_commit_group();
    tc05::bulk_wait_group_read0();
    return;
  }
  // splits > 1: the row's unnormalised O and (max, sum)
#pragma unroll 1
  for (int c = 0; c < G::kPartDims / 32; ++c) {
    uint32_t o[32];
    if (have) {
      tc05::tmem_ld32(tl + kColO + c * 32, o);
      tc05::tmem_ld_wait();
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = 0u;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q)
      *reinterpret_cast<uint4*>(orow + c * 32 + 4 * q) =
          make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
  }
  const float m_out = have ? m_run : SA_NEG_INF, l_out = have ? l_run : 0.0f;
  if (p.cluster_merge) {  // merged on chip after the cluster barrier
    float* ml = reinterpret_cast<float*>(sm + G::kOffMMl);
    ml[2 * row] = m_out;
    ml[2 * row + 1] = l_out;
    return;
  }
  const int64_t pidx = (static_cast<int64_t>(unit) * p.splits + split) * p.Hq + h;
  fence_proxy_async_smem();
  tc05::bulk_s2g(p.part_o + pidx * G::kD + part * G::kPartDims, orow, G::kPartDims * 4);
  tc05::bulk_commit_group();
  if (part == 0) {  // the same (max, sum) in every part: the combine kernel's layout
    p.part_ml[2 * pidx] = m_out;
    p.part_ml[2 * pidx + 1] = l_out;
  }
  tc05::bulk_wait_group_read0();
}

// The splits of one (unit, head block, part) are the CTAs of a cluster (rank =
// split).  Cluster CTA s merges head rows [128 s / C, 128 (s + 1) / C) of the
// part's dims, reading every CTA's staged O rows and (max, sum) through
// distributed shared memory:
//   y = sum_c 2^(m_c - M) O_c / (sum_c 2^(m_c - M) l_c [+ 2^(sink - M)]).
template <class G>
__device__ void fp8tc_cluster_merge(const Fp8TcParams& p, int unit, int hb, int part, uint8_t* sm) {
  const int C = p.splits;
  const uint32_t rank = cluster_rank();
  const int r0 = static_cast<int>(rank) * kHeads / C, r1 = (static_cast<int>(rank) + 1) * kHeads / C;
  const uint32_t o_base = smem_u32(sm + G::kOffMO), ml_base = smem_u32(sm + G::kOffMMl);
  float* wts = reinterpret_cast<float*>(sm + G::kOffMW);  // [128][kMaxClusterSplits]
  const int tid = static_cast<int>(threadIdx.x);
  const int b = unit / p.Sq, i = unit % p.Sq;
  if (tid < r1 - r0) {
    const int r = r0 + tid;
    float m[kMaxClusterSplits], l[kMaxClusterSplits];
    float M = SA_NEG_INF;
#pragma unroll
    for (int c = 0; c < kMaxClusterSplits; ++c) {
      m[c] = SA_NEG_INF;
      l[c] = 0.0f;
      if (c < C) {
        const float2 v = ld_cluster_f2(map_rank(ml_base + 8u * r, c));
        m[c] = v.x;
        l[c] = v.y;
        M = fmaxf(M, v.x);
      }
    }
    float L = 0.0f;
#pragma unroll
    for (int c = 0; c < kMaxClusterSplits; ++c) {
      m[c] = (M == SA_NEG_INF || m[c] == SA_NEG_INF) ? 0.0f : ex2(m[c] - M);  // weight
      L += m[c] * l[c];
    }
    if (p.sink && M != SA_NEG_INF) L += ex2(p.sink[hb * kHeads + r] * kLog2e - M);
    const float inv = (M == SA_NEG_INF || L == 0.0f) ? 0.0f : 1.0f / L;
#pragma unroll
    for (int c = 0; c < kMaxClusterSplits; ++c) wts[r * kMaxClusterSplits + c] = m[c] * inv;
  }
  __syncthreads();
  const int n = (r1 - r0) * (G::kPartDims / 4);
  for (int it = tid; it < n; it += kThreads) {
    const int r = r0 + it / (G::kPartDims / 4), k = it % (G::kPartDims / 4);
    const uint32_t src = o_base + static_cast<uint32_t>((r * G::kOStride + 4 * k) * 4);
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int c = 0; c < kMaxClusterSplits; ++c) {
      if (c >= C) break;
      const float w = wts[r * kMaxClusterSplits + c];
      if (w == 0.0f) continue;
      const float4 v = ld_cluster_f4(map_rank(src, c));
      acc.x = fmaf(v.x, w, acc.x);
      acc.y = fmaf(v.y, w, acc.y);
      acc.z = fmaf(v.z, w, acc.z);
      acc.w = fmaf(v.w, w, acc.w);
    }
    __nv_bfloat16* yp = static_cast<__nv_bfloat16*>(p.y) +
                        ((static_cast<int64_t>(b) * p.Hq + hb * kHeads + r) * p.Sq + i) * G::kD +
                        part * G::kPartDims + 4 * k;
    *reinterpret_cast<uint2*>(yp) =
        make_uint2(pack2<__nv_bfloat16>(acc.x, acc.y), pack2<__nv_bfloat16>(acc.z, acc.w));
  }
}

}  // namespace


// One CTA per (unit = (batch, query position), 128-head block, third of the
// output dims, key split): blockIdx.x = ((unit * hblocks + hb) * 3 + part) *
// splits + split, the splits of one output block adjacent (a cluster when
// they merge on chip).
template <class G, bool kCap, bool kBias>
__global__ void __launch_bounds__(kThreads, 1)
    fp8_tc05_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const Fp8TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + G::kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + G::kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + G::kOffAbort);
  uint32_t* valid = reinterpret_cast<uint32_t*>(sm + G::kOffValid);
  const int warp = static_cast<int>(threadIdx.x) >> 5, lane = static_cast<int>(threadIdx.x) & 31;
  int cta = static_cast<int>(blockIdx.x);
  const int split = cta % p.splits;
  cta /= p.splits;
  const int part = cta % G::kParts;
  cta /= G::kParts;
  const int hb = cta % p.hblocks;
  const int unit = cta / p.hblocks;
  const int t0 = split * p.chunk_tiles;
  int nt = p.tiles - t0;
  if (nt > p.chunk_tiles) nt = p.chunk_tiles;  // chunk_tiles <= kMaxTiles (host)
  if (nt < 0) nt = 0;

  if (warp == kWarpS) {
    tc05::tmem_alloc(tslot, kTmemCols);
    tc05::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&bars[kBarQ], 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[kBarFullS + s], 1);
      mbar_init(&bars[kBarFullPv + s], 1);
      mbar_init(&bars[kBarEmpty + s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kBarS + s], 1);
      mbar_init(&bars[kBarP + s], 128);
      mbar_init(&bars[kBarPv + s], 1);
      mbar_init(&bars[kBarDone + s], 1);
    }
    mbar_init(&bars[kBarO], 1);
    *abort_flag = 0;
    fence_mbar_init();
    // Q is an input of the call: its load may start before the kernels this
    // one depends on have finished
    tc05::prefetch_tmap(&tq);
    mbar_arrive_expect_tx(&bars[kBarQ], G::kChunks * kChunkBytes);
    const int b = unit / p.Sq, i = unit % p.Sq;
#pragma unroll 1
    for (int c = 0; c < G::kChunks; ++c)
      tc05::tma_load3(sm + G::kOffQ + c * kChunkBytes, &tq, 64 * c, i, b * p.Hq + hb * kHeads,
                      &bars[kBarQ]);
  }
  pdl_wait();  // the planned positions and the decoded keys
  // validity bit masks of this split's tiles: word 4j + k, bit i = key 32k + i
  const int64_t vbase = static_cast<int64_t>(unit) * p.n_cand_pad + static_cast<int64_t>(t0) * kKeys;
  for (int w = warp; w < 4 * nt; w += kThreads / 32) {
    const bool v = p.valid_u8 ? __ldg(p.valid_u8 + vbase + 32 * w + lane) != 0
                              : __ldg(p.pos + vbase + 32 * w + lane) >= 0;
    const uint32_t m = __ballot_sync(0xffffffffu, v);
    if (lane == 0) valid[w] = m;
  }
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  const uint32_t tmem = *tslot;

  if (warp == kWarpLoad) {
    if (lane == 0) fp8tc_producer<G>(&tk, p, unit, t0, nt, part, sm, bars, abort_flag);
  } else if (warp == kWarpS) {
    if (lane == 0) fp8tc_score_lane<G>(p, nt, sm, bars, tmem, abort_flag);
  } else if (warp == kWarpPv) {
    if (lane == 0) fp8tc_pv_lane<G>(p, nt, sm, bars, tmem, abort_flag);
  } else if (warp >= kWarpSoftmax) {
    fp8tc_softmax<G, kCap, kBias>(p, unit, hb, split, nt, part, valid, bars, tmem, abort_flag);
  }

  tc05::fence_before_sync();
  __syncwarp();
  if (p.splits > 1 && p.cluster_merge) {
    cluster_sync();  // every CTA's O rows staged
    fp8tc_cluster_merge<G>(p, unit, hb, part, sm);
    cluster_sync();  // no CTA leaves while another reads its shared memory
  } else {
    __syncthreads();
  }
  if (warp == kWarpS) {
    tc05::fence_after_sync();
    tc05::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- host side -----------------------------------------------------------------------------

int fp8_tc_max_tiles() { return kMaxTiles; }
size_t fp8_tc_decoded_row_bytes() { return kRowBytes; }

bool fp8_tc_supported(const GatherArgs& g) {
  if (g.fp8_warp_mma) return false;  // the caller asked for the warp-level MMA kernel
  if (g.bias) return false;          // an additive bias runs on the warp-level MMA kernel
  if (g.D != kD || g.Dv != kD || g.Hkv != 1 || g.Hq % kHeads != 0) return false;
  if (!(g.scale_log2 > 0.0f) || !std::isfinite(g.scale_log2)) return false;  // monotone logits
  if (g.n_cand < 1 || g.record_stride < 648 || g.record_stride % 8 != 0) return false;
  if (g.B * g.Hq * g.Sq >= (int64_t(1) << 31)) return false;
  return encode_tiled() != nullptr;
}

static bool bf16_map(CUtensorMap* m, const void* base, const cuuint64_t (&dims)[3],
                     const cuuint64_t (&strides)[2], const cuuint32_t (&box)[3]) {
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_tiled()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch that may begin while the previous kernel in the stream finishes
// (programmatic dependent launch; the kernel waits for that kernel's results
// itself, griddepcontrol.wait, before reading them), optionally as clusters
// of `cluster` CTAs.
template <typename K, typename... Args>
static int launch_pdl(K kernel, unsigned grid, unsigned block, size_t smem, cudaStream_t st,
                      unsigned cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  unsigned n = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess ? 0 : -1;
}

template <class G, bool kCap, bool kBias>
static bool set_smem() {
  return cudaFuncSetAttribute(fp8_tc05_kernel<G, kCap, kBias>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmem) == cudaSuccess;
}

// How many clusters of `c` CTAs of the attention kernel (geometry G) can be
// resident at once on this device (a cluster needs c SMs of one GPC)?  Asked
// once per geometry and size.
template <class G>
static int max_active_clusters(int c) {
  static std::once_flag once[kMaxClusterSplits + 1];
  static int ok[kMaxClusterSplits + 1];
  std::call_once(once[c], [c] {
    ok[c] = 0;
    if (!set_smem<G, false, false>() || !set_smem<G, true, false>() ||
        !set_smem<G, false, true>())
      return;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(c));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = G::kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(c);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fp8_tc05_kernel<G, false, false>, &cfg) == cudaSuccess)
      ok[c] = n;
    cudaGetLastError();  // a refused query leaves no sticky error behind
  });
  return ok[c];
}

// The splits of each output block merge on chip when they can form clusters
// and all `blocks` clusters are resident at once (a second wave of clusters
// would cost more than the separate combine).
bool fp8_tc_cluster_merge(int64_t splits, int64_t blocks) {
  if (splits < 2 || splits > kMaxClusterSplits) return false;
  return max_active_clusters<GeoFp8>(static_cast<int>(splits)) >= blocks;
}

int launch_fp8_tc(const GatherArgs& g, cudaStream_t st) {
  if (!fp8_tc_supported(g) || !g.fp8_kdec) return -1;
  const bool cluster = fp8_tc_cluster_merge(g.splits, g.units * (g.Hq / kHeads) * GeoFp8::kParts);
  if (g.splits > 1 && !cluster && (!g.part_o || !g.part_ml)) return -1;
  if (g.n_cand_pad % kKeys != 0 || g.chunk > kMaxTiles || g.chunk < 1) return -1;
  const int64_t rows = g.units * g.n_cand_pad;
  if (rows <= 0) return 0;
  // kernel 1: decoded rows [units, n_cand_pad, 576]
  DecodeParams d;
  d.recs = static_cast<const char*>(g.k);
  d.record_stride = g.record_stride;
  d.T = g.T;
  d.pos = g.pos;
  d.rows = rows;
  d.n_cand_pad = g.n_cand_pad;
  d.Sq = static_cast<int>(g.Sq);
  d.kdec = static_cast<__nv_bfloat16*>(g.fp8_kdec);
  d.err_word = g.err_word;
  d.own_positions = g.fp8_own_positions;
  d.after_plan = g.fp8_after_plan;
  d.pos_out = const_cast<int32_t*>(g.pos);
  d.idx = g.idx;
  d.idx_is_i64 = g.idx_is_i64;
  d.causal = g.causal;
  d.K = g.K;
  d.window = g.window;
  d.past_len = g.past_len;
  d.kv_len = g.kv_len;
  if (g.fp8_own_positions && (g.I != 1 || g.Hkv != 1 || (g.K > 0 && !g.idx))) return -1;
  const int64_t per_cta = 8 * kDecRecs;
  const size_t dsmem = kDecSmem;
  if (cudaFuncSetAttribute(fp8_gather_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(dsmem)) != cudaSuccess ||
      launch_pdl(fp8_gather_decode_kernel, static_cast<unsigned>((rows + per_cta - 1) / per_cta), 256,
                 dsmem, st, 1u, d) != 0)
    return -1;
  // kernel 2: Q as [B * Hq][Sq][576] in boxes of 64 dims x 1 position x 128
  // heads; decoded keys as [units][n_cand_pad][576] in boxes of 64 dims x 128 keys
  CUtensorMap tq, tk;
  const cuuint64_t qdims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(g.Sq),
                               static_cast<cuuint64_t>(g.B * g.Hq)};
  const cuuint64_t qstr[2] = {static_cast<cuuint64_t>(kRowBytes),
                              static_cast<cuuint64_t>(g.Sq * kRowBytes)};
  const cuuint32_t qbox[3] = {64, 1, static_cast<cuuint32_t>(kHeads)};
  const cuuint64_t kdims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(g.n_cand_pad),
                               static_cast<cuuint64_t>(g.units)};
  const cuuint64_t kstr[2] = {static_cast<cuuint64_t>(kRowBytes),
                              static_cast<cuuint64_t>(g.n_cand_pad * kRowBytes)};
  const cuuint32_t kbox[3] = {64, static_cast<cuuint32_t>(kKeys), 1};
  if (!bf16_map(&tq, g.q, qdims, qstr, qbox) || !bf16_map(&tk, g.fp8_kdec, kdims, kstr, kbox))
    return -1;
  Fp8TcParams p = {};
  p.pos = g.pos;
  p.n_cand_pad = g.n_cand_pad;
  p.y = g.y;
  p.part_o = g.part_o;
  p.part_ml = g.part_ml;
  p.sink = g.sink;
  p.err_word = g.err_word;
  p.B = static_cast<int>(g.B);
  p.Sq = static_cast<int>(g.Sq);
  p.Hq = static_cast<int>(g.Hq);
  p.hblocks = static_cast<int>(g.Hq / kHeads);
  p.splits = static_cast<int>(g.splits);
  p.chunk_tiles = static_cast<int>(g.chunk);
  p.tiles = static_cast<int>(g.tiles_per_unit);
  p.cluster_merge = cluster ? 1 : 0;
  p.scale_log2 = g.scale_log2;
  const float log2e = 1.4426950408889634f;
  p.k1 = g.softcap != 0.0f ? (g.scale_log2 / log2e) * g.inv_softcap : 0.0f;
  p.c_log2 = g.softcap * log2e;
  using G = GeoFp8;
  const unsigned grid = static_cast<unsigned>(g.units * p.hblocks * G::kParts * g.splits);
  const unsigned cl = cluster ? static_cast<unsigned>(g.splits) : 1u;
  if (!(g.softcap != 0.0f ? set_smem<G, true, false>() : set_smem<G, false, false>())) return -1;
  mark_event(g.ev_before, st);
  const int rc =
      g.softcap != 0.0f
          ? launch_pdl(fp8_tc05_kernel<G, true, false>, grid, kThreads, G::kSmem, st, cl, tq, tk, p)
          : launch_pdl(fp8_tc05_kernel<G, false, false>, grid, kThreads, G::kSmem, st, cl, tq, tk,
                       p);
  mark_event(g.ev_after, st);
  return rc;
}

// ---- compressed sparse attention rows (D = 512) on the same kernel -------------------------

bool csa_tc_supported(int64_t D, int64_t H, int q_dtype) {
  return D == GeoCsa::kD && H % kHeads == 0 && q_dtype == SA_BF16 && encode_tiled() != nullptr;
}

int csa_tc_max_tiles() { return kMaxTiles; }

// The assembled candidate rows [units, c_pad, 512] bf16 with their validity
// bytes: a (query, head block, half of the output dims, key split) per CTA,
// the query block read as [units * H][512] (one query position per unit).
int launch_csa_tc(const CsaArgs& a, cudaStream_t st, bool* merged) {
  using G = GeoCsa;
  const int64_t units = a.B * a.S;
  // the splits of an output block merge on chip when all blocks' clusters are resident at once
  const int64_t blocks = units * (a.H / kHeads) * G::kParts;
  const bool cluster = a.splits >= 2 && a.splits <= kMaxClusterSplits &&
                       max_active_clusters<G>(static_cast<int>(a.splits)) >= blocks;
  *merged = cluster || a.splits == 1;
  if (!csa_tc_supported(a.D, a.H, a.q_dtype) || a.c_pad % kKeys != 0 || a.chunk_tiles < 1 ||
      a.chunk_tiles > kMaxTiles || (a.splits > 1 && !cluster && (!a.part_o || !a.part_ml)))
    return -1;
  CUtensorMap tq, tk;
  const cuuint64_t qdims[3] = {static_cast<cuuint64_t>(G::kD), 1,
                               static_cast<cuuint64_t>(units * a.H)};
  const cuuint64_t qstr[2] = {static_cast<cuuint64_t>(G::kD * 2),
                              static_cast<cuuint64_t>(G::kD * 2)};
  const cuuint32_t qbox[3] = {64, 1, static_cast<cuuint32_t>(kHeads)};
  const cuuint64_t kdims[3] = {static_cast<cuuint64_t>(G::kD), static_cast<cuuint64_t>(a.c_pad),
                               static_cast<cuuint64_t>(units)};
  const cuuint64_t kstr[2] = {static_cast<cuuint64_t>(G::kD * 2),
                              static_cast<cuuint64_t>(a.c_pad * G::kD * 2)};
  const cuuint32_t kbox[3] = {64, static_cast<cuuint32_t>(kKeys), 1};
  if (!bf16_map(&tq, a.query, qdims, qstr, qbox) || !bf16_map(&tk, a.rows, kdims, kstr, kbox))
    return -1;
  Fp8TcParams p = {};
  p.pos = nullptr;
  p.valid_u8 = a.valid;
  p.bias = a.bias;
  p.bias_sb = a.bias_sb;
  p.bias_sh = a.bias_sh;
  p.bias_si = a.bias_si;
  p.bias_sk = a.bias_sk;
  p.bias_S = static_cast<int>(a.S);
  p.n_cand_pad = a.c_pad;
  p.y = a.y;
  p.part_o = a.part_o;
  p.part_ml = a.part_ml;
  p.sink = a.sink;
  p.err_word = a.err_word;
  p.B = static_cast<int>(units);
  p.Sq = 1;
  p.Hq = static_cast<int>(a.H);
  p.hblocks = static_cast<int>(a.H / kHeads);
  p.splits = static_cast<int>(a.splits);
  p.chunk_tiles = static_cast<int>(a.chunk_tiles);
  p.tiles = static_cast<int>(a.c_pad / kKeys);
  p.cluster_merge = cluster ? 1 : 0;
  p.scale_log2 = a.scale_log2;
  const unsigned grid = static_cast<unsigned>(units * p.hblocks * G::kParts * a.splits);
  const unsigned cl = cluster ? static_cast<unsigned>(a.splits) : 1u;
  const bool bias = a.bias != nullptr;
  if (!(bias ? set_smem<G, false, true>() : set_smem<G, false, false>())) return -1;
  mark_event(a.ev_before, st);
  const int rc =
      bias ? launch_pdl(fp8_tc05_kernel<G, false, true>, grid, kThreads, G::kSmem, st, cl, tq, tk, p)
           : launch_pdl(fp8_tc05_kernel<G, false, false>, grid, kThreads, G::kSmem, st, cl, tq, tk,
                        p);
  mark_event(a.ev_after, st);
  return rc;
}

}  // namespace sa
