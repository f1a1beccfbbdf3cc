// k_prefill.cu -- dense (causal) prefill attention on the fifth-generation
// tensor cores: tcgen05.mma with accumulators in tensor memory, operands
// staged by TMA.
//
// Semantics: ONNX Attention as the standard attention page gives it
// (onnx-runtime-ep-cuda standard_attention.rs, `attention_row`): with no
// past, query i of head h attends to keys 0..i (causal) of KV head h / g;
// score = scale * q.k, then softcap * tanh(score / softcap) when softcap is
// set, then the causal mask, an fp32 softmax, and the probability-weighted
// sum of V rows.
//
// GB300 design (one persistent CTA per SM, 12 warps):
//  * A work item is two 128-row query tiles that read the same K/V stream:
//    two query heads of one GQA group at the same positions, or (odd group
//    sizes) neighbouring entries of the group's (position tile, head) list.
//    Items go to CTAs in a snake order of decreasing causal length.
//  * Warp 0 (one lane) is the TMA producer: the two Q tiles, then K_0, V_0,
//    K_1, V_1, ... through a ring of 32 KB slots, every tile a set of
//    128-byte-swizzled 64-column slabs.
//  * Warp 1 owns the 512 TMEM columns and one lane issues every MMA:
//    S_x = Q_x K_j^T (128 x 128 x D, both operands K-major from shared
//    memory) and O_x += P_x V_j (P from tensor memory, V MN-major).
//  * Warps 4-7 and 8-11 are the softmax warpgroups of tiles a and b; thread
//    r owns row r (TMEM lane r).  Per KV tile it loads its S row, applies the
//    scale / softcap (tanh.approx) / mask, keeps a running maximum that is
//    raised only when a new score exceeds it by more than 2^8 (rescaling its
//    O row in TMEM then), writes P = 2^(s - m) as 16-bit pairs over the S
//    columns, and finally normalises its O row and stores it.
//  * P aliases S: the MMA issuing order PV_x(j) -> S_x(j+1) keeps the read of
//    P ahead of the next write of S.
//  * Every mbarrier wait is bounded; a stalled pipeline sets
//    SA_ERRBIT_TIMEOUT, stops every role, and still frees the tensor memory.
#include <cuda.h>

#include <cmath>
#include <mutex>
#include <type_traits>

#include "kernels.h"
#include "tc05.cuh"

namespace sa {

namespace {

constexpr int kThreads = 384;
constexpr int kTile = 128;          // query rows and keys per tile
constexpr int kSlabBytes = kTile * 128;  // 128 rows x 64 sixteen-bit columns
constexpr float kRescaleLog2 = 8.0f;     // lazy-maximum slack (factor 256)

template <int D>
struct PGeo {
  static constexpr int kSlabs = D / 64;
  static constexpr int kTileBytes = kSlabs * kSlabBytes;        // 16 or 32 KB
  static constexpr int kStages = D == 128 ? 4 : 8;              // K/V ring slots
  static constexpr int kOffQ = 0;                               // Q_a, Q_b
  static constexpr int kOffRing = 2 * kTileBytes;
  static constexpr int kOffBar = kOffRing + kStages * kTileBytes;
  // barriers: q_full, q_empty, kv_full[kStages], kv_empty[kStages],
  // s_full[2], p_full[2], o_full[2], done
  static constexpr int kBarQFull = 0, kBarQEmpty = 1, kBarKvFull = 2,
                       kBarKvEmpty = 2 + kStages, kBarS = 2 + 2 * kStages,
                       kBarP = kBarS + 2, kBarO = kBarP + 2, kBarDone = kBarO + 2,
                       kNumBars = kBarDone + 1;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemUsed = kOffAbort + 4;
  static constexpr int kSmem = kSmemUsed + 1024;                // 1024-byte alignment slack
  // tensor memory columns
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
  static constexpr uint32_t kTmemCols = 512;
};

// Kernel parameters (besides the three tensor maps).
struct PrefillKParams {
  void* y;
  uint32_t* err_word;
  int B, Hq, Hkv, S, g;
  int nq;             // query / key tiles per head: ceil(S / 128)
  int pairs;          // items per (b, kvh): ceil(nq * g / 2)
  int n_items;        // B * Hkv * pairs
  int causal;
  int softcap_on;     // selects the kernel instantiation
  float k1;           // score multiplier before tanh (scale / softcap), or 1
  float c_log2;       // log2-domain multiplier after it (softcap * log2e or scale * log2e)
};

struct Item {
  int b, kvh;
  int head[2], qt[2], n[2];
  int has_b;
  int n_max;
};

// Item w: (b, kvh) = w % (B * Hkv); its pair index counts down with w / (B *
// Hkv) so that longer causal items come first.  The group's query tiles are
// listed position-tile major, (qt, hh) -> qt * g + hh, and paired in order.
__device__ __forceinline__ Item item_of(int w, const PrefillKParams& p) {
  Item it;
  const int bk_n = p.B * p.Hkv;
  const int bk = w % bk_n;
  const int pair = p.pairs - 1 - w / bk_n;
  it.b = bk / p.Hkv;
  it.kvh = bk % p.Hkv;
  const int total = p.nq * p.g;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    const int e = 2 * pair + x;
    const int ee = e < total ? e : total - 1;
    it.qt[x] = ee / p.g;
    it.head[x] = it.kvh * p.g + ee % p.g;
    it.n[x] = p.causal ? it.qt[x] + 1 : p.nq;
  }
  it.has_b = (2 * pair + 1) < total;
  if (!it.has_b) it.n[1] = 0;
  it.n_max = it.n[0] > it.n[1] ? it.n[0] : it.n[1];
  return it;
}

// Snake assignment: round k of the persistent loop gives CTA c item
// k * G + c (even k) or k * G + G - 1 - c (odd k).
__device__ __forceinline__ int item_index(int k, int G) {
  const int c = static_cast<int>(blockIdx.x);
  return k * G + ((k & 1) ? G - 1 - c : c);
}

// Bounded wait that turns a timeout into a CTA-wide abort.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag, uint32_t* err_word) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity)) return true;
  *abort_flag = 1;
  if (err_word) atomicOr(err_word, static_cast<uint32_t>(SA_ERRBIT_TIMEOUT));
  return false;
}

// The same, with one verdict for the whole warp (its lanes then stay converged
// for the warp-collective tensor-memory instructions that follow).
__device__ __forceinline__ bool wait_or_abort_warp(uint64_t* bar, uint32_t parity,
                                                   volatile int* abort_flag, uint32_t* err_word) {
  const bool ok = wait_or_abort(bar, parity, abort_flag, err_word);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace

namespace {

// ---- role: TMA producer (one lane) ------------------------------------------------------

template <int D>
__device__ void prefill_producer(const CUtensorMap* tq, const CUtensorMap* tk,
                                 const CUtensorMap* tv, const PrefillKParams& p, uint8_t* sm,
                                 uint64_t* bars, volatile int* abort_flag) {
  using G = PGeo<D>;
  tc05::prefetch_tmap(tq);
  tc05::prefetch_tmap(tk);
  tc05::prefetch_tmap(tv);
  uint32_t kv_cnt = 0, q_cnt = 0;
  for (int k = 0;; ++k) {
    const int w = item_index(k, static_cast<int>(gridDim.x));
    if (w >= p.n_items) break;
    const Item it = item_of(w, p);
    if (q_cnt > 0 && !wait_or_abort(&bars[G::kBarQEmpty], (q_cnt - 1) & 1, abort_flag, p.err_word))
      break;
    mbar_arrive_expect_tx(&bars[G::kBarQFull], (it.has_b ? 2u : 1u) * G::kTileBytes);
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      if (x == 1 && !it.has_b) break;
#pragma unroll
      for (int s = 0; s < G::kSlabs; ++s)
        tc05::tma_load3(sm + G::kOffQ + x * G::kTileBytes + s * kSlabBytes, tq, s * 64,
                        it.qt[x] * kTile, it.b * p.Hq + it.head[x], &bars[G::kBarQFull]);
    }
    ++q_cnt;
    const int z = it.b * p.Hkv + it.kvh;
    bool stop = false;
    for (int j = 0; j < it.n_max && !stop; ++j) {
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        const uint32_t slot = kv_cnt % G::kStages, use = kv_cnt / G::kStages;
        if (use > 0 && !wait_or_abort(&bars[G::kBarKvEmpty + slot], (use - 1) & 1, abort_flag,
                                      p.err_word)) {
          stop = true;
          break;
        }
        mbar_arrive_expect_tx(&bars[G::kBarKvFull + slot], G::kTileBytes);
#pragma unroll
        for (int s = 0; s < G::kSlabs; ++s)
          tc05::tma_load3(sm + G::kOffRing + slot * G::kTileBytes + s * kSlabBytes,
                          kv ? tv : tk, s * 64, j * kTile, z, &bars[G::kBarKvFull + slot]);
        ++kv_cnt;
      }
    }
    if (stop) break;
  }
  if (*abort_flag) {
    // Let every copy already issued land before the CTA can exit.
    if (q_cnt > 0) mbar_wait(&bars[G::kBarQFull], (q_cnt - 1) & 1);
    for (uint32_t s = 0; s < G::kStages; ++s) {
      if (kv_cnt <= s) break;
      const uint32_t issued = (kv_cnt - s + G::kStages - 1) / G::kStages;
      mbar_wait(&bars[G::kBarKvFull + s], (issued - 1) & 1);
    }
  }
}

// ---- role: MMA issuer (one lane) ----------------------------------------------------

template <int D, bool kBf16>
__device__ void prefill_mma(const PrefillKParams& p, uint8_t* sm, uint64_t* bars, uint32_t tmem,
                            volatile int* abort_flag) {
  using G = PGeo<D>;
  constexpr uint32_t id_s = tc05::idesc_f16(kTile, kTile, kBf16, false, false);
  constexpr uint32_t id_o = tc05::idesc_f16(kTile, D, kBf16, false, true);
  const uint32_t sQ = smem_u32(sm + G::kOffQ), sRing = smem_u32(sm + G::kOffRing);
  const uint32_t colS[2] = {G::kColS0, G::kColS1}, colO[2] = {G::kColO0, G::kColO1};

  auto issue_s = [&](int x, uint32_t slot) {
    const uint32_t a0 = sQ + x * G::kTileBytes, b0 = sRing + slot * G::kTileBytes;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk / 4) * kSlabBytes + (kk % 4) * 32;
      tc05::mma_ss(tmem + colS[x], tc05::sw128_desc(a0 + off, 16, 1024),
                   tc05::sw128_desc(b0 + off, 16, 1024), id_s, kk > 0 ? 1u : 0u);
    }
  };
  auto issue_pv = [&](int x, uint32_t slot, bool acc) {
    const uint32_t v0 = sRing + slot * G::kTileBytes;
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk)
      tc05::mma_ts(tmem + colO[x], tmem + colS[x] + kk * 8,
                   tc05::sw128_desc(v0 + kk * 2048, kSlabBytes, 1024), id_o,
                   (acc || kk > 0) ? 1u : 0u);
  };

  uint32_t kv_cnt = 0, q_cnt = 0, p_cnt[2] = {0, 0};
  for (int k = 0;; ++k) {
    const int w = item_index(k, static_cast<int>(gridDim.x));
    if (w >= p.n_items) break;
    const Item it = item_of(w, p);
    if (!wait_or_abort(&bars[G::kBarQFull], q_cnt & 1, abort_flag, p.err_word)) break;
    ++q_cnt;
    uint32_t slotK = kv_cnt % G::kStages;
    if (!wait_or_abort(&bars[G::kBarKvFull + slotK], (kv_cnt / G::kStages) & 1, abort_flag,
                       p.err_word))
      break;
    ++kv_cnt;
    tc05::fence_after_sync();
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      if (it.n[x] > 0) {
        issue_s(x, slotK);
        tc05::commit(&bars[G::kBarS + x]);
      }
    }
    tc05::commit(&bars[G::kBarKvEmpty + slotK]);
    bool stop = false;
    for (int j = 0; j < it.n_max && !stop; ++j) {
      const uint32_t slotV = kv_cnt % G::kStages;
      if (!wait_or_abort(&bars[G::kBarKvFull + slotV], (kv_cnt / G::kStages) & 1, abort_flag,
                         p.err_word)) {
        stop = true;
        break;
      }
      ++kv_cnt;
      const bool has_next = j + 1 < it.n_max;
      if (has_next) {
        slotK = kv_cnt % G::kStages;
        if (!wait_or_abort(&bars[G::kBarKvFull + slotK], (kv_cnt / G::kStages) & 1, abort_flag,
                           p.err_word)) {
          stop = true;
          break;
        }
        ++kv_cnt;
      }
      tc05::fence_after_sync();
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (j < it.n[x]) {
          if (!wait_or_abort(&bars[G::kBarP + x], p_cnt[x] & 1, abort_flag, p.err_word)) {
            stop = true;
            break;
          }
          ++p_cnt[x];
          tc05::fence_after_sync();
          issue_pv(x, slotV, j > 0);
          if (j == it.n[x] - 1) tc05::commit(&bars[G::kBarO + x]);
        }
        if (has_next && j + 1 < it.n[x]) {
          issue_s(x, slotK);
          tc05::commit(&bars[G::kBarS + x]);
        }
      }
      if (stop) break;
      tc05::commit(&bars[G::kBarKvEmpty + slotV]);
      if (has_next) tc05::commit(&bars[G::kBarKvEmpty + slotK]);
    }
    if (stop) break;
    tc05::commit(&bars[G::kBarQEmpty]);
  }
  // Every MMA issued above completes before the tensor memory is released.
  tc05::commit(&bars[G::kBarDone]);
  mbar_wait(&bars[G::kBarDone], 0);
}

}  // namespace

namespace {

// ---- role: softmax warpgroup (tile x; thread = one query row) ---------------------------

// O row *= alpha, in tensor memory (warp-collective).
template <int D>
__device__ __forceinline__ void rescale_o_row(uint32_t tO, float alpha) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    tc05::tmem_ld32(tO + c * 32, o);
    tc05::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
    tc05::tmem_st32(tO + c * 32, o);
  }
  tc05::tmem_st_wait();
}

// In place over the 128 raw scores of a row: t = tanh(s * k1) (softcap) or
// t = s, masked columns (> rel) to -inf; returns max t.
template <bool kSoftcap, bool kMask>
__device__ __forceinline__ float score_pass(uint32_t (&r)[4][32], float k1, int rel) {
  float mx[4] = {SA_NEG_INF, SA_NEG_INF, SA_NEG_INF, SA_NEG_INF};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      float t = __uint_as_float(r[c][i]);
      if (kSoftcap) t = tanh_approx(t * k1);
      if (kMask && c * 32 + i > rel) t = SA_NEG_INF;
      r[c][i] = __float_as_uint(t);
      mx[i & 3] = fmaxf(mx[i & 3], t);
    }
  }
  return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
}

template <int D, typename T, bool kSoftcap>
__device__ void prefill_softmax(const PrefillKParams& p, uint64_t* bars, uint32_t tmem,
                                volatile int* abort_flag) {
  using G = PGeo<D>;
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const int x = (warp - 4) >> 2;
  const int row = ((warp & 3) << 5) | lane;
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_base + (x ? G::kColS1 : G::kColS0);
  const uint32_t tO = tmem + lane_base + (x ? G::kColO1 : G::kColO0);
  uint64_t* s_full = &bars[G::kBarS + x];
  uint64_t* p_full = &bars[G::kBarP + x];
  uint64_t* o_full = &bars[G::kBarO + x];
  const float c2 = p.c_log2;
  uint32_t s_cnt = 0, o_cnt = 0;

  for (int k = 0;; ++k) {
    const int w = item_index(k, static_cast<int>(gridDim.x));
    if (w >= p.n_items) break;
    const Item it = item_of(w, p);
    const int n = it.n[x];
    if (n == 0) continue;
    const int qi = it.qt[x] * kTile + row;
    const int lim = p.causal ? min(qi, p.S - 1) : p.S - 1;  // last visible key
    float m = SA_NEG_INF, l = 0.0f;
    bool stop = false;
    for (int j = 0; j < n; ++j) {
      if (!wait_or_abort_warp(s_full, s_cnt & 1, abort_flag, p.err_word)) {
        stop = true;
        break;
      }
      ++s_cnt;
      tc05::fence_after_sync();
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc05::tmem_ld32(tS + c * 32, r[c]);
      tc05::tmem_ld_wait();

      // scores -> (softcap) -> mask; row maximum
      const int rel = lim - j * kTile;  // columns above rel are masked
      const float mt =
          (rel < kTile - 1 ? score_pass<kSoftcap, true>(r, p.k1, rel)
                           : score_pass<kSoftcap, false>(r, p.k1, rel)) * c2;

      // lazy maximum: raise it only when the tile's maximum exceeds it by the slack
      const bool raise = mt > m + kRescaleLog2;
      const bool any_raise = __any_sync(0xffffffffu, raise);
      float alpha = 1.0f;
      if (raise) {
        alpha = ex2(m - mt);
        l *= alpha;
        m = mt;
      }
      const float neg_m = m == SA_NEG_INF ? 0.0f : -m;

      // probabilities, written over the S columns as 16-bit pairs
      float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2(fmaf(__uint_as_float(r[c][2 * i]), c2, neg_m));
          const float p1 = ex2(fmaf(__uint_as_float(r[c][2 * i + 1]), c2, neg_m));
          ls[i & 3] += p0 + p1;
          pk[i] = pack2<T>(p0, p1);
        }
        tc05::tmem_st16(tS + c * 16, pk);
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      // O (complete up to tile j - 1: its MMA preceded this S) follows the new maximum
      if (any_raise && j > 0) rescale_o_row<D>(tO, alpha);
      tc05::tmem_st_wait();
      tc05::fence_before_sync();
      mbar_arrive(p_full);
    }
    if (stop) break;

    // epilogue: O row / l -> y
    if (!wait_or_abort_warp(o_full, o_cnt & 1, abort_flag, p.err_word)) break;
    ++o_cnt;
    tc05::fence_after_sync();
    const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
    T* yrow = static_cast<T*>(p.y) +
              ((static_cast<int64_t>(it.b) * p.Hq + it.head[x]) * p.S + qi) * D;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tc05::tmem_ld32(tO + c * 32, o);
      tc05::tmem_ld_wait();
      if (qi < p.S) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack2<T>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        uint4* dst = reinterpret_cast<uint4*>(yrow + c * 32);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
      }
    }
  }
}

// ---- kernel -------------------------------------------------------------------------------

template <int D, typename T, bool kSoftcap>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc05_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv, const PrefillKParams p) {
  using G = PGeo<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + G::kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + G::kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + G::kOffAbort);
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);

  if (threadIdx.x == 0) {
    mbar_init(&bars[G::kBarQFull], 1);
    mbar_init(&bars[G::kBarQEmpty], 1);
    for (int s = 0; s < G::kStages; ++s) {
      mbar_init(&bars[G::kBarKvFull + s], 1);
      mbar_init(&bars[G::kBarKvEmpty + s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars[G::kBarS + x], 1);
      mbar_init(&bars[G::kBarP + x], 128);
      mbar_init(&bars[G::kBarO + x], 1);
    }
    mbar_init(&bars[G::kBarDone], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tc05::tmem_alloc(tslot, G::kTmemCols);
    tc05::tmem_relinquish();
  }
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    if (lane == 0) prefill_producer<D>(&tq, &tk, &tv, p, sm, bars, abort_flag);
  } else if (warp == 1) {
    if (lane == 0)
      prefill_mma<D, std::is_same<T, __nv_bfloat16>::value>(p, sm, bars, tmem, abort_flag);
  } else if (warp >= 4) {
    prefill_softmax<D, T, kSoftcap>(p, bars, tmem, abort_flag);
  }
  __syncwarp();
  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc05::fence_after_sync();
    tc05::tmem_dealloc(tmem, G::kTmemCols);
  }
}

}  // namespace

// ---- host side -----------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// [planes, rows, D] sixteen-bit tensor, boxes of 128 rows x 64 columns with the
// 128-byte swizzle; rows past the end read as zero.
static bool make_tile_map(CUtensorMap* m, const void* base, int dtype, int64_t D, int64_t rows,
                          int64_t planes) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(planes)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D * 2),
                                 static_cast<cuuint64_t>(rows * D * 2)};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kTile), 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m,
             dtype == SA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
             3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool al16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }

bool prefill_tc_supported(const PrefillTcArgs& a) {
  if (a.dtype != SA_BF16 && a.dtype != SA_F16) return false;
  if (a.D != 64 && a.D != 128) return false;
  if (!(a.scale > 0.0f) || !std::isfinite(a.scale) || !std::isfinite(a.softcap)) return false;
  if (!al16(a.q) || !al16(a.k) || !al16(a.v) || !al16(a.y)) return false;
  if (a.S < 1 || a.S > (int64_t(1) << 30)) return false;
  const int64_t nq = (a.S + kTile - 1) / kTile;
  const int64_t g = a.Hq / a.Hkv;
  const int64_t items = a.B * a.Hkv * ((nq * g + 1) / 2);
  if (items >= (int64_t(1) << 30) || a.B * a.Hq >= (int64_t(1) << 30)) return false;
  return encode_tiled() != nullptr;
}

template <int D, typename T>
static int launch_prefill_t(const PrefillTcArgs& a, cudaStream_t st) {
  using G = PGeo<D>;
  CUtensorMap tq, tk, tv;
  if (!make_tile_map(&tq, a.q, a.dtype, D, a.S, a.B * a.Hq) ||
      !make_tile_map(&tk, a.k, a.dtype, D, a.S, a.B * a.Hkv) ||
      !make_tile_map(&tv, a.v, a.dtype, D, a.S, a.B * a.Hkv))
    return -1;
  PrefillKParams p;
  p.y = a.y;
  p.err_word = a.err_word;
  p.B = static_cast<int>(a.B);
  p.Hq = static_cast<int>(a.Hq);
  p.Hkv = static_cast<int>(a.Hkv);
  p.S = static_cast<int>(a.S);
  p.g = static_cast<int>(a.Hq / a.Hkv);
  p.nq = static_cast<int>((a.S + kTile - 1) / kTile);
  p.pairs = (p.nq * p.g + 1) / 2;
  p.n_items = p.B * p.Hkv * p.pairs;
  p.causal = a.causal ? 1 : 0;
  const float log2e = 1.4426950408889634f;
  if (a.softcap != 0.0f) {
    const float cap = std::fabs(a.softcap);
    p.softcap_on = 1;
    p.k1 = a.scale / cap;
    p.c_log2 = cap * log2e;
  } else {
    p.softcap_on = 0;
    p.k1 = 1.0f;
    p.c_log2 = a.scale * log2e;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  const int grid = p.n_items < sms ? p.n_items : sms;
  auto kern = p.softcap_on ? prefill_tc05_kernel<D, T, true> : prefill_tc05_kernel<D, T, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmem) !=
      cudaSuccess)
    return -1;
  kern<<<grid, kThreads, G::kSmem, st>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_prefill_tc(const PrefillTcArgs& a, cudaStream_t st) {
  if (!prefill_tc_supported(a)) return -1;
  if (a.dtype == SA_BF16)
    return a.D == 128 ? launch_prefill_t<128, __nv_bfloat16>(a, st)
                      : launch_prefill_t<64, __nv_bfloat16>(a, st);
  return a.D == 128 ? launch_prefill_t<128, __half>(a, st) : launch_prefill_t<64, __half>(a, st);
}

}  // namespace sa
