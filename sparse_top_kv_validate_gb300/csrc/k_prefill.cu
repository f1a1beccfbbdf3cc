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
// GB300 design (one persistent CTA per SM; warps 0-3 service, 4-11 softmax):
//  * A work item is one 128-row query tile of one head; items go to CTAs in a
//    snake order of decreasing causal length, neighbouring heads of a GQA
//    group side by side so that their K/V reads meet in L2.
//  * Warp 0 (one lane) is the TMA producer: the item's Q tile (two buffers,
//    so the next item's Q arrives early), then the 128-key K and V tiles in
//    the order the MMA lanes consume them through a ring of slots; every tile
//    is a set of 128-byte-swizzled 64-column slabs.
//  * Warp 1 owns the tensor memory -- three 128-column score buffers and the
//    O accumulator.  Two lanes issue the MMAs: warp 1's lane issues S(g) =
//    Q K_g^T (128 x 128 x D, both operands K-major from shared memory) into
//    buffer g % 3 once K_g is in and the buffer's previous P has been read;
//    warp 3's lane issues O += P(g) V_g (P from tensor memory, V MN-major)
//    once P(g) and V_g are in.  tcgen05.mma issue returns only when the
//    tensor core can take the instruction, so with one issuing lane every
//    wait or commit of that lane was tensor-idle time; with two, each waits
//    only on its own inputs while the other keeps the queue fed.  (A 128 x 64
//    MMA costs as long as a 128 x 128 one, so score tiles stay 128 keys
//    wide.)
//  * Warp 2 (one lane) writes the present K/V outputs: the item that reads
//    K/V tile t as its last (diagonal) tile stores it from the ring with TMA.
//  * Two softmax warpgroups split each row's keys (keys 0-63 and 64-127 of a
//    tile); thread r of a group owns row r = TMEM lane r.  Per tile a thread
//    loads its scores, applies scale, softcap and mask, and writes
//    P = 2^(s - m) as 16-bit pairs over its own score columns; at the end the
//    groups add their row sums and each normalises and stores half the O
//    row.  With a softcap the logits are bounded and m is the constant 0
//    (exact: softmax is shift-invariant, and the bound keeps 2^logit and the
//    row sums inside fp32's normal range); otherwise m is a running maximum
//    shared by the groups and raised only when a tile's maximum exceeds it by
//    more than 2^8, O then rescaled in TMEM after the previous PV completed.
//  * The softcap's tanh runs on the FMA pipes as a fitted odd polynomial
//    (paired fp32 arithmetic) for about two thirds of every thread's scores
//    and on the MUFU tanh for the rest, so that neither pipe -- the MUFU one
//    also carries the exponentials -- bounds the kernel; a warp whose tile
//    holds a |score / softcap| outside the fitted range uses the MUFU tanh
//    throughout.
//  * Every mbarrier wait is bounded; a stalled pipeline sets
//    SA_ERRBIT_TIMEOUT, stops every role, and still frees the tensor memory.
#include <cuda.h>

#include <cmath>
#include <mutex>
#include <type_traits>
#include <utility>

#include "kernels.h"
#include "tc05.cuh"

namespace sa {

namespace {

#ifndef SA_PREFILL_GROUPS
#define SA_PREFILL_GROUPS 2
#endif
constexpr int kGroups = SA_PREFILL_GROUPS;  // softmax warpgroups, each a share of every key tile
constexpr int kThreads = 128 * (1 + kGroups);
constexpr int kTile = 128;               // query rows per tile; keys per K/V tile
constexpr int kGroupKeys = kTile / kGroups;  // keys of a tile per softmax warpgroup
constexpr int kSlabBytes = kTile * 128;  // 128 rows x 64 sixteen-bit columns
constexpr float kRescaleLog2 = 8.0f;     // lazy-maximum slack (factor 256)
constexpr int kSBufs = 3;                // score buffers in tensor memory
constexpr int kLead = kSBufs - 1;        // S(j + kLead) is issued before PV(j)
constexpr int kTanhTerms = 5;            // tanh(x) ~= x * sum_k c_k (x^2)^k
constexpr float kTanhPolyBound = 0.625f; // |x| range of the fit (abs error ~1e-7)
// Largest softcap * log2(e) for which 2^(logit) needs no offset: logits in
// [-97, 97] keep every probability a normal fp32 number and row sums over up
// to 2^30 keys below 2^127.
constexpr float kFixedOffsetMaxLog2 = 97.0f;

template <int D>
struct PGeo {
  static constexpr int kSlabs = D / 64;
  static constexpr int kTileBytes = kSlabs * kSlabBytes;        // 16 or 32 KB
#ifndef SA_PREFILL_QBUF
#define SA_PREFILL_QBUF 2
#endif
#ifndef SA_PREFILL_STAGES128
#define SA_PREFILL_STAGES128 4
#endif
  static constexpr int kQBufs = SA_PREFILL_QBUF;                // Q buffers (next item's Q early)
  static constexpr int kStages = D == 128 ? SA_PREFILL_STAGES128 : 8;  // K/V ring slots
  static constexpr int kOffQ = 0;
  static constexpr int kOffRing = kQBufs * kTileBytes;
  static constexpr int kOffXch = kOffRing + kStages * kTileBytes;  // [2 rounds][groups][128] f32
  static constexpr int kOffBar = kOffXch + 2 * kGroups * kTile * 4;
  // barriers: q_full[2], q_empty[2] (per Q buffer), kv_full[kStages],
  // kv_empty[kStages], s_full[3], p_full[3], pv_free[3] (per score buffer:
  // the PV that read its P has completed), o_full, xch[2] (softmax groups, per
  // exchange round parity), done[2] (per MMA lane).  A buffer is refilled
  // only after its previous contents were consumed, so no barrier that is
  // waited on phase by phase ever has two phases outstanding.
  static constexpr int kBarQFull = 0, kBarQEmpty = 2, kBarKvFull = 4,
                       kBarKvEmpty = kBarKvFull + kStages, kBarS = kBarKvEmpty + kStages,
                       kBarP = kBarS + kSBufs, kBarPv = kBarP + kSBufs, kBarO = kBarPv + kSBufs,
                       kBarXch = kBarO + 1, kBarDone = kBarXch + 2, kNumBars = kBarDone + 2;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemUsed = kOffAbort + 4;
  static constexpr int kSmem = kSmemUsed + 1024;                // 1024-byte alignment slack
  // tensor memory columns: score buffers 0, 1, 2, then O
  static constexpr uint32_t kColS = 0, kColO = kSBufs * kTile;
  static constexpr uint32_t kTmemCols = 512;
};

// Kernel parameters (besides the three tensor maps).
struct PrefillKParams {
  void* y;
  uint32_t* err_word;
  int write_present;  // bit 0: present_k, bit 1: present_v (through their tensor maps)
  int B, Hq, Hkv, S, g;
  int nq;             // query / key tiles per head: ceil(S / 128)
  int n_items;        // B * Hq * nq
  int causal;
  int softcap_on;     // 0 none, 1 softcap with a running maximum, 2 softcap, constant offset
  float k1;           // x = score * k1 (scale / softcap), or the raw score
  float c_log2;       // log2-domain multiplier of tanh(x) (softcap * log2e) or of x (scale * log2e)
  float tq[kTanhTerms];  // c_log2 * c_k: the tanh polynomial already in log2 units
  const int64_t* nonpad;  // nullable [B]: padding frontier (keys >= nonpad masked, causal
                          // offset nonpad - S)
};

// Last key query qi of batch b may see (< 0: none): S - 1, or the causal
// frontier (shifted by the padding frontier's offset), or the padding frontier.
__device__ __forceinline__ int last_key(const PrefillKParams& p, int b, int qi) {
  int lim = p.S - 1;
  int off = 0;
  if (p.nonpad) {
    const int64_t np = __ldg(p.nonpad + b);
    if (np >= 0 && np - 1 < lim) lim = static_cast<int>(np - 1);
    off = static_cast<int>(max(min(np - p.S, int64_t(1) << 30), -(int64_t(1) << 30)));
  }
  if (p.causal) lim = min(lim, qi + off);
  return lim;
}

struct Item {
  int b, h, kvh, qt, n;   // n: KV tiles the query tile reads
};

// Item w: (b, h) = w % (B * Hq), query tile counting down with w / (B * Hq) so
// that longer causal items come first.
__device__ __forceinline__ Item item_of(int w, const PrefillKParams& p) {
  Item it;
  const int bh_n = p.B * p.Hq;
  const int bh = w % bh_n;
  it.qt = p.nq - 1 - w / bh_n;
  it.b = bh / p.Hq;
  it.h = bh % p.Hq;
  it.kvh = it.h / p.g;
  if (!p.nonpad) {
    it.n = p.causal ? it.qt + 1 : p.nq;
  } else {
    // tiles up to the tile's last visible key; at least one (its rows may all
    // be masked, and then give 0)
    const int lim = last_key(p, it.b, min(it.qt * kTile + kTile - 1, p.S - 1));
    it.n = lim < 0 ? 1 : min(lim / kTile + 1, p.nq);
  }
  return it;
}

// Snake assignment: round k of the persistent loop gives CTA c item
// k * G + c (even k) or k * G + G - 1 - c (odd k).
__device__ __forceinline__ int item_index(int k, int G) {
  const int c = static_cast<int>(blockIdx.x);
  return k * G + ((k & 1) ? G - 1 - c : c);
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
  bool stop = false;
  for (int k = 0; !stop; ++k) {
    const int w = item_index(k, static_cast<int>(gridDim.x));
    if (w >= p.n_items) break;
    const Item it = item_of(w, p);
    // Q buffer qb is free once the last S MMA of its previous item has completed.
    const uint32_t qb = q_cnt % G::kQBufs, quse = q_cnt / G::kQBufs;
    if (quse > 0 &&
        !wait_or_abort(&bars[G::kBarQEmpty + qb], (quse - 1) & 1, abort_flag, p.err_word))
      break;
    mbar_arrive_expect_tx(&bars[G::kBarQFull + qb], G::kTileBytes);
#pragma unroll
    for (int s = 0; s < G::kSlabs; ++s)
      tc05::tma_load3(sm + G::kOffQ + qb * G::kTileBytes + s * kSlabBytes, tq, s * 64,
                      it.qt * kTile, it.b * p.Hq + it.h, &bars[G::kBarQFull + qb]);
    ++q_cnt;
    // K/V tiles in the order the MMA lane consumes them: K_0 .. K_(kLead-1),
    // then per tile j: K_(j+kLead) (if any), V_j.
    const int z = it.b * p.Hkv + it.kvh;
    const int n = it.n;
    for (int e = 0; e < 2 * n && !stop; ++e) {
      // entry e -> (is_v, t): the first kLead entries are K tiles; after them
      // the pairs (K_(j+kLead), V_j) while j + kLead < n, then the last V's.
      bool is_v;
      int t;
      const int nk0 = n < kLead ? n : kLead;
      if (e < nk0) {
        is_v = false;
        t = e;
      } else if (e < nk0 + 2 * (n - nk0)) {
        const int r = e - nk0;
        is_v = (r & 1) != 0;
        t = is_v ? r / 2 : r / 2 + kLead;
      } else {
        is_v = true;
        t = e - n;
      }
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
                        is_v ? tv : tk, s * 64, t * kTile, z, &bars[G::kBarKvFull + slot]);
      ++kv_cnt;
    }
  }
  if (*abort_flag) {
    // Let every copy already issued land before the CTA can exit.
    for (uint32_t qb = 0; qb < G::kQBufs; ++qb) {
      if (q_cnt <= qb) break;
      const uint32_t issued = (q_cnt - qb + G::kQBufs - 1) / G::kQBufs;
      mbar_wait(&bars[G::kBarQFull + qb], (issued - 1) & 1);
    }
    for (uint32_t s = 0; s < G::kStages; ++s) {
      if (kv_cnt <= s) break;
      const uint32_t issued = (kv_cnt - s + G::kStages - 1) / G::kStages;
      mbar_wait(&bars[G::kBarKvFull + s], (issued - 1) & 1);
    }
  }
}

// ---- role: present-KV writer (one lane) --------------------------------------------------

// Present K/V are exact copies of the inputs (there is no past).  K/V tile t
// of a (b, kvh) is read by the item of query tile t of the group's first
// head (its last tile when causal), which stores it from the ring to
// present_k / present_v -- one tile pair per item, so the stores spread over
// the whole grid.  Every ring slot takes two arrivals before it is refilled:
// the MMA lane's and this lane's, given once the store (if any) has finished
// reading shared memory.
template <int D>
__device__ void prefill_writer(const CUtensorMap* tpk, const CUtensorMap* tpv,
                               const PrefillKParams& p, uint8_t* sm, uint64_t* bars,
                               volatile int* abort_flag) {
  using G = PGeo<D>;
  uint32_t kv_cnt = 0;
  bool stop = false;
  for (int k = 0; !stop; ++k) {
    const int w = item_index(k, static_cast<int>(gridDim.x));
    if (w >= p.n_items) break;
    const Item it = item_of(w, p);
    const int n = it.n;
    const bool owner = p.write_present != 0 && it.h % p.g == 0;
    const int z = it.b * p.Hkv + it.kvh;
    const int nk0 = n < kLead ? n : kLead;
    for (int e = 0; e < 2 * n; ++e) {
      // the producer's entry order: K_0 .. K_(kLead-1), then (K_(j+kLead), V_j) pairs, then V's
      bool is_v;
      int t;
      if (e < nk0) {
        is_v = false;
        t = e;
      } else if (e < nk0 + 2 * (n - nk0)) {
        const int r = e - nk0;
        is_v = (r & 1) != 0;
        t = is_v ? r / 2 : r / 2 + kLead;
      } else {
        is_v = true;
        t = e - n;
      }
      const uint32_t slot = kv_cnt % G::kStages;
      if (!wait_or_abort(&bars[G::kBarKvFull + slot], (kv_cnt / G::kStages) & 1, abort_flag,
                         p.err_word)) {
        stop = true;
        break;
      }
      ++kv_cnt;
      if (owner && t == it.qt && ((p.write_present >> (is_v ? 1 : 0)) & 1)) {
        const uint8_t* src = sm + G::kOffRing + slot * G::kTileBytes;
#pragma unroll
        for (int s2 = 0; s2 < G::kSlabs; ++s2)
          tc05::tma_store3(is_v ? tpv : tpk, s2 * 64, t * kTile, z, src + s2 * kSlabBytes);
        tc05::bulk_commit_group();
        tc05::bulk_wait_group_read0();
      }
      mbar_arrive(&bars[G::kBarKvEmpty + slot]);
    }
  }
  tc05::bulk_wait_group0();  // every store has reached global memory
}

// ---- role: MMA issuer (one lane) ----------------------------------------------------

// Two lanes issue the MMAs, on different warps (and so different schedulers):
// the score lane S(g) for every KV tile g, as soon as its K tile is in and
// the buffer's previous P has been consumed; the PV lane O += P(g) V_g as soon
// as P(g) and V_g are in.  (tcgen05.mma issue returns only when the tensor
// core can take the instruction, so each lane waits only on its own
// dependencies while the other keeps the queue fed.)  Score buffers rotate
// with a tile count g that runs on across the CTA's items.
template <int D, bool kBf16, bool kScoreLane>
__device__ void prefill_mma(const PrefillKParams& p, uint8_t* sm, uint64_t* bars, uint32_t tmem,
                            volatile int* abort_flag) {
  using G = PGeo<D>;
  constexpr uint32_t id_s = tc05::idesc_f16(kTile, kTile, kBf16, false, false);
  constexpr uint32_t id_o = tc05::idesc_f16(kTile, D, kBf16, false, true);
  // Descriptors of Q buffer 0 and of ring slot 0; the start-address field
  // (16-byte units, bits 0-13) then only advances by the byte offset / 16.
  const uint64_t dQ = tc05::sw128_desc(smem_u32(sm + G::kOffQ), 16, 1024);
  const uint64_t dK = tc05::sw128_desc(smem_u32(sm + G::kOffRing), 16, 1024);
  const uint64_t dV = tc05::sw128_desc(smem_u32(sm + G::kOffRing), kSlabBytes, 1024);

  // S = Q . K^T into score buffer buf
  auto issue_s = [&](uint32_t qb, uint32_t slot, int buf) {
    const uint64_t a0 = dQ + ((qb * G::kTileBytes) >> 4), b0 = dK + ((slot * G::kTileBytes) >> 4);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = ((kk / 4) * kSlabBytes + (kk % 4) * 32) >> 4;
      tc05::mma_ss(tmem + G::kColS + buf * kTile, a0 + off, b0 + off, id_s, kk > 0 ? 1u : 0u);
    }
  };
  // O += P . V; P of group q's keys sits in the first half of that group's
  // score columns (each softmax group writes over its own scores).
  auto issue_pv = [&](uint32_t slot, int buf, bool acc) {
    const uint64_t v0 = dV + ((slot * G::kTileBytes) >> 4);
    const uint32_t a = tmem + G::kColS + buf * kTile;
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk)
      tc05::mma_ts(tmem + G::kColO,
                   a + (kk / (kGroupKeys / 16)) * kGroupKeys + (kk % (kGroupKeys / 16)) * 8,
                   v0 + ((kk * 2048) >> 4), id_o, (acc || kk > 0) ? 1u : 0u);
  };

  uint32_t kv_cnt = 0, q_cnt = 0, g = 0;
  uint32_t par = 0;  // bit b: parity of the next awaited phase of this lane's barrier b
  bool stop = false;
  for (int k = 0; !stop; ++k) {
    const int w = item_index(k, static_cast<int>(gridDim.x));
    if (w >= p.n_items) break;
    const Item it = item_of(w, p);
    const uint32_t qb = q_cnt % G::kQBufs;
    if (kScoreLane &&
        !wait_or_abort(&bars[G::kBarQFull + qb], (q_cnt / G::kQBufs) & 1, abort_flag, p.err_word))
      break;
    ++q_cnt;
    // Ring entries of this item, in the producer's order: K_0 .. K_(kLead-1),
    // then per tile j: K_(j+kLead) (if any), V_j.
    const uint32_t base = kv_cnt;
    const int n = it.n;
    kv_cnt += 2 * n;
    auto kidx = [&](int t) { return base + static_cast<uint32_t>(t < kLead ? t : 2 * t - kLead); };
    auto vidx = [&](int t) {
      return base + static_cast<uint32_t>(t < n - kLead ? kLead + 2 * t + 1 : n + t);
    };
    auto full = [&](uint32_t idx) {
      return wait_or_abort(&bars[G::kBarKvFull + idx % G::kStages], (idx / G::kStages) & 1,
                           abort_flag, p.err_word);
    };
    auto release = [&](uint32_t idx) { tc05::commit(&bars[G::kBarKvEmpty + idx % G::kStages]); };

    for (int j = 0; j < n; ++j, ++g) {
      const int buf = static_cast<int>(g % kSBufs);
      if (kScoreLane) {
        // the buffer's previous P (tile g - 3) must have been read by its PV
        const uint32_t ki = kidx(j);
        if ((g >= kSBufs &&
             !wait_or_abort(&bars[G::kBarPv + buf], (par >> buf) & 1, abort_flag, p.err_word)) ||
            !full(ki)) {
          stop = true;
          break;
        }
        if (g >= kSBufs) par ^= 1u << buf;
        tc05::fence_after_sync();
        issue_s(qb, ki % G::kStages, buf);
        tc05::commit(&bars[G::kBarS + buf]);
        release(ki);
        if (j == n - 1) tc05::commit(&bars[G::kBarQEmpty + qb]);
      } else {
        const uint32_t vi = vidx(j);
        if (!full(vi) ||
            !wait_or_abort(&bars[G::kBarP + buf], (par >> buf) & 1, abort_flag, p.err_word)) {
          stop = true;
          break;
        }
        par ^= 1u << buf;
        tc05::fence_after_sync();
        issue_pv(vi % G::kStages, buf, j > 0);
        tc05::commit(&bars[G::kBarPv + buf]);
        release(vi);
        if (j == n - 1) tc05::commit(&bars[G::kBarO]);
      }
    }
  }
  // Every MMA this lane issued completes before the tensor memory is released.
  uint64_t* done = &bars[G::kBarDone + (kScoreLane ? 0 : 1)];
  tc05::commit(done);
  mbar_wait(done, 0);
}

}  // namespace

namespace {

// ---- role: softmax warpgroups (group q owns keys [q, q + 1) * kGroupKeys of every tile) ----

// kCols columns of this thread's O row *= alpha, in tensor memory (warp-collective).
template <int kCols>
__device__ __forceinline__ void rescale_o(uint32_t tO, float alpha) {
  const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
  for (int c = 0; c < kCols / 16; ++c) {
    uint32_t o[16];
    tc05::tmem_ld16(tO + c * 16, o);
    tc05::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float lo, hi;
      f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), a2), lo,
                hi);
      o[2 * i] = __float_as_uint(lo);
      o[2 * i + 1] = __float_as_uint(hi);
    }
    tc05::tmem_st16(tO + c * 16, o);
  }
  tc05::tmem_st_wait();
}

// Pass 1 over a thread's 32 raw scores: x = s * k1 in place (softcap; else
// x = s); xmax = max of the unmasked x (columns <= rel; kNeedMax), amax =
// max |x| (softcap).
template <bool kSoftcap, bool kMask, bool kNeedMax>
__device__ __forceinline__ void score_pass(uint32_t (&r)[kGroupKeys], float k1, int rel,
                                           float& xmax, float& amax) {
  const uint64_t k1x2 = f2_pack(k1, k1);
  float mx[2] = {SA_NEG_INF, SA_NEG_INF}, ax[2] = {0.0f, 0.0f};
#pragma unroll
  for (int i = 0; i < kGroupKeys / 2; ++i) {
    float a = __uint_as_float(r[2 * i]), b = __uint_as_float(r[2 * i + 1]);
    if (kSoftcap) {
      f2_unpack(f2_mul(f2_pack(a, b), k1x2), a, b);
      r[2 * i] = __float_as_uint(a);
      r[2 * i + 1] = __float_as_uint(b);
      ax[i & 1] = max3(ax[i & 1], fabsf(a), fabsf(b));
    }
    if (kNeedMax) {
      if (kMask) {
        if (2 * i > rel) a = SA_NEG_INF;
        if (2 * i + 1 > rel) b = SA_NEG_INF;
      }
      mx[i & 1] = max3(mx[i & 1], a, b);
    }
  }
  xmax = fmaxf(mx[0], mx[1]);
  amax = fmaxf(ax[0], ax[1]);
}

// How the log2-domain logit of x is formed: c_log2 * x (no softcap), or
// c_log2 * tanh(x) with the first kPolyPairs pairs of a thread's scores on
// the polynomial and the rest on the MUFU tanh (kSplit: the two pipes then
// carry about the same load), or all on the MUFU tanh (a score outside the
// polynomial's range).
enum ScoreMode { kPlain = 0, kSplit = 1, kMufu = 2 };
constexpr int kPolyPairs = kGroupKeys * 11 / 32;  // of kGroupKeys / 2

__device__ __forceinline__ float poly_logit(float x, const float (&tq)[kTanhTerms]) {
  const float y = x * x;
  float q = tq[kTanhTerms - 1];
#pragma unroll
  for (int k = kTanhTerms - 2; k >= 0; --k) q = fmaf(q, y, tq[k]);
  return x * q;
}

// Pass 2: p = 2^(logit(x) - m), masked columns 0, written to tensor memory at
// tP as 16 columns of 16-bit pairs; returns the two partial sums.
template <int kMode, bool kMask, typename T>
__device__ __forceinline__ uint64_t exp_pass(const uint32_t (&r)[kGroupKeys], uint32_t tP, float c2,
                                             float neg_m, const float (&tq)[kTanhTerms], int rel) {
  const uint64_t c2x2 = f2_pack(c2, c2), nm2 = f2_pack(neg_m, neg_m);
  uint64_t ls[2] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f)};
  uint32_t pk[kGroupKeys / 2];
#pragma unroll
  for (int i = 0; i < kGroupKeys / 2; ++i) {
    const float x0 = __uint_as_float(r[2 * i]), x1 = __uint_as_float(r[2 * i + 1]);
    uint64_t v;
    if (kMode == kPlain) {
      v = f2_fma(f2_pack(x0, x1), c2x2, nm2);
    } else if (kMode == kMufu || i >= kPolyPairs) {
      v = f2_fma(f2_pack(tanh_approx(x0), tanh_approx(x1)), c2x2, nm2);
    } else {
      const uint64_t xx = f2_pack(x0, x1);
      const uint64_t y = f2_mul(xx, xx);
      uint64_t q = f2_fma(f2_pack(tq[4], tq[4]), y, f2_pack(tq[3], tq[3]));
      q = f2_fma(q, y, f2_pack(tq[2], tq[2]));
      q = f2_fma(q, y, f2_pack(tq[1], tq[1]));
      q = f2_fma(q, y, f2_pack(tq[0], tq[0]));
      v = f2_fma(xx, q, nm2);
    }
    float a, b;
    f2_unpack(v, a, b);
    if (kMask) {
      if (2 * i > rel) a = SA_NEG_INF;
      if (2 * i + 1 > rel) b = SA_NEG_INF;
    }
    a = ex2(a);
    b = ex2(b);
    ls[i & 1] = f2_add(ls[i & 1], f2_pack(a, b));
    pk[i] = pack2<T>(a, b);
  }
#pragma unroll
  for (int c = 0; c < kGroupKeys / 32; ++c)
    tc05::tmem_st16(tP + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[c * 16]));
  return f2_add(ls[0], ls[1]);
}

// Score variants: no softcap; softcap with a running maximum; softcap with the
// constant offset 0.  With |softcap| * log2(e) <= kFixedOffsetMaxLog2 every
// log2-domain logit lies within +-97, so 2^logit neither overflows nor
// underflows fp32, nor does a row sum over up to 2^30 keys: the shift-
// invariant softmax then needs no maximum at all (no cross-group exchange,
// no O rescale).
enum ScoreVariant { kVarPlain = 0, kVarSoftcapMax = 1, kVarSoftcapFixed = 2 };

template <int D, typename T, int kVariant>
__device__ void prefill_softmax(const PrefillKParams& p, uint8_t* sm, uint64_t* bars,
                                uint32_t tmem, volatile int* abort_flag) {
  using G = PGeo<D>;
  constexpr bool kSoftcap = kVariant != kVarPlain;
  constexpr bool kFixed = kVariant == kVarSoftcapFixed;
  constexpr int kOCols = D / kGroups;  // O columns normalised and stored by each group
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const int q = (warp - 4) >> 2;  // keys [q, q + 1) * kGroupKeys of every tile
  const int row = ((warp & 3) << 5) | lane;
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_base + G::kColS + q * kGroupKeys;  // + buffer * 128
  const uint32_t tO = tmem + lane_base + G::kColO + q * kOCols;
  float* xch = reinterpret_cast<float*>(sm + G::kOffXch);
  const float c2 = p.c_log2, k1 = p.k1;
  float tq[kTanhTerms];
#pragma unroll
  for (int k = 0; k < kTanhTerms; ++k) tq[k] = p.tq[k];
  // Phase parities as bit masks (bit b: next phase of buffer b's barrier):
  // s_full; pv_free, flipped when this thread hands a P to the PV lane (the PV
  // it starts then completes that barrier's next phase).  Score buffers rotate
  // with the tile count g across the CTA's items, as in the MMA lanes.
  uint32_t s_par = 0, pv_par = 0, o_cnt = 0, x_cnt = 0, g = 0;
  bool stop = false;

  // Share a value with the other groups of the same row (bounded; false on
  // abort); returns their maximum (kMax) or sum.
  auto exchange = [&](float v, bool kMax, float& out) -> bool {
    if (kGroups == 1) {  // the whole row is this thread's
      out = v;
      return true;
    }
    const uint32_t slot = x_cnt & 1;
    xch[(slot * kGroups + q) * kTile + row] = v;
    mbar_arrive(&bars[G::kBarXch + slot]);
    if (!wait_or_abort_warp(&bars[G::kBarXch + slot], (x_cnt >> 1) & 1, abort_flag, p.err_word))
      return false;
    ++x_cnt;
    const float* e = &xch[slot * kGroups * kTile + row];
    float acc = e[0];
#pragma unroll
    for (int g2 = 1; g2 < kGroups; ++g2) acc = kMax ? fmaxf(acc, e[g2 * kTile]) : acc + e[g2 * kTile];
    out = acc;
    return true;
  };

  for (int k = 0; !stop; ++k) {
    const int w = item_index(k, static_cast<int>(gridDim.x));
    if (w >= p.n_items) break;
    const Item it = item_of(w, p);
    const int qi = it.qt * kTile + row;
    const int lim = p.nonpad ? last_key(p, it.b, qi)                 // last visible key
                             : (p.causal ? min(qi, p.S - 1) : p.S - 1);
    float m = SA_NEG_INF, l = 0.0f;
    for (int j = 0; j < it.n; ++j, ++g) {
      const int buf = static_cast<int>(g % kSBufs);
      if (!wait_or_abort_warp(&bars[G::kBarS + buf], (s_par >> buf) & 1, abort_flag, p.err_word)) {
        stop = true;
        break;
      }
      s_par ^= 1u << buf;
      tc05::fence_after_sync();
      const uint32_t tSb = tS + buf * kTile;
      uint32_t r[kGroupKeys];
#pragma unroll
      for (int c = 0; c < kGroupKeys / 32; ++c)
        tc05::tmem_ld32(tSb + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[c * 32]));
      tc05::tmem_ld_wait();

      // pass 1: x, its masked maximum and its largest magnitude
      const int rel = lim - j * kTile - q * kGroupKeys;  // columns above rel are masked
      const bool masked = __any_sync(0xffffffffu, rel < kGroupKeys - 1);
      float xmax, amax;
      if (masked)
        score_pass<kSoftcap, true, !kFixed>(r, k1, rel, xmax, amax);
      else
        score_pass<kSoftcap, false, !kFixed>(r, k1, rel, xmax, amax);
      const int mode =
          !kSoftcap ? kPlain
                    : (__any_sync(0xffffffffu, amax > kTanhPolyBound) ? kMufu : kSplit);
      bool any_raise = false;
      float alpha = 1.0f;
      if (!kFixed) {
        float mt = SA_NEG_INF;
        if (xmax != SA_NEG_INF)
          mt = mode == kPlain   ? xmax * c2
               : mode == kSplit ? poly_logit(xmax, tq)
                                : tanh_approx(xmax) * c2;
        if (!exchange(mt, true, mt)) {
          stop = true;
          break;
        }
        // lazy maximum (every group takes the same decision from the same values)
        const bool raise = mt > m + kRescaleLog2;
        any_raise = __any_sync(0xffffffffu, raise);
        if (raise) {
          alpha = ex2(m - mt);
          l *= alpha;
          m = mt;
        }
      }
      const float neg_m = (kFixed || m == SA_NEG_INF) ? 0.0f : -m;

      // pass 2: probabilities over this group's own score columns
      uint64_t ls;
      if (mode == kPlain)
        ls = masked ? exp_pass<kPlain, true, T>(r, tSb, c2, neg_m, tq, rel)
                    : exp_pass<kPlain, false, T>(r, tSb, c2, neg_m, tq, rel);
      else if (mode == kSplit)
        ls = masked ? exp_pass<kSplit, true, T>(r, tSb, c2, neg_m, tq, rel)
                    : exp_pass<kSplit, false, T>(r, tSb, c2, neg_m, tq, rel);
      else
        ls = masked ? exp_pass<kMufu, true, T>(r, tSb, c2, neg_m, tq, rel)
                    : exp_pass<kMufu, false, T>(r, tSb, c2, neg_m, tq, rel);
      {
        float a, b;
        f2_unpack(ls, a, b);
        l += a + b;
      }
      // O follows the new maximum once PV(g - 1) has completed.  On its
      // buffer's pv_free barrier the phase before it, PV(g - 4), is complete
      // (the score lane waited for it before issuing S(g - 1)), so only
      // PV(g - 1)'s phase can be outstanding.
      if (!kFixed && any_raise && j > 0) {
        const int pb = static_cast<int>((g + kSBufs - 1) % kSBufs);
        if (!wait_or_abort_warp(&bars[G::kBarPv + pb], ((pv_par >> pb) & 1) ^ 1u, abort_flag,
                                p.err_word)) {
          stop = true;
          break;
        }
        tc05::fence_after_sync();
        rescale_o<kOCols>(tO, alpha);
      }
      tc05::tmem_st_wait();
      tc05::fence_before_sync();
      mbar_arrive(&bars[G::kBarP + buf]);
      pv_par ^= 1u << buf;
    }
    if (stop) break;

    // epilogue: the row sum is the groups' sums; this group stores O columns
    // [q * D / 4, (q + 1) * D / 4) / l
    float lt;
    if (!exchange(l, false, lt)) break;
    if (!wait_or_abort_warp(&bars[G::kBarO], o_cnt & 1, abort_flag, p.err_word)) break;
    ++o_cnt;
    tc05::fence_after_sync();
    const float inv_l = lt > 0.0f ? 1.0f / lt : 0.0f;
    T* yrow = static_cast<T*>(p.y) +
              ((static_cast<int64_t>(it.b) * p.Hq + it.h) * p.S + qi) * D + q * kOCols;
#pragma unroll
    for (int c = 0; c < kOCols / 16; ++c) {
      uint32_t o[16];
      tc05::tmem_ld16(tO + c * 16, o);
      tc05::tmem_ld_wait();
      if (qi < p.S) {
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          pk[i] = pack2<T>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        uint4* dst = reinterpret_cast<uint4*>(yrow + c * 16);
        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
  }
}

// ---- kernel -------------------------------------------------------------------------------

template <int D, typename T, int kVariant>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc05_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tpk,
                        const __grid_constant__ CUtensorMap tpv, const PrefillKParams p) {
  using G = PGeo<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + G::kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + G::kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + G::kOffAbort);
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[G::kBarQFull + i], 1);
      mbar_init(&bars[G::kBarQEmpty + i], 1);
      mbar_init(&bars[G::kBarXch + i], 128 * kGroups);
      mbar_init(&bars[G::kBarDone + i], 1);
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(&bars[G::kBarS + i], 1);
      mbar_init(&bars[G::kBarP + i], 128 * kGroups);
      mbar_init(&bars[G::kBarPv + i], 1);
    }
    for (int s = 0; s < G::kStages; ++s) {
      mbar_init(&bars[G::kBarKvFull + s], 1);
      mbar_init(&bars[G::kBarKvEmpty + s], 2);  // MMA lane + present writer
    }
    mbar_init(&bars[G::kBarO], 1);
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
      prefill_mma<D, std::is_same<T, __nv_bfloat16>::value, true>(p, sm, bars, tmem, abort_flag);
  } else if (warp == 3) {
    if (lane == 0)
      prefill_mma<D, std::is_same<T, __nv_bfloat16>::value, false>(p, sm, bars, tmem, abort_flag);
  } else if (warp == 2) {
    if (lane == 0) prefill_writer<D>(&tpk, &tpv, p, sm, bars, abort_flag);
  } else if (warp >= 4) {
    prefill_softmax<D, T, kVariant>(p, sm, bars, tmem, abort_flag);
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

EncodeTiledFn encode_tiled() {
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

// Least-squares fit of tanh(x) / x = sum_k c_k (x^2)^k over 0 < x <= B
// (Chebyshev nodes in x; normal equations in u = x^2 / B^2, solved in double
// by Gaussian elimination with partial pivoting).  Evaluated in fp32 with
// fused multiply-adds the polynomial stays within about 1e-7 of tanh on
// |x| <= B = kTanhPolyBound, below the MUFU tanh's own error.
static void fit_tanh_poly(double (&c)[kTanhTerms]) {
  constexpr int kNodes = 2048;
  const double B = kTanhPolyBound;
  const double pi = 3.14159265358979323846;
  double A[kTanhTerms][kTanhTerms + 1] = {};
  for (int i = 0; i < kNodes; ++i) {
    const double x = B * std::cos(pi * (i + 0.5) / (2.0 * kNodes));
    const double u = x * x / (B * B), f = std::tanh(x) / x;
    double pw[kTanhTerms];
    pw[0] = 1.0;
    for (int k = 1; k < kTanhTerms; ++k) pw[k] = pw[k - 1] * u;
    for (int r = 0; r < kTanhTerms; ++r) {
      for (int q = 0; q < kTanhTerms; ++q) A[r][q] += pw[r] * pw[q];
      A[r][kTanhTerms] += pw[r] * f;
    }
  }
  for (int col = 0; col < kTanhTerms; ++col) {
    int piv = col;
    for (int r = col + 1; r < kTanhTerms; ++r)
      if (std::fabs(A[r][col]) > std::fabs(A[piv][col])) piv = r;
    for (int q = 0; q <= kTanhTerms; ++q) std::swap(A[col][q], A[piv][q]);
    for (int r = 0; r < kTanhTerms; ++r) {
      if (r == col) continue;
      const double f = A[r][col] / A[col][col];
      for (int q = col; q <= kTanhTerms; ++q) A[r][q] -= f * A[col][q];
    }
  }
  double scale = 1.0;  // 1 / B^(2k): back from u to x^2
  for (int k = 0; k < kTanhTerms; ++k) {
    c[k] = A[k][kTanhTerms] / A[k][k] * scale;
    scale /= B * B;
  }
}

static const double* tanh_poly() {
  static std::once_flag once;
  static double c[kTanhTerms];
  std::call_once(once, [] { fit_tanh_poly(c); });
  return c;
}

bool prefill_tc_supported(const PrefillTcArgs& a) {
  if (a.dtype != SA_BF16 && a.dtype != SA_F16) return false;
  if (a.D != 64 && a.D != 128) return false;
  if (!(a.scale > 0.0f) || !std::isfinite(a.scale) || !std::isfinite(a.softcap)) return false;
  if (!al16(a.q) || !al16(a.k) || !al16(a.v) || !al16(a.y) || !al16(a.present_k) ||
      !al16(a.present_v))
    return false;
  if (a.S < 1 || a.S > (int64_t(1) << 30)) return false;
  const int64_t nq = (a.S + kTile - 1) / kTile;
  if (a.B * a.Hq * nq >= (int64_t(1) << 30)) return false;  // item indices in int
  return encode_tiled() != nullptr;
}

template <int D, typename T>
static int launch_prefill_t(const PrefillTcArgs& a, cudaStream_t st) {
  using G = PGeo<D>;
  CUtensorMap tq, tk, tv, tpk, tpv;
  if (!make_tile_map(&tq, a.q, a.dtype, D, a.S, a.B * a.Hq) ||
      !make_tile_map(&tk, a.k, a.dtype, D, a.S, a.B * a.Hkv) ||
      !make_tile_map(&tv, a.v, a.dtype, D, a.S, a.B * a.Hkv))
    return -1;
  tpk = tk;  // placeholders when no present output is requested
  tpv = tv;
  if ((a.present_k && !make_tile_map(&tpk, a.present_k, a.dtype, D, a.S, a.B * a.Hkv)) ||
      (a.present_v && !make_tile_map(&tpv, a.present_v, a.dtype, D, a.S, a.B * a.Hkv)))
    return -1;
  PrefillKParams p;
  p.y = a.y;
  p.err_word = a.err_word;
  p.write_present = (a.present_k ? 1 : 0) | (a.present_v ? 2 : 0);
  p.B = static_cast<int>(a.B);
  p.Hq = static_cast<int>(a.Hq);
  p.Hkv = static_cast<int>(a.Hkv);
  p.S = static_cast<int>(a.S);
  p.g = static_cast<int>(a.Hq / a.Hkv);
  p.nq = static_cast<int>((a.S + kTile - 1) / kTile);
  p.n_items = p.B * p.Hq * p.nq;
  p.causal = a.causal ? 1 : 0;
  p.nonpad = a.nonpad;
  const float log2e = 1.4426950408889634f;
  if (a.softcap != 0.0f) {
    const float cap = std::fabs(a.softcap);
    p.k1 = a.scale / cap;
    p.c_log2 = cap * log2e;
    p.softcap_on = p.c_log2 <= kFixedOffsetMaxLog2 ? 2 : 1;
    const double* c = tanh_poly();
    for (int k = 0; k < kTanhTerms; ++k)
      p.tq[k] = static_cast<float>(c[k] * static_cast<double>(cap) * 1.4426950408889634);
  } else {
    p.softcap_on = 0;
    p.k1 = 1.0f;
    p.c_log2 = a.scale * log2e;
    for (int k = 0; k < kTanhTerms; ++k) p.tq[k] = 0.0f;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  const int grid = p.n_items < sms ? p.n_items : sms;
  auto kern = p.softcap_on == 0   ? prefill_tc05_kernel<D, T, kVarPlain>
              : p.softcap_on == 1 ? prefill_tc05_kernel<D, T, kVarSoftcapMax>
                                  : prefill_tc05_kernel<D, T, kVarSoftcapFixed>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmem) !=
      cudaSuccess)
    return -1;
  kern<<<grid, kThreads, G::kSmem, st>>>(tq, tk, tv, tpk, tpv, p);
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
