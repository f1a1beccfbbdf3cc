// k_stream.cu -- persistent stream-K gather decode (f16 / bf16 storage) and
// the merge of units split across warps.
//
// Semantics: IndexShare `index_share_row` (onnx-runtime-ep-cuda
// src/kernels/index_share.rs): per output row, scaled QK scores over the
// candidate keys, a stable fp32 softmax in which a fully-masked row gives 0,
// probs . V.  ONNX Attention (standard_attention.rs) `attention_split` /
// `attention_combine`: partial (max, sum, unnormalised P.V) per key range,
// merged by a log-sum-exp combine in a fixed order.  Paged addressing:
// ferrum-kernels causal_attention.rs (16-token blocks through a table).
//
// GB300 design:
//  * Work = every unit's candidates cut into 16-key tiles laid end to end.
//    The grid is persistent (one CTA per SM); each warp owns one contiguous
//    range of tiles, so all SMs finish together whatever the unit lengths.
//  * Each warp runs its own 3-deep ring: a tile's 16 K rows and 16 V rows are
//    fetched by one bulk async copy per lane (a row each), completion counted
//    on the slot's mbarrier; rows are padded by 16 bytes so ldmatrix is
//    conflict-free; masked keys are not fetched.  With tensor maps (kTma) the
//    slots hold the 128-byte-swizzled layout instead: paged and dense tiles
//    (16 consecutive rows) arrive as D/64 TMA boxes of K and of V, selected
//    rows as tile::gather4 loads of four rows each, so a tile takes 4 or 16
//    copies in place of 32 (the per-row copies bounded the paged data path);
//    masked rows of a loaded tile get their V zeroed in shared memory.  The cache positions of a
//    tile (planned per index row by k_plan.cu, or read from the page table)
//    are prefetched one iteration ahead.  No CTA-wide barrier in the loop.
//  * Per tile: S^T = K . Q^T and O^T += V^T . P^T on the m16n8k16 tensor-core
//    MMA with keys as M and the GQA group as N (P^T from the S^T accumulator
//    by an in-register 8x8 transpose), online softmax in the log2 domain.
//  * A unit inside one warp's range is written directly; a unit split across
//    warps leaves one partial per warp, merged by stream_combine_kernel in
//    warp order (deterministic).
#include <cstdlib>
#include <cstring>

#include "gather_common.cuh"
#include "tc05.cuh"

namespace sa {

// kTma: the slot holds K then V as D/64 slabs of 16 rows x 128 bytes in the
// 128-byte swizzle (TMA boxes), every slot 1024-byte aligned; else rows padded
// to kRowStride.
template <int D, bool kTma = false>
struct SGeo {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kRowStride = kRowBytes + 16;        // padding: conflict-free ldmatrix
  static constexpr int kSlabs = D / 64;                    // kTma: 64-dim swizzled slabs
  static constexpr int kSlabBytes = 16 * 128;
  static constexpr int kHalfBytes = kTma ? kSlabs * kSlabBytes : 16 * kRowStride;
  static constexpr int kSlotBytes = 2 * kHalfBytes;        // 16 K rows then 16 V rows
  static constexpr int kWarps = (D <= 128) ? 8 : 4;        // warps per CTA
  static constexpr int kStages = (D == 64) ? 4 : 3;        // ring slots per warp
  static constexpr int kRingBytes = kStages * kSlotBytes;
  // per warp: ring | slot masks | full barriers
  static constexpr int kMaskOff = kRingBytes;
  static constexpr int kBarOff = (kMaskOff + kStages * 4 + 7) / 8 * 8;
  static constexpr int kAlign = kTma ? 1024 : 16;
  static constexpr int kWarpBytes = (kBarOff + kStages * 8 + kAlign - 1) / kAlign * kAlign;
  static constexpr int kThreads = kWarps * 32;
};

template <int D, bool kTma>
static size_t smem_bytes_t(int source, int64_t B) {
  size_t s = static_cast<size_t>(SGeo<D, kTma>::kWarps) * SGeo<D, kTma>::kWarpBytes;
  if (source == kPaged) s += static_cast<size_t>(B + 1) * 4;
  return s + (kTma ? 1024 : 0);  // + alignment of the dynamic base
}

size_t stream_smem_bytes(int D, int source, int64_t B) {
  switch (D) {
    case 64: return smem_bytes_t<64, false>(source, B);
    case 128: return smem_bytes_t<128, false>(source, B);
    default: return smem_bytes_t<256, false>(source, B);
  }
}

// Byte offset of 16-byte chunk c (of D / 8) of row r (< 16) in a kTma half.
__device__ __forceinline__ uint32_t swz_off(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

int stream_warps(int D) { return D <= 128 ? 8 : 4; }

// Paged requests keep a per-sequence tile prefix in shared memory.
int stream_max_batch_paged() { return 2048; }

// Unit geometry in the tile space.
struct TileUnit {
  int64_t u;    // unit index
  int64_t off;  // first tile of the unit
  int64_t tu;   // tiles of the unit
};

__device__ __forceinline__ TileUnit unit_of_tile(const GatherArgs& a, const int32_t* pref,
                                                 int64_t t) {
  TileUnit r;
  if (a.source != kPaged) {  // tile counts stay below 2^31 (checked on the host)
    r.u = static_cast<uint32_t>(t) / static_cast<uint32_t>(a.tiles_per_unit);
    r.off = r.u * a.tiles_per_unit;
    r.tu = a.tiles_per_unit;
    return r;
  }
  // pref[b] = tiles of sequences < b (per KV head); sequence b spans
  // [Hkv*pref[b], Hkv*pref[b+1]) with Hkv units of pref[b+1]-pref[b] tiles.
  int64_t lo = 0, hi = a.B;  // largest b with Hkv*pref[b] <= t (empty sequences skipped)
  while (hi - lo > 1) {
    const int64_t mid = (lo + hi) >> 1;
    if (a.Hkv * static_cast<int64_t>(pref[mid]) <= t) lo = mid;
    else hi = mid;
  }
  const int64_t tb = pref[lo + 1] - pref[lo];
  const int64_t base = a.Hkv * static_cast<int64_t>(pref[lo]);
  const int64_t kvh = static_cast<uint32_t>(t - base) / static_cast<uint32_t>(tb);
  r.u = lo * a.Hkv + kvh;
  r.off = base + kvh * tb;
  r.tu = tb;
  return r;
}

// Tile cursor: the unit of the current tile and what its rows need, advanced
// monotonically (a division only when it enters another unit).
struct Cursor {
  TileUnit tu;
  UnitInfo ui;
  int64_t nc;       // candidates of the unit
  int64_t rowbase;  // sparse/dense: first cache row of (b, kvh)
  int64_t prow;     // sparse: first planned position of the unit's index row
};

__device__ __forceinline__ void cursor_fill(const GatherArgs& a, Cursor& c) {
  c.ui = unit_info(a, c.tu.u);
  c.nc = (a.source == kPaged) ? static_cast<int64_t>(__ldg(a.ctx_len + c.ui.b)) : a.n_cand;
  c.rowbase = (c.ui.b * a.Hkv + c.ui.kvh) * a.T;
  c.prow = ((c.ui.b * a.I + c.ui.ih) * a.Sq + c.ui.i) * a.n_cand_pad;
}

__device__ __forceinline__ void cursor_to(const GatherArgs& a, const int32_t* pref, Cursor& c,
                                          int64_t t) {
  if (t >= c.tu.off && t < c.tu.off + c.tu.tu) return;
  if (a.source != kPaged && t >= c.tu.off && t < c.tu.off + 2 * c.tu.tu) {
    c.tu.u += 1;
    c.tu.off += c.tu.tu;
  } else {
    c.tu = unit_of_tile(a, pref, t);
  }
  cursor_fill(a, c);
}

// One lane's key of a tile, fetched ahead: the loaded word (planned position
// or page id) and what turns it into a cache row.
struct KeyRef {
  int64_t base;  // row = base + raw (sparse/dense) or raw * Hkv * page_tokens + base (paged)
  int32_t raw;   // -1: masked
};

__device__ __forceinline__ KeyRef key_load(const GatherArgs& a, const Cursor& cu, int64_t t,
                                           int lane) {
  KeyRef k;
  const int64_t c = (t - cu.tu.off) * 16 + (lane & 15);
  if (a.source == kSparse) {
    k.base = cu.rowbase;
    k.raw = __ldg(a.pos + cu.prow + c);
  } else if (a.source == kDense) {
    k.base = cu.rowbase;
    k.raw = (c < cu.nc && dense_visible(a, cu.ui.b, cu.ui.i, c)) ? static_cast<int32_t>(c) : -1;
  } else {
    // c < max_pages * page_tokens < 2^31 (checked on the host): 32-bit division
    const uint32_t c32 = static_cast<uint32_t>(c), pt = static_cast<uint32_t>(a.page_tokens);
    const uint32_t pi = c32 / pt;
    k.base = cu.ui.kvh * a.page_tokens + (c32 - pi * pt);
    k.raw = -1;
    if (c < cu.nc) {
      const int32_t pg = __ldg(a.block_table + cu.ui.b * a.max_pages + pi);
      k.raw = pg < 0 ? -2 : pg;  // -2: a bad table entry
    }
  }
  return k;
}

// Cache row of a prefetched key, or -1.
__device__ __forceinline__ int64_t key_row(const GatherArgs& a, const KeyRef& k) {
  if (k.raw == -1) return -1;
  if (a.source != kPaged) return k.base + k.raw;
  if (k.raw < 0 || k.raw >= a.num_pages) {
    if (a.err_word) atomicOr(a.err_word, SA_ERRBIT_PAGE);
    return -1;
  }
  return static_cast<int64_t>(k.raw) * a.Hkv * a.page_tokens + k.base;
}

// kBias: the request carries an additive bias (a separate instance, so that
// the common bias-free kernel keeps its registers).
template <typename T, int D, int NT, bool kTma, bool kBias>
__global__ void __launch_bounds__(SGeo<D, kTma>::kThreads, 1)
    gather_stream_kernel(const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv, GatherArgs a) {
  using G = SGeo<D, kTma>;
  constexpr int KS = D / 16;
  constexpr int NW = G::kWarps, S = G::kStages;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem =
      kTma ? reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023))
           : smem_raw;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;

  // ---- barriers and ring init --------------------------------------------------------
  if (threadIdx.x < NW) {
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + threadIdx.x * G::kWarpBytes + G::kBarOff);
#pragma unroll
    for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
  }
  // V rows of every slot start at zero: a masked key's row is never fetched,
  // and its probability 0 must multiply finite values.  (kTma slots get their
  // masked V rows zeroed after each load instead.)
  constexpr int kVz = G::kHalfBytes / 16;  // int4 per slot's V rows
  if (!kTma)
    for (int e = threadIdx.x; e < NW * S * kVz; e += blockDim.x) {
      const int w = e / (S * kVz), r = e % (S * kVz);
      uint4* vz = reinterpret_cast<uint4*>(smem + w * G::kWarpBytes + (r / kVz) * G::kSlotBytes +
                                           G::kHalfBytes);
      vz[r % kVz] = make_uint4(0, 0, 0, 0);
    }
  fence_proxy_async_smem();
  fence_mbar_init();
  // Everything above is independent of the previous kernel in the stream
  // (plan / append); from here on its results are read.
  pdl_wait();
  pdl_launch_dependents();  // the combine kernel may start launching
  __syncthreads();

  // ---- tile space -----------------------------------------------------------------
  int32_t* pref = reinterpret_cast<int32_t*>(smem + NW * G::kWarpBytes);
  int64_t NTt, R;
  if (a.source == kPaged) {
    // per-sequence tiles, exclusive prefix over the batch (every CTA computes
    // it): loads in parallel, then one warp scans 32 entries per step.
    for (int64_t b = threadIdx.x; b < a.B; b += blockDim.x) {
      const int64_t ctx = a.ctx_len[b];
      const bool ok = ctx >= 1 && ctx <= a.max_pages * a.page_tokens;
      if (!ok && blockIdx.x == 0 && a.err_word) atomicOr(a.err_word, SA_ERRBIT_PAGE);
      pref[b + 1] = ok ? static_cast<int32_t>((ctx + 15) / 16) : 0;
    }
    __syncthreads();
    if (warp == 0) {
      int32_t carry = 0;
      if (lane == 0) pref[0] = 0;
      for (int64_t b0 = 0; b0 < a.B; b0 += 32) {
        const int64_t b = b0 + lane;
        int32_t v = (b < a.B) ? pref[b + 1] : 0;
#pragma unroll
        for (int sh = 1; sh < 32; sh <<= 1) {
          const int32_t n = __shfl_up_sync(0xffffffffu, v, sh);
          if (lane >= sh) v += n;
        }
        if (b < a.B) pref[b + 1] = carry + v;
        carry += __shfl_sync(0xffffffffu, v, 31);
      }
    }
    __syncthreads();
    NTt = a.Hkv * static_cast<int64_t>(pref[a.B]);
    const int64_t gw_total = static_cast<int64_t>(gridDim.x) * NW;
    R = (NTt + gw_total - 1) / gw_total;
    if (R < 1) R = 1;
    if (blockIdx.x == 0) {
      // the combine kernel needs the same tile space
      for (int64_t b = threadIdx.x; b <= a.B; b += blockDim.x) a.pref_out[b] = pref[b];
      // sequences without tiles still need a (zero) output
      for (int64_t e = threadIdx.x; e < a.B * a.Hq * D; e += blockDim.x) {
        const int64_t b = e / (a.Hq * D);
        if (pref[b + 1] == pref[b]) static_cast<T*>(a.y)[e] = from_f32<T>(0.f);
      }
    }
  } else {
    NTt = a.units * a.tiles_per_unit;
    R = a.tiles_per_warp;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) a.meta[0] = R;

  // ---- this warp's tile range ----------------------------------------------------------
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * NW + warp;
  const int64_t t_begin = gw * R;
  int64_t t_end = t_begin + R;
  if (t_end > NTt) t_end = NTt;
  if (t_begin >= t_end) return;
  const int64_t ntiles = t_end - t_begin;

  unsigned char* wbase = smem + warp * G::kWarpBytes;
  const uint32_t ring_s = smem_u32(wbase);
  uint32_t* smask = reinterpret_cast<uint32_t*>(wbase + G::kMaskOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(wbase + G::kBarOff);
  const char* kb = static_cast<const char*>(a.k);
  const char* vb = static_cast<const char*>(a.v);

  // Issue cursor (runs S tiles ahead of compute) and its prefetched keys.
  Cursor ic;
  ic.tu = unit_of_tile(a, pref, t_begin);
  cursor_fill(a, ic);
  const int64_t first_u = ic.tu.u;  // unit of this warp's first tile (partial slot 0)

  // Copies of tile k into its ring slot: one bulk async copy per lane (lanes
  // 0-15 the K rows, 16-31 the V rows); bytes counted on the slot's barrier.
  auto issue = [&](int64_t k, const KeyRef& kr) {
    const int slot = static_cast<int>(k % S);
    const int64_t row = key_row(a, kr);
    const uint32_t m = __ballot_sync(0xffffffffu, row >= 0) & 0xffffu;
    fence_proxy_async_smem();  // this warp's reads of the slot precede the refill
    if (kTma) {
      const int first = m ? __ffs(m) - 1 : 0;
      const long long rf = __shfl_sync(0xffffffffu, static_cast<long long>(row), first);
      if (lane == 0) {
        smask[slot] = m;
        mbar_arrive_expect_tx(&full[slot], m ? 2u * 16u * G::kRowBytes : 0u);
      }
      __syncwarp();
      unsigned char* kd = wbase + slot * G::kSlotBytes;
      if (a.source == kSparse) {
        // scattered rows: op o = lane (< 8 * kSlabs) fetches rows 4q .. 4q + 3 of
        // slab h of K (kv = 0) or V; a masked key fetches the tile's first
        // valid row instead (its V row is zeroed after the load)
        const int q = lane & 3, h = (lane >> 2) % G::kSlabs, kv = lane / (4 * G::kSlabs);
        const int mine = static_cast<int>(row >= 0 ? row : rf);
        const int y0 = __shfl_sync(0xffffffffu, mine, 4 * q);
        const int y1 = __shfl_sync(0xffffffffu, mine, 4 * q + 1);
        const int y2 = __shfl_sync(0xffffffffu, mine, 4 * q + 2);
        const int y3 = __shfl_sync(0xffffffffu, mine, 4 * q + 3);
        if (m && lane < 8 * G::kSlabs)
          tc05::tma_gather4(kd + kv * G::kHalfBytes + h * G::kSlabBytes + q * 512, kv ? &tv : &tk,
                            64 * h, y0, y1, y2, y3, &full[slot]);
      } else if (m && lane == 0) {
        // consecutive rows (a page, or positions of a dense cache): row(l) = row(0) + l
        const int y = static_cast<int>(rf - first);
#pragma unroll
        for (int h = 0; h < G::kSlabs; ++h) {
          tc05::tma_load2(kd + h * G::kSlabBytes, &tk, 64 * h, y, &full[slot]);
          tc05::tma_load2(kd + G::kHalfBytes + h * G::kSlabBytes, &tv, 64 * h, y, &full[slot]);
        }
      }
      __syncwarp();
      return;
    }
    if (lane == 0) {
      smask[slot] = m;
      mbar_arrive_expect_tx(&full[slot], __popc(m) * 2u * G::kRowBytes);
    }
    __syncwarp();
    if (row >= 0) {
      const bool is_v = lane >= 16;
      unsigned char* dst = wbase + slot * G::kSlotBytes + (is_v ? 16 * G::kRowStride : 0) +
                           (lane & 15) * G::kRowStride;
      bulk_g2s(dst, (is_v ? vb : kb) + row * G::kRowBytes, G::kRowBytes, &full[slot]);
    }
  };
  auto load_key = [&](int64_t k) {
    cursor_to(a, pref, ic, t_begin + k);
    return key_load(a, ic, t_begin + k, lane);
  };
  for (int q = 0; q < S - 1; ++q)
    if (q < ntiles) issue(q, load_key(q));
  KeyRef next{0, -1};
  if (S - 1 < ntiles) next = load_key(S - 1);

  // ---- per-unit state -------------------------------------------------------------------
  uint32_t qf[NT][KS][2];
  float o[KS][NT][4];
  float m_run[NT][2], l_run[NT][2];
  Cursor cur;
  cur.tu.u = -1;
  cur.tu.off = 0;
  cur.tu.tu = 0;
  const float sl2 = a.scale_log2;
  const float cap = a.softcap, inv_cap = a.inv_softcap;

  auto start_unit = [&](int64_t t) {
    cursor_to(a, pref, cur, t);
    const T* qp = static_cast<const T*>(a.q);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int hh = nt * 8 + gid;
      const bool live = hh < a.hpu;
      const int64_t qoff =
          ((cur.ui.b * a.Hq + (cur.ui.h0 + (live ? hh : 0))) * a.Sq + cur.ui.i) * D;
      const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qp + qoff);
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        qf[nt][kk][0] = live ? __ldg(q32 + kk * 8 + tig) : 0u;
        qf[nt][kk][1] = live ? __ldg(q32 + kk * 8 + tig + 4) : 0u;
      }
      m_run[nt][0] = m_run[nt][1] = SA_NEG_INF;
      l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
    }
  };

  // End of a unit's tiles in this warp: write y directly when the whole unit
  // lies in this warp's range, else this warp's partial (slot 0 = the unit of
  // its first tile, slot 1 = the unit of its last tile).
  auto flush_unit = [&]() {
    float lsum[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float l = l_run[nt][j];
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) l += __shfl_xor_sync(0xffffffffu, l, sh);
        lsum[nt][j] = l;
      }
    const bool whole = cur.tu.off >= t_begin && cur.tu.off + cur.tu.tu <= t_end;
    const int64_t pbase = (gw * 2 + ((cur.tu.u == first_u) ? 0 : 1)) * a.hpu;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int hh = nt * 8 + 2 * tig + j;
        if (hh >= a.hpu) continue;
        if (whole) {
          const int64_t h = cur.ui.h0 + hh;
          const float M = m_run[nt][j];
          float L = lsum[nt][j];
          if (a.sink && M != SA_NEG_INF) L += ex2(a.sink[h] * kLog2e - M);
          const float inv = (M == SA_NEG_INF || L == 0.f) ? 0.f : 1.0f / L;
          T* yp = static_cast<T*>(a.y) + ((cur.ui.b * a.Hq + h) * a.Sq + cur.ui.i) * D;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            yp[mt * 16 + gid] = from_f32<T>(o[mt][nt][j] * inv);
            yp[mt * 16 + gid + 8] = from_f32<T>(o[mt][nt][2 + j] * inv);
          }
        } else {
          float* po = a.part_o + (pbase + hh) * D;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            po[mt * 16 + gid] = o[mt][nt][j];
            po[mt * 16 + gid + 8] = o[mt][nt][2 + j];
          }
          if (gid == 0) {
            a.part_ml[2 * (pbase + hh)] = m_run[nt][j];
            a.part_ml[2 * (pbase + hh) + 1] = lsum[nt][j];
          }
        }
      }
  };

  // ---- main loop ------------------------------------------------------------------
  bool timed_out = false;
  for (int64_t k = 0; k < ntiles; ++k) {
    const int64_t t = t_begin + k;
    __syncwarp();
    if (k + S - 1 < ntiles) {
      const KeyRef kr = next;
      if (k + S < ntiles) next = load_key(k + S);  // prefetch one tile further
      issue(k + S - 1, kr);
    }
    const int slot = static_cast<int>(k % S);
    if (!mbar_wait(&full[slot], static_cast<uint32_t>((k / S) & 1))) timed_out = true;
    if (cur.tu.u < 0 || t >= cur.tu.off + cur.tu.tu) {
      if (cur.tu.u >= 0) flush_unit();
      start_unit(t);
    }
    const uint32_t mask = smask[slot];
    if (mask == 0u) continue;
    const bool v_lo = (mask >> gid) & 1u, v_hi = (mask >> (gid + 8)) & 1u;
    const uint32_t kt = ring_s + slot * G::kSlotBytes;
    const uint32_t vt = kt + G::kHalfBytes;
    if (kTma && mask != 0xffffu) {
      // rows of the page past the context: V must hold finite values (zeros)
      unsigned char* vrow = wbase + slot * G::kSlotBytes + G::kHalfBytes;
      for (int e = lane; e < 16 * G::kSlabs * 8; e += 32) {
        const int r = e / (G::kSlabs * 8), rest = e % (G::kSlabs * 8);
        if (!((mask >> r) & 1u))
          *reinterpret_cast<uint4*>(vrow + (rest >> 3) * G::kSlabBytes + r * 128 + (rest & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }
    // S^T = K . Q^T
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
    {
      const uint32_t rbase = kt + (lane & 15) * G::kRowStride + (lane >> 4) * 16;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kTma ? kt + swz_off(lane & 15, 2 * kk + (lane >> 4)) : rbase + kk * 32, a0, a1, a2,
                a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma16816<T>(s[nt], a0, a1, a2, a3, qf[nt][kk][0], qf[nt][kk][1]);
      }
    }
    // additive bias ([IS] bias_at): keyed by the cache positions of this
    // lane's accumulator rows (keys gid and gid + 8 of the tile)
    int32_t j_lo = -1, j_hi = -1;
    if (kBias) {
      const int64_t c0 = (t - cur.tu.off) * 16 + gid;  // candidate of accumulator row gid
      if (a.source == kSparse) {
        if (v_lo) j_lo = __ldg(a.pos + cur.prow + c0);
        if (v_hi) j_hi = __ldg(a.pos + cur.prow + c0 + 8);
      } else {  // dense: the candidate is the key position
        if (v_lo) j_lo = static_cast<int32_t>(c0);
        if (v_hi) j_hi = static_cast<int32_t>(c0 + 8);
      }
    }
    uint32_t pb[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = s[nt][e];
        if (cap != 0.f) x = cap * tanh_fast(x * (sl2 * (1.0f / kLog2e)) * inv_cap) * kLog2e;
        else x = x * sl2;
        if (kBias) {
          const int32_t j = (e < 2) ? j_lo : j_hi;
          const int hh = nt * 8 + 2 * tig + (e & 1);
          if (j >= 0 && hh < a.hpu)
            x += kLog2e * bias_term(a, cur.ui.b, cur.ui.h0 + hh, cur.ui.i, j);
        }
        s[nt][e] = ((e < 2) ? v_lo : v_hi) ? x : SA_NEG_INF;
      }
      float tm0 = fmaxf(s[nt][0], s[nt][2]);
      float tm1 = fmaxf(s[nt][1], s[nt][3]);
#pragma unroll
      for (int sh = 4; sh < 32; sh <<= 1) {
        tm0 = fmaxf(tm0, __shfl_xor_sync(0xffffffffu, tm0, sh));
        tm1 = fmaxf(tm1, __shfl_xor_sync(0xffffffffu, tm1, sh));
      }
      const float mn0 = fmaxf(m_run[nt][0], tm0), mn1 = fmaxf(m_run[nt][1], tm1);
      const float mu0 = (mn0 == SA_NEG_INF) ? 0.f : mn0, mu1 = (mn1 == SA_NEG_INF) ? 0.f : mn1;
      const float al0 = ex2(m_run[nt][0] - mu0), al1 = ex2(m_run[nt][1] - mu1);
      m_run[nt][0] = mn0;
      m_run[nt][1] = mn1;
      const float p0 = ex2(s[nt][0] - mu0), p1 = ex2(s[nt][1] - mu1);
      const float p2 = ex2(s[nt][2] - mu0), p3 = ex2(s[nt][3] - mu1);
      l_run[nt][0] = l_run[nt][0] * al0 + (p0 + p2);
      l_run[nt][1] = l_run[nt][1] * al1 + (p1 + p3);
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        o[mt][nt][0] *= al0;
        o[mt][nt][1] *= al1;
        o[mt][nt][2] *= al0;
        o[mt][nt][3] *= al1;
      }
      pb[nt][0] = movm_t(pack2<T>(p0, p1));
      pb[nt][1] = movm_t(pack2<T>(p2, p3));
    }
    // O^T += V^T . P^T
    {
      const int vr = (lane & 7) + ((lane >> 4) << 3);
      const uint32_t rbase = vt + vr * G::kRowStride + ((lane >> 3) & 1) * 16;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(kTma ? vt + swz_off(vr, 2 * mt + ((lane >> 3) & 1)) : rbase + mt * 32, a0, a1,
                  a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma16816<T>(o[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
      }
    }
  }
  if (timed_out && lane == 0 && a.err_word) atomicOr(a.err_word, SA_ERRBIT_TIMEOUT);
  if (cur.tu.u >= 0) flush_unit();
}

// ---------------------------------------------------------------------------
// merge of split units: y = sum_w o_w 2^(m_w - M) / (sum_w l_w 2^(m_w - M) [+ sink])
// ---------------------------------------------------------------------------
// One 128-thread block per unit; a unit held wholly by one warp was written
// by the stream kernel and is skipped.  Warp w's partial of the unit sits in
// its slot 0 when the unit begins inside w's range, else in slot 1.
template <typename T, int D>
__global__ void __launch_bounds__(128) stream_combine_kernel(GatherArgs a) {
  constexpr int kMaxW = 64;  // partials merged per pass
  constexpr int kRegW = 8;   // up to this many partials: merged in registers
  pdl_wait();  // the stream kernel's partials and tile space
  const int64_t u = blockIdx.x;
  const int64_t R = a.meta[0];
  int64_t off, tu;
  if (a.source == kPaged) {
    const int64_t b = u / a.Hkv, kvh = u % a.Hkv;
    tu = a.pref_out[b + 1] - a.pref_out[b];
    off = a.Hkv * static_cast<int64_t>(a.pref_out[b]) + kvh * tu;
  } else {
    tu = a.tiles_per_unit;
    off = u * tu;
  }
  if (tu == 0) return;
  const int64_t w_lo = off / R, w_hi = (off + tu - 1) / R;
  if (w_lo == w_hi) return;  // written directly by the stream kernel
  const UnitInfo ui = unit_info(a, u);
  const int hpu = static_cast<int>(a.hpu);
  const int64_t nw = w_hi - w_lo + 1;
  if (nw <= kRegW) {
    // Few partials: every thread loads all it needs at once -- its float4 of
    // each partial and its head's (m, l) of each -- then merges in registers:
    // one round trip to L2 after the stream kernel ends.
    constexpr int kG2 = (16 * D / 4 + 127) / 128;
#pragma unroll
    for (int g = 0; g < kG2; ++g) {
      const int e = threadIdx.x + 128 * g;
      if (e >= hpu * D / 4) break;
      const int hh = (e * 4) / D, d = (e * 4) % D;
      float4 v[kRegW];
      float2 ml[kRegW];
#pragma unroll
      for (int wi = 0; wi < kRegW; ++wi) {
        if (wi < nw) {
          const int64_t w = w_lo + wi;
          const int64_t sb = (w * 2 + ((w * R >= off) ? 0 : 1)) * a.hpu + hh;
          v[wi] = __ldg(reinterpret_cast<const float4*>(a.part_o + sb * D + d));
          ml[wi] = __ldg(reinterpret_cast<const float2*>(a.part_ml) + sb);
        }
      }
      float M = SA_NEG_INF;
#pragma unroll
      for (int wi = 0; wi < kRegW; ++wi)
        if (wi < nw) M = fmaxf(M, ml[wi].x);
      const float Mu = (M == SA_NEG_INF) ? 0.f : M;
      float L = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int wi = 0; wi < kRegW; ++wi) {
        if (wi < nw && ml[wi].x != SA_NEG_INF) {
          const float f = ex2(ml[wi].x - Mu);
          L += ml[wi].y * f;
          acc.x = fmaf(v[wi].x, f, acc.x);
          acc.y = fmaf(v[wi].y, f, acc.y);
          acc.z = fmaf(v[wi].z, f, acc.z);
          acc.w = fmaf(v[wi].w, f, acc.w);
        }
      }
      if (a.sink && M != SA_NEG_INF) L += ex2(a.sink[ui.h0 + hh] * kLog2e - M);
      const float inv = (M == SA_NEG_INF || L == 0.f) ? 0.f : 1.0f / L;
      T* yp = static_cast<T*>(a.y) + ((ui.b * a.Hq + ui.h0 + hh) * a.Sq + ui.i) * D + d;
      yp[0] = from_f32<T>(acc.x * inv);
      yp[1] = from_f32<T>(acc.y * inv);
      yp[2] = from_f32<T>(acc.z * inv);
      yp[3] = from_f32<T>(acc.w * inv);
    }
    return;
  }
  __shared__ float sm_m[kMaxW][16], sm_l[kMaxW][16];
  __shared__ float sM[16], sL[16];
  if (threadIdx.x < hpu) {
    sM[threadIdx.x] = SA_NEG_INF;
    sL[threadIdx.x] = 0.f;
  }
  constexpr int kG = (16 * D / 4 + 127) / 128;  // float4 groups per thread (hpu <= 16)
  float4 acc[kG];
#pragma unroll
  for (int g = 0; g < kG; ++g) acc[g] = make_float4(0.f, 0.f, 0.f, 0.f);
  // Partials are merged in warp order, kMaxW at a time, as a running
  // (max, sum, output) exactly like the online softmax.
  for (int64_t w0 = 0; w0 < nw; w0 += kMaxW) {
    const int nwp = static_cast<int>(nw - w0 < kMaxW ? nw - w0 : kMaxW);
    __syncthreads();
    for (int t = threadIdx.x; t < nwp * hpu; t += blockDim.x) {
      const int wi = t / hpu, hh = t % hpu;
      const int64_t w = w_lo + w0 + wi;
      const int sl = (w * R >= off) ? 0 : 1;  // the unit begins inside w's range
      const float2 ml =
          __ldg(reinterpret_cast<const float2*>(a.part_ml) + (w * 2 + sl) * a.hpu + hh);
      sm_m[wi][hh] = ml.x;
      sm_l[wi][hh] = ml.y;
    }
    __syncthreads();
    // new running max per head, rescale of what is accumulated so far
    __shared__ float sScale[16];
    if (threadIdx.x < hpu) {
      const int hh = threadIdx.x;
      float M = sM[hh];
      for (int wi = 0; wi < nwp; ++wi) M = fmaxf(M, sm_m[wi][hh]);
      const float Mu = (M == SA_NEG_INF) ? 0.f : M;
      const float old = ex2(sM[hh] - Mu);
      float L = sL[hh] * old;
      for (int wi = 0; wi < nwp; ++wi) {
        const float f = ex2(sm_m[wi][hh] - Mu);
        sm_m[wi][hh] = f;  // now the partial's weight
        L += sm_l[wi][hh] * f;
      }
      sScale[hh] = old;
      sM[hh] = M;
      sL[hh] = L;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      const int e = threadIdx.x + 128 * g;
      if (e >= hpu * D / 4) break;
      const int hh = (e * 4) / D, d = (e * 4) % D;
      float4 s4 = acc[g];
      const float sc = sScale[hh];
      s4.x *= sc;
      s4.y *= sc;
      s4.z *= sc;
      s4.w *= sc;
#pragma unroll 4
      for (int wi = 0; wi < nwp; ++wi) {
        const int64_t w = w_lo + w0 + wi;
        const int sl = (w * R >= off) ? 0 : 1;
        const float f = sm_m[wi][hh];
        const float4 v = __ldg(reinterpret_cast<const float4*>(
            a.part_o + ((w * 2 + sl) * a.hpu + hh) * D + d));
        s4.x += v.x * f;
        s4.y += v.y * f;
        s4.z += v.z * f;
        s4.w += v.w * f;
      }
      acc[g] = s4;
    }
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < kG; ++g) {
    const int e = threadIdx.x + 128 * g;
    if (e >= hpu * D / 4) break;
    const int hh = (e * 4) / D, d = (e * 4) % D;
    const float M = sM[hh];
    float L = sL[hh];
    if (a.sink && M != SA_NEG_INF) L += ex2(a.sink[ui.h0 + hh] * kLog2e - M);
    const float inv = (M == SA_NEG_INF || L == 0.f) ? 0.f : 1.0f / L;
    T* yp = static_cast<T*>(a.y) + ((ui.b * a.Hq + ui.h0 + hh) * a.Sq + ui.i) * D + d;
    yp[0] = from_f32<T>(acc[g].x * inv);
    yp[1] = from_f32<T>(acc[g].y * inv);
    yp[2] = from_f32<T>(acc[g].z * inv);
    yp[3] = from_f32<T>(acc[g].w * inv);
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

// Launch with programmatic stream serialisation: the kernel may begin while
// the previous kernel in the stream finishes, and waits for its results
// itself (griddepcontrol.wait) before reading them.
template <typename K, typename... Args>
static int launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      Args... args) {
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
  return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess ? 0 : -1;
}

// K and V as 2-D tensors of 16-bit rows for the TMA-fed slots: page pools
// [num_pages, Hkv, page_tokens, D] and dense caches [B, Hkv, T, D] in boxes of
// 64 dims x 16 rows (a tile's rows are consecutive), selected-token caches in
// boxes one row high for tile::gather4.  All in the 128-byte swizzle.  False
// when the tensors cannot be described (then the per-row copies are used).
static bool kv_maps(const GatherArgs& a, int dtype, CUtensorMap* tk, CUtensorMap* tv) {
  if (a.row_copies) return false;  // the caller asked for the per-row copies
  if (a.D != 64 && a.D != 128 && a.D != 256) return false;
  if (a.source == kPaged && a.page_tokens % 16 != 0) return false;
  const int64_t rows =
      a.source == kPaged ? a.num_pages * a.Hkv * a.page_tokens : a.B * a.Hkv * a.T;
  if (rows < 16 || rows >= (int64_t(1) << 31)) return false;
  if ((reinterpret_cast<uintptr_t>(a.k) | reinterpret_cast<uintptr_t>(a.v)) & 15) return false;
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.D), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.D * 2)};
  const cuuint32_t box[2] = {64, a.source == kSparse ? 1u : 16u};
  const cuuint32_t es[2] = {1, 1};
  const CUtensorMapDataType dt =
      dtype == SA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const void* base[2] = {a.k, a.v};
  CUtensorMap* out[2] = {tk, tv};
  for (int i = 0; i < 2; ++i)
    if (enc(out[i], dt, 2, const_cast<void*>(base[i]), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  return true;
}

template <typename T, int D, int NT, bool kBias>
static int launch_stream_b(const GatherArgs& a, int dtype, int grid, cudaStream_t st) {
  CUtensorMap tk, tv;
  std::memset(&tk, 0, sizeof(tk));
  std::memset(&tv, 0, sizeof(tv));
  if (kv_maps(a, dtype, &tk, &tv)) {
    const size_t smem = smem_bytes_t<D, true>(a.source, a.B);
    if (cudaFuncSetAttribute(gather_stream_kernel<T, D, NT, true, kBias>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return -1;
    return launch_pdl(gather_stream_kernel<T, D, NT, true, kBias>, dim3(grid),
                      dim3(SGeo<D, true>::kThreads), smem, st, tk, tv, a);
  }
  const size_t smem = smem_bytes_t<D, false>(a.source, a.B);
  if (cudaFuncSetAttribute(gather_stream_kernel<T, D, NT, false, kBias>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return -1;
  return launch_pdl(gather_stream_kernel<T, D, NT, false, kBias>, dim3(grid),
                    dim3(SGeo<D, false>::kThreads), smem, st, tk, tv, a);
}

template <typename T, int D, int NT>
static int launch_stream_t(const GatherArgs& a, int dtype, int grid, cudaStream_t st) {
  // an additive bias (selected tokens) or attention mask (dense prefill)
  if (a.bias && a.source != kPaged) return launch_stream_b<T, D, NT, true>(a, dtype, grid, st);
  return launch_stream_b<T, D, NT, false>(a, dtype, grid, st);
}

int launch_gather_stream(const GatherArgs& a, int dtype, int grid, cudaStream_t st) {
  const bool two = a.hpu > 8;
  if (dtype == SA_BF16) {
    if (a.D == 64) return two ? launch_stream_t<__nv_bfloat16, 64, 2>(a, dtype, grid, st)
                              : launch_stream_t<__nv_bfloat16, 64, 1>(a, dtype, grid, st);
    if (a.D == 128) return two ? launch_stream_t<__nv_bfloat16, 128, 2>(a, dtype, grid, st)
                               : launch_stream_t<__nv_bfloat16, 128, 1>(a, dtype, grid, st);
    return launch_stream_t<__nv_bfloat16, 256, 1>(a, dtype, grid, st);
  }
  if (a.D == 64) return two ? launch_stream_t<__half, 64, 2>(a, dtype, grid, st)
                            : launch_stream_t<__half, 64, 1>(a, dtype, grid, st);
  if (a.D == 128) return two ? launch_stream_t<__half, 128, 2>(a, dtype, grid, st)
                             : launch_stream_t<__half, 128, 1>(a, dtype, grid, st);
  return launch_stream_t<__half, 256, 1>(a, dtype, grid, st);
}

int launch_stream_combine(const GatherArgs& a, int dtype, cudaStream_t st) {
  if (a.units == 0) return 0;
  const dim3 grid(static_cast<unsigned>(a.units)), blk(128);
  if (dtype == SA_BF16) {
    if (a.D == 64) return launch_pdl(stream_combine_kernel<__nv_bfloat16, 64>, grid, blk, 0, st, a);
    if (a.D == 128) return launch_pdl(stream_combine_kernel<__nv_bfloat16, 128>, grid, blk, 0, st, a);
    return launch_pdl(stream_combine_kernel<__nv_bfloat16, 256>, grid, blk, 0, st, a);
  }
  if (a.D == 64) return launch_pdl(stream_combine_kernel<__half, 64>, grid, blk, 0, st, a);
  if (a.D == 128) return launch_pdl(stream_combine_kernel<__half, 128>, grid, blk, 0, st, a);
  return launch_pdl(stream_combine_kernel<__half, 256>, grid, blk, 0, st, a);
}

}  // namespace sa
