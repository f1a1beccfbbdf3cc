// k_stream.cu -- persistent stream-K gather decode (f16 / bf16 storage).
//
// Semantics: IndexShare `index_share_row` (onnx-runtime-ep-cuda
// src/kernels/index_share.rs): per output row gather the valid prefix of the
// selected indices from the present cache, scaled QK scores, a stable fp32
// softmax in which a fully-masked row gives 0, probs . V; the present cache is
// past ++ current (`build_present`), and the row validation rules of
// `validate_indices` / `validate_index_rows`.  ONNX Attention
// (standard_attention.rs) `attention_split` / `attention_combine`: partial
// (max, sum, unnormalised P.V) per key range merged by a log-sum-exp combine
// in a fixed order.  Paged addressing: ferrum-kernels causal_attention.rs
// (16-token blocks through a table).
//
// GB300 design:
//  * Work = every unit's candidates cut into 16-key tiles, laid end to end.
//    The grid is persistent (one CTA per SM at the occupancy limit); each warp
//    owns one contiguous range of tiles, so all SMs finish together whatever
//    the per-unit lengths.
//  * Each warp runs its own 3-deep cp.async ring of tiles (16 K rows + 16 V
//    rows, 16-byte copies, XOR-swizzled so ldmatrix is conflict-free); masked
//    keys are zero-filled by the copy itself.  No CTA-wide barrier in the loop.
//  * Per tile: S^T = K . Q^T and O^T += V^T . P^T on the m16n8k16 tensor-core
//    MMA with keys as M and the GQA group as N (P^T via an in-register
//    transpose), online softmax in the log2 domain.
//  * A unit lying wholly inside one warp's range is written directly.  A unit
//    split across warps leaves one partial per warp; the last warp to finish
//    it (atomic ticket, no waiting) merges the partials in warp order, so the
//    result is deterministic.
//  * Optionally fused: index-row validation (each column's rule depends only
//    on its own value and its left neighbour's, so columns are checked in
//    parallel and the first failing column wins through an atomic max), and
//    the current token's K/V (read from the caller's buffer for positions
//    [write_pos, write_pos + C) and written into the cache).
#include "gather_common.cuh"

namespace sa {

template <int D>
struct SGeo {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kChunks = kRowBytes / 16;        // 16-byte chunks per row
  static constexpr int kRowsPerInst = 32 / kChunks;     // rows per warp copy instruction
  static constexpr int kTileBytes = 2 * 16 * kRowBytes; // 16 K rows then 16 V rows
  static constexpr int kWarps = (D <= 128) ? 8 : 4;
  static constexpr int kStages = 3;
  static constexpr int kIdxBuf = 256;                   // resolved candidates per warp
  static constexpr int kChunkTiles = kIdxBuf / 16;
  static constexpr int kWarpBytes = kStages * kTileBytes + kIdxBuf * 4 + 16;
};

size_t stream_smem_bytes(int D, int source, int64_t B) {
  size_t per = 0, warps = 0;
  switch (D) {
    case 64: per = SGeo<64>::kWarpBytes; warps = SGeo<64>::kWarps; break;
    case 128: per = SGeo<128>::kWarpBytes; warps = SGeo<128>::kWarps; break;
    default: per = SGeo<256>::kWarpBytes; warps = SGeo<256>::kWarps; break;
  }
  size_t s = per * warps;
  if (source == kPaged) s += static_cast<size_t>(B + 1) * 4;
  return s;
}

int stream_warps(int D) { return D <= 128 ? 8 : 4; }

// Paged requests keep a per-sequence tile prefix in shared memory.
int stream_max_batch_paged() { return 4096; }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Unit geometry in the tile space.
struct TileUnit {
  int64_t u;    // unit index
  int64_t off;  // first tile of the unit
  int64_t tu;   // tiles of the unit
};

__device__ __forceinline__ TileUnit unit_of_tile(const GatherArgs& a, const int32_t* pref,
                                                 int64_t t) {
  TileUnit r;
  if (a.source != kPaged) {
    r.u = t / a.tiles_per_unit;
    r.off = r.u * a.tiles_per_unit;
    r.tu = a.tiles_per_unit;
    return r;
  }
  // pref[b] = tiles of sequences < b (per KV head); sequence b spans
  // [Hkv*pref[b], Hkv*pref[b+1]) with Hkv units of pref[b+1]-pref[b] tiles.
  int64_t lo = 0, hi = a.B;  // find largest b with Hkv*pref[b] <= t
  while (hi - lo > 1) {
    const int64_t mid = (lo + hi) >> 1;
    if (a.Hkv * static_cast<int64_t>(pref[mid]) <= t) lo = mid;
    else hi = mid;
  }
  // skip sequences without tiles (their span is empty)
  const int64_t b = lo;
  const int64_t tb = pref[b + 1] - pref[b];
  const int64_t base = a.Hkv * static_cast<int64_t>(pref[b]);
  const int64_t kvh = (t - base) / tb;
  r.u = b * a.Hkv + kvh;
  r.off = base + kvh * tb;
  r.tu = tb;
  return r;
}

__device__ __forceinline__ int64_t n_cand_of(const GatherArgs& a, const UnitInfo& ui) {
  if (a.source == kPaged) return a.ctx_len[ui.b];
  return a.n_cand;
}

// Validation of one index column (exact per-column form of the row scan;
// see the file comment).  Returns the status code, 0 when the column passes;
// a -1 in column 0 returns the all-padding marker (reported only if no column
// of the row fails).
__device__ __forceinline__ int column_code(int64_t v, int64_t prev, int64_t col, int64_t bound) {
  if (v == -1) return col == 0 ? SA_IDX_ALL_PADDING : 0;
  if (v < -1) return SA_IDX_BELOW_SENTINEL;
  if (col > 0 && prev == -1) return SA_IDX_AFTER_PADDING;
  if (v >= bound) return SA_IDX_OUT_OF_RANGE;
  if (col > 0 && v == prev) return SA_IDX_DUPLICATE;
  if (col > 0 && v < prev) return SA_IDX_NOT_INCREASING;
  return 0;
}

// Global word a candidate's resolution depends on: the selected index (and,
// when validating, its left neighbour) for the sparse source, the block-table
// entry for the paged source.  Loaded in a separate pass so that every load of
// a chunk is in flight at once.
struct RawCand {
  int64_t v, prev;
};

__device__ __forceinline__ RawCand load_candidate(const GatherArgs& a, const UnitInfo& ui,
                                                  int64_t c, bool validate) {
  RawCand r{0, 0};
  if (a.source == kPaged) {
    if (c < a.max_pages * a.page_tokens)
      r.v = __ldg(a.block_table + ui.b * a.max_pages + c / a.page_tokens);
  } else if (a.source == kSparse && c >= a.window && c < a.n_cand) {
    const int64_t col = c - a.window;
    const int64_t off = ((ui.b * a.I + ui.ih) * a.Sq + ui.i) * a.K + col;
    r.v = a.idx_is_i64 ? __ldg(static_cast<const long long*>(a.idx) + off)
                       : static_cast<int64_t>(__ldg(static_cast<const int32_t*>(a.idx) + off));
    if (validate && col > 0)
      r.prev = a.idx_is_i64 ? __ldg(static_cast<const long long*>(a.idx) + off - 1)
                            : static_cast<int64_t>(__ldg(static_cast<const int32_t*>(a.idx) + off - 1));
  }
  return r;
}

// Cache row (>= 0), current-token row (<= -2, encoded as -2 - cur_row), or
// -1 for a masked / absent candidate, from the loaded word.  Also records the
// column check when asked.
__device__ __forceinline__ int32_t resolve_loaded(const GatherArgs& a, const UnitInfo& ui,
                                                  int64_t c, RawCand raw, bool validate,
                                                  int64_t irow) {
  if (a.source == kPaged) {
    const int64_t ctx = __ldg(a.ctx_len + ui.b);
    if (c >= ctx) return -1;
    const int64_t page = raw.v;
    if (page < 0 || page >= a.num_pages) {
      if (a.err_word) atomicOr(a.err_word, SA_ERRBIT_PAGE);
      return -1;
    }
    return static_cast<int32_t>((page * a.Hkv + ui.kvh) * a.page_tokens + c % a.page_tokens);
  }
  if (c >= a.n_cand) return -1;
  if (a.source == kDense) {
    if (a.causal && c > a.past_len + ui.i) return -1;
    return static_cast<int32_t>((ui.b * a.Hkv + ui.kvh) * a.T + c);
  }
  int64_t len = a.kv_len ? __ldg(a.kv_len + ui.b) : a.T;
  if (len > a.T) len = a.T;
  if (len < 0) len = 0;
  const int64_t wstart = len - a.window;
  int64_t t;
  if (c < a.window) {
    t = wstart + c;
    if (t < 0) return -1;
  } else {
    const int64_t col = c - a.window;
    t = raw.v;
    if (validate) {
      const int code = column_code(t, raw.prev, col, len);
      if (code) {
        const uint64_t key = (static_cast<uint64_t>(code == SA_IDX_ALL_PADDING ? a.K : col) << 8) |
                             static_cast<uint64_t>(code);
        atomicMax(a.vword + irow, static_cast<unsigned long long>(~key));
      }
    }
    if (t < 0 || t >= len) return -1;
    if (a.window > 0 && t >= wstart) return -1;
  }
  if (a.causal && t > a.past_len + ui.i) return -1;
  if (a.k_cur) {
    const int64_t wp = write_pos_of(a, ui.b);
    if (t >= wp && t < wp + a.C)
      return static_cast<int32_t>(-2 - ((ui.b * a.Hkv + ui.kvh) * a.C + (t - wp)));
  }
  return static_cast<int32_t>((ui.b * a.Hkv + ui.kvh) * a.T + t);
}

// Finish a row's fused validation: read-and-reset its word, record the code.
__device__ __forceinline__ void finish_validation(const GatherArgs& a, int64_t irow) {
  const unsigned long long w =
      atomicExch(reinterpret_cast<unsigned long long*>(a.vword) + irow, 0ull);
  const int code = w ? static_cast<int>((~w) & 0xff) : 0;
  if (a.row_status) a.row_status[irow] = static_cast<uint8_t>(code);
  if (code && a.err_word) atomicOr(a.err_word, static_cast<uint32_t>(code));
}

template <typename T, int D, int NT>
__global__ void __launch_bounds__(SGeo<D>::kWarps * 32, 1) gather_stream_kernel(GatherArgs a) {
  using G = SGeo<D>;
  constexpr int KS = D / 16;
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;

  // ---- tile space -----------------------------------------------------------------
  int32_t* pref = reinterpret_cast<int32_t*>(smem + G::kWarps * G::kWarpBytes);
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
    const int64_t gw_total = static_cast<int64_t>(gridDim.x) * G::kWarps;
    R = (NTt + gw_total - 1) / gw_total;
    // sequences without tiles still need a (zero) output
    if (blockIdx.x == 0) {
      for (int64_t e = threadIdx.x; e < a.B * a.Hq * D; e += blockDim.x) {
        const int64_t b = e / (a.Hq * D);
        if (pref[b + 1] == pref[b])
          static_cast<T*>(a.y)[e] = from_f32<T>(0.f);
      }
    }
  } else {
    NTt = a.units * a.tiles_per_unit;
    R = a.tiles_per_warp;
  }
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * G::kWarps + warp;
  const int64_t t_begin = gw * R;
  int64_t t_end = t_begin + R;
  if (t_end > NTt) t_end = NTt;
  if (t_begin >= t_end) return;

  unsigned char* ring = smem + warp * G::kWarpBytes;
  int32_t* kpos = reinterpret_cast<int32_t*>(ring + G::kStages * G::kTileBytes);
  uint32_t* smask = reinterpret_cast<uint32_t*>(kpos + G::kIdxBuf);
  const uint32_t ring_s = smem_u32(ring);
  const char* kb = static_cast<const char*>(a.k);
  const char* vb = static_cast<const char*>(a.v);
  const char* kc = static_cast<const char*>(a.k_cur);
  const char* vc = static_cast<const char*>(a.v_cur);
  const bool do_val = a.vword != nullptr && a.source == kSparse;
  const TileUnit first = unit_of_tile(a, pref, t_begin);

  // ---- candidate resolution for tiles [cb, cb + chunk) ----------------------------
  int64_t cb = t_begin;  // first tile held in kpos
  auto resolve_chunk = [&](int64_t c0) {
    constexpr int J = G::kIdxBuf / 32;  // candidates per lane
    const int64_t n = min(static_cast<int64_t>(G::kIdxBuf), (t_end - c0) * 16);
    RawCand raw[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {  // pass 1: every global load of the chunk
      const int64_t e = lane + 32 * j;
      raw[j].v = raw[j].prev = 0;
      if (e < n) {
        const int64_t t = c0 + (e >> 4);
        const TileUnit tu = unit_of_tile(a, pref, t);
        const UnitInfo ui = unit_info(a, tu.u);
        const bool val = do_val && (a.I != 1 || ui.kvh == 0);
        raw[j] = load_candidate(a, ui, (t - tu.off) * 16 + (e & 15), val);
      }
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {  // pass 2: resolve
      const int64_t e = lane + 32 * j;
      if (e < n) {
        const int64_t t = c0 + (e >> 4);
        const TileUnit tu = unit_of_tile(a, pref, t);
        const UnitInfo ui = unit_info(a, tu.u);
        const int64_t c = (t - tu.off) * 16 + (e & 15);
        const bool val = do_val && (a.I != 1 || ui.kvh == 0);
        const int64_t irow = (ui.b * a.I + ui.ih) * a.Sq + ui.i;
        kpos[e] = (c < n_cand_of(a, ui)) ? resolve_loaded(a, ui, c, raw[j], val, irow) : -1;
      }
    }
    __syncwarp();
  };

  // ---- issue the copies of tile ti into its ring slot -------------------------------
  auto issue = [&](int64_t ti) {
    if (ti - cb >= G::kChunkTiles) {
      cb = ti;
      resolve_chunk(cb);
    }
    const int slot = static_cast<int>((ti - t_begin) % G::kStages);
    const int32_t my = kpos[(ti - cb) * 16 + (lane & 15)];
    const uint32_t m = __ballot_sync(0xffffffffu, my != -1) & 0xffffu;
    if (lane == 0) smask[slot] = m;
    const uint32_t kdst = ring_s + slot * G::kTileBytes;
    const uint32_t vdst = kdst + 16 * G::kRowBytes;
    const int ch = lane % G::kChunks;
#pragma unroll
    for (int j = 0; j < 16 / G::kRowsPerInst; ++j) {
      const int r = j * G::kRowsPerInst + lane / G::kChunks;
      const int32_t rid = __shfl_sync(0xffffffffu, my, r);
      const char* ks;
      const char* vs;
      uint32_t nb = 16;
      if (rid >= 0) {
        ks = kb + static_cast<int64_t>(rid) * G::kRowBytes + ch * 16;
        vs = vb + static_cast<int64_t>(rid) * G::kRowBytes + ch * 16;
      } else if (rid <= -2) {
        ks = kc + static_cast<int64_t>(-2 - rid) * G::kRowBytes + ch * 16;
        vs = vc + static_cast<int64_t>(-2 - rid) * G::kRowBytes + ch * 16;
      } else {
        ks = kb;
        vs = vb;
        nb = 0;  // zero-fill
      }
      const uint32_t off = r * G::kRowBytes + ((ch ^ (r & 7)) << 4);
      cp_async16(kdst + off, ks, nb);
      cp_async16(vdst + off, vs, nb);
    }
  };

  resolve_chunk(cb);
#pragma unroll
  for (int s = 0; s < G::kStages - 1; ++s) {
    if (t_begin + s < t_end) issue(t_begin + s);
    cp_async_commit();
  }

  // ---- per-unit state --------------------------------------------------------------
  uint32_t qf[NT][KS][2];
  float o[KS][NT][4];
  float m_run[NT][2], l_run[NT][2];
  TileUnit cur;
  cur.u = -1;
  cur.off = 0;
  cur.tu = 0;
  UnitInfo cui;
  const float sl2 = a.scale_log2;
  const float cap = a.softcap, inv_cap = a.inv_softcap;

  auto start_unit = [&](const TileUnit& tu) {
    cur = tu;
    cui = unit_info(a, tu.u);
    const T* qp = static_cast<const T*>(a.q);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int hh = nt * 8 + gid;
      const bool live = hh < a.hpu;
      const int64_t qoff = ((cui.b * a.Hq + (cui.h0 + (live ? hh : 0))) * a.Sq + cui.i) * D;
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
    // fused append: the warp that starts a (b, kvh)'s first tile writes the
    // current token(s) into the cache (attention reads them from k_cur/v_cur)
    if (a.k_cur && tu.off >= t_begin && cui.h0 % a.g == 0) {
      const int64_t bh = cui.b * a.Hkv + cui.kvh;
      const int64_t wp = write_pos_of(a, cui.b);
      if (wp >= 0 && wp + a.C <= a.T) {
        const int64_t n16 = a.C * G::kChunks;
        for (int64_t e = lane; e < n16; e += 32) {
          const int64_t r = e / G::kChunks, cc = e % G::kChunks;
          const int4* ks = reinterpret_cast<const int4*>(kc + (bh * a.C + r) * G::kRowBytes) + cc;
          const int4* vs = reinterpret_cast<const int4*>(vc + (bh * a.C + r) * G::kRowBytes) + cc;
          int4* kd = reinterpret_cast<int4*>(const_cast<char*>(kb) + (bh * a.T + wp + r) * G::kRowBytes) + cc;
          int4* vd = reinterpret_cast<int4*>(const_cast<char*>(vb) + (bh * a.T + wp + r) * G::kRowBytes) + cc;
          *kd = __ldg(ks);
          *vd = __ldg(vs);
        }
      } else if (lane == 0 && a.err_word) {
        atomicOr(a.err_word, SA_ERRBIT_WRITE_POS);
      }
    }
  };

  // Write y for heads of unit `cur` from merged (M, L, O) held per lane.
  auto store_y = [&](int hh, int d, float M, float L, float acc) {
    const int64_t h = cui.h0 + hh;
    if (a.sink && M != SA_NEG_INF) L += ex2(a.sink[h] * kLog2e - M);
    const float out = (M == SA_NEG_INF || L == 0.f) ? 0.f : acc / L;
    static_cast<T*>(a.y)[((cui.b * a.Hq + h) * a.Sq + cui.i) * D + d] = from_f32<T>(out);
  };

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
    const bool val_unit = do_val && (a.I != 1 || cui.kvh == 0);
    const int64_t irow = (cui.b * a.I + cui.ih) * a.Sq + cui.i;
    const bool whole = cur.off >= t_begin && cur.off + cur.tu <= t_end;
    if (whole) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int hh = nt * 8 + 2 * tig + j;
          if (hh >= a.hpu) continue;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            store_y(hh, mt * 16 + gid, m_run[nt][j], lsum[nt][j], o[mt][nt][j]);
            store_y(hh, mt * 16 + gid + 8, m_run[nt][j], lsum[nt][j], o[mt][nt][2 + j]);
          }
        }
      if (val_unit && lane == 0) finish_validation(a, irow);
      return;
    }
    const int slot = (first.u == cur.u) ? 0 : 1;
    const int64_t pbase = (gw * 2 + slot) * a.hpu;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int hh = nt * 8 + 2 * tig + j;
        if (hh >= a.hpu) continue;
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
    __threadfence();
    __syncwarp();
    const int64_t w_lo = cur.off / R;
    const int64_t w_hi = (cur.off + cur.tu - 1) / R;
    unsigned int prev = 0;
    if (lane == 0) prev = atomicAdd(a.ticket + cur.u, 1u);
    prev = __shfl_sync(0xffffffffu, prev, 0);
    if (prev != static_cast<unsigned int>(w_hi - w_lo)) return;  // not the last warp
    __threadfence();
    // Last warp of the unit: merge every contributing warp's partial in warp
    // order.  (1) lane hh: M = max_w m_w and L = sum_w l_w 2^(m_w - M) of head
    // hh; (2) each lane accumulates float4 groups of the outputs over warps,
    // eight groups at a time, with all loads of one warp's partial in flight.
    float Mh = SA_NEG_INF, Lh = 0.f;
    if (lane < a.hpu) {
      for (int64_t w = w_lo; w <= w_hi; ++w) {
        const int sl = (unit_of_tile(a, pref, w * R).u == cur.u) ? 0 : 1;
        Mh = fmaxf(Mh, __ldcg(a.part_ml + 2 * ((w * 2 + sl) * a.hpu + lane)));
      }
      if (Mh != SA_NEG_INF) {
        for (int64_t w = w_lo; w <= w_hi; ++w) {
          const int sl = (unit_of_tile(a, pref, w * R).u == cur.u) ? 0 : 1;
          const float2 ml =
              __ldcg(reinterpret_cast<const float2*>(a.part_ml) + (w * 2 + sl) * a.hpu + lane);
          if (ml.x != SA_NEG_INF) Lh += ml.y * ex2(ml.x - Mh);
        }
        if (a.sink) Lh += ex2(a.sink[cui.h0 + lane] * kLog2e - Mh);
      }
    }
    const int64_t groups = a.hpu * D / 4;
    for (int64_t g0 = 0; g0 < groups; g0 += 32 * 8) {
      float4 acc[8];
      int hk[8];
      float Mk[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int64_t g = g0 + lane + 32 * k;
        hk[k] = g < groups ? static_cast<int>((g * 4) / D) : 0;
        Mk[k] = __shfl_sync(0xffffffffu, Mh, hk[k]);
        acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int64_t w = w_lo; w <= w_hi; ++w) {
        const int sl = (unit_of_tile(a, pref, w * R).u == cur.u) ? 0 : 1;
        const int64_t base = (w * 2 + sl) * a.hpu;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int64_t g = g0 + lane + 32 * k;
          if (g < groups) {
            const float m = __ldcg(a.part_ml + 2 * (base + hk[k]));
            const float4 v = __ldcg(reinterpret_cast<const float4*>(
                a.part_o + (base + hk[k]) * D + (g * 4) % D));
            const float f = (m == SA_NEG_INF) ? 0.f : ex2(m - Mk[k]);
            acc[k].x += v.x * f;
            acc[k].y += v.y * f;
            acc[k].z += v.z * f;
            acc[k].w += v.w * f;
          }
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int64_t g = g0 + lane + 32 * k;
        const float L = __shfl_sync(0xffffffffu, Lh, hk[k]);
        if (g < groups) {
          const float inv = (Mk[k] == SA_NEG_INF || L == 0.f) ? 0.f : 1.0f / L;
          const int64_t h = cui.h0 + hk[k];
          T* yp = static_cast<T*>(a.y) + ((cui.b * a.Hq + h) * a.Sq + cui.i) * D + (g * 4) % D;
          yp[0] = from_f32<T>(acc[k].x * inv);
          yp[1] = from_f32<T>(acc[k].y * inv);
          yp[2] = from_f32<T>(acc[k].z * inv);
          yp[3] = from_f32<T>(acc[k].w * inv);
        }
      }
    }
    if (lane == 0) {
      a.ticket[cur.u] = 0u;
      if (val_unit) finish_validation(a, irow);
    }
  };

  // ---- main loop ------------------------------------------------------------------
  for (int64_t t = t_begin; t < t_end; ++t) {
    __syncwarp();  // every lane is past the reads of the slot refilled below
    if (t + G::kStages - 1 < t_end) issue(t + G::kStages - 1);
    cp_async_commit();
    cp_async_wait<G::kStages - 1>();
    __syncwarp();
    if (t >= cur.off + cur.tu || cur.u < 0) {
      if (cur.u >= 0) flush_unit();
      start_unit(unit_of_tile(a, pref, t));
    }
    const int slot = static_cast<int>((t - t_begin) % G::kStages);
    const uint32_t mask = smask[slot];
    if (mask == 0u) continue;
    const bool v_lo = (mask >> gid) & 1u, v_hi = (mask >> (gid + 8)) & 1u;
    const uint32_t kt = ring_s + slot * G::kTileBytes;
    const uint32_t vt = kt + 16 * G::kRowBytes;
    // S^T = K . Q^T
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
    {
      const int r = lane & 15;
      const uint32_t rbase = kt + r * G::kRowBytes;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        const int chn = (kk * 2 + (lane >> 4)) ^ (r & 7);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(rbase + (chn << 4), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma16816<T>(s[nt], a0, a1, a2, a3, qf[nt][kk][0], qf[nt][kk][1]);
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
      const int r = (lane & 7) + ((lane >> 4) << 3);
      const uint32_t rbase = vt + r * G::kRowBytes;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int chn = (mt * 2 + ((lane >> 3) & 1)) ^ (r & 7);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(rbase + (chn << 4), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma16816<T>(o[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
      }
    }
  }
  cp_async_wait<0>();
  if (cur.u >= 0) flush_unit();
}

template <typename T, int D, int NT>
static int launch_stream_t(const GatherArgs& a, int grid, size_t smem, cudaStream_t st) {
  if (cudaFuncSetAttribute(gather_stream_kernel<T, D, NT>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return -1;
  gather_stream_kernel<T, D, NT><<<grid, SGeo<D>::kWarps * 32, smem, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_gather_stream(const GatherArgs& a, int dtype, int grid, cudaStream_t st) {
  const size_t smem = stream_smem_bytes(static_cast<int>(a.D), a.source, a.B);
  const bool two = a.hpu > 8;
  if (dtype == SA_BF16) {
    if (a.D == 64) return two ? launch_stream_t<__nv_bfloat16, 64, 2>(a, grid, smem, st)
                              : launch_stream_t<__nv_bfloat16, 64, 1>(a, grid, smem, st);
    if (a.D == 128) return two ? launch_stream_t<__nv_bfloat16, 128, 2>(a, grid, smem, st)
                               : launch_stream_t<__nv_bfloat16, 128, 1>(a, grid, smem, st);
    return launch_stream_t<__nv_bfloat16, 256, 1>(a, grid, smem, st);
  }
  if (a.D == 64) return two ? launch_stream_t<__half, 64, 2>(a, grid, smem, st)
                            : launch_stream_t<__half, 64, 1>(a, grid, smem, st);
  if (a.D == 128) return two ? launch_stream_t<__half, 128, 2>(a, grid, smem, st)
                             : launch_stream_t<__half, 128, 1>(a, grid, smem, st);
  return launch_stream_t<__half, 256, 1>(a, grid, smem, st);
}

}  // namespace sa
