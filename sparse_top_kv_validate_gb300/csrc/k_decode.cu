// k_decode.cu -- split-K gather decode over a KV cache (selected tokens or
// a page table), and the fixed-order combine of the split partials.
//
// Semantics: IndexShare `index_share_row` (onnx-runtime-ep-cuda
// src/kernels/index_share.rs) -- gather the valid prefix of a row's selected
// indices, scaled QK scores, a stable fp32 softmax in which a fully-masked row
// gives 0, probs . V; ONNX Attention `attention_split` / `attention_combine`
// (standard_attention.rs) -- FlashDecoding: each split of the keys yields
// (max, sum, unnormalised P.V) and a log-sum-exp combine merges the splits in
// a fixed order; paged addressing as in ferrum-kernels causal_attention.rs
// (16-token blocks through a table).
//
// GB300 design (not the pages' row-per-block kernel):
//  * A work unit is (batch, KV head or index head, query), serving every query
//    head that shares its index row and KV head, so each gathered K/V row is
//    read from HBM once for the whole GQA group.  Units are cut into splits of
//    `chunk` candidates (one CTA each).
//  * Candidate -> cache-row resolution (index row, window, masks, page table)
//    happens once per CTA into shared memory.
//  * K and V rows are fetched by bulk async copies (one 16-byte-aligned row per
//    copy, completion counted on an mbarrier) into a 3-deep ring of 64-key
//    stages; rows are padded by 16 bytes so ldmatrix reads are conflict-free.
//  * Each warp owns 16 keys of a stage and runs the tensor-core m16n8k16 MMA
//    with KEYS as the M dimension: S^T = K . Q^T (heads as N, so a GQA group of
//    8 fills N exactly), then O^T += V^T . P^T where P^T is produced from the
//    S^T accumulator by an in-register 8x8 transpose (movmatrix).  The online
//    softmax state of a head lives in the same lanes as its O^T columns, so
//    rescaling is thread-local.
//  * Warps merge in shared memory in warp order; splits merge in split order.
//    Results are deterministic run to run.
#include "common.cuh"
#include "kernels.h"

namespace sa {

// ---------------------------------------------------------------------------
// unit / candidate resolution (shared by the tensor-core and SIMT kernels)
// ---------------------------------------------------------------------------

struct UnitInfo {
  int64_t b, i, kvh, h0, ih;
};

__device__ __forceinline__ UnitInfo unit_info(const GatherArgs& a, int64_t unit) {
  UnitInfo u;
  u.i = unit % a.Sq;
  const int64_t r = unit / a.Sq;
  const int64_t grp = r % a.n_groups;
  u.b = r / a.n_groups;
  if (a.n_groups == a.Hkv) {  // one unit per KV head: the whole GQA group
    u.kvh = grp;
    u.h0 = grp * a.g;
  } else {                    // one unit per query head
    u.kvh = grp / a.g;
    u.h0 = grp;
  }
  u.ih = (a.I == 1) ? 0 : (a.I == a.Hkv ? u.kvh : u.h0);
  return u;
}

// Number of candidates of this unit (the per-batch context for paged units).
__device__ __forceinline__ int64_t unit_candidates(const GatherArgs& a, const UnitInfo& u) {
  if (a.source == kPaged) {
    int64_t ctx = a.ctx_len[u.b];
    const int64_t cap = a.max_pages * a.page_tokens;
    if (ctx < 1 || ctx > cap) return 0;
    return ctx;
  }
  return a.n_cand;
}

// Candidate c of the unit -> cache row id (row of D elements in k/v), or -1
// when the candidate is masked or absent.  Never returns an out-of-bounds row.
__device__ __forceinline__ int32_t resolve_candidate(const GatherArgs& a, const UnitInfo& u,
                                                     int64_t c) {
  if (a.source == kPaged) {
    const int64_t ctx = a.ctx_len[u.b];
    if (c >= ctx) return -1;
    const int32_t page = a.block_table[u.b * a.max_pages + c / a.page_tokens];
    if (page < 0 || page >= a.num_pages) {
      if (a.err_word) atomicOr(a.err_word, SA_ERRBIT_PAGE);
      return -1;
    }
    return static_cast<int32_t>((static_cast<int64_t>(page) * a.Hkv + u.kvh) * a.page_tokens +
                                c % a.page_tokens);
  }
  if (a.source == kDense) {
    if (a.causal && c > a.past_len + u.i) return -1;
    return static_cast<int32_t>((u.b * a.Hkv + u.kvh) * a.T + c);
  }
  int64_t len = a.kv_len ? a.kv_len[u.b] : a.T;
  if (len > a.T) len = a.T;
  const int64_t wstart = len - a.window;
  int64_t t;
  if (c < a.window) {
    t = wstart + c;
    if (t < 0) return -1;
  } else {
    const int64_t off = ((u.b * a.I + u.ih) * a.Sq + u.i) * a.K + (c - a.window);
    t = load_index(a.idx, off, a.idx_is_i64);
    if (t < 0 || t >= len) return -1;
    if (a.window > 0 && t >= wstart) return -1;  // already in the window
  }
  if (a.causal && t > a.past_len + u.i) return -1;
  return static_cast<int32_t>((u.b * a.Hkv + u.kvh) * a.T + t);
}

// ---------------------------------------------------------------------------
// tensor-core gather kernel (f16 / bf16 storage)
// ---------------------------------------------------------------------------

template <int D>
struct MmaCfg {
  static constexpr int kWarps = 4;
  static constexpr int kStageKeys = 16 * kWarps;
  static constexpr int kStages = 3;
  static constexpr int kRowBytes = D * 2;
  static constexpr int kRowStride = kRowBytes + 16;  // breaks ldmatrix bank conflicts
  static constexpr int kStageBytes = 2 * kStageKeys * kRowStride;
  static constexpr int kRingBytes = kStages * kStageBytes;
};

template <int D, int NT>
constexpr size_t mma_smem_bytes(int64_t chunk) {
  using Cfg = MmaCfg<D>;
  size_t merge = static_cast<size_t>(Cfg::kWarps) * (NT * 8) * (D + 2) * 4;
  size_t ring = Cfg::kRingBytes > merge ? Cfg::kRingBytes : merge;
  return ring + static_cast<size_t>(chunk) * 4 + Cfg::kStages * 8 + 16;
}

template <typename T, int D, int NT>
__global__ void __launch_bounds__(128) gather_mma_kernel(GatherArgs a) {
  using Cfg = MmaCfg<D>;
  constexpr int KS = D / 16;  // k-steps of the QK product, m-tiles of PV
  extern __shared__ __align__(128) unsigned char smem[];
  const int64_t split = blockIdx.x % a.splits;
  const int64_t unit = blockIdx.x / a.splits;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;

  size_t merge_bytes = static_cast<size_t>(Cfg::kWarps) * (NT * 8) * (D + 2) * 4;
  size_t ring_bytes = Cfg::kRingBytes > merge_bytes ? Cfg::kRingBytes : merge_bytes;
  int32_t* kpos = reinterpret_cast<int32_t*>(smem + ring_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ring_bytes + a.chunk * 4);

  const UnitInfo u = unit_info(a, unit);
  const int64_t n_cand = unit_candidates(a, u);
  const int64_t c0 = split * a.chunk;
  int64_t n_local = n_cand - c0;
  if (n_local > a.chunk) n_local = a.chunk;
  if (n_local < 0) n_local = 0;

  // Resolve this split's candidates to cache rows.
  for (int64_t c = tid; c < n_local; c += blockDim.x) kpos[c] = resolve_candidate(a, u, c0 + c);
  if (tid < Cfg::kStages) mbar_init(&bars[tid], 1);
  // Zero the V rows of the ring once: a masked key's slot is never copied
  // into, and its probability is 0, so its V row must hold finite values.
  for (int s = 0; s < Cfg::kStages; ++s) {
    uint4* vz = reinterpret_cast<uint4*>(smem + s * Cfg::kStageBytes +
                                         Cfg::kStageKeys * Cfg::kRowStride);
    for (int e = tid; e < Cfg::kStageKeys * Cfg::kRowStride / 16; e += blockDim.x)
      vz[e] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  fence_mbar_init();
  __syncthreads();

  const int n_stages = static_cast<int>((n_local + Cfg::kStageKeys - 1) / Cfg::kStageKeys);
  const char* kbase = static_cast<const char*>(a.k);
  const char* vbase = static_cast<const char*>(a.v);

  auto issue = [&](int st) {
    // warp 0 only
    const int buf = st % Cfg::kStages;
    unsigned char* kb = smem + buf * Cfg::kStageBytes;
    unsigned char* vb = kb + Cfg::kStageKeys * Cfg::kRowStride;
    const int64_t cbase = static_cast<int64_t>(st) * Cfg::kStageKeys;
    const int32_t r0 = (cbase + lane < n_local) ? kpos[cbase + lane] : -1;
    const int32_t r1 = (cbase + lane + 32 < n_local) ? kpos[cbase + lane + 32] : -1;
    const uint32_t n = __popc(__ballot_sync(0xffffffffu, r0 >= 0)) +
                       __popc(__ballot_sync(0xffffffffu, r1 >= 0));
    if (lane == 0) mbar_arrive_expect_tx(&bars[buf], n * 2u * Cfg::kRowBytes);
    __syncwarp();
    if (r0 >= 0) {
      bulk_g2s(kb + lane * Cfg::kRowStride, kbase + static_cast<int64_t>(r0) * Cfg::kRowBytes,
               Cfg::kRowBytes, &bars[buf]);
      bulk_g2s(vb + lane * Cfg::kRowStride, vbase + static_cast<int64_t>(r0) * Cfg::kRowBytes,
               Cfg::kRowBytes, &bars[buf]);
    }
    if (r1 >= 0) {
      bulk_g2s(kb + (lane + 32) * Cfg::kRowStride,
               kbase + static_cast<int64_t>(r1) * Cfg::kRowBytes, Cfg::kRowBytes, &bars[buf]);
      bulk_g2s(vb + (lane + 32) * Cfg::kRowStride,
               vbase + static_cast<int64_t>(r1) * Cfg::kRowBytes, Cfg::kRowBytes, &bars[buf]);
    }
  };

  if (warp == 0) {
    for (int st = 0; st < Cfg::kStages - 1 && st < n_stages; ++st) issue(st);
  }

  // Q^T as B fragments: b0 = Q[head gid][2tig..2tig+1], b1 = +8 dims.
  uint32_t qf[NT][KS][2];
  {
    const T* qp = static_cast<const T*>(a.q);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int hh = nt * 8 + gid;
      const bool live = hh < a.hpu;
      const int64_t qoff = ((u.b * a.Hq + (u.h0 + (live ? hh : 0))) * a.Sq + u.i) * D;
      const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qp + qoff);
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        qf[nt][kk][0] = live ? q32[(kk * 16 + 2 * tig) / 2] : 0u;
        qf[nt][kk][1] = live ? q32[(kk * 16 + 2 * tig + 8) / 2] : 0u;
      }
    }
  }

  float o[KS][NT][4];
#pragma unroll
  for (int mt = 0; mt < KS; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
  float m_run[NT][2], l_run[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = SA_NEG_INF;
    l_run[nt][0] = l_run[nt][1] = 0.f;
  }
  bool timed_out = false;
  const float sl2 = a.scale_log2;
  const float cap = a.softcap, inv_cap = a.inv_softcap;

  for (int st = 0; st < n_stages; ++st) {
    if (warp == 0 && st + Cfg::kStages - 1 < n_stages) issue(st + Cfg::kStages - 1);
    const int buf = st % Cfg::kStages;
    if (!mbar_wait(&bars[buf], static_cast<uint32_t>((st / Cfg::kStages) & 1))) timed_out = true;
    const unsigned char* kb = smem + buf * Cfg::kStageBytes;
    const unsigned char* vb = kb + Cfg::kStageKeys * Cfg::kRowStride;
    const int64_t cw = static_cast<int64_t>(st) * Cfg::kStageKeys + warp * 16;
    const bool v_lo = (cw + gid < n_local) && kpos[cw + gid] >= 0;
    const bool v_hi = (cw + gid + 8 < n_local) && kpos[cw + gid + 8] >= 0;
    if (__any_sync(0xffffffffu, v_lo || v_hi)) {
      // ---- S^T = K . Q^T over this warp's 16 keys -----------------------------
      float s[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
      const uint32_t ka = smem_u32(kb) + (warp * 16 + (lane & 15)) * Cfg::kRowStride +
                          (lane >> 4) * 16;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(ka + kk * 32, a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816<T>(s[nt], a0, a1, a2, a3, qf[nt][kk][0], qf[nt][kk][1]);
      }
      // ---- scale / softcap / mask, online softmax (log2 domain) ----------------
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
      // ---- O^T += V^T . P^T ------------------------------------------------------
      const uint32_t va = smem_u32(vb) +
                          (warp * 16 + (lane & 7) + ((lane >> 4) << 3)) * Cfg::kRowStride +
                          ((lane >> 3) & 1) * 16;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(va + mt * 32, a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816<T>(o[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
      }
    }
    __syncthreads();  // everyone is done with `buf` before it is refilled
  }
  if (timed_out && a.err_word) atomicOr(a.err_word, SA_ERRBIT_TIMEOUT);

  // ---- merge the warps (fixed warp order) ---------------------------------------
  constexpr int HP = NT * 8;
  float* sm_o = reinterpret_cast<float*>(smem);                     // [warps][HP][D]
  float* sm_m = sm_o + Cfg::kWarps * HP * D;                          // [warps][HP]
  float* sm_l = sm_m + Cfg::kWarps * HP;                              // [warps][HP]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float l = l_run[nt][j];
#pragma unroll
      for (int sh = 4; sh < 32; sh <<= 1) l += __shfl_xor_sync(0xffffffffu, l, sh);
      const int hh = nt * 8 + 2 * tig + j;
      if (gid == 0) {
        sm_m[warp * HP + hh] = m_run[nt][j];
        sm_l[warp * HP + hh] = l;
      }
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        sm_o[(warp * HP + hh) * D + mt * 16 + gid] = o[mt][nt][j];
        sm_o[(warp * HP + hh) * D + mt * 16 + gid + 8] = o[mt][nt][2 + j];
      }
    }
  }
  __syncthreads();

  const int64_t hpu = a.hpu;
  for (int64_t e = tid; e < hpu * D; e += blockDim.x) {
    const int hh = static_cast<int>(e / D);
    const int d = static_cast<int>(e % D);
    float M = SA_NEG_INF;
#pragma unroll
    for (int w = 0; w < Cfg::kWarps; ++w) M = fmaxf(M, sm_m[w * HP + hh]);
    float L = 0.f, acc = 0.f;
    if (M != SA_NEG_INF) {
#pragma unroll
      for (int w = 0; w < Cfg::kWarps; ++w) {
        const float f = ex2(sm_m[w * HP + hh] - M);
        L += sm_l[w * HP + hh] * f;
        acc += sm_o[(w * HP + hh) * D + d] * f;
      }
    }
    const int64_t h = u.h0 + hh;
    if (a.splits == 1) {
      if (a.sink && M != SA_NEG_INF) L += ex2(a.sink[h] * kLog2e - M);
      const float out = (M == SA_NEG_INF || L == 0.f) ? 0.f : acc / L;
      static_cast<T*>(a.y)[((u.b * a.Hq + h) * a.Sq + u.i) * D + d] = from_f32<T>(out);
    } else {
      const int64_t pidx = (unit * a.splits + split) * hpu + hh;
      a.part_o[pidx * D + d] = acc;
      if (d == 0) {
        a.part_ml[2 * pidx] = M;
        a.part_ml[2 * pidx + 1] = L;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// SIMT gather kernel (fp32 storage, or shapes the tensor-core kernel skips)
// ---------------------------------------------------------------------------
// One CTA per (unit, head, split); warps stride over candidates; lanes hold
// DPL dims each (d = lane + 32 * k).  fp32 FMA throughout.

template <typename T, int DPL>
__global__ void __launch_bounds__(128) gather_simt_kernel(GatherArgs a) {
  __shared__ float sm_o[4][DPL * 32];
  __shared__ float sm_ml[4][2];
  const int64_t split = blockIdx.x % a.splits;
  const int64_t rest = blockIdx.x / a.splits;
  const int64_t hh = rest % a.hpu;
  const int64_t unit = rest / a.hpu;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const UnitInfo u = unit_info(a, unit);
  const int64_t h = u.h0 + hh;
  const int64_t D = a.D;
  const int64_t n_cand = unit_candidates(a, u);
  const int64_t c0 = split * a.chunk;
  int64_t c1 = c0 + a.chunk;
  if (c1 > n_cand) c1 = n_cand;

  const T* qp = static_cast<const T*>(a.q) + ((u.b * a.Hq + h) * a.Sq + u.i) * D;
  float q[DPL], o[DPL];
#pragma unroll
  for (int k = 0; k < DPL; ++k) {
    const int64_t d = lane + 32 * k;
    q[k] = d < D ? to_f32<T>(qp[d]) : 0.f;
    o[k] = 0.f;
  }
  float m = SA_NEG_INF, l = 0.f;
  const T* kp = static_cast<const T*>(a.k);
  const T* vp = static_cast<const T*>(a.v);
  const float sl2 = a.scale_log2;
  for (int64_t c = c0 + warp; c < c1; c += 4) {
    const int32_t row = resolve_candidate(a, u, c);
    if (row < 0) continue;
    const T* kr = kp + static_cast<int64_t>(row) * D;
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k < DPL; ++k) {
      const int64_t d = lane + 32 * k;
      if (d < D) dot = fmaf(q[k], to_f32<T>(kr[d]), dot);
    }
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, sh);
    float x;
    if (a.softcap != 0.f) x = a.softcap * tanhf(dot * (sl2 / kLog2e) * a.inv_softcap) * kLog2e;
    else x = dot * sl2;
    const float mn = fmaxf(m, x);
    const float al = exp2f(m - mn);  // m == -inf -> 0
    const float p = exp2f(x - mn);
    l = l * al + p;
    const T* vr = vp + static_cast<int64_t>(row) * D;
#pragma unroll
    for (int k = 0; k < DPL; ++k) {
      const int64_t d = lane + 32 * k;
      o[k] = o[k] * al + (d < D ? p * to_f32<T>(vr[d]) : 0.f);
    }
    m = mn;
  }
#pragma unroll
  for (int k = 0; k < DPL; ++k) sm_o[warp][lane + 32 * k] = o[k];
  if (lane == 0) {
    sm_ml[warp][0] = m;
    sm_ml[warp][1] = l;
  }
  __syncthreads();
  if (warp != 0) return;
  float M = SA_NEG_INF;
  for (int w = 0; w < 4; ++w) M = fmaxf(M, sm_ml[w][0]);
  float L = 0.f;
  float f[4];
  for (int w = 0; w < 4; ++w) {
    f[w] = (M == SA_NEG_INF) ? 0.f : exp2f(sm_ml[w][0] - M);
    L += sm_ml[w][1] * f[w];
  }
  for (int k = 0; k < DPL; ++k) {
    const int64_t d = lane + 32 * k;
    if (d >= D) continue;
    float acc = 0.f;
    for (int w = 0; w < 4; ++w) acc += sm_o[w][lane + 32 * k] * f[w];
    if (a.splits == 1) {
      float LL = L;
      if (a.sink && M != SA_NEG_INF) LL += exp2f(a.sink[h] * kLog2e - M);
      const float out = (M == SA_NEG_INF || LL == 0.f) ? 0.f : acc / LL;
      static_cast<T*>(a.y)[((u.b * a.Hq + h) * a.Sq + u.i) * D + d] = from_f32<T>(out);
    } else {
      const int64_t pidx = (unit * a.splits + split) * a.hpu + hh;
      a.part_o[pidx * D + d] = acc;
      if (d == 0) {
        a.part_ml[2 * pidx] = M;
        a.part_ml[2 * pidx + 1] = L;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// combine: y = sum_s o_s 2^(m_s - M) / (sum_s l_s 2^(m_s - M) [+ sink term])
// ---------------------------------------------------------------------------

template <typename T>
__global__ void __launch_bounds__(128) combine_kernel(GatherArgs a) {
  const int64_t hh = blockIdx.x % a.hpu;
  const int64_t unit = blockIdx.x / a.hpu;
  const UnitInfo u = unit_info(a, unit);
  const int64_t h = u.h0 + hh;
  const int64_t D = a.Dv;
  const float* ml = a.part_ml + (unit * a.splits * a.hpu + hh) * 2;
  const int64_t mstride = a.hpu * 2;
  float M = SA_NEG_INF;
  for (int64_t s = 0; s < a.splits; ++s) M = fmaxf(M, ml[s * mstride]);
  float L = 0.f;
  if (M != SA_NEG_INF) {
    for (int64_t s = 0; s < a.splits; ++s) {
      const float ms = ml[s * mstride];
      if (ms != SA_NEG_INF) L += ml[s * mstride + 1] * ex2(ms - M);
    }
    if (a.sink) L += ex2(a.sink[h] * kLog2e - M);
  }
  const float inv = (M == SA_NEG_INF || L == 0.f) ? 0.f : 1.0f / L;
  T* yp = static_cast<T*>(a.y) + ((u.b * a.Hq + h) * a.Sq + u.i) * D;
  for (int64_t d = threadIdx.x; d < D; d += blockDim.x) {
    float acc = 0.f;
    if (M != SA_NEG_INF) {
      for (int64_t s = 0; s < a.splits; ++s) {
        const float ms = ml[s * mstride];
        if (ms == SA_NEG_INF) continue;
        acc += a.part_o[((unit * a.splits + s) * a.hpu + hh) * D + d] * ex2(ms - M);
      }
    }
    yp[d] = from_f32<T>(acc * inv);
  }
}

// ---------------------------------------------------------------------------
// paged: write the new token's K/V into the pool at token ctx - 1
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) paged_append_kernel(PagedAppendArgs a) {
  const int64_t row_bytes = a.D * a.esz;
  const int64_t n = a.B * a.Hkv * row_bytes;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t byte = e % row_bytes;
    const int64_t bh = e / row_bytes;
    const int64_t b = bh / a.Hkv, h = bh % a.Hkv;
    const int64_t ctx = a.ctx_len[b];
    if (ctx < 1 || ctx > a.max_pages * a.page_tokens) {
      if (byte == 0 && h == 0 && a.err_word) atomicOr(a.err_word, SA_ERRBIT_PAGE);
      continue;
    }
    const int64_t t = ctx - 1;
    const int32_t page = a.block_table[b * a.max_pages + t / a.page_tokens];
    if (page < 0 || page >= a.num_pages) {
      if (byte == 0 && h == 0 && a.err_word) atomicOr(a.err_word, SA_ERRBIT_PAGE);
      continue;
    }
    const int64_t dst = ((static_cast<int64_t>(page) * a.Hkv + h) * a.page_tokens +
                         t % a.page_tokens) * row_bytes + byte;
    const int64_t src = bh * row_bytes + byte;
    if (a.k_new)
      static_cast<unsigned char*>(a.k_pool)[dst] = static_cast<const unsigned char*>(a.k_new)[src];
    if (a.v_new)
      static_cast<unsigned char*>(a.v_pool)[dst] = static_cast<const unsigned char*>(a.v_new)[src];
  }
}

int launch_paged_append(const PagedAppendArgs& a, cudaStream_t st) {
  const int64_t n = a.B * a.Hkv * a.D * a.esz;
  if (n == 0) return 0;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  paged_append_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

template <typename T, int D, int NT>
static int launch_mma(const GatherArgs& a, cudaStream_t st) {
  const size_t smem = mma_smem_bytes<D, NT>(a.chunk);
  if (cudaFuncSetAttribute(gather_mma_kernel<T, D, NT>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(227 * 1024)) != cudaSuccess)
    return -1;
  const int64_t grid = a.units * a.splits;
  gather_mma_kernel<T, D, NT><<<static_cast<unsigned>(grid), 128, smem, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

template <typename T, int DPL>
static int launch_simt(const GatherArgs& a, cudaStream_t st) {
  const int64_t grid = a.units * a.hpu * a.splits;
  gather_simt_kernel<T, DPL><<<static_cast<unsigned>(grid), 128, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

template <typename T>
static int launch_simt_any(const GatherArgs& a, cudaStream_t st) {
  const int64_t dpl = (a.D + 31) / 32;
  if (dpl <= 1) return launch_simt<T, 1>(a, st);
  if (dpl <= 2) return launch_simt<T, 2>(a, st);
  if (dpl <= 4) return launch_simt<T, 4>(a, st);
  if (dpl <= 8) return launch_simt<T, 8>(a, st);
  if (dpl <= 16) return launch_simt<T, 16>(a, st);
  return -2;
}

template <typename T, int D, int NT>
static int occ_mma(const GatherArgs& a) {
  if (cudaFuncSetAttribute(gather_mma_kernel<T, D, NT>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(227 * 1024)) != cudaSuccess)
    return 1;
  int n = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gather_mma_kernel<T, D, NT>, 128,
                                                    mma_smem_bytes<D, NT>(a.chunk)) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

int gather_mma_occupancy(const GatherArgs& a, int dtype) {
  const bool two = a.hpu > 8;
  if (dtype == SA_BF16) {
    if (a.D == 64) return two ? occ_mma<__nv_bfloat16, 64, 2>(a) : occ_mma<__nv_bfloat16, 64, 1>(a);
    if (a.D == 128) return two ? occ_mma<__nv_bfloat16, 128, 2>(a) : occ_mma<__nv_bfloat16, 128, 1>(a);
    return occ_mma<__nv_bfloat16, 256, 1>(a);
  }
  if (a.D == 64) return two ? occ_mma<__half, 64, 2>(a) : occ_mma<__half, 64, 1>(a);
  if (a.D == 128) return two ? occ_mma<__half, 128, 2>(a) : occ_mma<__half, 128, 1>(a);
  return occ_mma<__half, 256, 1>(a);
}

// Whether the tensor-core kernel serves this request (mirrors the host plan).
bool gather_uses_mma(const GatherArgs& a, int dtype) {
  if (dtype != SA_F16 && dtype != SA_BF16) return false;
  if (!(a.D == 64 || a.D == 128 || a.D == 256)) return false;
  if (a.hpu > 16) return false;
  if (a.D == 256 && a.hpu > 8) return false;
  return true;
}

int launch_gather_decode(const GatherArgs& a, int dtype, cudaStream_t st) {
  if (a.units == 0) return 0;
  if (gather_uses_mma(a, dtype)) {
    const bool two = a.hpu > 8;
    if (dtype == SA_BF16) {
      if (a.D == 64) return two ? launch_mma<__nv_bfloat16, 64, 2>(a, st) : launch_mma<__nv_bfloat16, 64, 1>(a, st);
      if (a.D == 128) return two ? launch_mma<__nv_bfloat16, 128, 2>(a, st) : launch_mma<__nv_bfloat16, 128, 1>(a, st);
      return launch_mma<__nv_bfloat16, 256, 1>(a, st);
    }
    if (a.D == 64) return two ? launch_mma<__half, 64, 2>(a, st) : launch_mma<__half, 64, 1>(a, st);
    if (a.D == 128) return two ? launch_mma<__half, 128, 2>(a, st) : launch_mma<__half, 128, 1>(a, st);
    return launch_mma<__half, 256, 1>(a, st);
  }
  if (dtype == SA_F32) return launch_simt_any<float>(a, st);
  if (dtype == SA_F16) return launch_simt_any<__half>(a, st);
  if (dtype == SA_BF16) return launch_simt_any<__nv_bfloat16>(a, st);
  return -2;
}

int launch_combine(const GatherArgs& a, int dtype, cudaStream_t st) {
  if (a.splits <= 1 || a.units == 0) return 0;
  const unsigned grid = static_cast<unsigned>(a.units * a.hpu);
  if (dtype == SA_F32) combine_kernel<float><<<grid, 128, 0, st>>>(a);
  else if (dtype == SA_F16) combine_kernel<__half><<<grid, 128, 0, st>>>(a);
  else combine_kernel<__nv_bfloat16><<<grid, 128, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace sa
